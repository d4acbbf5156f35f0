// layout.cpp -- layout descriptor: validation and derived sizes (host only).
//
// Rules follow the review "BASP: Communication-Efficient Batch-Aware Sequence
// Parallelism for LLM Training" (evolve.pub): "Summary" (N = K*B ranks in B
// disjoint contiguous groups of K, peers drop from N-1 to K-1, B*S/N tokens
// per GPU), "Strengths" (the G-group form with B/G sequences per group) and
// FAQ "What are BASP's main limitations?" (N a multiple of B, heads divisible
// across group members, data parallelism when B > N).
#include <cstdlib>
#include <initializer_list>
#include <new>

#include "layout_internal.h"

namespace {

bool mul_ok(int64_t a, int64_t b, int64_t *out) {
    return !__builtin_mul_overflow(a, b, out);
}

}  // namespace

extern "C" basp_status basp_layout_create(int64_t B, int64_t S, int64_t Hq,
                                          int64_t Hkv, int64_t d, int64_t N,
                                          int64_t K, basp_dtype dtype,
                                          basp_layout **out) {
    const basp_layout_desc desc = {B, S, Hq, Hkv, d, N, K, dtype, BASP_ORDER_BSHD};
    return basp_layout_create_ex(&desc, out);
}

extern "C" basp_status basp_layout_create_ex(const basp_layout_desc *desc,
                                             basp_layout **out) {
    if (out == nullptr) return BASP_ERR_INVALID_ARG;
    *out = nullptr;
    if (desc == nullptr) return BASP_ERR_INVALID_ARG;
    int64_t B = desc->B, S = desc->S, Hq = desc->Hq, Hkv = desc->Hkv;
    int64_t d = desc->d, N = desc->N, K = desc->K;
    const basp_dtype dtype = desc->dtype;
    if (desc->order != BASP_ORDER_BSHD && desc->order != BASP_ORDER_SBHD)
        return BASP_ERR_INVALID_ARG;
    int64_t esz;
    switch (dtype) {
        case BASP_DTYPE_BF16: esz = 2; break;
        case BASP_DTYPE_FP16: esz = 2; break;
        case BASP_DTYPE_FP8: esz = 1; break;
        case BASP_DTYPE_FP32: esz = 4; break;
        default: return BASP_ERR_INVALID_ARG;
    }
    if (B < 0 || S < 0 || Hq < 1 || Hkv < 1 || d < 1 || N < 1 || K < 0)
        return BASP_ERR_INVALID_ARG;
    if (K == 0) {                       // the BASP rule: K = N / B
        if (B < 1) return BASP_ERR_INVALID_ARG;
        if (B > N) return BASP_ERR_BATCH_GT_RANKS;
        if (N % B != 0) return BASP_ERR_DIVISIBILITY;
        K = N / B;
    }
    if (N % K != 0) return BASP_ERR_DIVISIBILITY;
    const int64_t G = N / K;
    if (B % G != 0 || S % K != 0 || Hq % K != 0 || Hkv % K != 0)
        return BASP_ERR_DIVISIBILITY;

    // Every byte offset must fit comfortably in int64 (checked once here so
    // the planners and kernels can multiply freely).
    const int64_t H = Hq + 2 * Hkv;                     // packed QKV row
    int64_t t = 1;
    for (int64_t f : {B, S, H, d, esz, int64_t(4)}) {   // 4: send+recv, in+out
        if (!mul_ok(t, f, &t)) return BASP_ERR_TOO_LARGE;
    }
    if (t > (int64_t(1) << 60)) return BASP_ERR_TOO_LARGE;

    basp_layout *L = new (std::nothrow) basp_layout;
    if (L == nullptr) return BASP_ERR_INVALID_ARG;
    L->B = B; L->S = S; L->Hq = Hq; L->Hkv = Hkv; L->d = d; L->N = N; L->K = K;
    L->G = G;
    L->Bg = B / G;
    L->Sk = S / K;
    L->esz = esz;
    L->dtype = dtype;
    L->order = desc->order;
    *out = L;
    return BASP_OK;
}

extern "C" basp_status basp_layout_query(const basp_layout *L, basp_info *o) {
    if (L == nullptr || o == nullptr) return BASP_ERR_INVALID_ARG;
    o->B = L->B; o->S = L->S; o->Hq = L->Hq; o->Hkv = L->Hkv; o->d = L->d;
    o->N = L->N; o->K = L->K;
    o->groups = L->G;
    o->seqs_per_group = L->Bg;
    o->tokens_per_rank = L->Bg * L->Sk;
    o->elem_size = L->esz;
    o->elems_per_rank_q = L->Bg * L->Sk * L->Hq * L->d;
    o->elems_per_rank_kv = L->Bg * L->Sk * L->Hkv * L->d;
    o->peers = L->K - 1;
    o->bytes_per_peer_q = L->Bg * L->Sk * (L->Hq / L->K) * L->d * L->esz;
    o->bytes_per_peer_kv = L->Bg * L->Sk * (L->Hkv / L->K) * L->d * L->esz;
    o->bytes_q = basp::tensor_bytes(*L, L->Hq);
    o->bytes_kv = basp::tensor_bytes(*L, L->Hkv);
    const int64_t H3[3] = {L->Hq, L->Hkv, L->Hkv};
    o->workspace_bytes = basp::workspace_bytes(*L, H3, 3);
    o->staging_bytes = basp::workspace_bytes(*L, H3, 3);   // inputs + outputs
    o->foil_tokens_per_rank = L->B * L->S / L->K;
    o->order = L->order;
    o->bytes_qkv_packed = basp::tensor_bytes(*L, L->Hq + 2 * L->Hkv);
    return BASP_OK;
}

extern "C" void basp_layout_destroy(basp_layout *L) { delete L; }

extern "C" const char *basp_status_string(basp_status s) {
    switch (s) {
        case BASP_OK: return "ok";
        case BASP_ERR_INVALID_ARG: return "invalid argument";
        case BASP_ERR_DIVISIBILITY:
            return "shape breaks a divisibility rule (N%K, B%(N/K), S%K, Hq%K, Hkv%K)";
        case BASP_ERR_BATCH_GT_RANKS:
            return "micro-batch larger than the rank count: no BASP grouping (data parallelism)";
        case BASP_ERR_ALIGNMENT: return "pointer not aligned to the element size";
        case BASP_ERR_ALIASING: return "an output range overlaps another buffer";
        case BASP_ERR_WORKSPACE: return "workspace or staging buffer missing or too small";
        case BASP_ERR_CUDA: return "CUDA launch or copy failed";
        case BASP_ERR_TOO_LARGE: return "size beyond the library's index range";
    }
    return "unknown status";
}
