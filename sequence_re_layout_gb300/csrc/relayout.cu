// relayout.cu -- host side of the seq-sharded <-> head-sharded re-layout:
// stride tables, pass planning, launch, and the C-ABI entry points.  The one
// device kernel every pass launches is in relayout_kernel.cuh.
//
// The operation is the all-to-all of Ulysses / BASP attention (review "BASP:
// Communication-Efficient Batch-Aware Sequence Parallelism for LLM Training",
// evolve.pub, "Summary" and FAQ "What is Batch-Aware Sequence Parallelism
// (BASP)?"), done on one GPU where the N ranks are shards of one allocation,
// so the exchange is a permutation in HBM.
//
// Every buffer involved is a set of "rows": contiguous runs of
// L = (H/K)*d elements (one rank's head block of one token), addressed by five
// coordinates
//     g  group                      (G = N/K)
//     j  member holding the tokens  (K)   -- seq-sharded owner
//     jp member holding the heads   (K)   -- head-sharded owner
//     bl sequence within the group  (Bg = B/G)
//     sl token within the block     (S/K)
// and each buffer kind is a stride table over them (batch-first order shown;
// sequence-first order swaps [Bg] and [S/K] inside every table):
//     SEQ   seq-sharded  [G][K j][Bg][S/K sl][K jp][L]
//     HEAD  head-sharded [G][K jp][Bg][K j][S/K sl][L]
//     BYSRC send chunks  [G][K j][K jp][Bg][S/K][L]   (chunk jp of rank g*K+j)
//     BYDST recv chunks  [G][K jp][K j][Bg][S/K][L]   (slot j of rank g*K+jp)
// A pass copies every row from one kind to another.  The fused path is one
// pass SEQ -> HEAD (or back); the three-pass path is pack (SEQ -> BYSRC),
// exchange (BYSRC -> BYDST, whole chunks), unpack (BYDST -> HEAD), with the
// identity pass skipped on request when BYDST and HEAD address rows alike.
// Packed QKV input is three jobs whose SEQ rows stride over the packed row.
//
// Launch policy (all measured on GB300):
//   - one tile per CTA rather than a persistent grid (5-12% faster on HBM:
//     retiring CTAs let new ones start their loads while others drain their
//     stores): 16 KiB tiles of 256 threads, and 32 KiB tiles of 512 threads
//     for launches of at least 8 waves (+0.4-0.8% there);
//   - page-locked host buffers instead take a persistent grid of one
//     256-thread CTA per SM, which moves the most over the host link;
//   - programmatic dependent launch, so a kernel's CTAs may be scheduled while
//     the previous kernel on the stream drains (each waits with
//     griddepcontrol.wait before touching memory), hiding the launch gap
//     between back-to-back re-layouts (3-10% per step);
//   - an L2 prefetch of each CTA's tile before that wait, which overlaps the
//     first DRAM reads of a launch with the previous one's tail (+1% per step
//     at S=32768, +18% at S=1024).
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>

#include <nvtx3/nvToolsExt.h>

#include "layout_internal.h"
#include "relayout_kernel.cuh"
#include "scratch_cache.h"

namespace {

// An NVTX range named after the entry point, so profilers show each call
// (a no-op unless a tool is attached).
struct NvtxRange {
    explicit NvtxRange(const char *name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
};

// ---------------------------------------------------------------------------
// Host side: stride tables, pass planning, launch.
// ---------------------------------------------------------------------------

// Strides of the five coordinates for one buffer kind, in the unit `vpr` and
// `wseq` are given in (vectors of the launch's width).  `vpr` is one row (one rank's head block of one token);
// `wseq` is one whole token row on the seq-sharded side (K * vpr, or the
// packed QKV row).  Batch-first shards keep a sequence's tokens together;
// sequence-first shards interleave the group's sequences token by token.
void strides_of(const basp_layout &L, BufKind kind, int64_t vpr, int64_t wseq,
                int64_t s[5]) {
    const int64_t K = L.K, Bg = L.Bg, Sk = L.Sk;
    const bool sf = L.order == BASP_ORDER_SBHD;
    switch (kind) {
        case SEQ:     // [G][K j][Bg][Sk][row]  or  [G][K j][Sk][Bg][row]
            s[C_JP] = vpr;
            s[C_SL] = sf ? Bg * wseq : wseq;
            s[C_BL] = sf ? wseq : Sk * wseq;
            s[C_J] = Bg * Sk * wseq;
            s[C_G] = K * Bg * Sk * wseq;
            break;
        case HEAD:    // [G][K jp][Bg][K j][Sk][vpr]  or  [G][K jp][K j][Sk][Bg][vpr]
            s[C_SL] = sf ? Bg * vpr : vpr;
            s[C_J] = sf ? Sk * Bg * vpr : Sk * vpr;
            s[C_BL] = sf ? vpr : K * Sk * vpr;
            s[C_JP] = Bg * K * Sk * vpr;
            s[C_G] = K * Bg * K * Sk * vpr;
            break;
        case BYSRC:   // [G][K j][K jp][Bg][Sk][vpr]  or  ...[Sk][Bg][vpr]
            s[C_SL] = sf ? Bg * vpr : vpr;
            s[C_BL] = sf ? vpr : Sk * vpr;
            s[C_JP] = Bg * Sk * vpr;
            s[C_J] = K * Bg * Sk * vpr;
            s[C_G] = K * K * Bg * Sk * vpr;
            break;
        case BYDST:   // [G][K jp][K j][Bg][Sk][vpr]  or  ...[Sk][Bg][vpr]
            s[C_SL] = sf ? Bg * vpr : vpr;
            s[C_BL] = sf ? vpr : Sk * vpr;
            s[C_J] = Bg * Sk * vpr;
            s[C_JP] = K * Bg * Sk * vpr;
            s[C_G] = K * K * Bg * Sk * vpr;
            break;
    }
}

// Extent of a block digit.  In sequence-first order the group's sequences
// sit next to each other inside every token, so (sl, bl) merge into one row
// index of S/K * Bg rows whose stride is that of bl, and bl is no digit.
int64_t extent_of(const basp_layout &L, int c) {
    switch (c) {
        case C_G: return L.G;
        case C_J: return L.K;
        case C_JP: return L.K;
        case C_BL: return L.order == BASP_ORDER_SBHD ? 1 : L.Bg;
        default: return L.Sk;
    }
}

// Granlund-Montgomery constants for unsigned 32-bit division by D (1 <= D <
// 2^31), valid for dividends below 2^31: l = ceil(log2 D),
// m = floor(2^32 * (2^l - D) / D) + 1, and n / D == (umulhi(n, m) + n) >> l.
void udiv_magic(uint32_t D, uint32_t *m, uint32_t *l) {
    uint32_t ll = 0;
    while ((uint64_t(1) << ll) < D) ++ll;
    const uint64_t mm = ((uint64_t(1) << 32) * ((uint64_t(1) << ll) - D)) / D + 1;
    *m = uint32_t(mm);
    *l = ll;
}

struct TensorArg {
    const void *in;
    void *out;
    int64_t H;       // heads of this tensor
    int64_t seq_w;   // elements of one token row on the seq-sharded side
                     // (0: H * d; a packed QKV row is (Hq + 2*Hkv) * d)
    // extents of the buffers around `in` and `out`, in bytes relative to
    // the pointer (both 0: [0, the tensor's bytes)); bounds-checked builds
    // test every access against them
    int64_t in_lo, in_hi, out_lo, out_hi;
};

// [lo, hi) byte extent -> the vector indices whose whole vector lies inside.
int64_t vec_lo(int64_t lo, int vec) { return lo >= 0 ? (lo + vec - 1) / vec : -((-lo) / vec); }
int64_t vec_hi(int64_t hi, int vec) { return hi >= 0 ? hi / vec : -((-hi + vec - 1) / vec); }

int64_t seq_row_elems(const basp_layout &L, const TensorArg &t) {
    return t.seq_w > 0 ? t.seq_w : t.H * L.d;
}

struct Pass {
    BufKind from, to;
    int digit[4];     // block digits, outermost first; the row coordinate is sl
    int inner_fast;   // tiles interleave the innermost digit
};

// The passes of each path.  In the fused passes the head-block digit jp is
// innermost and interleaved: consecutive tiles take the K head blocks of the
// same tokens, so at any moment the CTAs in flight cover whole token rows on
// the seq-sharded side, where one rank's head block is a short segment of a
// longer row (measured on GB300: +0.5-2% for seq2head, within 0.5% for
// head2seq, against walking one head block at a time).  The three-pass
// passes take the destination's order, so consecutive tiles write
// consecutive memory.
constexpr Pass kFusedS2H = {SEQ, HEAD, {C_G, C_J, C_BL, C_JP}, 1};
constexpr Pass kFusedH2S = {HEAD, SEQ, {C_G, C_J, C_BL, C_JP}, 1};
constexpr Pass kPackS2H = {SEQ, BYSRC, {C_G, C_J, C_JP, C_BL}, 0};
constexpr Pass kExchS2H = {BYSRC, BYDST, {C_G, C_JP, C_J, C_BL}, 0};
constexpr Pass kUnpackS2H = {BYDST, HEAD, {C_G, C_JP, C_BL, C_J}, 0};
constexpr Pass kPackH2S = {HEAD, BYDST, {C_G, C_JP, C_J, C_BL}, 0};
constexpr Pass kExchH2S = {BYDST, BYSRC, {C_G, C_J, C_JP, C_BL}, 0};
constexpr Pass kUnpackH2S = {BYSRC, SEQ, {C_G, C_J, C_BL, C_JP}, 0};

// Widest vector (bytes) that divides the row length and every address.
int pick_vec(const basp_layout &L, const TensorArg *t, int n,
             const void *const *extra, int nextra) {
    int vec = 16;
    auto fits = [&](uintptr_t x) { return (x % uintptr_t(vec)) == 0; };
    while (vec > L.esz) {
        bool ok = true;
        for (int i = 0; i < n && ok; ++i) {
            const int64_t row_bytes = (t[i].H / L.K) * L.d * L.esz;
            const int64_t seq_bytes = seq_row_elems(L, t[i]) * L.esz;
            ok = fits(uintptr_t(row_bytes)) && fits(uintptr_t(seq_bytes)) &&
                 fits(uintptr_t(t[i].in)) && fits(uintptr_t(t[i].out));
        }
        for (int i = 0; i < nextra && ok; ++i) ok = fits(uintptr_t(extra[i]));
        if (ok) break;
        vec /= 2;
    }
    return vec;
}

basp_status plan(const basp_layout &L, const Pass &pass, const TensorArg *t,
                 int n, int vec, int tile_vec, Params *p) {
    std::memset(p, 0, sizeof(*p));
    uint64_t tiles = 0;
    int nj = 0;
    for (int i = 0; i < n; ++i) {
        const int64_t row_bytes = (t[i].H / L.K) * L.d * L.esz;
        const int64_t vpr = row_bytes / vec;
        const int64_t wseq = seq_row_elems(L, t[i]) * L.esz / vec;
        const bool sf = L.order == BASP_ORDER_SBHD;
        const int64_t rows = sf ? L.Sk * L.Bg : L.Sk;
        const int64_t vec_per_block = rows * vpr;
        if (vec_per_block == 0) continue;                    // empty tensor
        if (vec_per_block >= (int64_t(1) << 31)) return BASP_ERR_TOO_LARGE;
        Job &J = p->job[nj++];
        int64_t ss[5], ds[5];
        strides_of(L, pass.from, vpr, wseq, ss);
        strides_of(L, pass.to, vpr, wseq, ds);
        for (int k = 0; k < 4; ++k) {
            J.src_bs[k] = ss[pass.digit[k]];
            J.dst_bs[k] = ds[pass.digit[k]];
            J.radix[k] = uint32_t(extent_of(L, pass.digit[k]));
        }
        // rows: sl (batch-first) or the merged (sl, bl) (sequence-first)
        J.src_rs = sf ? ss[C_BL] : ss[C_SL];
        J.dst_rs = sf ? ds[C_BL] : ds[C_SL];
        J.src = static_cast<const unsigned char *>(t[i].in);
        J.dst = static_cast<unsigned char *>(t[i].out);
        {
            const int64_t tb = basp::tensor_bytes(L, t[i].H);
            const bool di = t[i].in_lo == 0 && t[i].in_hi == 0;
            const bool dd = t[i].out_lo == 0 && t[i].out_hi == 0;
            J.src_lo = vec_lo(di ? 0 : t[i].in_lo, vec);
            J.src_hi = vec_hi(di ? tb : t[i].in_hi, vec);
            J.dst_lo = vec_lo(dd ? 0 : t[i].out_lo, vec);
            J.dst_hi = vec_hi(dd ? tb : t[i].out_hi, vec);
        }
        J.vpr = uint32_t(vpr);
        udiv_magic(J.vpr, &J.vpr_magic, &J.vpr_shift);
        J.vec_per_block = uint32_t(vec_per_block);
        J.tiles_per_block = uint32_t((vec_per_block + tile_vec - 1) / tile_vec);
        J.tile_begin = uint32_t(tiles);
        J.inner_fast = uint32_t(pass.inner_fast);
        const uint64_t blocks = uint64_t(L.G) * L.K * L.K * uint64_t(extent_of(L, C_BL));
        tiles += blocks * J.tiles_per_block;
        if (tiles >= (uint64_t(1) << 31)) return BASP_ERR_TOO_LARGE;
    }
    p->njobs = nj;
    p->total_tiles = uint32_t(tiles);
    return BASP_OK;
}

// CTAs per SM of the persistent grid used on page-locked host buffers.  One
// per SM measured best on GB300 over NVLink-C2C (334 GB/s read+write at the
// Llama-3.2-1B S=8192 step against 295 with six; the host link's two-way
// limit measured with the copy engines is about 342).
constexpr int kHostCtasPerSm = 1;

// CTA slots of one wave on the current device: SMs x resident CTAs of the
// kernel (persistent: at most kHostCtasPerSm per SM).  Cached per device (a
// benign race: every thread computes the same value).
template <int VEC, int THREADS>
uint32_t wave_slots(bool persistent) {
    static std::atomic<int> cache[2][64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = 0;
    int slots = cache[persistent][dev].load(std::memory_order_relaxed);
    if (slots == 0) {
        int sms = 0, per_sm = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                &per_sm, basp_relayout_kernel<VEC, THREADS>, THREADS, 0) != cudaSuccess) {
            cudaGetLastError();           // clear the error this probe caused
            return 1;
        }
        int cap = persistent ? kHostCtasPerSm : per_sm;
        if (BASP_CTAS_PER_SM > 0 && cap > BASP_CTAS_PER_SM) cap = BASP_CTAS_PER_SM;
        if (cap > per_sm) cap = per_sm;
        slots = (sms > 0 ? sms : 1) * (cap > 0 ? cap : 1);
        cache[persistent][dev].store(slots, std::memory_order_relaxed);
    }
    return uint32_t(slots);
}

// One CTA per tile (device memory), or (persistent, host memory) a grid of
// kHostCtasPerSm CTAs per SM striding over the tiles.  The CTAs of a
// device-memory grid prefetch their tile into L2 first (BASP_PREFETCH: all of
// them, or those of the first wave); host memory is never prefetched.
template <int VEC, int THREADS = kThreads>
basp_status launch_vec(Params p, cudaStream_t stream, bool persistent) {
    const uint32_t slots = wave_slots<VEC, THREADS>(persistent);
    uint32_t grid = p.total_tiles < slots ? p.total_tiles : slots;
    if (BASP_GRID_ALL_TILES && !persistent) grid = p.total_tiles;
    p.prefetch_ctas = 0;
    if (!persistent && BASP_PREFETCH == 1) p.prefetch_ctas = slots;
    if (!persistent && BASP_PREFETCH == 2) p.prefetch_ctas = p.total_tiles;
#if BASP_PDL
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // the launch's own status: an error the caller left pending is not ours
    if (cudaLaunchKernelEx(&cfg, basp_relayout_kernel<VEC, THREADS>, p) != cudaSuccess) {
        cudaGetLastError();               // clear the error this launch set
        return BASP_ERR_CUDA;
    }
    return BASP_OK;
#else
    cudaGetLastError();                   // start from a clean error state
    basp_relayout_kernel<VEC, THREADS><<<grid, THREADS, 0, stream>>>(p);
    return cudaGetLastError() == cudaSuccess ? BASP_OK : BASP_ERR_CUDA;
#endif
}

basp_status run_pass(const basp_layout &L, const Pass &pass,
                     const TensorArg *t, int n, int vec, cudaStream_t stream,
                     bool persistent = false) {
    Params p;
    basp_status st = plan(L, pass, t, n, vec, kThreads * kUnroll, &p);
    if (st != BASP_OK || p.total_tiles == 0) return st;
    // A long launch (at least BASP_LARGE_WAVES waves of kThreads-thread CTAs)
    // runs kThreadsLarge-thread CTAs with tiles as many vectors longer:
    // measured on GB300, +0.4-0.5% from S=8192 up, while short launches
    // lose with them (2.6% at S=1024).  Host memory keeps the persistent
    // kThreads grid.
    if constexpr (kThreadsLarge != kThreads) {
        if (vec == 16 && !persistent &&
            uint64_t(p.total_tiles) >=
                uint64_t(BASP_LARGE_WAVES) * wave_slots<16, kThreads>(false)) {
            Params q;
            st = plan(L, pass, t, n, vec, kThreadsLarge * kUnroll, &q);
            if (st != BASP_OK) return st;
            return launch_vec<16, kThreadsLarge>(q, stream, false);
        }
    }
    switch (vec) {
        case 16: return launch_vec<16>(p, stream, persistent);
        case 8: return launch_vec<8>(p, stream, persistent);
        case 4: return launch_vec<4>(p, stream, persistent);
        case 2: return launch_vec<2>(p, stream, persistent);
        default: return launch_vec<1>(p, stream, persistent);
    }
}

bool overlaps(const void *a, int64_t na, const void *b, int64_t nb) {
    if (na <= 0 || nb <= 0 || a == nullptr || b == nullptr) return false;
    const uintptr_t x = uintptr_t(a), y = uintptr_t(b);
    return x < y + uintptr_t(nb) && y < x + uintptr_t(na);
}

// Gather the (input, output, heads) triples of one call and check pairing,
// alignment and aliasing.  The first pair has Hq heads (Q or O), the other
// two Hkv (K, V).
basp_status collect(const basp_layout *L, const void *a, const void *k,
                    const void *v, void *ao, void *ko, void *vo,
                    TensorArg *t, int *n) {
    if (L == nullptr) return BASP_ERR_INVALID_ARG;
    const TensorArg all[3] = {{a, ao, L->Hq}, {k, ko, L->Hkv}, {v, vo, L->Hkv}};
    *n = 0;
    for (const TensorArg &x : all) {
        if ((x.in == nullptr) != (x.out == nullptr)) return BASP_ERR_INVALID_ARG;
        if (x.in != nullptr) t[(*n)++] = x;
    }
    if (*n == 0) return BASP_ERR_INVALID_ARG;
    for (int i = 0; i < *n; ++i) {
        if (uintptr_t(t[i].in) % uintptr_t(L->esz) ||
            uintptr_t(t[i].out) % uintptr_t(L->esz))
            return BASP_ERR_ALIGNMENT;
    }
    for (int i = 0; i < *n; ++i) {
        const int64_t bi = basp::tensor_bytes(*L, t[i].H);
        for (int j = 0; j < *n; ++j) {
            const int64_t bj = basp::tensor_bytes(*L, t[j].H);
            if (overlaps(t[i].out, bi, t[j].in, bj)) return BASP_ERR_ALIASING;
            if (i != j && overlaps(t[i].out, bi, t[j].out, bj))
                return BASP_ERR_ALIASING;
        }
    }
    return BASP_OK;
}

int64_t region_bytes(const basp_layout &L, const TensorArg *t, int n) {
    int64_t H[3];
    for (int i = 0; i < n; ++i) H[i] = t[i].H;
    return basp::workspace_bytes(L, H, n);
}

// True when the receive-chunk layout of the three-pass path addresses every
// row exactly as the head-sharded layout does (one sequence per group, or
// sequence-first order): the unpack of seq2head and the pack of head2seq are
// then the identity and can be skipped.
bool recv_chunks_are_head_sharded(const basp_layout &L) {
    int64_t a[5], b[5];
    strides_of(L, BYDST, 1, L.K, a);
    strides_of(L, HEAD, 1, L.K, b);
    const bool sf = L.order == BASP_ORDER_SBHD;
    const int64_t ext[5] = {L.G, L.K, L.K, sf ? L.Sk * L.Bg : L.Bg, sf ? 1 : L.Sk};
    for (int c = 0; c < 5; ++c)
        if (ext[c] > 1 && a[c] != b[c]) return false;
    return true;
}

// The three-pass path with its identity pass skipped: seq2head packs into the
// workspace and exchanges straight into the head-sharded output; head2seq
// exchanges the head-sharded input into the workspace and unpacks from there.
// Needs one workspace region per tensor.
basp_status relayout_two_pass(const basp_layout &L, bool to_head,
                              const TensorArg *t, int n, void *ws,
                              size_t ws_bytes, cudaStream_t stream,
                              bool persistent) {
    int64_t need = 0;
    for (int i = 0; i < n; ++i) need += basp::align256(basp::tensor_bytes(L, t[i].H));
    if (need > 0 && (ws == nullptr || int64_t(ws_bytes) < need))
        return BASP_ERR_WORKSPACE;
    for (int i = 0; i < n; ++i) {
        const int64_t b = basp::tensor_bytes(L, t[i].H);
        if (overlaps(ws, need, t[i].in, b) || overlaps(ws, need, t[i].out, b))
            return BASP_ERR_ALIASING;
    }
    if (uintptr_t(ws) % uintptr_t(L.esz)) return BASP_ERR_ALIGNMENT;
    TensorArg first[3], second[3];
    unsigned char *w = static_cast<unsigned char *>(ws);
    for (int i = 0; i < n; ++i) {
        first[i] = {t[i].in, w, t[i].H};
        second[i] = {w, t[i].out, t[i].H};
        w += basp::align256(basp::tensor_bytes(L, t[i].H));
    }
    const void *extra[1] = {ws};
    const int vec = pick_vec(L, t, n, extra, 1);
    basp_status st = run_pass(L, to_head ? kPackS2H : kExchH2S, first, n, vec, stream,
                              persistent);
    if (st != BASP_OK) return st;
    return run_pass(L, to_head ? kExchS2H : kUnpackH2S, second, n, vec, stream,
                    persistent);
}

basp_status relayout(const basp_layout *L, basp_algo algo, bool to_head,
                     const void *a, const void *k, const void *v, void *ao,
                     void *ko, void *vo, void *ws, size_t ws_bytes,
                     cudaStream_t stream, bool persistent = false) {
    TensorArg t[3];
    int n = 0;
    basp_status st = collect(L, a, k, v, ao, ko, vo, t, &n);
    if (st != BASP_OK) return st;
    if (algo == BASP_ALGO_FUSED) {
        const int vec = pick_vec(*L, t, n, nullptr, 0);
        return run_pass(*L, to_head ? kFusedS2H : kFusedH2S, t, n, vec, stream,
                        persistent);
    }
    if (algo != BASP_ALGO_THREE_PASS && algo != BASP_ALGO_THREE_PASS_ELIDE)
        return BASP_ERR_INVALID_ARG;
    if (algo == BASP_ALGO_THREE_PASS_ELIDE && recv_chunks_are_head_sharded(*L))
        return relayout_two_pass(*L, to_head, t, n, ws, ws_bytes, stream, persistent);

    const int64_t need = region_bytes(*L, t, n);
    if (need > 0 && (ws == nullptr || int64_t(ws_bytes) < need))
        return BASP_ERR_WORKSPACE;
    for (int i = 0; i < n; ++i) {
        const int64_t b = basp::tensor_bytes(*L, t[i].H);
        if (overlaps(ws, need, t[i].in, b) || overlaps(ws, need, t[i].out, b))
            return BASP_ERR_ALIASING;
    }
    if (uintptr_t(ws) % uintptr_t(L->esz)) return BASP_ERR_ALIGNMENT;
    // workspace regions: [send 0][recv 0][send 1][recv 1]...
    TensorArg pack[3], exch[3], unpack[3];
    const void *extra[1] = {ws};
    unsigned char *w = static_cast<unsigned char *>(ws);
    for (int i = 0; i < n; ++i) {
        const int64_t r = basp::align256(basp::tensor_bytes(*L, t[i].H));
        unsigned char *send = w, *recv = w + r;
        w += 2 * r;
        pack[i] = {t[i].in, send, t[i].H};
        exch[i] = {send, recv, t[i].H};
        unpack[i] = {recv, t[i].out, t[i].H};
    }
    const int vec = pick_vec(*L, t, n, extra, 1);
    const Pass *passes[3] = {to_head ? &kPackS2H : &kPackH2S,
                             to_head ? &kExchS2H : &kExchH2S,
                             to_head ? &kUnpackS2H : &kUnpackH2S};
    const TensorArg *args[3] = {pack, exch, unpack};
    for (int s = 0; s < 3; ++s) {
        st = run_pass(*L, *passes[s], args[s], n, vec, stream, persistent);
        if (st != BASP_OK) return st;
    }
    return BASP_OK;
}

basp_status relayout_host(const basp_layout *L, basp_algo algo, bool to_head,
                          const void *a, const void *k, const void *v,
                          void *ao, void *ko, void *vo, void *staging,
                          size_t staging_bytes, void *ws, size_t ws_bytes,
                          cudaStream_t stream) {
    TensorArg t[3];
    int n = 0;
    basp_status st = collect(L, a, k, v, ao, ko, vo, t, &n);
    if (st != BASP_OK) return st;
    const int64_t need = region_bytes(*L, t, n);
    if (staging == nullptr && need > 0) {
        // Direct: every host buffer must be page-locked; the kernels reach it
        // through its device address (the same address under unified
        // addressing).  A persistent grid of one CTA per SM moves more over
        // the host link than one tile per CTA.
        const void *hp[6] = {a, k, v, ao, ko, vo};
        const void *dp[6] = {nullptr, nullptr, nullptr, nullptr, nullptr, nullptr};
        for (int x = 0; x < 6; ++x) {
            if (hp[x] == nullptr) continue;
            cudaPointerAttributes attr;
            if (cudaPointerGetAttributes(&attr, hp[x]) != cudaSuccess) {
                cudaGetLastError();
                return BASP_ERR_WORKSPACE;
            }
            if (attr.type != cudaMemoryTypeHost || attr.devicePointer == nullptr)
                return BASP_ERR_WORKSPACE;
            dp[x] = attr.devicePointer;
        }
        return relayout(L, algo, to_head, dp[0], dp[1], dp[2],
                        const_cast<void *>(dp[3]), const_cast<void *>(dp[4]),
                        const_cast<void *>(dp[5]), ws, ws_bytes, stream, true);
    }
    if (need > 0 && int64_t(staging_bytes) < need)
        return BASP_ERR_WORKSPACE;
    if (overlaps(staging, need, ws, int64_t(ws_bytes))) return BASP_ERR_ALIASING;
    // staging regions: [in 0][out 0][in 1][out 1]...
    const void *din[3] = {nullptr, nullptr, nullptr};
    void *dout[3] = {nullptr, nullptr, nullptr};
    unsigned char *sp = static_cast<unsigned char *>(staging);
    for (int i = 0; i < n; ++i) {
        const int64_t b = basp::tensor_bytes(*L, t[i].H);
        const int64_t r = basp::align256(b);
        din[i] = sp;
        dout[i] = sp + r;
        sp += 2 * r;
        if (b > 0 && cudaMemcpyAsync(sp - 2 * r, t[i].in, size_t(b),
                                     cudaMemcpyHostToDevice, stream) != cudaSuccess)
            return BASP_ERR_CUDA;
    }
    // Map the staged buffers back onto the (first, k, v) argument slots.
    const void *sa[3] = {nullptr, nullptr, nullptr};
    void *so[3] = {nullptr, nullptr, nullptr};
    int i = 0;
    if (a) { sa[0] = din[i]; so[0] = dout[i]; ++i; }
    if (k) { sa[1] = din[i]; so[1] = dout[i]; ++i; }
    if (v) { sa[2] = din[i]; so[2] = dout[i]; ++i; }
    st = relayout(L, algo, to_head, sa[0], sa[1], sa[2], so[0], so[1], so[2],
                  ws, ws_bytes, stream);
    if (st != BASP_OK) return st;
    for (int x = 0; x < n; ++x) {
        const int64_t b = basp::tensor_bytes(*L, t[x].H);
        if (b > 0 && cudaMemcpyAsync(t[x].out, dout[x], size_t(b),
                                     cudaMemcpyDeviceToHost, stream) != cudaSuccess)
            return BASP_ERR_CUDA;
    }
    return BASP_OK;
}

// Packed QKV: Q, K and V are three jobs of one fused launch whose
// seq-sharded side is the packed buffer, each starting at its own head offset
// inside the token row and striding over the whole row.
basp_status relayout_qkv(const basp_layout *L, bool to_head, const void *packed,
                         const void *q, const void *k, const void *v,
                         void *qo, void *ko, void *vo, cudaStream_t stream) {
    if (L == nullptr || packed == nullptr) return BASP_ERR_INVALID_ARG;
    const void *ptrs[3] = {to_head ? qo : q, to_head ? ko : k, to_head ? vo : v};
    for (const void *x : ptrs)
        if (x == nullptr) return BASP_ERR_INVALID_ARG;
    for (const void *x : ptrs)
        if (uintptr_t(x) % uintptr_t(L->esz)) return BASP_ERR_ALIGNMENT;
    if (uintptr_t(packed) % uintptr_t(L->esz)) return BASP_ERR_ALIGNMENT;
    const int64_t W = (L->Hq + 2 * L->Hkv) * L->d;
    const int64_t bytes[3] = {basp::tensor_bytes(*L, L->Hq),
                              basp::tensor_bytes(*L, L->Hkv),
                              basp::tensor_bytes(*L, L->Hkv)};
    const int64_t packed_bytes = basp::tensor_bytes(*L, L->Hq + 2 * L->Hkv);
    // outputs may overlap neither an input nor each other
    for (int i = 0; i < 3; ++i) {
        if (overlaps(ptrs[i], bytes[i], packed, packed_bytes)) return BASP_ERR_ALIASING;
        if (to_head)
            for (int j = 0; j < i; ++j)
                if (overlaps(ptrs[i], bytes[i], ptrs[j], bytes[j])) return BASP_ERR_ALIASING;
    }
    const int64_t off[3] = {0, L->Hq * L->d * L->esz, (L->Hq + L->Hkv) * L->d * L->esz};
    const int64_t H[3] = {L->Hq, L->Hkv, L->Hkv};
    TensorArg t[3];
    for (int i = 0; i < 3; ++i) {
        if (to_head) {
            t[i] = {static_cast<const unsigned char *>(packed) + off[i],
                    const_cast<void *>(ptrs[i]), H[i], W,
                    -off[i], packed_bytes - off[i], 0, 0};
        } else {
            t[i] = {ptrs[i],
                    static_cast<unsigned char *>(const_cast<void *>(packed)) + off[i],
                    H[i], W, 0, 0, -off[i], packed_bytes - off[i]};
        }
    }
    const int vec = pick_vec(*L, t, 3, nullptr, 0);
    return run_pass(*L, to_head ? kFusedS2H : kFusedH2S, t, 3, vec, stream);
}

}  // namespace

extern "C" basp_status basp_seq2head_qkv(const basp_layout *L, const void *qkv,
                                         void *q_out, void *k_out, void *v_out,
                                         cudaStream_t stream) {
    NvtxRange range("basp_seq2head_qkv");
    return relayout_qkv(L, true, qkv, nullptr, nullptr, nullptr, q_out, k_out,
                        v_out, stream);
}

extern "C" basp_status basp_head2seq_qkv(const basp_layout *L, const void *q,
                                         const void *k, const void *v,
                                         void *qkv_out, cudaStream_t stream) {
    NvtxRange range("basp_head2seq_qkv");
    return relayout_qkv(L, false, qkv_out, q, k, v, nullptr, nullptr, nullptr,
                        stream);
}

extern "C" basp_status basp_seq2head(const basp_layout *L, basp_algo algo,
                                     const void *q, const void *k, const void *v,
                                     void *q_out, void *k_out, void *v_out,
                                     void *ws, size_t ws_bytes, cudaStream_t stream) {
    NvtxRange range("basp_seq2head");
    return relayout(L, algo, true, q, k, v, q_out, k_out, v_out, ws, ws_bytes, stream);
}

extern "C" basp_status basp_head2seq(const basp_layout *L, basp_algo algo,
                                     const void *o, const void *k, const void *v,
                                     void *o_out, void *k_out, void *v_out,
                                     void *ws, size_t ws_bytes, cudaStream_t stream) {
    NvtxRange range("basp_head2seq");
    return relayout(L, algo, false, o, k, v, o_out, k_out, v_out, ws, ws_bytes, stream);
}

extern "C" basp_status basp_seq2head_host(const basp_layout *L, basp_algo algo,
                                          const void *q, const void *k, const void *v,
                                          void *q_out, void *k_out, void *v_out,
                                          void *staging, size_t staging_bytes,
                                          void *ws, size_t ws_bytes, cudaStream_t stream) {
    NvtxRange range("basp_seq2head_host");
    return relayout_host(L, algo, true, q, k, v, q_out, k_out, v_out, staging,
                         staging_bytes, ws, ws_bytes, stream);
}

extern "C" basp_status basp_head2seq_host(const basp_layout *L, basp_algo algo,
                                          const void *o, const void *k, const void *v,
                                          void *o_out, void *k_out, void *v_out,
                                          void *staging, size_t staging_bytes,
                                          void *ws, size_t ws_bytes, cudaStream_t stream) {
    NvtxRange range("basp_head2seq_host");
    return relayout_host(L, algo, false, o, k, v, o_out, k_out, v_out, staging,
                         staging_bytes, ws, ws_bytes, stream);
}

// ---------------------------------------------------------------------------
// basp_seq2head_noalloc: the three-pass seq2head with its scratch in a static
// device array, for callers that cannot allocate (see basp.h).
// ---------------------------------------------------------------------------

static __device__ __align__(256) unsigned char
    g_noalloc_scratch[BASP_NOALLOC_SCRATCH_BYTES];

namespace {

// The array's device address in the current context.  In host code the name
// g_noalloc_scratch is only a host-side stand-in, so the address is looked up
// with cudaGetSymbolAddress, with the caller's device current, once per
// context: the first call on a device does the lookup (which may load the
// library's device code there) and later calls reuse it.  The cache
// (scratch_cache.h) is keyed by the driver's context ID, which is never reused
// within a process, so a device reset (after which the device code is loaded
// afresh, perhaps at another address) leads to a new lookup rather than a
// stale address.
using CtxGetCurrentFn = CUresult (*)(CUcontext *);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long *);

struct DriverCtxQuery {
    CtxGetCurrentFn get_current = nullptr;
    CtxGetIdFn get_id = nullptr;
};

const DriverCtxQuery &driver_ctx_query() {
    static const DriverCtxQuery q = [] {
        DriverCtxQuery r;
        void *f = nullptr, *g = nullptr;
        cudaDriverEntryPointQueryResult qr1, qr2;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000,
                                             cudaEnableDefault, &qr1) == cudaSuccess &&
            cudaGetDriverEntryPointByVersion("cuCtxGetId", &g, 12000,
                                             cudaEnableDefault, &qr2) == cudaSuccess &&
            qr1 == cudaDriverEntryPointSuccess && qr2 == cudaDriverEntryPointSuccess) {
            r.get_current = reinterpret_cast<CtxGetCurrentFn>(f);
            r.get_id = reinterpret_cast<CtxGetIdFn>(g);
        } else {
            cudaGetLastError();
        }
        return r;
    }();
    return q;
}

// ID of the context current on this thread, or 0 if none is (or the driver
// cannot say).
unsigned long long current_ctx_id() {
    const DriverCtxQuery &q = driver_ctx_query();
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (q.get_current == nullptr || q.get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr)
        return 0;
    if (q.get_id(ctx, &id) != CUDA_SUCCESS) return 0;
    return id;
}

basp::ScratchAddressCache<64> g_noalloc_cache;

basp_status noalloc_scratch(void **out) {
    const bool ok = g_noalloc_cache.get(current_ctx_id, [](void **p) {
        if (cudaGetSymbolAddress(p, g_noalloc_scratch) == cudaSuccess) return true;
        cudaGetLastError();               // clear the error this lookup set
        return false;
    }, out);
    return ok ? BASP_OK : BASP_ERR_CUDA;
}

}  // namespace

extern "C" basp_status basp_seq2head_noalloc(const basp_layout *L,
                                             const void *q, const void *k, const void *v,
                                             void *q_out, void *k_out, void *v_out,
                                             cudaStream_t stream) {
    NvtxRange range("basp_seq2head_noalloc");
    TensorArg t[3];
    int n = 0;
    basp_status st = collect(L, q, k, v, q_out, k_out, v_out, t, &n);
    if (st != BASP_OK) return st;
    if (region_bytes(*L, t, n) > int64_t(BASP_NOALLOC_SCRATCH_BYTES))
        return BASP_ERR_WORKSPACE;
    void *scratch = nullptr;
    st = noalloc_scratch(&scratch);
    if (st != BASP_OK) return st;
    return relayout(L, BASP_ALGO_THREE_PASS, true, q, k, v, q_out, k_out, v_out,
                    scratch, size_t(BASP_NOALLOC_SCRATCH_BYTES), stream);
}

#if BASP_CHECK_BOUNDS
// Debug builds only (libbasp_debug.so, declared in basp_debug.h): read and
// clear the count of accesses the kernels found outside their buffers.
extern "C" basp_status basp_debug_bounds_violations(unsigned long long *count) {
    if (count == nullptr) return BASP_ERR_INVALID_ARG;
    const unsigned long long zero = 0;
    if (cudaDeviceSynchronize() != cudaSuccess ||
        cudaMemcpyFromSymbol(count, g_basp_bounds_violations, sizeof(*count)) != cudaSuccess ||
        cudaMemcpyToSymbol(g_basp_bounds_violations, &zero, sizeof(zero)) != cudaSuccess)
        return BASP_ERR_CUDA;
    return BASP_OK;
}
#endif
