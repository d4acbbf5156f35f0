/*
 * basp.h -- C ABI of libbasp: the sequence-sharded <-> head-sharded re-layout
 * of attention activations for Ulysses and BASP (batch-aware Ulysses sequence
 * parallelism), on one GPU.
 *
 * The operation.  The review "BASP: Communication-Efficient Batch-Aware
 * Sequence Parallelism for LLM Training" (evolve.pub), sections "Summary" and
 * "Key claims under review", and its FAQ "What is Batch-Aware Sequence
 * Parallelism (BASP)?": with micro-batch B and N = K*B ranks, the ranks form B
 * disjoint contiguous groups of K; each group owns one sequence and runs its
 * own K-way all-to-all during attention instead of one N-way all-to-all, and
 * every rank keeps B*S/N tokens.  Ulysses (fugumt.com related-papers entry
 * "DeepSpeed Ulysses") is the K = N case.  The same review's "Strengths"
 * section writes both as G groups with B/G sequences each; this library takes
 * that general form: G = N/K groups, Bg = B/G sequences per group.
 *
 * Buffers.  A "virtual-rank buffer" is the N rank shards of one tensor laid
 * back to back in one device allocation, rank 0 first.  Rank r = g*K + j is
 * member j of group g.  Logical tensor X[b][s][h][e] is [B, S, H, d],
 * row-major (batch-first).
 *   seq-sharded  shard of rank r: X[g*Bg + bl][j*S/K + sl][h][e],
 *                                  stored [Bg][S/K][H][d]   (bl, sl, h, e)
 *   head-sharded shard of rank r: X[g*Bg + bl][s][j*H/K + hl][e],
 *                                  stored [Bg][S][H/K][d]   (bl, s, hl, e)
 * Each shard holds B*S*H*d/N elements in both layouts, so both buffers of a
 * tensor have B*S*H*d elements.  Q and the attention output O have Hq heads;
 * K and V have Hkv heads (grouped-query attention).
 *
 * Conventions for every call below.
 *   - Elements are copied bit for bit (no rounding; NaN payloads, -0 and
 *     subnormals survive).  fp8 is a 1-byte word, bf16 and fp16 2-byte,
 *     fp32 4-byte.
 *   - Device pointers must be naturally aligned for the dtype; 16-byte
 *     alignment gives the 16-byte vector path, lesser alignment a narrower one.
 *   - A "device" buffer may also be page-locked host memory (cudaHostAlloc,
 *     cudaMallocHost, cudaHostRegister): under unified addressing the kernels
 *     read and write it in place over the host link, with no staging copy.
 *   - Output ranges may not overlap any input, output or workspace range
 *     (no in-place re-layout): BASP_ERR_ALIASING.
 *   - The caller owns every buffer.  Compute calls allocate nothing, never
 *     synchronise, and enqueue their kernels on `stream` (0 = legacy default
 *     stream).  Validation happens before anything is enqueued, so an error
 *     return means nothing was launched, except BASP_ERR_CUDA, which reports
 *     a failed launch or copy on `stream`.
 *   - A layout handle is immutable after creation; calls that share one
 *     handle may run concurrently from several host threads.
 *   - Kernels are launched with programmatic dependent launch: they may be
 *     scheduled while the previous kernel on `stream` drains, but wait for it
 *     (and its memory) before reading or writing any buffer, so ordering on
 *     `stream` is as usual.  Before that wait they ask L2 to fetch the lines
 *     of their input (prefetch.global.L2): this reads no value into the
 *     kernel, so an input the previous kernel is still writing is read only
 *     after it has finished, with its final contents.  They also release the
 *     next kernel early; a kernel the caller launches after them with the
 *     programmatic-serialisation attribute must wait
 *     (cudaGridDependencySynchronize) before reading their outputs, as CUDA
 *     requires of every such kernel.
 */
#ifndef BASP_H
#define BASP_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum basp_dtype {
    BASP_DTYPE_BF16 = 0,
    BASP_DTYPE_FP32 = 1,
    BASP_DTYPE_FP16 = 2,
    BASP_DTYPE_FP8 = 3      /* any 1-byte format (e4m3, e5m2, int8), copied as bytes */
} basp_dtype;

/* Token order inside every rank shard.  The BASP review fixes none;
 * batch-first is the default.  Sequence-first is the [S, B, H, d] activation
 * order of Megatron-style stacks: seq-sharded shards [S/K][Bg][H][d], head-sharded
 * shards [S][Bg][H/K][d].  With one sequence per group (every BASP layout) the
 * two orders store the same bytes. */
typedef enum basp_order {
    BASP_ORDER_BSHD = 0,
    BASP_ORDER_SBHD = 1
} basp_order;

typedef enum basp_algo {
    /* One pass: every element goes straight from its source place to its
     * destination place; Q, K and V (or O, K, V) in one kernel launch. */
    BASP_ALGO_FUSED = 0,
    /* The collective's shape: pack each rank's shard into K per-destination
     * contiguous send chunks, exchange the chunks between the members of each
     * group (recv chunk j of member j' = send chunk j' of member j, the
     * equal-split all-to-all convention), unpack.  Needs a workspace. */
    BASP_ALGO_THREE_PASS = 1,
    /* The three-pass path with the pass skipped that is the identity: when
     * each group holds one sequence (every BASP layout) or the order is
     * sequence-first, the receive chunks already sit in head-sharded order,
     * so seq2head exchanges straight into its output and head2seq exchanges
     * straight from its input (two passes, workspace of one region per
     * tensor).  Otherwise it runs all three passes like
     * BASP_ALGO_THREE_PASS. */
    BASP_ALGO_THREE_PASS_ELIDE = 2
} basp_algo;

typedef enum basp_status {
    BASP_OK = 0,
    BASP_ERR_INVALID_ARG = 1,      /* NULL handle/pointer pairing, bad dtype, negative size */
    BASP_ERR_DIVISIBILITY = 2,     /* N%K, B%(N/K), S%K, Hq%K or Hkv%K nonzero */
    BASP_ERR_BATCH_GT_RANKS = 3,   /* K = 0 (BASP rule) asked with B > N */
    BASP_ERR_ALIGNMENT = 4,        /* pointer not aligned to the element size */
    BASP_ERR_ALIASING = 5,         /* an output overlaps another range */
    BASP_ERR_WORKSPACE = 6,        /* workspace or staging missing or too small */
    BASP_ERR_CUDA = 7,             /* a CUDA launch or copy failed */
    BASP_ERR_TOO_LARGE = 8         /* a size beyond the library's index range */
} basp_status;

typedef struct basp_layout basp_layout;   /* opaque, host memory only */

typedef struct basp_info {
    int64_t B, S, Hq, Hkv, d, N, K;
    int64_t groups;               /* G = N / K                                 */
    int64_t seqs_per_group;       /* Bg = B / G                                */
    int64_t tokens_per_rank;      /* Bg * S / K = B * S / N, both layouts      */
    int64_t elem_size;            /* bytes per element                         */
    int64_t elems_per_rank_q;     /* B*S*Hq*d / N                              */
    int64_t elems_per_rank_kv;    /* B*S*Hkv*d / N                             */
    int64_t peers;                /* other ranks each rank exchanges with: K-1 */
    int64_t bytes_per_peer_q;     /* Bg*(S/K)*(Hq/K)*d*esz                     */
    int64_t bytes_per_peer_kv;    /* Bg*(S/K)*(Hkv/K)*d*esz                    */
    int64_t bytes_q;              /* whole Q (or O) buffer: B*S*Hq*d*esz       */
    int64_t bytes_kv;             /* whole K (or V) buffer: B*S*Hkv*d*esz      */
    int64_t workspace_bytes;      /* BASP_ALGO_THREE_PASS workspace for Q,K,V  */
    int64_t staging_bytes;        /* device staging for the *_host calls      */
    int64_t foil_tokens_per_rank; /* B*S/K: tokens per rank if every group of K
                                     held all B sequences (the "Ulysses with
                                     SP = N/B" alternative of the review's
                                     "Strengths" section, B*B*S/N at K = N/B) */
    int64_t order;                /* basp_order of the shards                  */
    int64_t bytes_qkv_packed;     /* packed QKV buffer: B*S*(Hq+2*Hkv)*d*esz   */
} basp_info;

/* Everything basp_layout_create takes, plus the token order. */
typedef struct basp_layout_desc {
    int64_t B, S, Hq, Hkv, d, N, K;
    basp_dtype dtype;
    basp_order order;
} basp_layout_desc;

/*
 * Create a layout handle.
 *   B, S        micro-batch size and sequence length (B >= 0, S >= 0; zero
 *               gives empty buffers and calls that launch nothing)
 *   Hq, Hkv     query / key-value head counts (>= 1)
 *   d           head dimension (>= 1)
 *   N           ranks (>= 1)
 *   K           group size.  K = N is Ulysses; K = N/B is BASP.  K = 0 asks
 *               for the BASP rule K = N/B: it needs 1 <= B <= N
 *               (BASP_ERR_BATCH_GT_RANKS when B > N, where the review's FAQ
 *               "What are BASP's main limitations?" falls back to data
 *               parallelism) and N % B == 0 (BASP_ERR_DIVISIBILITY).
 *   dtype       element type
 *   out         receives the handle; *out is NULL on error.
 * Rules (same FAQ: N must be a multiple of B; heads must divide evenly across
 * group members): N % K == 0, B % (N/K) == 0, S % K == 0, Hq % K == 0,
 * Hkv % K == 0, else BASP_ERR_DIVISIBILITY.  Host only; no CUDA call.
 */
basp_status basp_layout_create(int64_t B, int64_t S, int64_t Hq, int64_t Hkv,
                               int64_t d, int64_t N, int64_t K,
                               basp_dtype dtype, basp_layout **out);

/* As basp_layout_create, with the token order of the shards (desc->order);
 * basp_layout_create is this call with BASP_ORDER_BSHD.  BASP_ERR_INVALID_ARG
 * for a NULL desc or an unknown order.  Host only. */
basp_status basp_layout_create_ex(const basp_layout_desc *desc,
                                  basp_layout **out);

/* Fill *out with the derived sizes of a layout.  Host only. */
basp_status basp_layout_query(const basp_layout *layout, basp_info *out);

/* Free a handle (NULL is ignored).  Host only. */
void basp_layout_destroy(basp_layout *layout);

/*
 * seq-sharded -> head-sharded, before attention.
 *   q, k, v           device seq-sharded virtual-rank buffers (Hq, Hkv, Hkv
 *                     heads).  Any of the three may be NULL, with its output
 *                     NULL too; at least one pair must be given.
 *   q_out,k_out,v_out device head-sharded virtual-rank buffers.
 *   workspace         device scratch for BASP_ALGO_THREE_PASS, at least
 *                     info.workspace_bytes (enough for Q, K and V; fewer
 *                     tensors need only the sum of their own send and receive
 *                     regions).  Ignored (may be NULL) for BASP_ALGO_FUSED.
 *   stream            CUDA stream the kernels are enqueued on.
 */
basp_status basp_seq2head(const basp_layout *layout, basp_algo algo,
                          const void *q, const void *k, const void *v,
                          void *q_out, void *k_out, void *v_out,
                          void *workspace, size_t workspace_bytes,
                          cudaStream_t stream);

/*
 * head-sharded -> seq-sharded, after attention: the exact inverse of
 * basp_seq2head.  `o` is the attention output (Hq heads); `k`, `v` (Hkv heads)
 * are optional and serve the backward pass (gradients of K and V travel
 * this way).  Arguments as for basp_seq2head.
 */
basp_status basp_head2seq(const basp_layout *layout, basp_algo algo,
                          const void *o, const void *k, const void *v,
                          void *o_out, void *k_out, void *v_out,
                          void *workspace, size_t workspace_bytes,
                          cudaStream_t stream);

/*
 * Packed QKV forms (fused path, one launch).  A fused QKV projection writes one
 * activation whose every token row holds the Hq query heads, then the Hkv key
 * heads, then the Hkv value heads; its seq-sharded virtual-rank buffer has
 * shards [Bg][S/K][Hq+2*Hkv][d] (or [S/K][Bg][Hq+2*Hkv][d] for
 * BASP_ORDER_SBHD), info.bytes_qkv_packed bytes in all.
 *   basp_seq2head_qkv   packed seq-sharded `qkv` -> head-sharded q_out (Hq
 *                       heads), k_out, v_out (Hkv heads), the same buffers
 *                       basp_seq2head produces; no split copy first.
 *   basp_head2seq_qkv   the inverse: head-sharded q, k, v (in the backward
 *                       pass, the gradients dQ, dK, dV) -> one packed
 *                       seq-sharded buffer `qkv_out`.
 * All four pointers are required.  The BASP review describes no projection
 * layout; the head order inside the row is the plainest concatenation.
 */
basp_status basp_seq2head_qkv(const basp_layout *layout, const void *qkv,
                              void *q_out, void *k_out, void *v_out,
                              cudaStream_t stream);
basp_status basp_head2seq_qkv(const basp_layout *layout, const void *q,
                              const void *k, const void *v, void *qkv_out,
                              cudaStream_t stream);

/*
 * End-to-end forms for callers whose tensors live in host memory; the host
 * outputs are valid once `stream` has been synchronised.  Two modes:
 *   staged  (`staging` given): enqueue on `stream` the host->device copies of
 *           the inputs into `staging`, the re-layout, and the device->host
 *           copies of the results.  `staging` is caller-owned device memory
 *           of at least info.staging_bytes; host pointers should be
 *           page-locked for the copies to run asynchronously.
 *   direct  (`staging` NULL): every host buffer must be page-locked
 *           (cudaHostAlloc, cudaMallocHost, cudaHostRegister), else
 *           BASP_ERR_WORKSPACE; the kernels read the inputs and write the
 *           outputs in place over the host link, with no copies.  On GB300
 *           (NVLink-C2C) this is the faster mode.
 * Arguments otherwise as for basp_seq2head / basp_head2seq.
 */
basp_status basp_seq2head_host(const basp_layout *layout, basp_algo algo,
                               const void *q, const void *k, const void *v,
                               void *q_out, void *k_out, void *v_out,
                               void *staging, size_t staging_bytes,
                               void *workspace, size_t workspace_bytes,
                               cudaStream_t stream);
basp_status basp_head2seq_host(const basp_layout *layout, basp_algo algo,
                               const void *o, const void *k, const void *v,
                               void *o_out, void *k_out, void *v_out,
                               void *staging, size_t staging_bytes,
                               void *workspace, size_t workspace_bytes,
                               cudaStream_t stream);

/*
 * basp_seq2head_noalloc -- seq-sharded -> head-sharded through the three-pass
 * path (pack, exchange, unpack), with the scratch it needs taken from a buffer
 * built into the library instead of from the caller.  The paper has no
 * counterpart to this call; it exists for callers that cannot allocate device
 * memory when they need the re-layout: code that runs inside a host
 * framework's custom-op or plugin interface whose caching allocator owns all
 * device memory and hands out no scratch, and latency-bound serving loops that
 * ban cudaMalloc on their hot path because it can synchronise the device and
 * take milliseconds.  Such callers still pass their own inputs and outputs.
 *
 * The scratch is one file-scope __device__ array of
 * BASP_NOALLOC_SCRATCH_BYTES (32 MiB).  Every GPU on which the library's
 * device code is loaded holds it until the process exits.  A call needs
 * 2 * (bytes of each tensor it moves, each rounded up to 256) of it; a call
 * that needs more returns BASP_ERR_WORKSPACE and launches nothing (use
 * basp_seq2head with a workspace instead).  With Llama-3.2-1B heads
 * (Hq=32, Hkv=8, d=64, bf16, B=2) Q, K and V together fit up to S=1024.
 *
 * The first call on each device looks up the array's device address on that
 * device (cudaGetSymbolAddress, with that device current), which may load the
 * library's device code there; make that first call before any stream
 * capture.  The address is kept per CUDA context, keyed by the driver's
 * context ID: after a device reset the device has a new context, and the next
 * call looks the address up again instead of using the old one.  (As for any
 * CUDA library, nothing of it may be in use on the device while it is
 * reset.)  Every call shares the one array: calls whose kernels can overlap
 * on the GPU (different streams, or several host threads) race on it and
 * corrupt each other's results, so keep them on one stream.  Each call
 * writes every scratch byte before reading it, so nothing has to start at
 * zero and nothing is cleared between calls.  This call allocates nothing:
 * no cudaMalloc, cudaFree or allocating library routine.
 *
 * Arguments as for basp_seq2head with algo = BASP_ALGO_THREE_PASS and no
 * workspace.
 */
#define BASP_NOALLOC_SCRATCH_BYTES (32u << 20)
basp_status basp_seq2head_noalloc(const basp_layout *layout,
                                  const void *q, const void *k, const void *v,
                                  void *q_out, void *k_out, void *v_out,
                                  cudaStream_t stream);

/* Static English text for a status code. */
const char *basp_status_string(basp_status status);

#ifdef __cplusplus
}
#endif

#endif /* BASP_H */
