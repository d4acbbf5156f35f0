/*
 * basp_oracle.c -- CPU oracle for the BASP / Ulysses sequence<->head re-layout.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or calls
 * this file; only the tests, the package's smoke check and the benchmark's
 * CPU-baseline leg do.  It shares no code, header or constant with the CUDA
 * library.
 *
 * What it computes (plain definition, no blocking, no fusion):
 *
 *   The review "BASP: Communication-Efficient Batch-Aware Sequence Parallelism
 *   for LLM Training" (evolve.pub), section "Summary" and FAQ "What is
 *   Batch-Aware Sequence Parallelism (BASP)?": N ranks are split into disjoint,
 *   contiguous groups of K ranks; every group owns its own sequences and runs
 *   an independent K-way all-to-all during attention, and every rank keeps
 *   B*S/N tokens.  Ulysses (fugumt.com related-papers entry "DeepSpeed
 *   Ulysses") is the K = N case: one N-way all-to-all over a sequence-
 *   partitioned input.  The same review, section "Strengths" (Section IV.C of
 *   the paper), writes both as G groups holding B/G sequences each; here
 *   G = N/K and Bg = B/G.
 *
 *   Logical tensor X[b][s][h][e], b < B, s < S, h < H, e < d, row-major.
 *   Rank r = g*K + j (group g, member j).
 *     seq-sharded  (before attention): rank r holds X[g*Bg .. g*Bg+Bg-1]
 *                  [j*S/K .. (j+1)*S/K - 1][all H][all d], stored
 *                  [Bg][S/K][H][d].
 *     head-sharded (during attention): rank r holds X[g*Bg .. g*Bg+Bg-1]
 *                  [all S][j*H/K .. (j+1)*H/K - 1][all d], stored
 *                  [Bg][S][H/K][d].
 *   The N rank shards lie back to back, rank 0 first; each has
 *   P = Bg*(S/K)*H*d = B*S*H*d/N elements.
 *
 *   seq2head moves every element from its seq-sharded place to its
 *   head-sharded place; head2seq is the inverse.  Elements are opaque
 *   `esz`-byte words, so the result is a pure bit copy (no rounding).
 *
 * Readings where the BASP review and abstract are silent:
 *   - batch-first [B, S, H, d] order inside a shard (the *_ordered entry
 *     points also take the sequence-first [S, B, H, d] order of Megatron-style
 *     stacks: shards [S/K][Bg][H][d] and [S][Bg][H/K][d]);
 *   - member j of a group holds the j-th contiguous block of S/K tokens;
 *   - member j' receives the j'-th contiguous block of H/K heads.
 *
 * Return value: 0 on success, -1 if the shape breaks a divisibility rule
 * (N % K, B % (N/K), S % K, H % K -- the review's FAQ "What are BASP's main
 * limitations?" requires heads to divide evenly across group members).
 */
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

static int shape_ok(int64_t B, int64_t S, int64_t H, int64_t d, int64_t N,
                    int64_t K, int64_t esz)
{
    if (B < 0 || S < 0 || H < 1 || d < 1 || N < 1 || K < 1 || esz < 1)
        return 0;
    if (N % K != 0) return 0;
    if (B % (N / K) != 0) return 0;
    if (S % K != 0) return 0;
    if (H % K != 0) return 0;
    return 1;
}

/*
 * One source-driven walk over every element of the seq-sharded layout.
 * dir = 0: seq2head (read seq-sharded `a`, write head-sharded `b`).
 * dir = 1: head2seq (read head-sharded `b`, write seq-sharded `a`).
 * `a` and `b` are byte pointers; offsets below are in elements.
 * order = 0: batch-first shards ([Bg][S/K][H][d] and [Bg][S][H/K][d]);
 * order = 1: sequence-first shards ([S/K][Bg][H][d] and [S][Bg][H/K][d]), the
 *            [S, B, H, d] activation order of Megatron-style stacks.
 */
static int walk_ordered(int64_t B, int64_t S, int64_t H, int64_t d, int64_t N,
                        int64_t K, int64_t esz, unsigned char *a,
                        unsigned char *b, int dir, int order);

static int walk(int64_t B, int64_t S, int64_t H, int64_t d, int64_t N,
                int64_t K, int64_t esz, unsigned char *a, unsigned char *b,
                int dir)
{
    return walk_ordered(B, S, H, d, N, K, esz, a, b, dir, 0);
}

static int walk_ordered(int64_t B, int64_t S, int64_t H, int64_t d, int64_t N,
                        int64_t K, int64_t esz, unsigned char *a,
                        unsigned char *b, int dir, int order)
{
    if (!shape_ok(B, S, H, d, N, K, esz)) return -1;
    const int64_t G  = N / K;        /* groups                      */
    const int64_t Bg = B / G;        /* sequences per group         */
    const int64_t Sk = S / K;        /* tokens per rank, seq-sharded */
    const int64_t Hk = H / K;        /* heads per rank, head-sharded */
    const int64_t P  = Bg * Sk * H * d;  /* elements per rank shard */

    for (int64_t r_in = 0; r_in < N; ++r_in) {
        const int64_t g = r_in / K;      /* group of the source rank   */
        const int64_t j = r_in % K;      /* its place in the group     */
        for (int64_t bl = 0; bl < Bg; ++bl) {
            for (int64_t sl = 0; sl < Sk; ++sl) {
                const int64_t s = j * Sk + sl;           /* global token  */
                for (int64_t h = 0; h < H; ++h) {
                    const int64_t jp = h / Hk;           /* member that gets head h */
                    const int64_t hl = h % Hk;
                    const int64_t r_out = g * K + jp;
                    /* token position inside each shard, by order */
                    const int64_t t_in  = order ? sl * Bg + bl : bl * Sk + sl;
                    const int64_t t_out = order ? s * Bg + bl  : bl * S + s;
                    for (int64_t e = 0; e < d; ++e) {
                        const int64_t src = r_in * P + (t_in * H + h) * d + e;
                        const int64_t dst = r_out * P + (t_out * Hk + hl) * d + e;
                        if (dir == 0)
                            memcpy(b + dst * esz, a + src * esz, (size_t)esz);
                        else
                            memcpy(a + src * esz, b + dst * esz, (size_t)esz);
                    }
                }
            }
        }
    }
    return 0;
}

int basp_oracle_seq2head_ordered(int64_t B, int64_t S, int64_t H, int64_t d,
                                 int64_t N, int64_t K, int64_t esz, int order,
                                 const void *in, void *out)
{
    if (order != 0 && order != 1) return -1;
    return walk_ordered(B, S, H, d, N, K, esz, (unsigned char *)in,
                        (unsigned char *)out, 0, order);
}

int basp_oracle_head2seq_ordered(int64_t B, int64_t S, int64_t H, int64_t d,
                                 int64_t N, int64_t K, int64_t esz, int order,
                                 const void *in, void *out)
{
    if (order != 0 && order != 1) return -1;
    return walk_ordered(B, S, H, d, N, K, esz, (unsigned char *)out,
                        (unsigned char *)in, 1, order);
}

int basp_oracle_seq2head(int64_t B, int64_t S, int64_t H, int64_t d,
                         int64_t N, int64_t K, int64_t esz,
                         const void *in, void *out)
{
    return walk(B, S, H, d, N, K, esz, (unsigned char *)in,
                (unsigned char *)out, 0);
}

int basp_oracle_head2seq(int64_t B, int64_t S, int64_t H, int64_t d,
                         int64_t N, int64_t K, int64_t esz,
                         const void *in, void *out)
{
    return walk(B, S, H, d, N, K, esz, (unsigned char *)out,
                (unsigned char *)in, 1);
}

/*
 * Destination-driven single-element form, for sampled checks at sizes where a
 * full copy is not wanted.  Given the flat element index `o` of a head-sharded
 * buffer, return the flat element index of the seq-sharded buffer it comes
 * from (the same map read backwards serves head2seq).  Returns -1 for a bad
 * shape or an index out of range.
 */
int64_t basp_oracle_head_to_seq_index(int64_t B, int64_t S, int64_t H,
                                      int64_t d, int64_t N, int64_t K,
                                      int64_t o)
{
    if (!shape_ok(B, S, H, d, N, K, 1)) return -1;
    const int64_t G  = N / K;
    const int64_t Bg = B / G;
    const int64_t Sk = S / K;
    const int64_t Hk = H / K;
    const int64_t P  = Bg * Sk * H * d;
    if (o < 0 || o >= N * P) return -1;

    /* head-sharded place: rank r_out = g*K + jp, [bl][s][hl][e] */
    const int64_t r_out = o / P;
    int64_t rem = o % P;
    const int64_t e  = rem % d;   rem /= d;
    const int64_t hl = rem % Hk;  rem /= Hk;
    const int64_t s  = rem % S;   rem /= S;
    const int64_t bl = rem;
    const int64_t g  = r_out / K;
    const int64_t jp = r_out % K;

    /* seq-sharded place: rank r_in = g*K + j, [bl][sl][h][e] */
    const int64_t j  = s / Sk;
    const int64_t sl = s % Sk;
    const int64_t h  = jp * Hk + hl;
    const int64_t r_in = g * K + j;
    return r_in * P + ((bl * Sk + sl) * H + h) * d + e;
}

/*
 * All-core form, for timing the oracle on every host core (the single-thread
 * walk above stays the reference form; the tests check that both give the
 * same bytes).  The source rows -- the flattened (r_in, bl, sl) index, one
 * token of one rank's shard with all H heads -- are cut into `nthreads`
 * contiguous spans, one per POSIX thread.  Every element has exactly one
 * destination (the map is a bijection), so the threads write disjoint bytes
 * and need no locking.  Per element the destination is computed exactly as
 * in walk_ordered.
 */
struct span {
    int64_t B, S, H, d, N, K, esz;
    unsigned char *a, *b;
    int dir, order;
    int64_t lo, hi;           /* source rows [lo, hi) */
};

static void *walk_span(void *arg)
{
    const struct span *w = (const struct span *)arg;
    const int64_t K = w->K, H = w->H, d = w->d, esz = w->esz;
    const int64_t G  = w->N / K;
    const int64_t Bg = w->B / G;
    const int64_t Sk = w->S / K;
    const int64_t Hk = H / K;
    const int64_t P  = Bg * Sk * H * d;
    for (int64_t row = w->lo; row < w->hi; ++row) {
        const int64_t r_in = row / (Bg * Sk);
        const int64_t bl   = (row / Sk) % Bg;
        const int64_t sl   = row % Sk;
        const int64_t g = r_in / K;
        const int64_t j = r_in % K;
        const int64_t s = j * Sk + sl;
        const int64_t t_in  = w->order ? sl * Bg + bl : bl * Sk + sl;
        const int64_t t_out = w->order ? s * Bg + bl  : bl * w->S + s;
        for (int64_t h = 0; h < H; ++h) {
            const int64_t jp = h / Hk;
            const int64_t hl = h % Hk;
            const int64_t r_out = g * K + jp;
            for (int64_t e = 0; e < d; ++e) {
                const int64_t src = r_in * P + (t_in * H + h) * d + e;
                const int64_t dst = r_out * P + (t_out * Hk + hl) * d + e;
                if (w->dir == 0)
                    memcpy(w->b + dst * esz, w->a + src * esz, (size_t)esz);
                else
                    memcpy(w->a + src * esz, w->b + dst * esz, (size_t)esz);
            }
        }
    }
    return NULL;
}

static int walk_threads(int64_t B, int64_t S, int64_t H, int64_t d, int64_t N,
                        int64_t K, int64_t esz, unsigned char *a,
                        unsigned char *b, int dir, int order, int nthreads)
{
    if (!shape_ok(B, S, H, d, N, K, esz) || (order != 0 && order != 1) ||
        nthreads < 1)
        return -1;
    const int64_t rows = N * (B / (N / K)) * (S / K);
    if (nthreads > 1024) nthreads = 1024;
    if (rows < nthreads) nthreads = rows > 0 ? (int)rows : 1;
    struct span *w = (struct span *)malloc(sizeof(struct span) * (size_t)nthreads);
    pthread_t *tid = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    unsigned char *running = (unsigned char *)calloc((size_t)nthreads, 1);
    if (w == NULL || tid == NULL || running == NULL) {
        free(w);
        free(tid);
        free(running);
        return -1;
    }
    int rc = 0;
    for (int i = 0; i < nthreads; ++i) {
        const struct span x = {B, S, H, d, N, K, esz, a, b, dir, order,
                               rows * i / nthreads, rows * (i + 1) / nthreads};
        w[i] = x;
        if (i == 0) continue;              /* span 0 runs on this thread */
        if (pthread_create(&tid[i], NULL, walk_span, &w[i]) == 0)
            running[i] = 1;
        else
            walk_span(&w[i]);              /* no thread: do the span here */
    }
    walk_span(&w[0]);
    for (int i = 1; i < nthreads; ++i)
        if (running[i] && pthread_join(tid[i], NULL) != 0) rc = -1;
    free(running);
    free(w);
    free(tid);
    return rc;
}

int basp_oracle_seq2head_threads(int64_t B, int64_t S, int64_t H, int64_t d,
                                 int64_t N, int64_t K, int64_t esz, int order,
                                 int nthreads, const void *in, void *out)
{
    return walk_threads(B, S, H, d, N, K, esz, (unsigned char *)in,
                        (unsigned char *)out, 0, order, nthreads);
}

int basp_oracle_head2seq_threads(int64_t B, int64_t S, int64_t H, int64_t d,
                                 int64_t N, int64_t K, int64_t esz, int order,
                                 int nthreads, const void *in, void *out)
{
    return walk_threads(B, S, H, d, N, K, esz, (unsigned char *)out,
                        (unsigned char *)in, 1, order, nthreads);
}
