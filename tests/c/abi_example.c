/*
 * abi_example.c -- a C program that uses libbasp through include/basp.h only,
 * the way a C or C++ caller would (no Python).  Test program.
 *
 *   abi_example           host-only checks: layout rules, derived sizes,
 *                         validation errors (no GPU needed)
 *   abi_example gpu       also re-lays out Q, K, V and O in cudaMalloc'd
 *                         buffers on the current device and compares every
 *                         byte with the CPU oracle (libbasp_oracle.so)
 *
 * Exit status 0 on success; a message on stderr and status 1 otherwise.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "basp.h"

/* the oracle's entry points (test infrastructure, plain C) */
int basp_oracle_seq2head(int64_t B, int64_t S, int64_t H, int64_t d, int64_t N,
                         int64_t K, int64_t esz, const void *in, void *out);
int basp_oracle_head2seq(int64_t B, int64_t S, int64_t H, int64_t d, int64_t N,
                         int64_t K, int64_t esz, const void *in, void *out);

#define CHECK(cond, ...)                                                  \
    do {                                                                  \
        if (!(cond)) {                                                    \
            fprintf(stderr, "abi_example: " __VA_ARGS__);                 \
            fprintf(stderr, "\n");                                        \
            exit(1);                                                      \
        }                                                                 \
    } while (0)

static void host_checks(void) {
    basp_layout *L = NULL;
    basp_info info;
    /* BASP rule: K = N / B */
    CHECK(basp_layout_create(2, 8192, 32, 8, 64, 8, 0, BASP_DTYPE_BF16, &L) == BASP_OK,
          "create failed");
    CHECK(basp_layout_query(L, &info) == BASP_OK, "query failed");
    CHECK(info.K == 4 && info.groups == 2 && info.seqs_per_group == 1, "groups");
    CHECK(info.peers == 3, "peers %lld", (long long)info.peers);
    CHECK(info.tokens_per_rank * info.N == info.B * info.S, "tokens per rank");
    CHECK(info.bytes_per_peer_q == 2048LL * 8 * 64 * 2, "bytes per peer");
    basp_layout_destroy(L);
    /* rule violations leave *out NULL */
    L = (basp_layout *)1;
    CHECK(basp_layout_create(16, 64, 8, 8, 16, 8, 0, BASP_DTYPE_BF16, &L) ==
              BASP_ERR_BATCH_GT_RANKS && L == NULL, "B > N");
    CHECK(basp_layout_create(2, 62, 8, 8, 16, 8, 4, BASP_DTYPE_BF16, &L) ==
              BASP_ERR_DIVISIBILITY && L == NULL, "S %% K");
    CHECK(strlen(basp_status_string(BASP_ERR_ALIASING)) > 0, "status string");
    /* validation before any CUDA call: an output overlapping its input */
    CHECK(basp_layout_create(2, 64, 8, 8, 16, 4, 2, BASP_DTYPE_FP32, &L) == BASP_OK, "create");
    char *fake = (char *)(uintptr_t)(1ull << 40);
    CHECK(basp_seq2head(L, BASP_ALGO_FUSED, fake, NULL, NULL, fake + 64, NULL, NULL,
                        NULL, 0, 0) == BASP_ERR_ALIASING, "aliasing");
    basp_layout_destroy(L);
}

static void gpu_checks(void) {
    const int64_t B = 2, S = 512, Hq = 32, Hkv = 8, d = 64, N = 8, K = 4;
    const int64_t nq = B * S * Hq * d, nkv = B * S * Hkv * d;
    const int64_t n[4] = {nq, nkv, nkv, nq};
    uint16_t *h_in[4], *h_out[4], *h_ref[4];
    void *d_in[4], *d_out[4];
    for (int t = 0; t < 4; ++t) {
        h_in[t] = malloc(n[t] * 2);
        h_out[t] = malloc(n[t] * 2);
        h_ref[t] = malloc(n[t] * 2);
        CHECK(h_in[t] && h_out[t] && h_ref[t], "malloc");
        uint32_t x = 12345u + 7919u * (uint32_t)t;          /* xorshift bits */
        for (int64_t i = 0; i < n[t]; ++i) {
            x ^= x << 13; x ^= x >> 17; x ^= x << 5;
            h_in[t][i] = (uint16_t)x;
        }
        CHECK(cudaMalloc(&d_in[t], n[t] * 2) == cudaSuccess, "cudaMalloc");
        CHECK(cudaMalloc(&d_out[t], n[t] * 2) == cudaSuccess, "cudaMalloc");
        CHECK(cudaMemcpy(d_in[t], h_in[t], n[t] * 2, cudaMemcpyHostToDevice) == cudaSuccess,
              "H2D");
    }
    basp_layout *L = NULL;
    CHECK(basp_layout_create(B, S, Hq, Hkv, d, N, K, BASP_DTYPE_BF16, &L) == BASP_OK, "create");
    cudaStream_t s;
    CHECK(cudaStreamCreate(&s) == cudaSuccess, "stream");
    CHECK(basp_seq2head(L, BASP_ALGO_FUSED, d_in[0], d_in[1], d_in[2], d_out[0], d_out[1],
                        d_out[2], NULL, 0, s) == BASP_OK, "seq2head");
    CHECK(basp_head2seq(L, BASP_ALGO_FUSED, d_in[3], NULL, NULL, d_out[3], NULL, NULL,
                        NULL, 0, s) == BASP_OK, "head2seq");
    CHECK(cudaStreamSynchronize(s) == cudaSuccess, "sync");
    const int64_t H[4] = {Hq, Hkv, Hkv, Hq};
    for (int t = 0; t < 4; ++t) {
        CHECK(cudaMemcpy(h_out[t], d_out[t], n[t] * 2, cudaMemcpyDeviceToHost) == cudaSuccess,
              "D2H");
        if (t < 3)
            CHECK(basp_oracle_seq2head(B, S, H[t], d, N, K, 2, h_in[t], h_ref[t]) == 0, "oracle");
        else
            CHECK(basp_oracle_head2seq(B, S, H[t], d, N, K, 2, h_in[t], h_ref[t]) == 0, "oracle");
        CHECK(memcmp(h_out[t], h_ref[t], n[t] * 2) == 0, "tensor %d differs from the oracle", t);
        cudaFree(d_in[t]);
        cudaFree(d_out[t]);
        free(h_in[t]); free(h_out[t]); free(h_ref[t]);
    }
    cudaStreamDestroy(s);
    basp_layout_destroy(L);
}

int main(int argc, char **argv) {
    host_checks();
    if (argc > 1 && strcmp(argv[1], "gpu") == 0) gpu_checks();
    printf("abi_example ok\n");
    return 0;
}
