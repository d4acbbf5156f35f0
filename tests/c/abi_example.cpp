// abi_example.cpp -- the C++ layer (include/basp.hpp) as a C++ caller uses it.
// Test program.
//   abi_example_cpp        host-only: RAII layout, info, errors as exceptions
//   abi_example_cpp gpu    also a seq2head / head2seq round trip on the GPU,
//                          compared with the C oracle
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <vector>

#include <cuda_runtime_api.h>

#include "basp.hpp"

extern "C" int basp_oracle_seq2head(int64_t B, int64_t S, int64_t H, int64_t d, int64_t N,
                                    int64_t K, int64_t esz, const void *in, void *out);

#define CHECK(cond, msg)                                                   \
    do {                                                                   \
        if (!(cond)) {                                                     \
            std::fprintf(stderr, "abi_example_cpp: %s\n", msg);            \
            std::exit(1);                                                  \
        }                                                                  \
    } while (0)

static void host_checks() {
    basp::Layout L(2, 8192, 32, 8, 64, 8, 0);               // BASP rule
    CHECK(L.info().K == 4 && L.info().peers == 3, "derived sizes");
    basp::Layout moved = std::move(L);                      // ownership moves
    CHECK(moved.handle() != nullptr && L.handle() == nullptr, "move");
    bool threw = false;
    try {
        basp::Layout bad(2, 62, 8, 8, 16, 8, 4);             // S % K != 0
    } catch (const basp::Error &e) {
        threw = e.status() == BASP_ERR_DIVISIBILITY && std::strlen(e.what()) > 0;
    }
    CHECK(threw, "divisibility error as exception");
}

static void gpu_checks() {
    const int64_t B = 2, S = 256, Hq = 16, Hkv = 8, d = 32, N = 8, K = 8;
    const int64_t n = B * S * Hq * d;
    std::vector<uint16_t> h(n), out(n), ref(n), back(n);
    for (int64_t i = 0; i < n; ++i) h[i] = uint16_t(i * 2654435761u >> 7);
    void *din, *dout, *dback;
    CHECK(cudaMalloc(&din, n * 2) == cudaSuccess && cudaMalloc(&dout, n * 2) == cudaSuccess &&
          cudaMalloc(&dback, n * 2) == cudaSuccess, "cudaMalloc");
    CHECK(cudaMemcpy(din, h.data(), n * 2, cudaMemcpyHostToDevice) == cudaSuccess, "H2D");
    basp::Layout L(B, S, Hq, Hkv, d, N, K, BASP_DTYPE_BF16);
    L.seq2head(din, nullptr, nullptr, dout, nullptr, nullptr, 0);
    L.head2seq(dout, nullptr, nullptr, dback, nullptr, nullptr, 0);
    CHECK(cudaDeviceSynchronize() == cudaSuccess, "sync");
    CHECK(cudaMemcpy(out.data(), dout, n * 2, cudaMemcpyDeviceToHost) == cudaSuccess, "D2H");
    CHECK(cudaMemcpy(back.data(), dback, n * 2, cudaMemcpyDeviceToHost) == cudaSuccess, "D2H");
    CHECK(basp_oracle_seq2head(B, S, Hq, d, N, K, 2, h.data(), ref.data()) == 0, "oracle");
    CHECK(std::memcmp(out.data(), ref.data(), n * 2) == 0, "seq2head differs from the oracle");
    CHECK(std::memcmp(back.data(), h.data(), n * 2) == 0, "round trip differs");
    cudaFree(din); cudaFree(dout); cudaFree(dback);

    // host buffers through the C++ layer: page-locked, re-laid out in place
    // (no staging), then back; a pageable output is refused as an exception
    void *pin_in, *pin_out, *pin_back;
    CHECK(cudaMallocHost(&pin_in, n * 2) == cudaSuccess &&
          cudaMallocHost(&pin_out, n * 2) == cudaSuccess &&
          cudaMallocHost(&pin_back, n * 2) == cudaSuccess, "cudaMallocHost");
    std::memcpy(pin_in, h.data(), n * 2);
    L.seq2head_host(pin_in, nullptr, nullptr, pin_out, nullptr, nullptr, nullptr, 0, 0);
    L.head2seq_host(pin_out, nullptr, nullptr, pin_back, nullptr, nullptr, nullptr, 0, 0);
    CHECK(cudaDeviceSynchronize() == cudaSuccess, "sync");
    CHECK(std::memcmp(pin_out, ref.data(), n * 2) == 0, "host seq2head differs from the oracle");
    CHECK(std::memcmp(pin_back, h.data(), n * 2) == 0, "host round trip differs");
    bool threw = false;
    try {
        L.seq2head_host(pin_in, nullptr, nullptr, out.data(), nullptr, nullptr, nullptr, 0, 0);
    } catch (const basp::Error &e) {
        threw = e.status() == BASP_ERR_WORKSPACE;
    }
    CHECK(threw, "pageable host output in direct mode must be refused");
    cudaFreeHost(pin_in); cudaFreeHost(pin_out); cudaFreeHost(pin_back);
}

int main(int argc, char **argv) {
    host_checks();
    if (argc > 1 && std::strcmp(argv[1], "gpu") == 0) gpu_checks();
    std::printf("abi_example_cpp ok\n");
    return 0;
}
