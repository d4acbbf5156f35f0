// layout_internal.h -- the host-side layout descriptor behind the opaque
// basp_layout handle, and the pass planner's vocabulary.
#pragma once

#include <cstdint>

#include "basp.h"

struct basp_layout {
    int64_t B, S, Hq, Hkv, d, N, K;
    int64_t G;     // groups, N / K
    int64_t Bg;    // sequences per group, B / G
    int64_t Sk;    // tokens per rank in the seq-sharded layout, S / K
    int64_t esz;   // bytes per element
    basp_dtype dtype;
    basp_order order;
};

namespace basp {

// Bytes of one whole tensor with H heads.
inline int64_t tensor_bytes(const basp_layout &L, int64_t H) {
    return L.B * L.S * H * L.d * L.esz;
}

// Round up to a multiple of 256 bytes (workspace and staging regions).
inline int64_t align256(int64_t x) { return (x + 255) & ~int64_t(255); }

// Workspace of the three-pass path for tensors with head counts H[0..n-1]:
// one send and one receive region per tensor.
inline int64_t workspace_bytes(const basp_layout &L, const int64_t *H, int n) {
    int64_t w = 0;
    for (int i = 0; i < n; ++i) w += 2 * align256(tensor_bytes(L, H[i]));
    return w;
}

}  // namespace basp
