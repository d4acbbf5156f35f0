// relayout_kernel.cuh -- device side of the re-layout: the one copy kernel
// every pass launches, its job table and its load/store helpers.  Included
// once, by relayout.cu.
//
// Each CTA copies one tile of THREADS * kUnroll vectors: 16 KiB at 16-byte
// vectors and 256 threads, 32 KiB with the 512-thread CTAs of long launches.
// A tile lies inside one block of rows (fixed g, j, jp, bl); the block's
// source and destination bases come from its four digits times the job's
// stride tables, and vector i of the block sits in row i / vpr, column
// i % vpr.  Loads are non-coherent and skip L1; stores are plain (the written
// lines stay in L2 at normal priority).  Every thread issues its kUnroll
// loads before its stores.  Every CTA first prefetches its tile's source
// lines into L2; the ones resident before the previous kernel on the stream
// has finished do so while it drains, before they wait for it.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

namespace {

// Build-time tuning switches (-DBASP_...=); the defaults are the settings
// that measured best on GB300.  None of them changes what is copied where.
//   BASP_THREADS, BASP_UNROLL  tile shape: threads per CTA, vectors per thread
//   BASP_THREADS_LARGE         threads per CTA of long launches (0: always
//                              BASP_THREADS); BASP_LARGE_WAVES sets "long"
//   BASP_STORE_CS              evict-first stores (1) or plain stores (0)
//   BASP_RECOMPUTE_DST         recompute store offsets instead of keeping them
//   BASP_CTAS_PER_SM           cap on resident CTAs for persistent grids
//   BASP_PDL                   programmatic dependent launch
//   BASP_GRID_ALL_TILES        one CTA per tile (1) or a persistent grid (0)
//   BASP_PREFETCH              L2 prefetch of the first tile before the wait
//                              for the previous kernel: 0 none, 1 the CTAs of
//                              the first wave, 2 every CTA
//   BASP_CHECK_BOUNDS          debug build: every access is checked against
//                              its buffer's extent; an access outside it is
//                              counted (g_basp_bounds_violations) and skipped
#ifndef BASP_THREADS
#define BASP_THREADS 256
#endif
#ifndef BASP_UNROLL
#define BASP_UNROLL 4
#endif
#ifndef BASP_THREADS_LARGE
#define BASP_THREADS_LARGE 512
#endif
#ifndef BASP_LARGE_WAVES
#define BASP_LARGE_WAVES 8
#endif
#ifndef BASP_STORE_CS
#define BASP_STORE_CS 0         // plain stores: with the L2 prefetch they beat .cs
#endif
#ifndef BASP_RECOMPUTE_DST
#define BASP_RECOMPUTE_DST 0
#endif
#ifndef BASP_CTAS_PER_SM
#define BASP_CTAS_PER_SM 0      // 0: as many as fit
#endif
#ifndef BASP_PDL
#define BASP_PDL 1              // programmatic dependent launch (0: plain launch)
#endif
#ifndef BASP_CHECK_BOUNDS
#define BASP_CHECK_BOUNDS 0
#endif
#ifndef BASP_GRID_ALL_TILES
#define BASP_GRID_ALL_TILES 1   // 0: persistent grid (SMs x resident CTAs)
#endif
#ifndef BASP_PREFETCH
#define BASP_PREFETCH 2
#endif
constexpr int kThreads = BASP_THREADS;   // threads per CTA
// threads per CTA of launches of at least BASP_LARGE_WAVES waves of
// kThreads-thread CTAs (device memory, 16-byte vectors)
constexpr int kThreadsLarge = BASP_THREADS_LARGE > 0 ? BASP_THREADS_LARGE : BASP_THREADS;
constexpr int kUnroll = BASP_UNROLL;     // vectors in flight per thread
constexpr int kMaxJobs = 3;

enum Coord { C_G = 0, C_J = 1, C_JP = 2, C_BL = 3, C_SL = 4 };
enum BufKind { SEQ, HEAD, BYSRC, BYDST };

// One tensor's share of one launch.
struct Job {
    const unsigned char *src;
    unsigned char *dst;
    int64_t src_bs[4], dst_bs[4];   // block-digit strides, in vectors
    int64_t src_rs, dst_rs;         // row strides, in vectors
    uint32_t radix[4];              // block-digit radices; digit 3 fastest
    uint32_t vpr;                   // vectors per row
    uint32_t vpr_magic, vpr_shift;  // i / vpr == (umulhi(i, magic) + i) >> shift
    uint32_t vec_per_block;         // rows * vpr  (< 2^31)
    uint32_t tiles_per_block;
    uint32_t tile_begin;            // first tile of this job within the launch
    uint32_t inner_fast;            // 1: digit 3 varies fastest across tiles
    int64_t src_lo, src_hi;         // extent of the source buffer, in vectors
    int64_t dst_lo, dst_hi;         // from src / dst (checked in debug builds)
};

struct Params {
    Job job[kMaxJobs];
    int njobs;
    uint32_t total_tiles;
    uint32_t prefetch_ctas;   // CTAs below this index prefetch their first tile
};

template <int VEC> struct Word;
template <> struct Word<16> { using T = uint4; };
template <> struct Word<8> { using T = uint2; };
template <> struct Word<4> { using T = uint32_t; };
template <> struct Word<2> { using T = unsigned short; };
template <> struct Word<1> { using T = unsigned char; };

__device__ __forceinline__ uint4 load_stream(const uint4 *p) {
    uint4 v;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}
__device__ __forceinline__ uint2 load_stream(const uint2 *p) {
    uint2 v;
    asm("ld.global.nc.L1::no_allocate.v2.u32 {%0, %1}, [%2];"
        : "=r"(v.x), "=r"(v.y) : "l"(p));
    return v;
}
__device__ __forceinline__ uint32_t load_stream(const uint32_t *p) {
    uint32_t v;
    asm("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}
__device__ __forceinline__ unsigned char load_stream(const unsigned char *p) {
    unsigned short v;
    asm("ld.global.nc.L1::no_allocate.u8 %0, [%1];" : "=h"(v) : "l"(p));
    return static_cast<unsigned char>(v);
}
__device__ __forceinline__ unsigned short load_stream(const unsigned short *p) {
    unsigned short v;
    asm("ld.global.nc.L1::no_allocate.u16 %0, [%1];" : "=h"(v) : "l"(p));
    return v;
}

#if BASP_STORE_CS
#define BASP_ST "st.global.cs"
#else
#define BASP_ST "st.global"
#endif

__device__ __forceinline__ void store(uint4 *p, uint4 v) {
    asm volatile(BASP_ST ".v4.u32 [%0], {%1, %2, %3, %4};"
                 :: "l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}
__device__ __forceinline__ void store(uint2 *p, uint2 v) {
    asm volatile(BASP_ST ".v2.u32 [%0], {%1, %2};"
                 :: "l"(p), "r"(v.x), "r"(v.y) : "memory");
}
__device__ __forceinline__ void store(uint32_t *p, uint32_t v) {
    asm volatile(BASP_ST ".u32 [%0], %1;" :: "l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void store(unsigned char *p, unsigned char v) {
    const unsigned short w = v;
    asm volatile(BASP_ST ".u8 [%0], %1;" :: "l"(p), "h"(w) : "memory");
}
__device__ __forceinline__ void store(unsigned short *p, unsigned short v) {
    asm volatile(BASP_ST ".u16 [%0], %1;" :: "l"(p), "h"(v) : "memory");
}

#if BASP_CHECK_BOUNDS
__device__ unsigned long long g_basp_bounds_violations;
#endif

// One tile located: its job, the source and destination bases of its block
// (in vectors), and its vector range [i0, i1) within the block.
struct Tile {
    const Job *J;
    int64_t sb, db;
    uint32_t i0, i1;
};

// tile -> (job, block digits, tile within block).  Tiles run either block by
// block (inner_fast = 0) or with the innermost block digit varying fastest,
// so that consecutive tiles fill neighbouring row segments.
template <int THREADS>
__device__ __forceinline__ Tile locate(const Params &p, uint32_t t) {
    constexpr uint32_t kTile = uint32_t(THREADS * kUnroll);
    int jb = 0;
    if (p.njobs > 1 && t >= p.job[1].tile_begin) jb = 1;
    if (p.njobs > 2 && t >= p.job[2].tile_begin) jb = 2;
    const Job &J = p.job[jb];
    uint32_t lt = t - J.tile_begin;
    uint32_t tb, q;
    int64_t sb = 0, db = 0;
    if (J.inner_fast) {
        q = lt / J.radix[3];
        const uint32_t d3 = lt - q * J.radix[3];
        sb += int64_t(d3) * J.src_bs[3];
        db += int64_t(d3) * J.dst_bs[3];
        lt = q;
        q = lt / J.tiles_per_block;
        tb = lt - q * J.tiles_per_block;
        lt = q;
    } else {
        q = lt / J.tiles_per_block;
        tb = lt - q * J.tiles_per_block;
        lt = q;
        q = lt / J.radix[3];
        const uint32_t d3 = lt - q * J.radix[3];
        sb += int64_t(d3) * J.src_bs[3];
        db += int64_t(d3) * J.dst_bs[3];
        lt = q;
    }
#pragma unroll
    for (int k = 2; k >= 1; --k) {
        q = lt / J.radix[k];
        const uint32_t dgt = lt - q * J.radix[k];
        sb += int64_t(dgt) * J.src_bs[k];
        db += int64_t(dgt) * J.dst_bs[k];
        lt = q;
    }
    sb += int64_t(lt) * J.src_bs[0];
    db += int64_t(lt) * J.dst_bs[0];
    Tile T;
    T.J = &J;
    T.sb = sb;
    T.db = db;
    T.i0 = tb * kTile;
    T.i1 = min(T.i0 + kTile, J.vec_per_block);
    return T;
}

// Row and column of vector i of a block: row = i / vpr by the job's
// multiply-high constants, col = i - row * vpr.
__device__ __forceinline__ uint32_t row_of(const Job &J, uint32_t i) {
    return (__umulhi(i, J.vpr_magic) + i) >> J.vpr_shift;
}

// Ask L2 for the lines the tile will read.  A prefetch hands no value to the
// thread, so it may run before the previous kernel on the stream has finished:
// L2 is where every SM's accesses meet, so a line that kernel writes later is
// updated there, and the loads after griddepcontrol.wait see its final value.
template <int VEC, int THREADS>
__device__ __forceinline__ void prefetch_tile(const Tile &T) {
    using W = typename Word<VEC>::T;
    const Job &J = *T.J;
    const W *src = reinterpret_cast<const W *>(J.src) + T.sb;
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
        const uint32_t i = T.i0 + threadIdx.x + uint32_t(u * THREADS);
        if (i < T.i1) {
            const uint32_t row = row_of(J, i);
            const int64_t so = int64_t(row) * J.src_rs + (i - row * J.vpr);
#if BASP_CHECK_BOUNDS
            if (T.sb + so < J.src_lo || T.sb + so >= J.src_hi) continue;
#endif
            asm volatile("prefetch.global.L2 [%0];" :: "l"(src + so));
        }
    }
}

template <int VEC, int THREADS>
__device__ __forceinline__ void copy_tile(const Tile &T) {
    using W = typename Word<VEC>::T;
    const Job &J = *T.J;
    const W *src = reinterpret_cast<const W *>(J.src) + T.sb;
    W *dst = reinterpret_cast<W *>(J.dst) + T.db;
#if BASP_CHECK_BOUNDS
    for (int u = 0; u < kUnroll; ++u) {
        const uint32_t i = T.i0 + threadIdx.x + uint32_t(u * THREADS);
        if (i < T.i1) {
            const uint32_t row = row_of(J, i);
            const uint32_t col = i - row * J.vpr;
            const int64_t so = T.sb + int64_t(row) * J.src_rs + col;
            const int64_t dof = T.db + int64_t(row) * J.dst_rs + col;
            if (so < J.src_lo || so >= J.src_hi || dof < J.dst_lo || dof >= J.dst_hi) {
                atomicAdd(&g_basp_bounds_violations, 1ull);
                continue;
            }
            store(reinterpret_cast<W *>(J.dst) + dof,
                  load_stream(reinterpret_cast<const W *>(J.src) + so));
        }
    }
    (void)src;
    (void)dst;
#else
    W v[kUnroll];
#if !BASP_RECOMPUTE_DST
    int64_t doff[kUnroll];
#endif
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
        const uint32_t i = T.i0 + threadIdx.x + uint32_t(u * THREADS);
        if (i < T.i1) {
            const uint32_t row = row_of(J, i);
            const uint32_t col = i - row * J.vpr;
            v[u] = load_stream(src + (int64_t(row) * J.src_rs + col));
#if !BASP_RECOMPUTE_DST
            doff[u] = int64_t(row) * J.dst_rs + col;
#endif
        }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
        const uint32_t i = T.i0 + threadIdx.x + uint32_t(u * THREADS);
        if (i < T.i1) {
#if BASP_RECOMPUTE_DST
            const uint32_t row = row_of(J, i);
            store(dst + (int64_t(row) * J.dst_rs + (i - row * J.vpr)), v[u]);
#else
            store(dst + doff[u], v[u]);
#endif
        }
    }
#endif  // BASP_CHECK_BOUNDS
}

template <int VEC, int THREADS>
__global__ void __launch_bounds__(THREADS)
basp_relayout_kernel(const __grid_constant__ Params p) {
#if BASP_PDL
    // Launched with programmatic stream serialisation: the previous kernel on
    // the stream may still be running.  CTAs below p.prefetch_ctas (all of
    // them by default) warm L2 with their first tile's source lines: in the
    // CTAs resident that early the DRAM latency of the first loads overlaps
    // the previous kernel's tail, and in every CTA the line requests go out
    // ahead of the loads without holding registers.  Then every CTA waits for
    // that kernel (and its memory) before touching any buffer, and lets the
    // next kernel start its own launch.  The tile is located again after the
    // wait, so nothing stays live across it.
    if (blockIdx.x < p.prefetch_ctas && blockIdx.x < p.total_tiles)
        prefetch_tile<VEC, THREADS>(locate<THREADS>(p, blockIdx.x));
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" :::);
#endif
    for (uint32_t t = blockIdx.x; t < p.total_tiles; t += gridDim.x)
        copy_tile<VEC, THREADS>(locate<THREADS>(p, t));
}

}  // namespace
