// relayout_tma.cuh -- an alternative fused re-layout kernel that moves rows
// with the Tensor Memory Accelerator's bulk copies (cp.async.bulk) through
// shared memory instead of 16-byte register loads.  Built only with
// -DBASP_TMA=1 (included by relayout.cu under that switch) for comparison
// with the register-copy kernel of relayout_kernel.cuh.
//
// One warp per CTA copies one tile of up to kTmaTileBytes: `nrows` rows of one
// block.  The side whose rows are contiguous (the head-sharded side of the
// fused passes) moves as one bulk copy of nrows * row_bytes; the strided side
// moves as one bulk copy per row, issued by the 32 lanes in turn.  Loads
// complete on an mbarrier; its wait is bounded (a timed-out wait records an
// error code in g_basp_tma_error, keeps waiting a second bounded period for
// the copies in flight, and returns).  Stores are bulk-group copies that the
// issuing lane waits to have finished reading shared memory before the CTA
// exits.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

namespace {

constexpr int kTmaTileBytes = 16384;

struct RowJob {
    const unsigned char *src;
    unsigned char *dst;
    int64_t src_bs[4], dst_bs[4];   // block-digit strides, in bytes
    int64_t src_rs, dst_rs;         // row strides, in bytes
    uint32_t radix[4];
    uint32_t row_bytes;             // multiple of 16
    uint32_t rows;                  // rows per block
    uint32_t rows_per_tile;
    uint32_t tiles_per_block;
    uint32_t tile_begin;
};

struct RowParams {
    RowJob job[3];
    int njobs;
    uint32_t total_tiles;
};

__device__ unsigned int g_basp_tma_error;

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
    return ok != 0;
}

// Bounded wait for phase 0 of `bar`; false if it gave up.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t limit) {
    for (uint32_t i = 0; i < limit; ++i)
        if (mbar_try_wait(bar, 0)) return true;
    return false;
}

__device__ __forceinline__ void bulk_load(uint32_t smem, const void *gmem,
                                          uint32_t bytes, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes "
        "[%0], [%1], %2, [%3];"
        :: "r"(smem), "l"(gmem), "r"(bytes), "r"(bar) : "memory");
}

__device__ __forceinline__ void bulk_store(void *gmem, uint32_t smem, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;"
                 :: "l"(gmem), "r"(smem), "r"(bytes) : "memory");
}

__global__ void __launch_bounds__(32)
basp_relayout_tma_kernel(const __grid_constant__ RowParams p) {
    __shared__ __align__(128) unsigned char tile[kTmaTileBytes];
    __shared__ __align__(8) uint64_t bar_storage;
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" :::);

    const uint32_t lane = threadIdx.x;
    const uint32_t t = blockIdx.x;
    if (t >= p.total_tiles) return;
    int jb = 0;
    if (p.njobs > 1 && t >= p.job[1].tile_begin) jb = 1;
    if (p.njobs > 2 && t >= p.job[2].tile_begin) jb = 2;
    const RowJob &J = p.job[jb];

    // tile -> block digits (digit 3 fastest) and the tile's first row
    uint32_t lt = t - J.tile_begin;
    uint32_t q = lt / J.tiles_per_block;
    const uint32_t tb = lt - q * J.tiles_per_block;
    lt = q;
    int64_t sb = 0, db = 0;
#pragma unroll
    for (int k = 3; k >= 1; --k) {
        q = lt / J.radix[k];
        const uint32_t dgt = lt - q * J.radix[k];
        sb += int64_t(dgt) * J.src_bs[k];
        db += int64_t(dgt) * J.dst_bs[k];
        lt = q;
    }
    sb += int64_t(lt) * J.src_bs[0];
    db += int64_t(lt) * J.dst_bs[0];
    const uint32_t row0 = tb * J.rows_per_tile;
    const uint32_t nrows = min(J.rows_per_tile, J.rows - row0);
    const uint32_t bytes = nrows * J.row_bytes;
    const unsigned char *src = J.src + sb + int64_t(row0) * J.src_rs;
    unsigned char *dst = J.dst + db + int64_t(row0) * J.dst_rs;

    const uint32_t bar = uint32_t(__cvta_generic_to_shared(&bar_storage));
    const uint32_t sm = uint32_t(__cvta_generic_to_shared(tile));
    if (lane == 0) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" :: "r"(bar) : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                     :: "r"(bar), "r"(bytes) : "memory");
    }
    __syncwarp();
    if (J.src_rs == J.row_bytes) {                 // contiguous source rows
        if (lane == 0) bulk_load(sm, src, bytes, bar);
    } else {
        for (uint32_t r = lane; r < nrows; r += 32)
            bulk_load(sm + r * J.row_bytes, src + int64_t(r) * J.src_rs, J.row_bytes, bar);
    }
    if (!mbar_wait_bounded(bar, 1u << 22)) {
        if (lane == 0) atomicCAS(&g_basp_tma_error, 0u, 1u);
        mbar_wait_bounded(bar, 1u << 24);          // let the copies in flight land
        return;
    }
    if (J.dst_rs == J.row_bytes) {                 // contiguous destination rows
        if (lane == 0) bulk_store(dst, sm, bytes);
    } else {
        for (uint32_t r = lane; r < nrows; r += 32)
            bulk_store(dst + int64_t(r) * J.dst_rs, sm + r * J.row_bytes, J.row_bytes);
    }
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

}  // namespace
