// tl_kernel_common.cuh -- device building blocks of the GEMM kernel
// (tl_gemm.cu): tile geometry, bounded waits, tile order, shared-memory
// operand descriptors and the epilogue paths.
#pragma once
#include "tl_gemm.h"
#include "tl_ptx.cuh"

#include <cuda_bf16.h>

namespace tl {
namespace kc {

constexpr int kUmmaK = 16;
constexpr uint32_t kStageA = kBlockM * kBlockK * 2;  // 128 rows of A per CTA: 16 KiB
constexpr uint32_t kMnChunk = 64 * kBlockK * 2;      // 64 MN elements x 64 K rows = 8 KiB
constexpr uint32_t kTmemCols = 2 * kBlockN;          // two fp32 accumulators of 256 columns
constexpr int kThreads = 256;
constexpr int kFirstEpilogueWarp = 4;
// Epilogue staging: each of the 4 epilogue warps owns boxes of 32 output rows
// x 128 bytes (64 bf16 columns) for its TMA stores.
constexpr uint32_t kEpiBuf = 32 * 128;
constexpr uint32_t kBarBytes = 512;

static_assert(kBlockK * 2 == 128, "one K-block row must be one 128-byte swizzle row");

// Tile geometry.  Single CTA: 128 x 256 output tile, B = 256 rows of N per
// stage.  CTA pair (cta_group::2): 256 x 256 output tile; each CTA loads its
// own 128 rows of A and its own 128 rows (N) of B, and the pair's MMA reads
// both CTAs' shared memory.  EPI_BOXES staging boxes per epilogue warp.
template <bool PAIR, int EPI_BOXES>
struct Geo {
    static constexpr int kTileM = PAIR ? 2 * kBlockM : kBlockM;
    static constexpr int kBRows = PAIR ? kBlockN / 2 : kBlockN;
    static constexpr uint32_t kStageB = uint32_t(kBRows) * kBlockK * 2;
    static constexpr uint32_t kStageBytes = kStageA + kStageB;
    static constexpr uint32_t kEpiBytes = 4u * EPI_BOXES * kEpiBuf;
    // 6 stages in pair mode, with the epilogue's staging boxes beside them
    static constexpr int kStages = PAIR ? 6 : 4;
    static constexpr size_t kSmem = size_t(kStages) * kStageBytes + kEpiBytes + kBarBytes + 1024;
    static_assert(kSmem <= 232448, "shared memory budget");
};

struct WaitCtx {
    int32_t* err;
    uint64_t timeout_ns;
};

__device__ __noinline__ inline bool wait_slow(uint32_t bar, uint32_t parity, int32_t* err, int32_t code,
                                              bool stop_on_error, uint64_t timeout_ns) {
    const uint64_t t0 = global_timer_ns();
    for (uint32_t n = 1;; ++n) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((n & 255u) == 0) {
            if (stop_on_error && *reinterpret_cast<volatile int32_t*>(err) != 0) return false;
            if (global_timer_ns() - t0 > timeout_ns) {
                atomicOr(err, code);
                return false;
            }
        }
    }
}

// The MMA thread's waits use the base limit; the producer's wait for a free
// stage and the epilogue's wait for an accumulator (both downstream of the
// MMA thread) use twice that, so when a pipeline stalls the role nearest the
// stall reports first.
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, const WaitCtx& w, int32_t code,
                                             bool stop_on_error = true) {
    if (mbar_try_wait(bar, parity)) return true;
    const bool downstream = code == kErrProducerWait || code == kErrEpilogueWait;
    return wait_slow(bar, parity, w.err, code, stop_on_error, downstream ? 2 * w.timeout_ns : w.timeout_ns);
}

// Bounded wait with cluster-scope acquire (the dynamic tile queue).
__device__ __noinline__ inline bool wait_bounded_cluster(uint32_t bar, uint32_t parity, const WaitCtx& w,
                                                         int32_t code) {
    const uint64_t t0 = global_timer_ns();
    for (uint32_t n = 1;; ++n) {
        if (mbar_try_wait_cluster(bar, parity)) return true;
        if ((n & 255u) == 0) {
            if (*reinterpret_cast<volatile int32_t*>(w.err) != 0) return false;
            if (global_timer_ns() - t0 > 2 * w.timeout_ns) {
                atomicOr(w.err, code);
                return false;
            }
        }
    }
}

// Warp-uniform wait: lane 0 waits (bounded); then every lane observes the
// completed phase itself, which cannot move on before this warp arrives.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, const WaitCtx& w, int32_t code,
                                          int lane) {
    int ok = 1;
    if (lane == 0) ok = wait_bounded(bar, parity, w, code) ? 1 : 0;
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (!ok) return false;
    // lane 0 has seen the phase complete, so every lane's first test passes;
    // the bound only keeps the loop finite
    int mine = 0;
    for (int n = 0; n < (1 << 10) && !mine; ++n) mine = mbar_try_wait(bar, parity) ? 1 : 0;
    if (!mine) atomicOr(w.err, code);
    return __all_sync(0xffffffffu, mine) != 0;
}

// Output tile order: groups of `group` blocks along one dimension, walking
// the other dimension inside the group, so that the group's blocks of one
// operand stay in L2 while the other operand streams past once per group.
// raster 0: groups of m-blocks (m fastest); 1: groups of n-blocks.
__device__ __forceinline__ void tile_coords(int tile, int num_m, int num_n, int raster, int group, int& mb,
                                            int& nb) {
    const int outer = raster == 0 ? num_m : num_n;
    const int inner = raster == 0 ? num_n : num_m;
    const int group_tiles = group * inner;
    const int g = tile / group_tiles;
    const int first = g * group;
    const int width = min(group, outer - first);
    const int local = tile - g * group_tiles;
    const int a = first + local % width;
    const int b = local / width;
    mb = raster == 0 ? a : b;
    nb = raster == 0 ? b : a;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

// Shared-memory descriptor of UMMA_K step j (16 elements of K) of a stage
// operand: K-major rows advance 32 bytes inside the 128-byte swizzle row,
// MN-major operands advance 16 rows of 128 bytes.
__device__ __forceinline__ uint64_t operand_desc(bool mn_major, uint32_t base, int j) {
    return mn_major ? smem_desc_sw128(base + uint32_t(j) * 2048u, kMnChunk, 1024)
                    : smem_desc_sw128(base + uint32_t(j) * 32u, 16, 1024);
}

// ---- epilogues ---------------------------------------------------------------
// Warp q owns TMEM lanes 32q..32q+31 = output rows row0..row0+31 of the CTA's
// half tile; lane l holds row row0 + l.  t_row addresses the warp's lanes of
// the accumulator.

// bf16: per 64-column chunk, two tcgen05.ld, pack, write the lane's 128-byte
// row into a 128B-swizzled staging box (two per warp, alternating), and lane 0
// issues a TMA store of the 32 x 64 box at (col0 + 64c, row0).
__device__ __forceinline__ void epi_bf16_tma(const CUtensorMap* map, uint32_t t_row, uint32_t epi0, uint32_t& buf,
                                             int nchunks, int col0, int row0, int lane) {
    for (int c = 0; c < nchunks; ++c) {
        uint32_t w[32];
        uint32_t v[32];
        tmem_ld_32cols(t_row + uint32_t(c) * 64u, v);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 16; ++j) w[j] = pack_bf16x2(__uint_as_float(v[2 * j]), __uint_as_float(v[2 * j + 1]));
        tmem_ld_32cols(t_row + uint32_t(c) * 64u + 32u, v);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 16; ++j)
            w[16 + j] = pack_bf16x2(__uint_as_float(v[2 * j]), __uint_as_float(v[2 * j + 1]));
        const uint32_t sbuf = epi0 + buf * kEpiBuf;
        if (lane == 0) bulk_wait_group_read<1>();  // the store that last used sbuf has read it
        __syncwarp();
        const uint32_t row_addr = sbuf + uint32_t(lane) * 128u;
#pragma unroll
        for (int j = 0; j < 8; ++j)
            st_shared_v4(row_addr + ((uint32_t(j) ^ (uint32_t(lane) & 7u)) << 4), w[4 * j], w[4 * j + 1],
                         w[4 * j + 2], w[4 * j + 3]);
        fence_proxy_async_shared();
        __syncwarp();
        if (lane == 0) {
            tma_store_2d(map, sbuf, col0 + c * 64, row0);
            bulk_commit_group();
        }
        buf ^= 1u;
    }
}

// bf16 of (addend + accumulator), for a dX that is the next operator's dY:
// each lane reads its own row of the fp32 addend (ld `ld_add`) with 16-byte
// loads, issued before the chunk's TMEM loads so that the two latencies
// overlap, adds it in fp32 (round to nearest, as a reduce-add in L2 would)
// and rounds the sum to bf16 once.  Rows >= m_dim and columns >= n_dim read
// no addend; the TMA store clips them.
__device__ __forceinline__ void epi_bf16_add_tma(const CUtensorMap* map, uint32_t t_row, uint32_t epi0,
                                                 uint32_t& buf, int nchunks, int col0, int row0, int lane,
                                                 const float* addend, int64_t ld_add, int m_dim, int n_dim) {
    const int row = row0 + lane;
    const float* arow = addend + int64_t(row) * ld_add;
    for (int c = 0; c < nchunks; ++c) {
        const int cb = col0 + c * 64;
        float a[64];
        if (row < m_dim && cb + 64 <= n_dim) {
            const float4* src = reinterpret_cast<const float4*>(arow + cb);
#pragma unroll
            for (int q = 0; q < 16; ++q) {
                const float4 f = __ldg(src + q);
                a[4 * q] = f.x;
                a[4 * q + 1] = f.y;
                a[4 * q + 2] = f.z;
                a[4 * q + 3] = f.w;
            }
        } else {
#pragma unroll
            for (int e = 0; e < 64; ++e) a[e] = (row < m_dim && cb + e < n_dim) ? __ldg(arow + cb + e) : 0.0f;
        }
        uint32_t w[32];
        uint32_t v[32];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            tmem_ld_32cols(t_row + uint32_t(c) * 64u + 32u * uint32_t(h), v);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 16; ++j)
                w[16 * h + j] = pack_bf16x2(__fadd_rn(a[32 * h + 2 * j], __uint_as_float(v[2 * j])),
                                            __fadd_rn(a[32 * h + 2 * j + 1], __uint_as_float(v[2 * j + 1])));
        }
        const uint32_t sbuf = epi0 + buf * kEpiBuf;
        if (lane == 0) bulk_wait_group_read<1>();  // the store that last used sbuf has read it
        __syncwarp();
        const uint32_t row_addr = sbuf + uint32_t(lane) * 128u;
#pragma unroll
        for (int j = 0; j < 8; ++j)
            st_shared_v4(row_addr + ((uint32_t(j) ^ (uint32_t(lane) & 7u)) << 4), w[4 * j], w[4 * j + 1],
                         w[4 * j + 2], w[4 * j + 3]);
        fence_proxy_async_shared();
        __syncwarp();
        if (lane == 0) {
            tma_store_2d(map, sbuf, cb, row0);
            bulk_commit_group();
        }
        buf ^= 1u;
    }
}

// fp32 through TMA: per 32-column chunk, tcgen05.ld of the lane's row into a
// 128B-swizzled staging box (two per warp, alternating), and lane 0 issues a
// TMA store of the 32 x 32 box at (col0 + 32c, row0) -- or, with `add`, a TMA
// reduce-add of it into the values there, so that the read-modify-write
// happens in L2 on whole lines instead of as per-thread loads and stores.
__device__ __forceinline__ void epi_f32_tma(const CUtensorMap* map, uint32_t t_row, uint32_t epi0, uint32_t& buf,
                                            int nchunks, int col0, int row0, int lane, bool add) {
    // The output streams through L2 once per launch: evict it first, so that
    // it does not push out the operand blocks the tile order keeps resident.
    const uint64_t pol = l2_policy_evict_first();
    for (int c = 0; c < nchunks; ++c) {
        uint32_t v[32];
        tmem_ld_32cols(t_row + uint32_t(c) * 32u, v);
        tmem_ld_wait();
        const uint32_t sbuf = epi0 + buf * kEpiBuf;
        if (lane == 0) bulk_wait_group_read<1>();  // the copy that last used sbuf has read it
        __syncwarp();
        const uint32_t row_addr = sbuf + uint32_t(lane) * 128u;
#pragma unroll
        for (int j = 0; j < 8; ++j)
            st_shared_v4(row_addr + ((uint32_t(j) ^ (uint32_t(lane) & 7u)) << 4), v[4 * j], v[4 * j + 1],
                         v[4 * j + 2], v[4 * j + 3]);
        fence_proxy_async_shared();
        __syncwarp();
        if (lane == 0) {
            if (add) tma_reduce_add_2d_hint(map, sbuf, col0 + c * 32, row0, pol);
            else tma_store_2d_hint(map, sbuf, col0 + c * 32, row0, pol);
            bulk_commit_group();
        }
        buf ^= 1u;
    }
}

}  // namespace kc
}  // namespace tl
