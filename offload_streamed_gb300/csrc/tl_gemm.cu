// tl_gemm.cu -- persistent, warp-specialised bf16 GEMM for sm_103a.
//
// One CTA pair per two SMs (one CTA per SM without pairing) walks output
// tiles of 256 x 256 (128 x 256) in a grouped raster order.
//   warp 0      : TMA producer -- one thread loads the A and B slices of each
//                 64-deep K-block into a shared-memory ring (6 stages with a
//                 CTA pair, 4 for a single CTA).  B may come in two segments
//                 (two weight tiles in different ring slots).
//   warp 1      : MMA issuer -- one thread issues tcgen05.mma (M=256 across
//                 the pair or 128, N=256, K=16, bf16 x bf16 -> fp32) into one
//                 of two TMEM accumulators, and frees a ring stage with
//                 tcgen05.commit.
//   warp 2      : allocates / frees the 512 TMEM columns.
//   warps 4..7  : epilogue -- tcgen05.ld of the finished accumulator (each
//                 warp owns 32 TMEM lanes = 32 output rows), rounding to bf16
//                 or storing / adding fp32, while the MMA warp already fills
//                 the other accumulator.
// There is no split of the reduction dimension: every output element is
// reduced by one CTA in ascending K-block order, so a given element's value
// does not depend on the problem's other dimensions (forward Y is bit-exact
// between tiled and untiled runs).
//
// Every wait on an mbarrier is bounded (%globaltimer, 2 s).  On timeout the
// thread ORs an error bit into *err and its role stops; the other roles see
// the error word and stop too; the producer waits (time-bounded) for its own
// TMA loads to land, the MMA thread for its own MMAs, and TMEM is freed
// before the CTA exits.
#include "tl_gemm.h"
#include "tl_kernel_common.cuh"

#include <cudaTypedefs.h>

#include <algorithm>
#include <climits>
#include <cstdlib>
#include <mutex>

namespace tl {
namespace {

using namespace kc;

// Tensor maps of B segments 1.. (segment 0 is map_b).
struct BSegMaps {
    CUtensorMap m[GemmDesc::kMaxSeg - 1];
};

struct KParams {
    int32_t m_dim, n_dim, k_dim;
    int32_t num_m, num_n, num_k, num_tiles;
    int32_t raster, group;  // tile order (see kc::tile_coords)
    int32_t stream_shared;  // the streamed operand is read by several groups at once (see choose_tile_order)
    int32_t k_seg;          // reduction rows per B segment (INT32_MAX: one segment)
    void* d;
    int64_t ldd;
    int32_t accumulate;
    const float* addend;  // bf16 input-gradient kind: D = bf16(addend + A.B) (nullptr: no addend)
    int64_t ld_add;
    int32_t withhold_loads;
    int32_t* err;
    uint32_t* tile_counter;  // dynamic schedule (nullptr: static round robin)
    uint64_t timeout_ns;
};

template <bool A_MN, bool B_MN, bool OUT_F32, bool PAIR>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
                const __grid_constant__ CUtensorMap map_d, const __grid_constant__ BSegMaps segs,
                const KParams p) {
    using G = Geo<PAIR, 2>;
    const WaitCtx wc{p.err, p.timeout_ns};
    constexpr int S = G::kStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    constexpr int Q = 4;  // depth of the tile queue (dynamic schedule)
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S * G::kStageBytes + G::kEpiBytes);
    int32_t* tile_q = reinterpret_cast<int32_t*>(bars + 2 * S + 5 + 2 * Q);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tile_q + Q);
    static_assert((2 * S + 5 + 2 * Q) * 8 + 4 * Q + 4 <= int(kBarBytes), "barrier area");

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
    const int first_tile = PAIR ? int(cluster_id_x()) : int(blockIdx.x);
    const int tile_step = PAIR ? int(cluster_count_x()) : int(gridDim.x);
    const bool leader = (rank == 0);
    const uint32_t bar0 = smem_addr(bars);
    const uint32_t smem0 = smem_addr(smem);
    // barriers: full[s], empty[s], tmem_full[a], tmem_empty[a], drain.  With
    // a CTA pair, full[] and tmem_empty[] are used in the first CTA only.
    auto full_bar = [&](uint32_t s) { return bar0 + 8u * s; };
    auto empty_bar = [&](uint32_t s) { return bar0 + 8u * (S + s); };
    auto tfull_bar = [&](uint32_t a) { return bar0 + 8u * (2 * S + a); };
    auto tempty_bar = [&](uint32_t a) { return bar0 + 8u * (2 * S + 2 + a); };
    const uint32_t drain_bar = bar0 + 8u * (2 * S + 4);
    // Dynamic schedule: the first CTA's producer draws tiles from a device
    // counter and publishes them in a small queue (tile_q, in both CTAs of a
    // pair); queue_full[q] (every CTA) says slot q holds a tile id,
    // queue_empty[q] (first CTA) collects the readers' releases.  An id < 0
    // ends the sequence.  Without a counter every role walks the static
    // round robin first_tile, first_tile + tile_step, ...
    auto qfull_bar = [&](uint32_t q) { return bar0 + 8u * (2 * S + 5 + q); };
    auto qempty_bar = [&](uint32_t q) { return bar0 + 8u * (2 * S + 5 + Q + q); };
    const bool dynamic = p.tile_counter != nullptr;
    constexpr uint32_t kQueueReaders = PAIR ? 10u : 5u;  // MMA, peer producer, epilogue warps
    auto static_tile = [&](int it) {
        const int t = first_tile + it * tile_step;
        return t < p.num_tiles ? t : -1;
    };
    // first CTA's producer: draw and publish the tile of iteration `it`
    auto publish_tile = [&](int it) -> int {
        const uint32_t q = uint32_t(it) % Q, ph = (uint32_t(it) / Q) & 1u;
        if (!wait_bounded_cluster(qempty_bar(q), ph ^ 1u, wc, kErrTileQueueWait)) return -1;
        const uint32_t ticket = atomicAdd(p.tile_counter, 1u);
        const int t = ticket < uint32_t(p.num_tiles) ? int(ticket) : -1;
        // every cluster draws once past the end; the last such draw resets
        // the counter for the next launch
        if (ticket == uint32_t(p.num_tiles) + uint32_t(tile_step) - 1u) atomicExch(p.tile_counter, 0u);
        tile_q[q] = t;
        mbar_arrive_cluster(map_to_rank(qfull_bar(q), 0));
        if constexpr (PAIR) {
            st_shared_cluster_u32(map_to_rank(smem_addr(tile_q + q), 1), uint32_t(t));
            mbar_arrive_cluster(map_to_rank(qfull_bar(q), 1));
        }
        return t;
    };
    // every other role: read the tile of iteration `it` and release the slot
    auto take_tile = [&](int it) -> int {
        const uint32_t q = uint32_t(it) % Q, ph = (uint32_t(it) / Q) & 1u;
        if (!wait_bounded_cluster(qfull_bar(q), ph, wc, kErrTileQueueWait)) return -1;
        const int t = *reinterpret_cast<volatile int32_t*>(tile_q + q);
        mbar_arrive_cluster(map_to_rank(qempty_bar(q), 0));
        return t;
    };

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(tfull_bar(a), 1);
            mbar_init(tempty_bar(a), PAIR ? 8 : 4);  // one arrival per epilogue warp of the tile
        }
        mbar_init(drain_bar, 1);
        for (int q = 0; q < Q; ++q) {
            mbar_init(qfull_bar(q), 1);
            mbar_init(qempty_bar(q), kQueueReaders);
        }
        mbar_init_fence();
    }
    if (warp == 2) {
        tmem_alloc<PAIR>(smem_addr(tmem_slot), kTmemCols);
        tmem_relinquish<PAIR>();
    }
    tc_fence_before();
    if constexpr (PAIR) cluster_sync(); else __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer (each CTA loads its own halves) ----------------
            tma_prefetch_map(&map_a);
            tma_prefetch_map(&map_b);
            for (int j = 1; j < GemmDesc::kMaxSeg && j * p.k_seg < p.k_dim; ++j) tma_prefetch_map(&segs.m[j - 1]);
            // the tile order keeps a group of A blocks (raster 0) or of B
            // blocks (raster 1) in L2; the other operand streams through,
            // and leaves L2 first unless the groups in flight share it
            const uint64_t pol_s = p.stream_shared ? l2_policy_evict_normal() : l2_policy_evict_first();
            const uint64_t pol_a = p.raster == 0 ? l2_policy_evict_last() : pol_s;
            const uint64_t pol_b = p.raster == 0 ? pol_s : l2_policy_evict_last();
            uint32_t fills = 0;
            bool ok = true;
            for (int it = 0; ok; ++it) {
                const int tile = !dynamic ? static_tile(it) : leader ? publish_tile(it) : take_tile(it);
                if (tile < 0) break;
                if (p.withhold_loads != 0) break;  // the failure-path self-test withholds every load
                int mb, nb;
                tile_coords(tile, p.num_m, p.num_n, p.raster, p.group, mb, nb);
                const int m0 = mb * G::kTileM + int(rank) * kBlockM;
                const int n0 = nb * kBlockN + int(rank) * (PAIR ? G::kBRows : 0);
                for (int kb = 0; kb < p.num_k; ++kb, ++fills) {
                    const uint32_t s = fills % S;
                    const uint32_t ph = (fills / S) & 1u;
                    if (!wait_bounded(empty_bar(s), ph ^ 1u, wc, kErrProducerWait)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sa = smem0 + s * G::kStageBytes;
                    const uint32_t sb = sa + kStageA;
                    const int k0 = kb * kBlockK;
                    if (leader) mbar_arrive_expect_tx(full_bar(s), (PAIR ? 2u : 1u) * G::kStageBytes);
                    const uint32_t fb = PAIR ? map_to_rank(full_bar(s), 0) : full_bar(s);
                    auto load = [&](uint32_t dst, const CUtensorMap* m, int32_t x, int32_t y, uint64_t pol) {
                        if constexpr (PAIR) tma_load_2d_pair_hint(dst, m, fb, x, y, pol);
                        else tma_load_2d_hint(dst, m, fb, x, y, pol);
                    };
                    if (A_MN) {
                        load(sa, &map_a, m0, k0, pol_a);
                        load(sa + kMnChunk, &map_a, m0 + 64, k0, pol_a);
                    } else {
                        load(sa, &map_a, k0, m0, pol_a);
                    }
                    if (B_MN) {
#pragma unroll
                        for (int c = 0; c < G::kBRows / 64; ++c)
                            load(sb + c * kMnChunk, &map_b, n0 + 64 * c, k0, pol_b);
                    } else if (k0 < p.k_seg) {
                        load(sb, &map_b, k0, n0, pol_b);
                    } else {  // a further B segment
                        const int seg = k0 / p.k_seg;
                        load(sb, &segs.m[seg - 1], k0 - seg * p.k_seg, n0, pol_b);
                    }
                }
            }
            // Loads must land before the CTA may exit.  The first CTA's full[]
            // barriers count both CTAs' bytes, so its drain covers the pair.
            if (leader) {
                const uint32_t outstanding = fills < uint32_t(S) ? fills : uint32_t(S);
                for (uint32_t j = 0; j < outstanding; ++j) {
                    const uint32_t f = fills - 1 - j;
                    wait_bounded(full_bar(f % S), (f / S) & 1u, wc, kErrDrainWait, false);
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && leader) {
            // ---------------- MMA issuer (first CTA of the pair) ----------------
            constexpr uint32_t idesc = idesc_bf16_f32(G::kTileM, kBlockN, A_MN, B_MN);
            uint32_t fills = 0;
            bool ok = true;
            for (int it = 0; ok; ++it) {
                const int tile = dynamic ? take_tile(it) : static_tile(it);
                if (tile < 0) break;
                const uint32_t acc = it & 1;
                const uint32_t acc_ph = (it >> 1) & 1;
                if (!wait_bounded(tempty_bar(acc), acc_ph ^ 1u, wc, kErrMmaWaitTmem)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * kBlockN;
                for (int kb = 0; kb < p.num_k; ++kb, ++fills) {
                    const uint32_t s = fills % S;
                    const uint32_t ph = (fills / S) & 1u;
                    if (!wait_bounded(full_bar(s), ph, wc, kErrMmaWaitFull)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = smem0 + s * G::kStageBytes;
                    const uint32_t sb = sa + kStageA;
#pragma unroll
                    for (int j = 0; j < kBlockK / kUmmaK; ++j) {
                        const uint64_t ad = operand_desc(A_MN, sa, j);
                        const uint64_t bd = operand_desc(B_MN, sb, j);
                        if constexpr (PAIR) umma_bf16_pair(d_tmem, ad, bd, idesc, (kb | j) != 0 ? 1u : 0u);
                        else umma_bf16(d_tmem, ad, bd, idesc, (kb | j) != 0 ? 1u : 0u);
                    }
                    if constexpr (PAIR) umma_commit_pair(empty_bar(s), 0x3);
                    else umma_commit(empty_bar(s));
                }
                if (ok) {
                    if constexpr (PAIR) umma_commit_pair(tfull_bar(acc), 0x3);
                    else umma_commit(tfull_bar(acc));
                }
            }
            // The MMAs must complete before TMEM is freed (in both CTAs).
            if constexpr (PAIR) umma_commit_pair(drain_bar, 0x3);
            else umma_commit(drain_bar);
            wait_bounded(drain_bar, 0, wc, kErrDrainWait, false);
        }
    } else if (warp >= kFirstEpilogueWarp) {
        // ---------------- epilogue (each CTA stores its own 128 rows) ----------------
        // Outputs leave through swizzled staging boxes in shared memory: TMA
        // stores for bf16 and for a first fp32 dX, TMA reduce-adds (the add
        // done in L2) for an accumulated one.
        constexpr int kChunk = OUT_F32 ? 32 : 64;
        const int q = warp & 3;
        const uint32_t epi0 = smem0 + S * G::kStageBytes + uint32_t(q) * 2u * kEpiBuf;
        if (lane == 0) tma_prefetch_map(&map_d);
        uint32_t buf = 0;
        for (int it = 0;; ++it) {
            int tile;
            if (dynamic) {
                int t = 0;
                if (lane == 0) t = take_tile(it);
                tile = __shfl_sync(0xffffffffu, t, 0);
            } else {
                tile = static_tile(it);
            }
            if (tile < 0) break;
            const uint32_t acc = it & 1;
            const uint32_t acc_ph = (it >> 1) & 1;
            int mb, nb;
            tile_coords(tile, p.num_m, p.num_n, p.raster, p.group, mb, nb);
            const int row0 = mb * G::kTileM + int(rank) * kBlockM + q * 32;
            const int n0 = nb * kBlockN;
            int nchunks = 0;
            if (row0 < p.m_dim)  // warp-uniform
                while (nchunks * kChunk < kBlockN && n0 + nchunks * kChunk < p.n_dim) ++nchunks;
            if (!warp_wait(tfull_bar(acc), acc_ph, wc, kErrEpilogueWait, lane)) break;
            tc_fence_after();
            const uint32_t t_row = tmem_base + (uint32_t(q * 32) << 16) + acc * kBlockN;
            if constexpr (OUT_F32) {
                epi_f32_tma(&map_d, t_row, epi0, buf, nchunks, n0, row0, lane, p.accumulate != 0);
            } else if constexpr (!A_MN && !B_MN) {  // dX rounded to bf16, after the addend if any
                if (p.addend)
                    epi_bf16_add_tma(&map_d, t_row, epi0, buf, nchunks, n0, row0, lane, p.addend, p.ld_add,
                                     p.m_dim, p.n_dim);
                else
                    epi_bf16_tma(&map_d, t_row, epi0, buf, nchunks, n0, row0, lane);
            } else {
                epi_bf16_tma(&map_d, t_row, epi0, buf, nchunks, n0, row0, lane);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if (PAIR && !leader) mbar_arrive_cluster(map_to_rank(tempty_bar(acc), 0));
                else mbar_arrive(tempty_bar(acc));
            }
        }
        if (lane == 0) bulk_wait_group_all();  // stores complete before the CTA exits
        __syncwarp();
    }

    tc_fence_before();
    if constexpr (PAIR) cluster_sync(); else __syncthreads();
    if (warp == 2) {
        tc_fence_after();
        // The second CTA of a pair has not watched the MMAs: wait for the
        // drain commit that the first CTA multicast to it.
        if (PAIR && !leader) wait_bounded(drain_bar, 0, wc, kErrDrainWait, false);
        tmem_dealloc<PAIR>(tmem_base, kTmemCols);
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// 2-D tensor map: `inner` contiguous elements per row, `outer` rows `ld`
// elements apart, box of (128 bytes of elements) x box_outer, 128-byte
// swizzle, zero fill outside the tensor (loads) / clipping (stores).
bool make_map(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint64_t ld,
              uint32_t box_outer, std::string* why, bool f32 = false) {
    auto fn = encode_fn();
    if (!fn) {
        if (why) *why = "cuTensorMapEncodeTiled is unavailable from the driver";
        return false;
    }
    const uint32_t esize = f32 ? 4 : 2;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {ld * esize};
    cuuint32_t box[2] = {128 / esize, box_outer};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                    const_cast<void*>(base), dims, strides,
                    box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        if (why) *why = "cuTensorMapEncodeTiled failed with CUresult " + std::to_string(int(r));
        return false;
    }
    return true;
}

template <bool A_MN, bool B_MN, bool OUT_F32, bool PAIR>
cudaError_t launch_one(const CUtensorMap& ma, const CUtensorMap& mb, const CUtensorMap& md, const BSegMaps& segs,
                       const KParams& kp, int grid, cudaStream_t stream) {
    auto kern = gemm_kernel<A_MN, B_MN, OUT_F32, PAIR>;
    constexpr size_t smem = Geo<PAIR, 2>::kSmem;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(unsigned(grid), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = PAIR ? 2 : 1;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, ma, mb, md, segs, kp);
}

template <bool PAIR>
cudaError_t dispatch(const GemmDesc& g, const CUtensorMap& ma, const CUtensorMap& mb, const CUtensorMap& md,
                     const BSegMaps& segs, const KParams& kp, int grid, cudaStream_t stream) {
    if (!g.a_mn_major && g.b_mn_major)
        return launch_one<false, true, false, PAIR>(ma, mb, md, segs, kp, grid, stream);
    if (g.a_mn_major && g.b_mn_major) return launch_one<true, true, false, PAIR>(ma, mb, md, segs, kp, grid, stream);
    if (g.out == OutKind::BF16) return launch_one<false, false, false, PAIR>(ma, mb, md, segs, kp, grid, stream);
    return launch_one<false, false, true, PAIR>(ma, mb, md, segs, kp, grid, stream);
}


bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

// Choose the tile order that moves the fewest operand bytes from DRAM: keep
// a group of one operand's blocks (at most kL2Budget bytes) resident in L2
// and stream the other operand once per group.  The budget is a quarter of
// the L2: the persistent CTAs drift apart in K, so a group's blocks must
// share the cache with the streamed operand's slices in flight (32 MiB
// measured best or equal for all three GEMMs at the GPT-scale tile, against
// 16, 48, 64 and 128 MiB, under the power cap).
// When a group holds fewer tiles than the `concurrent` tiles in flight (long
// reductions, whose blocks are so large that a group holds one or two), one
// wave of tiles spans several groups, which walk the streamed operand's K
// slices together and read each slice from DRAM once: the streamed operand
// is then read once per wave of groups, not once per group, and its loads
// keep the L2's normal eviction priority instead of evict-first
// (`stream_shared`), or the groups after the first find it gone.  Measured
// resident at the power cap against groups counted one by one with
// evict-first: 64K-hidden forward 1520 -> 1726-1740 TFLOP/s (DRAM bytes per
// launch 14.7 -> 4.5 GB), its dX 1604-1620 -> 1681 (18.1 -> 12.6 GB), the
// 1T-width forward 1535-1551 -> 1582-1585; the GPT-scale GEMMs' groups exceed
// a wave, and their order is unchanged.
void choose_tile_order(int64_t k_dim, int tile_m, int num_m, int num_n, int concurrent, int32_t* raster,
                       int32_t* group, int32_t* stream_shared) {
    constexpr double kL2Budget = 32.0 * 1024 * 1024;
    const double a_blk = double(tile_m) * double(k_dim) * 2;
    const double b_blk = double(kBlockN) * double(k_dim) * 2;
    const double a_tot = a_blk * num_m, b_tot = b_blk * num_n;
    const int gm = std::max(1, std::min(num_m, int(kL2Budget / a_blk)));
    const int gn = std::max(1, std::min(num_n, int(kL2Budget / b_blk)));
    const double c = std::max(1, concurrent);
    // passes of the streamed operand: one per wave of groups
    auto passes = [&](int groups, int group_tiles) {
        const double per_wave = std::max(1.0, std::floor(c / group_tiles));
        return std::ceil(groups / per_wave);
    };
    const double t0 = a_tot + b_tot * passes((num_m + gm - 1) / gm, gm * num_n);
    const double t1 = b_tot + a_tot * passes((num_n + gn - 1) / gn, gn * num_m);
    if (t1 < t0) {
        *raster = 1;
        *group = gn;
        *stream_shared = gn * num_m < concurrent ? 1 : 0;
    } else {
        *raster = 0;
        *group = gm;
        *stream_shared = gm * num_n < concurrent ? 1 : 0;
    }
}

bool cta_pair_enabled() {
    static const bool pair = [] {
        const char* e = std::getenv("TILED_LINEAR_CTA_PAIR");
        return !(e && e[0] == '0');
    }();
    return pair;
}

std::string gemm_check(const GemmDesc& g) {
    if (g.m_dim < 1 || g.n_dim < 1 || g.k_dim < 1) return "GEMM sizes must be >= 1";
    if (g.m_dim > INT32_MAX / 2 || g.n_dim > INT32_MAX / 2 || g.k_dim > INT32_MAX / 2)
        return "GEMM size too large";
    if (!g.a || !g.b || !g.d || !g.err) return "null pointer";
    if (!aligned16(g.a) || !aligned16(g.b) || !aligned16(g.d))
        return "operand pointers must be 16-byte aligned";
    if (reinterpret_cast<uintptr_t>(g.err) & 3u) return "err pointer must be 4-byte aligned";
    if (reinterpret_cast<uintptr_t>(g.tile_counter) & 3u) return "tile counter must be 4-byte aligned";
    if (g.lda % 8 || g.ldb % 8 || g.ldd % 8)
        return "leading dimensions must be multiples of 8 elements";
    if ((g.a_mn_major ? g.m_dim : g.k_dim) > g.lda) return "A leading dimension too small";
    if (g.nseg <= 1 && (g.b_mn_major ? g.n_dim : g.k_dim) > g.ldb) return "B leading dimension too small";
    if (g.n_dim > g.ldd) return "D leading dimension too small";
    if (g.lda * 2 >= (int64_t(1) << 40) || g.ldb * 2 >= (int64_t(1) << 40))
        return "leading dimension too large";
    const int64_t tiles = ((g.m_dim + kBlockM - 1) / kBlockM) * ((g.n_dim + kBlockN - 1) / kBlockN);  // 1-CTA tiles bound pair tiles
    if (tiles > INT32_MAX) return "too many output tiles";
    const bool fwd = !g.a_mn_major && g.b_mn_major && g.out == OutKind::BF16;
    const bool dw = g.a_mn_major && g.b_mn_major && g.out == OutKind::BF16;
    const bool dx = !g.a_mn_major && !g.b_mn_major && g.out == OutKind::F32;
    const bool dx_bf16 = !g.a_mn_major && !g.b_mn_major && g.out == OutKind::BF16;
    if (!(fwd || dw || dx || dx_bf16)) return "unsupported operand-major / output combination";
    if (g.accumulate && g.out != OutKind::F32) return "accumulate needs fp32 output";
    if (g.addend) {
        if (!dx_bf16) return "an addend needs the bf16 input-gradient kind";
        if (!aligned16(g.addend)) return "addend pointer must be 16-byte aligned";
        if (g.ld_addend % 8 || g.ld_addend < g.n_dim) return "addend leading dimension must be a multiple of 8 and >= n";
        if (g.ld_addend * 4 >= (int64_t(1) << 40)) return "addend leading dimension too large";
    }
    if (g.nseg < 1 || g.nseg > GemmDesc::kMaxSeg) return "nseg must be in 1..4";
    if (g.nseg > 1) {
        if (g.b_mn_major) return "B segments need a K-major B";
        for (int j = 1; j < g.nseg; ++j)
            if (!g.bseg[j] || !aligned16(g.bseg[j])) return "B segment pointers must be non-null and 16-byte aligned";
        if (g.k_seg <= 0 || g.k_seg % kBlockK || g.k_seg * g.nseg != g.k_dim)
            return "k_seg must be a multiple of 64 with nseg * k_seg == k_dim";
        if (g.k_seg > g.ldb) return "B leading dimension too small";
    }
    return {};
}

cudaError_t gemm_launch(const GemmDesc& g, int num_sms, cudaStream_t stream, std::string* why) {
    std::string bad = gemm_check(g);
    if (!bad.empty()) {
        if (why) *why = bad;
        return cudaErrorInvalidValue;
    }
    const bool pair = cta_pair_enabled() && num_sms >= 2;
    const int tile_m = pair ? 2 * kBlockM : kBlockM;
    const uint32_t b_rows = pair ? kBlockN / 2 : kBlockN;
    CUtensorMap ma, mb;
    const bool ok_a = g.a_mn_major ? make_map(&ma, g.a, g.m_dim, g.k_dim, g.lda, 64, why)
                                   : make_map(&ma, g.a, g.k_dim, g.m_dim, g.lda, kBlockM, why);
    if (!ok_a) return cudaErrorInvalidValue;
    const int64_t k_b = g.nseg > 1 ? g.k_seg : g.k_dim;  // reduction rows held by b
    const bool ok_b = g.b_mn_major ? make_map(&mb, g.b, g.n_dim, k_b, g.ldb, 64, why)
                                   : make_map(&mb, g.b, k_b, g.n_dim, g.ldb, b_rows, why);
    if (!ok_b) return cudaErrorInvalidValue;
    BSegMaps segs;
    for (int j = 1; j < GemmDesc::kMaxSeg; ++j) {
        segs.m[j - 1] = mb;
        if (j < g.nseg && !make_map(&segs.m[j - 1], g.bseg[j], g.k_seg, g.n_dim, g.ldb, b_rows, why))
            return cudaErrorInvalidValue;
    }
    CUtensorMap md;
    if (!make_map(&md, g.d, g.n_dim, g.m_dim, g.ldd, 32, why, g.out == OutKind::F32)) return cudaErrorInvalidValue;

    KParams kp{};
    kp.m_dim = int32_t(g.m_dim);
    kp.n_dim = int32_t(g.n_dim);
    kp.k_dim = int32_t(g.k_dim);
    kp.num_m = int32_t((g.m_dim + tile_m - 1) / tile_m);
    kp.num_n = int32_t((g.n_dim + kBlockN - 1) / kBlockN);
    kp.num_k = int32_t((g.k_dim + kBlockK - 1) / kBlockK);
    kp.num_tiles = kp.num_m * kp.num_n;
    const int slots = pair ? num_sms / 2 : num_sms;  // tiles in flight at once
    choose_tile_order(g.k_dim, tile_m, kp.num_m, kp.num_n, slots, &kp.raster, &kp.group, &kp.stream_shared);
    kp.k_seg = g.nseg > 1 ? int32_t(g.k_seg) : INT32_MAX;
    kp.d = g.d;
    kp.ldd = g.ldd;
    kp.accumulate = g.accumulate ? 1 : 0;
    kp.addend = g.addend;
    kp.ld_add = g.ld_addend;
    kp.withhold_loads = g.withhold_loads ? 1 : 0;
    kp.err = g.err;
    // The dynamic schedule costs each tile a ticket draw and a publish to
    // the peer CTA before its first loads (~4.4k cycles measured at the
    // tile boundary); for short reductions the static round robin's
    // seamless tile starts outweigh the dynamic schedule's tighter L2 window
    // and tail.  Resident at the power cap, static against dynamic: 32
    // K-blocks (the 64K-hidden dW, T = 2048) +4.8 to +6.1 %, 64 K-blocks
    // +0.6 to +1.3 %, 128 K-blocks -1.1 %, long reductions -1 to -3 %.
    constexpr int kStaticMaxKBlocks = 64;
    kp.tile_counter = kp.num_k <= kStaticMaxKBlocks ? nullptr : g.tile_counter;
    kp.timeout_ns = g.timeout_ns;
    const int units = kp.num_tiles < slots ? kp.num_tiles : slots;
    const int grid = pair ? 2 * units : units;

    const cudaError_t e = pair ? dispatch<true>(g, ma, mb, md, segs, kp, grid, stream)
                               : dispatch<false>(g, ma, mb, md, segs, kp, grid, stream);
    if (e != cudaSuccess && why) *why = std::string("kernel launch: ") + cudaGetErrorString(e);
    return e;
}

}  // namespace tl
