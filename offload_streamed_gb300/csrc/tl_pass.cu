// tl_pass.cu -- persistent streamed pass: one launch runs the GEMMs of all N
// weight tiles of a forward or a backward pass while the copy streams move
// tiles in and gradients out.
//
// The pass is a flat list of output-tile jobs in pass order.  Forward: the
// Y_i = X.W_i tiles of i = 0..N-1.  Backward walks i = N-1..0 in groups of
// `gx` consecutive tiles: the dW_i = X^T.dY_i tiles of each tile of the
// group, then the dX tiles of the group, each accumulating dY_i.W_i^T over
// all gx tiles of the group in tensor memory (a reduction over gx*Mi) before
// one read-modify-write of dX -- gx times less dX traffic than one update
// per tile.  CTA pairs (clusters of
// 2, cta_group::2 MMAs, 256 x 256 tiles) take every C-th job, so all clusters
// move through the tiles together and one launch has one tail instead of one
// per tile.  Cross-engine dependencies are 32-bit sequence flags in device
// memory:
//  - before loading a W tile the producer waits (bounded) for the copy
//    stream's "ready" flag of that fetch;
//  - when every job that read a W tile is done (its MMAs completed), the last
//    one publishes "freed", which the copy stream waits on before reusing the
//    ring slot (the pages' release of a gathered tile after use);
//  - dW tiles go to a staging slot once the device->host stream has
//    "drained" its previous contents; when the last dW warp of the tile has
//    stored, "dwready" starts that tile's write-back;
//  - dX accumulation of group G waits until all dX stores of group G-1 are
//    done, which fixes the summation order.
// Every dependency points to an earlier job in the list and all clusters are
// resident, so the earliest unfinished job can always make progress.  Every
// wait is bounded; on a failure the kernel sets the error word and releases
// the copy streams' waits.
#include "tl_gemm.h"
#include "tl_kernel_common.cuh"

#include <cuda.h>

#include <algorithm>
#include <cstring>
#include <string>

namespace tl {
namespace {

using namespace kc;

constexpr uint32_t kFarAhead = 0x40000000u;

struct PassMaps {
    CUtensorMap a0;                    // fwd: X [T,K] K-major; bwd: dY [T,M] K-major (A of dX)
    CUtensorMap d0;                    // fwd: Y [T,M] bf16 store
    CUtensorMap a1;                    // bwd: X as M-major (A of dW; rows = K index)
    CUtensorMap b1;                    // bwd: dY [T,M] N-major (B of dW)
    CUtensorMap stage[kMaxPassStages]; // bwd: dW staging slots [K, Mi] bf16 store
    CUtensorMap w[kMaxPassSlots];      // ring slots [K, Mi]: fwd N-major (B of Y); bwd K-major (B of dX)
    CUtensorMap dx;                    // bwd: dX [T, K] fp32 store / reduce-add
};

// Job kind 0: the GEMM that reads W (fwd Y_i, bwd dX); kind 1: bwd dW_i.
struct PassParams {
    int32_t m_dim[2], n_dim[2], num_m[2], num_n[2], num_k[2], tiles[2], raster[2], group[2];
    int32_t N, Mi, jobs_per_tile, total_jobs;
    int32_t gx;            // backward: tiles per dX group
    int32_t jobs_per_group;  // backward: gx * tiles[1] + tiles[0]
    uint32_t fetch_base, stage_base;
    int32_t nslots, nstage;
    uint32_t* flags;
    uint32_t* done;
    uint32_t* dwdone;
    uint32_t* dxdone;
    int32_t* err;
    uint64_t timeout_ns, flag_timeout_ns;
};

// A job: kind 0 = the GEMM reading W (fwd Y tile, bwd dX tile of group G
// covering pass positions j .. j+gsz-1), kind 1 = bwd dW tile of position j.
struct Job {
    int kind, t, j, G, gsz;
};

template <bool BWD>
__device__ __forceinline__ Job decode_job(const PassParams& p, int w) {
    Job b;
    if (!BWD) {
        b.j = w / p.jobs_per_tile;
        b.t = w - b.j * p.jobs_per_tile;
        b.kind = 0;
        b.G = b.j;
        b.gsz = 1;
        return b;
    }
    const int full = p.N / p.gx;
    int r;
    if (w < full * p.jobs_per_group) {
        b.G = w / p.jobs_per_group;
        r = w - b.G * p.jobs_per_group;
        b.gsz = p.gx;
    } else {
        b.G = full;
        r = w - full * p.jobs_per_group;
        b.gsz = p.N - full * p.gx;
    }
    const int j0 = b.G * p.gx;
    if (r < b.gsz * p.tiles[1]) {
        b.kind = 1;
        b.j = j0 + r / p.tiles[1];
        b.t = r % p.tiles[1];
    } else {
        b.kind = 0;
        b.j = j0;
        b.t = r - b.gsz * p.tiles[1];
    }
    return b;
}

template <bool BWD>
__global__ void __launch_bounds__(kThreads, 1) pass_kernel(const __grid_constant__ PassMaps maps, const PassParams p) {
    using G = Geo<true, 2>;
    constexpr int S = G::kStages;
    constexpr int kParts = 8;  // epilogue warps per job: 4 per CTA, 2 CTAs
    const WaitCtx wc{p.err, p.timeout_ns};
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S * G::kStageBytes + G::kEpiBytes);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * S + 5);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const int first_job = int(cluster_id_x());
    const int job_step = int(cluster_count_x());
    const bool leader = (rank == 0);
    const uint32_t bar0 = smem_addr(bars);
    const uint32_t smem0 = smem_addr(smem);
    auto full_bar = [&](uint32_t s) { return bar0 + 8u * s; };
    auto empty_bar = [&](uint32_t s) { return bar0 + 8u * (S + s); };
    auto tfull_bar = [&](uint32_t a) { return bar0 + 8u * (2 * S + a); };
    auto tempty_bar = [&](uint32_t a) { return bar0 + 8u * (2 * S + 2 + a); };
    const uint32_t drain_bar = bar0 + 8u * (2 * S + 4);

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(tfull_bar(a), 1);
            mbar_init(tempty_bar(a), kParts);
        }
        mbar_init(drain_bar, 1);
        mbar_init_fence();
    }
    if (warp == 2) {
        tmem_alloc<true>(smem_addr(tmem_slot), kTmemCols);
        tmem_relinquish<true>();
    }
    tc_fence_before();
    cluster_sync();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer (each CTA loads its own halves) ----------------
            uint64_t pol_a[2], pol_b[2];
            for (int k = 0; k < 2; ++k) {
                pol_a[k] = p.raster[k] == 0 ? l2_policy_evict_last() : l2_policy_evict_first();
                pol_b[k] = p.raster[k] == 0 ? l2_policy_evict_first() : l2_policy_evict_last();
            }
            uint32_t fills = 0;
            bool ok = true;
            bool have_ready = false;
            uint32_t ready_f = 0;
            for (int w = first_job; ok && w < p.total_jobs; w += job_step) {
                const Job b = decode_job<BWD>(p, w);
                const int kind = b.kind;
                int mb, nb;
                tile_coords(b.t, p.num_m[kind], p.num_n[kind], p.raster[kind], p.group[kind], mb, nb);
                const int m0 = mb * G::kTileM + int(rank) * kBlockM;
                const int n0 = nb * kBlockN + int(rank) * G::kBRows;
                const int kpt = p.num_k[kind];                       // K-blocks per pass position
                const int nk = kind == 0 ? kpt * b.gsz : kpt;        // a dX job spans its group
                for (int kb = 0; kb < nk; ++kb, ++fills) {
                    // a dX job reduces its group's tiles in ascending tile
                    // order (the group's last pass position first)
                    const int seg = kind == 0 ? kb / kpt : 0;
                    const int jj = b.j + (kind == 0 ? b.gsz - 1 - seg : 0);  // pass position of this K-block
                    const int kbl = kb - seg * kpt;
                    const int i = BWD ? p.N - 1 - jj : jj;            // weight tile index
                    const uint32_t f = p.fetch_base + uint32_t(jj);
                    const int s = int(f % uint32_t(p.nslots));
                    if (kind == 0 && !(have_ready && ready_f == f)) {
                        if (!poll_geq(p.flags + kFlagReady + s, f + 1u, wc, kErrFlagWait, p.flag_timeout_ns)) {
                            ok = false;
                            break;
                        }
                        fence_proxy_async_global();  // the tile's bytes before our TMA reads of them
                        have_ready = true;
                        ready_f = f;
                    }
                    const uint32_t st = fills % S;
                    const uint32_t ph = (fills / S) & 1u;
                    if (!wait_bounded(empty_bar(st), ph ^ 1u, wc, kErrProducerWait)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sa = smem0 + st * G::kStageBytes;
                    const uint32_t sb = sa + kStageA;
                    const int k0 = kbl * kBlockK;
                    if (leader) mbar_arrive_expect_tx(full_bar(st), 2u * G::kStageBytes);
                    const uint32_t fb = map_to_rank(full_bar(st), 0);
                    if (!BWD) {  // Y_i = X . W_i : A K-major, B N-major
                        tma_load_2d_pair_hint(sa, &maps.a0, fb, k0, m0, pol_a[0]);
                        tma_load_2d_pair_hint(sb, &maps.w[s], fb, n0, k0, pol_b[0]);
                        tma_load_2d_pair_hint(sb + kMnChunk, &maps.w[s], fb, n0 + 64, k0, pol_b[0]);
                    } else if (kind == 0) {  // dX += dY_i . W_i^T : both K-major
                        tma_load_2d_pair_hint(sa, &maps.a0, fb, i * p.Mi + k0, m0, pol_a[0]);
                        tma_load_2d_pair_hint(sb, &maps.w[s], fb, k0, n0, pol_b[0]);
                    } else {  // dW_i = X^T . dY_i : A M-major, B N-major
                        tma_load_2d_pair_hint(sa, &maps.a1, fb, m0, k0, pol_a[1]);
                        tma_load_2d_pair_hint(sa + kMnChunk, &maps.a1, fb, m0 + 64, k0, pol_a[1]);
                        tma_load_2d_pair_hint(sb, &maps.b1, fb, i * p.Mi + n0, k0, pol_b[1]);
                        tma_load_2d_pair_hint(sb + kMnChunk, &maps.b1, fb, i * p.Mi + n0 + 64, k0, pol_b[1]);
                    }
                }
            }
            // The first CTA's full[] barriers count both CTAs' bytes, so its
            // drain covers the pair's loads in flight.
            if (leader) {
                const uint32_t outstanding = fills < uint32_t(S) ? fills : uint32_t(S);
                for (uint32_t q = 0; q < outstanding; ++q) {
                    const uint32_t f = fills - 1 - q;
                    wait_bounded(full_bar(f % S), (f / S) & 1u, wc, kErrDrainWait, false);
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && leader) {
            // ---------------- MMA issuer (first CTA of the pair) ----------------
            constexpr uint32_t idesc_fwd = idesc_bf16_f32(2 * kBlockM, kBlockN, false, true);
            constexpr uint32_t idesc_dx = idesc_bf16_f32(2 * kBlockM, kBlockN, false, false);
            constexpr uint32_t idesc_dw = idesc_bf16_f32(2 * kBlockM, kBlockN, true, true);
            uint32_t fills = 0;
            bool ok = true;
            int it = 0;
            for (int w = first_job; ok && w < p.total_jobs; w += job_step, ++it) {
                const Job b = decode_job<BWD>(p, w);
                const int kind = b.kind;
                const int nk = kind == 0 ? p.num_k[0] * b.gsz : p.num_k[kind];
                const bool a_mn = BWD && kind == 1;
                const bool b_mn = !BWD || kind == 1;
                const uint32_t idesc = !BWD ? idesc_fwd : (kind == 0 ? idesc_dx : idesc_dw);
                const uint32_t acc = it & 1;
                const uint32_t acc_ph = (it >> 1) & 1;
                if (!wait_bounded(tempty_bar(acc), acc_ph ^ 1u, wc, kErrMmaWaitTmem)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * kBlockN;
                for (int kb = 0; kb < nk; ++kb, ++fills) {
                    const uint32_t st = fills % S;
                    const uint32_t ph = (fills / S) & 1u;
                    if (!wait_bounded(full_bar(st), ph, wc, kErrMmaWaitFull)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = smem0 + st * G::kStageBytes;
                    const uint32_t sb = sa + kStageA;
#pragma unroll
                    for (int q = 0; q < kBlockK / kUmmaK; ++q)
                        umma_bf16_pair(d_tmem, operand_desc(a_mn, sa, q), operand_desc(b_mn, sb, q), idesc,
                                       (kb | q) != 0 ? 1u : 0u);
                    umma_commit_pair(empty_bar(st), 0x3);
                }
                if (ok) umma_commit_pair(tfull_bar(acc), 0x3);
            }
            umma_commit_pair(drain_bar, 0x3);
            wait_bounded(drain_bar, 0, wc, kErrDrainWait, false);
        }
    } else if (warp >= kFirstEpilogueWarp) {
        // ---------------- epilogue (each CTA stores its own 128 rows) ----------------
        const int q = warp & 3;
        const uint32_t epi0 = smem0 + S * G::kStageBytes + uint32_t(q) * 2u * kEpiBuf;
        uint32_t buf = 0;
        int it = 0;
        bool ok = true;
        bool have_drained = false;
        int drained_j = 0;
        for (int w = first_job; ok && w < p.total_jobs; w += job_step, ++it) {
            const Job b = decode_job<BWD>(p, w);
            const int kind = b.kind;
            const int j = b.j;
            const int i = BWD ? p.N - 1 - j : j;
            const uint32_t acc = it & 1;
            const uint32_t acc_ph = (it >> 1) & 1;
            int mb, nb;
            tile_coords(b.t, p.num_m[kind], p.num_n[kind], p.raster[kind], p.group[kind], mb, nb);
            const int row0 = mb * G::kTileM + int(rank) * kBlockM + q * 32;
            const int n0 = nb * kBlockN;
            const bool f32 = BWD && kind == 0;
            const int chunk = f32 ? 32 : 64;
            int nchunks = 0;
            if (row0 < p.m_dim[kind])  // warp-uniform
                while (nchunks * chunk < kBlockN && n0 + nchunks * chunk < p.n_dim[kind]) ++nchunks;
            const uint32_t sj = p.stage_base + uint32_t(j);
            const int g = int(sj % uint32_t(p.nstage > 0 ? p.nstage : 1));
            // ordering waits that do not depend on this job's accumulator
            if (BWD && kind == 1 && !(have_drained && drained_j == j) && sj >= uint32_t(p.nstage)) {
                int okw = 1;
                if (lane == 0)
                    okw = poll_geq(p.flags + kFlagDrained + g, sj - uint32_t(p.nstage) + 1u, wc, kErrFlagWait,
                                   p.flag_timeout_ns);
                okw = __shfl_sync(0xffffffffu, okw, 0);
                if (!okw) break;
                have_drained = true;
                drained_j = j;
            }
            if (BWD && kind == 0 && b.G > 0) {  // dX of the previous group fully stored
                int okw = 1;
                if (lane == 0) {
                    okw = poll_geq(p.dxdone + (b.G - 1), uint32_t(kParts * p.tiles[0]), wc, kErrFlagWait,
                                   p.flag_timeout_ns);
                    fence_proxy_async_global();  // before this lane's TMA reduce-adds of the same dX
                }
                okw = __shfl_sync(0xffffffffu, okw, 0);
                if (!okw) break;
            }
            if (!warp_wait(tfull_bar(acc), acc_ph, wc, kErrEpilogueWait, lane)) break;
            tc_fence_after();
            // The job's MMAs are complete: its reads of the W tiles are over.
            if (kind == 0 && leader && q == 0 && lane == 0) {
                for (int jj = j; jj < j + b.gsz; ++jj) {
                    const uint32_t f = p.fetch_base + uint32_t(jj);
                    const uint32_t prev = atomicAdd(p.done + jj, 1u);
                    if (prev + 1u == uint32_t(p.tiles[0]))
                        st_release_u32(p.flags + kFlagFreed + int(f % uint32_t(p.nslots)), f + 1u);
                }
            }
            const uint32_t t_row = tmem_base + (uint32_t(q * 32) << 16) + acc * kBlockN;
            if (!BWD) {
                epi_bf16_tma(&maps.d0, t_row, epi0, buf, nchunks, i * p.Mi + n0, row0, lane);
            } else if (kind == 1) {
                epi_bf16_tma(&maps.stage[g], t_row, epi0, buf, nchunks, n0, row0, lane);
                if (lane == 0) {
                    bulk_wait_group_all();  // this warp's part of dW_i is in global memory
                    fence_proxy_async_global();
                    __threadfence();
                    const uint32_t prev = atomicAdd(p.dwdone + j, 1u);
                    if (prev + 1u == uint32_t(kParts * p.tiles[1]))
                        st_release_u32(p.flags + kFlagDwReady + g, sj + 1u);
                }
            } else {
                epi_f32_tma(&maps.dx, t_row, epi0, buf, nchunks, n0, row0, lane, b.G > 0);
                if (lane == 0) {
                    bulk_wait_group_all();  // this warp's part of the dX tile is in global memory
                    fence_proxy_async_global();
                    __threadfence();
                    atomicAdd(p.dxdone + b.G, 1u);
                }
                __syncwarp();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if (!leader) mbar_arrive_cluster(map_to_rank(tempty_bar(acc), 0));
                else mbar_arrive(tempty_bar(acc));
            }
        }
        if (lane == 0) bulk_wait_group_all();
        __syncwarp();
    }

    tc_fence_before();
    cluster_sync();
    if (warp == 2) {
        tc_fence_after();
        if (!leader) wait_bounded(drain_bar, 0, wc, kErrDrainWait, false);
        tmem_dealloc<true>(tmem_base, kTmemCols);
    }
    // After a failure, let the copy streams' waits on this pass go through so
    // that nothing waits forever; the handle reports the error.
    if (threadIdx.x == 0 && leader && *reinterpret_cast<volatile int32_t*>(p.err) != 0) {
        for (int s = 0; s < p.nslots; ++s)
            st_release_u32(p.flags + kFlagFreed + s, p.fetch_base + uint32_t(p.N) + kFarAhead);
        for (int g = 0; g < p.nstage; ++g)
            st_release_u32(p.flags + kFlagDwReady + g, p.stage_base + uint32_t(p.N) + kFarAhead);
    }
}

template <bool BWD>
cudaError_t launch_pass(const PassMaps& maps, const PassParams& pp, int grid, cudaStream_t stream) {
    auto kern = pass_kernel<BWD>;
    constexpr size_t smem = Geo<true, 2>::kSmem;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(unsigned(grid), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, maps, pp);
}

void set_kind(PassParams& pp, int k, int64_t m_dim, int64_t n_dim, int64_t k_dim) {
    pp.m_dim[k] = int32_t(m_dim);
    pp.n_dim[k] = int32_t(n_dim);
    pp.num_m[k] = int32_t((m_dim + 2 * kBlockM - 1) / (2 * kBlockM));
    pp.num_n[k] = int32_t((n_dim + kBlockN - 1) / kBlockN);
    pp.num_k[k] = int32_t((k_dim + kBlockK - 1) / kBlockK);
    pp.tiles[k] = pp.num_m[k] * pp.num_n[k];
    choose_tile_order(k_dim, 2 * kBlockM, pp.num_m[k], pp.num_n[k], &pp.raster[k], &pp.group[k]);
}

}  // namespace

cudaError_t pass_preload() {
    cudaError_t e = cudaFuncSetAttribute(pass_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         int(Geo<true, 2>::kSmem));
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(pass_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                int(Geo<true, 2>::kSmem));
}

std::string pass_check(const PassDesc& d, int num_sms) {
    if (!cta_pair_enabled() || num_sms < 2) return "CTA pairs unavailable";
    if (d.T < 1 || d.K < 8 || d.Mi < 1 || d.N < 1) return "empty problem";
    if (d.Mi % kBlockN) return "tile width not a multiple of 256";
    if (d.N > kMaxPassTiles) return "too many tiles for the pass counters";
    if (d.nslots < 1 || d.nslots > kMaxPassSlots) return "ring has too many slots for a persistent pass";
    if (d.backward && (d.nstage < 1 || d.nstage > kMaxPassStages)) return "bad staging slot count";
    if (d.backward && (d.dx_group < 1 || d.dx_group > d.nslots)) return "dX group larger than the ring";
    if (d.T > (int64_t(1) << 30) || d.K > (int64_t(1) << 30) || int64_t(d.N) * d.Mi > (int64_t(1) << 34))
        return "problem too large";
    if (!d.flags || !d.done || !d.dwdone || !d.dxdone || !d.err || !d.x) return "null pointer";
    if (d.backward ? (!d.dy || !d.dx) : !d.y) return "null pointer";
    return {};
}

cudaError_t pass_launch(const PassDesc& d, int num_sms, cudaStream_t stream, std::string* why) {
    std::string bad = pass_check(d, num_sms);
    if (!bad.empty()) {
        if (why) *why = bad;
        return cudaErrorInvalidValue;
    }
    const int64_t T = d.T, K = d.K, Mi = d.Mi, M = int64_t(d.N) * d.Mi;
    PassMaps maps;
    std::memset(&maps, 0, sizeof(maps));
    PassParams pp{};
    bool ok = true;
    if (!d.backward) {
        ok = ok && make_tensor_map(&maps.a0, d.x, K, T, K, kBlockM, false, why);
        ok = ok && make_tensor_map(&maps.d0, d.y, M, T, M, 32, false, why);
        for (int s = 0; s < d.nslots; ++s) ok = ok && make_tensor_map(&maps.w[s], d.slots[s], Mi, K, Mi, 64, false, why);
        set_kind(pp, 0, T, Mi, K);
        pp.tiles[1] = 0;
        pp.jobs_per_tile = pp.tiles[0];
    } else {
        ok = ok && make_tensor_map(&maps.a0, d.dy, M, T, M, kBlockM, false, why);
        ok = ok && make_tensor_map(&maps.a1, d.x, K, T, K, 64, false, why);
        ok = ok && make_tensor_map(&maps.b1, d.dy, M, T, M, 64, false, why);
        for (int g = 0; g < d.nstage; ++g) ok = ok && make_tensor_map(&maps.stage[g], d.stages[g], Mi, K, Mi, 32, false, why);
        for (int s = 0; s < d.nslots; ++s)
            ok = ok && make_tensor_map(&maps.w[s], d.slots[s], Mi, K, Mi, kBlockN / 2, false, why);
        ok = ok && make_tensor_map(&maps.dx, d.dx, K, T, K, 32, true, why);
        set_kind(pp, 0, T, K, Mi);  // dX (per pass position; a job spans its group)
        set_kind(pp, 1, K, Mi, T);  // dW
        pp.jobs_per_tile = pp.tiles[0] + pp.tiles[1];
    }
    pp.gx = d.backward ? std::max(1, std::min(d.dx_group, d.N)) : 1;
    if (!ok) return cudaErrorInvalidValue;
    pp.N = d.N;
    pp.Mi = int32_t(d.Mi);
    if (d.backward) {
        pp.jobs_per_group = pp.gx * pp.tiles[1] + pp.tiles[0];
        const int full = d.N / pp.gx, rem = d.N - full * pp.gx;
        pp.total_jobs = full * pp.jobs_per_group + (rem > 0 ? rem * pp.tiles[1] + pp.tiles[0] : 0);
    } else {
        pp.jobs_per_group = pp.jobs_per_tile;
        pp.total_jobs = pp.jobs_per_tile * d.N;
    }
    pp.fetch_base = d.fetch_base;
    pp.stage_base = d.stage_base;
    pp.nslots = d.nslots;
    pp.nstage = d.nstage;
    pp.flags = d.flags;
    pp.done = d.done;
    pp.dwdone = d.dwdone;
    pp.dxdone = d.dxdone;
    pp.err = d.err;
    pp.timeout_ns = d.timeout_ns;
    pp.flag_timeout_ns = d.flag_timeout_ns;
    const int clusters = std::min(pp.total_jobs, num_sms / 2);
    const cudaError_t e = d.backward ? launch_pass<true>(maps, pp, 2 * clusters, stream)
                                     : launch_pass<false>(maps, pp, 2 * clusters, stream);
    if (e != cudaSuccess && why) *why = std::string("pass launch: ") + cudaGetErrorString(e);
    return e;
}

}  // namespace tl
