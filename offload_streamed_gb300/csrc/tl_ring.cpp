// tl_ring.cpp -- handle creation, the depth-d tile ring and the forward and
// backward schedules of the engine (see tl_engine.h for the resources).
//
// The copy of a tile into a ring slot waits for the free event of the slot's
// last reader, so the h2d stream runs up to d tiles ahead of the compute
// stream (aicassindra tm_zero_infinity, "Prefetch depth: how far ahead the
// pipeline must run"; pwwt.cn/news/5430303, "关键技术三", 动态预取器).  A slot
// whose reader has finished is refilled: that is the release of the gathered
// weights (gpu_zero_sharding, "End-to-end flow").  Backward runs the tiles in
// descending order (the backward pass walks the operators in reverse: same
// section), fetches every tile again (it was freed after forward), runs the
// weight-gradient GEMM first (it does not read W_i, so it overlaps the
// tile's fetch), hands the gradient tile to the d2h stream, and then
// accumulates dX with the W_i tile (pwwt.cn/news/5430303, "关键技术三",
// 后向传播中的重叠: gradients go back to slow memory while later operators
// compute).
//
// Also here: dX over groups of tiles that sit in the ring together; the dW
// staging slots lent to the forward as extra fetch slots; tile reuse across
// calls; chains of operators through one ring; the host waits of the host
// optimizer (tl_optimizer) and the file tier's fetch / write-back (tl_filetier).
#include "tl_engine.h"
#include "tl_unbound_error.h"

#include <cmath>
#include <cstring>
#include <new>

namespace tl {

std::string check_shape(int64_t K, int64_t M, int32_t N, int32_t d) {
    if (K < 8 || K % 8) return "K must be a positive multiple of 8";
    if (M < 1 || N < 1) return "M and N must be >= 1";
    if (M % N) return "M must be divisible by N";
    if ((M / N) % 8) return "M/N (tile width) must be a multiple of 8";
    if (d < -1) return "d must be >= -1";
    if (K > (int64_t(1) << 31) || M > (int64_t(1) << 34)) return "K or M too large";
    return {};
}

namespace {

size_t ring_slot_bytes(const std::vector<Shape>& ops) {
    size_t tb = 0;
    for (const Shape& o : ops) tb = std::max(tb, align_up(tile_bytes(o.K, o.Mi), kAlign));
    return tb;
}

int32_t total_tiles(const std::vector<Shape>& ops) {
    int32_t n = 0;
    for (const Shape& o : ops) n += o.N;
    return n;
}

// Slots a handle at depth d uses: d+1 weight slots (at most N) and min(2, N)
// dW staging slots.  With automatic depth the workspace decides (see
// create_ops): at least two weight slots and min(2, N) staging slots, and as
// many as N of each.
int32_t min_slots(int32_t N, int32_t d) {
    const int32_t w = d < 0 ? std::min(N, 2) : std::min(d, N - 1) + 1;
    return w + std::min(N, kMaxStage);
}

int32_t max_slots(int32_t N, int32_t d) { return d < 0 ? 2 * N : min_slots(N, d); }

}  // namespace

size_t workspace_for(const std::vector<Shape>& ops, int32_t d) {
    return kHeaderBytes + size_t(max_slots(total_tiles(ops), d)) * ring_slot_bytes(ops);
}

bool is_pinned_host(const void* p) {
    cudaPointerAttributes a{};
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return a.type == cudaMemoryTypeHost;
}

bool is_device_mem(const void* p, int device) {
    cudaPointerAttributes a{};
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) && a.device == device;
}

// Read the pinned mirror of the kernels' error word (written at the end of
// every call); a non-zero word makes the handle sticky-failed.
tl_status poll_error(tl_handle* h) {
    if (h->err_mirror && *reinterpret_cast<volatile int32_t*>(h->err_mirror) != 0)
        return fail(h, TL_ERR_TIMEOUT,
                    "a kernel's bounded wait timed out (error bits " +
                        std::to_string(*h->err_mirror) + ")");
    return TL_OK;
}

tl_status check_usable(tl_handle* h) {
    if (!h) return TL_ERR_STATE;
    if (h->sticky != TL_OK) return TL_ERR_STATE;
    return poll_error(h);
}

namespace {

const uint8_t* w_tile_src(const Op& o, int i) {
    const Shape& s = o.s;
    if (o.layout == TL_LAYOUT_TILE_MAJOR) return o.w_host + size_t(i) * tile_bytes(s.K, s.Mi);
    return o.w_host + size_t(i) * size_t(s.Mi) * 2;
}

uint8_t* dw_tile_dst(const Op& o, int i) {
    const Shape& s = o.s;
    if (o.layout == TL_LAYOUT_TILE_MAJOR) return o.dw_host + size_t(i) * tile_bytes(s.K, s.Mi);
    return o.dw_host + size_t(i) * size_t(s.Mi) * 2;
}

cudaError_t copy_w_tile(const Op& o, int i, void* dst, cudaStream_t st) {
    const Shape& s = o.s;
    if (o.layout == TL_LAYOUT_TILE_MAJOR)
        return cudaMemcpyAsync(dst, w_tile_src(o, i), tile_bytes(s.K, s.Mi), cudaMemcpyHostToDevice, st);
    return cudaMemcpy2DAsync(dst, size_t(s.Mi) * 2, w_tile_src(o, i), size_t(s.M) * 2,
                             size_t(s.Mi) * 2, size_t(s.K), cudaMemcpyHostToDevice, st);
}

cudaError_t copy_dw_tile(const Op& o, int i, const void* src, cudaStream_t st) {
    const Shape& s = o.s;
    if (o.layout == TL_LAYOUT_TILE_MAJOR)
        return cudaMemcpyAsync(dw_tile_dst(o, i), src, tile_bytes(s.K, s.Mi), cudaMemcpyDeviceToHost, st);
    return cudaMemcpy2DAsync(dw_tile_dst(o, i), size_t(s.M) * 2, src, size_t(s.Mi) * 2,
                             size_t(s.Mi) * 2, size_t(s.K), cudaMemcpyDeviceToHost, st);
}

// Host->device copy of W tile i of operator o into device slot dst on the
// h2d stream: from pinned host memory, or from the file tier's host slot
// once its reader has the tile there (the calling thread waits for that).
tl_status fetch_w_tile(tl_handle* h, const Op& o, int i, void* dst) {
    if (!h->tier) {
        TL_TRY(h, copy_w_tile(o, i, dst, h->h2d));
        return TL_OK;
    }
    std::string why;
    const int slot = h->tier->acquire_w(o.first + i, &why);
    if (slot < 0) return fail(h, TL_ERR_IO, why);
    TL_TRY(h, cudaMemcpyAsync(dst, h->tier->w_slot(slot), tile_bytes(o.s.K, o.s.Mi), cudaMemcpyHostToDevice, h->h2d));
    TL_TRY(h, cudaEventRecord(h->tier->w_event(slot), h->h2d));
    h->tier->release_w(slot);
    return TL_OK;
}

// Device->host copy of dW tile i of operator o from src on stream st: into
// pinned host memory, or into a file-tier host slot that a writer stores
// to the dW file once the copy is done (the calling thread waits for a free
// slot).
tl_status writeback_dw_tile(tl_handle* h, const Op& o, int i, const void* src, cudaStream_t st) {
    if (!h->tier) {
        TL_TRY(h, copy_dw_tile(o, i, src, st));
        return TL_OK;
    }
    std::string why;
    const int slot = h->tier->acquire_dw(&why);
    if (slot < 0) return fail(h, TL_ERR_IO, why);
    TL_TRY(h, cudaMemcpyAsync(h->tier->dw_slot(slot), src, tile_bytes(o.s.K, o.s.Mi), cudaMemcpyDeviceToHost, st));
    TL_TRY(h, cudaEventRecord(h->tier->dw_event(slot), st));
    h->tier->commit_dw(slot, o.first + i);
    return TL_OK;
}

// One launch per tile: slots 0..d free in order, holding no tile.
void reset_ring(tl_handle* h) {
    h->slot_q.clear();
    for (int s = 0; s <= h->d; ++s) h->slot_q.push_back(s);
    h->slot_tile.assign(h->slot.size(), -1);
}

// The dW staging slots double as weight slots for the forward, where they sit
// idle: slot index slot_cap + g is staging slot g.  A backward takes them out
// of the free queue (its dW GEMMs write them) and hands them back once their
// last write-back has left.
int staging_slot(const tl_handle* h, int g) { return h->slot_cap + g; }

void withdraw_staging(tl_handle* h) {
    std::deque<int> q;
    for (int sl : h->slot_q)
        if (sl < h->slot_cap) q.push_back(sl);
    h->slot_q.swap(q);
    for (int g = 0; g < h->nstage; ++g) h->slot_tile[size_t(staging_slot(h, g))] = -1;
}

// The slot for the next fetch: the one whose last reader was enqueued
// earliest (the fetch waits for that reader on the h2d stream).
int take_slot(tl_handle* h, bool ring_only = false) {
    for (auto it = h->slot_q.begin(); it != h->slot_q.end(); ++it)
        if (!ring_only || *it < h->slot_cap) {
            const int sl = *it;
            h->slot_q.erase(it);
            return sl;
        }
    return -1;
}

// With a host optimizer attached: the host waits before it queues a copy that
// reads tile g's W (until every submitted step has rewritten it) or writes
// tile g's dW (until every submitted job has read the last one).
tl_status opt_wait(tl_handle* h, int g, bool update) {
    if (!h->opt) return TL_OK;
    const bool ok = update ? tl::optimizer_wait_update(h->opt, g, kOptWaitSeconds)
                           : tl::optimizer_wait_read(h->opt, g, kOptWaitSeconds);
    if (!ok) return fail(h, TL_ERR_TIMEOUT, tl::optimizer_error(h->opt));
    return TL_OK;
}

}  // namespace

// Automatic depth: after the first forward call, the pages' rule
// d = ceil(t_fetch / t_layer) (tm_zero_infinity, "Prefetch depth"), with
// t_layer the call's mean per-tile GEMM time and t_fetch its slowest tile copy
// plus the handle's stall allowance: the host link occasionally stalls for
// tens of milliseconds, and a ring sized from mean times stops the GEMMs for
// the length of such a stall (same page, "Pitfalls": a mistuned prefetch
// stalls).  Bounded by the weight slots the workspace holds.
tl_status finish_auto_depth(tl_handle* h) {
    if (!h->auto_pending || h->fwd.last < 0) return TL_OK;
    CallSlot& c = h->fwd.ring[h->fwd.last];
    tl_status st = harvest(h, h->fwd, c, h->n_total);
    if (st != TL_OK) return st;
    const double layer = c.nk > 0 ? double(c.gemm1) / c.nk : 0.0;
    const double fetch = double(c.h2d_max) + h->stall_allowance_ms;
    int32_t dnew = h->slot_cap - 1;
    if (layer > 0) dnew = int32_t(std::min<double>(std::ceil(fetch / layer), double(h->slot_cap - 1)));
    dnew = std::max<int32_t>(std::min<int32_t>(1, h->slot_cap - 1), dnew);
    if (dnew != h->d) {
        // the first call's fetches are done before the new ring starts
        for (size_t s = 0; s < h->slot.size(); ++s) TL_TRY(h, cudaStreamWaitEvent(h->h2d, h->ev_free[s], 0));
        h->d = dnew;
        reset_ring(h);
    }
    h->auto_pending = false;
    return TL_OK;
}

namespace {

// dX is accumulated over groups of consecutive tiles, one launch per group,
// whenever the operator's depth min(d, N - 1) is at least 2 and the tile
// width splits into whole 64-deep K-blocks.  A group reduces at least 8192
// deep where the ring allows: g = max(2, ceil(8192 / Mi)), at most
// min(d, N - 1) and 4 (the GEMM's B segments); the last group of an
// operator may be smaller.  The bound uses the operator's own N, so that an
// operator groups its tiles the same way alone and inside a chain.
// A group holds its tiles' ring slots until its launch, so g <= d leaves at
// least one of the d + 1 slots fetching ahead while the group computes: at
// d = 1 a pair would hold the whole ring and stop the refetch during each dX
// launch (1T-width layer at d = 1: 994 TFLOP/s with pairs, 1155 with single
// tiles; the link-bound sweep point T = 2048 at d = 1: +6 to 8 %).  Larger
// groups mean fewer fp32 passes over dX; pairs stay for wide tiles (groups of
// three measured 1 % slower on the GPT-scale layer).  The groups depend on
// (N, Mi, d) alone, so a backward that reuses resident tiles and one that
// fetches them again agree bit for bit.
int dx_group(const tl_handle* h, const Shape& s) {
    const int d = std::min(h->d, s.N - 1);
    if (d < 2 || s.Mi % tl::kBlockK) return 1;
    const int want = std::max<int>(2, int((8192 + s.Mi - 1) / s.Mi));
    return std::min({want, d, int(tl::GemmDesc::kMaxSeg)});
}

tl_status launch(tl_handle* h, const tl::GemmDesc& g0, cudaStream_t st) {
    tl::GemmDesc g = g0;
    g.tile_counter = h->tile_counter;  // one word: launches on the compute stream are ordered
    std::string why;
    cudaError_t e = tl::gemm_launch(g, h->num_sms, st, &why);
    if (e != cudaSuccess) return fail(h, TL_ERR_CUDA, "GEMM launch: " + why);
    return TL_OK;
}

}  // namespace

tl_status create_ops(tl_handle** out, std::vector<Op> ops, int32_t d, void* ws, size_t ws_bytes, int device,
                     bool single_api, const FileArgs* file) {
    if (!out) {
        tl::set_unbound_error("out is NULL");
        return TL_ERR_INVALID;
    }
    *out = nullptr;
    std::string bad = ops.empty() ? "no operators" : "";
    std::vector<Shape> shapes;
    int32_t first = 0;
    for (size_t l = 0; l < ops.size() && bad.empty(); ++l) {
        Op& o = ops[l];
        bad = check_shape(o.s.K, o.s.M, o.s.N, d);
        if (bad.empty() && !file && (!o.w_host || !o.dw_host)) bad = "null pointer argument";
        if (bad.empty() && l > 0 && o.s.K != ops[l - 1].s.M) bad = "operator inputs must match the outputs before them";
        if (!bad.empty() && ops.size() > 1) bad = "operator " + std::to_string(l) + ": " + bad;
        o.s.Mi = o.s.M / std::max<int32_t>(o.s.N, 1);
        o.first = first;
        first += o.s.N;
        shapes.push_back(o.s);
    }
    if (bad.empty() && first > (1 << 20)) bad = "too many tiles";
    if (bad.empty() && !ws) bad = "null pointer argument";
    if (bad.empty() && device < 0) bad = "device must be >= 0";
    if (!bad.empty()) {
        tl::set_unbound_error(bad);
        return TL_ERR_INVALID;
    }
    const int32_t N = first;  // tiles over all operators
    const size_t tb = ring_slot_bytes(shapes);
    const size_t need = kHeaderBytes + size_t(min_slots(N, d)) * tb;
    if (ws_bytes < need || (reinterpret_cast<uintptr_t>(ws) % kAlign)) {
        tl::set_unbound_error("workspace too small or not 256-byte aligned (need " + std::to_string(need) +
                              " bytes)");
        return TL_ERR_WORKSPACE;
    }

    tl_handle* h = new (std::nothrow) tl_handle();
    if (!h) {
        tl::set_unbound_error("out of host memory");
        return TL_ERR_INVALID;
    }
    auto bail = [&](tl_status st) {
        tl::set_unbound_error(h->msg);
        tiled_linear_destroy(h);
        return st;
    };
    h->device = device;
    h->ops = ops;
    h->single_api = single_api;
    h->n_total = N;
    h->s = ops[0].s;
    h->layout = ops[0].layout;
    h->d_req = d;
    h->w_host = ops[0].w_host;
    h->dw_host = ops[0].dw_host;
    h->ws = static_cast<uint8_t*>(ws);
    h->ws_bytes = ws_bytes;

    DeviceGuard guard(device);
    if (guard.err != cudaSuccess) {
        h->msg = std::string("cudaSetDevice: ") + cudaGetErrorString(guard.err);
        return bail(TL_ERR_CUDA);
    }
    for (const Op& o : ops)
        if (!file && (!is_pinned_host(o.w_host) || !is_pinned_host(o.dw_host))) {
            h->msg = "w_host and dw_host must be pinned host memory";
            return bail(TL_ERR_NOT_PINNED);
        }
    if (!is_device_mem(ws, device)) {
        h->msg = "workspace is not device memory of the handle's device";
        return bail(TL_ERR_WORKSPACE);
    }

    // Carve the workspace: header (error word, tile counter), weight slots,
    // staging slots.  At a fixed depth: d+1 weight slots and min(2, N)
    // staging slots.  With automatic depth, every slot that fits, split evenly
    // between the two (at least 2 weight and min(2, N) staging slots, at most
    // N of each); the depth is chosen among the weight slots after the first
    // forward (finish_auto_depth), and every staging slot takes its turn, so
    // that a stalled write-back holds the backward up only once all of them
    // wait to drain.
    if (d >= 0) {
        h->slot_cap = std::min(d, N - 1) + 1;
        h->nstage = std::min(N, kMaxStage);
    } else {
        const int32_t fit = int32_t(std::min<size_t>(size_t(2 * N), (ws_bytes - kHeaderBytes) / tb));
        h->nstage = std::max(std::min(N, kMaxStage), std::min(N, fit / 2));
        h->slot_cap = std::max(std::min(N, 2), std::min(N, fit - h->nstage));
    }
    h->d = h->slot_cap - 1;
    h->auto_pending = (d < 0);
    h->stall_allowance_ms = kDefaultStallAllowanceMs;
    h->err_dev = reinterpret_cast<int32_t*>(h->ws);
    h->tile_counter = reinterpret_cast<uint32_t*>(h->ws + kTileCounterOffset);
    uint8_t* p = h->ws + kHeaderBytes;
    for (int s = 0; s < h->slot_cap; ++s, p += tb) h->slot.push_back(p);
    for (int g = 0; g < h->nstage; ++g, p += tb) h->stage.push_back(p);
    for (int g = 0; g < h->nstage; ++g) h->slot.push_back(h->stage[size_t(g)]);  // see staging_slot
    reset_ring(h);

    if (cudaMemset(h->ws, 0, kHeaderBytes) != cudaSuccess ||
        cudaHostAlloc(reinterpret_cast<void**>(&h->err_mirror), sizeof(int32_t), cudaHostAllocPortable) !=
            cudaSuccess) {
        h->msg = std::string("error-word setup: ") + cudaGetErrorString(cudaGetLastError());
        return bail(TL_ERR_CUDA);
    }
    *h->err_mirror = 0;
    if (cudaStreamCreateWithFlags(&h->h2d, cudaStreamNonBlocking) != cudaSuccess ||
        cudaStreamCreateWithFlags(&h->d2h, cudaStreamNonBlocking) != cudaSuccess) {
        h->msg = std::string("stream creation: ") + cudaGetErrorString(cudaGetLastError());
        return bail(TL_ERR_CUDA);
    }
    auto mk = [&](std::vector<cudaEvent_t>& v, int n) {
        v.assign(size_t(n), nullptr);
        for (auto& e : v)
            if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) return false;
        return true;
    };
    const int nbuf = h->slot_cap + h->nstage;
    if (!mk(h->ev_ready, nbuf) || !mk(h->ev_free, nbuf) || !mk(h->ev_dwdone, h->nstage) ||
        !mk(h->ev_drained, h->nstage)) {
        h->msg = std::string("event creation: ") + cudaGetErrorString(cudaGetLastError());
        return bail(TL_ERR_CUDA);
    }
    if (create_phase(h, h->fwd, N, false) != TL_OK || create_phase(h, h->bwd, N, true) != TL_OK)
        return bail(TL_ERR_CUDA);
    if (cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) {
        h->msg = "cudaDeviceGetAttribute(multiProcessorCount) failed";
        return bail(TL_ERR_CUDA);
    }
    if (file) {
        std::string why;
        h->tier = tl::FileTier::open(file->w_path, file->dw_path, N, tile_bytes(h->s.K, h->s.Mi), file->host_slots,
                                     file->io_threads, &why);
        if (!h->tier) {
            h->msg = "file tier: " + why;
            return bail(TL_ERR_IO);
        }
    }
    *out = h;
    return TL_OK;
}

// ---- one launch per tile, over the handle's operators in sequence ----------
// Forward: operator l computes ys[l][:, tile i] = X_l . W_{l,i}, X_0 = x and
// X_l = ys[l-1]; the ring streams the operators' tiles in that order, so the
// next operator's first tiles are fetched while this one's last tiles run.
tl_status forward_tiles(tl_handle* h, int64_t T, const void* x, void* const* ys, cudaStream_t cs) {
    tl_status st;
    CallSlot* tp = begin_call(h, h->fwd, &st);
    if (!tp) return st;
    CallSlot& t = *tp;
    int64_t h2d_bytes = 0;
    if (h->tier) {  // the file tier reads the tiles in the order this call fetches them
        h->tier->clear_requests();
        for (int g = 0; g < h->n_total; ++g) h->tier->request(g);
    }
    TL_TRY(h, cudaEventRecord(t.start, cs));
    for (size_t l = 0; l < h->ops.size(); ++l) {
        const Op& o = h->ops[l];
        const Shape& s = o.s;
        const void* xl = l == 0 ? x : ys[l - 1];
        for (int i = 0; i < s.N; ++i) {
            const int g = o.first + i;  // tile index in the handle's order
            if ((st = opt_wait(h, g, true)) != TL_OK) return st;
            // the pass's last d+1 tiles go to ring slots: a backward that
            // follows may take them from there (tile reuse)
            const int sl = take_slot(h, g >= h->n_total - (h->d + 1));
            if (sl < 0) return fail(h, TL_ERR_STATE, "internal: no ring slot to fetch into");
            h->slot_tile[size_t(sl)] = -1;
            TL_TRY(h, cudaStreamWaitEvent(h->h2d, h->ev_free[sl], 0));
            if (t.timed) TL_TRY(h, cudaEventRecord(t.ev[4][g], h->h2d));
            if ((st = fetch_w_tile(h, o, i, h->slot[sl])) != TL_OK) return st;
            h->slot_tile[size_t(sl)] = g;
            h2d_bytes += int64_t(tile_bytes(s.K, s.Mi));
            if (t.timed) TL_TRY(h, cudaEventRecord(t.ev[5][g], h->h2d));
            TL_TRY(h, cudaEventRecord(h->ev_ready[sl], h->h2d));

            TL_TRY(h, cudaStreamWaitEvent(cs, h->ev_ready[sl], 0));
            if (t.timed) TL_TRY(h, cudaEventRecord(t.ev[0][g], cs));
            tl::GemmDesc gd;
            gd.m_dim = T;
            gd.n_dim = s.Mi;
            gd.k_dim = s.K;
            gd.a = xl;
            gd.lda = s.K;
            gd.a_mn_major = false;
            gd.b = h->slot[sl];
            gd.ldb = s.Mi;
            gd.b_mn_major = true;
            gd.d = static_cast<uint8_t*>(ys[l]) + size_t(i) * size_t(s.Mi) * 2;
            gd.ldd = s.M;
            gd.out = tl::OutKind::BF16;
            gd.err = h->err_dev;
            if ((st = launch(h, gd, cs)) != TL_OK) return st;
            if (t.timed) TL_TRY(h, cudaEventRecord(t.ev[1][g], cs));
            TL_TRY(h, cudaEventRecord(h->ev_free[sl], cs));
            h->slot_q.push_back(sl);
        }
    }
    TL_TRY(h, cudaEventRecord(t.end, cs));
    TL_TRY(h, cudaMemcpyAsync(h->err_mirror, h->err_dev, sizeof(int32_t), cudaMemcpyDeviceToHost, cs));
    t.nk = h->n_total;
    t.depth = h->d;
    t.launches = h->n_total;
    t.h2d_bytes = h2d_bytes;
    t.d2h_bytes = 0;
    end_call(h->fwd, t);
    return TL_OK;
}

// Backward, operators in reverse and each one's tiles in descending order:
//   dW_{l,i} = X_l^T . dY_l[:, tile i] -> staging slot -> host (d2h stream)
//   dX_l (+)= dY_l[:, tile i] . W_{l,i}^T in fp32 (tile groups, see dx_group)
// dY_{L-1} = dy; for l < L-1, dY_l = bf16(dX_{l+1}): dX_l for l >= 1
// accumulates in scr_dx, and operator l's last dX launch adds its share to
// the fp32 sum of the earlier ones and writes the bf16 RNE of the total as
// dY_{l-1}, into scr_dy[(L - 1 - l) % 2] (two buffers, so that an operator
// never writes the dY it reads).  dX_0 goes to dx.
tl_status backward_tiles(tl_handle* h, int64_t T, const void* x, const void* const* ys, const void* dy,
                         float* dx, float* scr_dx, void* const* scr_dy, cudaStream_t cs) {
    tl_status st;
    const int L = int(h->ops.size());
    withdraw_staging(h);
    if (T == 0) {  // dW = X^T dY over an empty sum: zero
        if (h->opt) h->opt_order.clear();
        for (int l = L - 1; l >= 0; --l) {
            const Op& o = h->ops[size_t(l)];
            TL_TRY(h, cudaStreamWaitEvent(cs, h->ev_drained[0], 0));
            TL_TRY(h, cudaStreamWaitEvent(cs, h->ev_free[staging_slot(h, 0)], 0));
            TL_TRY(h, cudaMemsetAsync(h->stage[0], 0, tile_bytes(o.s.K, o.s.Mi), cs));
            for (int i = o.s.N - 1; i >= 0; --i) {
                const int g = o.first + i;
                if ((st = opt_wait(h, g, false)) != TL_OK) return st;
                if ((st = writeback_dw_tile(h, o, i, h->stage[0], cs)) != TL_OK) return st;
                if (h->opt) {
                    TL_TRY(h, cudaEventRecord(h->opt_ev_w[size_t(g)], cs));
                    TL_TRY(h, cudaEventRecord(h->opt_ev_dw[size_t(g)], cs));
                    h->opt_order.push_back(g);
                }
            }
            TL_TRY(h, cudaEventRecord(h->ev_drained[0], cs));
        }
        if (h->opt) h->opt_have_bwd = true;
        for (int g = 0; g < h->nstage; ++g) {
            TL_TRY(h, cudaEventRecord(h->ev_free[staging_slot(h, g)], cs));
            h->slot_q.push_back(staging_slot(h, g));
        }
        return TL_OK;
    }
    CallSlot* tp = begin_call(h, h->bwd, &st);
    if (!tp) return st;
    CallSlot& t = *tp;
    const int NT = h->n_total;
    // With reuse on, the longest prefix of the descending tile order that is
    // still resident in the ring (the last d+1 tiles a forward fetched) is
    // taken as it is; those slots leave the free queue until their dX launch.
    std::vector<int> resident(size_t(NT), -1);
    int reused = 0;
    if (h->reuse) {
        for (int sl = 0; sl <= h->d; ++sl)
            if (h->slot_tile[size_t(sl)] >= 0) resident[size_t(h->slot_tile[size_t(sl)])] = sl;
        while (reused < NT && resident[size_t(NT - 1 - reused)] >= 0) ++reused;
        std::deque<int> q;
        for (int sl : h->slot_q) {
            bool taken = false;
            for (int j = 0; j < reused; ++j) taken = taken || resident[size_t(NT - 1 - j)] == sl;
            if (!taken) q.push_back(sl);
        }
        h->slot_q.swap(q);
    }
    int64_t h2d_bytes = 0, d2h_bytes = 0;
    if (h->tier) {  // the tiles this call fetches, in its order (operators and tiles descending)
        h->tier->clear_requests();
        int pos = 0;
        for (int l = L - 1; l >= 0; --l)
            for (int i = h->ops[size_t(l)].s.N - 1; i >= 0; --i, ++pos)
                if (pos >= reused) h->tier->request(h->ops[size_t(l)].first + i);
    }
    int launches = 0;
    int jg = 0;  // position in the backward's tile order
    std::vector<bool> stage_ready(size_t(h->nstage), false);  // forward done with the staging slot
    if (h->opt) h->opt_order.clear();
    TL_TRY(h, cudaEventRecord(t.start, cs));
    for (int l = L - 1; l >= 0; --l) {
        const Op& o = h->ops[size_t(l)];
        const Shape& s = o.s;
        const void* xl = l == 0 ? x : ys[l - 1];
        const void* dyl = l == L - 1 ? dy : scr_dy[(L - 2 - l) % 2];
        float* dxl = l == 0 ? dx : scr_dx;
        const size_t tb = tile_bytes(s.K, s.Mi);
        // dX is accumulated over groups of tiles (i+g-1, ..., i) -- one
        // launch reducing over all of them, in ascending column order.
        const int gsz = dx_group(h, s);
        std::vector<int> pend;  // ring slots of the open group's tiles, highest tile first
        int dx_launches = 0;
        for (int j = 0; j < s.N; ++j, ++jg) {
            const int i = s.N - 1 - j;
            const int g = o.first + i;
            const int gs = int(h->stage_seq++ % uint64_t(h->nstage));
            int sl;
            if (jg < reused) {  // W_i is still in the ring
                sl = resident[size_t(g)];
                if (t.timed) TL_TRY(h, cudaEventRecord(t.ev[4][jg], h->h2d));
                if (t.timed) TL_TRY(h, cudaEventRecord(t.ev[5][jg], h->h2d));
            } else {  // refetch W_i
                if ((st = opt_wait(h, g, true)) != TL_OK) return st;
                sl = take_slot(h);
                if (sl < 0) return fail(h, TL_ERR_STATE, "internal: no ring slot to fetch into");
                h->slot_tile[size_t(sl)] = -1;
                TL_TRY(h, cudaStreamWaitEvent(h->h2d, h->ev_free[sl], 0));
                if (t.timed) TL_TRY(h, cudaEventRecord(t.ev[4][jg], h->h2d));
                if ((st = fetch_w_tile(h, o, i, h->slot[sl])) != TL_OK) return st;
                if (t.timed) TL_TRY(h, cudaEventRecord(t.ev[5][jg], h->h2d));
                TL_TRY(h, cudaEventRecord(h->ev_ready[sl], h->h2d));
                h->slot_tile[size_t(sl)] = g;
                h2d_bytes += int64_t(tb);
            }
            // the host W of tile g is no longer read by this call once the
            // h2d stream gets here
            if (h->opt) TL_TRY(h, cudaEventRecord(h->opt_ev_w[size_t(g)], h->h2d));

            // dW_i = X^T dY_i into staging slot gs (does not need W_i)
            TL_TRY(h, cudaStreamWaitEvent(cs, h->ev_drained[gs], 0));
            if (!stage_ready[size_t(gs)]) {  // the forward may have read a weight tile from it
                TL_TRY(h, cudaStreamWaitEvent(cs, h->ev_free[staging_slot(h, gs)], 0));
                stage_ready[size_t(gs)] = true;
            }
            if (t.timed) TL_TRY(h, cudaEventRecord(t.ev[0][jg], cs));
            tl::GemmDesc gw;
            gw.m_dim = s.K;
            gw.n_dim = s.Mi;
            gw.k_dim = T;
            gw.a = xl;
            gw.lda = s.K;
            gw.a_mn_major = true;
            gw.b = static_cast<const uint8_t*>(dyl) + size_t(i) * size_t(s.Mi) * 2;
            gw.ldb = s.M;
            gw.b_mn_major = true;
            gw.d = h->stage[gs];
            gw.ldd = s.Mi;
            gw.out = tl::OutKind::BF16;
            gw.err = h->err_dev;
            if ((st = launch(h, gw, cs)) != TL_OK) return st;
            ++launches;
            if (t.timed) TL_TRY(h, cudaEventRecord(t.ev[1][jg], cs));
            TL_TRY(h, cudaEventRecord(h->ev_dwdone[gs], cs));

            // write dW_i back on the d2h stream
            if ((st = opt_wait(h, g, false)) != TL_OK) return st;
            TL_TRY(h, cudaStreamWaitEvent(h->d2h, h->ev_dwdone[gs], 0));
            if (t.timed) TL_TRY(h, cudaEventRecord(t.ev[6][jg], h->d2h));
            if ((st = writeback_dw_tile(h, o, i, h->stage[gs], h->d2h)) != TL_OK) return st;
            if (t.timed) TL_TRY(h, cudaEventRecord(t.ev[7][jg], h->d2h));
            if (h->opt) {
                TL_TRY(h, cudaEventRecord(h->opt_ev_dw[size_t(g)], h->d2h));
                h->opt_order.push_back(g);
            }
            TL_TRY(h, cudaEventRecord(h->ev_drained[gs], h->d2h));
            d2h_bytes += int64_t(tb);
            if (jg >= NT - h->nstage) {
                // the staging slot's last write-back of this call: from here
                // it serves the next forward (in release order in the queue)
                TL_TRY(h, cudaEventRecord(h->ev_free[staging_slot(h, gs)], h->d2h));
                h->slot_q.push_back(staging_slot(h, gs));
            }

            if (int(pend.size()) + 1 < gsz && j + 1 < s.N) {
                // not the group's last (lowest) tile: its dX waits for the group
                pend.push_back(sl);
                if (t.timed) TL_TRY(h, cudaEventRecord(t.ev[2][jg], cs));
                if (t.timed) TL_TRY(h, cudaEventRecord(t.ev[3][jg], cs));
                t.dx_at[size_t(jg)] = 0;
                continue;
            }
            // dX (+)= sum over the group's tiles i, i+1, .. of dY_i W_i^T, fp32;
            // the first launch stores
            std::vector<int> grp(pend.rbegin(), pend.rend());  // ascending tile order from i+1
            grp.insert(grp.begin(), sl);                        // tile i first
            for (int gsl : grp) TL_TRY(h, cudaStreamWaitEvent(cs, h->ev_ready[gsl], 0));
            if (t.timed) TL_TRY(h, cudaEventRecord(t.ev[2][jg], cs));
            tl::GemmDesc gx;
            gx.m_dim = T;
            gx.n_dim = s.K;
            gx.k_dim = int64_t(grp.size()) * s.Mi;
            gx.a = static_cast<const uint8_t*>(dyl) + size_t(i) * size_t(s.Mi) * 2;
            gx.lda = s.M;
            gx.a_mn_major = false;
            gx.b = h->slot[sl];
            gx.ldb = s.Mi;
            gx.b_mn_major = false;
            if (grp.size() > 1) {  // reduction rows [j Mi, (j+1) Mi) are tile i+j's
                gx.nseg = int32_t(grp.size());
                gx.k_seg = s.Mi;
                for (size_t jj = 0; jj < grp.size(); ++jj) gx.bseg[jj] = h->slot[size_t(grp[jj])];
            }
            gx.ldd = s.K;
            gx.err = h->err_dev;
            if (l > 0 && j + 1 == s.N) {  // the operator's last dX launch: the previous one's dY in bf16
                gx.d = scr_dy[(L - 1 - l) % 2];
                gx.out = tl::OutKind::BF16;
                gx.addend = dx_launches > 0 ? dxl : nullptr;
                gx.ld_addend = s.K;
            } else {
                gx.d = dxl;
                gx.out = tl::OutKind::F32;
                gx.accumulate = dx_launches > 0;
            }
            if ((st = launch(h, gx, cs)) != TL_OK) return st;
            t.dx_at[size_t(jg)] = 1;
            ++dx_launches;
            ++launches;
            if (t.timed) TL_TRY(h, cudaEventRecord(t.ev[3][jg], cs));
            for (int psl : pend) {
                TL_TRY(h, cudaEventRecord(h->ev_free[psl], cs));
                h->slot_q.push_back(psl);
            }
            TL_TRY(h, cudaEventRecord(h->ev_free[sl], cs));
            h->slot_q.push_back(sl);
            pend.clear();
        }
    }
    // dW on the host is complete when `stream` is.
    for (int gi = 0; gi < h->nstage; ++gi) TL_TRY(h, cudaStreamWaitEvent(cs, h->ev_drained[gi], 0));
    TL_TRY(h, cudaEventRecord(t.end, cs));
    TL_TRY(h, cudaMemcpyAsync(h->err_mirror, h->err_dev, sizeof(int32_t), cudaMemcpyDeviceToHost, cs));
    if (h->opt) h->opt_have_bwd = true;
    t.nk = NT;
    t.depth = h->d;
    t.launches = launches;
    t.reused = reused;
    t.h2d_bytes = h2d_bytes;
    t.d2h_bytes = d2h_bytes;
    end_call(h->bwd, t);
    return TL_OK;
}

}  // namespace tl
