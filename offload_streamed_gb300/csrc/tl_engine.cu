// tl_engine.cu -- the prefetch / eviction engine behind the C ABI.
//
// Resources per handle: two copy streams (host->device, device->host), a ring
// of (d+1) device slots for weight tiles, min(2, N) device staging slots for
// gradient tiles, and events that order them:
//   ready[s]   copy of a tile into weight slot s has landed      (h2d -> compute)
//   free[s]    last reader of weight slot s has finished         (compute -> h2d)
//   dwdone[g]  gradient tile in staging slot g is complete       (compute -> d2h)
//   drained[g] staging slot g has been copied back to the host   (d2h -> compute)
// The copy of tile f into slot f % (d+1) waits for free[] of the fetch d+1
// earlier, so the h2d stream runs up to d tiles ahead of the compute stream
// (aicassindra tm_zero_infinity, "Prefetch depth: how far ahead the pipeline
// must run"; pwwt.cn/news/5430303, "关键技术三", 动态预取器).  A slot whose
// reader has finished is refilled: that is the release of the gathered
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
// calls; chains of operators through one ring; the hooks of the host
// optimizer (tl_optimizer: host waits before a tile's W is copied in or its
// dW overwritten) and of the file tier (tl_filetier: a tile's bytes pass
// through pinned host slots between a file and the same copies); the sampled
// per-launch and per-copy timing and the call timeline built from it; and
// the persistent-pass mode (tl_pass.cu).
#include "tiled_linear.h"
#include "tl_filetier.h"
#include "tl_gemm.h"
#include "tl_optimizer.h"

#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <deque>
#include <mutex>
#include <new>
#include <string>
#include <vector>

namespace {

// Workspace header: the kernels' error word, then the persistent pass's
// sequence flags and per-position counters (zeroed per call).
constexpr size_t kHeaderBytes = 65536;
constexpr size_t kTileCounterOffset = 64;
constexpr size_t kFlagsOffset = 256;
constexpr size_t kDoneOffset = 4096;
constexpr size_t kDwDoneOffset = kDoneOffset + 4 * size_t(tl::kMaxPassTiles);
constexpr size_t kDxDoneOffset = kDwDoneOffset + 4 * size_t(tl::kMaxPassTiles);
static_assert(kDxDoneOffset + 4 * size_t(tl::kMaxPassTiles) <= kHeaderBytes, "header layout");

// Stream memory operations (copy streams <-> persistent pass kernel).
using StreamValueFn = CUresult (*)(CUstream, CUdeviceptr, cuuint32_t, unsigned int);
struct MemOps {
    StreamValueFn write = nullptr, wait = nullptr;
};
const MemOps& memops() {
    static MemOps m;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuStreamWriteValue32", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            m.write = reinterpret_cast<StreamValueFn>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuStreamWaitValue32", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            m.wait = reinterpret_cast<StreamValueFn>(p);
    });
    return m;
}
constexpr unsigned kWaitGeq = 0x0;       // CU_STREAM_WAIT_VALUE_GEQ
constexpr unsigned kWriteDefault = 0x0;  // CU_STREAM_WRITE_VALUE_DEFAULT
constexpr size_t kAlign = 256;
constexpr int kMaxStage = 2;
constexpr int kAutoMaxDepth = 3;

thread_local std::string g_create_error;

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct Shape {
    int64_t K = 0, M = 0, Mi = 0;
    int32_t N = 0;
};

// Shape rules shared by workspace sizing and create.  Empty string = valid.
std::string check_shape(int64_t K, int64_t M, int32_t N, int32_t d) {
    if (K < 8 || K % 8) return "K must be a positive multiple of 8";
    if (M < 1 || N < 1) return "M and N must be >= 1";
    if (M % N) return "M must be divisible by N";
    if ((M / N) % 8) return "M/N (tile width) must be a multiple of 8";
    if (d < -1) return "d must be >= -1";
    if (K > (int64_t(1) << 31) || M > (int64_t(1) << 34)) return "K or M too large";
    return {};
}

int32_t slots_for(int32_t N, int32_t d) {
    const int32_t dd = d < 0 ? std::min(N - 1, kAutoMaxDepth) : std::min(d, N - 1);
    return dd + 1;
}

size_t tile_bytes(int64_t K, int64_t Mi) { return size_t(K) * size_t(Mi) * 2; }

// One tiled linear operator of a handle: Y [T, M] = X [T, K] . W, W split into
// N column tiles held in pinned host memory.  A handle runs one operator, or
// a chain of them (operator l's output is operator l+1's input); `first` is
// the index of the operator's first tile in the handle's tile order.
struct Op {
    Shape s;
    const uint8_t* w_host = nullptr;
    uint8_t* dw_host = nullptr;
    tl_layout layout = TL_LAYOUT_TILE_MAJOR;
    int32_t first = 0;
};

// Workspace of a handle over `ops`: the header, then d+1 ring slots and
// min(2, tiles) staging slots, each sized for the largest tile.
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
size_t workspace_for(const std::vector<Shape>& ops, int32_t d) {
    const int32_t n = total_tiles(ops);
    return kHeaderBytes + size_t(slots_for(n, d) + std::min(n, kMaxStage)) * ring_slot_bytes(ops);
}

constexpr int kTimingRing = 16;

// Timing events of one call.  Per tile: [0] kernel-1 start, [1] kernel-1 end,
// [2] kernel-2 start, [3] kernel-2 end, [4] h2d start, [5] h2d end, [6] d2h
// start, [7] d2h end.  Forward records [0],[1],[4],[5].
struct CallSlot {
    cudaEvent_t start = nullptr, end = nullptr;
    std::vector<cudaEvent_t> ev[8];
    std::vector<char> dx_at;  // backward: a dX launch closed a tile group at this position
    bool pending = false;  // recorded, not yet harvested
    bool harvested = false;
    int32_t nk = 0;        // kernel spans recorded (N per-tile launches, or 1 pass)
    int32_t depth = 0, launches = 0, reused = 0;
    bool timed = true;     // per-launch and per-copy events recorded (see tiled_linear_set_timing)
    int64_t h2d_bytes = 0, d2h_bytes = 0;
    float total = 0, gemm1 = 0, gemm2 = 0, h2d = 0, d2h = 0;
};

// A ring of call slots: a call reuses the slot of the call kTimingRing
// earlier, harvesting its timings first (that call finished long ago, so the
// host does not stall the device).  Harvested calls are added to the sums.
struct Phase {
    bool backward = false;
    std::vector<CallSlot> ring;
    uint64_t calls = 0;
    int last = -1;        // ring index of the last timed call
    int64_t sum_calls = 0, sum_timed = 0;
    double sum_total = 0, sum_gemm1 = 0, sum_gemm2 = 0, sum_h2d = 0, sum_d2h = 0;
};

}  // namespace

struct tl_handle {
    int device = 0;
    Shape s;                 // operator 0 (the persistent mode runs single operators only)
    std::vector<Op> ops;     // the operators, in forward order
    bool single_api = true;  // created by tiled_linear_create[_tilemajor] (else a chain)
    int32_t n_total = 0;     // tiles over all operators
    tl_layout layout = TL_LAYOUT_ROW_MAJOR;
    int32_t d_req = 0, d = 0, slot_cap = 0, nstage = 0;
    bool auto_pending = false;
    const uint8_t* w_host = nullptr;
    uint8_t* dw_host = nullptr;
    uint8_t* ws = nullptr;
    size_t ws_bytes = 0;
    int32_t* err_dev = nullptr;
    int32_t* err_mirror = nullptr;  // pinned host copy of *err_dev, refreshed per call
    std::vector<uint8_t*> slot, stage;
    cudaStream_t h2d = nullptr, d2h = nullptr;
    std::vector<cudaEvent_t> ev_ready, ev_free, ev_dwdone, ev_drained;
    uint64_t fetch_seq = 0, stage_seq = 0;
    // One launch per tile: the ring slots in the order their last readers
    // were enqueued (a fetch takes the front: the slot freed earliest), the
    // tile each slot holds (-1: none), and whether a backward takes the
    // tiles it starts with from the ring when they are still there.
    std::deque<int> slot_q;
    std::vector<int32_t> slot_tile;
    bool reuse = false;
    int32_t timing_every = 1;  // record per-launch / per-copy events on every n-th call
    // Host optimizer attached by tiled_linear_optimizer_create: its worker,
    // per-tile events the backward records (W read by the GPU, dW in host
    // memory) and the tile order of the last backward.
    tl::Optimizer* opt = nullptr;
    tl_optimizer* opt_owner = nullptr;  // the C object; its handle pointer is cleared on destroy
    std::vector<cudaEvent_t> opt_ev_w, opt_ev_dw;
    std::vector<int> opt_order;
    bool opt_have_bwd = false;  // a backward recorded the events since the last submit
    int num_sms = 0;
    bool persistent = false;  // whole passes as one persistent launch
    tl::FileTier* tier = nullptr;  // W and dW in files (tiled_linear_create_file), else in host memory
    uint32_t* flags = nullptr;
    uint32_t* done = nullptr;
    uint32_t* dwdone = nullptr;
    uint32_t* dxdone = nullptr;
    uint32_t* tile_counter = nullptr;   // dynamic tile schedule of the per-tile GEMMs (header word)
    cudaEvent_t ev_d2h_tail = nullptr;  // last dW write-back of the last backward call
    cudaEvent_t ev_call_done = nullptr; // end of the last call (calls share the pass counters)
    Phase fwd, bwd;
    tl_status sticky = TL_OK;
    std::string msg;
};

namespace {

struct DeviceGuard {
    int prev = -1;
    cudaError_t err = cudaSuccess;
    explicit DeviceGuard(int dev) {
        if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
        if (prev != dev) err = cudaSetDevice(dev);
    }
    ~DeviceGuard() {
        if (prev >= 0) cudaSetDevice(prev);
    }
};

tl_status fail(tl_handle* h, tl_status st, const std::string& what) {
    if (h) {
        h->msg = what;
        if (st == TL_ERR_CUDA || st == TL_ERR_TIMEOUT || st == TL_ERR_IO) h->sticky = st;
    }
    return st;
}

#define TL_TRY(h, call)                                                                   \
    do {                                                                                  \
        cudaError_t e_ = (call);                                                          \
        if (e_ != cudaSuccess)                                                            \
            return fail((h), TL_ERR_CUDA, std::string(#call) + ": " + cudaGetErrorString(e_)); \
    } while (0)

#define TL_CU(h, call)                                                                     \
    do {                                                                                   \
        CUresult r_ = (call);                                                              \
        if (r_ != CUDA_SUCCESS)                                                            \
            return fail((h), TL_ERR_CUDA, std::string(#call) + ": CUresult " + std::to_string(int(r_))); \
    } while (0)

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

tl_status create_phase(tl_handle* h, Phase& p, int n, bool backward) {
    p.backward = backward;
    p.ring.resize(kTimingRing);
    for (auto& c : p.ring) {
        c.dx_at.assign(size_t(n), 0);
        TL_TRY(h, cudaEventCreate(&c.start));
        TL_TRY(h, cudaEventCreate(&c.end));
        for (int k = 0; k < 8; ++k) {
            if (!backward && (k == 2 || k == 3 || k == 6 || k == 7)) continue;
            c.ev[k].assign(size_t(n), nullptr);
            for (auto& e : c.ev[k]) TL_TRY(h, cudaEventCreate(&e));
        }
    }
    return TL_OK;
}

void destroy_phase(Phase& p) {
    for (auto& c : p.ring) {
        if (c.start) cudaEventDestroy(c.start);
        if (c.end) cudaEventDestroy(c.end);
        for (auto& v : c.ev)
            for (auto e : v)
                if (e) cudaEventDestroy(e);
    }
    p.ring.clear();
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

float span_ms(cudaEvent_t a, cudaEvent_t b) {
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, a, b) != cudaSuccess) {
        cudaGetLastError();
        return 0.f;
    }
    return ms;
}

tl_status harvest(tl_handle* h, Phase& p, CallSlot& c, int n) {
    if (!c.pending) return TL_OK;
    TL_TRY(h, cudaEventSynchronize(c.end));
    c.total = span_ms(c.start, c.end);
    c.gemm1 = c.gemm2 = c.h2d = c.d2h = 0;
    if (!c.timed) {  // only counted: the sums describe the timed calls
        c.pending = false;
        c.harvested = true;
        p.sum_calls += 1;
        return TL_OK;
    }
    for (int i = 0; i < n; ++i) {
        if (i < c.nk) {
            c.gemm1 += span_ms(c.ev[0][i], c.ev[1][i]);
            if (p.backward && c.nk == n) c.gemm2 += span_ms(c.ev[2][i], c.ev[3][i]);
        }
        c.h2d += span_ms(c.ev[4][i], c.ev[5][i]);
        if (p.backward) c.d2h += span_ms(c.ev[6][i], c.ev[7][i]);
    }
    c.pending = false;
    c.harvested = true;
    p.sum_calls += 1;
    p.sum_timed += 1;
    p.sum_total += c.total;
    p.sum_gemm1 += c.gemm1;
    p.sum_gemm2 += c.gemm2;
    p.sum_h2d += c.h2d;
    p.sum_d2h += c.d2h;
    return TL_OK;
}

tl_status harvest_all(tl_handle* h, Phase& p) {
    for (auto& c : p.ring) {
        tl_status st = harvest(h, p, c, h->n_total);
        if (st != TL_OK) return st;
    }
    return TL_OK;
}

// Slot for the next call of phase p (harvesting the call that used it last).
CallSlot* begin_call(tl_handle* h, Phase& p, tl_status* st) {
    CallSlot& c = p.ring[p.calls % kTimingRing];
    *st = harvest(h, p, c, h->n_total);
    if (*st != TL_OK) return nullptr;
    c.timed = p.calls % uint64_t(h->timing_every) == 0;
    return &c;
}

void end_call(Phase& p, CallSlot& c) {
    c.pending = true;
    c.harvested = false;
    if (c.timed) p.last = int(p.calls % kTimingRing);
    p.calls += 1;
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
constexpr double kOptWaitSeconds = 600.0;

tl_status opt_wait(tl_handle* h, int g, bool update) {
    if (!h->opt) return TL_OK;
    const bool ok = update ? tl::optimizer_wait_update(h->opt, g, kOptWaitSeconds)
                           : tl::optimizer_wait_read(h->opt, g, kOptWaitSeconds);
    if (!ok) return fail(h, TL_ERR_TIMEOUT, tl::optimizer_error(h->opt));
    return TL_OK;
}

// Automatic depth: after the first forward call, d = ceil(t_fetch / t_layer)
// from that call's measured copy and kernel spans (tm_zero_infinity,
// "Prefetch depth"), bounded by the slots the workspace holds.
tl_status finish_auto_depth(tl_handle* h) {
    if (!h->auto_pending || h->fwd.last < 0) return TL_OK;
    CallSlot& c = h->fwd.ring[h->fwd.last];
    tl_status st = harvest(h, h->fwd, c, h->n_total);
    if (st != TL_OK) return st;
    const double fetch = c.h2d, layer = c.gemm1;
    int32_t dnew = 1;
    if (layer > 0) dnew = int32_t(std::ceil(fetch / layer));
    dnew = std::max<int32_t>(1, std::min<int32_t>(dnew, h->slot_cap - 1));
    if (h->slot_cap - 1 < 1) dnew = 0;
    if (dnew != h->d) {
        if (h->persistent) {
            // Every earlier fetch has been consumed (the first forward call has
            // finished); mark every slot free up to the next fetch so that the
            // new ring size starts clean.
            TL_TRY(h, cudaStreamSynchronize(h->h2d));
            for (int s = 0; s < tl::kMaxPassSlots; ++s)
                TL_CU(h, memops().write(reinterpret_cast<CUstream>(h->h2d),
                                        reinterpret_cast<CUdeviceptr>(h->flags + tl::kFlagFreed + s),
                                        uint32_t(h->fetch_seq), kWriteDefault));
        } else {
            for (size_t s = 0; s < h->slot.size(); ++s) TL_TRY(h, cudaStreamWaitEvent(h->h2d, h->ev_free[s], 0));
            h->fetch_seq = 0;
        }
        h->d = dnew;
        reset_ring(h);
    }
    h->auto_pending = false;
    return TL_OK;
}

// ---- persistent passes ------------------------------------------------------
CUstream cu(cudaStream_t s) { return reinterpret_cast<CUstream>(s); }
CUdeviceptr cuptr(const void* p) { return reinterpret_cast<CUdeviceptr>(p); }

// dX is accumulated over groups of consecutive tiles, one launch per group,
// whenever the ring holds several tiles (d >= 1) and the tile width splits
// into whole 64-deep K-blocks.  A group reduces at least 8192 deep where the
// ring allows: g = max(2, ceil(8192 / Mi)), at most d + 1, N and 4 (the
// GEMM's B segments); the last group of an operator may be smaller.  Pairs
// for wide tiles: a larger group holds more of the ring and delays the next
// fetches (groups of three measured 1 % slower on the GPT-scale layer), while
// narrow tiles need the depth (groups of three: +7 % on the FFN chain, whose
// down-projection has 1024-wide tiles).  Both launch modes use the same
// groups, so their dX agree bit for bit.
int dx_group(const tl_handle* h, const Shape& s) {
    if (h->d < 1 || s.N < 2 || s.Mi % tl::kBlockK) return 1;
    const int want = std::max<int>(2, int((8192 + s.Mi - 1) / s.Mi));
    return std::min({want, h->d + 1, s.N, int(tl::GemmDesc::kMaxSeg)});
}

tl::PassDesc pass_desc(const tl_handle* h, bool backward, int64_t T, uint64_t fetch_base, uint64_t stage_base) {
    tl::PassDesc d;
    d.backward = backward;
    d.T = T;
    d.K = h->s.K;
    d.Mi = h->s.Mi;
    d.N = h->s.N;
    d.nslots = h->d + 1;
    for (int i = 0; i < d.nslots && i < tl::kMaxPassSlots; ++i) d.slots[i] = h->slot[i];
    d.nstage = h->nstage;
    for (int g = 0; g < d.nstage && g < tl::kMaxPassStages; ++g) d.stages[g] = h->stage[g];
    d.fetch_base = uint32_t(fetch_base);
    d.stage_base = uint32_t(stage_base);
    d.dx_group = dx_group(h, h->s);
    d.flags = h->flags;
    d.done = h->done;
    d.dwdone = h->dwdone;
    d.dxdone = h->dxdone;
    d.err = h->err_dev;
    return d;
}

// Host->device fetches of the pass's tiles, in pass order, gated by the
// slots' "freed" flags and announced by "ready" flags.
tl_status enqueue_fetches(tl_handle* h, CallSlot& t, uint64_t base, bool backward) {
    const MemOps& mo = memops();
    const int N = h->s.N;
    const uint64_t nslots = uint64_t(h->d + 1);
    for (int j = 0; j < N; ++j) {
        const int i = backward ? N - 1 - j : j;
        const uint64_t f = base + uint64_t(j);
        const int sl = int(f % nslots);
        if (f >= nslots)
            TL_CU(h, mo.wait(cu(h->h2d), cuptr(h->flags + tl::kFlagFreed + sl), uint32_t(f - nslots + 1), kWaitGeq));
        TL_TRY(h, cudaEventRecord(t.ev[4][j], h->h2d));
        const tl_status st = fetch_w_tile(h, h->ops[0], i, h->slot[sl]);
        if (st != TL_OK) return st;
        TL_TRY(h, cudaEventRecord(t.ev[5][j], h->h2d));
        TL_CU(h, mo.write(cu(h->h2d), cuptr(h->flags + tl::kFlagReady + sl), uint32_t(f + 1), kWriteDefault));
    }
    return TL_OK;
}

tl_status launch_pass(tl_handle* h, const tl::PassDesc& d, cudaStream_t cs) {
    std::string why;
    if (tl::pass_launch(d, h->num_sms, cs, &why) != cudaSuccess) return fail(h, TL_ERR_CUDA, "pass launch: " + why);
    return TL_OK;
}

tl_status launch(tl_handle* h, const tl::GemmDesc& g0, cudaStream_t st) {
    tl::GemmDesc g = g0;
    g.tile_counter = h->tile_counter;  // one word: launches on the compute stream are ordered
    std::string why;
    cudaError_t e = tl::gemm_launch(g, h->num_sms, st, &why);
    if (e != cudaSuccess) return fail(h, TL_ERR_CUDA, "GEMM launch: " + why);
    return TL_OK;
}

// Create a handle over `ops` (one operator, or a chain) sharing one ring.
// W and dW in files instead of host memory (tiled_linear_create_file).
struct FileArgs {
    const char* w_path = nullptr;
    const char* dw_path = nullptr;
    int32_t host_slots = 0, io_threads = 0;
};

tl_status create_ops(tl_handle** out, std::vector<Op> ops, int32_t d, void* ws, size_t ws_bytes, int device,
                     bool single_api, const FileArgs* file = nullptr) {
    if (!out) {
        g_create_error = "out is NULL";
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
        g_create_error = bad;
        return TL_ERR_INVALID;
    }
    const int32_t N = first;  // tiles over all operators
    const size_t need = workspace_for(shapes, d);
    if (ws_bytes < need || (reinterpret_cast<uintptr_t>(ws) % kAlign)) {
        g_create_error = "workspace too small or not 256-byte aligned (need " + std::to_string(need) +
                         " bytes)";
        return TL_ERR_WORKSPACE;
    }

    tl_handle* h = new (std::nothrow) tl_handle();
    if (!h) {
        g_create_error = "out of host memory";
        return TL_ERR_INVALID;
    }
    auto bail = [&](tl_status st) {
        g_create_error = h->msg;
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

    // Carve the workspace: header (error word), weight slots, staging slots.
    const size_t tb = ring_slot_bytes(shapes);
    const int32_t min_slots = slots_for(N, d);
    const int32_t fit = int32_t(std::min<size_t>(size_t(N), (ws_bytes - kHeaderBytes) / tb - size_t(std::min(N, kMaxStage))));
    h->nstage = std::min(N, kMaxStage);
    h->slot_cap = d < 0 ? std::max(min_slots, std::min(fit, kAutoMaxDepth + 1)) : min_slots;
    h->slot_cap = std::min<int32_t>(h->slot_cap, N);
    h->d = h->slot_cap - 1;
    h->auto_pending = (d < 0);
    h->err_dev = reinterpret_cast<int32_t*>(h->ws);
    h->flags = reinterpret_cast<uint32_t*>(h->ws + kFlagsOffset);
    h->done = reinterpret_cast<uint32_t*>(h->ws + kDoneOffset);
    h->dwdone = reinterpret_cast<uint32_t*>(h->ws + kDwDoneOffset);
    h->dxdone = reinterpret_cast<uint32_t*>(h->ws + kDxDoneOffset);
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
    if (cudaEventCreateWithFlags(&h->ev_d2h_tail, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&h->ev_call_done, cudaEventDisableTiming) != cudaSuccess) {
        h->msg = "event creation failed";
        return bail(TL_ERR_CUDA);
    }
    // One launch per tile and per GEMM by default (the faster mode on the
    // GPT-scale layer: the separate dW and dX launches keep their operand
    // pairs L2-resident).  TILED_LINEAR_PERSISTENT=1 asks for whole passes as
    // one persistent launch, granted when the stream memory operations are
    // there and the shapes allow it (tile width a multiple of 256, at most 8
    // ring slots).
    {
        const char* env = std::getenv("TILED_LINEAR_PERSISTENT");
        const bool wanted = env && env[0] == '1';
        tl::PassDesc probe = pass_desc(h, false, 1, 0, 0);
        probe.nslots = h->slot_cap;
        probe.x = h->ws;
        probe.y = h->ws;
        const MemOps& mo = memops();
        if (wanted && single_api && !file && mo.write && mo.wait && tl::pass_check(probe, h->num_sms).empty()) {
            // the stream memory operations must work on this device
            if (mo.write(cu(h->h2d), cuptr(h->flags + tl::kNumFlags), 0u, kWriteDefault) == CUDA_SUCCESS &&
                cudaStreamSynchronize(h->h2d) == cudaSuccess && tl::pass_preload() == cudaSuccess)
                h->persistent = true;
            cudaGetLastError();
        }
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

// Forward as one persistent pass.  The caller's stream first waits for the
// handle's previous call (the pass counters are reused), then the counters of
// this pass are cleared and the kernel launched; the fetches run ahead on the
// h2d stream as far as the ring's "freed" flags allow.
tl_status forward_persistent(tl_handle* h, int64_t T, const void* x, void* y, cudaStream_t cs) {
    tl_status st;
    CallSlot* tp = begin_call(h, h->fwd, &st);
    if (!tp) return st;
    CallSlot& t = *tp;
    const Shape& s = h->s;
    const uint64_t base = h->fetch_seq;
    h->fetch_seq += uint64_t(s.N);
    TL_TRY(h, cudaStreamWaitEvent(cs, h->ev_call_done, 0));
    TL_TRY(h, cudaEventRecord(t.start, cs));
    TL_TRY(h, cudaMemsetAsync(h->done, 0, 4 * size_t(s.N), cs));
    // The kernel is launched before its fetches are queued: every flag wait
    // a copy stream holds must be satisfiable by a kernel already launched.
    tl::PassDesc d = pass_desc(h, false, T, base, 0);
    d.x = x;
    d.y = y;
    TL_TRY(h, cudaEventRecord(t.ev[0][0], cs));
    if ((st = launch_pass(h, d, cs)) != TL_OK) return st;
    TL_TRY(h, cudaEventRecord(t.ev[1][0], cs));
    if ((st = enqueue_fetches(h, t, base, false)) != TL_OK) return st;
    TL_TRY(h, cudaEventRecord(t.end, cs));
    TL_TRY(h, cudaEventRecord(h->ev_call_done, cs));
    TL_TRY(h, cudaMemcpyAsync(h->err_mirror, h->err_dev, sizeof(int32_t), cudaMemcpyDeviceToHost, cs));
    t.nk = 1;
    t.depth = h->d;
    t.launches = 1;
    t.h2d_bytes = int64_t(s.N) * int64_t(tile_bytes(s.K, s.Mi));
    t.d2h_bytes = 0;
    end_call(h->fwd, t);
    return TL_OK;
}

// Backward as one persistent pass; the dW write-backs are queued on the d2h
// stream, each gated by its staging slot's "dwready" flag, and the caller's
// stream waits for the last one.
tl_status backward_persistent(tl_handle* h, int64_t T, const void* x, const void* dy, float* dx,
                              cudaStream_t cs) {
    tl_status st;
    const Shape& s = h->s;
    const size_t tb = tile_bytes(s.K, s.Mi);
    if (T == 0) {  // dW = X^T dY over an empty sum: zero
        TL_TRY(h, cudaStreamWaitEvent(cs, h->ev_call_done, 0));
        TL_TRY(h, cudaStreamWaitEvent(cs, h->ev_d2h_tail, 0));
        TL_TRY(h, cudaMemsetAsync(h->stage[0], 0, tb, cs));
        for (int i = 0; i < s.N; ++i)
            if ((st = writeback_dw_tile(h, h->ops[0], i, h->stage[0], cs)) != TL_OK) return st;
        TL_TRY(h, cudaEventRecord(h->ev_call_done, cs));
        return TL_OK;
    }
    CallSlot* tp = begin_call(h, h->bwd, &st);
    if (!tp) return st;
    CallSlot& t = *tp;
    const MemOps& mo = memops();
    const uint64_t base = h->fetch_seq;
    h->fetch_seq += uint64_t(s.N);
    const uint64_t sbase = h->stage_seq;
    h->stage_seq += uint64_t(s.N);
    TL_TRY(h, cudaStreamWaitEvent(cs, h->ev_call_done, 0));
    TL_TRY(h, cudaEventRecord(t.start, cs));
    TL_TRY(h, cudaMemsetAsync(h->done, 0, (kDxDoneOffset - kDoneOffset) + 4 * size_t(s.N), cs));
    tl::PassDesc d = pass_desc(h, true, T, base, sbase);
    d.x = x;
    d.dy = dy;
    d.dx = dx;
    TL_TRY(h, cudaEventRecord(t.ev[0][0], cs));
    if ((st = launch_pass(h, d, cs)) != TL_OK) return st;
    TL_TRY(h, cudaEventRecord(t.ev[1][0], cs));
    if ((st = enqueue_fetches(h, t, base, true)) != TL_OK) return st;
    for (int j = 0; j < s.N; ++j) {
        const int i = s.N - 1 - j;
        const uint64_t sj = sbase + uint64_t(j);
        const int g = int(sj % uint64_t(h->nstage));
        TL_CU(h, mo.wait(cu(h->d2h), cuptr(h->flags + tl::kFlagDwReady + g), uint32_t(sj + 1), kWaitGeq));
        TL_TRY(h, cudaEventRecord(t.ev[6][j], h->d2h));
        if ((st = writeback_dw_tile(h, h->ops[0], i, h->stage[g], h->d2h)) != TL_OK) return st;
        TL_TRY(h, cudaEventRecord(t.ev[7][j], h->d2h));
        TL_CU(h, mo.write(cu(h->d2h), cuptr(h->flags + tl::kFlagDrained + g), uint32_t(sj + 1), kWriteDefault));
    }
    TL_TRY(h, cudaEventRecord(h->ev_d2h_tail, h->d2h));
    TL_TRY(h, cudaStreamWaitEvent(cs, h->ev_d2h_tail, 0));
    TL_TRY(h, cudaEventRecord(t.end, cs));
    TL_TRY(h, cudaEventRecord(h->ev_call_done, cs));
    TL_TRY(h, cudaMemcpyAsync(h->err_mirror, h->err_dev, sizeof(int32_t), cudaMemcpyDeviceToHost, cs));
    t.nk = 1;
    t.depth = h->d;
    t.launches = 1;
    t.h2d_bytes = int64_t(s.N) * int64_t(tb);
    t.d2h_bytes = int64_t(s.N) * int64_t(tb);
    end_call(h->bwd, t);
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

}  // namespace

extern "C" {

size_t tiled_linear_workspace_bytes(int64_t K, int64_t M, int32_t N, int32_t d) {
    if (!check_shape(K, M, N, d).empty()) return 0;
    return workspace_for({Shape{K, M, M / N, N}}, d);
}

static Op one_op(int64_t K, int64_t M, int32_t N, const void* w_host, void* dw_host, tl_layout layout) {
    Op o;
    o.s = Shape{K, M, N > 0 ? M / N : 0, N};
    o.w_host = static_cast<const uint8_t*>(w_host);
    o.dw_host = static_cast<uint8_t*>(dw_host);
    o.layout = layout;
    return o;
}

tl_status tiled_linear_create(tl_handle** out, int64_t K, int64_t M, int32_t N, int32_t d,
                              const void* w_host, void* dw_host, void* workspace_dev,
                              size_t workspace_bytes, int device) {
    return create_ops(out, {one_op(K, M, N, w_host, dw_host, TL_LAYOUT_ROW_MAJOR)}, d, workspace_dev,
                      workspace_bytes, device, true);
}

tl_status tiled_linear_create_tilemajor(tl_handle** out, int64_t K, int64_t M, int32_t N, int32_t d,
                                        const void* w_host, void* dw_host, void* workspace_dev,
                                        size_t workspace_bytes, int device) {
    return create_ops(out, {one_op(K, M, N, w_host, dw_host, TL_LAYOUT_TILE_MAJOR)}, d, workspace_dev,
                      workspace_bytes, device, true);
}

tl_status tiled_linear_create_file(tl_handle** out, int64_t K, int64_t M, int32_t N, int32_t d, const char* w_path,
                                   const char* dw_path, int32_t host_slots, int32_t io_threads, void* workspace_dev,
                                   size_t workspace_bytes, int device) {
    std::string bad;
    if (!w_path || !dw_path || !w_path[0] || !dw_path[0]) bad = "null or empty file path";
    else if (host_slots < 2 || host_slots > 64) bad = "host_slots must be in 2..64";
    else if (io_threads < 1 || io_threads > 64) bad = "io_threads must be in 1..64";
    else if (check_shape(K, M, N, d).empty() && (K * (M / N) * 2) % 4096)
        bad = "a tile (K * M/N * 2 bytes) must be a multiple of 4096 bytes for direct I/O";
    if (!bad.empty()) {
        g_create_error = bad;
        if (out) *out = nullptr;
        return TL_ERR_INVALID;
    }
    FileArgs fa;
    fa.w_path = w_path;
    fa.dw_path = dw_path;
    fa.host_slots = host_slots;
    fa.io_threads = io_threads;
    return create_ops(out, {one_op(K, M, N, nullptr, nullptr, TL_LAYOUT_TILE_MAJOR)}, d, workspace_dev,
                      workspace_bytes, device, true, &fa);
}

tl_status tiled_linear_file_sync(tl_handle* h) {
    if (!h) return TL_ERR_STATE;
    if (!h->tier) return fail(h, TL_ERR_INVALID, "the handle keeps W and dW in host memory");
    std::string why;
    if (!h->tier->sync(&why)) return fail(h, TL_ERR_IO, "file tier: " + why);
    return TL_OK;
}

tl_status tiled_linear_file_stats(const tl_handle* h, tl_file_stats* out) {
    if (!h || !out) return TL_ERR_INVALID;
    if (!h->tier) return TL_ERR_INVALID;
    const tl::FileTierStats st = h->tier->stats();
    std::memset(out, 0, sizeof(*out));
    out->read_bytes = st.read_bytes;
    out->write_bytes = st.write_bytes;
    out->read_seconds = st.read_s;
    out->write_seconds = st.write_s;
    out->fetch_wait_seconds = st.fetch_wait_s;
    out->writeback_wait_seconds = st.writeback_wait_s;
    out->host_slots = h->tier->host_slots();
    out->io_threads = h->tier->io_threads();
    return TL_OK;
}

static std::string chain_args(int32_t L, const int64_t* dims, const int32_t* n_tiles) {
    if (L < 1 || L > 64) return "L must be in 1..64";
    if (!dims || !n_tiles) return "null dims or n_tiles";
    return {};
}

size_t tiled_linear_chain_workspace_bytes(int32_t L, const int64_t* dims, const int32_t* n_tiles, int32_t d) {
    if (!chain_args(L, dims, n_tiles).empty()) return 0;
    std::vector<Shape> shapes;
    for (int l = 0; l < L; ++l) {
        if (!check_shape(dims[l], dims[l + 1], n_tiles[l], d).empty()) return 0;
        shapes.push_back(Shape{dims[l], dims[l + 1], dims[l + 1] / n_tiles[l], n_tiles[l]});
    }
    return workspace_for(shapes, d);
}

tl_status tiled_linear_chain_create(tl_handle** out, int32_t L, const int64_t* dims, const int32_t* n_tiles,
                                    int32_t d, const void* const* w_host, void* const* dw_host,
                                    void* workspace_dev, size_t workspace_bytes, int device) {
    std::string bad = chain_args(L, dims, n_tiles);
    if (bad.empty() && (!w_host || !dw_host)) bad = "null w_host or dw_host array";
    if (!bad.empty()) {
        g_create_error = bad;
        if (out) *out = nullptr;
        return TL_ERR_INVALID;
    }
    std::vector<Op> ops;
    for (int l = 0; l < L; ++l)
        ops.push_back(one_op(dims[l], dims[l + 1], n_tiles[l], w_host[l], dw_host[l], TL_LAYOUT_TILE_MAJOR));
    return create_ops(out, ops, d, workspace_dev, workspace_bytes, device, false);
}

// Shared argument checks of the call entry points.  Returns TL_OK or the
// status to return (with the handle's message set).
static tl_status call_prologue(tl_handle* h, int64_t T) {
    tl_status st = check_usable(h);
    if (st != TL_OK) return st;
    if (T < 0 || T > (int64_t(1) << 30)) return fail(h, TL_ERR_INVALID, "T out of range");
    return TL_OK;
}

static bool misaligned(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; }

tl_status tiled_linear_forward(tl_handle* h, int64_t T, const void* x_dev, void* y_dev, void* stream) {
    tl_status st = call_prologue(h, T);
    if (st != TL_OK) return st;
    if (!h->single_api) return fail(h, TL_ERR_INVALID, "a chain handle runs tiled_linear_chain_forward");
    if (T == 0) return TL_OK;
    if (!x_dev || !y_dev) return fail(h, TL_ERR_INVALID, "null x or y");
    if (misaligned(x_dev) || misaligned(y_dev)) return fail(h, TL_ERR_INVALID, "x and y must be 16-byte aligned");
    DeviceGuard guard(h->device);
    if (guard.err != cudaSuccess) return fail(h, TL_ERR_CUDA, "cudaSetDevice failed");
    if ((st = finish_auto_depth(h)) != TL_OK) return st;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    if (h->persistent) return forward_persistent(h, T, x_dev, y_dev, cs);
    void* ys[1] = {y_dev};
    return forward_tiles(h, T, x_dev, ys, cs);
}

tl_status tiled_linear_backward(tl_handle* h, int64_t T, const void* x_dev, const void* dy_dev,
                                float* dx_dev, void* stream) {
    tl_status st = call_prologue(h, T);
    if (st != TL_OK) return st;
    if (!h->single_api) return fail(h, TL_ERR_INVALID, "a chain handle runs tiled_linear_chain_backward");
    if (T > 0 && (!x_dev || !dy_dev || !dx_dev)) return fail(h, TL_ERR_INVALID, "null x, dy or dx");
    if (misaligned(x_dev) || misaligned(dy_dev) || misaligned(dx_dev))
        return fail(h, TL_ERR_INVALID, "x, dy and dx must be 16-byte aligned");
    DeviceGuard guard(h->device);
    if (guard.err != cudaSuccess) return fail(h, TL_ERR_CUDA, "cudaSetDevice failed");
    if ((st = finish_auto_depth(h)) != TL_OK) return st;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    if (h->persistent) return backward_persistent(h, T, x_dev, dy_dev, dx_dev, cs);
    return backward_tiles(h, T, x_dev, nullptr, dy_dev, dx_dev, nullptr, nullptr, cs);
}

size_t tiled_linear_chain_scratch_bytes(int64_t T, int32_t L, const int64_t* dims) {
    if (T < 0 || L < 1 || !dims) return 0;
    int64_t inner = 0;
    for (int l = 1; l < L; ++l) inner = std::max(inner, dims[l]);
    if (inner == 0) return 0;
    const size_t dy_bufs = L >= 3 ? 2 : 1;  // dY buffers: an operator between two others reads one, writes the other
    return align_up(size_t(T) * size_t(inner) * 4, kAlign) + dy_bufs * align_up(size_t(T) * size_t(inner) * 2, kAlign);
}

tl_status tiled_linear_chain_forward(tl_handle* h, int64_t T, const void* x_dev, void* const* y_dev,
                                     void* stream) {
    tl_status st = call_prologue(h, T);
    if (st != TL_OK) return st;
    if (h->single_api) return fail(h, TL_ERR_INVALID, "a single-operator handle runs tiled_linear_forward");
    if (T == 0) return TL_OK;
    if (!x_dev || !y_dev || misaligned(x_dev)) return fail(h, TL_ERR_INVALID, "null or misaligned x / y array");
    for (size_t l = 0; l < h->ops.size(); ++l)
        if (!y_dev[l] || misaligned(y_dev[l]))
            return fail(h, TL_ERR_INVALID, "y[" + std::to_string(l) + "] is null or not 16-byte aligned");
    DeviceGuard guard(h->device);
    if (guard.err != cudaSuccess) return fail(h, TL_ERR_CUDA, "cudaSetDevice failed");
    if ((st = finish_auto_depth(h)) != TL_OK) return st;
    return forward_tiles(h, T, x_dev, y_dev, static_cast<cudaStream_t>(stream));
}

tl_status tiled_linear_chain_backward(tl_handle* h, int64_t T, const void* x_dev, const void* const* y_dev,
                                      const void* dy_dev, float* dx_dev, void* scratch_dev,
                                      size_t scratch_bytes, void* stream) {
    tl_status st = call_prologue(h, T);
    if (st != TL_OK) return st;
    if (h->single_api) return fail(h, TL_ERR_INVALID, "a single-operator handle runs tiled_linear_backward");
    const int L = int(h->ops.size());
    float* scr_dx = nullptr;
    void* scr_dy[2] = {nullptr, nullptr};
    if (T > 0) {
        if (!x_dev || !dy_dev || !dx_dev || misaligned(x_dev) || misaligned(dy_dev) || misaligned(dx_dev))
            return fail(h, TL_ERR_INVALID, "x, dy and dx must be non-null and 16-byte aligned");
        if (L > 1) {
            if (!y_dev) return fail(h, TL_ERR_INVALID, "null y array");
            for (int l = 0; l + 1 < L; ++l)
                if (!y_dev[l] || misaligned(y_dev[l]))
                    return fail(h, TL_ERR_INVALID, "y[" + std::to_string(l) + "] is null or not 16-byte aligned");
            std::vector<int64_t> dims;
            dims.push_back(h->ops[0].s.K);
            for (const Op& o : h->ops) dims.push_back(o.s.M);
            const size_t need = tiled_linear_chain_scratch_bytes(T, L, dims.data());
            if (!scratch_dev || scratch_bytes < need || (reinterpret_cast<uintptr_t>(scratch_dev) % kAlign))
                return fail(h, TL_ERR_WORKSPACE, "scratch too small or not 256-byte aligned (need " +
                                                     std::to_string(need) + " bytes)");
            int64_t inner = 0;
            for (int l = 1; l < L; ++l) inner = std::max(inner, dims[size_t(l)]);
            scr_dx = static_cast<float*>(scratch_dev);
            scr_dy[0] = static_cast<uint8_t*>(scratch_dev) + align_up(size_t(T) * size_t(inner) * 4, kAlign);
            if (L >= 3) scr_dy[1] = static_cast<uint8_t*>(scr_dy[0]) + align_up(size_t(T) * size_t(inner) * 2, kAlign);
        }
    }
    DeviceGuard guard(h->device);
    if (guard.err != cudaSuccess) return fail(h, TL_ERR_CUDA, "cudaSetDevice failed");
    if ((st = finish_auto_depth(h)) != TL_OK) return st;
    return backward_tiles(h, T, x_dev, y_dev, dy_dev, dx_dev, scr_dx, scr_dy, static_cast<cudaStream_t>(stream));
}

struct tl_optimizer {
    tl_handle* h = nullptr;
    bool has_acc = false;
};

static void detach_optimizer(tl_handle* h) {
    if (h->opt_owner) {
        h->opt_owner->h = nullptr;
        h->opt_owner = nullptr;
    }
    if (!h->opt) return;
    tl::optimizer_delete(h->opt);  // waits for the submitted jobs
    h->opt = nullptr;
    for (auto* v : {&h->opt_ev_w, &h->opt_ev_dw}) {
        for (auto e : *v)
            if (e) cudaEventDestroy(e);
        v->clear();
    }
    h->opt_have_bwd = false;
}

tl_status tiled_linear_destroy(tl_handle* h) {
    if (!h) return TL_OK;
    tl_status st = h->sticky;
    {
        DeviceGuard guard(h->device);
        detach_optimizer(h);
        if (h->h2d) cudaStreamSynchronize(h->h2d);
        if (h->d2h) cudaStreamSynchronize(h->d2h);
        delete h->tier;  // stores the dW tiles still being written
        h->tier = nullptr;
        for (auto* v : {&h->ev_ready, &h->ev_free, &h->ev_dwdone, &h->ev_drained})
            for (auto e : *v) {
                if (e) {
                    cudaEventSynchronize(e);
                    cudaEventDestroy(e);
                }
            }
        for (Phase* p : {&h->fwd, &h->bwd})
            for (auto& c : p->ring)
                if (c.end) cudaEventSynchronize(c.end);
        destroy_phase(h->fwd);
        destroy_phase(h->bwd);
        if (h->ev_d2h_tail) cudaEventDestroy(h->ev_d2h_tail);
        if (h->ev_call_done) cudaEventDestroy(h->ev_call_done);
        if (h->h2d) cudaStreamDestroy(h->h2d);
        if (h->d2h) cudaStreamDestroy(h->d2h);
        if (h->err_mirror) cudaFreeHost(h->err_mirror);
        cudaGetLastError();
    }
    delete h;
    return st;
}

const char* tiled_linear_last_error(const tl_handle* h) {
    if (!h) return g_create_error.c_str();
    return h->msg.c_str();
}

tl_status tiled_linear_get_trace(tl_handle* h, int32_t backward, tl_trace_event* out, int32_t capacity,
                                 int32_t* count) {
    if (!h || !count || capacity < 0 || (capacity > 0 && !out)) return TL_ERR_INVALID;
    *count = 0;
    DeviceGuard guard(h->device);
    Phase& p = backward ? h->bwd : h->fwd;
    tl_status st = harvest_all(h, p);
    if (st != TL_OK) return st;
    if (p.last < 0) return TL_OK;
    const CallSlot& c = p.ring[size_t(p.last)];
    int32_t n = 0;
    auto add = [&](int32_t kind, int32_t tile, cudaEvent_t a, cudaEvent_t b) {
        const float t0 = span_ms(c.start, a), t1 = span_ms(c.start, b);
        if (n < capacity) out[n] = tl_trace_event{kind, tile, t0, t1};
        ++n;
    };
    const int NT = h->n_total;
    if (c.nk == 1 && NT > 1) {  // one persistent launch for the pass
        add(TL_TRACE_PASS, -1, c.ev[0][0], c.ev[1][0]);
    } else {
        for (int j = 0; j < c.nk; ++j) {
            const int tile = backward ? NT - 1 - j : j;
            add(backward ? TL_TRACE_DW_GEMM : TL_TRACE_FWD_GEMM, tile, c.ev[0][j], c.ev[1][j]);
            if (backward && c.dx_at[size_t(j)]) add(TL_TRACE_DX_GEMM, tile, c.ev[2][j], c.ev[3][j]);
        }
    }
    for (int j = 0; j < NT; ++j) {
        const int tile = backward ? NT - 1 - j : j;
        if (!backward || j >= c.reused) add(TL_TRACE_H2D, tile, c.ev[4][j], c.ev[5][j]);  // reused: no copy
        if (backward) add(TL_TRACE_D2H, tile, c.ev[6][j], c.ev[7][j]);
    }
    *count = n;
    return TL_OK;
}

tl_status tiled_linear_get_stats(tl_handle* h, void* out_v) {
    if (!h || !out_v) return TL_ERR_INVALID;
    tl_stats* out = static_cast<tl_stats*>(out_v);
    std::memset(out, 0, sizeof(*out));
    DeviceGuard guard(h->device);
    out->n_tiles = h->n_total;
    out->depth = h->d;
    tl_status st = harvest_all(h, h->fwd);
    if (st == TL_OK) st = harvest_all(h, h->bwd);
    if (st != TL_OK) return st;
    if (h->fwd.last >= 0) {
        const CallSlot& c = h->fwd.ring[h->fwd.last];
        out->fwd_valid = 1;
        out->fwd_total_ms = c.total;
        out->fwd_gemm_ms = c.gemm1;
        out->fwd_h2d_ms = c.h2d;
        out->fwd_wait_ms = c.total - c.gemm1;
        out->fwd_h2d_bytes = c.h2d_bytes;
        out->fwd_launches = c.launches;
        out->depth = c.depth;
    }
    if (h->bwd.last >= 0) {
        const CallSlot& c = h->bwd.ring[h->bwd.last];
        out->bwd_valid = 1;
        out->bwd_total_ms = c.total;
        out->bwd_gemm_ms = c.gemm1 + c.gemm2;
        out->bwd_dw_gemm_ms = c.nk == h->n_total ? c.gemm1 : 0.f;
        out->bwd_dx_gemm_ms = c.nk == h->n_total ? c.gemm2 : 0.f;
        out->bwd_h2d_ms = c.h2d;
        out->bwd_d2h_ms = c.d2h;
        out->bwd_wait_ms = c.total - c.gemm1 - c.gemm2;
        out->bwd_h2d_bytes = c.h2d_bytes;
        out->bwd_d2h_bytes = c.d2h_bytes;
        out->bwd_launches = c.launches;
        out->bwd_reused_tiles = c.reused;
    }
    out->fwd_calls = h->fwd.sum_calls;
    out->sum_fwd_total_ms = h->fwd.sum_total;
    out->sum_fwd_gemm_ms = h->fwd.sum_gemm1;
    out->sum_fwd_h2d_ms = h->fwd.sum_h2d;
    out->bwd_calls = h->bwd.sum_calls;
    out->sum_bwd_total_ms = h->bwd.sum_total;
    out->sum_bwd_dw_gemm_ms = h->bwd.sum_gemm1;
    out->sum_bwd_dx_gemm_ms = h->bwd.sum_gemm2;
    out->sum_bwd_h2d_ms = h->bwd.sum_h2d;
    out->sum_bwd_d2h_ms = h->bwd.sum_d2h;
    out->sum_bwd_gemm_ms = h->bwd.sum_gemm1 + h->bwd.sum_gemm2;
    out->persistent = h->persistent ? 1 : 0;
    out->fwd_timed_calls = h->fwd.sum_timed;
    out->bwd_timed_calls = h->bwd.sum_timed;
    out->timing_every = h->timing_every;
    int32_t word = 0;
    TL_TRY(h, cudaMemcpy(&word, h->err_dev, sizeof(word), cudaMemcpyDeviceToHost));
    if (word != 0)
        return fail(h, TL_ERR_TIMEOUT,
                    "a kernel's bounded wait timed out (error bits " + std::to_string(word) + ")");
    return h->sticky;
}

static std::string adam_config_error(const tl_adam_config* c) {
    if (!c) return "null config";
    if (!(c->lr >= 0.f) || !std::isfinite(c->lr)) return "lr must be finite and >= 0";
    if (!(c->beta1 >= 0.f && c->beta1 < 1.f) || !(c->beta2 >= 0.f && c->beta2 < 1.f))
        return "beta1 and beta2 must be in [0, 1)";
    if (!(c->eps > 0.f) || !std::isfinite(c->eps)) return "eps must be finite and > 0";
    if (!(c->weight_decay >= 0.f) || !std::isfinite(c->weight_decay)) return "weight_decay must be finite and >= 0";
    return {};
}

static tl::AdamHyper hyper(const tl_adam_config* c) {
    tl::AdamHyper hp;
    hp.lr = c->lr;
    hp.beta1 = c->beta1;
    hp.beta2 = c->beta2;
    hp.eps = c->eps;
    hp.weight_decay = c->weight_decay;
    return hp;
}

tl_status tiled_linear_adam_update(const tl_adam_config* cfg, int64_t step, int64_t n, float* master, float* m,
                                   float* v, const float* grad_acc, const void* grad_bf16, void* w_bf16) {
    if (!adam_config_error(cfg).empty() || step < 1 || n < 0) return TL_ERR_INVALID;
    if (n == 0) return TL_OK;
    if (!master || !m || !v || !grad_bf16 || !w_bf16) return TL_ERR_INVALID;
    tl::Block b;
    b.master = master;
    b.m = m;
    b.v = v;
    b.acc = const_cast<float*>(grad_acc);
    b.grad = static_cast<const uint16_t*>(grad_bf16);
    b.w = static_cast<uint16_t*>(w_bf16);
    b.rows = 1;
    b.cols = n;
    b.ld = n;
    tl::adam_rows(b, hyper(cfg), step, grad_acc != nullptr, 0, 1);
    return TL_OK;
}

tl_status tiled_linear_optimizer_create(tl_optimizer** out, tl_handle* h, const tl_adam_config* cfg,
                                        float* const* master, float* const* m, float* const* v,
                                        float* const* grad_acc) {
    if (!out) return TL_ERR_INVALID;
    *out = nullptr;
    tl_status st = check_usable(h);
    if (st != TL_OK) return st;
    const std::string bad = adam_config_error(cfg);
    if (!bad.empty()) return fail(h, TL_ERR_INVALID, "optimizer config: " + bad);
    if (h->persistent) return fail(h, TL_ERR_INVALID, "the host optimizer needs the per-tile launch mode");
    if (h->tier) return fail(h, TL_ERR_INVALID, "the host optimizer needs W and dW in host memory");
    if (h->opt) return fail(h, TL_ERR_STATE, "the handle already has an optimizer");
    if (!master || !m || !v) return fail(h, TL_ERR_INVALID, "null master, m or v array");
    std::vector<tl::Block> tiles;
    for (size_t l = 0; l < h->ops.size(); ++l) {
        const Op& o = h->ops[l];
        if (!master[l] || !m[l] || !v[l] || (grad_acc && !grad_acc[l]))
            return fail(h, TL_ERR_INVALID, "null parameter array for operator " + std::to_string(l));
        for (int i = 0; i < o.s.N; ++i) {
            const bool tm = o.layout == TL_LAYOUT_TILE_MAJOR;
            const size_t off = tm ? size_t(i) * size_t(o.s.K) * size_t(o.s.Mi) : size_t(i) * size_t(o.s.Mi);
            tl::Block b;
            b.master = master[l] + off;
            b.m = m[l] + off;
            b.v = v[l] + off;
            b.acc = grad_acc ? grad_acc[l] + off : nullptr;
            b.grad = reinterpret_cast<const uint16_t*>(o.dw_host) + off;
            b.w = reinterpret_cast<uint16_t*>(const_cast<uint8_t*>(o.w_host)) + off;
            b.rows = o.s.K;
            b.cols = o.s.Mi;
            b.ld = tm ? o.s.Mi : o.s.M;
            tiles.push_back(b);
        }
    }
    DeviceGuard guard(h->device);
    if (guard.err != cudaSuccess) return fail(h, TL_ERR_CUDA, "cudaSetDevice failed");
    auto* o = new (std::nothrow) tl_optimizer();
    if (!o) return fail(h, TL_ERR_INVALID, "out of host memory");
    h->opt_ev_w.assign(size_t(h->n_total), nullptr);
    h->opt_ev_dw.assign(size_t(h->n_total), nullptr);
    for (auto* vv : {&h->opt_ev_w, &h->opt_ev_dw})
        for (auto& e : *vv)
            if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) {
                detach_optimizer(h);
                delete o;
                return fail(h, TL_ERR_CUDA, "optimizer event creation failed");
            }
    try {
        h->opt = tl::optimizer_new(tiles, hyper(cfg), cfg->threads);
    } catch (const std::exception& e) {
        detach_optimizer(h);
        delete o;
        return fail(h, TL_ERR_INVALID, std::string("optimizer threads: ") + e.what());
    }
    h->opt_have_bwd = false;
    h->opt_owner = o;
    o->h = h;
    o->has_acc = grad_acc != nullptr;
    *out = o;
    return TL_OK;
}

static tl_status optimizer_submit_job(tl_optimizer* o, bool step) {
    if (!o || !o->h || !o->h->opt) return TL_ERR_STATE;
    tl_handle* h = o->h;
    tl_status st = check_usable(h);
    if (st != TL_OK) return st;
    if (!step && !o->has_acc) return fail(h, TL_ERR_INVALID, "accumulate needs a gradient accumulator");
    if (!h->opt_have_bwd) return fail(h, TL_ERR_STATE, "no backward since the last optimizer call");
    if (!tl::optimizer_submit(h->opt, step, h->opt_order, h->opt_ev_w, h->opt_ev_dw))
        return fail(h, TL_ERR_TIMEOUT, tl::optimizer_error(h->opt));
    h->opt_have_bwd = false;
    return TL_OK;
}

tl_status tiled_linear_optimizer_accumulate(tl_optimizer* o) { return optimizer_submit_job(o, false); }
tl_status tiled_linear_optimizer_step(tl_optimizer* o) { return optimizer_submit_job(o, true); }

tl_status tiled_linear_optimizer_wait(tl_optimizer* o) {
    if (!o || !o->h || !o->h->opt) return TL_ERR_STATE;
    if (!tl::optimizer_wait_all(o->h->opt, kOptWaitSeconds))
        return fail(o->h, TL_ERR_TIMEOUT, tl::optimizer_error(o->h->opt));
    return TL_OK;
}

tl_status tiled_linear_optimizer_stats(const tl_optimizer* o, int64_t* steps, double* busy_seconds) {
    if (!o || !o->h || !o->h->opt) return TL_ERR_STATE;
    if (steps) *steps = tl::optimizer_steps(o->h->opt);
    if (busy_seconds) *busy_seconds = tl::optimizer_busy_seconds(o->h->opt);
    return TL_OK;
}

tl_status tiled_linear_optimizer_destroy(tl_optimizer* o) {
    if (!o) return TL_OK;
    tl_status st = TL_OK;
    if (o->h && o->h->opt) {
        if (!tl::optimizer_error(o->h->opt).empty()) st = TL_ERR_TIMEOUT;
        DeviceGuard guard(o->h->device);
        detach_optimizer(o->h);
    }
    delete o;
    return st;
}

tl_status tiled_linear_set_tile_reuse(tl_handle* h, int32_t enable) {
    tl_status st = check_usable(h);
    if (st != TL_OK) return st;
    if (enable && h->persistent)
        return fail(h, TL_ERR_INVALID, "tile reuse needs the per-tile launch mode (TILED_LINEAR_PERSISTENT=1 is set)");
    h->reuse = enable != 0;
    return TL_OK;
}

tl_status tiled_linear_set_timing(tl_handle* h, int32_t every) {
    tl_status st = check_usable(h);
    if (st != TL_OK) return st;
    if (every < 1) return fail(h, TL_ERR_INVALID, "every must be >= 1");
    h->timing_every = every;
    return TL_OK;
}

tl_status tiled_linear_reset_stats(tl_handle* h) {
    if (!h) return TL_ERR_INVALID;
    DeviceGuard guard(h->device);
    tl_status st = harvest_all(h, h->fwd);
    if (st == TL_OK) st = harvest_all(h, h->bwd);
    if (st != TL_OK) return st;
    for (Phase* p : {&h->fwd, &h->bwd}) {
        p->sum_calls = 0;
        p->sum_timed = 0;
        p->sum_total = p->sum_gemm1 = p->sum_gemm2 = p->sum_h2d = p->sum_d2h = 0;
    }
    return TL_OK;
}

// ---- resident GEMMs --------------------------------------------------------
static tl_status raw_launch(const tl::GemmDesc& g0, void* stream) {
    tl::GemmDesc g = g0;
    // the caller's err buffer holds the error word and, next to it, the
    // tile counter of the dynamic schedule
    g.tile_counter = g.err ? reinterpret_cast<uint32_t*>(g.err + 1) : nullptr;
    std::string bad = tl::gemm_check(g);
    if (!bad.empty()) return TL_ERR_INVALID;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return TL_ERR_CUDA;
    std::string why;
    return tl::gemm_launch(g, sms, static_cast<cudaStream_t>(stream), &why) == cudaSuccess ? TL_OK
                                                                                           : TL_ERR_CUDA;
}

tl_status tiled_linear_gemm_forward(int64_t T, int64_t K, int64_t n, const void* x_dev, int64_t ldx,
                                    const void* w_dev, int64_t ldw, void* y_dev, int64_t ldy,
                                    int32_t* err_dev, void* stream) {
    tl::GemmDesc g;
    g.m_dim = T;
    g.n_dim = n;
    g.k_dim = K;
    g.a = x_dev;
    g.lda = ldx;
    g.a_mn_major = false;
    g.b = w_dev;
    g.ldb = ldw;
    g.b_mn_major = true;
    g.d = y_dev;
    g.ldd = ldy;
    g.out = tl::OutKind::BF16;
    g.err = err_dev;
    return raw_launch(g, stream);
}

tl_status tiled_linear_gemm_dw(int64_t T, int64_t K, int64_t n, const void* x_dev, int64_t ldx,
                               const void* dy_dev, int64_t lddy, void* dw_dev, int64_t lddw,
                               int32_t* err_dev, void* stream) {
    tl::GemmDesc g;
    g.m_dim = K;
    g.n_dim = n;
    g.k_dim = T;
    g.a = x_dev;
    g.lda = ldx;
    g.a_mn_major = true;
    g.b = dy_dev;
    g.ldb = lddy;
    g.b_mn_major = true;
    g.d = dw_dev;
    g.ldd = lddw;
    g.out = tl::OutKind::BF16;
    g.err = err_dev;
    return raw_launch(g, stream);
}

tl_status tiled_linear_gemm_dx(int64_t T, int64_t K, int64_t n, const void* dy_dev, int64_t lddy,
                               const void* w_dev, int64_t ldw, float* dx_dev, int64_t lddx,
                               int32_t accumulate, int32_t* err_dev, void* stream) {
    tl::GemmDesc g;
    g.m_dim = T;
    g.n_dim = K;
    g.k_dim = n;
    g.a = dy_dev;
    g.lda = lddy;
    g.a_mn_major = false;
    g.b = w_dev;
    g.ldb = ldw;
    g.b_mn_major = false;
    g.d = dx_dev;
    g.ldd = lddx;
    g.out = tl::OutKind::F32;
    g.accumulate = accumulate != 0;
    g.err = err_dev;
    return raw_launch(g, stream);
}

tl_status tiled_linear_gemm_dx_bf16(int64_t T, int64_t K, int64_t n, const void* dy_dev, int64_t lddy,
                                    const void* w_dev, int64_t ldw, const float* addend_dev, int64_t ld_add,
                                    void* dx_dev, int64_t lddx, int32_t* err_dev, void* stream) {
    tl::GemmDesc g;
    g.m_dim = T;
    g.n_dim = K;
    g.k_dim = n;
    g.a = dy_dev;
    g.lda = lddy;
    g.a_mn_major = false;
    g.b = w_dev;
    g.ldb = ldw;
    g.b_mn_major = false;
    g.d = dx_dev;
    g.ldd = lddx;
    g.out = tl::OutKind::BF16;
    g.addend = addend_dev;
    g.ld_addend = ld_add;
    g.err = err_dev;
    return raw_launch(g, stream);
}

tl_status tiled_linear_selftest_timeout(void* scratch_dev, size_t scratch_bytes, int64_t timeout_ns,
                                        void* stream) {
    constexpr size_t kNeed = 256 + 128 * 256 * 2;
    if (!scratch_dev || (reinterpret_cast<uintptr_t>(scratch_dev) & 255u) || scratch_bytes < kNeed ||
        timeout_ns <= 0 || timeout_ns > int64_t(10000000000))
        return TL_ERR_INVALID;
    auto* base = static_cast<uint8_t*>(scratch_dev);
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(base, 0, 2 * sizeof(int32_t), cs) != cudaSuccess) return TL_ERR_CUDA;
    // A 128 x 256 x 64 forward GEMM whose operands are never read: the
    // producer withholds every load, so the MMA thread's first bounded wait
    // runs out.
    tl::GemmDesc g;
    g.m_dim = 128;
    g.n_dim = 256;
    g.k_dim = 64;
    g.a = base + 256;
    g.lda = 64;
    g.a_mn_major = false;
    g.b = base + 256;
    g.ldb = 256;
    g.b_mn_major = true;
    g.d = base + 256;
    g.ldd = 256;
    g.out = tl::OutKind::BF16;
    g.err = reinterpret_cast<int32_t*>(base);
    g.timeout_ns = uint64_t(timeout_ns);
    g.withhold_loads = true;
    return raw_launch(g, stream);
}

tl_status tiled_linear_host_alloc(size_t bytes, void** out) {
    if (!out) return TL_ERR_INVALID;
    *out = nullptr;
    if (bytes == 0) return TL_ERR_INVALID;
    if (cudaHostAlloc(out, bytes, cudaHostAllocPortable) != cudaSuccess) {
        cudaGetLastError();
        *out = nullptr;
        return TL_ERR_CUDA;
    }
    return TL_OK;
}

tl_status tiled_linear_host_free(void* p) {
    if (!p) return TL_OK;
    return cudaFreeHost(p) == cudaSuccess ? TL_OK : TL_ERR_CUDA;
}

const char* tiled_linear_version(void) { return "tiled_linear 0.1 (sm_103a)"; }

}  // extern "C"
