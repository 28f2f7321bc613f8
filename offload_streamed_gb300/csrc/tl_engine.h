// tl_engine.h -- internals of the prefetch / eviction engine behind the C ABI,
// shared by its translation units:
//   tl_ring.cpp   handle creation, the depth-d tile ring, the forward and
//                 backward schedules (fetch, GEMMs, write-back), auto depth
//   tl_stats.cpp  the sampled per-launch and per-copy timing, call timelines
//                 and the stats / trace entry points
//   tl_hooks.cpp  the host optimizer's and the file tier's entry points
//   tl_abi.cpp    the remaining C entry points (create, calls, chains,
//                 destroy, resident GEMMs, pinned memory)
//
// Resources per handle: two copy streams (host->device, device->host), a ring
// of (d+1) device slots for weight tiles, min(2, N) device staging slots for
// gradient tiles, and events that order them:
//   ready[s]   copy of a tile into weight slot s has landed      (h2d -> compute)
//   free[s]    last reader of weight slot s has finished         (compute -> h2d)
//   dwdone[g]  gradient tile in staging slot g is complete       (compute -> d2h)
//   drained[g] staging slot g has been copied back to the host   (d2h -> compute)
#pragma once
#include "tiled_linear.h"
#include "tl_filetier.h"
#include "tl_gemm.h"
#include "tl_optimizer.h"

#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <deque>
#include <string>
#include <vector>

namespace tl {

// Workspace header: the kernels' error word at 0 and the dynamic tile
// schedule's counter at kTileCounterOffset.
constexpr size_t kHeaderBytes = 4096;
constexpr size_t kTileCounterOffset = 64;
constexpr size_t kAlign = 256;
constexpr int kMaxStage = 2;
// Host waits of the host optimizer's hooks (tl_optimizer) give up after this.
constexpr double kOptWaitSeconds = 600.0;
// Automatic depth: host-link stall the ring is sized to ride out by default
// (stalls of 25-55 ms were measured on a shared GB300 machine's host link).
constexpr double kDefaultStallAllowanceMs = 50.0;

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct Shape {
    int64_t K = 0, M = 0, Mi = 0;
    int32_t N = 0;
};

inline size_t tile_bytes(int64_t K, int64_t Mi) { return size_t(K) * size_t(Mi) * 2; }

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

// One operator over host buffers in `layout`.
inline Op one_op(int64_t K, int64_t M, int32_t N, const void* w_host, void* dw_host, tl_layout layout) {
    Op o;
    o.s = Shape{K, M, N > 0 ? M / N : 0, N};
    o.w_host = static_cast<const uint8_t*>(w_host);
    o.dw_host = static_cast<uint8_t*>(dw_host);
    o.layout = layout;
    return o;
}

// Shape rules shared by workspace sizing and create.  Empty string = valid.
std::string check_shape(int64_t K, int64_t M, int32_t N, int32_t d);
// Workspace of a handle over `ops` at depth d (auto: d < 0): the header, then
// the ring's slots and min(2, tiles) staging slots, each sized for the
// largest tile.
size_t workspace_for(const std::vector<Shape>& ops, int32_t d);

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
    int32_t nk = 0;        // kernel spans recorded (one per tile)
    int32_t depth = 0, launches = 0, reused = 0;
    bool timed = true;     // per-launch and per-copy events recorded (see tiled_linear_set_timing)
    int64_t h2d_bytes = 0, d2h_bytes = 0;
    float total = 0, gemm1 = 0, gemm2 = 0, h2d = 0, d2h = 0;
    float h2d_max = 0;     // slowest single tile copy host->device
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

}  // namespace tl

struct tl_handle {
    int device = 0;
    tl::Shape s;                 // operator 0
    std::vector<tl::Op> ops;     // the operators, in forward order
    bool single_api = true;      // created by tiled_linear_create[_tilemajor|_file] (else a chain)
    int32_t n_total = 0;         // tiles over all operators
    tl_layout layout = TL_LAYOUT_ROW_MAJOR;
    int32_t d_req = 0, d = 0, slot_cap = 0, nstage = 0;
    bool auto_pending = false;
    double stall_allowance_ms = 0;  // auto depth: host-link stall the ring is sized to ride out
    const uint8_t* w_host = nullptr;
    uint8_t* dw_host = nullptr;
    uint8_t* ws = nullptr;
    size_t ws_bytes = 0;
    int32_t* err_dev = nullptr;
    int32_t* err_mirror = nullptr;  // pinned host copy of *err_dev, refreshed per call
    std::vector<uint8_t*> slot, stage;
    cudaStream_t h2d = nullptr, d2h = nullptr;
    std::vector<cudaEvent_t> ev_ready, ev_free, ev_dwdone, ev_drained;
    uint64_t stage_seq = 0;
    // The ring slots in the order their last readers were enqueued (a fetch
    // takes the front: the slot freed earliest), the tile each slot holds
    // (-1: none), and whether a backward takes the tiles it starts with from
    // the ring when they are still there.
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
    tl::FileTier* tier = nullptr;  // W and dW in files (tiled_linear_create_file), else in host memory
    uint32_t* tile_counter = nullptr;  // dynamic tile schedule of the GEMMs (header word)
    tl::Phase fwd, bwd;
    tl_status sticky = TL_OK;
    std::string msg;
};

namespace tl {

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

// Record `what` on the handle; CUDA, timeout and I/O failures make it sticky.
inline tl_status fail(tl_handle* h, tl_status st, const std::string& what) {
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
            return ::tl::fail((h), TL_ERR_CUDA, std::string(#call) + ": " + cudaGetErrorString(e_)); \
    } while (0)

bool is_pinned_host(const void* p);
bool is_device_mem(const void* p, int device);

// ---- tl_stats.cpp ----
tl_status create_phase(tl_handle* h, Phase& p, int n, bool backward);
void destroy_phase(Phase& p);
float span_ms(cudaEvent_t a, cudaEvent_t b);
tl_status harvest(tl_handle* h, Phase& p, CallSlot& c, int n);
tl_status harvest_all(tl_handle* h, Phase& p);
CallSlot* begin_call(tl_handle* h, Phase& p, tl_status* st);
void end_call(Phase& p, CallSlot& c);

// ---- tl_ring.cpp ----
tl_status poll_error(tl_handle* h);
tl_status check_usable(tl_handle* h);
// W and dW in files instead of host memory (tiled_linear_create_file).
struct FileArgs {
    const char* w_path = nullptr;
    const char* dw_path = nullptr;
    int32_t host_slots = 0, io_threads = 0;
};
// Create a handle over `ops` (one operator, or a chain) sharing one ring.
tl_status create_ops(tl_handle** out, std::vector<Op> ops, int32_t d, void* ws, size_t ws_bytes, int device,
                     bool single_api, const FileArgs* file = nullptr);
tl_status finish_auto_depth(tl_handle* h);
tl_status forward_tiles(tl_handle* h, int64_t T, const void* x, void* const* ys, cudaStream_t cs);
tl_status backward_tiles(tl_handle* h, int64_t T, const void* x, const void* const* ys, const void* dy,
                         float* dx, float* scr_dx, void* const* scr_dy, cudaStream_t cs);

// ---- tl_hooks.cpp ----
// Detach and delete the handle's host optimizer (waits for its jobs).
void detach_optimizer(tl_handle* h);

}  // namespace tl
