// tl_abi.cpp -- the C entry points of the engine: workspace sizing, handle
// creation (one operator or a chain), forward / backward calls, destroy, the
// switches of a handle, the resident GEMMs, the failure-path self-test and
// pinned host memory.  The schedules themselves are in tl_ring.cpp.
#include "tl_engine.h"
#include "tl_unbound_error.h"

#include <cmath>
#include <cstring>

namespace tl {
namespace {
thread_local std::string g_unbound_error;
}  // namespace
void set_unbound_error(const std::string& why) { g_unbound_error = why; }
const char* unbound_error() { return g_unbound_error.c_str(); }
}  // namespace tl

using namespace tl;

extern "C" {

size_t tiled_linear_workspace_bytes(int64_t K, int64_t M, int32_t N, int32_t d) {
    if (!check_shape(K, M, N, d).empty()) return 0;
    return workspace_for({Shape{K, M, M / N, N}}, d);
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
        tl::set_unbound_error(bad);
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
        if (h->h2d) cudaStreamDestroy(h->h2d);
        if (h->d2h) cudaStreamDestroy(h->d2h);
        if (h->err_mirror) cudaFreeHost(h->err_mirror);
        cudaGetLastError();
    }
    delete h;
    return st;
}

const char* tiled_linear_last_error(const tl_handle* h) {
    if (!h) return tl::unbound_error();
    return h->msg.c_str();
}

tl_status tiled_linear_set_tile_reuse(tl_handle* h, int32_t enable) {
    tl_status st = check_usable(h);
    if (st != TL_OK) return st;
    h->reuse = enable != 0;
    return TL_OK;
}

tl_status tiled_linear_set_stall_allowance(tl_handle* h, double ms) {
    tl_status st = check_usable(h);
    if (st != TL_OK) return st;
    if (!(ms >= 0.0) || !std::isfinite(ms)) return fail(h, TL_ERR_INVALID, "the stall allowance must be finite and >= 0");
    h->stall_allowance_ms = ms;
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
