// tl_static.cu -- a streamed forward that allocates nothing.
//
// Some callers cannot allocate device memory at all: a plug-in running inside
// a host framework whose allocator owns every byte of the GPU, or a service
// that forbids allocation once it has started.  They still want to run the
// streamed forward.  tiled_linear_forward_static serves them: its scratch (one
// weight-tile slot and the kernels' timeout word) lives in the file-scope
// array below, which every GPU that loads this library holds until the process
// exits.  The caller passes only inputs, outputs and a stream.
//
// The entry point runs the same forward kernel, tile after tile in the same
// order, as tiled_linear_forward, so Y is identical.  Everything is ordered on
// the caller's stream (copy of tile i, then its GEMM, then the next copy):
// without a second stream there is no copy/compute overlap.
#include "tiled_linear.h"
#include "tl_gemm.h"
#include "tl_unbound_error.h"

#include <cuda.h>
#include <cuda_runtime.h>

#include <climits>
#include <mutex>
#include <string>

namespace {

constexpr size_t kStaticScratchBytes = size_t(32) << 20;  // 32 MiB per GPU
constexpr size_t kStatusBytes = 256;                      // timeout word, padded
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_tl_static_scratch[kStaticScratchBytes];

// Driver calls that name the current context (through the runtime's entry
// point query, as the rest of the library reaches driver calls).
using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);
struct CtxFns {
    CtxGetCurrentFn current = nullptr;
    CtxGetIdFn id = nullptr;
};
const CtxFns& ctx_fns() {
    static CtxFns f;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            f.current = reinterpret_cast<CtxGetCurrentFn>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            f.id = reinterpret_cast<CtxGetIdFn>(p);
    });
    return f;
}

// Id of the current thread's context (0 if it cannot be read: the address is
// then looked up on every call).
unsigned long long current_ctx_id() {
    const CtxFns& f = ctx_fns();
    CUcontext c = nullptr;
    unsigned long long id = 0;
    if (!f.current || !f.id || f.current(&c) != CUDA_SUCCESS || !c || f.id(c, &id) != CUDA_SUCCESS) return 0;
    return id;
}

struct DeviceScratch {
    unsigned long long ctx = 0;  // context the address belongs to
    void* addr = nullptr;
    int sms = 0;
};
std::mutex g_mu;
DeviceScratch g_dev[kMaxDevices];

// Device address of the static array in the current context of device `dev`
// (the current device).  In host code the array's name is only a host-side
// stand-in for the symbol, never a device address.  The address is kept per
// device and context: a context destroyed and created again (cudaDeviceReset)
// loads the module anew, possibly at another address, and is looked up again.
cudaError_t scratch_for_device(int dev, void** addr, int* sms) {
    const unsigned long long ctx = current_ctx_id();
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceScratch& d = g_dev[dev];
    if (!d.addr || ctx == 0 || d.ctx != ctx) {
        void* p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_tl_static_scratch);
        if (e != cudaSuccess) return e;
        int n = 0;
        e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        d.addr = p;
        d.sms = n;
        d.ctx = ctx;
    }
    *addr = d.addr;
    *sms = d.sms;
    return cudaSuccess;
}

bool pinned(const void* p) {
    cudaPointerAttributes a{};
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return a.type == cudaMemoryTypeHost;
}

// The reason of a refused or failed call, kept for tiled_linear_last_error(NULL).
tl_status reject(tl_status st, const std::string& why) {
    tl::set_unbound_error("tiled_linear_forward_static: " + why);
    return st;
}

}  // namespace

extern "C" tl_status tiled_linear_forward_static(int64_t T, int64_t K, int64_t M, int32_t N,
                                                 const void* w_host, const void* x_dev, void* y_dev,
                                                 int32_t* status_host, void* stream) {
    constexpr int64_t kMaxDim = INT32_MAX / 2;  // the GEMM's index range
    if (K < 8 || K % 8 || M < 1 || N < 1 || M % N || (M / N) % 8)
        return reject(TL_ERR_INVALID, "need K % 8 == 0, K >= 8, N >= 1, M % N == 0 and (M/N) % 8 == 0");
    if (T < 0 || T > kMaxDim || K > kMaxDim || M / N > kMaxDim)
        return reject(TL_ERR_INVALID, "T, K and M/N must each be at most 2^30 - 1");
    const int64_t Mi = M / N;
    // one tile, K * Mi * 2 bytes, beside the status word (no overflow: K and
    // Mi are below 2^30 here)
    if (K > int64_t((kStaticScratchBytes - kStatusBytes) / 2) / Mi)
        return reject(TL_ERR_WORKSPACE, "one weight tile (K * (M/N) * 2 bytes) exceeds the static slot of " +
                                            std::to_string(kStaticScratchBytes - kStatusBytes) + " bytes");
    const size_t tile = size_t(K) * size_t(Mi) * 2;
    if (!status_host) return reject(TL_ERR_INVALID, "status_host is required (a kernel timeout is reported there)");
    if (T > 0 && (!w_host || !x_dev || !y_dev)) return reject(TL_ERR_INVALID, "null pointer");
    if ((reinterpret_cast<uintptr_t>(x_dev) | reinterpret_cast<uintptr_t>(y_dev)) & 15u)
        return reject(TL_ERR_INVALID, "x and y must be 16-byte aligned");
    if (!pinned(status_host) || (T > 0 && !pinned(w_host)))
        return reject(TL_ERR_NOT_PINNED, "w_host and status_host must be pinned host memory");

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return reject(TL_ERR_CUDA, "no current device");
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    int sdev = -1;
    cudaError_t e = cudaStreamGetDevice(cs, &sdev);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return reject(TL_ERR_INVALID, std::string("stream: ") + cudaGetErrorString(e));
    }
    if (sdev != dev)
        return reject(TL_ERR_INVALID, "the stream belongs to device " + std::to_string(sdev) +
                                          ", not to the current device " + std::to_string(dev));
    void* scratch = nullptr;
    int sms = 0;
    if ((e = scratch_for_device(dev, &scratch, &sms)) != cudaSuccess)
        return reject(TL_ERR_CUDA, std::string("static scratch lookup: ") + cudaGetErrorString(e));

    auto* base = static_cast<unsigned char*>(scratch);
    int32_t* err = reinterpret_cast<int32_t*>(base);
    unsigned char* slot = base + kStatusBytes;

    // The array keeps the previous call's contents: the timeout word and the
    // tile counter must start at zero for this call.
    if ((e = cudaMemsetAsync(err, 0, 2 * sizeof(int32_t), cs)) != cudaSuccess)
        return reject(TL_ERR_CUDA, std::string("clearing the timeout word: ") + cudaGetErrorString(e));
    const auto* w = static_cast<const unsigned char*>(w_host);
    for (int32_t i = 0; T > 0 && i < N; ++i) {
        if ((e = cudaMemcpyAsync(slot, w + size_t(i) * tile, tile, cudaMemcpyHostToDevice, cs)) != cudaSuccess)
            return reject(TL_ERR_CUDA, std::string("tile copy: ") + cudaGetErrorString(e));
        tl::GemmDesc g;
        g.m_dim = T;
        g.n_dim = Mi;
        g.k_dim = K;
        g.a = x_dev;
        g.lda = K;
        g.a_mn_major = false;
        g.b = slot;
        g.ldb = Mi;
        g.b_mn_major = true;
        g.d = static_cast<unsigned char*>(y_dev) + size_t(i) * size_t(Mi) * 2;
        g.ldd = M;
        g.out = tl::OutKind::BF16;
        g.err = err;
        g.tile_counter = reinterpret_cast<uint32_t*>(err + 1);
        std::string why;
        if (tl::gemm_launch(g, sms, cs, &why) != cudaSuccess) return reject(TL_ERR_CUDA, "kernel launch: " + why);
    }
    if ((e = cudaMemcpyAsync(status_host, err, sizeof(int32_t), cudaMemcpyDeviceToHost, cs)) != cudaSuccess)
        return reject(TL_ERR_CUDA, std::string("status copy: ") + cudaGetErrorString(e));
    return TL_OK;
}
