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

#include <cuda_runtime.h>

#include <mutex>
#include <string>

namespace {

constexpr size_t kStaticScratchBytes = size_t(32) << 20;  // 32 MiB per GPU
constexpr size_t kStatusBytes = 256;                      // timeout word, padded
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_tl_static_scratch[kStaticScratchBytes];

std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};
int g_num_sms[kMaxDevices] = {};

// Device address of the static array on `dev` (current device), looked up
// once per device.  In host code the array's name is only a host-side stand-in
// for the symbol, never a device address.
cudaError_t scratch_for_device(int dev, void** addr, int* sms) {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_tl_static_scratch);
        if (e != cudaSuccess) return e;
        int n = 0;
        e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        g_scratch_addr[dev] = p;
        g_num_sms[dev] = n;
    }
    *addr = g_scratch_addr[dev];
    *sms = g_num_sms[dev];
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

// Errors are reported by status code only (the reason is in the comment at
// each return); the entry point keeps no other state.
tl_status reject(tl_status st, const char* /*why*/) { return st; }

}  // namespace

extern "C" tl_status tiled_linear_forward_static(int64_t T, int64_t K, int64_t M, int32_t N,
                                                 const void* w_host, const void* x_dev, void* y_dev,
                                                 int32_t* status_host, void* stream) {
    if (K < 8 || K % 8 || M < 1 || N < 1 || M % N || (M / N) % 8)
        return reject(TL_ERR_INVALID, "need K % 8 == 0, M % N == 0, (M/N) % 8 == 0");
    if (T < 0 || T > (int64_t(1) << 30)) return reject(TL_ERR_INVALID, "T out of range");
    const int64_t Mi = M / N;
    const size_t tile = size_t(K) * size_t(Mi) * 2;
    if (kStatusBytes + tile > kStaticScratchBytes)
        return reject(TL_ERR_WORKSPACE, "one weight tile does not fit the static slot");
    if (T == 0) return TL_OK;
    if (!w_host || !x_dev || !y_dev) return reject(TL_ERR_INVALID, "null pointer");
    if ((reinterpret_cast<uintptr_t>(x_dev) | reinterpret_cast<uintptr_t>(y_dev)) & 15u)
        return reject(TL_ERR_INVALID, "x and y must be 16-byte aligned");
    if (!pinned(w_host) || (status_host && !pinned(status_host)))
        return reject(TL_ERR_NOT_PINNED, "w_host and status_host must be pinned host memory");

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return reject(TL_ERR_CUDA, "no current device");
    void* scratch = nullptr;
    int sms = 0;
    cudaError_t e = scratch_for_device(dev, &scratch, &sms);
    if (e != cudaSuccess)
        return reject(TL_ERR_CUDA, "static scratch lookup failed");

    auto* base = static_cast<unsigned char*>(scratch);
    int32_t* err = reinterpret_cast<int32_t*>(base);
    unsigned char* slot = base + kStatusBytes;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);

    // The array keeps the previous call's contents: the timeout word must
    // start at zero for this call.
    if ((e = cudaMemsetAsync(err, 0, 2 * sizeof(int32_t), cs)) != cudaSuccess)
        return reject(TL_ERR_CUDA, "clearing the timeout word failed");
    const auto* w = static_cast<const unsigned char*>(w_host);
    for (int32_t i = 0; i < N; ++i) {
        if ((e = cudaMemcpyAsync(slot, w + size_t(i) * tile, tile, cudaMemcpyHostToDevice, cs)) != cudaSuccess)
            return reject(TL_ERR_CUDA, "tile copy failed");
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
        if (tl::gemm_launch(g, sms, cs, &why) != cudaSuccess)
            return reject(TL_ERR_CUDA, "kernel launch failed");
    }
    if (status_host &&
        (e = cudaMemcpyAsync(status_host, err, sizeof(int32_t), cudaMemcpyDeviceToHost, cs)) != cudaSuccess)
        return reject(TL_ERR_CUDA, "status copy failed");
    return TL_OK;
}
