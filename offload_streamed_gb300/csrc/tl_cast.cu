// tl_cast.cu -- fp32 -> bf16 (round to nearest even) over a contiguous array.
//
// In a chain of tiled linear operators the backward of operator l produces
// dX_l in fp32; operator l-1 takes it as its dY in bf16.  The conversion is a
// pure streaming pass (4 bytes read, 2 written per element): each thread
// moves 8 elements per step with 16-byte loads and one 16-byte store, and a
// grid of a few CTAs per SM strides over the array.
#include "tl_cast.h"

#include <cuda_bf16.h>

namespace tl {
namespace {

__global__ void __launch_bounds__(256) cast_kernel(const float4* __restrict__ src, uint4* __restrict__ dst,
                                                   int64_t n8) {
    const int64_t stride = int64_t(gridDim.x) * blockDim.x;
    for (int64_t k = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; k < n8; k += stride) {
        const float4 a = __ldcs(src + 2 * k);
        const float4 b = __ldcs(src + 2 * k + 1);
        __nv_bfloat162 p0 = __floats2bfloat162_rn(a.x, a.y);
        __nv_bfloat162 p1 = __floats2bfloat162_rn(a.z, a.w);
        __nv_bfloat162 p2 = __floats2bfloat162_rn(b.x, b.y);
        __nv_bfloat162 p3 = __floats2bfloat162_rn(b.z, b.w);
        uint4 o;
        o.x = *reinterpret_cast<uint32_t*>(&p0);
        o.y = *reinterpret_cast<uint32_t*>(&p1);
        o.z = *reinterpret_cast<uint32_t*>(&p2);
        o.w = *reinterpret_cast<uint32_t*>(&p3);
        dst[k] = o;
    }
}

}  // namespace

cudaError_t cast_f32_bf16(const float* src, void* dst, int64_t n, int num_sms, cudaStream_t stream,
                          std::string* why) {
    if (n % 8 || (reinterpret_cast<uintptr_t>(src) & 15u) || (reinterpret_cast<uintptr_t>(dst) & 15u)) {
        if (why) *why = "cast: n must be a multiple of 8 and both pointers 16-byte aligned";
        return cudaErrorInvalidValue;
    }
    if (n == 0) return cudaSuccess;
    const int64_t n8 = n / 8;
    const int64_t want = (n8 + 255) / 256;
    const int grid = int(want < int64_t(num_sms) * 4 ? want : int64_t(num_sms) * 4);
    cast_kernel<<<grid, 256, 0, stream>>>(reinterpret_cast<const float4*>(src), reinterpret_cast<uint4*>(dst), n8);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess && why) *why = cudaGetErrorString(e);
    return e;
}

}  // namespace tl
