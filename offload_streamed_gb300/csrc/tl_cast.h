// tl_cast.h -- internal: fp32 -> bf16 conversion between chained operators.
#pragma once
#include <cstdint>
#include <string>
#include <cuda_runtime.h>

namespace tl {

// dst[k] = bf16 round-to-nearest-even of src[k], k < n.  n % 8 == 0; both
// pointers 16-byte aligned.  Enqueued on `stream`.
cudaError_t cast_f32_bf16(const float* src, void* dst, int64_t n, int num_sms, cudaStream_t stream,
                          std::string* why);

}  // namespace tl
