// rmsnorm.h -- launcher of the normalisation before the block (rmsnorm.cu).
#pragma once

#include <cstdint>

#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace zffn {

// x[t][c] = bf16(h[t][c] * rsqrt(mean_c' h[t][c']^2 + eps) * gamma[c]) for
// h fp32 [T][H], gamma fp32 [H], x bf16 [T][H]; H % 4 == 0 and 16-byte
// aligned pointers (checked by the caller).
cudaError_t launch_rmsnorm_bf16(const float *h, const float *gamma, float eps, __nv_bfloat16 *x, int T,
                                int H, cudaStream_t s);

}  // namespace zffn
