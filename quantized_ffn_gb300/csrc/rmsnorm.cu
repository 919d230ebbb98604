// rmsnorm.cu -- the normalisation in front of the block: the residual stream
// h (fp32) becomes the block's bf16 input x = RMSNorm(h) * gamma, and the
// block's output is then added back into h (the residual entry points).  "Four
// bottlenecks, one CUDA backend...", section "Bottleneck 3 -- Gemma decode is
// launch-latency bound": the rms_norm and the residual accumulate around a
// block are folded into as few launches as possible.  The pages do not write
// RMSNorm out; the form used is x = h / sqrt(mean(h^2) + eps) * gamma.
//
// One block of 256 threads per row: float4 loads of the row, the sum of
// squares reduced in fp32 (warp shuffles, then one value per warp in shared
// memory), and a second pass over the row (from L1) that scales, multiplies by
// gamma and stores four bf16 at a time.  HBM-bound: 6 bytes per element.
#include "rmsnorm.h"

namespace zffn {

constexpr int kNormThreads = 256;

__global__ void __launch_bounds__(kNormThreads)
    rmsnorm_bf16_kernel(const float *__restrict__ h, const float *__restrict__ gamma, float eps,
                        __nv_bfloat16 *__restrict__ x, int H) {
    __shared__ float part[kNormThreads / 32];
    const int t = blockIdx.x;
    const float4 *row = reinterpret_cast<const float4 *>(h + (int64_t)t * H);
    const int n4 = H / 4;
    float ss = 0.0f;
    // (unrolled so that a thread's loads of the row are in flight together)
#pragma unroll 4
    for (int i = threadIdx.x; i < n4; i += kNormThreads) {
        const float4 v = __ldg(row + i);
        ss = fmaf(v.x, v.x, ss);
        ss = fmaf(v.y, v.y, ss);
        ss = fmaf(v.z, v.z, ss);
        ss = fmaf(v.w, v.w, ss);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = ss;
    __syncthreads();
    float tot = 0.0f;
#pragma unroll
    for (int w = 0; w < kNormThreads / 32; ++w) tot += part[w];
    const float r = rsqrtf(tot / (float)H + eps);
    const float4 *g4 = reinterpret_cast<const float4 *>(gamma);
    uint2 *out = reinterpret_cast<uint2 *>(x + (int64_t)t * H);
#pragma unroll 4
    for (int i = threadIdx.x; i < n4; i += kNormThreads) {
        const float4 v = __ldg(row + i);
        const float4 g = __ldg(g4 + i);
        const __nv_bfloat162 lo = __floats2bfloat162_rn(v.x * r * g.x, v.y * r * g.y);
        const __nv_bfloat162 hi = __floats2bfloat162_rn(v.z * r * g.z, v.w * r * g.w);
        uint2 pk;
        pk.x = *reinterpret_cast<const uint32_t *>(&lo);
        pk.y = *reinterpret_cast<const uint32_t *>(&hi);
        out[i] = pk;
    }
}

cudaError_t launch_rmsnorm_bf16(const float *h, const float *gamma, float eps, __nv_bfloat16 *x, int T,
                                int H, cudaStream_t s) {
    if (T < 1 || H < 4 || H % 4 != 0) return cudaErrorInvalidValue;
    rmsnorm_bf16_kernel<<<T, kNormThreads, 0, s>>>(h, gamma, eps, x, H);
    return cudaGetLastError();
}

}  // namespace zffn
