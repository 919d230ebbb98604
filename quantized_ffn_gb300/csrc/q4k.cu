// q4k.cu -- standalone Q4_K kernels: unpack to fp32 (bit-exact), the min/max
// quantiser, and the conversion of x to fp16 (with the zero fill of y that the
// tensor-core kernel's reductions add into).
#include "zffn_internal.cuh"

namespace zffn {

// ---------------------------------------------------------------------------
// Unpack.  One warp per 144-byte block; lane l owns code bytes 4l..4l+3 of the
// block, i.e. group g = l/8, positions p = 4(l%8)..+3: weights 64g+p.. (low
// nibbles, sub-block 2g) and 64g+32+p.. (high nibbles, sub-block 2g+1).
// d*sc and dmin*m are exact in fp32 and so is d*sc*q, so the single fused
// multiply-add rounds exactly once: the correctly rounded value.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) q4k_dequant_kernel(const uint8_t *__restrict__ blocks,
                                                          float *__restrict__ out, int64_t rows,
                                                          int64_t cols) {
    const int64_t nb = (cols + kQK - 1) / kQK;
    const int64_t total = rows * nb;
    const int lane = threadIdx.x & 31;
    const int64_t warp = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const int g = lane >> 3;
    const int p = 4 * (lane & 7);
    for (int64_t blk = warp; blk < total; blk += nwarps) {
        const int64_t r = blk / nb, b = blk % nb;
        const uint8_t *src = blocks + blk * kBlockBytes;
        // header and code bytes (byte loads: the buffer may have any alignment)
        uint32_t hd = src[0] | (src[1] << 8), hm = src[2] | (src[3] << 8);
        uint32_t s[3];
#pragma unroll
        for (int i = 0; i < 3; ++i)
            s[i] = src[4 + 4 * i] | (src[5 + 4 * i] << 8) | (src[6 + 4 * i] << 16) |
                   ((uint32_t)src[7 + 4 * i] << 24);
        const uint8_t *qs = src + 16 + 32 * g + p;
        const float d = half_bits_to_float(hd), dmin = half_bits_to_float(hm);
        int sc0, m0, sc1, m1;
        q4k_scale_min(s[0], s[1], s[2], 2 * g, sc0, m0);
        q4k_scale_min(s[0], s[1], s[2], 2 * g + 1, sc1, m1);
        const float ds0 = d * (float)sc0, dm0 = dmin * (float)m0;
        const float ds1 = d * (float)sc1, dm1 = dmin * (float)m1;
        float *o = out + r * cols + b * kQK;
        const int64_t lim = cols - b * kQK;   // valid columns in this block
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int q = qs[i];
            const int k0 = 64 * g + p + i, k1 = k0 + 32;
            if (k0 < lim) o[k0] = fmaf(ds0, (float)(q & 15), -dm0);
            if (k1 < lim) o[k1] = fmaf(ds1, (float)(q >> 4), -dm1);
        }
    }
}

cudaError_t launch_q4k_dequant(const void *blocks, float *out, int64_t rows, int64_t cols,
                               cudaStream_t s) {
    const int64_t nb = (cols + kQK - 1) / kQK;
    const int64_t warps = rows * nb;
    int64_t grid = (warps + 7) / 8;
    const int64_t cap = (int64_t)device_info().num_sms * 16;
    if (grid > cap) grid = cap;
    if (grid < 1) grid = 1;
    q4k_dequant_kernel<<<(unsigned)grid, 256, 0, s>>>(static_cast<const uint8_t *>(blocks), out,
                                                       rows, cols);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Min/max quantiser.  One warp per block; lane l owns weight 32j+l of every
// sub-block j, so sub-block minima and maxima are warp reductions (exact) and
// code byte 32g+l (low nibble: sub-block 2g, high: 2g+1) is lane-local.
// Every step uses IEEE round-to-nearest fp32 operations in the documented
// order, so the codes equal those of any other correct evaluation.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) q4k_quantize_kernel(const float *__restrict__ w,
                                                           uint8_t *__restrict__ blocks,
                                                           int64_t rows, int64_t cols) {
    const int64_t nb = (cols + kQK - 1) / kQK;
    const int64_t total = rows * nb;
    const int lane = threadIdx.x & 31;
    const int64_t warp = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t blk = warp; blk < total; blk += nwarps) {
        const int64_t r = blk / nb, b = blk % nb;
        const float *src = w + r * cols + b * kQK;
        const int64_t lim = cols - b * kQK;
        float v[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int k = 32 * j + lane;
            v[j] = k < lim ? src[k] : 0.0f;
        }
        float scale[8], mn[8];
        float max_scale = 0.0f, max_min = 0.0f;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            float lo = fminf(v[j], 0.0f), hi = v[j];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, o));
                hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, o));
            }
            scale[j] = __fdiv_rn(__fsub_rn(hi, lo), 15.0f);
            mn[j] = -lo;
            if (scale[j] > max_scale) max_scale = scale[j];
            if (mn[j] > max_min) max_min = mn[j];
        }
        const __half d16 = __float2half_rn(__fdiv_rn(max_scale, 63.0f));
        const __half dm16 = __float2half_rn(__fdiv_rn(max_min, 63.0f));
        const float d = __half2float(d16), dmin = __half2float(dm16);
        int sc[8], m[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float rs = d > 0.0f ? __fdiv_rn(scale[j], d) : 0.0f;
            const float rm = dmin > 0.0f ? __fdiv_rn(mn[j], dmin) : 0.0f;
            sc[j] = min(max(__float2int_rn(rs), 0), 63);
            m[j] = min(max(__float2int_rn(rm), 0), 63);
        }
        int q[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float ds = __fmul_rn(d, (float)sc[j]);
            const float dm = __fmul_rn(dmin, (float)m[j]);
            int c = 0;
            if (ds > 0.0f) c = min(max(__float2int_rn(__fdiv_rn(__fadd_rn(v[j], dm), ds)), 0), 15);
            q[j] = c;
        }
        uint8_t *dst = blocks + blk * kBlockBytes;
#pragma unroll
        for (int g = 0; g < 4; ++g) dst[16 + 32 * g + lane] = (uint8_t)(q[2 * g] | (q[2 * g + 1] << 4));
        if (lane < 12) {
            uint8_t byte;
            if (lane < 4)
                byte = (uint8_t)((sc[lane] & 63) | ((sc[lane + 4] >> 4) << 6));
            else if (lane < 8)
                byte = (uint8_t)((m[lane - 4] & 63) | ((m[lane] >> 4) << 6));
            else
                byte = (uint8_t)((sc[lane - 4] & 15) | ((m[lane - 4] & 15) << 4));
            dst[4 + lane] = byte;
        } else if (lane == 12) {
            const unsigned short db = __half_as_ushort(d16), mb = __half_as_ushort(dm16);
            dst[0] = (uint8_t)(db & 255);
            dst[1] = (uint8_t)(db >> 8);
            dst[2] = (uint8_t)(mb & 255);
            dst[3] = (uint8_t)(mb >> 8);
        }
    }
}

cudaError_t launch_q4k_quantize(const float *w, void *blocks, int64_t rows, int64_t cols,
                                cudaStream_t s) {
    const int64_t nb = (cols + kQK - 1) / kQK;
    int64_t grid = (rows * nb + 7) / 8;
    const int64_t cap = (int64_t)device_info().num_sms * 16;
    if (grid > cap) grid = cap;
    if (grid < 1) grid = 1;
    q4k_quantize_kernel<<<(unsigned)grid, 256, 0, s>>>(w, static_cast<uint8_t *>(blocks), rows,
                                                        cols);
    return cudaGetLastError();
}

// The tensor-core kernel's gate/up operand: x (bf16, n values, n % 8 == 0)
// as fp16; optionally y[0, ny) = 0 in the same pass (the reductions of the
// tensor-core kernel add into y).
__global__ void __launch_bounds__(256) x_to_f16_kernel(const uint4 *__restrict__ x, uint4 *__restrict__ x16,
                                                       int64_t n8, float4 *__restrict__ y, int64_t ny4,
                                                       float *ytail, int nytail) {
    // the block that consumes x16 and y may be scheduled now; it waits for
    // this grid's completion before it reads them
    if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n8; i += stride) {
        const uint4 v = x[i];
        x16[i] = make_uint4(bf16x2_to_f16x2_satfinite(v.x), bf16x2_to_f16x2_satfinite(v.y),
                            bf16x2_to_f16x2_satfinite(v.z), bf16x2_to_f16x2_satfinite(v.w));
    }
    if (y) {
        for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < ny4; i += stride)
            y[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (blockIdx.x == 0 && threadIdx.x < nytail) ytail[threadIdx.x] = 0.0f;
    }
}

cudaError_t launch_x_to_f16(const void *x, void *x16, int64_t n, float *y_zero, int64_t ny,
                            cudaStream_t s) {
    if (n % 8 != 0) return cudaErrorInvalidValue;
    const int64_t n8 = n / 8, ny4 = y_zero ? ny / 4 : 0;
    const int64_t work = n8 > ny4 ? n8 : ny4;
    int64_t grid = (work + 255) / 256;
    const int64_t cap = (int64_t)device_info().num_sms * 8;
    if (grid > cap) grid = cap;
    if (grid < 1) grid = 1;
    x_to_f16_kernel<<<(unsigned)grid, 256, 0, s>>>(
        static_cast<const uint4 *>(x), static_cast<uint4 *>(x16), n8, reinterpret_cast<float4 *>(y_zero), ny4,
        y_zero ? y_zero + 4 * ny4 : nullptr, y_zero ? (int)(ny - 4 * ny4) : 0);
    return cudaGetLastError();
}

}  // namespace zffn
