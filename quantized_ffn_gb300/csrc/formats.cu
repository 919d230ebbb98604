// formats.cu -- other block formats of W_down on the single-token paths.
//
// The routed layers of the pages keep their gate/up experts in Q4_K and
// their down experts in Q5_K or Q5_1 ("Four bottlenecks, one CUDA
// backend...", section "Bottleneck 2": one batched launch reads the chosen
// ids and runs the down matvec of every chosen expert in Q5_K or Q5_1; section
// "Bottleneck 4": Q5_K and Q6_K matrices next to Q4_K).  The pages name the
// formats but do not lay them out; the reading is the GGUF arrangement:
//   Q5_K  176 B / 256 weights: d, dmin (fp16), 12 scale bytes packed as Q4_K,
//         qh[32], qs[128]; code = Q4_K nibble + 16 * bit (k/32) of qh[k%32];
//         w = d*sc*q - dmin*m.
//   Q6_K  210 B / 256 weights: ql[128], qh[64], int8 scales[16], d (fp16);
//         weight k of half n (r = k%128, i = r/32, l = r%32): low 4 bits
//         from ql[64n + l + 32(i&1)] (low nibble for i < 2, else high), high
//         2 bits = bits 2i..2i+1 of qh[32n + l]; w = d * scales[k/16] * (q-32).
//   Q5_1  24 B / 32 weights: d, m (fp16), qh (32 bits), qs[16]; code j =
//         nibble j of qs (low for j < 16, high for j >= 16) + 16 * bit j of
//         qh; w = d*q + m.
// Every product is exact in fp32, so the dequantised values are bit-exact
// whatever the evaluation order (and whether or not a multiply and an add are
// fused): the exact product, then at most one rounding of the sum.
//
// Kernels:
//   dequant_fmt_kernel<F>: one thread per weight, fp32 out (bit-exact).
//   down_fmt_kernel<F>: y[n] = sum_p w_p * Wd_{e_p}[n] . h[p] for one token,
//     launched as a programmatic dependent of the Q4_K gate/up kernel of the
//     single-token path, which leaves h (fp32 [P][I]) in the workspace.  One
//     warp per output row at a time: lane t dequantises weight t of each
//     32-weight group of the row (the group's header bytes are broadcast
//     loads, its codes one byte per lane) and multiplies it by h, staged in
//     shared memory; the row's sum is one warp reduction.  The rows of the
//     grid are interleaved so that all warps stream the matrix together.
#include "formats.h"

#include "zffn_internal.cuh"

namespace zffn {

__host__ __device__ inline int fmt_block_weights(int f) { return f == kFmtQ5_1 ? 32 : 256; }
__host__ __device__ inline int fmt_block_bytes(int f) {
    return f == kFmtQ4_K ? 144 : f == kFmtQ5_K ? 176 : f == kFmtQ6_K ? 210 : 24;
}
__host__ __device__ int64_t fmt_row_bytes_hd(int f, int64_t cols) {
    const int bw = fmt_block_weights(f);
    return (cols + bw - 1) / bw * fmt_block_bytes(f);
}
int64_t fmt_row_bytes(int f, int64_t cols) { return fmt_row_bytes_hd(f, cols); }
bool fmt_valid(int f) { return f >= kFmtQ4_K && f <= kFmtQ5_1; }

__device__ __forceinline__ float fp16_at(const uint8_t *p) {
    return half_bits_to_float((uint32_t)p[0] | ((uint32_t)p[1] << 8));
}

// Value of weight k of the block at blk.
template <int F>
__device__ __forceinline__ float fmt_weight(const uint8_t *__restrict__ blk, int k) {
    if (F == kFmtQ6_K) {
        const int n = k >> 7, r = k & 127, i = r >> 5, l = r & 31;
        const uint32_t lb = __ldg(blk + 64 * n + l + 32 * (i & 1));
        const int lo = (int)((i < 2 ? lb : lb >> 4) & 15u);
        const int hi = (int)((__ldg(blk + 128 + 32 * n + l) >> (2 * i)) & 3u);
        const int sc = (int)(int8_t)__ldg(blk + 192 + (k >> 4));
        return fp16_at(blk + 208) * (float)(sc * ((lo | (hi << 4)) - 32));   // exact
    } else if (F == kFmtQ5_1) {
        const uint32_t qs = __ldg(blk + 8 + (k & 15));
        const uint32_t qh = __ldg(blk + 4 + (k >> 3));
        const int q = (int)(((k < 16 ? qs : qs >> 4) & 15u) | (((qh >> (k & 7)) & 1u) << 4));
        return fmaf(fp16_at(blk), (float)q, fp16_at(blk + 2));               // d*q exact
    } else {
        // Q4_K and Q5_K share the scale packing and the nibble arrangement
        const int j = k >> 5;
        const uint8_t *sb = blk + 4;
        int sc, m;
        if (j < 4) {
            sc = __ldg(sb + j) & 63;
            m = __ldg(sb + j + 4) & 63;
        } else {
            sc = (__ldg(sb + j + 4) & 15) | ((__ldg(sb + j - 4) >> 6) << 4);
            m = (__ldg(sb + j + 4) >> 4) | ((__ldg(sb + j) >> 6) << 4);
        }
        const uint8_t *qs = blk + (F == kFmtQ5_K ? 48 : 16);
        const uint32_t b = __ldg(qs + 32 * (k >> 6) + (k & 31));
        int q = (int)(((k & 32) ? b >> 4 : b) & 15u);
        if (F == kFmtQ5_K) q |= (int)((__ldg(blk + 16 + (k & 31)) >> j) & 1u) << 4;
        const float wq = (fp16_at(blk) * (float)sc) * (float)q;             // exact
        return wq - fp16_at(blk + 2) * (float)m;                             // one rounding
    }
}

template <int F>
__global__ void dequant_fmt_kernel(const uint8_t *__restrict__ blocks, float *__restrict__ out, int64_t rows,
                                   int64_t cols) {
    const int64_t rb = fmt_row_bytes_hd(F, cols);
    const int bw = fmt_block_weights(F), bb = fmt_block_bytes(F);
    const int64_t n = rows * cols;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = i / cols, c = i - r * cols;
        const uint8_t *blk = blocks + r * rb + (c / bw) * bb;
        out[i] = fmt_weight<F>(blk, (int)(c % bw));
    }
}

cudaError_t launch_dequant_fmt(int f, const void *blocks, float *out, int64_t rows, int64_t cols,
                               cudaStream_t s) {
    const int64_t n = rows * cols;
    const int threads = 256;
    const int64_t want = (n + threads - 1) / threads;
    const int blocks_n = (int)(want < 152 * 32 ? want : 152 * 32);
    const uint8_t *b = static_cast<const uint8_t *>(blocks);
    switch (f) {
    case kFmtQ4_K: dequant_fmt_kernel<kFmtQ4_K><<<blocks_n, threads, 0, s>>>(b, out, rows, cols); break;
    case kFmtQ5_K: dequant_fmt_kernel<kFmtQ5_K><<<blocks_n, threads, 0, s>>>(b, out, rows, cols); break;
    case kFmtQ6_K: dequant_fmt_kernel<kFmtQ6_K><<<blocks_n, threads, 0, s>>>(b, out, rows, cols); break;
    case kFmtQ5_1: dequant_fmt_kernel<kFmtQ5_1><<<blocks_n, threads, 0, s>>>(b, out, rows, cols); break;
    default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

constexpr int kDownWarps = 16;

// Shared memory: h of every expert slot, fp32 [P][I].
template <int F>
__global__ void __launch_bounds__(kDownWarps * 32) down_fmt_kernel(MatvecArgs a) {
    extern __shared__ __align__(16) float hs[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int H = a.H, I = a.I, P = a.k;
    const bool moe = a.ids != nullptr;
    // the next work in the stream may be scheduled as this grid's blocks leave
    if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    // h is written by the gate/up kernel: wait until that grid has completed
    asm volatile("griddepcontrol.wait;" ::: "memory");
    for (int i = threadIdx.x; i < P * I; i += blockDim.x) hs[i] = __ldcg(a.h + i);
    __syncthreads();
    const int64_t rb = fmt_row_bytes_hd(F, I);
    const int bw = fmt_block_weights(F), bb = fmt_block_bytes(F);
    const int groups = I / 32;
    const int64_t gw = (int64_t)gridDim.x * kDownWarps;
    for (int64_t n = (int64_t)warp * gridDim.x + blockIdx.x; n < H; n += gw) {
        float acc = 0.0f;
        for (int p = 0; p < P; ++p) {
            const int e = moe ? a.ids[p] : 0;
            if (e < 0 || e >= a.E) continue;
            const float wp = moe ? a.wts[p] : 1.0f;
            const uint8_t *row = a.Wd + ((int64_t)e * H + n) * rb;
            const float *hp = hs + (size_t)p * I;
            float part = 0.0f;
#pragma unroll 4
            for (int g = 0; g < groups; ++g) {
                const int c = g * 32 + lane;
                const float w = fmt_weight<F>(row + (c / bw) * bb, c % bw);
                part = fmaf(w, hp[c], part);
            }
            acc = fmaf(wp, part, acc);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
        if (lane == 0) a.y[n] = a.accumulate ? a.y[n] + acc : acc;
    }
}

size_t down_fmt_smem_bytes(int I, int k) { return (size_t)k * I * sizeof(float); }

cudaError_t launch_token_fmt(const MatvecArgs &a, int wd_fmt, cudaStream_t s) {
    if (a.T != 1 || !fmt_valid(wd_fmt) || wd_fmt == kFmtQ4_K || a.I % 64 != 0) return cudaErrorInvalidValue;
    const DeviceInfo &di = device_info();
    const size_t smem_a = gu_smem_total(a.H, a.I, a.k), smem_b = down_fmt_smem_bytes(a.I, a.k);
    if (smem_a > (size_t)di.max_smem_optin || smem_b > (size_t)di.max_smem_optin) return cudaErrorInvalidValue;
    const void *down = wd_fmt == kFmtQ5_K ? (const void *)down_fmt_kernel<kFmtQ5_K>
                     : wd_fmt == kFmtQ6_K ? (const void *)down_fmt_kernel<kFmtQ6_K>
                                          : (const void *)down_fmt_kernel<kFmtQ5_1>;
    cudaError_t e = cudaFuncSetAttribute(ffn_gu_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_a);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(down, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_b);
    if (e != cudaSuccess) return e;
    // the gate/up kernel's block size is its launch bound
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, ffn_gu_kernel);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(di.num_sms);
    cfg.blockDim = dim3(fa.maxThreadsPerBlock);
    cfg.stream = s;
    cfg.dynamicSmemBytes = smem_a;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    MatvecArgs args = a;
    e = cudaLaunchKernelEx(&cfg, ffn_gu_kernel, args);
    if (e != cudaSuccess) return e;
    cfg.blockDim = dim3(kDownWarps * 32);
    cfg.dynamicSmemBytes = smem_b;
    void *kargs[] = {&args};
    return cudaLaunchKernelExC(&cfg, down, kargs);
}

}  // namespace zffn
