// ffn_matvec.cu -- the memory-bound path for a single token (dense decode) and
// for a handful of (token, expert) pairs (MoE decode).
//
// One persistent launch (cooperative, one 512-thread block per SM) in two
// phases separated by a bounded grid barrier:
//   phase 1: for every pair p and intermediate row i, stream the W_gate and
//            W_up rows once, dot them with x (same input, one pass: "fuse the
//            same-input Q4_K matvec pairs", "Four bottlenecks, one CUDA
//            backend...", Bottleneck 3) and store h[p][i] = silu(g) * u
//            (fp32, a few tens of KB that stay in L2 and are consumed at once:
//            for one token the intermediate is small, "Fused SwiGLU MLP...",
//            FAQ "Does this affect decode?");
//   phase 2: stream the W_down rows: y[t][n] = sum_p w_p * Wd_{e_p}[n] . h[p].
// While phase 1 runs, every warp asks the L2 to prefetch the W_down rows it
// will read in phase 2, so the barrier and phase 2 overlap HBM traffic.
// Expert ids are read on the device ("Bottleneck 2"), never on the host.
//
// Lane layout for one 256-weight block: 8 lanes per block, 4 blocks per warp
// step.  Lane (b, s) owns code bytes 32g+16h .. +15 (g = s/2, h = s%2):
// weights 64g+16h+v (low nibbles, sub-block 2g) and 64g+32+16h+v (high
// nibbles, sub-block 2g+1), v = 0..15.  The dot product of a sub-block is
// d*sc*sum(q*x) - dmin*m*sum(x).  Vectors live in shared memory padded by 4
// floats every 64, which makes the lanes' 16-byte reads bank-conflict free.
#include "zffn_internal.cuh"

namespace zffn {

constexpr int kMvThreads = 512;
constexpr int kMvWarps = kMvThreads / 32;

__host__ __device__ inline int padded_len(int n) { return n + (n / 64) * 4; }
__device__ __forceinline__ int pad_index(int k) { return k + (k >> 6) * 4; }

// Partial dot product of one lane's 32 weights of a block with a padded vector.
struct BlockPart {
    float ds0, dm0, ds1, dm1;
};

__device__ __forceinline__ BlockPart decode_head(uint4 hd, int g) {
    BlockPart r;
    const float d = half_bits_to_float(hd.x), dmin = half_bits_to_float(hd.x >> 16);
    int sc, m;
    q4k_scale_min(hd.y, hd.z, hd.w, 2 * g, sc, m);
    r.ds0 = d * (float)sc;
    r.dm0 = dmin * (float)m;
    q4k_scale_min(hd.y, hd.z, hd.w, 2 * g + 1, sc, m);
    r.ds1 = d * (float)sc;
    r.dm1 = dmin * (float)m;
    return r;
}

// sums of q*x over the low and high nibbles of 16 code bytes
__device__ __forceinline__ void qx_sums(uint4 qs, const float *xlo, const float *xhi, float &slo,
                                        float &shi) {
    const uint32_t w[4] = {qs.x, qs.y, qs.z, qs.w};
    float a = 0.f, b = 0.f;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const float4 l4 = *reinterpret_cast<const float4 *>(xlo + 4 * u);
        const float4 h4 = *reinterpret_cast<const float4 *>(xhi + 4 * u);
        const uint32_t ww = w[u];
        a = fmaf((float)(ww & 15), l4.x, a);
        a = fmaf((float)((ww >> 8) & 15), l4.y, a);
        a = fmaf((float)((ww >> 16) & 15), l4.z, a);
        a = fmaf((float)((ww >> 24) & 15), l4.w, a);
        b = fmaf((float)((ww >> 4) & 15), h4.x, b);
        b = fmaf((float)((ww >> 12) & 15), h4.y, b);
        b = fmaf((float)((ww >> 20) & 15), h4.z, b);
        b = fmaf((float)((ww >> 28) & 15), h4.w, b);
    }
    slo = a;
    shi = b;
}

__device__ __forceinline__ void x_sums(const float *xlo, const float *xhi, float &slo, float &shi) {
    float a = 0.f, b = 0.f;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const float4 l4 = *reinterpret_cast<const float4 *>(xlo + 4 * u);
        const float4 h4 = *reinterpret_cast<const float4 *>(xhi + 4 * u);
        a += (l4.x + l4.y) + (l4.z + l4.w);
        b += (h4.x + h4.y) + (h4.z + h4.w);
    }
    slo = a;
    shi = b;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned *p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Bounded grid barrier over all blocks of this launch (co-resident by the
// cooperative launch).  bar[0] counts arrivals, bar[1] is the generation.
__device__ void grid_barrier(unsigned *bar, int *err) {
    __syncthreads();
    if (threadIdx.x == 0) {
        const unsigned gen = ld_acquire_u32(bar + 1);
        __threadfence();
        const unsigned arrived = atomicAdd(bar, 1u);
        if (arrived == gridDim.x - 1) {
            atomicExch(bar, 0u);
            __threadfence();
            atomicAdd(bar + 1, 1u);
        } else {
            const long long t0 = clock64();
            while (ld_acquire_u32(bar + 1) == gen) {
                if (clock64() - t0 > kWaitBudgetCycles) {
                    record_error(err, ZFFN_ERR_TIMEOUT);
                    break;
                }
                __nanosleep(32);
            }
        }
        __threadfence();
    }
    __syncthreads();
}

__global__ void __launch_bounds__(kMvThreads, 1) ffn_matvec_kernel(MatvecArgs a) {
    extern __shared__ __align__(16) float smem[];
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int gwarp = blockIdx.x * kMvWarps + warp;
    const int nwarps = gridDim.x * kMvWarps;
    const int H = a.H, I = a.I, k = a.k;
    const int P = a.T * k;                      // (token, slot) pairs
    const int nbH = H / kQK;
    const int nbI = (I + kQK - 1) / kQK;
    const int64_t rbH = (int64_t)nbH * kBlockBytes;
    const int64_t rbI = (int64_t)nbI * kBlockBytes;
    const int Hp = padded_len(H), Ip = padded_len(nbI * kQK);
    const int sub = lane & 7, g = sub >> 1, hh = sub & 1, bl = lane >> 3;
    const bool moe = a.ids != nullptr;

    auto expert_of = [&](int p) -> int { return moe ? a.ids[p] : 0; };

    // ---- L2 prefetch of this warp's phase-2 W_down rows --------------------
    if (lane == 0) {
        for (int task = gwarp; task < a.T * H; task += nwarps) {
            const int t = task / H, n = task % H;
            for (int j = 0; j < k; ++j) {
                const int e = expert_of(t * k + j);
                if (e < 0 || e >= a.E) continue;
                prefetch_l2_bulk(a.Wd + ((int64_t)e * H + n) * rbI, (uint32_t)rbI);
            }
        }
    }

    // ---- phase 1: h[p][i] = silu(Wg_e[i] . x_t) * (Wu_e[i] . x_t) ------------
    for (int idx = threadIdx.x; idx < a.T * Hp; idx += blockDim.x) {
        const int t = idx / Hp, kp = idx % Hp;
        // inverse of pad_index: position kp belongs to 68-float groups
        const int grp = kp / 68, off = kp % 68;
        float v = 0.f;
        if (off < 64) v = __bfloat162float(a.x[(int64_t)t * H + grp * 64 + off]);
        smem[idx] = v;
    }
    __syncthreads();

    for (int task = gwarp; task < P * I; task += nwarps) {
        const int p = task / I, i = task % I;
        const int e = expert_of(p);
        const int t = p / k;
        float gacc = 0.f, uacc = 0.f;
        if (e >= 0 && e < a.E) {
            const uint8_t *rg = a.Wg + ((int64_t)e * I + i) * rbH;
            const uint8_t *ru = a.Wu + ((int64_t)e * I + i) * rbH;
            const float *xs = smem + t * Hp;
#pragma unroll 4
            for (int b0 = 0; b0 < nbH; b0 += 4) {
                const int b = b0 + bl;
                if (b < nbH) {
                    const int64_t off = (int64_t)b * kBlockBytes;
                    const uint4 hg = __ldg(reinterpret_cast<const uint4 *>(rg + off));
                    const uint4 qg = __ldg(reinterpret_cast<const uint4 *>(rg + off + 16 + 32 * g + 16 * hh));
                    const uint4 hu = __ldg(reinterpret_cast<const uint4 *>(ru + off));
                    const uint4 qu = __ldg(reinterpret_cast<const uint4 *>(ru + off + 16 + 32 * g + 16 * hh));
                    const float *xlo = xs + pad_index(b * kQK + 64 * g + 16 * hh);
                    const float *xhi = xlo + 32;
                    float sxl, sxh;
                    x_sums(xlo, xhi, sxl, sxh);
                    float ql, qh;
                    const BlockPart pg = decode_head(hg, g);
                    qx_sums(qg, xlo, xhi, ql, qh);
                    gacc += pg.ds0 * ql - pg.dm0 * sxl + pg.ds1 * qh - pg.dm1 * sxh;
                    const BlockPart pu = decode_head(hu, g);
                    qx_sums(qu, xlo, xhi, ql, qh);
                    uacc += pu.ds0 * ql - pu.dm0 * sxl + pu.ds1 * qh - pu.dm1 * sxh;
                }
            }
        }
        gacc = warp_sum(gacc);
        uacc = warp_sum(uacc);
        if (lane == 0) {
            const float s = gacc / (1.0f + expf(-gacc));
            a.h[(int64_t)p * I + i] = s * uacc;
        }
    }

    grid_barrier(a.barrier, a.err);

    // ---- phase 2: y[t][n] = sum_j w_{t,j} * Wd_{e_{t,j}}[n] . h[t*k+j] ---------
    for (int idx = threadIdx.x; idx < P * Ip; idx += blockDim.x) {
        const int p = idx / Ip, kp = idx % Ip;
        const int grp = kp / 68, off = kp % 68;
        const int col = grp * 64 + off;
        float v = 0.f;
        if (off < 64 && col < I) v = __ldcg(a.h + (int64_t)p * I + col);
        smem[idx] = v;
    }
    __syncthreads();

    const int items = k * nbI;   // (slot, block) pairs per output row
    for (int task = gwarp; task < a.T * H; task += nwarps) {
        const int t = task / H, n = task % H;
        float acc = 0.f;
        for (int it0 = 0; it0 < items; it0 += 4) {
            const int it = it0 + bl;
            if (it < items) {
                const int j = it / nbI, b = it % nbI;
                const int p = t * k + j;
                const int e = expert_of(p);
                if (e >= 0 && e < a.E) {
                    const float wgt = moe ? a.wts[p] : 1.0f;
                    const uint8_t *rd = a.Wd + ((int64_t)e * H + n) * rbI + (int64_t)b * kBlockBytes;
                    const uint4 hd = __ldg(reinterpret_cast<const uint4 *>(rd));
                    const uint4 qd = __ldg(reinterpret_cast<const uint4 *>(rd + 16 + 32 * g + 16 * hh));
                    const float *hs = smem + p * Ip + pad_index(b * kQK + 64 * g + 16 * hh);
                    float sxl, sxh, ql, qh;
                    x_sums(hs, hs + 32, sxl, sxh);
                    qx_sums(qd, hs, hs + 32, ql, qh);
                    const BlockPart pd = decode_head(hd, g);
                    acc += wgt * (pd.ds0 * ql - pd.dm0 * sxl + pd.ds1 * qh - pd.dm1 * sxh);
                }
            }
        }
        acc = warp_sum(acc);
        if (lane == 0) {
            float *dst = a.y + (int64_t)t * H + n;
            *dst = a.accumulate ? *dst + acc : acc;
        }
    }
}

size_t matvec_smem_bytes(int T, int H, int I, int k) {
    const int nbI = (I + kQK - 1) / kQK;
    const size_t p1 = (size_t)T * padded_len(H);
    const size_t p2 = (size_t)T * k * padded_len(nbI * kQK);
    return 4 * (p1 > p2 ? p1 : p2);
}

cudaError_t launch_ffn_matvec(const MatvecArgs &a, cudaStream_t s) {
    const DeviceInfo &di = device_info();
    const size_t smem = matvec_smem_bytes(a.T, a.H, a.I, a.k);
    cudaError_t e = cudaFuncSetAttribute(ffn_matvec_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, ffn_matvec_kernel, kMvThreads, smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    const int grid = di.num_sms;   // one block per SM: co-resident by construction
    MatvecArgs args = a;
    void *params[] = {&args};
    return cudaLaunchCooperativeKernel((const void *)ffn_matvec_kernel, dim3(grid),
                                       dim3(kMvThreads), params, smem, s);
}

}  // namespace zffn
