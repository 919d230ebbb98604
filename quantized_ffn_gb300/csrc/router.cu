// router.cu -- the router of a routed (mixture-of-experts) layer on the
// device: router logits -> the top_k experts of each token -> softmax weights
// over the chosen logits, written to device buffers that the routed block
// reads as they are ("Four bottlenecks, one CUDA backend...", section
// "Bottleneck 2 -- MoE decode was paying for its routing twice": the layer
// computes router logits and picks the top-k experts; section "What's next,
// and what it's worth": a GPU-side step that drops the last router round-trip
// to the host).  The pages do not state the weighting; the softmax over the
// chosen k logits is the reading used here.
//
// One warp per token: top_k passes over the token's logits (held in registers
// when E <= 256), each a warp-wide maximum of 64-bit rank keys, then one
// warp-wide sum for the softmax.
#include "router.h"

#include <cstdint>

namespace zffn {

// Rank of an expert as one 64-bit key, larger = chosen first: the high word
// maps the logit to an unsigned integer in the order of the values (NaN
// lowest, -0 the same as +0), the low word is ~index, so that equal logits go
// to the lower index.  Every key of a row is distinct, so the j-th choice is
// the largest key below the (j-1)-th: no "taken" marks are needed.
__device__ __forceinline__ uint64_t router_key(float v, int e) {
    uint32_t r;
    if (v != v) {
        r = 0u;
    } else {
        const uint32_t u = __float_as_uint(v == 0.0f ? 0.0f : v);
        r = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    }
    return ((uint64_t)r << 32) | (uint64_t)(0xFFFFFFFFu - (uint32_t)e);
}

constexpr int kRouterWarps = 8;
constexpr int kRouterMaxK = 64;

// Largest 64-bit key over the warp: two 32-bit warp reductions (high words,
// then the low words of the lanes that hold the largest high word).
__device__ __forceinline__ uint64_t warp_max_key(uint64_t key) {
    const uint32_t hi = (uint32_t)(key >> 32), lo = (uint32_t)key;
    const uint32_t mhi = __reduce_max_sync(0xffffffffu, hi);
    const uint32_t mlo = __reduce_max_sync(0xffffffffu, hi == mhi ? lo : 0u);
    return ((uint64_t)mhi << 32) | mlo;
}

// R > 0: every lane holds the keys of experts lane, lane + 32, ... (E <= 32 R)
// in registers, read once; R == 0: any E, the logits are read again in every
// pass (from L1 after the first).
template <int R>
__global__ void __launch_bounds__(kRouterWarps * 32)
    moe_router_kernel(const float *__restrict__ logits, int T, int E, int k, int32_t *__restrict__ ids,
                      float *__restrict__ weights) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t = blockIdx.x * kRouterWarps + warp;
    if (t >= T) return;
    const float *l = logits + (int64_t)t * E;
    uint64_t keys[R > 0 ? R : 1];
    if (R > 0) {
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int e = lane + 32 * r;
            keys[r] = e < E ? router_key(__ldg(l + e), e) : 0ull;   // 0: below every key
        }
    }
    // choice j is kept by lane j % 32 in slot j / 32
    float val[kRouterMaxK / 32];
    int idx[kRouterMaxK / 32];
#pragma unroll
    for (int s = 0; s < kRouterMaxK / 32; ++s) { val[s] = 0.0f; idx[s] = 0; }
    uint64_t prev = ~0ull;
    float top = 0.0f;
    for (int j = 0; j < k; ++j) {
        uint64_t best = 0;
        if (R > 0) {
#pragma unroll
            for (int r = 0; r < R; ++r)
                if (keys[r] < prev && keys[r] > best) best = keys[r];
        } else {
            for (int e = lane; e < E; e += 32) {
                const uint64_t key = router_key(__ldg(l + e), e);
                if (key < prev && key > best) best = key;
            }
        }
        best = warp_max_key(best);
        prev = best;
        // (k <= E leaves a candidate in every pass; the clamp only keeps the
        // load in bounds whatever the key)
        int e = (int)(0xFFFFFFFFu - (uint32_t)best);
        e = e < 0 || e >= E ? 0 : e;
        const float v = __ldg(l + e);
        if (j == 0) top = v;
        if ((j & 31) == lane) {
#pragma unroll
            for (int s = 0; s < kRouterMaxK / 32; ++s)
                if (s == (j >> 5)) { val[s] = v; idx[s] = e; }
        }
    }
    // softmax over the chosen logits, relative to the largest
    float ex[kRouterMaxK / 32];
    float sum = 0.0f;
#pragma unroll
    for (int s = 0; s < kRouterMaxK / 32; ++s) {
        ex[s] = (s * 32 + lane < k) ? expf(val[s] - top) : 0.0f;
        sum += ex[s];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
#pragma unroll
    for (int s = 0; s < kRouterMaxK / 32; ++s) {
        const int j = s * 32 + lane;
        if (j < k) {
            ids[(int64_t)t * k + j] = idx[s];
            weights[(int64_t)t * k + j] = ex[s] / sum;
        }
    }
}

cudaError_t launch_moe_router(const float *logits, int T, int E, int k, int32_t *ids, float *weights,
                              cudaStream_t s) {
    if (T < 1 || E < 1 || k < 1 || k > E || k > kRouterMaxK) return cudaErrorInvalidValue;
    const int blocks = (T + kRouterWarps - 1) / kRouterWarps;
    if (E <= 32 * 4)
        moe_router_kernel<4><<<blocks, kRouterWarps * 32, 0, s>>>(logits, T, E, k, ids, weights);
    else if (E <= 32 * 8)
        moe_router_kernel<8><<<blocks, kRouterWarps * 32, 0, s>>>(logits, T, E, k, ids, weights);
    else
        moe_router_kernel<0><<<blocks, kRouterWarps * 32, 0, s>>>(logits, T, E, k, ids, weights);
    return cudaGetLastError();
}

}  // namespace zffn
