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
//     warp per output row at a time: the warp streams the row, a chunk of
//     whole 256-weight units at a time, through a shared-memory buffer; the
//     next chunk's words are loaded into registers (4-byte loads by all
//     lanes, all in flight) while the current chunk is computed.  Lane t
//     takes the eight weights 8t .. 8t+7 of each unit, which share one scale
//     (decoded once), and multiplies them by h, staged in shared memory; a
//     row's sum is one warp reduction.  The rows of the grid are interleaved
//     so that all warps stream the matrix together.
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
__device__ __forceinline__ float fmt_weight(const uint8_t *blk, int k) {
    if (F == kFmtQ6_K) {
        const int n = k >> 7, r = k & 127, i = r >> 5, l = r & 31;
        const uint32_t lb = (*(blk + 64 * n + l + 32 * (i & 1)));
        const int lo = (int)((i < 2 ? lb : lb >> 4) & 15u);
        const int hi = (int)(((*(blk + 128 + 32 * n + l)) >> (2 * i)) & 3u);
        const int sc = (int)(int8_t)(*(blk + 192 + (k >> 4)));
        return fp16_at(blk + 208) * (float)(sc * ((lo | (hi << 4)) - 32));   // exact
    } else if (F == kFmtQ5_1) {
        const uint32_t qs = (*(blk + 8 + (k & 15)));
        const uint32_t qh = (*(blk + 4 + (k >> 3)));
        const int q = (int)(((k < 16 ? qs : qs >> 4) & 15u) | (((qh >> (k & 7)) & 1u) << 4));
        return fmaf(fp16_at(blk), (float)q, fp16_at(blk + 2));               // d*q exact
    } else {
        // Q4_K and Q5_K share the scale packing and the nibble arrangement
        const int j = k >> 5;
        const uint8_t *sb = blk + 4;
        int sc, m;
        if (j < 4) {
            sc = (*(sb + j)) & 63;
            m = (*(sb + j + 4)) & 63;
        } else {
            sc = ((*(sb + j + 4)) & 15) | (((*(sb + j - 4)) >> 6) << 4);
            m = ((*(sb + j + 4)) >> 4) | (((*(sb + j)) >> 6) << 4);
        }
        const uint8_t *qs = blk + (F == kFmtQ5_K ? 48 : 16);
        const uint32_t b = qs[32 * (k >> 6) + (k & 31)];
        int q = (int)(((k & 32) ? b >> 4 : b) & 15u);
        if (F == kFmtQ5_K) q |= (int)(((*(blk + 16 + (k & 31))) >> j) & 1u) << 4;
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
constexpr int kDownBuf = 4096;         // bytes of a warp's row-chunk buffer

// 8 bytes at any shared-memory address p: three aligned words and two funnel
// shifts (the buffer has slack after its last byte).
__device__ __forceinline__ void load8(const uint8_t *p, uint32_t &lo, uint32_t &hi) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    const uint32_t *w = reinterpret_cast<const uint32_t *>(a & ~(uintptr_t)3);
    const uint32_t sh = (uint32_t)(a & 3) * 8;
    const uint32_t w0 = w[0], w1 = w[1], w2 = w[2];
    lo = __funnelshift_r(w0, w1, sh);
    hi = __funnelshift_r(w1, w2, sh);
}

// Byte i (0..7) of the pair (lo, hi).
__device__ __forceinline__ uint32_t byte8(uint32_t lo, uint32_t hi, int i) {
    return ((i < 4 ? lo : hi) >> (8 * (i & 3))) & 0xFFu;
}

// Dot product of eight weights with h: h is held as int16 per 32-element group (scale vs)
// with the fp32 sum of every 8 elements (hs8), and the codes go into int8
// lanes for dp2a; the offsets of the formats (the min of Q5_K, the -32 of
// Q6_K, the m of Q5_1) multiply hs8 instead of each weight.
//   Q4_K/Q5_K: sum w*h = d*sc * vs * sum(q*h_int) - dmin*m * hs8
//   Q6_K:      sum w*h = d*sc * (vs * sum(q*h_int) - 32 * hs8)
//   Q5_1:      sum w*h = d * vs * sum(q*h_int) + m * hs8
template <int F>
__device__ __forceinline__ float dot8i(const uint8_t *unit, int k0, uint4 hq, float vs, float hs8) {
    uint32_t c0, c1;   // the eight codes, one per byte (0..63)
    float a, b;        // result = a * isum + b
    if (F == kFmtQ6_K) {
        const int n = k0 >> 7, rr = k0 & 127, i = rr >> 5, l = rr & 31;
        uint32_t l0, l1, h0, h1;
        load8(unit + 64 * n + l + 32 * (i & 1), l0, l1);
        load8(unit + 128 + 32 * n + l, h0, h1);
        const int lsh = i < 2 ? 0 : 4, hsh = 2 * i;
        c0 = ((l0 >> lsh) & 0x0F0F0F0Fu) | (((h0 >> hsh) & 0x03030303u) << 4);
        c1 = ((l1 >> lsh) & 0x0F0F0F0Fu) | (((h1 >> hsh) & 0x03030303u) << 4);
        const float ds = fp16_at(unit + 208) * (float)(int)(int8_t)unit[192 + (k0 >> 4)];
        a = ds * vs;
        b = -32.0f * ds * hs8;
    } else if (F == kFmtQ5_1) {
        const uint8_t *blk = unit + (k0 >> 5) * 24;
        const int j0 = k0 & 31;
        uint32_t q0, q1;
        load8(blk + 8 + (j0 & 15), q0, q1);
        const uint32_t qh = (uint32_t)blk[4] | ((uint32_t)blk[5] << 8) | ((uint32_t)blk[6] << 16) |
                            ((uint32_t)blk[7] << 24);
        const int nsh = j0 < 16 ? 0 : 4;
        // four bits b0..b3 to the low bit of four bytes: b * (1 + 2^7 + 2^14 + 2^21)
        // puts bit i at bit 8i (the partial products do not overlap)
        const uint32_t b_lo = ((((qh >> j0) & 0xFu) * 0x00204081u) & 0x01010101u) << 4;
        const uint32_t b_hi = ((((qh >> (j0 + 4)) & 0xFu) * 0x00204081u) & 0x01010101u) << 4;
        c0 = ((q0 >> nsh) & 0x0F0F0F0Fu) | b_lo;
        c1 = ((q1 >> nsh) & 0x0F0F0F0Fu) | b_hi;
        a = fp16_at(blk) * vs;
        b = fp16_at(blk + 2) * hs8;
    } else {
        const int j = k0 >> 5;
        const uint8_t *sb = unit + 4;
        int sc, m;
        if (j < 4) {
            sc = sb[j] & 63;
            m = sb[j + 4] & 63;
        } else {
            sc = (sb[j + 4] & 15) | ((sb[j - 4] >> 6) << 4);
            m = (sb[j + 4] >> 4) | ((sb[j] >> 6) << 4);
        }
        uint32_t q0, q1;
        load8(unit + (F == kFmtQ5_K ? 48 : 16) + 32 * (k0 >> 6) + (k0 & 31), q0, q1);
        const int nsh = (k0 & 32) ? 4 : 0;
        c0 = (q0 >> nsh) & 0x0F0F0F0Fu;
        c1 = (q1 >> nsh) & 0x0F0F0F0Fu;
        if (F == kFmtQ5_K) {
            uint32_t e0, e1;
            load8(unit + 16 + (k0 & 31), e0, e1);
            c0 |= ((e0 >> j) & 0x01010101u) << 4;
            c1 |= ((e1 >> j) & 0x01010101u) << 4;
        }
        a = fp16_at(unit) * (float)sc * vs;
        b = -(fp16_at(unit + 2) * (float)m) * hs8;
    }
    int isum = __dp2a_lo((int)hq.x, (int)c0, 0);
    isum = __dp2a_hi((int)hq.y, (int)c0, isum);
    isum = __dp2a_lo((int)hq.z, (int)c1, isum);
    isum = __dp2a_hi((int)hq.w, (int)c1, isum);
    return fmaf(a, (float)isum, b);
}

// Each expert slot's h is held quantised in shared memory (layout in the
// kernel), followed by one row-chunk buffer per warp.  A warp walks one stream of chunks: for each of its output
// rows, for each valid expert slot, the row's whole 256-weight units a chunk
// at a time.  The words of the next chunk are loaded into registers (all of a
// lane's loads in flight) while the current chunk, already in the buffer, is
// computed: lane t takes weights 8t .. 8t+7 of each unit.
struct ChunkCursor {
    int64_t n;   // output row
    int p;       // expert slot
    int u0;      // first unit of the chunk
    bool done;
};

template <int F>
__global__ void __launch_bounds__(kDownWarps * 32, 1) down_fmt_kernel(MatvecArgs a) {
    // Shared memory: h as int16 [P*I], its scale per 32 elements (fp32
    // [P*I/32]) and its sum per 8 elements (fp32 [P*I/8]), then one row-chunk
    // buffer per warp.
    extern __shared__ __align__(16) uint8_t smem_raw[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int H = a.H, I = a.I, P = a.k;
    const bool moe = a.ids != nullptr;
    const int PI = P * I;
    int16_t *hq = reinterpret_cast<int16_t *>(smem_raw);
    float *hvs = reinterpret_cast<float *>(smem_raw + (size_t)PI * 2);
    float *hs8 = hvs + PI / 32;
    uint8_t *buf = reinterpret_cast<uint8_t *>(hs8 + PI / 8) + (size_t)warp * (kDownBuf + 16);
    // the next work in the stream may be scheduled as this grid's blocks leave
    if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    // h is written by the gate/up kernel: wait until that grid has completed
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // quantise h: warp w takes the 32-element groups w, w + 16, ...; lane t
    // element t of the group (loads of four groups issued together)
    for (int g0 = warp; g0 < PI / 32; g0 += 4 * kDownWarps) {
        float v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int g = g0 + u * kDownWarps;
            v[u] = g < PI / 32 ? __ldcg(a.h + (size_t)g * 32 + lane) : 0.0f;
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int g = g0 + u * kDownWarps;
            float mx = fabsf(v[u]);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            float s8 = v[u];
#pragma unroll
            for (int o = 4; o > 0; o >>= 1) s8 += __shfl_xor_sync(0xffffffffu, s8, o);
            if (g < PI / 32) {
                const float inv = mx > 0.0f ? 32767.0f / mx : 0.0f;
                hq[(size_t)g * 32 + lane] = (int16_t)__float2int_rn(v[u] * inv);
                if (lane == 0) hvs[g] = mx > 0.0f ? mx / 32767.0f : 0.0f;
                if ((lane & 7) == 0) hs8[(size_t)g * 4 + (lane >> 3)] = s8;
            }
        }
    }
    __syncthreads();
    const int64_t rb = fmt_row_bytes_hd(F, I);
    const int ub = (256 / fmt_block_weights(F)) * fmt_block_bytes(F);   // bytes of a unit
    const int nu = (I + 255) / 256;
    const int nuc = (kDownBuf - 4) / ub;                                 // units per chunk
    const int k0 = 8 * lane;
    const int64_t gw = (int64_t)gridDim.x * kDownWarps;
    const int64_t n_first = (int64_t)warp * gridDim.x + blockIdx.x;
    auto slot_valid = [&](int p) {
        const int e = moe ? a.ids[p] : 0;
        return e >= 0 && e < a.E;
    };
    auto next_slot = [&](int p) {            // first valid slot >= p (P if none)
        while (p < P && !slot_valid(p)) ++p;
        return p;
    };
    const int p_first = next_slot(0);
    if (p_first >= P) {
        // no valid expert slot: every output of this warp is zero
        for (int64_t n = n_first; n < H; n += gw)
            if (lane == 0 && !a.accumulate) a.y[n] = 0.0f;
        return;
    }
    auto advance = [&](ChunkCursor &c) {
        c.u0 += nuc;
        if (c.u0 < nu) return;
        c.u0 = 0;
        c.p = next_slot(c.p + 1);
        if (c.p < P) return;
        c.p = p_first;
        c.n += gw;
        c.done = c.n >= H;
    };
    // The bytes of chunk c: [src, end) of its row (the last unit may be cut
    // short by the row's end), read as the 4-byte words from the word holding
    // src up to end, plus the 0-3 tail bytes (W_down is 4-byte aligned: no
    // word starts before the matrix or ends after it).  At most kDownBuf / 128
    // words per lane.
    constexpr int kWords = kDownBuf / 128;
    uint32_t r[kWords];
    uint32_t rt = 0;
    auto chunk_src = [&](const ChunkCursor &c) {
        const int e = moe ? a.ids[c.p] : 0;
        return a.Wd + ((int64_t)e * H + c.n) * rb + (size_t)c.u0 * ub;
    };
    auto chunk_end = [&](const ChunkCursor &c) {
        const int e = moe ? a.ids[c.p] : 0;
        return a.Wd + ((int64_t)e * H + c.n) * rb + min((int64_t)min(nu, c.u0 + nuc) * ub, rb);
    };
    auto issue = [&](const ChunkCursor &c) {
        const uint8_t *src = chunk_src(c);
        const uintptr_t a0 = reinterpret_cast<uintptr_t>(src) & ~(uintptr_t)3;
        const size_t span = reinterpret_cast<uintptr_t>(chunk_end(c)) - a0;
        const int nwords = (int)(span / 4), tail = (int)(span % 4);
        const uint32_t *w32 = reinterpret_cast<const uint32_t *>(a0);
#pragma unroll
        for (int j = 0; j < kWords; ++j) {
            const int i = lane + 32 * j;
            r[j] = i < nwords ? __ldg(w32 + i) : 0u;
        }
        rt = lane < tail ? (uint32_t)__ldg(reinterpret_cast<const uint8_t *>(a0) + 4 * nwords + lane) : 0u;
    };
    ChunkCursor cur{n_first, p_first, 0, n_first >= H};
    if (!cur.done) issue(cur);
    float acc = 0.0f, part = 0.0f;
    while (!cur.done) {
        // the current chunk's words, loaded during the previous chunk's
        // compute, go to the buffer (after every lane finished reading it)
        const uint8_t *src = chunk_src(cur);
        const uintptr_t a0 = reinterpret_cast<uintptr_t>(src) & ~(uintptr_t)3;
        const size_t span = reinterpret_cast<uintptr_t>(chunk_end(cur)) - a0;
        const int nwords = (int)(span / 4), tail = (int)(span % 4);
        __syncwarp();
#pragma unroll
        for (int j = 0; j < kWords; ++j) {
            const int i = lane + 32 * j;
            if (i < nwords) reinterpret_cast<uint32_t *>(buf)[i] = r[j];
        }
        if (lane < tail) buf[4 * nwords + lane] = (uint8_t)rt;
        __syncwarp();
        // the next chunk's loads go out before this chunk is computed
        ChunkCursor nx = cur;
        advance(nx);
        if (!nx.done) issue(nx);
        const uint8_t *sb = buf + (reinterpret_cast<uintptr_t>(src) - a0);
        const size_t hbase = (size_t)cur.p * I;
        const int u1 = min(nu, cur.u0 + nuc);
        for (int u = cur.u0; u < u1; ++u) {
            const int c0 = u * 256 + k0;
            if (c0 >= I) continue;                  // past the row (I % 256 != 0)
            const size_t hc = hbase + c0;           // a multiple of 8
            const uint4 hv = *reinterpret_cast<const uint4 *>(hq + hc);
            part += dot8i<F>(sb + (size_t)(u - cur.u0) * ub, k0, hv, hvs[hc >> 5], hs8[hc >> 3]);
        }
        if (u1 >= nu) {                             // last chunk of this slot's row
            float w = 1.0f;
            if (moe) {
                w = a.wts[cur.p];
                if (a.down_scale) w *= a.down_scale[a.ids[cur.p]];
            }
            acc = fmaf(w, part, acc);
            part = 0.0f;
            if (nx.done || nx.n != cur.n) {         // last slot of this output row
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
                if (lane == 0) a.y[cur.n] = a.accumulate ? a.y[cur.n] + acc : acc;
                acc = 0.0f;
            }
        }
        cur = nx;
    }
}

size_t down_fmt_smem_bytes(int I, int k) {
    const size_t pi = (size_t)k * I;
    return pi * 2 + pi / 32 * 4 + pi / 8 * 4 + (size_t)kDownWarps * (kDownBuf + 16);
}

cudaError_t launch_token_fmt(const MatvecArgs &a, int wd_fmt, cudaStream_t s) {
    if (a.T != 1 || !fmt_valid(wd_fmt) || wd_fmt == kFmtQ4_K || a.I % 64 != 0) return cudaErrorInvalidValue;
    const DeviceInfo &di = device_info();
    const size_t smem_a = gu_smem_total(a.H, a.I, a.k), smem_b = down_fmt_smem_bytes(a.I, a.k);
    if (smem_a > (size_t)di.max_smem_optin || smem_b > (size_t)di.max_smem_optin) return cudaErrorInvalidValue;
    const void *down = wd_fmt == kFmtQ5_K ? (const void *)down_fmt_kernel<kFmtQ5_K>
                     : wd_fmt == kFmtQ6_K ? (const void *)down_fmt_kernel<kFmtQ6_K>
                                          : (const void *)down_fmt_kernel<kFmtQ5_1>;
    // Raise, never lower, each kernel's dynamic shared-memory limit (the
    // gate/up kernel is shared with the Q4_K single-token path).
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, ffn_gu_kernel);
    if (e == cudaSuccess) e = ensure_dynamic_smem((const void *)ffn_gu_kernel, smem_a);
    if (e == cudaSuccess) e = ensure_dynamic_smem(down, smem_b);
    if (e != cudaSuccess) return e;
    // (the gate/up kernel's block size is its launch bound: fa.maxThreadsPerBlock)
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
