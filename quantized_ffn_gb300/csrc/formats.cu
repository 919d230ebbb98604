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
//     single-token path, which leaves h (fp32 [P][I]) in the workspace.
//     Each block owns a contiguous range of output rows and has their bytes
//     of every chosen expert streamed into L2 before it waits for h.  h is
//     quantised in shared memory to int16 per 32 values.  Each warp streams
//     its rows (every valid expert slot's row of each) as one sequence of
//     256-weight units, eight to a chunk, one bulk copy per unit into
//     shared memory, two chunks ahead of the one being computed; a chunk is
//     one pass: four lanes per unit, 64 weights (two scales) per lane,
//     integer dot products by dp2a.
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

// Bytes of a 256-weight unit of W_down; the stride of a unit's slot in a
// warp's chunk buffer (a multiple of 16: a unit is copied as the aligned
// pieces that hold it, so a Q6_K unit may start up to 15 bytes into its
// slot); units per chunk (one pass of a warp).
__host__ __device__ constexpr int fmt_unit_bytes(int f) {
    return f == kFmtQ5_K ? 176 : f == kFmtQ6_K ? 210 : 192;
}
__host__ __device__ constexpr int fmt_slot_bytes(int f) { return f == kFmtQ6_K ? 240 : fmt_unit_bytes(f); }
__host__ __device__ constexpr int fmt_chunk_units(int) { return 8; }
constexpr int kChunkBufs = 3;      // chunk buffers per warp: two chunks in flight

// Four codes (one per byte of c) against four int16 values of h (two per
// word, in weight order), added to acc: exact.
__device__ __forceinline__ int dot_codes4(uint32_t c, uint32_t h01, uint32_t h23, int acc) {
    acc = __dp2a_lo((int)h01, (int)c, acc);
    return __dp2a_hi((int)h23, (int)c, acc);
}

// Bit i (i < 4) of b to bit 4 of byte i: the four shifted copies of b in the
// product do not overlap, and only the intended bit lands on each bit 4.
__device__ __forceinline__ uint32_t spread4_to_bit4(uint32_t b) {
    return ((b & 0xFu) * 0x02040810u) & 0x10101010u;
}

// 32 bytes at the even shared-memory address p: nine aligned words and
// eight funnel shifts.
__device__ __forceinline__ void load32_at(const uint8_t *p, uint32_t (&o)[8]) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    const uint32_t *w = reinterpret_cast<const uint32_t *>(a & ~(uintptr_t)3);
    const uint32_t sh = (uint32_t)(a & 3) * 8;
    uint32_t v[9];
#pragma unroll
    for (int i = 0; i < 9; ++i) v[i] = w[i];
#pragma unroll
    for (int i = 0; i < 8; ++i) o[i] = __funnelshift_r(v[i], v[i + 1], sh);
}

// 16 bytes of shared memory at the 32-bit shared address a.
__device__ __forceinline__ uint4 lds128(uint32_t a) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
    return v;
}

// Dot product of the 64 weights of part jp (weights 64jp .. 64jp+63: groups
// 2jp and 2jp+1 of 32) of one unit with h.  h is held as int16 (hline: the
// shared address of the 128-byte line of the part's 64 values with the
// line's swizzle in bits 4-6, so that piece i is at hline ^ (i << 4); vs:
// the scales of its two groups) with the fp32 sums of
// its four 16-value quarters (hs); the codes go into int8 lanes for dp2a and
// the formats' offsets (the min of Q5_K, the -32 of Q6_K, the m of Q5_1)
// multiply the sums of h instead of each weight.  Per group of 32:
//   Q5_K: d*sc*vs*sum(q*h_int) - dmin*m*(sum of h)
//   Q5_1: d*vs*sum(q*h_int) + m*(sum of h)
//   Q6_K: per 16 weights, d*sc*(vs*sum(q*h_int) - 32*(sum of h))
// u: the unit's first byte (16-byte aligned for Q5_K and Q5_1, even for
// Q6_K).  Independent partial sums keep the dp2a chains short.
template <int F>
__device__ __forceinline__ float dot64(const uint8_t *u, int jp, uint32_t hline, float2 vs, float4 hs) {
    uint32_t hw[32];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint4 v = lds128(hline ^ (uint32_t)(i << 4));
        hw[4 * i] = v.x;
        hw[4 * i + 1] = v.y;
        hw[4 * i + 2] = v.z;
        hw[4 * i + 3] = v.w;
    }
    if (F == kFmtQ5_K) {
        // sub-blocks j0 = 2jp and j0 + 1: their codes are the low and high
        // nibbles of the same 32 bytes, their fifth bits bits j0 and j0 + 1
        // of the same 32 bytes of qh
        const int j0 = 2 * jp;
        const uint4 hd = *reinterpret_cast<const uint4 *>(u);
        const uint32_t sc4 = jp < 2 ? (hd.y & 0x3F3F3F3Fu)
                                    : (hd.w & 0x0F0F0F0Fu) | ((hd.y >> 2) & 0x30303030u);
        const uint32_t m4 = jp < 2 ? (hd.z & 0x3F3F3F3Fu)
                                   : ((hd.w >> 4) & 0x0F0F0F0Fu) | ((hd.z >> 2) & 0x30303030u);
        const int sh = 8 * (j0 & 3);
        const float sc0 = (float)((sc4 >> sh) & 0xFFu), sc1 = (float)((sc4 >> (sh + 8)) & 0xFFu);
        const float m0 = (float)((m4 >> sh) & 0xFFu), m1 = (float)((m4 >> (sh + 8)) & 0xFFu);
        const uint4 qa = *reinterpret_cast<const uint4 *>(u + 48 + 32 * jp);
        const uint4 qb = *reinterpret_cast<const uint4 *>(u + 64 + 32 * jp);
        const uint4 ha = *reinterpret_cast<const uint4 *>(u + 16);
        const uint4 hb = *reinterpret_cast<const uint4 *>(u + 32);
        const uint32_t qs[8] = {qa.x, qa.y, qa.z, qa.w, qb.x, qb.y, qb.z, qb.w};
        const uint32_t qh[8] = {ha.x, ha.y, ha.z, ha.w, hb.x, hb.y, hb.z, hb.w};
        int is[4] = {0, 0, 0, 0};
#pragma unroll
        for (int w = 0; w < 8; ++w) {
            const uint32_t b = qh[w] >> j0;
            const uint32_t lo = (qs[w] & 0x0F0F0F0Fu) | ((b << 4) & 0x10101010u);
            const uint32_t hi = ((qs[w] >> 4) & 0x0F0F0F0Fu) | ((b << 3) & 0x10101010u);
            is[w & 1] = dot_codes4(lo, hw[2 * w], hw[2 * w + 1], is[w & 1]);
            is[2 + (w & 1)] = dot_codes4(hi, hw[16 + 2 * w], hw[17 + 2 * w], is[2 + (w & 1)]);
        }
        const float d = half_bits_to_float(hd.x & 0xFFFFu), dmin = half_bits_to_float(hd.x >> 16);
        const float r0 = fmaf((d * sc0) * vs.x, (float)(is[0] + is[1]), -(dmin * m0) * (hs.x + hs.y));
        const float r1 = fmaf((d * sc1) * vs.y, (float)(is[2] + is[3]), -(dmin * m1) * (hs.z + hs.w));
        return r0 + r1;
    } else if (F == kFmtQ5_1) {
        // blocks 2jp and 2jp + 1: 48 bytes from a 16-byte boundary
        const uint4 b0 = *reinterpret_cast<const uint4 *>(u + 48 * jp);
        const uint4 b1 = *reinterpret_cast<const uint4 *>(u + 48 * jp + 16);
        const uint4 b2 = *reinterpret_cast<const uint4 *>(u + 48 * jp + 32);
        const uint32_t W[12] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w, b2.x, b2.y, b2.z, b2.w};
        float r = 0.0f;
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const uint32_t hdr = W[6 * k], qh = W[6 * k + 1];
            int is[2] = {0, 0};
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                // weights 4w..4w+3: low nibbles; 16+4w..: high nibbles
                const uint32_t qs = W[6 * k + 2 + w];
                const uint32_t lo = (qs & 0x0F0F0F0Fu) | spread4_to_bit4(qh >> (4 * w));
                const uint32_t hi = ((qs >> 4) & 0x0F0F0F0Fu) | spread4_to_bit4(qh >> (16 + 4 * w));
                is[0] = dot_codes4(lo, hw[16 * k + 2 * w], hw[16 * k + 2 * w + 1], is[0]);
                is[1] = dot_codes4(hi, hw[16 * k + 8 + 2 * w], hw[16 * k + 9 + 2 * w], is[1]);
            }
            const float d = half_bits_to_float(hdr & 0xFFFFu), m = half_bits_to_float(hdr >> 16);
            const float vk = k ? vs.y : vs.x, sk = k ? hs.z + hs.w : hs.x + hs.y;
            r += fmaf(d * vk, (float)(is[0] + is[1]), m * sk);
        }
        return r;
    } else {
        // Q6_K: half n = jp / 2, quarters i0 = 2 (jp % 2) and i0 + 1: their
        // low bits are the same nibble of 64 consecutive bytes of ql (32
        // each), their high bits bits 2 i0 and 2 i0 + 2 of the same 32 bytes
        // of qh; one scale per 16 weights
        const int n = jp >> 1, i0 = 2 * (jp & 1);
        uint32_t l0[8], l1[8], qh[8];
        load32_at(u + 64 * n, l0);
        load32_at(u + 64 * n + 32, l1);
        load32_at(u + 128 + 32 * n, qh);
        const int lsh = 2 * i0, hsh = 2 * i0;
        int is[4] = {0, 0, 0, 0};
#pragma unroll
        for (int w = 0; w < 8; ++w) {
            const uint32_t c0 = ((l0[w] >> lsh) & 0x0F0F0F0Fu) | (((qh[w] >> hsh) & 0x03030303u) << 4);
            const uint32_t c1 = ((l1[w] >> lsh) & 0x0F0F0F0Fu) | (((qh[w] >> (hsh + 2)) & 0x03030303u) << 4);
            is[w >> 2] = dot_codes4(c0, hw[2 * w], hw[2 * w + 1], is[w >> 2]);
            is[2 + (w >> 2)] = dot_codes4(c1, hw[16 + 2 * w], hw[17 + 2 * w], is[2 + (w >> 2)]);
        }
        const uint32_t sa = *reinterpret_cast<const uint16_t *>(u + 192 + 4 * jp);
        const uint32_t sb = *reinterpret_cast<const uint16_t *>(u + 194 + 4 * jp);
        const float s0 = (float)(int)(int8_t)(sa & 0xFFu), s1 = (float)(int)(int8_t)(sa >> 8);
        const float s2 = (float)(int)(int8_t)(sb & 0xFFu), s3 = (float)(int)(int8_t)(sb >> 8);
        const float d = half_bits_to_float(*reinterpret_cast<const uint16_t *>(u + 208));
        const float r = s0 * fmaf(vs.x, (float)is[0], -32.0f * hs.x) + s1 * fmaf(vs.x, (float)is[1], -32.0f * hs.y) +
                        s2 * fmaf(vs.y, (float)is[2], -32.0f * hs.z) + s3 * fmaf(vs.y, (float)is[3], -32.0f * hs.w);
        return d * r;
    }
}

// q = n / d and r = n % d for 0 <= n < 2^24 and 1 <= d: the product with the
// rounded reciprocal rd is within one of the quotient (its relative error is
// below 2^-23 and n / d < 2^23 unless d == 1, where it is exact), and one
// correction step fixes it.
__device__ __forceinline__ int div_small(int n, int d, float rd, int &r) {
    int q = __float2int_rz((float)n * rd);
    r = n - q * d;
    if (r < 0) {
        --q;
        r += d;
    } else if (r >= d) {
        ++q;
        r -= d;
    }
    return q;
}

// Bulk copy global -> shared (16-byte aligned addresses, a multiple of 16
// bytes), counted on the barrier bar.
__device__ __forceinline__ void bulk_copy_to_smem(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(dst)),
                 "l"(src), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}

// Global -> shared copy of 4 bytes that bypasses the registers; src_bytes < 4
// reads only that many bytes and fills the rest with zeros.
__device__ __forceinline__ void cp_async4(uint32_t dst, const void *src, uint32_t src_bytes) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// every group but the last two committed is complete
__device__ __forceinline__ void cp_async_wait_ahead2() { asm volatile("cp.async.wait_group 2;" ::: "memory"); }

// Shared memory of the down kernel: h of every expert slot as int16 [P*I]
// (each 128-byte line's 16-byte pieces in the order piece ^ (line % 8), so
// that lanes reading the same piece of different lines use different
// banks), its scale per 32 values (fp32, P*I/32 rounded up to a multiple of
// 4) and its sums per 16 values (fp32 pairs [P*I/32]), the valid expert
// slots (index, weight and expert, 64 each) and their count, a barrier per
// chunk buffer, then the chunk buffers of every warp.
__host__ __device__ inline int down_fmt_ng_pad(int I, int k) { return ((k * I / 32) + 3) & ~3; }
__host__ __device__ inline size_t down_fmt_h_bytes(int I, int k) {
    const size_t pi = (size_t)k * I;
    return (pi * 2 + (size_t)down_fmt_ng_pad(I, k) * 4 + pi / 32 * 8 + 3 * 64 * 4 + 16 +
            (size_t)kDownWarps * kChunkBufs * 8 + 15) & ~(size_t)15;
}
size_t down_fmt_smem_bytes(int f, int I, int k) {
    return down_fmt_h_bytes(I, k) + (size_t)kDownWarps * kChunkBufs * fmt_chunk_units(f) * fmt_slot_bytes(f);
}

// A warp's work is one stream of units: for each of its output rows n (the
// block's rows n0 + warp, n0 + warp + kDownWarps, ...),
// for each valid expert slot, the row's 256-weight units in order.  The
// stream is cut into chunks of fmt_chunk_units units, whatever rows or slots
// they come from.  The next two chunks are copied into the warp's other
// buffers (cp.async, no registers held) while the current one is computed.
// In a chunk, lane t describes unit t: its address, length and where its h
// starts; in its pass, the eight groups of four lanes take the eight units,
// lane jp of a group the 64 weights 64jp.. of its unit.
struct UnitInfo {
    const uint8_t *src;   // first byte of the unit in W_down
    int nbytes;           // its length (the last unit of a Q5_1 row may be short)
    int hb;               // index of its first weight's h (slot * I + 256 * unit)
    int lim;              // valid weights in it (I - 256 * unit)
    int vi;               // index of its slot in the valid-slot table
};

template <int F>
__global__ void __launch_bounds__(kDownWarps * 32, 1) down_fmt_kernel(MatvecArgs a) {
    extern __shared__ __align__(128) uint8_t smem_raw[];
    constexpr int UB = fmt_unit_bytes(F), SB = fmt_slot_bytes(F), K = fmt_chunk_units(F);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int H = a.H, I = a.I, P = a.k;
    const bool moe = a.ids != nullptr;
    const int PI = P * I, NG = PI / 32;
    int16_t *hq = reinterpret_cast<int16_t *>(smem_raw);
    const uint32_t hq_s = smem_u32(hq);
    // the swizzled reads of h take its lines to start on 128-byte boundaries
    if (hq_s & 127u) {
        if (threadIdx.x == 0) record_error(a.err, ZFFN_ERR_UNSUPPORTED);
        return;
    }
    float *hvs = reinterpret_cast<float *>(smem_raw + (size_t)PI * 2);
    float2 *hs16 = reinterpret_cast<float2 *>(hvs + down_fmt_ng_pad(I, P));
    int *vslot = reinterpret_cast<int *>(hs16 + NG);
    float *wslot = reinterpret_cast<float *>(vslot + 64);
    int *eslot = reinterpret_cast<int *>(wslot + 64);
    int *nvalid = eslot + 64;             // the number of valid slots (16 bytes reserved)
    uint64_t *bars = reinterpret_cast<uint64_t *>(eslot + 68) + warp * kChunkBufs;
    uint8_t *buf = smem_raw + down_fmt_h_bytes(I, P) + (size_t)warp * kChunkBufs * K * SB;
    // the block's output rows [n0, n1)
    const int n0 = (int)((int64_t)H * blockIdx.x / gridDim.x);
    const int n1 = (int)((int64_t)H * (blockIdx.x + 1) / gridDim.x);
    const int64_t rb = fmt_row_bytes_hd(F, I);
    // the next work in the stream may be scheduled as this grid's blocks leave
    if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    // W_down does not depend on the gate/up kernel: the block's rows of every
    // valid expert slot (one contiguous range each) are streamed into L2 now,
    // while the gate/up kernel finishes (the whole 16-byte pieces inside
    // each range; the copies fetch the rest)
    if (warp == 0 && n1 > n0)
        for (int p = lane; p < P; p += 32) {
            const int e = moe ? a.ids[p] : 0;
            if (e < 0 || e >= a.E) continue;
            const uintptr_t lo = reinterpret_cast<uintptr_t>(a.Wd + ((int64_t)e * H + n0) * rb);
            const uintptr_t hi = reinterpret_cast<uintptr_t>(a.Wd + ((int64_t)e * H + n1) * rb);
            const uintptr_t lo16 = (lo + 15) & ~(uintptr_t)15, hi16 = hi & ~(uintptr_t)15;
            if (hi16 > lo16) prefetch_l2_bulk(reinterpret_cast<const void *>(lo16), (uint32_t)(hi16 - lo16));
        }
    // h is written by the gate/up kernel: wait until that grid has completed
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // the valid expert slots, in slot order, with their weights
    if (warp == 0) {
        int base = 0;
        for (int p0 = 0; p0 < P; p0 += 32) {
            const int p = p0 + lane;
            const int e = p < P ? (moe ? a.ids[p] : 0) : -1;
            const bool ok = e >= 0 && e < a.E;
            const uint32_t bal = __ballot_sync(0xffffffffu, ok);
            if (ok) {
                const int at = base + __popc(bal & ((1u << lane) - 1u));
                float w = 1.0f;
                if (moe) {
                    w = a.wts[p];
                    if (a.down_scale) w *= a.down_scale[e];
                }
                vslot[at] = p;
                wslot[at] = w;
                eslot[at] = e;
            }
            base += __popc(bal);
        }
        if (lane == 0) *nvalid = base;
    }
    if (threadIdx.x == 0) {
        uint64_t *all = reinterpret_cast<uint64_t *>(eslot + 68);
        for (int i = 0; i < kDownWarps * kChunkBufs; ++i) mbar_init(&all[i], 1);
        fence_mbarrier_init();
    }
    __syncthreads();
    const int V = *nvalid;
    // warp w takes the rows n0 + w, n0 + w + kDownWarps, ...
    const int gw = kDownWarps;
    const int n_first = n0 + warp;
    if (V == 0) {
        // no valid expert slot: every output is zero (V is the same for the
        // whole block, so every thread leaves here)
        if (lane == 0 && !a.accumulate)
            for (int n = n_first; n < n1; n += gw) a.y[n] = 0.0f;
        return;
    }
    const int nu = (I + 255) / 256;                  // units of one slot's row
    const int R = V * nu;                            // units of one output row
    const int rows = n_first < n1 ? (n1 - 1 - n_first) / gw + 1 : 0;
    const int S = rows * R;                          // units of the warp's stream
    const int nch = (S + K - 1) / K;
    // One bulk copy per unit when W_down is 16-byte aligned: the 16-byte
    // aligned range that holds the unit lies inside the matrix (its rows of
    // H % 256 == 0 units end it on a 16-byte boundary, whatever the format).
    // Else 4-byte copies of the words that hold the unit.
    const bool bulk = (reinterpret_cast<uintptr_t>(a.Wd) & 15) == 0;
    const uint32_t buf_s = (uint32_t)__cvta_generic_to_shared(buf);

    // stream position s -> (row, slot, unit): reciprocal divisions while
    // every position is below 2^24 (always, unless a launch has very few
    // blocks)
    const bool fdiv = S < (1 << 24);
    const float rR = 1.0f / (float)R, rnu = 1.0f / (float)nu;
    auto info = [&](int s) {
        UnitInfo ui{nullptr, 0, 0, 0, 0};
        if (s < S) {
            int ri, rem, vi, u;
            if (fdiv) {
                ri = div_small(s, R, rR, rem);
                vi = div_small(rem, nu, rnu, u);
            } else {
                ri = s / R;
                rem = s - ri * R;
                vi = rem / nu;
                u = rem - vi * nu;
            }
            const int p = vslot[vi];
            const int e = eslot[vi];
            const int n = n_first + ri * gw;
            ui.src = a.Wd + ((int64_t)e * H + n) * rb + (int64_t)u * UB;
            ui.nbytes = (int)min((int64_t)UB, rb - (int64_t)u * UB);
            ui.hb = p * I + 256 * u;
            ui.lim = I - 256 * u;
            ui.vi = vi;
        }
        return ui;
    };
    // copy chunk c (lane t < kc described by ui) into buffer b: the aligned
    // pieces (or words) from the one holding the unit's first byte to the
    // one holding its last, to the same alignment in the unit's slot
    auto issue = [&](const UnitInfo &ui, int kc, int b) {
        const uint32_t dst0 = buf_s + (uint32_t)(b * K * SB);
        const unsigned long long src = reinterpret_cast<unsigned long long>(ui.src);
        if (bulk) {
            const unsigned long long a0 = src & ~15ull;
            const unsigned long long a1 = (src + (unsigned long long)ui.nbytes + 15ull) & ~15ull;
            const uint32_t bytes = lane < kc ? (uint32_t)(a1 - a0) : 0u;
            uint32_t total = bytes;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) total += __shfl_xor_sync(0xffffffffu, total, o);
            if (lane == 0) mbar_arrive_expect_tx(&bars[b], total);
            __syncwarp();
            if (bytes)
                bulk_copy_to_smem(buf + (size_t)b * K * SB + (size_t)lane * SB, reinterpret_cast<const void *>(a0),
                                  bytes, &bars[b]);
        } else {
            for (int t = 0; t < kc; ++t) {
                const unsigned long long s_t = __shfl_sync(0xffffffffu, src, t);
                const int nb_t = __shfl_sync(0xffffffffu, ui.nbytes, t);
                const unsigned long long a0 = s_t & ~3ull;
                const int span = (int)(s_t - a0) + nb_t;
                for (int w = lane; 4 * w < span; w += 32) {
                    const int left = span - 4 * w;
                    cp_async4(dst0 + (uint32_t)(t * SB + 4 * w), reinterpret_cast<const void *>(a0 + 4ull * w),
                              left < 4 ? (uint32_t)left : 4u);
                }
            }
        }
    };

    // chunks c, c + 1 and c + 2 of the stream, as lane t < K describes them
    UnitInfo cur = info(lane < K ? lane : S);
    UnitInfo nx1 = info(lane < K ? K + lane : S);
    // quantise h: a pass of a warp takes four 32-value groups, eight lanes
    // per group and four consecutive values per lane (one 16-byte load);
    // warp w takes the passes w, w + 16, ..., eight of them with their loads
    // in flight together.  The scale is max|h| / 32767 of the group, so no
    // code leaves [-32767, 32767].
    {
        const int qg = lane >> 3, ql = lane & 7;
        const int npass = (NG + 3) / 4;
        for (int q0 = warp; q0 < npass; q0 += 8 * kDownWarps) {
            float4 v[8];
#pragma unroll
            for (int b = 0; b < 8; ++b) {
                const int grp = (q0 + b * kDownWarps) * 4 + qg;
                v[b] = grp < NG ? __ldcg(reinterpret_cast<const float4 *>(a.h + (size_t)grp * 32) + ql)
                                : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int b = 0; b < 8; ++b) {
                const int grp = (q0 + b * kDownWarps) * 4 + qg;
                float mx = fmaxf(fmaxf(fabsf(v[b].x), fabsf(v[b].y)), fmaxf(fabsf(v[b].z), fabsf(v[b].w)));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
                float s = (v[b].x + v[b].y) + (v[b].z + v[b].w);
                s += __shfl_xor_sync(0xffffffffu, s, 2);
                s += __shfl_xor_sync(0xffffffffu, s, 1);      // lanes 0-3: values 0-15, 4-7: 16-31
                const float s_hi = __shfl_down_sync(0xffffffffu, s, 4);
                if (grp < NG) {
                    const float inv = mx > 0.0f ? 32767.0f * __frcp_rn(mx) : 0.0f;
                    const int c0 = max(-32767, min(32767, __float2int_rn(v[b].x * inv)));
                    const int c1 = max(-32767, min(32767, __float2int_rn(v[b].y * inv)));
                    const int c2 = max(-32767, min(32767, __float2int_rn(v[b].z * inv)));
                    const int c3 = max(-32767, min(32767, __float2int_rn(v[b].w * inv)));
                    // byte 64 grp + 8 ql of the swizzled layout: line L, piece
                    // ((byte >> 4) & 7) ^ (L & 7)
                    const size_t byte = (size_t)grp * 64 + 8 * ql, line = byte >> 7;
                    const size_t at = (line << 7) | ((((byte >> 4) & 7) ^ (line & 7)) << 4) | (byte & 15);
                    *reinterpret_cast<uint2 *>(reinterpret_cast<uint8_t *>(hq) + at) =
                        make_uint2(((uint32_t)c0 & 0xFFFFu) | ((uint32_t)c1 << 16),
                                   ((uint32_t)c2 & 0xFFFFu) | ((uint32_t)c3 << 16));
                    if (ql == 0) {
                        hvs[grp] = mx * (1.0f / 32767.0f);
                        hs16[grp] = make_float2(s, s_hi);
                    }
                }
            }
        }
    }
    __syncthreads();
    // the first two chunks' copies go out once h is quantised (issued
    // earlier, they would hold up its loads)
    if (nch > 0) issue(cur, min(K, S), 0);
    cp_async_commit();
    if (nch > 1) issue(nx1, min(K, S - K), 1);
    cp_async_commit();
    const int g = lane >> 2, jp = lane & 3;
    float acc = 0.0f;
    int rrem = R;          // units left in the current output row
    int n_cur = n_first;   // the current output row
    for (int c = 0; c < nch; ++c) {
        const int kc = min(K, S - c * K);
        // every lane is done with chunk c - 1: its buffer takes chunk c + 2
        __syncwarp();
        const UnitInfo nx2 = info(lane < K ? (c + 2) * K + lane : S);
        if (c + 2 < nch) issue(nx2, min(K, S - (c + 2) * K), (c + 2) % kChunkBufs);
        cp_async_commit();
        if (bulk) {
            if (!mbar_wait(&bars[c % kChunkBufs], (uint32_t)((c / kChunkBufs) & 1), nullptr, a.err)) return;
        } else {
            cp_async_wait_ahead2();
        }
        __syncwarp();
        const uint8_t *cb = buf + (size_t)(c % kChunkBufs) * K * SB;
        // the value of this lane's part of unit g (weighted by its slot's weight)
        float v = 0.0f;
        {
            const int hb = __shfl_sync(0xffffffffu, cur.hb, g);
            const int lim = __shfl_sync(0xffffffffu, cur.lim, g);
            const int vi = __shfl_sync(0xffffffffu, cur.vi, g);
            const uint32_t off =
                (uint32_t)__shfl_sync(0xffffffffu, (uint32_t)reinterpret_cast<uintptr_t>(cur.src), g) &
                (bulk ? 15u : 3u);
            if (g < kc && 64 * jp < lim) {
                const int hi = hb + 64 * jp;
                v = wslot[vi] * dot64<F>(cb + (size_t)g * SB + off, jp,
                                         hq_s + 2u * (uint32_t)hi + ((uint32_t)(hi >> 6) & 7u) * 16u,
                                         *reinterpret_cast<const float2 *>(hvs + (hi >> 5)),
                                         *reinterpret_cast<const float4 *>(hs16 + (hi >> 5)));
            }
        }
        // add each unit's value to its output row; a row's sum is written
        // when its last unit has been added
        int g0 = 0;
        while (g0 < kc) {
            const int take = min(rrem, kc - g0);
            if (g >= g0 && g < g0 + take) acc += v;
            g0 += take;
            rrem -= take;
            if (rrem == 0) {
                float s = acc;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
                if (lane == 0) a.y[n_cur] = a.accumulate ? a.y[n_cur] + s : s;
                acc = 0.0f;
                rrem = R;
                n_cur += gw;
            }
        }
        cur = nx1;
        nx1 = nx2;
    }
}

cudaError_t launch_token_fmt(const MatvecArgs &a, int wd_fmt, cudaStream_t s) {
    if (a.T != 1 || !fmt_valid(wd_fmt) || wd_fmt == kFmtQ4_K || a.I % 64 != 0) return cudaErrorInvalidValue;
    const DeviceInfo &di = device_info();
    const size_t smem_a = gu_smem_total(a.H, a.I, a.k), smem_b = down_fmt_smem_bytes(wd_fmt, a.I, a.k);
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
