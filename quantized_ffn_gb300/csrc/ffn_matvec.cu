// ffn_matvec.cu -- the memory-bound path for one token: dense decode and the
// routed (mixture-of-experts) decode over the token's top_k experts.
//
// Two kernels in sequence, the second launched as a programmatic dependent
// of the first:
//   A (gate/up): for every (expert slot p, intermediate row i) owned by this
//            block, dot the W_gate and W_up rows with x (same input, one pass
//            over x: "fuse the same-input Q4_K matvec pairs", "Four
//            bottlenecks, one CUDA backend...", Bottleneck 3) and store
//            h[p][i] = silu(g) * u in fp32.  For one token the intermediate
//            is a few tens of KB that are consumed at once ("Fused SwiGLU
//            MLP...", FAQ "Does this affect decode?").
//   B (down): y[n] = sum_p w_p * Wd_{e_p}[n] . h[p] for the output rows of
//            this block.  Expert ids are read on the device ("Bottleneck 2").
// B's blocks start on the SMs that A's blocks leave; their reads of h wait
// (griddepcontrol) until A has completed, so the dependency is carried by the
// hardware's grid completion, not by a software grid barrier.  A is in turn a
// programmatic dependent of the work before it in the stream (typically the
// previous call's B): its blocks start as that work's blocks leave and wait
// for its completion before touching global memory, which takes the launch
// of A off the critical path of back-to-back calls.
//
// Data movement: every block of A first copies x into shared memory (a bulk
// copy that nothing else is queued behind: a weight stream started earlier
// delays these 8 KB by several microseconds).  Each warp then walks its rows
// on its own: its lane 0 copies the packed rows of the warp's next pass into
// one of the warp's two shared-memory slots (bulk copy, mbarrier) while the
// warp computes on the other.  No step synchronises more than one warp.  B
// reads h first and only then starts its own row copies, for the same reason.
//
// Arithmetic: the vector (x, later h) is stored in shared memory as int16 per
// 128-element half-block with one fp32 scale each (relative rounding error
// 2^-16 of the half-block's largest magnitude), plus the fp32 sum of every
// 32-element sub-block.  A sub-block's dot product is
//     d*sc * scale * sum(q * v_int) - dmin*m * sum(v)
// where sum(q * v_int) is exact in int32: the 4-bit codes are masked into
// int8 lanes (one LOP3 per four codes) and multiplied with int16 pairs by
// dp2a.  Each lane owns one half-block (128 weights) of a row at a time.
#include "zffn_internal.cuh"

namespace zffn {

constexpr int kDecWarps = 16;
constexpr int kDecThreads = kDecWarps * 32;
constexpr int kHalfBytes = 272;                         // 128 int16 + 16 pad

struct DecGeom {
    int P;            // expert slots of the token (dense: 1)
    int nbH, nbI;     // blocks per W_gate/W_up row, per W_down row
    int64_t rbH, rbI; // bytes per row
    int nhalf1, nhalf2;   // vector half-blocks of x and of h (all slots)
};

__host__ __device__ inline DecGeom dec_geom(int H, int I, int k) {
    DecGeom g;
    g.P = k;
    g.nbH = H / kQK;
    g.nbI = (I + kQK - 1) / kQK;
    g.rbH = (int64_t)g.nbH * kBlockBytes;
    g.rbI = (int64_t)g.nbI * kBlockBytes;
    g.nhalf1 = 2 * g.nbH;
    g.nhalf2 = g.P * 2 * g.nbI;
    return g;
}

// Shared memory of one block: the quantised vector (int16 half-blocks, their
// scales and sub-block sums).
__host__ __device__ inline size_t dec_smem_bytes(int nhalf) {
    return (size_t)nhalf * (kHalfBytes + 4 + 16);
}

// (defined below: shared memory of the gate/up and of the down kernel)
size_t gu_smem_total(int H, int I, int k);
size_t down_smem_total(int H, int I, int k);

size_t matvec_smem_bytes(int T, int H, int I, int k) {
    (void)T;
    const size_t sa = gu_smem_total(H, I, k), sb = down_smem_total(H, I, k);
    return sa > sb ? sa : sb;
}

struct DecVec {
    uint8_t *vec;
    float *vscale, *vsum;
};
__device__ __forceinline__ DecVec dec_vec(uint8_t *smem, int nhalf) {
    DecVec V;
    V.vec = smem;
    V.vscale = reinterpret_cast<float *>(smem + (size_t)nhalf * kHalfBytes);
    V.vsum = V.vscale + nhalf;
    return V;
}

// The 6-bit scales and mins of the four sub-blocks 4*hh .. 4*hh+3 of a
// block, one per byte: sub-block j < 4 keeps its scale and min in the low six
// bits of scale bytes j and 4+j; sub-block j >= 4 keeps their low four bits in
// the two nibbles of byte 4+j and their top two bits in the top bits of bytes
// j-4 and j.  hh is per lane, so both forms are computed and one is selected.
__device__ __forceinline__ void scales_mins4(const uint4 &hd, int hh, uint32_t &sc4, uint32_t &m4) {
    const uint32_t sc_lo = hd.y & 0x3F3F3F3Fu, m_lo = hd.z & 0x3F3F3F3Fu;
    const uint32_t sc_hi = (hd.w & 0x0F0F0F0Fu) | ((hd.y >> 2) & 0x30303030u);
    const uint32_t m_hi = ((hd.w >> 4) & 0x0F0F0F0Fu) | ((hd.z >> 2) & 0x30303030u);
    sc4 = hh ? sc_hi : sc_lo;
    m4 = hh ? m_hi : m_lo;
}

// Byte jj of v as a float, exactly: the byte becomes the low mantissa bits of
// 2^23 (one byte permute), then 2^23 is subtracted.
__device__ __forceinline__ float byte_to_float(uint32_t v, int jj) {
    const uint32_t f = __byte_perm(v, 0x4B000000u, 0x7650u + (uint32_t)jj);
    return __uint_as_float(f) - 8388608.0f;
}

// Integer part of the dot product of one half-block of codes (qv: the 64
// code bytes of half hh) with a quantised vector half-block in registers: the
// four sub-block sums of q * v_int (exact in int32).
__device__ __forceinline__ void half_block_isums(const uint4 (&qv4)[4], const uint4 (&xv)[16],
                                                 int (&acc)[4]) {
    int acc_a[4] = {0, 0, 0, 0}, acc_b[4] = {0, 0, 0, 0};
#pragma unroll
    for (int g = 0; g < 2; ++g) {            // the two 64-weight groups of the half
#pragma unroll
        for (int c = 0; c < 2; ++c) {        // 16 code bytes: weights 16c.. (low) and 32+16c.. (high)
            const uint4 qv = qv4[2 * g + c];
            const uint4 xlo0 = xv[8 * g + 2 * c], xlo1 = xv[8 * g + 2 * c + 1];
            const uint4 xhi0 = xv[8 * g + 4 + 2 * c], xhi1 = xv[8 * g + 4 + 2 * c + 1];
            const uint32_t qw[4] = {qv.x, qv.y, qv.z, qv.w};
            const uint32_t lo[8] = {xlo0.x, xlo0.y, xlo0.z, xlo0.w, xlo1.x, xlo1.y, xlo1.z, xlo1.w};
            const uint32_t hi[8] = {xhi0.x, xhi0.y, xhi0.z, xhi0.w, xhi1.x, xhi1.y, xhi1.z, xhi1.w};
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                const int ql = (int)(qw[w] & 0x0F0F0F0Fu);
                const int qh = (int)((qw[w] >> 4) & 0x0F0F0F0Fu);
                acc_a[2 * g] = __dp2a_lo((int)lo[2 * w], ql, acc_a[2 * g]);
                acc_b[2 * g] = __dp2a_hi((int)lo[2 * w + 1], ql, acc_b[2 * g]);
                acc_a[2 * g + 1] = __dp2a_lo((int)hi[2 * w], qh, acc_a[2 * g + 1]);
                acc_b[2 * g + 1] = __dp2a_hi((int)hi[2 * w + 1], qh, acc_b[2 * g + 1]);
            }
        }
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[j] = acc_a[j] + acc_b[j];
}

// Scale the sub-block sums: sum_j d*sc_j*vscale*isum_j - dmin*m_j*vsum_j.
__device__ __forceinline__ float half_block_scale(const uint4 &hd, int hh, const int (&acc)[4],
                                                  float vscale, const float (&vsum)[4]) {
    const float d = half_bits_to_float(hd.x), dmin = half_bits_to_float(hd.x >> 16);
    const float dv = d * vscale;
    uint32_t sc4, m4;
    scales_mins4(hd, hh, sc4, m4);
    float r = 0.0f, rm = 0.0f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        r = fmaf(byte_to_float(sc4, j), (float)acc[j], r);
        rm = fmaf(byte_to_float(m4, j), vsum[j], rm);
    }
    return fmaf(dv, r, -dmin * rm);
}

__device__ __forceinline__ void load_half(const DecVec &V, int hb, uint4 (&xv)[16], float &sc,
                                          float (&sm)[4]) {
    const uint4 *src = reinterpret_cast<const uint4 *>(V.vec + (size_t)hb * kHalfBytes);
#pragma unroll
    for (int i = 0; i < 16; ++i) xv[i] = src[i];
    sc = V.vscale[hb];
#pragma unroll
    for (int j = 0; j < 4; ++j) sm[j] = V.vsum[4 * hb + j];
}

// Quantise the half-blocks wi, wi + nw, wi + 2*nw, ... of a vector into V
// (warp wi of nw; each lane holds four values of a half-block): int16 values
// scaled by 32766 / max|v|, the half-block scale max|v| / 32766 and the fp32
// sum of every 32-element sub-block.  NT half-blocks are taken per round and
// computed without branches, so that their loads, shuffles and divisions
// overlap; only the stores are predicated.  load4(hb) returns this lane's
// four values of half-block hb.
template <int NT, class Load4>
__device__ __forceinline__ void quantize_vector(const DecVec &V, int nhalf, int wi, int nw, int lane,
                                                Load4 load4) {
    for (int b0 = wi; b0 < nhalf; b0 += NT * nw) {
        float4 v[NT];
        float m[NT], sm[NT];
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            const int hb = b0 + t * nw;
            v[t] = load4(hb < nhalf ? hb : b0);   // always a valid half-block
        }
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            m[t] = fmaxf(fmaxf(fabsf(v[t].x), fabsf(v[t].y)), fmaxf(fabsf(v[t].z), fabsf(v[t].w)));
            sm[t] = (v[t].x + v[t].y) + (v[t].z + v[t].w);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
#pragma unroll
            for (int t = 0; t < NT; ++t) m[t] = fmaxf(m[t], __shfl_xor_sync(0xffffffffu, m[t], o));
#pragma unroll
        for (int o = 4; o > 0; o >>= 1)
#pragma unroll
            for (int t = 0; t < NT; ++t) sm[t] += __shfl_xor_sync(0xffffffffu, sm[t], o);
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            const int hb = b0 + t * nw;
            const float inv = m[t] > 0.0f ? 32766.0f / m[t] : 0.0f;
            // round to nearest: |v * inv| <= 32766 < 2^22, so adding 1.5 * 2^23
            // leaves the rounded integer in the low mantissa bits
            const int q0 = __float_as_int(fmaf(v[t].x, inv, 12582912.0f)) - 0x4B400000;
            const int q1 = __float_as_int(fmaf(v[t].y, inv, 12582912.0f)) - 0x4B400000;
            const int q2 = __float_as_int(fmaf(v[t].z, inv, 12582912.0f)) - 0x4B400000;
            const int q3 = __float_as_int(fmaf(v[t].w, inv, 12582912.0f)) - 0x4B400000;
            if (hb < nhalf) {
                *reinterpret_cast<uint2 *>(V.vec + (size_t)hb * kHalfBytes + 8 * lane) =
                    make_uint2((uint32_t)(q0 & 0xFFFF) | ((uint32_t)q1 << 16),
                               (uint32_t)(q2 & 0xFFFF) | ((uint32_t)q3 << 16));
                if ((lane & 7) == 0) V.vsum[4 * hb + (lane >> 3)] = sm[t];
                if (lane == 0) V.vscale[hb] = m[t] > 0.0f ? m[t] / 32766.0f : 0.0f;
            }
        }
    }
}

// Half-block slots per row: the real count 2*nb rounded up to a power of two
// when it is at most 32, so that a warp holds 32 / slots whole rows.
__host__ __device__ inline int slots_per_row(int nb) {
    const int lr = 2 * nb;
    int lp = 1;
    while (lp < lr) lp <<= 1;
    return lp;
}

// Per-warp double buffer: slot bytes sized for the larger of a gate/up pass
// and a down row.
struct WarpRing {
    uint8_t *slot0, *slot1;
    uint64_t *bar0, *bar1;
    // selects rather than an indexed array, which would live in local memory
    __device__ __forceinline__ uint8_t *slot(int b) const { return b ? slot1 : slot0; }
    __device__ __forceinline__ uint64_t *bar(int b) const { return b ? bar1 : bar0; }
};
// The ring of warp w: its depth slots of slot_bytes each from slots, its two
// barriers from bars.  With depth 1 slot 1 aliases slot 0 and is unused.
__device__ __forceinline__ WarpRing warp_ring(uint8_t *slots, size_t slot_bytes, int depth, uint64_t *bars,
                                              int w) {
    WarpRing r;
    r.slot0 = slots + (size_t)w * depth * slot_bytes;
    r.slot1 = r.slot0 + (depth == 2 ? slot_bytes : 0);
    r.bar0 = bars + 2 * w;
    r.bar1 = bars + 2 * w + 1;
    return r;
}
__host__ __device__ inline int64_t dec_slot_bytes(const DecGeom &g, int Lp, bool down) {
    if (down) return (int64_t)g.P * g.rbI;
    const int rpc = Lp <= 32 ? 32 / Lp : 1;
    return 2 * (int64_t)rpc * g.rbH;
}

__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// ----------------------------------------------------------------------------
// A: gate and up rows -> h
// ----------------------------------------------------------------------------
// Shared memory: [x raw: bf16 (H*2), or with the RMSNorm folded in the fp32
// residual row and gamma (H*4 each) and 16 floats of reduction scratch] [x
// quantised (nhalf1 half-blocks)] [x bar] [per warp: 2 slot barriers, 2
// slots].
__host__ __device__ inline size_t gu_x_raw_bytes(int H, bool norm) {
    return ((size_t)H * (norm ? 8 : 2) + (norm ? 64 : 0) + 127) & ~(size_t)127;
}
__host__ __device__ inline size_t gu_smem_bytes(const DecGeom &g, int H, bool norm = false) {
    const int Lp = slots_per_row(g.nbH);
    const size_t slot = (size_t)((dec_slot_bytes(g, Lp, false) + 127) & ~(int64_t)127);
    size_t o = gu_x_raw_bytes(H, norm);
    o += (dec_smem_bytes(g.nhalf1) + 127) & ~(size_t)127;
    o += 8 + (size_t)kDecWarps * 2 * 8;
    o = (o + 127) & ~(size_t)127;
    o += (size_t)kDecWarps * 2 * slot;
    return o;
}

__global__ void __launch_bounds__(kDecThreads, 1) ffn_gu_kernel(MatvecArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    const DecGeom G = dec_geom(a.H, a.I, a.k);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int H = a.H, I = a.I, P = G.P;
    const bool moe = a.ids != nullptr;
    auto expert_of = [&](int p) -> int { return moe ? a.ids[p] : 0; };
    auto valid = [&](int e) -> bool { return e >= 0 && e < a.E; };
    const int64_t rows1 = (int64_t)P * I;
    const int r0 = (int)(rows1 * blockIdx.x / gridDim.x), r1 = (int)(rows1 * (blockIdx.x + 1) / gridDim.x);
    const int Lr = 2 * G.nbH;
    const int Lp = slots_per_row(G.nbH);

    // carve shared memory
    const bool norm = a.norm_in != nullptr;
    uint8_t *x_raw = smem;
    const float *gamma_s = reinterpret_cast<const float *>(smem + (size_t)H * 4);   // (norm only)
    float *norm_part = reinterpret_cast<float *>(smem + (size_t)H * 8);            // (norm only)
    size_t o = gu_x_raw_bytes(H, norm);
    const DecVec V = dec_vec(smem + o, G.nhalf1);
    o += (dec_smem_bytes(G.nhalf1) + 127) & ~(size_t)127;
    uint64_t *xbar = reinterpret_cast<uint64_t *>(smem + o);
    uint64_t *wbars = xbar + 1;
    o += 8 + (size_t)kDecWarps * 2 * 8;
    o = (o + 127) & ~(size_t)127;
    const size_t slot_bytes = (size_t)((dec_slot_bytes(G, Lp, false) + 127) & ~(int64_t)127);
    uint8_t *const slots = smem + o;
    const WarpRing ring = warp_ring(slots, slot_bytes, 2, wbars, warp);

    // the rows of a pass: rpc consecutive row pairs (Lr <= 32) or one
    const int rpc = Lr <= 32 ? 32 / Lp : 1;
    const int pass_stride = kDecWarps * rpc;
    // bytes of the pass starting at pair r (0: nothing to copy)
    auto pass_bytes = [&](int r) -> uint32_t {
        uint32_t bytes = 0;
        for (int t = 0; t < rpc && r + t < r1; ++t)
            if (valid(expert_of((r + t) / I))) bytes += 2 * (uint32_t)G.rbH;
        return bytes;
    };
    // copy the packed rows of the pass starting at pair r into slot b of rg
    auto issue = [&](const WarpRing &rg, int r, int b, uint32_t bytes) {
        mbar_arrive_expect_tx(rg.bar(b), bytes);
        for (int t = 0; t < rpc && r + t < r1; ++t) {
            const int p = (r + t) / I, i = (r + t) % I;
            const int e = expert_of(p);
            if (!valid(e)) continue;
            uint8_t *dst = rg.slot(b) + (size_t)t * 2 * G.rbH;
            bulk_g2s(dst, a.Wg + ((int64_t)e * I + i) * G.rbH, (uint32_t)G.rbH, rg.bar(b));
            bulk_g2s(dst + G.rbH, a.Wu + ((int64_t)e * I + i) * G.rbH, (uint32_t)G.rbH, rg.bar(b));
        }
    };
    const int first = r0 + warp * rpc;

    // This kernel may be launched as a programmatic dependent of the work
    // before it in the stream (the previous call's down kernel, say): its
    // blocks then start as that work's blocks leave, and wait here, before
    // touching global memory, until that work has completed.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (threadIdx.x == 0) {
        mbar_init(xbar, 1);
        for (int i = 0; i < 2 * kDecWarps; ++i) mbar_init(&wbars[i], 1);
        fence_mbarrier_init();
        const uint32_t xb = (uint32_t)(H * (norm ? 4 : 2));
        mbar_arrive_expect_tx(xbar, norm ? 2 * xb : xb);
        bulk_g2s(x_raw, norm ? static_cast<const void *>(a.norm_in) : static_cast<const void *>(a.x), xb, xbar);
        if (norm) bulk_g2s(x_raw + xb, a.gamma, xb, xbar);
    }
    __syncthreads();
    // the down-projection kernel may be scheduled as soon as SMs free up
    if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    // Each warp's first two passes, queued behind x.  A bulk copy stalls the
    // thread that issues it for a few hundred cycles whatever its size, so
    // every warp issues its own (in parallel) rather than one thread all.
    // bit b of pend: slot b holds a pass in flight; bit b of ph: its phase
    uint32_t pend = 0, ph = 0;
#pragma unroll
    for (int b = 0; b < 2; ++b) {
        const int r = first + b * pass_stride;
        const uint32_t bytes = r < r1 ? pass_bytes(r) : 0u;
        if (bytes && lane == 0) issue(ring, r, b, bytes);
        if (bytes) pend |= 1u << b;
    }
    __syncwarp();
    // quantise x (each warp its share of half-blocks)
    if (!mbar_wait(xbar, 0, nullptr, a.err)) return;
    if (norm) {
        // x = bf16(r * row * gamma), r = 1 / sqrt(mean(row^2) + eps), as the
        // RMSNorm kernel computes it (its reduction order aside)
        const float4 *row4 = reinterpret_cast<const float4 *>(x_raw);
        float ss = 0.0f;
        for (int i = threadIdx.x; i < H / 4; i += kDecThreads) {
            const float4 v = row4[i];
            ss = fmaf(v.x, v.x, ss);
            ss = fmaf(v.y, v.y, ss);
            ss = fmaf(v.z, v.z, ss);
            ss = fmaf(v.w, v.w, ss);
        }
#pragma unroll
        for (int o2 = 16; o2 > 0; o2 >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o2);
        if (lane == 0) norm_part[warp] = ss;
        __syncthreads();
        float tot = 0.0f;
#pragma unroll
        for (int w = 0; w < kDecWarps; ++w) tot += norm_part[w];
        const float r = rsqrtf(tot / (float)H + a.eps);
        const float4 *g4 = reinterpret_cast<const float4 *>(gamma_s);
        quantize_vector<4>(V, G.nhalf1, warp, kDecWarps, lane, [&](int hb) -> float4 {
            const float4 v = row4[hb * 32 + lane];
            const float4 g = g4[hb * 32 + lane];
            return make_float4(__bfloat162float(__float2bfloat16_rn(v.x * r * g.x)),
                               __bfloat162float(__float2bfloat16_rn(v.y * r * g.y)),
                               __bfloat162float(__float2bfloat16_rn(v.z * r * g.z)),
                               __bfloat162float(__float2bfloat16_rn(v.w * r * g.w)));
        });
    } else {
        quantize_vector<4>(V, G.nhalf1, warp, kDecWarps, lane, [&](int hb) -> float4 {
            const uint2 raw = *reinterpret_cast<const uint2 *>(x_raw + (size_t)(hb * 128 + 4 * lane) * 2);
            return make_float4(__uint_as_float(raw.x << 16), __uint_as_float(raw.x & 0xFFFF0000u),
                               __uint_as_float(raw.y << 16), __uint_as_float(raw.y & 0xFFFF0000u));
        });
    }
    __syncthreads();

    int lg = 0;
    while ((1 << lg) < Lp && (1 << lg) < 32) ++lg;
    const int q = Lr <= 32 ? (lane & (Lp - 1)) : lane;
    uint4 xr[16];
    float xs = 0.0f, xsum[4] = {0.f, 0.f, 0.f, 0.f};
    if (Lr <= 32 && q < Lr) load_half(V, q, xr, xs, xsum);

    int b = 0;
    for (int pp = first; pp < r1; pp += pass_stride, b ^= 1) {
        const bool have = (pend >> b) & 1;
        if (have && !mbar_wait(ring.bar(b), (ph >> b) & 1, nullptr, a.err)) return;
        if (have) ph ^= 1u << b;
        const uint8_t *slot = ring.slot(b);
        float g = 0.0f, u = 0.0f;
        int r;
        if (Lr <= 32) {
            const int t = lane >> lg;
            r = pp + t;
            if (have && r < r1 && q < Lr && valid(expert_of(r / I))) {
                const uint8_t *rowg = slot + (size_t)t * 2 * G.rbH + (size_t)(q >> 1) * kBlockBytes;
                const uint8_t *rowu = rowg + G.rbH;
                const uint4 hg = *reinterpret_cast<const uint4 *>(rowg);
                const uint4 hu = *reinterpret_cast<const uint4 *>(rowu);
                uint4 cg[4], cu[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    cg[i] = *reinterpret_cast<const uint4 *>(rowg + 16 + 64 * (q & 1) + 16 * i);
                    cu[i] = *reinterpret_cast<const uint4 *>(rowu + 16 + 64 * (q & 1) + 16 * i);
                }
                int ag[4], au[4];
                half_block_isums(cg, xr, ag);
                half_block_isums(cu, xr, au);
                g = half_block_scale(hg, q & 1, ag, xs, xsum);
                u = half_block_scale(hu, q & 1, au, xs, xsum);
            }
            for (int o2 = Lp >> 1; o2 > 0; o2 >>= 1) {
                g += __shfl_xor_sync(0xffffffffu, g, o2);
                u += __shfl_xor_sync(0xffffffffu, u, o2);
            }
        } else {
            r = pp;
            if (have && valid(expert_of(r / I))) {
                for (int qq = lane; qq < Lr; qq += 32) {
                    uint4 xv[16];
                    float vs, vsm[4];
                    load_half(V, qq, xv, vs, vsm);
                    const uint8_t *rowg = slot + (size_t)(qq >> 1) * kBlockBytes;
                    const uint8_t *rowu = rowg + G.rbH;
                    const uint4 hg = *reinterpret_cast<const uint4 *>(rowg);
                    const uint4 hu = *reinterpret_cast<const uint4 *>(rowu);
                    uint4 cg[4], cu[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        cg[i] = *reinterpret_cast<const uint4 *>(rowg + 16 + 64 * (qq & 1) + 16 * i);
                        cu[i] = *reinterpret_cast<const uint4 *>(rowu + 16 + 64 * (qq & 1) + 16 * i);
                    }
                    int ag[4], au[4];
                    half_block_isums(cg, xv, ag);
                    half_block_isums(cu, xv, au);
                    g += half_block_scale(hg, qq & 1, ag, vs, vsm);
                    u += half_block_scale(hu, qq & 1, au, vs, vsm);
                }
            }
#pragma unroll
            for (int o2 = 16; o2 > 0; o2 >>= 1) {
                g += __shfl_xor_sync(0xffffffffu, g, o2);
                u += __shfl_xor_sync(0xffffffffu, u, o2);
            }
        }
        // the slot is free once every lane has read it: refill it two passes on
        __syncwarp();
        {
            const int rn = pp + 2 * pass_stride;
            const uint32_t bytes = rn < r1 ? pass_bytes(rn) : 0u;
            if (bytes && lane == 0) issue(ring, rn, b, bytes);
            pend = (pend & ~(1u << b)) | (bytes ? 1u << b : 0u);
        }
        const bool writer = Lr <= 32 ? (q == 0 && r < r1) : lane == 0;
        if (writer) {
            const int p = r / I, i = r % I;
            a.h[(int64_t)p * I + i] = g / (1.0f + expf(-g)) * u;
        }
    }
}

// ----------------------------------------------------------------------------
// B: down rows, y = sum_p w_p * Wd_p . h_p
// ----------------------------------------------------------------------------
// Shared memory: [h quantised (nhalf2)] [per warp: 2 slot barriers] [per
// warp: 2 slots of one row of every expert slot].
__host__ __device__ inline size_t down_smem_bytes(const DecGeom &g, int depth) {
    const size_t slot = (size_t)((dec_slot_bytes(g, 0, true) + 127) & ~(int64_t)127);
    size_t o = (dec_smem_bytes(g.nhalf2) + 127) & ~(size_t)127;
    o += (size_t)kDecWarps * 2 * 8;
    o = (o + 127) & ~(size_t)127;
    o += (size_t)kDecWarps * depth * slot;
    return o;
}

__global__ void __launch_bounds__(kDecThreads, 1) ffn_down_kernel(MatvecArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    const DecGeom G = dec_geom(a.H, a.I, a.k);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int H = a.H, I = a.I, P = G.P;
    const bool moe = a.ids != nullptr;
    const int n0 = (int)((int64_t)H * blockIdx.x / gridDim.x), n1 = (int)((int64_t)H * (blockIdx.x + 1) / gridDim.x);

    const DecVec V = dec_vec(smem, G.nhalf2);
    size_t o = (dec_smem_bytes(G.nhalf2) + 127) & ~(size_t)127;
    uint64_t *wbars = reinterpret_cast<uint64_t *>(smem + o);
    o += (size_t)kDecWarps * 2 * 8;
    o = (o + 127) & ~(size_t)127;
    const size_t slot_bytes = (size_t)((dec_slot_bytes(G, 0, true) + 127) & ~(int64_t)127);
    uint8_t *const slots = smem + o;
    const int depth = a.ring_depth;
    const WarpRing ring = warp_ring(slots, slot_bytes, depth, wbars, warp);
    // bytes of a row: one W_down row per valid expert slot
    uint32_t row_bytes = 0;
    for (int p = 0; p < P; ++p) {
        const int e = moe ? a.ids[p] : 0;
        if (e >= 0 && e < a.E) row_bytes += (uint32_t)G.rbI;
    }
    // copy row n of every valid expert slot into slot b of rg
    auto issue = [&](const WarpRing &rg, int n, int b) {
        mbar_arrive_expect_tx(rg.bar(b), row_bytes);
        for (int p = 0; p < P; ++p) {
            const int e = moe ? a.ids[p] : 0;
            if (e < 0 || e >= a.E) continue;
            bulk_g2s(rg.slot(b) + (size_t)p * G.rbI, a.Wd + ((int64_t)e * H + n) * G.rbI, (uint32_t)G.rbI,
                     rg.bar(b));
        }
    };
    const int first = n0 + warp;
    if (threadIdx.x == 0) {
        for (int i = 0; i < 2 * kDecWarps; ++i) mbar_init(&wbars[i], 1);
        fence_mbarrier_init();
    }
    __syncthreads();
    // the next work in the stream (the next call's gate/up kernel, say) may
    // be scheduled as this kernel's blocks leave; it waits for this kernel's
    // completion itself
    if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    // W_down does not depend on the gate/up kernel: its rows are streamed
    // into L2 now, while the gate/up kernel finishes.  (Copies into shared
    // memory issued now would hold up the loads of h behind them.)  The rows
    // of one expert slot are contiguous: one request each.
    if (threadIdx.x == 0 && n1 > n0)
        for (int p = 0; p < P; ++p) {
            const int e = moe ? a.ids[p] : 0;
            if (e >= 0 && e < a.E)
                prefetch_l2_bulk(a.Wd + ((int64_t)e * H + n0) * G.rbI, (uint32_t)((n1 - n0) * G.rbI));
        }
    // h is written by the gate/up kernel: wait until that grid has completed
    // and its memory is visible
    asm volatile("griddepcontrol.wait;" ::: "memory");
    quantize_vector<8>(V, G.nhalf2, warp, kDecWarps, lane, [&](int hb) -> float4 {
        const int p = hb / (2 * G.nbI), hl = hb - p * (2 * G.nbI);
        const int col = hl * 128 + 4 * lane;
        // load from a valid address whatever the column, then zero past I
        const int colc = col < I ? col : 0;
        float4 v = __ldcg(reinterpret_cast<const float4 *>(a.h + (int64_t)p * I + colc));
        if (col >= I) v = make_float4(0.f, 0.f, 0.f, 0.f);
        return v;
    });
    // bit b of pend: slot b holds a row in flight; bit b of ph: its phase
    uint32_t pend = 0, ph = 0;
    for (int b = 0; b < depth; ++b) {
        const int n = first + b * kDecWarps;
        if (row_bytes && n < n1) {
            if (lane == 0) issue(ring, n, b);
            pend |= 1u << b;
        }
    }
    // a row's work items are its (slot p, half-block q) pairs
    const int Lr2 = 2 * G.nbI;
    const int items = P * Lr2;
    const int nrows = n1 - n0;
    // Every row of the block was asked for above when they fit the warps'
    // slots together: then each thread keeps one h half-block in registers
    // and runs it against several rows, so that the block reads h from
    // shared memory once instead of once per row; the warps' row sums are
    // added into y (zeroed here unless the call accumulates).
    const bool resident = row_bytes && nrows <= kDecWarps * depth;
    if (resident && !a.accumulate)
        for (int t = threadIdx.x; t < nrows; t += kDecThreads) a.y[n0 + t] = 0.0f;
    __syncthreads();
    if (resident) {
        const int WI = (items + 31) / 32;                   // warps covering the items once
        const int groups = WI <= kDecWarps ? kDecWarps / WI : 1;
        const int wi = WI <= kDecWarps ? warp % WI : warp;
        const int j = WI <= kDecWarps ? warp / WI : 0;      // this warp's rows: j, j + groups, ...
        const int stride = WI <= kDecWarps ? WI * 32 : kDecWarps * 32;
        if (j >= groups) return;
        for (int base = wi * 32; base < items; base += stride) {
            const int it = base + lane;
            const int p = it / Lr2, q = it - p * Lr2;
            const int e = it < items ? (moe ? a.ids[p] : 0) : -1;
            const bool iv = e >= 0 && e < a.E;
            uint4 xv[16];
            float xs = 0.0f, xsum[4] = {0.f, 0.f, 0.f, 0.f};
            if (iv) load_half(V, it, xv, xs, xsum);
            const float w = iv && moe ? (a.down_scale ? a.wts[p] * a.down_scale[e] : a.wts[p]) : 1.0f;
            for (int k = j; k < nrows; k += groups) {
                // row n0 + k went to slot k / kDecWarps of warp k % kDecWarps
                const int ow = k % kDecWarps, ob = k / kDecWarps;
                if (!mbar_wait(&wbars[2 * ow + ob], 0, nullptr, a.err)) return;
                float v = 0.0f;
                if (iv) {
                    const uint8_t *blk = slots + (size_t)(ow * depth + ob) * slot_bytes + (size_t)p * G.rbI +
                                         (size_t)(q >> 1) * kBlockBytes;
                    const uint4 hd = *reinterpret_cast<const uint4 *>(blk);
                    uint4 cq[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) cq[i] = *reinterpret_cast<const uint4 *>(blk + 16 + 64 * (q & 1) + 16 * i);
                    int ai[4];
                    half_block_isums(cq, xv, ai);
                    v = w * half_block_scale(hd, q & 1, ai, xs, xsum);
                }
#pragma unroll
                for (int o2 = 16; o2 > 0; o2 >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o2);
                if (lane == 0) atomicAdd(a.y + n0 + k, v);
            }
        }
        return;
    }

    // otherwise rows stream through the warps' slots: lanes take items lane,
    // lane + 32, ... of a row and the warp sums them
    int b = 0;
    for (int n = first; n < n1; n += kDecWarps, b = depth == 2 ? b ^ 1 : 0) {
        const bool have = (pend >> b) & 1;
        if (have && !mbar_wait(ring.bar(b), (ph >> b) & 1, nullptr, a.err)) return;
        if (have) ph ^= 1u << b;
        float acc = 0.0f;
        if (have) {
            for (int it = lane; it < items; it += 32) {
                const int p = it / Lr2, q = it - p * Lr2;
                const int e = moe ? a.ids[p] : 0;
                if (e < 0 || e >= a.E) continue;
                uint4 xv[16];
                float xs, xsum[4];
                load_half(V, it, xv, xs, xsum);
                const uint8_t *blk = ring.slot(b) + (size_t)p * G.rbI + (size_t)(q >> 1) * kBlockBytes;
                const uint4 hd = *reinterpret_cast<const uint4 *>(blk);
                uint4 cq[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) cq[i] = *reinterpret_cast<const uint4 *>(blk + 16 + 64 * (q & 1) + 16 * i);
                int ai[4];
                half_block_isums(cq, xv, ai);
                const float w = moe ? (a.down_scale ? a.wts[p] * a.down_scale[e] : a.wts[p]) : 1.0f;
                acc = fmaf(w, half_block_scale(hd, q & 1, ai, xs, xsum), acc);
            }
        }
        __syncwarp();
        {
            const int nn = n + depth * kDecWarps;
            const bool more = row_bytes && nn < n1;
            if (more && lane == 0) issue(ring, nn, b);
            pend = (pend & ~(1u << b)) | (more ? 1u << b : 0u);
        }
#pragma unroll
        for (int o2 = 16; o2 > 0; o2 >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o2);
        if (lane == 0) {
            float *dst = a.y + n;
            *dst = a.accumulate ? *dst + acc : acc;
        }
    }
}

// ----------------------------------------------------------------------------
// C: the routed single-token layer in one cooperative launch
// ----------------------------------------------------------------------------
// When every block's share of the token's expert weights fits in its shared
// memory (a routed layer's top_k experts: a few tens of MB for the whole
// GPU), one launch does both steps.  Every block first asks for all of its
// weights at once: x, its gate/up row pairs (in chunks of kTokChunkRows
// pairs, each on its own barrier) and its down rows of every chosen expert
// (bulk copies, one per contiguous range), so that the whole layer streams
// from HBM together and each warp starts as soon as its rows are in.  It then
// computes its h rows as in A, writes them to the workspace, meets the other
// blocks at a grid barrier, quantises all of h and computes its output rows
// as in B from the down rows already in shared memory.  The cooperative
// launch keeps every block resident, so the barrier's waits end; each is
// bounded all the same.
//
// Shared memory: [x raw bf16] [x quantised] [h quantised] [3 barriers, the
// slot table, a flag] [gate rows] [up rows] [down rows, slot-major], each region
// 128-byte aligned; the row regions are sized for the largest block share.
// Gate/up row pairs are copied and waited for in chunks of kTokChunkRows,
// each on its own barrier, so that a warp starts on its rows as soon as they
// have landed (at most kTokMaxChunks chunks per block).
constexpr int kTokChunkRows = 16, kTokMaxChunks = 16;
constexpr int kTokBars = 2 + kTokMaxChunks;   // x, down rows, gate/up chunks
__host__ __device__ inline int token_fused_rows1(const DecGeom &g, int I, int grid) {
    return (int)(((int64_t)g.P * I + grid - 1) / grid);
}
__host__ __device__ inline int token_fused_rows2(int H, int grid) { return (H + grid - 1) / grid; }
__host__ __device__ inline size_t token_fused_smem_bytes(const DecGeom &g, int H, int I, int grid) {
    size_t o = ((size_t)H * 2 + 127) & ~(size_t)127;
    o += (dec_smem_bytes(g.nhalf1) + 127) & ~(size_t)127;
    o += (dec_smem_bytes(g.nhalf2) + 127) & ~(size_t)127;
    o += kTokBars * 8 + 2 * 64 * 4 + 4;
    o = (o + 127) & ~(size_t)127;
    o += 2 * (size_t)token_fused_rows1(g, I, grid) * g.rbH;
    o = (o + 127) & ~(size_t)127;
    o += (size_t)g.P * token_fused_rows2(H, grid) * g.rbI;
    return o;
}

// One grid-wide barrier for the blocks of a cooperative launch, on a 64-bit
// arrival count in global memory (zero before the first use, never reset):
// the blocks of the n-th barrier on it arrive as counts n*nblocks ..
// (n+1)*nblocks - 1 and leave once the count has reached (n+1)*nblocks.
// Called by one thread of each block after the block's writes (ordered
// before it by a block barrier).  Bounded: on timeout the error word records
// ZFFN_ERR_TIMEOUT and false is returned.
__device__ __forceinline__ bool grid_barrier(unsigned long long *count, unsigned int nblocks, int *err) {
    __threadfence();
    const unsigned long long old = atomicAdd(count, 1ull);
    const unsigned long long target = (old / nblocks + 1) * nblocks;
    const long long t0 = clock64();
    for (;;) {
        unsigned long long v;
        asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(count) : "memory");
        if (v >= target) return true;
        if (clock64() - t0 > kWaitBudgetCycles) {
            record_error(err, ZFFN_ERR_TIMEOUT);
            return false;
        }
        __nanosleep(32);
    }
}

// Raise the transaction count of the current phase of bar (no arrival).
__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__global__ void __launch_bounds__(kDecThreads, 1) ffn_token_fused_kernel(MatvecArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    const DecGeom G = dec_geom(a.H, a.I, a.k);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int H = a.H, I = a.I, P = G.P;
    const int64_t rows1 = (int64_t)P * I;
    const int r0 = (int)(rows1 * blockIdx.x / gridDim.x), r1 = (int)(rows1 * (blockIdx.x + 1) / gridDim.x);
    const int n0 = (int)((int64_t)H * blockIdx.x / gridDim.x), n1 = (int)((int64_t)H * (blockIdx.x + 1) / gridDim.x);
    const int nr = r1 - r0, nd = n1 - n0;
    const int Lr = 2 * G.nbH, Lp = slots_per_row(G.nbH);

    // carve shared memory
    uint8_t *x_raw = smem;
    size_t o = ((size_t)H * 2 + 127) & ~(size_t)127;
    const DecVec V = dec_vec(smem + o, G.nhalf1);
    o += (dec_smem_bytes(G.nhalf1) + 127) & ~(size_t)127;
    const DecVec Vh = dec_vec(smem + o, G.nhalf2);
    o += (dec_smem_bytes(G.nhalf2) + 127) & ~(size_t)127;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + o);   // x, down rows, gate/up chunks
    int *s_e = reinterpret_cast<int *>(smem + o + kTokBars * 8);   // expert of slot p (or -1)
    float *s_w = reinterpret_cast<float *>(s_e + 64);          // its weight (routing * down scale)
    int *s_ok = reinterpret_cast<int *>(s_w + 64);             // the grid barrier's outcome
    o += kTokBars * 8 + 2 * 64 * 4 + 4;
    o = (o + 127) & ~(size_t)127;
    uint8_t *gu = smem + o;                                    // nr gate rows, then nr up rows
    o += 2 * (size_t)token_fused_rows1(G, I, gridDim.x) * G.rbH;
    o = (o + 127) & ~(size_t)127;
    uint8_t *dn = smem + o;                                    // [slot p][row n - n0]

    if (threadIdx.x == 0) {
        for (int i = 0; i < kTokBars; ++i) mbar_init(&bars[i], 1);
        fence_mbarrier_init();
    }
    __syncthreads();
    // every copy this block needs, issued by three warps in parallel
    if (warp == 0) {
        if (lane == 0) {
            mbar_arrive_expect_tx(&bars[0], (uint32_t)(H * 2));
            bulk_g2s(x_raw, a.x, (uint32_t)(H * 2), &bars[0]);
        }
    } else if (warp == 1) {
        // gate/up row pairs [r0, r1) in chunks of kTokChunkRows: lanes 2c and
        // 2c + 1 copy chunk c's rows of the (at most two) slots it touches,
        // one range of each matrix, counted on chunk c's barrier
        const int c = lane >> 1, part = lane & 1;
        const int cs = r0 + c * kTokChunkRows, ce = min(r1, cs + kTokChunkRows);
        int start = 0, end = 0, p = 0;
        if (cs < ce) {
            const int bound = (cs / I + 1) * I;   // the first slot boundary after cs
            start = part ? bound : cs;
            end = part ? ce : min(ce, bound);
            p = (part ? bound : cs) / I;
        }
        const int e = end > start ? a.ids[p] : -1;
        const bool ok = e >= 0 && e < a.E;
        const uint32_t bytes = ok ? (uint32_t)(2 * (int64_t)(end - start) * G.rbH) : 0u;
        if (bytes) mbar_expect_tx(&bars[2 + c], bytes);
        if (ok) {
            const int64_t row = (int64_t)e * I + (start - p * I);
            const uint32_t half = bytes / 2;
            bulk_g2s(gu + (size_t)(start - r0) * G.rbH, a.Wg + row * G.rbH, half, &bars[2 + c]);
            bulk_g2s(gu + (size_t)(nr + start - r0) * G.rbH, a.Wu + row * G.rbH, half, &bars[2 + c]);
        }
        __syncwarp();
        if (part == 0 && cs < ce) mbar_arrive(&bars[2 + c]);
    } else if (warp == 2) {
        // the slot table, and the bytes of the down rows [n0, n1) of every
        // valid slot (one range each, copied once this warp's part of step 1
        // is done: issued now, they would compete with the gate/up rows that
        // step 1 and the grid barrier wait for)
        uint32_t total = 0;
        for (int p = lane; p < P; p += 32) {
            const int e = a.ids[p];
            const bool ok = e >= 0 && e < a.E;
            s_e[p] = ok ? e : -1;
            float w = 0.0f;
            if (ok) {
                w = a.wts[p];
                if (a.down_scale) w *= a.down_scale[e];
            }
            s_w[p] = w;
            if (ok) total += (uint32_t)((int64_t)nd * G.rbI);
        }
#pragma unroll
        for (int s = 16; s > 0; s >>= 1) total += __shfl_xor_sync(0xffffffffu, total, s);
        if (lane == 0) mbar_arrive_expect_tx(&bars[1], total);
    }
    // quantise x
    if (!mbar_wait(&bars[0], 0, nullptr, a.err)) return;
    quantize_vector<4>(V, G.nhalf1, warp, kDecWarps, lane, [&](int hb) -> float4 {
        const uint2 raw = *reinterpret_cast<const uint2 *>(x_raw + (size_t)(hb * 128 + 4 * lane) * 2);
        return make_float4(__uint_as_float(raw.x << 16), __uint_as_float(raw.x & 0xFFFF0000u),
                           __uint_as_float(raw.y << 16), __uint_as_float(raw.y & 0xFFFF0000u));
    });
    __syncthreads();

    // step 1: h rows [r0, r1); the pairs of a pass as in the gate/up kernel
    // (kTokChunkRows is a multiple of a pass's pairs: one chunk per pass)
    {
        const int rpc = Lr <= 32 ? 32 / Lp : 1;
        int lg = 0;
        while ((1 << lg) < Lp && (1 << lg) < 32) ++lg;
        const int q = Lr <= 32 ? (lane & (Lp - 1)) : lane;
        uint4 xr[16];
        float xs = 0.0f, xsum[4] = {0.f, 0.f, 0.f, 0.f};
        if (Lr <= 32 && q < Lr) load_half(V, q, xr, xs, xsum);
        for (int t0 = warp * rpc; t0 < nr; t0 += kDecWarps * rpc) {
            if (!mbar_wait(&bars[2 + t0 / kTokChunkRows], 0, nullptr, a.err)) return;
            float g = 0.0f, u = 0.0f;
            int t;
            if (Lr <= 32) {
                t = t0 + (lane >> lg);
                if (t < nr && q < Lr && s_e[(r0 + t) / I] >= 0) {
                    const uint8_t *rowg = gu + (size_t)t * G.rbH + (size_t)(q >> 1) * kBlockBytes;
                    const uint8_t *rowu = rowg + (size_t)nr * G.rbH;
                    const uint4 hg = *reinterpret_cast<const uint4 *>(rowg);
                    const uint4 hu = *reinterpret_cast<const uint4 *>(rowu);
                    uint4 cg[4], cu[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        cg[i] = *reinterpret_cast<const uint4 *>(rowg + 16 + 64 * (q & 1) + 16 * i);
                        cu[i] = *reinterpret_cast<const uint4 *>(rowu + 16 + 64 * (q & 1) + 16 * i);
                    }
                    int ag[4], au[4];
                    half_block_isums(cg, xr, ag);
                    half_block_isums(cu, xr, au);
                    g = half_block_scale(hg, q & 1, ag, xs, xsum);
                    u = half_block_scale(hu, q & 1, au, xs, xsum);
                }
                for (int o2 = Lp >> 1; o2 > 0; o2 >>= 1) {
                    g += __shfl_xor_sync(0xffffffffu, g, o2);
                    u += __shfl_xor_sync(0xffffffffu, u, o2);
                }
            } else {
                t = t0;
                if (s_e[(r0 + t) / I] >= 0) {
                    for (int qq = lane; qq < Lr; qq += 32) {
                        uint4 xv[16];
                        float vs, vsm[4];
                        load_half(V, qq, xv, vs, vsm);
                        const uint8_t *rowg = gu + (size_t)t * G.rbH + (size_t)(qq >> 1) * kBlockBytes;
                        const uint8_t *rowu = rowg + (size_t)nr * G.rbH;
                        const uint4 hg = *reinterpret_cast<const uint4 *>(rowg);
                        const uint4 hu = *reinterpret_cast<const uint4 *>(rowu);
                        uint4 cg[4], cu[4];
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            cg[i] = *reinterpret_cast<const uint4 *>(rowg + 16 + 64 * (qq & 1) + 16 * i);
                            cu[i] = *reinterpret_cast<const uint4 *>(rowu + 16 + 64 * (qq & 1) + 16 * i);
                        }
                        int ag[4], au[4];
                        half_block_isums(cg, xv, ag);
                        half_block_isums(cu, xv, au);
                        g += half_block_scale(hg, qq & 1, ag, vs, vsm);
                        u += half_block_scale(hu, qq & 1, au, vs, vsm);
                    }
                }
#pragma unroll
                for (int o2 = 16; o2 > 0; o2 >>= 1) {
                    g += __shfl_xor_sync(0xffffffffu, g, o2);
                    u += __shfl_xor_sync(0xffffffffu, u, o2);
                }
            }
            const bool writer = Lr <= 32 ? (q == 0 && t < nr) : lane == 0;
            if (writer) {
                const int r = r0 + t;
                a.h[r] = g / (1.0f + expf(-g)) * u;   // h[p][i] at p * I + i = r
            }
        }
    }
    if (warp == 2 && nd > 0)
        for (int p = lane; p < P; p += 32) {
            const int e = s_e[p];
            if (e < 0) continue;
            bulk_g2s(dn + (size_t)p * nd * G.rbI, a.Wd + ((int64_t)e * H + n0) * G.rbI,
                     (uint32_t)((int64_t)nd * G.rbI), &bars[1]);
        }
    // every block's h rows (made visible by the barrier's fence), then all of h
    __syncthreads();
    if (threadIdx.x == 0) *s_ok = grid_barrier(a.gbar, gridDim.x, a.err) ? 1 : 0;
    __syncthreads();
    if (!*s_ok) return;
    quantize_vector<8>(Vh, G.nhalf2, warp, kDecWarps, lane, [&](int hb) -> float4 {
        const int p = hb / (2 * G.nbI), hl = hb - p * (2 * G.nbI);
        const int col = hl * 128 + 4 * lane;
        // load from a valid address whatever the column, then zero past I
        const int colc = col < I ? col : 0;
        float4 v = __ldcg(reinterpret_cast<const float4 *>(a.h + (int64_t)p * I + colc));
        if (col >= I) v = make_float4(0.f, 0.f, 0.f, 0.f);
        return v;
    });
    __syncthreads();

    // step 2: output rows [n0, n1) from the down rows in shared memory
    if (!mbar_wait(&bars[1], 0, nullptr, a.err)) return;
    const int Lr2 = 2 * G.nbI;
    const int items = P * Lr2;
    for (int n = n0 + warp; n < n1; n += kDecWarps) {
        float acc = 0.0f;
        for (int it = lane; it < items; it += 32) {
            const int p = it / Lr2, qh = it - p * Lr2;
            if (s_e[p] < 0) continue;
            uint4 xv[16];
            float xs, xsum[4];
            load_half(Vh, it, xv, xs, xsum);
            const uint8_t *blk = dn + ((size_t)p * nd + (n - n0)) * G.rbI + (size_t)(qh >> 1) * kBlockBytes;
            const uint4 hd = *reinterpret_cast<const uint4 *>(blk);
            uint4 cq[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) cq[i] = *reinterpret_cast<const uint4 *>(blk + 16 + 64 * (qh & 1) + 16 * i);
            int ai[4];
            half_block_isums(cq, xv, ai);
            acc = fmaf(s_w[p], half_block_scale(hd, qh & 1, ai, xs, xsum), acc);
        }
#pragma unroll
        for (int o2 = 16; o2 > 0; o2 >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o2);
        if (lane == 0) a.y[n] = a.accumulate ? a.y[n] + acc : acc;
    }
}

size_t gu_smem_total(int H, int I, int k) { return gu_smem_bytes(dec_geom(H, I, k), H); }
size_t matvec_smem_bytes_prenorm(int H, int I) {
    const size_t sa = gu_smem_bytes(dec_geom(H, I, 1), H, true), sb = down_smem_total(H, I, 1);
    return sa > sb ? sa : sb;
}
// The down kernel double-buffers its rows when that fits a block's shared
// memory, else it single-buffers (long rows).
int down_ring_depth(int H, int I, int k) {
    return down_smem_bytes(dec_geom(H, I, k), 2) <= (size_t)device_info().max_smem_optin ? 2 : 1;
}
size_t down_smem_total(int H, int I, int k) {
    return down_smem_bytes(dec_geom(H, I, k), down_ring_depth(H, I, k));
}

// The one-launch routed path applies when its barrier words are given and
// every block's share of the weights fits in its shared memory.
bool token_fused_fits_dims(int H, int I, int k) {
    if (k > 64) return false;
    const DeviceInfo &di = device_info();
    const DecGeom G = dec_geom(H, I, k);
    const int grid = di.num_sms;
    // a block's gate/up pairs: at most kTokMaxChunks chunks, each touching at
    // most two slots
    if (token_fused_rows1(G, I, grid) > kTokChunkRows * kTokMaxChunks || I < kTokChunkRows) return false;
    return token_fused_smem_bytes(G, H, I, grid) <= (size_t)di.max_smem_optin;
}
bool token_fused_fits(const MatvecArgs &a) {
    return a.T == 1 && a.ids && a.gbar && token_fused_fits_dims(a.H, a.I, a.k);
}

cudaError_t launch_ffn_matvec(const MatvecArgs &a, cudaStream_t s) {
    const DeviceInfo &di = device_info();
    if (a.T != 1) return cudaErrorInvalidValue;
    const DecGeom G = dec_geom(a.H, a.I, a.k);
    if (token_fused_fits(a)) {
        const size_t smem = token_fused_smem_bytes(G, a.H, a.I, di.num_sms);
        cudaError_t e = ensure_dynamic_smem((const void *)ffn_token_fused_kernel, smem);
        if (e != cudaSuccess) return e;
        MatvecArgs args = a;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(di.num_sms);   // one block per SM, all resident
        cfg.blockDim = dim3(kDecThreads);
        cfg.stream = s;
        cfg.dynamicSmemBytes = smem;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeCooperative;
        attr[0].val.cooperative = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        return cudaLaunchKernelEx(&cfg, ffn_token_fused_kernel, args);
    }
    const int depth = down_ring_depth(a.H, a.I, a.k);
    const size_t smem_a = gu_smem_bytes(G, a.H, a.norm_in != nullptr), smem_b = down_smem_bytes(G, depth);
    cudaError_t e = ensure_dynamic_smem((const void *)ffn_gu_kernel, smem_a);
    if (e == cudaSuccess) e = ensure_dynamic_smem((const void *)ffn_down_kernel, smem_b);
    if (e != cudaSuccess) return e;
    MatvecArgs args = a;
    args.ring_depth = depth;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(di.num_sms);   // one block per SM
    cfg.blockDim = dim3(kDecThreads);
    cfg.stream = s;
    cfg.dynamicSmemBytes = smem_a;
    // both kernels are programmatic dependents of what precedes them: the
    // gate/up kernel of the stream's previous work, the down kernel of the
    // gate/up kernel
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, ffn_gu_kernel, args);
    if (e != cudaSuccess) return e;
    cfg.dynamicSmemBytes = smem_b;
    return cudaLaunchKernelEx(&cfg, ffn_down_kernel, args);
}

}  // namespace zffn
