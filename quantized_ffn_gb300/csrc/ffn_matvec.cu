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
// B's blocks start on the SMs that A's blocks leave and stream their W_down
// rows into shared memory at once; only the reads of h wait (griddepcontrol)
// until A has completed.  The dependency between the two halves is thus
// carried by the hardware's grid completion, not by a software grid barrier
// polled over global memory.
//
// Data movement: one producer warp per block streams the packed weight rows
// into a ring of shared-memory stages with bulk asynchronous copies.  In A it
// starts once the consumers hold x, so that the small vector load does not
// queue behind the weight stream.  Consumer warps unpack from shared memory.
//
// Arithmetic: the vector (x, later h) is stored in shared memory as int16 per
// 128-element half-block with one fp32 scale each (relative rounding error
// 2^-16 of the half-block's largest magnitude), plus the fp32 sum of every
// 32-element sub-block.  A sub-block's dot product is
//     d*sc * scale * sum(q * v_int) - dmin*m * sum(v)
// where sum(q * v_int) is exact in int32: the 4-bit codes are masked into
// int8 lanes (one LOP3 per four codes) and multiplied with int16 pairs by
// dp2a.  Each lane owns one half-block (128 weights) of one row.
#include "zffn_internal.cuh"

namespace zffn {

constexpr int kMvConsumerWarps = 12;
constexpr int kMvConsumers = kMvConsumerWarps * 32;
constexpr int kMvThreads = kMvConsumers + 32;          // + producer warp
constexpr int kMvStages = 3;
constexpr int kMvStageBytes = 55296;                   // 54 KB, multiple of 16
constexpr int kMvMaxRows = 64;                          // rows per stage cap
constexpr int kHalfBytes = 272;                         // 128 int16 + 16 pad

struct MvGeom {
    int P;            // expert slots of the token (dense: 1)
    int nbH, nbI;     // blocks per W_gate/W_up row, per W_down row
    int64_t rbH, rbI; // bytes per row
    int R1, R2;       // rows per stage in phase 1 (row pairs) and phase 2
    int nhalf1, nhalf2;   // vector half-blocks in phase 1 and phase 2
};

// Half-block slots reserved per row: the real count 2*nb rounded up to a
// power of two (<= 32) or to a multiple of 32, so that rows never straddle
// a 32-lane chunk unevenly.
__host__ __device__ inline int slots_per_row(int nb) {
    const int lr = 2 * nb;
    if (lr > 32) return (lr + 31) & ~31;
    int lp = 1;
    while (lp < lr) lp <<= 1;
    return lp;
}

// Rows per stage: as many as fit (at most kMvMaxRows), trimmed so that the
// stage's 32-lane chunks split evenly over the consumer warps when that
// costs at most a quarter of the rows.
__host__ __device__ inline int rows_per_stage(int64_t bytes_per_row, int nmat, int nb) {
    int r = (int)(kMvStageBytes / bytes_per_row);
    if (r > kMvMaxRows) r = kMvMaxRows;
    const int lp = slots_per_row(nb);
    for (int t = r; t >= 1 && 4 * t >= 3 * r; --t) {
        const int chunks = (nmat * t * lp + 31) / 32;
        if (chunks % kMvConsumerWarps == 0) return t;
    }
    return r;
}

__host__ __device__ inline MvGeom mv_geom(int H, int I, int k) {
    MvGeom g;
    g.P = k;
    g.nbH = H / kQK;
    g.nbI = (I + kQK - 1) / kQK;
    g.rbH = (int64_t)g.nbH * kBlockBytes;
    g.rbI = (int64_t)g.nbI * kBlockBytes;
    g.R1 = rows_per_stage(2 * g.rbH, 2, g.nbH);
    g.R2 = rows_per_stage(g.rbI, 1, g.nbI);
    g.nhalf1 = 2 * g.nbH;
    g.nhalf2 = g.P * 2 * g.nbI;
    return g;
}

struct MvSmem {
    size_t ring, vec, vscale, vsum, acc, yacc, bars, total;
};

__host__ __device__ inline MvSmem mv_smem_layout(const MvGeom &g) {
    MvSmem L;
    size_t o = 0;
    const int nh = g.nhalf1 > g.nhalf2 ? g.nhalf1 : g.nhalf2;
    L.ring = o; o += (size_t)kMvStages * kMvStageBytes;
    L.vec = o; o += (size_t)nh * kHalfBytes;
    L.vscale = o; o += (size_t)nh * 4;
    L.vsum = o; o += (size_t)nh * 4 * 4;
    L.acc = o; o += 2 * kMvMaxRows * 4;
    L.yacc = o; o += kMvMaxRows * 4;
    o = (o + 15) & ~(size_t)15;
    L.bars = o; o += (2 * kMvStages + 1) * 8;
    L.total = o;
    return L;
}

size_t matvec_smem_bytes(int T, int H, int I, int k) {
    (void)T;
    const MvGeom g = mv_geom(H, I, k);
    if (g.R1 < 1 || g.R2 < 1) return (size_t)1 << 30;   // a row does not fit a stage
    return mv_smem_layout(g).total;
}

__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void consumers_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(kMvConsumers) : "memory");
}

// Quantise one 128-element half-block of a vector (one warp, 4 values per
// lane): int16 values, the half-block scale and the four sub-block sums.
__device__ __forceinline__ void quantize_half(const float4 v4, int lane, uint8_t *vec_hb,
                                              float *scale, float *sums) {
    const float v[4] = {v4.x, v4.y, v4.z, v4.w};
    float m = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    const float inv = m > 0.0f ? 32766.0f / m : 0.0f;
    int q[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) q[j] = __float2int_rn(v[j] * inv);
    const uint32_t w0 = (uint32_t)(q[0] & 0xFFFF) | ((uint32_t)q[1] << 16);
    const uint32_t w1 = (uint32_t)(q[2] & 0xFFFF) | ((uint32_t)q[3] << 16);
    *reinterpret_cast<uint2 *>(vec_hb + 8 * lane) = make_uint2(w0, w1);
    float s = (v[0] + v[1]) + (v[2] + v[3]);
#pragma unroll
    for (int o = 4; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if ((lane & 7) == 0) sums[lane >> 3] = s;
    if (lane == 0) *scale = m > 0.0f ? m / 32766.0f : 0.0f;
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

// Integer part of the dot product of one half-block of packed codes (half hh
// of the block at blk) with a quantised vector half-block in registers: the
// four sub-block sums of q * v_int (exact in int32).
__device__ __forceinline__ void half_block_isums(const uint8_t *blk, int hh, const uint4 (&xv)[16],
                                                 int (&acc)[4]) {
    const uint4 *qs = reinterpret_cast<const uint4 *>(blk + 16 + 64 * hh);
    int acc_a[4] = {0, 0, 0, 0}, acc_b[4] = {0, 0, 0, 0};
#pragma unroll
    for (int g = 0; g < 2; ++g) {            // the two 64-weight groups of the half
#pragma unroll
        for (int c = 0; c < 2; ++c) {        // 16 code bytes: weights 16c.. (low) and 32+16c.. (high)
            const uint4 qv = qs[2 * g + c];
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

// Dot product of one half-block of packed weights (header at blk, codes of
// half hh) with a quantised vector half-block held in registers (xv: 128
// int16), its scale and its four sub-block sums.
__device__ __forceinline__ float half_block_dot(const uint8_t *blk, int hh, const uint4 (&xv)[16],
                                                float vscale, const float (&vsum)[4]) {
    const uint4 hd = *reinterpret_cast<const uint4 *>(blk);
    int acc[4];
    half_block_isums(blk, hh, xv, acc);
    return half_block_scale(hd, hh, acc, vscale, vsum);
}

// Two rows at once (same half-block slot): independent work for the
// scheduler to interleave.
__device__ __forceinline__ void half_block_dot2(const uint8_t *blk0, const uint8_t *blk1, int hh,
                                                const uint4 (&xv)[16], float vscale,
                                                const float (&vsum)[4], float &r0, float &r1) {
    const uint4 hd0 = *reinterpret_cast<const uint4 *>(blk0);
    const uint4 hd1 = *reinterpret_cast<const uint4 *>(blk1);
    int acc0[4], acc1[4];
    half_block_isums(blk0, hh, xv, acc0);
    half_block_isums(blk1, hh, xv, acc1);
    r0 = half_block_scale(hd0, hh, acc0, vscale, vsum);
    r1 = half_block_scale(hd1, hh, acc1, vscale, vsum);
}

__device__ __forceinline__ void load_half(const uint8_t *vec, const float *vscale,
                                          const float *vsum, int hb, uint4 (&xv)[16], float &sc,
                                          float (&sm)[4]) {
    const uint4 *src = reinterpret_cast<const uint4 *>(vec + (size_t)hb * kHalfBytes);
#pragma unroll
    for (int i = 0; i < 16; ++i) xv[i] = src[i];
    sc = vscale[hb];
#pragma unroll
    for (int j = 0; j < 4; ++j) sm[j] = vsum[4 * hb + j];
}

// A lane keeps one vector half-block in registers when it always owns the
// same slot of a row: rows of at most 32 slots (slot = lane mod slots), or
// rows of several 32-slot chunks when the consumer warps split evenly into
// one class per chunk position.
__device__ __forceinline__ bool slot_resident(int Lp) {
    return Lp <= 32 || kMvConsumerWarps % (Lp >> 5) == 0;
}
__device__ __forceinline__ int lane_slot(int Lp, int warp, int lane) {
    return Lp <= 32 ? (lane & (Lp - 1)) : (warp % (Lp >> 5)) * 32 + lane;
}

// Shared-memory views of one block.
struct MvShared {
    uint8_t *ring, *vec;
    float *vscale, *vsum, *acc, *yacc;
    uint64_t *full, *empty, *xready;
};
__device__ __forceinline__ MvShared mv_shared(uint8_t *smem, const MvSmem &L) {
    MvShared S;
    S.ring = smem + L.ring;
    S.vec = smem + L.vec;
    S.vscale = reinterpret_cast<float *>(smem + L.vscale);
    S.vsum = reinterpret_cast<float *>(smem + L.vsum);
    S.acc = reinterpret_cast<float *>(smem + L.acc);      // [2][kMvMaxRows]
    S.yacc = reinterpret_cast<float *>(smem + L.yacc);    // [kMvMaxRows]
    S.full = reinterpret_cast<uint64_t *>(smem + L.bars);
    S.empty = S.full + kMvStages;
    S.xready = S.empty + kMvStages;
    return S;
}

// Quantise nhalf vector half-blocks into S; load4(hb) returns this lane's four
// values of half-block hb.  A warp issues the loads of up to 8 of its
// half-blocks before using any, so the vector arrives in one round trip.
template <class Load4>
__device__ __forceinline__ void quantize_vector(const MvShared &S, int nhalf, int warp, int lane,
                                                Load4 load4) {
    for (int b0 = warp; b0 < nhalf; b0 += 8 * kMvConsumerWarps) {
        float4 v[8];
#pragma unroll
        for (int t = 0; t < 8; ++t) {
            const int hb = b0 + t * kMvConsumerWarps;
            v[t] = load4(hb < nhalf ? hb : b0);   // always a valid half-block: no branch
        }
#pragma unroll
        for (int t = 0; t < 8; ++t) {
            const int hb = b0 + t * kMvConsumerWarps;
            if (hb < nhalf)
                quantize_half(v[t], lane, S.vec + (size_t)hb * kHalfBytes, S.vscale + hb, S.vsum + 4 * hb);
        }
    }
}

// The consumer side's copy of one vector half-block kept in registers.
struct VecReg {
    uint4 xr[16];
    float xs = 0.0f, xsum[4] = {0.f, 0.f, 0.f, 0.f};
};

// Load this lane's resident half-block of the vector starting at vec_base.
__device__ __forceinline__ void load_resident(const MvShared &S, VecReg &R, int nb, int vec_base,
                                              int warp, int lane) {
    const int Lp = slots_per_row(nb);
    if (!slot_resident(Lp)) return;
    const int q = lane_slot(Lp, warp, lane);
    if (q < 2 * nb) load_half(S.vec, S.vscale, S.vsum, vec_base + q, R.xr, R.xs, R.xsum);
}

// Process one stage: nmat matrices of nrows rows with nb blocks each; each
// row's dot product with the vector half-blocks starting at vec_base lands in
// acc[mat][row].  Rows hold slots_per_row(nb) slots (half-blocks, the real
// ones first).  With a resident vector the lane's half-block is already in R.
__device__ __forceinline__ void process_stage(const MvShared &S, const uint8_t *base, const VecReg &R,
                                              int nmat, int nrows, int nb, int64_t rb, int vec_base,
                                              int warp, int lane) {
    const int Lr = 2 * nb;
    const int Lp = slots_per_row(nb);
    const int nrg = nmat * nrows;
    auto write = [&](int rowg, float v, bool add) {
        const int mat = rowg >= nrows;
        float *dst = &S.acc[mat * kMvMaxRows + rowg - mat * nrows];
        if (add) atomicAdd(dst, v); else *dst = v;
    };
    if (Lp <= 32) {
        int lg = 0;
        while ((1 << lg) < Lp) ++lg;
        const int rpc = 32 >> lg;                     // rows per chunk
        const int chunks = (nrg + rpc - 1) / rpc;
        const int q = lane & (Lp - 1);
        // two chunks per pass (c and c + kMvConsumerWarps) for instruction-level parallelism
        for (int c = warp; c < chunks; c += 2 * kMvConsumerWarps) {
            const int c2 = c + kMvConsumerWarps;
            const int rowg = c * rpc + (lane >> lg), rowg2 = c2 * rpc + (lane >> lg);
            const bool v1 = rowg < nrg && q < Lr, v2 = c2 < chunks && rowg2 < nrg && q < Lr;
            float part = 0.0f, part2 = 0.0f;
            const int64_t off = (q >> 1) * kBlockBytes;
            if (v1 && v2)
                half_block_dot2(base + (int64_t)rowg * rb + off, base + (int64_t)rowg2 * rb + off, q & 1,
                                R.xr, R.xs, R.xsum, part, part2);
            else if (v1)
                part = half_block_dot(base + (int64_t)rowg * rb + off, q & 1, R.xr, R.xs, R.xsum);
            for (int o = Lp >> 1; o > 0; o >>= 1) {
                part += __shfl_xor_sync(0xffffffffu, part, o);
                part2 += __shfl_xor_sync(0xffffffffu, part2, o);
            }
            if (rowg < nrg && q == 0) write(rowg, part, false);
            if (c2 < chunks && rowg2 < nrg && q == 0) write(rowg2, part2, false);
        }
    } else if (slot_resident(Lp)) {
        const int cpr = Lp >> 5;
        const int q = lane_slot(Lp, warp, lane);
        const int rstep = kMvConsumerWarps / cpr;
        for (int rowg = warp / cpr; rowg < nrg; rowg += 2 * rstep) {
            const int rowg2 = rowg + rstep;
            float part = 0.0f, part2 = 0.0f;
            const int64_t off = (q >> 1) * kBlockBytes;
            if (q < Lr) {
                if (rowg2 < nrg)
                    half_block_dot2(base + (int64_t)rowg * rb + off, base + (int64_t)rowg2 * rb + off, q & 1,
                                    R.xr, R.xs, R.xsum, part, part2);
                else
                    part = half_block_dot(base + (int64_t)rowg * rb + off, q & 1, R.xr, R.xs, R.xsum);
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                part += __shfl_xor_sync(0xffffffffu, part, o);
                part2 += __shfl_xor_sync(0xffffffffu, part2, o);
            }
            if (lane == 0) {
                write(rowg, part, true);
                if (rowg2 < nrg) write(rowg2, part2, true);
            }
        }
    } else {
        const int cpr = Lp >> 5;
        for (int c = warp; c < nrg * cpr; c += kMvConsumerWarps) {
            const int rowg = c / cpr;
            const int q = (c - rowg * cpr) * 32 + lane;
            float part = 0.0f;
            if (q < Lr) {
                uint4 xv[16];
                float sc, sm[4];
                load_half(S.vec, S.vscale, S.vsum, vec_base + q, xv, sc, sm);
                part = half_block_dot(base + (int64_t)rowg * rb + (q >> 1) * kBlockBytes, q & 1, xv, sc, sm);
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
            if (lane == 0) write(rowg, part, true);
        }
    }
}

__device__ __forceinline__ void init_ring(const MvShared &S) {
    if (threadIdx.x == 0) {
        for (int st = 0; st < kMvStages; ++st) {
            mbar_init(&S.full[st], 1);
            mbar_init(&S.empty[st], 1);
        }
        mbar_init(S.xready, kMvConsumerWarps);
        fence_mbarrier_init();
    }
    __syncthreads();
}

// The producer waits (bounded) until the consumers released every stage,
// i.e. until every copy it issued has landed and been read.
__device__ __forceinline__ void drain_ring(const MvShared &S, uint32_t slot, uint32_t ph, int *err) {
    for (int st = 0; st < kMvStages; ++st) {
        mbar_wait(&S.empty[slot], ph ^ 1, nullptr, err, kWaitBudgetCycles / 8);
        if (++slot == kMvStages) { slot = 0; ph ^= 1; }
    }
}

// ----------------------------------------------------------------------------
// A: gate and up rows -> h
// ----------------------------------------------------------------------------
__global__ void __launch_bounds__(kMvThreads, 1) ffn_gu_kernel(MatvecArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    const MvGeom G = mv_geom(a.H, a.I, a.k);
    const MvShared S = mv_shared(smem, mv_smem_layout(G));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int I = a.I, P = G.P;
    const bool moe = a.ids != nullptr;
    auto expert_of = [&](int p) -> int { return moe ? a.ids[p] : 0; };
    auto valid = [&](int e) -> bool { return e >= 0 && e < a.E; };
    const int64_t rows1 = (int64_t)P * I;
    const int r0 = (int)(rows1 * blockIdx.x / gridDim.x), r1 = (int)(rows1 * (blockIdx.x + 1) / gridDim.x);

    init_ring(S);
    // the down-projection kernel may be scheduled as soon as SMs free up
    if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    if (warp == kMvConsumerWarps) {
        // ------------------------- producer -------------------------------
        if (lane == 0) {
            uint32_t slot = 0, ph = 0;
            bool ok = mbar_wait(S.xready, 0, nullptr, a.err);
            // stages: chunks of up to R1 rows within one slot p
            for (int r = r0; r < r1 && ok;) {
                const int p = r / I, i = r % I;
                const int cnt = min(min(G.R1, r1 - r), I - i);
                const int e = expert_of(p);
                if (valid(e)) {
                    if (!mbar_wait(&S.empty[slot], ph ^ 1, nullptr, a.err)) { ok = false; break; }
                    const uint32_t bytes = (uint32_t)(cnt * G.rbH);
                    mbar_arrive_expect_tx(&S.full[slot], 2 * bytes);
                    uint8_t *dst = S.ring + slot * kMvStageBytes;
                    bulk_g2s(dst, a.Wg + ((int64_t)e * I + i) * G.rbH, bytes, &S.full[slot]);
                    bulk_g2s(dst + bytes, a.Wu + ((int64_t)e * I + i) * G.rbH, bytes, &S.full[slot]);
                    if (++slot == kMvStages) { slot = 0; ph ^= 1; }
                }
                r += cnt;
            }
            drain_ring(S, slot, ph, a.err);
        }
        return;
    }

    // ----------------------------- consumers ---------------------------------
    const int tid = threadIdx.x;
    uint32_t slot = 0, ph = 0;
    bool ok = true;
    for (int t = tid; t < 3 * kMvMaxRows; t += kMvConsumers) S.acc[t] = 0.0f;   // acc and yacc
    quantize_vector(S, G.nhalf1, warp, lane, [&](int hb) -> float4 {
        const uint2 raw = *reinterpret_cast<const uint2 *>(a.x + hb * 128 + 4 * lane);
        return make_float4(__uint_as_float(raw.x << 16), __uint_as_float(raw.x & 0xFFFF0000u),
                           __uint_as_float(raw.y << 16), __uint_as_float(raw.y & 0xFFFF0000u));
    });
    // x is in: the weight stream may start now
    __syncwarp();
    if (lane == 0) mbar_arrive(S.xready);
    consumers_sync();
    VecReg R;
    load_resident(S, R, G.nbH, 0, warp, lane);
    for (int r = r0; r < r1 && ok;) {
        const int p = r / I, i = r % I;
        const int cnt = min(min(G.R1, r1 - r), I - i);
        const int e = expert_of(p);
        if (!valid(e)) {
            for (int t = tid; t < cnt; t += kMvConsumers) a.h[(int64_t)p * I + i + t] = 0.0f;
            r += cnt;
            continue;
        }
        if (!mbar_wait(&S.full[slot], ph, nullptr, a.err)) { ok = false; break; }
        process_stage(S, S.ring + slot * kMvStageBytes, R, 2, cnt, G.nbH, G.rbH, 0, warp, lane);
        consumers_sync();
        if (tid == 0) mbar_arrive(&S.empty[slot]);
        if (++slot == kMvStages) { slot = 0; ph ^= 1; }
        if (tid < cnt) {
            const float g = S.acc[tid], u = S.acc[kMvMaxRows + tid];
            a.h[(int64_t)p * I + i + tid] = g / (1.0f + expf(-g)) * u;
            S.acc[tid] = 0.0f;
            S.acc[kMvMaxRows + tid] = 0.0f;
        }
        consumers_sync();
        r += cnt;
    }
}

// ----------------------------------------------------------------------------
// B: down rows, y = sum_p w_p * Wd_p . h_p
// ----------------------------------------------------------------------------
__global__ void __launch_bounds__(kMvThreads, 1) ffn_down_kernel(MatvecArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    const MvGeom G = mv_geom(a.H, a.I, a.k);
    const MvShared S = mv_shared(smem, mv_smem_layout(G));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int H = a.H, I = a.I, P = G.P;
    const bool moe = a.ids != nullptr;
    auto expert_of = [&](int p) -> int { return moe ? a.ids[p] : 0; };
    auto valid = [&](int e) -> bool { return e >= 0 && e < a.E; };
    const int n0 = (int)((int64_t)H * blockIdx.x / gridDim.x), n1 = (int)((int64_t)H * (blockIdx.x + 1) / gridDim.x);

    init_ring(S);

    if (warp == kMvConsumerWarps) {
        // ---- producer: W_down does not depend on A, so it streams at once;
        // after two stages it waits until the consumers hold h, so that the
        // h loads do not queue behind the rest of the weight stream ----
        if (lane == 0) {
            uint32_t slot = 0, ph = 0;
            bool ok = true;
            int issued = 0;
            // for each chunk of up to R2 output rows, one stage per valid slot
            for (int n = n0; n < n1 && ok;) {
                const int cnt = min(G.R2, n1 - n);
                for (int p = 0; p < P && ok; ++p) {
                    const int e = expert_of(p);
                    if (!valid(e)) continue;
                    if (issued == 2 && !mbar_wait(S.xready, 0, nullptr, a.err)) { ok = false; break; }
                    if (!mbar_wait(&S.empty[slot], ph ^ 1, nullptr, a.err)) { ok = false; break; }
                    ++issued;
                    const uint32_t bytes = (uint32_t)(cnt * G.rbI);
                    mbar_arrive_expect_tx(&S.full[slot], bytes);
                    bulk_g2s(S.ring + slot * kMvStageBytes, a.Wd + ((int64_t)e * H + n) * G.rbI, bytes,
                             &S.full[slot]);
                    if (++slot == kMvStages) { slot = 0; ph ^= 1; }
                }
                n += cnt;
            }
            drain_ring(S, slot, ph, a.err);
        }
        return;
    }

    // ----------------------------- consumers ---------------------------------
    const int tid = threadIdx.x;
    uint32_t slot = 0, ph = 0;
    bool ok = true;
    for (int t = tid; t < 3 * kMvMaxRows; t += kMvConsumers) S.acc[t] = 0.0f;   // acc and yacc
    // h is written by the gate/up kernel: wait until that grid has completed
    // and its memory is visible
    asm volatile("griddepcontrol.wait;" ::: "memory");
    quantize_vector(S, G.nhalf2, warp, lane, [&](int hb) -> float4 {
        const int p = hb / (2 * G.nbI), hl = hb - p * (2 * G.nbI);
        const int col = hl * 128 + 4 * lane;
        // load from a valid address whatever the column, then zero past I
        const int colc = col < I ? col : 0;
        float4 v = __ldcg(reinterpret_cast<const float4 *>(a.h + (int64_t)p * I + colc));
        if (col >= I) v = make_float4(0.f, 0.f, 0.f, 0.f);
        return v;
    });
    __syncwarp();
    if (lane == 0) mbar_arrive(S.xready);
    consumers_sync();
    VecReg R;
    int loaded_p = -1;
    for (int n = n0; n < n1 && ok;) {
        const int cnt = min(G.R2, n1 - n);
        for (int p = 0; p < P && ok; ++p) {
            const int e = expert_of(p);
            if (!valid(e)) continue;
            if (p != loaded_p) {
                load_resident(S, R, G.nbI, p * 2 * G.nbI, warp, lane);
                loaded_p = p;
            }
            if (!mbar_wait(&S.full[slot], ph, nullptr, a.err)) { ok = false; break; }
            process_stage(S, S.ring + slot * kMvStageBytes, R, 1, cnt, G.nbI, G.rbI, p * 2 * G.nbI, warp,
                          lane);
            consumers_sync();
            if (tid == 0) mbar_arrive(&S.empty[slot]);
            if (++slot == kMvStages) { slot = 0; ph ^= 1; }
            if (tid < cnt) {
                const float w = moe ? a.wts[p] : 1.0f;
                S.yacc[tid] += w * S.acc[tid];
                S.acc[tid] = 0.0f;
            }
            consumers_sync();
        }
        if (tid < cnt) {
            float *dst = a.y + n + tid;
            *dst = a.accumulate ? *dst + S.yacc[tid] : S.yacc[tid];
            S.yacc[tid] = 0.0f;
        }
        consumers_sync();
        n += cnt;
    }
}

cudaError_t launch_ffn_matvec(const MatvecArgs &a, cudaStream_t s) {
    const DeviceInfo &di = device_info();
    if (a.T != 1) return cudaErrorInvalidValue;
    const size_t smem = matvec_smem_bytes(1, a.H, a.I, a.k);
    static int attr_device = -1;
    if (attr_device != di.device) {
        cudaError_t e = cudaFuncSetAttribute(ffn_gu_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(ffn_down_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)smem);
        if (e != cudaSuccess) return e;
        attr_device = di.device;
    } else {
        // the attribute holds the largest request so far; grow it when needed
        cudaFuncAttributes fa;
        if (cudaFuncGetAttributes(&fa, ffn_gu_kernel) == cudaSuccess &&
            (size_t)fa.maxDynamicSharedSizeBytes < smem) {
            cudaError_t e = cudaFuncSetAttribute(ffn_gu_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 (int)smem);
            if (e == cudaSuccess)
                e = cudaFuncSetAttribute(ffn_down_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
            if (e != cudaSuccess) return e;
        }
    }
    const int grid = di.num_sms;   // one block per SM
    MatvecArgs args = a;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kMvThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaError_t e = cudaLaunchKernelEx(&cfg, ffn_gu_kernel, args);
    if (e != cudaSuccess) return e;
    // the down kernel is a programmatic dependent of the gate/up kernel
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, ffn_down_kernel, args);
}

}  // namespace zffn
