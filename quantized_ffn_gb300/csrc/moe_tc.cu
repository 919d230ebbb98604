// moe_tc.cu -- the routed layer's tensor-core kernel for few tokens per expert.
//
// In a routed layer each expert sees only the tokens routed to it -- at the
// routed workload's 256 tokens, top-8 of 128 experts, about 16 per expert --
// so the expert's weights, streamed once from memory, meet a handful of token
// rows ("Four bottlenecks, one CUDA backend...", section "Bottleneck 2 -- MoE
// decode was paying for its routing twice": one batched call over the chosen
// experts, ids read on the device).  Here the weights are the MMA's M side
// (128 rows per UMMA) and an expert's group of up to 32 gathered token rows
// its N side, so every unpacked weight feeds only useful products and every
// Q4_K byte is read once per group:
//
//   for each 128-row block of the expert's intermediate chunk:
//       G = Wg_blk . Xg^T,  U = Wu_blk . Xg^T            (TMEM, [128 x 32])
//       h[:, blk] = fp16(silu(G) * U * 2^-8)               (epilogue -> SMEM)
//   for each 128-row block of the output:
//       Y = Wd_blk[:, chunk] . h^T                         (TMEM, [128 x 32])
//       y[token, blk] += weight * 2^8 * Y                  (fp32 reductions)
//
// Both products take fp16 operands: x (converted when it is gathered), the
// weights unpacked with the fp8 -> fp16 converter (zffn_internal.cuh), and the
// intermediate scaled by 2^-8 so that its fp16 range reaches 1.7e7 (values
// beyond saturate).  The SwiGLU intermediate of a group never leaves the SM.
//
// The unpacked weights never touch shared memory: each unpacking thread owns
// one weight row, which is one TMEM lane of the MMA's A operand, and writes
// its 64 fp16 values of a K step straight into tensor memory (tcgen05.st);
// the MMA reads A from there.  Four A stages live in TMEM next to the
// accumulators, so the unpackers run up to four K steps ahead of the tensor
// core, and shared memory holds only the packed blocks, x and h.
//
// Block roles (24 warps):
//   warps 0-3   epilogue for TMEM lane quadrants 0-3: SwiGLU -> h, Y -> y
//   warp 4      TMEM allocator and MMA issuer (one elected lane issues)
//   warp 5      producer: whole blocks of 128 weight rows (one TMA box per
//               matrix covers four K steps; a Q6_K W_down stage is copied in
//               16-byte pieces by the threads of warps 5 and 7)
//   warp 6      TMA producer: the group's x tiles [32 x 64] fp16
//   warps 8-23  unpackers, four groups of four warps (one per TMEM lane
//               quadrant) taking tasks in turn
//   warp 7      idle (Q6_K: second producer warp for the W_down rows)
#include <cstring>

#include <cudaTypedefs.h>

#include "formats.h"
#include "zffn_internal.cuh"

namespace zffn {
namespace mg {

// 32 bytes at the even shared address a: nine aligned words and eight funnel
// shifts.
__device__ __forceinline__ void ld_shared_32_even(uint32_t a, uint32_t (&o)[8]) {
    const uint32_t base = a & ~3u, sh = (a & 3u) * 8;
    uint32_t v[9];
#pragma unroll
    for (int i = 0; i < 9; ++i) asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v[i]) : "r"(base + 4 * i));
#pragma unroll
    for (int i = 0; i < 8; ++i) o[i] = __funnelshift_r(v[i], v[i + 1], sh);
}

// Bytes of one row's 256 W_down weights in format F (whole blocks: Q5_1 has
// eight 24-byte blocks per 256 weights); the down phase's packed boxes are
// [128 rows x WD_BOX(F) bytes].  All are multiples of 16 bytes, as TMA needs.
// Q6_K (210-byte blocks, rows at 2-byte alignment) has no tensor map: each
// row's block is copied as the 16-byte aligned range that holds it (224
// bytes) into a 224-byte slot, the block starting (address % 16) bytes into
// it.
template <int F>
__host__ __device__ constexpr int wd_box_bytes() {
    return F == kFmtQ5_K ? 176 : F == kFmtQ5_1 ? 192 : F == kFmtQ6_K ? 224 : 144;
}

constexpr int NG = 32;                       // token rows of a group (UMMA N)
constexpr int BM = 128;                      // weight rows of a UMMA (M)
constexpr int BK = 64;                       // K per step
constexpr int KSB = 4;                       // K steps per packed block step (256 weights)
constexpr int IC_MAX = 768;                  // intermediate columns of a work unit
constexpr int NUM_WARPS = 24;
constexpr int THREADS = NUM_WARPS * 32;
constexpr int NR = 4, NA = 4, NX = 8;        // packed, unpacked (TMEM), x stages
constexpr int R_BOX = BM * kBlockBytes;      // one whole-block box of 128 rows: 18432 bytes
constexpr int R_BYTES = 2 * R_BOX;           // gate + up (the down phase uses the first half)
constexpr int X_BYTES = NG * BK * 2;         // [32 x 64] fp16
constexpr int H_TILE = NG * BK * 2;          // h columns [64j, 64j + 64) of the group
constexpr int H_BYTES = (IC_MAX / BK) * H_TILE;
constexpr int OFF_R = 0;
constexpr int OFF_X = OFF_R + NR * R_BYTES;
constexpr int OFF_H = OFF_X + NX * X_BYTES;
constexpr int OFF_BAR = OFF_H + H_BYTES;
constexpr int N_BARS = 2 * NR + 2 * NA + 2 * NX + 4 + 4 + 2;
constexpr int SMEM_BYTES = OFF_BAR + N_BARS * 8 + 16 + 1024;   // + alignment slack
static_assert(OFF_X % 1024 == 0 && OFF_H % 1024 == 0, "swizzled tiles 1024-aligned");
static_assert(SMEM_BYTES <= 232448, "shared memory budget of one block");
static_assert(NG == 32, "one group row per lane of an epilogue warp");
// TMEM columns: gate / up / down accumulators, two of each, then the A
// stages: 64 columns each (a K step of 128 rows in fp16 pairs: gate rows in
// the first 32 columns and up rows in the next 32, or W_down rows in the first 32)
constexpr uint32_t COL_G = 0, COL_U = 2 * NG, COL_Y = 4 * NG, COL_A = 6 * NG, A_COLS = 64;
constexpr uint32_t TMEM_COLS = 512;
static_assert(COL_A + NA * A_COLS <= TMEM_COLS, "TMEM budget");
constexpr uint32_t IDESC = idesc_f16_f32(BM, NG);
constexpr float H_SCALE = 1.0f / 256.0f;     // the intermediate is held as h * 2^-8

enum Role { ROLE_EPI, ROLE_MMA, ROLE_WPROD, ROLE_XPROD, ROLE_UNPACK, ROLE_IDLE };
__device__ __forceinline__ int warp_role(int w) {
    if (w < 4) return ROLE_EPI;
    if (w == 4) return ROLE_MMA;
    if (w == 5) return ROLE_WPROD;
    if (w == 6) return ROLE_XPROD;
    if (w >= 8) return ROLE_UNPACK;
    return ROLE_IDLE;
}

struct Maps {
    CUtensorMap x;             // gathered rows, fp16 [P][H], boxes [32 rows x 64]
    CUtensorMap wg, wu, wd;    // byte matrices, boxes [128 rows x 144 bytes]
};

struct Params {
    const uint8_t *Wd;         // W_down (Q6_K: bulk-copied rows; else through maps.wd)
    int64_t rbI;               // bytes of a W_down row
    float *y;
    const int4 *tiles;         // {row_start, row_count, expert, 0}
    const int *n_tiles_dev;
    const int *row_token;
    const float *row_weight;
    int *err;
    int n_tiles_host;
    int H, I;
};

// Geometry of one work unit (a group of one expert's rows, one chunk of its
// intermediate width).  Both phases run over whole Q4_K blocks of the chunk:
// rows of the chunk past its width unpack as zeros (h = 0 there), so the down
// phase may run over the partial last block.
struct Unit {
    int row_start, rows, expert;
    int i0, ic;                // chunk start and width
    int n_ib, ks_g;            // 128-row intermediate blocks, K steps of each
    int n_hb, ks_y;            // 128-row output blocks, K steps of each
};

__device__ __forceinline__ Unit make_unit(const Params &p, int u, int n_tiles) {
    Unit un;
    const int t = u % n_tiles, c = u / n_tiles;
    const int4 v = p.tiles[t];
    un.row_start = v.x;
    un.rows = v.y;
    un.expert = v.z;
    un.i0 = c * IC_MAX;
    un.ic = min(IC_MAX, p.I - un.i0);
    const int nb = (un.ic + 255) / 256;
    un.n_ib = 2 * nb;
    un.ks_g = p.H / BK;
    un.n_hb = p.H / BM;
    un.ks_y = KSB * nb;
    return un;
}

// Two K steps (128 weights of one nibble half) of a W_down row in Q5_K or
// Q5_1, into the TMEM operand layout (column c of a K step holds weights 2c,
// 2c+1 as an fp16 pair).  The 5-bit code q4 + 16 q5 splits into the 4-bit
// part, turned into fp16 as for Q4_K, and the fifth bit, a second code 0/1
// through the same converter, added with 16 times the scale:
//     w = (q4 2^-9) (512 d sc) + (q5 2^-9) (8192 d sc) - dmin m   (Q5_K)
//     w = (q4 2^-9) (512 d) + (q5 2^-9) (8192 d) + m              (Q5_1)
// two roundings to fp16 instead of one.  row: the row's bytes of the packed
// stage; ks0: the first K step (even) within the 256 weights; h: nibble half.
// out[j][16]: the TMEM words of K step ks0 + j for this thread's half.
template <int F>
__device__ __forceinline__ void unpack_wd_pair_fmt(uint32_t row, int ks0, int h, uint32_t (&out)[2][16]) {
    if (F == kFmtQ6_K) {
        // row: the block's first byte (even).  K steps ks0, ks0 + 1 (ks0
        // even) are half n = ks0 / 2 of the block; task h of K step j is its
        // quarter i = 2j + h: low 4 bits from nibble j of ql[64n + 32h + l],
        // high 2 bits = bits 2i, 2i+1 of qh[32n + l], one int8 scale per 16
        // weights.  w = d sc (q4 + 16 q2 - 32) as
        //     (q4 2^-9) (512 d sc) - 32 d sc + (q2 2^-9) (8192 d sc)
        // (the high part through the same converter; two roundings to fp16).
        const int n = ks0 >> 1;
        uint32_t ql[8], qh[8];
        ld_shared_32_even(row + 64 * n + 32 * h, ql);
        ld_shared_32_even(row + 128 + 32 * n, qh);
        uint32_t dbits, s0, s1;
        asm volatile("ld.shared.u16 %0, [%1];" : "=r"(dbits) : "r"(row + 208));
        asm volatile("ld.shared.u16 %0, [%1];" : "=r"(s0) : "r"(row + 192 + 4 * ks0 + 2 * h));
        asm volatile("ld.shared.u16 %0, [%1];" : "=r"(s1) : "r"(row + 192 + 4 * (ks0 + 1) + 2 * h));
        const float d = half_bits_to_float(dbits);
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const uint32_t sp = j ? s1 : s0;
            const int i = 2 * j + h;
            uint32_t a[2], a16[2], b[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const float ds = d * (float)(int)(int8_t)((sp >> (8 * e)) & 0xFFu);
                a[e] = f16x2_splat_satfinite(512.0f * ds);
                a16[e] = f16x2_splat_satfinite(8192.0f * ds);
                b[e] = f16x2_splat_satfinite(-32.0f * ds);
            }
#pragma unroll
            for (int w = 0; w < 8; ++w) {
                const int e = w >> 2;   // weights 4w..4w+3: scale 0 for l < 16, 1 after
                uint32_t o0, o1, f0, f1;
                codes4_to_f16((ql[w] >> (4 * j)) & 0x0F0F0F0Fu, a[e], b[e], o0, o1);
                codes4_to_f16((qh[w] >> (2 * i)) & 0x03030303u, a16[e], 0u, f0, f1);
                out[j][2 * w] = fma_f16x2(0x3C003C00u, f0, o0);
                out[j][2 * w + 1] = fma_f16x2(0x3C003C00u, f1, o1);
            }
        }
    } else if (F == kFmtQ5_K) {
        const uint4 hd = ld_shared_v4(row);
        const uint4 qh0 = ld_shared_v4(row + 16), qh1 = ld_shared_v4(row + 32);
        const uint32_t qh[8] = {qh0.x, qh0.y, qh0.z, qh0.w, qh1.x, qh1.y, qh1.z, qh1.w};
        const float d = half_bits_to_float(hd.x), dmin = half_bits_to_float(hd.x >> 16);
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int g = ks0 + j, sb = 2 * g + h;
            int sc, m;
            q4k_scale_min(hd.y, hd.z, hd.w, sb, sc, m);
            const uint32_t a = f16x2_splat_satfinite(512.0f * (d * (float)sc));
            const uint32_t a16 = f16x2_splat_satfinite(8192.0f * (d * (float)sc));
            const uint32_t b = f16x2_splat_satfinite(-(dmin * (float)m));
            const uint4 c0 = ld_shared_v4(row + 48 + 32 * g), c1 = ld_shared_v4(row + 64 + 32 * g);
            const uint32_t w[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                uint32_t o0, o1, f0, f1;
                codes4_to_f16((w[i] >> (4 * h)) & 0x0F0F0F0Fu, a, b, o0, o1);
                // fifth bits of weights 4i..4i+3 of sub-block sb: bit sb of qh bytes 4i..4i+3
                const uint32_t zero = 0u;
                codes4_to_f16((qh[i] >> sb) & 0x01010101u, a16, zero, f0, f1);
                out[j][2 * i] = fma_f16x2(0x3C003C00u, f0, o0);      // 1.0 * fifth + low part
                out[j][2 * i + 1] = fma_f16x2(0x3C003C00u, f1, o1);
            }
        }
    } else {   // Q5_1: eight 24-byte blocks per 256 weights, two per K step
#pragma unroll
        for (int j = 0; j < 2; ++j) {
#pragma unroll
            for (int bb = 0; bb < 2; ++bb) {
                const uint32_t blk = row + 24u * (uint32_t)(2 * (ks0 + j) + bb);
                uint32_t dm, qh;
                uint2 qa, qb;
                asm volatile("ld.shared.b32 %0, [%1];" : "=r"(dm) : "r"(blk));
                asm volatile("ld.shared.b32 %0, [%1];" : "=r"(qh) : "r"(blk + 4));
                asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(qa.x), "=r"(qa.y) : "r"(blk + 8));
                asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(qb.x), "=r"(qb.y) : "r"(blk + 16));
                const float d = half_bits_to_float(dm);
                const uint32_t a = f16x2_splat_satfinite(512.0f * d);
                const uint32_t a16 = f16x2_splat_satfinite(8192.0f * d);
                const uint32_t b = (dm >> 16) | (dm & 0xFFFF0000u);   // m, both halves
                const uint32_t qs[4] = {qa.x, qa.y, qb.x, qb.y};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    // weights 16h + 4i .. +3 of the block: nibble h of qs bytes 4i..4i+3
                    uint32_t o0, o1, f0, f1;
                    codes4_to_f16((qs[i] >> (4 * h)) & 0x0F0F0F0Fu, a, b, o0, o1);
                    // their fifth bits, qh bits 16h + 4i .. +3, one per byte
                    const uint32_t hb = (((qh >> (16 * h + 4 * i)) & 15u) * 0x00204081u) & 0x01010101u;
                    const uint32_t zero = 0u;
                    codes4_to_f16(hb, a16, zero, f0, f1);
                    // columns 16 bb + 8 h + 2 i, +1 of the K step
                    out[j][8 * bb + 2 * i] = fma_f16x2(0x3C003C00u, f0, o0);
                    out[j][8 * bb + 2 * i + 1] = fma_f16x2(0x3C003C00u, f1, o1);
                }
            }
        }
    }
}

template <int F>
__global__ void __launch_bounds__(THREADS, 1) moe_group_kernel(const __grid_constant__ Maps maps, const Params p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + OFF_BAR);
    uint64_t *r_full = bars, *r_empty = bars + NR;
    uint64_t *a_full = bars + 2 * NR, *a_empty = a_full + NA;
    uint64_t *x_full = a_empty + NA, *x_empty = x_full + NX;
    uint64_t *g_full = x_empty + NX, *g_empty = g_full + 2;
    uint64_t *y_full = g_empty + 2, *y_empty = y_full + 2;
    uint64_t *h_full = y_empty + 2, *drain = h_full + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + N_BARS);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // (Q6_K: warp 7 shares the producer's row copies)
    const int role = F == kFmtQ6_K && warp == 7 ? ROLE_WPROD : warp_role(warp);
    const uint32_t s_r = smem_u32(smem + OFF_R);
    const uint32_t s_x = smem_u32(smem + OFF_X), s_h = smem_u32(smem + OFF_H);

    if (threadIdx.x == 0) {
        for (int i = 0; i < NR; ++i) {
            // (Q6_K: every thread of the two producer warps arrives)
            mbar_init(&r_full[i], F == kFmtQ6_K ? 64 : 1);
            mbar_init(&r_empty[i], 2 * 2 * 4);        // 2 K-step pairs x 2 tasks x 4 warps
        }
        for (int i = 0; i < NA; ++i) {
            mbar_init(&a_full[i], 2 * 4);             // 2 tasks x 4 warps
            mbar_init(&a_empty[i], 1);
        }
        for (int i = 0; i < NX; ++i) {
            mbar_init(&x_full[i], 1);
            mbar_init(&x_empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&g_full[i], 1);
            mbar_init(&g_empty[i], 4);
            mbar_init(&y_full[i], 1);
            mbar_init(&y_empty[i], 4);
        }
        mbar_init(h_full, 4);
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbarrier_init();
        prefetch_tensormap(&maps.x);
        prefetch_tensormap(&maps.wg);
        prefetch_tensormap(&maps.wu);
        if (F != kFmtQ6_K) prefetch_tensormap(&maps.wd);
    }
    if (role == ROLE_MMA) {
        tmem_alloc(tmem_slot, TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // This kernel is launched as a programmatic dependent of the kernel that
    // writes its tile table and gathered rows: wait for that grid's
    // completion before the first read of them.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    const int n_tiles = min(*p.n_tiles_dev, p.n_tiles_host);
    const int n_chunks = (p.I + IC_MAX - 1) / IC_MAX;
    const int n_units = n_tiles * n_chunks;
    const int m_units = (int)blockIdx.x < n_units
                            ? (n_units - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x : 0;
    auto unit_of = [&](int k) { return make_unit(p, (int)blockIdx.x + k * (int)gridDim.x, n_tiles); };

    if (role == ROLE_WPROD) {
        // ------------- producer: whole blocks of 128 weight rows -------------
        // Lane 0 of warp 5 issues the TMA boxes.  Q6_K: warps 5 and 7 both
        // run this loop and every one of their threads arrives once per stage
        // (the stage barrier expects 64 arrivals): on a gate/up stage lane 0
        // of warp 5 with the TMA bytes and the others plainly; on a W_down
        // stage each thread copies two rows' blocks in 16-byte pieces
        // (cp.async, no TMA: 128 small bulk copies a stage were bound by the
        // copy engine) and arrives when they have landed.
        const int pw = warp == 5 ? 0 : 1;                // producer warp index
        uint32_t ri = 0, rph = 0, issued = 0;
        bool ok = true;
        for (int k = 0; k < m_units && ok; ++k) {
            const Unit un = unit_of(k);
            const int nbs_g = un.ks_g / KSB, nbs_y = un.ks_y / KSB;
            for (int b = 0; b < un.n_ib * nbs_g + un.n_hb * nbs_y; ++b) {
                if (!mbar_wait(&r_empty[ri], rph ^ 1, abort_flag, p.err)) { ok = false; break; }
                uint8_t *rs = smem + OFF_R + ri * R_BYTES;
                if (b < un.n_ib * nbs_g) {
                    const int ib = b / nbs_g, kb = b % nbs_g;
                    const int row = un.expert * p.I + un.i0 + ib * BM;
                    if (pw == 0 && lane == 0) {
                        mbar_arrive_expect_tx(&r_full[ri], 2 * R_BOX);
                        tma_load_2d(rs, &maps.wg, &r_full[ri], kb * kBlockBytes, row);
                        tma_load_2d(rs + R_BOX, &maps.wu, &r_full[ri], kb * kBlockBytes, row);
                    } else if (F == kFmtQ6_K) {
                        mbar_arrive(&r_full[ri]);
                    }
                } else {
                    const int bb = b - un.n_ib * nbs_g;
                    const int hb = bb / nbs_y, kb = bb % nbs_y;
                    const int row = un.expert * p.H + hb * BM;
                    if (F == kFmtQ6_K) {
                        // row t = 64 pw + 32 q + lane: the 16-byte aligned
                        // range of its block, which starts at an even offset
                        // of at most 14 and so always spans 224 bytes (14
                        // pieces), inside the matrix (a 16-byte aligned
                        // W_down whose rows of H % 256 == 0 blocks end on a
                        // 16-byte boundary)
                        const uint32_t dst0 = smem_u32(rs);
#pragma unroll
                        for (int q = 0; q < BM / 64; ++q) {
                            const int t = 64 * pw + 32 * q + lane;
                            const uint64_t src = (reinterpret_cast<uint64_t>(p.Wd) +
                                                  (uint64_t)((int64_t)(row + t) * p.rbI) +
                                                  (uint64_t)(un.i0 / 256 + kb) * 210u) & ~15ull;
#pragma unroll
                            for (int c = 0; c < 14; ++c)
                                asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                                                 dst0 + (uint32_t)(t * wd_box_bytes<F>() + 16 * c)),
                                             "l"(src + 16ull * c)
                                             : "memory");
                        }
                        asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(&r_full[ri]))
                                     : "memory");
                    } else if (pw == 0 && lane == 0) {
                        mbar_arrive_expect_tx(&r_full[ri], BM * wd_box_bytes<F>());
                        tma_load_2d(rs, &maps.wd, &r_full[ri], (un.i0 / 256 + kb) * wd_box_bytes<F>(), row);
                    }
                }
                ++issued;
                if (++ri == NR) { ri = 0; rph ^= 1; }
            }
        }
        // every load issued here lands before the block may exit
        for (uint32_t i = 0; i < (uint32_t)NR && i < issued; ++i) {
            if (ri == 0) { ri = NR; rph ^= 1; }
            --ri;
            mbar_wait(&r_full[ri], rph, nullptr, p.err, kWaitBudgetCycles / 8);
        }
    } else if (role == ROLE_XPROD) {
        // ------------- TMA producer: x tiles of the group, one per gate/up K step -------------
        if (lane == 0) {
            uint32_t xi = 0, xph = 0, issued = 0;
            bool ok = true;
            for (int k = 0; k < m_units && ok; ++k) {
                const Unit un = unit_of(k);
                for (int s = 0; s < un.n_ib * un.ks_g; ++s) {
                    const int ks = s % un.ks_g;
                    if (!mbar_wait(&x_empty[xi], xph ^ 1, abort_flag, p.err)) { ok = false; break; }
                    mbar_arrive_expect_tx(&x_full[xi], X_BYTES);
                    tma_load_2d(smem + OFF_X + xi * X_BYTES, &maps.x, &x_full[xi], ks * BK, un.row_start);
                    ++issued;
                    if (++xi == NX) { xi = 0; xph ^= 1; }
                }
            }
            for (uint32_t i = 0; i < (uint32_t)NX && i < issued; ++i) {
                if (xi == 0) { xi = NX; xph ^= 1; }
                --xi;
                mbar_wait(&x_full[xi], xph, nullptr, p.err, kWaitBudgetCycles / 8);
            }
        }
    } else if (role == ROLE_MMA) {
        // ---------------- MMA issuer ----------------
        // One elected lane walks the program and issues every MMA and commit.
        const bool issuer = elect_one();
      if (issuer) {
        uint32_t ai = 0, aph = 0, xi = 0, xph = 0;
        uint32_t gb = 0, gph = 0, yb = 0, yph = 0;   // buffer index, per-buffer parity bits
        bool ok = true;
        auto commit = [&](uint64_t *bar) { tc_commit(bar); };
        const uint64_t dx0 = smem_desc_k_sw128(s_x);
        const uint64_t dh0 = smem_desc_k_sw128(s_h);
        for (int k = 0; k < m_units && ok; ++k) {
            const Unit un = unit_of(k);
            for (int ib = 0; ib < un.n_ib && ok; ++ib) {
                for (int ks = 0; ks < un.ks_g; ++ks) {
                    if (ks == 0) {
                        if (!mbar_wait(&g_empty[gb], ((gph >> gb) & 1) ^ 1, abort_flag, p.err)) { ok = false; break; }
                    }
                    if (!mbar_wait(&a_full[ai], aph, abort_flag, p.err) ||
                        !mbar_wait(&x_full[xi], xph, abort_flag, p.err)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t ta = tmem_base + COL_A + ai * A_COLS;
                    const uint64_t dx = dx0 + (uint64_t)((xi * X_BYTES) >> 4);
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk)
                        tc_mma_f16_ta(tmem_base + COL_G + gb * NG, ta + 8 * kk, dx + 2 * kk, IDESC,
                                      (ks | kk) != 0);
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk)
                        tc_mma_f16_ta(tmem_base + COL_U + gb * NG, ta + 32 + 8 * kk, dx + 2 * kk, IDESC,
                                      (ks | kk) != 0);
                    commit(&a_empty[ai]);
                    commit(&x_empty[xi]);
                    if (++ai == NA) { ai = 0; aph ^= 1; }
                    if (++xi == NX) { xi = 0; xph ^= 1; }
                    if (ks == un.ks_g - 1) {
                        commit(&g_full[gb]);
                        gph ^= 1u << gb;
                        gb ^= 1;
                    }
                }
            }
            for (int hb = 0; hb < un.n_hb && ok; ++hb) {
                for (int ks = 0; ks < un.ks_y; ++ks) {
                    if (ks == 0) {
                        // the unit's h is complete in shared memory before its first down step
                        if (hb == 0 && !mbar_wait(h_full, (uint32_t)k & 1, abort_flag, p.err)) { ok = false; break; }
                        if (!mbar_wait(&y_empty[yb], ((yph >> yb) & 1) ^ 1, abort_flag, p.err)) { ok = false; break; }
                    }
                    if (!mbar_wait(&a_full[ai], aph, abort_flag, p.err)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t ta = tmem_base + COL_A + ai * A_COLS;
                    const uint64_t dh = dh0 + (uint64_t)((ks * H_TILE) >> 4);
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk)
                        tc_mma_f16_ta(tmem_base + COL_Y + yb * NG, ta + 8 * kk, dh + 2 * kk, IDESC,
                                      (ks | kk) != 0);
                    commit(&a_empty[ai]);
                    if (++ai == NA) { ai = 0; aph ^= 1; }
                    if (ks == un.ks_y - 1) {
                        commit(&y_full[yb]);
                        yph ^= 1u << yb;
                        yb ^= 1;
                    }
                }
            }
        }
        // every MMA issued here completes before TMEM is released
        commit(drain);
      }
        __syncwarp();
        mbar_wait(drain, 0, nullptr, p.err, kWaitBudgetCycles / 8);
    } else if (role == ROLE_UNPACK) {
        // ------------- weight unpackers (four groups of 4 warps) -------------
        // The program's K steps go in pairs (2m, 2m+1: both in one Q4_K
        // block), and every pair has two 128-thread tasks: the gate rows and
        // the up rows (gate/up phase), or the low and the high nibbles of the
        // 128 W_down rows (down phase).  Group g takes task g % 2 of the pairs
        // with parity g / 2: groups 0-1 fill A stages 0-1, groups 2-3 stages
        // 2-3.  A task decodes its row's block header once for the four
        // sub-blocks of its two K steps.  Thread r of a task owns weight row r,
        // which is TMEM lane r: warp w writes lane quadrant w % 4 (the only one
        // it may access).
        const int uw = warp - 8;
        const uint32_t grp = (uint32_t)(uw / 4);
        const int task = (int)(grp & 1);
        const uint32_t pair_parity = grp >> 1;
        const int r = (uw % 4) * 32 + lane;             // weight row within the task
        const uint32_t t_row = tmem_base + ((uint32_t)((uw % 4) * 32) << 16);
        uint32_t pair = 0;                               // K-step pairs of the program so far
        bool ok = true;
        for (int k = 0; k < m_units && ok; ++k) {
            const Unit un = unit_of(k);
            const int n_g = un.n_ib * un.ks_g, n_steps = n_g + un.n_hb * un.ks_y;
            int blk = 0, ks = 0;                         // position within the phase
            for (int s = 0; s < n_steps && ok; s += 2, ++pair) {
                const bool gu = s < n_g;
                if (s == n_g) { blk = 0; ks = 0; }
                const int cur_blk = blk, cur_ks = ks;
                ks += 2;
                if (ks == (gu ? un.ks_g : un.ks_y)) { ks = 0; ++blk; }
                if ((pair & 1) != pair_parity) continue;
                const uint32_t bs = pair >> 1;           // packed block step
                const uint32_t ri = bs % NR, rph = (bs / NR) & 1;
                const uint32_t ai = (2 * pair) % NA, aph = ((2 * pair) / NA) & 1;
                const bool zero = gu && cur_blk * BM + r >= un.ic;
                if (!mbar_wait(&r_full[ri], rph, abort_flag, p.err)) { ok = false; break; }
                if (F != kFmtQ4_K && !gu) {
                    // W_down in Q5_K / Q5_1: the format's unpack reads the
                    // packed stage itself; the stage is released after it
                    if (!mbar_wait(&a_empty[ai], aph ^ 1, abort_flag, p.err) ||
                        !mbar_wait(&a_empty[ai + 1], aph ^ 1, abort_flag, p.err)) { ok = false; break; }
                    tc_fence_after();
                    uint32_t v[2][16];
                    // (Q6_K: where the row's block starts in its slot)
                    const uint32_t off =
                        F == kFmtQ6_K
                            ? (uint32_t)(((int64_t)(un.expert * p.H + cur_blk * BM + r) * p.rbI +
                                          (int64_t)(un.i0 / 256 + (cur_ks >> 2)) * 210) & 15)
                            : 0u;
                    unpack_wd_pair_fmt<F>(s_r + ri * R_BYTES + (uint32_t)(r * wd_box_bytes<F>()) + off, cur_ks & 3,
                                          task, v);
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&r_empty[ri]);
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        if ((cur_ks + j) * BK >= un.ic) {   // past the chunk's width: zeros
#pragma unroll
                            for (int i = 0; i < 16; ++i) v[j][i] = 0u;
                        }
                        const uint32_t dst = t_row + COL_A + (ai + j) * A_COLS;
                        if (F == kFmtQ5_K || F == kFmtQ6_K) {
                            tmem_st_32x32b_x16(dst + 16 * task, v[j]);
                        } else {   // Q5_1: columns 8 task .. +7 of each 32-weight block
                            const uint32_t v0[8] = {v[j][0], v[j][1], v[j][2], v[j][3], v[j][4], v[j][5], v[j][6], v[j][7]};
                            const uint32_t v1[8] = {v[j][8], v[j][9], v[j][10], v[j][11], v[j][12], v[j][13], v[j][14], v[j][15]};
                            tmem_st_32x32b_x8(dst + 8 * task, v0);
                            tmem_st_32x32b_x8(dst + 16 + 8 * task, v1);
                        }
                    }
                    tmem_st_wait();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) {
                        mbar_arrive(&a_full[ai]);
                        mbar_arrive(&a_full[ai + 1]);
                    }
                    continue;
                }
                uint4 hd = make_uint4(0, 0, 0, 0), c[4] = {hd, hd, hd, hd};
                if (!zero) {
                    const uint32_t src = s_r + ri * R_BYTES + (gu ? task * R_BOX : 0) + r * kBlockBytes;
                    hd = ld_shared_v4(src);
#pragma unroll
                    for (int i = 0; i < 4; ++i) c[i] = ld_shared_v4(src + 16 + 32 * (cur_ks & 3) + 16 * i);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&r_empty[ri]);
                if (!mbar_wait(&a_empty[ai], aph ^ 1, abort_flag, p.err) ||
                    !mbar_wait(&a_empty[ai + 1], aph ^ 1, abort_flag, p.err)) { ok = false; break; }
                tc_fence_after();
                uint32_t sa[4], sb[4];                   // sub-blocks 2 (ks & 3) .. +3
                if (gu) {
                    q4k_f16_scales4(hd, 2 * (cur_ks & 3), sa, sb);
                } else {
                    // down phase: only this task's nibble half of each K step,
                    // sub-blocks 2 (ks & 3) + task and 2 (ks & 3) + 2 + task
                    const float d = 512.0f * half_bits_to_float(hd.x), dmin = half_bits_to_float(hd.x >> 16);
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        int sc, m;
                        q4k_scale_min(hd.y, hd.z, hd.w, 2 * (cur_ks & 3) + 2 * j + task, sc, m);
                        sa[2 * j] = sa[2 * j + 1] = f16x2_splat_satfinite(d * (float)sc);
                        sb[2 * j] = sb[2 * j + 1] = f16x2_splat_satfinite(-(dmin * (float)m));
                    }
                }
#pragma unroll
                for (int j = 0; j < 2; ++j) {            // K step cur_ks + j, stage ai + j
                    const uint32_t w[8] = {c[2 * j].x, c[2 * j].y, c[2 * j].z, c[2 * j].w,
                                           c[2 * j + 1].x, c[2 * j + 1].y, c[2 * j + 1].z, c[2 * j + 1].w};
                    const uint32_t dst = t_row + COL_A + (ai + j) * A_COLS;
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        if (!gu && h != task) continue;  // down phase: one nibble half
                        uint32_t v[16];
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            codes4_to_f16((w[i] >> (4 * h)) & 0x0F0F0F0Fu, sa[2 * j + h], sb[2 * j + h],
                                          v[2 * i], v[2 * i + 1]);
                        if (!gu && (cur_ks + j) * BK >= un.ic) {   // past the chunk's width: zeros
#pragma unroll
                            for (int i = 0; i < 16; ++i) v[i] = 0u;
                        }
                        // gate/up: row's columns 32 task + 16 h; down: 16 h
                        tmem_st_32x32b_x16(dst + (gu ? 32 * task : 0) + 16 * h, v);
                    }
                }
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&a_full[ai]);
                    mbar_arrive(&a_full[ai + 1]);
                }
            }
        }
    } else if (role == ROLE_EPI) {
        // ---------------- epilogue (4 warps) ----------------
        const int q = warp;                           // TMEM lane quadrant of this warp
        const uint32_t t_lane = tmem_base + ((uint32_t)(q * 32) << 16);
        uint32_t gb = 0, gph = 0, yb = 0, yph = 0;
        bool ok = true;
        for (int k = 0; k < m_units && ok; ++k) {
            const Unit un = unit_of(k);
            // the group's rows: lane t holds row t's token and routing weight
            // (NG == 32: one row per lane), broadcast by shuffles below
            const bool v = lane < un.rows;
            const int my_tok = v ? p.row_token[un.row_start + lane] : 0;
            const float my_w = v ? p.row_weight[un.row_start + lane] * 256.0f : 0.0f;
            // ---- gate/up blocks: h = silu(G) * U, scaled, to shared memory
            for (int ib = 0; ib < un.n_ib; ++ib) {
                if (!mbar_wait(&g_full[gb], (gph >> gb) & 1, abort_flag, p.err)) { ok = false; break; }
                tc_fence_after();
                const int i = ib * BM + q * 32 + lane;        // intermediate column within the chunk
                const uint32_t hrow = s_h + (uint32_t)(i >> 6) * H_TILE + (uint32_t)(i & 7) * 2;
                const uint32_t chunk = (uint32_t)((i & 63) >> 3);
#pragma unroll
                for (int c = 0; c < NG; c += 16) {
                    uint32_t gr[16], ur[16];
                    tmem_ld_32x32b_x16(t_lane + COL_G + gb * NG + c, gr);
                    tmem_ld_32x32b_x16(t_lane + COL_U + gb * NG + c, ur);
                    tmem_ld_wait(gr);
                    tmem_ld_wait(ur);
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int t = c + j;
                        const float g = __uint_as_float(gr[j]), u = __uint_as_float(ur[j]);
                        const float h = __fdividef(g * u * H_SCALE, 1.0f + __expf(-g));
                        uint16_t hb16;
                        asm("cvt.rn.satfinite.f16.f32 %0, %1;" : "=h"(hb16) : "f"(h));
                        const uint32_t addr = hrow + (uint32_t)t * 128 + ((chunk ^ (uint32_t)(t & 7)) << 4);
                        asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"(hb16) : "memory");
                    }
                }
                fence_proxy_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&g_empty[gb]);
                    if (ib == un.n_ib - 1) mbar_arrive(h_full);
                }
                gph ^= 1u << gb;
                gb ^= 1;
            }
            // ---- down blocks: y[token, row] += weight * 2^8 * Y
            for (int hb = 0; hb < un.n_hb && ok; ++hb) {
                if (!mbar_wait(&y_full[yb], (yph >> yb) & 1, abort_flag, p.err)) { ok = false; break; }
                tc_fence_after();
                const int row = hb * BM + q * 32 + lane;      // output column
#pragma unroll
                for (int c = 0; c < NG; c += 16) {
                    uint32_t yr[16];
                    tmem_ld_32x32b_x16(t_lane + COL_Y + yb * NG + c, yr);
                    tmem_ld_wait(yr);
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int t = c + j;
                        const int tok = __shfl_sync(0xffffffffu, my_tok, t);
                        const float wt = __shfl_sync(0xffffffffu, my_w, t);
                        if (t < un.rows) {
                            float *dst = p.y + (int64_t)tok * p.H + row;
                            asm volatile("red.global.add.f32 [%0], %1;" ::"l"(dst), "f"(__uint_as_float(yr[j]) * wt)
                                         : "memory");
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&y_empty[yb]);
                yph ^= 1u << yb;
                yb ^= 1;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (role == ROLE_MMA) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

}  // namespace mg

static bool encode_map(PFN_cuTensorMapEncodeTiled_v12000 encode, CUtensorMap *m, CUtensorMapDataType dt,
                       const void *base, int64_t inner, int64_t rows, int64_t row_pitch, int box_inner,
                       int box_rows, CUtensorMapSwizzle sw) {
    const cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)row_pitch};
    const cuuint32_t box[2] = {(cuuint32_t)box_inner, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return encode(m, dt, 2, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int moe_group_rows() { return mg::NG; }

cudaError_t launch_moe_group(const TcArgs &a, int wd_fmt, cudaStream_t s) {
    if (wd_fmt != kFmtQ4_K && wd_fmt != kFmtQ5_K && wd_fmt != kFmtQ5_1 && wd_fmt != kFmtQ6_K)
        return cudaErrorInvalidValue;
    if (wd_fmt == kFmtQ6_K && (reinterpret_cast<uintptr_t>(a.Wd) & 15)) return cudaErrorInvalidValue;
    const DeviceInfo &di = device_info();
    if (a.H % 256 != 0 || a.I % 64 != 0) return cudaErrorInvalidValue;
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult qr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &qr) !=
            cudaSuccess || qr != cudaDriverEntryPointSuccess)
        return cudaErrorNotSupported;
    auto encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    mg::Maps maps;
    const int64_t rbH = q4k_row_bytes(a.H), rbI = fmt_row_bytes(wd_fmt, a.I);
    const int wd_box = wd_fmt == kFmtQ5_K ? mg::wd_box_bytes<kFmtQ5_K>()
                     : wd_fmt == kFmtQ5_1 ? mg::wd_box_bytes<kFmtQ5_1>() : mg::wd_box_bytes<kFmtQ4_K>();
    memset(&maps, 0, sizeof(maps));
    if (!encode_map(encode, &maps.x, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, a.x, a.H, a.x_rows, (int64_t)a.H * 2,
                    mg::BK, mg::NG, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_map(encode, &maps.wg, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.Wg, rbH, (int64_t)a.E * a.I, rbH,
                    kBlockBytes, mg::BM, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !encode_map(encode, &maps.wu, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.Wu, rbH, (int64_t)a.E * a.I, rbH,
                    kBlockBytes, mg::BM, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        (wd_fmt != kFmtQ6_K &&
         !encode_map(encode, &maps.wd, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.Wd, rbI, (int64_t)a.E * a.H, rbI,
                     wd_box, mg::BM, CU_TENSOR_MAP_SWIZZLE_NONE)))
        return cudaErrorInvalidValue;
    const void *fn = wd_fmt == kFmtQ5_K ? (const void *)mg::moe_group_kernel<kFmtQ5_K>
                   : wd_fmt == kFmtQ5_1 ? (const void *)mg::moe_group_kernel<kFmtQ5_1>
                   : wd_fmt == kFmtQ6_K ? (const void *)mg::moe_group_kernel<kFmtQ6_K>
                                        : (const void *)mg::moe_group_kernel<kFmtQ4_K>;
    cudaError_t e = ensure_dynamic_smem(fn, (size_t)mg::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    mg::Params p;
    p.Wd = a.Wd;
    p.rbI = rbI;
    p.y = a.y;
    p.tiles = a.tiles;
    p.n_tiles_dev = a.n_tiles_dev;
    p.row_token = a.row_token;
    p.row_weight = a.row_weight;
    p.err = a.err;
    p.n_tiles_host = a.n_tiles_host;
    p.H = a.H;
    p.I = a.I;
    const int n_chunks = (a.I + mg::IC_MAX - 1) / mg::IC_MAX;
    int64_t grid = (int64_t)a.n_tiles_host * n_chunks;
    if (grid > di.num_sms) grid = di.num_sms;
    if (grid < 1) return cudaSuccess;
    void *kargs[] = {&maps, &p};
    // a programmatic dependent of the kernel before it (the gather of the
    // routed rows, or the tile table of a dense call): its launch overlaps
    // that kernel's tail and it waits for its completion itself
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(mg::THREADS);
    cfg.dynamicSmemBytes = (size_t)mg::SMEM_BYTES;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelExC(&cfg, fn, kargs);
}

}  // namespace zffn
