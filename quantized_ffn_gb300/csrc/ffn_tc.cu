// ffn_tc.cu -- the fused prefill kernel on the 5th-generation tensor cores.
//
// What it computes, per (token tile, intermediate chunk) work unit:
//   for each 128-row slice s of the chunk:
//       [G | U] = X_tile . [W_gate rows ; W_up rows]^T        (tcgen05, TMEM)
//       h[:, s] = fp16( silu(G) * U / 16 )                      (epilogue)
//   for each 128-column slice n of the output:
//       Y = h . (16 W_down[n rows, chunk cols])^T              (tcgen05, TMEM)
//       y[token, n cols] += Y                                   (fp32 reductions in L2)
// This is the producer/consumer interleave along the intermediate dimension
// ("Fused SwiGLU MLP: ZINC RDNA4 Down-Projection Bandwidth", section "Why
// this fusion is harder than the last one"): a block of the intermediate is
// computed, staged on chip, and contracted by the down projection before the
// next block; only x and y touch device memory.  Q4_K weights are unpacked
// on chip on their way into the multiply (same page, FAQ "Why is fusing the
// SwiGLU intermediate harder..."): dedicated warps read the packed blocks and
// write fp16 operand tiles straight into shared memory; no unpacked copy of a
// weight ever exists in device memory.  The scale/min pair of a sub-block is
// decoded once per row and step, not per weight ("VGPR pressure caps the
// fused RDNA4 prefill GEMM at nine waves", section "The recoverable registers
// versus the stubborn ones"); accumulators live in tensor memory, not in
// registers, which removes the register-pressure problem at its root.
//
// Schedule.  The y reductions of a unit (4 MB for 256 tokens) leave the SM
// through a port of about 32 bytes per cycle, so a unit's down projection
// cannot keep pace with its own MMAs.  The MMA program therefore interleaves
// the down-projection jobs of unit i with the gate/up steps of unit i+1:
//   G(0) | Y(0,0) G(1)... Y(0,1) G(1)... ... Y(0,31) G(1)... | Y(1,0) G(2)... |
// (each Y job is followed by an equal share of the next unit's gate/up
// steps), so the y traffic is spread over the whole run.  TMEM holds one
// gate/up accumulator (256 columns), one down-projection accumulator (128
// columns) and a stash of the next unit's h (128 columns of fp16 pairs),
// copied into shared memory once the current unit's down projection has
// consumed the previous h.
//
// Block roles (24 warps; warp w runs on sub-partition w % 4):
//   warps 0-3   epilogue for TMEM lane quadrants 0-3: SwiGLU -> h stash,
//               h stash -> shared memory, down-projection tile -> y
//   warp 4      TMEM allocator and MMA issuer (one elected lane issues)
//   warp 5      TMA producer: packed Q4_K weight slices into a ring
//   warp 6      TMA producer: x tiles [128 x 64] fp16, 128-byte swizzle
//   warps 8-19  weight unpackers: packed slices -> fp16 tiles, 128-byte
//               swizzle
//   warps 7, 20-23  idle
// Every role walks the same step program (Prog below) in the same order.
#include <cudaTypedefs.h>

#include "zffn_internal.cuh"

namespace zffn {
namespace tc {

constexpr int BM = 128;                  // token rows per CTA per tile (UMMA M per CTA)
constexpr int BK = 64;                   // K per gate/up step (128 bytes of fp16)
constexpr int YK = 128;                  // K per down-projection step
constexpr int GU_ROWS = 128;             // intermediate rows per gate/up job
constexpr int NJ_GU = 256;               // UMMA N of a gate/up job (128 gate + 128 up rows)
constexpr int NJ_Y = 128;                // UMMA N of a down-projection job (output columns)
constexpr int A_BYTES = BM * BK * 2;     // 16 KB x tile per CTA
constexpr int HT_BYTES = BM * BK * 2;    // one 64-column slice of h: 16 KB
constexpr uint32_t COL_GU = 0, COL_Y = 256, COL_STASH = 384;   // TMEM columns
// Both products take fp16 operands: x (converted once per call), the weights
// (unpacked with the fp8 -> fp16 converter) and the intermediate.  The
// intermediate is held as h / W_SCALE (fp16 range to 1.05e6) and W_down as
// W_SCALE * w (sub-blocks up to d*sc = 8, dmin*m = 4094 in range; values
// beyond saturate), so the down product needs no rescaling: both factors are
// powers of two and change no significand.
constexpr float W_SCALE = 16.0f;
constexpr float H_SCALE = 1.0f / W_SCALE;
// Two fp32 values -> one fp16 pair (lo in the low half), nearest, clamped to
// the largest finite fp16.
__device__ __forceinline__ uint32_t pack_f16x2_satfinite(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}
// Unpack the 8 code words of one Q4_K weight row and K step (64 weights of
// sub-blocks 2g and 2g+1) into its swizzled fp16 row (128-byte swizzle),
// times ws (1, or W_SCALE for W_down).  Each code pair becomes (q0, q1) *
// 2^-9 exactly (codes_to_f16x2), and one fused fp16 multiply-add per pair
// gives  w = (q * 2^-9) * fp16(512 ws d sc) - fp16(ws dmin m),  rounded once
// to fp16: the sub-block's scale and offset are exact in fp32 before their
// rounding to fp16 (ws is a power of two); values beyond the fp16 range
// saturate at +-65504.  Chunks are stored as soon as they are formed.
__device__ __forceinline__ void unpack_row_to_smem_f16(uint4 hd, const uint32_t (&w)[8], int g, float ws,
                                                       uint32_t row_addr, int row) {
    const float d = ws * half_bits_to_float(hd.x), dmin = ws * half_bits_to_float(hd.x >> 16);
    int sc0, m0, sc1, m1;
    q4k_scale_min(hd.y, hd.z, hd.w, 2 * g, sc0, m0);
    q4k_scale_min(hd.y, hd.z, hd.w, 2 * g + 1, sc1, m1);
    const uint32_t a0 = f16x2_splat_satfinite(512.0f * (d * (float)sc0));
    const uint32_t b0 = f16x2_splat_satfinite(-(dmin * (float)m0));
    const uint32_t a1 = f16x2_splat_satfinite(512.0f * (d * (float)sc1));
    const uint32_t b1 = f16x2_splat_satfinite(-(dmin * (float)m1));
    constexpr uint32_t NIB = 0x0F0F0F0Fu;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        // words 2c, 2c+1: low nibbles are weights 8c..8c+7 of sub-block 2g,
        // high nibbles weights 32+8c..32+8c+7 of sub-block 2g+1
        const uint32_t l0 = w[2 * c] & NIB, l1 = w[2 * c + 1] & NIB;
        const uint32_t h0 = (w[2 * c] >> 4) & NIB, h1 = (w[2 * c + 1] >> 4) & NIB;
        st_shared_v4(row_addr + (((uint32_t)(c ^ (row & 7))) << 4),
                     fma_f16x2(codes_to_f16x2(l0), a0, b0), fma_f16x2(codes_to_f16x2(l0 >> 16), a0, b0),
                     fma_f16x2(codes_to_f16x2(l1), a0, b0), fma_f16x2(codes_to_f16x2(l1 >> 16), a0, b0));
        st_shared_v4(row_addr + (((uint32_t)((c + 4) ^ (row & 7))) << 4),
                     fma_f16x2(codes_to_f16x2(h0), a1, b1), fma_f16x2(codes_to_f16x2(h0 >> 16), a1, b1),
                     fma_f16x2(codes_to_f16x2(h1), a1, b1), fma_f16x2(codes_to_f16x2(h1 >> 16), a1, b1));
    }
}
// Down-projection accumulators.  While a block has a next unit, its down jobs
// use COL_Y (the gate/up accumulator is busy with the next unit), the first
// half of them alternating with the h stash (ybuf_of).  In a block's last unit
// the stash and the gate/up accumulator are free once its h is in shared
// memory, so its down jobs rotate over four 128-column buffers and the drain
// of one overlaps the MMAs of the next three.
constexpr int NYBUF = 4;
__device__ __forceinline__ uint32_t ybuf_col(int b) {
    return b == 0 ? COL_Y : b == 1 ? COL_STASH : b == 2 ? COL_GU : COL_GU + 128;
}
// The buffer of down job n (of NY) of a unit.  In a block's last unit the
// jobs rotate over all four.  Otherwise the stash is free from the moment the
// unit's h has gone to shared memory until the next unit's first gate/up job
// completes, which the program places after down job NY/2 - 1: jobs before
// it alternate between COL_Y and the stash, later ones use COL_Y.
__device__ __forceinline__ int ybuf_of(int n, int NY, bool last) {
    return last ? n % NYBUF : (n < NY / 2 ? (n & 1) : 0);
}
// Warp roles.  Warp w is scheduled by sub-partition w % 4.  The epilogue
// needs one warp per sub-partition, because a warp reads only the TMEM lane
// quadrant w % 4: warps 0-3.  The unpackers (warps 8-19, three groups of one
// warp per sub-partition) spread the arithmetic evenly over the four
// sub-partitions.  One lane of the MMA warp walks its program and issues the
// MMAs, without per-instruction divergence.
//
// Groups and B stages: group k takes the tasks with index k modulo
// UNPACK_GROUPS, and the waits on a stage's "empty" barrier test a phase
// parity only.  A group's wait for phase n of a stage is unambiguous only if
// phase n-1 has completed, which its own previous wait guarantees exactly
// when UNPACK_GROUPS <= the stages a CTA pair cycles through (NB); on a
// single CTA two tasks share a step, so each group keeps to one stage.
constexpr int NUM_WARPS = 24;
constexpr int THREADS = NUM_WARPS * 32;
constexpr int UNPACK_GROUP_WARPS = 4;    // one 128-thread task
constexpr int UNPACK_GROUPS = 3;         // groups take tasks in turn
enum Role { ROLE_EPI, ROLE_MMA, ROLE_WPROD, ROLE_XPROD, ROLE_UNPACK, ROLE_IDLE };
__device__ __forceinline__ int warp_role(int w) {
    if (w < 4) return ROLE_EPI;
    if (w == 4) return ROLE_MMA;
    if (w == 5) return ROLE_WPROD;
    if (w == 6) return ROLE_XPROD;
    if (w >= 8 && w < 8 + UNPACK_GROUPS * UNPACK_GROUP_WARPS) return ROLE_UNPACK;
    return ROLE_IDLE;
}
// 0..11 over the unpack warps 8..19
__device__ __forceinline__ int unpack_index(int w) { return w - 8; }
constexpr uint32_t TMEM_COLS = 512;
// y staging for the TMA reductions: per epilogue warp two buffers of
// [32 rows x Y_COLS fp32]; 32 columns use the 128-byte swizzle (chunk j of
// row r at j ^ (r % 8)), 16 columns the 64-byte swizzle (j ^ (r/2 % 4)).

// Geometry of one kernel variant.  PAIR: a cluster of two CTAs shares each
// 256-token tile; one UMMA of M = 256 covers both CTAs' rows, and the weight
// rows of every step are split between the CTAs.
//   gate/up step: ROWS_B weight rows x 64 K per CTA (pair: the leader the
//                 gate rows, its peer the up rows)
//   down step:    ROWS_Y W_down rows x 128 K per CTA, stored as two
//                 64-column halves
// Both kinds fill one B stage and take TASKS 128-thread unpack tasks, one
// 64-weight slice per thread.
template <bool PAIR>
struct Cfg {
    static constexpr int ROWS_B = PAIR ? 128 : 256;
    static constexpr int ROWS_Y = ROWS_B / 2;
    static constexpr int TASKS = ROWS_B / 128;
    static constexpr int TILE = PAIR ? 256 : 128;         // tokens per work-unit tile
    static constexpr int IC = 256;                        // intermediate columns per work unit
    static constexpr int N_HT = IC / BK;                  // 64-column slices of h
    static constexpr int NA = PAIR ? 3 : 2;               // x stages
    static constexpr int NB = PAIR ? 3 : 2;               // unpacked-weight stages
    static constexpr int NR = PAIR ? 5 : 3;               // packed-weight stages
    static constexpr int Y_COLS = PAIR ? 32 : 16;
    static constexpr int Y_BUF = 32 * Y_COLS * 4;
    static constexpr int B_BYTES = ROWS_B * BK * 2;       // = 2 * ROWS_Y * 128
    static constexpr int R_HDR_GU = ROWS_B * 16;          // gate/up: headers, then 32 code bytes a row
    static constexpr int R_HDR_Y = ROWS_Y * 16;           // down: headers, then 64 code bytes a row
    static constexpr int R_BYTES_GU = ROWS_B * 48;
    static constexpr int R_BYTES_Y = ROWS_Y * 80;
    static constexpr int R_BYTES = R_BYTES_GU;            // stage size (the larger)
    static constexpr int OFF_H = 0;
    static constexpr int OFF_A = OFF_H + N_HT * HT_BYTES;
    static constexpr int OFF_B = OFF_A + NA * A_BYTES;
    static constexpr int OFF_R = OFF_B + NB * B_BYTES;
    static constexpr int OFF_Y = ((OFF_R + NR * R_BYTES) + 1023) & ~1023;
    static constexpr int OFF_BAR = OFF_Y + 4 * 2 * Y_BUF;
    static constexpr int N_BARS = 2 * NA + 2 * NB + 2 * NR + 5 + 2 * NYBUF;
    static constexpr int SMEM_BYTES = OFF_BAR + N_BARS * 8 + 16 + 1024;   // + alignment slack
    static constexpr int EPI_ARRIVALS = PAIR ? 8 : 4;     // epilogue warps arriving per job
    static constexpr int B_ARRIVALS = (PAIR ? 2 : 1) * TASKS * UNPACK_GROUP_WARPS;
    static constexpr uint32_t IDESC_GU = idesc_f16_f32(PAIR ? 256 : 128, NJ_GU);   // fp16 x, W_gate, W_up
    static constexpr uint32_t IDESC_Y = idesc_f16_f32(PAIR ? 256 : 128, NJ_Y);     // fp16 h / 16, 16 W_down
    static_assert(R_BYTES_Y <= R_BYTES, "down-step slice fits a weight stage");
    static_assert(!PAIR || UNPACK_GROUPS <= NB, "parity waits on B stages stay unambiguous");
    static_assert(PAIR || UNPACK_GROUPS <= 2 * NB, "parity waits on B stages stay unambiguous");
    static_assert(SMEM_BYTES <= 232448, "shared memory budget of one block");
    static_assert(NA == NB, "x stage i goes with unpacked-weight stage i");
};

// Tensor maps: x tiles, y tiles, and the packed weights viewed as byte
// matrices [rows][row bytes] with two box shapes each: the 16-byte block
// headers and the code bytes of one step (32 for a gate/up step of 64
// weights, 64 for a down step of 128).
struct Maps {
    CUtensorMap x;
    CUtensorMap y;                          // fp32 [T][H], boxes of [32 rows x Y_COLS]
    CUtensorMap g_hdr, g_qs, u_hdr, u_qs;   // boxes of 128 rows
    CUtensorMap d_hdr, d_qs;                // boxes of ROWS_Y rows
};

struct Params {
    const uint8_t *Wg, *Wu, *Wd;
    float *y;
    const int4 *tiles;
    const int *n_tiles_dev;
    const int *row_token;
    const float *row_weight;
    int *err;
    int n_tiles_host;
    int T, H, I;
};

struct Tile {
    int row_start, row_count, expert;
};

// Work-unit geometry shared by every role.
struct Unit {
    Tile tile;    // the CTA's own token rows
    int i0;       // first intermediate column of the chunk
    int ic;       // columns in this chunk (multiple of 64)
};

template <bool PAIR>
__device__ __forceinline__ Unit make_unit(const Params &p, int u, int n_tiles, uint32_t rank) {
    Unit un;
    const int chunk = u / n_tiles;
    const int t = u % n_tiles;
    if (p.tiles) {
        const int4 v = p.tiles[t];
        un.tile.row_start = v.x;
        un.tile.row_count = v.y;
        un.tile.expert = v.z;
    } else {
        un.tile.row_start = t * Cfg<PAIR>::TILE + (int)rank * BM;
        un.tile.row_count = min(BM, p.T - un.tile.row_start);
        un.tile.expert = 0;
    }
    un.i0 = chunk * Cfg<PAIR>::IC;
    un.ic = min(Cfg<PAIR>::IC, p.I - un.i0);
    return un;
}

// The step program of one block, walked in the same order by every role.
// Units k = 0..m-1 of the block (global unit group + k * n_groups).  First
// the gate/up steps of unit 0 (two jobs of ksg steps); then, for each unit
// k, its NY down jobs (YS steps each), each followed by the next GU_PER_Y
// gate/up steps of unit k+1.  With a 256-wide chunk a unit has 2 * H/64
// gate/up steps and H/128 down jobs, so GU_PER_Y = 4 spreads the next unit's
// gate/up steps exactly over the current unit's down jobs.  The walk is
// incremental (no divisions): the MMA issuer's scalar work per step sits on
// the critical path of the tensor pipe.
constexpr int GU_PER_Y = 4;
struct Prog {
    int m, NY, YS, ksg;
    int blk;        // -1: leading gate/up steps of unit 0; k >= 0: down jobs of unit k
    int n, ys;      // down job and step within it
    int s, ks;      // gate/up job and step (of the unit whose gate/up steps run)
    int gb;         // gate/up steps left in the current share
    bool gu, done;
    __device__ __forceinline__ void start(int m_, int ksg_, int NY_, int YS_) {
        m = m_; ksg = ksg_; NY = NY_; YS = YS_;
        blk = -1; n = 0; ys = 0; s = 0; ks = 0; gb = 2 * ksg; gu = true; done = m <= 0;
    }
    // index (0..m-1) of the unit the current step belongs to
    __device__ __forceinline__ int unit() const { return gu ? blk + 1 : blk; }
    __device__ __forceinline__ bool gu_last() const { return ks == ksg - 1; }
    __device__ __forceinline__ void next_job() {
        gu = false;
        ys = 0;
        if (++n < NY) return;
        n = 0;
        s = 0;
        ks = 0;
        if (++blk >= m) done = true;
    }
    __device__ __forceinline__ void next() {
        if (gu) {
            if (++ks == ksg) { ks = 0; ++s; }
            if (--gb > 0) return;
            if (blk < 0) { blk = 0; n = 0; ys = 0; s = 0; ks = 0; gu = false; return; }
            next_job();
        } else {
            if (++ys < YS) return;
            if (blk + 1 < m) { gu = true; gb = GU_PER_Y; return; }
            next_job();
        }
    }
};

template <bool PAIR>
__global__ void __launch_bounds__(THREADS, 1)
    ffn_tc_kernel(const __grid_constant__ Maps maps, const Params p) {
    using C = Cfg<PAIR>;
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte alignment for the swizzled tiles
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);
    uint64_t *a_full = bars, *a_empty = bars + C::NA;
    uint64_t *b_full = bars + 2 * C::NA, *b_empty = b_full + C::NB;
    uint64_t *r_full = b_empty + C::NB, *r_empty = r_full + C::NR;
    uint64_t *g_full = r_empty + C::NR, *g_empty = g_full + 1;
    uint64_t *h_full = g_full + 2, *h_empty = g_full + 3, *drain = g_full + 4;
    uint64_t *y_full = g_full + 5, *y_empty = y_full + NYBUF;   // per down-projection buffer
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + C::N_BARS);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int role = warp_role(warp);
    const uint32_t rank = PAIR ? cluster_ctarank() : 0;
    const bool leader = rank == 0;
    const uint32_t s_h = smem_u32(smem + C::OFF_H);
    const uint32_t s_a = smem_u32(smem + C::OFF_A);
    const uint32_t s_b = smem_u32(smem + C::OFF_B);
    const uint32_t s_r = smem_u32(smem + C::OFF_R);
    // Arrive on a barrier that the MMA issuer waits on: the local one, or the
    // pair leader's copy at the same offset.
    auto arrive_leader = [&](uint64_t *bar) {
        if (PAIR) mbar_arrive_cluster(mapa_shared(smem_u32(bar), 0));
        else mbar_arrive(bar);
    };

    if (threadIdx.x == 0) {
        for (int i = 0; i < C::NA; ++i) {
            mbar_init(&a_full[i], 1);
            mbar_init(&a_empty[i], 1);
        }
        for (int i = 0; i < C::NB; ++i) {
            mbar_init(&b_full[i], C::B_ARRIVALS);
            mbar_init(&b_empty[i], 1);
        }
        for (int i = 0; i < C::NR; ++i) {
            mbar_init(&r_full[i], 1);
            mbar_init(&r_empty[i], C::TASKS * UNPACK_GROUP_WARPS);
        }
        mbar_init(g_full, 1);
        mbar_init(g_empty, C::EPI_ARRIVALS);
        for (int b = 0; b < NYBUF; ++b) {
            mbar_init(&y_full[b], 1);
            mbar_init(&y_empty[b], C::EPI_ARRIVALS);
        }
        mbar_init(h_full, C::EPI_ARRIVALS);
        mbar_init(h_empty, 1);
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbarrier_init();
        prefetch_tensormap(&maps.x);
        prefetch_tensormap(&maps.y);
        prefetch_tensormap(&maps.g_hdr);
        prefetch_tensormap(&maps.g_qs);
        prefetch_tensormap(&maps.u_hdr);
        prefetch_tensormap(&maps.u_qs);
        prefetch_tensormap(&maps.d_hdr);
        prefetch_tensormap(&maps.d_qs);
    }
    if (role == ROLE_MMA) {
        if (PAIR) {
            tmem_alloc_pair(tmem_slot, TMEM_COLS);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(tmem_slot, TMEM_COLS);
            tmem_relinquish();
        }
    }
    tc_fence_before();
    __syncthreads();
    if (PAIR) cluster_sync_all();      // both CTAs' barriers exist before any remote arrive
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    const int n_tiles = p.n_tiles_dev ? min(*p.n_tiles_dev, p.n_tiles_host) : p.n_tiles_host;
    const int n_chunks = (p.I + C::IC - 1) / C::IC;
    const int n_units = n_tiles * n_chunks;
    const int group = PAIR ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
    const int n_groups = PAIR ? (int)(gridDim.x >> 1) : (int)gridDim.x;
    const int m_units = group < n_units ? (n_units - group + n_groups - 1) / n_groups : 0;
    // Gate/up steps of a unit, steps of a K = 128 down job, down jobs.  The
    // chunk width is IC for every unit (I is a multiple of 256).
    const int ks_gu = p.H / BK;
    const int YS = C::IC / YK;
    const int NY = p.H / NJ_Y;
    auto unit_of = [&](int k) { return make_unit<PAIR>(p, group + k * n_groups, n_tiles, rank); };

    if (role == ROLE_WPROD) {
        // ------------- TMA producer: packed weights -------------
        if (lane == 0) {
            uint32_t ri = 0, rph = 0, r_issued = 0;
            Prog pg;
            pg.start(m_units, ks_gu, NY, YS);
            int cur = -1;
            Unit un{};
            for (; !pg.done; pg.next()) {
                if (pg.unit() != cur) { cur = pg.unit(); un = unit_of(cur); }
                const int e = un.tile.expert;
                if (!mbar_wait(&r_empty[ri], rph ^ 1, abort_flag, p.err)) break;
                uint8_t *rs = smem + C::OFF_R + ri * C::R_BYTES;
                if (pg.gu) {
                    const int s = pg.s, ks = pg.ks;
                    const int xcol = (ks >> 2) * kBlockBytes;
                    const int qcol = xcol + 16 + 32 * (ks & 3);
                    const int row = e * p.I + un.i0 + s * GU_ROWS;
                    mbar_arrive_expect_tx(&r_full[ri], C::R_BYTES_GU);
                    if (PAIR) {
                        // the leader unpacks the gate rows, its peer the up rows
                        const CUtensorMap *mh = leader ? &maps.g_hdr : &maps.u_hdr;
                        const CUtensorMap *mq = leader ? &maps.g_qs : &maps.u_qs;
                        tma_load_2d(rs, mh, &r_full[ri], xcol, row);
                        tma_load_2d(rs + C::R_HDR_GU, mq, &r_full[ri], qcol, row);
                    } else {
                        tma_load_2d(rs, &maps.g_hdr, &r_full[ri], xcol, row);
                        tma_load_2d(rs + 128 * 16, &maps.u_hdr, &r_full[ri], xcol, row);
                        tma_load_2d(rs + C::R_HDR_GU, &maps.g_qs, &r_full[ri], qcol, row);
                        tma_load_2d(rs + C::R_HDR_GU + 128 * 32, &maps.u_qs, &r_full[ri], qcol, row);
                    }
                } else {
                    // W_down rows n*128 + rank*ROWS_Y .. +ROWS_Y, chunk columns
                    // [i0 + 128*ys, +128): one Q4_K block per row, code bytes 64*ys..
                    const int xcol = (un.i0 >> 8) * kBlockBytes;
                    const int row = e * p.H + pg.n * NJ_Y + (int)rank * C::ROWS_Y;
                    mbar_arrive_expect_tx(&r_full[ri], C::R_BYTES_Y);
                    tma_load_2d(rs, &maps.d_hdr, &r_full[ri], xcol, row);
                    tma_load_2d(rs + C::R_HDR_Y, &maps.d_qs, &r_full[ri], xcol + 16 + 64 * pg.ys, row);
                }
                ++r_issued;
                if (++ri == C::NR) { ri = 0; rph ^= 1; }
            }
            // Before the block may exit, every load issued here must have
            // landed: wait (bounded) for the full barriers of the last stages
            // issued (a phase that completed long ago passes at once).
            for (uint32_t i = 0; i < (uint32_t)C::NR && i < r_issued; ++i) {
                if (ri == 0) { ri = C::NR; rph ^= 1; }
                --ri;
                mbar_wait(&r_full[ri], rph, nullptr, p.err, kWaitBudgetCycles / 8);
            }
        }
    } else if (role == ROLE_XPROD) {
        // ------------- TMA producer: x tiles of the gate/up steps -------------
        // (A dense call whose units fill every pair launches this kernel as
        // a programmatic dependent of the x conversion: x and y are read only
        // after that grid completes, the weight roles start at once.)
        // x stage i goes with unpacked-weight stage i: the step that uses
        // both releases both with one commit (b_empty), so this producer
        // walks every step of the program on the B ring's index and loads x
        // for the gate/up steps only.
        if (lane == 0) {
            asm volatile("griddepcontrol.wait;" ::: "memory");
            uint32_t bi = 0, bph = 0, apb = 0, issued = 0;
            Prog pg;
            pg.start(m_units, ks_gu, NY, YS);
            int cur = -1;
            Unit un{};
            for (; !pg.done; pg.next()) {
                // every step's stage is waited for, so that each wait tests
                // the phase right after the one the previous wait saw (parity
                // waits are unambiguous only then)
                if (!mbar_wait(&b_empty[bi], bph ^ 1, abort_flag, p.err)) break;
                if (pg.gu) {
                    if (pg.unit() != cur) { cur = pg.unit(); un = unit_of(cur); }
                    const int ks = pg.ks;
                    void *dst = smem + C::OFF_A + bi * A_BYTES;
                    if (PAIR) {
                        // both CTAs' tiles complete on the leader's barrier
                        if (leader) mbar_arrive_expect_tx(&a_full[bi], 2 * A_BYTES);
                        tma_load_2d_pair(dst, &maps.x, mapa_shared(smem_u32(&a_full[bi]), 0), ks * BK,
                                         un.tile.row_start);
                    } else {
                        mbar_arrive_expect_tx(&a_full[bi], A_BYTES);
                        tma_load_2d(dst, &maps.x, &a_full[bi], ks * BK, un.tile.row_start);
                    }
                    apb ^= 1u << bi;
                    issued |= 1u << bi;
                }
                if (++bi == C::NB) { bi = 0; bph ^= 1; }
            }
            // In a pair the x tiles complete on the leader's barriers, which the
            // leader's issuer has waited for before its final MMAs.
            if (!PAIR || leader) {
                for (int i = 0; i < C::NA; ++i)
                    if ((issued >> i) & 1)
                        mbar_wait(&a_full[i], ((apb >> i) & 1) ^ 1, nullptr, p.err, kWaitBudgetCycles / 8);
            }
        }
    } else if (role == ROLE_MMA) {
        // ---------------- MMA issuer (the pair's leader only) ----------------
        // One elected lane walks the program and issues every MMA and commit
        // (no divergence inside the loop); the rest of the warp waits for the
        // final drain.
        if (leader) {
          const bool issuer = elect_one();
          if (issuer) {
            uint32_t bi = 0, bph = 0, jg = 0;
            uint32_t apb = 0;    // bit i: parity of the uses of x stage i so far
            uint32_t yph = 0;    // bit b: parity of the uses of down buffer b so far
            int yb = 0;
            bool ok = true;
            auto commit = [&](uint64_t *bar) {
                if (PAIR) tc_commit_pair(bar); else tc_commit(bar);
            };
            auto mma = [&](uint32_t d, uint64_t da, uint64_t db, uint32_t idesc, bool acc) {
                if (PAIR) tc_mma_bf16_pair(d, da, db, idesc, acc);
                else tc_mma_bf16(d, da, db, idesc, acc);
            };
            // Descriptors advance by the stage strides (start address field in
            // 16-byte units); every operand lies below 256 KB.
            const uint64_t da0 = smem_desc_k_sw128(s_a), db0 = smem_desc_k_sw128(s_b);
            const uint64_t dh0 = smem_desc_k_sw128(s_h);
            constexpr uint64_t A_STEP = A_BYTES >> 4, B_STEP = C::B_BYTES >> 4;
            constexpr uint64_t HT_STEP = HT_BYTES >> 4, YH_STEP = (C::ROWS_Y * 128) >> 4;
            uint64_t db = db0;
            const uint32_t d_gu = tmem_base + COL_GU;
            uint32_t d_y = tmem_base + COL_Y;
            Prog pg;
            pg.start(m_units, ks_gu, NY, YS);
            for (; !pg.done && ok; pg.next()) {
                if (pg.gu) {
                    if (pg.ks == 0) {
                        if (!mbar_wait(g_empty, (jg & 1) ^ 1, abort_flag, p.err)) { ok = false; break; }
                        tc_fence_after();
                    }
                    if (!mbar_wait(&a_full[bi], (apb >> bi) & 1, abort_flag, p.err) ||
                        !mbar_wait(&b_full[bi], bph, abort_flag, p.err)) { ok = false; break; }
                    tc_fence_after();
                    const uint64_t da = da0 + bi * A_STEP;
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk)
                        mma(d_gu, da + 2 * kk, db + 2 * kk, C::IDESC_GU, (pg.ks | kk) != 0);
                    // one commit frees the step's x and weight stages
                    commit(&b_empty[bi]);
                    apb ^= 1u << bi;
                    if (++bi == C::NB) { bi = 0; bph ^= 1; db = db0; } else { db += B_STEP; }
                    if (pg.gu_last()) { commit(g_full); ++jg; }
                } else {
                    if (pg.ys == 0) {
                        // the first down job of a unit reads its h: wait until
                        // the epilogues placed all of it in shared memory
                        if (pg.n == 0 && !mbar_wait(h_full, (uint32_t)pg.blk & 1, abort_flag, p.err)) { ok = false; break; }
                        yb = ybuf_of(pg.n, NY, pg.blk == m_units - 1);
                        d_y = tmem_base + ybuf_col(yb);
                        if (!mbar_wait(&y_empty[yb], ((yph >> yb) & 1) ^ 1, abort_flag, p.err)) { ok = false; break; }
                        tc_fence_after();
                    }
                    if (!mbar_wait(&b_full[bi], bph, abort_flag, p.err)) { ok = false; break; }
                    tc_fence_after();
                    const uint64_t dh = dh0 + (uint64_t)(2 * pg.ys) * HT_STEP;
#pragma unroll
                    for (int kk = 0; kk < YK / 16; ++kk)
                        mma(d_y, dh + (kk / 4) * HT_STEP + 2 * (kk & 3), db + (kk / 4) * YH_STEP + 2 * (kk & 3),
                            C::IDESC_Y, (pg.ys | kk) != 0);
                    commit(&b_empty[bi]);
                    if (++bi == C::NB) { bi = 0; bph ^= 1; db = db0; } else { db += B_STEP; }
                    if (pg.ys == YS - 1) {
                        commit(&y_full[yb]);
                        yph ^= 1u << yb;
                        // h may be overwritten once the unit's last down MMAs finish
                        if (pg.n == NY - 1) commit(h_empty);
                    }
                }
            }
            // every MMA issued here completes before TMEM is released
            commit(drain);
          }
          __syncwarp();
          mbar_wait(drain, 0, nullptr, p.err, kWaitBudgetCycles / 8);
        }
    } else if (role == ROLE_UNPACK) {
        // ------------- weight unpackers (three groups of 4 warps) -------------
        // A step's weights are split into 128-thread tasks of one 64-weight
        // slice per thread; the groups take the tasks in turn, counted over
        // the whole program of this block.
        const int uw = unpack_index(warp);
        const uint32_t grp = (uint32_t)(uw / UNPACK_GROUP_WARPS);
        const int tt = (uw % UNPACK_GROUP_WARPS) * 32 + lane;    // thread within the task
        uint32_t bi = 0, bph = 0, ri = 0, rph = 0, gt = 0;
        bool ok = true;
        Prog pg;
        pg.start(m_units, ks_gu, NY, YS);
        int cur = -1;
        Unit un{};
        for (; !pg.done && ok; pg.next()) {
#pragma unroll
            for (int task = 0; task < C::TASKS; ++task, ++gt) {
                if (gt % UNPACK_GROUPS != grp) continue;
                if (pg.unit() != cur) { cur = pg.unit(); un = unit_of(cur); }
                const int f = task * 128 + tt;
                int row, half, g;
                uint32_t qoff, hdr_base;
                bool zero = false;
                if (pg.gu) {
                    const int s = pg.s, ks = pg.ks;
                    row = f;
                    half = 0;
                    g = ks & 3;
                    qoff = C::R_HDR_GU + row * 32;
                    const int grow = PAIR ? row : (row & 127);      // gate/up row within the job
                    zero = un.i0 + s * GU_ROWS + grow >= p.I;
                } else {
                    row = f % C::ROWS_Y;
                    half = f / C::ROWS_Y;
                    g = 2 * pg.ys + half;
                    qoff = C::R_HDR_Y + row * 64 + 32 * half;
                }
                hdr_base = row * 16;
                if (!mbar_wait(&r_full[ri], rph, abort_flag, p.err)) { ok = false; break; }
                uint4 hd = make_uint4(0, 0, 0, 0), q0 = hd, q1 = hd;
                if (!zero) {
                    const uint32_t rs = s_r + ri * C::R_BYTES;
                    hd = ld_shared_v4(rs + hdr_base);
                    // bank-conflict-free order of the two 16-byte reads
                    const int qfirst = (row >> 2) & 1;
                    const uint4 first = ld_shared_v4(rs + qoff + 16 * qfirst);
                    const uint4 second = ld_shared_v4(rs + qoff + 16 * (qfirst ^ 1));
                    q0 = qfirst ? second : first;
                    q1 = qfirst ? first : second;
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&r_empty[ri]);
                if (!mbar_wait(&b_empty[bi], bph ^ 1, abort_flag, p.err)) { ok = false; break; }
                const uint32_t rb = s_b + bi * C::B_BYTES + half * (C::ROWS_Y * 128) + sw128_row(row);
                const uint32_t w8[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
                unpack_row_to_smem_f16(hd, w8, g, pg.gu ? 1.0f : W_SCALE, rb, row);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) arrive_leader(&b_full[bi]);
            }
            if (++ri == C::NR) { ri = 0; rph ^= 1; }
            if (++bi == C::NB) { bi = 0; bph ^= 1; }
        }
    } else if (role == ROLE_EPI) {
        // ---------------- epilogue (4 warps) ----------------
        // y (zero-filled by the x conversion of a dense call) is touched only
        // after the grid before this one has completed
        asm volatile("griddepcontrol.wait;" ::: "memory");
        const int q = warp & 3;                      // TMEM lane quadrant of this warp
        const int row = q * 32 + lane;               // token row within the CTA's tile
        const uint32_t lane_bits = (uint32_t)(q * 32) << 16;
        const uint32_t t_lane = tmem_base + lane_bits;
        const uint32_t s_y = smem_u32(smem + C::OFF_Y), s_base = smem_u32(smem);
        // dense tiles: y slices go through swizzled shared memory and one TMA
        // reduction per warp and slice; routed tiles scatter rows, so each
        // thread adds its own row with vector reductions
        const bool tma_y = p.tiles == nullptr;
        uint32_t jg = 0;
        uint32_t yph = 0;        // bit b: parity of the uses of down buffer b so far
        bool ok = true;
        Prog pg;
        pg.start(m_units, ks_gu, NY, YS);
        int cur = -1;
        Unit un{};
        bool valid = false, warp_live = false;
        int token = 0, warp_row0 = 0;
        float wgt = 1.0f;
        for (; !pg.done && ok; pg.next()) {
            if (pg.gu) {
                if (!pg.gu_last()) continue;
                // ---- gate/up job complete: h = silu(G) * U -> the TMEM stash
                const int s = pg.s;
                if (!mbar_wait(g_full, jg & 1, abort_flag, p.err)) { ok = false; break; }
                tc_fence_after();
#pragma unroll 1
                for (int c = 0; c < GU_ROWS; c += 16) {
                    uint32_t gr[16], ur[16], hw[8];
                    tmem_ld_32x32b_x16(t_lane + COL_GU + c, gr);
                    tmem_ld_32x32b_x16(t_lane + COL_GU + GU_ROWS + c, ur);
                    tmem_ld_wait(gr);
                    tmem_ld_wait(ur);
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const float g0 = __uint_as_float(gr[2 * j]), g1 = __uint_as_float(gr[2 * j + 1]);
                        const float u0 = __uint_as_float(ur[2 * j]), u1 = __uint_as_float(ur[2 * j + 1]);
                        const float h0 = __fdividef(g0 * u0 * H_SCALE, 1.0f + __expf(-g0));
                        const float h1 = __fdividef(g1 * u1 * H_SCALE, 1.0f + __expf(-g1));
                        hw[j] = pack_f16x2_satfinite(h0, h1);
                    }
                    // stash column s*64 + c/2 holds h columns s*128 + c, +1
                    tmem_st_32x32b_x8(t_lane + COL_STASH + s * 64 + c / 2, hw);
                }
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) arrive_leader(g_empty);
                ++jg;
                continue;
            }
            if (pg.n == 0 && pg.ys == 0) {
                // ---- start of unit blk's down jobs: its h, stashed in TMEM by
                // the gate/up jobs, goes to shared memory once the previous
                // unit's down MMAs have finished reading the old h
                if (!mbar_wait(h_empty, ((uint32_t)pg.blk & 1) ^ 1, abort_flag, p.err)) { ok = false; break; }
                tc_fence_after();
#pragma unroll 1
                for (int t = 0; t < C::N_HT; ++t) {
                    uint32_t hw[32];
                    tmem_ld_32x32b_x32(t_lane + COL_STASH + t * 32, hw);
                    tmem_ld_wait(hw);
                    const uint32_t tile_base = s_h + t * HT_BYTES + sw128_row(row);
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        st_shared_v4(tile_base + ((uint32_t)(j ^ (row & 7)) << 4), hw[4 * j], hw[4 * j + 1],
                                     hw[4 * j + 2], hw[4 * j + 3]);
                }
                fence_proxy_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) arrive_leader(h_full);
                // this row's destination for the unit's down jobs
                if (pg.blk != cur) { cur = pg.blk; un = unit_of(cur); }
                valid = row < un.tile.row_count;
                token = 0;
                wgt = 1.0f;
                if (valid) {
                    const int xr = un.tile.row_start + row;
                    token = p.row_token ? p.row_token[xr] : xr;
                    wgt = p.row_weight ? p.row_weight[xr] : 1.0f;
                }
                warp_row0 = un.tile.row_start + q * 32;
                warp_live = warp_row0 < p.T;
            }
            if (pg.ys != YS - 1) continue;
            // ---- down job n complete: Y tile -> y[token, n*128 ..]
            const int yb = ybuf_of(pg.n, NY, pg.blk == m_units - 1);
            const uint32_t ycol = ybuf_col(yb);
            if (!mbar_wait(&y_full[yb], (yph >> yb) & 1, abort_flag, p.err)) { ok = false; break; }
            tc_fence_after();
            const int ncol = pg.n * NJ_Y;
            if (tma_y) {
                // Pairs of staging boxes: a warp's two buffers are refilled once
                // the previous pair's reductions have read them; one proxy fence
                // and one bulk group cover a pair.  One 32-column TMEM load
                // fills 32 / Y_COLS boxes.
                constexpr int BOX_PER_LD = 32 / C::Y_COLS;
                const int sw = C::Y_COLS == 32 ? (lane & 7) : ((lane >> 1) & 3);
                const uint32_t buf0 = s_y + (uint32_t)(q * 2 * C::Y_BUF);
                const uint32_t rowoff = (uint32_t)lane * (C::Y_COLS * 4);
#pragma unroll 1
                for (int c = 0; c < NJ_Y; c += 32) {
                    const int box0 = (c / C::Y_COLS) & 1;         // buffer of this load's first box
                    if (box0 == 0) {
                        if (lane == 0) bulk_wait_group_read<0>();
                        __syncwarp();
                    }
                    uint32_t yv[32];
                    tmem_ld_32x32b_x32(t_lane + ycol + c, yv);
                    tmem_ld_wait(yv);
#pragma unroll
                    for (int e = 0; e < 32; e += 4) {
                        const int bx = box0 + e / C::Y_COLS, j = (e % C::Y_COLS) / 4;
                        st_shared_v4(buf0 + bx * C::Y_BUF + rowoff + (((uint32_t)(j ^ sw)) << 4),
                                     yv[e], yv[e + 1], yv[e + 2], yv[e + 3]);
                    }
                    if (box0 + BOX_PER_LD == 2) {
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0 && warp_live) {
                            const int col0 = ncol + c + 32 - 2 * C::Y_COLS;   // first column of the pair
                            tma_reduce_add_2d(&maps.y, smem + (buf0 - s_base), col0, warp_row0);
                            tma_reduce_add_2d(&maps.y, smem + (buf0 + C::Y_BUF - s_base), col0 + C::Y_COLS,
                                              warp_row0);
                            bulk_commit_group();
                        }
                    }
                }
            } else {
                float *yrow = p.y + (int64_t)token * p.H + ncol;
#pragma unroll 1
                for (int c = 0; c < NJ_Y; c += 32) {
                    uint32_t yr[32];
                    tmem_ld_32x32b_x32(t_lane + ycol + c, yr);
                    tmem_ld_wait(yr);
                    if (valid) {
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            const float v0 = __uint_as_float(yr[4 * j]) * wgt;
                            const float v1 = __uint_as_float(yr[4 * j + 1]) * wgt;
                            const float v2 = __uint_as_float(yr[4 * j + 2]) * wgt;
                            const float v3 = __uint_as_float(yr[4 * j + 3]) * wgt;
                            asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(yrow + c + 4 * j),
                                         "f"(v0), "f"(v1), "f"(v2), "f"(v3)
                                         : "memory");
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) arrive_leader(&y_empty[yb]);
            yph ^= 1u << yb;
        }
        // the reductions must have finished before the block exits
        if (lane == 0) bulk_wait_group_all();
        __syncwarp();
    }

    // Every role is done: all MMAs were consumed by the epilogues (or the
    // launch is aborting, in which case the issuer waited for its MMAs).  In a
    // pair, neither CTA leaves while the leader's MMAs may still read the
    // peer's shared memory or the peer may still arrive on the leader's barriers.
    tc_fence_before();
    __syncthreads();
    if (PAIR) cluster_sync_all();
    if (role == ROLE_MMA) {
        __syncwarp();
        tc_fence_after();
        if (PAIR) tmem_dealloc_pair(tmem_base, TMEM_COLS);
        else tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

}  // namespace tc

static PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    }
    return fn;
}

static bool encode_bytes_map(PFN_cuTensorMapEncodeTiled_v12000 encode, CUtensorMap *m,
                             const void *base, int64_t row_bytes, int64_t rows, int box_bytes,
                             int box_rows) {
    const cuuint64_t dims[2] = {(cuuint64_t)row_bytes, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
    const cuuint32_t box[2] = {(cuuint32_t)box_bytes, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box,
                  estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

cudaError_t launch_ffn_tc(const TcArgs &a, cudaStream_t s) {
    const DeviceInfo &di = device_info();
    auto encode = get_encode_fn();
    if (!encode) return cudaErrorNotSupported;
    // Dense prefill with at least one full pair tile runs on CTA pairs.
    const bool pair = a.tiles == nullptr && a.T >= 256 && di.num_sms >= 2;
    const int rows_y = pair ? tc::Cfg<true>::ROWS_Y : tc::Cfg<false>::ROWS_Y;
    tc::Maps maps;
    {
        const cuuint64_t dims[2] = {(cuuint64_t)a.H, (cuuint64_t)a.x_rows};
        const cuuint64_t strides[1] = {(cuuint64_t)a.H * 2};
        const cuuint32_t box[2] = {tc::BK, tc::BM};
        const cuuint32_t estr[2] = {1, 1};
        CUresult r = encode(&maps.x, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void *>(a.x),
                            dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    }
    {
        const cuuint64_t dims[2] = {(cuuint64_t)a.H, (cuuint64_t)a.T};
        const cuuint64_t strides[1] = {(cuuint64_t)a.H * 4};
        const int ycols = pair ? tc::Cfg<true>::Y_COLS : tc::Cfg<false>::Y_COLS;
        const cuuint32_t box[2] = {(cuuint32_t)ycols, 32};
        const cuuint32_t estr[2] = {1, 1};
        CUresult r = encode(&maps.y, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, a.y, dims, strides, box,
                            estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                            ycols == 32 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    }
    const int64_t rbH = q4k_row_bytes(a.H), rbI = q4k_row_bytes(a.I);
    const int64_t gu_rows = (int64_t)a.E * a.I, d_rows = (int64_t)a.E * a.H;
    if (!encode_bytes_map(encode, &maps.g_hdr, a.Wg, rbH, gu_rows, 16, tc::GU_ROWS) ||
        !encode_bytes_map(encode, &maps.g_qs, a.Wg, rbH, gu_rows, 32, tc::GU_ROWS) ||
        !encode_bytes_map(encode, &maps.u_hdr, a.Wu, rbH, gu_rows, 16, tc::GU_ROWS) ||
        !encode_bytes_map(encode, &maps.u_qs, a.Wu, rbH, gu_rows, 32, tc::GU_ROWS) ||
        !encode_bytes_map(encode, &maps.d_hdr, a.Wd, rbI, d_rows, 16, rows_y) ||
        !encode_bytes_map(encode, &maps.d_qs, a.Wd, rbI, d_rows, 64, rows_y))
        return cudaErrorInvalidValue;
    const void *fn = pair ? (const void *)tc::ffn_tc_kernel<true> : (const void *)tc::ffn_tc_kernel<false>;
    const int smem = pair ? tc::Cfg<true>::SMEM_BYTES : tc::Cfg<false>::SMEM_BYTES;
    {
        cudaError_t e = ensure_dynamic_smem(fn, (size_t)smem);
        if (e != cudaSuccess) return e;
    }
    tc::Params p;
    p.Wg = a.Wg;
    p.Wu = a.Wu;
    p.Wd = a.Wd;
    p.y = a.y;
    p.tiles = a.tiles;
    p.n_tiles_dev = a.n_tiles_dev;
    p.row_token = a.row_token;
    p.row_weight = a.row_weight;
    p.err = a.err;
    p.T = a.T;
    p.H = a.H;
    p.I = a.I;
    const int n_chunks = (a.I + (pair ? tc::Cfg<true>::IC : tc::Cfg<false>::IC) - 1) /
                         (pair ? tc::Cfg<true>::IC : tc::Cfg<false>::IC);
    if (pair) {
        p.n_tiles_host = (a.T + 255) / 256;
        const int64_t units = (int64_t)p.n_tiles_host * n_chunks;
        int64_t pairs = di.num_sms / 2;
        // a programmatic dependent of the x conversion when the units fill
        // every pair (measured: earlier start pays there, costs with idle pairs)
        const bool early = units >= pairs;
        if (units < pairs) pairs = units;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)(2 * pairs));
        cfg.blockDim = dim3(tc::THREADS);
        cfg.dynamicSmemBytes = (size_t)smem;
        cfg.stream = s;
        cudaLaunchAttribute attr[2];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[1].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = early ? 2 : 1;
        return cudaLaunchKernelEx(&cfg, tc::ffn_tc_kernel<true>, maps, p);
    }
    p.n_tiles_host = a.n_tiles_host;
    const int64_t units = (int64_t)a.n_tiles_host * n_chunks;
    int grid = di.num_sms;
    if (units < grid) grid = (int)units;
    if (grid < 1) return cudaSuccess;
    if (a.tiles || units < di.num_sms) {
        // routed tiles: every role reads the tile table, so no early start;
        // nor with idle SMs (as for pairs)
        tc::ffn_tc_kernel<false><<<grid, tc::THREADS, smem, s>>>(maps, p);
        return cudaGetLastError();
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(tc::THREADS);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, tc::ffn_tc_kernel<false>, maps, p);
}

}  // namespace zffn
