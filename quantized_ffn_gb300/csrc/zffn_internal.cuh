// zffn_internal.cuh -- shared pieces of the CUDA library: Q4_K unpacking on the
// device, PTX wrappers for mbarrier / TMA / tcgen05, bounded waits, launch
// declarations.  Library-internal; the public interface is include/zffn.h.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "zffn.h"

namespace zffn {

// ---------------------------------------------------------------------------
// Q4_K on the device.  144 bytes per 256 weights: fp16 d, fp16 dmin, 12 bytes
// of 6-bit (scale, min) pairs, 128 bytes of 4-bit codes (byte 32g+l holds
// weight 64g+l in its low nibble and 64g+32+l in its high nibble).
// ---------------------------------------------------------------------------
constexpr int kQK = 256;
constexpr int kBlockBytes = 144;

__host__ __device__ inline int64_t q4k_row_bytes(int64_t cols) {
    return ((cols + kQK - 1) / kQK) * kBlockBytes;
}

// Scales as three little-endian words: s0 = bytes 0..3, s1 = 4..7, s2 = 8..11.
// Sub-block j < 4: scale = low 6 bits of byte j, min = low 6 bits of byte j+4.
// Sub-block j >= 4: low 4 bits in the nibbles of byte j+4, top 2 bits in the
// spare top bits of byte j-4 (scale) and byte j (min).
__device__ __forceinline__ void q4k_scale_min(uint32_t s0, uint32_t s1, uint32_t s2, int j,
                                              int &sc, int &m) {
    if (j < 4) {
        sc = (s0 >> (8 * j)) & 63;
        m = (s1 >> (8 * j)) & 63;
    } else {
        const int jj = j - 4;
        sc = ((s2 >> (8 * jj)) & 15) | (((s0 >> (8 * jj + 6)) & 3) << 4);
        m = ((s2 >> (8 * jj + 4)) & 15) | (((s1 >> (8 * jj + 6)) & 3) << 4);
    }
}

__device__ __forceinline__ float half_bits_to_float(uint32_t bits16) {
    return __half2float(__ushort_as_half((unsigned short)(bits16 & 0xFFFFu)));
}

// ---------------------------------------------------------------------------
// Device error word and bounded waits.
// ---------------------------------------------------------------------------
// Budget of a bounded wait in SM clock cycles (about two seconds at boost
// clock): far above any legitimate wait inside one launch.
constexpr long long kWaitBudgetCycles = 4000000000LL;

__device__ __forceinline__ void record_error(int *err, int code) {
    if (err) atomicCAS(err, 0, code);
}

// ---------------------------------------------------------------------------
// PTX wrappers (sm_100 family).
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void fence_mbarrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
// The same test, allowed to suspend the thread for up to `ns` nanoseconds
// while the phase is incomplete: a waiting thread then takes no issue slots
// from the warps that share its scheduler.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t *bar, uint32_t parity, uint32_t ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(ns)
        : "memory");
    return ok != 0;
}
constexpr uint32_t kWaitSuspendNs = 20000;

// Wait for the phase with the given parity to complete.  Gives up after
// `budget` SM cycles (or as soon as another role raised *abort), records
// ZFFN_ERR_TIMEOUT, raises *abort and returns false.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, volatile int *abort,
                                          int *err, long long budget = kWaitBudgetCycles) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (!mbar_try_wait_sleep(bar, parity, kWaitSuspendNs)) {
        if ((abort && *abort) || clock64() - t0 > budget) {
            record_error(err, ZFFN_ERR_TIMEOUT);
            if (abort) *abort = 1;
            return false;
        }
    }
    return true;
}

// One lane of the (fully active) warp is elected; the rest get false.
__device__ __forceinline__ bool elect_one() {
    uint32_t e;
    asm volatile("{\n\t.reg .pred p;\n\telect.sync _|p, 0xffffffff;\n\tselp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(e));
    return e != 0;
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// 2-D TMA tile load global -> shared, completion counted on `bar` (bytes).
__device__ __forceinline__ void tma_load_2d(void *smem_dst, const CUtensorMap *map, uint64_t *bar,
                                            int c0, int c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1)
        : "memory");
}

// 2-D TMA tile reduction shared -> global: global += tile (fp32 add), tracked
// by the issuing thread's bulk-async group.
__device__ __forceinline__ void tma_reduce_add_2d(const CUtensorMap *map, const void *smem_src,
                                                  int c0, int c1) {
    asm volatile(
        "cp.reduce.async.bulk.tensor.2d.global.shared::cta.add.tile.bulk_group"
        " [%0, {%2, %3}], [%1];" ::"l"(reinterpret_cast<uint64_t>(map)),
        "r"(smem_u32(smem_src)), "r"(c0), "r"(c1)
        : "memory");
}
__device__ __forceinline__ void bulk_commit_group() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Wait until at most N of this thread's bulk groups still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_group_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
// Wait until all of this thread's bulk groups have completed.
__device__ __forceinline__ void bulk_wait_group_all() {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Ask for [gptr, gptr + bytes) to be brought into L2 (bytes a multiple of 16).
__device__ __forceinline__ void prefetch_l2_bulk(const void *gptr, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(gptr), "r"(bytes) : "memory");
}

// ---- tcgen05 ---------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t *dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem desc] * B[smem desc]^T, bf16 inputs, fp32 accumulate.
__device__ __forceinline__ void tc_mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// The same with A read from tensor memory: `a_tmem` addresses lane 0 of the
// first of the K/2 columns holding A's M rows (one row per lane, two 16-bit
// elements per 32-bit column).
__device__ __forceinline__ void tc_mma_f16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                              uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive once on `bar` when every tcgen05 op this thread issued so far completes.
__device__ __forceinline__ void tc_commit(uint64_t *bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}

// ---- CTA pairs (cluster of 2, tcgen05 cta_group::2) ------------------------
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// shared::cluster address of the same shared variable in CTA `rank`
__device__ __forceinline__ uint32_t mapa_shared(uint32_t saddr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                     : "memory");
}
// Arrive on a barrier given by its cluster address (possibly in the peer CTA).
// Default (CTA-scope release) semantics: callers that publish shared-memory
// writes to the tensor cores fence them to the async proxy first.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
// TMA load into this CTA's shared memory whose completion is counted on a
// barrier that may live in the peer CTA of the pair (cluster address).
__device__ __forceinline__ void tma_load_2d_pair(void *smem_dst, const CUtensorMap *map,
                                                 uint32_t bar_cluster_addr, int c0, int c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster_addr), "r"(c0), "r"(c1)
        : "memory");
}
__device__ __forceinline__ void tmem_alloc_pair(uint32_t *dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}
// Pair MMA: D (both CTAs' TMEM) (+)= A (both CTAs' rows) * B (rows split
// between the CTAs)^T.  Issued by one thread of the pair's even CTA.
__device__ __forceinline__ void tc_mma_bf16_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                                 uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Arrive once on the barrier at this shared offset in both CTAs of the pair
// when every tcgen05 op issued so far by this thread completes.
__device__ __forceinline__ void tc_commit_pair(uint64_t *bar) {
    const uint16_t mask = 0x3;
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
        " [%0], %1;" ::"r"(smem_u32(bar)),
        "h"(mask)
        : "memory");
}

// 32 lanes x 32 consecutive 32-bit columns; thread i of the warp gets lane
// (base + i), registers = columns.  The registers are undefined until
// tmem_ld_wait(r) returns.
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
}
__device__ __forceinline__ void tmem_ld_32x32b_x16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}
__device__ __forceinline__ void tmem_ld_wait(uint32_t (&r)[16]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15])
                 :
                 : "memory");
}
__device__ __forceinline__ void tmem_st_32x32b_x8(uint32_t taddr, const uint32_t (&r)[8]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr),
                 "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
                 : "memory");
}
__device__ __forceinline__ void tmem_st_32x32b_x16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
                 ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
                 "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
                 : "memory");
}
__device__ __forceinline__ void tmem_st_wait() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
// Wait for every tcgen05.ld of this thread; the registers of `r` are passed
// through the wait so that no use of them can be scheduled before it.
__device__ __forceinline__ void tmem_ld_wait(uint32_t (&r)[32]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
                 :
                 : "memory");
}

// Shared-memory matrix descriptor, K-major, 128-byte swizzle: rows of 128 bytes
// (64 bf16), groups of 8 rows 1024 bytes apart; the tile starts 1024-aligned.
__device__ __forceinline__ uint64_t smem_desc_k_sw128(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);  // start address
    d |= (uint64_t)1 << 16;                    // leading byte offset (unused here)
    d |= (uint64_t)(1024 >> 4) << 32;          // stride byte offset: 8-row groups
    d |= (uint64_t)1 << 46;                    // descriptor version (sm_100 family)
    d |= (uint64_t)2 << 61;                    // 128-byte swizzle
    return d;
}

// Instruction descriptor: kind::f16 with A = B = fp16 (format code 0),
// D = fp32, both K-major.
__host__ __device__ constexpr uint32_t idesc_f16_f32(int M, int N) {
    return (1u << 4)                          // D format f32
           | ((uint32_t)(N >> 3) << 17)       // N / 8
           | ((uint32_t)(M >> 4) << 24);      // M / 16
}


// Two 4-bit codes as fp16: the low 16 bits of `v` hold two bytes, each a code
// 0..15.  Read as an e4m3 bit pattern, a byte 0000qqqq is q * 2^-9 exactly
// (exponent field 0: subnormal (q & 7) / 8 * 2^-6; exponent field 1 for
// q >= 8: (1 + (q & 7) / 8) * 2^-6), so the fp8 -> fp16 converter turns the
// pair into fp16 (q0 * 2^-9, q1 * 2^-9) without rounding.
__device__ __forceinline__ uint32_t codes_to_f16x2(uint32_t v) {
    uint32_t r;
    asm("{\n\t.reg .b16 t;\n\tcvt.u16.u32 t, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, t;\n\t}" : "=r"(r) : "r"(v));
    return r;
}
// a * b + c on fp16 pairs, rounded once.
__device__ __forceinline__ uint32_t fma_f16x2(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t r;
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(c));
    return r;
}
// fp32 -> fp16 (nearest), clamped to the largest finite fp16, in both halves.
__device__ __forceinline__ uint32_t f16x2_splat_satfinite(float v) {
    uint32_t r;
    asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %1;" : "=r"(r) : "f"(v));
    return r;
}

// bf16 pair (one 32-bit word) -> fp16 pair: both widen exactly to fp32, then
// round to fp16 (nearest, saturating at +-65504).
__device__ __forceinline__ uint32_t bf16x2_to_f16x2_satfinite(uint32_t w) {
    uint32_t r;
    asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;"
        : "=r"(r)
        : "f"(__uint_as_float(w & 0xFFFF0000u)), "f"(__uint_as_float(w << 16)));
    return r;
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}


// ---------------------------------------------------------------------------
// Q4_K -> fp16 operand tiles of the tensor-core kernels.
// ---------------------------------------------------------------------------
// Byte offset of row r in a [rows x 64] bf16 tile laid out K-major with the
// 128-byte swizzle (groups of 8 rows, 1024 bytes apart); 16-byte chunk c of
// the row sits at chunk position c ^ (r % 8).
__device__ __forceinline__ uint32_t sw128_row(int r) {
    return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128);
}

__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}




// Four code bytes (each a code 0..15) -> the fp16 weights of bytes 0-1 (o0) and
// 2-3 (o1): w = (q * 2^-9) * a + b with a, b fp16 pairs (see codes_to_f16x2).
__device__ __forceinline__ void codes4_to_f16(uint32_t v, uint32_t a, uint32_t b, uint32_t &o0, uint32_t &o1) {
    uint32_t c0, c1;
    asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\tcvt.rn.f16x2.e4m3x2 %0, l;\n\t"
        "cvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
        : "=r"(c0), "=r"(c1)
        : "r"(v));
    o0 = fma_f16x2(c0, a, b);
    o1 = fma_f16x2(c1, a, b);
}

// fp16 scale and offset pairs (512 d sc, -dmin m) of the four sub-blocks
// sb0 .. sb0+3 of a Q4_K block header (sb0 = 0 or 4).
__device__ __forceinline__ void q4k_f16_scales4(uint4 hd, int sb0, uint32_t (&a)[4], uint32_t (&b)[4]) {
    const float d = 512.0f * half_bits_to_float(hd.x), dmin = half_bits_to_float(hd.x >> 16);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        int sc, m;
        q4k_scale_min(hd.y, hd.z, hd.w, sb0 + j, sc, m);
        a[j] = f16x2_splat_satfinite(d * (float)sc);
        b[j] = f16x2_splat_satfinite(-(dmin * (float)m));
    }
}

// ---------------------------------------------------------------------------
// Host-side launchers (defined in the kernel translation units).
// ---------------------------------------------------------------------------
struct DeviceInfo {
    int device = -1;
    int num_sms = 0;
    int max_smem_optin = 0;
    int *err_word = nullptr;   // device error word of this device
};
const DeviceInfo &device_info();   // current device (cached per device)
void set_last_error(const char *what);   // text returned by zffn_last_error()
// Raise `fn`'s dynamic shared-memory limit on the current device to at least
// `bytes` (never lowers it).  Thread-safe: one lock covers the check, the
// attribute call and the per-device record of the largest request so far.
cudaError_t ensure_dynamic_smem(const void *fn, size_t bytes);

cudaError_t launch_q4k_dequant(const void *blocks, float *out, int64_t rows, int64_t cols,
                               cudaStream_t s);
cudaError_t launch_q4k_quantize(const float *w, void *blocks, int64_t rows, int64_t cols,
                                cudaStream_t s);
// x (bf16, n values, n % 8 == 0, 16-byte aligned) -> x16 (fp16, saturating);
// if y_zero is not null, also y_zero[0, ny) = 0.
cudaError_t launch_x_to_f16(const void *x, void *x16, int64_t n, float *y_zero, int64_t ny,
                            cudaStream_t s);

// Single-token path: a gate/up kernel (SwiGLU into an on-device strip h)
// followed by a down-projection kernel launched as its programmatic
// dependent.
struct MatvecArgs {
    const __nv_bfloat16 *x;      // [T][H]
    const uint8_t *Wg, *Wu, *Wd; // expert-stacked
    const int32_t *ids;          // [T][k] or nullptr (dense: expert 0, weight 1)
    const float *wts;            // [T][k] or nullptr
    const float *down_scale;     // [E] scale of each expert's down projection, or nullptr
    float *y;                    // [T][H]
    float *h;                    // workspace [T*k][I]
    int *err;
    int T, H, I, E, k;
    bool accumulate;             // y += result instead of y = result
    int ring_depth;              // set by the launcher: row buffers per warp in the down kernel
    unsigned long long *gbar;    // routed only: the one-launch path's grid-barrier count (zero
                                 // before its first use), or nullptr for the two-kernel path
    // Dense only, or nullptr: the gate/up kernel builds x itself as
    // bf16(RMSNorm(norm_in) * gamma) from this fp32 row (x is then unused)
    const float *norm_in;
    const float *gamma;
    float eps;
};
size_t matvec_smem_bytes(int T, int H, int I, int k);
// The same with the RMSNorm folded into the gate/up kernel (dense, T = 1).
size_t matvec_smem_bytes_prenorm(int H, int I);
// The one-launch routed single-token path fits these sizes on this device.
bool token_fused_fits_dims(int H, int I, int k);
cudaError_t launch_ffn_matvec(const MatvecArgs &a, cudaStream_t s);

// Tensor-core fused prefill path.
struct TcArgs {
    const void *x;               // fp16 rows (dense x converted, or the gathered MoE rows)
    int64_t x_rows;              // rows of x visible to the tensor map
    const uint8_t *Wg, *Wu, *Wd;
    float *y;                    // [T][H], zero-filled before the launch
    // Dense: tiles == nullptr, tokens taken as x rows.  MoE: tile table and
    // per-row (token, weight) maps produced on the device by the router pass.
    const int4 *tiles;           // {row_start, row_count, expert, 0}
    const int *n_tiles_dev;      // device count of tiles
    const int *row_token;        // x row -> token
    const float *row_weight;     // x row -> routing weight
    int n_tiles_host;            // dense: exact count; MoE: upper bound
    int *err;
    int T, H, I;
    int E;                       // experts stacked in Wg/Wu/Wd (dense: 1)
};
cudaError_t launch_ffn_tc(const TcArgs &a, cudaStream_t s);
// Routed layer with few rows per expert: groups of at most moe_group_rows()
// gathered rows of one expert, weights as the MMA's M side (moe_tc.cu).
int moe_group_rows();
// wd_fmt: the W_down block format (Q4_K, Q5_K or Q5_1; a.Wd rows of its row bytes)
cudaError_t launch_moe_group(const TcArgs &a, int wd_fmt, cudaStream_t s);

// MoE routing on the device: bucket (token, slot) pairs by expert, build the
// tile table and the row maps, gather x rows per expert.
struct RouteArgs {
    const int32_t *ids;
    const float *wts;
    const float *down_scale;   // [E] or nullptr: multiplies each row's routing weight
    const __nv_bfloat16 *x;
    int T, H, E, k;
    int *counts;        // [E]
    int *offsets;       // [E + 1]
    int *cursors;       // [E]
    int4 *tiles;        // [max_tiles]
    int *n_tiles;       // [1]
    int *row_token;     // [T*k]
    float *row_weight;  // [T*k]
    __half *x_perm;     // [T*k][H] gathered rows, converted to fp16
    int max_tiles;
    int tile_rows;      // rows per tile: 128 (prefill kernel) or the grouped kernel's group
    float *y_zero;      // [ny] set to zero by the gather kernel (the block then adds into it), or nullptr
    int64_t ny;
};
cudaError_t launch_moe_route(const RouteArgs &a, cudaStream_t s);
// The tile table of a dense block run as one expert: groups of `rows`
// consecutive tokens, row_token[i] = i, row_weight[i] = 1.
cudaError_t launch_dense_groups(int T, int rows, int4 *tiles, int *n_tiles, int *row_token, float *row_weight,
                                cudaStream_t s);

cudaError_t launch_wait_timeout_selftest(int64_t budget_cycles, int *err, cudaStream_t s);

}  // namespace zffn
