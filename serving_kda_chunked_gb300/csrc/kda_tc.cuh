// kda_tc.cuh -- thin inline-PTX wrappers for Blackwell (sm_103a) tensor-core
// kernels: tcgen05 MMA / TMEM, mbarriers, bulk async copies.
//
// Descriptor formats used here (checked on GB300 with a layout probe):
//  * shared-memory matrix descriptor (64 bit): bits 0-13 start address >> 4,
//    16-29 leading byte offset >> 4, 32-45 stride byte offset >> 4, bits 46-47
//    version = 1, bits 61-63 layout (0 = no swizzle, 2 = 128-byte swizzle).
//    - K-major, 128B swizzle: rows of 128 bytes, 8-row atoms of 1024 bytes
//      (SBO = 1024, LBO unused = 16); a K step inside the row adds its byte
//      offset to the start address.
//    - no swizzle (either major-ness): 8 x 16-byte core matrices; LBO is the
//      stride between core matrices along K, SBO the stride along M/N.
//    - MN-major, 128B swizzle: LBO = stride between 64-element MN atoms,
//      SBO = stride between 8-row K groups (1024).
//  * instruction descriptor (kind::f16 / kind::tf32): bits 4-5 D format
//    (1 = f32), 7-9 A format, 10-12 B format (f16 = 0, bf16 = 1, tf32 = 2),
//    13 negate A, 15 A major (1 = MN), 16 B major, 17-22 N >> 3, 24-28 M >> 4.
//  * an M = 64 accumulator occupies TMEM lanes 0-15 of each 32-lane quadrant:
//    row m lives in lane (m / 16) * 32 + m % 16.  M = 128 uses lane = row.
#pragma once

#include <stdint.h>

namespace kda {
namespace tc {

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

// ---- descriptors -------------------------------------------------------------
enum : uint32_t { LAYOUT_NONE = 0, LAYOUT_SW128 = 2 };
enum : uint32_t { FMT_F16 = 0, FMT_BF16 = 1, FMT_TF32 = 2 };

__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo,
                                          uint32_t layout) {
    return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | ((uint64_t)layout << 61);
}
// K-major, 128-byte swizzle (rows of 128 bytes, 1024-byte 8-row atoms).
__device__ __forceinline__ uint64_t sdesc_k_sw128(uint32_t saddr) {
    return sdesc(saddr, 16, 1024, LAYOUT_SW128);
}
// The same descriptor moved by `bytes` (a multiple of 16): only the start
// address field changes, and shared addresses stay below 2^18, so the sum
// never carries out of that 14-bit field.
__device__ __forceinline__ uint64_t sdesc_add(uint64_t desc, uint32_t bytes) {
    return desc + (uint64_t)(bytes >> 4);
}
__host__ __device__ constexpr uint32_t idesc(uint32_t M, uint32_t N, uint32_t afmt,
                                             uint32_t bfmt, uint32_t a_mn, uint32_t b_mn,
                                             uint32_t neg_a = 0) {
    return (1u << 4) | (afmt << 7) | (bfmt << 10) | (neg_a << 13) | (a_mn << 15) |
           (b_mn << 16) | ((N >> 3) << 17) | ((M >> 4) << 24);
}

// ---- warp-uniform values and one elected lane ---------------------------------
// tcgen05.mma takes its TMEM address and matrix descriptors from uniform
// registers.  A value the compiler cannot prove warp-uniform is converted
// before every MMA, which measured ~150-200 cycles per instruction on GB300;
// with uniform operands, an unrolled issue loop and one elected lane, eight
// MMAs issue in ~350 cycles in total.  So every operand of an MMA is passed
// through warp_uniform() in converged code, and the MMAs are issued inside
// `if (elect_one())` by the whole (converged) warp's elected lane -- always the
// same lane, so that its tcgen05.commit tracks every MMA it issued.
__device__ __forceinline__ uint32_t warp_uniform(uint32_t x) {
    return __shfl_sync(0xffffffffu, x, 0);
}
__device__ __forceinline__ bool elect_one() {
    uint32_t pred = 0;
    asm volatile("{\n.reg .b32 rx;\n.reg .pred px;\nelect.sync rx|px, 0xffffffff;\n"
                 "selp.b32 %0, 1, 0, px;\n}" : "=r"(pred));
    return pred != 0;
}

// ---- MMA -----------------------------------------------------------------------
__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t id,
                                        uint32_t accumulate) {
    asm volatile("{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}"
                 :: "r"(d_tmem), "l"(a), "l"(b), "r"(id), "r"(accumulate) : "memory");
}
__device__ __forceinline__ void mma_tf32(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t id,
                                         uint32_t accumulate) {
    asm volatile("{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
                 "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n}"
                 :: "r"(d_tmem), "l"(a), "l"(b), "r"(id), "r"(accumulate) : "memory");
}
// tf32 MMA with the A operand in tensor memory (M rows in lanes, one tf32
// element of K per 32-bit column; the K step moves the address by 8 columns)
// and B in shared memory.
__device__ __forceinline__ void mma_tf32_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t b,
                                                uint32_t id, uint32_t accumulate) {
    asm volatile("{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
                 "tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n}"
                 :: "r"(d_tmem), "r"(a_tmem), "l"(b), "r"(id), "r"(accumulate) : "memory");
}
// Arrive on an mbarrier once every tcgen05 operation issued so far by this
// thread has completed.
__device__ __forceinline__ void mma_commit(uint64_t *mbar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 :: "r"(smem_addr(mbar)) : "memory");
}
__device__ __forceinline__ void fence_before_sync() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_after_sync() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Make generic-proxy shared-memory writes visible to the async proxy (MMA, bulk copy).
__device__ __forceinline__ void fence_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---- TMEM --------------------------------------------------------------------
// One full warp allocates; the base address is written to *dst (shared).
template <uint32_t NCOLS>
__device__ __forceinline__ void tmem_alloc(uint32_t *dst) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 :: "r"(smem_addr(dst)), "n"(NCOLS) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
template <uint32_t NCOLS>
__device__ __forceinline__ void tmem_dealloc(uint32_t base) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;"
                 :: "r"(base), "n"(NCOLS) : "memory");
}
// 32 lanes x 16 consecutive 32-bit columns (one column per register).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 "
                 "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                   "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]),
                   "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
                 : "r"(taddr) : "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
// 32 lanes x 32 consecutive 32-bit columns from registers (one column per
// register); complete once tcgen05.wait::st returns.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
                 "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
                 "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
                 :: "r"(taddr),
                    "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]),
                    "f"(v[7]), "f"(v[8]), "f"(v[9]), "f"(v[10]), "f"(v[11]), "f"(v[12]), "f"(v[13]),
                    "f"(v[14]), "f"(v[15]), "f"(v[16]), "f"(v[17]), "f"(v[18]), "f"(v[19]),
                    "f"(v[20]), "f"(v[21]), "f"(v[22]), "f"(v[23]), "f"(v[24]), "f"(v[25]),
                    "f"(v[26]), "f"(v[27]), "f"(v[28]), "f"(v[29]), "f"(v[30]), "f"(v[31])
                 : "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
// Registers filled by tcgen05.ld are defined only after tcgen05.wait::ld.
// Passing them through an empty volatile asm after the wait stops the
// compiler from moving their uses above it when the load was issued early.
template <int N>
__device__ __forceinline__ void reg_fence(float (&v)[N]) {
#pragma unroll
    for (int i = 0; i < N; ++i) asm volatile("" : "+f"(v[i]));
}
// TMEM address of (lane quadrant base of this warp, column).
__device__ __forceinline__ uint32_t tmem_at(uint32_t base, int warp, int col) {
    return base + ((uint32_t)((warp & 3) * 32) << 16) + (uint32_t)col;
}

// ---- mbarriers -----------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t *mbar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(smem_addr(mbar)), "r"(count)
                 : "memory");
}
__device__ __forceinline__ void mbar_fence_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *mbar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                 :: "r"(smem_addr(mbar)), "r"(bytes) : "memory");
}
// Bounded wait for the phase with the given parity to complete.  Returns
// false if the limit ran out (the caller records the error and unwinds).
__device__ __forceinline__ bool mbar_wait(uint64_t *mbar, uint32_t parity,
                                          uint32_t limit = (1u << 22)) {
    const uint32_t a = smem_addr(mbar);
    for (uint32_t it = 0; it < limit; ++it) {
        uint32_t done;
        asm volatile("{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
                     "selp.b32 %0, 1, 0, p;\n}" : "=r"(done) : "r"(a), "r"(parity) : "memory");
        if (done) return true;
    }
    return false;
}

// ---- bulk async copy (global -> shared), completion counted on an mbarrier ----
__device__ __forceinline__ void bulk_g2s(void *smem_dst, const void *gmem_src, uint32_t bytes,
                                         uint64_t *mbar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 :: "r"(smem_addr(smem_dst)), "l"(gmem_src), "r"(bytes), "r"(smem_addr(mbar))
                 : "memory");
}

// ---- named barriers (subsets of the CTA) -------------------------------------
__device__ __forceinline__ void bar_sync(uint32_t id, uint32_t nthreads) {
    asm volatile("bar.sync %0, %1;" :: "r"(id), "r"(nthreads) : "memory");
}

// ---- byte offsets of canonical layouts ---------------------------------------
// K-major 128B-swizzled tile whose rows hold 128 bytes: byte offset of the
// 16-byte chunk `chunk` (0..7) of row `row`.
__host__ __device__ __forceinline__ uint32_t sw128_off(uint32_t row, uint32_t chunk) {
    return (row >> 3) * 1024u + (row & 7u) * 128u + ((chunk ^ (row & 7u)) << 4);
}

}  // namespace tc
}  // namespace kda
