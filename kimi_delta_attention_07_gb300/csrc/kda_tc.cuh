// Blackwell (sm_103a) building blocks for the tensor-core chunk path:
// mbarriers, bulk copies, TMEM allocation, tcgen05.mma with shared-memory
// operands, tcgen05.ld, and the 128-byte-swizzled K-major operand layout.
// Hand-written inline PTX; no CUTLASS.
#pragma once

#include <stdint.h>

namespace kda {
namespace tc {

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

// ---- mbarrier -----------------------------------------------------------------

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return done != 0;
}
// Wait for the phase of `parity` to complete, giving up after ~max_cycles SM
// clocks.  Returns false on timeout (the caller records an error and exits).
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity,
                                          long long max_cycles = 4000000000LL) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (clock64() - t0 > max_cycles) return false;
    }
    return true;
}

// ---- bulk copy (global -> shared, completes on an mbarrier) ---------------------
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes,
                                         uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// ---- bulk copy (shared -> global, bulk-group completion) -----------------------
// dst, src 16-byte aligned; bytes a multiple of 16.  The issuing thread tracks
// completion: bulk_wait_read() returns once every committed copy has read its
// shared-memory source, bulk_wait_all() once the writes are done.
__device__ __forceinline__ void bulk_s2g(void *dst, const void *src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst),
                 "r"(smem_u32(src)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_all() {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// ---- TMA tensor copy (3-D tile, global -> shared, completes on an mbarrier) ----------
// tmap: generic address of a CUtensorMap kernel parameter; c0 (innermost) must
// keep the copied row 16-byte aligned (here always 0).
__device__ __forceinline__ void tma_load_3d(void *dst, const void *tmap, int c0, int c1, int c2,
                                            uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
        "l"(tmap), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
        : "memory");
}

// Prefetch the same tile into L2 only (no shared memory, no barrier).
__device__ __forceinline__ void tma_prefetch_3d(const void *tmap, int c0, int c1, int c2) {
    asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(tmap),
                 "r"(c0), "r"(c1), "r"(c2)
                 : "memory");
}
__device__ __forceinline__ void prefetch_l2(const void *p) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p) : "memory");
}

// ---- named barrier `id` (1..15; 0 is __syncthreads): returns once `count`
// threads (whole warps) have arrived at it.
__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// named barrier `id` with an AND-reduction of `pred` over its `count` threads
__device__ __forceinline__ bool named_bar_and(uint32_t id, uint32_t count, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}\n"
        : "=r"(r)
        : "r"((uint32_t)pred), "r"(id), "r"(count)
        : "memory");
    return r != 0;
}

// ---- fences -----------------------------------------------------------------------
// generic-proxy shared-memory writes -> visible to the tensor core (async proxy)
__device__ __forceinline__ void fence_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// ---- ready flags between kernels that run at the same time ---------------------------
// The writer publishes once its data is written: its own bulk copies complete
// (bulk_wait_all) and the other threads' stores ordered before it by a CTA
// barrier; the proxy fence orders the bulk copies' writes before the release.
__device__ __forceinline__ void flag_publish(int32_t *p) {
    asm volatile("fence.proxy.async.global;\n\tst.release.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(1)
                 : "memory");
}
__device__ __forceinline__ int32_t flag_peek(const int32_t *p) {
    int32_t v;
    asm volatile("ld.relaxed.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ int32_t flag_load_acquire(const int32_t *p) {
    int32_t v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
// The reader: once a relaxed read has seen the flag, this fence makes it an
// acquire, and the proxy fence orders the bulk copies issued next after it.
__device__ __forceinline__ void flag_acquire() {
    asm volatile("fence.acq_rel.gpu;\n\tfence.proxy.async.global;" ::: "memory");
}
// Wait until *p is nonzero with acquiring reads (an acquiring read costs its
// thread one L2 round trip; a fence after a relaxed read costs about twice
// that, more with copies in flight), giving up after ~max_cycles SM clocks;
// the proxy fence orders the bulk copies issued next after it.  False on
// timeout.
__device__ __forceinline__ bool flag_wait(const int32_t *p, long long max_cycles = 4000000000LL) {
    if (!flag_load_acquire(p)) {
        const long long t0 = clock64();
        while (!flag_load_acquire(p)) {
            if (clock64() - t0 > max_cycles) return false;
        }
    }
    asm volatile("fence.proxy.async.global;" ::: "memory");
    return true;
}
// A counter that kernels running at the same time raise as they finish.
__device__ __forceinline__ void count_release(int32_t *p) {
    asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(1) : "memory");
}
__device__ __forceinline__ bool count_wait(const int32_t *p, int32_t target,
                                           long long max_cycles = 4000000000LL) {
    const long long t0 = clock64();
    while (flag_peek(p) < target) {
        if (clock64() - t0 > max_cycles) return false;
        __nanosleep(256);
    }
    flag_acquire();
    return true;
}

// ---- TMEM ---------------------------------------------------------------------------
// Executed by one full warp; the TMEM base address is written to *dst.
__device__ __forceinline__ void tmem_alloc(uint32_t *dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(dst)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

// 32 consecutive fp32 columns of this thread's TMEM lane (warp w reads lanes
// 32*(w%4) .. 32*(w%4)+31; taddr carries that lane base in bits 16..31).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&r)[32]) {
    uint32_t *u = reinterpret_cast<uint32_t *>(r);
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(u[0]), "=r"(u[1]), "=r"(u[2]), "=r"(u[3]), "=r"(u[4]), "=r"(u[5]), "=r"(u[6]),
          "=r"(u[7]), "=r"(u[8]), "=r"(u[9]), "=r"(u[10]), "=r"(u[11]), "=r"(u[12]),
          "=r"(u[13]), "=r"(u[14]), "=r"(u[15]), "=r"(u[16]), "=r"(u[17]), "=r"(u[18]),
          "=r"(u[19]), "=r"(u[20]), "=r"(u[21]), "=r"(u[22]), "=r"(u[23]), "=r"(u[24]),
          "=r"(u[25]), "=r"(u[26]), "=r"(u[27]), "=r"(u[28]), "=r"(u[29]), "=r"(u[30]),
          "=r"(u[31])
        : "r"(taddr));
}
// 16 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&r)[16]) {
    uint32_t *u = reinterpret_cast<uint32_t *>(r);
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(u[0]), "=r"(u[1]), "=r"(u[2]), "=r"(u[3]), "=r"(u[4]), "=r"(u[5]), "=r"(u[6]),
          "=r"(u[7]), "=r"(u[8]), "=r"(u[9]), "=r"(u[10]), "=r"(u[11]), "=r"(u[12]),
          "=r"(u[13]), "=r"(u[14]), "=r"(u[15])
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// ---- UMMA operand layout: K-major, 128-byte swizzle, bf16 ------------------------------
//
// A [rows x K] operand tile (K a multiple of 64) is stored as K/64 "K-blocks",
// each [rows][64] bf16 = rows x 128 bytes; 8-row groups form 1024-byte swizzle
// atoms in which the 16-byte chunk c of row r sits at chunk position c ^ (r % 8).
// Tiles start on a 1024-byte boundary.

__host__ __device__ __forceinline__ uint32_t sw128_off(int row, int k, int rows) {
    const int kb = k >> 6, kk = k & 63;
    return (uint32_t)(kb * rows * 128 + row * 128 + ((((kk >> 3) ^ (row & 7))) << 4) +
                      ((kk & 7) << 1));
}

// Shared-memory matrix descriptor of a K-major SW128 tile starting at saddr.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);  // start address >> 4
    d |= (uint64_t)1 << 16;                    // leading byte offset (unused: swizzled K-major)
    d |= (uint64_t)(1024 >> 4) << 32;          // stride byte offset: one 8-row atom
    d |= (uint64_t)1 << 46;                    // tcgen05 descriptor version
    d |= (uint64_t)2 << 61;                    // 128-byte swizzle
    return d;
}

// Instruction descriptor, kind::f16: bf16 A and B (both K-major), fp32 D.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) |
           ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// High 32 bits of every SW128 K-major descriptor used here (stride byte
// offset 1024, tcgen05 version bit, 128-byte swizzle); see sw128_desc.
constexpr uint32_t kDescHi = (uint32_t)(1024 >> 4) | (1u << 14) | (2u << 29);

__device__ __forceinline__ uint32_t sw128_desc_lo(uint32_t saddr) {
    return ((saddr & 0x3FFFFu) >> 4) | (1u << 16);
}

// Operands of mma_tile:
//   K-major SW128: [rows][K] in K-blocks of 64 (see sw128_off); ROWS = rows of
//     the tile; a K=16 step moves the start address by 32 bytes inside the
//     swizzle atom (next K-block: +ROWS * 128 bytes).
//   MN-major SW128: [K][MN] with MN split in 64-element blocks of K rows x 128
//     bytes (the same byte formula as sw128_off(k, mn, K)); block stride
//     (leading byte offset) = K * 128, 8-row groups 1024 bytes apart; a K=16
//     step moves the start address by 2048 bytes.
template <bool MN_MAJOR, int ROWS_OR_K>
__device__ __forceinline__ uint32_t operand_lo(uint32_t saddr, int s) {
    if (MN_MAJOR)
        return (((saddr & 0x3FFFFu) >> 4) | ((uint32_t)((ROWS_OR_K * 128) >> 4) << 16)) + (uint32_t)(s * 128);
    return sw128_desc_lo(saddr) + (uint32_t)((s >> 2) * ROWS_OR_K * 8 + (s & 3) * 2);
}

// D[M x N] (+)= A[M x K] * B[N x K]^T on SW128 tiles, issued by one thread.
// AROWS / BROWS: rows of a K-major operand tile; for an MN-major operand
// (A_MN / B_MN) pass K.  The descriptors of the K steps differ only in their
// low word (start address), by constants.
template <int M, int N, int K, int AROWS, int BROWS, bool A_MN = false, bool B_MN = false>
__device__ __forceinline__ void mma_tile(uint32_t d_tmem, uint32_t a_saddr, uint32_t b_saddr,
                                         bool accumulate) {
    constexpr uint32_t idesc =
        idesc_bf16(M, N) | (A_MN ? (1u << 15) : 0u) | (B_MN ? (1u << 16) : 0u);
#pragma unroll
    for (int s = 0; s < K / 16; ++s) {
        const uint64_t ad = ((uint64_t)kDescHi << 32) | (uint64_t)operand_lo<A_MN, AROWS>(a_saddr, s);
        const uint64_t bd = ((uint64_t)kDescHi << 32) | (uint64_t)operand_lo<B_MN, BROWS>(b_saddr, s);
        mma_bf16(d_tmem, ad, bd, idesc, (accumulate || s > 0) ? 1u : 0u);
    }
}

// B operand with N = 32, MN-major, 64-byte swizzle: one 64-byte row per K
// index, element (n, k) at sw64_off(k, n); 8-row groups 512 bytes apart, a K=16
// step moves the start address by 1024 bytes.  Tiles start on a 1024-byte
// boundary.
__host__ __device__ __forceinline__ uint32_t sw64_off(int k, int n) {
    return (uint32_t)(k * 64 + ((((n >> 3) ^ ((k >> 1) & 3))) << 4) + ((n & 7) << 1));
}
constexpr uint32_t kDescHiSw64 = (uint32_t)(512 >> 4) | (1u << 14) | (4u << 29);

// D[M x 32] (+)= A[M x K] * B[32 x K]^T, A as in mma_tile, B as above.
template <int M, int K, int AROWS, bool A_MN = false>
__device__ __forceinline__ void mma_tile_n32(uint32_t d_tmem, uint32_t a_saddr, uint32_t b_saddr,
                                             bool accumulate) {
    constexpr uint32_t idesc = idesc_bf16(M, 32) | (A_MN ? (1u << 15) : 0u) | (1u << 16);
    const uint32_t b_lo = (b_saddr & 0x3FFFFu) >> 4;
#pragma unroll
    for (int s = 0; s < K / 16; ++s) {
        const uint64_t ad = ((uint64_t)kDescHi << 32) | (uint64_t)operand_lo<A_MN, AROWS>(a_saddr, s);
        const uint64_t bd = ((uint64_t)kDescHiSw64 << 32) | (uint64_t)(b_lo + (uint32_t)(s * 64));
        mma_bf16(d_tmem, ad, bd, idesc, (accumulate || s > 0) ? 1u : 0u);
    }
}

__device__ __forceinline__ void mma_commit(uint64_t *bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}

}  // namespace tc
}  // namespace kda
