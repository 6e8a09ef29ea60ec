// cp_ptx.cuh -- thin inline-PTX wrappers for sm_103a: mbarriers, TMA tensor
// loads, tcgen05 (TMEM allocation, MMA, commit, TMEM load/store) and fences.
// Internal to libcpattn; formats follow the public PTX ISA (shared-memory
// matrix descriptor and the kind::f16 instruction descriptor of tcgen05.mma).
#pragma once
#include <cstdint>
#include <cuda.h>

namespace cpattn {

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar_addr, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar_addr), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait for the phase of parity `parity` to complete.  Returns false
// (and raises *abort_flag) when `timeout_ns` elapses or when another thread
// has already raised *abort_flag; every caller then unwinds.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                          uint64_t timeout_ns) {
    const uint32_t a = smem_u32(bar);
    if (mbar_try_wait(a, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(a, parity)) return true;
        if ((it & 31u) == 0u) {
            if (*abort_flag) return false;
            if (global_timer_ns() - t0 > timeout_ns) {
                *abort_flag = 1;
                return false;
            }
        }
    }
}

// mbar_wait by every lane of a warp with one warp-wide answer: a lane that
// gave up (timeout or abort) makes the whole warp give up, so the warp never
// splits around the warp-collective tcgen05 instructions that follow.  Lanes
// still spinning see the raised abort flag and stop as well.
__device__ __forceinline__ bool mbar_wait_warp(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                               uint64_t timeout_ns) {
    const bool ok = mbar_wait(bar, parity, abort_flag, timeout_ns);
    return __all_sync(0xffffffffu, ok);
}

// ---------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}
// 4-D tiled load into shared memory; completion is signalled on `bar` as
// transaction bytes.  c0 is the innermost coordinate (elements).
__device__ __forceinline__ void tma_load_4d(void *smem_dst, const CUtensorMap *map, uint64_t *bar, int c0,
                                            int c1, int c2, int c3) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
        : "memory");
}

// 2-D tiled load (innermost coordinate c0 in elements).
__device__ __forceinline__ void tma_load_2d(void *smem_dst, const CUtensorMap *map, uint64_t *bar, int c0, int c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1)
        : "memory");
}

// ---------------------------------------------------------------- tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t *smem_result, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(smem_result)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor (tcgen05): start address >> 4 in [0,14),
// leading byte offset >> 4 in [16,30), stride byte offset >> 4 in [32,46),
// fixed 0b001 in [46,49), base offset 0, relative LBO, swizzle mode in
// [61,64) (2 = 128-byte swizzle).
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32;
    d |= static_cast<uint64_t>(1u) << 46;
    d |= static_cast<uint64_t>(2u) << 61;
    return d;
}

// Instruction descriptor, kind::f16: D fp32 (bits 4-5 = 1), A and B bf16
// (bits 7-9 = 1, 10-12 = 1), A/B major in bits 15/16 (0 = K-major,
// 1 = MN-major), N >> 3 in bits 17-22, M >> 4 in bits 24-28.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(uint32_t M, uint32_t N, uint32_t a_mn_major,
                                                      uint32_t b_mn_major) {
    return (1u << 4) | (1u << 7) | (1u << 10) | (a_mn_major << 15) | (b_mn_major << 16) | ((N >> 3) << 17) |
           ((M >> 4) << 24);
}

// S = Q K^T for one 128-row tile: D/16 MMAs (K = 16 each) over the 128-byte
// swizzled K-major tiles whose descriptors for k-step 0 are `a` and `b`; k-step
// kk starts (kk / 4) * 16 KB + (kk % 4) * 32 B further (descriptor units of
// 16 B: (kk / 4) * 1024 + (kk % 4) * 2).  The first MMA overwrites D.
template <int NK>
__device__ __forceinline__ void umma_qk_group(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc) {
    static_assert(NK == 4 || NK == 8, "head dim 64 or 128");
    if (NK == 8) {
        asm volatile(
            "{\n\t.reg .pred t, f;\n\t.reg .b64 a1, b1;\n\t"
            "setp.ne.b32 t, %4, 0;\n\tsetp.eq.b32 f, %4, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, f;\n\t"
            "add.s64 a1, %1, 2;\n\tadd.s64 b1, %2, 2;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], a1, b1, %3, t;\n\t"
            "add.s64 a1, %1, 4;\n\tadd.s64 b1, %2, 4;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], a1, b1, %3, t;\n\t"
            "add.s64 a1, %1, 6;\n\tadd.s64 b1, %2, 6;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], a1, b1, %3, t;\n\t"
            "add.s64 a1, %1, 1024;\n\tadd.s64 b1, %2, 1024;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], a1, b1, %3, t;\n\t"
            "add.s64 a1, %1, 1026;\n\tadd.s64 b1, %2, 1026;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], a1, b1, %3, t;\n\t"
            "add.s64 a1, %1, 1028;\n\tadd.s64 b1, %2, 1028;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], a1, b1, %3, t;\n\t"
            "add.s64 a1, %1, 1030;\n\tadd.s64 b1, %2, 1030;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], a1, b1, %3, t;\n\t"
            "}" ::"r"(d_tmem),
            "l"(a), "l"(b), "r"(idesc), "r"(1u)
            : "memory");
    } else {
        asm volatile(
            "{\n\t.reg .pred t, f;\n\t.reg .b64 a1, b1;\n\t"
            "setp.ne.b32 t, %4, 0;\n\tsetp.eq.b32 f, %4, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, f;\n\t"
            "add.s64 a1, %1, 2;\n\tadd.s64 b1, %2, 2;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], a1, b1, %3, t;\n\t"
            "add.s64 a1, %1, 4;\n\tadd.s64 b1, %2, 4;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], a1, b1, %3, t;\n\t"
            "add.s64 a1, %1, 6;\n\tadd.s64 b1, %2, 6;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], a1, b1, %3, t;\n\t"
            "}" ::"r"(d_tmem),
            "l"(a), "l"(b), "r"(idesc), "r"(1u)
            : "memory");
    }
}
// O (+)= P V for one 128-row tile and 128 keys: 8 MMAs (K = 16 keys each), P
// read from TMEM starting at column `a_tmem` (8 columns per k-step), V from
// the MN-major swizzled tile whose descriptor for keys 0..15 is `b` (next 16
// keys: +2048 B, i.e. +128 in descriptor units).  `acc` = 0 overwrites O with
// the first product.
__device__ __forceinline__ void umma_pv_group(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                              uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred t, p;\n\t.reg .b64 b1;\n\t.reg .b32 a1;\n\t"
        "setp.ne.b32 t, %5, 0;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t"
        "add.u32 a1, %1, 8;\n\tadd.s64 b1, %2, 128;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], [a1], b1, %3, t;\n\t"
        "add.u32 a1, %1, 16;\n\tadd.s64 b1, %2, 256;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], [a1], b1, %3, t;\n\t"
        "add.u32 a1, %1, 24;\n\tadd.s64 b1, %2, 384;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], [a1], b1, %3, t;\n\t"
        "add.u32 a1, %1, 32;\n\tadd.s64 b1, %2, 512;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], [a1], b1, %3, t;\n\t"
        "add.u32 a1, %1, 40;\n\tadd.s64 b1, %2, 640;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], [a1], b1, %3, t;\n\t"
        "add.u32 a1, %1, 48;\n\tadd.s64 b1, %2, 768;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], [a1], b1, %3, t;\n\t"
        "add.u32 a1, %1, 56;\n\tadd.s64 b1, %2, 896;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], [a1], b1, %3, t;\n\t"
        "}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc), "r"(1u)
        : "memory");
}

// D = A B^T over NK k-steps of 16 (K = 16 NK) with both operands K-major,
// 128-byte swizzled: k-step kk starts (kk / 4) swizzle atoms + (kk % 4) * 32 B
// further in each operand, an atom of A being AU and of B being BU descriptor
// units (16 B; a 128-row atom is 1024 units, a 64-row atom 512).  The first
// MMA overwrites D.
template <int NK, int AU, int BU>
__device__ __forceinline__ void umma_ss_kgroup(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc) {
    static_assert(NK == 4 || NK == 8, "head dim 64 or 128");
    if (NK == 8) {
        asm volatile(
            "{\n\t.reg .pred t, f;\n\t.reg .b64 a1, b1;\n\t"
            "setp.ne.b32 t, %4, 0;\n\tsetp.eq.b32 f, %4, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, f;\n\t"
            "add.s64 a1, %1, 2;\n\tadd.s64 b1, %2, 2;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], a1, b1, %3, t;\n\t"
            "add.s64 a1, %1, 4;\n\tadd.s64 b1, %2, 4;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], a1, b1, %3, t;\n\t"
            "add.s64 a1, %1, 6;\n\tadd.s64 b1, %2, 6;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], a1, b1, %3, t;\n\t"
            "add.s64 a1, %1, %5;\n\tadd.s64 b1, %2, %9;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], a1, b1, %3, t;\n\t"
            "add.s64 a1, %1, %6;\n\tadd.s64 b1, %2, %10;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], a1, b1, %3, t;\n\t"
            "add.s64 a1, %1, %7;\n\tadd.s64 b1, %2, %11;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], a1, b1, %3, t;\n\t"
            "add.s64 a1, %1, %8;\n\tadd.s64 b1, %2, %12;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], a1, b1, %3, t;\n\t"
            "}" ::"r"(d_tmem),
            "l"(a), "l"(b), "r"(idesc), "r"(1u), "n"(AU), "n"(AU + 2), "n"(AU + 4), "n"(AU + 6), "n"(BU),
            "n"(BU + 2), "n"(BU + 4), "n"(BU + 6)
            : "memory");
    } else {
        asm volatile(
            "{\n\t.reg .pred t, f;\n\t.reg .b64 a1, b1;\n\t"
            "setp.ne.b32 t, %4, 0;\n\tsetp.eq.b32 f, %4, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, f;\n\t"
            "add.s64 a1, %1, 2;\n\tadd.s64 b1, %2, 2;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], a1, b1, %3, t;\n\t"
            "add.s64 a1, %1, 4;\n\tadd.s64 b1, %2, 4;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], a1, b1, %3, t;\n\t"
            "add.s64 a1, %1, 6;\n\tadd.s64 b1, %2, 6;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], a1, b1, %3, t;\n\t"
            "}" ::"r"(d_tmem),
            "l"(a), "l"(b), "r"(idesc), "r"(1u)
            : "memory");
    }
}
// D (+)= A B over K = 64 (4 k-steps of 16): A read from TMEM starting at
// column `a_tmem` (8 columns of packed bf16 pairs per k-step), B from an
// MN-major swizzled tile whose descriptor for rows 0..15 is `b` (next 16
// rows: +2048 B = +128 units).  `acc` = 0 overwrites D with the first product.
__device__ __forceinline__ void umma_ts_k64(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                            uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred t, p;\n\t.reg .b64 b1;\n\t.reg .b32 a1;\n\t"
        "setp.ne.b32 t, %5, 0;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t"
        "add.u32 a1, %1, 8;\n\tadd.s64 b1, %2, 128;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], [a1], b1, %3, t;\n\t"
        "add.u32 a1, %1, 16;\n\tadd.s64 b1, %2, 256;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], [a1], b1, %3, t;\n\t"
        "add.u32 a1, %1, 24;\n\tadd.s64 b1, %2, 384;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], [a1], b1, %3, t;\n\t"
        "}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc), "r"(1u)
        : "memory");
}

// umma_ts_k64 with the A operand's four k-steps at TMEM columns a, a+8, a+32,
// a+40 (two 16-column blocks 32 columns apart).
__device__ __forceinline__ void umma_ts_k64_split(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                                  uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred t, p;\n\t.reg .b64 b1;\n\t.reg .b32 a1;\n\t"
        "setp.ne.b32 t, %5, 0;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t"
        "add.u32 a1, %1, 8;\n\tadd.s64 b1, %2, 128;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], [a1], b1, %3, t;\n\t"
        "add.u32 a1, %1, 32;\n\tadd.s64 b1, %2, 256;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], [a1], b1, %3, t;\n\t"
        "add.u32 a1, %1, 40;\n\tadd.s64 b1, %2, 384;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], [a1], b1, %3, t;\n\t"
        "}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc), "r"(1u)
        : "memory");
}

// Arrive once on `bar` when every tcgen05 operation issued so far by this
// thread has completed.
__device__ __forceinline__ void umma_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

#define CP_R8(a, i) "=r"(a[i]), "=r"(a[i + 1]), "=r"(a[i + 2]), "=r"(a[i + 3]), "=r"(a[i + 4]), "=r"(a[i + 5]), \
                    "=r"(a[i + 6]), "=r"(a[i + 7])
#define CP_W8(a, i) "r"(a[i]), "r"(a[i + 1]), "r"(a[i + 2]), "r"(a[i + 3]), "r"(a[i + 4]), "r"(a[i + 5]), \
                    "r"(a[i + 6]), "r"(a[i + 7])

// Load 32 consecutive 32-bit TMEM columns of this thread's lane (warp-wide,
// 32x32b shape) and wait for completion inside the same asm statement, so the
// compiler cannot touch the registers early.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : CP_R8(r, 0), CP_R8(r, 8), CP_R8(r, 16), CP_R8(r, 24)
        : "r"(taddr)
        : "memory");
}
// Load 16 consecutive 32-bit TMEM columns of this thread's lane and wait.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : CP_R8(r, 0), CP_R8(r, 8)
        : "r"(taddr)
        : "memory");
}
// Two 32-column loads in flight before one wait (64 columns).
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, uint32_t (&r)[64]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%64];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,"
        "%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%65];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : CP_R8(r, 0), CP_R8(r, 8), CP_R8(r, 16), CP_R8(r, 24), CP_R8(r, 32), CP_R8(r, 40), CP_R8(r, 48),
          CP_R8(r, 56)
        : "r"(taddr), "r"(taddr + 32u)
        : "memory");
}
// Four 32-column loads in flight before one wait (128 columns, two arrays).
__device__ __forceinline__ void tmem_ld128(uint32_t taddr, uint32_t (&a)[64], uint32_t (&b)[64]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%128];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,"
        "%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%129];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%64,%65,%66,%67,%68,%69,%70,%71,%72,%73,%74,%75,%76,%77,%78,%79,"
        "%80,%81,%82,%83,%84,%85,%86,%87,%88,%89,%90,%91,%92,%93,%94,%95}, [%130];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%96,%97,%98,%99,%100,%101,%102,%103,%104,%105,%106,%107,%108,%109,%110,%111,"
        "%112,%113,%114,%115,%116,%117,%118,%119,%120,%121,%122,%123,%124,%125,%126,%127}, [%131];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : CP_R8(a, 0), CP_R8(a, 8), CP_R8(a, 16), CP_R8(a, 24), CP_R8(a, 32), CP_R8(a, 40), CP_R8(a, 48),
          CP_R8(a, 56), CP_R8(b, 0), CP_R8(b, 8), CP_R8(b, 16), CP_R8(b, 24), CP_R8(b, 32), CP_R8(b, 40),
          CP_R8(b, 48), CP_R8(b, 56)
        : "r"(taddr), "r"(taddr + 32u), "r"(taddr + 64u), "r"(taddr + 96u)
        : "memory");
}
// Store 64 consecutive columns (two arrays of 32) and wait once.
__device__ __forceinline__ void tmem_st64(uint32_t taddr, const uint32_t (&a)[32], const uint32_t (&b)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,"
        "%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33};\n\t"
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%1], "
        "{%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,"
        "%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63,%64,%65};\n\t"
        "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
        "r"(taddr + 32u), CP_W8(a, 0), CP_W8(a, 8), CP_W8(a, 16), CP_W8(a, 24), CP_W8(b, 0), CP_W8(b, 8),
        CP_W8(b, 16), CP_W8(b, 24)
        : "memory");
}
// Issue a 64-column load (two x32 shapes) WITHOUT waiting; the registers must
// not be read before tmem_wait_ld(r) on the same array.
__device__ __forceinline__ void tmem_ld64_nowait(uint32_t taddr, uint32_t (&r)[64]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%64];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,"
        "%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%65];"
        : CP_R8(r, 0), CP_R8(r, 8), CP_R8(r, 16), CP_R8(r, 24), CP_R8(r, 32), CP_R8(r, 40), CP_R8(r, 48),
          CP_R8(r, 56)
        : "r"(taddr), "r"(taddr + 32u)
        : "memory");
}
#define CP_RW8(a, i) "+r"(a[i]), "+r"(a[i + 1]), "+r"(a[i + 2]), "+r"(a[i + 3]), "+r"(a[i + 4]), "+r"(a[i + 5]), \
                     "+r"(a[i + 6]), "+r"(a[i + 7])
// Wait for every outstanding tcgen05.ld of this thread; the registers of `r`
// are declared as produced here, so the compiler cannot read them earlier.
__device__ __forceinline__ void tmem_wait_ld(uint32_t (&r)[64]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : CP_RW8(r, 0), CP_RW8(r, 8), CP_RW8(r, 16), CP_RW8(r, 24), CP_RW8(r, 32), CP_RW8(r, 40),
                   CP_RW8(r, 48), CP_RW8(r, 56)
                 :
                 : "memory");
}
// Issue a 32-column load WITHOUT waiting; read `r` only after tmem_wait_ld32(r).
__device__ __forceinline__ void tmem_ld32_nowait(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : CP_R8(r, 0), CP_R8(r, 8), CP_R8(r, 16), CP_R8(r, 24)
        : "r"(taddr)
        : "memory");
}
// Wait for every outstanding tcgen05.ld of this thread, declaring `r` produced here.
__device__ __forceinline__ void tmem_wait_ld32(uint32_t (&r)[32]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : CP_RW8(r, 0), CP_RW8(r, 8), CP_RW8(r, 16), CP_RW8(r, 24)
                 :
                 : "memory");
}
// Issue a 16-column store without waiting (tmem_wait_st completes it).
__device__ __forceinline__ void tmem_st16_nowait(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
        CP_W8(r, 0), CP_W8(r, 8)
        : "memory");
}
// Issue a 32-column store without waiting (tmem_wait_st completes it).
__device__ __forceinline__ void tmem_st32_nowait(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        CP_W8(r, 0), CP_W8(r, 8), CP_W8(r, 16), CP_W8(r, 24)
        : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
// Store 32 consecutive 32-bit TMEM columns of this thread's lane and wait.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n\t"
        "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
        CP_W8(r, 0), CP_W8(r, 8), CP_W8(r, 16), CP_W8(r, 24)
        : "memory");
}

// ---------------------------------------------------------------- packed fp32 math
// Two fp32 values in one 64-bit register (low word = first).
__device__ __forceinline__ uint64_t f2_pack(uint32_t lo_bits, uint32_t hi_bits) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(lo_bits), "r"(hi_bits));
    return r;
}
__device__ __forceinline__ uint64_t f2_packf(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float &lo, float &hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// 32-byte global store (8 fp32); the address must be 32-byte aligned.
__device__ __forceinline__ void st_global_v8(float *p, float a, float b, float c, float d, float e, float f, float g,
                                             float h) {
    asm volatile("st.global.v8.f32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "f"(a), "f"(b), "f"(c),
                 "f"(d), "f"(e), "f"(f), "f"(g), "f"(h)
                 : "memory");
}

// 32-byte global load (8 fp32); the address must be 32-byte aligned.
__device__ __forceinline__ void ld_global_v8(const float *p, float (&r)[8]) {
    asm volatile("ld.global.v8.f32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=f"(r[0]), "=f"(r[1]), "=f"(r[2]), "=f"(r[3]), "=f"(r[4]), "=f"(r[5]), "=f"(r[6]), "=f"(r[7])
                 : "l"(p)
                 : "memory");
}
__device__ __forceinline__ void prefetch_l2(const void *p) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p) : "memory");
}

// ---------------------------------------------------------------- misc
__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    // low 16 bits <- lo, high 16 bits <- hi (round to nearest even)
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

}  // namespace cpattn
