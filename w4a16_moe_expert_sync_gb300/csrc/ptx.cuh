// ptx.cuh -- inline-PTX wrappers for sm_103a: mbarrier, TMA bulk copies,
// tcgen05 (TMEM allocation, MMA with the A operand in tensor memory,
// TMEM loads/stores) and the shared-memory matrix descriptor.
#pragma once

#include <cstdint>

#include <cuda.h>
#include <cuda_runtime.h>

namespace w4 {

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ------------------------------------------------- gpu-scope synchronisation
// Acquire-release fence at gpu scope: releases this thread's earlier writes
// (and those ordered before it by CTA-scope synchronisation) to a thread
// that reads a later write of this thread and then acquires, and acquires
// what such a write published.
__device__ __forceinline__ void fence_acq_rel_gpu()
{
    asm volatile("fence.acq_rel.gpu;" ::: "memory");
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

// The barrier helpers come in two forms: by pointer, and by 32-bit shared
// address (suffix _a) for loops that keep their barriers' addresses in
// registers.
__device__ __forceinline__ bool mbar_try_wait_a(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity)
{
    return mbar_try_wait_a(smem_u32(bar), parity);
}

// try_wait with a suspend-time hint: the thread is suspended until the phase
// completes or about `hint_ns` elapse, so a waiting warp does not spin on the
// issue slots the working warps of its sub-partition need.
__device__ __forceinline__ bool mbar_try_wait_sleep_a(uint32_t bar, uint32_t parity,
                                                      uint32_t hint_ns)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t *bar, uint32_t parity,
                                                    uint32_t hint_ns)
{
    return mbar_try_wait_sleep_a(smem_u32(bar), parity, hint_ns);
}

// A pipeline wait with a time limit.  Returns false (and raises the CTA's
// abort flag and the device status bit) when the phase did not complete
// within `limit_ns`, or when another role of the CTA has already aborted.
// Each try suspends the thread for up to 20 us; between tries the abort
// flag and the clock are checked.
// Suspend-time hint of a retried try_wait, in ns.
#ifndef W4_WAIT_HINT_NS
#define W4_WAIT_HINT_NS 20000u
#endif

__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                          int32_t *dev_status, int32_t timeout_bit,
                                          uint64_t limit_ns = 1000000000ull)
{
    if (mbar_try_wait(bar, parity))
        return true;
    // Every retry is one suspending try_wait and a branch; the abort flag and
    // the clock are looked at on every 16th retry only, so waiting warps take
    // few issue slots from the working ones.
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
#ifdef W4_WAIT_NOHINT
        if (mbar_try_wait(bar, parity))
            return true;
#else
        if (mbar_try_wait_sleep(bar, parity, W4_WAIT_HINT_NS))
            return true;
#endif
#ifdef W4_WAIT_BACKOFF_NS
        __nanosleep(W4_WAIT_BACKOFF_NS);
#endif
        if ((it & 15u) == 0) {
            if (*abort_flag)
                return false;
            if (global_timer_ns() - t0 > limit_ns) {
                *abort_flag = 1;
                if (dev_status)
                    atomicOr(dev_status, timeout_bit);
                return false;
            }
        }
    }
}

// A pipeline wait by a whole warp with warp-uniform control flow: every lane
// probes the phase (so every lane observes its completion) and one vote
// decides each branch, so the loop needs no divergence handling.  Same time
// limit and abort handling as mbar_wait.
__device__ __forceinline__ bool mbar_wait_warp_a(uint32_t bar, uint32_t parity,
                                                 volatile int *abort_flag, int32_t *dev_status,
                                                 int32_t timeout_bit,
                                                 uint64_t limit_ns = 1000000000ull)
{
    const unsigned full = 0xffffffffu;
    if (__all_sync(full, mbar_try_wait_a(bar, parity)))
        return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        if (__all_sync(full, mbar_try_wait_sleep_a(bar, parity, W4_WAIT_HINT_NS)))
            return true;
        if ((it & 15u) == 0) {
            if (__any_sync(full, *abort_flag != 0))
                return false;
            if (__any_sync(full, global_timer_ns() - t0 > limit_ns)) {
                if ((threadIdx.x & 31) == 0) {
                    *abort_flag = 1;
                    if (dev_status)
                        atomicOr(dev_status, timeout_bit);
                }
                return false;
            }
        }
    }
}

__device__ __forceinline__ bool mbar_wait_warp(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                               int32_t *dev_status, int32_t timeout_bit,
                                               uint64_t limit_ns = 1000000000ull)
{
    return mbar_wait_warp_a(smem_u32(bar), parity, abort_flag, dev_status, timeout_bit, limit_ns);
}

// One arrival per warp, made by an elected lane without a branch (call with
// the warp converged, after whatever the arrival must publish).
__device__ __forceinline__ void mbar_arrive_elect_a(uint32_t bar)
{
    asm volatile(
        "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
        "@e mbarrier.arrive.shared::cta.b64 _, [%0];\n\t}" ::"r"(bar)
        : "memory");
}

__device__ __forceinline__ void mbar_arrive_elect(uint64_t *bar)
{
    mbar_arrive_elect_a(smem_u32(bar));
}

// A pipeline wait for roles whose wake-up latency matters little (producers
// running ahead, an epilogue waiting for a whole unit): between tries the
// thread sleeps `backoff_ns`, so a waiting warp takes almost no issue slots
// from the working warps of its sub-partition.  Same time limit and abort
// handling as mbar_wait.
__device__ __forceinline__ bool mbar_wait_lazy(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                               int32_t *dev_status, int32_t timeout_bit,
                                               uint32_t backoff_ns,
                                               uint64_t limit_ns = 1000000000ull)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        __nanosleep(backoff_ns);
        if (mbar_try_wait(bar, parity))
            return true;
        if ((it & 15u) == 0) {
            if (*abort_flag)
                return false;
            if (global_timer_ns() - t0 > limit_ns) {
                *abort_flag = 1;
                if (dev_status)
                    atomicOr(dev_status, timeout_bit);
                return false;
            }
        }
    }
}

// ------------------------------------------------------------ TMA / bulk
__device__ __forceinline__ uint64_t l2_policy_evict_first()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap *map)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 2-D tiled TMA load (coordinates: x = innermost, in elements) completing on
// an mbarrier, with an L2 cache policy.
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int x, int y,
                                            uint64_t *bar, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// Prefetch of one 2-D tile (the tensor map's box at x, y) from global memory
// into L2; no shared memory, no completion.  Coordinates as tma_load_2d.
__device__ __forceinline__ void tma_prefetch_2d(const CUtensorMap *map, int x, int y)
{
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y)
                 : "memory");
}

// Prefetch of `bytes` (a multiple of 16) at the 16-byte aligned src into L2.
__device__ __forceinline__ void bulk_prefetch_l2(const void *src, uint32_t bytes)
{
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// 2-D tiled TMA load without a cache hint.
__device__ __forceinline__ void tma_load_2d_nohint(void *dst, const CUtensorMap *map, int x, int y,
                                                   uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

// Four rows r0..r3 (any order, any rows of the tensor) of one box column
// starting at x, gathered by a 2-D tensor map whose box is one row high, into
// four consecutive box rows at dst.
__device__ __forceinline__ void tma_gather4(void *dst, const CUtensorMap *map, int x, int r0,
                                            int r1, int r2, int r3, uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cta.global.tile::gather4.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(r0), "r"(r1), "r"(r2), "r"(r3),
        "r"(smem_u32(bar))
        : "memory");
}

// Contiguous bulk copy global -> shared (both 16-byte aligned, size % 16 == 0).
// 1-D bulk copy global -> shared without a cache hint; dst, src 16-byte
// aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_load_nohint(void *dst, const void *src, uint32_t bytes,
                                                 uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// 3-D tile copy global -> shared (coordinates innermost first).
__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *map, int x, int y, int z,
                                            uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void bulk_load(void *dst, const void *src, uint32_t bytes,
                                          uint64_t *bar, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// Make generic-proxy shared-memory writes visible to the async proxy
// (tensor-core operand reads).
__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------- tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t *dst_smem, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish()
{
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before()
{
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after()
{
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Arrive (once) on `bar` when every tcgen05 operation issued so far by this
// thread has completed.
__device__ __forceinline__ void tc_commit(uint64_t *bar)
{
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]^T, kind::f16 (fp16 or bf16 in, fp32 out).
__device__ __forceinline__ void tc_mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// The same MMA and commit issued by one elected lane of a converged warp.
// With the whole warp on the same path its operands stay warp-uniform (in
// uniform registers), which makes the issue several times cheaper than from a
// lone lane in a divergent branch.
__device__ __forceinline__ void tc_mma_ts_elect(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                                uint32_t idesc, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p, e;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Up to four MMAs as in tc_mma4_ts_commit_elect, without the commit.
__device__ __forceinline__ void tc_mma4_ts_elect(uint32_t d_tmem, uint32_t a_tmem, uint64_t b0,
                                                 uint64_t b1, uint64_t b2, uint64_t b3,
                                                 uint32_t idesc, int n, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred e, q0, q1, q2, q3, acc, on;\n\t"
        ".reg .b32 a1, a2, a3;\n\t"
        "add.u32 a1, %1, 8;\n\tadd.u32 a2, %1, 16;\n\tadd.u32 a3, %1, 24;\n\t"
        "setp.ne.b32 acc, %7, 0;\n\t"
        "setp.eq.b32 on, %7, %7;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "setp.gt.and.s32 q0, %8, 0, e;\n\t"
        "setp.gt.and.s32 q1, %8, 1, e;\n\t"
        "setp.gt.and.s32 q2, %8, 2, e;\n\t"
        "setp.gt.and.s32 q3, %8, 3, e;\n\t"
        "@q0 tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %6, acc;\n\t"
        "@q1 tcgen05.mma.cta_group::1.kind::f16 [%0], [a1], %3, %6, on;\n\t"
        "@q2 tcgen05.mma.cta_group::1.kind::f16 [%0], [a2], %4, %6, on;\n\t"
        "@q3 tcgen05.mma.cta_group::1.kind::f16 [%0], [a3], %5, %6, on;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b0), "l"(b1), "l"(b2), "l"(b3), "r"(idesc), "r"(accumulate), "r"(n)
        : "memory");
}

// Up to four MMAs (A in tensor memory, B from shared memory, one D) and a
// commit of this thread's tcgen05 work to `bar`, all from one elected lane of
// a converged warp: MMA t is issued when t < n, with a_tmem + 8 t and
// b_desc + b_step[t]; the first adds to D only when `accumulate` is set, the
// others always.  One elect and one issue sequence for the group keeps the
// per-MMA cost of the issuing warp low.
__device__ __forceinline__ void tc_mma4_ts_commit_elect(uint32_t d_tmem, uint32_t a_tmem,
                                                        uint64_t b0, uint64_t b1, uint64_t b2,
                                                        uint64_t b3, uint32_t idesc, int n,
                                                        uint32_t accumulate, uint64_t *bar)
{
    asm volatile(
        "{\n\t.reg .pred e, q0, q1, q2, q3, acc, on;\n\t"
        ".reg .b32 a1, a2, a3;\n\t"
        "add.u32 a1, %1, 8;\n\tadd.u32 a2, %1, 16;\n\tadd.u32 a3, %1, 24;\n\t"
        "setp.ne.b32 acc, %7, 0;\n\t"
        "setp.eq.b32 on, %7, %7;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "setp.gt.and.s32 q0, %8, 0, e;\n\t"
        "setp.gt.and.s32 q1, %8, 1, e;\n\t"
        "setp.gt.and.s32 q2, %8, 2, e;\n\t"
        "setp.gt.and.s32 q3, %8, 3, e;\n\t"
        "@q0 tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %6, acc;\n\t"
        "@q1 tcgen05.mma.cta_group::1.kind::f16 [%0], [a1], %3, %6, on;\n\t"
        "@q2 tcgen05.mma.cta_group::1.kind::f16 [%0], [a2], %4, %6, on;\n\t"
        "@q3 tcgen05.mma.cta_group::1.kind::f16 [%0], [a3], %5, %6, on;\n\t"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%9];\n\t}" ::"r"(
            d_tmem),
        "r"(a_tmem), "l"(b0), "l"(b1), "l"(b2), "l"(b3), "r"(idesc), "r"(accumulate), "r"(n),
        "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void tc_commit_elect(uint64_t *bar)
{
    asm volatile(
        "{\n\t.reg .pred e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(
            smem_u32(bar))
        : "memory");
}

// Instruction descriptor for kind::f16: fp16 A and B (both K-major), fp32
// accumulator, M = 128, N in [16, 256] step 16.
__host__ __device__ constexpr uint32_t idesc_f16_f32(uint32_t M, uint32_t N)
{
    return (1u << 4)                // D format: fp32
           | (0u << 7)              // A format: fp16
           | (0u << 10)             // B format: fp16
           | (0u << 15)             // A K-major
           | (0u << 16)             // B K-major
           | ((N >> 3) << 17)       // N / 8
           | ((M >> 4) << 24);      // M / 16
}

// Instruction descriptor for kind::f16 with both operands bf16 (bf16 = true)
// or both fp16, fp32 accumulator, K-major A and B.
__host__ __device__ constexpr uint32_t idesc_16bit_f32(uint32_t M, uint32_t N, bool bf16)
{
    return idesc_f16_f32(M, N) | (bf16 ? ((1u << 7) | (1u << 10)) : 0u);
}

// Shared-memory matrix descriptor, K-major, 128-byte swizzle: rows of 128 B,
// 8-row atoms of 1024 B (stride between atoms = SBO = 1024 B).
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t smem_addr)
{
    uint64_t d = 0;
    d |= static_cast<uint64_t>((smem_addr & 0x3FFFFu) >> 4);   // start address
    d |= static_cast<uint64_t>(1) << 16;                       // LBO (unused here)
    d |= static_cast<uint64_t>(1024 >> 4) << 32;               // SBO
    d |= static_cast<uint64_t>(1) << 46;                       // descriptor version
    d |= static_cast<uint64_t>(2) << 61;                       // SWIZZLE_128B
    return d;
}

// 32 lanes x 8 columns of 32 bit (thread i: lane quarter base + i).
__device__ __forceinline__ void tmem_st_32x32b_x8(uint32_t taddr, const uint32_t (&r)[8])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(
            taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
        : "memory");
}

// 32 lanes x 16 columns of 32 bit (thread i: lane quarter base + i).
__device__ __forceinline__ void tmem_st_32x32b_x16(uint32_t taddr, const uint32_t (&r)[16])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15])
        : "memory");
}

// 32 lanes x 32 columns of 32 bit: thread i of the warp writes lane
// (warp quarter base + i), columns [col, col + 32).
__device__ __forceinline__ void tmem_st_32x32b_x32(uint32_t taddr, const uint32_t (&r)[32])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
        "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(
            taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
        "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
        "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

__device__ __forceinline__ void tmem_wait_st()
{
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Load 8 consecutive 32-bit columns of this thread's lane and wait for them.
__device__ __forceinline__ void tmem_ld_32x32b_x8(uint32_t taddr, uint32_t (&r)[8])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7])
        : "r"(taddr)
        : "memory");
}

// Load 16 consecutive 32-bit columns of this thread's lane and wait for them.
__device__ __forceinline__ void tmem_ld_32x32b_x16(uint32_t taddr, uint32_t (&r)[16])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15}, [%16];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}

// Four loads of 8 columns each (at four TMEM addresses of this warp's lane
// quarter) followed by one wait, so the four round trips overlap.
// Two 32x32b.x8 loads (columns t0 .. t0+7 and t1 .. t1+7 of the warp's lane
// quarter) into r[0..7] and r[8..15], then wait for both.
__device__ __forceinline__ void tmem_ld_2x_32x32b_x8(uint32_t t0, uint32_t t1, uint32_t (&r)[16])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%16];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%8, %9, %10, %11, %12, %13, %14, %15}, [%17];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(t0), "r"(t1)
        : "memory");
}

__device__ __forceinline__ void tmem_ld_4x_32x32b_x8(uint32_t t0, uint32_t t1, uint32_t t2,
                                                     uint32_t t3, uint32_t (&r)[32])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%32];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%8, %9, %10, %11, %12, %13, %14, %15}, [%33];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%16, %17, %18, %19, %20, %21, %22, %23}, [%34];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%24, %25, %26, %27, %28, %29, %30, %31}, [%35];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
          "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
          "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(t0), "r"(t1), "r"(t2), "r"(t3)
        : "memory");
}

// Load 32 consecutive 32-bit columns of this thread's lane and wait for them.
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
        "%28, %29, %30, %31}, [%32];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr)
        : "memory");
}

// Programmatic dependent launch.  pdl_wait: block until the grid this one
// depends on (the preceding kernel in the stream, when this kernel was
// launched as its dependent) has completed and its writes are visible; a
// no-op otherwise.  pdl_trigger: allow the next dependent kernel to start
// launching; it still waits for this grid's completion in its own pdl_wait.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

}  // namespace w4
