// ptx.cuh -- thin inline-PTX wrappers for sm_103a: mbarriers, TMA / bulk
// copies, tcgen05 (TMEM allocation, MMA, commit, loads), global timer.
//
// Every wait in this library is bounded: bounded_wait() gives up after a
// wall-time limit (kWaitTimeoutNs unless a test asks for a shorter one) or
// when the CTA's abort flag is raised, so a broken hand-off ends the kernel
// with an error status instead of a hang.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#define IDX_DEVI __device__ __forceinline__

namespace idx {

constexpr uint64_t kWaitTimeoutNs = 2000000000ull;  // 2 s: far beyond any legal wait

IDX_DEVI uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

IDX_DEVI uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

IDX_DEVI void record_status(uint32_t* status, uint32_t bits) {
    if (status) atomicOr(status, bits);
}

// ------------------------------------------------- programmatic dependent launch

// Block until every grid this launch depends on has completed and its
// memory operations are visible (no-op when launched without a dependency).
IDX_DEVI void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Allow the next launch on the stream (a programmatic dependent) to begin.
IDX_DEVI void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ------------------------------------------------------------------ mbarrier

IDX_DEVI void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

// Make mbarrier initialisation visible to the async proxy (TMA, tcgen05).
IDX_DEVI void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

IDX_DEVI void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

IDX_DEVI void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

IDX_DEVI bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// As mbar_try_wait, but the thread may sleep in hardware (issuing nothing)
// until the phase completes or about `hint_ns` nanoseconds pass, so waiting
// warps leave their scheduler's issue slots to the warps doing work.
IDX_DEVI bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity, uint32_t hint_ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}

// Wait for the phase of `bar` with the given parity to complete.  Returns
// false (and raises *abort) when `limit_ns` of wall time pass or *abort is
// already set.
IDX_DEVI bool bounded_wait(uint64_t* bar, uint32_t parity, volatile int* abort,
                           uint64_t limit_ns = kWaitTimeoutNs) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    const uint32_t hint = limit_ns < 200000ull ? (uint32_t)limit_ns : 200000u;
    while (true) {
        if (mbar_try_wait_sleep(bar, parity, hint)) return true;
        if (*abort) return false;
        if (globaltimer_ns() - t0 > limit_ns) {
            *abort = 1;
            return false;
        }
    }
}

// ------------------------------------------------------------- TMA / bulk

// 2D tiled TMA load of one box into shared memory, completing on `bar`.
IDX_DEVI void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y)
        : "memory");
}

// Untiled bulk copy global -> shared (16-byte aligned, size a multiple of 16).
IDX_DEVI void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// Order this thread's generic-proxy shared-memory writes before later
// async-proxy reads of them (tensor-core operands, bulk copies).
IDX_DEVI void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// Bring the line holding `ptr` into L2 (no register result, nothing waits on it).
IDX_DEVI void prefetch_l2(const void* ptr) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<uint64_t>(ptr)) : "memory");
}

IDX_DEVI void prefetch_tensormap(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ----------------------------------------------------------------- tcgen05

IDX_DEVI void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {  // whole warp
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}

IDX_DEVI void tmem_relinquish() {  // whole warp
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

IDX_DEVI void tmem_dealloc(uint32_t taddr, uint32_t ncols) {  // whole warp
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

IDX_DEVI void tc_fence_before_sync() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

IDX_DEVI void tc_fence_after_sync() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem desc] * B[smem desc]^T, FP8 operands, f32 accumulator.
IDX_DEVI void mma_f8f6f4(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                         uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive once on `bar` when every tcgen05 op issued so far by this thread is done.
IDX_DEVI void mma_commit(uint64_t* bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}

// 32 consecutive f32 columns of this thread's TMEM lane (32x32b shape, x32),
// waited for inside the same statement so the registers are valid on return.
// 16 consecutive f32 columns of this thread's TMEM lane (32x32b shape, x16),
// waited for inside the same statement.
IDX_DEVI void tmem_load_16cols(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];\n\t"
        "tcgen05.wait::ld.sync.aligned;\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

IDX_DEVI void tmem_load_32cols(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n\t"
        "tcgen05.wait::ld.sync.aligned;\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// Shared-memory matrix descriptor for a K-major operand in the 128-byte
// swizzle layout that a TMA load with CU_TENSOR_MAP_SWIZZLE_128B writes:
// rows of 128 bytes, 8-row (1024-byte) swizzle atoms stacked along M/N.
// The buffer must be 1024-byte aligned; a K offset inside the 128-byte row
// is applied by advancing the start address.
IDX_DEVI uint64_t desc_kmajor_sw128(uint32_t saddr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);  // start address / 16
    d |= static_cast<uint64_t>(1) << 16;                   // leading byte offset (unused)
    d |= static_cast<uint64_t>(1024 >> 4) << 32;           // stride byte offset: 8 rows
    d |= static_cast<uint64_t>(1) << 46;                   // descriptor version (tcgen05)
    d |= static_cast<uint64_t>(2) << 61;                   // 128-byte swizzle
    return d;
}

// Instruction descriptor: E4M3 x E4M3 -> F32, both K-major, dense, M x N.
IDX_DEVI uint32_t idesc_e4m3_f32(uint32_t M, uint32_t N) {
    return (1u << 4)            // D format F32
           | (0u << 7)          // A format E4M3
           | (0u << 10)         // B format E4M3
           | ((N >> 3) << 17)   // N / 8
           | ((M >> 4) << 24);  // M / 16
}

}  // namespace idx
