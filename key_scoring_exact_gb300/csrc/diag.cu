// diag.cu -- diagnostics of include/idx_diag.h: the tcgen05 FP8 tensor-core
// peak probe that the scoring's roofline is measured against, and the test
// hook that shortens the scoring kernel's wait limit.
#include <cstdio>

#include "../../include/idx_diag.h"
#include "idx_internal.h"
#include "ptx.cuh"

namespace idx {

namespace {

thread_local WaitTestHook g_hook = {0ull, 0};

constexpr int kProbeThreads = 128;
constexpr uint32_t kProbeA = 128 * 128;      // A: 128 rows of 128 bytes (E4M3, K = 128)
constexpr uint32_t kProbeB = 256 * 128;      // B: up to 256 rows of 128 bytes
constexpr uint32_t kProbeSmem = 120 * 1024;  // more than half an SM's shared memory: one CTA per SM

// One CTA per SM: thread 0 issues n_mma back-to-back M = 128 x N x K = 32
// kind::f8f6f4 MMAs (E4M3 x E4M3 -> f32) from shared memory into TMEM,
// alternating between two 256-column accumulators every 8 MMAs (as the
// scoring does per tile), commits, waits for completion, and writes the
// elapsed wall time (ns) and SM clocks of its CTA.
__global__ void __launch_bounds__(kProbeThreads, 1)
k_probe_fp8(int n_mma, uint32_t n_cols, unsigned long long* out_ns, unsigned long long* out_clk) {
    extern __shared__ uint8_t raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
    __shared__ uint64_t bar;
    __shared__ uint32_t tslot;
    __shared__ int abort_flag;
    // E4M3 1.0 in every operand byte: finite sums whatever the accumulation.
    for (uint32_t i = threadIdx.x; i < (kProbeA + kProbeB) / 4; i += kProbeThreads)
        reinterpret_cast<uint32_t*>(sm)[i] = 0x38383838u;
    fence_proxy_async_smem();
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    if ((threadIdx.x >> 5) == 0) {
        tmem_alloc(&tslot, 512);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tb = tslot;
    if (threadIdx.x == 0) {
        const uint32_t idesc = idesc_e4m3_f32(128, n_cols);
        const uint32_t a = smem_u32(sm), b = smem_u32(sm + kProbeA);
        const uint64_t t0 = globaltimer_ns();
        const long long c0 = clock64();
        for (int i = 0; i < n_mma; ++i) {
            const uint32_t kk = (uint32_t)(i & 3) * 32;
            const uint32_t d = tb + (uint32_t)((i >> 3) & 1) * 256;
            mma_f8f6f4(d, desc_kmajor_sw128(a + kk), desc_kmajor_sw128(b + kk), idesc, (i & 3) ? 1u : 0u);
        }
        mma_commit(&bar);
        const bool done = bounded_wait(&bar, 0, reinterpret_cast<volatile int*>(&abort_flag));
        const long long c1 = clock64();
        const uint64_t t1 = globaltimer_ns();
        out_ns[blockIdx.x] = done ? (unsigned long long)(t1 - t0) : 0ull;
        out_clk[blockIdx.x] = done ? (unsigned long long)(c1 - c0) : 0ull;
    }
    tc_fence_before_sync();
    __syncthreads();
    if ((threadIdx.x >> 5) == 0) {
        tc_fence_after_sync();
        tmem_dealloc(tb, 512);
    }
}

}  // namespace

WaitTestHook wait_test_hook() { return g_hook; }

}  // namespace idx

using namespace idx;

extern "C" {

idx_status idx_probe_fp8_mma(int n_mma, int n_cols, unsigned long long* out_ns, unsigned long long* out_clk,
                             int n_out, void* stream) {
    if (n_mma < 8 || n_mma > (1 << 22) || !out_ns || !out_clk) return IDX_ERR_ARG;
    if (n_cols < 16 || n_cols > 256 || n_cols % 16 != 0) return IDX_ERR_ARG;
    int dev = 0, sms = 0, major = 0, minor = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
        (void)cudaGetLastError();
        return IDX_ERR_CUDA;
    }
    if (major != 10 || minor != 3) return IDX_ERR_UNSUPPORTED;
    if (n_out < sms) return IDX_ERR_ARG;
    if (cudaFuncSetAttribute(k_probe_fp8, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kProbeSmem) !=
        cudaSuccess) {
        (void)cudaGetLastError();
        return IDX_ERR_CUDA;
    }
    k_probe_fp8<<<sms, kProbeThreads, kProbeSmem, static_cast<cudaStream_t>(stream)>>>(n_mma, (uint32_t)n_cols,
                                                                                       out_ns, out_clk);
    if (cudaGetLastError() != cudaSuccess) return IDX_ERR_CUDA;
    return IDX_OK;
}

idx_status idx_test_set_wait_limit(unsigned long long wait_ns, int drop_query_handoff) {
    g_hook.wait_ns = wait_ns;
    g_hook.drop_query_handoff = drop_query_handoff ? 1 : 0;
    return IDX_OK;
}

}  // extern "C"
