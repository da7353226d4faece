// stage.cu -- gathers a fused call's per-step inputs from page-locked host
// memory into the workspace with one kernel.  On a Grace-Blackwell node the
// host memory is reached over the coherent chip-to-chip link, so one launch
// whose threads read the buffers directly replaces one copy-engine transfer
// (several microseconds of fixed cost each) per buffer.
#include "idx_internal.h"
#include "ptx.cuh"

namespace idx {

namespace {

constexpr int kStageThreads = 256;

// A programmatic dependent of the kernel before it on the stream (the
// previous call's selection, which allows it at its start): each thread reads
// its first 16 bytes from host memory at once, over the link's latency, then
// waits for that kernel to finish before it writes the workspace that kernel
// may still read.
__global__ void __launch_bounds__(kStageThreads) k_stage(StagePlan plan) {
    pdl_launch_dependents();  // the scoring kernel may launch now; it waits for this grid's end
    const StageCopy cp = plan.c[blockIdx.y];
    const uint32_t n16 = cp.bytes / 16, n4 = cp.bytes / 4;
    const uint32_t stride = gridDim.x * kStageThreads;
    const uint32_t t0 = blockIdx.x * kStageThreads + threadIdx.x;
    const uint4* s16 = static_cast<const uint4*>(cp.src);
    uint4* d16 = static_cast<uint4*>(cp.dst);
    uint4 first = make_uint4(0u, 0u, 0u, 0u);
    if (t0 < n16) first = s16[t0];
    pdl_wait();
    if (t0 < n16) d16[t0] = first;
    for (uint32_t i = t0 + stride; i < n16; i += stride) d16[i] = s16[i];
    const uint32_t* s4 = static_cast<const uint32_t*>(cp.src);
    uint32_t* d4 = static_cast<uint32_t*>(cp.dst);
    for (uint32_t i = 4 * n16 + t0; i < n4; i += stride) d4[i] = s4[i];
}

}  // namespace

cudaError_t launch_stage(const StagePlan& plan, cudaStream_t stream) {
    if (plan.n < 1 || plan.n > kStageMaxCopies) return cudaErrorInvalidValue;
    uint32_t most = 0;
    for (int i = 0; i < plan.n; ++i) most = plan.c[i].bytes > most ? plan.c[i].bytes : most;
    uint32_t blocks = (most / 16 + kStageThreads - 1) / kStageThreads;
    blocks = blocks < 1 ? 1 : (blocks > 64 ? 64 : blocks);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(blocks, (unsigned)plan.n, 1);
    cfg.blockDim = dim3(kStageThreads, 1, 1);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k_stage, plan);
}

}  // namespace idx
