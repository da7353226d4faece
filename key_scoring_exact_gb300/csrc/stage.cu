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

__global__ void __launch_bounds__(kStageThreads) k_stage(StagePlan plan) {
    pdl_launch_dependents();  // the scoring kernel may launch now; it waits for this grid's end
    const StageCopy cp = plan.c[blockIdx.y];
    const uint32_t n16 = cp.bytes / 16, n4 = cp.bytes / 4;
    const uint32_t stride = gridDim.x * kStageThreads;
    const uint32_t t0 = blockIdx.x * kStageThreads + threadIdx.x;
    const uint4* s16 = static_cast<const uint4*>(cp.src);
    uint4* d16 = static_cast<uint4*>(cp.dst);
    for (uint32_t i = t0; i < n16; i += stride) d16[i] = s16[i];
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
    k_stage<<<dim3(blocks, (unsigned)plan.n), kStageThreads, 0, stream>>>(plan);
    return cudaGetLastError();
}

}  // namespace idx
