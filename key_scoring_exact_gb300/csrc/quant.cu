// quant.cu -- the stand-alone FP8 query quantisation (idx_quantize_query):
// one warp per (row, head), the same device code the scoring kernel uses.
#include "idx_internal.h"
#include "quant.cuh"

namespace idx {

namespace {

constexpr int kQuantWarps = 8;

__global__ void __launch_bounds__(kQuantWarps * 32)
k_quantize(const uint16_t* __restrict__ q, const float* __restrict__ head_w, int pairs,
           uint8_t* __restrict__ q8, float* __restrict__ w_out) {
    const int lane = threadIdx.x & 31;
    const int pp = blockIdx.x * kQuantWarps + (threadIdx.x >> 5);
    if (pp >= pairs) return;  // warp-uniform
    const uint2 raw = reinterpret_cast<const uint2*>(q)[(int64_t)pp * 32 + lane];
    float scale;
    const uint32_t codes = quantize_head_lane(raw, &scale);
    reinterpret_cast<uint32_t*>(q8)[(int64_t)pp * 32 + lane] = codes;
    if (lane == 0) w_out[pp] = __fmul_rn(head_w[pp], scale);
}

}  // namespace

cudaError_t launch_quantize(const void* q, const float* head_w, int R, uint8_t* q8, float* w_out,
                            cudaStream_t stream) {
    const int pairs = R * kHeads;
    k_quantize<<<(pairs + kQuantWarps - 1) / kQuantWarps, kQuantWarps * 32, 0, stream>>>(
        static_cast<const uint16_t*>(q), head_w, pairs, q8, w_out);
    return cudaGetLastError();
}

}  // namespace idx
