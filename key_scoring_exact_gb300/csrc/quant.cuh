// quant.cuh -- on-device FP8 (E4M3) quantisation of a bf16 index query, one
// scale per (row, head), the scale folded into the head weight.  Shared by
// the scoring kernel (which quantises each group's query into its MMA
// operand) and the stand-alone quantisation kernel.
//
// The recipe is the per-token FP8 quantisation of "[Perf] [MI355X]
// minimax_m31" (section "Modifications", o_proj bullet) -- amax / 448, a
// reciprocal, clamp, round to nearest even -- applied per head: amax = max |q|
// over the head's 128 elements, scale = amax / 448, inv = 1 / scale (both
// correctly rounded f32 divisions, once per head), code = E4M3(q * inv) (f32
// product, converted to nearest even and saturated at +-448); w' = w * scale.
// An all-zero head gets scale 0: codes 0, w' = 0.
#pragma once

#include <cuda_fp8.h>

#include <cstdint>

namespace idx {

// One (row, head) held by a warp, four bf16 elements per lane (lane l holds
// elements 4l .. 4l + 3 as two 32-bit words).  Returns the lane's four codes
// packed little-endian and leaves the head's scale in *scale.
__device__ __forceinline__ uint32_t quantize_head_lane(uint2 raw, float* scale) {
    float x[4];
    x[0] = __uint_as_float(raw.x << 16);
    x[1] = __uint_as_float(raw.x & 0xFFFF0000u);
    x[2] = __uint_as_float(raw.y << 16);
    x[3] = __uint_as_float(raw.y & 0xFFFF0000u);
    const float a = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
    // non-negative floats order like their bit patterns
    const float amax = __uint_as_float(__reduce_max_sync(0xFFFFFFFFu, __float_as_uint(a)));
    const float s = __fdiv_rn(amax, 448.0f);
    *scale = s;
    if (!(s > 0.0f)) return 0u;
    const float inv = __fdiv_rn(1.0f, s);
    uint32_t codes = 0;
#pragma unroll
    for (int i = 0; i < 4; i += 2) {
        const __nv_fp8x2_storage_t c = __nv_cvt_float2_to_fp8x2(
            make_float2(__fmul_rn(x[i], inv), __fmul_rn(x[i + 1], inv)), __NV_SATFINITE, __NV_E4M3);
        codes |= (uint32_t)c << (8 * i);
    }
    return codes;
}

}  // namespace idx
