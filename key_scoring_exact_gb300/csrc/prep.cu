// prep.cu -- per-launch preparation for the scoring kernel.
//
//  1. The query.  The scoring MMAs run on FP8 (E4M3) operands.  A bf16 query
//     element has 8 significant bits and E4M3 only 4, so each (row, head)
//     vector is scaled by a power of two 2^e that brings its largest element
//     into (224, 448] and then split exactly into two E4M3 terms:
//         x * 2^e = hi + lo,  hi = RN_e4m3(x * 2^e),  lo = x * 2^e - hi.
//     For every element whose scaled magnitude is at least 2^-2, lo is a
//     multiple of the element's bf16 ulp no larger than 8 ulps, so it is an
//     E4M3 value and the split is exact; smaller elements lose at most 2^-10
//     (scaled) to E4M3's subnormal grid -- below 4e-6 of the head's largest
//     element.  K.hi + K.lo then equals K.(x * 2^e) up to that, and 2^-e > 0
//     commutes with the ReLU, so it is folded into the head weight:
//         w'[r,h] = w[r,h] * 2^-e[r,h].
//     An E4M3 query is used as is (hi = q, no lo term, w' = w).
//  2. The plan.  Consecutive rows of one request form groups of at most four
//     rows that score the request's keys in one pass, as in "sgl-amd-mono-
//     upstream PR 18" (GLM-5.3 indexer launch), section "Modifications / 2. A
//     request's rows scored together"; each group's keys are cut into 128-key
//     tiles (two 64-token pages) numbered in one sequence of work items.
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "idx_internal.h"
#include "ptx.cuh"

namespace idx {

namespace {

constexpr int kPrepThreads = 256;
constexpr int kPairsPerBlock = kPrepThreads / 32;  // one warp per (row, head)

__device__ __forceinline__ float e4m3_pair_to_float(uint16_t codes, int which) {
    __half2_raw h2 = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(codes), __NV_E4M3);
    __half_raw h;
    h.x = which ? h2.y : h2.x;
    return __half2float(__half(h));
}

__device__ __forceinline__ uint16_t to_e4m3_pair(float a, float b) {
    return static_cast<uint16_t>(__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3));
}

__device__ __forceinline__ float pow2f(int e) {  // e in [-126, 127]: exact 2^e
    return __int_as_float((e + 127) << 23);
}

__device__ void split_query(int qtype, const void* q, const float* head_w, int R, uint8_t* q8,
                            float* wq) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int pair = blockIdx.x * kPairsPerBlock + warp;  // r * 64 + h
    if (pair >= R * kHeads) return;
    uint32_t* hi_out = reinterpret_cast<uint32_t*>(q8) + (size_t)pair * (kDim / 4);
    uint32_t* lo_out = reinterpret_cast<uint32_t*>(q8 + (size_t)R * kHeads * kDim) + (size_t)pair * (kDim / 4);
    const float w = head_w[pair];
    if (qtype == IDX_Q_E4M3) {
        hi_out[lane] = reinterpret_cast<const uint32_t*>(q)[(size_t)pair * 32 + lane];
        lo_out[lane] = 0u;
        if (lane == 0) wq[pair] = w;
        return;
    }
    const uint2 raw = reinterpret_cast<const uint2*>(q)[(size_t)pair * 32 + lane];
    float x[4];
    x[0] = __uint_as_float(raw.x << 16);
    x[1] = __uint_as_float(raw.x & 0xFFFF0000u);
    x[2] = __uint_as_float(raw.y << 16);
    x[3] = __uint_as_float(raw.y & 0xFFFF0000u);
    float amax = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
    int e = 0;
    if (amax > 0.0f && amax <= 3.0e38f) {
        int E;
        const float m = frexpf(amax, &E);  // amax = m * 2^E, m in [0.5, 1)
        e = (m <= 0.875f) ? 9 - E : 8 - E;  // amax * 2^e in (224, 448]
        e = max(-126, min(126, e));
    }
    const float sc = pow2f(e);
    float xs[4], hi[4], lo[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) xs[i] = x[i] * sc;
    const uint16_t h01 = to_e4m3_pair(xs[0], xs[1]);
    const uint16_t h23 = to_e4m3_pair(xs[2], xs[3]);
    hi[0] = e4m3_pair_to_float(h01, 0);
    hi[1] = e4m3_pair_to_float(h01, 1);
    hi[2] = e4m3_pair_to_float(h23, 0);
    hi[3] = e4m3_pair_to_float(h23, 1);
#pragma unroll
    for (int i = 0; i < 4; ++i) lo[i] = __fsub_rn(xs[i], hi[i]);
    const uint16_t l01 = to_e4m3_pair(lo[0], lo[1]);
    const uint16_t l23 = to_e4m3_pair(lo[2], lo[3]);
    hi_out[lane] = (uint32_t)h01 | ((uint32_t)h23 << 16);
    lo_out[lane] = (uint32_t)l01 | ((uint32_t)l23 << 16);
    if (lane == 0) wq[pair] = w * pow2f(-e);
}

// One warp builds the plan.  Rows r and r-1 share a group run when they have
// the same request; a run is cut into groups of kGroupRows rows.
__device__ void build_plan(const int32_t* seq_lens, const int32_t* row_req, int R, int max_pages,
                           int64_t len_bound, Plan* plan, uint32_t* status) {
    __shared__ int s_gid[kMaxRows];
    if (threadIdx.x >= 32) return;
    const int lane = threadIdx.x;
    const unsigned full = 0xFFFFFFFFu;
    // A row may not be longer than its block table or the score buffer.
    const int64_t cap = (int64_t)max_pages * kPage < len_bound ? (int64_t)max_pages * kPage : len_bound;
    int carry_seg = 0, carry_req = -1, n_groups = 0;
    bool bad = false;
    for (int base = 0; base < R; base += 32) {
        const int r = base + lane;
        const bool valid = r < R;
        const int req = valid ? row_req[r] : -1;
        int len = valid ? seq_lens[r] : 0;
        if (valid) {
            if (len < 0 || (int64_t)len > cap || req < 0) bad = true;
            len = len < 0 ? 0 : ((int64_t)len > cap ? (int)cap : len);
            if (req < 0) len = 0;
            plan->row_len[r] = len;
        }
        int prev_req = __shfl_up_sync(full, req, 1);
        if (lane == 0) prev_req = carry_req;
        const bool seg_start = valid && (r == 0 || req != prev_req);
        const unsigned upto = full >> (31 - lane);  // lanes 0..lane
        const unsigned starts = __ballot_sync(full, seg_start) & upto;
        const int seg = starts ? base + (31 - __clz(starts)) : carry_seg;
        const bool gstart = valid && ((r - seg) % kGroupRows == 0);
        const unsigned gs = __ballot_sync(full, gstart);
        const int gid = n_groups + __popc(gs & upto) - 1;
        if (valid) s_gid[r] = gid;
        if (gstart) {
            plan->g_req[gid] = req;
            plan->g_r0[gid] = r;
        }
        n_groups += __popc(gs);
        carry_seg = __shfl_sync(full, seg, 31);
        carry_req = __shfl_sync(full, req, 31);
    }
    __syncwarp();
    if (__any_sync(full, bad) && lane == 0) record_status(status, kStatusBounds);
    int item = 0;
    for (int base = 0; base < n_groups; base += 32) {
        const int g = base + lane;
        int ntiles = 0;
        if (g < n_groups) {
            const int r0 = plan->g_r0[g];
            int nr = 0, glen = 0;
            for (int i = 0; i < kGroupRows && r0 + i < R; ++i) {
                if (s_gid[r0 + i] != g) break;
                ++nr;
                glen = max(glen, plan->row_len[r0 + i]);
            }
            plan->g_nr[g] = nr;
            plan->g_len[g] = glen;
            ntiles = (glen + kTileKeys - 1) / kTileKeys;
        }
        int incl = ntiles;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(full, incl, o);
            if (lane >= o) incl += v;
        }
        if (g < n_groups) plan->g_item[g] = item + incl - ntiles;
        item += __shfl_sync(full, incl, 31);
    }
    if (lane == 0) {
        plan->g_item[n_groups] = item;
        plan->n_groups = n_groups;
        plan->n_items = item;
    }
}

__global__ void __launch_bounds__(kPrepThreads) k_prep(int qtype, const void* q, const float* head_w,
                                                       const int32_t* seq_lens, const int32_t* row_req,
                                                       int R, int max_pages, int64_t len_bound, uint8_t* q8,
                                                       float* wq, Plan* plan, uint32_t* status, int n_qblocks) {
    pdl_launch_dependents();  // the scoring kernel may start its set-up now
    if ((int)blockIdx.x == n_qblocks) {
        build_plan(seq_lens, row_req, R, max_pages, len_bound, plan, status);
        return;
    }
    split_query(qtype, q, head_w, R, q8, wq);
}

}  // namespace

cudaError_t launch_prep(const ScoreArgs& a) {
    static int configured_device = -1;
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (configured_device != dev) {
        // Same shared-memory carve-out as the scoring kernel that follows, so
        // an SM need not drain and reconfigure between the two launches.
        err = cudaFuncSetAttribute(k_prep, cudaFuncAttributePreferredSharedMemoryCarveout,
                                   cudaSharedmemCarveoutMaxShared);
        if (err != cudaSuccess) return err;
        configured_device = dev;
    }
    const int n_qblocks = (a.R * kHeads + kPairsPerBlock - 1) / kPairsPerBlock;
    k_prep<<<n_qblocks + 1, kPrepThreads, 0, a.stream>>>(
        a.qtype, a.q, a.head_w, a.seq_lens, a.row_req, a.R, a.max_pages, a.len_bound,
        reinterpret_cast<uint8_t*>(a.ws + a.L.q8), reinterpret_cast<float*>(a.ws + a.L.wq),
        reinterpret_cast<Plan*>(a.ws + a.L.plan), reinterpret_cast<uint32_t*>(a.ws + a.L.status),
        n_qblocks);
    return cudaGetLastError();
}

}  // namespace idx
