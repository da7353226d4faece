// select.cu -- exact top-k of each row by a multi-slice radix select.
//
// "sgl-amd-mono-upstream PR 18" (GLM-5.3 indexer launch), section
// "Modifications / 3. Every row's exact top-2048 on up to 64 slices": a row's
// keys are split into slices of contiguous positions, each slice holds its
// keys as radix keys in on-chip memory, and for each digit (from the top)
// every slice publishes the histogram of its keys under the prefix found so
// far and reads every other slice's, finds the digit that holds the remaining
// k-th key and the count above it.
//
// On GB300 a row is one thread-block cluster (16 CTAs, else 8): the slices are
// the cluster's CTAs and the all-gather is a read of the other CTAs' shared
// memory (DSMEM) after a hardware cluster barrier, so no slice ever spins on
// another.  The radix key is the order-preserving uint32 image of the f32
// score (-0 folded into +0, NaN below every number).  Four 8-bit digit rounds
// give the exact k-th largest image T and the number kr of keys equal to T
// that the list takes; each slice then counts its keys above / at T, the
// counts of earlier slices give its output offsets, and warps write positions
// in order with ballot ranks: keys above T first, then ties, each in
// ascending position.
#include <cooperative_groups.h>

#include "idx_internal.h"
#include "ptx.cuh"

namespace cg = cooperative_groups;

namespace idx {

namespace {

constexpr int kThreads = kSelectThreads;  // 256: one thread per histogram bin
constexpr int kWarps = kThreads / 32;
constexpr int kBins = 256;
constexpr int kMaxSmemKeys = 12288;       // per slice; longer slices re-read global memory

__device__ __forceinline__ uint32_t radix_key(float x) {
    uint32_t b = __float_as_uint(x);
    if ((b & 0x7FFFFFFFu) > 0x7F800000u) return 0u;  // NaN: below every number
    if (b == 0x80000000u) b = 0u;                    // -0 == +0
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

struct SliceView {
    const float* g;        // this slice's scores in global memory
    const uint32_t* s;     // radix keys held in shared memory
    int n_smem;            // keys [0, n_smem) are in shared memory
    __device__ __forceinline__ uint32_t operator()(int i) const {
        return i < n_smem ? s[i] : radix_key(__ldg(g + i));
    }
};

__device__ __forceinline__ uint32_t lanemask_lt() {
    uint32_t m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

template <int CL>
__global__ void __launch_bounds__(kThreads)
k_select(const float* __restrict__ scores, int64_t stride, const int32_t* __restrict__ row_lens,
         int k, int32_t* __restrict__ out, uint32_t* status, int smem_keys) {
    cg::cluster_group cluster = cg::this_cluster();
    const int c = (int)cluster.block_rank();
    const int row = blockIdx.y;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    extern __shared__ uint32_t keys_s[];
    __shared__ uint32_t hist[2][kBins];
    __shared__ uint32_t wsum[kWarps];
    __shared__ uint32_t pick[2];             // digit, count above it
    __shared__ uint32_t counts[2];           // this slice: keys > T, keys == T (read remotely)
    __shared__ uint32_t wcnt[2][kWarps];     // per-warp counts, then exclusive offsets
    __shared__ uint32_t base[2];             // keys > T / == T in earlier slices

    int64_t n = row_lens[row];
    if (n < 0 || n > stride) {
        if (c == 0 && tid == 0) record_status(status, kStatusBounds);
        n = n < 0 ? 0 : stride;
    }
    int32_t* dst = out + (int64_t)row * k;
    if (n <= k) {  // uniform over the cluster: no barrier is skipped by a subset
        if (c == 0)
            for (int j = tid; j < k; j += kThreads) dst[j] = j < n ? j : -1;
        return;
    }

    // ---- slice plan: one slice per kSliceKeys keys, at most CL slices -------
    int64_t ns = (n + kSliceKeys - 1) / kSliceKeys;
    if (ns > CL) ns = CL;
    int64_t per = (n + ns - 1) / ns;
    per = (per + 3) & ~int64_t(3);  // slice starts stay 16-byte aligned
    const int64_t start = (int64_t)c * per;
    const int cnt = (int)(start < n ? (n - start < per ? n - start : per) : 0);
    const float* src = scores + (int64_t)row * stride + start;

    // ---- radix keys into shared memory ---------------------------------------
    const int n_smem = cnt < smem_keys ? cnt : smem_keys;
    {
        const int nv = n_smem >> 2;
        const float4* src4 = reinterpret_cast<const float4*>(src);
        uint4* dst4 = reinterpret_cast<uint4*>(keys_s);
        for (int i = tid; i < nv; i += kThreads) {
            const float4 v = __ldg(src4 + i);
            dst4[i] = make_uint4(radix_key(v.x), radix_key(v.y), radix_key(v.z), radix_key(v.w));
        }
        for (int i = (nv << 2) + tid; i < n_smem; i += kThreads) keys_s[i] = radix_key(__ldg(src + i));
    }
    const SliceView key{src, keys_s, n_smem};

    // ---- digit rounds -------------------------------------------------------
    uint32_t prefix = 0, mask = 0;
    uint32_t kr = (uint32_t)k;  // rank still to find among keys under the prefix
#pragma unroll 1
    for (int round = 0; round < 4; ++round) {
        const int shift = 24 - 8 * round;
        uint32_t* h = hist[round & 1];
        h[tid] = 0;
        __syncthreads();
        const int span = (cnt + 31) & ~31;  // whole warps stay converged for match_any
        for (int i = tid; i < span; i += kThreads) {
            uint32_t u = 0;
            bool hit = false;
            if (i < cnt) {
                u = key(i);
                hit = (u & mask) == prefix;
            }
            const uint32_t active = __ballot_sync(0xFFFFFFFFu, hit);
            if (hit) {
                const uint32_t d = (u >> shift) & 0xFFu;
                const uint32_t peers = __match_any_sync(active, d);
                if (lane == __ffs(peers) - 1) atomicAdd(&h[d], (uint32_t)__popc(peers));
            }
        }
        cluster.sync();  // every slice's histogram of this round is complete

        // Bin tid summed over the cluster's slices.
        uint32_t tot = 0;
#pragma unroll 4
        for (int r = 0; r < CL; ++r) tot += cluster.map_shared_rank(h, r)[tid];
        // Suffix sums over bins (digit >= tid): within the warp from lane 31
        // down, then plus the totals of the warps holding higher bins.
        uint32_t incl = tot;  // sum of bins >= tid within this warp
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t t = __shfl_down_sync(0xFFFFFFFFu, incl, o);
            if (lane + o < 32) incl += t;
        }
        if (lane == 0) wsum[warp] = incl;  // total of this warp's bins
        __syncthreads();
        uint32_t above_warps = 0;
        for (int w = warp + 1; w < kWarps; ++w) above_warps += wsum[w];
        incl += above_warps;                 // keys with digit >= tid
        const uint32_t excl = incl - tot;    // keys with digit > tid
        if (excl < kr && incl >= kr) {
            pick[0] = (uint32_t)tid;
            pick[1] = excl;
        }
        __syncthreads();
        prefix |= pick[0] << shift;
        mask |= 0xFFu << shift;
        kr -= pick[1];
    }
    const uint32_t T = prefix;  // the k-th largest radix key of the row

    // ---- this slice's counts, per warp over contiguous sub-ranges ----------
    const int wspan = ((cnt + kWarps - 1) / kWarps + 31) & ~31;
    const int w_lo = min(cnt, warp * wspan), w_hi = min(cnt, w_lo + wspan);
    uint32_t n_gt = 0, n_eq = 0;
    for (int i = w_lo + lane; i < w_hi; i += 32) {
        const uint32_t u = key(i);
        n_gt += u > T;
        n_eq += u == T;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        n_gt += __shfl_xor_sync(0xFFFFFFFFu, n_gt, o);
        n_eq += __shfl_xor_sync(0xFFFFFFFFu, n_eq, o);
    }
    if (lane == 0) {
        wcnt[0][warp] = n_gt;
        wcnt[1][warp] = n_eq;
    }
    __syncthreads();
    if (tid == 0) {
        uint32_t a = 0, b = 0;
        for (int w = 0; w < kWarps; ++w) {
            const uint32_t x = wcnt[0][w], y = wcnt[1][w];
            wcnt[0][w] = a;
            wcnt[1][w] = b;
            a += x;
            b += y;
        }
        counts[0] = a;
        counts[1] = b;
    }
    cluster.sync();  // every slice's counts are published
    if (tid < 2) {
        uint32_t b = 0;
        for (int r = 0; r < c; ++r) b += cluster.map_shared_rank(counts, r)[tid];
        base[tid] = b;
    }
    __syncthreads();

    // ---- ordered writes -----------------------------------------------------
    const uint32_t gt_total = (uint32_t)k - kr;  // keys above T in the whole row
    uint32_t pos_gt = base[0] + wcnt[0][warp];
    uint32_t pos_eq = gt_total + base[1] + wcnt[1][warp];
    const uint32_t lt = lanemask_lt();
    for (int i0 = w_lo; i0 < w_hi; i0 += 32) {
        const int i = i0 + lane;
        const uint32_t u = i < w_hi ? key(i) : 0u;
        const bool gt = i < w_hi && u > T;
        const bool eq = i < w_hi && u == T;
        const uint32_t bg = __ballot_sync(0xFFFFFFFFu, gt);
        const uint32_t be = __ballot_sync(0xFFFFFFFFu, eq);
        if (gt) {
            const uint32_t pg = pos_gt + __popc(bg & lt);
            if (pg < gt_total) dst[pg] = (int32_t)(start + i);
        }
        if (eq) {
            const uint32_t pe = pos_eq + __popc(be & lt);
            if (pe < (uint32_t)k) dst[pe] = (int32_t)(start + i);
        }
        pos_gt += __popc(bg);
        pos_eq += __popc(be);
    }
    cluster.sync();  // no slice leaves while another may still read its counts
}

template <int CL>
cudaError_t launch_cluster(const SelectArgs& a, int smem_keys) {
    static int configured_device = -1;
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (configured_device != dev) {
        if (CL > 8) {
            err = cudaFuncSetAttribute(k_select<CL>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
            if (err != cudaSuccess) return err;
        }
        err = cudaFuncSetAttribute(k_select<CL>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   kMaxSmemKeys * 4);
        if (err != cudaSuccess) return err;
        configured_device = dev;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(CL, (unsigned)a.R, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = (size_t)smem_keys * 4;
    cfg.stream = a.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CL;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k_select<CL>, a.scores, a.score_stride, a.row_lens, a.k, a.indices,
                              a.status, smem_keys);
}

}  // namespace

cudaError_t launch_select(const SelectArgs& a) {
    // Keys per slice for the longest row the launch may see.
    const int64_t bound = a.max_len > 0 ? a.max_len : 1;
    auto smem_for = [&](int cl) {
        int64_t ns = (bound + kSliceKeys - 1) / kSliceKeys;
        if (ns > cl) ns = cl;
        int64_t per = ((bound + ns - 1) / ns + 3) & ~int64_t(3);
        return (int)(per < kMaxSmemKeys ? per : kMaxSmemKeys);
    };
    static int cluster16_ok = -1;
    if (cluster16_ok < 0) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(16, 1, 1);
        cfg.blockDim = dim3(kThreads, 1, 1);
        cfg.dynamicSmemBytes = (size_t)kMaxSmemKeys * 4;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 16;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int nclusters = 0;
        cudaError_t e1 = cudaFuncSetAttribute(k_select<16>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        cudaError_t e2 = cudaFuncSetAttribute(k_select<16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                              kMaxSmemKeys * 4);
        cudaError_t e3 = (e1 == cudaSuccess && e2 == cudaSuccess)
                             ? cudaOccupancyMaxActiveClusters(&nclusters, k_select<16>, &cfg)
                             : cudaErrorInvalidValue;
        cluster16_ok = (e3 == cudaSuccess && nclusters > 0) ? 1 : 0;
        (void)cudaGetLastError();  // a refused query leaves no sticky error
    }
    if (cluster16_ok) return launch_cluster<16>(a, smem_for(16));
    return launch_cluster<8>(a, smem_for(8));
}

}  // namespace idx
