// select.cu -- exact top-k of each row by a multi-slice radix select.
//
// "sgl-amd-mono-upstream PR 18" (GLM-5.3 indexer launch), section
// "Modifications / 3. Every row's exact top-2048 on up to 64 slices": a row's
// keys are split into slices of contiguous positions, each slice holds its
// keys as radix keys on chip, and for each digit (from the top) every slice
// contributes the histogram of its keys under the prefix found so far; the
// digit holding the remaining k-th key and the count above it follow.
//
// GB300 form:
//  * A row is one thread-block cluster (16 CTAs, else 8).  The slices are the
//    cluster's CTAs; a row short enough for one slice runs on one CTA alone.
//  * A slice's keys live in shared memory (loaded with float4 reads issued
//    together), as the order-preserving uint32 image of the f32 score (-0
//    folded into +0, NaN below every number).  The rounds run one compact
//    loop body, so a one-shot launch does not refetch unrolled code.
//  * Digits of 11, 11 and 10 bits: three rounds give the exact k-th largest
//    image T and the number kr of keys equal to T that the list takes.
//  * Histograms are built in shared memory with warp-aggregated atomics (the
//    lanes sharing a hot digit add once), then added into CTA 0's copy with
//    distributed-shared-memory reductions; after one hardware cluster barrier
//    every slice reads the totals back and scans them.  No slice spins on
//    another; every wait is a cluster barrier.
//  * Each slice then counts its keys above / at T; the counts of earlier
//    slices give its output offsets, and positions are written in order:
//    keys above T first, then ties, each in ascending position.
#include "idx_internal.h"
#include "ptx.cuh"

namespace idx {

namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
constexpr int kBinsMax = 2048;
constexpr int kSliceTarget = 4096;  // keys per slice the launcher aims for
constexpr int kSliceCapMax = 32768; // keys one slice can hold (128 KB of shared memory)
constexpr int kMaxChunks = kSliceCapMax / (4 * kThreads);
constexpr int kMaxCluster = 16;
constexpr uint32_t kFull = 0xFFFFFFFFu;

// ---------------------------------------------------------------- cluster PTX

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_arrive() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// shared::cluster address of `p` (a shared variable) in CTA `rank` of the cluster
__device__ __forceinline__ uint32_t map_rank(const void* p, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
    return r;
}
__device__ __forceinline__ void red_add_remote(uint32_t addr, uint32_t v) {
    asm volatile("red.shared::cluster.add.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t ld_remote(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}
__device__ __forceinline__ void st_remote(uint32_t addr, uint32_t v) {
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

__device__ __forceinline__ uint32_t radix_key(float x) {
    uint32_t b = __float_as_uint(x);
    if ((b & 0x7FFFFFFFu) > 0x7F800000u) return 0u;  // NaN: below every number
    if (b == 0x80000000u) b = 0u;                    // -0 == +0
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// Add one key per lane (where `hit`) to histogram h: the lanes that share
// the first hit lane's digit add together (the hot bin of a concentrated
// score distribution), the rest alone.
__device__ __forceinline__ void hist_add(uint32_t* h, bool hit, uint32_t d, int lane) {
    const uint32_t m = __ballot_sync(kFull, hit);
    if (m == 0) return;
    const int leader = __ffs(m) - 1;
    const uint32_t dl = __shfl_sync(kFull, d, leader);
    const uint32_t same = __ballot_sync(kFull, hit && d == dl);
    if (lane == leader) atomicAdd(&h[dl], (uint32_t)__popc(same));
    if (hit && !((same >> lane) & 1u)) atomicAdd(&h[d], 1u);
}

struct Shared {
    uint32_t hloc[kBinsMax];             // this slice's histogram of the round
    uint32_t htot[3][kBinsMax];          // cluster totals (CTA 0's copy is the one used)
    uint32_t ctot[3][kBinsMax / 32];     // coarse totals: 32 fine bins each (CTA 0's copy)
    uint32_t cloc[kBinsMax / 32];        // this slice's coarse histogram
    uint32_t cnt[2][kMaxCluster];        // per-slice counts above / at T (CTA 0's copy)
    uint32_t pick[2];
    uint32_t woff[2][kMaxChunks * kWarps];  // per (chunk, warp) counts, then offsets
    uint32_t tot[2];                     // this slice's counts above / at T
    uint32_t base[2];                    // counts of the earlier slices
};

// Warp 0: find the digit holding rank kr (counting from the largest digit)
// from nc coarse totals (32 digits each) and, inside the chosen coarse bin,
// its 32 fine totals.  coarse(i) / fine(i) read totals; the result goes to
// S.pick (digit, keys above it).
template <typename Coarse, typename Fine>
__device__ __forceinline__ void pick_digit_warp(int nc, uint32_t kr, Shared& S, int lane, Coarse coarse,
                                                Fine fine) {
    const int cpl = nc / 32;  // coarse bins per lane: 2 or 1; lane L holds nc-1-(L*cpl+q)
    uint32_t cv[2] = {0u, 0u}, s = 0;
    for (int q = 0; q < cpl; ++q) {
        cv[q] = coarse(nc - 1 - (lane * cpl + q));
        s += cv[q];
    }
    uint32_t incl = s;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t v = __shfl_up_sync(kFull, incl, o);
        if (lane >= o) incl += v;
    }
    uint32_t above = incl - s;
    int cb = -1;
    uint32_t cabove = 0;
    for (int q = 0; q < cpl; ++q) {
        if (above < kr && above + cv[q] >= kr) {
            cb = nc - 1 - (lane * cpl + q);
            cabove = above;
        }
        above += cv[q];
    }
    const uint32_t who = __ballot_sync(kFull, cb >= 0);
    const int src = who ? __ffs(who) - 1 : 0;
    cb = __shfl_sync(kFull, cb, src);
    cabove = __shfl_sync(kFull, cabove, src);
    if (cb < 0) cb = 0;  // unreachable when kr <= the keys under the prefix
    // fine bins of coarse bin cb, descending: lane L holds digit cb*32 + 31 - L
    const int d = cb * 32 + 31 - lane;
    const uint32_t f = fine(d);
    uint32_t finc = f;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t v = __shfl_up_sync(kFull, finc, o);
        if (lane >= o) finc += v;
    }
    const uint32_t fab = cabove + finc - f;
    if (fab < kr && fab + f >= kr) {
        S.pick[0] = (uint32_t)d;
        S.pick[1] = fab;
    }
}

// One digit round (digit = (key >> shift) & (nb - 1)) over the slice's keys
// whose bits above the digit equal `prefix` under `mask`.  Leaves the digit
// holding rank kr and the count above it in S.pick.  One copy of this code
// serves all rounds.
__device__ __noinline__ void digit_round(const uint32_t* __restrict__ keys, int cnt, uint32_t prefix,
                                         uint32_t mask, int shift, int nb, uint32_t kr, bool single, int r,
                                         Shared& S) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int bpt = nb / kThreads;  // fine bins per thread: 4 or 2
    const int tpc = 32 / bpt;       // threads per coarse bin: 8 or 16
    for (int q = 0; q < bpt; ++q) S.hloc[tid * bpt + q] = 0;
    __syncthreads();
    const uint32_t dm = (uint32_t)nb - 1;
    const int n4 = (cnt + 3) >> 2;
    const int span = (n4 + 31) & ~31;  // whole warps take each trip
#pragma unroll 1
    for (int i4 = tid; i4 < span; i4 += kThreads) {
        uint4 u = make_uint4(0, 0, 0, 0);
        if (i4 < n4) u = reinterpret_cast<const uint4*>(keys)[i4];
        const int i = 4 * i4;
        hist_add(S.hloc, i + 0 < cnt && (u.x & mask) == prefix, (u.x >> shift) & dm, lane);
        hist_add(S.hloc, i + 1 < cnt && (u.y & mask) == prefix, (u.y >> shift) & dm, lane);
        hist_add(S.hloc, i + 2 < cnt && (u.z & mask) == prefix, (u.z >> shift) & dm, lane);
        hist_add(S.hloc, i + 3 < cnt && (u.w & mask) == prefix, (u.w >> shift) & dm, lane);
    }
    __syncthreads();
    // coarse sums of 32 fine bins (tpc consecutive threads)
    uint32_t fv[4] = {0u, 0u, 0u, 0u}, part = 0;
    for (int q = 0; q < bpt; ++q) {
        fv[q] = S.hloc[tid * bpt + q];
        part += fv[q];
    }
    for (int o = 1; o < tpc; o <<= 1) part += __shfl_xor_sync(kFull, part, o);
    if (single) {
        if (tid % tpc == 0) S.cloc[tid / tpc] = part;
        __syncthreads();
        if (warp == 0)
            pick_digit_warp(nb / 32, kr, S, lane, [&](int i) { return S.cloc[i]; },
                            [&](int i) { return S.hloc[i]; });
    } else {
        const uint32_t rf = map_rank(&S.htot[r][0], 0), rc = map_rank(&S.ctot[r][0], 0);
        for (int q = 0; q < bpt; ++q)
            if (fv[q]) red_add_remote(rf + 4 * (tid * bpt + q), fv[q]);
        if (tid % tpc == 0 && part) red_add_remote(rc + 4 * (tid / tpc), part);
        cluster_arrive();
        cluster_wait();
        if (warp == 0)
            pick_digit_warp(nb / 32, kr, S, lane, [&](int i) { return ld_remote(rc + 4 * i); },
                            [&](int i) { return ld_remote(rf + 4 * i); });
    }
    __syncthreads();
}

template <int CL>
__global__ void __launch_bounds__(kThreads)
k_select(const float* __restrict__ scores, int64_t stride, const int32_t* __restrict__ row_lens,
         int k, int32_t* __restrict__ out, uint32_t* status, int slice_cap) {
    extern __shared__ __align__(16) uint32_t keys_s[];  // slice_cap radix keys
    __shared__ Shared S;
    const uint32_t c = cluster_ctarank();
    const int row = blockIdx.y;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    int64_t n = row_lens[row];
    if (n < 0 || n > stride) {
        if (c == 0 && tid == 0) record_status(status, kStatusBounds);
        n = n < 0 ? 0 : stride;
    }
    if (n > (int64_t)CL * slice_cap) {  // the launcher sizes slice_cap for the longest row
        if (c == 0 && tid == 0) record_status(status, kStatusBounds);
        n = (int64_t)CL * slice_cap;
    }
    int32_t* dst = out + (int64_t)row * k;
    if (n <= k) {  // uniform over the cluster: no barrier is skipped by a subset
        if (c == 0)
            for (int j = tid; j < k; j += kThreads) dst[j] = j < n ? j : -1;
        return;
    }

    // ---- slice plan ------------------------------------------------------
    int64_t ns = (n + kSliceTarget - 1) / kSliceTarget;
    if (ns > CL) ns = CL;
    int64_t per = (n + ns - 1) / ns;
    per = (per + 3) & ~int64_t(3);  // slice starts stay 16-byte aligned
    if (per > slice_cap) per = slice_cap;
    const bool single = ns == 1;
    if (single && c != 0) return;   // one CTA serves the row; no cluster barrier is used
    const int64_t start = (int64_t)c * per;
    const int cnt = (int)(start < n ? (n - start < per ? n - start : per) : 0);
    const float* src = scores + (int64_t)row * stride + start;

    if (!single) {
        if (c == 0) {
            uint32_t* h = &S.htot[0][0];
            for (int i = tid; i < 3 * kBinsMax; i += kThreads) h[i] = 0;
            uint32_t* hc = &S.ctot[0][0];
            for (int i = tid; i < 3 * (kBinsMax / 32); i += kThreads) hc[i] = 0;
        }
        cluster_arrive();  // CTA 0's zeroed totals are released; waited on before the first add
    }

    // ---- radix keys into shared memory: four float4 reads in flight -----
    {
        const int n4 = cnt >> 2;
        const float4* src4 = reinterpret_cast<const float4*>(src);
        uint4* k4 = reinterpret_cast<uint4*>(keys_s);
#pragma unroll 1
        for (int b = 0; b < n4; b += 4 * kThreads) {
            float4 v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int i = b + u * kThreads + tid;
                if (i < n4) v[u] = __ldg(src4 + i);
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int i = b + u * kThreads + tid;
                if (i < n4)
                    k4[i] = make_uint4(radix_key(v[u].x), radix_key(v[u].y), radix_key(v[u].z),
                                       radix_key(v[u].w));
            }
        }
        const int tail = cnt & 3;
        if (tid < 4) keys_s[4 * n4 + tid] = tid < tail ? radix_key(__ldg(src + 4 * n4 + tid)) : 0u;
    }
    __syncthreads();
    if (!single) cluster_wait();

    // ---- digit rounds: bits 31..21, 20..10, 9..0 ----------------------------
    uint32_t prefix = 0, mask = 0, kr = (uint32_t)k;
    digit_round(keys_s, cnt, prefix, mask, 21, 2048, kr, single, 0, S);
    prefix |= S.pick[0] << 21;
    mask |= 0x7FFu << 21;
    kr -= S.pick[1];
    digit_round(keys_s, cnt, prefix, mask, 10, 2048, kr, single, 1, S);
    prefix |= S.pick[0] << 10;
    mask |= 0x7FFu << 10;
    kr -= S.pick[1];
    digit_round(keys_s, cnt, prefix, mask, 0, 1024, kr, single, 2, S);
    prefix |= S.pick[0];
    kr -= S.pick[1];
    const uint32_t T = prefix;            // the k-th largest radix key of the row
    const uint32_t gt_total = (uint32_t)k - kr;

    // ---- counts per (chunk, warp), in position order.  Chunk j holds
    //      positions [2048 j, 2048 j + 2048); thread tid covers 4 of them. ----
    const int nchunks = (cnt + 4 * kThreads - 1) / (4 * kThreads);
#pragma unroll 1
    for (int j = 0; j < nchunks; ++j) {
        const int i = 4 * (j * kThreads + tid);
        const uint4 u = i < cnt ? reinterpret_cast<const uint4*>(keys_s)[j * kThreads + tid]
                                : make_uint4(0, 0, 0, 0);
        const uint32_t g = (i < cnt && u.x > T) + (i + 1 < cnt && u.y > T) + (i + 2 < cnt && u.z > T) +
                           (i + 3 < cnt && u.w > T);
        const uint32_t e = (i < cnt && u.x == T) + (i + 1 < cnt && u.y == T) + (i + 2 < cnt && u.z == T) +
                           (i + 3 < cnt && u.w == T);
        const uint32_t ga = __reduce_add_sync(kFull, g), ea = __reduce_add_sync(kFull, e);
        if (lane == 0) {
            S.woff[0][j * kWarps + warp] = ga;
            S.woff[1][j * kWarps + warp] = ea;
        }
    }
    __syncthreads();
    if (warp == 0) {  // exclusive offsets over (chunk, warp) in position order
        for (int a = 0; a < 2; ++a) {
            uint32_t carry = 0;
            for (int b0 = 0; b0 < nchunks * kWarps; b0 += 32) {
                const int b = b0 + lane;
                const uint32_t v = b < nchunks * kWarps ? S.woff[a][b] : 0u;
                uint32_t inc = v;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const uint32_t x = __shfl_up_sync(kFull, inc, o);
                    if (lane >= o) inc += x;
                }
                if (b < nchunks * kWarps) S.woff[a][b] = carry + inc - v;
                carry += __shfl_sync(kFull, inc, 31);
            }
            if (lane == 0) S.tot[a] = carry;
        }
    }
    __syncthreads();
    if (single) {
        if (tid < 2) S.base[tid] = 0;
    } else {
        if (tid < 2) st_remote(map_rank(&S.cnt[tid][c], 0), S.tot[tid]);
        cluster_arrive();
        cluster_wait();  // every slice's counts are in CTA 0
        if (warp == 0) {  // lanes 0..15: counts above T, 16..31: counts at T
            const int a = lane >> 4, r = lane & 15;
            uint32_t v = (uint32_t)r < c ? ld_remote(map_rank(&S.cnt[a][r], 0)) : 0u;
#pragma unroll
            for (int o = 1; o < 16; o <<= 1) v += __shfl_xor_sync(kFull, v, o);
            if (r == 0) S.base[a] = v;
        }
        __syncthreads();
        cluster_arrive();  // done reading CTA 0; waited on before leaving
    }
    __syncthreads();

    // ---- ordered writes --------------------------------------------------------
#pragma unroll 1
    for (int j = 0; j < nchunks; ++j) {
        const int i = 4 * (j * kThreads + tid);
        const uint4 u4 = i < cnt ? reinterpret_cast<const uint4*>(keys_s)[j * kThreads + tid]
                                 : make_uint4(0, 0, 0, 0);
        const uint32_t uu[4] = {u4.x, u4.y, u4.z, u4.w};
        uint32_t g = 0, e = 0;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            g += i + q < cnt && uu[q] > T;
            e += i + q < cnt && uu[q] == T;
        }
        // exclusive prefix of the lanes before this one
        uint32_t gi = g, ei = e;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t a = __shfl_up_sync(kFull, gi, o);
            const uint32_t b = __shfl_up_sync(kFull, ei, o);
            if (lane >= o) {
                gi += a;
                ei += b;
            }
        }
        uint32_t pg = S.base[0] + S.woff[0][j * kWarps + warp] + gi - g;
        uint32_t pe = gt_total + S.base[1] + S.woff[1][j * kWarps + warp] + ei - e;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            if (i + q >= cnt) break;
            if (uu[q] > T) {
                if (pg < gt_total) dst[pg] = (int32_t)(start + i + q);
                ++pg;
            } else if (uu[q] == T) {
                if (pe < (uint32_t)k) dst[pe] = (int32_t)(start + i + q);
                ++pe;
            }
        }
    }
    if (!single) cluster_wait();  // CTA 0 outlives every remote read of its memory
}

int slice_cap_for(int cl, int64_t max_len) {
    int64_t ns = (max_len + kSliceTarget - 1) / kSliceTarget;
    if (ns > cl) ns = cl;
    if (ns < 1) ns = 1;
    int64_t per = ((max_len + ns - 1) / ns + 3) & ~int64_t(3);
    if (per < 4) per = 4;
    return (int)(per < kSliceCapMax ? per : kSliceCapMax);
}

template <int CL>
cudaError_t launch_c(const SelectArgs& a) {
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
                                   kSliceCapMax * 4 + 16);
        if (err != cudaSuccess) return err;
        err = cudaFuncSetAttribute(k_select<CL>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                   cudaSharedmemCarveoutMaxShared);
        if (err != cudaSuccess) return err;
        configured_device = dev;
    }
    const int cap = slice_cap_for(CL, a.max_len);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(CL, (unsigned)a.R, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = (size_t)cap * 4 + 16;
    cfg.stream = a.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CL;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k_select<CL>, a.scores, a.score_stride, a.row_lens, a.k, a.indices,
                              a.status, cap);
}

bool cluster16_supported() {
    static int ok = -1;
    if (ok < 0) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(16, 1, 1);
        cfg.blockDim = dim3(kThreads, 1, 1);
        cfg.dynamicSmemBytes = kSliceCapMax * 4 + 16;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 16;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int nclusters = 0;
        cudaError_t e = cudaFuncSetAttribute(k_select<16>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(k_select<16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     kSliceCapMax * 4 + 16);
        if (e == cudaSuccess) e = cudaOccupancyMaxActiveClusters(&nclusters, k_select<16>, &cfg);
        ok = (e == cudaSuccess && nclusters > 0) ? 1 : 0;
        (void)cudaGetLastError();  // a refused query leaves no sticky error
    }
    return ok == 1;
}

}  // namespace

int64_t select_max_len(int cluster) { return (int64_t)cluster * kSliceCapMax; }

cudaError_t launch_select(const SelectArgs& a) {
    if (cluster16_supported()) {
        if (a.max_len > select_max_len(16)) return cudaErrorInvalidValue;
        return launch_c<16>(a);
    }
    if (a.max_len > select_max_len(8)) return cudaErrorInvalidValue;
    return launch_c<8>(a);
}

}  // namespace idx
