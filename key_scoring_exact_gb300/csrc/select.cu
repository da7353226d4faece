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
//    lanes sharing a hot digit add once); each slice then adds its non-zero
//    bins into every slice's own totals with distributed-shared-memory
//    reductions, so after one hardware cluster barrier each slice scans its
//    local totals.  No slice spins on another; every wait is a cluster
//    barrier.
//  * After the first round, when the bin that holds the k-th key has at most
//    8,192 keys across the row, every slice appends its keys of that bin to a
//    candidate array in CTA 0 (a remote atomic reserves the room), and CTA 0
//    alone runs the last two rounds on them, then writes T and kr into every
//    slice: two rounds without a cluster barrier each.  A fuller bin takes
//    the last two rounds on all slices as above.
//  * Each slice then counts its keys above / at T and adds the counts to every
//    later slice; after one more barrier the counts of earlier slices give its
//    output offsets, and positions are written in order: keys above T first,
//    then ties, each in ascending position.
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
constexpr int kCandCap = 8192;      // candidates CTA 0 resolves alone after the first round
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
__device__ __forceinline__ void st_remote(uint32_t addr, uint32_t v) {
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t atom_add_remote(uint32_t addr, uint32_t v) {
    uint32_t old;
    asm volatile("atom.shared::cluster.add.u32 %0, [%1], %2;" : "=r"(old) : "r"(addr), "r"(v) : "memory");
    return old;
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
    uint32_t htot[3][kBinsMax];          // totals of every slice, one buffer per round
    uint32_t cnt[2][kMaxCluster];        // counts above / at T of every earlier slice
    uint32_t wsum[kWarps];
    uint32_t pick[3];                    // digit, keys above it, keys in it
    uint32_t cand_n;                     // candidates gathered so far (CTA 0's copy)
    uint32_t bcast[2];                   // T and kr, written by CTA 0 into every slice
    uint32_t woff[2][kMaxChunks * kWarps];  // per (chunk, warp) counts, then offsets
    uint32_t tot[2];                     // this slice's counts above / at T
    uint32_t base[2];                    // counts of the earlier slices
};

// One digit round (digit = (key >> shift) & (nb - 1)) over the slice's keys
// whose bits above the digit equal `prefix` under `mask`.  Leaves the digit
// holding rank kr (counted from the largest digit) and the number of keys
// above it in S.pick.  One copy of this code serves all rounds.
__device__ __noinline__ void digit_round(const uint32_t* __restrict__ keys, int cnt, uint32_t prefix,
                                         uint32_t mask, int shift, int nb, uint32_t kr, bool single, int r,
                                         int nslices, Shared& S) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int b = tid; b < nb; b += kThreads) S.hloc[b] = 0;
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
    const uint32_t* totals = S.hloc;
    if (!single) {
        // every non-zero bin into every slice's totals for this round
        for (int b = tid; b < nb; b += kThreads) {
            const uint32_t v = S.hloc[b];
            if (v)
                for (int t = 0; t < nslices; ++t) red_add_remote(map_rank(&S.htot[r][b], (uint32_t)t), v);
        }
        cluster_arrive();
        cluster_wait();
        totals = S.htot[r];
    }
    // Scan in descending digit order: thread tid holds digits nb-1-(bpt*tid+q).
    const int bpt = nb / kThreads;  // 2 or 1
    uint32_t tv[2] = {0u, 0u}, sum = 0;
    for (int q = 0; q < bpt; ++q) {
        tv[q] = totals[nb - 1 - (bpt * tid + q)];
        sum += tv[q];
    }
    uint32_t incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t x = __shfl_up_sync(kFull, incl, o);
        if (lane >= o) incl += x;
    }
    if (lane == 31) S.wsum[warp] = incl;
    __syncthreads();
    if (warp == 0) {  // exclusive prefix of the warp totals
        const uint32_t wv = S.wsum[lane];
        uint32_t wi = wv;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t x = __shfl_up_sync(kFull, wi, o);
            if (lane >= o) wi += x;
        }
        S.wsum[lane] = wi - wv;
    }
    __syncthreads();
    uint32_t above = S.wsum[warp] + incl - sum;
    for (int q = 0; q < bpt; ++q) {
        if (above < kr && above + tv[q] >= kr) {
            S.pick[0] = (uint32_t)(nb - 1 - (bpt * tid + q));
            S.pick[1] = above;
            S.pick[2] = tv[q];
        }
        above += tv[q];
    }
    __syncthreads();
}

template <int CL>
__global__ void __launch_bounds__(kThreads)
k_select(const float* __restrict__ scores, int64_t len_cap, const int32_t* __restrict__ row_lens,
         int64_t stride, int k, int32_t* __restrict__ out, uint32_t* status, int slice_cap) {
    extern __shared__ __align__(16) uint32_t keys_s[];  // slice_cap radix keys
    __shared__ Shared S;
    const uint32_t c = cluster_ctarank();
    const int row = blockIdx.y;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    int64_t n = row_lens[row];
    if (n < 0 || n > len_cap) {
        if (c == 0 && tid == 0) record_status(status, kStatusBounds);
        n = n < 0 ? 0 : len_cap;
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
        uint32_t* h = &S.htot[0][0];
        for (int i = tid; i < 3 * kBinsMax; i += kThreads) h[i] = 0;
        if (tid < 2 * kMaxCluster) (&S.cnt[0][0])[tid] = 0;
        if (tid == 0) S.cand_n = 0;
        __syncthreads();
        cluster_arrive();  // zeroed totals are released; waited on before the first add
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

    // ---- digit rounds: bits 31..21, then 20..10 and 9..0 ----------------------
    uint32_t prefix = 0, mask = 0, kr = (uint32_t)k;
    digit_round(keys_s, cnt, prefix, mask, 21, 2048, kr, single, 0, CL, S);
    prefix |= S.pick[0] << 21;
    mask |= 0x7FFu << 21;
    kr -= S.pick[1];
    const uint32_t in_bin = S.pick[2];  // keys of the row that share the first digit of T
    if (!single && in_bin <= (uint32_t)kCandCap) {
        // Few keys share the first digit: every slice sends those keys' values
        // to CTA 0, which finds the exact k-th largest among them alone, then
        // writes it (and the ties to take) into every slice.
        uint32_t* cand = keys_s + ((slice_cap + 4 + 3) & ~3);
        uint32_t mine = 0;
        const int n4 = (cnt + 3) >> 2;
        for (int i4 = tid; i4 < n4; i4 += kThreads) {
            const uint4 u = reinterpret_cast<const uint4*>(keys_s)[i4];
            const int i = 4 * i4;
            mine += (i + 0 < cnt && (u.x & mask) == prefix) + (i + 1 < cnt && (u.y & mask) == prefix) +
                    (i + 2 < cnt && (u.z & mask) == prefix) + (i + 3 < cnt && (u.w & mask) == prefix);
        }
        uint32_t incl = mine;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t x = __shfl_up_sync(kFull, incl, o);
            if (lane >= o) incl += x;
        }
        if (lane == 31) S.wsum[warp] = incl;
        __syncthreads();
        if (warp == 0) {
            const uint32_t wv = S.wsum[lane];
            uint32_t wi = wv;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t x = __shfl_up_sync(kFull, wi, o);
                if (lane >= o) wi += x;
            }
            S.wsum[lane] = wi - wv;
            if (lane == 31 && wi) S.tot[0] = atom_add_remote(map_rank(&S.cand_n, 0), wi);  // reserve
            if (lane == 31 && !wi) S.tot[0] = 0;
        }
        __syncthreads();
        {
            uint32_t at = S.tot[0] + S.wsum[warp] + incl - mine;
            const uint32_t rc = map_rank(cand, 0);
            for (int i4 = tid; i4 < n4; i4 += kThreads) {
                const uint4 u = reinterpret_cast<const uint4*>(keys_s)[i4];
                const int i = 4 * i4;
                if (i + 0 < cnt && (u.x & mask) == prefix) st_remote(rc + 4 * at++, u.x);
                if (i + 1 < cnt && (u.y & mask) == prefix) st_remote(rc + 4 * at++, u.y);
                if (i + 2 < cnt && (u.z & mask) == prefix) st_remote(rc + 4 * at++, u.z);
                if (i + 3 < cnt && (u.w & mask) == prefix) st_remote(rc + 4 * at++, u.w);
            }
        }
        cluster_arrive();
        cluster_wait();  // every candidate has landed in CTA 0
        if (c == 0) {
            const int nc = (int)S.cand_n;  // == in_bin
            digit_round(cand, nc, prefix, mask, 10, 2048, kr, true, 1, CL, S);
            uint32_t p2 = prefix | (S.pick[0] << 10), k2 = kr - S.pick[1];
            digit_round(cand, nc, p2, mask | (0x7FFu << 10), 0, 1024, k2, true, 2, CL, S);
            p2 |= S.pick[0];
            k2 -= S.pick[1];
            if (tid < 2 * CL) st_remote(map_rank(&S.bcast[tid & 1], (uint32_t)(tid >> 1)), (tid & 1) ? k2 : p2);
        }
        cluster_arrive();
        cluster_wait();  // T and kr are in every slice
        prefix = S.bcast[0];
        kr = S.bcast[1];
    } else {
        digit_round(keys_s, cnt, prefix, mask, 10, 2048, kr, single, 1, CL, S);
        prefix |= S.pick[0] << 10;
        mask |= 0x7FFu << 10;
        kr -= S.pick[1];
        digit_round(keys_s, cnt, prefix, mask, 0, 1024, kr, single, 2, CL, S);
        prefix |= S.pick[0];
        kr -= S.pick[1];
    }
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
        // this slice's counts into every later slice
        if (tid < 2 * kMaxCluster) {
            const int a = tid / kMaxCluster, t = tid % kMaxCluster;
            if ((uint32_t)t > c && t < CL) st_remote(map_rank(&S.cnt[a][c], (uint32_t)t), S.tot[a]);
        }
        cluster_arrive();
        cluster_wait();  // every earlier slice's counts have landed; no remote access follows
        if (warp == 0) {  // lanes 0..15: counts above T, 16..31: counts at T
            const int a = lane >> 4, r = lane & 15;
            uint32_t v = (uint32_t)r < c ? S.cnt[a][r] : 0u;
#pragma unroll
            for (int o = 1; o < 16; o <<= 1) v += __shfl_xor_sync(kFull, v, o);
            if (r == 0) S.base[a] = v;
        }
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
                                   (kSliceCapMax + 8) * 4 + kCandCap * 4);
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
    cfg.dynamicSmemBytes = (size_t)((cap + 4 + 3) & ~3) * 4 + (size_t)kCandCap * 4;
    cfg.stream = a.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CL;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const int64_t cap_len = a.len_cap < a.score_stride ? a.len_cap : a.score_stride;
    return cudaLaunchKernelEx(&cfg, k_select<CL>, a.scores, cap_len, a.row_lens, a.score_stride, a.k, a.indices,
                              a.status, cap);
}

bool cluster16_supported() {
    static int ok = -1;
    if (ok < 0) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(16, 1, 1);
        cfg.blockDim = dim3(kThreads, 1, 1);
        cfg.dynamicSmemBytes = (kSliceCapMax + 8) * 4 + kCandCap * 4;
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
                                     (kSliceCapMax + 8) * 4 + kCandCap * 4);
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
