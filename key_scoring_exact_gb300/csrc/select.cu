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
//  * A row is one thread-block cluster of 16, 8, 4, 2 or 1 CTAs, the size
//    chosen per launch (one CTA when the longest row has at most 12,288
//    keys; otherwise the largest whose slices hold the longest row and whose
//    clusters for all rows are resident at once).  The slices are the
//    cluster's CTAs; slice c covers positions [c P, (c + 1) P) with P fixed by
//    the launch's length bound, so its score loads go out together with the
//    read of the row's length; a row of at most P keys runs on one CTA alone.
//  * The launch is a programmatic dependent of the kernel before it (the
//    scoring): it waits for that grid before reading a score, and at once
//    allows the next launch (the next scoring) to start on the SMs it leaves
//    free.
//  * A slice's keys live in shared memory, as the order-preserving uint32
//    image of the f32 score (-0 folded into +0, NaN below every number).
//  * Digits of 11, 11 and 10 bits give the exact k-th largest image T and
//    the number kr of keys equal to T that the list takes.  The first
//    round's histogram is built while the slice is loaded.
//  * Histograms are built in shared memory with plain atomic adds (on this
//    hardware faster than aggregating equal digits within a warp first, even
//    when the scores crowd into a few bins).  The slices' histograms are
//    summed by reduce-scatter and all-gather: bin b belongs to slice
//    b / (bins / slices), every slice adds its non-zero bins there with a
//    distributed-shared-memory reduction, and after one hardware cluster
//    barrier each thread reads its four bins' totals from their owner with
//    one 16-byte remote load, then the block scans them.  No slice spins on
//    another; every wait is a cluster barrier.
//  * Leader path (a split row whose first digit's threshold bin holds at
//    most kLeadCap keys, the usual case): each thread scans its own run of
//    positions once, counting its keys above that bin and marking those in
//    it; the marked keys (the candidates) go to the leader, the last slice,
//    as (radix key, row position) pairs, with each slice's count above the
//    bin.  After one cluster barrier the leader finds the two lower digits
//    among the candidates with its own barriers only (one pass when the
//    second digit's bin holds a single candidate, which is then T), counts
//    each slice's candidates above and at T, and sends every slice T, kr and
//    the keys above / at T in the slices before it; one more cluster barrier
//    and every slice writes its part of the list.
//  * Otherwise two more cluster rounds: in the last one each thread scans its
//    own run, counting its keys above the 22-bit prefix and marking those
//    that match it; each slice sends its count above the prefix and its
//    non-zero last-digit bins (at most 8 of them) to the other slices with the
//    round's histogram, so after that round's barrier every slice knows how
//    many keys above T and at T the slices before it hold.  Only when some
//    slice has more non-zero bins does one more exchange (and barrier) follow.
//  * One block scan of the threads' packed (above T, at T) counts gives their
//    offsets, and the positions are written in order: keys above T first,
//    then ties, each in ascending position (or, for the slot variant, the
//    cache slots those positions map to; for the tagged variant, each entry
//    beside the launch's tag in one 8-byte store).
#include "idx_internal.h"
#include "ptx.cuh"

namespace idx {

namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
static_assert(kThreads >= 256 && kThreads <= 1024 && kThreads % 256 == 0, "block size");
constexpr int kLoadUnroll = 4096 / kThreads;  // float4 reads in flight per thread (16K keys a CTA)
constexpr int kBinsMax = 2048;
constexpr int kSliceTarget = 4096;  // keys per slice the launcher aims for
constexpr int kSingleMax = 12288;   // rows up to this long run on one CTA each (no cluster barrier)
constexpr int kSliceCapMax = 32768; // keys one slice can hold (128 KB of shared memory)
constexpr int kMaxCluster = 16;
constexpr uint32_t kMail = 8;  // last-digit bins a slice sends to the later slices
constexpr uint32_t kLeadCap = 4096;  // candidate keys the leader slice takes (else three cluster rounds)
constexpr uint32_t kFull = 0xFFFFFFFFu;
static_assert(kSliceCapMax / kThreads <= 32, "a thread's keys fit one 32-bit mask");

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
__device__ __forceinline__ void st_remote2(uint32_t addr, uint32_t a, uint32_t b) {  // addr 8-byte aligned
    asm volatile("st.shared::cluster.v2.u32 [%0], {%1, %2};" ::"r"(addr), "r"(a), "r"(b) : "memory");
}
__device__ __forceinline__ uint32_t atom_add_remote(uint32_t addr, uint32_t v) {
    uint32_t old;
    asm volatile("atom.shared::cluster.add.u32 %0, [%1], %2;" : "=r"(old) : "r"(addr), "r"(v) : "memory");
    return old;
}
__device__ __forceinline__ uint4 ld_remote4(uint32_t addr) {  // addr 16-byte aligned
    uint4 v;
    asm volatile("ld.shared::cluster.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr));
    return v;
}

__device__ __forceinline__ uint32_t radix_key(float x) {
    uint32_t b = __float_as_uint(x);
    if ((b & 0x7FFFFFFFu) > 0x7F800000u) return 0u;  // NaN: below every number
    if (b == 0x80000000u) b = 0u;                    // -0 == +0
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

struct __align__(16) Shared {
    uint32_t hloc[kBinsMax];             // this slice's histogram of the round
    uint32_t htot[3][kBinsMax];          // totals of every slice, one buffer per round
    uint32_t cnt[2][kMaxCluster];        // counts above / at T of every earlier slice
    uint32_t mail[kMaxCluster][kMail];   // last round: slice t's non-zero bins, (bin << 16) | count
    uint32_t mail_n[kMaxCluster];        // last round: slice t's non-zero bins (> kMail: not all sent)
    uint32_t mail_above[kMaxCluster];    // last round: slice t's keys above the prefix
    uint32_t nz, above;                  // this slice's non-zero last-round bins, keys above the prefix
    uint32_t base[3];                    // keys above / at T before this slice; 1 if a slice sent too many bins
    uint32_t wsum[kWarps];
    uint32_t pick[3];                    // digit, keys above it, keys in it
    // leader path (slice 0 resolves the rest of T from the first digit's bin)
    uint32_t gt0[kMaxCluster];           // leader: keys above the first digit's bin, per slice
    uint32_t gtc[kMaxCluster];           // leader: candidates above T, per slice
    uint32_t eqc[kMaxCluster];           // leader: candidates equal to T, per slice
    uint32_t ncand;                      // leader: candidates received
    uint32_t lead[4];                    // from the leader: T, kr, keys above / at T before this slice
    uint32_t bin_min, bin_max;           // one-CTA rows: least and largest key in the first digit's bin
};
// 16-byte vector reads of the histograms, local and remote
static_assert(offsetof(Shared, hloc) % 16 == 0 && offsetof(Shared, htot) % 16 == 0 &&
                  (kBinsMax * sizeof(uint32_t)) % 16 == 0, "histograms need 16-byte alignment");

// Exclusive prefix sum over the block in thread order; *total gets the sum.
// Ends with a barrier, so S.wsum may be reused right after.
__device__ __forceinline__ uint32_t block_scan(uint32_t v, uint32_t* total, Shared& S) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    uint32_t incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t x = __shfl_up_sync(kFull, incl, o);
        if (lane >= o) incl += x;
    }
    if (lane == 31) S.wsum[warp] = incl;
    __syncthreads();
    const uint32_t wv = lane < kWarps ? S.wsum[lane] : 0u;
    uint32_t wi = wv;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t x = __shfl_up_sync(kFull, wi, o);
        if (lane >= o) wi += x;
    }
    const uint32_t before = __shfl_sync(kFull, wi - wv, warp);
    *total = __shfl_sync(kFull, wi, 31);
    __syncthreads();
    return before + incl - v;
}

// One digit round (digit = (key >> shift) & (nb - 1)) over the slice's keys
// whose bits above the digit equal `prefix` under `mask` (or over S.hloc as
// built by the caller, when `have_hist`).  Leaves the digit holding rank kr
// (counted from the largest digit), the number of keys above it and the
// number in it in S.pick.
//
// The `last` round also prepares the ordered writes: each thread scans its
// own run of positions [4 j0, 4 j1) and leaves its keys above the prefix in
// *above and, in *cmask, which of its keys match the prefix (bit 4 (j - j0)
// + q for position 4 j + q); the slice's count above the prefix and its
// non-zero bins (up to kMail of them, with their counts) go to the other
// slices ahead of the round's cluster barrier.
__device__ __forceinline__ void digit_round(const uint32_t* __restrict__ keys, int cnt, uint32_t prefix,
                                         uint32_t mask, int shift, int nb, uint32_t kr, bool single, int r,
                                         int nslices, bool have_hist, Shared& S, bool last = false,
                                         uint32_t c = 0, int j0 = 0, int j1 = 0, uint32_t* above_out = nullptr,
                                         uint32_t* cmask_out = nullptr, bool tie_check = false) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (!have_hist && last) {
        for (int b = tid; b < nb; b += kThreads) S.hloc[b] = 0;
        if (tid == 0) {
            S.nz = 0;
            S.above = 0;
        }
        __syncthreads();
        const uint32_t dm = (uint32_t)nb - 1;
        uint32_t above = 0, cm = 0;
        for (int j = j0; j < j1; ++j) {
            const uint4 u = reinterpret_cast<const uint4*>(keys)[j];
            const uint32_t uu[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                if (4 * j + q < cnt) {
                    const uint32_t hi = uu[q] & mask;
                    if (hi == prefix) {
                        atomicAdd(&S.hloc[(uu[q] >> shift) & dm], 1u);
                        cm |= 1u << (4 * (j - j0) + q);
                    } else {
                        above += (uint32_t)(hi > prefix);
                    }
                }
            }
        }
        *above_out = above;
        *cmask_out = cm;
        above = __reduce_add_sync(kFull, above);
        if (lane == 0 && above) atomicAdd(&S.above, above);
    } else if (!have_hist && tie_check) {
        // As the branch below, over the thread's own run; besides the
        // histogram it marks the keys under the prefix, counts those above it
        // and finds their least and largest key (S.bin_min, S.bin_max).
        for (int b = tid; b < nb; b += kThreads) S.hloc[b] = 0;
        __syncthreads();
        const uint32_t dm = (uint32_t)nb - 1;
        uint32_t above = 0, cm = 0, lo = 0xFFFFFFFFu, hi_key = 0u;
        for (int j = j0; j < j1; ++j) {
            const uint4 u = reinterpret_cast<const uint4*>(keys)[j];
            const uint32_t uu[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                if (4 * j + q < cnt) {
                    const uint32_t hi = uu[q] & mask;
                    if (hi == prefix) {
                        atomicAdd(&S.hloc[(uu[q] >> shift) & dm], 1u);
                        cm |= 1u << (4 * (j - j0) + q);
                        lo = min(lo, uu[q]);
                        hi_key = max(hi_key, uu[q]);
                    } else {
                        above += (uint32_t)(hi > prefix);
                    }
                }
            }
        }
        *above_out = above;
        *cmask_out = cm;
        lo = __reduce_min_sync(kFull, lo);
        hi_key = __reduce_max_sync(kFull, hi_key);
        if (lane == 0) {
            atomicMin(&S.bin_min, lo);
            atomicMax(&S.bin_max, hi_key);
        }
    } else if (!have_hist) {
        for (int b = tid; b < nb; b += kThreads) S.hloc[b] = 0;
        __syncthreads();
        const uint32_t dm = (uint32_t)nb - 1;
        const int n4 = (cnt + 3) >> 2;
#pragma unroll 1
        for (int i4 = tid; i4 < n4; i4 += kThreads) {
            const uint4 u = reinterpret_cast<const uint4*>(keys)[i4];
            const int i = 4 * i4;
            if (i + 0 < cnt && (u.x & mask) == prefix) atomicAdd(&S.hloc[(u.x >> shift) & dm], 1u);
            if (i + 1 < cnt && (u.y & mask) == prefix) atomicAdd(&S.hloc[(u.y >> shift) & dm], 1u);
            if (i + 2 < cnt && (u.z & mask) == prefix) atomicAdd(&S.hloc[(u.z >> shift) & dm], 1u);
            if (i + 3 < cnt && (u.w & mask) == prefix) atomicAdd(&S.hloc[(u.w >> shift) & dm], 1u);
        }
    }
    __syncthreads();
    // every key under the prefix is the same: the caller has T, no scan needed
    if (tie_check && S.bin_min == S.bin_max) return;
    // Scan in descending digit order: thread tid < nb / bpt holds the bpt
    // digits b0 .. b0 + bpt - 1 (tv[q] = digit b0 + q), b0 = nb - bpt (tid + 1),
    // so threads in order cover the digits from the largest down; others none.
    constexpr int kBptMax = kBinsMax / kThreads < 4 ? 4 : kBinsMax / kThreads;
    const int bpt = nb / kThreads < 4 ? 4 : nb / kThreads;
    const int b0 = nb - bpt * (tid + 1);
    uint32_t tv[kBptMax];
#pragma unroll
    for (int q = 0; q < kBptMax; ++q) tv[q] = 0u;
    if (single) {
        if (b0 >= 0) {
#pragma unroll
            for (int q4 = 0; q4 < kBptMax / 4; ++q4) {
                if (4 * q4 < bpt) {
                    const uint4 t4 = *reinterpret_cast<const uint4*>(&S.hloc[b0 + 4 * q4]);
                    tv[4 * q4 + 0] = t4.x;
                    tv[4 * q4 + 1] = t4.y;
                    tv[4 * q4 + 2] = t4.z;
                    tv[4 * q4 + 3] = t4.w;
                }
            }
        }
    } else {
        // Bin b's total lives in slice b / (nb / nslices): each slice adds its
        // non-zero bins there (one remote add per bin), and after the barrier
        // every thread reads its bins' totals from their owner, four at a time.
        const int per_owner = nb / nslices;
        for (int b = tid; b < nb; b += kThreads) {
            const uint32_t v = S.hloc[b];
            if (v) {
                S.hloc[b] = 0u;  // the leader's rounds start from a zero histogram
                red_add_remote(map_rank(&S.htot[r][b], (uint32_t)(b / per_owner)), v);
                if (last) {
                    const uint32_t slot = atomicAdd(&S.nz, 1u);
                    if (slot < kMail)
                        for (int t = (int)c + 1; t < nslices; ++t)
                            st_remote(map_rank(&S.mail[c][slot], (uint32_t)t), ((uint32_t)b << 16) | v);
                }
            }
        }
        if (last) {
            __syncthreads();  // S.nz and S.above are final
            if (tid < nslices && tid != (int)c) {
                st_remote(map_rank(&S.mail_n[c], (uint32_t)tid), S.nz);
                st_remote(map_rank(&S.mail_above[c], (uint32_t)tid), S.above);
            }
        }
        cluster_arrive();
        cluster_wait();
        if (b0 >= 0) {
            const uint32_t own = (uint32_t)(b0 / per_owner);
#pragma unroll
            for (int q4 = 0; q4 < kBptMax / 4; ++q4) {
                if (4 * q4 < bpt) {
                    const uint4 t4 = ld_remote4(map_rank(&S.htot[r][b0 + 4 * q4], own));
                    tv[4 * q4 + 0] = t4.x;
                    tv[4 * q4 + 1] = t4.y;
                    tv[4 * q4 + 2] = t4.z;
                    tv[4 * q4 + 3] = t4.w;
                }
            }
        }
    }
    uint32_t sum = 0;
#pragma unroll
    for (int q = 0; q < kBptMax; ++q) sum += tv[q];
    // The warps' totals, then only the warp whose prefix reaches kr scans its
    // threads (digits run from the largest down in thread order).
    const uint32_t wtot = __reduce_add_sync(kFull, sum);
    if (lane == 0) S.wsum[warp] = wtot;
    __syncthreads();
    const uint32_t wv = lane < kWarps ? S.wsum[lane] : 0u;
    uint32_t wi = wv;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t x = __shfl_up_sync(kFull, wi, o);
        if (lane >= o) wi += x;
    }
    const uint32_t wbefore = __shfl_sync(kFull, wi - wv, warp);
    const uint32_t wafter = __shfl_sync(kFull, wi, warp);
    if (wbefore < kr && wafter >= kr) {  // warp-uniform
        uint32_t incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t x = __shfl_up_sync(kFull, incl, o);
            if (lane >= o) incl += x;
        }
        uint32_t above = wbefore + incl - sum;
#pragma unroll
        for (int q = kBptMax - 1; q >= 0; --q) {
            if (q < bpt) {
                if (above < kr && above + tv[q] >= kr) {
                    S.pick[0] = (uint32_t)(b0 + q);
                    S.pick[1] = above;
                    S.pick[2] = tv[q];
                }
                above += tv[q];
            }
        }
    }
    __syncthreads();
}

// The leader's digit round over its n candidates (radix keys in cand[i].x)
// whose bits under `mask` equal `prefix`: a histogram of digit (key >> shift)
// & (nb - 1) in S.hloc (zero on entry and on return), then the digit holding
// rank kr (counted from the largest) with the keys above it and in it in
// S.pick.  Only this CTA's barriers are used.
__device__ __forceinline__ void cand_round(const uint2* cand, int n, uint32_t prefix, uint32_t mask, int shift,
                                        int nb, uint32_t kr, Shared& S) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t dm = (uint32_t)nb - 1;
    for (int i = tid; i < n; i += kThreads) {
        const uint32_t u = cand[i].x;
        if ((u & mask) == prefix) atomicAdd(&S.hloc[(u >> shift) & dm], 1u);
    }
    __syncthreads();
    // thread tid holds digits b0 .. b0 + bpt - 1, from the largest down in thread order
    const int bpt = nb / kThreads < 1 ? 1 : nb / kThreads;  // 2 or 1
    const int b0 = nb - bpt * (tid + 1);
    uint32_t t0 = 0, t1 = 0;
    if (b0 >= 0) {
        t0 = S.hloc[b0];
        S.hloc[b0] = 0u;
        if (bpt == 2) {
            t1 = S.hloc[b0 + 1];
            S.hloc[b0 + 1] = 0u;
        }
    }
    const uint32_t sum = t0 + t1;
    const uint32_t wtot = __reduce_add_sync(kFull, sum);
    if (lane == 0) S.wsum[warp] = wtot;
    __syncthreads();
    const uint32_t wv = lane < kWarps ? S.wsum[lane] : 0u;
    uint32_t wi = wv;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t x = __shfl_up_sync(kFull, wi, o);
        if (lane >= o) wi += x;
    }
    const uint32_t wbefore = __shfl_sync(kFull, wi - wv, warp);
    const uint32_t wafter = __shfl_sync(kFull, wi, warp);
    if (wbefore < kr && wafter >= kr) {  // warp-uniform
        uint32_t incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t x = __shfl_up_sync(kFull, incl, o);
            if (lane >= o) incl += x;
        }
        uint32_t above = wbefore + incl - sum;
        if (bpt == 2) {  // the higher digit first
            if (above < kr && above + t1 >= kr) {
                S.pick[0] = (uint32_t)(b0 + 1);
                S.pick[1] = above;
                S.pick[2] = t1;
            }
            above += t1;
        }
        if (above < kr && above + t0 >= kr) {
            S.pick[0] = (uint32_t)b0;
            S.pick[1] = above;
            S.pick[2] = t0;
        }
    }
    __syncthreads();
}

// Words of a slice's radix keys in shared memory (a multiple of 4).
__host__ __device__ constexpr int slice_words(int cap) { return (cap + 4 + 3) & ~3; }

// List entries as positions, or as physical cache slots of the row's request;
// with `pairs`, each entry is written as a tagged pair instead.
struct SlotMap {
    const int32_t* table;    // [n_req][max_pages] page ids, or null for positions
    const int32_t* row_req;  // [R]
    int max_pages;
    long long* pairs;        // [R][k] tagged pairs, or null: entries into `out`
    uint32_t tag;
};

__device__ __forceinline__ int32_t list_entry(const int32_t* page_row, int64_t pos) {
    return page_row ? page_row[pos / kPage] * kPage + (int32_t)(pos % kPage) : (int32_t)pos;
}

// Entry j of the row's list: an int32, or the pair {entry, tag} (the int32
// words in that order) in one 8-byte store, so that a reader that sees the
// launch's tag in a pair sees that launch's entry beside it.
__device__ __forceinline__ void put_entry(int32_t* dst, long long* pdst, uint32_t tag, int64_t j, int32_t e) {
    if (pdst)
        pdst[j] = (long long)(((unsigned long long)tag << 32) | (unsigned long long)(uint32_t)e);
    else
        dst[j] = e;
}

template <int CL>
__global__ void __launch_bounds__(kThreads)
k_select(const float* __restrict__ scores, int64_t len_cap, const int32_t* __restrict__ row_lens,
         int64_t stride, int k, int32_t* __restrict__ out, uint32_t* status, int slice_cap, SlotMap sm) {
    // slice_cap radix keys (+ 4); after them, in clusters of more than one
    // CTA, the leader's (radix key, row position) of every candidate
    extern __shared__ __align__(16) uint32_t keys_s[];
    __shared__ Shared S;
    const uint32_t c = cluster_ctarank();
    const int row = blockIdx.y;
    const int tid = threadIdx.x;
    // The next launch on the stream (the next step's scoring) may start setting
    // up on the SMs this launch leaves free; it waits for this grid to finish
    // before it reads or writes anything in global memory.
    pdl_launch_dependents();
    // Shared-memory set-up, which reads no global memory, overlaps the wait.
    for (int i = tid; i < kBinsMax; i += kThreads) S.hloc[i] = 0;
    {
        uint32_t* h = &S.htot[0][0];
        for (int i = tid; i < 3 * kBinsMax; i += kThreads) h[i] = 0;
    }
    if (tid < 2 * kMaxCluster) (&S.cnt[0][0])[tid] = 0;
    if (tid < kMaxCluster) {
        S.gt0[tid] = 0;
        S.gtc[tid] = 0;
        S.eqc[tid] = 0;
    }
    if (tid == 0) {
        S.ncand = 0;
        S.bin_min = 0xFFFFFFFFu;
        S.bin_max = 0u;
    }
    // This launch is itself a programmatic dependent of the kernel before it
    // (the scoring): wait for that grid before reading a score.
    pdl_wait();

    // Slice c covers positions [c * slice_cap, (c + 1) * slice_cap) of the row
    // (slice_cap is fixed by the launch's length bound), so its score loads
    // are issued together with the read of the row's length.
    const int64_t start = (int64_t)c * slice_cap;
    const float* src = scores + (int64_t)row * stride + start;
    const int64_t lim64 = len_cap - start;  // keys of this slice inside the score buffer
    const int lim = lim64 <= 0 ? 0 : (lim64 < slice_cap ? (int)lim64 : slice_cap);
    const int lim4 = lim >> 2;
    const float4* src4 = reinterpret_cast<const float4*>(src);
    float4 v[kLoadUnroll];
#pragma unroll
    for (int u = 0; u < kLoadUnroll; ++u) {
        const int i = u * kThreads + tid;
        if (i < lim4) v[u] = __ldg(src4 + i);
    }

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
    long long* pdst = sm.pairs ? sm.pairs + (int64_t)row * k : nullptr;
    const int32_t* page_row = sm.table ? sm.table + (int64_t)sm.row_req[row] * sm.max_pages : nullptr;
    if (n <= k) {  // uniform over the cluster: no barrier is skipped by a subset
        if (c == 0)
            for (int j = tid; j < k; j += kThreads) put_entry(dst, pdst, sm.tag, j, j < n ? list_entry(page_row, j) : -1);
        return;
    }
    const bool single = CL == 1 || n <= slice_cap;  // one CTA a row: always (rows are cut to its slice above)
    if (single && c != 0) return;   // one CTA serves the row; no cluster barrier is used
    const int cnt = (int)(start < n ? (n - start < slice_cap ? n - start : slice_cap) : 0);

    __syncthreads();  // the shared memory zeroed before the grid wait is visible to every thread
    if (!single) cluster_arrive();  // zeroed totals are released; waited on before the first add

    // ---- radix keys into shared memory and the first round's histogram
    //      (bits 31..21), 16K keys' reads in flight ---------------------------------
    {
        const int n4 = cnt >> 2;
        uint4* k4 = reinterpret_cast<uint4*>(keys_s);
#pragma unroll 1
        for (int b = 0; b < n4; b += kLoadUnroll * kThreads) {
            if (b > 0) {
#pragma unroll
                for (int u = 0; u < kLoadUnroll; ++u) {
                    const int i = b + u * kThreads + tid;
                    if (i < n4) v[u] = __ldg(src4 + i);
                }
            }
#pragma unroll
            for (int u = 0; u < kLoadUnroll; ++u) {
                const int i = b + u * kThreads + tid;
                if (i < n4) {
                    const uint4 key = make_uint4(radix_key(v[u].x), radix_key(v[u].y), radix_key(v[u].z),
                                                 radix_key(v[u].w));
                    k4[i] = key;
                    atomicAdd(&S.hloc[key.x >> 21], 1u);
                    atomicAdd(&S.hloc[key.y >> 21], 1u);
                    atomicAdd(&S.hloc[key.z >> 21], 1u);
                    atomicAdd(&S.hloc[key.w >> 21], 1u);
                }
            }
        }
        const int tail = cnt & 3;
        if (tid < 4) {
            const uint32_t key = tid < tail ? radix_key(__ldg(src + 4 * n4 + tid)) : 0u;
            keys_s[4 * n4 + tid] = key;
            if (tid < tail) atomicAdd(&S.hloc[key >> 21], 1u);
        }
    }
    __syncthreads();
    if (!single) cluster_wait();

    // ---- digit rounds: bits 31..21, then 20..10 and 9..0; thread tid owns the
    //      slice's positions [4 j0, 4 j1) in the last round and the writes -------
    const int n4 = (cnt + 3) >> 2;
    const int m4 = (n4 + kThreads - 1) / kThreads;
    const int j0 = tid * m4 < n4 ? tid * m4 : n4;
    const int j1 = j0 + m4 < n4 ? j0 + m4 : n4;
    uint32_t kr = (uint32_t)k;
    digit_round(keys_s, cnt, 0u, 0u, 21, 2048, kr, single, 0, CL, true, S);
    uint32_t prefix = S.pick[0] << 21, mask = 0x7FFu << 21;
    kr -= S.pick[1];
    uint32_t T, gt_total, base_gt = 0, base_eq = 0, above = 0, cmask = 0, d_last = 0;
    const bool lead = CL > 1 && !single && S.pick[2] <= kLeadCap;  // the same in every slice of the row
    if (lead) {
        // The leader is the last slice: a decode row's top keys crowd into its
        // most recent positions, so most candidates stay in the leader's own
        // shared memory.
        constexpr uint32_t kLeader = (uint32_t)CL - 1;
        uint2* cand = reinterpret_cast<uint2*>(keys_s + slice_words(slice_cap));
        // ---- leader path: the keys in the first digit's threshold bin (the
        //      row's candidates) go to the leader, which finds T among them with
        //      CTA barriers only and sends every slice T and its offsets.
        //      Each thread scans its own run once: keys above the bin are
        //      counted, keys in it are marked (bit 4 (j - j0) + q for position
        //      4 j + q) and sent to the leader as (radix key, row position).
        const int lane = tid & 31;
        for (int j = j0; j < j1; ++j) {
            const uint4 u = reinterpret_cast<const uint4*>(keys_s)[j];
            const uint32_t uu[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                if (4 * j + q < cnt) {
                    const uint32_t hi = uu[q] & mask;
                    if (hi == prefix) cmask |= 1u << (4 * (j - j0) + q);
                    else above += (uint32_t)(hi > prefix);
                }
            }
        }
        const uint32_t m = (uint32_t)__popc(cmask);
        uint32_t incl = m;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t x = __shfl_up_sync(kFull, incl, o);
            if (lane >= o) incl += x;
        }
        uint32_t at = 0;
        if (lane == 31 && incl) at = atom_add_remote(map_rank(&S.ncand, kLeader), incl);
        at = __shfl_sync(kFull, at, 31) + incl - m;
        for (uint32_t b = cmask; b; b &= b - 1, ++at) {
            const int i = 4 * j0 + (__ffs(b) - 1);
            if (at < kLeadCap)
                st_remote2(map_rank(&cand[at], kLeader), keys_s[i], (uint32_t)(start + i));
        }
        const uint32_t wa = __reduce_add_sync(kFull, above);
        if (lane == 0 && wa) red_add_remote(map_rank(&S.gt0[c], kLeader), wa);
        cluster_arrive();
        cluster_wait();  // every candidate and count has reached the leader
        if (c == kLeader) {
            const int n_c = (int)(S.ncand < kLeadCap ? S.ncand : kLeadCap);
            cand_round(cand, n_c, prefix, mask, 10, 2048, kr, S);
            prefix |= S.pick[0] << 10;
            mask |= 0x7FFu << 10;
            kr -= S.pick[1];
            uint32_t t_key;
            if (S.pick[2] == 1) {
                // one candidate has the 22-bit prefix: it is T, and the others
                // compare with T as their 22-bit prefixes do
                for (int i = tid; i < n_c; i += kThreads) {
                    const uint2 e = cand[i];
                    const int sl = (int)(e.y / (uint32_t)slice_cap);
                    const uint32_t hi = e.x & mask;
                    if (hi > prefix) {
                        atomicAdd(&S.gtc[sl], 1u);
                    } else if (hi == prefix) {
                        atomicAdd(&S.eqc[sl], 1u);
                        S.pick[0] = e.x;
                    }
                }
                __syncthreads();
                t_key = S.pick[0];
                kr = 1;
            } else {
                cand_round(cand, n_c, prefix, mask, 0, 1024, kr, S);
                t_key = prefix | S.pick[0];
                kr -= S.pick[1];
                for (int i = tid; i < n_c; i += kThreads) {
                    const uint2 e = cand[i];
                    const int sl = (int)(e.y / (uint32_t)slice_cap);
                    if (e.x > t_key) atomicAdd(&S.gtc[sl], 1u);
                    else if (e.x == t_key) atomicAdd(&S.eqc[sl], 1u);
                }
                __syncthreads();
            }
            if (tid < CL) {
                uint32_t bg = 0, be = 0;
                for (int t = 0; t < tid; ++t) {
                    bg += S.gt0[t] + S.gtc[t];
                    be += S.eqc[t];
                }
                const uint32_t dst4 = map_rank(&S.lead[0], (uint32_t)tid);
                st_remote(dst4, t_key);
                st_remote(dst4 + 4, kr);
                st_remote(dst4 + 8, bg);
                st_remote(dst4 + 12, be);
            }
        }
        cluster_arrive();
        cluster_wait();  // T and the offsets have reached every slice
        T = S.lead[0];
        kr = S.lead[1];
        base_gt = S.lead[2];
        base_eq = S.lead[3];
        gt_total = (uint32_t)k - kr;
    } else {
        // ---- two more cluster rounds (bits 20..10, then 9..0).  In a launch of
        //      one CTA a row, the first of them also checks whether every key in
        //      the first digit's threshold bin is the same (a tie-heavy row: many
        //      keys of one value); then T is that key, the pass has marked the
        //      bin's keys and counted those above it, and the last round is not
        //      needed.
        constexpr bool kTieCheck = CL == 1;  // rows on one CTA each (launches of short rows)
        digit_round(keys_s, cnt, prefix, mask, 10, 2048, kr, single, 1, CL, false, S, false, c, j0, j1, &above,
                    &cmask, kTieCheck);
        if (kTieCheck && S.bin_min == S.bin_max) {
            T = S.bin_min;  // kr of the bin's keys, all equal to T, complete the list
        } else {
            prefix |= S.pick[0] << 10;
            mask |= 0x7FFu << 10;
            kr -= S.pick[1];
            digit_round(keys_s, cnt, prefix, mask, 0, 1024, kr, single, 2, CL, false, S, true, c, j0, j1, &above,
                        &cmask);
            d_last = S.pick[0];
            T = prefix | d_last;  // the k-th largest radix key of the row
            kr -= S.pick[1];
        }
        gt_total = (uint32_t)k - kr;
    }

    // ---- this thread's counts above and at T, packed (above < 2^11, at <=
    //      slice_cap < 2^16), scanned in thread order; only the marked keys
    //      are looked at again --------------------------------------------------
    uint32_t gt = above, eq = 0;
    for (uint32_t m = cmask; m; m &= m - 1) {
        const uint32_t u = keys_s[4 * j0 + (__ffs(m) - 1)];
        gt += (uint32_t)(u > T);
        eq += (uint32_t)(u == T);
    }
    const uint32_t mine = (gt << 16) | eq;
    if (!single && !lead && (tid >> 5) == 0) {
        // Keys above / at T in the slices before this one, from what they sent
        // with the last round (lane t: slice t), unless a slice had more
        // non-zero bins than it could send.
        const int lane = tid & 31;
        uint32_t n_t = 0, g_t = 0, e_t = 0;
        if (lane < CL) {
            n_t = lane == (int)c ? S.nz : S.mail_n[lane];
            if (lane < (int)c) {
                g_t = S.mail_above[lane];
                const uint32_t ne = n_t < kMail ? n_t : kMail;
                for (uint32_t e = 0; e < ne; ++e) {
                    const uint32_t x = S.mail[lane][e];
                    if ((x >> 16) > d_last) g_t += x & 0xFFFFu;
                    else if ((x >> 16) == d_last) e_t += x & 0xFFFFu;
                }
            }
        }
        const uint32_t ovf = __any_sync(kFull, n_t > kMail) ? 1u : 0u;
        g_t = __reduce_add_sync(kFull, g_t);
        e_t = __reduce_add_sync(kFull, e_t);
        if (lane == 0) {
            S.base[0] = g_t;
            S.base[1] = e_t;
            S.base[2] = ovf;
        }
    }
    uint32_t total;
    const uint32_t off = block_scan(mine, &total, S);  // its barriers also publish S.base
    if (!single && !lead && !S.base[2]) {
        base_gt = S.base[0];
        base_eq = S.base[1];
    } else if (!single && !lead) {
        // this slice's counts into every later slice (kept apart: a row's ties
        // may outnumber 2^16)
        if (tid > (int)c && tid < CL) {
            st_remote(map_rank(&S.cnt[0][c], (uint32_t)tid), total >> 16);
            st_remote(map_rank(&S.cnt[1][c], (uint32_t)tid), total & 0xFFFFu);
        }
        cluster_arrive();
        cluster_wait();  // every earlier slice's counts have landed; no remote access follows
        for (int t = 0; t < (int)c; ++t) {
            base_gt += S.cnt[0][t];
            base_eq += S.cnt[1][t];
        }
    }
    // ---- ordered writes --------------------------------------------------------
    if (mine) {
        uint32_t pg = base_gt + (off >> 16);
        uint32_t pe = gt_total + base_eq + (off & 0xFFFFu);
        for (int j = j0; j < j1; ++j) {
            const uint4 u = reinterpret_cast<const uint4*>(keys_s)[j];
            const uint32_t uu[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int i = 4 * j + q;
                if (i >= cnt) break;
                if (uu[q] > T) {
                    if (pg < gt_total) put_entry(dst, pdst, sm.tag, pg, list_entry(page_row, start + i));
                    ++pg;
                } else if (uu[q] == T) {
                    if (pe < (uint32_t)k) put_entry(dst, pdst, sm.tag, pe, list_entry(page_row, start + i));
                    ++pe;
                }
            }
        }
    }
}

// ---- the pages' list order --------------------------------------------------
//
// "sgl-amd-mono-upstream PR 18", section "Modifications / 3", Order: the
// pages' radix stops at the first of the threshold's 12- and 24-bit prefixes
// whose keys fit the candidate room, else at 32 bits, and its list is the keys
// whose prefix is above the threshold's, in position order, then the prefix's
// keys above the threshold, then the ties.  The pages do not size the room;
// the caller gives it.  Given a row's list in this library's order (keys above
// T, then ties, each in ascending position) this launch finds T (the smallest
// image on the list), counts the row's keys sharing T's 12- and 24-bit
// prefixes, and partitions the list stably into the three parts.
constexpr int kOrderThreads = 512;
constexpr int kOrderWarps = kOrderThreads / 32;

// Exclusive sums over the block in thread order of three counts at once.
__device__ __forceinline__ void order_scan3(uint32_t (&v)[3], uint32_t (&tot)[3], uint32_t* ws) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    uint32_t inc[3];
#pragma unroll
    for (int c = 0; c < 3; ++c) {
        inc[c] = v[c];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t x = __shfl_up_sync(kFull, inc[c], o);
            if (lane >= o) inc[c] += x;
        }
        if (lane == 31) ws[c * kOrderWarps + warp] = inc[c];
    }
    __syncthreads();
#pragma unroll
    for (int c = 0; c < 3; ++c) {
        const uint32_t wv = lane < kOrderWarps ? ws[c * kOrderWarps + lane] : 0u;
        uint32_t wi = wv;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t x = __shfl_up_sync(kFull, wi, o);
            if (lane >= o) wi += x;
        }
        const uint32_t before = __shfl_sync(kFull, wi - wv, warp);
        tot[c] = __shfl_sync(kFull, wi, 31);
        v[c] = before + inc[c] - v[c];
    }
    __syncthreads();
}

__global__ void __launch_bounds__(kOrderThreads)
k_prefix_order(const float* __restrict__ scores, int64_t len_cap, const int32_t* __restrict__ row_lens, int64_t stride,
               int k, int64_t room, int32_t* __restrict__ out) {
    __shared__ int32_t lst[IDX_MAX_K];
    __shared__ uint32_t img[IDX_MAX_K];
    __shared__ uint32_t ws[3 * kOrderWarps];
    const int row = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    pdl_launch_dependents();
    pdl_wait();  // the selection's list is complete
    int64_t n = row_lens[row];
    n = n < 0 ? 0 : (n > len_cap ? len_cap : n);
    if (n <= k) return;  // every key, then -1: the same in every order
    int32_t* dst = out + (int64_t)row * k;
    const float* srow = scores + (int64_t)row * stride;
    // the list, its keys' images, and T: the smallest image on it
    uint32_t tmin = 0xFFFFFFFFu;
    for (int j = tid; j < k; j += kOrderThreads) {
        const int32_t p = dst[j];
        const uint32_t u = (p >= 0 && p < n) ? radix_key(srow[p]) : 0xFFFFFFFFu;
        lst[j] = p;
        img[j] = u;
        tmin = min(tmin, u);
    }
    tmin = __reduce_min_sync(kFull, tmin);
    if (lane == 0) ws[warp] = tmin;
    __syncthreads();
    const uint32_t T = __reduce_min_sync(kFull, lane < kOrderWarps ? ws[lane] : 0xFFFFFFFFu);
    __syncthreads();
    // the row's keys sharing T's 12- and 24-bit prefixes
    uint32_t c12 = 0, c24 = 0;
    const int n4 = (int)((n + 3) >> 2);
    const float4* src4 = reinterpret_cast<const float4*>(srow);
    for (int i = tid; i < n4; i += kOrderThreads) {
        const float4 v = __ldcg(src4 + i);
        const float f[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            if (4 * (int64_t)i + q < n) {
                const uint32_t u = radix_key(f[q]);
                c12 += (uint32_t)((u >> 20) == (T >> 20));
                c24 += (uint32_t)((u >> 8) == (T >> 8));
            }
        }
    }
    c12 = __reduce_add_sync(kFull, c12);
    c24 = __reduce_add_sync(kFull, c24);
    if (lane == 0) {
        ws[warp] = c12;
        ws[kOrderWarps + warp] = c24;
    }
    __syncthreads();
    const uint32_t n12 = __reduce_add_sync(kFull, lane < kOrderWarps ? ws[lane] : 0u);
    const uint32_t n24 = __reduce_add_sync(kFull, lane < kOrderWarps ? ws[kOrderWarps + lane] : 0u);
    __syncthreads();
    const int sh = (int64_t)n12 <= room ? 20 : ((int64_t)n24 <= room ? 8 : 0);
    const uint32_t tp = T >> sh;
    // stable partition of the list: prefix above (0), prefix equal and above T (1), ties (2)
    const int per = (k + kOrderThreads - 1) / kOrderThreads;
    const int j0 = min(k, tid * per), j1 = min(k, j0 + per);
    uint32_t cnt[3] = {0u, 0u, 0u};
    for (int j = j0; j < j1; ++j) {
        const uint32_t u = img[j];
        cnt[(u >> sh) > tp ? 0 : (u > T ? 1 : 2)] += 1u;
    }
    uint32_t tot[3];
    order_scan3(cnt, tot, ws);
    uint32_t at[3] = {cnt[0], tot[0] + cnt[1], tot[0] + tot[1] + cnt[2]};
    for (int j = j0; j < j1; ++j) {
        const uint32_t u = img[j];
        const int c = (u >> sh) > tp ? 0 : (u > T ? 1 : 2);
        dst[at[c]++] = lst[j];
    }
}

}  // namespace

cudaError_t launch_prefix_order(const SelectArgs& a, int64_t room) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)a.R, 1, 1);
    cfg.blockDim = dim3(kOrderThreads, 1, 1);
    cfg.stream = a.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const int64_t cap_len = a.len_cap < a.score_stride ? a.len_cap : a.score_stride;
    return cudaLaunchKernelEx(&cfg, k_prefix_order, a.scores, cap_len, a.row_lens, a.score_stride, a.k, room, a.indices);
}

namespace {

int slice_cap_for(int cl, int64_t max_len) {
    int64_t ns = (max_len + kSliceTarget - 1) / kSliceTarget;
    if (ns > cl) ns = cl;
    if (ns < 1) ns = 1;
    int64_t per = ((max_len + ns - 1) / ns + 3) & ~int64_t(3);
    if (per < 4) per = 4;
    return (int)(per < kSliceCapMax ? per : kSliceCapMax);
}

// Dynamic shared memory of k_select<CL>: the slice's keys, then (CL > 1)
// the leader's candidate buffer.
template <int CL>
constexpr size_t slice_bytes(int cap) {
    return (size_t)slice_words(cap) * 4 + (CL > 1 ? (size_t)kLeadCap * sizeof(uint2) : 0);
}

// Once per device (and host thread: setting the attributes is idempotent):
// cluster and shared-memory attributes of k_select<CL>.
template <int CL>
cudaError_t configure(int dev) {
    static thread_local int configured_device = -1;
    if (configured_device == dev) return cudaSuccess;
    cudaError_t err = cudaSuccess;
    if (CL > 8) {
        err = cudaFuncSetAttribute(k_select<CL>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (err != cudaSuccess) return err;
    }
    err = cudaFuncSetAttribute(k_select<CL>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)slice_bytes<CL>(kSliceCapMax));
    if (err != cudaSuccess) return err;
    err = cudaFuncSetAttribute(k_select<CL>, cudaFuncAttributePreferredSharedMemoryCarveout,
                               cudaSharedmemCarveoutMaxShared);
    if (err != cudaSuccess) return err;
    configured_device = dev;
    return cudaSuccess;
}

template <int CL>
cudaError_t launch_c(const SelectArgs& a) {
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    err = configure<CL>(dev);
    if (err != cudaSuccess) return err;
    const int cap = slice_cap_for(CL, a.max_len);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(CL, (unsigned)a.R, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = slice_bytes<CL>(cap);
    cfg.stream = a.stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CL;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    // a programmatic dependent of the kernel before it (k_select waits for it)
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    const int64_t cap_len = a.len_cap < a.score_stride ? a.len_cap : a.score_stride;
    const SlotMap sm{a.slot_table, a.slot_row_req, a.slot_max_pages, a.pairs, a.tag};
    return cudaLaunchKernelEx(&cfg, k_select<CL>, a.scores, cap_len, a.row_lens, a.score_stride, a.k, a.indices,
                              a.status, cap, sm);
}

// Clusters of CL CTAs (slices of `cap` keys) that can be resident at once on
// this device; 0 when the size is refused.  Cached per host thread and
// (device, CL, cap).
template <int CL>
int max_active_clusters(int cap) {
    static thread_local int cached_dev = -1, cached_cap = -1, cached = 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    if (dev == cached_dev && cap == cached_cap) return cached;
    int n = 0;
    cudaError_t e = configure<CL>(dev);
    if (e == cudaSuccess) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(CL, 1, 1);
        cfg.blockDim = dim3(kThreads, 1, 1);
        cfg.dynamicSmemBytes = slice_bytes<CL>(cap);
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = CL;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        e = cudaOccupancyMaxActiveClusters(&n, k_select<CL>, &cfg);
    }
    if (e != cudaSuccess) n = 0;
    (void)cudaGetLastError();  // a refused query leaves no sticky error
    cached_dev = dev;
    cached_cap = cap;
    cached = n;
    return n;
}

}  // namespace

int64_t select_max_len(int cluster) { return (int64_t)cluster * kSliceCapMax; }

// The cluster size: one CTA per row when the longest row has at most
// kSingleMax keys (its three passes over the keys cost less than the cluster
// barriers of a split row); otherwise the largest of 16, 8, 4, 2, 1 CTAs, but
// no more than the longest row's slices of kSliceTarget keys, whose slices
// hold the longest row and whose clusters for all rows are resident at once;
// when no size fits the rows in one wave, the smallest size that holds the
// row (the most rows at once).  A row's slices then do more work each, but
// every CTA's time is mostly fixed latencies (barriers, exchanges), so fewer
// waves win.
cudaError_t launch_select(const SelectArgs& a) {
    if (a.max_len <= kSingleMax && max_active_clusters<1>(slice_cap_for(1, a.max_len)) > 0) return launch_c<1>(a);
    int chosen = 0;
    const int sizes[] = {16, 8, 4, 2, 1};
    // no more CTAs than the longest row has slices of kSliceTarget keys: extra
    // CTAs would hold no keys yet take part in every cluster barrier
    const int64_t want = (a.max_len + kSliceTarget - 1) / kSliceTarget;
    for (int cl : sizes) {
        if (cl > 1 && (int64_t)(cl / 2) >= want) continue;
        if (a.max_len > select_max_len(cl)) break;  // smaller clusters cannot hold the row either
        const int cap = slice_cap_for(cl, a.max_len);
        int active = 0;
        switch (cl) {
            case 16: active = max_active_clusters<16>(cap); break;
            case 8: active = max_active_clusters<8>(cap); break;
            case 4: active = max_active_clusters<4>(cap); break;
            case 2: active = max_active_clusters<2>(cap); break;
            default: active = max_active_clusters<1>(cap); break;
        }
        if (active <= 0) continue;  // size refused on this device
        chosen = cl;
        if (a.R <= active) break;
    }
    switch (chosen) {
        case 16: return launch_c<16>(a);
        case 8: return launch_c<8>(a);
        case 4: return launch_c<4>(a);
        case 2: return launch_c<2>(a);
        case 1: return launch_c<1>(a);
        default: return cudaErrorInvalidValue;  // no cluster size holds the row
    }
}

}  // namespace idx
