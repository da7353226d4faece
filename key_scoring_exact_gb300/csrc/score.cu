// score.cu -- paged key scoring on the 5th-generation tensor cores.
//
// For every group of (at most four consecutive) rows of one request and every
// 128-key tile of that request's keys:
//
//     D[key, (row, head)] = sum_d K[key, d] * Q'[(row, head), d]     (tcgen05)
//     s[row, key] = scale[key] * sum_h w'[row, h] * max(D[key, (row, h)], 0)
//
// which is the indexer score sum_h w * ReLU(q . (k * scale)) once the key's
// scale (>= 0) and the query's power-of-two factor are taken out of the ReLU
// (see prep.cu).  Every key of a request is read from HBM once per group, as
// "sgl-amd-mono-upstream PR 18" (GLM-5.3 indexer launch), section
// "Modifications / 2. A request's rows scored together" asks; its LDS batches
// of whole pages become TMA loads of whole 64-token pages into a ring of
// shared-memory stages.
//
// Keys sit on the MMA's M dimension (128 lanes of TMEM = 128 keys) and the
// group's (row, head) pairs on N (<= 256 columns), so the epilogue reads one
// key per thread and reduces over heads inside the thread: no cross-lane sums,
// and each warp stores 32 consecutive scores of a row.
//
// Warp roles (one CTA per SM, persistent over a contiguous range of tiles):
//   warp 0     TMA producer: the group's query (E4M3 hi/lo parts), then per
//              tile two key pages (TMA, 128-byte swizzle) + their scales
//              (bulk copy) into stage s of an 8-stage ring.
//   warp 1     TMEM allocator and MMA issuer: 4 (E4M3 query) or 8 (bf16 query,
//              hi and lo terms) kind::f8f6f4 MMAs of K = 32 per tile into one
//              of two TMEM accumulators.
//   warps 2-9  epilogue: tcgen05.ld the accumulator, ReLU, head-weighted sum,
//              times the key scale, masked coalesced f32 stores.
#include "idx_internal.h"
#include "ptx.cuh"

namespace idx {

namespace {

constexpr int kStages = 8;
constexpr int kEpiWarps = 8;
constexpr int kScoreThreads = 64 + kEpiWarps * 32;
constexpr uint32_t kQRows = kGroupRows * kHeads;           // 256
constexpr uint32_t kQPartBytes = kQRows * kDim;            // 32 KB
constexpr uint32_t kPageKeyBytes = kPage * kDim;           // 8 KB
constexpr uint32_t kPageScaleBytes = kPage * 4;            // 256 B
constexpr uint32_t kStageBytes = kTileKeys * kDim;         // 16 KB
constexpr uint32_t kStageScaleBytes = kTileKeys * 4;       // 512 B
constexpr uint32_t kAccCols = 256;
constexpr uint32_t kTmemCols = 2 * kAccCols;

constexpr uint32_t kOffQHi = 0;
constexpr uint32_t kOffQLo = kOffQHi + kQPartBytes;
constexpr uint32_t kOffStages = kOffQLo + kQPartBytes;
constexpr uint32_t kOffScales = kOffStages + kStages * kStageBytes;
constexpr uint32_t kOffWq = kOffScales + kStages * kStageScaleBytes;
constexpr uint32_t kWqPerWarp = 2 * kHeads;                 // two rows of head weights
constexpr uint32_t kOffBars = kOffWq + kEpiWarps * kWqPerWarp * 4;
constexpr uint32_t kNumBars = 2 * kStages + 4 + 3;
constexpr uint32_t kOffMisc = kOffBars + kNumBars * 8;
constexpr uint32_t kSmemUsed = kOffMisc + 16;
constexpr uint32_t kSmemBytes = kSmemUsed + 1024;  // slack for 1024-byte alignment
static_assert(kSmemBytes <= 232448, "shared memory budget");
static_assert(kOffStages % 1024 == 0 && kOffQLo % 1024 == 0, "swizzle atoms need 1024-byte alignment");

struct ScoreParams {
    const Plan* plan;
    const float* wq;
    const float* k_scale;
    const int32_t* block_table;
    int64_t pool_pages;
    int max_pages;
    int R;
    int two_terms;  // 1: bf16 query split into hi + lo E4M3 terms
    float* scores;
    int64_t score_stride;
    uint32_t* status;
};

// The group that holds work item `it`: the last g with g_item[g] <= it.
__device__ __forceinline__ int find_group(const Plan* plan, int it) {
    int lo = 0, hi = plan->n_groups;  // g_item[lo] <= it < g_item[hi]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (plan->g_item[mid] <= it) lo = mid; else hi = mid;
    }
    return lo;
}

__global__ void __launch_bounds__(kScoreThreads, 1)
k_score(const __grid_constant__ CUtensorMap keys_map, const __grid_constant__ CUtensorMap q_map,
        const ScoreParams p) {
    const Plan* plan = p.plan;
    const int n_items = plan->n_items;
    const int n_groups = plan->n_groups;
    const int it0 = (int)(((int64_t)blockIdx.x * n_items) / gridDim.x);
    const int it1 = (int)(((int64_t)(blockIdx.x + 1) * n_items) / gridDim.x);
    if (it0 >= it1 || n_groups < 1) return;

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* q_hi = smem + kOffQHi;
    uint8_t* q_lo = smem + kOffQLo;
    uint8_t* stages = smem + kOffStages;
    float* scales = reinterpret_cast<float*>(smem + kOffScales);
    float* wq_s = reinterpret_cast<float*>(smem + kOffWq);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBars);
    uint64_t* full = bars;                    // [kStages] keys + scales landed
    uint64_t* empty = bars + kStages;         // [kStages] MMA done and scales read
    uint64_t* tfull = bars + 2 * kStages;     // [2] accumulator ready
    uint64_t* tempty = tfull + 2;             // [2] accumulator drained
    uint64_t* qfull = tempty + 2;             // group query landed
    uint64_t* qempty = qfull + 1;             // MMAs on the group query done
    uint64_t* drain = qempty + 1;             // final MMA completion (abort path)
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1 + kEpiWarps);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&tfull[a], 1);
            mbar_init(&tempty[a], kEpiWarps);
        }
        mbar_init(qfull, 1);
        mbar_init(qempty, 1);
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
        prefetch_tensormap(&keys_map);
        prefetch_tensormap(&q_map);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            int g = find_group(plan, it0), cur_g = -1, qi = 0, li = 0;
            for (int it = it0; it < it1; ++it, ++li) {
                while (g + 1 < n_groups && it >= plan->g_item[g + 1]) ++g;
                if (g != cur_g) {
                    if (!bounded_wait(qempty, (qi & 1) ^ 1, abort_flag)) break;
                    const int r0 = plan->g_r0[g], nr = plan->g_nr[g];
                    mbar_arrive_expect_tx(qfull, (uint32_t)nr * kPageKeyBytes * (p.two_terms ? 2u : 1u));
                    for (int i = 0; i < nr; ++i) {
                        tma_load_2d(q_hi + i * kPageKeyBytes, &q_map, qfull, 0, (r0 + i) * kHeads);
                        if (p.two_terms)
                            tma_load_2d(q_lo + i * kPageKeyBytes, &q_map, qfull, 0,
                                        (p.R + r0 + i) * kHeads);
                    }
                    cur_g = g;
                    ++qi;
                }
                const int s = li % kStages;
                if (!bounded_wait(&empty[s], ((li / kStages) & 1) ^ 1, abort_flag)) break;
                const int t = it - plan->g_item[g];
                const int req = plan->g_req[g];
                const int npages = (plan->g_len[g] + kPage - 1) / kPage;
                int ids[2];
                uint32_t bytes = 0;
                for (int hh = 0; hh < 2; ++hh) {
                    const int pidx = 2 * t + hh;
                    ids[hh] = -1;
                    if (pidx < npages) {
                        const int id = p.block_table[(int64_t)req * p.max_pages + pidx];
                        if (id < 0 || (int64_t)id >= p.pool_pages) {
                            record_status(p.status, kStatusBounds);
                        } else {
                            ids[hh] = id;
                            bytes += kPageKeyBytes + kPageScaleBytes;
                        }
                    }
                }
                mbar_arrive_expect_tx(&full[s], bytes);
                for (int hh = 0; hh < 2; ++hh) {
                    if (ids[hh] < 0) continue;
                    tma_load_2d(stages + s * kStageBytes + hh * kPageKeyBytes, &keys_map, &full[s], 0,
                                ids[hh] * kPage);
                    bulk_load(scales + s * kTileKeys + hh * kPage, p.k_scale + (int64_t)ids[hh] * kPage,
                              kPageScaleBytes, &full[s]);
                }
            }
            if (*abort_flag) {
                // Let every copy this thread started land before the CTA exits.
                int dummy = 0;
                const int first = li > kStages ? li - kStages : 0;
                for (int j = first; j < li; ++j)
                    bounded_wait(&full[j % kStages], (j / kStages) & 1, &dummy);
                if (qi > 0) bounded_wait(qfull, (qi - 1) & 1, &dummy);
            }
        }
    } else if (warp == 1) {
        // -------------------------------------------------------- MMA issuer
        if (lane == 0) {
            int g = find_group(plan, it0), cur_g = -1, qi = 0, li = 0;
            uint32_t idesc = 0;
            const uint32_t a0 = smem_u32(stages), bh = smem_u32(q_hi), bl = smem_u32(q_lo);
            for (int it = it0; it < it1; ++it, ++li) {
                while (g + 1 < n_groups && it >= plan->g_item[g + 1]) ++g;
                if (g != cur_g) {
                    if (cur_g >= 0) mma_commit(qempty);
                    if (!bounded_wait(qfull, qi & 1, abort_flag)) break;
                    tc_fence_after_sync();
                    idesc = idesc_e4m3_f32(128, (uint32_t)plan->g_nr[g] * kHeads);
                    cur_g = g;
                    ++qi;
                }
                const int s = li % kStages, acc = li & 1;
                if (!bounded_wait(&tempty[acc], ((li >> 1) & 1) ^ 1, abort_flag)) break;
                tc_fence_after_sync();
                if (!bounded_wait(&full[s], (li / kStages) & 1, abort_flag)) break;
                tc_fence_after_sync();
                const uint32_t d = tmem_base + (uint32_t)acc * kAccCols;
                const uint32_t a = a0 + (uint32_t)s * kStageBytes;
#pragma unroll
                for (int kk = 0; kk < kDim / 32; ++kk)
                    mma_f8f6f4(d, desc_kmajor_sw128(a + kk * 32), desc_kmajor_sw128(bh + kk * 32), idesc,
                               kk > 0 ? 1u : 0u);
                if (p.two_terms) {
#pragma unroll
                    for (int kk = 0; kk < kDim / 32; ++kk)
                        mma_f8f6f4(d, desc_kmajor_sw128(a + kk * 32), desc_kmajor_sw128(bl + kk * 32),
                                   idesc, 1u);
                }
                mma_commit(&empty[s]);
                mma_commit(&tfull[acc]);
            }
            // Every MMA issued here must finish before TMEM is released.
            int dummy = 0;
            mma_commit(drain);
            bounded_wait(drain, 0, &dummy);
        }
    } else {
        // ---------------------------------------------------------- epilogue
        const int e = warp - 2;            // 0..7
        const int quad = warp & 3;         // TMEM lanes this warp may read
        const int half = e >> 2;           // rows half, half + 2
        const int key = quad * 32 + lane;  // key of the tile this thread owns
        float* wq_w = wq_s + e * kWqPerWarp;
        int g = find_group(plan, it0), cur_g = -1, li = 0;
        int r0 = 0, nr = 0;
        int rlen[2] = {0, 0};
        for (int it = it0; it < it1; ++it, ++li) {
            while (g + 1 < n_groups && it >= plan->g_item[g + 1]) ++g;
            if (g != cur_g) {
                // Each warp keeps its own copy of its rows' head weights, so no
                // barrier across warps is needed here.
                __syncwarp();
                r0 = plan->g_r0[g];
                nr = plan->g_nr[g];
                for (int j = 0; j < 2; ++j) {
                    const int rr = half + 2 * j;
                    rlen[j] = rr < nr ? plan->row_len[r0 + rr] : 0;
                    if (rr < nr) {
                        wq_w[j * kHeads + lane] = p.wq[(int64_t)(r0 + rr) * kHeads + lane];
                        wq_w[j * kHeads + 32 + lane] = p.wq[(int64_t)(r0 + rr) * kHeads + 32 + lane];
                    }
                }
                __syncwarp();
                cur_g = g;
            }
            const int s = li % kStages, acc = li & 1;
            if (!bounded_wait(&tfull[acc], (li >> 1) & 1, abort_flag)) break;
            tc_fence_after_sync();
            // The stage cannot be refilled before this warp releases it, so its
            // `full` phase is still the current one: observe it, then read the
            // scales the bulk copy wrote.
            if (!bounded_wait(&full[s], (li / kStages) & 1, abort_flag)) break;
            const float sc = scales[s * kTileKeys + key];
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
            const int64_t pos = (int64_t)(it - plan->g_item[g]) * kTileKeys + key;
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int rr = half + 2 * j;
                if (rr >= nr) break;  // warp-uniform
                const uint32_t taddr = tmem_base + ((uint32_t)(quad * 32) << 16) +
                                       (uint32_t)acc * kAccCols + (uint32_t)rr * kHeads;
                const float* w = wq_w + j * kHeads;
                float v[32];
                float sum = 0.0f;
                tmem_load_32cols(taddr, v);
#pragma unroll
                for (int h = 0; h < 32; ++h) sum = fmaf(w[h], fmaxf(v[h], 0.0f), sum);
                tmem_load_32cols(taddr + 32, v);
#pragma unroll
                for (int h = 0; h < 32; ++h) sum = fmaf(w[32 + h], fmaxf(v[h], 0.0f), sum);
                const float out = __fadd_rn(sum * sc, 0.0f);  // -0 -> +0
                if (pos < rlen[j]) p.scores[(int64_t)(r0 + rr) * p.score_stride + pos] = out;
            }
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[acc]);
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    if (threadIdx.x == 0 && *abort_flag) record_status(p.status, kStatusTimeout);
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

}  // namespace

cudaError_t launch_score(const ScoreArgs& a, const CUtensorMap& keys_map, const CUtensorMap& q_map) {
    static int configured_device = -1;
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (configured_device != dev) {
        err = cudaFuncSetAttribute(k_score, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
        if (err != cudaSuccess) return err;
        configured_device = dev;
    }
    ScoreParams p;
    p.plan = reinterpret_cast<const Plan*>(a.ws + a.L.plan);
    p.wq = reinterpret_cast<const float*>(a.ws + a.L.wq);
    p.k_scale = a.k_scale;
    p.block_table = a.block_table;
    p.pool_pages = a.pool_pages;
    p.max_pages = a.max_pages;
    p.R = a.R;
    p.two_terms = a.qtype == IDX_Q_BF16 ? 1 : 0;
    p.scores = a.scores;
    p.score_stride = a.score_stride;
    p.status = reinterpret_cast<uint32_t*>(a.ws + a.L.status);
    k_score<<<a.num_sms, kScoreThreads, kSmemBytes, a.stream>>>(keys_map, q_map, p);
    return cudaGetLastError();
}

}  // namespace idx
