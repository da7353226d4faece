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
//   warps 2-17 epilogue, one (row, TMEM lane quadrant) per warp: tcgen05.ld
//              the row's 64 head columns (two halves), ReLU, head-weighted sum
//              (packed f32x2 FMAs), times the key scale, masked coalesced f32
//              stores; then the accumulator goes back to the MMA issuer.
//
// The launch is a programmatic dependent of the prep kernel: barrier set-up,
// TMEM allocation and descriptor prefetch overlap the prep kernel's tail, and
// nothing it wrote is read before griddepcontrol.wait.
#include "idx_internal.h"
#include "ptx.cuh"

namespace idx {

namespace {

constexpr int kStages = 8;
constexpr int kEpiWarps = 16;                              // 4 rows x 4 TMEM lane quadrants
constexpr int kScoreThreads = 64 + kEpiWarps * 32;         // 576
constexpr uint32_t kQRows = kGroupRows * kHeads;           // 256
constexpr uint32_t kQPartBytes = kQRows * kDim;            // 32 KB
constexpr uint32_t kPageKeyBytes = kPage * kDim;           // 8 KB
constexpr uint32_t kPageScaleBytes = kPage * 4;            // 256 B
constexpr uint32_t kStageBytes = kTileKeys * kDim;         // 16 KB
constexpr uint32_t kStageScaleBytes = kTileKeys * 4;       // 512 B
constexpr uint32_t kAccCols = 256;
constexpr uint32_t kTmemCols = 2 * kAccCols;
constexpr int kPlanCacheGroups = 256;                      // plan entries kept in shared memory
constexpr int kPlanCacheRows = kMaxRows;

constexpr uint32_t kOffQHi = 0;
constexpr uint32_t kOffQLo = kOffQHi + kQPartBytes;
constexpr uint32_t kOffStages = kOffQLo + kQPartBytes;
constexpr uint32_t kOffScales = kOffStages + kStages * kStageBytes;
constexpr uint32_t kOffWq = kOffScales + kStages * kStageScaleBytes;
constexpr uint32_t kOffPlan = kOffWq + kEpiWarps * kHeads * 4;
constexpr uint32_t kPlanInts = 5 * kPlanCacheGroups + 1 + kPlanCacheRows;
constexpr uint32_t kOffBars = kOffPlan + kPlanInts * 4 + 4;
constexpr uint32_t kNumBars = 2 * kStages + 4 + 3;
constexpr uint32_t kOffMisc = kOffBars + kNumBars * 8;
constexpr uint32_t kSmemUsed = kOffMisc + 16;
constexpr uint32_t kSmemBytes = kSmemUsed + 1024;  // slack for 1024-byte alignment
static_assert(kSmemBytes <= 232448, "shared memory budget");
static_assert(kOffStages % 1024 == 0 && kOffQLo % 1024 == 0, "swizzle atoms need 1024-byte alignment");
static_assert(kOffBars % 8 == 0, "mbarrier alignment");

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

// The plan, read from shared memory when it fits there, else from global.
struct PlanView {
    const int* item;  // [n_groups + 1]
    const int* req;
    const int* r0;
    const int* nr;
    const int* len;
    const int* row_len;
    int n_groups;
    // The group that holds work item `it`: the last g with item[g] <= it.
    __device__ __forceinline__ int find(int it) const {
        int lo = 0, hi = n_groups;
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (item[mid] <= it) lo = mid; else hi = mid;
        }
        return lo;
    }
};

__device__ __forceinline__ uint64_t pack2(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ float2 unpack2(uint64_t v) {
    float lo, hi;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
    return make_float2(lo, hi);
}
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

__global__ void __launch_bounds__(kScoreThreads, 1)
k_score(const __grid_constant__ CUtensorMap keys_map, const __grid_constant__ CUtensorMap q_map,
        const ScoreParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* q_hi = smem + kOffQHi;
    uint8_t* q_lo = smem + kOffQLo;
    uint8_t* stages = smem + kOffStages;
    float* scales = reinterpret_cast<float*>(smem + kOffScales);
    float* wq_s = reinterpret_cast<float*>(smem + kOffWq);
    int* plan_s = reinterpret_cast<int*>(smem + kOffPlan);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBars);
    uint64_t* full = bars;                    // [kStages] keys + scales landed
    uint64_t* empty = bars + kStages;         // [kStages] MMAs done (seen by the epilogue), scales read
    uint64_t* tfull = bars + 2 * kStages;     // [2] accumulator ready
    uint64_t* tempty = tfull + 2;             // [2] accumulator drained
    uint64_t* qfull = tempty + 2;             // group query landed
    uint64_t* qempty = qfull + 1;             // MMAs on the group query done
    uint64_t* drain = qempty + 1;             // final MMA completion
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // ---- set-up that needs nothing from the prep kernel --------------------
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kEpiWarps);  // every epilogue warp, after its MMA-done wait
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
    pdl_wait();               // the prep kernel's plan and query are complete and visible
    pdl_launch_dependents();  // the selection may be scheduled as SMs free up

    // ---- the plan: one coalesced copy into shared memory ------------------
    const Plan* plan = p.plan;
    const int n_items = plan->n_items;
    const int n_groups = plan->n_groups;
    PlanView pv;
    pv.n_groups = n_groups;
    if (n_groups <= kPlanCacheGroups) {
        int* it_s = plan_s;
        int* rq_s = it_s + kPlanCacheGroups + 1;
        int* r0_s = rq_s + kPlanCacheGroups;
        int* nr_s = r0_s + kPlanCacheGroups;
        int* ln_s = nr_s + kPlanCacheGroups;
        for (int i = threadIdx.x; i <= n_groups; i += kScoreThreads) {
            it_s[i] = plan->g_item[i];
            if (i < n_groups) {
                rq_s[i] = plan->g_req[i];
                r0_s[i] = plan->g_r0[i];
                nr_s[i] = plan->g_nr[i];
                ln_s[i] = plan->g_len[i];
            }
        }
        pv.item = it_s;
        pv.req = rq_s;
        pv.r0 = r0_s;
        pv.nr = nr_s;
        pv.len = ln_s;
    } else {
        pv.item = plan->g_item;
        pv.req = plan->g_req;
        pv.r0 = plan->g_r0;
        pv.nr = plan->g_nr;
        pv.len = plan->g_len;
    }
    {
        int* rl_s = plan_s + 5 * kPlanCacheGroups + 1;
        for (int i = threadIdx.x; i < p.R && i < kPlanCacheRows; i += kScoreThreads) rl_s[i] = plan->row_len[i];
        pv.row_len = p.R <= kPlanCacheRows ? rl_s : plan->row_len;
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;
    const int it0 = (int)(((int64_t)blockIdx.x * n_items) / gridDim.x);
    const int it1 = (int)(((int64_t)(blockIdx.x + 1) * n_items) / gridDim.x);
    const bool has_work = it0 < it1 && n_groups >= 1;

    if (!has_work) {
        // nothing to do; fall through to the common teardown
    } else if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        // The whole warp fetches block-table entries, one page per lane and
        // up to 16 tiles at a time, so the page ids of a batch arrive in one
        // round trip; lane 0 waits on the ring and issues the copies.
        int g = pv.find(it0), cur_g = -1, qi = 0, issued = 0;
        int req = 0, npages = 0, gbeg = 0, gend = 0;
        bool stop = false;
        int it = it0;
        while (it < it1 && !stop) {
            while (g + 1 < n_groups && it >= pv.item[g + 1]) ++g;
            if (g != cur_g) {
                req = pv.req[g];
                npages = (pv.len[g] + kPage - 1) / kPage;
                gbeg = pv.item[g];
                gend = pv.item[g + 1];
                if (lane == 0) {
                    if (!bounded_wait(qempty, (qi & 1) ^ 1, abort_flag)) {
                        stop = true;
                    } else {
                        const int r0 = pv.r0[g], nr = pv.nr[g];
                        mbar_arrive_expect_tx(qfull, (uint32_t)nr * kPageKeyBytes * (p.two_terms ? 2u : 1u));
                        for (int i = 0; i < nr; ++i) {
                            tma_load_2d(q_hi + i * kPageKeyBytes, &q_map, qfull, 0, (r0 + i) * kHeads);
                            if (p.two_terms)
                                tma_load_2d(q_lo + i * kPageKeyBytes, &q_map, qfull, 0,
                                            (p.R + r0 + i) * kHeads);
                        }
                        ++qi;
                    }
                }
                stop = __shfl_sync(0xFFFFFFFFu, stop ? 1 : 0, 0) != 0;
                cur_g = g;
                if (stop) break;
            }
            const int nb = min(16, min(it1, gend) - it);
            const int t0 = it - gbeg;
            int id = -1;
            if (lane < 2 * nb) {
                const int pidx = 2 * t0 + lane;
                if (pidx < npages) {
                    const int v = p.block_table[(int64_t)req * p.max_pages + pidx];
                    if (v < 0 || (int64_t)v >= p.pool_pages) record_status(p.status, kStatusBounds);
                    else id = v;
                }
            }
            for (int b = 0; b < nb; ++b) {
                const int id0 = __shfl_sync(0xFFFFFFFFu, id, 2 * b);
                const int id1 = __shfl_sync(0xFFFFFFFFu, id, 2 * b + 1);
                if (lane == 0) {
                    const int s = issued % kStages;
                    if (!bounded_wait(&empty[s], ((issued / kStages) & 1) ^ 1, abort_flag)) {
                        stop = true;
                    } else {
                        const uint32_t bytes = (id0 >= 0 ? kPageKeyBytes + kPageScaleBytes : 0u) +
                                               (id1 >= 0 ? kPageKeyBytes + kPageScaleBytes : 0u);
                        mbar_arrive_expect_tx(&full[s], bytes);
                        if (id0 >= 0) {
                            tma_load_2d(stages + s * kStageBytes, &keys_map, &full[s], 0, id0 * kPage);
                            bulk_load(scales + s * kTileKeys, p.k_scale + (int64_t)id0 * kPage,
                                      kPageScaleBytes, &full[s]);
                        }
                        if (id1 >= 0) {
                            tma_load_2d(stages + s * kStageBytes + kPageKeyBytes, &keys_map, &full[s], 0,
                                        id1 * kPage);
                            bulk_load(scales + s * kTileKeys + kPage, p.k_scale + (int64_t)id1 * kPage,
                                      kPageScaleBytes, &full[s]);
                        }
                        ++issued;
                    }
                }
                stop = __shfl_sync(0xFFFFFFFFu, stop ? 1 : 0, 0) != 0;
                if (stop) break;
            }
            it += nb;
        }
        if (lane == 0 && *abort_flag) {
            // Let every copy this thread started land before the CTA exits.
            int dummy = 0;
            const int first = issued > kStages ? issued - kStages : 0;
            for (int j = first; j < issued; ++j) bounded_wait(&full[j % kStages], (j / kStages) & 1, &dummy);
            if (qi > 0) bounded_wait(qfull, (qi - 1) & 1, &dummy);
        }
    } else if (warp == 1) {
        // -------------------------------------------------------- MMA issuer
        if (lane == 0) {
            const uint32_t a0 = smem_u32(stages), bh = smem_u32(q_hi), bl = smem_u32(q_lo);
            const int nmma = p.two_terms ? 8 : 4;
            int g = pv.find(it0), qi = 0;
            int gend = pv.item[g + 1];  // first work item past the current group
            uint32_t idesc = 0;
            bool ok = true;
            for (int it = it0, li = 0; it < it1; ++it, ++li) {
                if (it == it0 || it >= gend) {
                    if (it != it0) {
                        mma_commit(qempty);  // the previous group's query may be replaced
                        while (g + 1 < n_groups && it >= pv.item[g + 1]) ++g;
                        gend = pv.item[g + 1];
                    }
                    if (!bounded_wait(qfull, qi & 1, abort_flag)) { ok = false; break; }
                    tc_fence_after_sync();
                    idesc = idesc_e4m3_f32(128, (uint32_t)pv.nr[g] * kHeads);
                    ++qi;
                }
                if (!bounded_wait(&tempty[li & 1], ((li >> 1) & 1) ^ 1, abort_flag)) { ok = false; break; }
                tc_fence_after_sync();
                if (!bounded_wait(&full[li % kStages], (li / kStages) & 1, abort_flag)) { ok = false; break; }
                const uint32_t d = tmem_base + (uint32_t)(li & 1) * kAccCols;
                const uint32_t a = a0 + (uint32_t)(li % kStages) * kStageBytes;
                for (int k = 0; k < nmma; ++k) {  // K slice k % 4 of the hi (k < 4) or lo term
                    const uint32_t kk = (uint32_t)(k & 3) * 32;
                    mma_f8f6f4(d, desc_kmajor_sw128(a + kk), desc_kmajor_sw128((k < 4 ? bh : bl) + kk), idesc,
                               k > 0 ? 1u : 0u);
                }
                mma_commit(&tfull[li & 1]);
            }
            (void)ok;
            // Every MMA issued here must finish before TMEM is released.
            int dummy = 0;
            mma_commit(drain);
            bounded_wait(drain, 0, &dummy);
        }
    } else {
        // ---------------------------------------------------------- epilogue
        const int e = warp - 2;            // 0..15
        const int quad = warp & 3;         // TMEM lanes this warp may read
        const int rr = e >> 2;             // the group row this warp reduces
        const int key = quad * 32 + lane;  // key of the tile this thread owns
        float* w = wq_s + e * kHeads;      // this warp's copy of its row's head weights
        int g = pv.find(it0), li = 0;
        int gend = -1, gbeg = 0, r0 = 0, nr = 0, rlen = 0;
        for (int it = it0; it < it1; ++it, ++li) {
            if (it >= gend) {
                while (g + 1 < n_groups && it >= pv.item[g + 1]) ++g;
                gbeg = pv.item[g];
                gend = pv.item[g + 1];
                __syncwarp();
                r0 = pv.r0[g];
                nr = pv.nr[g];
                rlen = rr < nr ? pv.row_len[r0 + rr] : 0;
                if (rr < nr) {
                    w[lane] = p.wq[(int64_t)(r0 + rr) * kHeads + lane];
                    w[32 + lane] = p.wq[(int64_t)(r0 + rr) * kHeads + 32 + lane];
                }
                __syncwarp();
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
            if (rr < nr) {  // warp-uniform
                const int64_t pos = (int64_t)(it - gbeg) * kTileKeys + key;
                const uint32_t taddr = tmem_base + ((uint32_t)(quad * 32) << 16) +
                                       (uint32_t)acc * kAccCols + (uint32_t)rr * kHeads;
                uint64_t a[4] = {0ull, 0ull, 0ull, 0ull};  // four packed (2 x f32) partial sums
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    float v[32];
                    tmem_load_32cols(taddr + 32 * hf, v);
#pragma unroll
                    for (int h = 0; h < 32; h += 8) {
                        const float4 w0 = *reinterpret_cast<const float4*>(w + 32 * hf + h);
                        const float4 w1 = *reinterpret_cast<const float4*>(w + 32 * hf + h + 4);
                        a[0] = ffma2(pack2(w0.x, w0.y), pack2(fmaxf(v[h + 0], 0.0f), fmaxf(v[h + 1], 0.0f)), a[0]);
                        a[1] = ffma2(pack2(w0.z, w0.w), pack2(fmaxf(v[h + 2], 0.0f), fmaxf(v[h + 3], 0.0f)), a[1]);
                        a[2] = ffma2(pack2(w1.x, w1.y), pack2(fmaxf(v[h + 4], 0.0f), fmaxf(v[h + 5], 0.0f)), a[2]);
                        a[3] = ffma2(pack2(w1.z, w1.w), pack2(fmaxf(v[h + 6], 0.0f), fmaxf(v[h + 7], 0.0f)), a[3]);
                    }
                }
                const float2 s0 = unpack2(a[0]), s1 = unpack2(a[1]), s2 = unpack2(a[2]), s3 = unpack2(a[3]);
                const float sum = ((s0.x + s0.y) + (s1.x + s1.y)) + ((s2.x + s2.y) + (s3.x + s3.y));
                const float out = __fadd_rn(sum * sc, 0.0f);  // -0 -> +0
                if (pos < rlen) p.scores[(int64_t)(r0 + rr) * p.score_stride + pos] = out;
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
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)a.num_sms, 1, 1);
    cfg.blockDim = dim3(kScoreThreads, 1, 1);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = a.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k_score, keys_map, q_map, p);
}

}  // namespace idx
