// score.cu -- paged key scoring on the 5th-generation tensor cores.
//
// For every group of (at most four consecutive) rows of one request and every
// 128-key tile of that request's keys:
//
//     D[key, (row, head)] = sum_d K[key, d] * Q'[(row, head), d]     (tcgen05)
//     s[row, key] = scale[key] * sum_h w'[row, h] * max(D[key, (row, h)], 0)
//
// which is the indexer score sum_h w * ReLU(q . (k * scale)) once the key's
// scale (>= 0) and the query's power-of-two factor are taken out of the ReLU.
// Every key of a request is read from HBM once per group, as "sgl-amd-mono-
// upstream PR 18" (GLM-5.3 indexer launch), section "Modifications / 2. A
// request's rows scored together" asks; its LDS batches of whole pages become
// TMA loads of whole 64-token pages into a ring of shared-memory stages.
//
// The query on FP8 tensor cores.  A bf16 query element has 8 significant bits
// and E4M3 only 4, so each (row, head) vector is scaled by a power of two 2^e
// that brings its largest element into [128, 256) and split exactly into two
// E4M3 terms: x * 2^e = hi + lo, hi = RN_e4m3(x * 2^e), lo = x * 2^e - hi.
// For every element whose scaled magnitude is at least 2^-2, lo is a multiple
// of the element's bf16 ulp no larger than 8 ulps, so it is an E4M3 value and
// the split is exact; smaller elements lose at most 2^-10 (scaled) to E4M3's
// subnormal grid -- below 8e-6 of the head's largest element.  The two terms
// accumulate into one TMEM accumulator, and 2^-e > 0 commutes with the ReLU,
// so it is folded into the head weight: w'[r,h] = w[r,h] * 2^-e[r,h].  An
// E4M3 query is used as is (hi = q, no lo term, w' = w).
//
// Keys sit on the MMA's M dimension (128 lanes of TMEM = 128 keys) and the
// group's (row, head) pairs on N (<= 256 columns), so the epilogue reads one
// key per thread and reduces over heads inside the thread: no cross-lane sums,
// and each warp stores 32 consecutive scores of a row.
//
// Two launches per call:
//   k_qprep    (small) splits every row's query once into the two E4M3 terms,
//              laid out as the shared-memory operand (swizzled), and w', in
//              the workspace; with new keys it first stores them.
//   k_score    one CTA per SM, persistent over a contiguous range of tiles:
//   all        build the plan in shared memory: consecutive rows of one
//              request form groups of at most four rows, each group's keys
//              are cut into 128-key tiles numbered as work items.
//   warp 0     TMA producer: the whole warp fetches block-table entries (one
//              page per lane), lane 0 issues per tile two key pages (TMA,
//              128-byte swizzle) + their scales (bulk copy) into stage s of a
//              7-stage ring.
//   warp 1     TMEM allocator and MMA issuer: at each group one bulk copy of
//              the group's prepared operand and w' into shared memory, then
//              4 (E4M3 query) or 8 (bf16 query, hi and lo terms)
//              kind::f8f6f4 MMAs of K = 32 per tile into one of two TMEM
//              accumulators.
//   warps 2-17 epilogue, per tile one (row, TMEM lane quadrant) per warp:
//              tcgen05.ld the row's 64 head columns, ReLU, head-weighted sum
//              (packed f32x2 FMAs), times the key scale, masked coalesced f32
//              stores.  Without a prepared operand (the no-allocation entry
//              point has no room for one) these warps split the group's query
//              themselves at each group.
//
// Launch chaining: k_qprep waits for the kernel before it (griddepcontrol.wait)
// and then lets k_score launch as its programmatic dependent, so every input
// written before the call is complete when k_score starts: it builds its plan
// and starts its key loads at once, and its MMA warp waits for k_qprep's grid
// before copying an operand.  Without a prepared operand k_score itself waits
// for the kernel before it before touching global memory.  Each CTA lets the
// next launch (the selection) start once its scores are written.  Launches
// of many tiles per CTA use a second instantiation whose epilogue keeps half
// of its row's head weights in registers (kRegW below).
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "idx_internal.h"
#include "ptx.cuh"
#include "quant.cuh"

namespace idx {

namespace {

constexpr int kStages = 7;
constexpr int kEpiWarps = 16;                              // 4 rows x 4 TMEM lane quadrants
constexpr int kScoreThreads = 64 + kEpiWarps * 32;         // 576
constexpr uint32_t kQRows = kGroupRows * kHeads;           // 256
constexpr uint32_t kQPartBytes = kQRows * kDim;            // 32 KB
constexpr uint32_t kQRowBytes = kHeads * kDim;             // 8 KB: one row's operand term
constexpr uint32_t kPageKeyBytes = kPage * kDim;           // 8 KB
constexpr uint32_t kPageScaleBytes = kPage * 4;            // 256 B
constexpr uint32_t kStageBytes = kTileKeys * kDim;         // 16 KB
constexpr uint32_t kStageScaleBytes = kTileKeys * 4;       // 512 B
constexpr uint32_t kAccCols = 256;
constexpr int kRegWTilesPerCta = 12;  // launches of at least this many tiles per CTA keep weights in registers
constexpr uint32_t kTmemCols = 2 * kAccCols;

constexpr uint32_t kOffQHi = 0;
constexpr uint32_t kOffQLo = kOffQHi + kQPartBytes;
constexpr uint32_t kOffStages = kOffQLo + kQPartBytes;
constexpr uint32_t kOffScales = kOffStages + kStages * kStageBytes;
constexpr uint32_t kOffWq = kOffScales + kStages * kStageScaleBytes;   // [2][256] f32, by group parity
constexpr uint32_t kOffPlan = kOffWq + 2 * kQRows * 4;
// plan: item[kMaxRows+1], req, r0, nr, len [kMaxRows] each, row_len[kMaxRows], gid[kMaxRows]
constexpr uint32_t kPlanInts = (kMaxRows + 1) + 4 * kMaxRows + 2 * kMaxRows;
constexpr uint32_t kOffBars = ((kOffPlan + kPlanInts * 4) + 7) & ~7u;
constexpr uint32_t kNumBars = 2 * kStages + 4 + 4;
constexpr uint32_t kOffMisc = kOffBars + kNumBars * 8;
constexpr uint32_t kSmemUsed = kOffMisc + 16;
constexpr uint32_t kSmemBytes = kSmemUsed + 1024;  // slack for 1024-byte alignment
static_assert(kSmemBytes <= 232448, "shared memory budget");
static_assert(kOffStages % 1024 == 0 && kOffQLo % 1024 == 0, "swizzle atoms need 1024-byte alignment");

struct ScoreParams {
    int qtype;
    const void* q;
    const float* head_w;
    const int32_t* seq_lens;
    const int32_t* row_req;
    int R;
    int64_t len_cap;  // rows are cut to this many keys (block table and score buffer)
    const float* k_scale;
    const int32_t* block_table;
    int64_t pool_pages;
    int max_pages;
    float* scores;
    int64_t score_stride;
    uint32_t* status;
    uint8_t* qop;            // the rows' prepared operands (k_qprep), or null: split in the kernel
    const uint8_t* new_k;    // with qop: k_qprep stores each row's new key and scale in its slot
    const float* new_scale;
    uint8_t* k_cache_w;      // the cache, written by that store
    float* k_scale_w;
    int inputs_ready;        // k_qprep lets the scoring launch before its own grid wait
    int table_prefetch;      // k_qprep prefetches long rows' block-table entries into L2
    uint64_t wait_ns;        // wall-time limit of every role's waits (kWaitTimeoutNs in normal use)
    int drop_query_handoff;  // test only: the epilogue never signals the query operand
};

struct PlanSmem {
    int* item;     // [n_groups + 1] first work item of each group
    int* req;      // request of each group
    int* r0;       // first row of each group
    int* nr;       // rows in each group
    int* len;      // longest row of each group
    int* row_len;  // [R] clamped row lengths
    int* gid;      // [R] group of each row (scratch)
};

__device__ __forceinline__ int find_group(const PlanSmem& pl, int n_groups, int it) {
    int lo = 0, hi = n_groups;  // item[lo] <= it < item[hi]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (pl.item[mid] <= it) lo = mid; else hi = mid;
    }
    return lo;
}

// Warp 0: group rows r and r-1 when they have the same request, at most
// kGroupRows rows a group; tiles of each group numbered in one sequence.
__device__ void build_plan(const ScoreParams& p, const PlanSmem& pl, int* n_groups_out, int* n_items_out) {
    const int lane = threadIdx.x & 31;
    const unsigned full = 0xFFFFFFFFu;
    const int R = p.R;
    int carry_seg = 0, carry_req = -1, n_groups = 0;
    bool bad = false;
    for (int base = 0; base < R; base += 32) {
        const int r = base + lane;
        const bool valid = r < R;
        const int req = valid ? __ldcg(p.row_req + r) : -1;  // through L2 (read before the grid wait)
        int len = valid ? __ldcg(p.seq_lens + r) : 0;
        if (valid) {
            if (len < 0 || (int64_t)len > p.len_cap || req < 0) bad = true;
            len = len < 0 ? 0 : ((int64_t)len > p.len_cap ? (int)p.len_cap : len);
            if (req < 0) len = 0;
            pl.row_len[r] = len;
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
        if (valid) pl.gid[r] = gid;
        if (gstart) {
            pl.req[gid] = req;
            pl.r0[gid] = r;
        }
        n_groups += __popc(gs);
        carry_seg = __shfl_sync(full, seg, 31);
        carry_req = __shfl_sync(full, req, 31);
    }
    __syncwarp();
    if (blockIdx.x == 0 && __any_sync(full, bad) && lane == 0) record_status(p.status, kStatusBounds);
    int item = 0;
    for (int base = 0; base < n_groups; base += 32) {
        const int g = base + lane;
        int ntiles = 0;
        if (g < n_groups) {
            const int r0 = pl.r0[g];
            int nr = 0, glen = 0;
            for (int i = 0; i < kGroupRows && r0 + i < R; ++i) {
                if (pl.gid[r0 + i] != g) break;
                ++nr;
                glen = max(glen, pl.row_len[r0 + i]);
            }
            pl.nr[g] = nr;
            pl.len[g] = glen;
            ntiles = (glen + kTileKeys - 1) / kTileKeys;
        }
        int incl = ntiles;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(full, incl, o);
            if (lane >= o) incl += v;
        }
        if (g < n_groups) pl.item[g] = item + incl - ntiles;
        item += __shfl_sync(full, incl, 31);
    }
    if (lane == 0) {
        pl.item[n_groups] = item;
        *n_groups_out = n_groups;
        *n_items_out = item;
    }
}

__device__ __forceinline__ uint16_t to_e4m3_pair(float a, float b) {
    return static_cast<uint16_t>(__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3));
}

// 2 ReLU(x) = x + |x|: one add (the absolute value is an operand modifier)
// on the FMA pipe instead of a max on the half-rate ALU pipe; exact, and a NaN
// passes through as it does in the definition's ReLU.
__device__ __forceinline__ float relu2(float x) { return __fadd_rn(x, fabsf(x)); }

// x rounded to the nearest E4M3 value, ties to even, as an f32, for |x| < 448
// (the value whose code cvt.rn.satfinite.e4m3x2.f32 gives): in E4M3's
// normal range (|x| >= 2^-6) the f32 mantissa is rounded to 3 bits in the
// integer unit; below it to a multiple of 2^-9 (E4M3's subnormal spacing) by
// adding and subtracting 1.5 * 2^14.
__device__ __forceinline__ float round_e4m3(float x) {
    const uint32_t u = __float_as_uint(x);
    const uint32_t rn = (u + 0x7FFFFu + ((u >> 20) & 1u)) & 0xFFF00000u;
    const float sub = __fsub_rn(__fadd_rn(x, 24576.0f), 24576.0f);
    return fabsf(x) >= 0.015625f ? __uint_as_float(rn) : sub;
}

__device__ __forceinline__ float pow2f(int e) {  // e in [-126, 127]: exact 2^e
    return __int_as_float((e + 127) << 23);
}

// Byte offset of 4-byte group `lane` of B-operand row n in the K-major
// 128-byte-swizzle layout (8-row atoms of 1024 bytes, 16-byte chunks XOR row).
__device__ __forceinline__ uint32_t swz_off(int n, int lane) {
    return (uint32_t)((n >> 3) * 1024 + (n & 7) * 128 + ((((lane >> 2) ^ (n & 7)) & 7) << 4) + ((lane & 3) << 2));
}

// One (row, head) vector of a bf16 query split exactly into hi + lo E4M3
// terms after scaling by 2^ex (warp-collective: lane l holds elements 4l ..
// 4l + 3 as two packed bf16 pairs in `raw`).  Returns the lane's four hi and
// four lo codes and 2^-ex, the factor folded into the head weight.
struct PairSplit {
    uint32_t hi, lo;
    float inv_scale;
};
__device__ __forceinline__ PairSplit split_pair(uint2 raw) {
    float x[4];
    x[0] = __uint_as_float(raw.x << 16);
    x[1] = __uint_as_float(raw.x & 0xFFFF0000u);
    x[2] = __uint_as_float(raw.y << 16);
    x[3] = __uint_as_float(raw.y & 0xFFFF0000u);
    // Largest exponent field of the 128 elements (one warp reduction); the
    // largest element lies in [2^(E-127), 2^(E-126)).
    const uint32_t e01 = max((raw.x >> 7) & 0xFFu, (raw.x >> 23) & 0xFFu);
    const uint32_t e23 = max((raw.y >> 7) & 0xFFu, (raw.y >> 23) & 0xFFu);
    const int emax = (int)__reduce_max_sync(0xFFFFFFFFu, max(e01, e23));
    // 2^ex brings the largest element into [128, 256) (<= 448).
    const int ex = max(-126, min(126, 134 - emax));
    const float sc = pow2f(ex);
    float xs[4], lo[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        xs[i] = x[i] * sc;
        lo[i] = __fsub_rn(xs[i], round_e4m3(xs[i]));
    }
    PairSplit r;
    r.hi = (uint32_t)to_e4m3_pair(xs[0], xs[1]) | ((uint32_t)to_e4m3_pair(xs[2], xs[3]) << 16);
    r.lo = (uint32_t)to_e4m3_pair(lo[0], lo[1]) | ((uint32_t)to_e4m3_pair(lo[2], lo[3]) << 16);
    r.inv_scale = pow2f(-ex);
    return r;
}

// The epilogue warps split the query of a group (rows r0 .. r0+nr-1) into
// the hi / lo operand buffers and write w' for each (row, head) (launches
// without a prepared operand: idx_score_noalloc).  Not inlined: it is off the
// usual path, and inlined it would push the tile loop's registers past the
// cap.
__device__ __noinline__ void split_group_query(const ScoreParams& p, int r0, int nr, uint8_t* q_hi, uint8_t* q_lo,
                                  float* wq, int e, int lane) {
    const int pairs = nr * kHeads;
    if (p.qtype != IDX_Q_BF16) {
        // One E4M3 term: the query's codes as given (IDX_Q_E4M3), or quantised
        // here with the scale folded into w' (IDX_Q_BF16_FP8).  A warp's pairs
        // are loaded eight at a time.
        constexpr int kBatch1 = 8;
        const bool quant = p.qtype == IDX_Q_BF16_FP8;
        for (int p0 = e; p0 < pairs; p0 += kEpiWarps * kBatch1) {
            uint2 raw[kBatch1];
            float wv[kBatch1];
#pragma unroll
            for (int b = 0; b < kBatch1; ++b) {
                const int pp = p0 + b * kEpiWarps;
                raw[b] = make_uint2(0, 0);
                wv[b] = 0.0f;
                if (pp < pairs) {
                    const int64_t src = (int64_t)r0 * kHeads + pp;
                    if (quant)
                        raw[b] = reinterpret_cast<const uint2*>(p.q)[src * 32 + lane];
                    else
                        raw[b].x = reinterpret_cast<const uint32_t*>(p.q)[src * 32 + lane];
                    wv[b] = p.head_w[src];
                }
            }
#pragma unroll
            for (int b = 0; b < kBatch1; ++b) {
                const int pp = p0 + b * kEpiWarps;
                if (pp >= pairs) break;  // warp-uniform
                uint32_t codes = raw[b].x;
                float wq_b = wv[b];
                if (quant) {
                    float scale;
                    codes = quantize_head_lane(raw[b], &scale);
                    wq_b = __fmul_rn(wv[b], scale);
                }
                *reinterpret_cast<uint32_t*>(q_hi + swz_off(pp, lane)) = codes;
                if (lane == 0) wq[pp] = wq_b;
            }
        }
        return;
    }
    constexpr int kBatch = 8;  // pairs whose loads are in flight together
    for (int p0 = e; p0 < pairs; p0 += kEpiWarps * kBatch) {
        uint2 raw[kBatch];
        float wv[kBatch];
#pragma unroll
        for (int b = 0; b < kBatch; ++b) {
            const int pp = p0 + b * kEpiWarps;
            raw[b] = make_uint2(0, 0);
            wv[b] = 0.0f;
            if (pp < pairs) {
                const int64_t src = (int64_t)r0 * kHeads + pp;
                raw[b] = reinterpret_cast<const uint2*>(p.q)[src * 32 + lane];
                wv[b] = p.head_w[src];
            }
        }
#pragma unroll
        for (int b = 0; b < kBatch; ++b) {
            const int pp = p0 + b * kEpiWarps;
            if (pp >= pairs) break;  // warp-uniform
            const PairSplit sp = split_pair(raw[b]);
            const uint32_t off = swz_off(pp, lane);
            *reinterpret_cast<uint32_t*>(q_hi + off) = sp.hi;
            *reinterpret_cast<uint32_t*>(q_lo + off) = sp.lo;
            if (lane == 0) wq[pp] = wv[b] * sp.inv_scale;
        }
    }
}

// ---- k_qprep: the query operand of every row, once per call ----------------
//
// Row r's operand in the workspace, in the shared-memory layout the scoring
// copies verbatim (K-major, 128-byte swizzle, 1024-byte atoms of 8 heads):
//   hi [R][8192 B] at qop, lo [R][8192 B] at qop + R * 8192 (bf16 query only),
//   w' [R][64] f32 at qop + 2 * R * 8192.
// A group of rows r0 .. r0 + nr - 1 is then one contiguous run of each.
constexpr int kQprepThreads = 256;
constexpr int kPrefetchMinPages = 256;  // rows of at least 16,384 keys get their block table prefetched
constexpr int kQprepPairsPerWarp = 1;

__global__ void __launch_bounds__(kQprepThreads) k_qprep(const ScoreParams p) {
    // Wait for the kernel before this one, then let the scoring launch (a
    // programmatic dependent) start: every input written before this call is
    // then complete, so the scoring may read the inputs other than this
    // kernel's operands before its own grid wait.  When the caller guarantees
    // that those inputs (block table, lengths, row map, key cache and scales)
    // were complete when the call was enqueued, the scoring may launch at
    // once, so that its set-up, plan and first key pages overlap the kernel
    // before this one; the query and head weights, which that kernel may
    // still be writing, are read here only after the wait, and the scoring
    // writes no score before this grid has completed.
    if (p.inputs_ready) pdl_launch_dependents();
    pdl_wait();
    if (!p.inputs_ready) pdl_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int warp_g = blockIdx.x * (kQprepThreads / 32) + (threadIdx.x >> 5);
    const int pairs = p.R * kHeads;
    // Row warp_g's length and request, for the block-table prefetch below
    // (plain calls only: with inputs complete at enqueue the scoring reads its
    // block table while the kernel before this one still runs).
    const bool pf = warp_g < p.R && p.table_prefetch;
    int pf_len = 0, pf_req = -1;
    if (pf) {
        pf_len = __ldcg(p.seq_lens + warp_g);
        pf_req = __ldcg(p.row_req + warp_g);
    }
    if (p.new_k && warp_g < p.R) {
        // The keys this call writes ("sgl-amd-mono-upstream PR 18", section
        // "Modifications / 2", keys this launch writes): row r's key goes to its
        // own slot, position seq_lens[r] - 1 of its request, so that every row
        // of the request -- in any row group -- scores it.  The scoring's
        // producer waits for this grid before its first page load.
        const int r = warp_g;
        const int len = __ldcg(p.seq_lens + r), req = __ldcg(p.row_req + r);
        if (len >= 1 && (int64_t)len <= p.len_cap && req >= 0) {
            const int pos = len - 1;
            const int v = __ldcg(p.block_table + (int64_t)req * p.max_pages + pos / kPage);
            if (v >= 0 && (int64_t)v < p.pool_pages) {
                reinterpret_cast<uint32_t*>(p.k_cache_w + (int64_t)v * kPageKeyBytes + (pos % kPage) * kDim)[lane] =
                    reinterpret_cast<const uint32_t*>(p.new_k + (int64_t)r * kDim)[lane];
                if (lane == 0) p.k_scale_w[(int64_t)v * kPage + pos % kPage] = p.new_scale[r];
            } else if (lane == 0) {
                record_status(p.status, kStatusBounds);
            }
        }
    }
    uint8_t* hi = p.qop;
    uint8_t* lo = p.qop + (int64_t)p.R * kQRowBytes;
    float* wq = reinterpret_cast<float*>(p.qop + 2 * (int64_t)p.R * kQRowBytes);
    uint2 raw[kQprepPairsPerWarp];
    float wv[kQprepPairsPerWarp];
#pragma unroll
    for (int b = 0; b < kQprepPairsPerWarp; ++b) {
        const int pp = warp_g * kQprepPairsPerWarp + b;
        raw[b] = make_uint2(0u, 0u);
        wv[b] = 0.0f;
        if (pp < pairs) {
            if (p.qtype == IDX_Q_E4M3) raw[b].x = reinterpret_cast<const uint32_t*>(p.q)[(int64_t)pp * 32 + lane];
            else raw[b] = reinterpret_cast<const uint2*>(p.q)[(int64_t)pp * 32 + lane];
            wv[b] = p.head_w[pp];
        }
    }
#pragma unroll
    for (int b = 0; b < kQprepPairsPerWarp; ++b) {
        const int pp = warp_g * kQprepPairsPerWarp + b;
        if (pp >= pairs) break;  // warp-uniform
        const int64_t off = (int64_t)(pp / kHeads) * kQRowBytes + swz_off(pp % kHeads, lane);
        float w_out = wv[b];
        if (p.qtype == IDX_Q_BF16) {
            const PairSplit sp = split_pair(raw[b]);
            *reinterpret_cast<uint32_t*>(hi + off) = sp.hi;
            *reinterpret_cast<uint32_t*>(lo + off) = sp.lo;
            w_out = wv[b] * sp.inv_scale;
        } else if (p.qtype == IDX_Q_BF16_FP8) {
            float scale;
            *reinterpret_cast<uint32_t*>(hi + off) = quantize_head_lane(raw[b], &scale);
            w_out = __fmul_rn(wv[b], scale);
        } else {
            *reinterpret_cast<uint32_t*>(hi + off) = raw[b].x;
        }
        if (lane == 0) wq[pp] = w_out;
    }
    // The block-table entries of every long row into L2, so that the scoring's
    // producers (which read them right after building their plan) find them
    // there: a long row's table is otherwise a DRAM miss by the time the next
    // call reads it.  Short rows' tables are few lines and stay in L2.
    if (pf) {
        const int64_t n = min((int64_t)pf_len, p.len_cap);
        const int npages = (int)((n + kPage - 1) / kPage);
        if (npages >= kPrefetchMinPages && pf_req >= 0) {
            const int32_t* row = p.block_table + (int64_t)pf_req * p.max_pages;
            for (int e = lane * 32; e < npages; e += 1024) prefetch_l2(row + e);
            if (lane == 0) prefetch_l2(row + npages - 1);
        }
    }
}

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

// kRegW: the epilogue keeps the first 32 head weights of its row in registers
// for a group's tiles and reads the TMEM accumulator 16 columns at a time
// (room for them under the register cap of 18 warps); the weights' broadcast
// shared-memory reads otherwise share the shared-memory pipe with the tensor
// core's operand reads in every tile.  It pays when a CTA has many tiles.
template <bool kRegW>
__global__ void __launch_bounds__(kScoreThreads, 1)
k_score(const __grid_constant__ CUtensorMap keys_map, const ScoreParams p) {
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
    uint64_t* qfull = tempty + 2;             // the group's query operand written
    uint64_t* drain = qfull + 1;              // final MMA completion
    uint64_t* qcopy = drain + 1;              // the group's prepared operand copied in
    uint64_t* grp_ready = qcopy + 1;          // every epilogue warp is done with the previous group
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);
    int* counts = reinterpret_cast<int*>(smem + kOffMisc + 8);  // n_groups, n_items

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    PlanSmem pl;
    pl.item = plan_s;
    pl.req = pl.item + kMaxRows + 1;
    pl.r0 = pl.req + kMaxRows;
    pl.nr = pl.r0 + kMaxRows;
    pl.len = pl.nr + kMaxRows;
    pl.row_len = pl.len + kMaxRows;
    pl.gid = pl.row_len + kMaxRows;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kEpiWarps);  // every epilogue warp, after its MMA-done wait
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&tfull[a], 1);
            mbar_init(&tempty[a], kEpiWarps);
        }
        mbar_init(qfull, kEpiWarps);
        mbar_init(drain, 1);
        mbar_init(qcopy, 1);
        mbar_init(grp_ready, kEpiWarps);
        *abort_flag = 0;
        fence_mbar_init();
        prefetch_tensormap(&keys_map);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    // Launched as a programmatic dependent of the kernel before it on the
    // stream.  With a prepared operand that kernel is k_qprep, which lets this
    // grid launch only once every kernel before it has completed (or at once,
    // when the caller guarantees those inputs complete at enqueue): the plan
    // inputs, block table and keys are read at once (through L2), and the
    // MMA warp waits for k_qprep to finish (griddepcontrol.wait) before
    // copying the operand.  Without one, wait for the kernel before before
    // reading an input or writing a score.
    if (!p.qop) pdl_wait();
    if (warp == 0) build_plan(p, pl, &counts[0], &counts[1]);
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;
    const int n_groups = counts[0], n_items = counts[1];
    const int it0 = (int)(((int64_t)blockIdx.x * n_items) / gridDim.x);
    const int it1 = (int)(((int64_t)(blockIdx.x + 1) * n_items) / gridDim.x);
    const bool has_work = it0 < it1 && n_groups >= 1;

    if (!has_work) {
        // nothing to do; fall through to the common teardown
    } else if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        // The whole warp fetches block-table entries, one page per lane and
        // up to 16 tiles at a time, so the page ids of a batch arrive in one
        // round trip; lane 0 waits on the ring and issues the copies.  When
        // k_qprep stores this call's keys, the pages are loaded only after it
        // has completed.
        if (p.new_k) pdl_wait();
        int g = find_group(pl, n_groups, it0), issued = 0;
        bool stop = false;
        int it = it0;
        while (it < it1 && !stop) {
            while (g + 1 < n_groups && it >= pl.item[g + 1]) ++g;
            const int req = pl.req[g];
            const int npages = (pl.len[g] + kPage - 1) / kPage;
            const int nb = min(16, min(it1, pl.item[g + 1]) - it);
            const int t0 = it - pl.item[g];
            int id = -1;
            if (lane < 2 * nb) {
                const int pidx = 2 * t0 + lane;
                if (pidx < npages) {
                    const int v = __ldcg(p.block_table + (int64_t)req * p.max_pages + pidx);
                    if (v < 0 || (int64_t)v >= p.pool_pages) record_status(p.status, kStatusBounds);
                    else id = v;
                }
            }
            for (int b = 0; b < nb; ++b) {
                const int id0 = __shfl_sync(0xFFFFFFFFu, id, 2 * b);
                const int id1 = __shfl_sync(0xFFFFFFFFu, id, 2 * b + 1);
                if (lane == 0) {
                    const int s = issued % kStages;
                    if (!bounded_wait(&empty[s], ((issued / kStages) & 1) ^ 1, abort_flag, p.wait_ns)) {
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
        }
    } else if (warp == 1) {
        // -------------------------------------------------------- MMA issuer
        if (lane == 0) {
            const uint32_t a0 = smem_u32(stages), bh = smem_u32(q_hi), bl = smem_u32(q_lo);
            const int nmma = p.qtype == IDX_Q_BF16 ? 8 : 4;  // hi and lo terms, or one E4M3 term
            int g = find_group(pl, n_groups, it0), qi = 0;
            int gend = -1;  // first work item past the current group
            uint32_t idesc = 0;
            bool copy_pending = false;
            for (int it = it0, li = 0; it < it1; ++it, ++li) {
                if (it >= gend) {
                    while (g + 1 < n_groups && it >= pl.item[g + 1]) ++g;
                    gend = pl.item[g + 1];
                    if (p.qop) {
                        // Copy the group's prepared operand and w' in, once every
                        // epilogue warp is done with the previous group (so its
                        // MMAs have completed and its w' is no longer read).
                        if (qi > 0 && !bounded_wait(grp_ready, (qi - 1) & 1, abort_flag, p.wait_ns)) break;
                        if (qi == 0) pdl_wait();  // k_qprep has written every operand
                        if (!p.drop_query_handoff) {
                            const int r0g = pl.r0[g], nrg = pl.nr[g];
                            const bool two = p.qtype == IDX_Q_BF16;
                            const uint32_t term = (uint32_t)nrg * kQRowBytes;
                            mbar_arrive_expect_tx(qcopy, term * (two ? 2u : 1u) + (uint32_t)nrg * kHeads * 4u);
                            bulk_load(q_hi, p.qop + (int64_t)r0g * kQRowBytes, term, qcopy);
                            if (two) bulk_load(q_lo, p.qop + ((int64_t)p.R + r0g) * kQRowBytes, term, qcopy);
                            bulk_load(wq_s, p.qop + 2 * (int64_t)p.R * kQRowBytes + (int64_t)r0g * kHeads * 4,
                                      (uint32_t)nrg * kHeads * 4u, qcopy);
                            copy_pending = true;
                        }
                        if (!bounded_wait(qcopy, qi & 1, abort_flag, p.wait_ns)) break;
                        copy_pending = false;
                    } else if (!bounded_wait(qfull, qi & 1, abort_flag, p.wait_ns)) {
                        break;  // the epilogue has written this group's query operand
                    }
                    tc_fence_after_sync();
                    idesc = idesc_e4m3_f32(128, (uint32_t)pl.nr[g] * kHeads);
                    ++qi;
                }
                if (!bounded_wait(&tempty[li & 1], ((li >> 1) & 1) ^ 1, abort_flag, p.wait_ns)) break;
                tc_fence_after_sync();
                if (!bounded_wait(&full[li % kStages], (li / kStages) & 1, abort_flag, p.wait_ns)) break;
                const uint32_t d = tmem_base + (uint32_t)(li & 1) * kAccCols;
                const uint32_t a = a0 + (uint32_t)(li % kStages) * kStageBytes;
                for (int k = 0; k < nmma; ++k) {  // K slice k % 4 of the hi (k < 4) or lo term
                    const uint32_t kk = (uint32_t)(k & 3) * 32;
                    mma_f8f6f4(d, desc_kmajor_sw128(a + kk), desc_kmajor_sw128((k < 4 ? bh : bl) + kk), idesc,
                               k > 0 ? 1u : 0u);
                }
                mma_commit(&tfull[li & 1]);
            }
            // Every MMA issued here must finish before TMEM is released, and an
            // operand copy in flight before the CTA leaves.
            int dummy = 0;
            mma_commit(drain);
            bounded_wait(drain, 0, &dummy);
            if (copy_pending) bounded_wait(qcopy, (qi & 1), &dummy);
        }
    } else {
        // ---------------------------------------------------------- epilogue
        const int e = warp - 2;            // 0..15
        const int quad = warp & 3;         // TMEM lanes this warp may read
        const int rr = e >> 2;             // the group row this warp reduces
        const int key = quad * 32 + lane;  // key of the tile this thread owns
        int g = find_group(pl, n_groups, it0), li = 0, qi = 0;
        int gend = -1, gbeg = 0, r0 = 0, nr = 0, rlen = 0;
        const float* w = wq_s;
        uint64_t wr[kRegW ? 16 : 1];  // kRegW: w' of heads 0..31 of this warp's row, packed pairs
        for (int it = it0; it < it1; ++it, ++li) {
            if (it >= gend) {
                // A new group.  Every MMA that read the previous group's query has
                // completed (this warp waited for the last one's accumulator), so
                // the operand can be rewritten.
                while (g + 1 < n_groups && it >= pl.item[g + 1]) ++g;
                gbeg = pl.item[g];
                gend = pl.item[g + 1];
                r0 = pl.r0[g];
                nr = pl.nr[g];
                rlen = rr < nr ? pl.row_len[r0 + rr] : 0;
                if (p.qop) {
                    // the MMA warp copies the prepared operand and w' in once
                    // every epilogue warp is done with the previous group
                    if (qi > 0) {
                        fence_proxy_async_smem();  // this warp's reads of w' -> the copy's writes
                        __syncwarp();
                        if (lane == 0) mbar_arrive(grp_ready);
                    }
                    if (!bounded_wait(qcopy, qi & 1, abort_flag, p.wait_ns)) break;
                    w = wq_s + rr * kHeads;
                } else {
                    float* wbuf = wq_s + (qi & 1) * kQRows;
                    split_group_query(p, r0, nr, q_hi, q_lo, wbuf, e, lane);
                    fence_proxy_async_smem();  // generic-proxy writes -> the tensor core's operand reads
                    __syncwarp();
                    if (lane == 0 && !p.drop_query_handoff) mbar_arrive(qfull);
                    if (!bounded_wait(qfull, qi & 1, abort_flag, p.wait_ns)) break;  // every warp's w' is written
                    w = wbuf + rr * kHeads;
                }
                if constexpr (kRegW) {
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const float4 x = *reinterpret_cast<const float4*>(w + 4 * j);
                        wr[2 * j] = pack2(x.x, x.y);
                        wr[2 * j + 1] = pack2(x.z, x.w);
                    }
                }
                ++qi;
            }
            const int s = li % kStages, acc = li & 1;
            if (!bounded_wait(&tfull[acc], (li >> 1) & 1, abort_flag, p.wait_ns)) break;
            tc_fence_after_sync();
            // The stage cannot be refilled before this warp releases it, so its
            // `full` phase is still the current one: observe it, then read the
            // scales the bulk copy wrote.
            if (!bounded_wait(&full[s], (li / kStages) & 1, abort_flag, p.wait_ns)) break;
            const float sc = scales[s * kTileKeys + key];
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
            if (rr < nr) {  // warp-uniform
                const int64_t pos = (int64_t)(it - gbeg) * kTileKeys + key;
                const uint32_t taddr = tmem_base + ((uint32_t)(quad * 32) << 16) +
                                       (uint32_t)acc * kAccCols + (uint32_t)rr * kHeads;
                uint64_t a[4] = {0ull, 0ull, 0ull, 0ull};  // four packed (2 x f32) partial sums
                // Heads in the same order either way: a[j] takes head pairs
                // (8 i + 2 j, 8 i + 2 j + 1) for i = 0 .. 7.
                if constexpr (kRegW) {
#pragma unroll
                    for (int ch = 0; ch < 4; ++ch) {  // 16 head columns at a time
                        float v[16];
                        tmem_load_16cols(taddr + 16 * ch, v);
                        if (ch == 3) {
                            // every column of this warp is in registers: release
                            // the accumulator before the last chunk's arithmetic
                            tc_fence_before_sync();
                            __syncwarp();
                            if (lane == 0) mbar_arrive(&tempty[acc]);
                        }
#pragma unroll
                        for (int h = 0; h < 16; h += 8) {
                            uint64_t wp[4];
                            if (ch < 2) {
#pragma unroll
                                for (int j = 0; j < 4; ++j) wp[j] = wr[(16 * ch + h) / 2 + j];
                            } else {
                                const float4 w0 = *reinterpret_cast<const float4*>(w + 16 * ch + h);
                                const float4 w1 = *reinterpret_cast<const float4*>(w + 16 * ch + h + 4);
                                wp[0] = pack2(w0.x, w0.y);
                                wp[1] = pack2(w0.z, w0.w);
                                wp[2] = pack2(w1.x, w1.y);
                                wp[3] = pack2(w1.z, w1.w);
                            }
                            a[0] = ffma2(wp[0], pack2(relu2(v[h + 0]), relu2(v[h + 1])), a[0]);
                            a[1] = ffma2(wp[1], pack2(relu2(v[h + 2]), relu2(v[h + 3])), a[1]);
                            a[2] = ffma2(wp[2], pack2(relu2(v[h + 4]), relu2(v[h + 5])), a[2]);
                            a[3] = ffma2(wp[3], pack2(relu2(v[h + 6]), relu2(v[h + 7])), a[3]);
                        }
                    }
                } else {
#pragma unroll
                    for (int hf = 0; hf < 2; ++hf) {
                        float v[32];
                        tmem_load_32cols(taddr + 32 * hf, v);
                        if (hf == 1) {
                            // every column of this warp is in registers: release the
                            // accumulator before the second half's arithmetic
                            tc_fence_before_sync();
                            __syncwarp();
                            if (lane == 0) mbar_arrive(&tempty[acc]);
                        }
#pragma unroll
                        for (int h = 0; h < 32; h += 8) {
                            const float4 w0 = *reinterpret_cast<const float4*>(w + 32 * hf + h);
                            const float4 w1 = *reinterpret_cast<const float4*>(w + 32 * hf + h + 4);
                            a[0] = ffma2(pack2(w0.x, w0.y), pack2(relu2(v[h + 0]), relu2(v[h + 1])), a[0]);
                            a[1] = ffma2(pack2(w0.z, w0.w), pack2(relu2(v[h + 2]), relu2(v[h + 3])), a[1]);
                            a[2] = ffma2(pack2(w1.x, w1.y), pack2(relu2(v[h + 4]), relu2(v[h + 5])), a[2]);
                            a[3] = ffma2(pack2(w1.z, w1.w), pack2(relu2(v[h + 6]), relu2(v[h + 7])), a[3]);
                        }
                    }
                }
                const float2 s0 = unpack2(a[0]), s1 = unpack2(a[1]), s2 = unpack2(a[2]), s3 = unpack2(a[3]);
                const float sum = ((s0.x + s0.y) + (s1.x + s1.y)) + ((s2.x + s2.y) + (s3.x + s3.y));
                // the terms carry 2 ReLU(d): halve the sum (exact), then the scale
                const float out = __fadd_rn((sum * 0.5f) * sc, 0.0f);  // -0 -> +0
                if (pos < rlen) p.scores[(int64_t)(r0 + rr) * p.score_stride + pos] = out;
            } else {
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(&tempty[acc]);
            }
        }
    }

    // This CTA's scores are written: the selection (a programmatic dependent)
    // may launch onto the SMs the scoring frees; it waits for the whole grid.
    pdl_launch_dependents();
    tc_fence_before_sync();
    __syncthreads();
    if (threadIdx.x == 0 && *abort_flag) record_status(p.status, kStatusTimeout);
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

}  // namespace

cudaError_t launch_score(const ScoreArgs& a, const CUtensorMap& keys_map) {
    static thread_local int configured_device = -1;  // per host thread: setting the attribute is idempotent
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (configured_device != dev) {
        err = cudaFuncSetAttribute(k_score<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
        if (err != cudaSuccess) return err;
        err = cudaFuncSetAttribute(k_score<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
        if (err != cudaSuccess) return err;
        configured_device = dev;
    }
    ScoreParams p;
    p.qtype = a.qtype;
    p.q = a.q;
    p.head_w = a.head_w;
    p.seq_lens = a.seq_lens;
    p.row_req = a.row_req;
    p.R = a.R;
    p.len_cap = a.len_bound < (int64_t)a.max_pages * kPage ? a.len_bound : (int64_t)a.max_pages * kPage;
    p.k_scale = a.k_scale;
    p.block_table = a.block_table;
    p.pool_pages = a.pool_pages;
    p.max_pages = a.max_pages;
    p.scores = a.scores;
    p.score_stride = a.score_stride;
    p.status = reinterpret_cast<uint32_t*>(a.ws + a.L.status);
    p.qop = a.L.qop ? reinterpret_cast<uint8_t*>(a.ws + a.L.qop) : nullptr;
    if (a.new_k && !p.qop) return cudaErrorInvalidValue;  // the store is k_qprep's
    p.inputs_ready = a.inputs_ready && p.qop ? 1 : 0;
    p.table_prefetch = a.table_prefetch && !a.inputs_ready ? 1 : 0;
    p.new_k = a.new_k;
    p.new_scale = a.new_scale;
    p.k_cache_w = const_cast<uint8_t*>(a.k_cache);
    p.k_scale_w = const_cast<float*>(a.k_scale);
    const WaitTestHook hook = wait_test_hook();
    p.wait_ns = hook.wait_ns ? hook.wait_ns : kWaitTimeoutNs;
    p.drop_query_handoff = hook.drop_query_handoff;
    // Tiles per CTA, at least (the rows form at least ceil(R / 4) groups, each
    // of up to len_cap keys): the register-held weights from 12 on.
    const int64_t tiles = (int64_t)((a.R + kGroupRows - 1) / kGroupRows) * ((p.len_cap + kTileKeys - 1) / kTileKeys);
    const bool reg_w = tiles >= (int64_t)kRegWTilesPerCta * a.num_sms;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)a.num_sms, 1, 1);
    cfg.blockDim = dim3(kScoreThreads, 1, 1);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = a.stream;
    // Every launch is a programmatic dependent of the kernel before it on the
    // stream: its CTAs may launch (on SMs that kernel leaves free) once that
    // kernel allows it.  k_qprep and, without a prepared operand, k_score wait
    // for it (griddepcontrol.wait) before reading an input it may write; the
    // selection allows its dependent at its start, the host call's gather
    // kernel too; any other kernel before it simply completes first.
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (p.qop) {
        // the rows' operands first, as the scoring's predecessor on the stream
        const int pairs = p.R * kHeads;
        const int per_cta = (kQprepThreads / 32) * kQprepPairsPerWarp;
        cudaLaunchConfig_t qc = {};
        qc.gridDim = dim3((unsigned)((pairs + per_cta - 1) / per_cta), 1, 1);
        qc.blockDim = dim3(kQprepThreads, 1, 1);
        qc.stream = a.stream;
        qc.attrs = attr;
        qc.numAttrs = 1;
        const cudaError_t e = cudaLaunchKernelEx(&qc, k_qprep, p);
        if (e != cudaSuccess) return e;
    }
    return reg_w ? cudaLaunchKernelEx(&cfg, k_score<true>, keys_map, p)
                 : cudaLaunchKernelEx(&cfg, k_score<false>, keys_map, p);
}

}  // namespace idx
