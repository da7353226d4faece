// idx_internal.h -- workspace layout and the launchers each kernel file
// exports to the C-ABI layer (idx_api.cu).  Host and device visible.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/idx.h"

namespace idx {

constexpr int kHeads = IDX_HEADS;
constexpr int kDim = IDX_DIM;
constexpr int kPage = IDX_PAGE;
constexpr int kMaxRows = IDX_MAX_ROWS;
constexpr int kGroupRows = IDX_GROUP_ROWS;
constexpr int kTileKeys = 128;             // keys per MMA tile (two pages)
constexpr int kSliceKeys = 1024;           // selection: one slice per this many keys
constexpr int kSelectThreads = 256;

// Device status bits, OR-ed into the workspace status word.
constexpr uint32_t kStatusBounds = 1u;   // block-table id outside the pool / row too long
constexpr uint32_t kStatusTimeout = 2u;  // a bounded wait gave up

// Workspace layout: the status word; the rows' prepared query operands (hi
// and lo E4M3 terms of 8 KB and 64 f32 head weights a row, for the scoring
// calls); then (optionally) an f32 score matrix.
struct WsLayout {
    size_t status;   // uint32 status word
    size_t qop;      // [R] prepared query operands (0: none)
    size_t scores;   // f32 [R][score_stride] (optional)
    size_t end;
    int64_t score_stride;
};

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

constexpr size_t kQopRowBytes = 2 * 8192 + 64 * 4;

inline WsLayout ws_layout(int R, int64_t max_len, int with_scores, int with_qop = 1) {
    WsLayout L{};
    L.status = 0;
    L.score_stride = (max_len + 3) / 4 * 4;
    if (L.score_stride < 4) L.score_stride = 4;
    L.qop = with_qop ? 1024 : 0;
    L.scores = with_qop ? align_up(1024 + kQopRowBytes * (size_t)R, 1024) : 1024;
    L.end = with_scores ? align_up(L.scores + sizeof(float) * (size_t)R * (size_t)L.score_stride, 1024) : L.scores;
    return L;
}

// ---- launchers (each defined next to its kernel) --------------------------

struct ScoreArgs {
    int qtype;
    const void* q;
    const float* head_w;
    const uint8_t* k_cache;
    const float* k_scale;
    int64_t pool_pages;
    const int32_t* block_table;
    int max_pages;
    const int32_t* seq_lens;
    const int32_t* row_req;
    int R;
    float* scores;
    int64_t score_stride;
    int64_t len_bound;  // rows are clamped to this many keys (the score buffer's width)
    char* ws;
    WsLayout L;
    cudaStream_t stream;
    int num_sms;
    // Keys this call stores: row r's key new_k[r] (128 E4M3 codes) and scale
    // new_scale[r] go to its own cache slot, position seq_lens[r] - 1 of its
    // request, before any row scores them (null: no store).  The cache
    // pointers above are then written.
    const uint8_t* new_k = nullptr;
    const float* new_scale = nullptr;
    // The caller guarantees that the block table, lengths, row map, key cache
    // and scales are complete when the call is enqueued (no kernel that may
    // still be running writes them): the scoring may then launch before
    // k_qprep's grid wait and read them while the kernel before the call
    // still runs.
    bool inputs_ready = false;
    // k_qprep prefetches long rows' block-table entries into L2 (off when the
    // table was written just before the call and is in L2 already).
    bool table_prefetch = true;
};

cudaError_t launch_score(const ScoreArgs& a, const CUtensorMap& keys_map);

// Test hook of the calling host thread (diag.cu): a wall-time limit for the
// scoring kernel's waits (0 = the normal kWaitTimeoutNs) and whether the
// epilogue leaves out its signal that the query operand is written, so that
// a test can make a bounded wait run out without a fault.
struct WaitTestHook {
    uint64_t wait_ns;
    int drop_query_handoff;
};
WaitTestHook wait_test_hook();

struct SelectArgs {
    const float* scores;
    int64_t score_stride;
    const int32_t* row_lens;
    int R;
    int k;
    int32_t* indices;
    uint32_t* status;     // may be null
    int64_t max_len;      // bound on row lengths (launch shape)
    int64_t len_cap;      // rows longer than this are cut to it (and reported)
    cudaStream_t stream;
    // When slot_table is set, list entries are physical cache slots
    // (slot_table[row_req[r]][pos / page] * page + pos % page) instead of positions.
    const int32_t* slot_table = nullptr;
    const int32_t* slot_row_req = nullptr;
    int slot_max_pages = 0;
    // When pairs is set, entry j of row r goes to pairs[r][j] as the int32
    // words {entry, tag} (one 8-byte store) instead of indices[r][j].
    long long* pairs = nullptr;
    uint32_t tag = 0;
};

cudaError_t launch_select(const SelectArgs& a);
// After launch_select on the same stream: each row's list rearranged into the
// pages' prefix order for candidate room `room` (position lists only).
cudaError_t launch_prefix_order(const SelectArgs& a, int64_t room);

// Device copies of host buffers the GPU can address (page-locked, mapped):
// every source and destination 16-byte aligned, every size a multiple of 4.
constexpr int kStageMaxCopies = 5;
struct StageCopy {
    const void* src;
    void* dst;
    uint32_t bytes;
};
struct StagePlan {
    StageCopy c[kStageMaxCopies];
    int n;
};
cudaError_t launch_stage(const StagePlan& plan, cudaStream_t stream);

// FP8 query quantisation of a bf16 query [R][64][128] (quant.cuh).
cudaError_t launch_quantize(const void* q, const float* head_w, int R, uint8_t* q8, float* w_out,
                            cudaStream_t stream);
// Longest row the selection handles with clusters of `cluster` CTAs.
int64_t select_max_len(int cluster);
constexpr int64_t kSelectMaxLen = 16 * 512 * 4 * 16;  // 524,288 keys (16-CTA clusters)

}  // namespace idx
