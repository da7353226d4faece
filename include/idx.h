/*
 * idx.h -- C ABI of the GB300 index chain: paged FP8 key scoring and exact
 * top-k selection for sparse-attention decode.
 *
 * The operation is the one of "sgl-amd-mono-upstream PR 18" (GLM-5.3 indexer
 * launch): section "Modifications / 2. A request's rows scored together"
 * (every row of a request scores that request's paged index keys in one pass,
 * each key read once) and section "Modifications / 3. Every row's exact
 * top-2048 on up to 64 slices" (radix select with all-gathered digit
 * histograms).  The score is the indexer's
 *
 *     s[r, j] = sum_h w[r, h] * ReLU( q[r, h, :] . (k[j, :] * scale[j]) )
 *
 * with k an FP8 E4M3 key, scale its f32 per-key scale, q a bf16 (or E4M3)
 * query row of H = 64 heads of D = 128 dims, accumulated in f32.
 *
 * Conventions for every entry point:
 *  - All array pointers are DEVICE pointers owned by the caller; the library
 *    allocates nothing and keeps no pointer after the call returns.
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream).  Work is
 *    enqueued asynchronously; no entry point synchronises except
 *    idx_check_status.
 *  - A returned idx_status reports argument errors found on the host before
 *    anything is enqueued (nothing is launched then) and launch errors.
 *    Errors found by the kernels (a block-table entry outside the pool, a row
 *    longer than its block table, a wait that timed out) are OR-ed into a
 *    status word in the workspace and read with idx_check_status.
 *  - Shapes are fixed: IDX_HEADS heads, IDX_DIM dims, IDX_PAGE tokens a page.
 */
#ifndef IDX_H
#define IDX_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define IDX_HEADS 64      /* index heads per query row */
#define IDX_DIM 128       /* index head dimension */
#define IDX_PAGE 64       /* tokens per key-cache page */
#define IDX_MAX_K 2048    /* largest k of the top-k */
#define IDX_MAX_ROWS 1024 /* most query rows in one call */
#define IDX_GROUP_ROWS 4  /* rows of one request scored in one pass */
#define IDX_MAX_TOPK_LEN 524288 /* longest row the top-k selection takes */

typedef enum {
    IDX_OK = 0,
    IDX_ERR_ARG = -1,       /* a NULL pointer, a size out of range */
    IDX_ERR_ALIGN = -2,     /* a pointer or stride that breaks the alignment rule */
    IDX_ERR_WORKSPACE = -3, /* workspace NULL or smaller than idx_workspace_bytes */
    IDX_ERR_CUDA = -4,      /* a CUDA call failed (launch, attribute, ...) */
    IDX_ERR_TIMEOUT = -5,   /* device: a bounded wait gave up */
    IDX_ERR_BOUNDS = -6,    /* device: block-table id outside the pool, or a row
                               longer than its block table (row treated as shorter) */
    IDX_ERR_UNSUPPORTED = -7 /* no sm_103a device, or a missing driver feature */
} idx_status;

typedef enum {
    IDX_Q_BF16 = 0,     /* q holds bf16 values */
    IDX_Q_E4M3 = 1,     /* q holds FP8 E4M3 codes; any per-(row, head) scale of q
                           is the caller's to fold into head_w */
    IDX_Q_BF16_FP8 = 2  /* q holds bf16 values that the scoring quantises to
                           E4M3 on the device, one scale per (row, head) folded
                           into head_w, as idx_quantize_query does; the scores
                           are those of the quantised query */
} idx_qtype;

/* Bytes of workspace the calls below need for R rows, rows of at most
 * `max_len` keys and top-k size k.  `with_scores` != 0 adds room for an f32
 * score matrix [R][round_up(max_len, 4)], used by idx_score_topk when the
 * caller passes scores == NULL.  The workspace must be 1024-byte aligned and
 * zeroed once before its first use (idx_workspace_init does that). */
size_t idx_workspace_bytes(int R, int64_t max_len, int k, int with_scores);

/* Zero the workspace's status word (asynchronously on `stream`). */
idx_status idx_workspace_init(void *workspace, size_t ws_bytes, void *stream);

/*
 * idx_score -- score every key of each row's request against the row.
 *
 *  qtype        IDX_Q_BF16, IDX_Q_E4M3 or IDX_Q_BF16_FP8
 *  q            [R][IDX_HEADS][IDX_DIM] bf16 or E4M3, 16-byte aligned
 *  head_w       [R][IDX_HEADS] f32
 *  k_cache      [pool_pages][IDX_PAGE][IDX_DIM] E4M3 codes, 16-byte aligned
 *  k_scale      [pool_pages][IDX_PAGE] f32, 16-byte aligned; every scale >= 0
 *               (the scale is taken out of the ReLU)
 *  pool_pages   pages in the pool (1 .. 2^25)
 *  block_table  [n_req][max_pages] int32: page ids of request i's keys in
 *               position order (key j of a request is page j/64, slot j%64)
 *  max_pages    row stride of block_table
 *  seq_lens     [R] int32: keys visible to row r (its request's first seq_lens[r])
 *  row_req      [R] int32: request of row r.  Consecutive rows of one request
 *               are scored together, IDX_GROUP_ROWS at a time.
 *  scores       [R][score_stride] f32 out: scores[r][j] for j < seq_lens[r];
 *               entries at j >= seq_lens[r] are left untouched.  -0 is written
 *               as +0.  16-byte aligned, score_stride a multiple of 4 and at
 *               least the longest row.
 *  workspace    >= idx_workspace_bytes(R, score_stride, 1, 0) bytes
 *
 * Errors: IDX_ERR_ARG (NULL pointer, R outside [1, IDX_MAX_ROWS], bad sizes),
 * IDX_ERR_ALIGN, IDX_ERR_WORKSPACE, IDX_ERR_UNSUPPORTED, IDX_ERR_CUDA.
 */
idx_status idx_score(int qtype, const void *q, const float *head_w,
                     const uint8_t *k_cache, const float *k_scale, int64_t pool_pages,
                     const int32_t *block_table, int max_pages,
                     const int32_t *seq_lens, const int32_t *row_req, int R,
                     float *scores, int64_t score_stride,
                     void *workspace, size_t ws_bytes, void *stream);

/*
 * idx_topk -- exact top-k list of each row of a score matrix.
 *
 * The list of row r (n = row_lens[r] scores) holds the positions whose score
 * is strictly above the k-th largest score, in ascending position, then the
 * positions whose score equals it, in ascending position, until k entries.
 * Rows with n <= k list 0..n-1 and pad with -1.  Scores compare as f32 with
 * -0 == +0; a NaN ranks below every number (finite inputs are expected).
 *
 *  scores       [R][score_stride] f32, 16-byte aligned, score_stride % 4 == 0
 *  row_lens     [R] int32, each in [0, min(score_stride, IDX_MAX_TOPK_LEN)];
 *               a longer row is cut to that length and reported as
 *               IDX_ERR_BOUNDS by idx_check_status
 *  k            1 .. IDX_MAX_K
 *  indices      [R][k] int32 out
 *  workspace    status word holder (>= idx_workspace_bytes(R, score_stride, k, 0)
 *               bytes, else IDX_ERR_WORKSPACE); may be NULL, then device errors
 *               are not reported
 *
 * Errors: IDX_ERR_ARG, IDX_ERR_ALIGN, IDX_ERR_WORKSPACE, IDX_ERR_CUDA.
 */
idx_status idx_topk(const float *scores, int64_t score_stride, const int32_t *row_lens,
                    int R, int k, int32_t *indices,
                    void *workspace, size_t ws_bytes, void *stream);

/*
 * idx_score_topk -- idx_score then idx_topk on the same stream, with no host
 * round trip in between.  scores may be NULL: the scores then live in the
 * workspace (size it with with_scores = 1) and score_stride is ignored.
 * max_len bounds the longest row (used for the launch shape and workspace);
 * it must not exceed IDX_MAX_TOPK_LEN (IDX_ERR_ARG), and rows longer than
 * max_len are cut to it (IDX_ERR_BOUNDS).
 */
idx_status idx_score_topk(int qtype, const void *q, const float *head_w,
                          const uint8_t *k_cache, const float *k_scale, int64_t pool_pages,
                          const int32_t *block_table, int max_pages,
                          const int32_t *seq_lens, const int32_t *row_req, int R,
                          int64_t max_len, int k, int32_t *indices,
                          float *scores, int64_t score_stride,
                          void *workspace, size_t ws_bytes, void *stream);

/*
 * idx_score_topk_ready -- idx_score_topk (same arguments, scores, lists and
 * errors) for a caller whose block_table, seq_lens, row_req, k_cache and
 * k_scale are complete when the call is enqueued: written by the host, by
 * copies or by kernels that have finished, and by no kernel that may still
 * be running.  q and head_w may still come from the kernel just before the
 * call on the stream.  The scoring launch then starts on the SMs that kernel
 * leaves free and builds its plan, reads the block table and fetches its
 * first key pages while that kernel runs; it reads q and head_w and writes
 * scores only after that kernel has completed.  In a sequence of decode
 * steps whose paged-cache metadata is prepared ahead, this overlaps each
 * step's scoring set-up with the previous step's selection
 * ("sgl-amd-mono-upstream PR 18", section "Motivation": the indexer launch
 * is the whole chain, so its fixed latencies are the cost at small sizes).
 * With inputs that break the condition the scores race with their writer
 * and are undefined.
 */
idx_status idx_score_topk_ready(int qtype, const void *q, const float *head_w,
                                const uint8_t *k_cache, const float *k_scale, int64_t pool_pages,
                                const int32_t *block_table, int max_pages,
                                const int32_t *seq_lens, const int32_t *row_req, int R,
                                int64_t max_len, int k, int32_t *indices,
                                float *scores, int64_t score_stride,
                                void *workspace, size_t ws_bytes, void *stream);

/*
 * idx_score_topk_slots -- idx_score_topk whose lists hold physical cache
 * slots instead of logical positions: a list entry for position p of row r
 * is block_table[row_req[r]][p / IDX_PAGE] * IDX_PAGE + p % IDX_PAGE, the
 * row of the paged key cache that holds the key, which is what a sparse
 * attention over the same paged cache gathers ("sgl-amd-mono-upstream PR 18",
 * the consumer's slot format); -1 padding stays -1.  The list order, the
 * arguments and the errors are those of idx_score_topk (slots in place of
 * indices).
 */
idx_status idx_score_topk_slots(int qtype, const void *q, const float *head_w,
                                const uint8_t *k_cache, const float *k_scale, int64_t pool_pages,
                                const int32_t *block_table, int max_pages,
                                const int32_t *seq_lens, const int32_t *row_req, int R,
                                int64_t max_len, int k, int32_t *slots,
                                float *scores, int64_t score_stride,
                                void *workspace, size_t ws_bytes, void *stream);

/*
 * idx_score_topk_tagged -- idx_score_topk whose lists are written as tagged
 * pairs, the hand-off of "sgl-amd-mono-upstream PR 11" (GLM-5.3-Flash
 * monokernel hand-offs), section "3. The selected tokens are tagged pairs": a
 * consumer polls the list entries themselves for the launch's tag instead of a
 * separate ready flag written after them.  Entry j of row r is
 *
 *     pairs[r][j] = ((uint64_t)tag << 32) | (uint32_t)entry
 *
 * i.e. the int32 words {entry, tag} in that order in memory, stored with one
 * 8-byte store, so a reader that finds `tag` in a pair (with an 8-byte load)
 * finds this launch's entry beside it.  entry is the list entry of
 * idx_score_topk (a logical position), or with slots != 0 that of
 * idx_score_topk_slots (a physical cache slot); -1 padding is stored as
 * {-1, tag}, so a short row is complete once all k pairs carry the tag.  The
 * caller picks the tag (a step counter, say) and must not reuse the tag of a
 * launch whose pairs a reader might still mistake for this one's.
 *
 *  tag          32-bit launch tag
 *  slots        0: positions, else physical cache slots
 *  pairs        [R][k] int64 out, 8-byte aligned (else IDX_ERR_ALIGN)
 *
 * The other arguments, the list order and the errors are those of
 * idx_score_topk.
 */
idx_status idx_score_topk_tagged(int qtype, const void *q, const float *head_w,
                                 const uint8_t *k_cache, const float *k_scale, int64_t pool_pages,
                                 const int32_t *block_table, int max_pages,
                                 const int32_t *seq_lens, const int32_t *row_req, int R,
                                 int64_t max_len, int k, uint32_t tag, int slots, int64_t *pairs,
                                 float *scores, int64_t score_stride,
                                 void *workspace, size_t ws_bytes, void *stream);

/*
 * idx_score_topk_newkeys -- idx_score_topk for a step whose rows bring new
 * index keys: "sgl-amd-mono-upstream PR 18", section "Modifications / 2",
 * keys this launch writes.  Row r's own key (its request's position
 * seq_lens[r] - 1, the slot the row writes) is new_k[r] with scale
 * new_scale[r]; the call stores it in the cache and every row of the request
 * scores it, in whichever group of rows that row falls (an 8-row draft chain
 * spans two groups, and the second group scores the first group's new keys).
 * The store comes first, so the cache may hold anything at those slots before
 * the call (stale or poisoned values).
 *
 *  k_cache, k_scale  as in idx_score, and written: slot seq_lens[r] - 1 of
 *               request row_req[r] receives row r's key and scale (rows of one
 *               request name distinct slots; rows with seq_lens[r] == 0 store
 *               nothing; a slot whose block-table entry lies outside the pool
 *               is skipped and reported as IDX_ERR_BOUNDS)
 *  new_k        [R][IDX_DIM] E4M3 codes, 16-byte aligned
 *  new_scale    [R] f32, >= 0
 *
 * The other arguments, the outputs and the errors are those of
 * idx_score_topk.
 */
idx_status idx_score_topk_newkeys(int qtype, const void *q, const float *head_w,
                                  uint8_t *k_cache, float *k_scale, int64_t pool_pages,
                                  const int32_t *block_table, int max_pages,
                                  const int32_t *seq_lens, const int32_t *row_req, int R,
                                  const uint8_t *new_k, const float *new_scale,
                                  int64_t max_len, int k, int32_t *indices,
                                  float *scores, int64_t score_stride,
                                  void *workspace, size_t ws_bytes, void *stream);

/*
 * idx_score_topk_prefix_order -- idx_score_topk whose lists are in the
 * pages' order ("sgl-amd-mono-upstream PR 18", section "Modifications / 3",
 * Order, and section "Modifications / 0", the list check): the pages' radix
 * stops at the first of the threshold's 12- and 24-bit prefixes whose keys
 * fit the candidate room, else at all 32 bits.  With T the k-th largest
 * score's order-preserving 32-bit image (as the selection uses it) and P the
 * first of T's 12- and 24-bit prefixes shared by at most `room` of the row's
 * keys (else all 32 bits), row r's list is
 *     the keys whose image's prefix is above P, in ascending position;
 *     then the keys with prefix P above T, in ascending position;
 *     then the keys equal to T, in ascending position, until k entries.
 * It holds the same keys as idx_score_topk's list; at 32 bits (room 0, or
 * T's prefixes shared too widely) it is that list.  The pages do not size
 * the room; the caller gives it.  Rows with at most k keys are as in
 * idx_score_topk.
 *
 *  room      the candidate room, >= 0 (else IDX_ERR_ARG)
 *  indices   [R][k] int32 out, logical positions
 *
 * The other arguments and the errors are those of idx_score_topk.  One more
 * launch after the selection reads each row's scores once more.
 */
idx_status idx_score_topk_prefix_order(int qtype, const void *q, const float *head_w,
                                       const uint8_t *k_cache, const float *k_scale, int64_t pool_pages,
                                       const int32_t *block_table, int max_pages,
                                       const int32_t *seq_lens, const int32_t *row_req, int R,
                                       int64_t max_len, int k, int64_t room, int32_t *indices,
                                       float *scores, int64_t score_stride,
                                       void *workspace, size_t ws_bytes, void *stream);

/*
 * idx_quantize_query -- the FP8 (E4M3) query of a bf16 index query, one scale
 * per (row, head), as IDX_Q_BF16_FP8 scoring uses it.  The recipe is the
 * per-token FP8 quantisation of "[Perf] [MI355X] minimax_m31" (section
 * "Modifications", o_proj bullet) -- amax / 448, a reciprocal, clamp, round to
 * nearest even -- applied per head: amax = max |q| over the head's IDX_DIM
 * elements, scale = amax / 448 and inv = 1 / scale (correctly rounded f32
 * divisions), q8 = E4M3(q * inv) (f32 product, nearest even, saturated at
 * +-448); w_out = head_w * scale (f32).  A head whose elements are all zero gets
 * codes 0 and weight 0.  Inputs are expected finite.
 *
 *  q       [R][IDX_HEADS][IDX_DIM] bf16, device, 8-byte aligned
 *  head_w  [R][IDX_HEADS] f32, device
 *  q8      [R][IDX_HEADS][IDX_DIM] E4M3 codes out, device, 4-byte aligned
 *  w_out   [R][IDX_HEADS] f32 out, device
 *
 * Asynchronous on `stream`.  Errors: IDX_ERR_ARG, IDX_ERR_ALIGN, IDX_ERR_CUDA.
 */
idx_status idx_quantize_query(const void *q, const float *head_w, int R, uint8_t *q8, float *w_out,
                              void *stream);

/*
 * idx_host_workspace_bytes -- workspace bytes idx_score_topk_host needs for R
 * rows of at most max_len keys, k, and a block table of n_req x max_pages.
 * Returns 0 for arguments out of range.
 */
size_t idx_host_workspace_bytes(int R, int64_t max_len, int k, int n_req, int max_pages);

/*
 * idx_score_topk_host -- the fused call (idx_score_topk) with the per-step
 * inputs and the output in HOST memory: the key cache and its scales stay in
 * device memory (the serving cache), while the query, head weights, block
 * table (n_req x max_pages), row lengths, row map and the [R][k] indices are
 * host buffers.  The call brings the inputs into the workspace, runs the
 * scoring and the selection on `stream` (the scores live in the workspace),
 * and returns the indices to indices_host.  Page-locked buffers that the
 * driver maps into the device's address space (16-byte aligned inputs) are
 * read by one gather kernel and the indices written by the selection kernel
 * directly, over the CPU-GPU link; other host buffers go through
 * cudaMemcpyAsync.  Everything is asynchronous: the indices are in
 * indices_host once the stream has reached the end of the call (synchronise
 * it, or wait on an event recorded after the call), and the host must not
 * modify the inputs before then.
 *
 * The gather kernel and the scoring kernel are programmatic dependents of
 * the kernel before each on `stream` (as every scoring launch is): the gather
 * may read the host buffers as soon as that kernel allows dependents to
 * launch (this library's selection does so at its start; a kernel that never
 * does simply completes first), and waits for it to complete before writing
 * the workspace.  So the host buffers must hold this call's inputs when the
 * call is made.
 *
 *  workspace  device memory, 1024-byte aligned, >= idx_host_workspace_bytes
 *             (R, max_len, k, n_req, max_pages), zeroed once by idx_workspace_init
 *
 * Errors: those of idx_score_topk, all checked before anything is launched;
 * IDX_ERR_ARG for a null host pointer or a size out of range, IDX_ERR_CUDA
 * when a copy cannot be queued.
 */
idx_status idx_score_topk_host(int qtype, const void *q_host, const float *head_w_host,
                               const uint8_t *k_cache, const float *k_scale, int64_t pool_pages,
                               const int32_t *block_table_host, int n_req, int max_pages,
                               const int32_t *seq_lens_host, const int32_t *row_req_host, int R,
                               int64_t max_len, int k, int32_t *indices_host,
                               void *workspace, size_t ws_bytes, void *stream);

/*
 * idx_score_noalloc -- idx_score for callers that cannot allocate device
 * memory, with no workspace argument.  The indexer launch this library
 * follows has no counterpart to this entry point; it exists for callers such
 * as a serving loop replaying a captured CUDA graph, an allocator-less
 * embedding, or code inside a memory pool that forbids new allocations,
 * which cannot obtain (or size) a workspace buffer.
 *
 * Arguments, layouts and results are those of idx_score minus the workspace.
 * Instead of a workspace, the call uses one fixed scratch array in device
 * memory that the library declares statically (1 KB holding the call's status
 * word; every device that loads the library holds it until the process
 * exits).  Nothing is allocated: no cudaMalloc, no cudaFree, no allocating
 * library routine.
 *
 *  - R must be in [1, IDX_NOALLOC_MAX_ROWS]; larger R returns IDX_ERR_ARG.
 *  - The first call in a CUDA context (normally a device's primary context)
 *    looks up the array's device address with that context current; make
 *    that first call before any stream capture.  After a device reset the
 *    next call looks the address up again.
 *  - All calls share the one array.  Calls whose work overlaps on the GPU
 *    (different streams without ordering, or several host threads) share its
 *    status word; nothing else is shared, and nothing needs clearing.
 *  - Device-detected problems (a block-table id outside the pool, a row
 *    longer than its block table or the score buffer) are handled as in
 *    idx_score but not reported: there is no status word to read them from.
 */
#define IDX_NOALLOC_MAX_ROWS IDX_MAX_ROWS
idx_status idx_score_noalloc(int qtype, const void *q, const float *head_w,
                             const uint8_t *k_cache, const float *k_scale, int64_t pool_pages,
                             const int32_t *block_table, int max_pages,
                             const int32_t *seq_lens, const int32_t *row_req, int R,
                             float *scores, int64_t score_stride, void *stream);

/* Wait for `stream`, read and clear the workspace status word, and return the
 * first device error recorded since the last call (IDX_OK if none). */
idx_status idx_check_status(void *workspace, void *stream);

/* A short English name for a status code. */
const char *idx_status_str(int status);

/* Library version, major * 10000 + minor * 100 + patch. */
int idx_version(void);

#ifdef __cplusplus
}
#endif

#endif /* IDX_H */
