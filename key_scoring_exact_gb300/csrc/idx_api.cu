// idx_api.cu -- the C ABI declared in include/idx.h: host-side argument
// checks, workspace layout, TMA descriptors and the launch sequence.
// No entry point allocates device memory or synchronises (except
// idx_check_status); all work goes to the caller's stream.
#include <cstdio>
#include <cstring>
#include <mutex>

#include "idx_internal.h"

namespace idx {
namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
        (void)cudaGetLastError();
    });
    return fn;
}

struct DeviceInfo {
    int ok = 0;  // sm_103
    int num_sms = 0;
};

// Cached per host thread, so concurrent callers share no mutable state.
idx_status device_info(DeviceInfo* out) {
    static thread_local DeviceInfo cache[64];
    static thread_local int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        (void)cudaGetLastError();
        return IDX_ERR_CUDA;
    }
    if (dev < 0 || dev >= 64) return IDX_ERR_UNSUPPORTED;
    if (!cached[dev]) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            (void)cudaGetLastError();
            return IDX_ERR_CUDA;
        }
        cache[dev].ok = (major == 10 && minor == 3);
        cache[dev].num_sms = sms;
        cached[dev] = 1;
    }
    *out = cache[dev];
    return out->ok ? IDX_OK : IDX_ERR_UNSUPPORTED;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// 2D uint8 tensor map: rows of 128 bytes, boxes of 64 rows, 128-byte swizzle.
idx_status make_rows_map(CUtensorMap* map, const void* base, uint64_t rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return IDX_ERR_UNSUPPORTED;
    const cuuint64_t dims[2] = {(cuuint64_t)kDim, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)kDim};
    const cuuint32_t box[2] = {(cuuint32_t)kDim, (cuuint32_t)kPage};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? IDX_OK : IDX_ERR_CUDA;
}

idx_status check_score_args(int qtype, const void* q, const float* head_w, const uint8_t* k_cache,
                            const float* k_scale, int64_t pool_pages, const int32_t* block_table,
                            int max_pages, const int32_t* seq_lens, const int32_t* row_req, int R,
                            void* workspace) {
    if (qtype != IDX_Q_BF16 && qtype != IDX_Q_E4M3 && qtype != IDX_Q_BF16_FP8) return IDX_ERR_ARG;
    if (!q || !head_w || !k_cache || !k_scale || !block_table || !seq_lens || !row_req) return IDX_ERR_ARG;
    if (R < 1 || R > kMaxRows) return IDX_ERR_ARG;
    if (pool_pages < 1 || pool_pages > (int64_t(1) << 25)) return IDX_ERR_ARG;
    if (max_pages < 1 || (int64_t)max_pages * kPage > INT32_MAX) return IDX_ERR_ARG;
    if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(k_scale, 16)) return IDX_ERR_ALIGN;
    if (!workspace) return IDX_ERR_WORKSPACE;
    if (!aligned(workspace, 1024)) return IDX_ERR_ALIGN;
    return IDX_OK;
}

idx_status to_status(cudaError_t e) {
    if (e == cudaSuccess) return IDX_OK;
    (void)cudaGetLastError();
    return IDX_ERR_CUDA;
}

idx_status run_score(const ScoreArgs& a) {
    CUtensorMap keys_map;
    idx_status st = make_rows_map(&keys_map, a.k_cache, (uint64_t)a.pool_pages * kPage);
    if (st != IDX_OK) return st;
    return to_status(launch_score(a, keys_map));
}

// ---------------------------------------------------------------------------
// Scratch for idx_score_noalloc: a fixed device array instead of a caller
// workspace.  It holds the part of the workspace layout the scoring kernel
// uses (its status word); every device that loads this library keeps it for
// the life of the process.
constexpr size_t kNoallocScratchBytes = 1024;  // the status word's block of the workspace layout

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

// The current CUDA context's unique id (driver entry points fetched at run
// time: the library does not link the driver library); 0 when unavailable.
unsigned long long current_context_id() {
    using GetCurrentFn = CUresult (*)(CUcontext*);
    using GetIdFn = CUresult (*)(CUcontext, unsigned long long*);
    static GetCurrentFn get_current = nullptr;
    static GetIdFn get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<GetCurrentFn>(p);
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<GetIdFn>(p);
        (void)cudaGetLastError();
    });
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS)
        return 0;
    return id;
}

// The array's device address in the current context (in host code the
// array's name is only a stand-in for it), looked up once per context with
// that context current: a device reset or another context gets a lookup of
// its own, so no address outlives the context it belongs to.  Without a
// context id the address is looked up on every call (that allocates nothing).
idx_status noalloc_scratch(char** out) {
    static std::mutex mu;
    constexpr int kSlots = 16;
    static unsigned long long ids[kSlots] = {0};
    static char* addrs[kSlots] = {nullptr};
    static int next = 0;
    unsigned long long id = current_context_id();  // 0 before the device's context is made current
    std::lock_guard<std::mutex> lock(mu);
    if (id != 0)
        for (int i = 0; i < kSlots; ++i)
            if (ids[i] == id) {
                *out = addrs[i];
                return IDX_OK;
            }
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {  // makes the context current
        (void)cudaGetLastError();
        return IDX_ERR_CUDA;
    }
    if (id == 0) id = current_context_id();
    if (id != 0) {
        ids[next] = id;
        addrs[next] = static_cast<char*>(p);
        next = (next + 1) % kSlots;
    }
    *out = static_cast<char*>(p);
    return IDX_OK;
}

}  // namespace
}  // namespace idx

using namespace idx;

namespace {
// Host-buffer fused call: the fused call's workspace (scores inside), then
// device copies of the per-step inputs and of the output indices.
struct HostLayout {
    size_t q, w, bt, lens, rreq, idx, end;
};
HostLayout host_layout(int R, int64_t max_len, int k, int n_req, int max_pages) {
    HostLayout H{};
    size_t at = ws_layout(R, max_len, 1).end;
    auto take = [&at](size_t bytes) {
        const size_t p = at;
        at = align_up(at + bytes, 256);
        return p;
    };
    H.q = take((size_t)R * kHeads * kDim * 2);
    H.w = take((size_t)R * kHeads * 4);
    H.bt = take((size_t)n_req * (size_t)max_pages * 4);
    H.lens = take((size_t)R * 4);
    H.rreq = take((size_t)R * 4);
    H.idx = take((size_t)R * (size_t)k * 4);
    H.end = align_up(at, 1024);
    return H;
}

// The device address of a host buffer the GPU can reach (page-locked and
// mapped into the device's address space), or null (pageable memory).
const void* mapped(const void* host) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, host) != cudaSuccess) {
        (void)cudaGetLastError();
        return nullptr;
    }
    return a.type == cudaMemoryTypeHost ? a.devicePointer : nullptr;
}
}  // namespace

// The fused call; with `slots` the lists hold physical cache slots, with
// `pairs` they are written as tagged pairs (indices unused).
static idx_status score_topk_impl(int qtype, const void* q, const float* head_w, const uint8_t* k_cache,
                          const float* k_scale, int64_t pool_pages, const int32_t* block_table, int max_pages,
                          const int32_t* seq_lens, const int32_t* row_req, int R, int64_t max_len, int k,
                          int32_t* indices, float* scores, int64_t score_stride, void* workspace,
                          size_t ws_bytes, void* stream, bool slots, long long* pairs = nullptr,
                          uint32_t tag = 0, const uint8_t* new_k = nullptr, const float* new_scale = nullptr,
                          int64_t prefix_room = -1, bool inputs_ready = false, bool table_prefetch = true) {
    idx_status st = check_score_args(qtype, q, head_w, k_cache, k_scale, pool_pages, block_table, max_pages,
                                     seq_lens, row_req, R, workspace);
    if (st != IDX_OK) return st;
    if ((!indices && !pairs) || k < 1 || k > IDX_MAX_K || max_len < 1) return IDX_ERR_ARG;
    if (pairs && !aligned(pairs, 8)) return IDX_ERR_ALIGN;
    const int64_t cap = (int64_t)max_pages * kPage;
    if (max_len > cap) max_len = cap;
    if (max_len > kSelectMaxLen) return IDX_ERR_ARG;
    DeviceInfo dev;
    st = device_info(&dev);
    if (st != IDX_OK) return st;
    const int with_scores = scores == nullptr;
    const WsLayout L = ws_layout(R, max_len, with_scores);
    if (ws_bytes < L.end) return IDX_ERR_WORKSPACE;
    char* ws = static_cast<char*>(workspace);
    if (with_scores) {
        scores = reinterpret_cast<float*>(ws + L.scores);
        score_stride = L.score_stride;
    } else {
        if (score_stride < max_len || score_stride % 4 != 0 || !aligned(scores, 16)) return IDX_ERR_ALIGN;
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    ScoreArgs a{qtype, q, head_w, k_cache, k_scale, pool_pages, block_table, max_pages, seq_lens, row_req,
                R, scores, score_stride, max_len, ws, L, s, dev.num_sms};
    a.new_k = new_k;
    a.new_scale = new_scale;
    a.inputs_ready = inputs_ready;
    a.table_prefetch = table_prefetch;
    st = run_score(a);
    if (st != IDX_OK) return st;
    // Each row's selection covers the keys its scores were written for.
    SelectArgs sel{scores, score_stride, seq_lens, R, k, indices,
                   reinterpret_cast<uint32_t*>(ws + L.status), max_len, max_len, s};
    if (slots) {
        sel.slot_table = block_table;
        sel.slot_row_req = row_req;
        sel.slot_max_pages = max_pages;
    }
    sel.pairs = pairs;
    sel.tag = tag;
    const cudaError_t e = launch_select(sel);
    if (e != cudaSuccess || prefix_room < 0) return to_status(e);
    return to_status(launch_prefix_order(sel, prefix_room));
}

extern "C" {

size_t idx_workspace_bytes(int R, int64_t max_len, int k, int with_scores) {
    (void)k;
    if (R < 1 || R > kMaxRows || max_len < 0) return 0;
    return ws_layout(R, max_len, with_scores).end;
}

idx_status idx_workspace_init(void* workspace, size_t ws_bytes, void* stream) {
    if (!workspace || ws_bytes < 256) return IDX_ERR_WORKSPACE;
    return to_status(cudaMemsetAsync(workspace, 0, 256, static_cast<cudaStream_t>(stream)));
}

idx_status idx_score(int qtype, const void* q, const float* head_w, const uint8_t* k_cache,
                     const float* k_scale, int64_t pool_pages, const int32_t* block_table, int max_pages,
                     const int32_t* seq_lens, const int32_t* row_req, int R, float* scores,
                     int64_t score_stride, void* workspace, size_t ws_bytes, void* stream) {
    idx_status st = check_score_args(qtype, q, head_w, k_cache, k_scale, pool_pages, block_table, max_pages,
                                     seq_lens, row_req, R, workspace);
    if (st != IDX_OK) return st;
    if (!scores) return IDX_ERR_ARG;
    if (score_stride < 4 || score_stride % 4 != 0) return IDX_ERR_ALIGN;
    if (!aligned(scores, 16)) return IDX_ERR_ALIGN;
    DeviceInfo dev;
    st = device_info(&dev);
    if (st != IDX_OK) return st;
    const WsLayout L = ws_layout(R, score_stride, 0);
    if (ws_bytes < L.end) return IDX_ERR_WORKSPACE;
    ScoreArgs a{qtype, q, head_w, k_cache, k_scale, pool_pages, block_table, max_pages, seq_lens, row_req,
                R, scores, score_stride, score_stride, static_cast<char*>(workspace), L,
                static_cast<cudaStream_t>(stream), dev.num_sms};
    return run_score(a);
}

idx_status idx_topk(const float* scores, int64_t score_stride, const int32_t* row_lens, int R, int k,
                    int32_t* indices, void* workspace, size_t ws_bytes, void* stream) {
    if (!scores || !row_lens || !indices) return IDX_ERR_ARG;
    if (R < 1 || R > kMaxRows || k < 1 || k > IDX_MAX_K) return IDX_ERR_ARG;
    if (score_stride < 4 || score_stride % 4 != 0 || !aligned(scores, 16)) return IDX_ERR_ALIGN;
    uint32_t* status = nullptr;
    if (workspace) {
        if (ws_bytes < ws_layout(R, score_stride, 0, 0).end) return IDX_ERR_WORKSPACE;
        status = static_cast<uint32_t*>(workspace);
    }
    DeviceInfo dev;
    idx_status st = device_info(&dev);
    if (st != IDX_OK) return st;
    const int64_t bound = score_stride < kSelectMaxLen ? score_stride : kSelectMaxLen;
    SelectArgs s{scores, score_stride, row_lens, R, k, indices, status, bound, score_stride,
                 static_cast<cudaStream_t>(stream)};
    return to_status(launch_select(s));
}

idx_status idx_score_topk(int qtype, const void* q, const float* head_w, const uint8_t* k_cache,
                          const float* k_scale, int64_t pool_pages, const int32_t* block_table, int max_pages,
                          const int32_t* seq_lens, const int32_t* row_req, int R, int64_t max_len, int k,
                          int32_t* indices, float* scores, int64_t score_stride, void* workspace,
                          size_t ws_bytes, void* stream) {
    return score_topk_impl(qtype, q, head_w, k_cache, k_scale, pool_pages, block_table, max_pages, seq_lens, row_req,
                           R, max_len, k, indices, scores, score_stride, workspace, ws_bytes, stream, false);
}

idx_status idx_score_topk_ready(int qtype, const void* q, const float* head_w, const uint8_t* k_cache,
                                const float* k_scale, int64_t pool_pages, const int32_t* block_table,
                                int max_pages, const int32_t* seq_lens, const int32_t* row_req, int R,
                                int64_t max_len, int k, int32_t* indices, float* scores, int64_t score_stride,
                                void* workspace, size_t ws_bytes, void* stream) {
    return score_topk_impl(qtype, q, head_w, k_cache, k_scale, pool_pages, block_table, max_pages, seq_lens, row_req,
                           R, max_len, k, indices, scores, score_stride, workspace, ws_bytes, stream, false,
                           nullptr, 0, nullptr, nullptr, -1, true);
}

idx_status idx_score_topk_slots(int qtype, const void* q, const float* head_w, const uint8_t* k_cache,
                                const float* k_scale, int64_t pool_pages, const int32_t* block_table,
                                int max_pages, const int32_t* seq_lens, const int32_t* row_req, int R,
                                int64_t max_len, int k, int32_t* slots, float* scores, int64_t score_stride,
                                void* workspace, size_t ws_bytes, void* stream) {
    return score_topk_impl(qtype, q, head_w, k_cache, k_scale, pool_pages, block_table, max_pages, seq_lens, row_req,
                           R, max_len, k, slots, scores, score_stride, workspace, ws_bytes, stream, true);
}

idx_status idx_score_topk_tagged(int qtype, const void* q, const float* head_w, const uint8_t* k_cache,
                                 const float* k_scale, int64_t pool_pages, const int32_t* block_table,
                                 int max_pages, const int32_t* seq_lens, const int32_t* row_req, int R,
                                 int64_t max_len, int k, uint32_t tag, int slots, int64_t* pairs, float* scores,
                                 int64_t score_stride, void* workspace, size_t ws_bytes, void* stream) {
    if (!pairs) return IDX_ERR_ARG;
    return score_topk_impl(qtype, q, head_w, k_cache, k_scale, pool_pages, block_table, max_pages, seq_lens, row_req,
                           R, max_len, k, nullptr, scores, score_stride, workspace, ws_bytes, stream, slots != 0,
                           reinterpret_cast<long long*>(pairs), tag);
}

idx_status idx_score_topk_newkeys(int qtype, const void* q, const float* head_w, uint8_t* k_cache, float* k_scale,
                                  int64_t pool_pages, const int32_t* block_table, int max_pages,
                                  const int32_t* seq_lens, const int32_t* row_req, int R, const uint8_t* new_k,
                                  const float* new_scale, int64_t max_len, int k, int32_t* indices, float* scores,
                                  int64_t score_stride, void* workspace, size_t ws_bytes, void* stream) {
    if (!new_k || !new_scale) return IDX_ERR_ARG;
    if (!aligned(new_k, 16) || !aligned(new_scale, 4)) return IDX_ERR_ALIGN;
    return score_topk_impl(qtype, q, head_w, k_cache, k_scale, pool_pages, block_table, max_pages, seq_lens, row_req,
                           R, max_len, k, indices, scores, score_stride, workspace, ws_bytes, stream, false, nullptr, 0,
                           new_k, new_scale);
}

idx_status idx_score_topk_prefix_order(int qtype, const void* q, const float* head_w, const uint8_t* k_cache,
                                       const float* k_scale, int64_t pool_pages, const int32_t* block_table,
                                       int max_pages, const int32_t* seq_lens, const int32_t* row_req, int R,
                                       int64_t max_len, int k, int64_t room, int32_t* indices, float* scores,
                                       int64_t score_stride, void* workspace, size_t ws_bytes, void* stream) {
    if (room < 0) return IDX_ERR_ARG;
    return score_topk_impl(qtype, q, head_w, k_cache, k_scale, pool_pages, block_table, max_pages, seq_lens, row_req,
                           R, max_len, k, indices, scores, score_stride, workspace, ws_bytes, stream, false, nullptr, 0,
                           nullptr, nullptr, room);
}

idx_status idx_quantize_query(const void* q, const float* head_w, int R, uint8_t* q8, float* w_out,
                              void* stream) {
    if (!q || !head_w || !q8 || !w_out) return IDX_ERR_ARG;
    if (R < 1 || R > kMaxRows) return IDX_ERR_ARG;
    if (!aligned(q, 8) || !aligned(head_w, 4) || !aligned(q8, 4) || !aligned(w_out, 4)) return IDX_ERR_ALIGN;
    DeviceInfo dev;
    const idx_status st = device_info(&dev);
    if (st != IDX_OK) return st;
    return to_status(launch_quantize(q, head_w, R, q8, w_out, static_cast<cudaStream_t>(stream)));
}

size_t idx_host_workspace_bytes(int R, int64_t max_len, int k, int n_req, int max_pages) {
    if (R < 1 || R > kMaxRows || max_len < 1 || k < 1 || k > IDX_MAX_K || n_req < 1 || max_pages < 1) return 0;
    return host_layout(R, max_len, k, n_req, max_pages).end;
}

namespace {
// One host-buffer call: where each input goes in the workspace, which of
// them the stage kernel gathers over the host link (page-locked, mapped
// buffers) and which the copy engine copies, and where the indices go.
struct HostCall {
    int qtype, R, max_pages, k;
    const uint8_t* k_cache;
    const float* k_scale;
    int64_t pool_pages, max_len;
    char* ws;
    size_t ws_bytes;
    HostLayout H;
    StagePlan plan;
    struct {
        const void* host;
        size_t off, bytes;
    } copy[kStageMaxCopies];  // inputs the copy engine takes
    int n_copy;
    int32_t* indices_host;
    int32_t* idx_out;  // mapped host indices, or the workspace's (then copied back)
};

// Every launch and copy of one host-buffer call, in stream order.
idx_status host_launches(const HostCall& c, cudaStream_t s) {
    for (int i = 0; i < c.n_copy; ++i) {
        if (cudaMemcpyAsync(c.ws + c.copy[i].off, c.copy[i].host, c.copy[i].bytes, cudaMemcpyHostToDevice, s) !=
            cudaSuccess) {
            (void)cudaGetLastError();
            return IDX_ERR_CUDA;
        }
    }
    if (c.plan.n > 0 && launch_stage(c.plan, s) != cudaSuccess) {
        (void)cudaGetLastError();
        return IDX_ERR_CUDA;
    }
    const HostLayout& H = c.H;
    // The gather and the scoring kernel are each a programmatic dependent of
    // the kernel before them: the gather reads the host buffers while the
    // previous call's selection runs, the scoring's CTAs set up while the
    // gather runs; each waits for its predecessor before writing (and the
    // scoring before reading what the gather wrote).
    // (the gather has just written the block table: it is in L2, no prefetch)
    const idx_status st =
        score_topk_impl(c.qtype, c.ws + H.q, reinterpret_cast<const float*>(c.ws + H.w), c.k_cache, c.k_scale,
                        c.pool_pages, reinterpret_cast<const int32_t*>(c.ws + H.bt), c.max_pages,
                        reinterpret_cast<const int32_t*>(c.ws + H.lens), reinterpret_cast<const int32_t*>(c.ws + H.rreq),
                        c.R, c.max_len, c.k, c.idx_out, nullptr, 0, c.ws, c.ws_bytes, s, false, nullptr, 0, nullptr,
                        nullptr, -1, false, false);
    if (st != IDX_OK) return st;
    int32_t* idx_dev = reinterpret_cast<int32_t*>(c.ws + H.idx);
    if (c.idx_out == idx_dev && cudaMemcpyAsync(c.indices_host, idx_dev, (size_t)c.R * (size_t)c.k * 4,
                                                cudaMemcpyDeviceToHost, s) != cudaSuccess) {
        (void)cudaGetLastError();
        return IDX_ERR_CUDA;
    }
    return IDX_OK;
}

}  // namespace

idx_status idx_score_topk_host(int qtype, const void* q_host, const float* head_w_host, const uint8_t* k_cache,
                               const float* k_scale, int64_t pool_pages, const int32_t* block_table_host,
                               int n_req, int max_pages, const int32_t* seq_lens_host,
                               const int32_t* row_req_host, int R, int64_t max_len, int k,
                               int32_t* indices_host, void* workspace, size_t ws_bytes, void* stream) {
    if (!q_host || !head_w_host || !block_table_host || !seq_lens_host || !row_req_host || !indices_host)
        return IDX_ERR_ARG;
    if (qtype != IDX_Q_BF16 && qtype != IDX_Q_E4M3 && qtype != IDX_Q_BF16_FP8) return IDX_ERR_ARG;
    if (R < 1 || R > kMaxRows || n_req < 1 || max_pages < 1 || k < 1 || k > IDX_MAX_K || max_len < 1)
        return IDX_ERR_ARG;
    if (!workspace) return IDX_ERR_WORKSPACE;
    if (!aligned(workspace, 1024)) return IDX_ERR_ALIGN;
    HostCall c{};
    c.qtype = qtype;
    c.R = R;
    c.max_pages = max_pages;
    c.k = k;
    c.k_cache = k_cache;
    c.k_scale = k_scale;
    c.pool_pages = pool_pages;
    c.max_len = max_len;
    c.ws = static_cast<char*>(workspace);
    c.ws_bytes = ws_bytes;
    c.H = host_layout(R, max_len, k, n_req, max_pages);
    if (ws_bytes < c.H.end) return IDX_ERR_WORKSPACE;
    // every argument check of the fused call, before anything is launched
    const idx_status pre =
        check_score_args(qtype, c.ws + c.H.q, reinterpret_cast<const float*>(c.ws + c.H.w), k_cache, k_scale,
                         pool_pages, reinterpret_cast<const int32_t*>(c.ws + c.H.bt), max_pages,
                         reinterpret_cast<const int32_t*>(c.ws + c.H.lens),
                         reinterpret_cast<const int32_t*>(c.ws + c.H.rreq), R, workspace);
    if (pre != IDX_OK) return pre;
    if ((max_len < (int64_t)max_pages * kPage ? max_len : (int64_t)max_pages * kPage) > kSelectMaxLen)
        return IDX_ERR_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // Inputs in page-locked, mapped host memory are gathered by one kernel that
    // reads them over the host link; any other buffer is copied by the copy engine.
    const struct {
        const void* host;
        size_t off, bytes;
    } in[kStageMaxCopies] = {
        {q_host, c.H.q, (size_t)R * kHeads * kDim * (qtype == IDX_Q_E4M3 ? 1 : 2)},
        {head_w_host, c.H.w, (size_t)R * kHeads * 4},
        {block_table_host, c.H.bt, (size_t)n_req * (size_t)max_pages * 4},
        {seq_lens_host, c.H.lens, (size_t)R * 4},
        {row_req_host, c.H.rreq, (size_t)R * 4},
    };
    for (const auto& b : in) {
        const void* d = mapped(b.host);
        if (d && aligned(d, 16) && b.bytes % 4 == 0 && b.bytes < (1ull << 31)) {
            c.plan.c[c.plan.n++] = StageCopy{d, c.ws + b.off, (uint32_t)b.bytes};
        } else {
            c.copy[c.n_copy].host = b.host;
            c.copy[c.n_copy].off = b.off;
            c.copy[c.n_copy].bytes = b.bytes;
            ++c.n_copy;
        }
    }
    // The selection writes the indices straight into mapped host memory.
    c.indices_host = indices_host;
    c.idx_out = reinterpret_cast<int32_t*>(c.ws + c.H.idx);
    const void* out_map = mapped(indices_host);
    if (out_map && aligned(out_map, 4)) c.idx_out = const_cast<int32_t*>(static_cast<const int32_t*>(out_map));
    return host_launches(c, s);
}

idx_status idx_check_status(void* workspace, void* stream) {
    if (!workspace) return IDX_ERR_WORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint32_t word = 0;
    if (cudaMemcpyAsync(&word, workspace, sizeof word, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess ||
        cudaMemsetAsync(workspace, 0, sizeof word, s) != cudaSuccess) {
        (void)cudaGetLastError();
        return IDX_ERR_CUDA;
    }
    if (word & kStatusTimeout) return IDX_ERR_TIMEOUT;
    if (word & kStatusBounds) return IDX_ERR_BOUNDS;
    return IDX_OK;
}

const char* idx_status_str(int status) {
    switch (status) {
        case IDX_OK: return "ok";
        case IDX_ERR_ARG: return "invalid argument";
        case IDX_ERR_ALIGN: return "misaligned pointer or stride";
        case IDX_ERR_WORKSPACE: return "workspace missing or too small";
        case IDX_ERR_CUDA: return "CUDA error";
        case IDX_ERR_TIMEOUT: return "device wait timed out";
        case IDX_ERR_BOUNDS: return "block-table id or row length out of bounds";
        case IDX_ERR_UNSUPPORTED: return "unsupported device or driver";
        default: return "unknown status";
    }
}

idx_status idx_score_noalloc(int qtype, const void* q, const float* head_w, const uint8_t* k_cache,
                             const float* k_scale, int64_t pool_pages, const int32_t* block_table,
                             int max_pages, const int32_t* seq_lens, const int32_t* row_req, int R,
                             float* scores, int64_t score_stride, void* stream) {
    if (R < 1 || R > IDX_NOALLOC_MAX_ROWS) return IDX_ERR_ARG;  // the static scratch holds this many rows
    // The checks of idx_score, minus the workspace (the scratch array is 256-byte aligned).
    if (qtype != IDX_Q_BF16 && qtype != IDX_Q_E4M3 && qtype != IDX_Q_BF16_FP8) return IDX_ERR_ARG;
    if (!q || !head_w || !k_cache || !k_scale || !block_table || !seq_lens || !row_req) return IDX_ERR_ARG;
    if (pool_pages < 1 || pool_pages > (int64_t(1) << 25)) return IDX_ERR_ARG;
    if (max_pages < 1 || (int64_t)max_pages * kPage > INT32_MAX) return IDX_ERR_ARG;
    if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(k_scale, 16)) return IDX_ERR_ALIGN;
    if (!scores) return IDX_ERR_ARG;
    if (score_stride < 4 || score_stride % 4 != 0) return IDX_ERR_ALIGN;
    if (!aligned(scores, 16)) return IDX_ERR_ALIGN;
    DeviceInfo dev;
    idx_status st = device_info(&dev);
    if (st != IDX_OK) return st;
    char* scratch = nullptr;
    st = noalloc_scratch(&scratch);
    if (st != IDX_OK) return st;
    const WsLayout L = ws_layout(R, score_stride, 0, 0);  // the status word only: the query is split in the kernel
    if (L.end > kNoallocScratchBytes) return IDX_ERR_WORKSPACE;
    ScoreArgs a{qtype, q, head_w, k_cache, k_scale, pool_pages, block_table, max_pages, seq_lens, row_req,
                R, scores, score_stride, score_stride, scratch, L, static_cast<cudaStream_t>(stream), dev.num_sms};
    return run_score(a);
}

int idx_version(void) { return 100; }

}  // extern "C"
