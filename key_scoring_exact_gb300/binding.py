"""ctypes binding of libidx.so (include/idx.h), for torch CUDA tensors.

Argument marshalling only: every function checks dtypes, devices and shapes,
passes raw device pointers and the current CUDA stream, and turns a non-zero
status into an exception.  All computation happens in the library's kernels;
there is no CPU fallback, and loading fails loudly when the library is missing.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

HEADS, DIM, PAGE, MAX_K, MAX_ROWS, GROUP_ROWS = 64, 128, 64, 2048, 1024, 4
Q_BF16, Q_E4M3, Q_BF16_FP8 = 0, 1, 2
OK = 0
STATUS = {0: "IDX_OK", -1: "IDX_ERR_ARG", -2: "IDX_ERR_ALIGN", -3: "IDX_ERR_WORKSPACE",
          -4: "IDX_ERR_CUDA", -5: "IDX_ERR_TIMEOUT", -6: "IDX_ERR_BOUNDS", -7: "IDX_ERR_UNSUPPORTED"}

EXPORTS = ("idx_workspace_bytes", "idx_workspace_init", "idx_score", "idx_topk", "idx_score_topk",
           "idx_check_status", "idx_status_str", "idx_version", "idx_score_noalloc",
           "idx_host_workspace_bytes", "idx_score_topk_host", "idx_quantize_query", "idx_score_topk_slots",
           "idx_score_topk_tagged", "idx_score_topk_newkeys", "idx_score_topk_prefix_order",
           "idx_score_topk_ready")
DIAG_EXPORTS = ("idx_probe_fp8_mma", "idx_test_set_wait_limit")   # include/idx_diag.h

_lib = None


class IdxError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__("%s failed: %s (%d)" % (where, STATUS.get(status, "?"), status))


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = False) -> ctypes.CDLL:
    """Load libidx.so (optionally building it first). Raises if it is absent."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.LIB
    if not os.path.exists(path):
        if not build_if_missing:
            raise ImportError("libidx.so is not built (%s); run key_scoring_exact_gb300.build.build()" % path)
        _build.build()
    lib = ctypes.CDLL(path)
    p, i32, i64, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
    lib.idx_workspace_bytes.restype = sz
    lib.idx_workspace_bytes.argtypes = [i32, i64, i32, i32]
    lib.idx_workspace_init.restype = i32
    lib.idx_workspace_init.argtypes = [p, sz, p]
    score_common = [i32, p, p, p, p, i64, p, i32, p, p, i32]
    lib.idx_score.restype = i32
    lib.idx_score.argtypes = score_common + [p, i64, p, sz, p]
    lib.idx_topk.restype = i32
    lib.idx_topk.argtypes = [p, i64, p, i32, i32, p, p, sz, p]
    lib.idx_score_topk.restype = i32
    lib.idx_score_topk.argtypes = score_common + [i64, i32, p, p, i64, p, sz, p]
    lib.idx_score_topk_slots.restype = i32
    lib.idx_score_topk_slots.argtypes = score_common + [i64, i32, p, p, i64, p, sz, p]
    lib.idx_score_topk_ready.restype = i32
    lib.idx_score_topk_ready.argtypes = score_common + [i64, i32, p, p, i64, p, sz, p]
    lib.idx_score_topk_prefix_order.restype = i32
    lib.idx_score_topk_prefix_order.argtypes = score_common + [i64, i32, i64, p, p, i64, p, sz, p]
    lib.idx_score_topk_newkeys.restype = i32
    lib.idx_score_topk_newkeys.argtypes = score_common + [p, p, i64, i32, p, p, i64, p, sz, p]
    lib.idx_score_topk_tagged.restype = i32
    lib.idx_score_topk_tagged.argtypes = score_common + [i64, i32, ctypes.c_uint32, i32, p, p, i64, p, sz, p]
    lib.idx_check_status.restype = i32
    lib.idx_check_status.argtypes = [p, p]
    lib.idx_status_str.restype = ctypes.c_char_p
    lib.idx_status_str.argtypes = [i32]
    lib.idx_version.restype = i32
    lib.idx_version.argtypes = []
    lib.idx_score_noalloc.restype = i32
    lib.idx_score_noalloc.argtypes = score_common + [p, i64, p]
    lib.idx_quantize_query.restype = i32
    lib.idx_quantize_query.argtypes = [p, p, i32, p, p, p]
    lib.idx_host_workspace_bytes.restype = sz
    lib.idx_host_workspace_bytes.argtypes = [i32, i64, i32, i32, i32]
    lib.idx_score_topk_host.restype = i32
    lib.idx_score_topk_host.argtypes = [i32, p, p, p, p, i64, p, i32, i32, p, p, i32, i64, i32, p, p, sz, p]
    lib.idx_probe_fp8_mma.restype = i32
    lib.idx_probe_fp8_mma.argtypes = [i32, i32, p, p, i32, p]
    lib.idx_test_set_wait_limit.restype = i32
    lib.idx_test_set_wait_limit.argtypes = [ctypes.c_ulonglong, i32]
    _lib = lib
    return lib


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _dev(t: torch.Tensor, name: str, dtype=None) -> int:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if dtype is not None and t.dtype not in (dtype if isinstance(dtype, tuple) else (dtype,)):
        raise ValueError("%s has dtype %s" % (name, t.dtype))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    return t.data_ptr()


def _check(st: int, where: str) -> None:
    if st != OK:
        raise IdxError(st, where)


def workspace_bytes(R: int, max_len: int, k: int = MAX_K, with_scores: bool = False) -> int:
    return int(load().idx_workspace_bytes(int(R), int(max_len), int(k), 1 if with_scores else 0))


def new_workspace(R: int, max_len: int, k: int = MAX_K, with_scores: bool = False,
                  device=None, stream=None) -> torch.Tensor:
    """A zero-initialised, 1024-byte aligned workspace tensor (allocated by torch)."""
    n = workspace_bytes(R, max_len, k, with_scores)
    if n == 0:
        raise ValueError("invalid workspace request")
    raw = torch.zeros(n + 1024, dtype=torch.uint8, device=device or "cuda")
    off = (-raw.data_ptr()) % 1024
    ws = raw[off:off + n]
    _check(load().idx_workspace_init(ws.data_ptr(), n, _stream(stream)), "idx_workspace_init")
    return ws


def _qtype(q: torch.Tensor, quantize_q: bool = False) -> int:
    if q.dtype == torch.bfloat16:
        return Q_BF16_FP8 if quantize_q else Q_BF16
    if q.dtype in (torch.uint8, torch.float8_e4m3fn):
        if quantize_q:
            raise ValueError("quantize_q needs a bfloat16 query")
        return Q_E4M3
    raise ValueError("q must be bfloat16 or E4M3 (uint8 / float8_e4m3fn)")


def quantize_query(q, head_w, q8=None, w_out=None, stream=None):
    """idx_quantize_query: the FP8 query of a bf16 query [R, 64, 128], one
    scale per (row, head) folded into the head weights.  Returns (q8 uint8
    [R, 64, 128], w_out f32 [R, 64])."""
    R = q.shape[0]
    if q.dtype != torch.bfloat16 or tuple(q.shape) != (R, HEADS, DIM) or tuple(head_w.shape) != (R, HEADS):
        raise ValueError("q must be bfloat16 [R, 64, 128] and head_w [R, 64]")
    q8 = q8 if q8 is not None else torch.empty(q.shape, dtype=torch.uint8, device=q.device)
    w_out = w_out if w_out is not None else torch.empty(head_w.shape, dtype=torch.float32, device=q.device)
    st = load().idx_quantize_query(_dev(q, "q", torch.bfloat16), _dev(head_w, "head_w", torch.float32), int(R),
                                   _dev(q8, "q8", torch.uint8), _dev(w_out, "w_out", torch.float32),
                                   _stream(stream))
    _check(st, "idx_quantize_query")
    return q8, w_out


def _score_common(q, head_w, k_cache, k_scale, block_table, seq_lens, row_req, quantize_q=False):
    R = q.shape[0]
    if tuple(q.shape) != (R, HEADS, DIM) or tuple(head_w.shape) != (R, HEADS):
        raise ValueError("q must be [R, 64, 128] and head_w [R, 64]")
    if k_cache.dim() != 3 or tuple(k_cache.shape[1:]) != (PAGE, DIM):
        raise ValueError("k_cache must be [pool_pages, 64, 128]")
    if tuple(k_scale.shape) != tuple(k_cache.shape[:2]):
        raise ValueError("k_scale must be [pool_pages, 64]")
    if block_table.dim() != 2 or seq_lens.shape != (R,) or row_req.shape != (R,):
        raise ValueError("block_table [n_req, max_pages], seq_lens [R], row_req [R]")
    return [_qtype(q, quantize_q), _dev(q, "q"), _dev(head_w, "head_w", torch.float32),
            _dev(k_cache, "k_cache", (torch.uint8, torch.float8_e4m3fn)),
            _dev(k_scale, "k_scale", torch.float32), int(k_cache.shape[0]),
            _dev(block_table, "block_table", torch.int32), int(block_table.shape[1]),
            _dev(seq_lens, "seq_lens", torch.int32), _dev(row_req, "row_req", torch.int32), int(R)]


def score(q, head_w, k_cache, k_scale, block_table, seq_lens, row_req, scores, workspace, stream=None,
          quantize_q=False):
    """idx_score: scores[r, j] for j < seq_lens[r] (f32 [R, stride], stride % 4 == 0).
    quantize_q: score the on-device FP8 quantisation of a bf16 query."""
    args = _score_common(q, head_w, k_cache, k_scale, block_table, seq_lens, row_req, quantize_q)
    if scores.dim() != 2 or scores.shape[0] != q.shape[0]:
        raise ValueError("scores must be [R, stride]")
    st = load().idx_score(*args, _dev(scores, "scores", torch.float32), int(scores.shape[1]),
                          _dev(workspace, "workspace", torch.uint8), workspace.numel(), _stream(stream))
    _check(st, "idx_score")


def score_noalloc(q, head_w, k_cache, k_scale, block_table, seq_lens, row_req, scores, stream=None):
    """idx_score_noalloc: idx_score without a workspace, for callers that
    cannot allocate; it uses the library's one static scratch array (its
    status word), and device-side bounds problems are not reported."""
    args = _score_common(q, head_w, k_cache, k_scale, block_table, seq_lens, row_req)
    if scores.dim() != 2 or scores.shape[0] != q.shape[0]:
        raise ValueError("scores must be [R, stride]")
    st = load().idx_score_noalloc(*args, _dev(scores, "scores", torch.float32), int(scores.shape[1]),
                                  _stream(stream))
    _check(st, "idx_score_noalloc")


def topk(scores, row_lens, k, indices, workspace=None, stream=None):
    """idx_topk: indices[r] = exact top-k list of scores[r, :row_lens[r]]."""
    R = scores.shape[0]
    if indices.shape != (R, k):
        raise ValueError("indices must be [R, k]")
    ws = _dev(workspace, "workspace", torch.uint8) if workspace is not None else None
    st = load().idx_topk(_dev(scores, "scores", torch.float32), int(scores.shape[1]),
                         _dev(row_lens, "row_lens", torch.int32), int(R), int(k),
                         _dev(indices, "indices", torch.int32), ws,
                         workspace.numel() if workspace is not None else 0, _stream(stream))
    _check(st, "idx_topk")


def score_topk(q, head_w, k_cache, k_scale, block_table, seq_lens, row_req, max_len, k, indices,
               workspace, scores=None, stream=None, quantize_q=False, slots=False, inputs_ready=False):
    """idx_score_topk: scoring then selection on one stream.  With scores=None
    the scores live in the workspace (size it with with_scores=True).
    quantize_q: score the on-device FP8 quantisation of a bf16 query.
    slots: the lists hold physical cache slots (idx_score_topk_slots).
    inputs_ready: idx_score_topk_ready -- the block table, lengths, row map,
    key cache and scales are complete when the call is enqueued (no running
    kernel writes them), so the scoring's set-up overlaps the kernel before."""
    if slots and inputs_ready:
        raise ValueError("slots and inputs_ready are separate entry points")
    args = _score_common(q, head_w, k_cache, k_scale, block_table, seq_lens, row_req, quantize_q)
    if indices.shape != (q.shape[0], k):
        raise ValueError("indices must be [R, k]")
    sp = _dev(scores, "scores", torch.float32) if scores is not None else None
    stride = int(scores.shape[1]) if scores is not None else 0
    name = "idx_score_topk_slots" if slots else ("idx_score_topk_ready" if inputs_ready else "idx_score_topk")
    st = getattr(load(), name)(*args, int(max_len), int(k), _dev(indices, "indices", torch.int32), sp,
                               stride, _dev(workspace, "workspace", torch.uint8), workspace.numel(),
                               _stream(stream))
    _check(st, name)


def score_topk_tagged(q, head_w, k_cache, k_scale, block_table, seq_lens, row_req, max_len, k, tag, pairs,
                      workspace, scores=None, stream=None, quantize_q=False, slots=False):
    """idx_score_topk_tagged: as score_topk, the lists written into `pairs`
    ([R, k] int64) as tagged pairs (tag << 32) | uint32(entry)."""
    args = _score_common(q, head_w, k_cache, k_scale, block_table, seq_lens, row_req, quantize_q)
    if pairs.shape != (q.shape[0], k):
        raise ValueError("pairs must be [R, k]")
    sp = _dev(scores, "scores", torch.float32) if scores is not None else None
    stride = int(scores.shape[1]) if scores is not None else 0
    st = load().idx_score_topk_tagged(*args, int(max_len), int(k), int(tag) & 0xFFFFFFFF, 1 if slots else 0,
                                      _dev(pairs, "pairs", torch.int64), sp, stride,
                                      _dev(workspace, "workspace", torch.uint8), workspace.numel(), _stream(stream))
    _check(st, "idx_score_topk_tagged")


def score_topk_prefix_order(q, head_w, k_cache, k_scale, block_table, seq_lens, row_req, max_len, k, room, indices,
                            workspace, scores=None, stream=None, quantize_q=False):
    """idx_score_topk_prefix_order: as score_topk, each list in the pages'
    prefix order for candidate room `room`."""
    args = _score_common(q, head_w, k_cache, k_scale, block_table, seq_lens, row_req, quantize_q)
    if indices.shape != (q.shape[0], k):
        raise ValueError("indices must be [R, k]")
    sp = _dev(scores, "scores", torch.float32) if scores is not None else None
    stride = int(scores.shape[1]) if scores is not None else 0
    st = load().idx_score_topk_prefix_order(*args, int(max_len), int(k), int(room),
                                            _dev(indices, "indices", torch.int32), sp, stride,
                                            _dev(workspace, "workspace", torch.uint8), workspace.numel(),
                                            _stream(stream))
    _check(st, "idx_score_topk_prefix_order")


def score_topk_newkeys(q, head_w, k_cache, k_scale, block_table, seq_lens, row_req, new_k, new_scale, max_len, k,
                       indices, workspace, scores=None, stream=None, quantize_q=False):
    """idx_score_topk_newkeys: as score_topk, after storing row r's new key
    new_k[r] ([R, 128] E4M3 codes) and scale new_scale[r] in its own slot
    (position seq_lens[r] - 1 of its request); k_cache and k_scale are written."""
    args = _score_common(q, head_w, k_cache, k_scale, block_table, seq_lens, row_req, quantize_q)
    R = q.shape[0]
    if tuple(new_k.shape) != (R, DIM) or tuple(new_scale.shape) != (R,) or indices.shape != (R, k):
        raise ValueError("new_k must be [R, 128], new_scale [R], indices [R, k]")
    sp = _dev(scores, "scores", torch.float32) if scores is not None else None
    stride = int(scores.shape[1]) if scores is not None else 0
    st = load().idx_score_topk_newkeys(*args, _dev(new_k, "new_k", (torch.uint8, torch.float8_e4m3fn)),
                                       _dev(new_scale, "new_scale", torch.float32), int(max_len), int(k),
                                       _dev(indices, "indices", torch.int32), sp, stride,
                                       _dev(workspace, "workspace", torch.uint8), workspace.numel(), _stream(stream))
    _check(st, "idx_score_topk_newkeys")


def host_workspace_bytes(R: int, max_len: int, k: int, n_req: int, max_pages: int) -> int:
    return int(load().idx_host_workspace_bytes(int(R), int(max_len), int(k), int(n_req), int(max_pages)))


def new_host_workspace(R: int, max_len: int, k: int, n_req: int, max_pages: int, device=None,
                       stream=None) -> torch.Tensor:
    """A zero-initialised, 1024-byte aligned workspace for score_topk_host."""
    n = host_workspace_bytes(R, max_len, k, n_req, max_pages)
    if n == 0:
        raise ValueError("invalid workspace request")
    raw = torch.zeros(n + 1024, dtype=torch.uint8, device=device or "cuda")
    off = (-raw.data_ptr()) % 1024
    ws = raw[off:off + n]
    _check(load().idx_workspace_init(ws.data_ptr(), n, _stream(stream)), "idx_workspace_init")
    return ws


def _host(t: torch.Tensor, name: str, dtype=None) -> int:
    if not isinstance(t, torch.Tensor) or t.is_cuda:
        raise ValueError("%s must be a host (CPU) tensor" % name)
    if dtype is not None and t.dtype not in (dtype if isinstance(dtype, tuple) else (dtype,)):
        raise ValueError("%s has dtype %s" % (name, t.dtype))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    return t.data_ptr()


def score_topk_host(q, head_w, k_cache, k_scale, block_table, seq_lens, row_req, max_len, k, indices,
                    workspace, stream=None, quantize_q=False):
    """idx_score_topk_host: q, head_w, block_table, seq_lens, row_req and the
    [R, k] indices are host tensors (pin them for asynchronous copies); the
    key cache, its scales and the workspace are device tensors.  Asynchronous:
    read `indices` after synchronising the stream."""
    R = q.shape[0]
    if tuple(q.shape) != (R, HEADS, DIM) or tuple(head_w.shape) != (R, HEADS):
        raise ValueError("q must be [R, 64, 128] and head_w [R, 64]")
    if k_cache.dim() != 3 or tuple(k_cache.shape[1:]) != (PAGE, DIM) or tuple(k_scale.shape) != tuple(k_cache.shape[:2]):
        raise ValueError("k_cache must be [pool_pages, 64, 128] and k_scale [pool_pages, 64]")
    if block_table.dim() != 2 or seq_lens.shape != (R,) or row_req.shape != (R,) or indices.shape != (R, k):
        raise ValueError("block_table [n_req, max_pages], seq_lens/row_req [R], indices [R, k]")
    st = load().idx_score_topk_host(
        _qtype(q, quantize_q), _host(q, "q"), _host(head_w, "head_w", torch.float32),
        _dev(k_cache, "k_cache", (torch.uint8, torch.float8_e4m3fn)), _dev(k_scale, "k_scale", torch.float32),
        int(k_cache.shape[0]), _host(block_table, "block_table", torch.int32), int(block_table.shape[0]),
        int(block_table.shape[1]), _host(seq_lens, "seq_lens", torch.int32), _host(row_req, "row_req", torch.int32),
        int(R), int(max_len), int(k), _host(indices, "indices", torch.int32),
        _dev(workspace, "workspace", torch.uint8), workspace.numel(), _stream(stream))
    _check(st, "idx_score_topk_host")


def check_status(workspace, stream=None) -> int:
    """Synchronise the stream and return (and clear) the device status."""
    return int(load().idx_check_status(_dev(workspace, "workspace", torch.uint8), _stream(stream)))


def scores_view(workspace: torch.Tensor, R: int, max_len: int) -> torch.Tensor:
    """The [R, stride] f32 score matrix that idx_score_topk keeps in the
    workspace when called with scores=None (layout of idx_workspace_bytes)."""
    lib = load()
    no_scores = int(lib.idx_workspace_bytes(int(R), int(max_len), 1, 0))
    stride = max(4, (int(max_len) + 3) // 4 * 4)
    n = R * stride
    return workspace[no_scores:no_scores + 4 * n].view(torch.float32).view(R, stride)


def probe_fp8_mma(n_mma: int = 8192, n_cols: int = 256, stream=None) -> dict:
    """idx_probe_fp8_mma: back-to-back tcgen05 FP8 MMAs (M = 128, N = n_cols,
    K = 32) on every SM; returns the device's rate and the per-MMA time."""
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    ns = torch.zeros(sms, dtype=torch.int64, device="cuda")
    clk = torch.zeros(sms, dtype=torch.int64, device="cuda")
    _check(load().idx_probe_fp8_mma(int(n_mma), int(n_cols), ns.data_ptr(), clk.data_ptr(), sms, _stream(stream)),
           "idx_probe_fp8_mma")
    torch.cuda.synchronize()
    ns_h, clk_h = ns.cpu().tolist(), clk.cpu().tolist()
    if min(ns_h) <= 0:
        raise RuntimeError("idx_probe_fp8_mma: a CTA's wait gave up")
    worst = max(ns_h)
    flops = 2.0 * 128 * n_cols * 32 * n_mma * sms
    return {"tflops": flops / (worst * 1e-9) / 1e12, "ns_per_mma": worst / n_mma,
            "clk_per_mma": max(clk_h) / n_mma, "sms": sms, "n_mma": n_mma, "n_cols": n_cols,
            "mhz": max(clk_h) / worst * 1e3}


def test_set_wait_limit(wait_ns: int, drop_query_handoff: bool = False) -> None:
    """idx_test_set_wait_limit (test only): this thread's later scoring
    launches give up waiting after wait_ns (0 = the normal 2 s); with
    drop_query_handoff the kernel's query hand-off is never signalled."""
    _check(load().idx_test_set_wait_limit(int(wait_ns), 1 if drop_query_handoff else 0), "idx_test_set_wait_limit")
