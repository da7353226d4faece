"""CPU oracle for the paged key scoring and exact top-k selection.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package.  The GPU library (``key_scoring_exact_gb300``) never imports it, and
this package imports nothing from the GPU library.

Contents:
  * ``oracle.c`` -- f64 scores by the literal indexer formula and a sort-based
    exact top-k list (see that file's header for the definitions followed);
  * ``brute.py`` -- a pure-Python brute-force selection for tiny inputs.

The C file is compiled with gcc into ``oracle/_build/liboracle.so`` and called
through ctypes with NumPy arrays.  Plain double arithmetic, no fast-math.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_SO = os.path.join(_HERE, "_build", "liboracle.so")
_lock = threading.Lock()
_lib = None

OK, ERR_ARG, ERR_BOUNDS = 0, -1, -6


def build(force: bool = False) -> str:
    """Compile oracle.c into a shared library (C99, -O2, no fast-math)."""
    os.makedirs(os.path.dirname(_SO), exist_ok=True)
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + ".tmp.%d" % os.getpid()
        subprocess.check_call(
            ["gcc", "-std=c99", "-O2", "-fPIC", "-shared", "-fno-fast-math",
             "-ffp-contract=off", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_SO)
            p = ctypes.c_void_p
            i32, i64 = ctypes.c_int32, ctypes.c_int64
            lib.oracle_e4m3_to_f64.restype = ctypes.c_double
            lib.oracle_e4m3_to_f64.argtypes = [ctypes.c_uint8]
            lib.oracle_bf16_to_f64.restype = ctypes.c_double
            lib.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
            common = [i32, p, p, p, p, i64, p, i32, p, p, i32, i32, i32, i32]
            lib.oracle_scores.restype = i32
            lib.oracle_scores.argtypes = common + [p, i64]
            lib.oracle_score_positions.restype = i32
            lib.oracle_score_positions.argtypes = common + [i32, p, i64, p]
            lib.oracle_topk.restype = i32
            lib.oracle_topk.argtypes = [p, i64, i32, p]
            lib.oracle_topk_rows.restype = i32
            lib.oracle_topk_rows.argtypes = [p, i64, p, i32, i32, p]
            lib.oracle_f32_to_e4m3.restype = ctypes.c_uint8
            lib.oracle_f32_to_e4m3.argtypes = [ctypes.c_float]
            lib.oracle_slots.restype = None
            lib.oracle_slots.argtypes = [p, i32, i32, p, i32, p, i32, p]
            lib.oracle_quantize_query.restype = None
            lib.oracle_quantize_query.argtypes = [p, p, i32, i32, i32, p, p]
            lib.oracle_tagged.restype = None
            lib.oracle_tagged.argtypes = [p, i64, ctypes.c_uint32, p]
            lib.oracle_prefix_order.restype = i32
            lib.oracle_prefix_order.argtypes = [p, i64, i32, i64, p]
            lib.oracle_store_keys.restype = i32
            lib.oracle_store_keys.argtypes = [p, p, i64, p, i32, p, p, i32, p, p, i32, i32]
            _lib = lib
    return _lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _c(a, dtype) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a), dtype=dtype)


def e4m3_to_f64(codes) -> np.ndarray:
    """Decode E4M3 codes (any shape of uint8) to float64, one by one."""
    lib = _load()
    c = _c(codes, np.uint8)
    out = np.empty(c.shape, np.float64)
    flat = out.reshape(-1)
    for i, v in enumerate(c.reshape(-1).tolist()):
        flat[i] = lib.oracle_e4m3_to_f64(v)
    return out


def bf16_to_f64(bits) -> np.ndarray:
    """Decode bf16 bit patterns (uint16) to float64, one by one."""
    lib = _load()
    c = _c(bits, np.uint16)
    out = np.empty(c.shape, np.float64)
    flat = out.reshape(-1)
    for i, v in enumerate(c.reshape(-1).tolist()):
        flat[i] = lib.oracle_bf16_to_f64(v)
    return out


def f32_to_e4m3(values) -> np.ndarray:
    """Encode f32 values (any shape) as E4M3 codes, one by one: nearest,
    ties to even, saturated at +-448, NaN to the NaN code."""
    lib = _load()
    c = _c(values, np.float32)
    out = np.empty(c.shape, np.uint8)
    flat = out.reshape(-1)
    for i, v in enumerate(c.reshape(-1).tolist()):
        flat[i] = lib.oracle_f32_to_e4m3(v)
    return out


def quantize_query(q_bits, head_w):
    """FP8 query of a bf16 index query, one scale per (row, head):
    returns (codes [R, H, D] uint8, w' [R, H] float32)."""
    lib = _load()
    q = _c(q_bits, np.uint16)
    w = _c(head_w, np.float32)
    R, H, D = q.shape
    q8 = np.empty(q.shape, np.uint8)
    wo = np.empty((R, H), np.float32)
    lib.oracle_quantize_query(_ptr(q), _ptr(w), R, H, D, _ptr(q8), _ptr(wo))
    return q8, wo


def slots(idx, block_table, row_req, page: int = 64) -> np.ndarray:
    """Logical positions [R, k] (-1 = padding) as physical cache slots."""
    lib = _load()
    i = _c(idx, np.int32)
    bt = _c(block_table, np.int32)
    rr = _c(row_req, np.int32)
    out = np.empty(i.shape, np.int32)
    lib.oracle_slots(_ptr(i), i.shape[0], i.shape[1], _ptr(bt), bt.shape[1], _ptr(rr), int(page), _ptr(out))
    return out


def store_keys(k_cache, k_scale, block_table, seq_lens, row_req, new_k, new_scale, page: int = 64):
    """The cache after the step's stores: row r's key new_k[r] and scale
    new_scale[r] in its slot, position seq_lens[r] - 1 of its request.
    Returns new (k_cache, k_scale) arrays; the inputs are not changed."""
    lib = _load()
    kc = np.array(k_cache, np.uint8, copy=True, order="C")
    ks = np.array(k_scale, np.float32, copy=True, order="C")
    bt = _c(block_table, np.int32)
    ln = _c(seq_lens, np.int32)
    rr = _c(row_req, np.int32)
    nk = _c(new_k, np.uint8)
    ns = _c(new_scale, np.float32)
    st = lib.oracle_store_keys(_ptr(kc), _ptr(ks), kc.shape[0], _ptr(bt), bt.shape[1], _ptr(ln), _ptr(rr),
                               ln.shape[0], _ptr(nk), _ptr(ns), int(page), kc.shape[2])
    if st != OK:
        raise ValueError("oracle_store_keys: a slot's page is outside the pool")
    return kc, ks


def tagged(entries, tag: int) -> np.ndarray:
    """List entries (positions or slots, -1 = padding) as tagged pairs: int64
    words whose low 32 bits hold the entry and whose high 32 bits the tag."""
    lib = _load()
    e = _c(entries, np.int32)
    out = np.empty(e.shape, np.int64)
    lib.oracle_tagged(_ptr(e), e.size, int(tag) & 0xFFFFFFFF, _ptr(out))
    return out


class Problem:
    """The scoring inputs as contiguous NumPy arrays.

    q:            [R, H, D] uint16 (bf16 bits) or uint8 (E4M3 codes)
    head_w:       [R, H] float32
    k_cache:      [pool_pages, P, D] uint8 (E4M3 codes)
    k_scale:      [pool_pages, P] float32
    block_table:  [n_req, max_pages] int32
    seq_lens:     [R] int32   keys visible to each row
    row_req:      [R] int32   request of each row
    """

    def __init__(self, q, q_is_e4m3, head_w, k_cache, k_scale, block_table, seq_lens, row_req):
        self.q_is_e4m3 = bool(q_is_e4m3)
        self.q = _c(q, np.uint8 if q_is_e4m3 else np.uint16)
        self.head_w = _c(head_w, np.float32)
        self.k_cache = _c(k_cache, np.uint8)
        self.k_scale = _c(k_scale, np.float32)
        self.block_table = _c(block_table, np.int32)
        self.seq_lens = _c(seq_lens, np.int32)
        self.row_req = _c(row_req, np.int32)
        self.R, self.H, self.D = self.q.shape
        self.P = self.k_cache.shape[1]
        assert self.k_cache.shape[2] == self.D
        assert self.head_w.shape == (self.R, self.H)
        assert self.k_scale.shape == self.k_cache.shape[:2]

    def _common(self):
        return [int(self.q_is_e4m3), _ptr(self.q), _ptr(self.head_w), _ptr(self.k_cache),
                _ptr(self.k_scale), int(self.k_cache.shape[0]), _ptr(self.block_table),
                int(self.block_table.shape[1]), _ptr(self.seq_lens), _ptr(self.row_req),
                self.R, self.H, self.D, self.P]


def scores(pb: Problem) -> np.ndarray:
    """f64 scores [R, max(seq_lens)]; entries at j >= seq_lens[r] are NaN."""
    lib = _load()
    width = int(pb.seq_lens.max()) if pb.R else 0
    out = np.full((pb.R, max(width, 1)), np.nan, np.float64)
    st = lib.oracle_scores(*pb._common(), _ptr(out), out.shape[1])
    if st != OK:
        raise ValueError("oracle_scores failed with status %d" % st)
    return out[:, :width]


def score_positions(pb: Problem, row: int, positions) -> np.ndarray:
    """f64 scores of one row at the given key positions."""
    lib = _load()
    pos = _c(positions, np.int64)
    out = np.empty(pos.shape[0], np.float64)
    st = lib.oracle_score_positions(*pb._common(), int(row), _ptr(pos), pos.shape[0], _ptr(out))
    if st != OK:
        raise ValueError("oracle_score_positions failed with status %d" % st)
    return out


def topk(row_scores, k: int) -> np.ndarray:
    """Exact top-k list of one row of f32 scores (all of them count)."""
    lib = _load()
    s = _c(row_scores, np.float32)
    out = np.empty(k, np.int32)
    st = lib.oracle_topk(_ptr(s), s.shape[0], int(k), _ptr(out))
    if st != OK:
        raise ValueError("oracle_topk failed with status %d" % st)
    return out


def prefix_order(row_scores, k: int, room: int) -> np.ndarray:
    """One row's list in the pages' prefix order: the radix stops at the
    threshold's 12- or 24-bit prefix once the row's keys sharing it number at
    most `room`, else at 32 bits (oracle_topk's order)."""
    lib = _load()
    s = _c(row_scores, np.float32)
    out = np.empty(k, np.int32)
    st = lib.oracle_prefix_order(_ptr(s), s.shape[0], int(k), int(room), _ptr(out))
    if st != OK:
        raise ValueError("oracle_prefix_order failed with status %d" % st)
    return out


def topk_rows(scores_2d, lens, k: int) -> np.ndarray:
    """Exact top-k lists [R, k] of rows of an f32 matrix with per-row lengths."""
    lib = _load()
    s = _c(scores_2d, np.float32)
    ln = _c(lens, np.int32)
    R = ln.shape[0]
    assert s.shape[0] == R and (R == 0 or int(ln.max(initial=0)) <= s.shape[1])
    out = np.empty((R, k), np.int32)
    st = lib.oracle_topk_rows(_ptr(s), s.shape[1], _ptr(ln), R, int(k), _ptr(out))
    if st != OK:
        raise ValueError("oracle_topk_rows failed with status %d" % st)
    return out
