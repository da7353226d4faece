"""The C-ABI library loads on a CPU-only host and exports every entry point
that include/idx.h declares; host-only calls behave as documented."""
import ctypes
import os
import re

import pytest

from key_scoring_exact_gb300 import binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "idx.h")
DIAG_HEADER = os.path.join(ROOT, "include", "idx_diag.h")


def _declared(header=HEADER):
    text = open(header).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(idx_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return ctypes.CDLL(build.LIB)


def test_header_declares_the_api():
    names = _declared()
    for n in ("idx_score", "idx_topk", "idx_score_topk", "idx_workspace_bytes", "idx_check_status"):
        assert n in names
    assert set(names) == set(binding.EXPORTS)


def test_diag_header_declares_the_diagnostics():
    assert set(_declared(DIAG_HEADER)) == set(binding.DIAG_EXPORTS)


def test_every_declared_symbol_is_exported(lib):
    for name in _declared() + _declared(DIAG_HEADER):
        assert hasattr(lib, name), name


def test_diag_argument_errors_need_no_gpu(lib):
    lib.idx_probe_fp8_mma.restype = ctypes.c_int
    p = ctypes.c_void_p
    lib.idx_probe_fp8_mma.argtypes = [ctypes.c_int, ctypes.c_int, p, p, ctypes.c_int, p]
    fake = ctypes.c_void_p(1024)
    assert lib.idx_probe_fp8_mma(4, 256, fake, fake, 200, None) == -1      # too few MMAs
    assert lib.idx_probe_fp8_mma(64, 250, fake, fake, 200, None) == -1     # N not a multiple of 16
    assert lib.idx_probe_fp8_mma(64, 256, None, fake, 200, None) == -1     # null output
    lib.idx_test_set_wait_limit.restype = ctypes.c_int
    lib.idx_test_set_wait_limit.argtypes = [ctypes.c_ulonglong, ctypes.c_int]
    assert lib.idx_test_set_wait_limit(0, 0) == 0


def test_host_only_calls(lib):
    lib.idx_workspace_bytes.restype = ctypes.c_size_t
    lib.idx_workspace_bytes.argtypes = [ctypes.c_int, ctypes.c_int64, ctypes.c_int, ctypes.c_int]
    a = lib.idx_workspace_bytes(4, 131072, 2048, 0)
    b = lib.idx_workspace_bytes(4, 131072, 2048, 1)
    assert a > 0 and b >= a + 4 * 4 * 131072
    assert lib.idx_workspace_bytes(0, 100, 2048, 0) == 0
    lib.idx_status_str.restype = ctypes.c_char_p
    assert lib.idx_status_str(0) == b"ok"
    assert lib.idx_status_str(-6).startswith(b"block-table")
    assert lib.idx_version() >= 100


def test_argument_errors_need_no_gpu(lib):
    lib.idx_topk.restype = ctypes.c_int
    p = ctypes.c_void_p
    lib.idx_topk.argtypes = [p, ctypes.c_int64, p, ctypes.c_int, ctypes.c_int, p, p, ctypes.c_size_t, p]
    assert lib.idx_topk(None, 16, None, 1, 8, None, None, 0, None) == -1       # NULL pointers
    fake = ctypes.c_void_p(1024)
    assert lib.idx_topk(fake, 16, fake, 1, 0, fake, None, 0, None) == -1      # k = 0
    assert lib.idx_topk(fake, 16, fake, 1, 4096, fake, None, 0, None) == -1   # k > 2048
    assert lib.idx_topk(fake, 18, fake, 1, 8, fake, None, 0, None) == -2      # stride % 4


def test_host_entry_sizes_and_argument_errors(lib):
    """The host-buffer fused call: its workspace holds the fused call's
    workspace (scores inside) plus device copies of the inputs and indices;
    null host pointers and sizes out of range are refused before any copy."""
    lib.idx_host_workspace_bytes.restype = ctypes.c_size_t
    lib.idx_host_workspace_bytes.argtypes = [ctypes.c_int, ctypes.c_int64, ctypes.c_int, ctypes.c_int,
                                             ctypes.c_int]
    lib.idx_workspace_bytes.restype = ctypes.c_size_t
    lib.idx_workspace_bytes.argtypes = [ctypes.c_int, ctypes.c_int64, ctypes.c_int, ctypes.c_int]
    h = lib.idx_host_workspace_bytes(4, 131072, 2048, 1, 2048)
    fused = lib.idx_workspace_bytes(4, 131072, 2048, 1)
    inputs = 4 * 64 * 128 * 2 + 4 * 64 * 4 + 2048 * 4 + 2 * 4 * 4 + 4 * 2048 * 4
    assert h >= fused + inputs and h % 1024 == 0
    assert lib.idx_host_workspace_bytes(0, 100, 2048, 1, 2) == 0
    assert lib.idx_host_workspace_bytes(4, 100, 4096, 1, 2) == 0
    assert lib.idx_host_workspace_bytes(4, 100, 2048, 0, 2) == 0
    p, i32, i64, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
    lib.idx_score_topk_host.restype = ctypes.c_int
    lib.idx_score_topk_host.argtypes = [i32, p, p, p, p, i64, p, i32, i32, p, p, i32, i64, i32, p, p, sz, p]
    buf = (ctypes.c_char * 4096)()
    hp = ctypes.cast(buf, p)
    fake = ctypes.c_void_p(1024)
    args = [0, hp, hp, fake, fake, 8, hp, 1, 4, hp, hp, 1, 256, 16, hp, fake, 1 << 30, None]
    bad_q = list(args)
    bad_q[1] = None
    assert lib.idx_score_topk_host(*bad_q) == -1                 # null host query
    bad_k = list(args)
    bad_k[13] = 0
    assert lib.idx_score_topk_host(*bad_k) == -1                 # k = 0
    bad_t = list(args)
    bad_t[0] = 7
    assert lib.idx_score_topk_host(*bad_t) == -1                 # query type
    small = list(args)
    small[16] = 1024
    assert lib.idx_score_topk_host(*small) == -3                 # workspace too small
    odd = list(args)
    odd[15] = ctypes.c_void_p(1024 + 256)
    assert lib.idx_score_topk_host(*odd) == -2                   # workspace alignment
    # the fused call's own checks also run before anything is launched
    kc = list(args)
    kc[3] = ctypes.c_void_p(1024 + 1)
    assert lib.idx_score_topk_host(*kc) == -2                    # key cache alignment
    pool = list(args)
    pool[5] = 0
    assert lib.idx_score_topk_host(*pool) == -1                  # empty page pool
    long_rows = list(args)
    long_rows[8], long_rows[12] = 10000, 600000                  # rows past the selection's 524,288 keys
    assert lib.idx_score_topk_host(*long_rows) == -1


def test_tagged_and_newkeys_argument_errors_need_no_gpu(lib):
    """idx_score_topk_tagged and idx_score_topk_newkeys refuse a null or
    misaligned output or key array before anything is launched."""
    p, i32, i64, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
    common = [i32, p, p, p, p, i64, p, i32, p, p, i32]
    lib.idx_score_topk_tagged.restype = i32
    lib.idx_score_topk_tagged.argtypes = common + [i64, i32, ctypes.c_uint32, i32, p, p, i64, p, sz, p]
    lib.idx_score_topk_newkeys.restype = i32
    lib.idx_score_topk_newkeys.argtypes = common + [p, p, i64, i32, p, p, i64, p, sz, p]
    fake = ctypes.c_void_p(1 << 20)
    base = [0, fake, fake, fake, fake, 8, fake, 4, fake, fake, 2]
    tag = lambda pairs: lib.idx_score_topk_tagged(*base, 256, 16, 7, 0, pairs, None, 0, fake, 1 << 30, None)
    assert tag(None) == -1                               # no output
    assert tag(ctypes.c_void_p((1 << 20) + 4)) == -2     # pairs not 8-byte aligned
    newk = lambda nk, ns: lib.idx_score_topk_newkeys(*base, nk, ns, 256, 16, fake, None, 0, fake, 1 << 30, None)
    assert newk(None, fake) == -1                        # no new keys
    assert newk(fake, None) == -1                        # no new scales
    assert newk(ctypes.c_void_p((1 << 20) + 8), fake) == -2  # keys not 16-byte aligned
    bad_type = list(base)
    bad_type[0] = 9
    assert lib.idx_score_topk_newkeys(*bad_type, fake, fake, 256, 16, fake, None, 0, fake, 1 << 30, None) == -1


def test_ready_entry_point_argument_errors_need_no_gpu(lib):
    """idx_score_topk_ready takes idx_score_topk's arguments and refuses the
    same errors before anything is launched: no output, k out of range, a
    misaligned key cache, a bad query type (the workspace size is checked after
    the device query, as in idx_score_topk)."""
    p, i32, i64, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
    common = [i32, p, p, p, p, i64, p, i32, p, p, i32]
    lib.idx_score_topk_ready.restype = i32
    lib.idx_score_topk_ready.argtypes = common + [i64, i32, p, p, i64, p, sz, p]
    fake = ctypes.c_void_p(1 << 20)
    base = [0, fake, fake, fake, fake, 8, fake, 4, fake, fake, 2]

    def call(b=base, max_len=256, k=16, idx=fake, ws_bytes=1 << 30):
        return lib.idx_score_topk_ready(*b, max_len, k, idx, None, 0, fake, ws_bytes, None)

    assert call(idx=None) == -1                          # no output
    assert call(k=0) == -1 and call(k=4096) == -1        # k outside [1, 2048]
    bad_cache = list(base)
    bad_cache[3] = ctypes.c_void_p((1 << 20) + 1)
    assert call(b=bad_cache) == -2                       # key cache not 16-byte aligned
    bad_type = list(base)
    bad_type[0] = 9
    assert call(b=bad_type) == -1                        # query type
