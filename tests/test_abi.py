"""The C-ABI library loads on a CPU-only host and exports every entry point
that include/idx.h declares; host-only calls behave as documented."""
import ctypes
import os
import re

import pytest

from key_scoring_exact_gb300 import binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "idx.h")


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(idx_[a-z_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return ctypes.CDLL(build.LIB)


def test_header_declares_the_api():
    names = _declared()
    for n in ("idx_score", "idx_topk", "idx_score_topk", "idx_workspace_bytes", "idx_check_status"):
        assert n in names
    assert set(names) == set(binding.EXPORTS)


def test_every_declared_symbol_is_exported(lib):
    for name in _declared():
        assert hasattr(lib, name), name


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
