"""idx_score_noalloc: scoring for callers that cannot allocate device memory.

Some callers cannot call cudaMalloc or size a workspace: a serving loop that
replays a captured CUDA graph, an embedding without a device allocator, or code
running under a memory pool that forbids new allocations.  idx_score_noalloc
serves them from one scratch array the library declares statically.  This
test calls it through the C ABI twice in a row and checks each result against
idx_score (the workspace entry point) within the score tolerance the other
tests use.  It lives in a file of its own, collected last, and passes both
alone in a fresh process and after the rest of the suite.
"""
import numpy as np
import pytest
import torch

from key_scoring_exact_gb300 import binding
from key_scoring_exact_gb300 import workloads as W
from tests import checks
from tests.gpu_util import device_inputs, stride_for

pytestmark = pytest.mark.gpu


def _row_errors(a, b, lens):
    return [checks.row_score_error(a[r, :n], b[r, :n].astype(np.float64)) for r, n in enumerate(lens)]


def test_noalloc_matches_workspace_entry_point_twice():
    lib = binding.load()
    cases = [W.make_workload([W.chain(5000), [3000], [130]], "random", seed=71),
             W.make_workload([W.chain(2000, 4) for _ in range(3)], "recent", seed=72, recent_keys=300)]
    for w in cases:
        t = device_inputs(w)
        lens = w.seq_lens.tolist()
        stride = stride_for(w.max_len)
        ref = torch.zeros(w.R, stride, dtype=torch.float32, device="cuda")
        ws = binding.new_workspace(w.R, stride)
        binding.score(t["q"], t["head_w"], t["k_cache"], t["k_scale"], t["block_table"], t["seq_lens"],
                      t["row_req"], ref, ws)
        assert binding.check_status(ws) == 0
        refn = ref.cpu().numpy()
        for call in range(2):
            out = torch.full((w.R, stride), -1.0, dtype=torch.float32, device="cuda")
            st = lib.idx_score_noalloc(
                0, t["q"].data_ptr(), t["head_w"].data_ptr(), t["k_cache"].data_ptr(),
                t["k_scale"].data_ptr(), w.pool_pages, t["block_table"].data_ptr(), w.max_pages,
                t["seq_lens"].data_ptr(), t["row_req"].data_ptr(), w.R, out.data_ptr(), stride,
                torch.cuda.current_stream().cuda_stream)
            assert st == 0, "call %d returned %d" % (call, st)
            torch.cuda.synchronize()
            errs = _row_errors(out.cpu().numpy(), refn, lens)
            assert max(errs) <= checks.SCORE_TOL, (call, errs)


def test_noalloc_rejects_too_many_rows():
    lib = binding.load()
    w = W.make_workload([[4] for _ in range(binding.MAX_ROWS + 1)], "random", seed=73)
    t = device_inputs(w)
    out = torch.zeros(w.R, 100, dtype=torch.float32, device="cuda")
    st = lib.idx_score_noalloc(0, t["q"].data_ptr(), t["head_w"].data_ptr(), t["k_cache"].data_ptr(),
                               t["k_scale"].data_ptr(), w.pool_pages, t["block_table"].data_ptr(),
                               w.max_pages, t["seq_lens"].data_ptr(), t["row_req"].data_ptr(), w.R,
                               out.data_ptr(), 100, torch.cuda.current_stream().cuda_stream)
    assert st == -1  # IDX_ERR_ARG: more rows than the entry point takes
