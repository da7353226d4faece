"""The device-timeout path of the scoring kernel, made to run out on purpose
without a fault: a test-only wall-time limit of 1 ms on every wait and the
query-operand hand-off left unsignalled (idx_test_set_wait_limit).  The
kernel must give up, stop every role, drain its own copies and MMAs, release
its tensor memory and record IDX_ERR_TIMEOUT, which idx_check_status returns;
the call must return promptly, and the next normal call on the same stream
must give the oracle's scores and lists."""
import time

import numpy as np
import pytest
import torch

import oracle
from key_scoring_exact_gb300 import binding
from key_scoring_exact_gb300 import workloads as W
from tests import checks
from tests.gpu_util import device_inputs, problem, stride_for

pytestmark = pytest.mark.gpu

TIMEOUT = -5


def _fused(w, t, ws, scores, idx, stream):
    binding.score_topk(t["q"], t["head_w"], t["k_cache"], t["k_scale"], t["block_table"], t["seq_lens"],
                       t["row_req"], w.max_len, w.k, idx, ws, scores=scores, stream=stream)


@pytest.mark.parametrize("qtype_fp8", [False, True])
def test_wait_that_runs_out_is_reported_and_the_next_call_is_exact(qtype_fp8):
    w = W.make_workload([W.chain(3000, 2), [700], W.chain(9000, 4)], "random", seed=91, k=256,
                        q_is_e4m3=qtype_fp8)
    t = device_inputs(w)
    stream = torch.cuda.Stream()
    stride = stride_for(w.max_len)
    ws = binding.new_workspace(w.R, w.max_len, w.k, stream=stream)
    scores = torch.zeros(w.R, stride, dtype=torch.float32, device="cuda")
    idx = torch.full((w.R, w.k), -7, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()

    binding.test_set_wait_limit(1_000_000, drop_query_handoff=True)   # 1 ms, hand-off never signalled
    try:
        t0 = time.perf_counter()
        _fused(w, t, ws, scores, idx, stream)
        st = binding.check_status(ws, stream)          # synchronises the stream
        elapsed = time.perf_counter() - t0
    finally:
        binding.test_set_wait_limit(0, False)
    assert st == TIMEOUT, "status %d, expected IDX_ERR_TIMEOUT" % st
    assert elapsed < 1.0, "the timed-out call took %.3f s" % elapsed

    # the status word was cleared by the read; the next normal call is exact
    scores.zero_()
    _fused(w, t, ws, scores, idx, stream)
    assert binding.check_status(ws, stream) == 0
    s = scores.cpu().numpy()
    ref = oracle.scores(problem(w))
    lens = w.seq_lens.tolist()
    errs = checks.score_errors(s, ref, lens)
    assert max(errs) <= checks.SCORE_TOL, errs
    got = idx.cpu().numpy()
    for r, n in enumerate(lens):
        assert np.array_equal(got[r], oracle.topk(s[r, :n], w.k)), "row %d" % r
