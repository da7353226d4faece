"""idx_score_topk_ready: the fused call for inputs that are complete when the
call is enqueued.  The scoring launch may then start (plan, block table,
first key pages) while the kernel before it on the stream still runs, so the
tests check every way that overlap could go wrong: scores and lists against
the oracle on configurations 1-4; calls back to back on one stream with the
scores in one shared workspace, each scoring starting while the previous
selection still reads that workspace; a query written by the kernel just
before the call (allowed by the contract); ready and plain calls mixed; two
and sixteen row groups."""
import numpy as np
import pytest
import torch

import oracle
from key_scoring_exact_gb300 import binding
from key_scoring_exact_gb300 import workloads as W
from tests import checks
from tests.gpu_util import device_inputs, gpu_fused, problem, stride_for

pytestmark = pytest.mark.gpu


def _call(w, t, idx, ws, scores=None, stream=None, ready=True):
    binding.score_topk(t["q"], t["head_w"], t["k_cache"], t["k_scale"], t["block_table"], t["seq_lens"],
                       t["row_req"], w.max_len, w.k, idx, ws, scores=scores, stream=stream, inputs_ready=ready)


def _lists_exact(w, s, got):
    for r, n in enumerate(w.seq_lens.tolist()):
        exp = oracle.topk(s[r, :n], w.k)
        assert np.array_equal(got[r], exp), "row %d list differs" % r
        assert checks.list_invariants(got[r], s[r, :n], w.k) == []


@pytest.mark.parametrize("idx", [1, 2, 3, 4])
def test_ready_configs(idx):
    """Every score within 1e-4 of the f64 oracle, every list bit-exact."""
    w = W.make_config(idx)
    t = device_inputs(w)
    scores = torch.zeros(w.R, stride_for(w.max_len), dtype=torch.float32, device="cuda")
    got = torch.full((w.R, w.k), -7, dtype=torch.int32, device="cuda")
    ws = binding.new_workspace(w.R, w.max_len, w.k)
    _call(w, t, got, ws, scores=scores)
    assert binding.check_status(ws) == 0
    s = scores.cpu().numpy()
    errs = checks.score_errors(s, oracle.scores(problem(w)), w.seq_lens.tolist())
    assert max(errs) <= checks.SCORE_TOL, errs
    _lists_exact(w, s, got.cpu().numpy())


def test_ready_chain_shares_a_workspace():
    """Twelve calls back to back on one stream with no synchronisation,
    cycling through three workloads of different shapes, every call's scores
    in one shared workspace: each scoring launch starts while the previous
    selection still reads that workspace, and must not write a score before
    it has finished.  Every call's lists equal its workload's own."""
    loads = [W.make_config(3), W.make_config(4), W.make_config(2)]
    tens = [device_inputs(w) for w in loads]
    refs = []
    for w, t in zip(loads, tens):
        _, ref, st = gpu_fused(w, t, in_workspace=True)
        assert st == 0
        refs.append(ref)
    torch.cuda.synchronize()
    R = max(w.R for w in loads)
    max_len = max(w.max_len for w in loads)
    ws = binding.new_workspace(R, max_len, 2048, with_scores=True)
    stream = torch.cuda.Stream()
    outs = []
    for i in range(12):
        w, t = loads[i % 3], tens[i % 3]
        idx = torch.full((w.R, w.k), -7, dtype=torch.int32, device="cuda")
        _call(w, t, idx, ws, stream=stream)
        outs.append(idx)
    stream.synchronize()
    assert binding.check_status(ws, stream) == 0
    for i, idx in enumerate(outs):
        assert np.array_equal(idx.cpu().numpy(), refs[i % 3]), "call %d" % i


def test_ready_query_from_the_kernel_before():
    """The contract lets the query and head weights come from the kernel just
    before the call: here a copy kernel rewrites both between calls on the
    same stream, and each call's lists equal those of the query it was
    given."""
    w = W.make_config(3)
    t = device_inputs(w)
    variants = []
    g = torch.Generator().manual_seed(31)
    for v in range(3):
        q = (torch.randn(t["q"].shape, generator=g) * (1.0 + v)).to(torch.bfloat16).cuda()
        hw = (torch.rand(t["head_w"].shape, generator=g) / 8).cuda()
        tv = dict(t, q=q, head_w=hw)
        _, ref, st = gpu_fused(w, tv)
        assert st == 0
        variants.append((q, hw, ref))
    torch.cuda.synchronize()
    q_buf = torch.empty_like(t["q"])
    w_buf = torch.empty_like(t["head_w"])
    tb = dict(t, q=q_buf, head_w=w_buf)
    ws = binding.new_workspace(w.R, w.max_len, w.k, with_scores=True)
    stream = torch.cuda.Stream()
    outs = []
    with torch.cuda.stream(stream):
        for i in range(6):
            q, hw, _ = variants[i % 3]
            q_buf.copy_(q)
            w_buf.copy_(hw)
            idx = torch.full((w.R, w.k), -7, dtype=torch.int32, device="cuda")
            _call(w, tb, idx, ws, stream=stream)
            outs.append(idx)
    stream.synchronize()
    assert binding.check_status(ws, stream) == 0
    for i, idx in enumerate(outs):
        assert np.array_equal(idx.cpu().numpy(), variants[i % 3][2]), "call %d" % i


def test_ready_and_plain_calls_mixed():
    """Ready and plain calls alternating on one stream through one workspace
    give the same lists as each other and as the oracle's selection."""
    w = W.make_config(4)
    t = device_inputs(w)
    _, ref, st = gpu_fused(w, t, in_workspace=True)
    assert st == 0
    ws = binding.new_workspace(w.R, w.max_len, w.k, with_scores=True)
    stream = torch.cuda.Stream()
    outs = []
    for i in range(8):
        idx = torch.full((w.R, w.k), -7, dtype=torch.int32, device="cuda")
        _call(w, t, idx, ws, stream=stream, ready=(i % 2 == 0))
        outs.append(idx)
    stream.synchronize()
    assert binding.check_status(ws, stream) == 0
    for i, idx in enumerate(outs):
        assert np.array_equal(idx.cpu().numpy(), ref), "call %d" % i


def test_ready_chain_of_eight_rows():
    """Two row groups of one request through idx_score_topk_ready: every
    score within 1e-4 of the oracle, every list exact."""
    w = W.make_extra("chain8")
    t = device_inputs(w)
    scores = torch.zeros(w.R, stride_for(w.max_len), dtype=torch.float32, device="cuda")
    got = torch.full((w.R, w.k), -7, dtype=torch.int32, device="cuda")
    ws = binding.new_workspace(w.R, w.max_len, w.k)
    _call(w, t, got, ws, scores=scores)
    assert binding.check_status(ws) == 0
    s = scores.cpu().numpy()
    errs = checks.score_errors(s, oracle.scores(problem(w)), w.seq_lens.tolist())
    assert max(errs) <= checks.SCORE_TOL, errs
    _lists_exact(w, s, got.cpu().numpy())


def test_ready_sixteen_requests():
    """16 requests x 4 rows x 131K keys (16 row groups, the selection in two
    waves of clusters) through idx_score_topk_ready, twice back to back on one
    stream: sampled scores within 1e-4 of the oracle, every list exact and the
    same in both calls."""
    w = W.make_config(5)
    t = device_inputs(w)
    scores = torch.zeros(w.R, stride_for(w.max_len), dtype=torch.float32, device="cuda")
    ws = binding.new_workspace(w.R, w.max_len, w.k)
    stream = torch.cuda.Stream()
    outs = []
    for _ in range(2):
        got = torch.full((w.R, w.k), -7, dtype=torch.int32, device="cuda")
        _call(w, t, got, ws, scores=scores, stream=stream)
        outs.append(got)
    stream.synchronize()
    assert binding.check_status(ws, stream) == 0
    s = scores.cpu().numpy()
    pb = problem(w)
    rng = np.random.default_rng(5)
    for r, n in enumerate(w.seq_lens.tolist()):
        pos = np.unique(np.concatenate([[0, 127, 128, n - 1], rng.integers(0, n, 12),
                                        np.argsort(-s[r, :n])[:4]])).astype(np.int64)
        ref = oracle.score_positions(pb, r, pos)
        assert np.max(np.abs(s[r, pos] - ref)) <= checks.SCORE_TOL * np.max(np.abs(ref)), r
    _lists_exact(w, s, outs[0].cpu().numpy())
    assert np.array_equal(outs[0].cpu().numpy(), outs[1].cpu().numpy())
