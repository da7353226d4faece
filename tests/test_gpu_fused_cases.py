"""The fused call (idx_score_topk) on layouts that stress the hand-off between
the scoring's row groups and the selection: every list bit-exact against the
oracle's selection of the GPU's own scores -- rows at and around k in one
group, groups without keys, hundreds of one-row requests (several groups per
scoring CTA), k from 1 to 2048, ties spread over every slice of a row, an
all-tied row, the longest row, and calls of different shapes back to back
through one workspace."""
import numpy as np
import pytest
import torch

import oracle
from key_scoring_exact_gb300 import binding
from key_scoring_exact_gb300 import workloads as W
from tests import checks
from tests.gpu_util import device_inputs, gpu_fused, problem

pytestmark = pytest.mark.gpu


def _lists_exact(w, s, got):
    for r, n in enumerate(w.seq_lens.tolist()):
        exp = oracle.topk(s[r, :n], w.k)
        assert np.array_equal(got[r], exp), "row %d (len %d) list differs" % (r, n)


def _scores_ok(w, s):
    ref = oracle.scores(problem(w))
    errs = checks.score_errors(s, ref, w.seq_lens.tolist())
    assert max(errs) <= checks.SCORE_TOL, errs


@pytest.mark.parametrize("layout", [
    [[2047, 2048, 2049, 6000]],          # rows of one group either side of k
    [[0, 0, 0], [300]],                  # a group without keys
    [[0], [5000], [0, 3000], [1]],       # empty and short rows beside long ones
    [[2048] * 4, [2049] * 3],
])
def test_rows_around_k(layout):
    w = W.make_workload(layout, "random", seed=3 + len(layout))
    s, got, st = gpu_fused(w)
    assert st == 0
    _scores_ok(w, s)
    _lists_exact(w, s, got)


def test_many_groups_per_cta():
    """300 single-row requests of 800 to 3,080 keys (some under k): several
    row groups per scoring CTA, one selection cluster per row."""
    rng = np.random.default_rng(7)
    lens = rng.integers(100, 385, size=300) * 8
    w = W.make_workload([[int(n)] for n in lens], "random", seed=11)
    s, got, st = gpu_fused(w)
    assert st == 0
    _lists_exact(w, s, got)


@pytest.mark.parametrize("k", [1, 7, 100, 2047, 2048])
def test_various_k(k):
    w = W.make_workload([W.chain(20000, 4), [k], [k + 1], [300]], "random", seed=20 + k, k=k)
    s, got, st = gpu_fused(w)
    assert st == 0
    _lists_exact(w, s, got)


def test_all_tied_row_longer_than_the_list():
    """All-zero keys: every score 0 and every key ties, so each list is the
    first k positions in order."""
    w = W.make_workload([[40000, 39000]], "zeros", seed=5)
    s, got, st = gpu_fused(w)
    assert st == 0
    assert np.all(s[0, :40000] == 0.0)
    for r in range(2):
        assert np.array_equal(got[r], np.arange(2048)), r
    _lists_exact(w, s, got)


def test_ties_across_slices():
    """The tie cache at 60K keys: each of 4 values is held by ~15K keys spread
    over every slice of the row; the list takes the first ties in position
    order."""
    w = W.make_workload([W.chain(60000, 4)], "ties", seed=9)
    s, got, st = gpu_fused(w)
    assert st == 0
    _lists_exact(w, s, got)


def test_longest_row():
    """One row of 524,288 keys (the longest the fused call takes) beside a
    short one; scores sampled against the oracle."""
    w = W.make_workload([[524288], [5000]], "random", seed=13)
    s, got, st = gpu_fused(w)
    assert st == 0
    pb = problem(w)
    pos = np.unique(np.concatenate([np.arange(0, 524288, 4099), np.argsort(-s[0, :524288])[:16]]))
    ref = oracle.score_positions(pb, 0, pos.astype(np.int64))
    assert np.max(np.abs(s[0, pos] - ref)) <= checks.SCORE_TOL * np.max(np.abs(ref))
    _lists_exact(w, s, got)


def test_back_to_back_mixed_shapes_one_workspace():
    """Calls of different shapes through one workspace, one after another on
    one stream: each gives its own exact lists."""
    big = W.make_workload([W.chain(30000, 4), [8000], [1000]], "recent", seed=41)
    ws = binding.new_workspace(big.R, big.max_len, big.k)
    cases = [big,
             W.make_workload([[25000, 24000]], "ties", seed=42),
             W.make_workload([[3000], [0], [12000]], "random", seed=43),
             big]
    for i, w in enumerate(cases):
        t = device_inputs(w)
        idx = torch.full((w.R, w.k), -7, dtype=torch.int32, device="cuda")
        sc = torch.zeros(w.R, (big.max_len + 3) // 4 * 4, dtype=torch.float32, device="cuda")
        binding.score_topk(t["q"], t["head_w"], t["k_cache"], t["k_scale"], t["block_table"], t["seq_lens"],
                           t["row_req"], big.max_len, w.k, idx, ws, scores=sc)
        assert binding.check_status(ws) == 0
        _lists_exact(w, sc.cpu().numpy(), idx.cpu().numpy())
