"""GPU scoring (idx_score) against the f64 oracle.

Bound (from "sgl-amd-mono-upstream PR 18", section "Modifications / 0. An
exact top-k check"): per row, max |gpu - f64| <= 1e-4 * max |f64|; an
all-zero reference row must come out exactly zero.  Covers request layouts
(1..9 rows, groups split at 4 rows, interleaved requests), ragged lengths at
page / tile boundaries, the E4M3 query path, the tie / zero / recent caches,
untouched entries past each row's length, bad block-table ids and run-to-run
determinism."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from key_scoring_exact_gb300 import binding
from key_scoring_exact_gb300 import workloads as W
from tests import checks
from tests.gpu_util import device_inputs, gpu_scores, problem, stride_for

pytestmark = pytest.mark.gpu

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "ragged_lengths.json")))
SENTINEL = -12345.0


def _assert_scores(w, s):
    ref = oracle.scores(problem(w))
    lens = w.seq_lens.tolist()
    errs = checks.score_errors(s, ref, lens)
    worst = max(errs) if errs else 0.0
    assert worst <= checks.SCORE_TOL, "worst row error %.3g (rows %s)" % (worst, errs)
    for r, n in enumerate(lens):
        assert np.all(s[r, n:] == SENTINEL), "row %d: entries past its length were written" % r
    return worst


def test_single_row_small():
    w = W.make_workload([[300]], "random", seed=1)
    s, st = gpu_scores(w, sentinel=SENTINEL)
    assert st == 0
    _assert_scores(w, s)


@pytest.mark.parametrize("layout", [
    [[1000]],
    [[1000, 999]],
    [W.chain(1500, 3)],
    [W.chain(2000, 4)],
    [W.chain(2000, 5)],                 # split into groups of 4 + 1
    [W.chain(700, 9)],                  # 4 + 4 + 1
    [[900], W.chain(1200, 4), [64], [65, 1]],
])
def test_request_layouts(layout):
    w = W.make_workload(layout, "random", seed=len(layout) * 7 + sum(map(len, layout)))
    s, st = gpu_scores(w, sentinel=SENTINEL)
    assert st == 0
    _assert_scores(w, s)


def test_interleaved_requests():
    # Rows of one request that are not adjacent score in separate groups.
    w = W.make_workload([[500], [800]], "random", seed=4)
    perm = torch.tensor([0, 1, 0, 1], dtype=torch.long)
    w.q = torch.cat([w.q, w.q.flip(0)])
    w.head_w = torch.cat([w.head_w, w.head_w.flip(0)])
    w.seq_lens = w.seq_lens[perm].clone()
    w.row_req = w.row_req[perm].clone()
    s, st = gpu_scores(w, sentinel=SENTINEL)
    assert st == 0
    _assert_scores(w, s)


@pytest.mark.parametrize("n", sorted(set(GOLDEN["page_boundary"][:6] + GOLDEN["tile_boundary"])))
def test_ragged_lengths(n):
    w = W.make_workload([[n, max(1, n - 1)]], "random", seed=n)
    s, st = gpu_scores(w, sentinel=SENTINEL)
    assert st == 0
    _assert_scores(w, s)


@pytest.mark.parametrize("cache", ["ties", "zeros", "recent"])
def test_caches(cache):
    w = W.make_workload([W.chain(5000)], cache, seed=21, recent_keys=1000)
    s, st = gpu_scores(w, sentinel=SENTINEL)
    assert st == 0
    _assert_scores(w, s)
    if cache == "zeros":
        for r, n in enumerate(w.seq_lens.tolist()):
            assert np.all(s[r, :n] == 0.0) and not np.any(np.signbit(s[r, :n]))


def test_e4m3_query():
    w = W.make_workload([W.chain(3000), [777]], "random", seed=8, q_is_e4m3=True)
    s, st = gpu_scores(w, sentinel=SENTINEL)
    assert st == 0
    _assert_scores(w, s)


def test_config1_full():
    w = W.make_config(1)
    s, st = gpu_scores(w, sentinel=SENTINEL)
    assert st == 0
    worst = _assert_scores(w, s)
    print("1 row x 4,096 keys: worst relative score error %.3g" % worst)


def test_bad_block_id_is_reported():
    w = W.make_workload([[300]], "random", seed=2)
    w.block_table[0, 1] = w.pool_pages + 5
    s, st = gpu_scores(w, sentinel=SENTINEL)
    assert st == -6  # IDX_ERR_BOUNDS


def test_row_longer_than_block_table_is_reported():
    w = W.make_workload([[300]], "random", seed=2)
    w.seq_lens[0] = w.max_pages * 64 + 10
    t = device_inputs(w)
    scores = torch.full((1, stride_for(w.max_pages * 64 + 10)), SENTINEL, device="cuda")
    ws = binding.new_workspace(1, scores.shape[1])
    binding.score(t["q"], t["head_w"], t["k_cache"], t["k_scale"], t["block_table"], t["seq_lens"],
                  t["row_req"], scores, ws)
    assert binding.check_status(ws) == -6


def test_deterministic():
    w = W.make_workload([W.chain(4000), [2500]], "random", seed=6)
    t = device_inputs(w)
    a, _ = gpu_scores(w, t)
    for _ in range(3):
        b, _ = gpu_scores(w, t)
        assert np.array_equal(a, b)


def test_host_argument_errors():
    w = W.make_workload([[100]], "random", seed=1)
    t = device_inputs(w)
    scores = torch.zeros(1, 100, device="cuda")
    ws = binding.new_workspace(1, 100)
    with pytest.raises(binding.IdxError) as e:
        binding.score(t["q"], t["head_w"], t["k_cache"], t["k_scale"], t["block_table"], t["seq_lens"],
                      t["row_req"], torch.zeros(1, 102, device="cuda"), ws)  # stride % 4 != 0
    assert e.value.status == -2
    with pytest.raises(binding.IdxError) as e:
        binding.score(t["q"], t["head_w"], t["k_cache"], t["k_scale"], t["block_table"], t["seq_lens"],
                      t["row_req"], scores, ws[:64])  # workspace too small
    assert e.value.status == -3
