"""The FP8-query path: idx_quantize_query bit-exact against the oracle's
quantiser, and scoring with IDX_Q_BF16_FP8 (quantisation inside the scoring
kernel) against the oracle's scores of the oracle-quantised query, with the
lists bit-exact against the oracle's selection of the GPU's own scores."""
import numpy as np
import pytest
import torch

import oracle
from key_scoring_exact_gb300 import binding
from key_scoring_exact_gb300 import workloads as W
from tests import checks
from tests.gpu_util import device_inputs, stride_for

pytestmark = pytest.mark.gpu


def _bits(q_bf16: torch.Tensor) -> np.ndarray:
    return q_bf16.contiguous().view(torch.int16).numpy().view(np.uint16)


def _special_heads(R=3):
    """Random heads over several magnitudes, plus all-zero heads, one-element
    heads, and heads whose quotients land on E4M3 ties."""
    rng = np.random.default_rng(77)
    q = (rng.standard_normal((R, 64, 128)) * np.exp2(rng.integers(-20, 20, (R, 64, 1)))).astype(np.float32)
    q[0, 0] = 0.0
    q[0, 1] = 0.0
    q[0, 1, 99] = -7.5
    # exact ties: amax = 448 * 2^k, the other elements halfway between E4M3 values times 2^k
    vals = oracle.e4m3_to_f64(np.arange(0x7F, dtype=np.uint8)).reshape(-1)
    mids = ((vals[:-1] + vals[1:]) / 2).astype(np.float32)
    for h in range(2, 10):
        k = float(h - 6)
        row = rng.choice(mids, 128) * rng.choice([-1.0, 1.0], 128)
        row[0] = 448.0
        q[1, h] = (row * 2.0 ** k).astype(np.float32)
    return torch.from_numpy(q).to(torch.bfloat16)


def test_quantize_bit_exact():
    q = _special_heads()
    w = torch.from_numpy(np.random.default_rng(78).uniform(-1, 1, (3, 64)).astype(np.float32))
    ref8, refw = oracle.quantize_query(_bits(q), w.numpy())
    q8, wo = binding.quantize_query(q.cuda(), w.cuda())
    assert np.array_equal(q8.cpu().numpy(), ref8)
    assert np.array_equal(wo.cpu().numpy().view(np.uint32), refw.view(np.uint32))


def _quantised_problem(w: W.Workload) -> oracle.Problem:
    q8, wq = oracle.quantize_query(_bits(w.q), w.head_w.numpy())
    return oracle.Problem(q8, True, wq, w.k_cache.numpy(), w.k_scale.numpy(), w.block_table.numpy(),
                          w.seq_lens.numpy(), w.row_req.numpy())


@pytest.mark.parametrize("cfg", [1, 2, 4])
def test_quantised_fused_matches_oracle(cfg):
    w = W.make_config(cfg)
    t = device_inputs(w)
    idx = torch.full((w.R, w.k), -7, dtype=torch.int32, device="cuda")
    s = torch.zeros(w.R, stride_for(w.max_len), dtype=torch.float32, device="cuda")
    ws = binding.new_workspace(w.R, w.max_len, w.k)
    binding.score_topk(t["q"], t["head_w"], t["k_cache"], t["k_scale"], t["block_table"], t["seq_lens"],
                       t["row_req"], w.max_len, w.k, idx, ws, scores=s, quantize_q=True)
    assert binding.check_status(ws) == 0
    s, got = s.cpu().numpy(), idx.cpu().numpy()
    ref = oracle.scores(_quantised_problem(w))
    errs = checks.score_errors(s, ref, w.seq_lens.tolist())
    assert max(errs) <= checks.SCORE_TOL, errs
    for r, n in enumerate(w.seq_lens.tolist()):
        assert np.array_equal(got[r], oracle.topk(s[r, :n], w.k)), "row %d" % r


def test_quantised_scores_at_128k_sampled():
    w = W.make_config(3)
    t = device_inputs(w)
    s = torch.zeros(w.R, stride_for(w.max_len), dtype=torch.float32, device="cuda")
    ws = binding.new_workspace(w.R, stride_for(w.max_len))
    binding.score(t["q"], t["head_w"], t["k_cache"], t["k_scale"], t["block_table"], t["seq_lens"],
                  t["row_req"], s, ws, quantize_q=True)
    assert binding.check_status(ws) == 0
    s = s.cpu().numpy()
    pb = _quantised_problem(w)
    rng = np.random.default_rng(79)
    for r, n in enumerate(w.seq_lens.tolist()):
        pos = np.unique(np.concatenate([[0, 63, 64, 127, 128, n - 1], rng.integers(0, n, 60),
                                        np.argsort(-s[r, :n])[:8]])).astype(np.int64)
        ref = oracle.score_positions(pb, r, pos)
        assert np.max(np.abs(s[r, pos] - ref)) / np.max(np.abs(ref)) <= checks.SCORE_TOL


def test_quantised_host_call_matches_device_call():
    w = W.make_config(2)
    t = device_inputs(w)
    idx = torch.full((w.R, w.k), -7, dtype=torch.int32, device="cuda")
    ws = binding.new_workspace(w.R, w.max_len, w.k, with_scores=True)
    binding.score_topk(t["q"], t["head_w"], t["k_cache"], t["k_scale"], t["block_table"], t["seq_lens"],
                       t["row_req"], w.max_len, w.k, idx, ws, quantize_q=True)
    hws = binding.new_host_workspace(w.R, w.max_len, w.k, w.block_table.shape[0], w.block_table.shape[1])
    out = torch.full((w.R, w.k), -7, dtype=torch.int32).pin_memory()
    binding.score_topk_host(w.q.pin_memory(), w.head_w.pin_memory(), t["k_cache"], t["k_scale"],
                            w.block_table.pin_memory(), w.seq_lens.pin_memory(), w.row_req.pin_memory(),
                            w.max_len, w.k, out, hws, quantize_q=True)
    torch.cuda.synchronize()
    assert np.array_equal(out.numpy(), idx.cpu().numpy())
