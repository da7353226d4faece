"""Helpers for the GPU parity tests: move a workload to the device, run the
library through its C ABI, and build the oracle's view of the same inputs."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from key_scoring_exact_gb300 import binding
from key_scoring_exact_gb300 import workloads as W

FIELDS = ("q", "head_w", "k_cache", "k_scale", "block_table", "seq_lens", "row_req")


def device_inputs(w: W.Workload, dev="cuda"):
    return {f: getattr(w, f).to(dev) for f in FIELDS}


def problem(w: W.Workload) -> oracle.Problem:
    return oracle.Problem(w.q_bits().numpy(), w.q_is_e4m3, w.head_w.numpy(), w.k_cache.numpy(),
                          w.k_scale.numpy(), w.block_table.numpy(), w.seq_lens.numpy(),
                          w.row_req.numpy())


def stride_for(max_len: int) -> int:
    return max(4, (int(max_len) + 3) // 4 * 4)


def gpu_scores(w: W.Workload, t=None, sentinel: float = -12345.0):
    """idx_score; returns (scores [R, stride] numpy, status)."""
    t = t or device_inputs(w)
    stride = stride_for(w.max_len)
    scores = torch.full((w.R, stride), sentinel, dtype=torch.float32, device="cuda")
    ws = binding.new_workspace(w.R, stride)
    binding.score(t["q"], t["head_w"], t["k_cache"], t["k_scale"], t["block_table"], t["seq_lens"],
                  t["row_req"], scores, ws)
    st = binding.check_status(ws)
    return scores.cpu().numpy(), st


def gpu_topk(scores_np: np.ndarray, lens, k: int):
    s = torch.from_numpy(np.ascontiguousarray(scores_np, np.float32)).cuda()
    if s.shape[1] % 4:
        pad = torch.zeros(s.shape[0], 4 - s.shape[1] % 4, dtype=torch.float32, device="cuda")
        s = torch.cat([s, pad], 1).contiguous()
    ln = torch.as_tensor(np.asarray(lens, np.int32)).cuda()
    idx = torch.full((s.shape[0], k), -7, dtype=torch.int32, device="cuda")
    ws = binding.new_workspace(s.shape[0], s.shape[1], k)
    binding.topk(s, ln, k, idx, ws)
    st = binding.check_status(ws)
    return idx.cpu().numpy(), st


def gpu_fused(w: W.Workload, t=None, in_workspace: bool = False):
    """idx_score_topk; returns (scores, indices, status)."""
    t = t or device_inputs(w)
    max_len = w.max_len
    idx = torch.full((w.R, w.k), -7, dtype=torch.int32, device="cuda")
    if in_workspace:
        ws = binding.new_workspace(w.R, max_len, w.k, with_scores=True)
        binding.score_topk(t["q"], t["head_w"], t["k_cache"], t["k_scale"], t["block_table"],
                           t["seq_lens"], t["row_req"], max_len, w.k, idx, ws)
        scores = binding.scores_view(ws, w.R, max_len).clone()
    else:
        scores = torch.zeros(w.R, stride_for(max_len), dtype=torch.float32, device="cuda")
        ws = binding.new_workspace(w.R, max_len, w.k)
        binding.score_topk(t["q"], t["head_w"], t["k_cache"], t["k_scale"], t["block_table"],
                           t["seq_lens"], t["row_req"], max_len, w.k, idx, ws, scores=scores)
    st = binding.check_status(ws)
    return scores.cpu().numpy(), idx.cpu().numpy(), st
