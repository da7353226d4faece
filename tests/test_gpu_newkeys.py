"""idx_score_topk_newkeys: the keys a step writes ("sgl-amd-mono-upstream PR
18", section "Modifications / 2", keys this launch writes).  Each row's own
key is stored in its slot and scored by every row of its request, in every
row group.  The rows' slots are poisoned in the cache first (NaN codes,
scale 1e30, as the pages' check poisons the step's cached scales), so a row
that scored a slot before its store would be off by ~1e30.  Checks: the
cache afterwards equals the oracle's store, the scores are within 1e-4 of
the oracle's scores of that cache, and the lists are bit-exact."""
import numpy as np
import pytest
import torch

import oracle
from key_scoring_exact_gb300 import binding
from key_scoring_exact_gb300 import workloads as W
from tests import checks
from tests.gpu_util import stride_for

pytestmark = pytest.mark.gpu

E4M3_NAN = 0x7F


@pytest.mark.parametrize("layout,query", [
    ([W.chain(20000, 8), [3000]], "bf16"),   # an 8-row draft chain: two row groups, each scoring the other's keys
    ([W.chain(9000, 4), [700], W.chain(5000, 3)], "bf16"),
    ([W.chain(6000, 6)], "e4m3"),
    ([W.chain(6000, 6), [2500]], "bf16_fp8"),
])
def test_new_keys_stored_and_scored_by_every_row(layout, query):
    w = W.make_workload(layout, "random", seed=sum(map(sum, layout)) % 97, q_is_e4m3=query == "e4m3")
    R = w.R
    g = torch.Generator().manual_seed(123)
    new_k = torch.randn(R, 128, generator=g).to(torch.float8_e4m3fn).view(torch.uint8)
    new_scale = torch.rand(R, generator=g) * 1.5 + 0.5
    kc, ks = w.k_cache.clone(), w.k_scale.clone()
    bt = w.block_table.numpy()
    for r, (n, q) in enumerate(zip(w.seq_lens.tolist(), w.row_req.tolist())):
        pg = bt[q, (n - 1) // 64]
        kc[pg, (n - 1) % 64] = E4M3_NAN
        ks[pg, (n - 1) % 64] = 1e30
    want_k, want_s = oracle.store_keys(kc.numpy(), ks.numpy(), bt, w.seq_lens.numpy(), w.row_req.numpy(),
                                       new_k.numpy(), new_scale.numpy())

    dev = {f: getattr(w, f).cuda() for f in ("q", "head_w", "block_table", "seq_lens", "row_req")}
    kc_d, ks_d = kc.cuda(), ks.cuda()
    scores = torch.zeros(R, stride_for(w.max_len), dtype=torch.float32, device="cuda")
    idx = torch.full((R, w.k), -7, dtype=torch.int32, device="cuda")
    ws = binding.new_workspace(R, w.max_len, w.k)
    binding.score_topk_newkeys(dev["q"], dev["head_w"], kc_d, ks_d, dev["block_table"], dev["seq_lens"],
                               dev["row_req"], new_k.cuda(), new_scale.cuda(), w.max_len, w.k, idx, ws,
                               scores=scores, quantize_q=query == "bf16_fp8")
    assert binding.check_status(ws) == 0
    assert np.array_equal(kc_d.cpu().numpy(), want_k)
    # bit patterns: the pool's unused slots hold NaN scales
    assert np.array_equal(ks_d.cpu().numpy().view(np.uint32), want_s.view(np.uint32))

    s = scores.cpu().numpy()
    if query == "bf16_fp8":   # the scores of the query as the device quantises it (idx_quantize_query)
        q8, wq = oracle.quantize_query(w.q_bits().numpy(), w.head_w.numpy())
        pb = oracle.Problem(q8, True, wq, want_k, want_s, bt, w.seq_lens.numpy(), w.row_req.numpy())
    else:
        pb = oracle.Problem(w.q_bits().numpy(), w.q_is_e4m3, w.head_w.numpy(), want_k, want_s, bt,
                            w.seq_lens.numpy(), w.row_req.numpy())
    ref = oracle.scores(pb)
    errs = checks.score_errors(s, ref, w.seq_lens.tolist())
    assert max(errs) <= checks.SCORE_TOL, errs
    got = idx.cpu().numpy()
    for r, n in enumerate(w.seq_lens.tolist()):
        assert np.array_equal(got[r], oracle.topk(s[r, :n], w.k)), "row %d" % r
