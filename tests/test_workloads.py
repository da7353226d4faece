"""The synthetic input recipes: shapes, poisoning, cache structure, determinism."""
import numpy as np
import pytest
import torch

from key_scoring_exact_gb300 import workloads as W


def test_config1_shapes_and_poison():
    w = W.make_config(1)
    assert w.R == 1 and w.seq_lens.tolist() == [4096]
    assert w.q.dtype == torch.bfloat16 and tuple(w.q.shape) == (1, 64, 128)
    pages = w.block_table[0]
    used = pages[pages >= 0].long()
    assert used.numel() == 64
    unused = torch.ones(w.pool_pages, dtype=torch.bool)
    unused[used] = False
    assert unused.sum() == W.EXTRA_POISON_PAGES
    assert torch.all(w.k_cache[unused] == W.E4M3_NAN)
    assert torch.all(torch.isnan(w.k_scale[unused]))
    s = w.k_scale[used]
    assert torch.all((s >= 0.5) & (s <= 2.0))
    assert torch.all((w.head_w >= 0) & (w.head_w <= 1 / 8))


def test_chain_lengths_and_tail_poison():
    w = W.make_workload([W.chain(300)], "random", seed=1)
    assert w.seq_lens.tolist() == [297, 298, 299, 300]
    last = int(w.block_table[0, (300 - 1) // 64])
    assert torch.all(w.k_cache[last, 300 % 64:] == W.E4M3_NAN)
    assert torch.all(torch.isnan(w.k_scale[last, 300 % 64:]))
    assert not torch.any(torch.isnan(w.k_scale[last, :300 % 64]))


def test_tie_cache_structure():
    w = W.make_config(2)
    assert w.seq_lens.tolist() == [8189, 8190, 8191, 8192]
    keys = w.k_cache[w.block_table[0].long()].reshape(-1, 128)[:8192]
    scl = w.k_scale[w.block_table[0].long()].reshape(-1)[:8192]
    for j in range(4):
        assert torch.all(keys[j::4] == keys[j]) and torch.all(scl[j::4] == scl[j])
    assert len({tuple(keys[j].tolist()) for j in range(4)}) == 4


def test_recent_cache_scales():
    w = W.make_workload([W.chain(5000)], "recent", seed=3, recent_keys=1000)
    scl = w.k_scale[w.block_table[0].long()].reshape(-1)[:5000]
    assert torch.all(scl[:4000] <= 2.0) and torch.all(scl[4000:] >= 4.0)


def test_mixed_lengths():
    for seed in range(1, 30):
        lens = W.mixed_lengths(seed)
        assert len(lens) == 16 and sum(1 for v in lens if v < 2048) >= 3
        assert min(lens) >= 512 and max(lens) <= 131072


def test_config4_has_zero_request():
    w = W.make_config(4)
    assert w.R == 17 and w.row_req.tolist() == list(range(17))
    assert w.seq_lens[16] == 8192
    zpages = w.block_table[16][w.block_table[16] >= 0].long()
    assert torch.all(w.k_cache[zpages] == 0)


def test_deterministic():
    a = W.make_workload([[500, 400], [70]], "random", seed=5)
    b = W.make_workload([[500, 400], [70]], "random", seed=5)
    for f in ("q", "head_w", "k_cache", "block_table", "seq_lens", "row_req"):
        assert torch.equal(getattr(a, f), getattr(b, f))
    assert torch.equal(a.k_scale.nan_to_num(-1), b.k_scale.nan_to_num(-1))


def test_rotation_copies():
    w = W.make_workload([[300]], "random", seed=6)
    big, tables = W.with_rotation(w, 3)
    assert big.pool_pages == 3 * w.pool_pages and tables.shape[0] == 3
    for c in range(3):
        pg = tables[c, 0][tables[c, 0] >= 0].long()
        assert torch.equal(big.k_cache[pg], w.k_cache[w.block_table[0][:pg.numel()].long()])


def test_e4m3_query_variant():
    w = W.make_workload([[100]], "random", seed=8, q_is_e4m3=True)
    assert w.q.dtype == torch.uint8 and w.q_bits().dtype == torch.uint8
