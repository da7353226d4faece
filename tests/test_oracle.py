"""Pins for the CPU oracle: each checks it against something other than itself.

 * E4M3 / bf16 decoding against torch's float8_e4m3fn / bfloat16 casts (a
   library routine) and closed-form codes of the format;
 * scores against a hand-worked example (tests/golden/hand_example.json),
   closed forms (one-hot query and key, all-zero keys, all-negative dots, the
   tie cache's four values), an independent NumPy f64 einsum over torch-decoded
   operands, and invariances of the paging (any page placement, same scores);
 * the selection against a pure-Python brute force on tiny inputs, its special
   cases, and list invariants on larger random rows;
 * the checker's negative controls (a winner swapped with the best loser, two
   entries swapped, one score's bits flipped) must each be caught, as in
   "sgl-amd-mono-upstream PR 18" (GLM-5.3 indexer launch), section
   "Modifications / 0. An exact top-k check".
"""
import json
import math
import os
import random

import numpy as np
import pytest
import torch

import oracle
from oracle import brute
from key_scoring_exact_gb300 import workloads as W
from tests import checks

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def problem_of(w: W.Workload) -> oracle.Problem:
    return oracle.Problem(w.q_bits().numpy(), w.q_is_e4m3, w.head_w.numpy(), w.k_cache.numpy(),
                          w.k_scale.numpy(), w.block_table.numpy(), w.seq_lens.numpy(),
                          w.row_req.numpy())


# ----------------------------------------------------------------- formats

def test_e4m3_all_codes_match_torch():
    codes = np.arange(256, dtype=np.uint8)
    got = oracle.e4m3_to_f64(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float32).double().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert nan.sum() == 2  # 0x7F and 0xFF
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def test_e4m3_closed_forms():
    f = oracle.e4m3_to_f64
    assert f(np.uint8(0x38)) == 1.0
    assert f(np.uint8(0x7E)) == 448.0
    assert f(np.uint8(0x01)) == 2.0 ** -9          # smallest subnormal
    assert f(np.uint8(0x07)) == 7 * 2.0 ** -9      # largest subnormal
    assert f(np.uint8(0x08)) == 2.0 ** -6          # smallest normal
    assert f(np.uint8(0x44)) == 3.0
    assert f(np.uint8(0xC4)) == -3.0
    assert f(np.uint8(0x80)) == 0.0 and np.signbit(f(np.uint8(0x80)))
    assert np.isnan(f(np.uint8(0x7F))) and np.isnan(f(np.uint8(0xFF)))


def test_bf16_matches_torch():
    rng = np.random.default_rng(0)
    bits = np.concatenate([rng.integers(0, 1 << 16, 4000, dtype=np.uint16),
                           np.array([0x0000, 0x8000, 0x3F80, 0xC000, 0x0001, 0x7F7F], np.uint16)])
    got = oracle.bf16_to_f64(bits)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


# ------------------------------------------------------------------ scores

def _hand_problem():
    d = json.load(open(os.path.join(GOLDEN, "hand_example.json")))
    pb = oracle.Problem(np.array(d["q_bits"], np.uint16), False, np.array(d["head_w"], np.float32),
                        np.array(d["k_cache_codes"], np.uint8), np.array(d["k_scale"], np.float32),
                        np.array(d["block_table"], np.int32), np.array(d["seq_lens"], np.int32),
                        np.array(d["row_req"], np.int32))
    return d, pb


def test_hand_example_scores():
    d, pb = _hand_problem()
    s = oracle.scores(pb)
    for r, exp in enumerate(d["expected_scores"]):
        n = len(exp)
        assert np.array_equal(s[r, :n], np.array(exp)), (r, s[r], exp)
        assert np.all(np.isnan(s[r, n:]))


def test_hand_example_topk():
    d, pb = _hand_problem()
    s = oracle.scores(pb)
    for k, lists in d["expected_topk"].items():
        for r, exp in enumerate(lists):
            n = d["seq_lens"][r]
            assert oracle.topk(s[r, :n].astype(np.float32), int(k)).tolist() == exp
            assert brute.topk(s[r, :n].astype(np.float32).tolist(), int(k)) == exp


def _tiny(H=3, D=5, P=4, lens=(7,), seed=0, q_e4m3=False):
    """A small random problem at any shape, one request, shuffled pages."""
    rng = np.random.default_rng(seed)
    n = max(lens)
    pages = (n + P - 1) // P
    pool = pages + 3
    perm = rng.permutation(pool)
    kc = np.full((pool, P, D), 0x7F, np.uint8)
    ks = np.full((pool, P), np.nan, np.float32)
    codes = torch.randn(pages * P, D, generator=torch.Generator().manual_seed(seed)).to(
        torch.float8_e4m3fn).view(torch.uint8).numpy().reshape(pages, P, D)
    scl = rng.uniform(0.5, 2.0, (pages, P)).astype(np.float32)
    for lp in range(pages):
        kc[perm[lp]] = codes[lp]
        ks[perm[lp]] = scl[lp]
    bt = perm[:pages].astype(np.int32)[None, :]
    R = len(lens)
    qf = torch.randn(R, H, D, generator=torch.Generator().manual_seed(seed + 1))
    q = (qf.to(torch.float8_e4m3fn).view(torch.uint8) if q_e4m3
         else qf.to(torch.bfloat16).view(torch.int16)).numpy()
    w = rng.uniform(0, 1 / 8, (R, H)).astype(np.float32)
    return oracle.Problem(q, q_e4m3, w, kc, ks, bt, np.array(lens, np.int32), np.zeros(R, np.int32))


def _einsum_scores(pb: oracle.Problem) -> np.ndarray:
    """The same definition through library routines: torch casts decode the
    operands, NumPy einsum contracts in f64."""
    if pb.q_is_e4m3:
        q = torch.from_numpy(pb.q).view(torch.float8_e4m3fn).double().numpy()
    else:
        q = torch.from_numpy(pb.q.view(np.int16)).view(torch.bfloat16).double().numpy()
    kv = torch.from_numpy(pb.k_cache).view(torch.float8_e4m3fn).double().numpy()
    kv = kv * pb.k_scale.astype(np.float64)[:, :, None]
    out = np.full((pb.R, int(pb.seq_lens.max())), np.nan)
    for r in range(pb.R):
        n = int(pb.seq_lens[r])
        pages = pb.block_table[pb.row_req[r]]
        keys = kv[pages].reshape(-1, pb.D)[:n]                      # [n, D] logical order
        dots = np.einsum("hd,jd->hj", q[r], keys)
        out[r, :n] = np.einsum("h,hj->j", pb.head_w[r].astype(np.float64), np.maximum(dots, 0.0))
    return out


@pytest.mark.parametrize("seed,shape,q_e4m3", [
    (0, dict(H=3, D=5, P=4, lens=(7,)), False),
    (1, dict(H=8, D=16, P=8, lens=(33, 40, 1)), False),
    (2, dict(H=4, D=32, P=16, lens=(65, 64)), True),
    (3, dict(H=64, D=128, P=64, lens=(130,)), False),
])
def test_scores_match_einsum(seed, shape, q_e4m3):
    pb = _tiny(seed=seed, q_e4m3=q_e4m3, **shape)
    got = oracle.scores(pb)
    ref = _einsum_scores(pb)
    for r, n in enumerate(pb.seq_lens):
        np.testing.assert_allclose(got[r, :n], ref[r, :n], rtol=1e-12, atol=1e-12)


def test_scores_one_hot_closed_form():
    # q[h] = c_h * e_{d_h}, key j = v_j * e_{d_j}: dot = c*v*scale on a shared
    # dim, else 0; s = sum_h w_h * max(dot, 0).
    H, D, P = 2, 4, 2
    q = np.zeros((1, H, D), np.uint16)
    q[0, 0, 1] = 0x4000  # 2.0
    q[0, 1, 3] = 0xC000  # -2.0
    kc = np.zeros((2, P, D), np.uint8)
    kc[0, 0, 1] = 0x38   # key 0 = 1.0 * e1
    kc[0, 1, 3] = 0x38   # key 1 = 1.0 * e3
    kc[1, 0, 3] = 0xB8   # key 2 = -1.0 * e3
    kc[1, 1, 0] = 0x48   # key 3 = 4.0 * e0 (orthogonal to both heads)
    ks = np.array([[0.5, 2.0], [1.5, 3.0]], np.float32)
    w = np.array([[0.25, 0.75]], np.float32)
    pb = oracle.Problem(q, False, w, kc, ks, np.array([[0, 1]], np.int32),
                        np.array([4], np.int32), np.array([0], np.int32))
    s = oracle.scores(pb)[0]
    assert s.tolist() == [0.25 * 2.0 * 1.0 * 0.5, 0.0, 0.75 * (-2.0) * (-1.0) * 1.5, 0.0]


def test_scores_zero_keys_and_negative_dots():
    w = W.make_workload([[300]], "zeros", seed=3)
    s = oracle.scores(problem_of(w))
    assert np.all(s[0, :300] == 0.0)
    pb = _tiny(H=4, D=8, P=4, lens=(9,), seed=5)
    kv = torch.from_numpy(pb.k_cache).view(torch.float8_e4m3fn).float()
    pb.k_cache = (-kv.abs()).to(torch.float8_e4m3fn).view(torch.uint8).numpy()   # keys <= 0
    qf = torch.from_numpy(pb.q.view(np.int16)).view(torch.bfloat16).float()
    pb.q = qf.abs().to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)    # q >= 0
    s = oracle.scores(pb)[0, :9]
    assert np.all(s == 0.0)


def test_tie_cache_has_four_values():
    w = W.make_workload([[523, 520]], "ties", seed=11, k=8)
    s = oracle.scores(problem_of(w))
    for r, n in enumerate(w.seq_lens.tolist()):
        row = s[r, :n]
        vals = np.unique(row)
        assert len(vals) <= 4
        for j in range(4):
            assert np.all(row[j::4] == row[j])


def test_paging_invariance():
    # The same logical keys under a contiguous and a shuffled placement.
    a = W.make_workload([[200, 150]], "random", seed=9, shuffle_pages=False)
    b = W.make_workload([[200, 150]], "random", seed=9, shuffle_pages=True)
    assert torch.equal(a.k_cache[a.block_table[0, :4].long()], b.k_cache[b.block_table[0, :4].long()])
    sa = oracle.scores(problem_of(a))
    sb = oracle.scores(problem_of(b))
    assert np.array_equal(sa, sb, equal_nan=True)


def test_score_positions_agree_with_full_rows():
    w = W.make_workload([[700, 650]], "recent", seed=4, recent_keys=100)
    pb = problem_of(w)
    full = oracle.scores(pb)
    pos = np.array([0, 1, 63, 64, 127, 128, 599, 600, 649], np.int64)
    got = oracle.score_positions(pb, 1, pos)
    assert np.array_equal(got, full[1, pos])


def test_poisoned_reads_are_detected():
    # A row that claims more keys than its request holds reads poison: NaN.
    w = W.make_workload([[100]], "random", seed=2)
    w.seq_lens[0] = 128        # keys 100..127 are poisoned slots of the last page
    s = oracle.scores(problem_of(w))[0]
    assert np.all(np.isfinite(s[:100])) and np.all(np.isnan(s[100:128]))


def test_out_of_range_page_is_an_error():
    w = W.make_workload([[100]], "random", seed=2)
    w.seq_lens[0] = 129        # needs a third page; the block table holds -1 there
    with pytest.raises(ValueError):
        oracle.scores(problem_of(w))


# --------------------------------------------------------------- selection

def _levels_row(rng, n, levels):
    vals = rng.choice(levels, size=n)
    return vals.astype(np.float32)


@pytest.mark.parametrize("seed", range(40))
def test_topk_matches_bruteforce_tiny(seed):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(0, 13))
    k = int(rng.integers(1, 6))
    levels = [np.float32(-1.5), np.float32(0.0), np.float32(2.25)]
    if seed % 5 == 0:
        levels += [np.float32(np.nan), np.float32(-0.0)]
    row = _levels_row(rng, n, levels)
    assert oracle.topk(row, k).tolist() == brute.topk(row.tolist(), k)


@pytest.mark.parametrize("seed", range(8))
def test_topk_matches_bruteforce_small_random(seed):
    rng = np.random.default_rng(100 + seed)
    n = int(rng.integers(20, 200))
    k = int(rng.integers(1, n + 5))
    row = rng.integers(-6, 7, n).astype(np.float32) / 4  # many ties
    assert oracle.topk(row, k).tolist() == brute.topk(row.tolist(), k)


def test_topk_special_cases():
    k = 16
    assert oracle.topk(np.zeros(0, np.float32), k).tolist() == [-1] * k
    assert oracle.topk(np.ones(10, np.float32), k).tolist() == list(range(10)) + [-1] * 6
    assert oracle.topk(np.ones(k, np.float32), k).tolist() == list(range(k))
    assert oracle.topk(np.full(100, 3.0, np.float32), k).tolist() == list(range(k))
    distinct = np.random.default_rng(1).permutation(100).astype(np.float32)
    got = oracle.topk(distinct, k)
    assert sorted(got.tolist()) == sorted(np.argsort(-distinct)[:k].tolist())
    # no ties: the keys above the k-th largest ascend, then the k-th itself
    assert np.all(np.diff(got[:-1]) > 0)
    assert distinct[got[-1]] == np.sort(distinct)[-k]
    # -0 and +0 tie: the earlier position wins
    assert oracle.topk(np.array([-0.0, 0.0, -1.0], np.float32), 1).tolist() == [0]
    assert oracle.topk(np.array([0.0, -0.0, -1.0], np.float32), 1).tolist() == [0]
    # NaN ranks below every number
    assert oracle.topk(np.array([np.nan, -np.inf, np.nan], np.float32), 1).tolist() == [1]


@pytest.mark.parametrize("n,k", [(5000, 2048), (2049, 2048), (70000, 2048), (4097, 1)])
def test_topk_invariants(n, k):
    rng = np.random.default_rng(n + k)
    row = (rng.standard_normal(n) * 3).astype(np.float32)
    row[rng.integers(0, n, n // 10)] = np.float32(1.0)     # a big tie block
    lst = oracle.topk(row, k)
    assert checks.list_invariants(lst, row, k) == []


def test_topk_rows_matches_single_rows():
    rng = np.random.default_rng(7)
    s = rng.standard_normal((3, 50)).astype(np.float32)
    lens = np.array([50, 3, 0], np.int32)
    out = oracle.topk_rows(s, lens, 8)
    for r in range(3):
        assert out[r].tolist() == oracle.topk(s[r, :lens[r]], 8).tolist()


# --------------------------------------------------------- negative controls

def _scored_row(seed=0, n=6000, k=2048):
    rng = np.random.default_rng(seed)
    row = rng.standard_normal(n).astype(np.float32)
    row[::37] = np.float32(0.5)
    return row, oracle.topk(row, k), k


def test_negative_control_winner_swapped_with_best_loser():
    row, lst, k = _scored_row()
    bad = lst.copy()
    losers = np.setdiff1d(np.arange(row.shape[0]), lst)
    best_loser = losers[np.argmax(row[losers])]
    bad[-1] = best_loser
    assert not np.array_equal(bad, lst)
    assert checks.list_invariants(bad, row, k) != []


def test_negative_control_two_entries_swapped():
    row, lst, k = _scored_row(1)
    bad = lst.copy()
    bad[[3, 10]] = bad[[10, 3]]
    assert not np.array_equal(bad, lst)
    assert checks.list_invariants(bad, row, k) != []


def test_negative_control_score_bits_flipped():
    row, lst, k = _scored_row(2)
    flipped = row.copy()
    j = int(lst[0])
    flipped.view(np.uint32)[j] ^= np.uint32(0x40000000)   # an exponent bit
    ref = row.astype(np.float64)
    assert checks.row_score_error(flipped, ref) > checks.SCORE_TOL
    # and the list of the flipped scores differs from the original list
    assert not np.array_equal(oracle.topk(flipped, k), lst) or flipped[j] > row[j]


def test_missed_counts():
    row, lst, k = _scored_row(3)
    assert checks.missed(lst, row, k) == 0
    bad = lst.copy()
    losers = np.setdiff1d(np.arange(row.shape[0]), lst)
    bad[0] = losers[0]
    assert checks.missed(bad, row, k) == 1


def test_oracle_planted_mistake_is_caught():
    """A plausible oracle bug (dropping the ReLU) fails the einsum pin."""
    pb = _tiny(H=6, D=8, P=4, lens=(23,), seed=21)
    ref = _einsum_scores(pb)
    q = torch.from_numpy(pb.q.view(np.int16)).view(torch.bfloat16).double().numpy()
    kv = torch.from_numpy(pb.k_cache).view(torch.float8_e4m3fn).double().numpy()
    kv = kv * pb.k_scale.astype(np.float64)[:, :, None]
    keys = kv[pb.block_table[0]].reshape(-1, pb.D)[:23]
    no_relu = np.einsum("h,hj->j", pb.head_w[0].astype(np.float64), np.einsum("hd,jd->hj", q[0], keys))
    assert np.max(np.abs(no_relu - ref[0])) > 1e-3


# ---------------------------------------------------------------- FP8 query quantisation

def _torch_e4m3_codes(x32: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(x32, np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def _e4m3_midpoints() -> np.ndarray:
    """Every value halfway between two neighbouring finite non-negative E4M3
    values (an exact tie), with both signs."""
    vals = oracle.e4m3_to_f64(np.arange(0x7F, dtype=np.uint8)).reshape(-1)
    mids = (vals[:-1] + vals[1:]) / 2
    return np.concatenate([mids, -mids]).astype(np.float32)


def test_e4m3_encode_matches_torch_cast():
    """The oracle's encoder (nearest by exhaustive comparison, ties to even)
    against torch's cast on every finite bf16 value below the saturation
    point (|x| < 464, where the cast does not overflow), every exact tie and
    its neighbours, and random f32 values."""
    bits = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)
    vals = (bits.astype(np.uint32) << 16).view(np.float32)
    vals = vals[np.isfinite(vals) & (np.abs(vals) < 464)]
    mids = _e4m3_midpoints()
    near = np.concatenate([np.nextafter(mids, np.float32(np.inf)), np.nextafter(mids, np.float32(-np.inf))])
    rng = np.random.default_rng(9)
    rnd = (rng.standard_normal(20000) * np.exp2(rng.integers(-12, 8, 20000))).astype(np.float32)
    rnd = rnd[np.abs(rnd) < 464]
    x = np.concatenate([vals, mids, near, rnd]).astype(np.float32)
    assert np.array_equal(oracle.f32_to_e4m3(x), _torch_e4m3_codes(x))


def test_e4m3_encode_saturates_and_keeps_nan():
    x = np.array([448.0, 463.9, 464.0, 500.0, 1e30, -464.0, -1e30, np.nan], np.float32)
    assert oracle.f32_to_e4m3(x).tolist() == [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0xFE, 0x7F]


def _bf16_bits(x: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_quantize_exact_powers_of_two():
    """Heads made of E4M3 values times 2^k with one element at 448 * 2^k: the
    scale is exactly 2^k, so the codes are the E4M3 values and w' = w 2^k."""
    rng = np.random.default_rng(31)
    R, H, D = 2, 5, 128
    codes = rng.integers(0, 0x7F, (R, H, D)).astype(np.uint8)
    codes[rng.random((R, H, D)) < 0.5] |= 0x80
    codes[codes == 0x80] = 0x00
    codes[codes == 0xFF] = 0x7E
    codes[..., 7] = 0x7E                         # the head's largest magnitude: 448
    codes[..., 0x7F & 9] &= 0x7F                 # keep one position non-negative
    vals = oracle.e4m3_to_f64(codes).astype(np.float32)
    ks = rng.integers(-20, 20, (R, H)).astype(np.float32)
    q = vals * np.exp2(ks)[:, :, None]
    w = rng.uniform(0.1, 2.0, (R, H)).astype(np.float32)
    q8, wo = oracle.quantize_query(_bf16_bits(q), w)
    assert np.array_equal(q8, codes)
    assert np.array_equal(wo, (w * np.exp2(ks)).astype(np.float32))


def test_quantize_zero_and_single_element_heads():
    R, H, D = 1, 3, 128
    q = np.zeros((R, H, D), np.float32)
    q[0, 1, 17] = -3.0
    q[0, 2, 5] = 0.013671875
    w = np.array([[1.5, 2.0, -0.5]], np.float32)
    q8, wo = oracle.quantize_query(_bf16_bits(q), w)
    assert not q8[0, 0].any() and wo[0, 0] == 0.0                     # an all-zero head
    assert q8[0, 1, 17] == 0xFE and np.count_nonzero(q8[0, 1]) == 1   # -448
    assert q8[0, 2, 5] == 0x7E and np.count_nonzero(q8[0, 2]) == 1
    assert wo[0, 1] == np.float32(2.0) * (np.float32(3.0) / np.float32(448.0))
    assert wo[0, 2] == np.float32(-0.5) * (np.float32(0.013671875) / np.float32(448.0))


def _quant_properties_hold(q32, w, q8, wo) -> bool:
    """Properties of any correct per-head amax/448 quantisation: the largest
    element maps to +-448, w' / w is the head's scale, and every element is
    reproduced within half an E4M3 step at its magnitude (times the scale),
    give or take the f32 rounding of the quotient (2^-24 relative, well
    below the 1e-5 of the half step allowed here)."""
    amax = np.abs(q32).max(-1)
    scale = (wo / w).astype(np.float64)
    if not np.allclose(scale, amax.astype(np.float64) / 448, rtol=1e-6, atol=0):
        return False
    top = np.take_along_axis(q8, np.abs(q32).argmax(-1)[..., None], -1)[..., 0] & 0x7F
    if not np.all(top == 0x7E):
        return False
    dec = oracle.e4m3_to_f64(q8)
    mag = np.maximum(np.abs(dec), 2.0 ** -6)
    half_step = np.exp2(np.floor(np.log2(mag)) - 4)      # half the spacing: 3 mantissa bits
    err = np.abs(dec * scale[..., None] - q32.astype(np.float64))
    return bool(np.all(err <= half_step * scale[..., None] * (1 + 1e-5) + 1e-30))


def test_quantize_properties_and_symmetries():
    rng = np.random.default_rng(47)
    R, H, D = 3, 64, 128
    q32 = (rng.standard_normal((R, H, D)) * np.exp2(rng.integers(-6, 6, (R, H, 1)))).astype(np.float32)
    q32 = torch.from_numpy(q32).to(torch.bfloat16).float().numpy()
    w = rng.uniform(0.05, 1.0, (R, H)).astype(np.float32)
    q8, wo = oracle.quantize_query(_bf16_bits(q32), w)
    assert _quant_properties_hold(q32, w, q8, wo)
    # negation flips the sign bits of the non-zero codes and keeps the weights
    n8, nw = oracle.quantize_query(_bf16_bits(-q32), w)
    nz = (q8 & 0x7F) != 0
    assert np.array_equal(n8[nz], q8[nz] ^ 0x80) and np.array_equal(nw, wo)
    # a power-of-two factor leaves the codes and scales the weights exactly
    p8, pw = oracle.quantize_query(_bf16_bits(q32 * np.float32(2.0 ** -5)), w)
    assert np.array_equal(p8, q8) and np.array_equal(pw, (wo * np.float32(2.0 ** -5)).astype(np.float32))


def test_quantize_planted_mistake_is_caught():
    """Codes from a wrong divisor (amax / 447) or weights missing the scale
    fail the property check."""
    rng = np.random.default_rng(48)
    q32 = torch.from_numpy(rng.standard_normal((1, 8, 128)).astype(np.float32)).to(torch.bfloat16).float().numpy()
    w = np.ones((1, 8), np.float32)
    q8, wo = oracle.quantize_query(_bf16_bits(q32), w)
    amax = np.abs(q32).max(-1, keepdims=True)
    wrong = oracle.f32_to_e4m3((q32 / (amax / np.float32(447))).astype(np.float32))
    assert not _quant_properties_hold(q32, w, wrong, wo)
    assert not _quant_properties_hold(q32, w, q8, w)


# ---------------------------------------------------------------- physical slots

def test_slots_worked_example_and_closed_forms():
    """Pages of 64 keys: request 0's block table [5, 2, 9] puts position 0 in
    slot 5 * 64 = 320, position 63 in 383, position 64 in page 2 (slot 128)
    and position 130 in page 9 at row 2 (slot 578); an identity table maps
    every position to itself; padding stays -1."""
    bt = np.array([[5, 2, 9], [0, 1, 2]], np.int32)
    idx = np.array([[0, 63, 64, 130, -1], [0, 63, 64, 130, -1]], np.int32)
    got = oracle.slots(idx, bt, np.array([0, 1], np.int32))
    assert got.tolist() == [[320, 383, 128, 578, -1], [0, 63, 64, 130, -1]]
    ident = np.arange(64, dtype=np.int32)[None, :]
    pos = np.random.default_rng(3).integers(0, 64 * 64, (3, 50)).astype(np.int32)
    assert np.array_equal(oracle.slots(pos, ident, np.zeros(3, np.int32)), pos)


def test_tagged_pairs_worked_example_and_layout():
    """oracle_tagged ("sgl-amd-mono-upstream PR 11", section "3. The selected
    tokens are tagged pairs"): worked values written out by hand, and the pair
    read back as its two little-endian int32 words {entry, tag}."""
    e = np.array([5, -1, 0x7FFFFFFF, 0, 2048], np.int32)
    got = oracle.tagged(e, 7)
    assert got.tolist() == [0x0000000700000005, 0x00000007FFFFFFFF, 0x000000077FFFFFFF,
                            0x0000000700000000, 0x0000000700000800]
    # the top tag bit: the int64 goes negative, the words stay {entry, tag}
    top = oracle.tagged(np.array([3, -1], np.int32), 0xFFFFFFFF)
    assert top.tolist() == [-(1 << 32) + 3, -1]
    rng = np.random.default_rng(4)
    ent = rng.integers(-1, 1 << 31, size=1000).astype(np.int32)
    for tag in (0, 1, 123456789, 0xFFFFFFFF):
        words = oracle.tagged(ent, tag).view(np.int32).reshape(-1, 2)   # little-endian host
        assert np.array_equal(words[:, 0], ent)
        assert np.all(words[:, 1].view(np.uint32) == np.uint32(tag))


def test_store_keys_worked_example():
    """oracle_store_keys ("sgl-amd-mono-upstream PR 18", section "Modifications
    / 2", keys this launch writes): each row's key lands in the slot of its
    request's position seq_lens[r] - 1, found through the block table, and
    nothing else changes.  The expected cache is written by hand."""
    P, D = 64, 128
    rng = np.random.default_rng(8)
    kc = rng.integers(0, 256, size=(3, P, D), dtype=np.uint8)
    ks = rng.random((3, P), dtype=np.float32)
    bt = np.array([[2, 0], [1, -1]], np.int32)       # request 0: page 2 then page 0; request 1: page 1
    lens = np.array([70, 65, 0, 10], np.int32)        # rows 0..2 of request 0, row 3 of request 1
    rreq = np.array([0, 0, 0, 1], np.int32)
    nk = rng.integers(0, 256, size=(4, D), dtype=np.uint8)
    ns = np.array([0.5, 1.5, 9.0, 2.5], np.float32)
    got_k, got_s = oracle.store_keys(kc, ks, bt, lens, rreq, nk, ns)
    want_k, want_s = kc.copy(), ks.copy()
    want_k[0, 5] = nk[0]      # row 0: position 69 = page index 1 -> page 0, slot 5
    want_s[0, 5] = 0.5
    want_k[0, 0] = nk[1]      # row 1: position 64 -> page 0, slot 0
    want_s[0, 0] = 1.5
    want_k[1, 9] = nk[3]      # row 3: position 9 of request 1 -> page 1, slot 9 (row 2 has no key)
    want_s[1, 9] = 2.5
    assert np.array_equal(got_k, want_k) and np.array_equal(got_s, want_s)
    assert np.array_equal(kc, oracle.store_keys(kc, ks, bt, lens * 0, rreq, nk, ns)[0])  # no keys: no change


def test_stored_keys_are_what_the_rows_score():
    """After the store, the score of each new key is the one-hot closed form
    of that key (head 0 only, w = 1): scale * e4m3(code) * q where positive;
    with the slot poisoned and no store, the same score is not finite."""
    P, D, H = 64, 128, 64
    R = 3
    kc = np.zeros((2, P, D), np.uint8)
    ks = np.ones((2, P), np.float32)
    bt = np.array([[1, 0]], np.int32)
    lens = np.array([70, 71, 72], np.int32)
    rreq = np.zeros(R, np.int32)
    kc[0, 5:8] = 0x7F                                  # the rows' slots poisoned (NaN codes, huge scales)
    ks[0, 5:8] = 1e30
    nk = np.zeros((R, D), np.uint8)
    nk[:, 3] = [0x38, 0x40, 0x44]                      # 1.0, 2.0, 3.0 in E4M3, at dim 3
    ns = np.array([0.5, 1.5, 2.0], np.float32)
    q = np.zeros((R, H, D), np.float32)
    q[:, 0, 3] = 1.0
    qb = (torch.from_numpy(q).to(torch.bfloat16).view(torch.uint16).numpy())
    w = np.zeros((R, H), np.float32)
    w[:, 0] = 1.0
    kc2, ks2 = oracle.store_keys(kc, ks, bt, lens, rreq, nk, ns)
    s = oracle.scores(oracle.Problem(qb, False, w, kc2, ks2, bt, lens, rreq))
    for r in range(R):
        for j, (code_val, sc) in enumerate([(1.0, 0.5), (2.0, 1.5), (3.0, 2.0)]):
            pos = 69 + j
            if pos < lens[r]:
                assert s[r, pos] == code_val * sc, (r, pos, s[r, pos])
    poisoned = oracle.scores(oracle.Problem(qb, False, w, kc, ks, bt, lens, rreq))
    assert not np.isfinite(poisoned[2, 69:72]).any()


def test_prefix_order_worked_example():
    """The pages' list order, worked by hand.  k = 3 over [1.5000001, 1.0, 1.5,
    0.5, 0.25, 3.0]: T = 1.5 (image 0xBFC00000).  The keys sharing T's 12-bit
    prefix 0xBFC are 1.5000001 and 1.5, and they share the 24-bit prefix too.
    With room >= 2 the radix stops at 12 bits: 3.0 (prefix 0xC04, position 5),
    then 1.5000001 (prefix 0xBFC, above T, position 0), then the tie at 2.
    With room 1 it runs to 32 bits: the specification's order, 0, 5, 2."""
    s = np.array([1.5000001, 1.0, 1.5, 0.5, 0.25, 3.0], np.float32)
    assert s[0] > s[2]
    assert oracle.prefix_order(s, 3, 2).tolist() == [5, 0, 2]
    assert oracle.prefix_order(s, 3, 100).tolist() == [5, 0, 2]
    assert oracle.prefix_order(s, 3, 1).tolist() == [0, 5, 2]
    assert oracle.topk(s, 3).tolist() == [0, 5, 2]
    # a 24-bit stop: 1.5 + 2^-12 shares T's 12-bit prefix but not its 24-bit one
    s2 = np.array([1.5 + 2.0 ** -12, 1.5000001, 1.5, 0.5, 3.0, 1.0], np.float32)
    # sorted: 3.0 (4), 1.5+2^-12 (0), 1.5000001 (1), 1.5 (2): k = 4 gives T = 1.5
    # 12-bit keys: positions 0, 1, 2 (3 keys); 24-bit keys: positions 1, 2 (2 keys)
    assert oracle.prefix_order(s2, 4, 2).tolist() == [0, 4, 1, 2]   # 24-bit stop: 0 and 4 are above 0xBFC000
    assert oracle.prefix_order(s2, 4, 3).tolist() == [4, 0, 1, 2]   # 12-bit stop
    assert oracle.prefix_order(s2, 4, 1).tolist() == [0, 1, 4, 2]   # 32 bits: the specification's order
    assert oracle.topk(s2, 4).tolist() == [0, 1, 4, 2]


def test_prefix_order_properties():
    """At every stop the list holds oracle_topk's set; room 0 (no prefix can
    stop: T's own key shares it) gives oracle_topk's list exactly; short rows
    are oracle_topk's."""
    rng = np.random.default_rng(21)
    for trial in range(30):
        n = int(rng.integers(1, 3000))
        k = int(rng.integers(1, 400))
        levels = rng.integers(2, 50)
        s = (rng.integers(0, levels, n) * rng.choice([1.0, 1.0 / 3.0, 1e-3])).astype(np.float32)
        s += rng.standard_normal(n).astype(np.float32) * rng.choice([0.0, 1e-6, 1e-2])
        ref = oracle.topk(s, k)
        assert np.array_equal(oracle.prefix_order(s, k, 0), ref)
        for room in (1, 7, 64, 1 << 20):
            got = oracle.prefix_order(s, k, room)
            assert sorted(got.tolist()) == sorted(ref.tolist()), (trial, room)
