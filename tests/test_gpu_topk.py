"""GPU selection (idx_topk) against the oracle's sort-based list, bit-exact.

Score rows cover the page / tile boundaries and the lengths around k from
tests/golden/ragged_lengths.json, tie-heavy and all-zero rows, rows whose top
crowds into their last keys, special values, and rows long enough that a
slice no longer fits in shared memory."""
import json
import os

import numpy as np
import pytest

import oracle
from tests import checks
from tests.gpu_util import gpu_topk

pytestmark = pytest.mark.gpu

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "ragged_lengths.json")))
LENGTHS = sorted(set(GOLDEN["page_boundary"] + GOLDEN["around_k"] + GOLDEN["tile_boundary"]
                     + [0, 2, 8192, 131072, 131069, 250000]))


def _check_rows(scores, lens, k, got):
    for r, n in enumerate(lens):
        exp = oracle.topk(scores[r, :n], k)
        if not np.array_equal(got[r], exp):
            bad = np.nonzero(got[r] != exp)[0]
            raise AssertionError("row %d (n=%d): %d entries differ, first at %d: got %d want %d"
                                 % (r, n, bad.size, bad[0], got[r][bad[0]], exp[bad[0]]))


@pytest.mark.parametrize("n", LENGTHS)
def test_random_lengths(n):
    rng = np.random.default_rng(n)
    k = 2048
    s = rng.standard_normal((1, max(n, 4))).astype(np.float32) * 10
    got, st = gpu_topk(s, [n], k)
    assert st == 0
    _check_rows(s, [n], k, got)


def test_mixed_rows_one_launch():
    rng = np.random.default_rng(1)
    lens = [0, 1, 500, 2047, 2048, 2049, 3000, 8192, 40000, 131072, 65, 100000]
    width = max(lens)
    s = rng.standard_normal((len(lens), width)).astype(np.float32)
    got, st = gpu_topk(s, lens, 2048)
    assert st == 0
    _check_rows(s, lens, 2048, got)


@pytest.mark.parametrize("levels", [1, 2, 4, 17])
def test_tie_heavy(levels):
    rng = np.random.default_rng(levels)
    vals = rng.standard_normal(levels).astype(np.float32)
    n = 50000
    s = vals[rng.integers(0, levels, n)][None, :]
    got, st = gpu_topk(s, [n], 2048)
    assert st == 0
    _check_rows(s, [n], 2048, got)


def test_concentrated_values():
    """Every score in one quarter-binade: the first 11-bit digit leaves all
    keys in one bin, so the threshold comes from the two lower digits, whose
    histograms hold every key of the row."""
    rng = np.random.default_rng(5)
    n = 100000
    lens = [n, n, n]
    s = np.empty((3, n), np.float32)
    s[0] = 1.0 + 0.25 * rng.random(n, dtype=np.float32) * np.float32(0.999)      # spread over 21 bits
    s[1] = np.float32(1.0) + np.float32(2 ** -12) * rng.integers(0, 8, n)        # spread over the last 11 bits
    s[2] = np.float32(3.0)                                                         # one value
    s[2, 77777] = np.float32(3.5)
    got, st = gpu_topk(s, lens, 2048)
    assert st == 0
    _check_rows(s, lens, 2048, got)


@pytest.mark.parametrize("n_tied", [1, 37, 300, 512, 513, 900])
def test_ties_at_the_threshold(n_tied):
    """A few hundred keys equal to the k-th score, spread over every slice of a
    long row: the list takes them in position order across the slices."""
    rng = np.random.default_rng(1000 + n_tied)
    n = 120000
    s = rng.standard_normal(n).astype(np.float32)
    v = np.float32(np.sort(s)[::-1][2047 - n_tied // 2])  # near rank 2048
    s[rng.choice(n, n_tied, replace=False)] = v
    got, st = gpu_topk(s[None, :], [n], 2048)
    assert st == 0
    _check_rows(s[None, :], [n], 2048, got)


def test_all_zero_row_is_iota():
    s = np.zeros((1, 10000), np.float32)
    got, st = gpu_topk(s, [10000], 2048)
    assert st == 0
    assert np.array_equal(got[0], np.arange(2048))


def test_recent_crowded():
    rng = np.random.default_rng(5)
    n = 131072
    s = np.abs(rng.standard_normal(n)).astype(np.float32)
    s[-4096:] *= 8
    got, st = gpu_topk(s[None, :], [n], 2048)
    assert st == 0
    _check_rows(s[None, :], [n], 2048, got)
    assert checks.list_invariants(got[0], s, 2048) == []


def test_special_values():
    rng = np.random.default_rng(9)
    n = 9000
    s = rng.standard_normal(n).astype(np.float32)
    s[::7] = -0.0
    s[::11] = 0.0
    s[::13] = np.nan
    s[5] = np.inf
    s[6] = -np.inf
    s[100:3000] = np.float32(2.0)  # a tie block crossing the threshold
    got, st = gpu_topk(s[None, :], [n], 2048)
    assert st == 0
    _check_rows(s[None, :], [n], 2048, got)


@pytest.mark.parametrize("k", [1, 7, 100, 1000, 2048])
def test_various_k(k):
    rng = np.random.default_rng(k)
    lens = [5, 3000, 70000]
    s = (rng.integers(-50, 50, (3, 70000)) / 8).astype(np.float32)
    got, st = gpu_topk(s, lens, k)
    assert st == 0
    _check_rows(s, lens, k, got)


def test_scores_past_row_length_are_ignored():
    rng = np.random.default_rng(3)
    s = rng.standard_normal((2, 8000)).astype(np.float32)
    s[0, 5000:] = np.float32(1e30)
    s[1, 7000:] = np.nan
    got, st = gpu_topk(s, [5000, 7000], 2048)
    assert st == 0
    _check_rows(s, [5000, 7000], 2048, got)


def test_row_longer_than_stride_is_reported():
    s = np.ones((1, 64), np.float32)
    got, st = gpu_topk(s, [1000], 8)
    assert st == -6  # IDX_ERR_BOUNDS: the row is clamped to the stride
    assert np.array_equal(got[0], np.arange(8))


def test_deterministic_replays():
    rng = np.random.default_rng(11)
    s = (rng.integers(0, 5, (4, 60000))).astype(np.float32)
    a, _ = gpu_topk(s, [60000, 59999, 30000, 2049], 2048)
    for _ in range(5):
        b, _ = gpu_topk(s, [60000, 59999, 30000, 2049], 2048)
        assert np.array_equal(a, b)


def test_longest_row():
    """A row of the largest length the selection takes (IDX_MAX_TOPK_LEN =
    524,288 keys: 16 slices of 32,768), plus a second row of half of it."""
    rng = np.random.default_rng(524)
    n = 524288
    s = (rng.standard_normal((2, n)) * 3).astype(np.float32)
    lens = [n, n // 2]
    got, st = gpu_topk(s, lens, 2048)
    assert st == 0
    _check_rows(s, lens, 2048, got)



@pytest.mark.parametrize("n", [20000, 131072])
@pytest.mark.parametrize("placement", ["spread", "first_keys", "last_keys"])
@pytest.mark.parametrize("c1", [600, 8192])
def test_crowded_first_digit(n, placement, c1):
    """c1 keys share the k-th key's first digit (scores in [1, 1.25)), 1,000
    lie above it and the rest below; the crowded bin sits spread over the
    row, in its first keys (one or two slices) or in its last keys, and a
    few of its keys tie at the threshold."""
    rng = np.random.default_rng(c1 + n + len(placement))
    s = rng.uniform(0.1, 0.9, n).astype(np.float32)            # below the bin
    if placement == "spread":
        pos = rng.choice(n, 1000 + c1, replace=False)
    elif placement == "first_keys":
        pos = rng.permutation(1000 + c1)
    else:
        pos = n - 1 - rng.permutation(1000 + c1)
    above, cand = pos[:1000], pos[1000:]
    s[above] = rng.uniform(2.0, 4.0, 1000).astype(np.float32)  # above the bin
    s[cand] = (1.0 + 0.2499 * rng.random(c1)).astype(np.float32)
    v = np.sort(s)[::-1][2047]
    s[cand[:17]] = v                                           # ties at the threshold
    got, st = gpu_topk(s[None, :], [n], 2048)
    assert st == 0
    _check_rows(s[None, :], [n], 2048, got)


@pytest.mark.parametrize("placement", ["spread", "first_keys"])
@pytest.mark.parametrize("c1", [4096, 4097, 8192, 8193])
def test_leader_capacity_boundary(placement, c1):
    """A split row whose first digit's threshold bin holds exactly the 4,096
    candidates the leader slice takes, or more (then the two further cluster
    rounds run instead; 8,192 and 8,193 are bins as large as 16 requests x 4
    rows of random keys produce); spread over the row or crowded into its
    first slices, far from the leader (the last slice)."""
    n = 131072
    rng = np.random.default_rng(c1 + len(placement))
    s = rng.uniform(0.1, 0.9, n).astype(np.float32)
    pos = rng.choice(n, 1000 + c1, replace=False) if placement == "spread" else rng.permutation(1000 + c1)
    s[pos[:1000]] = rng.uniform(2.0, 4.0, 1000).astype(np.float32)
    s[pos[1000:]] = (1.0 + 0.2499 * rng.random(c1)).astype(np.float32)
    got, st = gpu_topk(s[None, :], [n], 2048)
    assert st == 0
    _check_rows(s[None, :], [n], 2048, got)


@pytest.mark.parametrize("n", [30000, 131072])
@pytest.mark.parametrize("distinct", [1, 3, 8, 9, 40, 1024])
def test_last_digit_bins(n, distinct):
    """The k-th key shares its top 22 bits with 3,000 keys spread over the
    row, whose last 10 bits take `distinct` values: a slice with at most 8
    non-zero last-digit bins sends them with the last round, one with more
    makes every slice exchange its counts once more."""
    rng = np.random.default_rng(n + distinct)
    s = rng.uniform(0.1, 0.9, n).astype(np.float32)
    pos = rng.choice(n, 4000, replace=False)
    s[pos[:1000]] = rng.uniform(2.0, 4.0, 1000).astype(np.float32)
    low = rng.choice(1024, distinct, replace=False)
    bits = np.uint32(0x3F800000) + low[rng.integers(0, distinct, 3000)].astype(np.uint32)
    s[pos[1000:]] = bits.view(np.float32)          # 1.0 + low / 2^23: one 22-bit prefix
    got, st = gpu_topk(s[None, :], [n], 2048)
    assert st == 0
    _check_rows(s[None, :], [n], 2048, got)


@pytest.mark.parametrize("R,n", [(64, 20000), (200, 13000), (6, 12288), (6, 12289)])
def test_row_count_and_length_mixes(R, n):
    """Launches whose rows the launcher places on one CTA each (up to 12,288
    keys), on clusters of 2 (64 rows of 20,000 keys: larger clusters would
    not all be resident) or on one CTA each again (200 rows)."""
    rng = np.random.default_rng(R * n)
    s = rng.standard_normal((R, n)).astype(np.float32)
    lens = [n - (r % 3) for r in range(R)]
    got, st = gpu_topk(s, lens, 2048)
    assert st == 0
    _check_rows(s, lens, 2048, got)


def _bin_row(n, n_bin, values, n_above, seed):
    """A row of n keys: n_above keys well above, n_bin keys in one first-digit
    bin ([1.0, 1.25): the top 11 bits of the radix image agree) taking the
    given values in turn, the rest far below."""
    rng = np.random.default_rng(seed)
    s = rng.uniform(0.01, 0.1, n).astype(np.float32)
    pos = rng.permutation(n)
    s[pos[:n_above]] = rng.uniform(4.0, 8.0, n_above).astype(np.float32)
    vals = np.asarray(values, dtype=np.float32)
    s[pos[n_above:n_above + n_bin]] = vals[np.arange(n_bin) % vals.size]
    return s


@pytest.mark.parametrize("n,n_bin,n_above", [(8192, 2048, 0), (8192, 2048, 1000), (8189, 2047, 2047),
                                             (12288, 5000, 10), (8192, 511, 1700), (8192, 512, 1700),
                                             (4000, 3000, 0)])
def test_one_cta_bin_of_equal_keys(n, n_bin, n_above):
    """Rows on one CTA whose first digit's threshold bin holds only equal keys
    (as in the tie cache): T is that key, found without the two lower digit
    rounds when the bin holds at least 512 keys; the lists are the oracle's,
    whether the bin's keys all make the list or only some of them."""
    s = _bin_row(n, n_bin, [1.125], n_above, n + n_bin + n_above)[None, :]
    got, st = gpu_topk(s, [n], 2048)
    assert st == 0
    _check_rows(s, [n], 2048, got)


@pytest.mark.parametrize("values", [[1.125, 1.0625], [1.125, np.nextafter(np.float32(1.125), np.float32(2))],
                                    [1.0, 1.1, 1.2, 1.24]])
@pytest.mark.parametrize("n_above", [0, 1500])
def test_one_cta_crowded_bin_of_several_values(values, n_above):
    """A crowded threshold bin on one CTA whose keys are not all equal (two
    values one ulp apart among them): the check finds them unequal and the
    two lower digit rounds pick T; the lists are the oracle's."""
    n = 8192
    s = _bin_row(n, 3000, values, n_above, 7 + n_above + len(values))[None, :]
    got, st = gpu_topk(s, [n], 2048)
    assert st == 0
    _check_rows(s, [n], 2048, got)


def test_short_tied_row_beside_split_rows():
    """A tie-cache-like row short enough to run on one CTA of a cluster launch
    (its other slices leave at once), beside rows split over the cluster."""
    rows, lens = [], [8192, 131072, 9000, 60000]
    width = max(lens)
    for i, n in enumerate(lens):
        if n <= 9000:
            r = _bin_row(n, 2500, [1.125], 300 * i, 40 + i)
        else:
            r = np.random.default_rng(50 + i).standard_normal(n).astype(np.float32)
        rows.append(np.pad(r, (0, width - n)))
    s = np.stack(rows)
    got, st = gpu_topk(s, lens, 2048)
    assert st == 0
    _check_rows(s, lens, 2048, got)
