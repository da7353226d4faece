"""Pure-Python brute-force selection for tiny inputs (test infrastructure).

It rebuilds the exact top-k list from the definition alone, with no sort: a
key is in the top-k set when fewer than k other keys beat it, where key i beats
key j if its score is larger, or equal and at a lower position (NaN scores
rank below every number and tie with each other).  The list then holds the
set's keys strictly above the set's lowest score in ascending position,
followed by the set's keys tied with that score, in ascending position.  Rows
with n <= k keep every key and pad with -1.

The definitions come from "sgl-amd-mono-upstream PR 18" (GLM-5.3 indexer
launch), section "Modifications / 0. An exact top-k check" (the exact top-k
set by score descending, then position) and the list order of this library
(keys above the k-th score first, then its ties, each in position order).
Quadratic: for n up to a few hundred only.
"""
from __future__ import annotations

import math


def _above(a: float, b: float) -> bool:
    if math.isnan(a):
        return False
    if math.isnan(b):
        return True
    return a > b


def _tied(a: float, b: float) -> bool:
    if math.isnan(a) or math.isnan(b):
        return math.isnan(a) and math.isnan(b)
    return a == b


def _beats(s, i: int, j: int) -> bool:
    return _above(s[i], s[j]) or (_tied(s[i], s[j]) and i < j)


def topk(scores, k: int) -> list[int]:
    s = [float(x) for x in scores]
    n = len(s)
    if n <= k:
        return list(range(n)) + [-1] * (k - n)
    beaten_by = [sum(1 for i in range(n) if i != j and _beats(s, i, j)) for j in range(n)]
    chosen = [j for j in range(n) if beaten_by[j] < k]
    assert len(chosen) == k
    last = next(j for j in range(n) if beaten_by[j] == k - 1)
    t = s[last]
    above = [j for j in chosen if _above(s[j], t)]
    tied = [j for j in chosen if _tied(s[j], t)]
    return sorted(above) + sorted(tied)
