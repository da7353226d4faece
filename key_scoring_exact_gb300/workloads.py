"""Seeded synthetic inputs for the index chain (scoring + exact top-k).

This module only draws inputs: random query rows, head weights, a paged FP8
key cache with per-key scales, a shuffled block table, row lengths and the
row -> request map.  It holds none of the scoring or selection arithmetic, and
both the GPU path and the CPU oracle are fed from it.

Shapes and distributions follow the workloads of "sgl-amd-mono-upstream PR 18"
(GLM-5.3 indexer launch), section "Modifications / 0. An exact top-k check":
random keys, a tie cache of four repeated keys, all-zero keys, and a cache
whose last 4,096 keys carry 8x scales; row sets of one request's draft chain
(4 verify rows) and of mixed single-row requests, some under 2,048 keys.
Page size 64 tokens, 64 index heads of dimension 128, top-2048.

Every cache is poisoned where no valid read may land: unused physical pages
and the slots past a request's last key hold the E4M3 NaN code 0x7F with a NaN
scale, and block-table entries past a request's pages are -1.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Sequence

import torch

HEADS = 64
DIM = 128
PAGE = 64
TOPK = 2048
E4M3_NAN = 0x7F
EXTRA_POISON_PAGES = 8

CACHE_KINDS = ("random", "ties", "zeros", "recent")


@dataclasses.dataclass
class Workload:
    """One batch of index-chain inputs, all on the CPU.

    q            [R, 64, 128] bfloat16, or uint8 E4M3 codes when q_is_e4m3
    head_w       [R, 64] float32
    k_cache      [pool_pages, 64, 128] uint8 E4M3 codes
    k_scale      [pool_pages, 64] float32
    block_table  [n_req, max_pages] int32 (-1 past a request's pages)
    seq_lens     [R] int32, keys visible to each row
    row_req      [R] int32, request of each row
    req_keys     [n_req] keys held by each request (the longest of its rows)
    """

    name: str
    q: torch.Tensor
    q_is_e4m3: bool
    head_w: torch.Tensor
    k_cache: torch.Tensor
    k_scale: torch.Tensor
    block_table: torch.Tensor
    seq_lens: torch.Tensor
    row_req: torch.Tensor
    req_keys: list
    k: int = TOPK
    recipe: str = ""

    @property
    def R(self) -> int:
        return int(self.q.shape[0])

    @property
    def pool_pages(self) -> int:
        return int(self.k_cache.shape[0])

    @property
    def max_pages(self) -> int:
        return int(self.block_table.shape[1])

    @property
    def max_len(self) -> int:
        return int(self.seq_lens.max().item()) if self.R else 0

    def q_bits(self) -> torch.Tensor:
        """q as raw bits: uint16 for bf16, uint8 for E4M3."""
        return self.q if self.q_is_e4m3 else self.q.view(torch.int16).view(torch.uint16)

    def unique_key_bytes(self) -> int:
        """Bytes of key codes + scales a launch must read, each key once."""
        return sum(self.req_keys) * (DIM + 4)

    def row_keys(self) -> int:
        """Row-key pairs scored (sum of the rows' lengths)."""
        return int(self.seq_lens.sum().item())


def _e4m3_codes(x: torch.Tensor) -> torch.Tensor:
    """Round f32 to E4M3 (nearest-even, as torch's float8_e4m3fn cast) -> codes."""
    return x.to(torch.float8_e4m3fn).view(torch.uint8)


def make_workload(requests: Sequence[Sequence[int]], cache: str = "random", seed: int = 0,
                  q_is_e4m3: bool = False, k: int = TOPK, name: str = "custom",
                  cache_per_request: Sequence[str] | None = None,
                  recent_keys: int = 4096, recent_factor: float = 8.0,
                  shuffle_pages: bool = True, extra_pages: int = EXTRA_POISON_PAGES) -> Workload:
    """Build a workload from per-request row lengths.

    requests[i] lists the lengths seen by request i's rows (consecutive rows).
    cache is one of CACHE_KINDS (or give one per request in cache_per_request).
    """
    g = torch.Generator().manual_seed(int(seed))
    kinds = list(cache_per_request) if cache_per_request is not None else [cache] * len(requests)
    assert len(kinds) == len(requests)
    for kd in kinds:
        if kd not in CACHE_KINDS:
            raise ValueError("unknown cache kind %r" % kd)
    lens = [int(x) for rl in requests for x in rl]
    row_req = [i for i, rl in enumerate(requests) for _ in rl]
    R = len(lens)
    req_keys = [max([int(x) for x in rl], default=0) for rl in requests]
    req_pages = [(n + PAGE - 1) // PAGE for n in req_keys]
    used = sum(req_pages)
    pool_pages = used + int(extra_pages)
    max_pages = max(req_pages + [1])

    k_cache = torch.full((pool_pages, PAGE, DIM), E4M3_NAN, dtype=torch.uint8)
    k_scale = torch.full((pool_pages, PAGE), float("nan"), dtype=torch.float32)
    # The page placement has its own stream, so key values do not depend on it.
    gp = torch.Generator().manual_seed(int(seed) * 1000003 + 1)
    perm = torch.randperm(pool_pages, generator=gp) if shuffle_pages else torch.arange(pool_pages)
    block_table = torch.full((len(requests), max_pages), -1, dtype=torch.int32)

    cursor = 0
    for i, (n, npg, kd) in enumerate(zip(req_keys, req_pages, kinds)):
        phys = perm[cursor:cursor + npg]
        cursor += npg
        block_table[i, :npg] = phys.to(torch.int32)
        if n == 0:
            continue
        if kd == "ties":
            base = _e4m3_codes(torch.randn(4, DIM, generator=g))
            base_scale = torch.rand(4, generator=g) * 1.5 + 0.5
            sel = torch.arange(n) % 4
            codes, scales = base[sel], base_scale[sel]
        elif kd == "zeros":
            codes = torch.zeros(n, DIM, dtype=torch.uint8)
            scales = torch.rand(n, generator=g) * 1.5 + 0.5
        else:
            codes = _e4m3_codes(torch.randn(n, DIM, generator=g))
            scales = torch.rand(n, generator=g) * 1.5 + 0.5
            if kd == "recent":
                scales[max(0, n - recent_keys):] *= recent_factor
        full = torch.full((npg * PAGE, DIM), E4M3_NAN, dtype=torch.uint8)
        full[:n] = codes
        fscale = torch.full((npg * PAGE,), float("nan"), dtype=torch.float32)
        fscale[:n] = scales
        k_cache[phys] = full.view(npg, PAGE, DIM)
        k_scale[phys] = fscale.view(npg, PAGE)

    if q_is_e4m3:
        q = _e4m3_codes(torch.randn(R, HEADS, DIM, generator=g))
    else:
        q = torch.randn(R, HEADS, DIM, generator=g).to(torch.bfloat16)
    head_w = torch.rand(R, HEADS, generator=g) / 8.0
    return Workload(name=name, q=q, q_is_e4m3=q_is_e4m3, head_w=head_w, k_cache=k_cache,
                    k_scale=k_scale, block_table=block_table,
                    seq_lens=torch.tensor(lens, dtype=torch.int32),
                    row_req=torch.tensor(row_req, dtype=torch.int32), req_keys=req_keys, k=k)


def chain(n_keys: int, rows: int = 4) -> list[int]:
    """A draft chain of `rows` verify rows: row i sees n_keys - rows + 1 + i keys."""
    return [n_keys - rows + 1 + i for i in range(rows)]


def mixed_lengths(seed: int, n: int = 16, lo: int = 512, hi: int = 131072,
                  short_below: int = 2048, min_short: int = 3) -> list[int]:
    """n log-uniform lengths in [lo, hi]; if fewer than min_short fall under
    short_below, the first ones are redrawn uniformly from [lo, short_below-1]."""
    g = torch.Generator().manual_seed(int(seed) * 7919 + 17)
    u = torch.rand(n, generator=g, dtype=torch.float64)
    lens = [int(round(math.exp(math.log(lo) + float(x) * (math.log(hi) - math.log(lo))))) for x in u]
    lens = [min(max(v, lo), hi) for v in lens]
    short = sum(1 for v in lens if v < short_below)
    i = 0
    while short < min_short and i < n:
        if lens[i] >= short_below:
            lens[i] = int(torch.randint(lo, short_below, (1,), generator=g).item())
            short += 1
        i += 1
    return lens


# The five configurations: (description, builder).
CONFIG_RECIPES = {
    1: "1 request, 1 row, 4,096 keys; random E4M3 keys N(0,1), scales U(0.5,2); "
       "bf16 q N(0,1); head_w U(0,1)/8; shuffled 64-token pages; k=2048",
    2: "1 request, 4 verify rows seeing 8,189..8,192 keys; tie cache (4 key vectors "
       "repeated, position j uses vector j mod 4); bf16 q; k=2048",
    3: "1 request, 4 verify rows seeing 131,069..131,072 keys; random keys, scales "
       "U(0.5,2), the last 4,096 keys' scales x8; bf16 q; k=2048",
    4: "17 single-row requests: 16 log-uniform lengths in [512, 131,072] (>=3 under "
       "2,048) with random keys, plus one all-zero-key request of 8,192 keys; k=2048",
    5: "16 requests x 4 verify rows at 131,069..131,072 keys; random keys, scales "
       "U(0.5,2), shuffled pages; k=2048",
}


# Workloads beside the five configurations (measured by the benchmark as
# extras): an MTP draft chain of 8 verify rows, whose rows form two groups of
# four that score the same keys.
EXTRA_RECIPES = {
    "chain8": "1 request, 8 verify rows seeing 131,065..131,072 keys; random keys, scales "
              "U(0.5,2), shuffled pages; bf16 q; k=2048",
}


def make_extra(name: str, seed: int = 6, q_is_e4m3: bool = False) -> Workload:
    """One of EXTRA_RECIPES."""
    if name == "chain8":
        w = make_workload([chain(131072, 8)], "random", seed, q_is_e4m3, name="chain8")
    else:
        raise ValueError("extra workloads: %s" % ", ".join(EXTRA_RECIPES))
    w.recipe = EXTRA_RECIPES[name]
    return w


def make_config(idx: int, seed: int | None = None, q_is_e4m3: bool = False) -> Workload:
    """Configuration idx (1..5) with its fixed seed (= idx unless given)."""
    s = idx if seed is None else seed
    if idx == 1:
        w = make_workload([[4096]], "random", s, q_is_e4m3, name="cfg1")
    elif idx == 2:
        w = make_workload([chain(8192)], "ties", s, q_is_e4m3, name="cfg2")
    elif idx == 3:
        w = make_workload([chain(131072)], "recent", s, q_is_e4m3, name="cfg3")
    elif idx == 4:
        lens = mixed_lengths(s)
        reqs = [[n] for n in lens] + [[8192]]
        kinds = ["random"] * len(lens) + ["zeros"]
        w = make_workload(reqs, seed=s, q_is_e4m3=q_is_e4m3, name="cfg4", cache_per_request=kinds)
    elif idx == 5:
        w = make_workload([chain(131072) for _ in range(16)], "random", s, q_is_e4m3, name="cfg5")
    else:
        raise ValueError("configurations are numbered 1..5")
    w.recipe = CONFIG_RECIPES[idx]
    return w


def with_rotation(w: Workload, copies: int) -> tuple[Workload, torch.Tensor]:
    """Replicate the page pool `copies` times; return the enlarged workload and
    one block table per copy ([copies, n_req, max_pages]).  Successive launches
    that cycle through the copies read distinct memory, so a working set larger
    than the L2 cache streams from HBM."""
    pool = w.pool_pages
    kc = w.k_cache.repeat(copies, 1, 1)
    ks = w.k_scale.repeat(copies, 1)
    tables = []
    for c in range(copies):
        bt = w.block_table.clone()
        bt[bt >= 0] += c * pool
        tables.append(bt)
    out = dataclasses.replace(w, k_cache=kc, k_scale=ks, block_table=tables[0].clone())
    return out, torch.stack(tables)
