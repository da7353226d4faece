#!/usr/bin/env python3
"""Benchmark of the index chain: paged key scoring + exact top-2048.

One step = one idx_score_topk launch sequence (scoring, selection) over
one batch of synthetic inputs that are already resident in HBM.  The default
workload is 1 request with 4 verify rows at 131,069..131,072 keys (E4M3 keys
with per-key scales whose last 4,096 keys are 8x, bf16 query, 64 heads x 128,
k = 2048).  Successive steps cycle through enough copies of the key cache
to exceed 2.1 x L2 (17 copies, 294 MB), so keys stream from HBM.

Timing: W untimed warm-up steps, then about 0.8 s of untimed replays while
nvidia-smi starts sampling the clocks, then 7 trials of exactly K steps
replayed from CUDA graphs (a barrier + max over ranks under torchrun); each
trial is bracketed by CUDA events on the launching stream, behind a short
idle kernel so the host has queued the trial before the first event, and the
reported time per step is the median over the trials.  For the per-kernel
roofline, each of the two kernels is then replayed alone from a graph of its
own launches, bracketed by CUDA events.  The FP8 tensor-core rate the scoring
is measured against comes from idx_probe_fp8_mma on the same GPU in the same
run.

Prints one JSON line.  `--impl reference` times the CPU oracle instead (the
plain f64 scoring and sort-based selection) on a bounded sample.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = "µs per indexer launch (score + exact top-2048) at 4 rows, 8K/128K keys; keys/s"
UNIT = "us"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
L2_BYTES = 129 * 1024 * 1024
COPIES = 16
TRIALS = 7


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10000)
    ap.add_argument("--warmup", type=int, default=8)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", type=int, default=3, help="workload configuration 1..5")
    ap.add_argument("--workload", default=None, help="an extra workload instead of --config (chain8)")
    ap.add_argument("--no-chain8", action="store_true", help="skip the 8-row chain measurement")
    ap.add_argument("--copies", type=int, default=COPIES)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-8k", action="store_true")
    ap.add_argument("--no-fp8q", action="store_true", help="skip the FP8-query measurement")
    ap.add_argument("--no-newkeys", action="store_true", help="skip the new-key-store measurement")
    ap.add_argument("--no-ready", action="store_true",
                    help="skip the measurement through idx_score_topk_ready")
    ap.add_argument("--no-batch", action="store_true", help="skip the 64-row measurement")
    ap.add_argument("--no-warm", action="store_true", help="skip the L2-resident measurement")
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="CPU-baseline sample budget")
    return ap.parse_args()


# ---------------------------------------------------------------- distributed

def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
        return dist, rank, world, local
    return None, 0, 1, 0


def barrier(dist):
    if dist is not None:
        dist.barrier()


def max_over_ranks(dist, x: float) -> float:
    if dist is None:
        return x
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# --------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi clock / throttle-reason sampling every 200 ms."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.result = {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["not sampled"]}
        self.path = os.path.join("/tmp", "idx_clocks_%d_%d.csv" % (os.getpid(), gpu_index))

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.Q,
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self) -> dict:
        self.result = self._stop()
        return self.result

    def _stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), float(parts[3]) if parts[3] not in ("[N/A]", "N/A") else 0.0,
                             parts[5], parts[6], parts[7], parts[8]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        reasons = sorted({n for r in rows for n, v in zip(names, r[3:]) if v.lower() == "active"})
        loaded = [r for r in rows if r[2] > 0] or rows
        return {"sm_mhz": statistics.median(r[0] for r in loaded), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows), "power_w_max": max(r[2] for r in rows)}


# ---------------------------------------------------------------------- peaks

def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured"
    return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


def fp8_peak(stream, tries: int = 3) -> dict:
    """The FP8 tcgen05 MMA rate of this GPU, measured now: the best of a few
    runs of idx_probe_fp8_mma (M = 128 x N = 256 x K = 32, the scoring's MMA
    shape, back to back on every SM)."""
    from key_scoring_exact_gb300 import binding
    best = None
    for _ in range(tries):
        r = binding.probe_fp8_mma(8192, 256, stream=stream)
        if best is None or r["tflops"] > best["tflops"]:
            best = r
    best["source"] = "idx_probe_fp8_mma in this run (best of %d)" % tries
    return best


def mma_roofline(st, t_score: float, hbm_floor_s: float, fp8: dict) -> dict:
    """The scoring's tensor-core side: algorithmic flops (2 * 64 * 128 per
    row-key) and the flops the MMAs execute (twice that for a bf16 query,
    split exactly into two E4M3 terms), each against the measured FP8 rate,
    and which floor binds the kernel."""
    alg = st.alg_flops()
    executed = alg * (1 if st.w.q_is_e4m3 or st.quantize_q else 2)
    peak = fp8["tflops"] * 1e12
    floors = {"hbm_us": hbm_floor_s * 1e6, "mma_alg_us": alg / peak * 1e6, "mma_executed_us": executed / peak * 1e6}
    binding_floor = max(floors, key=floors.get)
    return {"alg_flops": alg, "executed_flops": executed, "fp8_peak_tflops": fp8["tflops"],
            "fp8_peak_source": fp8["source"], "fp8_ns_per_mma": fp8["ns_per_mma"], "fp8_probe_mhz": fp8["mhz"],
            "alg_tflops": alg / t_score / 1e12, "executed_tflops": executed / t_score / 1e12,
            "alg_frac": alg / t_score / peak, "executed_frac": executed / t_score / peak,
            "floors": floors, "binding_floor": binding_floor,
            "frac_of_binding_floor": floors[binding_floor] / 1e6 / t_score}


def ncu_traffic(kernel: str, source: str):
    """DRAM bytes (read + write) per launch of `kernel` from the committed ncu
    summary, or None when the kernel's source has changed since the capture."""
    import hashlib
    p = os.path.join(ROOT, "profiles", "traffic.json")
    src = os.path.join(ROOT, "key_scoring_exact_gb300", "csrc", source)
    if not os.path.exists(p) or not os.path.exists(src):
        return None
    rec = json.load(open(p)).get(kernel)
    if not rec:
        return None
    if hashlib.sha256(open(src, "rb").read()).hexdigest() != rec.get("source_sha256"):
        return None
    return rec.get("dram_bytes_per_launch")


# ------------------------------------------------------------ the GPU bench

class Step:
    """Device buffers for one configuration and its rotation copies."""

    def __init__(self, w, copies, dev):
        from key_scoring_exact_gb300 import binding, workloads as W
        self.binding = binding
        self.w = w
        big, tables = W.with_rotation(w, copies)
        self.copies = copies
        self.q = w.q.to(dev)
        self.head_w = w.head_w.to(dev)
        self.k_cache = big.k_cache.to(dev)
        self.k_scale = big.k_scale.to(dev)
        self.tables = [tables[c].contiguous().to(dev) for c in range(copies)]
        self.seq_lens = w.seq_lens.to(dev)
        self.row_req = w.row_req.to(dev)
        self.R, self.k, self.max_len = w.R, w.k, w.max_len
        self.stride = (self.max_len + 3) // 4 * 4
        self.scores = torch.zeros(self.R, self.stride, dtype=torch.float32, device=dev)
        self.idx = torch.zeros(self.R, self.k, dtype=torch.int32, device=dev)
        self.ws = binding.new_workspace(self.R, self.max_len, self.k, device=dev)

    quantize_q = False  # score the on-device FP8 quantisation of the bf16 query

    new_keys = None  # (new_k [R, 128] E4M3 codes, new_scale [R]): each step stores its rows' keys first

    inputs_ready = False  # idx_score_topk_ready: metadata and keys complete when each call is enqueued

    def fused(self, c, stream=None):
        b = self.binding
        if self.new_keys is not None:
            b.score_topk_newkeys(self.q, self.head_w, self.k_cache, self.k_scale, self.tables[c % self.copies],
                                 self.seq_lens, self.row_req, self.new_keys[0], self.new_keys[1], self.max_len,
                                 self.k, self.idx, self.ws, scores=self.scores, stream=stream,
                                 quantize_q=self.quantize_q)
            return
        b.score_topk(self.q, self.head_w, self.k_cache, self.k_scale, self.tables[c % self.copies],
                     self.seq_lens, self.row_req, self.max_len, self.k, self.idx, self.ws,
                     scores=self.scores, stream=stream, quantize_q=self.quantize_q,
                     inputs_ready=self.inputs_ready)

    def score_only(self, c, stream=None):
        self.binding.score(self.q, self.head_w, self.k_cache, self.k_scale, self.tables[c % self.copies],
                           self.seq_lens, self.row_req, self.scores, self.ws, stream=stream,
                           quantize_q=self.quantize_q)

    def select_only(self, stream=None):
        self.binding.topk(self.scores, self.seq_lens, self.k, self.idx, self.ws, stream=stream)

    def key_bytes(self):
        return self.w.unique_key_bytes()

    def alg_bytes_score(self):
        """HBM bytes the scoring must move: every key + scale once, the query,
        head weights and block-table entries in, one f32 score per (row, key) out."""
        w = self.w
        pages = sum((n + 63) // 64 for n in w.req_keys)
        return (self.key_bytes() + w.R * 64 * 128 * (1 if w.q_is_e4m3 else 2) + w.R * 64 * 4
                + pages * 4 + 4 * w.row_keys())

    def alg_bytes_select(self):
        """HBM bytes of the selection: every score read once, k indices written."""
        return 4 * self.w.row_keys() + 4 * self.R * self.k

    def alg_flops(self):
        """MMA flops of the algorithm: 2 * 64 heads * 128 dims per (row, key)."""
        return 2 * 64 * 128 * self.w.row_keys()


def capture(stream, fn, n):
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for i in range(n):
            fn(i)
    return g


def _idle(stream, us: float = 100.0):
    """A short spin kernel on the stream: while it runs, the host queues the
    next trial, so the trial's first event is not followed by launch latency."""
    with torch.cuda.stream(stream):
        torch.cuda._sleep(int(us * 2000))


def time_graph_steps(st: Step, steps: int, stream, dist, sampler=None, trials: int = TRIALS,
                     settle_s: float = 0.8):
    """`trials` timed trials of exactly `steps` fused steps each, replayed from
    CUDA graphs and bracketed by CUDA events on the launching stream.
    Consecutive steps use consecutive key-cache copies (trials of up to 256
    steps continue the rotation where the previous trial stopped).  With a
    sampler, the clocks are sampled from `settle_s` seconds of untimed replays
    before the first trial until the last one ends.  Returns (median seconds
    per step over the trials, per-trial seconds per step)."""
    G = 255 // st.copies * st.copies if st.copies <= 255 else st.copies  # a whole number of rotations
    cache = {}

    def graph(n, start):
        key = (n, start % st.copies)
        if key not in cache:
            cache[key] = capture(stream, lambda i: st.fused(start + i, stream), n)
        return cache[key]

    plan = []
    for t in range(trials):
        if steps <= 256:
            plan.append([graph(steps, t * steps)])   # one graph; the rotation continues across trials
        else:
            full, rem = divmod(steps, G)             # starts at copy 0
            plan.append([graph(G, 0)] * full + ([graph(rem, 0)] if rem else []))
    for gl in plan:                                  # upload + warm every graph
        for g in gl:
            g.replay()
    torch.cuda.synchronize()
    if sampler is not None:
        sampler.start()
        t_end = time.perf_counter() + settle_s
        while time.perf_counter() < t_end:
            for g in plan[0]:
                g.replay()
            torch.cuda.synchronize()
    barrier(dist)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in plan]
    for (e0, e1), gl in zip(ev, plan):
        _idle(stream)
        e0.record(stream)
        for g in gl:
            g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    if sampler is not None:
        sampler.stop()
    barrier(dist)
    torch.cuda.synchronize()
    per = [e0.elapsed_time(e1) / 1e3 / steps for e0, e1 in ev]
    return statistics.median(per), per


def per_kernel_times(st: Step, n: int, stream):
    """Average launch duration of each kernel: n scoring launches (rotating
    key-cache copies) replayed from one graph, then n selection launches from
    another, each bracketed by CUDA events on the launching stream.  Timing
    each kernel in a graph of its own keeps the launch pipelined, as it is in
    the fused steps; events placed between the two kernels of every step
    would add the launch latency to both.  Returns mean seconds of each."""
    out = []
    for body in (lambda i: st.score_only(i, stream), lambda i: st.select_only(stream)):
        g = capture(stream, body, n)
        g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        g.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        out.append(e0.elapsed_time(e1) / 1e3 / n)
        del g
    return out[0], out[1]


def copies_for(w, minimum: int) -> int:
    """Key-cache copies whose total exceeds 2.1 x L2."""
    need = int(np.ceil(2.1 * L2_BYTES / max(1, w.unique_key_bytes())))
    return max(minimum, need)


def e2e_time(st: Step, steps: int, stream):
    """Through the public C ABI with host buffers: each step is one
    idx_score_topk_host call, which copies that step's inputs (query, head
    weights, block table, row lengths, row map) from pinned host memory,
    runs the scoring and the selection, and copies the indices back to pinned
    host memory.  The key cache is device-resident state (the serving KV
    cache), not a per-step input.  Steps are issued back to back on one
    stream; the timed region ends once the last step's indices are on the
    host."""
    w = st.w
    host_q, host_w = w.q.contiguous().pin_memory(), w.head_w.contiguous().pin_memory()
    host_tables = [t.cpu().contiguous().pin_memory() for t in st.tables]
    host_lens, host_req = w.seq_lens.contiguous().pin_memory(), w.row_req.contiguous().pin_memory()
    out_host = torch.empty(st.R, st.k, dtype=torch.int32).pin_memory()
    b = st.binding
    n_req, max_pages = host_tables[0].shape
    ws = b.new_host_workspace(st.R, st.max_len, st.k, n_req, max_pages)
    h2d = (host_q.numel() * host_q.element_size() + host_w.numel() * 4 + host_tables[0].numel() * 4
           + 2 * st.R * 4)
    d2h = st.R * st.k * 4

    def one(i):
        b.score_topk_host(host_q, host_w, st.k_cache, st.k_scale, host_tables[i % st.copies], host_lens,
                          host_req, st.max_len, st.k, out_host, ws, stream=stream)

    with torch.cuda.stream(stream):
        for i in range(3):
            one(i)
        torch.cuda.synchronize()
        if b.check_status(ws, stream) != 0:
            raise RuntimeError("device status in the end-to-end warm-up")
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(steps):
            one(i)
        e1.record(stream)
        torch.cuda.synchronize()
    return e0.elapsed_time(e1) / 1e3 / steps, h2d, d2h


# ------------------------------------------------------------ CPU oracle leg

def _oracle_problem(w, keys_per_row: int):
    import oracle
    lens = w.seq_lens.numpy()
    sample = np.minimum(lens, max(1, int(keys_per_row))).astype(np.int32)
    pb = oracle.Problem(w.q_bits().numpy(), w.q_is_e4m3, w.head_w.numpy(), w.k_cache.numpy(),
                        w.k_scale.numpy(), w.block_table.numpy(), sample, w.row_req.numpy())
    return pb, sample


def _oracle_run(w, keys_per_row: int, threads: int = 1):
    """Oracle scores of every row over its first keys_per_row keys, then the
    sort-based top-k of those scores.  With threads > 1 the unchanged oracle
    calls run on a pool of host threads (the C oracle releases the GIL):
    scores over (row, key-chunk) tasks, then one top-k per row.  Returns
    (seconds, row-keys done)."""
    import oracle
    pb, sample = _oracle_problem(w, keys_per_row)
    if threads <= 1:
        t0 = time.perf_counter()
        s = oracle.scores(pb)
        for r in range(w.R):
            oracle.topk(s[r, :sample[r]].astype(np.float32), w.k)
        return time.perf_counter() - t0, int(sample.sum())
    from concurrent.futures import ThreadPoolExecutor
    tasks = []
    for r in range(w.R):
        n = int(sample[r])
        chunk = max(64, -(-n * w.R // (4 * threads)))
        tasks += [(r, a, min(n, a + chunk)) for a in range(0, n, chunk)]
    t0 = time.perf_counter()
    with ThreadPoolExecutor(max_workers=threads) as ex:
        parts = list(ex.map(lambda t: oracle.score_positions(pb, t[0], np.arange(t[1], t[2])), tasks))
        rows = [np.concatenate([p for t, p in zip(tasks, parts) if t[0] == r] or [np.zeros(0)])
                for r in range(w.R)]
        list(ex.map(lambda r: oracle.topk(rows[r].astype(np.float32), w.k), range(w.R)))
    return time.perf_counter() - t0, int(sample.sum())


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_launch_time(w, budget_s: float, threads: int = 1):
    """The oracle as it stands, timed on a bounded sample sized to take about
    budget_s seconds of CPU work, scaled to one whole launch (per row-key),
    on `threads` host threads."""
    lens = w.seq_lens.numpy()
    t, done = _oracle_run(w, 256)                       # calibration, one thread
    per_rowkey = t / done
    keys = int(min(lens.max(), max(256, budget_s / per_rowkey / w.R)))
    t, done = _oracle_run(w, keys, threads)
    total = float(lens.sum())
    desc = ("all %d rows over their first %d keys: %d of %d row-keys (%.3g of the launch), "
            "time scaled by row-keys, %d host thread%s" % (w.R, keys, done, int(total), done / total, threads,
                                                          "" if threads == 1 else "s"))
    return t * total / done, desc


def reference_main(args, w):
    dist, rank, world, _ = dist_setup(args)
    if rank != 0:
        return
    # the whole run (warm-up + steps) stays within about two minutes
    per_step = max(0.02, min(20.0, 120.0 / max(1, args.steps + args.warmup)))
    cores = host_cores()
    times = []
    desc = ""
    for i in range(args.warmup + args.steps):
        t, desc = oracle_launch_time(w, per_step * cores, cores)
        if i >= args.warmup:
            times.append(t)
    us = float(np.mean(times)) * 1e6
    line = {"impl": "reference", "metric": METRIC, "value": us, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": us / 1e3, "higher_is_better": False,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_desc(w, args),
            "cpu_baseline": {"value": us, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": desc},
            "e2e": {"value": us, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def config_desc(w, args):
    return {"workload": w.recipe, "rows": w.R,
            "requests": len(w.req_keys), "keys_per_row": [int(x) for x in w.seq_lens.tolist()][:8],
            "heads": 64, "dim": 128, "page": 64, "k": w.k, "query": "bf16" if not w.q_is_e4m3 else "e4m3",
            "l2": "inputs rotate over %d key-cache copies (%.0f MB > 2x L2)" % (
                args.copies, args.copies * w.unique_key_bytes() / 1e6),
            "parallelism": "replicas" if args.gpus > 1 else "1 GPU"}


def main():
    args = parse()
    from key_scoring_exact_gb300 import workloads as W
    w = W.make_extra(args.workload) if args.workload else W.make_config(args.config)
    args.copies = copies_for(w, args.copies)   # the same rotation (and config line) in both arms
    if args.impl == "reference":
        reference_main(args, w)
        return
    if not torch.cuda.is_available():
        print(json.dumps({"error": "no CUDA device"}))
        sys.exit(1)
    dist, rank, world, local = dist_setup(args)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    from key_scoring_exact_gb300 import binding
    binding.load(build_if_missing=True)
    stream = torch.cuda.Stream(device=dev)
    st = Step(w, args.copies, dev)

    sampler = ClockSampler(local)
    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            st.fused(i, stream)
        torch.cuda.synchronize()
        if binding.check_status(st.ws, stream) != 0:
            raise RuntimeError("device status after warm-up")
        sec, trial_secs = time_graph_steps(st, args.steps, stream, dist, sampler)
    clocks = sampler.result
    sec = max_over_ranks(dist, sec)
    with torch.cuda.stream(stream):
        t_score, t_select = per_kernel_times(st, min(args.steps, 256), stream)
        status = binding.check_status(st.ws, stream)
    if status != 0:
        raise RuntimeError("device status %d after the timed steps" % status)

    hbm, bf16, bf16_sus, src = peaks()
    with torch.cuda.stream(stream):
        fp8 = fp8_peak(stream)
    score_bytes = st.alg_bytes_score()
    select_bytes = st.alg_bytes_select()
    roof_score = {"kernel": "k_score", "bound": "hbm",
                  "achieved": score_bytes / t_score / 1e9, "peak": hbm, "unit": "GB/s",
                  "frac": score_bytes / t_score / 1e9 / hbm, "traffic": ncu_traffic("k_score", "score.cu"),
                  "alg_bytes": score_bytes, "us": t_score * 1e6, "peak_source": src}
    roof_select = {"kernel": "k_select", "bound": "hbm",
                   "achieved": select_bytes / t_select / 1e9, "peak": hbm, "unit": "GB/s",
                   "frac": select_bytes / t_select / 1e9 / hbm, "traffic": ncu_traffic("k_select", "select.cu"),
                   "alg_bytes": select_bytes, "us": t_select * 1e6, "peak_source": src}
    dominant, other = (roof_score, roof_select) if t_score >= t_select else (roof_select, roof_score)
    fused_bytes = st.key_bytes() + 4 * st.R * st.k
    line = {
        "metric": METRIC, "value": sec * 1e6, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": sec * 1e3, "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "e4m3 MMA, f32 accumulate, u32 radix", "data": "synthetic",
        "config": config_desc(w, args),
        "keys_per_s": world * w.row_keys() / sec,
        "unique_keys_per_s": world * sum(w.req_keys) / sec,
        "roofline": dominant,
        "roofline_other": other,
        "roofline_fused": {"alg_bytes": fused_bytes, "roof_us": fused_bytes / hbm / 1e3,
                           "frac": fused_bytes / hbm / 1e3 / (sec * 1e6)},
        "mma": mma_roofline(st, t_score, score_bytes / (hbm * 1e9), fp8),
        "trials": {"n": len(trial_secs), "steps_each": args.steps,
                   "per_step_us": [round(x * 1e6, 3) for x in trial_secs],
                   "mean_us": float(np.mean(trial_secs)) * 1e6, "statistic": "median"},
        "gpu_launches": 3 * args.steps,           # per timed trial (query prep, scoring, selection per step)
        "gpu_launches_all_trials": 3 * args.steps * len(trial_secs),
        "clocks": clocks,
    }
    if not args.no_8k:
        w8 = W.make_config(2)
        st8 = Step(w8, copies_for(w8, args.copies), dev)
        with torch.cuda.stream(stream):
            for i in range(3):
                st8.fused(i, stream)
            sec8, _ = time_graph_steps(st8, min(args.steps, 1024), stream, None)
        line["also_8k"] = {"workload": w8.recipe, "us": sec8 * 1e6,
                           "keys_per_s": w8.row_keys() / sec8}
        del st8
    if not args.no_warm:
        # the same workload with a single key-cache copy, which stays in L2
        # between steps (the figure beside the rotated, HBM-bound one)
        stw = Step(w, 1, dev)
        with torch.cuda.stream(stream):
            for i in range(3):
                stw.fused(i, stream)
            secw, _ = time_graph_steps(stw, min(args.steps, 4096), stream, None)
        line["also_warm_l2"] = {"workload": w.recipe + "; one key-cache copy, resident in L2 between steps",
                                "us": secw * 1e6, "keys_per_s": w.row_keys() / secw}
        del stw
    if not args.no_batch:
        # batch context: 16 requests x 4 verify rows (64 rows, 277 MB of keys)
        wb = W.make_config(5)
        stb = Step(wb, copies_for(wb, 2), dev)
        with torch.cuda.stream(stream):
            for i in range(3):
                stb.fused(i, stream)
            secb, _ = time_graph_steps(stb, min(args.steps, 64), stream, None)
            tb_score, tb_select = per_kernel_times(stb, min(args.steps, 32), stream)
        line["also_64_rows"] = {"workload": wb.recipe, "us": secb * 1e6, "scoring_us": tb_score * 1e6,
                                "selection_us": tb_select * 1e6,
                                "scoring_gbs_of_keys": wb.unique_key_bytes() / tb_score / 1e9,
                                "keys_per_s": wb.row_keys() / secb}
        del stb
    if not args.no_chain8 and not args.workload:
        # an MTP chain of 8 verify rows: two groups of four rows whose key
        # reads run on different CTAs at the same time (the second from L2)
        wc = W.make_extra("chain8")
        stc = Step(wc, copies_for(wc, 2), dev)
        with torch.cuda.stream(stream):
            for i in range(3):
                stc.fused(i, stream)
            secc, _ = time_graph_steps(stc, min(args.steps, 1024), stream, None)
            tc_score, tc_select = per_kernel_times(stc, min(args.steps, 256), stream)
        line["also_chain8"] = {"workload": wc.recipe, "us": secc * 1e6, "scoring_us": tc_score * 1e6,
                               "selection_us": tc_select * 1e6, "keys_per_s": wc.row_keys() / secc,
                               "dram_read_bytes_per_scoring_launch": ncu_traffic("k_score_chain8", "score.cu"),
                               "unique_key_bytes": wc.unique_key_bytes()}
        del stc
    if not args.no_fp8q and not w.q_is_e4m3:
        # the same workload with the query quantised to E4M3 on the device (one
        # E4M3 term: half the MMAs); scores are those of the quantised query
        st.quantize_q = True
        with torch.cuda.stream(stream):
            for i in range(3):
                st.fused(i, stream)
            secq, _ = time_graph_steps(st, min(args.steps, 4096), stream, None)
            tq_score, _ = per_kernel_times(st, min(args.steps, 256), stream)
        st.quantize_q = False
        line["also_fp8_query"] = {"workload": w.recipe + "; query quantised to E4M3 on the device per (row, head)",
                                  "us": secq * 1e6, "scoring_us": tq_score * 1e6,
                                  "keys_per_s": w.row_keys() / secq}
    if not args.no_newkeys:
        # the same workload as a decode step that brings its rows' own keys:
        # every step stores each row's key in its slot, then scores and selects
        g = torch.Generator().manual_seed(7)
        st.new_keys = (torch.randn(w.R, 128, generator=g).to(torch.float8_e4m3fn).view(torch.uint8).to(dev),
                       (torch.rand(w.R, generator=g) * 1.5 + 0.5).to(dev))
        with torch.cuda.stream(stream):
            for i in range(3):
                st.fused(i, stream)
            secn, _ = time_graph_steps(st, min(args.steps, 4096), stream, None)
        st.new_keys = None
        line["also_new_keys"] = {"workload": w.recipe + "; each step first stores its rows' new keys "
                                 "(idx_score_topk_newkeys)", "us": secn * 1e6, "keys_per_s": w.row_keys() / secn}
    if not args.no_ready:
        # the same workloads through idx_score_topk_ready: the block tables,
        # lengths, row map and key cache are written once before the timed
        # steps, so each call's scoring set-up may overlap the previous
        # call's selection
        ready = {}
        st.inputs_ready = True
        with torch.cuda.stream(stream):
            for i in range(3):
                st.fused(i, stream)
            secr, _ = time_graph_steps(st, min(args.steps, 4096), stream, None)
        st.inputs_ready = False
        ready["us"] = secr * 1e6
        ready["keys_per_s"] = w.row_keys() / secr
        if not args.no_8k and not args.workload and args.config == 3:
            w8 = W.make_config(2)
            st8 = Step(w8, copies_for(w8, args.copies), dev)
            st8.inputs_ready = True
            with torch.cuda.stream(stream):
                for i in range(3):
                    st8.fused(i, stream)
                sec8r, _ = time_graph_steps(st8, min(args.steps, 1024), stream, None)
            ready["us_4x8k"] = sec8r * 1e6
            del st8
        line["also_inputs_ready"] = dict({"workload": w.recipe + "; through idx_score_topk_ready (block tables, "
                                          "lengths, row map and keys complete before each call)"}, **ready)
    if not args.no_e2e:
        e2e_sec, h2d, d2h = e2e_time(st, min(args.steps, 200), stream)
        line["e2e"] = {"value": e2e_sec * 1e6, "unit": UNIT, "h2d_bytes_per_step": h2d,
                       "d2h_bytes_per_step": d2h}
    if rank == 0 and not args.no_cpu_baseline and world == 1:
        cores = host_cores()
        t1, desc1 = oracle_launch_time(w, args.cpu_seconds)
        tn, descn = oracle_launch_time(w, args.cpu_seconds, cores)
        line["cpu_baseline"] = {"value": tn * 1e6, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": descn,
                                "one_core": {"value": t1 * 1e6, "cores": 1, "sample": desc1}}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
