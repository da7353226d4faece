"""The five configurations end to end through idx_score_topk (the launch the
benchmark times): every score within 1e-4 of the f64 oracle (the largest
configuration on sampled positions), and every row's list bit-exact against
the oracle's selection of the GPU's own scores."""
import numpy as np
import pytest
import torch

import oracle
from key_scoring_exact_gb300 import binding
from key_scoring_exact_gb300 import workloads as W
from tests import checks
from tests.gpu_util import device_inputs, gpu_fused, problem, stride_for

pytestmark = pytest.mark.gpu


def _lists_exact(w, s, got):
    for r, n in enumerate(w.seq_lens.tolist()):
        exp = oracle.topk(s[r, :n], w.k)
        assert np.array_equal(got[r], exp), "row %d list differs" % r
        assert checks.list_invariants(got[r], s[r, :n], w.k) == []


@pytest.mark.parametrize("idx", [1, 2, 3, 4])
def test_config_full(idx):
    w = W.make_config(idx)
    s, got, st = gpu_fused(w)
    assert st == 0
    ref = oracle.scores(problem(w))
    errs = checks.score_errors(s, ref, w.seq_lens.tolist())
    assert max(errs) <= checks.SCORE_TOL, errs
    print("%s: worst relative score error %.3g" % (w.recipe, max(errs)))
    _lists_exact(w, s, got)


def test_config5_sampled():
    w = W.make_config(5)
    s, got, st = gpu_fused(w)
    assert st == 0
    pb = problem(w)
    rng = np.random.default_rng(55)
    worst = 0.0
    for r, n in enumerate(w.seq_lens.tolist()):
        pos = np.unique(np.concatenate([[0, 1, 63, 64, 127, 128, n - 2, n - 1],
                                        rng.integers(0, n, 40),
                                        np.argsort(-s[r, :n])[:8]])).astype(np.int64)
        ref = oracle.score_positions(pb, r, pos)
        # the row's largest reference score, from its top GPU candidates
        denom = np.max(np.abs(ref))
        err = np.max(np.abs(s[r, pos] - ref)) / denom
        worst = max(worst, err)
    assert worst <= checks.SCORE_TOL, worst
    print("16 requests x 4 rows x 131K keys: worst sampled relative score error %.3g" % worst)
    _lists_exact(w, s, got)


def test_chain_of_eight_rows():
    """An MTP draft chain of 8 verify rows at 131K keys (two groups of four
    rows scoring the same keys): every score within 1e-4, every list exact."""
    w = W.make_extra("chain8")
    s, got, st = gpu_fused(w)
    assert st == 0
    ref = oracle.scores(problem(w))
    errs = checks.score_errors(s, ref, w.seq_lens.tolist())
    assert max(errs) <= checks.SCORE_TOL, errs
    _lists_exact(w, s, got)


def test_scores_in_workspace():
    w = W.make_config(1)
    s1, got1, st1 = gpu_fused(w)
    s2, got2, st2 = gpu_fused(w, in_workspace=True)
    assert st1 == 0 and st2 == 0
    n = w.seq_lens[0].item()
    assert np.array_equal(s1[:, :n], s2[:, :n]) and np.array_equal(got1, got2)


def test_config3_e4m3_query():
    w = W.make_config(3, q_is_e4m3=True)
    s, got, st = gpu_fused(w)
    assert st == 0
    ref = oracle.scores(problem(w))
    errs = checks.score_errors(s, ref, w.seq_lens.tolist())
    assert max(errs) <= checks.SCORE_TOL, errs
    _lists_exact(w, s, got)


def test_fused_replay_determinism():
    w = W.make_config(2)
    t = device_inputs(w)
    s0, g0, _ = gpu_fused(w, t)
    for _ in range(10):
        s1, g1, _ = gpu_fused(w, t)
        assert np.array_equal(s0, s1) and np.array_equal(g0, g1)


def test_fused_calls_share_one_workspace():
    """One workspace across fused calls of different shapes: each call's
    lists equal the oracle's lists of its own scores (nothing a call leaves
    in the workspace changes the next one)."""
    ws = binding.new_workspace(17, 131072, 2048)
    for cfg in (2, 4, 1, 2, 3):
        w = W.make_config(cfg)
        t = device_inputs(w)
        idx = torch.full((w.R, w.k), -7, dtype=torch.int32, device="cuda")
        scores = torch.zeros(w.R, stride_for(w.max_len), dtype=torch.float32, device="cuda")
        binding.score_topk(t["q"], t["head_w"], t["k_cache"], t["k_scale"], t["block_table"],
                           t["seq_lens"], t["row_req"], w.max_len, w.k, idx, ws, scores=scores)
        assert binding.check_status(ws) == 0
        _lists_exact(w, scores.cpu().numpy(), idx.cpu().numpy())


@pytest.mark.parametrize("cfg,pinned", [(2, True), (4, True), (1, False)])
def test_host_buffer_call_matches_device_call(cfg, pinned):
    """idx_score_topk_host (inputs and indices in host memory, page-locked or
    not) gives the device call's lists."""
    w = W.make_config(cfg)
    t = device_inputs(w)
    _, ref, st = gpu_fused(w, t)
    assert st == 0
    host = lambda x: x.contiguous().pin_memory() if pinned else x.contiguous()
    ws = binding.new_host_workspace(w.R, w.max_len, w.k, w.block_table.shape[0], w.block_table.shape[1])
    out = host(torch.full((w.R, w.k), -7, dtype=torch.int32))
    binding.score_topk_host(host(w.q), host(w.head_w), t["k_cache"], t["k_scale"], host(w.block_table),
                            host(w.seq_lens), host(w.row_req), w.max_len, w.k, out, ws)
    torch.cuda.synchronize()
    assert binding.check_status(ws) == 0
    assert np.array_equal(out.numpy(), ref)


def test_host_buffer_calls_on_a_stream():
    """On an explicit stream with every buffer page-locked, idx_score_topk_host
    calls issued back to back with no synchronisation (each call's gather
    reading its host inputs while the previous call's selection still runs),
    alternating workloads of different shapes and inputs, each into its own
    host indices and all through one workspace per shape, give the device
    call's lists."""
    loads = [W.make_config(4), W.make_config(2), W.make_config(4, seed=44), W.make_config(1), W.make_config(4)]
    refs, args = [], []
    for w in loads:
        t = device_inputs(w)
        _, ref, st = gpu_fused(w, t)
        assert st == 0
        refs.append(ref)
        pin = lambda x: x.contiguous().pin_memory()
        ws = binding.new_host_workspace(w.R, w.max_len, w.k, w.block_table.shape[0], w.block_table.shape[1])
        out = pin(torch.full((w.R, w.k), -7, dtype=torch.int32))
        args.append((pin(w.q), pin(w.head_w), t["k_cache"], t["k_scale"], pin(w.block_table), pin(w.seq_lens),
                     pin(w.row_req), w.max_len, w.k, out, ws))
    stream = torch.cuda.Stream()
    binding.score_topk_host(*args[0], stream=stream)
    stream.synchronize()
    args[0][9].fill_(-7)
    for a in args:
        binding.score_topk_host(*a, stream=stream)
    stream.synchronize()
    for a, ref in zip(args, refs):
        assert binding.check_status(a[10], stream) == 0
        assert np.array_equal(a[9].numpy(), ref)


def test_back_to_back_calls_share_a_workspace():
    """Fused device calls issued back to back on one stream with no
    synchronisation, alternating two workloads, all with the scores in one
    shared workspace: each scoring launch may start while the previous
    selection runs (a programmatic dependent of it) and must not overwrite
    the scores that selection still reads.  Every call's lists equal the
    workload's own."""
    loads = [W.make_config(3), W.make_config(4)]
    tens = [device_inputs(w) for w in loads]
    refs = []
    for w, t in zip(loads, tens):
        _, ref, st = gpu_fused(w, t, in_workspace=True)
        assert st == 0
        refs.append(ref)
    R = max(w.R for w in loads)
    max_len = max(w.max_len for w in loads)
    ws = binding.new_workspace(R, max_len, 2048, with_scores=True)
    stream = torch.cuda.Stream()
    outs = []
    for i in range(6):
        w, t = loads[i % 2], tens[i % 2]
        idx = torch.full((w.R, w.k), -7, dtype=torch.int32, device="cuda")
        binding.score_topk(t["q"], t["head_w"], t["k_cache"], t["k_scale"], t["block_table"], t["seq_lens"],
                           t["row_req"], w.max_len, w.k, idx, ws, stream=stream)
        outs.append(idx)
    stream.synchronize()
    assert binding.check_status(ws, stream) == 0
    for i, idx in enumerate(outs):
        assert np.array_equal(idx.cpu().numpy(), refs[i % 2]), "call %d" % i


def test_host_buffer_call_argument_error():
    """An argument error of the fused call (a key cache that is not 16-byte
    aligned) is returned by the host-buffer call before it launches anything,
    and the stream stays usable: the next call gives the device call's
    lists."""
    w = W.make_config(1)
    t = device_inputs(w)
    _, ref, st = gpu_fused(w, t)
    assert st == 0
    pin = lambda x: x.contiguous().pin_memory()
    q, hw, bt, sl, rq = pin(w.q), pin(w.head_w), pin(w.block_table), pin(w.seq_lens), pin(w.row_req)
    out = pin(torch.full((w.R, w.k), -7, dtype=torch.int32))
    ws = binding.new_host_workspace(w.R, w.max_len, w.k, w.block_table.shape[0], w.block_table.shape[1])
    stream = torch.cuda.Stream()
    lib = binding.load()

    def call(kc_offset):
        return lib.idx_score_topk_host(0, q.data_ptr(), hw.data_ptr(), t["k_cache"].data_ptr() + kc_offset,
                                       t["k_scale"].data_ptr(), t["k_cache"].shape[0], bt.data_ptr(),
                                       bt.shape[0], bt.shape[1], sl.data_ptr(), rq.data_ptr(), w.R, w.max_len,
                                       w.k, out.data_ptr(), ws.data_ptr(), ws.numel(), stream.cuda_stream)
    assert call(0) == 0 and call(0) == 0
    assert call(1) == -2                   # IDX_ERR_ALIGN
    with torch.cuda.stream(stream):
        assert not torch.cuda.is_current_stream_capturing()
    out.fill_(-7)
    assert call(0) == 0
    stream.synchronize()
    assert binding.check_status(ws, stream) == 0
    assert np.array_equal(out.numpy(), ref)


@pytest.mark.parametrize("cfg", [2, 4])
def test_slot_lists(cfg):
    """idx_score_topk_slots: the same lists as idx_score_topk, each position
    replaced by its physical cache slot (the oracle's mapping)."""
    w = W.make_config(cfg)
    t = device_inputs(w)
    _, pos, st = gpu_fused(w, t)
    assert st == 0
    got = torch.full((w.R, w.k), -7, dtype=torch.int32, device="cuda")
    ws = binding.new_workspace(w.R, w.max_len, w.k, with_scores=True)
    binding.score_topk(t["q"], t["head_w"], t["k_cache"], t["k_scale"], t["block_table"], t["seq_lens"],
                       t["row_req"], w.max_len, w.k, got, ws, slots=True)
    assert binding.check_status(ws) == 0
    want = oracle.slots(pos, w.block_table.numpy(), w.row_req.numpy())
    assert np.array_equal(got.cpu().numpy(), want)


@pytest.mark.parametrize("slots", [False, True])
def test_tagged_pairs(slots):
    """idx_score_topk_tagged: every pair is the oracle's tagged pair of the
    oracle's list of the GPU's own scores (positions, or cache slots), padding
    included; a second launch with another tag rewrites every pair."""
    w = W.make_workload([W.chain(20000, 4), [1500], [0, 9000]], "recent", seed=77)
    t = device_inputs(w)
    stride = stride_for(w.max_len)
    ws = binding.new_workspace(w.R, w.max_len, w.k)
    for tag in (0xABCD1234, 0xFFFFFFFF):
        scores = torch.zeros(w.R, stride, dtype=torch.float32, device="cuda")
        pairs = torch.full((w.R, w.k), 0x5555555555555555, dtype=torch.int64, device="cuda")
        binding.score_topk_tagged(t["q"], t["head_w"], t["k_cache"], t["k_scale"], t["block_table"],
                                  t["seq_lens"], t["row_req"], w.max_len, w.k, tag, pairs, ws, scores=scores,
                                  slots=slots)
        assert binding.check_status(ws) == 0
        s = scores.cpu().numpy()
        lists = np.stack([oracle.topk(s[r, :n], w.k) for r, n in enumerate(w.seq_lens.tolist())])
        if slots:
            lists = oracle.slots(lists, w.block_table.numpy(), w.row_req.numpy())
        assert np.array_equal(pairs.cpu().numpy(), oracle.tagged(lists, tag))


@pytest.mark.parametrize("cfg", [1, 2, 3, 4])
@pytest.mark.parametrize("room", [0, 64, 1024, 1 << 20])
def test_prefix_order_lists(cfg, room):
    """idx_score_topk_prefix_order: every list equals the oracle's list in the
    pages' prefix order (of the GPU's own scores) for the given candidate room;
    room 0 gives idx_score_topk's lists."""
    w = W.make_config(cfg)
    t = device_inputs(w)
    scores = torch.zeros(w.R, stride_for(w.max_len), dtype=torch.float32, device="cuda")
    idx = torch.full((w.R, w.k), -7, dtype=torch.int32, device="cuda")
    ws = binding.new_workspace(w.R, w.max_len, w.k)
    binding.score_topk_prefix_order(t["q"], t["head_w"], t["k_cache"], t["k_scale"], t["block_table"],
                                    t["seq_lens"], t["row_req"], w.max_len, w.k, room, idx, ws, scores=scores)
    assert binding.check_status(ws) == 0
    s = scores.cpu().numpy()
    got = idx.cpu().numpy()
    differ = 0
    for r, n in enumerate(w.seq_lens.tolist()):
        assert np.array_equal(got[r], oracle.prefix_order(s[r, :n], w.k, room)), "row %d" % r
        differ += int(not np.array_equal(got[r], oracle.topk(s[r, :n], w.k)))
    if room == 0:
        assert differ == 0
    if room == 1 << 20 and cfg in (1, 4):
        assert differ > 0, "the prefix order should differ from the specification's order here"


def test_host_buffer_call_e4m3_query():
    """idx_score_topk_host with an E4M3 query (one byte per element)."""
    w = W.make_workload([W.chain(5000)], "random", seed=91, q_is_e4m3=True)
    t = device_inputs(w)
    _, ref, st = gpu_fused(w, t)
    assert st == 0
    ws = binding.new_host_workspace(w.R, w.max_len, w.k, w.block_table.shape[0], w.block_table.shape[1])
    out = torch.full((w.R, w.k), -7, dtype=torch.int32).pin_memory()
    binding.score_topk_host(w.q.pin_memory(), w.head_w.pin_memory(), t["k_cache"], t["k_scale"],
                            w.block_table.pin_memory(), w.seq_lens.pin_memory(), w.row_req.pin_memory(),
                            w.max_len, w.k, out, ws)
    torch.cuda.synchronize()
    assert binding.check_status(ws) == 0
    assert np.array_equal(out.numpy(), ref)


def test_most_rows():
    """The largest row count (IDX_MAX_ROWS = 1,024 rows): 300 requests of 1 to
    7 rows (groups of up to four, so many CTAs start in the middle of a
    request), rows from 0 to 700 keys (k = 256), end to end through the fused
    call."""
    rng = np.random.default_rng(1024)
    reqs, total = [], 0
    while total < 1024:
        nr = int(min(rng.integers(1, 8), 1024 - total))
        base = int(rng.integers(0, 700))
        reqs.append([max(0, base - j) for j in range(nr)][::-1])
        total += nr
    w = W.make_workload(reqs, "random", seed=1024, k=256, extra_pages=2)
    assert w.R == 1024
    s, got, st = gpu_fused(w)
    assert st == 0
    ref = oracle.scores(problem(w))
    errs = checks.score_errors(s, ref, w.seq_lens.tolist())
    assert max(errs) <= checks.SCORE_TOL
    _lists_exact(w, s, got)


def test_concurrent_host_threads():
    """Four host threads call the fused entry point at once, each on its own
    stream and workspace (ctypes releases the GIL during the call): every
    call returns the single-threaded lists."""
    import threading
    ws_cfg = [W.make_config(2), W.make_config(1)]
    refs, inputs = [], []
    for w in ws_cfg:
        t = device_inputs(w)
        _, ref, st = gpu_fused(w, t)
        assert st == 0
        refs.append(ref)
        inputs.append((w, t))
    errors = []

    def worker(j):
        try:
            w, t = inputs[j % 2]
            stream = torch.cuda.Stream()
            ws = binding.new_workspace(w.R, w.max_len, w.k, with_scores=True)
            for _ in range(20):
                idx = torch.full((w.R, w.k), -7, dtype=torch.int32, device="cuda")
                with torch.cuda.stream(stream):
                    binding.score_topk(t["q"], t["head_w"], t["k_cache"], t["k_scale"], t["block_table"],
                                       t["seq_lens"], t["row_req"], w.max_len, w.k, idx, ws, stream=stream)
                stream.synchronize()
                if binding.check_status(ws, stream) != 0 or not np.array_equal(idx.cpu().numpy(), refs[j % 2]):
                    errors.append(j)
                    return
        except Exception as exc:  # reported below
            errors.append(repr(exc))

    threads = [threading.Thread(target=worker, args=(j,)) for j in range(4)]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    assert not errors, errors
