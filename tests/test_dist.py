"""The multi-process (torchrun) path of bench.py on CPU, world size 2 over
gloo: the rendezvous, the barrier and the max over ranks that bracket the
timed region, and the reference arm, which rank 0 alone runs and prints.
The path shards by request with no collective on the data path ("replicas
only"), so these host-side pieces are all there is to cover without GPUs."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    sys.path.insert(0, ROOT)
    import bench
    dist, r, w, local = bench.dist_setup(None)
    assert (r, w, local) == (rank, world, rank)
    bench.barrier(dist)
    got = bench.max_over_ranks(dist, 10.0 + 5.0 * rank)   # rank-specific step times
    bench.barrier(dist)
    with open(os.path.join(out_dir, "rank%d.json" % rank), "w") as f:
        json.dump({"max": got, "backend": dist.get_backend()}, f)
    dist.destroy_process_group()


def test_barrier_and_max_over_two_ranks(tmp_path):
    port = _free_port()
    ctx = mp.get_context("spawn")
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, str(tmp_path))) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    for r in range(2):
        res = json.load(open(tmp_path / ("rank%d.json" % r)))
        assert res == {"max": 15.0, "backend": "gloo"}


def test_reference_arm_under_torchrun():
    """`torchrun --nproc-per-node 2 bench.py --impl reference`: both ranks
    exit 0 and only rank 0 prints its one JSON line."""
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0", "--config", "1"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["config"]["parallelism"] == "replicas"
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
