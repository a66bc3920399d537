"""The N > 1 host path of bench.py, on CPU with the gloo backend.

The layer runs as independent replicas, one per GPU, with no collective on
the data path.  What the ranks share is host logic only: a barrier around the
timed region, the whole-job reduction (slowest rank's time, summed bytes) and
rank 0 alone printing the line.  These tests run that logic as two gloo ranks.
"""
import json
import multiprocessing as mp
import os
import socket
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _gather_worker(rank: int, world: int, port: int, out):
    sys.path.insert(0, ROOT)
    import torch
    import bench
    torch.distributed.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                                         world_size=world)
    try:
        # rank r: times (r + 1, 10 - r), sizes (100 (r + 1), 7)
        times, sizes = bench.gather_replicas([rank + 1.0, 10.0 - rank], [100.0 * (rank + 1), 7.0], world)
        out.put((rank, times, sizes))
    finally:
        torch.distributed.destroy_process_group()


def test_gather_replicas_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.gather_replicas([1.5, 2], [3, 4.25], 1) == ([1.5, 2.0], [3.0, 4.25])


def test_gather_replicas_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_gather_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(out.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, times, sizes in got:
        # every rank sees the slowest time of each entry and the summed sizes
        assert times == [2.0, 10.0], (rank, times)
        assert sizes == [300.0, 14.0], (rank, sizes)


def test_reference_arm_under_torchrun_prints_one_line_from_rank_0():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl", "reference",
           "--gpus", "2", "--steps", "1", "--warmup", "3"]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference"
    assert line["n_gpus"] == 2
    assert line["steps"] == 1 and line["warmup"] == 3
    assert line["value"] > 0 and line["e2e"]["value"] == line["value"]
    assert line["cpu_baseline"]["kind"] == "oracle"
