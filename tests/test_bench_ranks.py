"""bench.py's multi-rank logic on CPU: two gloo ranks, no GPU.

With N GPUs every rank runs its own batch (weak scaling, no collective on
the data path); the only cross-rank steps are the barrier and taking the
slowest rank's time.  These tests run that reduction on two gloo ranks and
check the whole-job number built from it.
"""

import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms = [0.080, 0.095][rank]                      # rank 1 is the slower one
    slowest = bench.max_over_ranks(dist, ms, "cpu")
    gbs = bench.job_gbs(537_460_992, world, slowest)
    dist.barrier()
    dist.destroy_process_group()
    q.put((rank, slowest, gbs))


def test_two_gloo_ranks_take_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, slowest, gbs in res:
        assert slowest == pytest.approx(0.095)
        assert gbs == pytest.approx(2 * 537_460_992 / 0.095e-3 / 1e9)


def test_single_process_needs_no_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(None, 1.5, "cpu") == 1.5
    assert bench.job_gbs(1_000_000_000, 1, 1.0) == pytest.approx(1000.0)


def test_reference_arm_under_torchrun_prints_one_line_from_rank_0(tmp_path):
    # two gloo ranks of the oracle arm: rank 0 prints the JSON line, rank 1 exits quietly
    env = dict(os.environ, PYTHONPATH=ROOT)
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
           "--steps", "1", "--warmup", "0", "--history", "256"]
    r = subprocess.run(cmd, capture_output=True, text=True, env=env, timeout=600, cwd=tmp_path)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    import json
    j = json.loads(lines[0])
    assert j["impl"] == "reference" and j["n_gpus"] == 2 and j["value"] > 0
    # the oracle on every core of the affinity set, one process each with BLAS at one thread
    cb = j["cpu_baseline"]
    assert cb["cores"] == len(os.sched_getaffinity(0)) and cb["kind"] == "oracle"
    assert 0 < cb["busy"] <= cb["cores"] + 0.5 and cb["best_ms"] <= cb["median_ms"]
    assert cb["blas_threads"] == "1"                     # pinned when bench.py runs as a script
    assert cb["value"] == j["value"] and j["e2e"]["h2d_bytes_per_step"] == 0
