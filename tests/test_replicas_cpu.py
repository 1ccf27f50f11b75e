"""The multi-GPU path of bench.py is replicas of the same step (the path
does not exchange data): every rank times its own step, the job's time is
the slowest rank's, and the value counts every rank's units.  This runs
that host logic in two gloo ranks on the CPU."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as tdist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    tdist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        tdist.barrier()
        ms = bench.max_over_ranks(1.0 + rank, tdist, "cpu")   # rank 1 is the slower replica
        q.put((rank, ms, bench.job_value(world, 1000.0, ms)))
        tdist.barrier()
    finally:
        tdist.destroy_process_group()


def test_two_gloo_replicas_time_by_the_slowest_and_count_all_units():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    out = sorted(q.get(timeout=10) for _ in range(2))
    for rank, ms, value in out:
        assert ms == 2.0
        assert value == pytest.approx(2 * 1000.0 / 2e-3)


def test_single_process_is_unchanged():
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    assert bench.max_over_ranks(1.25, None, "cpu") == 1.25
    assert bench.job_value(1, 500.0, 2.0) == pytest.approx(2.5e5)


def test_reference_arm_under_torchrun_prints_one_line_from_rank_0():
    """The launch the harness uses for N > 1 (torch.distributed.run, one
    process per rank, 127.0.0.1 rendezvous), here for the reference arm on the
    CPU: rank 0 times the oracle and prints the one JSON line, the other rank
    exits 0 without output."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), "bench.py",
           "--impl", "reference", "--gpus", "2", "--workload", "1", "--steps", "3",
           "--warmup", "3"]
    r = subprocess.run(cmd, cwd=root, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["steps"] == 3
