"""The multi-process (replica) logic of bench.py on CPU: two gloo ranks meet
at the barrier, agree on the slowest rank's time, and the whole-job rate
counts every rank's work over that time. Under torchrun the reference arm
runs on rank 0 alone; other ranks exit without work."""
import json
import os
import socket
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        t_local = [0.25, 0.75][rank]
        bench.rank_barrier(world)
        t = bench.max_over_ranks(t_local, world, "cpu")
        rate = bench.whole_job_rate(1e9, 10, world, t)
        out.put((rank, t, rate))
    finally:
        dist.destroy_process_group()


def test_two_ranks_agree_on_the_slowest_time():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, world, port, out)) for r in range(world)]
    for pr in procs:
        pr.start()
    res = sorted(out.get(timeout=120) for _ in range(world))
    for pr in procs:
        pr.join(timeout=60)
        assert pr.exitcode == 0
    assert [r[1] for r in res] == [0.75, 0.75]
    # 2 ranks x 10 steps x 1e9 bytes over 0.75 s
    assert all(abs(r[2] - 2 * 10 / 0.75) < 1e-9 for r in res)


def test_single_process_needs_no_group():
    assert bench.max_over_ranks(1.5, 1) == 1.5
    bench.rank_barrier(1)
    assert bench.whole_job_rate(2e9, 4, 1, 2.0) == 4.0


@pytest.mark.parametrize("rank", [0, 1])
def test_reference_arm_runs_on_rank_zero_only(rank):
    env = dict(os.environ, RANK=str(rank), WORLD_SIZE="2", LOCAL_RANK=str(rank),
               MASTER_ADDR="127.0.0.1", MASTER_PORT=str(_free_port()))
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "q8_0_256x1024", "--steps", "1", "--warmup", "3", "--cpu-budget", "0.2"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    if rank == 0:
        assert len(lines) == 1
        d = json.loads(lines[0])
        assert d["impl"] == "reference" and d["value"] > 0
        assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"
    else:
        assert lines == []
