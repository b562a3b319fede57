"""The N > 1 host path of bench.py (replicas only: every rank runs the whole
path on its own GPU; the job rate is all ranks' units over the slowest
rank's time), on the CPU with gloo, world size 2."""

import json
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


def _worker(rank, world, port, out):
    import torch.distributed as dist

    sys.path.insert(0, ROOT)
    import bench

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r took 10 + 5 r ms: every rank sees the slowest
        got = bench.max_over_ranks(10.0 + 5.0 * rank, world, "cpu")
        out.put((rank, got))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    world, port = 2, _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    results = dict(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert results == {0: 15.0, 1: 15.0}


def test_whole_job_rate_and_single_rank():
    sys.path.insert(0, ROOT)
    import bench

    # 8.3 M pixels per rank, 2 ranks, slowest rank 10 ms -> 1.66 G pixels/s
    assert bench.whole_job_rate(8_294_400, 10.0, 2) == pytest.approx(1.65888e9)
    assert bench.max_over_ranks(3.5, 1, "cpu") == 3.5


@pytest.mark.slow
def test_reference_arm_prints_on_rank_zero_only():
    # launched as torchrun would: RANK / WORLD_SIZE in the environment; only
    # rank 0 times the oracle and prints the line, the other exits 0 silently
    outs = []
    for rank in range(2):
        env = dict(os.environ, RANK=str(rank), WORLD_SIZE="2", LOCAL_RANK=str(rank),
                   MASTER_ADDR="127.0.0.1")
        r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--gpus", "2",
                            "--steps", "1", "--warmup", "0"], cwd=ROOT, env=env,
                           capture_output=True, text=True, timeout=600)
        assert r.returncode == 0, r.stderr[-2000:]
        outs.append(r.stdout.strip())
    assert outs[1] == ""
    line = json.loads(outs[0].splitlines()[-1])
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["value"] > 0 and line["cpu_baseline"]["kind"] == "oracle"
