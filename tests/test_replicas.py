"""The multi-GPU path is independent replicas (no collective on the data path):
bench.py under torchrun times each rank's steps and reports the whole job as
the units all ranks processed over the slowest rank's time.  Its host-side
logic runs here as two gloo ranks on the CPU."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        # rank 1 is the slow replica in the device-resident timing, rank 0 in e2e
        ms = [10.0 + 5.0 * rank, 20.0 - 4.0 * rank]
        out = bench.max_over_ranks(ms, dist, torch.device("cpu"))
        q.put((rank, out, bench.job_rate(1e9, 4, world, out[0])))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_rate_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict()
    for _ in procs:
        rank, out, rate = q.get(timeout=120)
        res[rank] = (out, rate)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    # both ranks see the max of each timing
    assert res[0][0] == res[1][0] == [15.0, 20.0]
    # 2 replicas x 4 steps x 1e9 units in 15 ms = 533.3 G units/s
    assert abs(res[0][1] - 2 * 4 * 1e9 / 15e-3 / 1e9) < 1e-9


@pytest.mark.parametrize("rank", [0, 1])
def test_reference_arm_prints_on_rank_zero_only(rank):
    env = dict(os.environ, RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE="2",
               MASTER_ADDR="127.0.0.1", MASTER_PORT=str(_free_port()))
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "tiny_mixed", "--gpus", "2", "--steps", "1", "--warmup", "0"],
                       capture_output=True, text=True, env=env, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [x for x in r.stdout.splitlines() if x.strip()]
    if rank == 0:
        assert len(lines) == 1
        d = json.loads(lines[0])
        assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    else:
        assert lines == []
