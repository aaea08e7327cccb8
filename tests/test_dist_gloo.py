"""The N > 1 host path of bench.py on CPU: two gloo ranks (independent replicas),
the timing barrier, the max-over-ranks reduction and the whole-job aggregate."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ws, r, local = bench._dist()
        assert (ws, r, local) == (world, rank, rank)
        bench._barrier(ws)
        my_ms = 10.0 + 5.0 * rank          # rank 1 is the slow one
        mx = bench._max_over_ranks(my_ms, ws, "cpu")
        # whole-job value: every rank's tokens over the slowest rank's time
        tokens_per_rank = 256 * 7
        value = tokens_per_rank * ws / (mx / 1e3)
        # the reference arm prints only on rank 0; other ranks return 0 without work
        rc = bench.run_reference(type("A", (), {"steps": 1, "warmup": 3, "gpus": ws})()) if r != 0 else 0
        q.put((rank, mx, value, rc))
    finally:
        dist.destroy_process_group()


def test_two_rank_timing_reduction():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, mx, value, rc in res:
        assert mx == 15.0
        assert value == pytest.approx(256 * 7 * 2 / 0.015)
        assert rc == 0


def test_bench_gpus_2_launches_two_ranks():
    """bench.py --gpus 2 run without a launcher starts two ranks itself (torch.distributed.run
    on 127.0.0.1); with the reference arm rank 0 prints one line carrying n_gpus 2 and the
    other rank exits 0 without work."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = {k: v for k, v in os.environ.items() if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK")}
    r = subprocess.run([sys.executable, "bench.py", "--gpus", "2", "--impl", "reference", "--steps", "1",
                        "--warmup", "3"], cwd=root, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip().startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    line = json.loads(lines[0])
    assert line["n_gpus"] == 2 and line["impl"] == "reference" and line["value"] > 0
