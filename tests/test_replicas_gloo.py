"""The benchmark's N>1 path on the CPU: two ranks over gloo, launched the way
torchrun launches them (RANK / WORLD_SIZE / MASTER_* in the environment).
The replicas share no data; what they do exchange is a barrier before each
timed region and the maximum of their elapsed times after it, and the
whole-job throughput divides every rank's bytes by that maximum.  The CPU
(oracle) arm runs on rank 0 alone and the other ranks exit without work."""
import argparse
import contextlib
import io
import json
import multiprocessing as mp
import os
import socket
import time

import pytest

WORLD = 2


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, port, q):
    try:
        os.environ.update(RANK=str(rank), WORLD_SIZE=str(WORLD), LOCAL_RANK=str(rank),
                          MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
        import bench
        r, world, local = bench._rank_world()
        assert (r, world, local) == (rank, WORLD, rank)
        group = bench.Replicas(world, backend="gloo", device="cpu")
        # each rank's timed region lasts a different time; all of them must
        # report the slowest one
        elapsed = 0.010 * (rank + 1)
        group.barrier()
        t_max = group.max(elapsed)
        e2e_max = group.max(3.0 - rank)
        value = bench.aggregate_gbs(1e9, 10, world, t_max)
        group.barrier()
        group.close()
        out = io.StringIO()
        args = argparse.Namespace(workload="w8a8_block128_qkv_m8_k4096_n4096+1024+1024", rows=None,
                                  steps=2, warmup=3)
        t0 = time.perf_counter()
        with contextlib.redirect_stdout(out):
            bench.run_reference(args, rank, world, budget_s=0.5)
        q.put((rank, t_max, e2e_max, value, out.getvalue(), time.perf_counter() - t0, None))
    except BaseException as e:  # report to the parent instead of hanging it
        q.put((rank, None, None, None, "", 0.0, repr(e)))


def test_two_replicas_over_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, port, q)) for r in range(WORLD)]
    for p in procs:
        p.start()
    try:
        got = {}
        for _ in range(WORLD):
            rank, t_max, e2e_max, value, text, dt, err = q.get(timeout=240)
            assert err is None, f"rank {rank}: {err}"
            got[rank] = (t_max, e2e_max, value, text, dt)
    finally:
        for p in procs:
            p.join(timeout=30)
            if p.is_alive():
                p.kill()
    for rank in range(WORLD):
        t_max, e2e_max, value, _, _ = got[rank]
        assert t_max == pytest.approx(0.010 * WORLD)
        assert e2e_max == pytest.approx(3.0)
        # 1e9 bytes x 10 steps x 2 ranks over the slowest rank's 20 ms
        assert value == pytest.approx(1e9 * 10 * WORLD / (0.010 * WORLD) / 1e9)
    assert got[1][3] == "" and got[1][4] < 5.0  # rank 1 does no CPU-arm work
    lines = got[0][3].strip().splitlines()
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == WORLD and line["value"] > 0
    assert line["e2e"]["value"] == line["value"] and line["cpu_baseline"]["kind"] == "oracle"
    assert all(p.exitcode == 0 for p in procs)
