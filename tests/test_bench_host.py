"""Host-side pieces of bench.py that run without a GPU: the argument checks,
the rank environment, the whole-job throughput, and the DRAM-traffic records
it reports beside the roofline (each must name a workload, match the current
kernel source, and sit just above that launch's algorithmic bytes, since a
record far above them would mean re-reads or a stale number)."""
import os
import subprocess
import sys

import pytest

import bench
from quantized_decode_linear_gb300 import synthetic as syn

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _algorithmic_bytes(wl, rows):
    """bytes one launch of the dominant kernel must move, from the shapes"""
    if isinstance(wl, syn.W8A8Workload):
        n, k = wl.n, wl.k
        kb = k // 128
        w_scales = sum(n_s if wl.fmt == syn.PER_ROW else -(-n_s // 128) * kb for n_s in wl.segments) * 4
        a_scales = rows * (1 if wl.fmt == syn.PER_ROW else kb) * 4
        return n * k + w_scales + rows * k + a_scales + rows * n * 4
    if isinstance(wl, syn.Int4Workload):
        n = wl.nq + 2 * wl.nkv
        return wl.k * n // 2 + 8 * (wl.k // wl.group) * n + 4 * rows * wl.k + 4 * rows * n
    raise AssertionError(f"no traffic record expected for {wl.name}")


def test_traffic_records_are_current_and_near_the_algorithmic_bytes():
    kernel_src = {"w8a8": "w8a8_gemm_tc.cu", "int4": "int4_qkv_cc.cu"}
    assert bench.TRAFFIC
    for key, rec in bench.TRAFFIC.items():
        name, rows = key.rsplit("@", 1)
        wl = syn.WORKLOADS[name]
        assert rec["src"] == bench._src_hash([kernel_src[name.split("_")[0]]]), key
        alg = _algorithmic_bytes(wl, int(rows))
        assert alg <= rec["bytes"] <= 1.01 * alg, (key, rec["bytes"], alg)


def test_headline_algorithmic_bytes():
    # 25,165,824 weight codes + 6,144 scales + 32,768 codes + 1,024 act scales + 196,608 output
    wl = syn.WORKLOADS[syn.HEADLINE]
    assert _algorithmic_bytes(wl, 8) == 25_402_368


def test_aggregate_throughput_counts_every_rank():
    assert bench.aggregate_gbs(1e9, 10, 1, 1.0) == pytest.approx(10.0)
    assert bench.aggregate_gbs(1e9, 10, 4, 2.0) == pytest.approx(20.0)


def test_rank_environment(monkeypatch):
    for v in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(v, raising=False)
    assert bench._rank_world() == (0, 1, 0)
    monkeypatch.setenv("RANK", "3")
    monkeypatch.setenv("WORLD_SIZE", "8")
    monkeypatch.setenv("LOCAL_RANK", "3")
    assert bench._rank_world() == (3, 8, 3)


def test_single_replica_needs_no_process_group():
    g = bench.Replicas(1, backend="gloo", device="cpu")
    g.barrier()
    assert g.max(2.5) == 2.5
    g.close()


@pytest.mark.parametrize("args,msg", [
    (["--warmup", "2"], "--warmup >= 3"),
    (["--steps", "0"], "--steps >= 1"),
    (["--workload", "no_such_workload"], "unknown workload"),
])
def test_bench_rejects_bad_arguments(args, msg):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py")] + args, capture_output=True, text=True,
                       timeout=120)
    assert r.returncode == 2 and msg in r.stderr, (r.returncode, r.stderr[-400:])
