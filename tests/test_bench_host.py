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
    assert bench.TRAFFIC
    for key, rec in bench.TRAFFIC.items():
        name, rows = key.rsplit("@", 1)
        wl = syn.WORKLOADS[name]
        assert rec["src"] == bench._src_hash([rec["file"]]), key
        alg = _algorithmic_bytes(wl, int(rows))
        # within 3%: ncu empties the caches before a captured launch, so the
        # outputs that split-K ranks add into atomically are read back from DRAM
        assert alg <= rec["bytes"] <= 1.03 * alg, (key, rec["bytes"], alg)


def test_source_hash_covers_code_not_comments():
    """a traffic record stays valid across comment and layout edits, not code edits"""
    base = "int f(int x) {\n    return x + 1;  // one\n}\n/* block\n comment */\nconst char *s = \"a // b\";\n"
    same = "int f(int x)\n{\n  return x + 1;  // another comment\n}\nconst char *s = \"a // b\";\n"
    other = base.replace("x + 1", "x + 2")
    lit = base.replace("a // b", "a // c")
    assert bench._code_only(base) == bench._code_only(same)
    assert bench._code_only(base) != bench._code_only(other)
    assert bench._code_only(base) != bench._code_only(lit)  # a // inside a string literal is code


def test_qkv_algorithmic_bytes():
    # 25,165,824 weight codes + 6,144 scales + 32,768 codes + 1,024 act scales + 196,608 output
    wl = syn.WORKLOADS["w8a8_block128_qkv_m8_k4096_n4096+1024+1024"]
    assert _algorithmic_bytes(wl, 8) == 25_402_368


def test_headline_is_the_gate_up_sweep():
    """the metric is quoted on the largest workload: gate/up, K = 8192,
    N = 14336 + 14336, every row bucket from 1 to 256"""
    wl = syn.WORKLOADS[syn.HEADLINE]
    assert (wl.k, wl.segments, wl.fmt) == (8192, (14336, 14336), syn.BLOCK128)
    assert wl.rows == (1, 2, 4, 8, 16, 32, 64, 128, 256)
    # weights 234,881,024 + scales 2 * 112 * 64 * 4 = 57,344; one row adds
    # 8192 codes + 64 act scales * 4 + 28672 * 4 output bytes
    assert _algorithmic_bytes(wl, 1) == 234_881_024 + 57_344 + 8192 + 256 + 114_688


def test_block_steps_are_whole_k_step_sequences():
    for k in (1, 3, 20, 249, 250, 251, 1000, 100000):
        b = bench.block_steps(k)
        assert b % k == 0 and b >= min(250, k) and b >= k
    assert bench.block_steps(20) == 260 and bench.block_steps(100000) == 100000


def test_clock_parse_uses_loaded_samples():
    rows = ["0, 2070, 2070, 150.0, 0x0, Not Active, Not Active, Not Active, Not Active, 0",
            "0, 1900, 2070, 900.5, 0x4, Not Active, Not Active, Not Active, Active, 100",
            "0, 2000, 2070, 950.0, 0x0, Not Active, Not Active, Not Active, Not Active, 97",
            "garbage"]
    c = bench.ClockSampler.parse("\n".join(rows))
    assert c["samples"] == 3 and c["samples_under_load"] == 2
    assert c["sm_mhz"] == 1950.0 and c["sm_max_mhz"] == 2070.0
    assert c["reasons"] == ["sw_power_cap"] and c["power_w_max"] == 950.0


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
