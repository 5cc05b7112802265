"""Host-side tests of the C ABI: the library loads without a GPU, exports every
symbol include/qdl.h declares, the ctypes structs match the C layout, and every
validation rule of w8a8_decode.rs / fused_int4_qkv.rs rejects bad arguments
before any device work (no call here reaches the device)."""
import ctypes
import os
import re
import subprocess

import pytest

import quantized_decode_linear_gb300 as qdl
from quantized_decode_linear_gb300 import build as qbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "qdl.h")

INVALID, SCRATCH, UNSUPPORTED = 1, 2, 3
DEV = 0x7F0000000000  # a 256-byte aligned fake device address; never dereferenced


@pytest.fixture(scope="module")
def lib():
    qbuild.build()
    return qdl.load()


def _declared():
    src = open(HEADER).read()
    return sorted(set(re.findall(r"QDL_API\s+[\w\s\*]*?\b(qdl_\w+)\s*\(", src)))


def test_exports_every_declared_symbol(lib):
    names = _declared()
    assert len(names) >= 11
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(qdl.EXPORTS) == names


def test_struct_layout_matches_c(tmp_path):
    prog = tmp_path / "sz.c"
    prog.write_text(f'''#include <stdio.h>
#include <stddef.h>
#include "{HEADER}"
int main(void) {{
  printf("%zu %zu %zu %zu %zu %zu %zu %zu\\n", sizeof(qdl_fp8_segment), sizeof(qdl_w8a8_weight),
         offsetof(qdl_w8a8_weight, count), offsetof(qdl_w8a8_weight, n1),
         offsetof(qdl_w8a8_weight, magic), sizeof(qdl_plan), offsetof(qdl_plan, resident_clusters),
         offsetof(qdl_plan, proj_streamk));
  return 0;
}}
''')
    exe = tmp_path / "sz"
    subprocess.run(["gcc", str(prog), "-o", str(exe)], check=True)
    got = [int(v) for v in subprocess.run([str(exe)], capture_output=True, text=True).stdout.split()]
    W = qdl.W8A8WeightDesc
    P = qdl.Plan
    want = [ctypes.sizeof(qdl.Fp8Segment), ctypes.sizeof(W), W.count.offset, W.n1.offset,
            W.magic.offset, ctypes.sizeof(P), P.resident_clusters.offset, P.proj_streamk.offset]
    assert got == want


def test_status_strings(lib):
    for code, name in qdl.STATUS_NAMES.items():
        assert lib.qdl_status_string(code).decode() == name


def test_scratch_bytes(lib):
    # W8a8Scratch::alloc: 256 * max_k and 256 * max(ceil(max_k / 128), 1) * 4
    assert qdl.scratch_bytes(0) == (0, 1024)
    assert qdl.scratch_bytes(100) == (25600, 1024)
    assert qdl.scratch_bytes(128) == (32768, 1024)
    assert qdl.scratch_bytes(4096) == (256 * 4096, 256 * 32 * 4)
    assert qdl.scratch_bytes(4097) == (256 * 4097, 256 * 33 * 4)
    big = 2**32 - 1  # the group count must not wrap in 32 bits
    assert qdl.scratch_bytes(big) == (256 * big, 256 * 2**25 * 4)


# ---------------------------------------------------------------- weight descriptor

def _segs(specs, fmt=qdl.PER_ROW):
    arr = (qdl.Fp8Segment * 3)()
    for i, spec in enumerate(specs):
        n, k = spec[0], spec[1]
        w = spec[2] if len(spec) > 2 else DEV + i * 0x100000
        s = spec[3] if len(spec) > 3 else DEV + 0x8000000 + i * 0x1000
        f = spec[4] if len(spec) > 4 else fmt
        arr[i] = qdl.Fp8Segment(w, s, n, k, f)
    return arr


def _init(lib, specs, count=None, fmt=qdl.PER_ROW):
    desc = qdl.W8A8WeightDesc()
    st = lib.qdl_w8a8_weight_init(ctypes.byref(desc), _segs(specs, fmt),
                                  len(specs) if count is None else count)
    return st, desc, lib.qdl_last_error().decode()


def test_weight_init_ok_and_boundaries(lib):
    st, d, _ = _init(lib, [(4096, 4096)], fmt=qdl.BLOCK128)
    assert st == 0 and (d.n, d.n1, d.n2, d.count) == (4096, 4096, 4096, 1)
    st, d, _ = _init(lib, [(4096, 4096), (1024, 4096), (1000, 4096)], fmt=qdl.BLOCK128)
    assert st == 0 and (d.n, d.n1, d.n2) == (6120, 4096, 5120)
    st, d, _ = _init(lib, [(32, 256), (40, 256)])
    assert st == 0 and (d.n, d.n1, d.n2) == (72, 32, 72)


@pytest.mark.parametrize("specs,count,fmt,code,msg", [
    ([(16, 128)], 0, qdl.PER_ROW, INVALID, "0 segments, want 1..=3"),
    ([(16, 128)] * 3, 4, qdl.PER_ROW, INVALID, "4 segments, want 1..=3"),
    ([(16, 100)], None, qdl.PER_ROW, INVALID, "K=100 is not a positive multiple of 128"),
    ([(16, 0)], None, qdl.PER_ROW, INVALID, "K=0 is not a positive multiple of 128"),
    ([(16, 128), (16, 256)], None, qdl.PER_ROW, INVALID, "segment 1 is [16, 256]"),
    ([(16, 128), (16, 128, None, None, qdl.BLOCK128)], None, qdl.PER_ROW, INVALID, "segment 1 is"),
    ([(0, 128)], None, qdl.PER_ROW, INVALID, "segment 0 is empty"),
    ([(16, 128), (16, 128, 0)], None, qdl.PER_ROW, INVALID, "segment 1 is empty"),
    ([(16, 128, DEV, 0)], None, qdl.PER_ROW, INVALID, "segment 0 is empty"),
    ([(24, 128), (16, 128)], None, qdl.PER_ROW, INVALID, "segment 0 has 24 rows, not a multiple of 16"),
    ([(128, 128), (64, 128), (8, 128)], None, qdl.BLOCK128, INVALID,
     "segment 1 has 64 rows, not a multiple of 128"),
    ([(16, 128, DEV + 8)], None, qdl.PER_ROW, INVALID, "16-byte"),
    ([(16, 128, DEV, DEV + 2)], None, qdl.PER_ROW, INVALID, "4-byte"),
    ([(16, 128)], None, 7, INVALID, "is not per-row or 128x128 block"),
])
def test_weight_init_rejects(lib, specs, count, fmt, code, msg):
    st, _, err = _init(lib, specs, count, fmt)
    assert st == code and msg in err, (st, err)


def test_last_segment_may_be_ragged(lib):
    st, d, _ = _init(lib, [(16, 128), (7, 128)])
    assert st == 0 and d.n == 23
    st, d, _ = _init(lib, [(128, 128), (128, 128), (5, 128)], fmt=qdl.BLOCK128)
    assert st == 0 and d.n == 261


# ---------------------------------------------------------------- act quant

def _aq(lib, fmt=qdl.PER_ROW, x=DEV, ldx=4096, rows=8, k=4096, q=DEV + 0x1000000,
        s=DEV + 0x2000000, qb=256 * 4096, sb=256 * 32 * 4):
    st = lib.qdl_act_quant(fmt, x, ldx, rows, k, q, s, qb, sb, None)
    return st, lib.qdl_last_error().decode()


@pytest.mark.parametrize("kw,code,msg", [
    (dict(rows=0), INVALID, "0 rows, want 1..=256"),
    (dict(rows=257), INVALID, "257 rows, want 1..=256"),
    (dict(k=4000, ldx=4000), INVALID, "K=4000"),
    (dict(k=0, ldx=0), INVALID, "K=0"),
    (dict(k=65536 + 128, ldx=65536 + 128, qb=1 << 30, sb=1 << 30), INVALID, "K=65664"),
    (dict(ldx=4000), INVALID, "x stride=4000"),
    (dict(ldx=4100), INVALID, "x stride=4100"),
    (dict(x=0), INVALID, "x is NULL"),
    (dict(x=DEV + 8), INVALID, "x must be 16-byte aligned"),
    (dict(q=0), SCRATCH, "do not fit the scratch"),
    (dict(qb=8 * 4096 - 1), SCRATCH, "8 rows of K=4096 do not fit the scratch"),
    (dict(fmt=qdl.PER_ROW, sb=8 * 4 - 1), SCRATCH, "do not fit"),
    (dict(fmt=qdl.BLOCK128, sb=8 * 32 * 4 - 4), SCRATCH, "do not fit"),
    (dict(s=0), INVALID, "scale pointer is NULL"),
    (dict(q=DEV + 4), INVALID, "16-byte"),
    (dict(fmt=5), INVALID, "not per-row or 128x128 block"),
])
def test_act_quant_rejects(lib, kw, code, msg):
    st, err = _aq(lib, **kw)
    assert st == code and msg in err, (st, err)


def test_act_quant_silu_checks_both_strides(lib):
    args = dict(rows=4, k=256, q=DEV + 0x1000000, s=DEV + 0x2000000, qb=1 << 20, sb=1 << 16)

    def call(gate, up, ldg, ldu):
        st = lib.qdl_act_quant_silu(qdl.BLOCK128, gate, up, ldg, ldu, args["rows"], args["k"],
                                    args["q"], args["s"], args["qb"], args["sb"], None)
        return st, lib.qdl_last_error().decode()

    assert call(DEV, DEV, 256, 250) == (INVALID, call(DEV, DEV, 256, 250)[1])
    assert "up stride=250" in call(DEV, DEV, 256, 250)[1]
    assert "gate stride=100" in call(DEV, DEV, 100, 256)[1]
    assert "up is NULL" in call(DEV, 0, 256, 256)[1]


# ---------------------------------------------------------------- GEMV

def _weight(lib, fmt=qdl.BLOCK128):
    st, d, _ = _init(lib, [(4096, 4096), (1024, 4096), (1024, 4096)], fmt=fmt)
    assert st == 0
    return d


def _gemv(lib, d, rows=8, q=DEV + 0x1000000, s=DEV + 0x2000000, qb=1 << 24, sb=1 << 20,
          out=DEV + 0x4000000, dtype=qdl.OUT_F32, ldc=6144):
    st = lib.qdl_w8a8_gemv(ctypes.byref(d), q, s, qb, sb, rows, out, dtype, ldc, None)
    return st, lib.qdl_last_error().decode()


@pytest.mark.parametrize("kw,code,msg", [
    (dict(rows=0), INVALID, "not available for 0 rows of [6144, 4096] Block128"),
    (dict(rows=300), INVALID, "not available for 300 rows"),
    (dict(qb=8 * 4096 - 1), SCRATCH, "not available for 8 rows"),
    (dict(sb=8 * 32 * 4 - 1), SCRATCH, "not available"),
    (dict(ldc=6143), INVALID, "ldc=6143 < N=6144"),
    (dict(dtype=4), INVALID, "output dtype 4"),
    (dict(out=0), INVALID, "output is NULL"),
    (dict(out=DEV + 2), INVALID, "misaligned"),
])
def test_gemv_rejects(lib, kw, code, msg):
    st, err = _gemv(lib, _weight(lib), **kw)
    assert st == code and msg in err, (st, err)


def test_gemv_rejects_uninitialised_weight(lib):
    st, err = _gemv(lib, qdl.W8A8WeightDesc())
    assert st == INVALID and "qdl_w8a8_weight_init" in err


def test_proj_checks_input(lib):
    d = _weight(lib)
    st = lib.qdl_w8a8_proj(ctypes.byref(d), DEV, 4095, 8, DEV + 0x4000000, 0, 6144,
                           DEV + 0x1000000, DEV + 0x2000000, 1 << 24, 1 << 20, None)
    assert st == INVALID and "x stride=4095" in lib.qdl_last_error().decode()


def test_projections_refuse_k_beyond_the_quantiser(lib):
    """the projections quantise their activations, so a weight whose K exceeds
    QDL_MAX_K (what the quantiser covers) is refused by every projection entry
    point before any device work, as qdl_act_quant refuses it"""
    k = 65536 + 128
    st, d, _ = _init(lib, [(16, k)])
    assert st == 0
    big = 1 << 30
    st = lib.qdl_w8a8_proj(ctypes.byref(d), DEV, k, 1, DEV + 0x4000000, 0, 16,
                           DEV + 0x1000000, DEV + 0x2000000, big, big, None)
    assert st == INVALID and "K=65664" in lib.qdl_last_error().decode()
    st = lib.qdl_w8a8_proj_silu(ctypes.byref(d), DEV, DEV, k, k, 1, DEV + 0x4000000, 0, 16,
                                DEV + 0x1000000, DEV + 0x2000000, big, big, None)
    assert st == INVALID and "K=65664" in lib.qdl_last_error().decode()
    st = lib.qdl_w8a8_proj_static(ctypes.byref(d), DEV, k, 1, DEV + 0x4000000, 0, 16, None)
    assert st == INVALID and "K=65664" in lib.qdl_last_error().decode()


def test_accumulating_output_is_gemv_only(lib):
    """QDL_OUT_F32_ADD (out += y) is accepted by qdl_w8a8_gemv's checks but
    not by the projections, which pick accumulation themselves"""
    d = _weight(lib)
    st = lib.qdl_w8a8_proj(ctypes.byref(d), DEV, 4096, 8, DEV + 0x4000000, qdl.OUT_F32_ADD, 6144,
                           DEV + 0x1000000, DEV + 0x2000000, 1 << 24, 1 << 20, None)
    assert st == INVALID and "output dtype 2 is not F32, BF16 or F32_DETERMINISTIC" in lib.qdl_last_error().decode()
    st, err = _gemv(lib, d, dtype=qdl.OUT_F32_ADD, ldc=6143)  # fails on ldc, after the dtype check passed
    assert st == INVALID and "ldc=6143" in err, err


# ---------------------------------------------------------------- INT4

def _int4(lib, x=DEV, m=1, k=4096, nq=4096, nkv=1024, group=128, qw=None, sc=None, zr=None, out=None):
    arr = lambda v, base: (ctypes.c_void_p * 3)(*([base + i * 0x100000 for i in range(3)] if v is None else v))
    st = lib.qdl_int4_qkv_gemv(x, m, k, nq, nkv, group, arr(qw, DEV + 0x1000000), arr(sc, DEV + 0x2000000),
                               arr(zr, DEV + 0x3000000), arr(out, DEV + 0x4000000), None)
    return st, lib.qdl_last_error().decode()


@pytest.mark.parametrize("kw,msg", [
    (dict(m=0), "m=0"),
    (dict(group=0), "group=0"),
    (dict(group=24, k=48), "group=24"),
    (dict(k=4000), "k=4000"),
    (dict(nq=4100), "nq=4100"),
    (dict(nkv=0), "nkv=0"),
    (dict(x=0), "NULL"),
    (dict(x=DEV + 4), "x must be 16-byte aligned"),
    (dict(qw=[DEV, 0, DEV]), "projection 1 has a NULL pointer"),
    (dict(sc=[DEV, DEV, DEV + 4]), "projection 2 misaligned"),
])
def test_int4_rejects(lib, kw, msg):
    st, err = _int4(lib, **kw)
    assert st == INVALID and msg in err, (st, err)


# ---------------------------------------------------------------- KV-cache quantisers

def _kv(lib, fn, **kw):
    a = dict(x=DEV, tokens=64, dim=128, group=64, q=DEV + 0x1000000, s=DEV + 0x2000000, z=DEV + 0x3000000,
             out=DEV + 0x4000000)
    a.update(kw)
    if fn == "q8":
        st = lib.qdl_kv_quant_int8(a["x"], a["tokens"], a["dim"], a["q"], a["s"], None)
    elif fn == "d8":
        st = lib.qdl_kv_dequant_int8(a["q"], a["s"], a["tokens"], a["dim"], a["out"], None)
    elif fn == "q4":
        st = lib.qdl_kv_quant_int4(a["x"], a["tokens"], a["dim"], a["group"], a["q"], a["s"], a["z"], None)
    else:
        st = lib.qdl_kv_dequant_int4(a["q"], a["s"], a["z"], a["tokens"], a["dim"], a["group"], a["out"], None)
    return st, lib.qdl_last_error().decode()


@pytest.mark.parametrize("fn,kw,msg", [
    ("q8", dict(tokens=0), "tokens=0"),
    ("q8", dict(dim=130), "head_dim=130"),
    ("q8", dict(x=0), "NULL"),
    ("q8", dict(x=DEV + 4), "x must be 16-byte"),
    ("q8", dict(q=DEV + 2), "4-byte aligned"),
    ("d8", dict(out=DEV + 8), "out 16-byte aligned"),
    ("d8", dict(s=0), "NULL"),
    ("q4", dict(group=0), "group=0"),
    ("q4", dict(group=12), "group=12"),
    ("q4", dict(tokens=3, dim=4, group=8), "group=8"),
    ("q4", dict(z=0), "NULL"),
    ("d4", dict(dim=2), "head_dim=2"),
    ("d4", dict(q=DEV + 1), "4-byte"),
])
def test_kv_rejects(lib, fn, kw, msg):
    st, err = _kv(lib, fn, **kw)
    assert st == INVALID and msg in err, (st, err)


def test_kv_rejects_oversized(lib):
    st, err = _kv(lib, "q8", tokens=1 << 20, dim=4096)
    assert st == UNSUPPORTED and "exceeds 2^31" in err, (st, err)


# ---------------------------------------------------------------- weight preparation

def _wq(lib, **kw):
    a = dict(fmt=0, w=DEV, dtype=0, ldw=256, n=64, k=256, codes=DEV + 0x1000000, scales=DEV + 0x2000000)
    a.update(kw)
    st = lib.qdl_fp8_weight_quant(a["fmt"], a["w"], a["dtype"], a["ldw"], a["n"], a["k"], a["codes"], a["scales"],
                                  None)
    return st, lib.qdl_last_error().decode()


@pytest.mark.parametrize("kw,msg", [
    (dict(fmt=2), "format=2"),
    (dict(dtype=3), "w_dtype=3"),
    (dict(n=0), "n=0"),
    (dict(k=200, ldw=256), "k=200"),
    (dict(k=0), "k=0"),
    (dict(ldw=128), "ldw=128"),
    (dict(dtype=1, ldw=260), "multiple of 8"),
    (dict(ldw=258), "multiple of 4"),
    (dict(w=0), "NULL"),
    (dict(w=DEV + 8), "16-byte"),
    (dict(codes=DEV + 4), "codes 8-byte"),
    (dict(scales=DEV + 2), "scales 4-byte"),
])
def test_fp8_weight_quant_rejects(lib, kw, msg):
    st, err = _wq(lib, **kw)
    assert st == INVALID and msg in err, (st, err)


@pytest.mark.parametrize("kw,msg", [
    (dict(k=0), "k=0"),
    (dict(n=12), "n=12"),
    (dict(n=0), "n=0"),
    (dict(nib=0), "NULL"),
    (dict(nib=DEV + 4), "8-byte"),
    (dict(qw=DEV + 2), "4-byte"),
])
def test_awq_pack_rejects(lib, kw, msg):
    a = dict(nib=DEV, k=16, n=64, qw=DEV + 0x1000000)
    a.update(kw)
    st = lib.qdl_awq_pack(a["nib"], a["k"], a["n"], a["qw"], None)
    err = lib.qdl_last_error().decode()
    assert st == INVALID and msg in err, (st, err)


@pytest.mark.parametrize("rows,qb,code,msg", [
    (65537, 1 << 24, INVALID, "not available for 65537 rows"),
    (1000, 256 * 4096 - 1, SCRATCH, "not available for 1000 rows"),
    (100, 100 * 4096 - 1, SCRATCH, "not available for 100 rows"),
])
def test_proj_row_limits(lib, rows, qb, code, msg):
    """projections take up to QDL_MAX_PROJ_ROWS rows in passes of 256 through
    a scratch that holds min(rows, 256) rows"""
    d = _weight(lib)
    st = lib.qdl_w8a8_proj(ctypes.byref(d), DEV, 4096, rows, DEV + 0x4000000, 0, 6144,
                           DEV + 0x1000000, DEV + 0x2000000, qb, 1 << 20, None)
    err = lib.qdl_last_error().decode()
    assert st == code and msg in err, (st, err)


def _static(lib, d, rows=8, x=DEV, ldx=4096, out=DEV + 0x4000000, dtype=qdl.OUT_F32, ldc=6144):
    st = lib.qdl_w8a8_proj_static(ctypes.byref(d), x, ldx, rows, out, dtype, ldc, None)
    return st, lib.qdl_last_error().decode()


@pytest.mark.parametrize("kw,code,msg", [
    (dict(rows=0), INVALID, "0 rows, want 1..=256"),
    (dict(rows=257), INVALID, "257 rows, want 1..=256"),
    (dict(ldc=6143), INVALID, "ldc=6143 < N=6144"),
    (dict(dtype=qdl.OUT_F32_ADD), INVALID, "output dtype 2"),
    (dict(out=0), INVALID, "output is NULL"),
    (dict(out=DEV + 2), INVALID, "misaligned"),
    (dict(x=0), INVALID, "x is NULL"),
    (dict(ldx=4095), INVALID, "x stride=4095"),
    (dict(x=DEV + 8), INVALID, "x must be 16-byte aligned"),
])
def test_proj_static_rejects(lib, kw, code, msg):
    """the no-allocation projection checks everything before it looks up its
    scratch or launches"""
    st, err = _static(lib, _weight(lib), **kw)
    assert st == code and msg in err, (st, err)


def test_proj_static_scratch_limit(lib):
    # 256 rows of K = 16384: 4 MiB of codes plus the scales exceed the 4 MiB buffer
    st, d, _ = _init(lib, [(128, 16384)], fmt=qdl.BLOCK128)
    assert st == 0
    st, err = _static(lib, d, rows=256, ldx=16384, ldc=128)
    assert st == UNSUPPORTED and "static scratch" in err, (st, err)
    # K = 15872 is the largest that fits at 256 rows: the call gets past the
    # scratch check and stops at the next one (an ldc below N, on purpose)
    st, d, _ = _init(lib, [(128, 15872)], fmt=qdl.BLOCK128)
    assert st == 0
    st, err = _static(lib, d, rows=256, ldx=15872, ldc=127)
    assert st == INVALID and "ldc=127 < N=128" in err, (st, err)


def test_proj_static_rejects_uninitialised_weight(lib):
    st, err = _static(lib, qdl.W8A8WeightDesc())
    assert st == INVALID and "qdl_w8a8_weight_init" in err


def test_plan_rejects(lib):
    d = _weight(lib)
    plan = qdl.Plan()
    assert lib.qdl_w8a8_plan(ctypes.byref(d), 8, None) == INVALID
    assert "plan is NULL" in lib.qdl_last_error().decode()
    for rows in (0, 257):
        assert lib.qdl_w8a8_plan(ctypes.byref(d), rows, ctypes.byref(plan)) == INVALID
        assert f"{rows} rows, want 1..=256" in lib.qdl_last_error().decode()
    assert lib.qdl_w8a8_plan(ctypes.byref(qdl.W8A8WeightDesc()), 8, ctypes.byref(plan)) == INVALID
    assert "qdl_w8a8_weight_init" in lib.qdl_last_error().decode()


# ---------------------------------------------------------------- Python binding checks

def _wobj(lib):
    return qdl.W8A8Weight(_weight(lib), [])


def test_binding_refuses_host_tensors(lib):
    import torch
    w = _wobj(lib)
    x = torch.zeros((8, 4096), dtype=torch.bfloat16)
    out = torch.zeros((8, 6144), dtype=torch.float32)
    q = torch.zeros((8, 4096), dtype=torch.uint8)
    s = torch.zeros((8, 32), dtype=torch.float32)
    with pytest.raises(ValueError, match="x: expected a CUDA tensor"):
        qdl.w8a8_proj(w, x, 8, out, q, s, stream=0)
    with pytest.raises(ValueError, match="expected a CUDA tensor"):
        qdl.kv_quant_int8(torch.zeros((4, 128)), 4, 128, torch.zeros((4, 128), dtype=torch.int8),
                          torch.zeros(4), stream=0)


@pytest.mark.parametrize("case", ["bf16_tensor_for_f32_out", "short_out", "short_x_rows", "int4_out", "kv_scale",
                                  "weight_scales", "fp8_codes"])
def test_binding_refuses_buffers_too_small_for_the_call(lib, case, monkeypatch):
    """each buffer must hold every byte the call will touch from its first
    element; these are refused in Python, before the library is called (host
    tensors stand in for device ones here, and the library is never reached)"""
    import torch
    monkeypatch.setattr(torch.Tensor, "is_cuda", property(lambda self: True))
    monkeypatch.setattr(qdl, "load", lambda path=None: pytest.fail("the library was called"))
    w = _wobj(lib)
    f32, bf16, u8 = torch.float32, torch.bfloat16, torch.uint8
    x = torch.zeros((8, 4096), dtype=bf16)
    q, s = torch.zeros((8, 4096), dtype=u8), torch.zeros((8, 32), dtype=f32)
    with pytest.raises(ValueError, match="storage holds"):
        if case == "bf16_tensor_for_f32_out":
            qdl.w8a8_proj(w, x, 8, torch.zeros((8, 6144), dtype=bf16), q, s, stream=0)
        elif case == "short_out":
            qdl.w8a8_gemv(w, q, s, 8, torch.zeros((8, 6144), dtype=f32)[1:], stream=0)
        elif case == "short_x_rows":
            qdl.w8a8_proj(w, torch.zeros((4, 4096), dtype=bf16), 8, torch.zeros((8, 6144), dtype=f32), q, s,
                          stream=0)
        elif case == "int4_out":
            outs = [torch.zeros((2, 128)), torch.zeros((2, 64)), torch.zeros((1, 64))]
            qdl.int4_qkv_gemv(torch.zeros((2, 256)), 2, 256, 128, 64, 128,
                              [torch.zeros((256, n // 8), dtype=torch.int32) for n in (128, 64, 64)],
                              [torch.zeros((2, n)) for n in (128, 64, 64)],
                              [torch.zeros((2, n)) for n in (128, 64, 64)], outs, stream=0)
        elif case == "kv_scale":
            qdl.kv_quant_int4(torch.zeros((4, 128)), 4, 128, 64, torch.zeros(256, dtype=u8), torch.zeros(7),
                              torch.zeros(8), stream=0)
        elif case == "weight_scales":
            qdl.w8a8_weight_init([(torch.zeros((256, 256), dtype=u8), torch.zeros(3))], qdl.BLOCK128)
        elif case == "fp8_codes":
            qdl.fp8_weight_quant(qdl.PER_ROW, torch.zeros((4, 256)), qdl.IN_F32, 256, 4, 256,
                                 torch.zeros((3, 256), dtype=u8), torch.zeros(4), stream=0)


def test_binding_views_are_measured_from_their_first_element(lib, monkeypatch):
    """a view in the middle of a larger buffer may use the storage after it,
    and the up half of a [rows, 2K] gate/up buffer is exactly large enough"""
    import torch
    w = _wobj(lib)
    buf = torch.zeros((8, 2 * 4096), dtype=torch.bfloat16)
    q, s = torch.zeros((8, 4096), dtype=torch.uint8), torch.zeros((8, 32))
    out = torch.zeros((8 * 6144 + 64,))[64:].view(8, 6144)
    seen = []
    monkeypatch.setattr(torch.Tensor, "is_cuda", property(lambda self: True))

    class Lib:  # records the call instead of making it
        def qdl_w8a8_proj_silu(self, *a):
            seen.append(a)
            return 0
    monkeypatch.setattr(qdl, "load", lambda path=None: Lib())
    qdl.w8a8_proj_silu(w, buf[:, :4096], buf[:, 4096:], 8, out, q, s, stream=0)
    assert len(seen) == 1
    # the up view starts K elements into the buffer; ld_gate = ld_up = 2K
    assert seen[0][2] - seen[0][1] == 4096 * 2 and seen[0][3] == seen[0][4] == 8192
    with pytest.raises(ValueError, match="up: the call touches"):
        qdl.w8a8_proj_silu(w, buf[:, :4096], buf[:, 4097:], 8, out, q, s, ld_up=8192, stream=0)


def test_binding_passes_raw_pointers_to_the_library_checks(lib):
    w = _wobj(lib)
    with pytest.raises(qdl.QdlError, match="rows"):
        qdl.w8a8_proj_static(w, DEV, 0, DEV + 0x4000000, ldx=4096, ldc=6144, stream=0)


def test_c_program_links_and_gets_validation_errors(lib, tmp_path):
    """the boundary used from C, without Python: a program that includes
    qdl.h, links libqdl.so and makes calls that are refused on the host"""
    prog = tmp_path / "use.c"
    prog.write_text(f'''#include <stdio.h>
#include <string.h>
#include "{HEADER}"
int main(void) {{
  size_t qb = 0, sb = 0;
  if (qdl_scratch_bytes(4096, &qb, &sb) != QDL_OK || qb != 256u * 4096 || sb != 256u * 32 * 4) return 1;
  qdl_fp8_segment seg[3];
  memset(seg, 0, sizeof seg);
  const unsigned long long dev = 0x7F0000000000ull;
  unsigned n[3] = {{4096, 1024, 1024}};
  for (int i = 0; i < 3; ++i) {{
    seg[i].weight = (const void *)(dev + 0x100000ull * i);
    seg[i].scale = (const float *)(dev + 0x8000000ull + 0x1000ull * i);
    seg[i].n = n[i];
    seg[i].k = 4096;
    seg[i].format = QDL_SCALE_BLOCK128;
  }}
  qdl_w8a8_weight w;
  if (qdl_w8a8_weight_init(&w, seg, 3) != QDL_OK || w.n != 6144) return 2;
  qdl_status st = qdl_w8a8_proj(&w, (const void *)dev, 4096, 0, (void *)(dev + 0x4000000ull), QDL_OUT_F32, 6144,
                                (unsigned char *)(dev + 0x1000000ull), (float *)(dev + 0x2000000ull), qb, sb, 0);
  printf("%d %s | %s\\n", (int)st, qdl_status_string(st), qdl_last_error());
  return st == QDL_ERR_INVALID_ARG ? 0 : 3;
}}
''')
    exe = tmp_path / "use"
    libdir = os.path.dirname(qdl.LIB_PATH)
    subprocess.run(["gcc", str(prog), "-o", str(exe), f"-L{libdir}", "-lqdl", f"-Wl,-rpath,{libdir}"], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, (r.returncode, r.stdout, r.stderr)
    assert r.stdout.startswith("1 QDL_ERR_INVALID_ARG | ") and "0 rows" in r.stdout, r.stdout
