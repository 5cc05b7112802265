"""qdl oracle: plain, slow CPU reference of the quantized decode-time linear layer.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  It shares no code with
the CUDA library: the C source here is compiled with gcc into its own shared
object and loaded with ctypes.

Functions and what they follow (the C source restates each in a comment):

* ``e4m3_encode`` / ``e4m3_decode`` -- OCP FP8 E4M3, round to nearest even,
  saturating at +-448.
* ``expf`` / ``silu_mul`` -- the library's written exp specification (Cody and
  Waite reduction, degree-7 Taylor polynomial) and SiLU(gate) * up.
* ``act_quant`` / ``act_quant_silu`` -- w8a8_decode.rs, ``w8a8_act_quant`` and
  ``w8a8_act_quant_silu``: scale = absmax / 448 per token row or per 128-group.
* ``w8a8_gemv`` / ``w8a8_gemv_sampled`` -- w8a8_decode.rs, ``w8a8_gemv`` over
  1..3 segments (``W8a8Weight::boundaries``), dequantise-then-dot in double.
* ``int4_qkv`` -- fused_int4_qkv.rs, ``fused_int4_qkv_{q,k,v}`` with
  ``unpack_awq_qkv`` and the shift table ``QKV_AWQ_SHIFTS``.
* ``kv_quant_int8`` / ``kv_dequant_int8`` / ``kv_quant_int4`` /
  ``kv_dequant_int4`` -- kv_cache_quant.wgsl: per-token symmetric int8 (the
  page's "FP8" and INT8 per-token kernels) and per-group asymmetric INT4 with
  two codes per byte.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

PER_ROW = 0
BLOCK128 = 1

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qdl_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liborc.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP when available) and return the path."""
    srcs = [_SRC, os.path.join(_HERE, "qdl_oracle.h")]
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= max(os.path.getmtime(s) for s in srcs)):
        return _LIB_PATH
    os.makedirs(_BUILD_DIR, exist_ok=True)
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    base = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math",
            "-fPIC", "-shared", "-Wall", "-o", tmp, _SRC]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:] + ["-lm"], check=True,
                       capture_output=True, text=True)
    except subprocess.CalledProcessError:
        subprocess.run(base + ["-lm"], check=True, capture_output=True, text=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            I = ctypes.c_int
            S = ctypes.c_size_t
            lib.orc_e4m3_encode_n.argtypes = [P, S, P]
            lib.orc_e4m3_decode_n.argtypes = [P, S, P]
            lib.orc_expf_n.argtypes = [P, S, P]
            lib.orc_silu_mul_n.argtypes = [P, P, S, P]
            lib.orc_act_quant.argtypes = [I, P, S, I, I, P, P]
            lib.orc_act_quant_silu.argtypes = [I, P, S, P, S, I, I, P, P]
            lib.orc_w8a8_gemv.argtypes = [I, P, P, I, I, I, P, P, P, P, P]
            lib.orc_w8a8_gemv_sampled.argtypes = [I, P, P, I, I, I, P, P, P, P, P, I, P, P]
            lib.orc_int4_qkv.argtypes = [P, I, I, I, I, I, P, P, P, P, P]
            lib.orc_kv_quant_int8.argtypes = [P, I, I, P, P]
            lib.orc_kv_dequant_int8.argtypes = [P, P, I, I, P]
            lib.orc_kv_quant_int4.argtypes = [P, S, I, P, P, P]
            lib.orc_kv_dequant_int4.argtypes = [P, P, P, S, I, P]
            lib.orc_fp8_weight_quant.argtypes = [I, P, S, I, I, P, P]
            lib.orc_awq_pack.argtypes = [P, I, I, P]
            lib.orc_num_threads.restype = I
            lib.orc_set_num_threads.argtypes = [I]
            _lib = lib
    return _lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _c(a, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


def num_threads() -> int:
    return _load().orc_num_threads()


def set_num_threads(n: int) -> None:
    """threads for the oracle's later parallel loops (timing only; results do
    not depend on it)"""
    _load().orc_set_num_threads(int(n))


def e4m3_encode(v) -> np.ndarray:
    v = _c(v, np.float32)
    out = np.empty(v.shape, np.uint8)
    _load().orc_e4m3_encode_n(_ptr(v), v.size, _ptr(out))
    return out


def e4m3_decode(c) -> np.ndarray:
    c = _c(c, np.uint8)
    out = np.empty(c.shape, np.float32)
    _load().orc_e4m3_decode_n(_ptr(c), c.size, _ptr(out))
    return out


def expf(x) -> np.ndarray:
    x = _c(x, np.float32)
    out = np.empty(x.shape, np.float32)
    _load().orc_expf_n(_ptr(x), x.size, _ptr(out))
    return out


def silu_mul(g, u) -> np.ndarray:
    g = _c(g, np.float32)
    u = _c(u, np.float32)
    assert g.shape == u.shape
    out = np.empty(g.shape, np.float32)
    _load().orc_silu_mul_n(_ptr(g), _ptr(u), g.size, _ptr(out))
    return out


def _scales_per_row(fmt: int, k: int) -> int:
    return 1 if fmt == PER_ROW else k // 128


def act_quant(fmt: int, x_bits, k: int):
    """x_bits: uint16 bf16 bit patterns [rows, ldx].  Returns (q [rows, k], s)."""
    x = _c(x_bits, np.uint16)
    rows, ldx = x.shape
    q = np.empty((rows, k), np.uint8)
    s = np.empty((rows, _scales_per_row(fmt, k)), np.float32)
    _load().orc_act_quant(fmt, _ptr(x), ldx, rows, k, _ptr(q), _ptr(s))
    return q, (s[:, 0].copy() if fmt == PER_ROW else s)


def act_quant_silu(fmt: int, gate_bits, up_bits, k: int):
    """gate_bits/up_bits: uint16 bf16 [rows, ld_*] (may be column views of one
    buffer).  Returns (q [rows, k], s)."""
    g = np.asarray(gate_bits)
    u = np.asarray(up_bits)
    assert g.dtype == np.uint16 and u.dtype == np.uint16
    rows = g.shape[0]
    # strided row views are allowed: pass the row stride, keep columns contiguous
    for a in (g, u):
        assert a.strides[1] == 2, "columns must be contiguous"
    q = np.empty((rows, k), np.uint8)
    s = np.empty((rows, _scales_per_row(fmt, k)), np.float32)
    _load().orc_act_quant_silu(fmt, g.ctypes.data, g.strides[0] // 2,
                               u.ctypes.data, u.strides[0] // 2, rows, k, _ptr(q), _ptr(s))
    return q, (s[:, 0].copy() if fmt == PER_ROW else s)


def _segment_arrays(segments):
    ws = [_c(w, np.uint8) for w, _ in segments]
    ss = [_c(s, np.float32) for _, s in segments]
    n = np.array([w.shape[0] for w in ws], np.int32)
    wp = (ctypes.c_void_p * len(ws))(*[_ptr(w) for w in ws])
    sp = (ctypes.c_void_p * len(ss))(*[_ptr(s) for s in ss])
    return ws, ss, n, wp, sp


def w8a8_gemv(fmt: int, q, sa, segments):
    """segments: list of (codes uint8 [n_s, K], scale f32 [n_s] or
    [ceil(n_s/128), K/128]).  Returns (y, bound), both float64 [rows, N]."""
    q = _c(q, np.uint8)
    sa = _c(sa, np.float32)
    rows, k = q.shape
    ws, ss, n, wp, sp = _segment_arrays(segments)
    N = int(n.sum())
    y = np.empty((rows, N), np.float64)
    b = np.empty((rows, N), np.float64)
    _load().orc_w8a8_gemv(fmt, _ptr(q), _ptr(sa), rows, k, len(ws), wp, sp, _ptr(n),
                          _ptr(y), _ptr(b))
    return y, b


def w8a8_gemv_sampled(fmt: int, q, sa, segments, rows_idx, cols_idx):
    q = _c(q, np.uint8)
    sa = _c(sa, np.float32)
    rows, k = q.shape
    ws, ss, n, wp, sp = _segment_arrays(segments)
    ri = _c(rows_idx, np.int32)
    ci = _c(cols_idx, np.int32)
    y = np.empty(ri.shape, np.float64)
    b = np.empty(ri.shape, np.float64)
    _load().orc_w8a8_gemv_sampled(fmt, _ptr(q), _ptr(sa), rows, k, len(ws), wp, sp, _ptr(n),
                                  _ptr(ri), _ptr(ci), ri.size, _ptr(y), _ptr(b))
    return y, b


def int4_qkv(x, nq: int, nkv: int, group: int, qw, sc, zr):
    """x f32 [m, k]; qw/sc/zr: 3-lists (q, k, v) of uint32 [k, n/8] and f32
    [k/group, n].  Returns (outs, bounds): 3-lists of float64 [m, n]."""
    x = _c(x, np.float32)
    m, k = x.shape
    qw = [_c(a, np.uint32) for a in qw]
    sc = [_c(a, np.float32) for a in sc]
    zr = [_c(a, np.float32) for a in zr]
    ns = [nq, nkv, nkv]
    outs = [np.empty((m, n), np.float64) for n in ns]
    bounds = [np.empty((m, n), np.float64) for n in ns]
    arr = lambda xs: (ctypes.c_void_p * 3)(*[_ptr(a) for a in xs])
    _load().orc_int4_qkv(_ptr(x), m, k, nq, nkv, group, arr(qw), arr(sc), arr(zr),
                         arr(outs), arr(bounds))
    return outs, bounds


def kv_quant_int8(x):
    """x f32 [tokens, dim] -> (codes int8 [tokens, dim], scales f32 [tokens])."""
    x = _c(x, np.float32)
    t, d = x.shape
    q = np.empty((t, d), np.int8)
    s = np.empty((t,), np.float32)
    _load().orc_kv_quant_int8(_ptr(x), t, d, _ptr(q), _ptr(s))
    return q, s


def kv_dequant_int8(q, s):
    q = _c(q, np.int8)
    s = _c(s, np.float32)
    t, d = q.shape
    out = np.empty((t, d), np.float32)
    _load().orc_kv_dequant_int8(_ptr(q), _ptr(s), t, d, _ptr(out))
    return out


def kv_quant_int4(x, group: int):
    """x f32 (any shape, flattened) -> (packed uint8 [n/2], scale f32 [n/group],
    zero f32 [n/group])."""
    x = _c(x, np.float32).reshape(-1)
    n = x.size
    assert group > 0 and group % 2 == 0 and n % group == 0
    packed = np.empty((n // 2,), np.uint8)
    sc = np.empty((n // group,), np.float32)
    zr = np.empty((n // group,), np.float32)
    _load().orc_kv_quant_int4(_ptr(x), n, group, _ptr(packed), _ptr(sc), _ptr(zr))
    return packed, sc, zr


def kv_dequant_int4(packed, scale, zero, n: int, group: int):
    packed = _c(packed, np.uint8).reshape(-1)
    scale = _c(scale, np.float32)
    zero = _c(zero, np.float32)
    out = np.empty((n,), np.float32)
    _load().orc_kv_dequant_int4(_ptr(packed), _ptr(scale), _ptr(zero), n, group, _ptr(out))
    return out


def fp8_weight_quant(fmt: int, w):
    """w f32 [n, k] (k % 128 == 0) -> (codes uint8 [n, k], scales f32 [n] for
    PER_ROW or [ceil(n/128), k/128] for BLOCK128)."""
    w = _c(w, np.float32)
    n, k = w.shape
    assert k % 128 == 0
    codes = np.empty((n, k), np.uint8)
    scales = np.empty((n,) if fmt == 0 else ((n + 127) // 128, k // 128), np.float32)
    _load().orc_fp8_weight_quant(fmt, _ptr(w), k, n, k, _ptr(codes), _ptr(scales))
    return codes, scales


def awq_pack(nib):
    """nib uint8 [k, n] (codes 0..15, n % 8 == 0) -> uint32 [k, n/8] in the
    AWQ shift order."""
    nib = _c(nib, np.uint8)
    k, n = nib.shape
    assert n % 8 == 0
    qw = np.empty((k, n // 8), np.uint32)
    _load().orc_awq_pack(_ptr(nib), k, n, _ptr(qw))
    return qw
