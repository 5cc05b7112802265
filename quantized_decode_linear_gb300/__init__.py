"""Python binding of libqdl, the quantized decode-time linear layer for GB300.

Thin argument marshalling over the C ABI declared in ``include/qdl.h``: every
function here has the C entry point's name without the ``qdl_`` prefix, takes
torch CUDA tensors (or raw device pointers) and the current CUDA stream, and
calls the library through ctypes.  All computation happens in the library's
CUDA kernels; there is no host fallback.  If the library cannot be loaded the
call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

PER_ROW = 0
BLOCK128 = 1
OUT_F32 = 0
OUT_BF16 = 1
OUT_F32_ADD = 2  # qdl_w8a8_gemv only: out += y
OUT_F32_DETERMINISTIC = 3  # f32, split-K partials reduced in a fixed order (reproducible bits)
MAX_ROWS = 256
K_UNIT = 128

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "libqdl.so")

STATUS_NAMES = {0: "QDL_OK", 1: "QDL_ERR_INVALID_ARG", 2: "QDL_ERR_SCRATCH_TOO_SMALL",
                3: "QDL_ERR_UNSUPPORTED", 4: "QDL_ERR_CUDA", 5: "QDL_ERR_DEVICE_TIMEOUT"}

# every symbol include/qdl.h declares
EXPORTS = ("qdl_w8a8_weight_init", "qdl_scratch_bytes", "qdl_act_quant", "qdl_act_quant_silu",
           "qdl_w8a8_gemv", "qdl_w8a8_proj", "qdl_w8a8_proj_silu", "qdl_int4_qkv_gemv",
           "qdl_w8a8_proj_static", "qdl_w8a8_plan", "qdl_check_device_fault", "qdl_selftest_bounded_wait",
           "qdl_kv_quant_int8", "qdl_kv_dequant_int8", "qdl_kv_quant_int4", "qdl_kv_dequant_int4",
           "qdl_fp8_weight_quant", "qdl_awq_pack", "qdl_last_error", "qdl_status_string")


class QdlError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status
        self.message = message


class Fp8Segment(ctypes.Structure):
    _fields_ = [("weight", ctypes.c_void_p), ("scale", ctypes.c_void_p), ("n", ctypes.c_uint32),
                ("k", ctypes.c_uint32), ("format", ctypes.c_int32)]


class Plan(ctypes.Structure):
    _fields_ = [("kernel", ctypes.c_int32), ("mma_n", ctypes.c_uint32), ("tiles", ctypes.c_uint32),
                ("split_k", ctypes.c_uint32), ("stages", ctypes.c_uint32), ("threads", ctypes.c_uint32),
                ("smem_bytes", ctypes.c_uint32), ("resident_clusters", ctypes.c_int32),
                ("proj_launches", ctypes.c_uint32), ("proj_accumulates", ctypes.c_uint32),
                ("proj_streamk", ctypes.c_uint32)]

    def as_dict(self):
        return {f: getattr(self, f) for f, _ in self._fields_}


class W8A8WeightDesc(ctypes.Structure):
    _fields_ = [("segs", Fp8Segment * 3), ("count", ctypes.c_uint32), ("n", ctypes.c_uint32),
                ("k", ctypes.c_uint32), ("format", ctypes.c_int32), ("n1", ctypes.c_uint32),
                ("n2", ctypes.c_uint32), ("magic", ctypes.c_uint32)]


_lock = threading.Lock()
_lib = None


def load(path: str | None = None) -> ctypes.CDLL:
    """Load libqdl.so (built by ``quantized_decode_linear_gb300.build``)."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(f"libqdl.so is not built ({p}); run quantized_decode_linear_gb300.build.build()")
        lib = ctypes.CDLL(p)
        P, U32, I32, SZ = ctypes.c_void_p, ctypes.c_uint32, ctypes.c_int32, ctypes.c_size_t
        sig = {
            "qdl_w8a8_weight_init": [P, P, U32],
            "qdl_scratch_bytes": [U32, P, P],
            "qdl_act_quant": [I32, P, U32, U32, U32, P, P, SZ, SZ, P],
            "qdl_act_quant_silu": [I32, P, P, U32, U32, U32, U32, P, P, SZ, SZ, P],
            "qdl_w8a8_gemv": [P, P, P, SZ, SZ, U32, P, I32, U32, P],
            "qdl_w8a8_proj": [P, P, U32, U32, P, I32, U32, P, P, SZ, SZ, P],
            "qdl_w8a8_proj_silu": [P, P, P, U32, U32, U32, P, I32, U32, P, P, SZ, SZ, P],
            "qdl_int4_qkv_gemv": [P, U32, U32, U32, U32, U32, P, P, P, P, P],
            "qdl_w8a8_proj_static": [P, P, U32, U32, P, I32, U32, P],
            "qdl_fp8_weight_quant": [I32, P, I32, U32, U32, U32, P, P, P],
            "qdl_awq_pack": [P, U32, U32, P, P],
            "qdl_kv_quant_int8": [P, U32, U32, P, P, P],
            "qdl_kv_dequant_int8": [P, P, U32, U32, P, P],
            "qdl_kv_quant_int4": [P, U32, U32, U32, P, P, P, P],
            "qdl_kv_dequant_int4": [P, P, P, U32, U32, U32, P, P],
            "qdl_check_device_fault": [P],
            "qdl_w8a8_plan": [P, U32, P],
            "qdl_selftest_bounded_wait": [P, P, P, SZ, SZ, U32, P, U32, P],
            "qdl_last_error": [],
            "qdl_status_string": [ctypes.c_int],
        }
        for name, args in sig.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = ctypes.c_char_p if name in ("qdl_last_error", "qdl_status_string") else ctypes.c_int
        if path is None:
            _lib = lib
        return lib


def last_error() -> str:
    return _call("qdl_last_error").decode()


def _check(status: int):
    if status != 0:
        raise QdlError(status, last_error())


def _ptr(t, name: str = "tensor", nbytes: int | None = None) -> int | None:
    """device address of a CUDA tensor, or a raw device pointer (int) passed
    through; None -> NULL.  With `nbytes`, the bytes the call reads or writes
    from the tensor's first element must lie inside the tensor's storage, so
    that a buffer too small for the call (or of a narrower dtype than the call
    assumes) is refused here instead of being overrun on the device."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if nbytes is not None:
        avail = t.untyped_storage().nbytes() - t.storage_offset() * t.element_size()
        if nbytes > avail:
            raise ValueError(f"{name}: the call touches {nbytes} bytes from its first element, "
                             f"but its storage holds {avail}")
    if not t.is_cuda:
        raise ValueError(f"{name}: expected a CUDA tensor, got one on {t.device}")
    return t.data_ptr()


def _call(name: str, *args):
    """calls the library's `name` with arguments marshalled (and checked)
    beforehand"""
    return getattr(load(), name)(*args)


def _rows_span(rows: int, ld: int, width: int, elt: int) -> int:
    """bytes of `rows` rows of `width` elements at a row stride of `ld`"""
    return max(0, (rows - 1) * ld + width) * elt if rows > 0 else 0


def _out_elt(out_dtype: int) -> int:
    return 2 if out_dtype == OUT_BF16 else 4


def _nbytes(t) -> int:
    return t.numel() * t.element_size()


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


# ---------------------------------------------------------------- W8A8


class W8A8Weight:
    """A validated W8A8 weight (C struct qdl_w8a8_weight) plus references to
    the tensors it points at, so they outlive the descriptor."""

    def __init__(self, desc: W8A8WeightDesc, tensors):
        self.desc = desc
        self._tensors = tensors

    @property
    def n(self) -> int:
        return self.desc.n

    @property
    def k(self) -> int:
        return self.desc.k

    @property
    def format(self) -> int:
        return self.desc.format


def w8a8_weight_init(segments, fmt: int) -> W8A8Weight:
    """segments: list of (codes uint8 [n, k] CUDA tensor, f32 scales)."""
    segs = (Fp8Segment * max(1, len(segments)))()
    keep = []
    for i, (w, s) in enumerate(segments):
        n, k = w.shape[0], w.shape[1]
        s_bytes = (n if fmt == PER_ROW else -(-n // 128) * (k // 128)) * 4
        segs[i] = Fp8Segment(_ptr(w, f"segment {i} codes", n * k), _ptr(s, f"segment {i} scales", s_bytes), n, k,
                             fmt)
        keep += [w, s]
    desc = W8A8WeightDesc()
    _check(_call("qdl_w8a8_weight_init", ctypes.byref(desc), segs, len(segments)))
    return W8A8Weight(desc, keep)


def w8a8_plan(w: W8A8Weight, rows: int) -> dict:
    """Kernel and work split that qdl_w8a8_gemv would use for `rows` rows."""
    p = Plan()
    _check(_call("qdl_w8a8_plan", ctypes.byref(w.desc), rows, ctypes.byref(p)))
    return p.as_dict()


def scratch_bytes(max_k: int):
    q = ctypes.c_size_t()
    s = ctypes.c_size_t()
    _check(_call("qdl_scratch_bytes", max_k, ctypes.byref(q), ctypes.byref(s)))
    return q.value, s.value


def act_quant(fmt: int, x, rows: int, k: int, q, q_scale, ldx: int | None = None, stream=None):
    ldx = x.stride(0) if ldx is None else ldx
    _check(_call("qdl_act_quant", fmt, _ptr(x, "x", _rows_span(rows, ldx, k, 2)), ldx, rows, k, _ptr(q, "q"),
                 _ptr(q_scale, "q_scale"), _nbytes(q), _nbytes(q_scale), _stream(stream)))


def act_quant_silu(fmt: int, gate, up, rows: int, k: int, q, q_scale, ld_gate: int | None = None,
                   ld_up: int | None = None, stream=None):
    ld_gate = gate.stride(0) if ld_gate is None else ld_gate
    ld_up = up.stride(0) if ld_up is None else ld_up
    _check(_call("qdl_act_quant_silu", fmt, _ptr(gate, "gate", _rows_span(rows, ld_gate, k, 2)),
                 _ptr(up, "up", _rows_span(rows, ld_up, k, 2)), ld_gate, ld_up, rows, k,
                 _ptr(q, "q"), _ptr(q_scale, "q_scale"), _nbytes(q), _nbytes(q_scale),
                 _stream(stream)))


def w8a8_gemv(w: W8A8Weight, q, q_scale, rows: int, out, out_dtype: int = OUT_F32,
              ldc: int | None = None, stream=None):
    ldc = out.stride(0) if ldc is None else ldc
    o = _ptr(out, "out", _rows_span(rows, ldc, w.n, _out_elt(out_dtype)))
    _check(_call("qdl_w8a8_gemv", ctypes.byref(w.desc), _ptr(q, "q"), _ptr(q_scale, "q_scale"), _nbytes(q),
                 _nbytes(q_scale), rows, o, out_dtype, ldc, _stream(stream)))


def w8a8_proj(w: W8A8Weight, x, rows: int, out, q, q_scale, out_dtype: int = OUT_F32,
              ldx: int | None = None, ldc: int | None = None, stream=None):
    ldx = x.stride(0) if ldx is None else ldx
    ldc = out.stride(0) if ldc is None else ldc
    xp = _ptr(x, "x", _rows_span(rows, ldx, w.k, 2))
    o = _ptr(out, "out", _rows_span(rows, ldc, w.n, _out_elt(out_dtype)))
    _check(_call("qdl_w8a8_proj", ctypes.byref(w.desc), xp, ldx, rows, o, out_dtype, ldc, _ptr(q, "q"),
                 _ptr(q_scale, "q_scale"), _nbytes(q), _nbytes(q_scale), _stream(stream)))


def w8a8_proj_silu(w: W8A8Weight, gate, up, rows: int, out, q, q_scale, out_dtype: int = OUT_F32,
                   ld_gate: int | None = None, ld_up: int | None = None, ldc: int | None = None,
                   stream=None):
    ld_gate = gate.stride(0) if ld_gate is None else ld_gate
    ld_up = up.stride(0) if ld_up is None else ld_up
    ldc = out.stride(0) if ldc is None else ldc
    gp = _ptr(gate, "gate", _rows_span(rows, ld_gate, w.k, 2))
    up_ = _ptr(up, "up", _rows_span(rows, ld_up, w.k, 2))
    o = _ptr(out, "out", _rows_span(rows, ldc, w.n, _out_elt(out_dtype)))
    _check(_call("qdl_w8a8_proj_silu", ctypes.byref(w.desc), gp, up_, ld_gate, ld_up, rows, o, out_dtype, ldc,
                 _ptr(q, "q"), _ptr(q_scale, "q_scale"), _nbytes(q), _nbytes(q_scale),
                 _stream(stream)))


STATIC_SCRATCH_BYTES = 4 << 20


def w8a8_proj_static(w: W8A8Weight, x, rows: int, out, out_dtype: int = OUT_F32,
                     ldx: int | None = None, ldc: int | None = None, stream=None):
    """qdl_w8a8_proj without caller scratch, for callers that cannot allocate
    device memory (a plugin handed only input and output buffers, or a decode
    loop that must not risk cudaMalloc's synchronisation or failure).  Uses the
    library's built-in 4 MiB device array, shared by every call: calls that may
    overlap on the GPU must be serialised by the caller.  Make the first call on
    each device before any stream capture (it looks up the array's address)."""
    ldx = x.stride(0) if ldx is None else ldx
    ldc = out.stride(0) if ldc is None else ldc
    xp = _ptr(x, "x", _rows_span(rows, ldx, w.k, 2))
    o = _ptr(out, "out", _rows_span(rows, ldc, w.n, _out_elt(out_dtype)))
    _check(_call("qdl_w8a8_proj_static", ctypes.byref(w.desc), xp, ldx, rows, o, out_dtype, ldc,
                 _stream(stream)))


# ---------------------------------------------------------------- INT4


def int4_qkv_gemv(x, m: int, k: int, nq: int, nkv: int, group: int, qw, sc, zr, out, stream=None):
    """qw/sc/zr/out: 3-sequences (q, k, v) of CUDA tensors or device pointers."""
    ns = (nq, nkv, nkv)
    groups = k // group if group > 0 else 0

    def arr(name, xs, nbytes):
        return (ctypes.c_void_p * 3)(*[_ptr(t, f"{name}[{p}]", nbytes(ns[p])) for p, t in enumerate(xs)])

    _check(_call("qdl_int4_qkv_gemv", _ptr(x, "x", 4 * m * k), m, k, nq, nkv, group,
                 arr("qw", qw, lambda n: k * (n // 8) * 4), arr("sc", sc, lambda n: groups * n * 4),
                 arr("zr", zr, lambda n: groups * n * 4), arr("out", out, lambda n: 4 * m * n),
                 _stream(stream)))


IN_F32, IN_BF16 = 0, 1


def fp8_weight_quant(fmt: int, w, w_dtype: int, ldw: int, n: int, k: int, codes, scales, stream=None):
    """FP8 weight [n, k] with per-row ([n]) or 128x128-block ([ceil(n/128), k/128])
    f32 scales, absmax / 448, from f32 or bf16 w [n, ldw]."""
    s_bytes = (n if fmt == PER_ROW else -(-n // 128) * (k // 128)) * 4
    _check(_call("qdl_fp8_weight_quant", fmt, _ptr(w, "w", _rows_span(n, ldw, k, 2 if w_dtype == IN_BF16 else 4)),
                 w_dtype, ldw, n, k, _ptr(codes, "codes", n * k),
                 _ptr(scales, "scales", s_bytes), _stream(stream)))


def awq_pack(nib, k: int, n: int, qw, stream=None):
    """uint8 codes [k, n] -> uint32 [k, n/8] in the AWQ shift order."""
    _check(_call("qdl_awq_pack", _ptr(nib, "nib", k * n), k, n, _ptr(qw, "qw", k * (n // 8) * 4), _stream(stream)))


def kv_quant_int8(x, tokens: int, head_dim: int, q, scale, stream=None):
    """KV-cache per-token int8: x f32 [tokens, head_dim] -> q int8, scale f32 [tokens]."""
    n = tokens * head_dim
    _check(_call("qdl_kv_quant_int8", _ptr(x, "x", 4 * n), tokens, head_dim, _ptr(q, "q", n),
                 _ptr(scale, "scale", 4 * tokens), _stream(stream)))


def kv_dequant_int8(q, scale, tokens: int, head_dim: int, out, stream=None):
    n = tokens * head_dim
    _check(_call("qdl_kv_dequant_int8", _ptr(q, "q", n), _ptr(scale, "scale", 4 * tokens), tokens, head_dim,
                 _ptr(out, "out", 4 * n), _stream(stream)))


def kv_quant_int4(x, tokens: int, head_dim: int, group: int, packed, scale, zero, stream=None):
    """KV-cache per-group INT4: packed uint8 [tokens*head_dim/2], scale/zero f32 [tokens*head_dim/group]."""
    n = tokens * head_dim
    g = n // group if group > 0 else 0
    _check(_call("qdl_kv_quant_int4", _ptr(x, "x", 4 * n), tokens, head_dim, group, _ptr(packed, "packed", n // 2),
                 _ptr(scale, "scale", 4 * g), _ptr(zero, "zero", 4 * g), _stream(stream)))


def kv_dequant_int4(packed, scale, zero, tokens: int, head_dim: int, group: int, out, stream=None):
    n = tokens * head_dim
    g = n // group if group > 0 else 0
    _check(_call("qdl_kv_dequant_int4", _ptr(packed, "packed", n // 2), _ptr(scale, "scale", 4 * g),
                 _ptr(zero, "zero", 4 * g), tokens, head_dim, group, _ptr(out, "out", 4 * n),
                 _stream(stream)))


def selftest_bounded_wait(w: W8A8Weight, q, q_scale, rows: int, out, limit_us: int = 20000,
                          stream=None) -> int:
    """Run the GEMV with one pipeline stage withheld so that its bounded waits
    give up; returns the status (QDL_ERR_DEVICE_TIMEOUT = 5 when they did)."""
    o = _ptr(out, "out", _rows_span(rows, w.n, w.n, 4))
    return _call("qdl_selftest_bounded_wait", ctypes.byref(w.desc), _ptr(q, "q"), _ptr(q_scale, "q_scale"), _nbytes(q),
                 _nbytes(q_scale), rows, o, limit_us, _stream(stream))


def check_device_fault(stream=None):
    _check(_call("qdl_check_device_fault", _stream(stream)))
