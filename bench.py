#!/usr/bin/env python3
"""Benchmark of the quantized decode-time linear layer on one GB300 (or N
independent replicas, one per GPU, under torchrun).

One step = one full decode projection call on one batch of synthetic input:
activation quantisation (optionally SiLU-fused) plus the GEMV over all
segments, for W8A8 workloads; the fused INT4 QKV GEMV for the AWQ workload.
Steps are replayed from CUDA graphs; the weights rotate over enough copies
that the working set is several times the L2 cache, so every step streams its
weights from HBM.

Prints one JSON line (rank 0).  `--impl reference` times the CPU oracle on a
bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "quantized decode GEMV µs/call & weight-stream GB/s (% of GB300 HBM roofline)"
DETERMINISTIC = False  # --deterministic: W8A8 projections with QDL_OUT_F32_DETERMINISTIC output
FALLBACK_HBM_GBS = 6800.0

# DRAM traffic per launch of the dominant kernel from one ncu capture
# (dram__bytes_read.sum + dram__bytes_write.sum), keyed by workload and rows;
# valid only while the hash of the kernel's code (comments excluded) matches.
# Source: profiles/.
TRAFFIC = {
    "w8a8_block128_gateup_k8192_n14336+14336@1": {"bytes": 235109632 + 170752, "file": "w8a8_gemm_tc.cu",
                                                  "src": "c94992fe805862c4"},
    "w8a8_block128_gateup_k8192_n14336+14336@2": {"bytes": 235226368 + 124416, "file": "w8a8_gemm_tc.cu",
                                                  "src": "c94992fe805862c4"},
    "w8a8_block128_gateup_k8192_n14336+14336@4": {"bytes": 235474944 + 378880, "file": "w8a8_gemm_tc.cu",
                                                  "src": "c94992fe805862c4"},
    "w8a8_block128_gateup_k8192_n14336+14336@8": {"bytes": 235969536 + 74752, "file": "w8a8_gemm_tc.cu",
                                                  "src": "c94992fe805862c4"},
    "w8a8_block128_gateup_k8192_n14336+14336@16": {"bytes": 236955904 + 123136, "file": "w8a8_gemm_tc.cu",
                                                   "src": "c94992fe805862c4"},
    "w8a8_block128_gateup_k8192_n14336+14336@32": {"bytes": 242545664 + 2216704, "file": "w8a8_gemm_tc.cu",
                                                   "src": "c94992fe805862c4"},
    "w8a8_block128_gateup_k8192_n14336+14336@64": {"bytes": 245203200 + 3141120, "file": "w8a8_gemm_tc.cu",
                                                   "src": "c94992fe805862c4"},
    "w8a8_block128_gateup_k8192_n14336+14336@128": {"bytes": 246682112 + 5856768, "file": "w8a8_gemm_tc.cu",
                                                    "src": "c94992fe805862c4"},
    "w8a8_block128_gateup_k8192_n14336+14336@256": {"bytes": 266647808 + 4793344, "file": "w8a8_gemm_tc.cu",
                                                    "src": "c94992fe805862c4"},
    "int4_awq_qkv_k4096_nq4096_nkv1024_g128@1": {"bytes": 14220800 + 0, "file": "int4_qkv_cc.cu",
                                                 "src": "9a4ee01b88bafbf2"},
    "int4_awq_qkv_k4096_nq4096_nkv1024_g128@4": {"bytes": 14359296 + 0, "file": "int4_qkv_cc.cu",
                                                 "src": "9a4ee01b88bafbf2"},
}


def _nvtx_push(torch, name):
    """NVTX range around a timed region (visible to ncu --nvtx and nsys)"""
    try:
        torch.cuda.nvtx.range_push(name)
    except Exception:
        pass


def _nvtx_pop(torch):
    try:
        torch.cuda.nvtx.range_pop()
    except Exception:
        pass


def _rank_world():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), \
        int(os.environ.get("LOCAL_RANK", "0"))


class Replicas:
    """N independent replicas of the step, one process per GPU under torchrun.
    The replicas exchange nothing on the data path: the only collectives are
    a barrier before each timed region and the maximum of the ranks' elapsed
    times after it.  `backend`/`device` are NCCL on the GPU; the same code runs
    over gloo on the CPU."""

    def __init__(self, world, backend="nccl", device="cuda"):
        self.world, self.device, self.dist = world, device, None
        if world > 1:
            import torch.distributed as dist
            dist.init_process_group(backend)
            self.dist = dist

    def barrier(self):
        if self.dist:
            self.dist.barrier()

    def max(self, v):
        """the maximum of `v` over all ranks"""
        if not self.dist:
            return float(v)
        import torch
        t = torch.tensor([float(v)], dtype=torch.float64, device=self.device)
        self.dist.all_reduce(t, op=self.dist.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.dist:
            self.dist.destroy_process_group()
            self.dist = None


def aggregate_gbs(bytes_per_step, steps, world, seconds):
    """whole-job throughput: the bytes every rank streamed over the slowest
    rank's time"""
    return bytes_per_step * steps * world / seconds / 1e9


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def _code_only(text):
    """C/CUDA source with comments removed and whitespace collapsed: what a
    DRAM-traffic record depends on (string and character literals kept)"""
    out, i, n, quote = [], 0, len(text), None
    while i < n:
        c = text[i]
        if quote:
            out.append(c)
            if c == "\\" and i + 1 < n:
                out.append(text[i + 1])
                i += 2
                continue
            if c == quote:
                quote = None
            i += 1
        elif c in "\"'":
            quote = c
            out.append(c)
            i += 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def _src_hash(names):
    """hash of the named csrc files' code, comments and layout excluded"""
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "quantized_decode_linear_gb300", "csrc", n), encoding="utf-8") as f:
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


# ---------------------------------------------------------------- workloads

class W8A8Case:
    """Device buffers for one W8A8 workload at `rows` token rows."""

    @staticmethod
    def device_weights(wl, torch, qdl, syn, l2_bytes):
        """the workload's weight, uploaded once, in enough copies that the
        copies together are at least 4x the L2 cache; shared by every row
        count of a sweep"""
        segs = syn.w8a8_weights(wl)
        weight_bytes = sum(c.nbytes + s.nbytes for c, s in segs)
        copies = max(1, math.ceil(4 * l2_bytes / weight_bytes))
        base = [(torch.from_numpy(c).cuda(), torch.from_numpy(s).cuda()) for c, s in segs]
        weights = [qdl.w8a8_weight_init(base, wl.fmt)]
        for _ in range(copies - 1):
            weights.append(qdl.w8a8_weight_init([(c.clone(), s.clone()) for c, s in base], wl.fmt))
        return {"segs": segs, "weights": weights, "weight_bytes": weight_bytes, "copies": copies}

    def __init__(self, wl, rows, torch, qdl, syn, l2_bytes, shared=None):
        self.wl, self.rows = wl, rows
        shared = shared or self.device_weights(wl, torch, qdl, syn, l2_bytes)
        segs = shared["segs"]
        self.weight_bytes, self.copies, self.weights = shared["weight_bytes"], shared["copies"], shared["weights"]
        xb = syn.w8a8_activations(wl, rows)
        self.x_host = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).pin_memory()
        self.x = self.x_host.cuda()
        k = wl.k
        self.q = torch.empty((rows, k), dtype=torch.uint8, device="cuda")
        spr = 1 if wl.fmt == qdl.PER_ROW else k // 128
        self.s = torch.empty((rows, spr), dtype=torch.float32, device="cuda")
        self.out = torch.empty((rows, wl.n), dtype=torch.float32, device="cuda")
        self.out_host = torch.empty((rows, wl.n), dtype=torch.float32).pin_memory()
        self.qdl = qdl
        n, K = wl.n, k
        w_scales = sum(s.nbytes for _, s in segs)
        x_bytes = rows * (2 * K if wl.silu else K) * 2
        # algorithmic bytes of one fused call: weights + weight scales + bf16 input + f32 output
        self.step_bytes = n * K + w_scales + x_bytes + rows * n * 4
        # the scratch holds every row, so a projection of more than 256 rows
        # quantises them 256 at a time and makes one GEMV launch over all of
        # them (streaming the weights once)
        self.chunks = [(d, min(256, rows - d)) for d in range(0, rows, 256)]
        # of the GEMV launch: weights + scales + e4m3 activations + act scales + output
        self.gemv_bytes = n * K + w_scales + rows * K + rows * spr * 4 + rows * n * 4
        self.gemv_launches = 1
        plans = [qdl.w8a8_plan(self.weights[0], min(rows, 256))]
        self.launches_per_step = len(self.chunks) + 1  # the quantiser per 256 rows, then the GEMV
        # the GEMV as the projection runs it: with split K it adds into the
        # zeroed f32 output
        self.out_dtype = qdl.OUT_F32_DETERMINISTIC if DETERMINISTIC else qdl.OUT_F32
        self.dom_dtypes = [qdl.OUT_F32_ADD if pl["proj_accumulates"] and not DETERMINISTIC else qdl.OUT_F32
                           for pl in plans]
        self.kernel = "w8a8_streamk_kernel" if plans[0]["proj_streamk"] else "w8a8_gemm_tc_kernel"
        self.kernel_src = ["w8a8_gemm_tc.cu"]
        if rows > 256:  # the public GEMV takes at most 256 rows: the whole projection is the dominant step
            self.kernel = "act_quant_g128_kernel + w8a8_gemm_tc_kernel"

    def step(self, i):
        w = self.weights[i % self.copies]
        wl, k, qdl = self.wl, self.wl.k, self.qdl
        if wl.silu:
            qdl.w8a8_proj_silu(w, self.x[:, :k], self.x[:, k:], self.rows, self.out, self.q, self.s,
                               ld_gate=2 * k, ld_up=2 * k, out_dtype=self.out_dtype)
        else:
            qdl.w8a8_proj(w, self.x, self.rows, self.out, self.q, self.s, out_dtype=self.out_dtype)

    def dominant(self, i):
        if self.rows > 256:
            return self.step(i)
        w = self.weights[i % self.copies]
        self.qdl.w8a8_gemv(w, self.q, self.s, self.rows, self.out, out_dtype=self.dom_dtypes[0])

    def e2e_step(self, i):
        self.x.copy_(self.x_host, non_blocking=True)
        self.step(i)
        self.out_host.copy_(self.out, non_blocking=True)

    def e2e_bytes(self):
        return self.x_host.numel() * 2, self.out_host.numel() * 4

    def describe(self):
        wl = self.wl
        return {"workload": wl.name, "rows": self.rows, "k": wl.k, "n_segments": list(wl.segments),
                "scale_format": "per_row" if wl.fmt == 0 else "block128", "silu_fused": wl.silu,
                "out_dtype": "f32 deterministic" if DETERMINISTIC else "f32", "weight_copies": self.copies,
                "l2": f"inputs larger than L2: weights rotate over {self.copies} copies "
                      f"({self.copies * self.weight_bytes / 1e6:.0f} MB)"}


class Int4Case:
    @staticmethod
    def device_weights(wl, torch, qdl, syn, l2_bytes):
        ws = syn.int4_weights(wl)
        weight_bytes = sum(a.nbytes for w in ws for a in w)
        copies = max(1, math.ceil(4 * l2_bytes / weight_bytes))
        base = [[torch.from_numpy(a.view(np.int32) if a.dtype == np.uint32 else a).cuda() for a in w]
                for w in ws]
        sets = [base] + [[[a.clone() for a in w] for w in base] for _ in range(copies - 1)]
        return {"sets": sets, "weight_bytes": weight_bytes, "copies": copies}

    def __init__(self, wl, rows, torch, qdl, syn, l2_bytes, shared=None):
        self.wl, self.rows = wl, rows
        shared = shared or self.device_weights(wl, torch, qdl, syn, l2_bytes)
        self.weight_bytes, self.copies, self.sets = shared["weight_bytes"], shared["copies"], shared["sets"]
        x = syn.int4_activations(wl, rows)
        self.x_host = torch.from_numpy(x).pin_memory()
        self.x = self.x_host.cuda()
        self.outs = [torch.empty((rows, n), device="cuda") for n in (wl.nq, wl.nkv, wl.nkv)]
        self.out_hosts = [torch.empty((rows, n)).pin_memory() for n in (wl.nq, wl.nkv, wl.nkv)]
        self.qdl = qdl
        n_tot = wl.nq + 2 * wl.nkv
        self.step_bytes = self.weight_bytes + x.nbytes + rows * n_tot * 4
        self.gemv_bytes = self.step_bytes
        # the library's dispatch for widths multiple of 32: up to 4 rows the
        # CUDA-core stream-K kernel (f32 products), else (group 128) tcgen05
        # passes of 16 rows (f16 operands); each is an output-zeroing launch
        # and the GEMV
        if rows <= 4:
            self.gemv_launches = 1
            self.kernel, self.kernel_src, self.dtype = "int4_qkv_sk_kernel", ["int4_qkv_cc.cu"], "f32"
        else:
            self.gemv_launches = math.ceil(rows / 16)
            self.kernel, self.kernel_src, self.dtype = "int4_qkv_tc_kernel", ["int4_qkv_tc.cu"], "f16"
        self.launches_per_step = 2 * self.gemv_launches

    def step(self, i):
        s = self.sets[i % self.copies]
        wl = self.wl
        self.qdl.int4_qkv_gemv(self.x, self.rows, wl.k, wl.nq, wl.nkv, wl.group, [w[0] for w in s],
                               [w[1] for w in s], [w[2] for w in s], self.outs)

    dominant = step

    def e2e_step(self, i):
        self.x.copy_(self.x_host, non_blocking=True)
        self.step(i)
        for h, d in zip(self.out_hosts, self.outs):
            h.copy_(d, non_blocking=True)

    def e2e_bytes(self):
        return self.x_host.numel() * 4, sum(h.numel() * 4 for h in self.out_hosts)

    def describe(self):
        wl = self.wl
        return {"workload": wl.name, "rows": self.rows, "k": wl.k, "nq": wl.nq, "nkv": wl.nkv,
                "group": wl.group, "weight_copies": self.copies,
                "l2": f"inputs larger than L2: weights rotate over {self.copies} copies "
                      f"({self.copies * self.weight_bytes / 1e6:.0f} MB)"}


class KvCase:
    """KV-cache quantiser workload: a step quantises one block of rows and
    dequantises another (long untouched) block; blocks rotate over enough
    copies that every step streams from HBM."""

    @staticmethod
    def device_weights(wl, torch, qdl, syn, l2_bytes):
        return None

    def __init__(self, wl, rows, torch, qdl, syn, l2_bytes, shared=None):
        self.wl, self.rows, self.qdl = wl, rows, qdl
        n = rows * wl.head_dim
        self.n = n
        x = syn.kv_values(wl, rows)
        self.int4 = wl.group > 0
        code_bytes = n // 2 if self.int4 else n
        side = (n // wl.group) * 8 if self.int4 else rows * 4  # scales (+ zeros)
        per_copy = 4 * n + code_bytes + side + 4 * n
        self.copies = max(2, math.ceil(4 * l2_bytes / per_copy))
        dev = torch.from_numpy(x).cuda()
        self.x = [dev] + [dev.clone() for _ in range(self.copies - 1)]
        self.out = [torch.empty_like(dev) for _ in range(self.copies)]
        if self.int4:
            self.q = [torch.empty((n // 2,), dtype=torch.uint8, device="cuda") for _ in range(self.copies)]
            self.s = [torch.empty((n // wl.group,), dtype=torch.float32, device="cuda") for _ in range(self.copies)]
            self.z = [torch.empty((n // wl.group,), dtype=torch.float32, device="cuda") for _ in range(self.copies)]
        else:
            self.q = [torch.empty((rows, wl.head_dim), dtype=torch.int8, device="cuda") for _ in range(self.copies)]
            self.s = [torch.empty((rows,), dtype=torch.float32, device="cuda") for _ in range(self.copies)]
            self.z = [None] * self.copies
        for i in range(self.copies):  # every block holds valid codes before the first dequantisation
            self._quant(i)
        self.x_host = torch.from_numpy(x).pin_memory()
        self.out_host = torch.empty(x.shape, dtype=torch.float32).pin_memory()
        self.weight_bytes = 0
        # algorithmic bytes: quantise (read x, write codes + side data) and
        # dequantise (read codes + side data, write values)
        self.gemv_bytes = 4 * n + code_bytes + side
        self.step_bytes = self.gemv_bytes + code_bytes + side + 4 * n
        self.gemv_launches, self.launches_per_step = 1, 2
        self.kernel = "kv_quant_int4_kernel" if self.int4 else "kv_quant_int8_kernel"
        self.kernel_src = ["kv_quant.cu"]
        self.dtype = "u4" if self.int4 else "int8"

    def _quant(self, i):
        wl, r, d = self.wl, self.rows, self.wl.head_dim
        if self.int4:
            self.qdl.kv_quant_int4(self.x[i], r, d, wl.group, self.q[i], self.s[i], self.z[i])
        else:
            self.qdl.kv_quant_int8(self.x[i], r, d, self.q[i], self.s[i])

    def _dequant(self, i):
        wl, r, d = self.wl, self.rows, self.wl.head_dim
        if self.int4:
            self.qdl.kv_dequant_int4(self.q[i], self.s[i], self.z[i], r, d, wl.group, self.out[i])
        else:
            self.qdl.kv_dequant_int8(self.q[i], self.s[i], r, d, self.out[i])

    def step(self, i):
        self._quant(i % self.copies)
        self._dequant((i + self.copies // 2) % self.copies)

    def dominant(self, i):
        self._quant(i % self.copies)

    def e2e_step(self, i):
        c = i % self.copies
        self.x[c].copy_(self.x_host, non_blocking=True)
        self._quant(c)
        self._dequant(c)
        self.out_host.copy_(self.out[c], non_blocking=True)

    def e2e_bytes(self):
        return self.x_host.numel() * 4, self.out_host.numel() * 4

    def describe(self):
        wl = self.wl
        return {"workload": wl.name, "rows": self.rows, "head_dim": wl.head_dim,
                "codec": f"int4 group {wl.group}" if self.int4 else "int8 per token",
                "copies": self.copies,
                "l2": f"inputs larger than L2: blocks rotate over {self.copies} copies "
                      f"({self.copies * (8 * self.n) / 1e6:.0f} MB of values)"}


class PrepCase:
    """Weight preparation workload: one step quantises a bf16 weight to FP8
    (fp8) or packs 4-bit codes into AWQ words (awq); buffers rotate over
    enough copies that every step streams from HBM."""

    @staticmethod
    def device_weights(wl, torch, qdl, syn, l2_bytes):
        return None

    def __init__(self, wl, rows, torch, qdl, syn, l2_bytes, shared=None):
        self.wl, self.rows, self.qdl = wl, rows, qdl
        self.fp8 = wl.prep == "fp8"
        if self.fp8:
            src = syn.prep_weight_bf16(wl)
            in_bytes = src.nbytes
            nsc = wl.n if wl.scale_format == 0 else ((wl.n + 127) // 128) * (wl.k // 128)
            out_bytes = wl.n * wl.k + 4 * nsc
            dev = torch.from_numpy(src.view(np.int16)).cuda().view(torch.bfloat16)
            self.host_in = torch.from_numpy(src.view(np.int16)).view(torch.bfloat16).pin_memory()
        else:
            src = syn.prep_codes(wl)
            in_bytes = src.nbytes
            out_bytes = wl.k * wl.n // 2
            dev = torch.from_numpy(src).cuda()
            self.host_in = torch.from_numpy(src).pin_memory()
        self.copies = max(1, math.ceil(4 * l2_bytes / (in_bytes + out_bytes))) if in_bytes + out_bytes < 4 * l2_bytes else 1
        self.src = [dev] + [dev.clone() for _ in range(self.copies - 1)]
        if self.fp8:
            shape = (wl.n,) if wl.scale_format == 0 else ((wl.n + 127) // 128, wl.k // 128)
            self.codes = [torch.empty((wl.n, wl.k), dtype=torch.uint8, device="cuda") for _ in range(self.copies)]
            self.scales = [torch.empty(shape, dtype=torch.float32, device="cuda") for _ in range(self.copies)]
            self.host_out = torch.empty((wl.n, wl.k), dtype=torch.uint8).pin_memory()
        else:
            self.codes = [torch.empty((wl.k, wl.n // 8), dtype=torch.int32, device="cuda") for _ in range(self.copies)]
            self.host_out = torch.empty((wl.k, wl.n // 8), dtype=torch.int32).pin_memory()
        self.weight_bytes = in_bytes
        self.gemv_bytes = self.step_bytes = in_bytes + out_bytes
        self.gemv_launches, self.launches_per_step = 1, 1
        self.kernel = "fp8_weight_quant_kernel" if self.fp8 else "awq_pack_kernel"
        self.kernel_src = ["weight_quant.cu"]
        self.dtype = "e4m3" if self.fp8 else "u4"

    def _call(self, c):
        wl = self.wl
        if self.fp8:
            self.qdl.fp8_weight_quant(wl.scale_format, self.src[c], self.qdl.IN_BF16, wl.k, wl.n, wl.k,
                                      self.codes[c], self.scales[c])
        else:
            self.qdl.awq_pack(self.src[c], wl.k, wl.n, self.codes[c])

    def step(self, i):
        self._call(i % self.copies)

    dominant = step

    def e2e_step(self, i):
        c = i % self.copies
        self.src[c].copy_(self.host_in, non_blocking=True)
        self._call(c)
        self.host_out.copy_(self.codes[c], non_blocking=True)

    def e2e_bytes(self):
        return self.host_in.numel() * self.host_in.element_size(), self.host_out.numel() * self.host_out.element_size()

    def describe(self):
        wl = self.wl
        d = {"workload": wl.name, "n": wl.n, "k": wl.k, "copies": self.copies,
             "l2": f"inputs larger than L2: {self.copies} cop{'y' if self.copies == 1 else 'ies'} of "
                   f"{self.step_bytes / 1e6:.0f} MB moved per step"}
        if self.fp8:
            d.update(input="bf16", scale_format="per_row" if wl.scale_format == 0 else "block128")
        return d


# ---------------------------------------------------------------- timing helpers

def _graph(torch, fn, start, count):
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(start, start + count):
            fn(i)
    return g


class GraphBlock:
    """`fn(i)` for `steps` consecutive step indices, captured into CUDA
    graphs: up to four distinct graphs of `chunk` calls replayed in turn, plus
    one remainder graph.  `replay()` issues all `steps` calls."""

    def __init__(self, torch, fn, steps, chunk):
        c = min(chunk, steps)
        self.full, rem = divmod(steps, c)
        self.main = [_graph(torch, fn, j * c, c) for j in range(min(self.full, 4))]
        self.tail = _graph(torch, fn, self.full * c, rem) if rem else None
        self.steps = steps

    def replay(self):
        for r in range(self.full):
            self.main[r % len(self.main)].replay()
        if self.tail is not None:
            self.tail.replay()


def block_steps(k_steps):
    """steps per captured block: a whole number of K-step sequences, at least
    250 calls so that graph launches are rare against the work"""
    return k_steps * max(1, math.ceil(250 / k_steps))


def time_region(torch, stream, group, fn, k_steps, region_s, repeats, name):
    """Median device time per step of `fn` over `repeats` timed regions.  Each
    region replays a captured block of whole K-step sequences until at least
    `region_s` seconds have been timed (exactly K steps, once, when
    region_s <= 0), bracketed by a barrier and synchronisations, with CUDA
    events on the launching stream; the slowest rank's time counts."""
    unit = k_steps if region_s <= 0 else block_steps(k_steps)
    blk = GraphBlock(torch, fn, unit, unit if unit <= 1000 else 250)
    blk.replay()  # the first replay uploads the graphs
    torch.cuda.synchronize()
    blocks = 1
    if region_s > 0:
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        blk.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        blocks = max(1, math.ceil(region_s / max(e0.elapsed_time(e1) / 1e3, 1e-9)))
    per_step = []
    for _ in range(max(1, repeats)):
        group.barrier()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        _nvtx_push(torch, name)
        e0.record(stream)
        for _ in range(blocks):
            blk.replay()
        e1.record(stream)
        _nvtx_pop(torch)
        torch.cuda.synchronize()
        per_step.append(group.max(e0.elapsed_time(e1) / 1e3) / (blocks * unit))
    del blk
    return {"s_per_step": statistics.median(per_step), "min": min(per_step), "max": max(per_step),
            "steps_per_region": blocks * unit, "repeats": len(per_step)}


class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap,utilization.gpu")

    def __init__(self, gpu_index):
        self.proc = None
        self.gpu = gpu_index

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        return self.parse(out)

    @staticmethod
    def parse(out):
        """median SM clock and throttle reasons from nvidia-smi CSV rows;
        samples with the GPU under 50% busy are gaps between timed regions
        (graph capture, host work) and count only in `samples`"""
        sm, loaded, mx, power, reasons = [], [], None, [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [v.strip() for v in line.split(",")]
            if len(f) < 10:
                continue
            try:
                mhz, mx, w, util = float(f[1]), float(f[2]), float(f[3]), float(f[9])
            except ValueError:
                continue
            sm.append(mhz)
            power.append(w)
            if util >= 50.0:
                loaded.append(mhz)
            for nm, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        use = loaded or sm
        return {"sm_mhz": statistics.median(use) if use else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm), "samples_under_load": len(loaded),
                "power_w_max": max(power) if power else None}


# ---------------------------------------------------------------- oracle timing

def _oracle_step_fn(wl, rows, syn, fraction):
    """returns (fn, bytes_equiv, sample description) for one oracle step on a
    fraction of the workload's output columns"""
    import oracle
    if hasattr(wl, "prep"):
        if wl.prep == "fp8":
            take = max(128, int(round(wl.n * fraction / 128)) * 128)
            w = syn.prep_weight_bf16(wl, take)
            w32 = (w.astype(np.uint32) << 16).view(np.float32)
            nsc = take if wl.scale_format == 0 else (take // 128) * (wl.k // 128)

            def fn():
                oracle.fp8_weight_quant(wl.scale_format, w32)
            return fn, take * wl.k * 3 + 4 * nsc, f"quantise {take} of {wl.n} rows"
        take = max(1, int(round(wl.k * fraction)))
        nib = syn.prep_codes(wl, take)

        def fn():
            oracle.awq_pack(nib)
        return fn, take * wl.n * 3 // 2, f"pack {take} of {wl.k} rows"
    if hasattr(wl, "head_dim"):
        take = max(64, int(round(rows * fraction)))
        x = syn.kv_values(wl, take)
        n = take * wl.head_dim

        def fn():
            if wl.group:
                p, sc, zr = oracle.kv_quant_int4(x, wl.group)
                oracle.kv_dequant_int4(p, sc, zr, n, wl.group)
            else:
                q, s = oracle.kv_quant_int8(x)
                oracle.kv_dequant_int8(q, s)
        code = n // 2 if wl.group else n
        side = (n // wl.group) * 8 if wl.group else take * 4
        return fn, 8 * n + 2 * (code + side), f"quantise + dequantise {take} of {rows} rows"
    if hasattr(wl, "fmt"):
        segs = syn.w8a8_weights(wl)
        xb = syn.w8a8_activations(wl, rows)
        n = wl.n
        cols = max(1, int(round(n * fraction)))
        rng = np.random.default_rng(0)
        ci = np.sort(rng.choice(n, cols, replace=False)).astype(np.int32)
        r_idx = np.repeat(np.arange(rows, dtype=np.int32), cols)
        c_idx = np.tile(ci, rows)
        step_bytes = W8A8Bytes(wl, rows, segs)

        def fn():
            if wl.silu:
                q, s = oracle.act_quant_silu(wl.fmt, xb[:, :wl.k], xb[:, wl.k:], wl.k)
            else:
                q, s = oracle.act_quant(wl.fmt, xb, wl.k)
            oracle.w8a8_gemv_sampled(wl.fmt, q, s, segs, r_idx, c_idx)
        return fn, step_bytes * cols / n, f"act quant of all {rows} rows + GEMV of {cols} of {n} output columns"
    ws = syn.int4_weights(wl)
    x = syn.int4_activations(wl, rows)
    # oracle INT4 on a column slice of each projection
    ns = (wl.nq, wl.nkv, wl.nkv)
    take = [max(8, int(round(n * fraction / 8)) * 8) for n in ns]
    sl = [(w[0][:, :t // 8].copy(), w[1][:, :t].copy(), w[2][:, :t].copy()) for w, t in zip(ws, take)]
    total_bytes = sum(a.nbytes for w in ws for a in w) + x.nbytes + rows * sum(ns) * 4

    def fn():
        oracle.int4_qkv(x, take[0], take[1], wl.group, [s[0] for s in sl], [s[1] for s in sl],
                        [s[2] for s in sl])
    frac = sum(take) / sum(ns)
    return fn, total_bytes * frac, f"all {rows} rows x {sum(take)} of {sum(ns)} output columns"


def W8A8Bytes(wl, rows, segs):
    w_scales = sum(s.nbytes for _, s in segs)
    return wl.n * wl.k + w_scales + rows * (2 * wl.k if wl.silu else wl.k) * 2 + rows * wl.n * 4


def _time_oracle(wl, rows, syn, budget_s):
    import oracle
    fn, b, desc = _oracle_step_fn(wl, rows, syn, 1.0 / 256)
    fn()  # the first call may load (or build) the oracle library
    t0 = time.perf_counter()
    fn()
    t_probe = time.perf_counter() - t0
    frac = min(1.0, (1.0 / 256) * max(1.0, budget_s / max(t_probe, 1e-3)))
    fn, b, desc = _oracle_step_fn(wl, rows, syn, frac)
    # repeat a sample that finishes early (the whole workload, for the small
    # ones) until about budget_s of CPU time has passed
    reps, t0 = 0, time.perf_counter()
    while True:
        fn()
        reps += 1
        dt = time.perf_counter() - t0
        if dt >= budget_s or frac < 1.0:
            break
    if reps > 1:
        desc = f"{desc}, repeated {reps} times"
    return {"value": b * reps / dt / 1e9, "unit": "GB/s", "cores": oracle.num_threads(), "kind": "oracle",
            "sample": desc, "seconds": dt}


# ---------------------------------------------------------------- arms

# The metric is quoted on the gate/up M sweep; these other workloads are
# timed more briefly in the same run and reported under "extra".
EXTRA = [("w8a8_block128_qkv_m8_k4096_n4096+1024+1024", 8),
         ("w8a8_perrow_m1_k1024_n1024", 1),
         ("w8a8_perrow_silu_down_m64_k14336_n4096", 64),
         ("int4_awq_qkv_k4096_nq4096_nkv1024_g128", 1),
         ("int4_awq_qkv_k4096_nq4096_nkv1024_g128", 4),
         ("int4_awq_qkv_k4096_nq4096_nkv1024_g128", 16)]


def _rows_list(args, wl):
    return [args.rows] if args.rows else list(wl.rows)


def _core_config(wl, rows_list, world):
    """the workload's shape keys, the same in both arms' JSON lines"""
    c = {"workload": wl.name, "rows": rows_list if len(rows_list) > 1 else rows_list[0]}
    if hasattr(wl, "fmt"):
        c.update(k=wl.k, n_segments=list(wl.segments), scale_format="per_row" if wl.fmt == 0 else "block128",
                 silu_fused=wl.silu, out_dtype="f32 deterministic" if DETERMINISTIC else "f32")
    elif hasattr(wl, "nq"):
        c.update(k=wl.k, nq=wl.nq, nkv=wl.nkv, group=wl.group)
    c["parallelism"] = "replicas" if world > 1 else "single"
    if len(rows_list) > 1:
        c["step"] = f"one decode call at each of the {len(rows_list)} row counts"
    return c


def run_reference(args, rank, world, budget_s=120.0):
    """times the oracle on rank 0 alone; one step is the oracle on a bounded
    sample of every row count of the workload, sized so the whole warm-up +
    timed run takes about `budget_s`"""
    if rank != 0:
        return
    from quantized_decode_linear_gb300 import synthetic as syn
    import oracle
    wl = syn.WORKLOADS[args.workload]
    rows_list = _rows_list(args, wl)
    per_rows = budget_s / max(1, args.steps + args.warmup) / len(rows_list)
    fns = []
    for rows in rows_list:
        fn, b, desc = _oracle_step_fn(wl, rows, syn, 1.0 / 512)
        t0 = time.perf_counter()
        fn()
        t_probe = max(time.perf_counter() - t0, 1e-4)
        frac = min(1.0, max(1.0 / 4096, (1.0 / 512) * per_rows / t_probe))
        fns.append((rows,) + _oracle_step_fn(wl, rows, syn, frac))
    for _ in range(args.warmup):
        for _, fn, _, _ in fns:
            fn()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        for _, fn, _, _ in fns:
            fn()
    dt = time.perf_counter() - t0
    step_bytes = sum(b for _, _, b, _ in fns)
    value = step_bytes * args.steps / dt / 1e9
    desc = "; ".join(f"rows={r}: {d}" for r, _, _, d in fns)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f32" if hasattr(wl, "head_dim") else "f64",
            "data": "synthetic",
            "config": _core_config(wl, rows_list, world),
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": oracle.num_threads(), "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def _case_class(wl):
    return (PrepCase if hasattr(wl, "prep") else W8A8Case if hasattr(wl, "fmt") else
            KvCase if hasattr(wl, "head_dim") else Int4Case)


def _measure_case(torch, stream, group, case, args, world, regions):
    """times one workload at one row count: the decode steps, the dominant
    kernel alone, the steps end to end with host copies, and warm L2"""
    K, W = args.steps, args.warmup
    for i in range(W):  # untimed warm-up steps (eager calls; also loads every kernel)
        case.step(i)
    torch.cuda.synchronize()
    r_steps, r_dom, r_e2e, r_warm = regions
    t = {"steps": time_region(torch, stream, group, case.step, K, r_steps[0], r_steps[1], "qdl timed steps"),
         "dominant": time_region(torch, stream, group, case.dominant, K, r_dom[0], r_dom[1],
                                 "qdl dominant kernel")}
    if r_e2e[1] > 0:
        t["e2e"] = time_region(torch, stream, group, case.e2e_step, K, r_e2e[0], r_e2e[1], "qdl end-to-end steps")
    if r_warm[1] > 0:
        t["warm"] = time_region(torch, stream, group, lambda i: case.step(0), K, r_warm[0], r_warm[1],
                                "qdl warm L2")
    return t


def _fp8_peak_tflops():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return 2.0 * float(json.load(f)["bf16_tflops"]), "measured bf16 burst x 2 (nominal fp8/bf16 ratio)"
    except Exception:
        return 2.0 * 1900.0, "fallback bf16 x 2"


def _summary(case, t, peak, world):
    """per-row-count figures of one measured case"""
    s = t["steps"]["s_per_step"]
    d = t["dominant"]["s_per_step"] / case.gemv_launches
    key = f"{case.wl.name}@{case.rows}"
    tr = TRAFFIC.get(key)
    traffic = tr["bytes"] if tr and [tr.get("file")] == case.kernel_src and \
        tr.get("src") == _src_hash(case.kernel_src) else None
    r = {"rows": case.rows, "us_per_call": s * 1e6, "gbs": case.step_bytes / s / 1e9 * world,
         "hbm_frac_step": case.step_bytes / s / 1e9 / peak,
         "us_spread": [t["steps"]["min"] * 1e6, t["steps"]["max"] * 1e6],
         "steps_timed": t["steps"]["steps_per_region"] * t["steps"]["repeats"],
         "kernel": case.kernel, "kernel_us": d * 1e6,
         "kernel_gbs": case.gemv_bytes / case.gemv_launches / d / 1e9,
         "kernel_frac": case.gemv_bytes / case.gemv_launches / d / 1e9 / peak,
         "traffic": traffic, "launches_per_step": case.launches_per_step}
    if isinstance(case, W8A8Case):
        flops = 2.0 * case.rows * case.wl.n * case.wl.k
        fp8_peak, _ = _fp8_peak_tflops()
        r["kernel_tflops"] = flops / case.gemv_launches / d / 1e12
        r["kernel_fp8_frac"] = r["kernel_tflops"] / fp8_peak
    if "e2e" in t:
        r["e2e_us_per_call"] = t["e2e"]["s_per_step"] * 1e6
    if "warm" in t:
        r["warm_l2_us_per_call"] = t["warm"]["s_per_step"] * 1e6
    return r


def run_gpu(args, rank, world, local_rank):
    import torch
    import quantized_decode_linear_gb300 as qdl
    from quantized_decode_linear_gb300 import build as qbuild
    from quantized_decode_linear_gb300 import synthetic as syn

    qbuild.build()
    torch.cuda.set_device(local_rank)
    group = Replicas(world)
    props = torch.cuda.get_device_properties(local_rank)
    l2 = getattr(props, "L2_cache_size", 0) or 126 * 2**20
    stream = torch.cuda.current_stream()
    peak, peak_kind = _peaks()
    rs = args.region_s
    main_regions = ((rs, args.repeats), (rs / 2, args.repeats), (rs / 2, 3), (rs / 4, 3))
    if rs <= 0:
        main_regions = ((0, 1), (0, 1), (0, 1), (0, 1))

    wl = syn.WORKLOADS[args.workload]
    Case = _case_class(wl)
    rows_list = _rows_list(args, wl)
    shared = Case.device_weights(wl, torch, qdl, syn, l2)
    clocks = ClockSampler(local_rank)
    clocks.start()
    time.sleep(0.3)
    sweep, cases = [], []
    for rows in rows_list:
        case = Case(wl, rows, torch, qdl, syn, l2, shared)
        t = _measure_case(torch, stream, group, case, args, world, main_regions)
        sweep.append(_summary(case, t, peak, world))
        h2d, d2h = case.e2e_bytes()
        cases.append((case.step_bytes, case.gemv_bytes, case.gemv_launches, case.launches_per_step, h2d, d2h,
                      t, case.describe(), case.kernel, getattr(case, "dtype", "e4m3")))
        del case
    extra = {}
    if args.extra:
        ex_regions = ((rs * 0.3, 3), (rs * 0.3, 3), (rs * 0.2, 1), (0.0, 0)) if rs > 0 else \
            ((0, 1), (0, 1), (0, 0), (0, 0))
        for name, rows in EXTRA:
            ewl = syn.WORKLOADS[name]
            EC = _case_class(ewl)
            ec = EC(ewl, rows, torch, qdl, syn, l2)
            et = _measure_case(torch, stream, group, ec, args, world, ex_regions)
            extra[f"{name}@{rows}"] = _summary(ec, et, peak, world)
            del ec
            torch.cuda.empty_cache()
    clk = clocks.stop()

    # one step = one decode call at every row count of the sweep
    step_s = sum(c[6]["steps"]["s_per_step"] for c in cases)
    step_bytes = sum(c[0] for c in cases)
    dom_s = sum(c[6]["dominant"]["s_per_step"] for c in cases)
    dom_bytes = sum(c[1] for c in cases)
    dom_launches = sum(c[2] for c in cases)
    traffic = [r["traffic"] for r in sweep]
    value = aggregate_gbs(step_bytes, 1, world, step_s)
    sw = len(rows_list) > 1
    cfg = _core_config(wl, rows_list, world)
    for key in ("weight_copies", "copies", "l2"):
        if key in cases[0][7]:
            cfg[key] = cases[0][7][key]
    cfg["timing"] = (f"median over {main_regions[0][1]} regions of >= {main_regions[0][0]:.2f} s, each "
                     f"whole {args.steps}-step sequences replayed from CUDA graphs" if rs > 0 else
                     f"{args.steps} steps, one region")
    kernels = sorted({r["kernel"] for r in sweep})
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": step_s * 1e3,
        "us_per_call": step_s * 1e6 / len(rows_list),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": cases[0][9], "data": "synthetic",
        "config": cfg,
        "roofline": {"bound": "hbm", "achieved": dom_bytes / dom_s / 1e9, "peak": peak, "unit": "GB/s",
                     "frac": dom_bytes / dom_s / 1e9 / peak,
                     "traffic": (sum(traffic) / dom_launches if all(v is not None for v in traffic)
                                 else None),
                     "kernel": " + ".join(kernels), "peak_source": f"{peak_kind} hbm_gbs",
                     "kernel_us": dom_s / dom_launches * 1e6,
                     "algorithmic_bytes_per_launch": dom_bytes / dom_launches,
                     "note": ("per launch, averaged over the sweep: the dominant launches' algorithmic bytes "
                              "and event times summed over the row counts" if sw else "per launch")},
        "hbm_frac_step": value / world / peak,
        "sweep": sweep,
        "gpu_launches": sum(c[3] * c[6]["steps"]["steps_per_region"] * c[6]["steps"]["repeats"] for c in cases),
        "gpu_launches_note": "library kernels in all timed step regions",
        "clocks": clk,
    }
    if all("e2e" in c[6] for c in cases):
        e2e_s = sum(c[6]["e2e"]["s_per_step"] for c in cases)
        line["e2e"] = {"value": aggregate_gbs(step_bytes, 1, world, e2e_s), "unit": "GB/s",
                       "h2d_bytes_per_step": sum(c[4] for c in cases),
                       "d2h_bytes_per_step": sum(c[5] for c in cases),
                       "us_per_step": e2e_s * 1e6,
                       "method": "graphs of copy-in from pinned host memory, call, copy-out"}
    if all("warm" in c[6] for c in cases):
        warm_s = sum(c[6]["warm"]["s_per_step"] for c in cases)
        line["warm_l2"] = {"value": aggregate_gbs(step_bytes, 1, world, warm_s), "unit": "GB/s",
                           "us_per_step": warm_s * 1e6,
                           "method": "same steps, one weight copy reused by every call (L2-resident when it fits)"}
    fp8_peak, fp8_src = _fp8_peak_tflops()
    line["fp8_peak_tflops"] = {"value": fp8_peak, "source": fp8_src}
    if extra:
        line["extra"] = extra
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = _cpu_baseline_rows(wl, rows_list, syn)
    if rank == 0:
        print(json.dumps(line), flush=True)
    group.close()


def _cpu_baseline_rows(wl, rows_list, syn, budget_s=12.0, single_budget_s=4.0):
    """the oracle on all host cores over a sample of every row count (the
    budget split evenly), plus a shorter single-threaded sample of the first"""
    import oracle
    parts = [_time_oracle(wl, r, syn, budget_s / len(rows_list)) for r in rows_list]
    secs = sum(p["seconds"] for p in parts)
    gb = sum(p["value"] * p["seconds"] for p in parts)
    line = {"value": gb / secs, "unit": "GB/s", "cores": parts[0]["cores"], "kind": "oracle",
            "sample": "; ".join(f"rows={r}: {p['sample']}" for r, p in zip(rows_list, parts)), "seconds": secs}
    cores = oracle.num_threads()
    oracle.set_num_threads(1)
    try:
        one = _time_oracle(wl, rows_list[0], syn, single_budget_s)
    finally:
        oracle.set_num_threads(cores)
    line["single_thread"] = {k: one[k] for k in ("value", "cores", "sample", "seconds")}
    line["single_thread"]["rows"] = rows_list[0]
    return line


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="qdl", choices=["qdl", "reference"])
    ap.add_argument("--workload", default=None,
                    help="one workload (all its row counts unless --rows); default: the gate/up sweep "
                         "plus the other workloads under 'extra'")
    ap.add_argument("--rows", type=int, default=None)
    ap.add_argument("--region-s", type=float, default=1.0,
                    help="seconds per timed region of the decode steps (the dominant kernel and e2e take half); "
                         "0: time exactly --steps steps once")
    ap.add_argument("--repeats", type=int, default=5, help="timed regions per measurement (median reported)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--deterministic", action="store_true",
                    help="W8A8 projections write f32 with the fixed-order split-K reduction")
    args = ap.parse_args()
    global DETERMINISTIC
    DETERMINISTIC = args.deterministic
    if args.steps < 1 or args.warmup < 3:
        ap.error("need --steps >= 1 and --warmup >= 3")
    if args.repeats < 1:
        ap.error("need --repeats >= 1")
    from quantized_decode_linear_gb300 import synthetic as syn
    args.extra = args.workload is None and args.rows is None
    args.workload = args.workload or syn.HEADLINE
    if args.workload not in syn.WORKLOADS:
        ap.error(f"unknown workload; choose from {sorted(syn.WORKLOADS)}")
    rank, world, local_rank = _rank_world()
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_gpu(args, rank, world, local_rank)


if __name__ == "__main__":
    main()
