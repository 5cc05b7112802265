"""GPU parity: W8A8 GEMV and the fused decode projections against the oracle
(w8a8_decode.rs: w8a8_gemv, w8a8_proj, W8a8Weight::boundaries).

Outputs must be within 2e-3 * sum_k |x_hat w_hat| of the oracle's double
result; activation codes are bit-exact (test_gpu_act_quant.py), so both sides
see the same x_hat.  Small shapes compare every output; full-size workloads
compare a sample of outputs the oracle computes one by one."""
import functools

import numpy as np
import pytest
import torch

import oracle
import quantized_decode_linear_gb300 as qdl
from quantized_decode_linear_gb300 import synthetic as syn
from _gpu import BF16_REL, bf16_dev, check_close, dev, f32_bits_equal, host, scratch, upload_weight

pytestmark = pytest.mark.gpu

ROWS = [1, 2, 7, 8, 9, 16, 17, 33, 64, 100, 128, 129, 256]


def _segments(fmt, k, sizes, seed, std=0.02):
    return [syn.fp8_weight(n, k, fmt, std, seed + i) for i, n in enumerate(sizes)]


def _aligned_sizes(fmt, sizes):
    a = 16 if fmt == qdl.PER_ROW else 128
    return [n if i == len(sizes) - 1 else (n + a - 1) // a * a for i, n in enumerate(sizes)]


@pytest.mark.parametrize("fmt", [qdl.PER_ROW, qdl.BLOCK128])
@pytest.mark.parametrize("rows", ROWS)
def test_gemv_small_all_outputs(fmt, rows):
    k = 384
    sizes = _aligned_sizes(fmt, [256, 128, 200])
    segs = _segments(fmt, k, sizes, seed=rows)
    x = syn.bf16_normal((rows, k), seed=100 + rows)
    qo, so = oracle.act_quant(fmt, x, k)
    yo, bo = oracle.w8a8_gemv(fmt, qo, so, segs)
    w, _keep = upload_weight(segs, fmt)
    q = dev(qo)
    s = dev(so if fmt == qdl.BLOCK128 else so[:, None])
    out = torch.full((rows, w.n), float("nan"), device="cuda")
    qdl.w8a8_gemv(w, q, s, rows, out)
    torch.cuda.synchronize()
    check_close(host(out), yo, bo, what=f"fmt={fmt} rows={rows}")


@pytest.mark.parametrize("fmt", [qdl.PER_ROW, qdl.BLOCK128])
@pytest.mark.parametrize("sizes,k", [([16], 128), ([48], 256), ([7], 128), ([128, 128, 5], 256),
                                     ([256, 1000], 1024), ([4096, 1024, 1024], 4096)])
@pytest.mark.parametrize("rows", [1, 8, 16, 40])
def test_proj_segments_and_ragged_n(fmt, sizes, k, rows):
    sizes = _aligned_sizes(fmt, sizes)
    segs = _segments(fmt, k, sizes, seed=7 + len(sizes))
    ldx = k + 8
    x = syn.bf16_normal((rows, ldx), seed=rows * 3 + k)
    qo, so = oracle.act_quant(fmt, x, k)
    yo, bo = oracle.w8a8_gemv(fmt, qo, so, segs)
    w, _keep = upload_weight(segs, fmt)
    ldc = w.n + 5
    out = torch.full((rows, ldc), -7.0, device="cuda")
    q, s = scratch(rows, k, fmt)
    qdl.w8a8_proj(w, bf16_dev(x), rows, out, q, s, ldx=ldx, ldc=ldc)
    torch.cuda.synchronize()
    o = host(out)
    assert np.all(o[:, w.n:] == -7.0), "columns past N were written"
    assert np.array_equal(host(q), qo)
    check_close(o[:, :w.n], yo, bo, what=f"fmt={fmt} sizes={sizes} rows={rows}")


@pytest.mark.parametrize("fmt", [qdl.PER_ROW, qdl.BLOCK128])
@pytest.mark.parametrize("n,k,rows", [(384, 384, 3), (256, 8192, 8), (6144, 4096, 8), (1024, 14336, 64),
                                      (2048, 4096, 100), (640, 1024, 256), (1000, 2048, 33), (128, 8192, 128),
                                      (768, 2048, 20)])
def test_gemv_accumulating_output(fmt, n, k, rows):
    """QDL_OUT_F32_ADD adds y to the values already in out, with the split-K
    partial sums added atomically (shapes cover unsplit and split plans, and,
    for Block128 with 17 to 128 rows, the stream-K kernel with tiles shared
    by two CTAs and ragged N)"""
    segs = _segments(fmt, k, [n], seed=n + rows)
    x = syn.bf16_normal((rows, k), seed=7 + rows)
    qo, so = oracle.act_quant(fmt, x, k)
    yo, bo = oracle.w8a8_gemv(fmt, qo, so, segs)
    w, _keep = upload_weight(segs, fmt)
    base = np.random.default_rng(n).normal(0.0, 1.0, (rows, n)).astype(np.float32)
    out = dev(base)
    qdl.w8a8_gemv(w, dev(qo), dev(so if fmt == qdl.BLOCK128 else so[:, None]), rows, out,
                  out_dtype=qdl.OUT_F32_ADD)
    torch.cuda.synchronize()
    # the additions into out each round once more (at most split + 1 of them)
    check_close(host(out), base.astype(np.float64) + yo, bo + 2 ** -18 * np.abs(base) / 2e-3,
                what=f"fmt={fmt} split={qdl.w8a8_plan(w, rows)['split_k']}")


@pytest.mark.parametrize("rows", [64, 128, 256])
def test_gemv_accumulating_output_whole_tiles(rows):
    """QDL_OUT_F32_ADD on a weight wide enough that CTAs own whole output
    tiles (20480 rows in 160 tiles of K = 1024): a tile with a single writer
    must still add to what out held, not overwrite it"""
    fmt, n, k = qdl.BLOCK128, 20480, 1024
    segs = _segments(fmt, k, [n], seed=rows + 5)
    x = syn.bf16_normal((rows, k), seed=rows + 6)
    qo, so = oracle.act_quant(fmt, x, k)
    yo, bo = oracle.w8a8_gemv(fmt, qo, so, segs)
    w, _keep = upload_weight(segs, fmt)
    base = np.random.default_rng(rows).normal(0.0, 1.0, (rows, n)).astype(np.float32)
    out = dev(base)
    qdl.w8a8_gemv(w, dev(qo), dev(so), rows, out, out_dtype=qdl.OUT_F32_ADD)
    torch.cuda.synchronize()
    check_close(host(out), base.astype(np.float64) + yo, bo + 2 ** -18 * np.abs(base) / 2e-3,
                what=f"rows={rows} whole tiles")


@pytest.mark.parametrize("fmt", [qdl.PER_ROW, qdl.BLOCK128])
def test_bf16_output(fmt):
    rows, k = 9, 512
    segs = _segments(fmt, k, [256, 128], seed=3)
    x = syn.bf16_normal((rows, k), seed=4)
    qo, so = oracle.act_quant(fmt, x, k)
    yo, bo = oracle.w8a8_gemv(fmt, qo, so, segs)
    w, _keep = upload_weight(segs, fmt)
    out = torch.zeros((rows, w.n), dtype=torch.bfloat16, device="cuda")
    q, s = scratch(rows, k, fmt)
    qdl.w8a8_proj(w, bf16_dev(x), rows, out, q, s, out_dtype=qdl.OUT_BF16)
    torch.cuda.synchronize()
    check_close(host(out.float()), yo, bo, extra_rel=BF16_REL, what="bf16 out")


@pytest.mark.parametrize("fmt", [qdl.PER_ROW, qdl.BLOCK128])
@pytest.mark.parametrize("rows", [9, 100])
def test_bf16_output_unaligned_rows(fmt, rows):
    """bf16 output with a row stride of N + 3 elements: rows that start off an
    8-byte boundary take the element-wise stores, ragged N included; columns
    past N are not written"""
    k = 512
    segs = _segments(fmt, k, _aligned_sizes(fmt, [256, 130]), seed=rows + 7)
    x = syn.bf16_normal((rows, k), seed=rows + 8)
    qo, so = oracle.act_quant(fmt, x, k)
    yo, bo = oracle.w8a8_gemv(fmt, qo, so, segs)
    w, _keep = upload_weight(segs, fmt)
    ldc = w.n + 3
    out = torch.full((rows, ldc), -5.0, dtype=torch.bfloat16, device="cuda")
    q, s = scratch(rows, k, fmt)
    qdl.w8a8_proj(w, bf16_dev(x), rows, out, q, s, out_dtype=qdl.OUT_BF16, ldc=ldc)
    torch.cuda.synchronize()
    o = host(out.float())
    assert np.all(o[:, w.n:] == -5.0), "columns past N were written"
    check_close(o[:, :w.n], yo, bo, extra_rel=BF16_REL, what=f"bf16 ldc=N+3 fmt={fmt} rows={rows}")


def test_segment_identities_on_gpu():
    """3 segments == 3 single-segment calls concatenated; rows == single-row calls"""
    fmt, k, rows = qdl.BLOCK128, 256, 5
    segs = _segments(fmt, k, [128, 128, 64], seed=11)
    x = syn.bf16_normal((rows, k), seed=12)
    qo, so = oracle.act_quant(fmt, x, k)
    q, s = dev(qo), dev(so)
    w, _k1 = upload_weight(segs, fmt)
    full = torch.empty((rows, w.n), device="cuda")
    qdl.w8a8_gemv(w, q, s, rows, full)
    parts = []
    for seg in segs:
        ws, _k2 = upload_weight([seg], fmt)
        o = torch.empty((rows, ws.n), device="cuda")
        qdl.w8a8_gemv(ws, q, s, rows, o)
        parts.append(o)
    torch.cuda.synchronize()
    yo, bo = oracle.w8a8_gemv(fmt, qo, so, segs)
    check_close(host(full), yo, bo)
    check_close(host(torch.cat(parts, 1)), yo, bo)


# ---------------------------------------------------------------- full-size workloads

def _samples(rows, n, segments, count, seed):
    rng = np.random.default_rng(seed)
    r = [0, rows - 1, 0, rows - 1]
    c = [0, n - 1, n - 1, 0]
    start = 0
    for sz in segments:  # first and last column of every segment
        r += [rng.integers(rows), rng.integers(rows)]
        c += [start, start + sz - 1]
        start += sz
    r = np.array(r + list(rng.integers(0, rows, count)), np.int32)
    c = np.array(c + list(rng.integers(0, n, count)), np.int32)
    return r, c


def _full_workload(name, rows_list=None, samples=1500):
    wl = syn.WORKLOADS[name]
    segs = syn.w8a8_weights(wl)
    w, _keep = upload_weight(segs, wl.fmt)
    for rows in rows_list or wl.rows:
        xb = syn.w8a8_activations(wl, rows)
        q, s = scratch(rows, wl.k, wl.fmt)
        out = torch.empty((rows, wl.n), device="cuda")
        if wl.silu:
            d = bf16_dev(xb)
            qdl.w8a8_proj_silu(w, d[:, :wl.k], d[:, wl.k:], rows, out, q, s, ld_gate=2 * wl.k,
                               ld_up=2 * wl.k)
            qo, so = oracle.act_quant_silu(wl.fmt, xb[:, :wl.k], xb[:, wl.k:], wl.k)
        else:
            qdl.w8a8_proj(w, bf16_dev(xb), rows, out, q, s)
            qo, so = oracle.act_quant(wl.fmt, xb, wl.k)
        torch.cuda.synchronize()
        assert np.array_equal(host(q), qo), f"{name} rows={rows}: activation codes differ"
        sh = host(s)
        assert f32_bits_equal(sh[:, 0] if wl.fmt == qdl.PER_ROW else sh, so)
        r, c = _samples(rows, wl.n, wl.segments, samples, seed=rows)
        ys, bs = oracle.w8a8_gemv_sampled(wl.fmt, qo, so, segs, r, c)
        o = host(out)
        check_close(o[r, c], ys, bs, what=f"{name} rows={rows}")
        assert np.all(np.isfinite(o))


def test_full_perrow_m1_k1024_n1024_every_output():
    wl = syn.WORKLOADS["w8a8_perrow_m1_k1024_n1024"]
    segs = syn.w8a8_weights(wl)
    w, _keep = upload_weight(segs, wl.fmt)
    xb = syn.w8a8_activations(wl, 1)
    q, s = scratch(1, wl.k, wl.fmt)
    out = torch.empty((1, wl.n), device="cuda")
    qdl.w8a8_proj(w, bf16_dev(xb), 1, out, q, s)
    torch.cuda.synchronize()
    qo, so = oracle.act_quant(wl.fmt, xb, wl.k)
    yo, bo = oracle.w8a8_gemv(wl.fmt, qo, so, segs)
    check_close(host(out), yo, bo)


def test_full_block128_qkv_m8():
    _full_workload("w8a8_block128_qkv_m8_k4096_n4096+1024+1024")


def test_large_projections_back_to_back():
    """A 16-token projection over 16 MB of weights or more releases the next
    call's kernels at its start, and its split-K ranks add into the zeroed
    output without a cluster.  Back-to-back calls over two such weights, with
    no host synchronisation between them and one activation scratch, must each
    match the oracle: no kernel may read or write shared data before the call
    ahead of it has finished."""
    wl = syn.WORKLOADS["w8a8_block128_qkv_m8_k4096_n4096+1024+1024"]
    rows, k = 8, wl.k
    segs = [syn.w8a8_weights(wl), _segments(wl.fmt, k, wl.segments, seed=900)]
    weights = [upload_weight(sg, wl.fmt) for sg in segs]
    xs = [syn.w8a8_activations(wl, rows), syn.bf16_normal((rows, k), seed=901)]
    xd = [bf16_dev(x) for x in xs]
    refs = [oracle.act_quant(wl.fmt, x, k) for x in xs]
    q, s = scratch(rows, k, wl.fmt)
    outs = [torch.empty((rows, wl.n), device="cuda") for _ in range(4)]
    torch.cuda.synchronize()
    for rep in range(3):
        for i, out in enumerate(outs):
            qdl.w8a8_proj(weights[i % 2][0], xd[i % 2], rows, out, q, s)
        torch.cuda.synchronize()
        for i, out in enumerate(outs):
            qo, so = refs[i % 2]
            r, c = _samples(rows, wl.n, wl.segments, 400, seed=10 * rep + i)
            ys, bs = oracle.w8a8_gemv_sampled(wl.fmt, qo, so, segs[i % 2], r, c)
            o = host(out)
            check_close(o[r, c], ys, bs, what=f"repeat {rep} call {i}")
            assert np.all(np.isfinite(o))


def test_full_perrow_silu_down_m64():
    _full_workload("w8a8_perrow_silu_down_m64_k14336_n4096")


def test_full_block128_gateup_sweep():
    _full_workload("w8a8_block128_gateup_k8192_n14336+14336", samples=600)


@pytest.mark.parametrize("fmt", [qdl.PER_ROW, qdl.BLOCK128])
@pytest.mark.parametrize("rows", [8, 64, 256])
def test_back_to_back_calls_share_the_scratch(fmt, rows):
    """three projections queued with no host wait, each quantising into the
    same scratch that the previous call's GEMV reads: every GEMV must read
    its own call's codes and scales, never the previous call's (the kernels
    overlap under programmatic launch, so a scale read scheduled before the
    dependency wait would see the stale values)"""
    k = 512
    sizes = _aligned_sizes(fmt, [256, 128, 72])
    segs = _segments(fmt, k, sizes, seed=rows + 40)
    w, _keep = upload_weight(segs, fmt)
    q, s = scratch(rows, k, fmt)
    xs = [syn.bf16_normal((rows, k), seed=rows + 50 + i) for i in range(3)]
    outs = [torch.full((rows, w.n), float("nan"), device="cuda") for _ in xs]
    for x, out in zip(xs, outs):
        qdl.w8a8_proj(w, bf16_dev(x), rows, out, q, s)
    torch.cuda.synchronize()
    for i, (x, out) in enumerate(zip(xs, outs)):
        qo, so = oracle.act_quant(fmt, x, k)
        yo, bo = oracle.w8a8_gemv(fmt, qo, so, segs)
        check_close(host(out), yo, bo, what=f"fmt={fmt} rows={rows} call {i}")


@pytest.mark.parametrize("fmt", [qdl.PER_ROW, qdl.BLOCK128])
@pytest.mark.parametrize("rows", [257, 300, 600])
def test_proj_beyond_256_rows(fmt, rows):
    """prefill-shaped calls: passes of 256 rows through one 256-row scratch,
    ragged last pass, row stride beyond K; every output against the oracle"""
    k = 512
    sizes = _aligned_sizes(fmt, [256, 128, 72])
    segs = _segments(fmt, k, sizes, seed=rows)
    ldx = k + 16
    x = syn.bf16_normal((rows, ldx), seed=rows + 5)
    qo, so = oracle.act_quant(fmt, x, k)
    yo, bo = oracle.w8a8_gemv(fmt, qo, so, segs)
    w, _keep = upload_weight(segs, fmt)
    q, s = scratch(256, k, fmt)
    out = torch.full((rows, w.n), float("nan"), device="cuda")
    qdl.w8a8_proj(w, bf16_dev(x), rows, out, q, s, ldx=ldx)
    torch.cuda.synchronize()
    check_close(host(out), yo, bo, what=f"fmt={fmt} rows={rows}")


def test_proj_silu_beyond_256_rows_bf16():
    """SiLU-fused projection over 300 rows with bf16 output (ldc > N)"""
    fmt, k, rows = qdl.PER_ROW, 384, 300
    segs = _segments(fmt, k, [272], seed=3)
    xb = syn.bf16_normal((rows, 2 * k), seed=11)
    qo, so = oracle.act_quant_silu(fmt, xb[:, :k], xb[:, k:], k)
    yo, bo = oracle.w8a8_gemv(fmt, qo, so, segs)
    w, _keep = upload_weight(segs, fmt)
    q, s = scratch(256, k, fmt)
    ldc = w.n + 8
    out = torch.full((rows, ldc), float("nan"), device="cuda", dtype=torch.bfloat16)
    d = bf16_dev(xb)
    qdl.w8a8_proj_silu(w, d[:, :k], d[:, k:], rows, out, q, s, out_dtype=qdl.OUT_BF16, ld_gate=2 * k,
                       ld_up=2 * k, ldc=ldc)
    torch.cuda.synchronize()
    o = host(out.float())[:, :w.n]
    check_close(o, yo, bo, extra_rel=BF16_REL, what="silu rows=300 bf16")
    assert torch.isnan(out[:, w.n:].float()).all()


@functools.lru_cache(maxsize=1)
def _gateup_segments():
    return syn.w8a8_weights(syn.WORKLOADS["w8a8_block128_gateup_k8192_n14336+14336"])


def _every_tile_samples(rows, n, seed):
    """one output column per 128-wide output tile for every token row (a
    random column inside the tile, the tile's last column for the ragged
    end), so that every (token row, tile) pair is compared"""
    rng = np.random.default_rng(seed)
    tiles = (n + 127) // 128
    r = np.repeat(np.arange(rows, dtype=np.int32), tiles)
    t = np.tile(np.arange(tiles, dtype=np.int64), rows)
    c = np.minimum(t * 128 + rng.integers(0, 128, t.size), n - 1).astype(np.int32)
    return r, c


@pytest.mark.parametrize("rows", [32, 64, 128, 256])
def test_full_gateup_every_tile_every_row(rows):
    """the gate/up workload at the row counts whose GEMV splits tiles between
    CTAs (stream-K ranges at 17-128 rows, cluster split-K at 256): every token
    row of every 128-row output tile is compared with the oracle, so a tile
    whose shared partial sums went wrong cannot be missed"""
    wl = syn.WORKLOADS["w8a8_block128_gateup_k8192_n14336+14336"]
    segs = _gateup_segments()
    w, _keep = upload_weight(segs, wl.fmt)
    xb = syn.w8a8_activations(wl, rows)
    q, s = scratch(rows, wl.k, wl.fmt)
    out = torch.empty((rows, wl.n), device="cuda")
    qdl.w8a8_proj(w, bf16_dev(xb), rows, out, q, s)
    torch.cuda.synchronize()
    qo, so = oracle.act_quant(wl.fmt, xb, wl.k)
    assert np.array_equal(host(q), qo)
    r, c = _every_tile_samples(rows, wl.n, seed=rows)
    assert len(np.unique(c // 128)) == (wl.n + 127) // 128
    ys, bs = oracle.w8a8_gemv_sampled(wl.fmt, qo, so, segs, r, c)
    o = host(out)
    check_close(o[r, c], ys, bs, what=f"gate/up rows={rows}, every tile")
    assert np.all(np.isfinite(o))


@pytest.mark.parametrize("name,rows", [("w8a8_block128_qkv_m8_k4096_n4096+1024+1024", 8),
                                       ("w8a8_block128_qkv_m8_k4096_n4096+1024+1024", 64),
                                       ("w8a8_block128_gateup_k8192_n14336+14336", 16)])
def test_deterministic_f32_projection(name, rows):
    """QDL_OUT_F32_DETERMINISTIC: on shapes where the f32 projection adds
    split-K partials with atomics (the plan says it accumulates), repeated
    calls give identical bits and match the oracle"""
    wl = syn.WORKLOADS[name]
    segs = _gateup_segments() if wl.k == 8192 else syn.w8a8_weights(wl)
    w, _keep = upload_weight(segs, wl.fmt)
    assert qdl.w8a8_plan(w, rows)["proj_accumulates"] == 1
    xb = syn.bf16_normal((rows, wl.k), seed=rows + 77)
    x = bf16_dev(xb)
    q, s = scratch(rows, wl.k, wl.fmt)
    outs = []
    for _ in range(3):
        out = torch.full((rows, wl.n), float("nan"), device="cuda")
        qdl.w8a8_proj(w, x, rows, out, q, s, out_dtype=qdl.OUT_F32_DETERMINISTIC)
        outs.append(out)
    torch.cuda.synchronize()
    first = host(outs[0])
    for o in outs[1:]:
        assert f32_bits_equal(first, host(o)), "deterministic output differs between identical calls"
    qo, so = oracle.act_quant(wl.fmt, xb, wl.k)
    r, c = _every_tile_samples(rows, wl.n, seed=rows)
    ys, bs = oracle.w8a8_gemv_sampled(wl.fmt, qo, so, segs, r, c)
    check_close(first[r, c], ys, bs, what=f"{name} rows={rows} deterministic")


@pytest.mark.parametrize("fmt", [qdl.PER_ROW, qdl.BLOCK128])
@pytest.mark.parametrize("rows,dtype", [(257, qdl.OUT_F32), (300, qdl.OUT_BF16), (600, qdl.OUT_F32),
                                        (513, qdl.OUT_F32_DETERMINISTIC)])
def test_proj_beyond_256_rows_one_launch(fmt, rows, dtype):
    """prefill-shaped calls whose scratch holds every row: the rows are
    quantised 256 at a time and one GEMV launch covers them all (token blocks
    of 256); ragged last block, row stride beyond K, ldc beyond N; every
    output against the oracle, columns past N untouched"""
    k = 512
    sizes = _aligned_sizes(fmt, [256, 128, 72])
    segs = _segments(fmt, k, sizes, seed=rows + 1)
    ldx = k + 16
    x = syn.bf16_normal((rows, ldx), seed=rows + 9)
    qo, so = oracle.act_quant(fmt, x, k)
    yo, bo = oracle.w8a8_gemv(fmt, qo, so, segs)
    w, _keep = upload_weight(segs, fmt)
    q, s = scratch(rows, k, fmt)
    ldc = w.n + 4
    tdt = torch.bfloat16 if dtype == qdl.OUT_BF16 else torch.float32
    out = torch.full((rows, ldc), -3.0, device="cuda", dtype=tdt)
    qdl.w8a8_proj(w, bf16_dev(x), rows, out, q, s, ldx=ldx, ldc=ldc, out_dtype=dtype)
    torch.cuda.synchronize()
    o = host(out.float())
    assert np.all(o[:, w.n:] == -3.0), "columns past N were written"
    assert np.array_equal(host(q), qo)
    check_close(o[:, :w.n], yo, bo, extra_rel=BF16_REL if dtype == qdl.OUT_BF16 else 0.0,
                what=f"fmt={fmt} rows={rows}")


def test_full_gateup_512_rows_one_launch():
    """the gate/up workload at 512 rows through one GEMV launch: every token
    row of every 128-row tile compared with the oracle"""
    wl = syn.WORKLOADS["w8a8_block128_gateup_k8192_n14336+14336"]
    rows = 512
    segs = _gateup_segments()
    w, _keep = upload_weight(segs, wl.fmt)
    xb = syn.bf16_normal((rows, wl.k), seed=512)
    q, s = scratch(rows, wl.k, wl.fmt)
    out = torch.empty((rows, wl.n), device="cuda")
    qdl.w8a8_proj(w, bf16_dev(xb), rows, out, q, s)
    torch.cuda.synchronize()
    qo, so = oracle.act_quant(wl.fmt, xb, wl.k)
    assert np.array_equal(host(q), qo)
    r, c = _every_tile_samples(rows, wl.n, seed=rows)
    ys, bs = oracle.w8a8_gemv_sampled(wl.fmt, qo, so, segs, r, c)
    check_close(host(out)[r, c], ys, bs, what="gate/up rows=512 one launch")
