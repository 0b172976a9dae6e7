"""K splits of the DP4A GEMV: clusters of ks blocks share a tile range, each
block summing its 1/ks of the K chunks, the leader adding the ranks' per-row
sums in rank order.  Forced through W4_TUNE_K_SPLITS and compared with the
unsplit launch and the oracle:
  - per-row INT4: exact integer partial sums, so y is bit-identical to the
    unsplit GEMV ("Jetson Orin AGX INT4 推理优化实践", §"INT32 accumulator 是否
    安全": the int32 sums are exact in any order);
  - Q4_0, I8G32, Q6G32: fp32 group sums added in another order, within the
    tolerance of the summed term magnitudes ("在香橙派上跑 Gemma4", §3.1, §3.2).
Paths covered (K is split for one and two tokens): fused quantize, codes in
shared or global memory, the RMSNorm prologue, the gated epilogue with a
residual, two tokens, and a cluster with several rounds and more rows than the
staged per-row parameters.
"""
import numpy as np
import pytest

import oracle
from bit_quantized_decode_gb300 import workloads as wl
from helpers import RTOL_GROUP, RTOL_W4, check_close, cuda_ok, dev, group_scale, host, q4_0_scales, w4_scale

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not cuda_ok(), reason="needs a CUDA GPU")]


@pytest.fixture(scope="module")
def lib():
    import torch  # noqa: F401

    from bit_quantized_decode_gb300 import _lib
    _lib.load()
    _lib.clear_device_error()
    yield _lib
    for k in _lib.TUNE_KEYS:
        _lib.set_tuning(k, 0)
    assert _lib.device_error() == 0


def _run(lib, ks, fn, **tune):
    """Call fn() with K splits forced to ks (1: none) and the other tuning keys given."""
    import torch
    lib.set_tuning("k_splits", ks)
    for k, v in tune.items():
        lib.set_tuning(k, v)
    try:
        out = fn()
        torch.cuda.synchronize()
        return out
    finally:
        lib.set_tuning("k_splits", 0)
        for k in tune:
            lib.set_tuning(k, 0)


def _w4(lib, g, N, K):
    import torch
    W = wl.weights(g, N, K)
    q, sw = oracle.quantize_rows_int4(W)
    b = wl.bias(g, N)
    w = torch.empty(lib.w4_repacked_bytes(N, K), dtype=torch.uint8, device="cuda")
    lib.w4_repack([dev(oracle.pack_int4(q).view(np.int32))], K, w)
    return q, sw, b, w


def _plan_splits(lib, fmt, M, N, K, **kw):
    return lib.w4_plan(fmt, M, N, K, lib.w4_describe_device(), **kw)["k_splits"]


@pytest.mark.parametrize("M,N,K,ks", [(1, 512, 3584, 2), (1, 512, 3584, 4), (2, 200, 1536, 2), (2, 1000, 18944, 8),
                                      (1, 96, 1024, 2)])
def test_w4_linear_split_bit_identical(lib, M, N, K, ks):
    import torch
    g = wl.rng(900 + M + N + K + ks)
    q, sw, b, w = _w4(lib, g, N, K)
    x = wl.activations(g, M, K, outliers=(M == 1))
    swd, bd, xd = dev(sw), dev(b), dev(x)

    def call():
        y = torch.empty((M, N), device="cuda")
        qx = torch.empty((M, K), dtype=torch.int8, device="cuda")
        sx = torch.empty(M, device="cuda")
        lib.w4a8_linear(w, swd, bd, xd, y, qx, sx)
        return host(y), host(qx), host(sx)

    old = lib.get_tuning("k_splits")
    lib.set_tuning("k_splits", ks)
    assert _plan_splits(lib, "w4", M, N, K) == ks
    lib.set_tuning("k_splits", old)
    y1, _, _ = _run(lib, 1, call)
    yk, qk, sk = _run(lib, ks, call)
    assert np.array_equal(yk.view(np.uint32), y1.view(np.uint32))
    y_ref, qx_ref, sx_ref, acc = oracle.w4a8_linear(oracle.pack_int4(q), sw, x, b)
    assert np.array_equal(qk, qx_ref) and np.array_equal(sk.view(np.uint32), sx_ref.view(np.uint32))
    check_close(yk, y_ref, w4_scale(acc, sw, sx_ref, b), RTOL_W4, f"split {ks}")


def test_w4_gemv_on_codes_split_and_many_rounds(lib):
    """Codes input (shared-memory and global-memory paths), eight blocks in
    clusters of two: 625 tiles per cluster range of about 157 tiles, three
    rounds and 1256 rows per cluster, past the staged per-row parameters."""
    import torch
    M, N, K = 2, 5000, 1536
    g = wl.rng(77)
    q = wl.int_codes(g, (N, K), -8, 7)
    qx = wl.int_codes(g, (M, K), -127, 127)
    sw = wl.positive_scales(g, N, 1e-3, 3e-3)
    sx = wl.positive_scales(g, M, 1e-2, 2e-2)
    b = wl.bias(g, N)
    w = torch.empty(lib.w4_repacked_bytes(N, K), dtype=torch.uint8, device="cuda")
    lib.w4_repack([dev(oracle.pack_int4(q).view(np.int32))], K, w)
    args = [dev(sw), dev(b), dev(qx), dev(sx)]

    def call():
        y = torch.empty((M, N), device="cuda")
        lib.w4a8_gemv(w, args[0], args[1], args[2], args[3], y)
        return host(y)

    y1 = _run(lib, 1, call, grid_blocks=8)
    y2 = _run(lib, 2, call, grid_blocks=8)
    assert np.array_equal(y1.view(np.uint32), y2.view(np.uint32))
    acc = oracle.gemv_w4a8_acc(oracle.pack_int4(q), qx)
    y_ref = oracle.epilogue_w4a8(acc, sw, sx, b)
    check_close(y2, y_ref, w4_scale(acc, sw, sx, b), RTOL_W4, "codes, split 2, 8 blocks")


def test_w4_fused_norm_glu_residual_split(lib):
    """RMSNorm prologue, then a gated linear with a residual, K split in four."""
    import torch
    M, I, K = 1, 300, 3584
    g = wl.rng(31)
    Wg, Wu = wl.weights(g, I, K), wl.weights(g, I, K)
    qg, swg = oracle.quantize_rows_int4(Wg)
    qu, swu = oracle.quantize_rows_int4(Wu)
    bg, bu = wl.bias(g, I), wl.bias(g, I)
    gam = wl.norm_weight(g, K)
    x = wl.residual_stream(g, M, K)
    h = wl.residual_stream(g, M, I)
    w = torch.empty(lib.w4_glu_repacked_bytes(I, K), dtype=torch.uint8, device="cuda")
    lib.w4_repack_glu(dev(oracle.pack_int4(qg).view(np.int32)), dev(oracle.pack_int4(qu).view(np.int32)), K, w)
    sw, b = dev(np.concatenate([swg, swu])), dev(np.concatenate([bg, bu]))
    xd, hd, gd = dev(x), dev(h), dev(gam)

    def call():
        y = torch.empty((M, I), device="cuda")
        qx = torch.empty((M, K), dtype=torch.int8, device="cuda")
        sx = torch.empty(M, device="cuda")
        fz = lib.fusion(gd, 1e-6, lib.W4_GLU_SILU, hd)
        lib.w4a8_linear_fused(w, sw, b, xd, y, qx, sx, fz)
        return host(y)

    y1 = _run(lib, 1, call)
    y4 = _run(lib, 4, call)
    assert np.array_equal(y1.view(np.uint32), y4.view(np.uint32))


@pytest.mark.parametrize("fmt,M,N,K,ks", [("q4_0", 1, 2560, 1536, 2), ("q4_0", 1, 1536, 6144, 4),
                                          ("q4_0", 2, 333, 1536, 2), ("i8g32", 2, 700, 1536, 2),
                                          ("q6g32", 1, 512, 1536, 2)])
def test_group_formats_split_within_tolerance(lib, fmt, M, N, K, ks):
    import torch
    g = wl.rng(500 + N + K + ks)
    x = wl.activations(g, M, K)
    b = wl.bias(g, N)
    qx_ref, sx_ref = oracle.quantize_act_int8(x)
    if fmt == "q4_0":
        blocks = oracle.quantize_q4_0(wl.weights(g, N, K, 0.03))
        y_ref, acc = oracle.gemv_q4_0(blocks, qx_ref, sx_ref, b, want_acc=True)
        scale = group_scale(acc, q4_0_scales(blocks), sx_ref, b)
        w = torch.empty(lib.q4_0_repacked_bytes(N, K), dtype=torch.uint8, device="cuda")
        lib.q4_0_repack([dev(blocks)], K, w)
    else:
        q, d = oracle.quantize_i8g32(wl.weights(g, N, K))
        y_ref, acc = oracle.gemv_i8g32(q, d, qx_ref, sx_ref, b, want_acc=True)
        scale = group_scale(acc, d.view(np.float16).astype(np.float64), sx_ref, b)
        nbytes = lib.i8g32_repacked_bytes(N, K) if fmt == "i8g32" else lib.q6g32_repacked_bytes(N, K)
        w = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
        getattr(lib, f"{fmt}_repack")([dev(q)], [dev(d.view(np.int16))], K, w)
    bd, xd = dev(b), dev(x)

    def call():
        y = torch.empty((M, N), device="cuda")
        qx = torch.empty((M, K), dtype=torch.int8, device="cuda")
        sx = torch.empty(M, device="cuda")
        getattr(lib, f"{fmt}_linear")(w, bd, xd, y, qx, sx)
        return host(y)

    for ksplit in (1, ks):
        check_close(_run(lib, ksplit, call), y_ref, scale, RTOL_GROUP, f"{fmt} split {ksplit}")
