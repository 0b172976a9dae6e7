"""The 6-bit packed lm_head format (Q6G32): the I8G32 values in 6 bits.

The repack must be lossless (decoded on the CPU from the documented layout),
and the GEMV and fused linear must give the I8G32 results bit for bit (same
codes, same group order) and the oracle's within the group-format tolerance.
"""
import numpy as np
import pytest

import oracle
from bit_quantized_decode_gb300 import workloads as wl
from helpers import RTOL_GROUP, check_close, cuda_ok, decode_q6g32, dev, group_scale, host

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not cuda_ok(), reason="needs a CUDA GPU")]


@pytest.fixture(scope="module")
def lib():
    import torch  # noqa: F401

    from bit_quantized_decode_gb300 import _lib
    _lib.load()
    _lib.clear_device_error()
    yield _lib
    assert _lib.device_error() == 0


def _packs(lib, q_shards, d_shards, K):
    import torch
    N = sum(q.shape[0] for q in q_shards)
    w6 = torch.empty(lib.q6g32_repacked_bytes(N, K), dtype=torch.uint8, device="cuda")
    lib.q6g32_repack([dev(q) for q in q_shards], [dev(d.view(np.int16)) for d in d_shards], K, w6)
    w8 = torch.empty(lib.i8g32_repacked_bytes(N, K), dtype=torch.uint8, device="cuda")
    lib.i8g32_repack([dev(q) for q in q_shards], [dev(d.view(np.int16)) for d in d_shards], K, w8)
    return w6, w8


def test_q6g32_bytes_per_weight(lib):
    assert lib.q6g32_repacked_bytes(262144, 1536) == 262144 * 1536 * 13 // 16
    assert lib.q6g32_repacked_bytes(9, 64) == 16 * 2 * 26


@pytest.mark.parametrize("shards,K", [((256,), 1536), ((100, 37), 64), ((5,), 32)])
def test_q6g32_repack_lossless(lib, shards, K):
    g = wl.rng(sum(shards) + K)
    qs, ds = [], []
    for n in shards:
        qs.append(wl.int_codes(g, (n, K), -32, 31))
        ds.append((wl.positive_scales(g, n * (K // 32)).astype(np.float16)).view(np.uint16).reshape(n, K // 32))
    w6, _ = _packs(lib, qs, ds, K)
    q, d = decode_q6g32(host(w6), sum(shards), K)
    assert np.array_equal(q, np.concatenate(qs))
    assert np.array_equal(d, np.concatenate(ds).view(np.float16).astype(np.float64))


@pytest.mark.parametrize("M,N,K", [(1, 4096, 1536), (3, 77, 1536), (8, 600, 3584), (16, 40, 256), (1, 3, 32)])
def test_q6g32_gemv_matches_i8g32_and_oracle(lib, M, N, K):
    import torch
    g = wl.rng(23 * M + N + K)
    W = wl.weights(g, N, K)
    b = wl.bias(g, N)
    x = wl.activations(g, M, K)
    q, d = oracle.quantize_i8g32(W)
    qx, sx = oracle.quantize_act_int8(x)
    y_ref, acc = oracle.gemv_i8g32(q, d, qx, sx, b, want_acc=True)
    w6, w8 = _packs(lib, [q], [d], K)
    y6 = torch.empty((M, N), dtype=torch.float32, device="cuda")
    y8 = torch.empty((M, N), dtype=torch.float32, device="cuda")
    lib.q6g32_gemv(w6, dev(b), dev(qx), dev(sx), y6)
    lib.i8g32_gemv(w8, dev(b), dev(qx), dev(sx), y8)
    check_close(host(y6), y_ref, group_scale(acc, d.view(np.float16).astype(np.float64), sx, b), RTOL_GROUP,
                "q6g32_gemv")
    assert np.array_equal(host(y6).view(np.uint32), host(y8).view(np.uint32))


def test_q6g32_accumulators_bit_exact(lib):
    """Unit scales, no bias, extreme codes: y = sum_g acc_g exactly (|sums| < 2^24)."""
    import torch
    M, N, K = 2, 64, 1536
    g = wl.rng(29)
    q = wl.int_codes(g, (N, K), -32, 31)
    q[0] = -32
    q[1] = 31
    d = np.full((N, K // 32), 0x3C00, np.uint16)
    qx = wl.int_codes(g, (M, K), -127, 127)
    qx[0] = -127
    w6, _ = _packs(lib, [q], [d], K)
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    lib.q6g32_gemv(w6, None, dev(qx), dev(np.ones(M, np.float32)), y)
    acc = oracle.gemv_i8g32(q, d, qx, np.ones(M, np.float32), None, want_acc=True)[1]
    assert np.array_equal(host(y).astype(np.int64), acc.sum(axis=2).astype(np.int64))


@pytest.mark.parametrize("M,N,K", [(1, 262144 // 16, 1536), (4, 300, 1536)])
def test_q6g32_linear_fused(lib, M, N, K):
    import torch
    g = wl.rng(31 * M + N)
    W = wl.weights(g, N, K)
    b = wl.bias(g, N)
    x = wl.activations(g, M, K)
    q, d = oracle.quantize_i8g32(W)
    qx_ref, sx_ref = oracle.quantize_act_int8(x)
    y_ref, acc = oracle.gemv_i8g32(q, d, qx_ref, sx_ref, b, want_acc=True)
    w6, w8 = _packs(lib, [q], [d], K)
    outs = []
    for fn, w in ((lib.q6g32_linear, w6), (lib.i8g32_linear, w8)):
        y = torch.empty((M, N), dtype=torch.float32, device="cuda")
        qx = torch.empty((M, K), dtype=torch.int8, device="cuda")
        sx = torch.empty(M, dtype=torch.float32, device="cuda")
        fn(w, dev(b), dev(x), y, qx, sx)
        assert np.array_equal(host(qx), qx_ref)
        outs.append(host(y))
    check_close(outs[0], y_ref, group_scale(acc, d.view(np.float16).astype(np.float64), sx_ref, b), RTOL_GROUP,
                "q6g32_linear")
    assert np.array_equal(outs[0].view(np.uint32), outs[1].view(np.uint32))


def test_quantlinear_q6g32(lib):
    import torch

    from bit_quantized_decode_gb300 import QuantLinear
    N, K = 512, 1536
    W = torch.randn((N, K), generator=torch.Generator(device="cuda").manual_seed(3), device="cuda") * 0.02
    b = torch.randn(N, generator=torch.Generator(device="cuda").manual_seed(4), device="cuda") * 0.01
    x = torch.randn((1, K), generator=torch.Generator(device="cuda").manual_seed(5), device="cuda")
    q6 = QuantLinear.from_float("q6g32", [W], [b])
    q8 = QuantLinear.from_float("i8g32", [W], [b])
    assert q6.weight_bytes * 16 == N * K * 13
    assert np.array_equal(host(q6(x)).view(np.uint32), host(q8(x)).view(np.uint32))
