"""The multi-token per-row INT4 GEMV on the tensor cores (by default M = 3..16;
the tests force it for any M, one token included).

The accumulators must be the exact integer sums (read out through unit
scales), y must agree with the oracle within the per-row INT4 tolerance and
be bit-identical to the DP4A path on the same codes (both finish with
fmaf(s_w s_x, (float)acc, b)).  Shapes cover one and several K splits (the
cluster reduction), a partial last 128-row group, K not a multiple of the
256-wide K block (and shorter than one), the split forced by K > 16384, and the largest magnitudes
a split may reach.
"""
import numpy as np
import pytest

import oracle
from bit_quantized_decode_gb300 import workloads as wl
from helpers import RTOL_W4, check_close, cuda_ok, dev, host, w4_scale

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not cuda_ok(), reason="needs a CUDA GPU")]


@pytest.fixture(scope="module")
def lib():
    import torch  # noqa: F401

    from bit_quantized_decode_gb300 import _lib
    _lib.load()
    _lib.clear_device_error()
    yield _lib
    _lib.set_tuning("tc_min_m", 0)
    assert _lib.device_error() == 0


def _prep(lib, q, K):
    import torch
    N = q.shape[0]
    w = torch.empty(lib.w4_repacked_bytes(N, K), dtype=torch.uint8, device="cuda")
    lib.w4_repack([dev(oracle.pack_int4(q).view(np.int32))], K, w)
    return w


def _gemv(lib, w, sw, b, qx, sx, M, N, tc=True):
    import torch
    lib.set_tuning("tc_min_m", 1 if tc else 17)
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    lib.w4a8_gemv(w, sw, b, qx, sx, y)
    lib.set_tuning("tc_min_m", 0)
    return host(y)


@pytest.mark.parametrize("M,N,K", [(8, 256, 256), (16, 300, 3584), (12, 4608, 3584), (9, 3584, 18944),
                                   (16, 128, 96), (10, 1000, 6144), (16, 136, 32), (5, 384, 640),
                                   (6, 200, 224), (7, 1000, 3584), (1, 264, 1088)])
def test_tc_accumulators_bit_exact(lib, M, N, K):
    """Unit scales, no bias: y is (float)acc, exact while |acc| < 2^24."""
    g = wl.rng(3 * M + N + K)
    q = wl.int_codes(g, (N, K), -8, 7)
    qx = wl.int_codes(g, (M, K), -127, 127)
    acc = oracle.gemv_w4a8_acc(oracle.pack_int4(q), qx)
    assert np.abs(acc).max() < 2 ** 24
    w = _prep(lib, q, K)
    ones_n = dev(np.ones(N, np.float32))
    ones_m = dev(np.ones(M, np.float32))
    y = _gemv(lib, w, ones_n, None, dev(qx), ones_m, M, N)
    assert np.array_equal(y.astype(np.int64), acc.astype(np.int64))


def test_tc_extreme_magnitudes(lib):
    """Every product at +-1016 over K = 32768 (two splits of 16384): the
    tensor cores sum the biased nibbles n = q + 8 against the codes' high and
    low halves, whose partial sums reach 15 * 8 * 16384 and 15 * 15 * 16384,
    below 2^24; the total 33,292,288 is rounded only by the final conversion,
    exactly as in the oracle."""
    M, N, K = 16, 256, 32768
    q = np.full((N, K), -8, np.int8)
    q[1::2] = 7
    qx = np.full((M, K), -127, np.int8)
    qx[1::2] = 127
    acc = oracle.gemv_w4a8_acc(oracle.pack_int4(q), qx)
    w = _prep(lib, q, K)
    y = _gemv(lib, w, dev(np.ones(N, np.float32)), None, dev(qx), dev(np.ones(M, np.float32)), M, N)
    assert np.array_equal(y.view(np.uint32), acc.astype(np.float32).view(np.uint32))


@pytest.mark.parametrize("M,N,K", [(8, 512, 3584), (16, 4608, 3584), (13, 3584, 18944), (16, 1000, 1536),
                                   (5, 3584, 18944), (6, 4608, 3584), (7, 640, 1536), (2, 300, 3584)])
def test_tc_matches_oracle_and_dp4a(lib, M, N, K):
    g = wl.rng(5 * M + N + K)
    W = wl.weights(g, N, K)
    x = wl.activations(g, M, K, outliers=True)
    b = wl.bias(g, N)
    q, sw = oracle.quantize_rows_int4(W)
    y_ref, qx, sx, acc = oracle.w4a8_linear(oracle.pack_int4(q), sw, x, b)
    w = _prep(lib, q, K)
    args = (w, dev(sw), dev(b), dev(qx), dev(sx), M, N)
    y_tc = _gemv(lib, *args, tc=True)
    check_close(y_tc, y_ref, w4_scale(acc, sw, sx, b), RTOL_W4, "tensor-core w4a8_gemv")
    y_dp = _gemv(lib, *args, tc=False)
    assert np.array_equal(y_tc.view(np.uint32), y_dp.view(np.uint32))


@pytest.mark.parametrize("M,N,K", [(8, 4608, 3584), (16, 3584, 18944), (11, 37888 // 4, 3584),
                                   (5, 3584, 18944), (7, 4608, 3584)])
def test_tc_linear_fused_api(lib, M, N, K):
    """w4a8_linear with many tokens: the activation quantizer, then the
    tensor-core GEMV (chained); codes and scales bit-exact."""
    import torch
    g = wl.rng(7 * M + N + K)
    W = wl.weights(g, N, K)
    x = wl.activations(g, M, K)
    b = wl.bias(g, N)
    q, sw = oracle.quantize_rows_int4(W)
    y_ref, qx_ref, sx_ref, acc = oracle.w4a8_linear(oracle.pack_int4(q), sw, x, b)
    w = _prep(lib, q, K)
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    qx = torch.empty((M, K), dtype=torch.int8, device="cuda")
    sx = torch.empty(M, dtype=torch.float32, device="cuda")
    lib.w4a8_linear(w, dev(sw), dev(b), dev(x), y, qx, sx, lib.W4_FLAG_PDL)
    assert np.array_equal(host(sx).view(np.uint32), sx_ref.view(np.uint32))
    assert np.array_equal(host(qx), qx_ref)
    check_close(host(y), y_ref, w4_scale(acc, sw, sx_ref, b), RTOL_W4, "w4a8_linear (tensor cores)")


def test_tc_large_k_split_sampled_rows(lib):
    """152 row groups (one block each by count) with K = 18944 > 16384: the
    split is forced by K.  Oracle on a sample of rows."""
    M, N, K = 8, 152 * 128, 18944
    g = wl.rng(99)
    q = g.integers(-8, 8, size=(N, K), dtype=np.int8)
    qx = wl.int_codes(g, (M, K), -127, 127)
    w = _prep(lib, q, K)
    y = _gemv(lib, w, dev(np.ones(N, np.float32)), None, dev(qx), dev(np.ones(M, np.float32)), M, N)
    rows = np.sort(g.choice(N, 64, replace=False))
    acc = oracle.gemv_w4a8_acc(oracle.pack_int4(q[rows]), qx)
    assert np.array_equal(y[:, rows].astype(np.int64), acc.astype(np.int64))


def test_tc_largest_k_eight_splits(lib):
    """K = 131072, the largest K the library takes: eight K splits of 16384
    (a cluster of eight), whose partial sums fill the weight ring exactly;
    the accumulators stay bit-exact (unit scales)."""
    M, N, K = 8, 128, 131072
    g = wl.rng(2024)
    q = wl.int_codes(g, (N, K), -8, 7)
    qx = wl.int_codes(g, (M, K), -127, 127)
    acc = oracle.gemv_w4a8_acc(oracle.pack_int4(q), qx)
    w = _prep(lib, q, K)
    y = _gemv(lib, w, dev(np.ones(N, np.float32)), None, dev(qx), dev(np.ones(M, np.float32)), M, N)
    assert np.array_equal(y.view(np.uint32), acc.astype(np.float32).view(np.uint32))
