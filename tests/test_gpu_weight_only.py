"""The weight-only paths on float activations ([Orin-INT4] §"为什么 INT4 float
解包不快"): per-row INT4 unpacked to float (w4a32_gemv, on the W4 bytes the
DP4A path reads) and per-row INT8 (w8a32_gemv).

The INT8 weight quantizer and the repack are integer work: bit-exact against
the oracle and a CPU decoder of the documented layout.  The GEMVs accumulate
fp32 products in an unspecified order, so y is compared with the oracle's
fp64 result within the bound fp32 summation gives: each lane's running sum is
at most 2C + 64 additions deep (C = K/32 chunks), so
|y - y_ref| <= (2C + 64) 2^-24 s_w sum_i |q_i x_i| + 2^-23 (|y_ref| + |b|).
"""
import numpy as np
import pytest

import oracle
from bit_quantized_decode_gb300 import workloads as wl
from helpers import cuda_ok, decode_i8_units, dev, host

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not cuda_ok(), reason="needs a CUDA GPU")]

U = 2.0 ** -24


@pytest.fixture(scope="module")
def lib():
    import torch  # noqa: F401

    from bit_quantized_decode_gb300 import _lib
    _lib.load()
    _lib.clear_device_error()
    yield _lib
    assert _lib.device_error() == 0


def _bound(q, sw, x, b, y_ref, K):
    C = K // 32
    terms = np.abs(x.astype(np.float64)) @ np.abs(q.astype(np.float64)).T * np.abs(sw.astype(np.float64))[None, :]
    bb = 0.0 if b is None else np.abs(b.astype(np.float64))[None, :]
    return (2 * C + 64) * U * terms + 2 * U * (np.abs(y_ref) + bb)


def _close(y, y_ref, bound, what):
    err = np.abs(np.asarray(y, np.float64) - y_ref)
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"{what}: {bad.sum()} of {err.size} outside; worst at {i}: gpu {y[i]!r} "
                             f"ref {y_ref[i]!r} bound {bound[i]!r}")


def _w8(lib, q_shards, K):
    import torch
    N = sum(q.shape[0] for q in q_shards)
    w = torch.full((lib.w8_repacked_bytes(N, K),), 0xAB, dtype=torch.uint8, device="cuda")
    lib.w8_repack([dev(q) for q in q_shards], K, w)
    return w


def test_w8_quantize_rows_matches_oracle(lib):
    import torch
    g = wl.rng(41)
    N, K = 300, 1536
    W = wl.weights(g, N, K)
    W[7] = 0.0
    q_ref, sw_ref = oracle.quantize_rows_int8(W)
    q = torch.empty((N, K), dtype=torch.int8, device="cuda")
    sw = torch.empty(N, dtype=torch.float32, device="cuda")
    lib.w8_quantize_rows(dev(W), q, sw)
    assert np.array_equal(host(q), q_ref)
    assert np.array_equal(host(sw).view(np.uint32), sw_ref.view(np.uint32))


def test_w8_repack_lossless_with_shards(lib):
    g = wl.rng(42)
    K = 96
    shards = [wl.int_codes(g, (n, K), -127, 127) for n in (5, 8, 3)]
    w = _w8(lib, shards, K)
    N = 16
    assert w.numel() == 16 * K
    dec = decode_i8_units(host(w), N, K)
    assert np.array_equal(dec, np.concatenate(shards))


@pytest.mark.parametrize("M,N,K", [(1, 4608, 3584), (2, 300, 18944), (4, 264, 1536), (3, 77, 96), (1, 9, 32)])
def test_w4a32_matches_oracle(lib, M, N, K):
    """INT4 weights in the W4 layout, unpacked to float, on unquantized x."""
    import torch
    g = wl.rng(43 + M + N + K)
    q, sw = oracle.quantize_rows_int4(wl.weights(g, N, K))
    x = wl.activations(g, M, K, outliers=True)
    b = wl.bias(g, N)
    w = torch.empty(lib.w4_repacked_bytes(N, K), dtype=torch.uint8, device="cuda")
    lib.w4_repack([dev(oracle.pack_int4(q).view(np.int32))], K, w)
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    lib.w4a32_gemv(w, dev(sw), dev(b), dev(x), y, lib.W4_FLAG_PDL)
    y_ref = oracle.gemv_weight_only(q, sw, x, b)
    _close(host(y), y_ref, _bound(q, sw, x, b, y_ref, K), "w4a32")


def test_w4a32_extreme_codes(lib):
    """Every nibble value, -8 and 7 included, with unit scales and x = 1: y is
    the exact row sum of the codes."""
    import torch
    N, K = 16, 256
    q = np.tile(np.arange(-8, 8, dtype=np.int8), (N, K // 16))
    q[1::2] = -8
    q[2] = 7
    w = torch.empty(lib.w4_repacked_bytes(N, K), dtype=torch.uint8, device="cuda")
    lib.w4_repack([dev(oracle.pack_int4(q).view(np.int32))], K, w)
    y = torch.empty((1, N), dtype=torch.float32, device="cuda")
    lib.w4a32_gemv(w, dev(np.ones(N, np.float32)), None, dev(np.ones((1, K), np.float32)), y)
    assert np.array_equal(host(y)[0], q.astype(np.float64).sum(axis=1).astype(np.float32))


@pytest.mark.parametrize("M,N,K", [(1, 4608, 3584), (2, 300, 18944), (4, 264, 1536), (3, 77, 96)])
def test_w8a32_matches_oracle(lib, M, N, K):
    import torch
    g = wl.rng(44 + M + N + K)
    q, sw = oracle.quantize_rows_int8(wl.weights(g, N, K))
    x = wl.activations(g, M, K, outliers=True)
    b = wl.bias(g, N)
    w = _w8(lib, [q], K)
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    lib.w8a32_gemv(w, dev(sw), dev(b), dev(x), y)
    y_ref = oracle.gemv_weight_only(q, sw, x, b)
    _close(host(y), y_ref, _bound(q, sw, x, b, y_ref, K), "w8a32")


def test_w8a32_extreme_codes(lib):
    """Codes -127 and 127 (and every value between) with unit scales and x = 1."""
    import torch
    N, K = 8, 256
    q = ((np.arange(N * K) % 255) - 127).reshape(N, K).astype(np.int8)
    q[0] = -127
    q[1] = 127
    w = _w8(lib, [q], K)
    y = torch.empty((1, N), dtype=torch.float32, device="cuda")
    lib.w8a32_gemv(w, dev(np.ones(N, np.float32)), None, dev(np.ones((1, K), np.float32)), y)
    assert np.array_equal(host(y)[0], q.astype(np.float64).sum(axis=1).astype(np.float32))


def test_weight_only_argument_errors(lib):
    import torch
    K = 64
    w = torch.zeros(lib.w4_repacked_bytes(8, K), dtype=torch.uint8, device="cuda")
    sw = torch.ones(8, dtype=torch.float32, device="cuda")
    x = torch.zeros((5, K), dtype=torch.float32, device="cuda")
    y = torch.empty((5, 8), dtype=torch.float32, device="cuda")
    with pytest.raises(lib.W4Error) as e:
        lib.w4a32_gemv(w, sw, None, x, y)
    assert e.value.status == 2          # more than four tokens
    with pytest.raises(lib.W4Error) as e:
        lib.w8a32_gemv(w, None, None, x[:1], y[:1])
    assert e.value.status == 1
