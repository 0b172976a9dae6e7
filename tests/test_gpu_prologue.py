"""The fused activation prologue (quantize inside the GEMV launch).

Codes and scales must be bit-exact against the oracle and y within
tolerance of it, on inputs that stress the quantizer: many possible ties
(the exact fallback), all-zero and tiny-scale tokens, outliers; for every
register bucket of the prologue and its two-pass form, and for the three
weight formats.  The fused launch must also give y bit-identical to the
two-launch path (a8_quantize, then the GEMV on the int8 codes): the per-row
sums run in the same order.
"""
import numpy as np
import pytest

import oracle
from bit_quantized_decode_gb300 import workloads as wl
from helpers import (RTOL_GROUP, RTOL_W4, check_close, cuda_ok, dev, group_scale, host, q4_0_scales,
                     w4_scale)

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not cuda_ok(), reason="needs a CUDA GPU")]


@pytest.fixture(scope="module")
def lib():
    import torch  # noqa: F401

    from bit_quantized_decode_gb300 import _lib
    _lib.load()
    _lib.clear_device_error()
    yield _lib
    assert _lib.device_error() == 0


def _bufs(M, N, K):
    import torch
    return (torch.empty((M, N), dtype=torch.float32, device="cuda"),
            torch.empty((M, K), dtype=torch.int8, device="cuda"),
            torch.empty(M, dtype=torch.float32, device="cuda"))


def _activations(g, M, K, kind):
    x = wl.activations(g, M, K, outliers=True)
    if kind == "ties":
        # token 0: scale exactly 1 and every third entry on a half-integer
        x[0] = (np.arange(K) % 255 - 127).astype(np.float32)
        x[0, 1::3] += np.float32(0.5)
        x[0] = np.clip(x[0], -127.0, 127.0)
        x[0, 0] = np.float32(127.0)
    elif kind == "zero_tiny":
        x[0] = 0.0
        if M > 1:
            x[1] *= np.float32(1e-32)
    return x


# (M, N, K): register buckets 1/5 .. 5/5 of the prologue, the two-pass form
# (16 x 1536, 4 x 18944), fewer tiles than SMs, a single tile
W4_SHAPES = [(1, 512, 3584, "normal"), (1, 3584, 18944, "ties"), (1, 700, 768, "ties"),
             (2, 50, 3584, "zero_tiny"), (4, 100, 18944, "normal"), (16, 24, 1536, "ties"),
             (3, 7, 32, "zero_tiny"), (8, 1000, 6144, "normal"), (1, 64, 12288, "ties")]


@pytest.mark.parametrize("M,N,K,kind", W4_SHAPES)
def test_w4a8_fused_prologue(lib, M, N, K, kind):
    g = wl.rng(31 * M + N + K)
    W = wl.weights(g, N, K)
    x = _activations(g, M, K, kind)
    b = wl.bias(g, N)
    q, sw = oracle.quantize_rows_int4(W)
    y_ref, qx_ref, sx_ref, acc = oracle.w4a8_linear(oracle.pack_int4(q), sw, x, b)
    import torch
    w = torch.empty(lib.w4_repacked_bytes(N, K), dtype=torch.uint8, device="cuda")
    lib.w4_repack([dev(oracle.pack_int4(q).view(np.int32))], K, w)
    swd, bd = dev(sw), dev(b)
    y, qx, sx = _bufs(M, N, K)
    lib.w4a8_linear(w, swd, bd, dev(x), y, qx, sx, lib.W4_FLAG_PDL)
    assert np.array_equal(host(sx).view(np.uint32), sx_ref.view(np.uint32))
    assert np.array_equal(host(qx), qx_ref)
    check_close(host(y), y_ref, w4_scale(acc, sw, sx_ref, b), RTOL_W4, "w4a8_linear")
    y2, _, _ = _bufs(M, N, K)
    lib.w4a8_gemv(w, swd, bd, qx, sx, y2)
    assert np.array_equal(host(y).view(np.uint32), host(y2).view(np.uint32))


@pytest.mark.parametrize("M,N,K,kind", [(1, 2560, 1536, "ties"), (2, 100, 6144, "zero_tiny"),
                                        (1, 9, 32, "normal")])
def test_q4_0_fused_prologue(lib, M, N, K, kind):
    g = wl.rng(37 * M + N + K)
    W = wl.weights(g, N, K, 0.03)
    x = _activations(g, M, K, kind)
    blocks = oracle.quantize_q4_0(W)
    qx_ref, sx_ref = oracle.quantize_act_int8(x)
    y_ref, acc = oracle.gemv_q4_0(blocks, qx_ref, sx_ref, None, want_acc=True)
    import torch
    w = torch.empty(lib.q4_0_repacked_bytes(N, K), dtype=torch.uint8, device="cuda")
    lib.q4_0_repack([dev(blocks)], K, w)
    y, qx, sx = _bufs(M, N, K)
    lib.q4_0_linear(w, None, dev(x), y, qx, sx)
    assert np.array_equal(host(qx), qx_ref)
    check_close(host(y), y_ref, group_scale(acc, q4_0_scales(blocks), sx_ref, None), RTOL_GROUP, "q4_0_linear")
    y2, _, _ = _bufs(M, N, K)
    lib.q4_0_gemv(w, None, qx, sx, y2)
    assert np.array_equal(host(y).view(np.uint32), host(y2).view(np.uint32))


@pytest.mark.parametrize("M,N,K,kind", [(1, 4096, 1536, "ties"), (3, 5, 64, "zero_tiny")])
def test_i8g32_fused_prologue(lib, M, N, K, kind):
    g = wl.rng(41 * M + N + K)
    W = wl.weights(g, N, K)
    x = _activations(g, M, K, kind)
    b = wl.bias(g, N)
    q, d = oracle.quantize_i8g32(W)
    qx_ref, sx_ref = oracle.quantize_act_int8(x)
    y_ref, acc = oracle.gemv_i8g32(q, d, qx_ref, sx_ref, b, want_acc=True)
    import torch
    w = torch.empty(lib.i8g32_repacked_bytes(N, K), dtype=torch.uint8, device="cuda")
    lib.i8g32_repack([dev(q)], [dev(d.view(np.int16))], K, w)
    bd = dev(b)
    y, qx, sx = _bufs(M, N, K)
    lib.i8g32_linear(w, bd, dev(x), y, qx, sx)
    assert np.array_equal(host(qx), qx_ref)
    check_close(host(y), y_ref, group_scale(acc, d.view(np.float16).astype(np.float64), sx_ref, b), RTOL_GROUP,
                "i8g32_linear")
    y2, _, _ = _bufs(M, N, K)
    lib.i8g32_gemv(w, bd, qx, sx, y2)
    assert np.array_equal(host(y).view(np.uint32), host(y2).view(np.uint32))
