"""Oracle parity at the workloads' full shapes, every output row compared.

The smaller parity tests cover each format's arithmetic; these run the
launches the benchmark times, at sizes whose blocks take the branches small
shapes never reach:
  - per-row INT4 lm_head 152064 x 3584 ("Jetson Orin AGX INT4 推理优化实践",
    §模型尺寸, VOCAB 152064) on two blocks per SM at one and two tokens; also
    five tokens (the tensor-core path over 1188 row groups);
  - per-row INT4 fused gate/up 37888 x 3584 at one token;
  - the int8 group lm_head 262144 x 1536 ("在香橙派上跑 Gemma4", §3.2) in its
    int8 (I8G32) and 6-bit (Q6G32) layouts: four rounds per block and 1725
    rows per block, past the rows whose scales and bias are staged in shared
    memory, so the epilogue reads them from global memory;
  - Q4_0 with 160000 rows of K = 1536: 1053 rows per block, also uncached.
Weights are N(0, sigma) draws quantized by the oracle on the host (in row
chunks), x ~ N(0, 1); codes and scales are bit-exact, y within the stated
tolerances of the summed term magnitudes.
"""
import numpy as np
import pytest

import oracle
from bit_quantized_decode_gb300 import workloads as wl
from helpers import RTOL_GROUP, RTOL_W4, check_close, cuda_ok, dev, group_scale, host, q4_0_scales, w4_scale

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not cuda_ok(), reason="needs a CUDA GPU")]

ROWS_PER_DRAW = 8192


@pytest.fixture(scope="module")
def lib():
    import torch  # noqa: F401

    from bit_quantized_decode_gb300 import _lib
    _lib.load()
    _lib.clear_device_error()
    yield _lib
    assert _lib.device_error() == 0


def _draw_rows(g, N, K, sigma, quantize):
    """quantize(W chunk) for N(0, sigma) weights drawn ROWS_PER_DRAW rows at a time."""
    parts = []
    for r0 in range(0, N, ROWS_PER_DRAW):
        n = min(ROWS_PER_DRAW, N - r0)
        W = (g.standard_normal((n, K), dtype=np.float32) * np.float32(sigma)).astype(np.float32)
        parts.append(quantize(W))
    return parts


def _linear_buffers(M, N, K):
    import torch
    return (torch.empty((M, N), dtype=torch.float32, device="cuda"),
            torch.empty((M, K), dtype=torch.int8, device="cuda"),
            torch.empty(M, dtype=torch.float32, device="cuda"))


def _w4_case(lib, seed, N, K):
    import torch
    g = wl.rng(seed)
    parts = _draw_rows(g, N, K, 0.02, oracle.quantize_rows_int4)
    q = np.concatenate([p[0] for p in parts])
    sw = np.concatenate([p[1] for p in parts])
    b = wl.bias(g, N)
    packed = oracle.pack_int4(q)
    w = torch.empty(lib.w4_repacked_bytes(N, K), dtype=torch.uint8, device="cuda")
    lib.w4_repack([dev(packed.view(np.int32))], K, w)
    return g, packed, sw, b, w


@pytest.mark.parametrize("name,N,K,Ms", [("lm_head", 152064, 3584, (1, 2, 5)), ("gate_up", 37888, 3584, (1,))])
def test_w4_full_shape(lib, name, N, K, Ms):
    g, packed, sw, b, w = _w4_case(lib, 4100 + N, N, K)
    swd, bd = dev(sw), dev(b)
    for M in Ms:
        x = wl.activations(g, M, K)
        y_ref, qx_ref, sx_ref, acc = oracle.w4a8_linear(packed, sw, x, b)
        y, qx, sx = _linear_buffers(M, N, K)
        lib.w4a8_linear(w, swd, bd, dev(x), y, qx, sx)
        assert np.array_equal(host(sx).view(np.uint32), sx_ref.view(np.uint32))
        assert np.array_equal(host(qx), qx_ref)
        check_close(host(y), y_ref, w4_scale(acc, sw, sx_ref, b), RTOL_W4, f"{name} {N}x{K} M={M}")


@pytest.fixture(scope="module")
def lm_head_i8g32():
    """The Gemma-E2B lm_head at full size: int8 codes in [-32, 31] and fp16
    group scales of N(0, 0.02) weights, bias N(0, 0.01)."""
    N, K = 262144, 1536
    g = wl.rng(4262)
    parts = _draw_rows(g, N, K, 0.02, oracle.quantize_i8g32)
    q = np.concatenate([p[0] for p in parts])
    d = np.concatenate([p[1] for p in parts])
    b = wl.bias(g, N)
    x = wl.activations(g, 1, K)
    qx_ref, sx_ref = oracle.quantize_act_int8(x)
    y_ref, acc = oracle.gemv_i8g32(q, d, qx_ref, sx_ref, b, want_acc=True)
    scale = group_scale(acc, d.view(np.float16).astype(np.float64), sx_ref, b)
    return N, K, q, d, b, x, qx_ref, sx_ref, y_ref, scale


@pytest.mark.parametrize("layout", ["i8g32", "q6g32"])
def test_group_lm_head_full_shape(lib, lm_head_i8g32, layout):
    import torch
    N, K, q, d, b, x, qx_ref, sx_ref, y_ref, scale = lm_head_i8g32
    nbytes = lib.i8g32_repacked_bytes(N, K) if layout == "i8g32" else lib.q6g32_repacked_bytes(N, K)
    w = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    getattr(lib, f"{layout}_repack")([dev(q)], [dev(d.view(np.int16))], K, w)
    y, qx, sx = _linear_buffers(1, N, K)
    getattr(lib, f"{layout}_linear")(w, dev(b), dev(x), y, qx, sx)
    assert np.array_equal(host(qx), qx_ref)
    assert np.array_equal(host(sx).view(np.uint32), sx_ref.view(np.uint32))
    check_close(host(y), y_ref, scale, RTOL_GROUP, f"{layout} lm_head {N}x{K}")


def test_q4_0_past_the_staged_rows(lib):
    import torch
    N, K = 160000, 1536
    g = wl.rng(4160)
    blocks = np.concatenate(_draw_rows(g, N, K, 0.03, oracle.quantize_q4_0))
    b = wl.bias(g, N)
    x = wl.activations(g, 1, K)
    qx_ref, sx_ref = oracle.quantize_act_int8(x)
    y_ref, acc = oracle.gemv_q4_0(blocks, qx_ref, sx_ref, b, want_acc=True)
    w = torch.empty(lib.q4_0_repacked_bytes(N, K), dtype=torch.uint8, device="cuda")
    lib.q4_0_repack([dev(blocks)], K, w)
    y, qx, sx = _linear_buffers(1, N, K)
    lib.q4_0_linear(w, dev(b), dev(x), y, qx, sx)
    assert np.array_equal(host(qx), qx_ref)
    check_close(host(y), y_ref, group_scale(acc, q4_0_scales(blocks), sx_ref, b), RTOL_GROUP, f"q4_0 {N}x{K}")
