"""Parity of the CUDA path (through the C ABI) against the CPU oracle.

Bit-exact: activation codes and scales, weight codes and scales, repacked
layouts (decoded on the CPU), and the int32 accumulators (read out through
GEMVs with unit scales).  fp32 outputs: within 1e-5 (per-row INT4) or 1e-4
(group formats) of the summed term magnitudes, the tolerances the method
states for this path.
"""
import numpy as np
import pytest

import oracle
from bit_quantized_decode_gb300 import workloads as wl
from helpers import (RTOL_GROUP, RTOL_W4, check_close, cuda_ok, decode_group_plane, decode_i8_units,
                     decode_w4_units, dev, group_scale, host, q4_0_scales, w4_scale)

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not cuda_ok(), reason="needs a CUDA GPU")]


@pytest.fixture(scope="module")
def lib():
    import torch  # noqa: F401

    from bit_quantized_decode_gb300 import _lib
    _lib.load()
    _lib.clear_device_error()
    yield _lib
    assert _lib.device_error() == 0


def _torch():
    import torch
    return torch


# ------------------------------------------------------ activation quant
@pytest.mark.parametrize("M,K,outliers", [(1, 3584, True), (3, 1536, False), (16, 18944, False), (2, 32, False),
                                           (1, 8192, True), (8, 8192, True), (5, 32768, False), (4, 32800, True),
                                           (6, 32800, False), (2, 40960, False)])
def test_a8_quantize_bit_exact(lib, M, K, outliers):
    """Codes and scales bit-exact; five or more tokens with 8192 <= K <= 32768
    take the kernel with four blocks per token (a cluster sharing the token's
    absmax), the rest one block per token."""
    torch = _torch()
    g = wl.rng(100 + M + K)
    x = wl.activations(g, M, K, outliers)
    qx_ref, sx_ref = oracle.quantize_act_int8(x)
    qx = torch.empty((M, K), dtype=torch.int8, device="cuda")
    sx = torch.empty(M, dtype=torch.float32, device="cuda")
    lib.a8_quantize(dev(x), qx, sx)
    assert np.array_equal(host(sx).view(np.uint32), sx_ref.view(np.uint32))
    assert np.array_equal(host(qx), qx_ref)


def test_a8_quantize_ties_zero_and_tiny(lib):
    torch = _torch()
    K = 64
    x = np.zeros((4, K), np.float32)
    x[0, :8] = [127.0, 0.5, 1.5, 2.5, -0.5, -1.5, -127.0, 63.5]     # exact ties, s = 1
    # row 1 stays all zero: s = 0, codes 0
    x[2] = np.float32(1e-30) * np.arange(-32, 32, dtype=np.float32)  # tiny magnitudes
    x[3] = -np.float32(3.0e38) * (np.arange(K) % 3 == 0)            # near the top of fp32
    qx_ref, sx_ref = oracle.quantize_act_int8(x)
    qx = torch.empty((4, K), dtype=torch.int8, device="cuda")
    sx = torch.empty(4, dtype=torch.float32, device="cuda")
    lib.a8_quantize(dev(x), qx, sx)
    assert np.array_equal(host(sx).view(np.uint32), sx_ref.view(np.uint32))
    assert np.array_equal(host(qx), qx_ref)
    assert host(qx)[0, :8].tolist() == [127, 0, 2, 2, 0, -2, -127, 64]


# ------------------------------------------------------- weight quant
@pytest.mark.parametrize("N,K", [(512, 3584), (13, 96), (8, 18944)])
def test_w4_quantize_rows_bit_exact(lib, N, K):
    torch = _torch()
    W = wl.weights(wl.rng(N + K), N, K)
    W[min(3, N - 1)] = 0.0
    q_ref, sw_ref = oracle.quantize_rows_int4(W)
    packed = torch.empty((N, K // 8), dtype=torch.int32, device="cuda")
    sw = torch.empty(N, dtype=torch.float32, device="cuda")
    lib.w4_quantize_rows(dev(W), packed, sw)
    assert np.array_equal(host(sw).view(np.uint32), sw_ref.view(np.uint32))
    assert np.array_equal(host(packed).view(np.uint32), oracle.pack_int4(q_ref))


@pytest.mark.parametrize("N,K", [(2560, 1536), (7, 64)])
def test_q4_0_quantize_bit_exact(lib, N, K):
    torch = _torch()
    W = wl.weights(wl.rng(7 * N + K), N, K, 0.03)
    W[0, :32] = 0.0                               # a zero block: d = 0, all nibbles 8
    blocks = torch.empty((N, K // 32, 18), dtype=torch.uint8, device="cuda")
    lib.q4_0_quantize(dev(W), blocks)
    assert np.array_equal(host(blocks), oracle.quantize_q4_0(W))


@pytest.mark.parametrize("N,K", [(1024, 1536), (5, 32)])
def test_i8g32_quantize_bit_exact(lib, N, K):
    torch = _torch()
    W = wl.weights(wl.rng(3 * N + K), N, K)
    q_ref, d_ref = oracle.quantize_i8g32(W)
    q = torch.empty((N, K), dtype=torch.int8, device="cuda")
    d = torch.empty((N, K // 32), dtype=torch.int16, device="cuda")
    lib.i8g32_quantize(dev(W), q, d)
    assert np.array_equal(host(q), q_ref)
    assert np.array_equal(host(d).view(np.uint16), d_ref)


# ------------------------------------------------------------- repack
def _w4_canonical(g, rows, K):
    q = wl.int_codes(g, (rows, K), -8, 7)
    return q, oracle.pack_int4(q)


@pytest.mark.parametrize("shards,K", [((3584, 512, 512), 3584), ((5, 11, 3), 64), ((1,), 32)])
def test_w4_repack_lossless_with_shards(lib, shards, K):
    torch = _torch()
    g = wl.rng(sum(shards) + K)
    qs, ps = zip(*[_w4_canonical(g, n, K) for n in shards])
    N = sum(shards)
    out = torch.full((lib.w4_repacked_bytes(N, K),), 0xAB, dtype=torch.uint8, device="cuda")
    lib.w4_repack([dev(p.view(np.int32)) for p in ps], K, out)
    raw = host(out)
    assert np.array_equal(decode_w4_units(raw, N, K), np.concatenate(qs))
    # padded rows of the last tile are zero
    T = (N + 7) // 8
    if T * 8 > N:
        units = raw.reshape(T, K // 32, 8, 16)
        assert np.all(units[-1, :, N - (T - 1) * 8:, :] == 0)


def test_q4_0_repack_lossless_with_shards(lib):
    torch = _torch()
    K = 1536
    shards = (2048, 256, 256)
    g = wl.rng(5)
    blocks = [oracle.quantize_q4_0(wl.weights(g, n, K, 0.03)) for n in shards]
    N = sum(shards)
    out = torch.empty(lib.q4_0_repacked_bytes(N, K), dtype=torch.uint8, device="cuda")
    lib.q4_0_repack([dev(b) for b in blocks], K, out)
    raw = host(out)
    allb = np.concatenate(blocks)
    ref = oracle.dequantize_q4_0(allb, K) / np.repeat(np.where(q4_0_scales(allb) == 0, 1, q4_0_scales(allb)), 32, 1)
    assert np.array_equal(decode_w4_units(raw, N, K, biased=False).astype(np.float64), ref)
    assert np.array_equal(decode_group_plane(raw, N, K, 16), q4_0_scales(allb))


def test_i8g32_repack_lossless(lib):
    torch = _torch()
    K = 1536
    shards = (100, 37)
    g = wl.rng(6)
    qd = [oracle.quantize_i8g32(wl.weights(g, n, K)) for n in shards]
    N = sum(shards)
    out = torch.empty(lib.i8g32_repacked_bytes(N, K), dtype=torch.uint8, device="cuda")
    lib.i8g32_repack([dev(q) for q, _ in qd], [dev(d.view(np.int16)) for _, d in qd], K, out)
    raw = host(out)
    assert np.array_equal(decode_i8_units(raw, N, K), np.concatenate([q for q, _ in qd]))
    assert np.array_equal(decode_group_plane(raw, N, K, 32),
                          np.concatenate([d for _, d in qd]).view(np.float16).astype(np.float64))


# ----------------------------------------------------------- W4 GEMV
def _prep_w4(lib, q_shards, sw, bias, K):
    torch = _torch()
    N = sum(q.shape[0] for q in q_shards)
    w = torch.empty(lib.w4_repacked_bytes(N, K), dtype=torch.uint8, device="cuda")
    lib.w4_repack([dev(oracle.pack_int4(q).view(np.int32)) for q in q_shards], K, w)
    return w, dev(sw), (None if bias is None else dev(bias))


@pytest.mark.parametrize("M,N,K", [(1, 512, 3584), (1, 8, 32), (1, 13, 96), (2, 300, 1536), (3, 77, 3584),
                                   (4, 600, 18944), (8, 64, 6144), (16, 40, 3584), (16, 9, 18944), (5, 1000, 256)])
def test_w4a8_accumulators_bit_exact(lib, M, N, K):
    """Unit scales, no bias: y is (float)acc, exact while |acc| < 2^24."""
    torch = _torch()
    g = wl.rng(M * 1000 + N + K)
    q = wl.int_codes(g, (N, K), -8, 7)
    qx = wl.int_codes(g, (M, K), -127, 127)
    acc = oracle.gemv_w4a8_acc(oracle.pack_int4(q), qx)
    assert np.abs(acc).max() < 2**24
    w, sw, _ = _prep_w4(lib, [q], np.ones(N, np.float32), None, K)
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    lib.w4a8_gemv(w, sw, None, dev(qx), dev(np.ones(M, np.float32)), y)
    assert np.array_equal(host(y), acc.astype(np.float32))


def test_w4a8_worst_case_rows(lib):
    """The page's worst case: all -8 weights against all -127 / +127 codes."""
    torch = _torch()
    for K, bound in ((3584, 3_641_344), (18944, 19_247_104)):
        q = np.full((8, K), -8, np.int8)
        qx = np.stack([np.full(K, -127, np.int8), np.full(K, 127, np.int8)])
        w, sw, _ = _prep_w4(lib, [q], np.ones(8, np.float32), None, K)
        y = torch.empty((2, 8), dtype=torch.float32, device="cuda")
        lib.w4a8_gemv(w, sw, None, dev(qx), dev(np.ones(2, np.float32)), y)
        assert np.all(host(y)[0] == bound) and np.all(host(y)[1] == -bound)


@pytest.mark.parametrize("M,N,K", [(1, 512, 3584), (2, 4608, 3584), (3, 129, 18944), (16, 256, 1536)])
def test_w4a8_gemv_outputs(lib, M, N, K):
    torch = _torch()
    g = wl.rng(M + 2 * N + 3 * K)
    W = wl.weights(g, N, K)
    x = wl.activations(g, M, K, outliers=True)
    b = wl.bias(g, N)
    q, sw = oracle.quantize_rows_int4(W)
    y_ref, qx, sx, acc = oracle.w4a8_linear(oracle.pack_int4(q), sw, x, b)
    w, swd, bd = _prep_w4(lib, [q], sw, b, K)
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    lib.w4a8_gemv(w, swd, bd, dev(qx), dev(sx), y)
    check_close(host(y), y_ref, w4_scale(acc, sw, sx, b), RTOL_W4, "w4a8_gemv")


@pytest.mark.parametrize("M,N,K", [(1, 512, 3584), (1, 3584, 18944), (2, 50, 3584), (4, 1000, 18944),
                                   (8, 333, 6144), (16, 64, 3584), (16, 24, 18944), (3, 7, 32)])
def test_w4a8_linear_fused(lib, M, N, K):
    """Quantize + GEMV in one call: codes bit-exact, y within tolerance.
    (16 x 18944 does not fit in shared memory and takes the two-kernel path.)"""
    torch = _torch()
    g = wl.rng(11 * M + N + K)
    W = wl.weights(g, N, K)
    x = wl.activations(g, M, K, outliers=(M == 1))
    b = wl.bias(g, N)
    q, sw = oracle.quantize_rows_int4(W)
    y_ref, qx_ref, sx_ref, acc = oracle.w4a8_linear(oracle.pack_int4(q), sw, x, b)
    w, swd, bd = _prep_w4(lib, [q], sw, b, K)
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    qx = torch.empty((M, K), dtype=torch.int8, device="cuda")
    sx = torch.empty(M, dtype=torch.float32, device="cuda")
    lib.w4a8_linear(w, swd, bd, dev(x), y, qx, sx)
    assert np.array_equal(host(sx).view(np.uint32), sx_ref.view(np.uint32))
    assert np.array_equal(host(qx), qx_ref)
    check_close(host(y), y_ref, w4_scale(acc, sw, sx_ref, b), RTOL_W4, "w4a8_linear")


@pytest.mark.parametrize("M,N,K", [(3, 77, 3584), (4, 600, 18944), (3, 129, 18944), (4, 1000, 3584)])
def test_w4a8_dp4a_three_and_four_tokens(lib, M, N, K):
    """Three and four tokens run on the tensor cores by default; the DP4A
    kernels for them (fused prologue, codes in shared or global memory) stay
    reachable through W4_TUNE_TC_MIN_M and are checked here the same way."""
    torch = _torch()
    g = wl.rng(13 * M + N + K)
    W = wl.weights(g, N, K)
    x = wl.activations(g, M, K)
    b = wl.bias(g, N)
    q, sw = oracle.quantize_rows_int4(W)
    y_ref, qx_ref, sx_ref, acc = oracle.w4a8_linear(oracle.pack_int4(q), sw, x, b)
    w, swd, bd = _prep_w4(lib, [q], sw, b, K)
    lib.set_tuning("tc_min_m", 17)
    try:
        y = torch.empty((M, N), dtype=torch.float32, device="cuda")
        qx = torch.empty((M, K), dtype=torch.int8, device="cuda")
        sx = torch.empty(M, dtype=torch.float32, device="cuda")
        lib.w4a8_linear(w, swd, bd, dev(x), y, qx, sx)
        y2 = torch.empty((M, N), dtype=torch.float32, device="cuda")
        lib.w4a8_gemv(w, swd, bd, qx, sx, y2)
    finally:
        lib.set_tuning("tc_min_m", 0)
    assert np.array_equal(host(qx), qx_ref)
    check_close(host(y), y_ref, w4_scale(acc, sw, sx_ref, b), RTOL_W4, "dp4a linear")
    check_close(host(y2), y_ref, w4_scale(acc, sw, sx_ref, b), RTOL_W4, "dp4a gemv")


def test_w4a8_linear_deterministic_and_pdl(lib):
    torch = _torch()
    M, N, K = 1, 37888, 3584
    g = wl.rng(77)
    q = wl.int_codes(g, (N, K), -8, 7)
    sw = wl.positive_scales(g, N)
    b = wl.bias(g, N)
    x = dev(wl.activations(g, M, K))
    w, swd, bd = _prep_w4(lib, [q], sw, b, K)
    outs = []
    for flags in (0, 0, lib.W4_FLAG_PDL):
        y = torch.empty((M, N), dtype=torch.float32, device="cuda")
        qx = torch.empty((M, K), dtype=torch.int8, device="cuda")
        sx = torch.empty(M, dtype=torch.float32, device="cuda")
        lib.w4a8_linear(w, swd, bd, x, y, qx, sx, flags)
        outs.append(host(y))
    assert np.array_equal(outs[0].view(np.uint32), outs[1].view(np.uint32))
    assert np.array_equal(outs[0].view(np.uint32), outs[2].view(np.uint32))


# ---------------------------------------------------------- Q4_0 GEMV
def _prep_q4_0(lib, blocks_shards, K):
    torch = _torch()
    N = sum(b.shape[0] for b in blocks_shards)
    w = torch.empty(lib.q4_0_repacked_bytes(N, K), dtype=torch.uint8, device="cuda")
    lib.q4_0_repack([dev(b) for b in blocks_shards], K, w)
    return w


@pytest.mark.parametrize("M,N,K", [(1, 2560, 1536), (2, 100, 6144), (16, 40, 1536), (1, 9, 32)])
def test_q4_0_group_accumulators_bit_exact(lib, M, N, K):
    """Blocks with d = 1 and unit s_x: y = sum_g acc_g exactly."""
    torch = _torch()
    g = wl.rng(5 * M + N + K)
    nib = wl.int_codes(g, (N, K // 32, 32), 0, 15).astype(np.uint8)
    blocks = np.zeros((N, K // 32, 18), np.uint8)
    blocks[:, :, 0], blocks[:, :, 1] = 0x00, 0x3C
    blocks[:, :, 2:] = nib[:, :, :16] | (nib[:, :, 16:] << 4)
    qx = wl.int_codes(g, (M, K), -127, 127)
    ones = np.ones(M, np.float32)
    y_ref, acc = oracle.gemv_q4_0(blocks, qx, ones, None, want_acc=True)
    w = _prep_q4_0(lib, [blocks], K)
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    lib.q4_0_gemv(w, None, dev(qx), dev(ones), y)
    assert np.array_equal(host(y).astype(np.int64), acc.sum(axis=2).astype(np.int64))


@pytest.mark.parametrize("M,N,K", [(1, 2560, 1536), (1, 12288, 1536), (1, 1536, 6144), (4, 333, 1536),
                                   (16, 64, 6144), (3, 5, 64)])
def test_q4_0_linear(lib, M, N, K):
    torch = _torch()
    g = wl.rng(13 * M + N + K)
    W = wl.weights(g, N, K, 0.03)
    x = wl.activations(g, M, K)
    b = wl.bias(g, N) if N % 2 else None           # bias present on odd N only: both paths covered
    blocks = oracle.quantize_q4_0(W)
    qx_ref, sx_ref = oracle.quantize_act_int8(x)
    y_ref, acc = oracle.gemv_q4_0(blocks, qx_ref, sx_ref, b, want_acc=True)
    w = _prep_q4_0(lib, [blocks], K)
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    qx = torch.empty((M, K), dtype=torch.int8, device="cuda")
    sx = torch.empty(M, dtype=torch.float32, device="cuda")
    lib.q4_0_linear(w, None if b is None else dev(b), dev(x), y, qx, sx)
    assert np.array_equal(host(qx), qx_ref)
    check_close(host(y), y_ref, group_scale(acc, q4_0_scales(blocks), sx_ref, b), RTOL_GROUP, "q4_0_linear")
    # the int8-input entry point gives the same result within tolerance
    y2 = torch.empty((M, N), dtype=torch.float32, device="cuda")
    lib.q4_0_gemv(w, None if b is None else dev(b), qx, sx, y2)
    check_close(host(y2), y_ref, group_scale(acc, q4_0_scales(blocks), sx_ref, b), RTOL_GROUP, "q4_0_gemv")


# --------------------------------------------------------- i8g32 GEMV
@pytest.mark.parametrize("M,N,K", [(1, 4096, 1536), (2, 77, 1536), (16, 32, 1536), (1, 3, 32)])
def test_i8g32_linear(lib, M, N, K):
    torch = _torch()
    g = wl.rng(17 * M + N + K)
    W = wl.weights(g, N, K)
    x = wl.activations(g, M, K)
    b = wl.bias(g, N)
    q, d = oracle.quantize_i8g32(W)
    qx_ref, sx_ref = oracle.quantize_act_int8(x)
    y_ref, acc = oracle.gemv_i8g32(q, d, qx_ref, sx_ref, b, want_acc=True)
    w = torch.empty(lib.i8g32_repacked_bytes(N, K), dtype=torch.uint8, device="cuda")
    lib.i8g32_repack([dev(q)], [dev(d.view(np.int16))], K, w)
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    qx = torch.empty((M, K), dtype=torch.int8, device="cuda")
    sx = torch.empty(M, dtype=torch.float32, device="cuda")
    lib.i8g32_linear(w, dev(b), dev(x), y, qx, sx)
    assert np.array_equal(host(qx), qx_ref)
    check_close(host(y), y_ref, group_scale(acc, d.view(np.float16).astype(np.float64), sx_ref, b), RTOL_GROUP,
                "i8g32_linear")


# ------------------------------------------ group formats past eight tokens
def _group_weights(lib, fmt, W, K):
    """fmt weights from the oracle's quantizer, repacked on the device, with the
    oracle GEMV on them and their group scales."""
    torch = _torch()
    N = W.shape[0]
    if fmt == "q4_0":
        blocks = oracle.quantize_q4_0(W)
        return (_prep_q4_0(lib, [blocks], K),
                lambda qx, sx, b: oracle.gemv_q4_0(blocks, qx, sx, b, want_acc=True), q4_0_scales(blocks))
    q, d = oracle.quantize_i8g32(W)
    size, repack = ((lib.q6g32_repacked_bytes, lib.q6g32_repack) if fmt == "q6g32"
                    else (lib.i8g32_repacked_bytes, lib.i8g32_repack))
    w = torch.empty(size(N, K), dtype=torch.uint8, device="cuda")
    repack([dev(q)], [dev(d.view(np.int16))], K, w)
    return (w, lambda qx, sx, b: oracle.gemv_i8g32(q, d, qx, sx, b, want_acc=True),
            d.view(np.float16).astype(np.float64))


@pytest.mark.parametrize("fmt", ["q4_0", "i8g32", "q6g32"])
@pytest.mark.parametrize("M,N,K,t", [(16, 1000, 1536, 0), (13, 77, 6144, 0), (10, 9728, 1536, 0), (12, 300, 1536, 0),
                                     (9, 300, 1536, 8), (16, 5, 64, 4)])
def test_group_formats_past_eight_tokens(lib, fmt, M, N, K, t):
    """More than eight tokens run as two launches of the eight-token kernel
    over the same weights (tokens 0-7, then the rest), and as launches of at
    most t tokens under W4_TUNE_GROUP_LAUNCH_TOKENS = t: every token's
    codes and scale bit-exact, y within the group tolerance through both entry
    points, and each token's y bit-identical to the same token in a call of
    one launch of the same kernel on the same path (every launch of a call runs
    the first launch's kernel; the group sums' fp32 order depends on it)."""
    torch = _torch()
    g = wl.rng(41 * M + N + K + t)
    W = wl.weights(g, N, K, 0.03)
    x = wl.activations(g, M, K, outliers=True)
    b = wl.bias(g, N)
    w, ref, scales = _group_weights(lib, fmt, W, K)
    qx_ref, sx_ref = oracle.quantize_act_int8(x)
    y_ref, acc = ref(qx_ref, sx_ref, b)
    tol = group_scale(acc, scales, sx_ref, b)
    linear, gemv = getattr(lib, f"{fmt}_linear"), getattr(lib, f"{fmt}_gemv")
    device = lib.w4_describe_device()

    def bufs(m):
        return (torch.empty((m, N), dtype=torch.float32, device="cuda"),
                torch.empty((m, K), dtype=torch.int8, device="cuda"),
                torch.empty(m, dtype=torch.float32, device="cuda"))

    lib.set_tuning("group_launch_tokens", t)
    try:
        p = lib.w4_plan(fmt, M, N, K, device)
        c = t if t else 8
        assert p["gemv_launches"] == (M + c - 1) // c
        y, qx, sx = bufs(M)
        linear(w, dev(b), dev(x), y, qx, sx)
        assert np.array_equal(host(qx), qx_ref) and np.array_equal(host(sx), sx_ref)
        check_close(host(y), y_ref, tol, RTOL_GROUP, f"{fmt}_linear M={M}")
        yg = torch.empty((M, N), dtype=torch.float32, device="cuda")
        gemv(w, dev(b), qx, sx, yg)
        check_close(host(yg), y_ref, tol, RTOL_GROUP, f"{fmt}_gemv M={M}")
        def bucket(m):
            return 1 if m <= 1 else 2 if m <= 2 else 4 if m <= 4 else 8 if m <= 8 else 16

        for lo in range(0, M, c):
            hi = min(M, lo + c)
            q = lib.w4_plan(fmt, hi - lo, N, K, device)
            assert q["gemv_launches"] == 1
            ys, qxs, sxs = bufs(hi - lo)
            linear(w, dev(b), dev(x[lo:hi]), ys, qxs, sxs)
            assert np.array_equal(host(qxs), qx_ref[lo:hi])
            same_kernel = bucket(hi - lo) == bucket(c)
            if same_kernel and q["path"] == p["path"]:
                assert np.array_equal(host(ys).view(np.uint32), host(y)[lo:hi].view(np.uint32)), (lo, hi)
            yc = torch.empty((hi - lo, N), dtype=torch.float32, device="cuda")
            gemv(w, dev(b), qx[lo:hi], sx[lo:hi], yc)
            if same_kernel:
                assert np.array_equal(host(yc).view(np.uint32), host(yg)[lo:hi].view(np.uint32)), (lo, hi)
    finally:
        lib.set_tuning("group_launch_tokens", 0)


def test_i8g32_accumulators_bit_exact(lib):
    torch = _torch()
    M, N, K = 2, 50, 1536
    g = wl.rng(19)
    q = wl.int_codes(g, (N, K), -32, 31)
    d = np.full((N, K // 32), 0x3C00, np.uint16)
    qx = wl.int_codes(g, (M, K), -127, 127)
    ones = np.ones(M, np.float32)
    _, acc = oracle.gemv_i8g32(q, d, qx, ones, None, want_acc=True)
    w = torch.empty(lib.i8g32_repacked_bytes(N, K), dtype=torch.uint8, device="cuda")
    lib.i8g32_repack([dev(q)], [dev(d.view(np.int16))], K, w)
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    lib.i8g32_gemv(w, None, dev(qx), dev(ones), y)
    assert np.array_equal(host(y).astype(np.int64), acc.sum(axis=2).astype(np.int64))


# ------------------------------------------------------------ edges
def test_empty_calls_are_noops(lib):
    torch = _torch()
    y = torch.full((1, 8), 7.0, device="cuda")
    z8 = torch.zeros((1, 32), dtype=torch.int8, device="cuda")
    w = torch.zeros(lib.w4_repacked_bytes(8, 32), dtype=torch.uint8, device="cuda")
    sw = torch.ones(8, device="cuda")
    # M = 0 and N = 0 launch nothing and leave outputs untouched
    assert lib.load().w4a8_gemv(w.data_ptr(), sw.data_ptr(), None, z8.data_ptr(), sw.data_ptr(), 0, 8, 32,
                                y.data_ptr(), None) == 0
    assert lib.load().w4a8_gemv(w.data_ptr(), sw.data_ptr(), None, z8.data_ptr(), sw.data_ptr(), 1, 0, 32,
                                y.data_ptr(), None) == 0
    torch.cuda.synchronize()
    assert torch.all(y == 7.0)


def test_quantlinear_shard_fusion_matches_separate_shards(lib):
    """Fused q/k/v (one repack, one launch) equals three separate linears."""
    torch = _torch()
    from bit_quantized_decode_gb300 import QuantLinear
    K = 3584
    rows = (3584, 512, 512)
    g = wl.rng(23)
    Ws = [dev(wl.weights(g, n, K)) for n in rows]
    bs = [dev(wl.bias(g, n)) for n in rows]
    x = dev(wl.activations(g, 1, K))
    fused = QuantLinear.from_float("w4", Ws, bs)
    y = host(fused(x))
    parts = [host(QuantLinear.from_float("w4", [W], [b])(x)) for W, b in zip(Ws, bs)]
    assert np.array_equal(y.view(np.uint32), np.concatenate(parts, axis=1).view(np.uint32))
