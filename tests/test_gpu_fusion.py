"""Operators fused around the decode linear: RMSNorm in front of the
quantizer, the gated MLP activation (SiLU, GELU tanh) and the residual add
after the epilogue ([Orin-INT4] §"后续还能继续优化什么" item 1,
[310B-Gemma4] §4.2).

Parity with the oracle:
  * the activation codes and scales of a normalized token are bit-exact.  The
    one step that is not order-independent, the sum of squares, is rounded once
    to fp32 on both sides (the kernel's compensated sum is within about
    d^2 2^-48 of the exact value, d its summation depth), so a token can differ
    only when the exact sum lies that close to an fp32 rounding boundary; the
    test measures that distance from the oracle's inputs and, for such a token
    alone, allows a scale one ulp away and codes one step away;
  * y within the per-format tolerance (same as the plain linears);
  * gated outputs within the bound the arithmetic gives: the gate and up
    values each within the linear's tolerance, propagated through the
    activation (|act'| <= 1.2 for both), plus a few fp32 roundings.
Consistency with the separate kernels: the fused output equals the plain
linear followed by w4_rmsnorm/w4_glu/w4_add (same arithmetic) bit for bit
wherever the linear's own result is order-independent (W4's integer sums).
"""
import math

import numpy as np
import pytest

import oracle
from bit_quantized_decode_gb300 import workloads as wl
from helpers import RTOL_GROUP, RTOL_W4, cuda_ok, dev, group_scale, host, q4_0_scales, w4_scale

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not cuda_ok(), reason="needs a CUDA GPU")]

EPS = 1e-6


@pytest.fixture(scope="module")
def lib():
    import torch  # noqa: F401

    from bit_quantized_decode_gb300 import _lib
    _lib.load()
    _lib.clear_device_error()
    yield _lib
    _lib.set_tuning("tc_min_m", 0)
    assert _lib.device_error() == 0


# ------------------------------------------------------------ helpers
def _sum_margin(row) -> float:
    """Relative distance of the exact sum of squares of an fp32 row from the
    nearest fp32 rounding boundary (math.fsum: the exact sum correctly rounded
    to double; each square is exact in double)."""
    S = math.fsum(float(v) * float(v) for v in row)
    if S == 0.0:
        return math.inf
    s32 = np.float32(S)
    lo = np.nextafter(s32, np.float32(-np.inf))
    hi = np.nextafter(s32, np.float32(np.inf))
    m1 = (float(s32) + float(lo)) / 2.0
    m2 = (float(s32) + float(hi)) / 2.0
    return min(abs(S - m1), abs(S - m2)) / S


def _ambiguous(x, per_thread):
    """Tokens whose sum of squares lies within the kernels' error bound of an
    fp32 rounding boundary (bound 4 d^2 2^-48, d = squares per thread + tree depth)."""
    d = per_thread + 10
    band = 4.0 * d * d * 2.0 ** -48
    return [_sum_margin(x[m]) < band for m in range(x.shape[0])]


def _check_codes(qx, sx, qx_ref, sx_ref, amb, what):
    for m in range(qx_ref.shape[0]):
        if not amb[m]:
            assert sx[m].view(np.uint32) == sx_ref[m].view(np.uint32), f"{what}: sx of token {m}"
            assert np.array_equal(qx[m], qx_ref[m]), f"{what}: codes of token {m}"
        else:
            assert abs(float(sx[m]) - float(sx_ref[m])) <= 4 * np.spacing(sx_ref[m]), f"{what}: sx of token {m}"
            assert np.abs(qx[m].astype(int) - qx_ref[m].astype(int)).max() <= 1, f"{what}: codes of token {m}"
    assert sum(amb) <= 1, "inputs chosen too close to rounding boundaries"


def _close(y, y_ref, bound, what):
    err = np.abs(np.asarray(y, np.float64) - y_ref)
    bad = err > bound + 1e-30
    if bad.any():
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"{what}: {bad.sum()} of {err.size} outside; worst at {i}: gpu {y[i]!r} "
                             f"ref {y_ref[i]!r} bound {bound[i]!r}")


class Layer:
    """One linear in a given format: device weights and the oracle."""

    def __init__(self, lib, fmt, g, N, K, with_bias=True):
        import torch
        self.fmt, self.N, self.K = fmt, N, K
        W = wl.weights(g, N, K)
        self.b = wl.bias(g, N) if with_bias else None
        self.bd = None if self.b is None else dev(self.b)
        self.sw = self.swd = None
        if fmt == "w4":
            self.q, self.sw = oracle.quantize_rows_int4(W)
            self.swd = dev(self.sw)
            self.w = torch.empty(lib.w4_repacked_bytes(N, K), dtype=torch.uint8, device="cuda")
            lib.w4_repack([dev(oracle.pack_int4(self.q).view(np.int32))], K, self.w)
        elif fmt == "q4_0":
            self.blocks = oracle.quantize_q4_0(W)
            self.w = torch.empty(lib.q4_0_repacked_bytes(N, K), dtype=torch.uint8, device="cuda")
            lib.q4_0_repack([dev(self.blocks)], K, self.w)
        else:
            self.q, self.d = oracle.quantize_i8g32(W)
            nb = lib.i8g32_repacked_bytes(N, K) if fmt == "i8g32" else lib.q6g32_repacked_bytes(N, K)
            self.w = torch.empty(nb, dtype=torch.uint8, device="cuda")
            rep = lib.i8g32_repack if fmt == "i8g32" else lib.q6g32_repack
            rep([dev(self.q)], [dev(self.d.view(np.int16))], K, self.w)

    def ref(self, qx, sx):
        """(y fp64, error bound) of the linear on codes qx, sx."""
        if self.fmt == "w4":
            acc = oracle.gemv_w4a8_acc(oracle.pack_int4(self.q), qx)
            return oracle.epilogue_w4a8(acc, self.sw, sx, self.b), RTOL_W4 * w4_scale(acc, self.sw, sx, self.b)
        if self.fmt == "q4_0":
            y, acc = oracle.gemv_q4_0(self.blocks, qx, sx, self.b, want_acc=True)
            return y, RTOL_GROUP * group_scale(acc, q4_0_scales(self.blocks), sx, self.b)
        y, acc = oracle.gemv_i8g32(self.q, self.d, qx, sx, self.b, want_acc=True)
        return y, RTOL_GROUP * group_scale(acc, self.d.view(np.float16).astype(np.float64), sx, self.b)

    def fused(self, lib, x, y, qx, sx, fz, flags=0):
        if self.fmt == "w4":
            lib.w4a8_linear_fused(self.w, self.swd, self.bd, x, y, qx, sx, fz, flags)
        else:
            getattr(lib, f"{self.fmt}_linear_fused")(self.w, self.bd, x, y, qx, sx, fz, flags)

    def gemv(self, lib, qx, sx, y):
        if self.fmt == "w4":
            lib.w4a8_gemv(self.w, self.swd, self.bd, qx, sx, y)
        else:
            getattr(lib, f"{self.fmt}_gemv")(self.w, self.bd, qx, sx, y)


def _bufs(M, N, K):
    import torch
    return (torch.empty((M, N), dtype=torch.float32, device="cuda"),
            torch.empty((M, K), dtype=torch.int8, device="cuda"),
            torch.empty(M, dtype=torch.float32, device="cuda"))


# --------------------------------------------------------- RMSNorm prologue
@pytest.mark.parametrize("M,K", [(1, 3584), (3, 1536), (16, 3584), (2, 18944), (1, 40960), (5, 96)])
def test_rms_a8_quantize_matches_oracle(lib, M, K):
    """The standalone normalize+quantize kernel (registers up to 20480 values
    per token, three passes beyond)."""
    import torch
    g = wl.rng(1000 + M * 7 + K)
    x = wl.residual_stream(g, M, K)
    gam = wl.norm_weight(g, K)
    qx_ref, sx_ref = oracle.quantize_act_int8(oracle.rmsnorm_f32(x, gam, EPS))
    qx = torch.empty((M, K), dtype=torch.int8, device="cuda")
    sx = torch.empty(M, dtype=torch.float32, device="cuda")
    lib.rms_a8_quantize(dev(x), dev(gam), EPS, qx, sx)
    amb = _ambiguous(x, 4 * ((K // 4 + 511) // 512))
    _check_codes(host(qx), host(sx), qx_ref, sx_ref, amb, "rms_a8_quantize")


def test_rmsnorm_kernel_matches_oracle(lib):
    """w4_rmsnorm (fp32 out) equals the oracle's fp32 steps bit for bit."""
    import torch
    M, K = 4, 3584
    g = wl.rng(77)
    x = wl.residual_stream(g, M, K)
    gam = wl.norm_weight(g, K)
    ref = oracle.rmsnorm_f32(x, gam, EPS)
    out = torch.empty((M, K), dtype=torch.float32, device="cuda")
    lib.w4_rmsnorm(dev(x), dev(gam), EPS, out)
    amb = _ambiguous(x, 4 * ((K // 4 + 511) // 512))
    got = host(out)
    for m in range(M):
        if not amb[m]:
            assert np.array_equal(got[m].view(np.uint32), ref[m].view(np.uint32))
        else:
            assert np.allclose(got[m], ref[m], rtol=4e-7, atol=0)


@pytest.mark.parametrize("fmt", ["w4", "q4_0", "i8g32", "q6g32"])
@pytest.mark.parametrize("M,N,K", [(1, 4608, 3584), (2, 1000, 1536), (4, 264, 3584), (3, 520, 6144), (1, 77, 96),
                                   (1, 300, 18944)])
def test_norm_linear_fused(lib, fmt, M, N, K):
    """RMSNorm fused into the GEMV prologue (one to four tokens, x and the norm
    weight in registers; longer x falls back to the separate kernel): codes
    and scales bit-exact, y within the format's tolerance, and y bit-identical
    to rms_a8_quantize followed by the plain GEMV."""
    import torch
    g = wl.rng(2000 + M * 13 + N + K)
    L = Layer(lib, fmt, g, N, K)
    x = wl.residual_stream(g, M, K)
    gam = wl.norm_weight(g, K)
    qx_ref, sx_ref = oracle.quantize_act_int8(oracle.rmsnorm_f32(x, gam, EPS))
    xd, gd = dev(x), dev(gam)
    y, qx, sx = _bufs(M, N, K)
    fz = lib.fusion(norm_weight=gd, eps=EPS)
    L.fused(lib, xd, y, qx, sx, fz)
    amb = _ambiguous(x, 4 * ((K // 4 + 255) // 256))
    _check_codes(host(qx), host(sx), qx_ref, sx_ref, amb, f"{fmt} fused norm")
    y_ref, bound = L.ref(qx_ref, sx_ref)
    if not any(amb):
        _close(host(y), y_ref, bound, f"{fmt} fused norm linear")
    # the same codes through the separate kernels give the same bits
    qx2 = torch.empty_like(qx)
    sx2 = torch.empty_like(sx)
    lib.rms_a8_quantize(xd, gd, EPS, qx2, sx2)
    y2 = torch.empty_like(y)
    L.gemv(lib, qx2, sx2, y2)
    if np.array_equal(host(qx2), host(qx)) and np.array_equal(host(sx2), host(sx)):
        assert np.array_equal(host(y).view(np.uint32), host(y2).view(np.uint32))


def test_norm_linear_tensor_cores(lib):
    """Many tokens: normalize+quantize kernel, then the tensor-core GEMV."""
    import torch
    M, N, K = 16, 4608, 3584
    g = wl.rng(31)
    L = Layer(lib, "w4", g, N, K)
    x = wl.residual_stream(g, M, K)
    gam = wl.norm_weight(g, K)
    qx_ref, sx_ref = oracle.quantize_act_int8(oracle.rmsnorm_f32(x, gam, EPS))
    y, qx, sx = _bufs(M, N, K)
    lib.set_tuning("tc_min_m", 1)
    L.fused(lib, dev(x), y, qx, sx, lib.fusion(norm_weight=dev(gam), eps=EPS), lib.W4_FLAG_PDL)
    lib.set_tuning("tc_min_m", 0)
    amb = _ambiguous(x, 4 * ((K // 4 + 511) // 512))
    _check_codes(host(qx), host(sx), qx_ref, sx_ref, amb, "tensor-core norm")
    y_ref, bound = L.ref(qx_ref, sx_ref)
    if not any(amb):
        _close(host(y), y_ref, bound, "tensor-core norm linear")


# ------------------------------------------------------------ gated MLP
class GatedLayer:
    """Gate and up halves of a gated MLP (W4 or Q4_0), paired by *_repack_glu,
    and the same halves concatenated [gate; up] for the plain linear."""

    def __init__(self, lib, fmt, g, I, K):
        import torch
        self.fmt, self.I, self.K = fmt, I, K
        self.gate = Layer(lib, fmt, g, I, K)
        self.up = Layer(lib, fmt, g, I, K)
        self.bd = dev(np.concatenate([self.gate.b, self.up.b]))
        if fmt == "w4":
            self.swd = dev(np.concatenate([self.gate.sw, self.up.sw]))
            pg = dev(oracle.pack_int4(self.gate.q).view(np.int32))
            pu = dev(oracle.pack_int4(self.up.q).view(np.int32))
            self.wp = torch.empty(lib.w4_glu_repacked_bytes(I, K), dtype=torch.uint8, device="cuda")
            lib.w4_repack_glu(pg, pu, K, self.wp)
            self.wc = torch.empty(lib.w4_repacked_bytes(2 * I, K), dtype=torch.uint8, device="cuda")
            lib.w4_repack([pg, pu], K, self.wc)
        else:
            bg, bu = dev(self.gate.blocks), dev(self.up.blocks)
            self.wp = torch.empty(lib.q4_0_glu_repacked_bytes(I, K), dtype=torch.uint8, device="cuda")
            lib.q4_0_repack_glu(bg, bu, K, self.wp)
            self.wc = torch.empty(lib.q4_0_repacked_bytes(2 * I, K), dtype=torch.uint8, device="cuda")
            lib.q4_0_repack([bg, bu], K, self.wc)

    def run(self, lib, w, x, y, qx, sx, fz=None, flags=0):
        if self.fmt == "w4":
            lib.w4a8_linear_fused(w, self.swd, self.bd, x, y, qx, sx, fz, flags)
        else:
            lib.q4_0_linear_fused(w, self.bd, x, y, qx, sx, fz, flags)

    def ref(self, qx, sx, kind):
        yg, eg = self.gate.ref(qx, sx)
        yu, eu = self.up.ref(qx, sx)
        act = oracle.glu(yg, yu, kind)
        act_g = oracle.glu(yg, np.ones_like(yg), kind)
        ulp = 2.0 ** -23
        bound = 1.2 * np.abs(yu) * (eg + ulp * np.abs(yg)) + np.abs(act_g) * (eu + ulp * np.abs(yu)) \
            + 8 * ulp * np.abs(act)
        return act, bound


@pytest.mark.parametrize("fmt,kind", [("w4", 1), ("w4", 2), ("q4_0", 1), ("q4_0", 2)])
@pytest.mark.parametrize("M,I,K", [(1, 2368, 3584), (3, 101, 1536), (4, 3, 256), (16, 1000, 3584), (8, 516, 96),
                                   (12, 260, 1536)])
def test_glu_linear(lib, fmt, kind, M, I, K):
    """Gate/up paired per tile, the activation in the epilogue: within the
    propagated bound of the oracle, and equal to the plain linear on the
    [gate; up] layout followed by w4_glu -- bit for bit for W4 (integer
    accumulators), within the same bound for Q4_0 (its fp32 group sums merge
    in an order that depends on where a row's tile falls)."""
    import torch
    g = wl.rng(3000 + 17 * M + I + K + kind)
    L = GatedLayer(lib, fmt, g, I, K)
    x = wl.activations(g, M, K, outliers=True)
    xd = dev(x)
    y, qx, sx = _bufs(M, I, K)
    L.run(lib, L.wp, xd, y, qx, sx, lib.fusion(glu=kind))
    qx_ref, sx_ref = oracle.quantize_act_int8(x)
    assert np.array_equal(host(qx), qx_ref) and np.array_equal(host(sx), sx_ref)
    act, bound = L.ref(qx_ref, sx_ref, kind)
    _close(host(y), act, bound, f"{fmt} glu {kind}")
    y2, qx2, sx2 = _bufs(M, 2 * I, K)
    L.run(lib, L.wc, xd, y2, qx2, sx2)
    out = torch.empty((M, I), dtype=torch.float32, device="cuda")
    lib.w4_glu(y2, kind, out)
    if fmt == "w4":
        assert np.array_equal(host(out).view(np.uint32), host(y).view(np.uint32))
    else:
        _close(host(out), act, bound, f"{fmt} glu {kind}, separate kernels")


def test_glu_linear_tensor_cores_and_uncached_rows(lib):
    """W4 gated linear on the tensor cores (M = 16 and 6) and, at one token, with
    more rows per block than the staged parameter cache (I = 80000)."""
    import torch
    for M, I, K, tc in ((16, 4736, 3584, True), (6, 1000, 1536, True), (1, 80000, 64, False)):
        g = wl.rng(4000 + I)
        L = GatedLayer(lib, "w4", g, I, K)
        x = wl.activations(g, M, K)
        y, qx, sx = _bufs(M, I, K)
        lib.set_tuning("tc_min_m", 1 if tc else 17)
        L.run(lib, L.wp, dev(x), y, qx, sx, lib.fusion(glu=1), lib.W4_FLAG_PDL)
        lib.set_tuning("tc_min_m", 0)
        qx_ref, sx_ref = oracle.quantize_act_int8(x)
        act, bound = L.ref(qx_ref, sx_ref, 1)
        _close(host(y), act, bound, f"glu M={M} I={I}")


# ------------------------------------------------------------- residual
@pytest.mark.parametrize("fmt,M,N,K,tc", [("w4", 1, 3584, 3584, False), ("w4", 2, 3584, 18944, False),
                                          ("q4_0", 3, 1536, 6144, False), ("w4", 16, 3584, 3584, True),
                                          ("i8g32", 1, 200, 1536, False), ("w4", 7, 1000, 3584, True),
                                          ("w4", 4, 264, 3584, False), ("w4", 3, 520, 6144, False),
                                          ("q4_0", 12, 1536, 6144, False), ("q6g32", 16, 300, 1536, False),
                                          ("i8g32", 9, 1000, 1536, False)])
def test_residual_linear_in_place(lib, fmt, M, N, K, tc):
    """y = residual + linear(x), with the residual buffer as the output (the
    decoder's in-place update): within the linear's tolerance plus the final
    fp32 add, and bit-identical to the plain linear followed by w4_add."""
    import torch
    g = wl.rng(5000 + M + N + K)
    L = Layer(lib, fmt, g, N, K)
    x = wl.activations(g, M, K)
    h = wl.residual_stream(g, M, N)
    hd = dev(h)
    y, qx, sx = _bufs(M, N, K)
    lib.set_tuning("tc_min_m", 1 if tc else 17)
    L.fused(lib, dev(x), hd, qx, sx, lib.fusion(residual=hd), lib.W4_FLAG_PDL)
    L.fused(lib, dev(x), y, qx, sx, None, lib.W4_FLAG_PDL)
    lib.set_tuning("tc_min_m", 0)
    qx_ref, sx_ref = oracle.quantize_act_int8(x)
    y_ref, bound = L.ref(qx_ref, sx_ref)
    _close(host(hd), h.astype(np.float64) + y_ref, bound + 2.0 ** -24 * (np.abs(h) + np.abs(y_ref)),
           f"{fmt} residual")
    out = torch.empty((M, N), dtype=torch.float32, device="cuda")
    lib.w4_add(dev(h), y, out)
    assert np.array_equal(host(out).view(np.uint32), host(hd).view(np.uint32))


# ------------------------------------------------------- all three at once
def test_norm_glu_linear_one_token(lib):
    """The gate/up linear of a decoder layer: RMSNorm prologue and SwiGLU
    epilogue in one launch."""
    M, I, K = 1, 1184, 3584
    g = wl.rng(6000)
    L = GatedLayer(lib, "w4", g, I, K)
    x = wl.residual_stream(g, M, K)
    gam = wl.norm_weight(g, K)
    y, qx, sx = _bufs(M, I, K)
    L.run(lib, L.wp, dev(x), y, qx, sx, lib.fusion(norm_weight=dev(gam), eps=EPS, glu=1))
    qx_ref, sx_ref = oracle.quantize_act_int8(oracle.rmsnorm_f32(x, gam, EPS))
    amb = _ambiguous(x, 4 * ((K // 4 + 255) // 256))
    _check_codes(host(qx), host(sx), qx_ref, sx_ref, amb, "norm+glu")
    if not any(amb):
        act, bound = L.ref(qx_ref, sx_ref, 1)
        _close(host(y), act, bound, "norm+glu")


# --------------------------------------------------------- argument checks
def test_fusion_argument_errors(lib):
    import torch
    M, N, K = 1, 64, 256
    g = wl.rng(7)
    L = Layer(lib, "w4", g, N, K)
    x = dev(wl.activations(g, M, K))
    y, qx, sx = _bufs(M, N, K)
    gam = torch.ones(K + 4, dtype=torch.float32, device="cuda")
    with pytest.raises(lib.W4Error) as e:
        L.fused(lib, x, y, qx, sx, lib.fusion(norm_weight=gam[:K], eps=0.0))
    assert e.value.status == 1
    with pytest.raises(lib.W4Error) as e:
        L.fused(lib, x, y, qx, sx, lib.fusion(norm_weight=gam[1:K + 1], eps=EPS))
    assert e.value.status == 3
    with pytest.raises(lib.W4Error) as e:
        L.fused(lib, x, y, qx, sx, lib.fusion(glu=3))
    assert e.value.status == 1
    L8 = Layer(lib, "i8g32", g, N, K)
    with pytest.raises(lib.W4Error) as e:
        L8.fused(lib, x, y, qx, sx, lib.fusion(glu=1))
    assert e.value.status == 2
    # N = 0 with a norm: the codes only
    y0 = torch.empty((M, 0), dtype=torch.float32, device="cuda")
    lib.w4a8_linear_fused(L.w, L.swd, L.bd, x, y0, qx, sx, lib.fusion(norm_weight=gam[:K], eps=EPS))
    qx_ref, sx_ref = oracle.quantize_act_int8(oracle.rmsnorm_f32(host(x), np.ones(K, np.float32), EPS))
    amb = _ambiguous(host(x), 8)
    _check_codes(host(qx), host(sx), qx_ref, sx_ref, amb, "N = 0")
