"""Pins the CPU oracle to facts fixed outside itself.

Each test checks an oracle function against a value the pages print (fixtures
under tests/golden/, each citing its page and section), a closed form, a
library routine (numpy), or brute force on a tiny input.  None retypes the
oracle's own formula.  A dropped term, a wrong sign, a swapped operand or a
wrong rounding mode in the oracle fails at least one of them.
"""
import os

import numpy as np
import pytest

import oracle
from bit_quantized_decode_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _kv(name):
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, v = line.split()
            out[k] = int(v)
    return out


# ----------------------------------------------------------- int32 bound
def test_int32_worst_case_row_matches_page():
    g = _kv("orin_int4_worked.txt")
    H = g["H"]
    assert g["max_abs_qw"] * g["max_abs_qx"] == g["max_term"]
    packed = oracle.pack_int4(np.full((1, H), -8, np.int8))
    acc_pos = oracle.gemv_w4a8_acc(packed, np.full((1, H), -127, np.int8))
    acc_neg = oracle.gemv_w4a8_acc(packed, np.full((1, H), 127, np.int8))
    assert int(acc_pos[0, 0]) == g["row_bound"]
    assert int(acc_neg[0, 0]) == -g["row_bound"]
    assert g["row_bound"] < g["int32_max"] == 2**31 - 1


def test_int32_bound_at_intermediate_size():
    K = wl.QWEN7B_INTERMEDIATE
    packed = oracle.pack_int4(np.full((1, K), -8, np.int8))
    acc = oracle.gemv_w4a8_acc(packed, np.full((1, K), -127, np.int8))
    assert int(acc[0, 0]) == K * 1016 == 19_247_104


def test_int32_overflow_is_reported():
    # The largest K whose worst case still fits int32 is floor((2^31-1)/1016).
    kmax = (2**31 - 1) // 1016
    assert kmax == 2_113_665
    K_ok = kmax - kmax % 8             # 2_113_664: worst case fits
    K_bad = K_ok + 8                   # 2_113_672: worst case overflows
    for K, ok in ((K_ok, True), (K_bad, False)):
        packed = oracle.pack_int4(np.full((1, K), -8, np.int8))
        qx = np.full((1, K), -127, np.int8)
        if ok:
            assert int(oracle.gemv_w4a8_acc(packed, qx)[0, 0]) == K * 1016
        else:
            with pytest.raises(oracle.OracleError) as e:
                oracle.gemv_w4a8_acc(packed, qx)
            assert e.value.rc == oracle.ORC_ERR_INT32_OVERFLOW


# --------------------------------------------------------------- packing
def test_packing_words_match_diagram():
    with open(os.path.join(GOLDEN, "orin_int4_packing.txt")) as f:
        rows = [l.split() for l in f if l.strip() and not l.startswith("#")]
    for r in rows:
        w = np.array([int(v) for v in r[:8]], np.int8)[None, :]
        word = int(r[8], 16)
        assert int(oracle.pack_int4(w)[0, 0]) == word
        assert np.array_equal(oracle.unpack_int4(np.array([[word]], np.uint32), 8), w)


def test_packing_roundtrip_every_value_every_position():
    q = np.zeros((16 * 8, 8), np.int8)
    for v in range(-8, 8):
        for pos in range(8):
            q[(v + 8) * 8 + pos, pos] = v
    packed = oracle.pack_int4(q)
    assert np.array_equal(oracle.unpack_int4(packed, 8), q)
    # nibble `pos` of each word holds the value, every other nibble is 0
    for v in range(-8, 8):
        for pos in range(8):
            assert int(packed[(v + 8) * 8 + pos, 0]) == (v & 0xF) << (4 * pos)


def test_pack_rejects_out_of_range_codes():
    with pytest.raises(oracle.OracleError):
        oracle.pack_int4(np.array([[8, 0, 0, 0, 0, 0, 0, 0]], np.int8))


def test_row_bytes_match_page_table():
    g = _kv("orin_int4_worked.txt")
    assert oracle.row_weight_bytes(g["H"], 16) == g["row_bytes_fp16"]
    assert oracle.row_weight_bytes(g["H"], 8) == g["row_bytes_int8"]
    assert oracle.row_weight_bytes(g["H"], 4) == g["row_bytes_int4"]
    # and the canonical packed row really occupies that many bytes
    assert oracle.pack_int4(np.zeros((1, g["H"]), np.int8)).nbytes == g["row_bytes_int4"]


# ------------------------------------------------------------------ DP4A
def test_dp4a_matches_numpy_dot():
    g = np.random.default_rng(1)
    for _ in range(2000):
        a = g.integers(-128, 128, 4, dtype=np.int64)
        b = g.integers(-128, 128, 4, dtype=np.int64)
        c = int(g.integers(-(2**20), 2**20))
        aw = int(np.array(a, np.int8).view(np.uint32)[0])
        bw = int(np.array(b, np.int8).view(np.uint32)[0])
        assert oracle.dp4a(aw, bw, c) == c + int(np.dot(a, b))
    # extreme bytes
    assert oracle.dp4a(0x80808080, 0x80808080, 0) == 4 * 128 * 128
    assert oracle.dp4a(0x7F7F7F7F, 0x80808080, 0) == -4 * 127 * 128


def test_gemv_acc_equals_numpy_integer_matmul():
    g = np.random.default_rng(2)
    for (M, N, K) in ((1, 7, 64), (3, 5, 256), (2, 1, 3584)):
        q = wl.int_codes(g, (N, K), -8, 7)
        qx = wl.int_codes(g, (M, K), -127, 127)
        ref = qx.astype(np.int64) @ q.astype(np.int64).T
        acc = oracle.gemv_w4a8_acc(oracle.pack_int4(q), qx)
        assert np.array_equal(acc.astype(np.int64), ref)
        # the same sums built from the DP4A primitive, four products at a time
        qw_bytes = q.view(np.uint8).reshape(N, K // 4, 4)
        qx_bytes = qx.view(np.uint8).reshape(M, K // 4, 4)
        m, j = M - 1, N - 1
        s = 0
        for t in range(K // 4):
            s = oracle.dp4a(int(qw_bytes[j, t].view(np.uint32)[0]), int(qx_bytes[m, t].view(np.uint32)[0]), s)
        assert s == int(ref[m, j])


# ------------------------------------------------------- activation quant
def test_activation_quant_hand_cases():
    # s = 127/127 = 1: codes are the rounded values, ties to even, clipped at 127
    x = np.array([[127.0, 0.5, 1.5, 2.5, -0.5, -1.5, -127.0, 63.5]], np.float32)
    qx, sx = oracle.quantize_act_int8(x)
    assert sx[0] == np.float32(1.0)
    assert qx.tolist() == [[127, 0, 2, 2, 0, -2, -127, 64]]
    # s = 254/127 = 2
    qx, sx = oracle.quantize_act_int8(np.array([[254.0, 1.0, 3.0, 5.0, -254.0]], np.float32))
    assert sx[0] == np.float32(2.0)
    assert qx.tolist() == [[127, 0, 2, 2, -127]]


def test_activation_quant_zero_token():
    qx, sx = oracle.quantize_act_int8(np.zeros((2, 64), np.float32))
    assert np.all(qx == 0) and np.all(sx == 0)


def test_activation_quant_properties_on_random_tokens():
    g = np.random.default_rng(3)
    x = wl.activations(g, 4, 3584, outliers=True)
    qx, sx = oracle.quantize_act_int8(x)
    for m in range(4):
        amax = np.abs(x[m]).max()
        assert sx[m] == np.float32(amax) / np.float32(127)
        # the element equal to the absmax maps to +-127 exactly
        i = int(np.abs(x[m]).argmax())
        assert int(qx[m, i]) == (127 if x[m, i] > 0 else -127)
        # reconstruction error at most half a step, codes within [-127, 127]
        err = np.abs(x[m].astype(np.float64) - float(sx[m]) * qx[m].astype(np.float64))
        assert err.max() <= 0.5 * float(sx[m]) * (1 + 1e-6)
        assert qx[m].min() >= -127 and qx[m].max() <= 127
        # sign is kept
        nz = qx[m] != 0
        assert np.all(np.sign(qx[m][nz]) == np.sign(x[m][nz]))


# ------------------------------------------------------- weight quant
def test_weight_quant_exact_grid():
    s = np.float32(2.0**-6)
    k = np.array([[-7, -3, 0, 1, 7, 5, -1, 2]], np.int8)
    q, sw = oracle.quantize_rows_int4(k.astype(np.float32) * s)
    assert sw[0] == s and np.array_equal(q, k)


def test_weight_quant_properties():
    g = np.random.default_rng(4)
    W = wl.weights(g, 16, 512)
    W[3] = 0.0
    q, sw = oracle.quantize_rows_int4(W)
    assert sw[3] == 0 and np.all(q[3] == 0)
    for j in range(16):
        if j == 3:
            continue
        assert sw[j] == np.float32(np.abs(W[j]).max()) / np.float32(7)
        i = int(np.abs(W[j]).argmax())
        assert int(q[j, i]) == (7 if W[j, i] > 0 else -7)
        err = np.abs(W[j].astype(np.float64) - float(sw[j]) * q[j].astype(np.float64))
        assert err.max() <= 0.5 * float(sw[j]) * (1 + 1e-6)
        assert q[j].min() >= -8 and q[j].max() <= 7


# ------------------------------------------------- whole linear vs brute force
def test_lossless_special_case_equals_float_gemv():
    """W on an exact grid k*s and integer x with max 127 quantize without loss,
    so the quantized linear equals the float linear exactly."""
    g = np.random.default_rng(5)
    N, K = 8, 64
    s = np.float32(2.0**-7)
    k = wl.int_codes(g, (N, K), -7, 7)
    k[:, 0] = 7                                    # every row reaches the top code
    W = k.astype(np.float32) * s
    x = wl.int_codes(g, (2, K), -127, 127).astype(np.float32)
    x[:, 5] = 127.0
    b = (wl.int_codes(g, N, -50, 50).astype(np.float32) * np.float32(2.0**-4))
    y, qx, sx, acc = oracle.w4a8_linear(oracle.pack_int4(oracle.quantize_rows_int4(W)[0]),
                                        oracle.quantize_rows_int4(W)[1], x, b)
    ref = x.astype(np.float64) @ W.astype(np.float64).T + b.astype(np.float64)
    assert np.array_equal(y, ref)


@pytest.mark.parametrize("M,N,K", [(1, 8, 64), (3, 5, 32), (2, 8, 256)])
def test_quantized_linear_within_analytic_error_bound(M, N, K):
    """|y_q - y| <= sum_i |W||dx| + |dW||x| + |dW||dx| with |dW| <= s_w/2, |dx| <= s_x/2."""
    g = np.random.default_rng(10 + M * N + K)
    W = wl.weights(g, N, K, 0.5)
    x = wl.activations(g, M, K)
    b = wl.bias(g, N)
    q, sw = oracle.quantize_rows_int4(W)
    y, qx, sx, acc = oracle.w4a8_linear(oracle.pack_int4(q), sw, x, b)
    ref = x.astype(np.float64) @ W.astype(np.float64).T + b.astype(np.float64)
    aW = np.abs(W.astype(np.float64))
    ax = np.abs(x.astype(np.float64))
    dW = 0.5 * sw.astype(np.float64)[:, None] * (1 + 1e-6)
    dx = 0.5 * sx.astype(np.float64)[:, None] * (1 + 1e-6)
    bound = np.zeros((M, N))
    for m in range(M):
        for j in range(N):
            bound[m, j] = np.sum(aW[j] * dx[m] + dW[j] * ax[m] + dW[j] * dx[m])
    assert np.all(np.abs(y - ref) <= bound + 1e-9)
    # and the bound is not vacuous: it is far below the output scale
    assert bound.max() < 0.5 * np.abs(ax @ aW.T).max()


def test_scale_factoring_identity():
    """sum_i (s_W q_W)(s_x q_x) equals s_W s_x acc (dyadic scales: exact in fp64)."""
    g = np.random.default_rng(6)
    K = 512
    q = wl.int_codes(g, (3, K), -8, 7)
    qx = wl.int_codes(g, (1, K), -127, 127)
    sw = np.array([2.0**-5, 2.0**-9, 0.375], np.float32)
    sx = np.array([2.0**-3], np.float32)
    acc = oracle.gemv_w4a8_acc(oracle.pack_int4(q), qx)
    y = oracle.epilogue_w4a8(acc, sw, sx, None)
    direct = np.array([[np.sum((float(sw[j]) * q[j].astype(np.float64)) * (float(sx[0]) * qx[0].astype(np.float64)))
                        for j in range(3)]])
    assert np.array_equal(y, direct)


def test_bias_and_operand_order():
    """One nonzero weight and one nonzero activation pick out a single term."""
    K, N = 64, 4
    q = np.zeros((N, K), np.int8)
    q[2, 17] = -5
    qx = np.zeros((1, K), np.int8)
    qx[0, 17] = 3
    qx[0, 18] = 100
    acc = oracle.gemv_w4a8_acc(oracle.pack_int4(q), qx)
    assert acc.tolist() == [[0, 0, -15, 0]]
    y = oracle.epilogue_w4a8(acc, np.array([1, 1, 0.5, 1], np.float32), np.array([2.0], np.float32),
                             np.array([1, 2, 3, 4], np.float32))
    assert y.tolist() == [[1.0, 2.0, -15.0 + 3.0, 4.0]]


# ------------------------------------------------------------------ fp16
def test_half_to_float_exhaustive_against_numpy():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float32)
    got = np.array([oracle.half_to_float(int(b)) for b in bits], np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def test_float_to_half_against_numpy():
    g = np.random.default_rng(7)
    vals = np.concatenate([
        g.standard_normal(20000).astype(np.float32) * np.float32(10.0) ** g.integers(-9, 6, 20000).astype(np.float32),
        np.array([0.0, -0.0, 65504.0, 65519.0, 65520.0, 70000.0, -70000.0, 2.0**-24, 2.0**-25,
                  3 * 2.0**-26, 2.0**-14, 2.0**-14 - 2.0**-25, 1.0 + 2.0**-11, 1.0 + 3 * 2.0**-11,
                  np.inf, -np.inf], np.float32),
    ]).astype(np.float32)
    with np.errstate(over="ignore"):
        ref = vals.astype(np.float16).view(np.uint16)
    got = np.array([oracle.float_to_half(float(v)) for v in vals], np.uint16)
    assert np.array_equal(got, ref)


# ------------------------------------------------------------------ Q4_0
def test_q4_0_block_layout_matches_page():
    g = _kv("gemma_q4_0_block.txt")
    assert oracle.q4_0_block_bytes() == g["block_bytes"] == g["nibble_bytes"] + g["scale_bytes"]
    assert oracle.quantize_q4_0(np.zeros((1, 64), np.float32)).shape == (1, 2, g["block_bytes"])
    assert g["lm_head_rows"] * g["lm_head_cols"] * 2 // 10**6 == g["lm_head_bf16_mb"]


def test_q4_0_hand_block():
    # absmax 8 -> d = fp16(1.0); values w -> clip(round(w), -8, 7); +8 clips to 7
    w = np.array([[8.0, -8.0, 0.4, 0.5, 1.5, -2.5, 3.0, -7.0] + [0.0] * 24], np.float32)
    blk = oracle.quantize_q4_0(w)[0, 0]
    assert int(blk[0]) | (int(blk[1]) << 8) == 0x3C00
    vals = [7, -8, 0, 0, 2, -2, 3, -7] + [0] * 24
    n = [v + 8 for v in vals]
    assert [int(b) for b in blk[2:]] == [n[i] | (n[i + 16] << 4) for i in range(16)]
    assert np.array_equal(oracle.dequantize_q4_0(oracle.quantize_q4_0(w), 32)[0], np.array(vals, np.float64))


def test_q4_0_exact_grid_roundtrip():
    g = np.random.default_rng(8)
    k = wl.int_codes(g, (4, 96), -8, 7)
    k[:, ::32] = -8                                   # each block reaches -8: absmax = 8 d
    d = np.float32(2.0**-5)
    W = k.astype(np.float32) * d
    assert np.array_equal(oracle.dequantize_q4_0(oracle.quantize_q4_0(W), 96), W.astype(np.float64))


def test_q4_0_gemv_against_dequantized_float_gemv():
    g = np.random.default_rng(9)
    M, N, K = 2, 6, 160
    blocks = oracle.quantize_q4_0(wl.weights(g, N, K, 0.03))
    x = wl.activations(g, M, K)
    qx, sx = oracle.quantize_act_int8(x)
    b = wl.bias(g, N)
    y, acc = oracle.gemv_q4_0(blocks, qx, sx, b, want_acc=True)
    Wd = oracle.dequantize_q4_0(blocks, K)
    ref = (qx.astype(np.float64) * sx.astype(np.float64)[:, None]) @ Wd.T + b.astype(np.float64)
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-12)
    # the group accumulators are the integer dot products of each 32-block
    dbits = blocks[:, :, 0].astype(np.uint16) | (blocks[:, :, 1].astype(np.uint16) << 8)
    dval = dbits.view(np.float16).astype(np.float64)
    vals = np.rint(Wd / np.repeat(np.where(dval == 0, 1.0, dval), 32, axis=1)).astype(np.int64)
    for m in range(M):
        for j in range(N):
            for gi in range(K // 32):
                sl = slice(32 * gi, 32 * gi + 32)
                assert acc[m, j, gi] == int(np.dot(vals[j, sl], qx[m, sl].astype(np.int64)))


def test_q4_0_quant_error_bound():
    g = np.random.default_rng(11)
    W = wl.weights(g, 8, 256, 0.03)
    Wd = oracle.dequantize_q4_0(oracle.quantize_q4_0(W), 256)
    for j in range(8):
        for gi in range(8):
            sl = slice(32 * gi, 32 * gi + 32)
            amax = float(np.abs(W[j, sl]).max())
            d = float(np.float16(np.float32(amax) / np.float32(8)))
            w = W[j, sl].astype(np.float64)
            err = np.abs(w - Wd[j, sl])
            # half a step, except where w/d lies above 7.5 and clips to 7: there the
            # error is w - 7d, at most absmax - 7d (about one step; d is rounded to fp16)
            clipped = w / d > 7.5
            assert np.all(err[~clipped] <= 0.5 * d * (1 + 1e-6))
            assert np.all(err[clipped] <= amax - 7 * d + 1e-12)
            assert amax - 7 * d <= d * (1 + 2.0**-8) + 1e-12   # fp16 rounding: amax <= 8d(1+2^-11)
            assert np.all(Wd[j, sl][clipped] == 7 * d)


# ------------------------------------------------------------------ i8g32
def test_i8g32_hand_group():
    w = np.array([[32.0, -32.0, 0.5, 1.5, -31.0] + [0.0] * 27], np.float32)
    q, d = oracle.quantize_i8g32(w)
    assert int(d[0, 0]) == 0x3C00
    assert q[0, :5].tolist() == [31, -32, 0, 2, -31]


def test_i8g32_gemv_against_numpy():
    g = np.random.default_rng(12)
    M, N, K = 3, 5, 128
    q, d = oracle.quantize_i8g32(wl.weights(g, N, K))
    assert q.min() >= -32 and q.max() <= 31
    x = wl.activations(g, M, K)
    qx, sx = oracle.quantize_act_int8(x)
    b = wl.bias(g, N)
    y, acc = oracle.gemv_i8g32(q, d, qx, sx, b, want_acc=True)
    dd = d.view(np.float16).astype(np.float64)
    Wd = q.astype(np.float64) * np.repeat(dd, 32, axis=1)
    ref = (qx.astype(np.float64) * sx.astype(np.float64)[:, None]) @ Wd.T + b.astype(np.float64)
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-12)
    ref_acc = np.einsum("mgi,ngi->mng", qx.reshape(M, K // 32, 32).astype(np.int64),
                        q.reshape(N, K // 32, 32).astype(np.int64))
    assert np.array_equal(acc.astype(np.int64), ref_acc)


# ------------------------------------------------ operators around the linear
# RMSNorm and the gated MLP activations ([Orin-INT4] §"后续还能继续优化什么"
# item 1; [310B-Gemma4] §4.2), pinned by invariants and closed forms.

def test_rmsnorm_scale_invariant_bit_exact():
    """With eps = 0, scaling x by 4 (exact in fp32) scales S by 16 and r by
    1/4 exactly (correct rounding commutes with powers of two), so the output
    is bit-identical.  A missing square root, a missing square or a mean taken
    over |x| instead of x^2 breaks this."""
    g = wl.rng(11)
    x = g.standard_normal((3, 1536)).astype(np.float32)
    gam = (1.0 + 0.1 * g.standard_normal(1536)).astype(np.float32)
    a = oracle.rmsnorm_f32(x, gam, 0.0)
    b = oracle.rmsnorm_f32(4.0 * x, gam, 0.0)
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
    c = oracle.rmsnorm_f32(0.25 * x, gam, 0.0)
    assert np.array_equal(a.view(np.uint32), c.view(np.uint32))


@pytest.mark.parametrize("K", [32, 3584, 18944])
def test_rmsnorm_one_hot_closed_form(K):
    """x = v e_0, g = 1, eps = 0: ms = v^2 / K, so out_0 = sign(v) sqrt(K) and
    every other element is 0.  A mean over K - 1 or a sum without the 1/K
    fails."""
    for v in (3.0, -0.0625, 1234.5):
        x = np.zeros((1, K), np.float32)
        x[0, 0] = v
        out = oracle.rmsnorm_f32(x, np.ones(K, np.float32), 0.0)
        assert abs(out[0, 0] - np.sign(v) * np.sqrt(K)) <= 2 * np.spacing(np.float32(np.sqrt(K)))
        assert np.all(out[0, 1:] == 0)


def test_rmsnorm_eps_closed_form():
    """x = c everywhere and eps = c^2: ms + eps = 2 c^2, so out = 1 / sqrt(2)
    (to fp32 rounding).  eps added after the square root, or omitted, gives
    another value."""
    for c in (0.5, 2.0, 0.125):
        x = np.full((1, 256), c, np.float32)
        out = oracle.rmsnorm_f32(x, np.ones(256, np.float32), c * c)
        assert np.allclose(out, 1.0 / np.sqrt(2.0), rtol=3e-7, atol=0)


def test_rmsnorm_unit_mean_square_and_gamma_per_element():
    """With g = 1 and eps = 0 the output has mean square 1; with a random g
    every element is exactly fl(out1_i * g_i) (the weight multiplies last,
    element by element, not a shifted or reversed g)."""
    g = wl.rng(12)
    x = (3.0 * g.standard_normal((2, 3584))).astype(np.float32)
    one = oracle.rmsnorm_f32(x, np.ones(3584, np.float32), 0.0)
    ms = np.mean(one.astype(np.float64) ** 2, axis=1)
    assert np.all(np.abs(ms - 1.0) < 1e-5)
    gam = g.standard_normal(3584).astype(np.float32)
    out = oracle.rmsnorm_f32(x, gam, 0.0)
    assert np.array_equal(out.view(np.uint32), (one * gam[None, :]).astype(np.float32).view(np.uint32))


def test_rmsnorm_tokens_independent():
    g = wl.rng(13)
    x = g.standard_normal((4, 512)).astype(np.float32)
    x[2] *= 100.0
    gam = g.standard_normal(512).astype(np.float32)
    allm = oracle.rmsnorm_f32(x, gam, 1e-6)
    for m in range(4):
        assert np.array_equal(allm[m], oracle.rmsnorm_f32(x[m:m + 1], gam, 1e-6)[0])


def test_silu_against_logistic_and_identity():
    """SwiGLU: act(v) = v * logistic(v) (scipy's expit, a library routine),
    and the exact identity silu(-v) = silu(v) - v; the up factor multiplies."""
    special = pytest.importorskip("scipy.special")
    v = np.linspace(-30, 30, 6001)
    one = np.ones_like(v)
    s = oracle.glu(v, one, oracle.GLU_SILU)
    assert np.allclose(s, v * special.expit(v), rtol=1e-14, atol=1e-300)
    assert np.allclose(oracle.glu(-v, one, oracle.GLU_SILU), s - v, rtol=0, atol=1e-13)
    u = np.linspace(-2, 2, 6001)
    assert np.allclose(oracle.glu(v, u, oracle.GLU_SILU), s * u, rtol=1e-15, atol=0)
    assert oracle.glu(np.array([0.0]), np.array([5.0]), oracle.GLU_SILU)[0] == 0.0


def test_gelu_tanh_against_erf_gelu():
    """GELU(tanh): the identity act(v) - act(-v) = v, and the known accuracy
    of the tanh form against the exact v * Phi(v) (math.erf): within 5e-4
    everywhere and about 4.7e-4 at its worst near |v| = 2.7, so a dropped cubic
    term (error 0.034) or a wrong constant (0.09) fails."""
    import math
    v = np.linspace(-12, 12, 24001)
    one = np.ones_like(v)
    a = oracle.glu(v, one, oracle.GLU_GELU_TANH)
    assert np.allclose(a - oracle.glu(-v, one, oracle.GLU_GELU_TANH), v, rtol=0, atol=1e-12)
    exact = np.array([0.5 * t * (1.0 + math.erf(t / math.sqrt(2.0))) for t in v])
    err = np.abs(a - exact)
    assert err.max() < 5e-4
    assert err.max() > 4e-4
    u = np.full_like(v, -3.0)
    assert np.allclose(oracle.glu(v, u, oracle.GLU_GELU_TANH), -3.0 * a, rtol=1e-15, atol=0)


# -------------------------------------- weight-only paths (float activations)
# [Orin-INT4] §"为什么 INT4 float 解包不快": weight-only INT8 and INT4 with float
# unpacking, the two paths the page measures against INT4 DP4A.

def test_quantize_rows_int8_exact_grid_and_extremes():
    """Rows on the grid k * s (k in [-127, 127]) with the absmax at 127 s
    quantize exactly; the absmax maps to +-127; an all-zero row gives s = 0."""
    g = wl.rng(21)
    s = np.float32(2.0 ** -7)
    k = g.integers(-127, 128, size=(4, 256))
    k[:, 0] = 127
    k[1, 0] = -127
    W = (k * s).astype(np.float32)
    q, sw = oracle.quantize_rows_int8(W)
    assert np.all(sw == s)
    assert np.array_equal(q.astype(int), k)
    q0, s0 = oracle.quantize_rows_int8(np.zeros((1, 64), np.float32))
    assert s0[0] == 0 and not q0.any()
    Wr = wl.weights(g, 8, 512)
    qr, swr = oracle.quantize_rows_int8(Wr)
    assert np.all(np.abs(qr.astype(int)).max(axis=1) == 127)
    assert np.all(np.abs(Wr - qr * swr[:, None]) <= swr[:, None] / 2 * (1 + 1e-6))


def test_gemv_weight_only_against_numpy():
    """The weight-only linear against numpy's float64 matmul (a library routine)
    on the same integer codes, scales and bias."""
    g = wl.rng(22)
    M, N, K = 3, 40, 640
    q = g.integers(-127, 128, size=(N, K)).astype(np.int8)
    sw = wl.positive_scales(g, N)
    x = wl.activations(g, M, K, outliers=True)
    b = wl.bias(g, N)
    y = oracle.gemv_weight_only(q, sw, x, b)
    ref = (x.astype(np.float64) @ q.astype(np.float64).T) * sw.astype(np.float64)[None, :] + b[None, :]
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-12)
    # a single term: catches a swapped operand or a dropped scale or bias
    q1 = np.zeros((2, 32), np.int8)
    q1[1, 5] = -3
    x1 = np.zeros((1, 32), np.float32)
    x1[0, 5] = 0.5
    y1 = oracle.gemv_weight_only(q1, np.array([1.0, 0.25], np.float32), x1, np.array([0.0, 2.0], np.float32))
    assert y1[0, 0] == 0.0 and y1[0, 1] == 0.25 * -1.5 + 2.0


def test_weight_only_int4_equals_float_reconstruction():
    """INT4 codes through the weight-only linear equal the float GEMV of the
    reconstructed weights s_w q (exact products in fp64): the float-unpack
    path computes the dequantized weights' product with unquantized x."""
    g = wl.rng(23)
    W = wl.weights(g, 16, 256)
    q, sw = oracle.quantize_rows_int4(W)
    x = wl.activations(g, 2, 256)
    y = oracle.gemv_weight_only(q, sw, x)
    Wd = q.astype(np.float64) * sw.astype(np.float64)[:, None]
    assert np.allclose(y, x.astype(np.float64) @ Wd.T, rtol=1e-12, atol=1e-12)
