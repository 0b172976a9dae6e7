"""The library's host-side quantizers (w4_quantize_rows_host, q4_0_quantize_host,
i8g32_quantize_host) against the oracle, byte for byte, on the CPU.

These are the library's own C++ (no oracle code): the oracle is the
definition ("Jetson Orin AGX INT4 推理优化实践" §"从 FP 线性层到 INT4 DP4A 的数学
推导" for per-row INT4; "在香橙派上跑 Gemma4" §3.1 and §3.2 for Q4_0 and the
int8 group format).  Cases: the workloads' distributions, all-zero rows and
blocks, exact ties of the quotient, fp16 scales that are subnormal, that round
at a tie, and that overflow to infinity, and group magnitudes spread over
every fp16 binade.
"""
import numpy as np
import pytest

import oracle
from bit_quantized_decode_gb300 import workloads as wl


@pytest.fixture(scope="module")
def lib():
    from bit_quantized_decode_gb300 import _lib, build
    build.build()
    _lib.load()
    return _lib


def _spread_blocks(g, N, K, lo_exp=-32, hi_exp=20):
    """Weights whose 32-blocks have magnitudes 2^e, e uniform in [lo_exp, hi_exp)."""
    W = g.standard_normal((N, K // 32, 32)).astype(np.float32)
    e = g.uniform(lo_exp, hi_exp, size=(N, K // 32, 1))
    return (W * np.exp2(e)).astype(np.float32).reshape(N, K)


@pytest.mark.parametrize("N,K,sigma", [(64, 3584, 0.02), (13, 96, 1.0), (3, 8, 0.3)])
def test_w4_rows_host_equals_oracle(lib, N, K, sigma):
    W = wl.weights(wl.rng(N + K), N, K, sigma)
    W[min(2, N - 1)] = 0.0                                    # a zero row: s_w = 0, codes 0
    packed, sw = lib.w4_quantize_rows_host(W)
    q_ref, sw_ref = oracle.quantize_rows_int4(W)
    assert np.array_equal(sw.view(np.uint32), sw_ref.view(np.uint32))
    assert np.array_equal(packed, oracle.pack_int4(q_ref))


def test_w4_rows_host_ties_and_magnitudes(lib):
    K = 64
    W = np.zeros((4, K), np.float32)
    W[0, :9] = [7.0, 0.5, 1.5, 2.5, -0.5, -1.5, -2.5, 6.5, -7.0]    # s = 1: exact ties both ways
    W[1] = np.float32(1e-44) * np.arange(-32, 32, dtype=np.float32)  # subnormal weights
    W[2] = np.float32(3.0e38) * np.sin(np.arange(K, dtype=np.float32))
    W[3] = _spread_blocks(wl.rng(9), 1, K, -140, 120)[0]
    packed, sw = lib.w4_quantize_rows_host(W)
    q_ref, sw_ref = oracle.quantize_rows_int4(W)
    assert np.array_equal(sw.view(np.uint32), sw_ref.view(np.uint32))
    assert np.array_equal(packed, oracle.pack_int4(q_ref))
    assert oracle.unpack_int4(packed[:1], K)[0, :9].tolist() == [7, 0, 2, 2, 0, -2, -2, 6, -7]


@pytest.mark.parametrize("N,K,sigma", [(40, 1536, 0.03), (5, 64, 1.0)])
def test_q4_0_host_equals_oracle(lib, N, K, sigma):
    W = wl.weights(wl.rng(3 * N + K), N, K, sigma)
    W[0, :32] = 0.0                                           # a zero block: d = 0, nibbles 8
    assert np.array_equal(lib.q4_0_quantize_host(W), oracle.quantize_q4_0(W))


@pytest.mark.parametrize("N,K,sigma", [(40, 1536, 0.02), (5, 64, 1.0)])
def test_i8g32_host_equals_oracle(lib, N, K, sigma):
    W = wl.weights(wl.rng(5 * N + K), N, K, sigma)
    W[-1, 32:64] = 0.0
    q, d = lib.i8g32_quantize_host(W)
    q_ref, d_ref = oracle.quantize_i8g32(W)
    assert np.array_equal(q, q_ref)
    assert np.array_equal(d, d_ref)


def test_group_scales_over_every_fp16_binade(lib):
    """Block magnitudes from 2^-32 (the fp16 scale underflows to zero or a
    subnormal) to 2^20 (it overflows to infinity): the scale rounding and the
    codes against it match the oracle everywhere."""
    g = wl.rng(31)
    W = _spread_blocks(g, 256, 1024)
    assert np.array_equal(lib.q4_0_quantize_host(W), oracle.quantize_q4_0(W))
    q, d = lib.i8g32_quantize_host(W)
    q_ref, d_ref = oracle.quantize_i8g32(W)
    assert np.array_equal(q, q_ref) and np.array_equal(d, d_ref)
    # the sweep reached subnormal, normal and infinite scales
    dh = d.view(np.float16).astype(np.float64)
    assert (dh[(dh > 0) & (dh < 2.0 ** -14)]).size > 0 and np.isinf(dh).any() and (dh >= 1.0).any()


def test_group_scale_ties_round_to_even(lib):
    """absmax / 8 exactly halfway between two fp16 values: round to the even one."""
    K = 32
    # fp16 spacing at 1.0 is 2^-10; 1 + 2^-11 is a tie (-> 1.0), 1 + 3*2^-11 -> 1 + 2^-9
    mags = np.array([1.0 + 2.0 ** -11, 1.0 + 3 * 2.0 ** -11, 2.0 ** -24 * 1.5, 2.0 ** -24 * 2.5], np.float64)
    W = np.zeros((len(mags), K), np.float32)
    W[:, 0] = (8.0 * mags).astype(np.float32)
    W[:, 1:] = W[:, :1] * np.linspace(-0.9, 0.9, K - 1, dtype=np.float32)
    blocks = lib.q4_0_quantize_host(W)
    assert np.array_equal(blocks, oracle.quantize_q4_0(W))
    d = (blocks[:, 0, 0].astype(np.uint16) | (blocks[:, 0, 1].astype(np.uint16) << 8))
    assert d.tolist() == [0x3C00, 0x3C02, 0x0002, 0x0002]
