"""GPU checks of the boundary's helper entry points.

- The host quantizers (library C++) and the device quantizers (CUDA) give the
  same bytes on the same weights; the CPU suite pins the host ones to the
  oracle, so all three agree.
- w4_hbm_read reads every byte once: its XOR checksum equals numpy's over a
  buffer with a ragged tail (a last chunk shorter than a ring slot).
- w4_last_device_error reads the same word as w4_device_error.
- The timeout path of the bounded waits: a kernel whose wait nothing
  completes (the per-warp ring form and the K-split leader's cluster-scope
  form) ends by itself, sets the wait-timeout code in the error word, and the
  context keeps computing correct results afterwards.  No GPU fault is made.
"""
import numpy as np
import pytest

import oracle
from bit_quantized_decode_gb300 import workloads as wl
from helpers import cuda_ok, dev, host

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not cuda_ok(), reason="needs a CUDA GPU")]


@pytest.fixture(scope="module")
def lib():
    import torch  # noqa: F401

    from bit_quantized_decode_gb300 import _lib
    _lib.load()
    _lib.clear_device_error()
    yield _lib
    assert _lib.device_error() == 0


@pytest.mark.parametrize("N,K", [(600, 3584), (9, 64)])
def test_host_and_device_quantizers_agree(lib, N, K):
    import torch
    g = wl.rng(N * 7 + K)
    W = wl.weights(g, N, K, 0.03)
    W[1, :40] = 0.0
    Wd = dev(W)
    packed_h, sw_h = lib.w4_quantize_rows_host(W)
    packed = torch.empty((N, K // 8), dtype=torch.int32, device="cuda")
    sw = torch.empty(N, dtype=torch.float32, device="cuda")
    lib.w4_quantize_rows(Wd, packed, sw)
    assert np.array_equal(host(packed).view(np.uint32), packed_h)
    assert np.array_equal(host(sw).view(np.uint32), sw_h.view(np.uint32))
    blocks = torch.empty((N, K // 32, 18), dtype=torch.uint8, device="cuda")
    lib.q4_0_quantize(Wd, blocks)
    assert np.array_equal(host(blocks), lib.q4_0_quantize_host(W))
    q = torch.empty((N, K), dtype=torch.int8, device="cuda")
    d = torch.empty((N, K // 32), dtype=torch.int16, device="cuda")
    lib.i8g32_quantize(Wd, q, d)
    q_h, d_h = lib.i8g32_quantize_host(W)
    assert np.array_equal(host(q), q_h)
    assert np.array_equal(host(d).view(np.uint16), d_h)


@pytest.mark.parametrize("nbytes", [64 << 20, (3 << 20) + 4096 * 5 + 48, 16])
def test_hbm_read_checksum(lib, nbytes):
    import torch
    g = wl.rng(nbytes % 1000)
    words = g.integers(0, 2**32, size=nbytes // 4, dtype=np.uint64).astype(np.uint32)
    buf = dev(words.view(np.int32))
    sink = torch.full((1,), 12345, dtype=torch.int32, device="cuda")
    expect = int(np.bitwise_xor.reduce(words))
    for _ in range(2):                          # the sink is cleared by every call
        lib.hbm_read(buf, sink)
        assert int(host(sink).view(np.uint32)[0]) == expect


def test_last_device_error_alias(lib):
    assert lib.last_device_error() == lib.device_error() == 0


@pytest.mark.parametrize("cluster", [False, True])
def test_wait_timeout_sets_the_error_word_and_the_context_survives(lib, cluster):
    import time

    import torch
    lib.clear_device_error()
    t0 = time.perf_counter()
    lib.selftest_wait_timeout(cluster, 2000)
    torch.cuda.synchronize()
    assert time.perf_counter() - t0 < 5.0                     # the wait gave up by itself
    assert lib.device_error() == lib.WAIT_TIMEOUT_CODE
    lib.clear_device_error()
    # the context is usable: a GEMV on codes right after gives the oracle's sums
    g = wl.rng(4242)
    M, N, K = 2, 64, 256
    q = wl.int_codes(g, (N, K), -8, 7)
    qx = wl.int_codes(g, (M, K), -127, 127)
    w = torch.empty(lib.w4_repacked_bytes(N, K), dtype=torch.uint8, device="cuda")
    lib.w4_repack([dev(oracle.pack_int4(q).view(np.int32))], K, w)
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    lib.w4a8_gemv(w, dev(np.ones(N, np.float32)), None, dev(qx), dev(np.ones(M, np.float32)), y)
    assert np.array_equal(host(y), oracle.gemv_w4a8_acc(oracle.pack_int4(q), qx).astype(np.float32))
    assert lib.device_error() == 0
