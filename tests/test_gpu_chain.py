"""The chained decode-linear launch (w4a8_linear_chain) against per-linear
launches and the oracle.  Chains compute every linear exactly as
w4a8_linear does (same tiling, same reduction order), so outputs must be
bit-identical; with each input aliasing the previous output the chain must
still order every read after the producing linear."""
import numpy as np
import pytest

import oracle
from bit_quantized_decode_gb300 import workloads as wl
from helpers import RTOL_W4, check_close, cuda_ok, dev, host, w4_scale

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not cuda_ok(), reason="needs a CUDA GPU")]


@pytest.fixture(scope="module")
def lib():
    from bit_quantized_decode_gb300 import _lib
    _lib.load()
    _lib.clear_device_error()
    yield _lib
    assert _lib.device_error() == 0


def _linear(lib, g, N, K):
    import torch
    q = wl.int_codes(g, (N, K), -8, 7)
    sw = wl.positive_scales(g, N, 1e-3, 3e-3)
    b = wl.bias(g, N)
    w = torch.empty(lib.w4_repacked_bytes(N, K), dtype=torch.uint8, device="cuda")
    lib.w4_repack([dev(oracle.pack_int4(q).view(np.int32))], K, w)
    return q, sw, b, w, dev(sw), dev(b)


@pytest.mark.parametrize("M", [1, 2, 3, 4])
def test_chain_matches_single_launches_and_oracle(lib, M):
    import torch
    g = wl.rng(40 + M)
    shapes = [(4608, 3584), (3584, 3584), (1000, 3584), (3584, 18944), (13, 64), (512, 3584)]
    lins = [_linear(lib, g, N, K) for N, K in shapes]
    xs = [dev(wl.activations(g, M, K, outliers=True)) for _, K in shapes]
    ys = [torch.full((M, N), float("nan"), device="cuda") for N, _ in shapes]
    qxs = [torch.empty((M, K), dtype=torch.int8, device="cuda") for _, K in shapes]
    sxs = [torch.empty(M, dtype=torch.float32, device="cuda") for _ in shapes]
    descs = lib.make_chain_descs([(L[3], L[4], L[5], x, y, qx, sx) for L, x, y, qx, sx in zip(lins, xs, ys, qxs, sxs)])
    ws = torch.zeros(lib.chain_workspace_bytes(), dtype=torch.uint8, device="cuda")
    lib.w4a8_linear_chain(descs, M, ws)
    torch.cuda.synchronize()
    for (q, sw, b, w, swd, bd), x, y, qx, sx, (N, K) in zip(lins, xs, ys, qxs, sxs, shapes):
        y1 = torch.empty((M, N), device="cuda")
        q1 = torch.empty((M, K), dtype=torch.int8, device="cuda")
        s1 = torch.empty(M, device="cuda")
        lib.w4a8_linear(w, swd, bd, x, y1, q1, s1)
        assert np.array_equal(host(y).view(np.uint32), host(y1).view(np.uint32))
        y_ref, qx_ref, sx_ref, acc = oracle.w4a8_linear(oracle.pack_int4(q), sw, host(x), b)
        assert np.array_equal(host(qx), qx_ref) and np.array_equal(host(sx).view(np.uint32), sx_ref.view(np.uint32))
        check_close(host(y), y_ref, w4_scale(acc, sw, sx_ref, b), RTOL_W4, f"chain {N}x{K}")
    # the workspace's arrival count is back to zero, ready for the next call
    assert host(ws.view(torch.int32)).tolist() == [0] * (ws.numel() // 4)


@pytest.mark.parametrize("M", [1, 3])
def test_true_chain_aliasing_outputs_as_inputs(lib, M):
    """One buffer holds every activation: linear i writes rows of it that linear i+1 reads."""
    import torch
    g = wl.rng(90 + M)
    Ks = [3584, 3584, 3584, 3584, 3584]
    shapes = [(3584, 3584)] * 5
    lins = [_linear(lib, g, N, K) for N, K in shapes]
    bufs = [dev(wl.activations(g, M, 3584))] + [torch.zeros((M, 3584), device="cuda") for _ in shapes]
    descs = lib.make_chain_descs([(L[3], L[4], L[5], bufs[i], bufs[i + 1], None, None) for i, L in enumerate(lins)])
    ws = torch.zeros(lib.chain_workspace_bytes(), dtype=torch.uint8, device="cuda")
    for _ in range(3):                    # the workspace is reused across calls
        lib.w4a8_linear_chain(descs, M, ws)
    torch.cuda.synchronize()
    x = bufs[0]
    for i, (q, sw, b, w, swd, bd) in enumerate(lins):
        y1 = torch.empty((M, 3584), device="cuda")
        lib.w4a8_linear(w, swd, bd, x, y1, torch.empty((M, 3584), dtype=torch.int8, device="cuda"),
                        torch.empty(M, device="cuda"))
        assert np.array_equal(host(bufs[i + 1]).view(np.uint32), host(y1).view(np.uint32)), i
        # and against the oracle on the same fp32 input
        y_ref, _, sx_ref, acc = oracle.w4a8_linear(oracle.pack_int4(q), sw, host(x), b)
        check_close(host(y1), y_ref, w4_scale(acc, sw, sx_ref, b), RTOL_W4, f"link {i}")
        x = y1


@pytest.mark.parametrize("prefetch_kb,stages", [(1, 2), (64, 3), (4096, 0)])
def test_chain_producer_limits(lib, prefetch_kb, stages):
    """The weight stream of the chain with two ring slots per warp and no L2
    prefetch, with a short lookahead, and with a 4 MB lookahead per block
    (past the end of the chain): the outputs stay bit-identical to single
    launches.  A linear with 80000 rows takes two rounds per block and more
    rows than the staged per-row parameters."""
    import torch
    lib.set_tuning("chain_prefetch_kb", prefetch_kb)
    lib.set_tuning("max_stages", stages)
    try:
        M = 1
        g = wl.rng(300 + prefetch_kb + stages)
        shapes = [(80000, 64), (3584, 18944), (13, 64), (4608, 3584)]
        lins = [_linear(lib, g, N, K) for N, K in shapes]
        xs = [dev(wl.activations(g, M, K)) for _, K in shapes]
        ys = [torch.full((M, N), float("nan"), device="cuda") for N, _ in shapes]
        descs = lib.make_chain_descs([(L[3], L[4], L[5], x, y, None, None) for L, x, y in zip(lins, xs, ys)])
        ws = torch.zeros(lib.chain_workspace_bytes(), dtype=torch.uint8, device="cuda")
        for _ in range(2):
            lib.w4a8_linear_chain(descs, M, ws)
        torch.cuda.synchronize()
        for (q, sw, b, w, swd, bd), x, y, (N, K) in zip(lins, xs, ys, shapes):
            y1 = torch.empty((M, N), device="cuda")
            lib.w4a8_linear(w, swd, bd, x, y1, torch.empty((M, K), dtype=torch.int8, device="cuda"),
                            torch.empty(M, device="cuda"))
            assert np.array_equal(host(y).view(np.uint32), host(y1).view(np.uint32)), (N, K)
        assert host(ws.view(torch.int32)).tolist() == [0] * (ws.numel() // 4)
    finally:
        lib.set_tuning("chain_prefetch_kb", 0)
        lib.set_tuning("max_stages", 0)
