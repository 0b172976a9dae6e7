"""The chain entry point that allocates nothing (w4a8_linear_chain_noalloc).

Some callers cannot allocate device memory where they call the library: an
engine whose memory planner owns every allocation, or code that must not call
cudaMalloc while a stream is captured into a CUDA graph.  For them the chain
keeps its grid-barrier state in a fixed array inside the library.  Here the
outputs of that entry point, on two calls in a row, must agree with the
workspace entry point's bit for bit (the same kernel on the same inputs),
and the oracle's within the tests' fp32 tolerance.  A call with a bad
descriptor returns its error and leaves the next call unaffected.  This file is
collected last so that a run stopping at its first failure has run all else.
"""
import numpy as np
import pytest

import oracle
from bit_quantized_decode_gb300 import workloads as wl
from helpers import RTOL_W4, check_close, cuda_ok, dev, host, w4_scale

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not cuda_ok(), reason="needs a CUDA GPU")]


def test_chain_noalloc_matches_workspace_chain_twice():
    import torch

    from bit_quantized_decode_gb300 import _lib
    _lib.load()
    assert _lib.load().w4_chain_noalloc_scratch_bytes() >= _lib.chain_workspace_bytes()
    M = 2
    g = wl.rng(2024)
    shapes = [(4608, 3584), (3584, 3584), (3584, 18944), (1000, 3584)]
    lins = []
    for N, K in shapes:
        q = wl.int_codes(g, (N, K), -8, 7)
        sw = wl.positive_scales(g, N, 1e-3, 3e-3)
        b = wl.bias(g, N)
        w = torch.empty(_lib.w4_repacked_bytes(N, K), dtype=torch.uint8, device="cuda")
        _lib.w4_repack([dev(oracle.pack_int4(q).view(np.int32))], K, w)
        lins.append((q, sw, b, w, dev(sw), dev(b)))
    xs = [dev(wl.activations(g, M, K)) for _, K in shapes]

    def outputs():
        return [torch.full((M, N), float("nan"), device="cuda") for N, _ in shapes]

    # the existing entry point, with a caller workspace
    ref = outputs()
    descs = _lib.make_chain_descs([(L[3], L[4], L[5], x, y, None, None) for L, x, y in zip(lins, xs, ref)])
    ws = torch.zeros(_lib.chain_workspace_bytes(), dtype=torch.uint8, device="cuda")
    _lib.w4a8_linear_chain(descs, M, ws)
    torch.cuda.synchronize()

    for call in range(2):
        got = outputs()
        d2 = _lib.make_chain_descs([(L[3], L[4], L[5], x, y, None, None) for L, x, y in zip(lins, xs, got)])
        _lib.w4a8_linear_chain_noalloc(d2, M)
        torch.cuda.synchronize()
        for (q, sw, b, *_), x, y, yr, (N, K) in zip(lins, xs, got, ref, shapes):
            # the same kernel on the same inputs: bit for bit, and within the tests' tolerance of the oracle
            assert torch.equal(y, yr), f"call {call}, {N}x{K}"
            y_ref, _, sx, acc = oracle.w4a8_linear(oracle.pack_int4(q), sw, host(x), b)
            check_close(host(y), y_ref, w4_scale(acc, sw, sx, b), RTOL_W4, f"call {call}, {N}x{K}")
    assert _lib.device_error() == 0


def test_chain_noalloc_rejects_a_bad_descriptor_then_runs():
    """A call that fails its checks returns the status and enqueues nothing;
    the next valid call still matches the workspace chain."""
    import torch

    from bit_quantized_decode_gb300 import _lib
    _lib.load()
    M, N, K = 1, 1024, 3584
    g = wl.rng(77)
    q = wl.int_codes(g, (N, K), -8, 7)
    sw, b = wl.positive_scales(g, N, 1e-3, 3e-3), wl.bias(g, N)
    w = torch.empty(_lib.w4_repacked_bytes(N, K), dtype=torch.uint8, device="cuda")
    _lib.w4_repack([dev(oracle.pack_int4(q).view(np.int32))], K, w)
    x = dev(wl.activations(g, M, K))
    swd, bd = dev(sw), dev(b)
    bad = _lib.make_chain_descs([(w, swd, bd, x, torch.empty((M, N), device="cuda"), None, None)])
    bad[0].K = 48                                               # not a multiple of 32
    assert _lib.load().w4a8_linear_chain_noalloc(bad, 1, M, None) == 2
    ref = torch.empty((M, N), device="cuda")
    ws = torch.zeros(_lib.chain_workspace_bytes(), dtype=torch.uint8, device="cuda")
    _lib.w4a8_linear_chain(_lib.make_chain_descs([(w, swd, bd, x, ref, None, None)]), M, ws)
    got = torch.empty((M, N), device="cuda")
    _lib.w4a8_linear_chain_noalloc(_lib.make_chain_descs([(w, swd, bd, x, got, None, None)]), M)
    torch.cuda.synchronize()
    assert torch.equal(got, ref)
    assert _lib.device_error() == 0
