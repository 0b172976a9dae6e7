"""The chain entry point that allocates nothing (w4a8_linear_chain_noalloc).

Some callers cannot allocate device memory where they call the library: an
engine whose memory planner owns every allocation, or code that must not call
cudaMalloc while a stream is captured into a CUDA graph.  For them the chain
keeps its grid-barrier state in a fixed array inside the library.  Here the
outputs of that entry point, on two calls in a row, must agree with the
workspace entry point's within the tests' fp32 tolerance.  This file is
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
            _, _, sx, acc = oracle.w4a8_linear(oracle.pack_int4(q), sw, host(x), b)
            scale = w4_scale(acc, sw, sx, b)
            check_close(host(y), host(yr).astype(np.float64), scale, RTOL_W4, f"call {call}, {N}x{K}")
    assert _lib.device_error() == 0
