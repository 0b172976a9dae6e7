"""The RMSNorm's sum of squares, checked on the host.

The definition takes S = sum_i x_i^2 rounded once to fp32 from its exact
value.  The fused prologue gets it from a compensated (hi, lo) pair of fp32
per thread: each square split exactly into fl(x^2) and its FMA error, hi
accumulated through an error-free sum, the small parts added into lo; then a
butterfly over the warp and a merge over the eight warps in warp order, and
S = fl(hi + lo).  Its error stays near d^2 2^-48 of S for a reduction of
depth d, so it returns the exactly rounded S except when S lies that close to
an fp32 rounding boundary.  The reduction tree (256 threads, float4 i = t +
256 k per thread, x y z w in order) is replayed here in numpy fp32, whose
operations round to nearest even as the kernels' do, and compared with the
exact sum rounded once (rational arithmetic).
"""
from fractions import Fraction

import numpy as np

F = np.float32
THREADS = 256


def two_sum(a, b):
    s = (a + b).astype(F)
    bp = (s - a).astype(F)
    e = ((a - (s - bp).astype(F)).astype(F) + (b - bp).astype(F)).astype(F)
    return s, e


def sq_acc(x, hi, lo):
    p = (x * x).astype(F)
    pe = (x.astype(np.float64) * x.astype(np.float64) - p.astype(np.float64)).astype(F)   # fma(x, x, -p): exact
    s, e = two_sum(hi, p)
    return s, (lo + (e + pe).astype(F)).astype(F)


def pair_merge(hi, lo, hi2, lo2):
    s, e = two_sum(hi, hi2)
    return s, (lo + (lo2 + e).astype(F)).astype(F)


def kernel_sum(x):
    K4 = x.size // 4
    nit = -(-K4 // THREADS)
    v = np.zeros(nit * THREADS * 4, F)
    v[: x.size] = x
    v = v.reshape(nit, THREADS, 4)                 # [it][thread][component]
    hi = np.zeros(THREADS, F)
    lo = np.zeros(THREADS, F)
    for it in range(nit):
        for c in range(4):
            hi, lo = sq_acc(v[it, :, c], hi, lo)
    hi = hi.reshape(8, 32)
    lo = lo.reshape(8, 32)
    lanes = np.arange(32)
    for off in (16, 8, 4, 2, 1):                   # every lane merges its partner's pair
        hi, lo = pair_merge(hi, lo, hi[:, lanes ^ off], lo[:, lanes ^ off])
    h, l = hi[0, :1], lo[0, :1]
    for w in range(1, 8):
        h, l = pair_merge(h, l, hi[w, :1], lo[w, :1])
    return F((h + l).astype(F)[0])


def exact_rounded(x):
    """sum x^2 exactly, then rounded once to fp32 (nearest, ties to even)."""
    S = sum(Fraction(float(v)) ** 2 for v in x)
    f = F(float(S))
    cands = [np.nextafter(f, F(-np.inf)), f, np.nextafter(f, F(np.inf))]
    best = min(cands, key=lambda c: (abs(Fraction(float(c)) - S), int(np.array(c).view(np.uint32)) & 1))
    return F(best), S


def test_compensated_sum_is_the_exactly_rounded_sum():
    rng = np.random.default_rng(31)
    near = 0
    for K in (96, 1536, 3584, 10240):
        for trial in range(12):
            x = (rng.standard_normal(K) * rng.choice([1e-3, 1.0, 4.0, 300.0])).astype(F)
            if trial % 3 == 0:
                x[rng.integers(0, K, 3)] *= F(50.0)
            got = kernel_sum(x)
            want, S = exact_rounded(x)
            if got != want:
                # allowed only within the pair's error of a rounding boundary
                mid = (Fraction(float(got)) + Fraction(float(want))) / 2
                assert abs(S - mid) <= S * Fraction(2) ** -36, (K, trial, got, want)
                near += 1
    assert near <= 1


def test_plain_fp32_accumulation_would_not_be_exact():
    """The same tree with plain fp32 adds misses the exactly rounded sum on
    these inputs, so the comparison above can tell the two apart."""
    rng = np.random.default_rng(32)
    misses = 0
    for _ in range(20):
        x = rng.standard_normal(3584).astype(F)
        want, _ = exact_rounded(x)
        v = np.zeros(4 * 256 * 4, F)
        v[: x.size] = x
        part = np.zeros(256, F)
        for it in range(4):
            for c in range(4):
                q = v.reshape(4, 256, 4)[it, :, c]
                part = (part + (q * q).astype(F)).astype(F)
        total = F(0)
        for p in part:
            total = F(total + p)
        misses += int(total != want)
    assert misses > 0
