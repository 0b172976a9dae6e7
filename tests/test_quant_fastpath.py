"""The activation quantizer's fast path, checked on the host in IEEE fp32.

The definition of a code is q = clip(rint(fl(x / s)), -127, 127) with
s = fl(max|x| / 127) and the quotient rounded to fp32 once.  The kernels
instead form t = fl(x * fl(1 / s)), round it with the 1.5 * 2^23 addition, and
fall back to the IEEE quotient when d = t - rint(t) satisfies
d^2 >= fl(0.49997^2) (a possible tie).  The claim is that whenever the
fallback is not taken, the fast code equals the definition.  numpy float32
arithmetic rounds each operation to nearest even, as the kernels' .rn
operations do, so the fast path is restated here operation by operation and
compared with the definition on random tokens and on values built to sit
exactly at, and one ulp either side of, every half-integer quotient.
"""
import numpy as np

F = np.float32
BIG = F(12582912.0)                 # 1.5 * 2^23
TIE2 = F(0.2499700009)              # fl(0.49997^2), the kernels' constant


def definition(x, s):
    q = np.rint((x / s).astype(np.float32))
    return np.clip(q, -127, 127).astype(np.int32)


def fast_path(x, s):
    """Codes and the 'no tie' flag of the packed fast path."""
    r = (F(1.0) / s).astype(np.float32)
    t = (x * r).astype(np.float32)
    big = (t + BIG).astype(np.float32)
    rt = (big - BIG).astype(np.float32)
    d = t.astype(np.float64) - rt.astype(np.float64)         # exact: t and rint(t) are close fp32 values
    ok = d * d < np.float64(TIE2)                            # the sign of the kernels' FMA d*d - TIE2
    code = rt.astype(np.int32)
    return code, ok


def check(x, s):
    q_ref = definition(x, s)
    q, ok = fast_path(x, s)
    assert np.all(q[ok] == q_ref[ok]), (x[ok][q[ok] != q_ref[ok]][:5], s)
    return ok


def test_random_tokens():
    rng = np.random.default_rng(11)
    taken = 0
    total = 0
    for scale in (1e-3, 1.0, 37.0, 1e4):
        for _ in range(40):
            x = (rng.standard_normal(3584) * scale).astype(np.float32)
            x[rng.integers(0, 3584, 4)] *= F(20.0)
            s = (np.abs(x).max() / F(127.0)).astype(np.float32)
            ok = check(x, s)
            taken += int(ok.sum())
            total += ok.size
    assert taken > 0.999 * total          # the fallback is rare


def test_values_at_and_beside_every_half_integer_quotient():
    rng = np.random.default_rng(12)
    close = fallback = 0
    for _ in range(200):
        amax = F(rng.uniform(0.01, 100.0))
        s = (amax / F(127.0)).astype(np.float32)
        k = np.arange(-127, 127, dtype=np.float64) + 0.5
        base = (k * np.float64(s)).astype(np.float32)
        xs = [base]
        up = dn = base
        for _ in range(3):                 # three ulps up and three down
            up = np.nextafter(up, np.float32(np.inf))
            dn = np.nextafter(dn, np.float32(-np.inf))
            xs += [up, dn]
        x = np.concatenate(xs).astype(np.float32)
        x = x[np.abs(x) <= amax]
        ok = check(x, s)
        # the fast path was taken for some values within 1e-4 of a half-integer quotient
        quot = x.astype(np.float64) / np.float64(s)
        dist = np.abs(quot - np.floor(quot) - 0.5)
        close += int((ok & (dist < 1e-4)).sum())
        fallback += int((~ok).sum())
    assert close > 0 and fallback > 0


def test_margin_covers_the_reciprocal_error():
    """|fl(x fl(1/s)) - x/s| <= |x/s| (2^-24 + 2^-24 + 2^-48) <= 1.6e-5 for
    |x/s| <= 128, and fl(x/s) is within 2^-18 of x/s there: both below the
    3e-5 margin the tie test keeps (0.5 - 0.49997)."""
    bound = 128 * (2.0 ** -24 + 2.0 ** -24 + 2.0 ** -48)
    assert bound < 1.6e-5 and bound + 2.0 ** -18 < 0.5 - np.sqrt(np.float64(TIE2))
