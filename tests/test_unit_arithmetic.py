"""The GEMV inner loops' integer identities, checked on the host.

For one 32-weight unit (the device layouts documented in include/w4a8.h) and
32 int8 codes, the kernels form the exact group sum sum_i q_i x_i from DP4A on
masked bytes:
  W4     biased nibbles n = q + 8:  B + A / 16 - 8 sum x,  B = sum of low
         nibbles times codes, A = sum of high nibbles (kept in place, i.e.
         times 16) times codes (dp4a with unsigned weight bytes);
  Q4_0   4-bit two's complement: 16 sum q x from signed bytes
         (w << 4) & 0xF0F0F0F0 and w & 0xF0F0F0F0;
  Q6G32  n = q + 32 = lo + 16 hi: the W4 sums on the low plane, plus 16 times
         the 2-bit high parts summed by class, minus 32 sum x;
and the weight-only paths turn a byte into fp32 by placing it in the mantissa
of 2^23.  Each is restated operation by operation and compared with the
int64 dot product.  The GPU parity tests check the kernels end to end.
"""
import numpy as np


def sbytes(w: int):
    return [((w >> (8 * i)) & 0xFF) - (256 if (w >> (8 * i)) & 0x80 else 0) for i in range(4)]


def ubytes(w: int):
    return [(w >> (8 * i)) & 0xFF for i in range(4)]


def dp4a_us(a: int, b: int, c: int) -> int:
    """dp4a.u32.s32: unsigned bytes of a times signed bytes of b, plus c."""
    return c + sum(x * y for x, y in zip(ubytes(a), sbytes(b)))


def dp4a_ss(a: int, b: int, c: int) -> int:
    return c + sum(x * y for x, y in zip(sbytes(a), sbytes(b)))


def words(b: np.ndarray):
    """Little-endian 32-bit words of a byte array."""
    return [int(v) for v in b.astype(np.uint8).view("<u4")]


def nibble_unit(vals):
    """16-byte unit: word w holds weight 8w+b in the low nibble of byte b and
    weight 8w+4+b in the high nibble (vals already 0..15)."""
    out = np.zeros(16, np.uint8)
    for w in range(4):
        for b in range(4):
            out[4 * w + b] = (vals[8 * w + b] & 15) | ((vals[8 * w + 4 + b] & 15) << 4)
    return words(out)


def high_plane(hi):
    """8-byte unit of 2-bit high parts: weight 16h+4s+b in bits 2s..2s+1 of
    byte b of word h."""
    out = np.zeros(8, np.uint8)
    for h in range(2):
        for s in range(4):
            for b in range(4):
                out[4 * h + b] |= (hi[16 * h + 4 * s + b] & 3) << (2 * s)
    return words(out)


def unit4(w, x):
    B = A = 0
    for k in range(4):
        B = dp4a_us(w[k] & 0x0F0F0F0F, x[2 * k], B)
        A = dp4a_us(w[k] & 0xF0F0F0F0, x[2 * k + 1], A)
    return B, A


def bytesum(v: int) -> int:
    return sum(sbytes(v))


def rand_case(rng, lo, hi):
    q = rng.integers(lo, hi + 1, size=32)
    x = rng.integers(-127, 128, size=32)
    return q, x, words(x.astype(np.int8).view(np.uint8))


def test_w4_biased_nibbles():
    rng = np.random.default_rng(21)
    cases = [rand_case(rng, -8, 7) for _ in range(300)]
    cases.append((np.full(32, -8), np.full(32, 127), words(np.full(32, 127, np.int8).view(np.uint8))))
    for q, x, xw in cases:
        w = nibble_unit(q + 8)
        B, A = unit4(w, xw)
        assert A % 16 == 0
        assert B + (A >> 4) - 8 * sum(bytesum(v) for v in xw) == int(np.dot(q, x))


def test_q4_0_signed_nibbles():
    rng = np.random.default_rng(22)
    for q, x, xw in [rand_case(rng, -8, 7) for _ in range(300)]:
        w = nibble_unit(q & 15)                       # two's complement nibbles
        g = 0
        for k in range(4):
            g = dp4a_ss((w[k] << 4) & 0xF0F0F0F0, xw[2 * k], g)
            g = dp4a_ss(w[k] & 0xF0F0F0F0, xw[2 * k + 1], g)
        assert g % 16 == 0 and g >> 4 == int(np.dot(q, x))


def test_q6g32_planes():
    rng = np.random.default_rng(23)
    cases = [rand_case(rng, -32, 31) for _ in range(300)]
    cases.append((np.full(32, 31), np.full(32, -127), words(np.full(32, -127, np.int8).view(np.uint8))))
    for q, x, xw in cases:
        n = q + 32
        w = nibble_unit(n & 15)
        hv = high_plane(n >> 4)
        B, A = unit4(w, xw)
        s0 = dp4a_us(hv[1] & 0x03030303, xw[4], dp4a_us(hv[0] & 0x03030303, xw[0], 0))
        s1 = dp4a_us(hv[1] & 0x0C0C0C0C, xw[5], dp4a_us(hv[0] & 0x0C0C0C0C, xw[1], 0))
        s2 = dp4a_us(hv[1] & 0x30303030, xw[6], dp4a_us(hv[0] & 0x30303030, xw[2], 0))
        s3 = dp4a_us(hv[1] & 0xC0C0C0C0, xw[7], dp4a_us(hv[0] & 0xC0C0C0C0, xw[3], 0))
        hs = s0 + (s1 >> 2) + (s2 >> 4) + (s3 >> 6)
        g = B + (A >> 4) + 16 * hs - 32 * sum(bytesum(v) for v in xw)
        assert g == int(np.dot(q, x))


def test_weight_only_byte_to_float():
    b = np.arange(256, dtype=np.uint32)
    f = (np.uint32(0x4B000000) | b).view(np.float32)      # 2^23 + byte, exactly
    assert np.array_equal(f.astype(np.float64), 2.0 ** 23 + b)
    # W4F: a nibble n = q + 8 minus fl(2^23 + 8) is q; W8F: (q ^ 0x80) minus fl(2^23 + 128) is q
    w4 = (f[:16] + np.float32(-8388616.0)).astype(np.float32)
    assert np.array_equal(w4, np.arange(-8, 8, dtype=np.float32))
    q8 = np.arange(-128, 128)
    biased = (q8.astype(np.int8).view(np.uint8) ^ 0x80).astype(np.uint32)
    w8 = ((np.uint32(0x4B000000) | biased).view(np.float32) + np.float32(-8388736.0)).astype(np.float32)
    assert np.array_equal(w8, q8.astype(np.float32))
