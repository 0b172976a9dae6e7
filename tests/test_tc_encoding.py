"""The operand encoding of the tensor-core GEMV, checked on the host.

The tensor-core path (kind::f8f6f4, e4m3 operands) is exact only if its bit
manipulations produce e4m3 bytes whose values are the integers it means,
scaled by 2^-9, and if every partial sum stays exactly representable in fp32.
These tests restate the kernel's byte manipulations and check them against an
e4m3 decoder written from the OCP 8-bit floating point definition (sign bit,
4 exponent bits with bias 7, 3 mantissa bits, subnormals at exponent 0; the
value of S.1111.111 is NaN).  The GPU parity tests check the same path end to
end (bit-exact accumulators).
"""
import numpy as np


def e4m3_value(byte: int) -> float:
    s = -1.0 if byte & 0x80 else 1.0
    e = (byte >> 3) & 0xF
    m = byte & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:
        return s * (m / 8.0) * 2.0 ** -6
    return s * (1.0 + m / 8.0) * 2.0 ** (e - 7)


def split4(c: int):
    """The kernel's split of four int8 codes (one 32-bit word) into the e4m3
    bytes of h = x >> 4 (sign-magnitude) and l = x & 15."""
    lo = c & 0x0F0F0F0F
    u = (c >> 4) & 0x0F0F0F0F                      # h + 16 for negative h
    bm = ((u & 0x08080808) >> 3) * 0xFF            # 0xFF in the bytes of negative h
    m = ((u ^ (bm & 0x0F0F0F0F)) + (bm & 0x01010101)) & 0xFFFFFFFF
    hi = m | (bm & 0x80808080)
    return hi & 0xFFFFFFFF, lo


def nibbles_to_e4m3(word: int):
    """The kernel's two masks: the low and the high nibble of each byte of a
    word of biased nibbles, each as an e4m3 byte."""
    return word & 0x0F0F0F0F, (word >> 4) & 0x0F0F0F0F


def bytes_of(w: int):
    return [(w >> (8 * i)) & 0xFF for i in range(4)]


def test_biased_nibbles_are_e4m3_multiples_of_2_to_the_minus_9():
    for n in range(16):
        assert e4m3_value(n) == n * 2.0 ** -9
    rng = np.random.default_rng(3)
    for w in rng.integers(0, 2 ** 32, size=2000, dtype=np.uint64):
        w = int(w)
        a, b = nibbles_to_e4m3(w)
        for i, (x, y) in enumerate(zip(bytes_of(a), bytes_of(b))):
            byte = (w >> (8 * i)) & 0xFF
            assert e4m3_value(x) == (byte & 15) * 2.0 ** -9
            assert e4m3_value(y) == (byte >> 4) * 2.0 ** -9


def test_code_split_is_exact_for_every_int8():
    for x in range(-128, 128):
        h, l = x >> 4, x & 15
        assert x == 16 * h + l and -8 <= h <= 7 and 0 <= l <= 15
        # the same code in every byte position of a word, and beside other codes
        for pos in range(4):
            word = ((x & 0xFF) << (8 * pos)) | (0x7F << (8 * ((pos + 1) % 4)))
            hi, lo = split4(word)
            assert e4m3_value(bytes_of(hi)[pos]) == h * 2.0 ** -9
            assert e4m3_value(bytes_of(lo)[pos]) == l * 2.0 ** -9
    rng = np.random.default_rng(4)
    for w in rng.integers(0, 2 ** 32, size=2000, dtype=np.uint64):
        hi, lo = split4(int(w))
        for b, hb, lb in zip(bytes_of(int(w)), bytes_of(hi), bytes_of(lo)):
            x = b - 256 if b >= 128 else b
            assert e4m3_value(hb) == (x >> 4) * 2.0 ** -9 and e4m3_value(lb) == (x & 15) * 2.0 ** -9


def test_partial_sums_stay_exact_in_fp32():
    """Products n h 2^-18 and n l 2^-18 are multiples of 2^-18; a split of at
    most 16384 K keeps every partial sum below 64 in magnitude, where fp32
    (24-bit significand) holds every multiple of 2^-18 exactly."""
    max_split_k = 16384
    worst = max(15 * 15, 15 * 8) * max_split_k * 2.0 ** -18
    assert worst < 64
    # fp32 represents every multiple of 2^-18 in [0, 64) exactly
    ks = np.array([0, 1, 2 ** 23, 2 ** 24 - 1], dtype=np.float64)
    assert np.all(np.float32(ks * 2.0 ** -18).astype(np.float64) == ks * 2.0 ** -18)
    # an fp32 running sum of the worst products reaches the exact total
    n, l = 15, 15
    acc = np.float32(0.0)
    step = np.float32(n * l * 2.0 ** -18)
    for _ in range(max_split_k):
        acc = np.float32(acc + step)
    assert float(acc) == n * l * max_split_k * 2.0 ** -18
    # the epilogue's integer: 16 S_h + S_l - 8 sum x, times 2^18 each, in int32
    assert 16 * 15 * 8 * max_split_k + 15 * 15 * max_split_k + 8 * 127 * max_split_k < 2 ** 31
