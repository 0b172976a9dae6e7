// Host-side weight quantizers of the C ABI (w4_quantize_rows_host,
// q4_0_quantize_host, i8g32_quantize_host): plain C++ over host memory for
// loaders that hold float weights on the host.  Every decision is the one the
// device kernels take (prep_kernels.cu): IEEE fp32 division, round half to
// even to an integer, and fp16 scales rounded to nearest even, so the bytes
// are identical.  Compiled without contraction or fast math.
#include <cmath>
#include <cstdint>
#include <cstring>

#include "../../include/w4a8.h"

namespace {

uint32_t bits_of(float f)
{
    uint32_t u;
    std::memcpy(&u, &f, 4);
    return u;
}

float float_of(uint32_t u)
{
    float f;
    std::memcpy(&f, &u, 4);
    return f;
}

// Round the significand bits r >> shift to nearest, ties to even.
uint32_t round_shift(uint32_t r, int shift)
{
    const uint32_t q = r >> shift;
    const uint32_t rem = r & ((1u << shift) - 1u);
    const uint32_t half = 1u << (shift - 1);
    return (rem > half || (rem == half && (q & 1u))) ? q + 1u : q;
}

// IEEE binary32 -> binary16, round to nearest even (a carry out of the
// significand moves into the exponent field, which is the correct encoding).
uint16_t to_half(float f)
{
    const uint32_t u = bits_of(f);
    const uint32_t sign = (u >> 16) & 0x8000u;
    const uint32_t a = u & 0x7fffffffu;
    if (a >= 0x7f800000u) return static_cast<uint16_t>(sign | (a > 0x7f800000u ? 0x7e00u : 0x7c00u));
    if (a >= 0x477ff000u) return static_cast<uint16_t>(sign | 0x7c00u);    // >= 65520 rounds to infinity
    if (a >= 0x38800000u)                                                  // a normal half: rebias by 127 - 15
        return static_cast<uint16_t>(sign | round_shift(a - 0x38000000u, 13));
    const int e = static_cast<int>(a >> 23);
    if (e < 102) return static_cast<uint16_t>(sign);                       // below 2^-25: zero
    // subnormal half: the value in units of 2^-24 (may round up to 0x400, the least normal)
    const uint32_t m = (a & 0x7fffffu) | 0x800000u;
    return static_cast<uint16_t>(sign | round_shift(m, 126 - e));
}

// IEEE binary16 -> binary32 (exact).
float from_half(uint16_t h)
{
    const uint32_t sign = static_cast<uint32_t>(h & 0x8000u) << 16;
    const uint32_t e = (h >> 10) & 0x1fu;
    const uint32_t m = h & 0x3ffu;
    if (e == 0x1f) return float_of(sign | 0x7f800000u | (m << 13));
    if (e != 0) return float_of(sign | ((e + 112u) << 23) | (m << 13));
    // zero or subnormal: m * 2^-24, exact in binary32
    const float v = static_cast<float>(m) * float_of(0x33800000u);
    return sign ? -v : v;
}

// clip(rint(v / s), lo, hi) in fp32; s == 0 gives 0.
int quant_code(float v, float s, int lo, int hi)
{
    if (s == 0.0f) return 0;
    const float t = std::rint(v / s);
    if (t != t) return 0;                              // a NaN quotient converts to 0, as on the device
    if (t > static_cast<float>(hi)) return hi;
    if (t < static_cast<float>(lo)) return lo;
    return static_cast<int>(t);
}

float abs_max(const float* v, int n)
{
    float mx = 0.0f;
    for (int i = 0; i < n; ++i) mx = std::fmax(mx, std::fabs(v[i]));
    return mx;
}

w4_status check(const float* W, int N, int K, int kmod, const void* o1, const void* o2)
{
    if (N < 0 || K <= 0) return W4_ERR_INVALID_ARG;
    if (K % kmod != 0) return W4_ERR_UNSUPPORTED_SHAPE;
    if (N == 0) return W4_OK;
    if (!W || !o1 || !o2) return W4_ERR_INVALID_ARG;
    return W4_OK;
}

}  // namespace

extern "C" {

// "Jetson Orin AGX INT4 推理优化实践", §"从 FP 线性层到 INT4 DP4A 的数学推导":
// s_w = max|W_j| / 7, q = clip(rint(W / s_w), -8, 7), weight k of a word in
// bits 4k..4k+3 (§"DP4A 做了什么").
w4_status w4_quantize_rows_host(const float* W, int N, int K, uint32_t* packed, float* s_w)
{
    const w4_status st = check(W, N, K, 8, packed, s_w);
    if (st != W4_OK || N == 0) return st;
    for (int j = 0; j < N; ++j) {
        const float* row = W + static_cast<size_t>(j) * K;
        const float s = abs_max(row, K) / 7.0f;
        s_w[j] = s;
        uint32_t* out = packed + static_cast<size_t>(j) * (K / 8);
        for (int w = 0; w < K / 8; ++w) {
            uint32_t word = 0;
            for (int k = 0; k < 8; ++k)
                word |= (static_cast<uint32_t>(quant_code(row[8 * w + k], s, -8, 7)) & 0xfu) << (4 * k);
            out[w] = word;
        }
    }
    return W4_OK;
}

// "在香橙派上跑 Gemma4", §3.1: 18-byte blocks of 32 weights, fp16 d =
// fp16(max|w| / 8) little endian, then byte i = n_i | n_{i+16} << 4 with
// n = clip(rint(w / d), -8, 7) + 8 against the stored d.
w4_status q4_0_quantize_host(const float* W, int N, int K, uint8_t* blocks)
{
    const w4_status st = check(W, N, K, 32, blocks, blocks);
    if (st != W4_OK || N == 0) return st;
    const size_t nb = static_cast<size_t>(N) * (K / 32);
    for (size_t b = 0; b < nb; ++b) {
        const float* v = W + b * 32;
        const uint16_t dh = to_half(abs_max(v, 32) / 8.0f);
        const float d = from_half(dh);
        uint8_t* blk = blocks + b * 18;
        blk[0] = static_cast<uint8_t>(dh & 0xffu);
        blk[1] = static_cast<uint8_t>(dh >> 8);
        for (int i = 0; i < 16; ++i) {
            const uint32_t lo = static_cast<uint32_t>(quant_code(v[i], d, -8, 7) + 8);
            const uint32_t hi = static_cast<uint32_t>(quant_code(v[i + 16], d, -8, 7) + 8);
            blk[2 + i] = static_cast<uint8_t>(lo | (hi << 4));
        }
    }
    return W4_OK;
}

// "在香橙派上跑 Gemma4", §3.2 (int8 weights, one fp16 scale per group of 32):
// d = fp16(max|w| / 32), q = clip(rint(w / d), -32, 31).
w4_status i8g32_quantize_host(const float* W, int N, int K, int8_t* q, uint16_t* d)
{
    const w4_status st = check(W, N, K, 32, q, d);
    if (st != W4_OK || N == 0) return st;
    const size_t nb = static_cast<size_t>(N) * (K / 32);
    for (size_t b = 0; b < nb; ++b) {
        const float* v = W + b * 32;
        const uint16_t dh = to_half(abs_max(v, 32) / 32.0f);
        const float df = from_half(dh);
        d[b] = dh;
        for (int i = 0; i < 32; ++i) q[b * 32 + i] = static_cast<int8_t>(quant_code(v[i], df, -32, 31));
    }
    return W4_OK;
}

}  // extern "C"
