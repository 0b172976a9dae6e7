// Per-token INT8 activation code, q = clip(rint(x / s), -127, 127) with the
// quotient x / s rounded to fp32 first (IEEE division), as the definition
// ("Jetson Orin AGX INT4 推理优化实践", §"从 FP 线性层到 INT4 DP4A 的数学推导")
// is taken here.  Bit-identical to rintf(x / s) in IEEE fp32, but computed
// with one multiply by r = fl(1/s) except near ties:
//
//   |fl(x * r) - x / s| <= |x / s| * (2^-24 + 2^-24 + 2^-48) <= 1.6e-5 for
//   |x / s| <= 128, and fl(x / s) lies within half an ulp (<= 2^-18) of x / s.
//   So when t = fl(x * r) is farther than 3e-5 from every half-integer, t,
//   x / s and fl(x / s) all round to the same integer, and rint(t) is the
//   answer.  Otherwise (a possible tie, probability ~6e-5 for random data)
//   the exact quotient __fdiv_rn(x, s) decides.  Scales below 2^-100, where
//   r could overflow, always take the exact path.
#pragma once
#include <cstdint>

namespace w4k {

struct A8Scale {
    float s;   // the token's scale max|x| / 127
    float r;   // fl(1 / s), or 0 when the exact path must be used throughout
};

// Out of line: once per token, and its IEEE division need not sit in every
// quantizer's instruction stream.
static __device__ __noinline__ A8Scale a8_scale(float amax)
{
    A8Scale k;
    k.s = __fdiv_rn(amax, 127.0f);
    k.r = k.s >= 7.888609052e-31f ? __frcp_rn(k.s) : 0.0f;   // 2^-100
    return k;
}

__device__ __forceinline__ int a8_code(float v, const A8Scale& k)
{
    if (k.s == 0.0f) return 0;
    int q;
    if (k.r != 0.0f) {
        const float t = v * k.r;
        q = __float2int_rn(t);
        if (fabsf(t - __int2float_rn(q)) >= 0.49997f) q = __float2int_rn(__fdiv_rn(v, k.s));
    } else {
        q = __float2int_rn(__fdiv_rn(v, k.s));
    }
    return q > 127 ? 127 : (q < -127 ? -127 : q);
}

// Fast code for the common case, branch-free: t = fl(x * r) rounded half to
// even by adding and removing 1.5 * 2^23 (exact for |t| < 2^22).  `tie` is
// set when t lies within 3e-5 of a half-integer, where the exact quotient
// must decide (a8_code).  Valid only when k.r != 0.
__device__ __forceinline__ int a8_code_fast(float v, const A8Scale& k, bool& tie)
{
    const float t = __fmul_rn(v, k.r);
    const float big = __fadd_rn(t, 12582912.0f);
    const float rf = __fsub_rn(big, 12582912.0f);
    tie |= fabsf(__fsub_rn(t, rf)) >= 0.49997f;
    return __float_as_int(big) - 0x4B400000;
}

// Packed pairs of fp32 (sm_100 and later): one instruction performs two IEEE
// fp32 operations, each rounded exactly as its scalar form.
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi)
{
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ uint32_t f2_lo(uint64_t v) { return static_cast<uint32_t>(v); }
__device__ __forceinline__ uint32_t f2_hi(uint64_t v) { return static_cast<uint32_t>(v >> 32); }
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b)
{
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b)
{
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c)
{
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

// Low bytes of four ints, packed little-endian into one word.
__device__ __forceinline__ uint32_t pack_low_bytes(int a, int b, int c, int d)
{
    return __byte_perm(__byte_perm(a, b, 0x0040), __byte_perm(c, d, 0x0040), 0x5410);
}

// Four codes, fast path; sets `tie` if any of them needs a8_pack4 instead.
__device__ __forceinline__ uint32_t a8_pack4_fast(float4 v, const A8Scale& k, bool& tie)
{
    return pack_low_bytes(a8_code_fast(v.x, k, tie), a8_code_fast(v.y, k, tie), a8_code_fast(v.z, k, tie),
                          a8_code_fast(v.w, k, tie));
}

// The fast path of a8_pack4_fast on packed pairs, with the same roundings:
// t = fl(x * r), big = fl(t + 1.5 * 2^23) (so rint(t) is in big's low
// mantissa bits and the code is big's low byte), d = t - rint(t) exactly,
// and the tie test d^2 - 0.49997^2 >= 0, whose sign one FMA gets exactly.
// The sign bit of `ok` is cleared when some code of the four may be a tie
// (|d| within ~1e-8 of 0.49997 or above).  rr holds r in both halves.
__device__ __forceinline__ uint32_t a8_pack4_fast2(float4 v, uint64_t rr, uint32_t& ok)
{
    const uint64_t kBig = f2_pack(12582912.0f, 12582912.0f);
    const uint64_t kNegBig = f2_pack(-12582912.0f, -12582912.0f);
    const uint64_t kNegOne = f2_pack(-1.0f, -1.0f);
    const uint64_t kNegTie = f2_pack(-0.2499700009f, -0.2499700009f);   // -(0.49997^2)
    const uint64_t t01 = f2_mul(f2_pack(v.x, v.y), rr);
    const uint64_t t23 = f2_mul(f2_pack(v.z, v.w), rr);
    const uint64_t b01 = f2_add(t01, kBig);
    const uint64_t b23 = f2_add(t23, kBig);
    const uint64_t d01 = f2_fma(f2_add(b01, kNegBig), kNegOne, t01);
    const uint64_t d23 = f2_fma(f2_add(b23, kNegBig), kNegOne, t23);
    const uint64_t e01 = f2_fma(d01, d01, kNegTie);
    const uint64_t e23 = f2_fma(d23, d23, kNegTie);
    ok &= f2_lo(e01) & f2_hi(e01) & f2_lo(e23) & f2_hi(e23);
    return __byte_perm(__byte_perm(f2_lo(b01), f2_hi(b01), 0x0040), __byte_perm(f2_lo(b23), f2_hi(b23), 0x0040),
                       0x5410);
}

// The exact path for one word, out of line: it runs for about one word in
// 10^4 (possible ties, tiny scales), and inlined into every unrolled group of
// the quantizers its IEEE divisions would crowd the hot loop out of the
// instruction cache.
static __device__ __noinline__ uint32_t a8_pack4_exact(float4 v, A8Scale k);

// True when the fast path may not be used at all for this scale.
__device__ __forceinline__ bool a8_needs_exact(const A8Scale& k) { return k.s != 0.0f && k.r == 0.0f; }

__device__ __forceinline__ uint32_t a8_pack4(float4 v, const A8Scale& k)
{
    return (static_cast<uint32_t>(a8_code(v.x, k)) & 0xffu) | ((static_cast<uint32_t>(a8_code(v.y, k)) & 0xffu) << 8) |
           ((static_cast<uint32_t>(a8_code(v.z, k)) & 0xffu) << 16) |
           ((static_cast<uint32_t>(a8_code(v.w, k)) & 0xffu) << 24);
}

static __device__ __noinline__ uint32_t a8_pack4_exact(float4 v, A8Scale k) { return a8_pack4(v, k); }

}  // namespace w4k
