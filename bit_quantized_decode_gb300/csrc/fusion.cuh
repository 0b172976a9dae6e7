// Operators fused around the decode linear: RMSNorm in front of the
// activation quantizer, the gated MLP activation and the residual add after
// the epilogue.  "Jetson Orin AGX INT4 推理优化实践" §"后续还能继续优化什么"
// item 1 lists RMSNorm, quantization, linear, SwiGLU and the residual add as
// operators still separated by kernel boundaries; "在香橙派上跑 Gemma4" §4.2
// names add+rmsnorm and gelu+mul as the fusions to make.  The operators are
// the usual ones of the models those pages run:
//   RMSNorm:  r = 1 / sqrt(S / K + eps) with S = sum x^2 rounded once to fp32,
//             out = (x * r) * g, every step an IEEE fp32 operation;
//   SwiGLU:   act = g / (1 + exp(-g)) * u;
//   GELU-tanh gated: act = g / 2 * (1 + tanh(sqrt(2/pi) (g + 0.044715 g^3))) * u.
#pragma once
#include <cstdint>

#include "internal.h"

namespace w4k {

// Error-free sum (Knuth): s + e == a + b exactly, s = fl(a + b).
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e)
{
    s = __fadd_rn(a, b);
    const float bp = __fsub_rn(s, a);
    e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bp)), __fsub_rn(b, bp));
}

// Compensated sum of squares in a (hi, lo) pair of fp32: x*x = p + pe exactly
// (one FMA), p joins hi through an error-free sum, the small parts add into
// lo.  Over a tree of depth d the pair's error stays near d^2 2^-48 of the
// sum, so fl(hi + lo) is the correctly rounded S except when S lies within
// about 2^-38 (relative) of a rounding boundary.
__device__ __forceinline__ void sq_acc(float x, float& hi, float& lo)
{
    const float p = __fmul_rn(x, x);
    const float pe = __fmaf_rn(x, x, -p);
    float s, e;
    two_sum(hi, p, s, e);
    hi = s;
    lo = __fadd_rn(lo, __fadd_rn(e, pe));
}

__device__ __forceinline__ void sq_acc4(const float4& v, float& hi, float& lo)
{
    sq_acc(v.x, hi, lo);
    sq_acc(v.y, hi, lo);
    sq_acc(v.z, hi, lo);
    sq_acc(v.w, hi, lo);
}

__device__ __forceinline__ void pair_merge(float& hi, float& lo, float hi2, float lo2)
{
    float s, e;
    two_sum(hi, hi2, s, e);
    hi = s;
    lo = __fadd_rn(lo, __fadd_rn(lo2, e));
}

// Warp-wide merge of (hi, lo); lane 0's pair is the warp's sum.
__device__ __forceinline__ void warp_pair_sum(float& hi, float& lo)
{
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float h2 = __shfl_xor_sync(0xffffffffu, hi, off);
        const float l2 = __shfl_xor_sync(0xffffffffu, lo, off);
        pair_merge(hi, lo, h2, l2);
    }
}

// r = 1 / sqrt(fl(hi + lo) / K + eps), each operation correctly rounded.
__device__ __forceinline__ float rms_scale(float hi, float lo, int K, float eps)
{
    const float S = __fadd_rn(hi, lo);
    const float ms = __fdiv_rn(S, static_cast<float>(K));
    return __frcp_rn(__fsqrt_rn(__fadd_rn(ms, eps)));
}

__device__ __forceinline__ float4 rms_apply(const float4& x, float r, const float4& g)
{
    return make_float4(__fmul_rn(__fmul_rn(x.x, r), g.x), __fmul_rn(__fmul_rn(x.y, r), g.y),
                       __fmul_rn(__fmul_rn(x.z, r), g.z), __fmul_rn(__fmul_rn(x.w, r), g.w));
}

// Gated activation of one (gate, up) pair, in fp32 with the library's expf /
// tanhf (accurate, not the fast intrinsics).
__device__ __forceinline__ float glu_act(int kind, float g, float u)
{
    if (kind == GLU_SILU) return __fmul_rn(__fdiv_rn(g, __fadd_rn(1.0f, expf(-g))), u);
    const float g3 = __fmul_rn(__fmul_rn(g, g), g);
    const float t = tanhf(__fmul_rn(0.7978845608028654f, __fadd_rn(g, __fmul_rn(0.044715f, g3))));
    return __fmul_rn(__fmul_rn(__fmul_rn(0.5f, g), __fadd_rn(1.0f, t)), u);
}

// The same, out of line: the GEMV epilogues run it once per output, and its
// library calls stay out of the kernels' instruction footprint.
static __device__ __noinline__ float glu_act_call(int kind, float g, float u) { return glu_act(kind, g, u); }

}  // namespace w4k
