// Activation quantization, load-time weight quantizers and repack kernels.
//
// Quantization decisions are taken in IEEE fp32 with correctly rounded
// division (__fdiv_rn) and round-half-to-even conversion (__float2int_rn),
// so the codes are reproducible bit for bit by any IEEE implementation.
#include <cuda_fp16.h>

#include "fusion.cuh"
#include "internal.h"
#include "ptx.cuh"
#include "quant_a8.cuh"

namespace w4k {

// ---------------------------------------------------------------- helpers
__device__ __forceinline__ float warp_max(float v)
{
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
    return v;
}

__device__ __forceinline__ float abs_max4(float4 v)
{
    return fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
}

// clip(rint(v / s), lo, hi); s == 0 gives 0.
__device__ __forceinline__ int quant_code(float v, float s, int lo, int hi)
{
    if (s == 0.0f) return 0;
    int q = __float2int_rn(__fdiv_rn(v, s));
    return q > hi ? hi : (q < lo ? lo : q);
}

// ------------------------------------------------ per-token INT8 activations
// "Jetson Orin AGX INT4 推理优化实践", §"从 FP 线性层到 INT4 DP4A 的数学推导":
// s^x = max|x| / 127, q^x = clip(round(x / s^x), -127, 127).  One block per
// token.  Codes come from the fast path (multiply by fl(1/s), packed pairs)
// and, for words with a possible tie or a tiny scale, the exact quotient; the
// result is bit-identical to the definition (quant_a8.cuh).  The token stays
// in registers (NIT float4 per thread) when it fits, else it is read twice.
// Launched with programmatic dependent launch it waits for the previous
// kernel before reading x and lets the next kernel start at once.
constexpr int kQuantThreads = 512;
constexpr int kQuantWarps = kQuantThreads / 32;

// RMSNorm scale of one token over the block (fusion.cuh): the thread's
// compensated sum of squares (hi, lo) merged per warp, then over the warps in
// order.  Every thread returns r.  Two block barriers (red2 is reused).
__device__ __forceinline__ float block_rms_scale(float hi, float lo, int K, float eps, float* red2)
{
    warp_pair_sum(hi, lo);
    const int tid = threadIdx.x;
    if ((tid & 31) == 0) {
        red2[2 * (tid >> 5)] = hi;
        red2[2 * (tid >> 5) + 1] = lo;
    }
    __syncthreads();
    hi = red2[0];
    lo = red2[1];
#pragma unroll
    for (int w = 1; w < kQuantWarps; ++w) pair_merge(hi, lo, red2[2 * w], red2[2 * w + 1]);
    __syncthreads();
    return rms_scale(hi, lo, K, eps);
}

// kNorm: RMSNorm(x; gamma, eps) first (fusion.cuh), then the quantizer on the
// normalized values; gamma is read with x.  Without room in registers the
// token is read three times (sum of squares, absmax, codes).
template <int NIT, bool kNorm>
__global__ void __launch_bounds__(kQuantThreads) a8_quantize_kernel(const float* __restrict__ x,
                                                                    const float* __restrict__ gamma, float eps,
                                                                    int K, int8_t* __restrict__ qx,
                                                                    float* __restrict__ sx)
{
    __shared__ float red[kQuantWarps];
    __shared__ float red2[2 * kQuantWarps];
    constexpr bool kRegs = NIT > 0;
    constexpr int kN = kRegs ? NIT : 1;
    const int m = blockIdx.x;
    const int tid = threadIdx.x;
    const float4* xr = reinterpret_cast<const float4*>(x + static_cast<size_t>(m) * K);
    const float4* gr = reinterpret_cast<const float4*>(gamma);
    const int K4 = K >> 2;
    pdl_launch_dependents();
    // the norm weight does not depend on the previous kernel: load it first
    float4 gv[kNorm && kRegs ? kN : 1];
    if constexpr (kNorm && kRegs) {
#pragma unroll
        for (int it = 0; it < NIT; ++it) {
            const int i = tid + it * kQuantThreads;
            gv[it] = i < K4 ? __ldg(gr + i) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
    pdl_wait();
    float4 v[kN];
    float r = 1.0f;
    float mx = 0.0f;
    if constexpr (kRegs) {
#pragma unroll
        for (int it = 0; it < NIT; ++it) {
            const int i = tid + it * kQuantThreads;
            v[it] = i < K4 ? __ldcg(xr + i) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        if constexpr (kNorm) {
            float hi = 0.0f, lo = 0.0f;
#pragma unroll
            for (int it = 0; it < NIT; ++it) sq_acc4(v[it], hi, lo);
            r = block_rms_scale(hi, lo, K, eps, red2);
#pragma unroll
            for (int it = 0; it < NIT; ++it) v[it] = rms_apply(v[it], r, gv[it]);
        }
#pragma unroll
        for (int it = 0; it < NIT; ++it) mx = fmaxf(mx, abs_max4(v[it]));
    } else {
        if constexpr (kNorm) {
            float hi = 0.0f, lo = 0.0f;
            for (int i = tid; i < K4; i += kQuantThreads) sq_acc4(__ldcg(xr + i), hi, lo);
            r = block_rms_scale(hi, lo, K, eps, red2);
            for (int i = tid; i < K4; i += kQuantThreads) mx = fmaxf(mx, abs_max4(rms_apply(__ldcg(xr + i), r, __ldg(gr + i))));
        } else {
            for (int i = tid; i < K4; i += kQuantThreads) mx = fmaxf(mx, abs_max4(__ldcg(xr + i)));
        }
    }
    mx = warp_max(mx);
    if ((tid & 31) == 0) red[tid >> 5] = mx;
    __syncthreads();
    float amax = 0.0f;
#pragma unroll
    for (int w = 0; w < kQuantWarps; ++w) amax = fmaxf(amax, red[w]);
    const A8Scale ks = a8_scale(amax);
    const bool all_exact = a8_needs_exact(ks);
    const uint64_t rr = f2_pack(ks.r, ks.r);
    uint32_t* out = reinterpret_cast<uint32_t*>(qx + static_cast<size_t>(m) * K);
    auto code = [&](float4 f) -> uint32_t {
        uint32_t ok = 0xffffffffu;
        const uint32_t q = a8_pack4_fast2(f, rr, ok);
        return (all_exact || (ok >> 31) == 0) ? a8_pack4_exact(f, ks) : q;
    };
    if constexpr (kRegs) {
#pragma unroll
        for (int it = 0; it < NIT; ++it) {
            const int i = tid + it * kQuantThreads;
            if (i < K4) out[i] = code(v[it]);
        }
    } else {
        for (int i = tid; i < K4; i += kQuantThreads) {
            float4 f = __ldcg(xr + i);
            if constexpr (kNorm) f = rms_apply(f, r, __ldg(gr + i));
            out[i] = code(f);
        }
    }
    if (tid == 0) sx[m] = ks.s;
}

// Long tokens (8192 <= K <= 32768) and five or more of them: kQuantCluster
// blocks per token, in one thread-block cluster.  Block r reads quarter r of the token's float4 words
// into registers and takes its absmax; the blocks read one another's maxima
// through distributed shared memory, so each holds the token's absmax, and
// each quantizes its own quarter with a8_scale of that absmax: the codes and
// the scale are the single-block kernel's, bit for bit (a maximum does not
// depend on its order).  A block leaves only after every block has read its
// maximum (the second half of the last cluster barrier).  Measured on the 7B
// step (K = 18944 quantizer ahead of the down projection), against one block
// per token: 0.003 / 0.020 / 0.008 ms faster at 5 / 8 / 16 tokens, 0.018 ms
// slower at 3 (the cluster launch and its barriers outweigh the shorter read
// when there are few tokens).
constexpr int kQuantCluster = 4;
constexpr int kQuantClusterMinTokens = 5;

template <int NIT>
__global__ void __launch_bounds__(kQuantThreads) a8_quantize_cluster_kernel(const float* __restrict__ x, int K,
                                                                            int8_t* __restrict__ qx,
                                                                            float* __restrict__ sx)
{
    __shared__ float red[kQuantWarps];
    __shared__ float part;
    const int m = blockIdx.x / kQuantCluster;
    const int r = blockIdx.x - m * kQuantCluster;           // = rank in the cluster
    const int tid = threadIdx.x;
    const int K4 = K >> 2;
    const int q0 = r * K4 / kQuantCluster;
    const int q1 = (r + 1) * K4 / kQuantCluster;
    const float4* xr = reinterpret_cast<const float4*>(x + static_cast<size_t>(m) * K);
    pdl_launch_dependents();
    pdl_wait();
    float4 v[NIT];
    float mx = 0.0f;
#pragma unroll
    for (int it = 0; it < NIT; ++it) {
        const int i = q0 + tid + it * kQuantThreads;
        v[it] = i < q1 ? __ldcg(xr + i) : make_float4(0.f, 0.f, 0.f, 0.f);
        mx = fmaxf(mx, abs_max4(v[it]));
    }
    mx = warp_max(mx);
    if ((tid & 31) == 0) red[tid >> 5] = mx;
    __syncthreads();
    if (tid == 0) {
        float a = 0.0f;
#pragma unroll
        for (int w = 0; w < kQuantWarps; ++w) a = fmaxf(a, red[w]);
        part = a;
    }
    cluster_sync();                       // every block's maximum is written
    float amax = 0.0f;
#pragma unroll
    for (int c = 0; c < kQuantCluster; ++c)
        amax = fmaxf(amax, __uint_as_float(ld_cluster_u32(mapa_shared(smem_u32(&part), static_cast<uint32_t>(c)))));
    cluster_arrive_release();             // done with the other blocks' shared memory
    const A8Scale ks = a8_scale(amax);
    const bool all_exact = a8_needs_exact(ks);
    const uint64_t rr = f2_pack(ks.r, ks.r);
    uint32_t* out = reinterpret_cast<uint32_t*>(qx + static_cast<size_t>(m) * K);
#pragma unroll
    for (int it = 0; it < NIT; ++it) {
        const int i = q0 + tid + it * kQuantThreads;
        if (i < q1) {
            uint32_t ok = 0xffffffffu;
            const uint32_t q = a8_pack4_fast2(v[it], rr, ok);
            out[i] = (all_exact || (ok >> 31) == 0) ? a8_pack4_exact(v[it], ks) : q;
        }
    }
    if (r == 0 && tid == 0) sx[m] = ks.s;
    cluster_wait_acquire();
}

namespace {

cudaLaunchConfig_t token_launch(int M, bool pdl, cudaStream_t s, cudaLaunchAttribute* attr)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(M));
    cfg.blockDim = dim3(kQuantThreads);
    cfg.stream = s;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = pdl ? attr : nullptr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cfg;
}

template <bool kNorm>
cudaError_t launch_quant(const float* x, const float* gamma, float eps, int M, int K, int8_t* qx, float* sx, bool pdl,
                         cudaStream_t s)
{
    const int nit = (K / 4 + kQuantThreads - 1) / kQuantThreads;
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = token_launch(M, pdl, s, attr);
    if (nit <= 2) return cudaLaunchKernelEx(&cfg, a8_quantize_kernel<2, kNorm>, x, gamma, eps, K, qx, sx);
    if (nit <= 4) return cudaLaunchKernelEx(&cfg, a8_quantize_kernel<4, kNorm>, x, gamma, eps, K, qx, sx);
    if (nit <= 10) return cudaLaunchKernelEx(&cfg, a8_quantize_kernel<10, kNorm>, x, gamma, eps, K, qx, sx);
    if constexpr (!kNorm) {
        if (nit <= 16) return cudaLaunchKernelEx(&cfg, a8_quantize_kernel<16, kNorm>, x, gamma, eps, K, qx, sx);
    }
    return cudaLaunchKernelEx(&cfg, a8_quantize_kernel<0, kNorm>, x, gamma, eps, K, qx, sx);
}

}  // namespace

cudaError_t launch_a8_quantize(const float* x, int M, int K, int8_t* qx, float* sx, bool pdl, cudaStream_t s)
{
    const int per_block = (K / 4 + kQuantCluster - 1) / kQuantCluster;     // float4 words of a quarter
    if (M >= kQuantClusterMinTokens && K >= 8192 && per_block <= 4 * kQuantThreads) {
        cudaLaunchAttribute attr[2];
        cudaLaunchConfig_t cfg = token_launch(M, pdl, s, attr);
        cfg.gridDim = dim3(static_cast<unsigned>(M * kQuantCluster));
        attr[cfg.numAttrs].id = cudaLaunchAttributeClusterDimension;
        attr[cfg.numAttrs].val.clusterDim.x = kQuantCluster;
        attr[cfg.numAttrs].val.clusterDim.y = 1;
        attr[cfg.numAttrs].val.clusterDim.z = 1;
        cfg.attrs = attr;
        ++cfg.numAttrs;
        if (per_block <= 2 * kQuantThreads)
            return cudaLaunchKernelEx(&cfg, a8_quantize_cluster_kernel<2>, x, K, qx, sx);
        return cudaLaunchKernelEx(&cfg, a8_quantize_cluster_kernel<4>, x, K, qx, sx);
    }
    return launch_quant<false>(x, nullptr, 0.0f, M, K, qx, sx, pdl, s);
}

cudaError_t launch_rms_a8_quantize(const float* x, const float* gamma, float eps, int M, int K, int8_t* qx,
                                   float* sx, bool pdl, cudaStream_t s)
{
    return launch_quant<true>(x, gamma, eps, M, K, qx, sx, pdl, s);
}

// ----------------------------------------- the fused operators on their own
// RMSNorm to fp32 (one block per token, same arithmetic as the fused
// prologue), the gated activation of a [M][2I] gate|up output, and an
// elementwise add: the separate kernels a decoder runs without the fusions.
__global__ void __launch_bounds__(kQuantThreads) rmsnorm_kernel(const float* __restrict__ x,
                                                                const float* __restrict__ gamma, float eps, int K,
                                                                float* __restrict__ out)
{
    __shared__ float red2[2 * kQuantWarps];
    pdl_launch_dependents();
    pdl_wait();
    const int m = blockIdx.x;
    const float4* xr = reinterpret_cast<const float4*>(x + static_cast<size_t>(m) * K);
    const float4* gr = reinterpret_cast<const float4*>(gamma);
    float4* orow = reinterpret_cast<float4*>(out + static_cast<size_t>(m) * K);
    const int K4 = K >> 2;
    float hi = 0.0f, lo = 0.0f;
    for (int i = threadIdx.x; i < K4; i += kQuantThreads) sq_acc4(__ldcg(xr + i), hi, lo);
    const float r = block_rms_scale(hi, lo, K, eps, red2);
    for (int i = threadIdx.x; i < K4; i += kQuantThreads) orow[i] = rms_apply(__ldcg(xr + i), r, __ldg(gr + i));
}

__global__ void glu_kernel(const float* __restrict__ gu, int kind, int I, long long n, float* __restrict__ out)
{
    pdl_launch_dependents();
    pdl_wait();
    const long long k = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (k >= n) return;
    const long long m = k / I;
    const long long j = k - m * I;
    const float* row = gu + m * 2 * I;
    out[k] = glu_act_call(kind, __ldcg(row + j), __ldcg(row + I + j));
}

__global__ void add_kernel(const float* __restrict__ a, const float* __restrict__ b, long long n,
                           float* __restrict__ out)
{
    pdl_launch_dependents();
    pdl_wait();
    const long long k = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (k < n) out[k] = __fadd_rn(__ldcg(a + k), __ldcg(b + k));
}

cudaError_t launch_rmsnorm(const float* x, const float* gamma, float eps, int M, int K, float* out, bool pdl,
                           cudaStream_t s)
{
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = token_launch(M, pdl, s, attr);
    return cudaLaunchKernelEx(&cfg, rmsnorm_kernel, x, gamma, eps, K, out);
}

cudaError_t launch_glu(const float* gu, int kind, int M, int I, float* out, bool pdl, cudaStream_t s)
{
    const long long n = static_cast<long long>(M) * I;
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = token_launch(1, pdl, s, attr);
    cfg.gridDim = dim3(static_cast<unsigned>((n + 255) / 256));
    cfg.blockDim = dim3(256);
    return cudaLaunchKernelEx(&cfg, glu_kernel, gu, kind, I, n, out);
}

cudaError_t launch_add(const float* a, const float* b, long long n, float* out, bool pdl, cudaStream_t s)
{
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = token_launch(1, pdl, s, attr);
    cfg.gridDim = dim3(static_cast<unsigned>((n + 255) / 256));
    cfg.blockDim = dim3(256);
    return cudaLaunchKernelEx(&cfg, add_kernel, a, b, n, out);
}

// ------------------------------------------------------ per-row INT4 weights
// s^W_j = max|W_j| / 7, q = clip(rint(W / s^W_j), -8, 7), eight codes per
// uint32 with weight k in bits 4k..4k+3 (§"DP4A 做了什么").  One warp per row.
__global__ void __launch_bounds__(256) w4_quantize_rows_kernel(const float* __restrict__ W, int N, int K,
                                                              uint32_t* __restrict__ packed, float* __restrict__ sw)
{
    const int row = blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= N) return;
    const float4* wr = reinterpret_cast<const float4*>(W + static_cast<size_t>(row) * K);
    float mx = 0.0f;
    for (int i = lane; i < K / 4; i += 32) mx = fmaxf(mx, abs_max4(wr[i]));
    mx = warp_max(mx);
    const float s = __fdiv_rn(mx, 7.0f);
    if (lane == 0) sw[row] = s;
    uint32_t* out = packed + static_cast<size_t>(row) * (K / 8);
    for (int wi = lane; wi < K / 8; wi += 32) {
        const float4 v0 = wr[2 * wi], v1 = wr[2 * wi + 1];
        const float v[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
        uint32_t word = 0;
#pragma unroll
        for (int k = 0; k < 8; ++k) word |= (static_cast<uint32_t>(quant_code(v[k], s, -8, 7)) & 0xfu) << (4 * k);
        out[wi] = word;
    }
}

cudaError_t launch_w4_quantize_rows(const float* W, int N, int K, uint32_t* packed, float* s_w, cudaStream_t s)
{
    w4_quantize_rows_kernel<<<(N + 7) / 8, 256, 0, s>>>(W, N, K, packed, s_w);
    return cudaGetLastError();
}

// ------------------------------------------------------ per-row INT8 weights
// The weight-only INT8 path ("Jetson Orin AGX INT4 推理优化实践", §"为什么 INT4
// float 解包不快"): s^W_j = max|W_j| / 127, q = clip(rint(W / s^W_j), -127, 127),
// one int8 per weight [N][K].  One warp per row.
__global__ void __launch_bounds__(256) w8_quantize_rows_kernel(const float* __restrict__ W, int N, int K,
                                                              int8_t* __restrict__ q, float* __restrict__ sw)
{
    const int row = blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= N) return;
    const float4* wr = reinterpret_cast<const float4*>(W + static_cast<size_t>(row) * K);
    float mx = 0.0f;
    for (int i = lane; i < K / 4; i += 32) mx = fmaxf(mx, abs_max4(wr[i]));
    mx = warp_max(mx);
    const float s = __fdiv_rn(mx, 127.0f);
    if (lane == 0) sw[row] = s;
    uint32_t* out = reinterpret_cast<uint32_t*>(q + static_cast<size_t>(row) * K);
    for (int i = lane; i < K / 4; i += 32) {
        const float4 v = wr[i];
        out[i] = (static_cast<uint32_t>(quant_code(v.x, s, -127, 127)) & 0xffu) |
                 ((static_cast<uint32_t>(quant_code(v.y, s, -127, 127)) & 0xffu) << 8) |
                 ((static_cast<uint32_t>(quant_code(v.z, s, -127, 127)) & 0xffu) << 16) |
                 ((static_cast<uint32_t>(quant_code(v.w, s, -127, 127)) & 0xffu) << 24);
    }
}

cudaError_t launch_w8_quantize_rows(const float* W, int N, int K, int8_t* q, float* s_w, cudaStream_t s)
{
    w8_quantize_rows_kernel<<<(N + 7) / 8, 256, 0, s>>>(W, N, K, q, s_w);
    return cudaGetLastError();
}

// ---------------------------------------------------------------- Q4_0
// "在香橙派上跑 Gemma4", §3.1: 32 weights per block, 16 bytes of nibbles and an
// fp16 scale; d = fp16(max|w| / 8), n = clip(rint(w / d), -8, 7) + 8.  Block
// bytes: d (little endian), then byte i = element i | element (i+16) << 4.
__global__ void __launch_bounds__(256) q4_0_quantize_kernel(const float* __restrict__ W, int N, int K,
                                                           uint8_t* __restrict__ blocks)
{
    const int G = K / 32;
    const long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (idx >= static_cast<long long>(N) * G) return;
    const float4* wp = reinterpret_cast<const float4*>(W + idx * 32);
    float v[32];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float4 t = wp[i];
        v[4 * i] = t.x; v[4 * i + 1] = t.y; v[4 * i + 2] = t.z; v[4 * i + 3] = t.w;
    }
    float mx = 0.0f;
#pragma unroll
    for (int i = 0; i < 32; ++i) mx = fmaxf(mx, fabsf(v[i]));
    const __half dh = __float2half_rn(__fdiv_rn(mx, 8.0f));
    const float d = __half2float(dh);
    // 18-byte blocks are 2-byte aligned: store them as nine 16-bit words
    // (little endian: the scale first, then nibble bytes 2j and 2j+1).
    uint16_t* blk = reinterpret_cast<uint16_t*>(blocks + idx * 18);
    blk[0] = __half_as_ushort(dh);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        uint32_t pair = 0;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int i = 2 * j + h;
            const uint32_t lo = static_cast<uint32_t>(quant_code(v[i], d, -8, 7) + 8);
            const uint32_t hi = static_cast<uint32_t>(quant_code(v[i + 16], d, -8, 7) + 8);
            pair |= (lo | (hi << 4)) << (8 * h);
        }
        blk[1 + j] = static_cast<uint16_t>(pair);
    }
}

cudaError_t launch_q4_0_quantize(const float* W, int N, int K, uint8_t* blocks, cudaStream_t s)
{
    const long long n = static_cast<long long>(N) * (K / 32);
    q4_0_quantize_kernel<<<static_cast<unsigned>((n + 255) / 256), 256, 0, s>>>(W, N, K, blocks);
    return cudaGetLastError();
}

// ---------------------------------------------------------------- i8g32
// "在香橙派上跑 Gemma4", §3.2: int8 weights with one fp16 scale per group;
// here d = fp16(max|w| / 32), q = clip(rint(w / d), -32, 31).
__global__ void __launch_bounds__(256) i8g32_quantize_kernel(const float* __restrict__ W, int N, int K,
                                                            int8_t* __restrict__ q, uint16_t* __restrict__ d)
{
    const int G = K / 32;
    const long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (idx >= static_cast<long long>(N) * G) return;
    const float4* wp = reinterpret_cast<const float4*>(W + idx * 32);
    float v[32];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float4 t = wp[i];
        v[4 * i] = t.x; v[4 * i + 1] = t.y; v[4 * i + 2] = t.z; v[4 * i + 3] = t.w;
    }
    float mx = 0.0f;
#pragma unroll
    for (int i = 0; i < 32; ++i) mx = fmaxf(mx, fabsf(v[i]));
    const __half dh = __float2half_rn(__fdiv_rn(mx, 32.0f));
    const float df = __half2float(dh);
    d[idx] = __half_as_ushort(dh);
    uint32_t w[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        w[i] = 0;
#pragma unroll
        for (int b = 0; b < 4; ++b)
            w[i] |= (static_cast<uint32_t>(quant_code(v[4 * i + b], df, -32, 31)) & 0xffu) << (8 * b);
    }
    uint4* out = reinterpret_cast<uint4*>(q + idx * 32);
    out[0] = make_uint4(w[0], w[1], w[2], w[3]);
    out[1] = make_uint4(w[4], w[5], w[6], w[7]);
}

cudaError_t launch_i8g32_quantize(const float* W, int N, int K, int8_t* q, uint16_t* d, cudaStream_t s)
{
    const long long n = static_cast<long long>(N) * (K / 32);
    i8g32_quantize_kernel<<<static_cast<unsigned>((n + 255) / 256), 256, 0, s>>>(W, N, K, q, d);
    return cudaGetLastError();
}

// ---------------------------------------------------------------- repack
// Fused-shard row lookup: row j of the fused matrix is row j - row0[s] of
// shard s.  Returns -1 for rows past the end (tile padding).
__device__ __forceinline__ int shard_of(const ShardTable& st, int row, int& local)
{
    if (st.glu_rows > 0) {
        // gated pairing: kernel row -> gate (shard 0) or up (shard 1) row
        const int pr = glu_param_row(row, st.glu_rows);
        if (pr < 0) return -1;
        local = pr < st.glu_rows ? pr : pr - st.glu_rows;
        return pr < st.glu_rows ? 0 : 1;
    }
    for (int s = 0; s < st.n; ++s) {
        if (row < st.row0[s + 1]) {
            local = row - st.row0[s];
            return s;
        }
    }
    return -1;
}

// Canonical word (weight k in nibble k) -> device word: byte b holds weight b
// in its low nibble and weight b+4 in its high nibble.
__device__ __forceinline__ uint32_t spread4(uint32_t v)
{
    return (v & 0xfu) | ((v & 0xf0u) << 4) | ((v & 0xf00u) << 8) | ((v & 0xf000u) << 12);
}

// The device stores every nibble biased, n = q + 8, which for a 4-bit two's
// complement q is q with its top bit flipped.
__device__ __forceinline__ uint32_t interleave_w4(uint32_t canon)
{
    return (spread4(canon & 0xffffu) | (spread4(canon >> 16) << 4)) ^ 0x88888888u;
}

// One thread per unit (t, c, r) -> out unit index ((t*C + c)*8 + r).
__global__ void w4_repack_kernel(const ShardTable st, int N, int K, long long units, uint4* __restrict__ out)
{
    const long long u = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (u >= units) return;
    const int C = K / 32;
    const int r = static_cast<int>(u % kRows);
    const long long tc = u / kRows;
    const int c = static_cast<int>(tc % C);
    const long long t = tc / C;
    const long long row = t * kRows + r;
    uint4 o = make_uint4(0, 0, 0, 0);
    int local = 0;
    const int s = row < N ? shard_of(st, static_cast<int>(row), local) : -1;
    if (s >= 0) {
        const uint32_t* src = static_cast<const uint32_t*>(st.p[s]) + static_cast<size_t>(local) * (K / 8) + c * 4;
        o.x = interleave_w4(src[0]);
        o.y = interleave_w4(src[1]);
        o.z = interleave_w4(src[2]);
        o.w = interleave_w4(src[3]);
    }
    out[u] = o;
}

// Q4_0 nibble n (value n - 8) -> 4-bit two's complement of n - 8, i.e. n ^ 8.
__global__ void q4_0_repack_kernel(const ShardTable st, int N, int K, long long units, uint4* __restrict__ out,
                                   uint16_t* __restrict__ plane)
{
    const long long u = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (u >= units) return;
    const int C = K / 32;
    const int r = static_cast<int>(u % kRows);
    const long long tc = u / kRows;
    const int c = static_cast<int>(tc % C);
    const long long t = tc / C;
    const long long row = t * kRows + r;
    uint4 o = make_uint4(0, 0, 0, 0);
    uint16_t dbits = 0;
    int local = 0;
    const int s = row < N ? shard_of(st, static_cast<int>(row), local) : -1;
    if (s >= 0) {
        const uint8_t* blk = static_cast<const uint8_t*>(st.p[s]) + (static_cast<size_t>(local) * C + c) * 18;
        dbits = static_cast<uint16_t>(blk[0] | (blk[1] << 8));
        uint32_t v4[32];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const uint32_t byte = blk[2 + i];
            v4[i] = (byte & 0xfu) ^ 8u;
            v4[i + 16] = (byte >> 4) ^ 8u;
        }
        uint32_t w[4];
#pragma unroll
        for (int wi = 0; wi < 4; ++wi) {
            w[wi] = 0;
#pragma unroll
            for (int b = 0; b < 4; ++b) w[wi] |= (v4[8 * wi + b] | (v4[8 * wi + b + 4] << 4)) << (8 * b);
        }
        o = make_uint4(w[0], w[1], w[2], w[3]);
    }
    out[u] = o;
    plane[u] = dbits;
}

__global__ void i8g32_repack_kernel(const ShardTable st, int N, int K, long long units, uint4* __restrict__ out,
                                    uint16_t* __restrict__ plane)
{
    const long long u = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (u >= units) return;
    const int C = K / 32;
    const int r = static_cast<int>(u % kRows);
    const long long tc = u / kRows;
    const int c = static_cast<int>(tc % C);
    const long long t = tc / C;
    const long long row = t * kRows + r;
    uint4 o0 = make_uint4(0, 0, 0, 0), o1 = o0;
    uint16_t dbits = 0;
    int local = 0;
    const int s = row < N ? shard_of(st, static_cast<int>(row), local) : -1;
    if (s >= 0) {
        const uint4* src = reinterpret_cast<const uint4*>(static_cast<const int8_t*>(st.p[s]) +
                                                          static_cast<size_t>(local) * K + c * 32);
        o0 = src[0];
        o1 = src[1];
        if (plane != nullptr) dbits = static_cast<const uint16_t*>(st.p2[s])[static_cast<size_t>(local) * C + c];
    }
    out[2 * u] = o0;
    out[2 * u + 1] = o1;
    if (plane != nullptr) plane[u] = dbits;     // per-row INT8 (W8F) has no scale plane
}

// Q6G32: the i8g32 codes q in [-32, 31], biased n = q + 32 (6 bits), packed
// into a low plane (n & 15, same nibble places as the per-row INT4 unit: word
// w, byte b holds weight 8w+b low and 8w+4+b high) and a high plane (n >> 4,
// two bits: word h, byte b, bits 2s..2s+1 hold weight 16h+4s+b).
__global__ void q6g32_repack_kernel(const ShardTable st, int N, int K, long long units, uint4* __restrict__ lo,
                                    uint2* __restrict__ hi, uint16_t* __restrict__ plane)
{
    const long long u = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (u >= units) return;
    const int C = K / 32;
    const int r = static_cast<int>(u % kRows);
    const long long tc = u / kRows;
    const int c = static_cast<int>(tc % C);
    const long long t = tc / C;
    const long long row = t * kRows + r;
    uint32_t lw[4] = {0u, 0u, 0u, 0u};
    uint32_t hw[2] = {0u, 0u};
    uint16_t dbits = 0;
    int local = 0;
    const int s = row < N ? shard_of(st, static_cast<int>(row), local) : -1;
    if (s >= 0) {
        const int8_t* src = static_cast<const int8_t*>(st.p[s]) + static_cast<size_t>(local) * K + c * 32;
        uint32_t n[32];
#pragma unroll
        for (int k = 0; k < 32; ++k) n[k] = static_cast<uint32_t>(src[k] + 32) & 63u;
#pragma unroll
        for (int w = 0; w < 4; ++w)
#pragma unroll
            for (int b = 0; b < 4; ++b)
                lw[w] |= ((n[8 * w + b] & 15u) | ((n[8 * w + 4 + b] & 15u) << 4)) << (8 * b);
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int s2 = 0; s2 < 4; ++s2)
#pragma unroll
                for (int b = 0; b < 4; ++b) hw[h] |= (n[16 * h + 4 * s2 + b] >> 4) << (8 * b + 2 * s2);
        dbits = static_cast<const uint16_t*>(st.p2[s])[static_cast<size_t>(local) * C + c];
    }
    lo[u] = make_uint4(lw[0], lw[1], lw[2], lw[3]);
    hi[u] = make_uint2(hw[0], hw[1]);
    plane[u] = dbits;
}

static inline unsigned blocks_for(long long n, int t) { return static_cast<unsigned>((n + t - 1) / t); }

cudaError_t launch_q6g32_repack(const ShardTable& st, int N, int K, void* out, cudaStream_t s)
{
    const long long T = (N + kRows - 1) / kRows;
    const long long units = T * (K / 32) * kRows;
    uint8_t* base = static_cast<uint8_t*>(out);
    q6g32_repack_kernel<<<blocks_for(units, 256), 256, 0, s>>>(st, N, K, units, reinterpret_cast<uint4*>(base),
                                                              reinterpret_cast<uint2*>(base + units * 16),
                                                              reinterpret_cast<uint16_t*>(base + units * 24));
    return cudaGetLastError();
}

cudaError_t launch_w4_repack(const ShardTable& st, int N, int K, void* out, cudaStream_t s)
{
    const long long T = (N + kRows - 1) / kRows;
    const long long units = T * (K / 32) * kRows;
    w4_repack_kernel<<<blocks_for(units, 256), 256, 0, s>>>(st, N, K, units, static_cast<uint4*>(out));
    return cudaGetLastError();
}

cudaError_t launch_q4_0_repack(const ShardTable& st, int N, int K, void* out, cudaStream_t s)
{
    const long long T = (N + kRows - 1) / kRows;
    const long long units = T * (K / 32) * kRows;
    uint4* o = static_cast<uint4*>(out);
    uint16_t* plane = reinterpret_cast<uint16_t*>(static_cast<uint8_t*>(out) + units * 16);
    q4_0_repack_kernel<<<blocks_for(units, 256), 256, 0, s>>>(st, N, K, units, o, plane);
    return cudaGetLastError();
}

cudaError_t launch_i8g32_repack(const ShardTable& st, int N, int K, void* out, cudaStream_t s)
{
    const long long T = (N + kRows - 1) / kRows;
    const long long units = T * (K / 32) * kRows;
    uint4* o = static_cast<uint4*>(out);
    uint16_t* plane = reinterpret_cast<uint16_t*>(static_cast<uint8_t*>(out) + units * 32);
    i8g32_repack_kernel<<<blocks_for(units, 256), 256, 0, s>>>(st, N, K, units, o, plane);
    return cudaGetLastError();
}

// Per-row INT8 weights: the I8G32 unit layout without its scale plane.
cudaError_t launch_w8_repack(const ShardTable& st, int N, int K, void* out, cudaStream_t s)
{
    const long long T = (N + kRows - 1) / kRows;
    const long long units = T * (K / 32) * kRows;
    i8g32_repack_kernel<<<blocks_for(units, 256), 256, 0, s>>>(st, N, K, units, static_cast<uint4*>(out), nullptr);
    return cudaGetLastError();
}

}  // namespace w4k
