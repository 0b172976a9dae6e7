// Streaming decode GEMV for packed weights on sm_103a.
//
// What it computes ("Jetson Orin AGX INT4 推理优化实践", §"从 FP 线性层到 INT4 DP4A
// 的数学推导"; "在香橙派上跑 Gemma4", §3.1 and §3.2):
//   W4:    acc[m][j] = sum_i q_w[j][i] qx[m][i] (exact int32),
//          y = fmaf(s_w[j] * sx[m], (float)acc, b[j])
//   Q4_0, I8G32: acc_g = exact int32 sum over 32-block g,
//          y = fmaf(sx[m], sum_g d_g * acc_g, b[j])
//
// How (GB300 design, not the pages'):
//   * One thread block of 8 warps per SM, sized (shared memory <= ~113 KB,
//     <= 128 registers) so that the next GEMV in the stream can be resident
//     beside it: with programmatic dependent launch the next kernel starts,
//     prefetches its weights and waits at griddepcontrol.wait while this one
//     finishes.
//   * Each block owns a contiguous, balanced range of 8-row tiles, processed
//     in rounds; each round's lines (8 rows x 32 weights) are split evenly
//     among the warps.  Every warp runs its own ring of shared-memory slots
//     fed by 1-D bulk (TMA) copies (lane 0 issues, evict-first L2 policy,
//     bounded mbarrier waits).  The first slices are issued before the
//     dependency wait and the activation prologue.
//   * Per-row INT4 weights are stored biased (nibble n = q + 8): with
//     w & 0x0F0F0F0F and w & 0xF0F0F0F0 a 32-bit word yields four unsigned
//     bytes n and four bytes 16n, fed to DP4A (u8 x s8) against the matching
//     int8 activations -- two LOP3 and two DP4A per eight weights.  The bias
//     is removed exactly once per row in the epilogue with the activation
//     code sum: sum n x = sum q x + 8 sum x.  Q4_0 nibbles, whose scale
//     changes every 32 weights, are stored as 4-bit two's complement instead:
//     (w << 4) & 0xF0F0F0F0 and w & 0xF0F0F0F0 are four signed bytes 16q each,
//     and the group sum is shifted back exactly.  Both are the page's "two
//     int8x4, two DP4A per 8 weights" (§"DP4A 做了什么") with the sign
//     extension folded into an offset or a byte position.
//   * Lane l works on line (l >> 1) of a 16-line pass and on rows 4(l & 1) ..
//     4(l & 1) + 3, so one activation chunk feeds four rows (the page's
//     r-rows-per-block reuse, §"o2-all 和 o4-all 为什么能加速", done per lane).
//     Lanes read their four units in an XOR-permuted order so shared-memory
//     reads are conflict-free; the permutation is undone by a shuffle
//     butterfly at the end of each tile.
//   * Tiles split between warps are merged in shared memory in warp order
//     (deterministic); the epilogue writes y coalesced.
//   * Operators around the linear (fusion.cuh) are runtime branches of the
//     same instantiation: RMSNorm in the quantize prologue (one to four
//     tokens), the gated activation over gate/up rows paired per tile, and the
//     residual add in the epilogue.  One instantiation keeps consecutive
//     launches on the same instruction-cache lines.
//   * Code that runs once per launch (prologue, epilogue) is on the critical
//     path and meets cold instruction-cache lines, so rare paths (the
//     quantizer's exact tie path, the token scale, the gated activation) are
//     out-of-line functions, and tile ranges come from the host without a
//     division.
//   * FMT_W4F / FMT_W8F (xmode X_F32) are the weight-only baselines on float
//     activations: the same streaming, with every weight unpacked to fp32.
#pragma once
#include <cuda_fp16.h>

#include <type_traits>

#include "fusion.cuh"
#include "internal.h"
#include "ptx.cuh"
#include "quant_a8.cuh"

namespace w4k {

constexpr uint64_t kWaitTimeoutNs = 250ull * 1000ull * 1000ull;

// DP4A with unsigned bytes in a and signed bytes in b.
__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c)
{
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// Sum of the four signed bytes of a word.
__device__ __forceinline__ int bytesum(uint32_t w) { return __dp4a(static_cast<int>(w), 0x01010101, 0); }

// 4-bit units: B = sum n x over the low nibbles, A = sum 16 n x over the high
// nibbles of one 16-byte unit (32 weights) against its 32 activations.
__device__ __forceinline__ void unit4(const uint4 w, const uint4 x0, const uint4 x1, int& B, int& A)
{
    B = dp4a_us(w.x & 0x0F0F0F0Fu, x0.x, 0);
    A = dp4a_us(w.x & 0xF0F0F0F0u, x0.y, 0);
    B = dp4a_us(w.y & 0x0F0F0F0Fu, x0.z, B);
    A = dp4a_us(w.y & 0xF0F0F0F0u, x0.w, A);
    B = dp4a_us(w.z & 0x0F0F0F0Fu, x1.x, B);
    A = dp4a_us(w.z & 0xF0F0F0F0u, x1.y, A);
    B = dp4a_us(w.w & 0x0F0F0F0Fu, x1.z, B);
    A = dp4a_us(w.w & 0xF0F0F0F0u, x1.w, A);
}

// unit4 accumulated in place: B += sum n x (low nibbles), A += sum 16 n x
// (high nibbles), each a chain of four DP4A through its accumulator, so a
// line costs no separate adds; the row's sum n x is B + (A >> 4), formed once
// per tile (A stays a multiple of 16 and, over a row of K weights, within
// 16 * 15 * 127 * K / 2 < 2^31 for K <= 131072).
__device__ __forceinline__ void unit4_acc(const uint4 w, const uint4 x0, const uint4 x1, int& B, int& A)
{
    B = dp4a_us(w.x & 0x0F0F0F0Fu, x0.x, B);
    A = dp4a_us(w.x & 0xF0F0F0F0u, x0.y, A);
    B = dp4a_us(w.y & 0x0F0F0F0Fu, x0.z, B);
    A = dp4a_us(w.y & 0xF0F0F0F0u, x0.w, A);
    B = dp4a_us(w.z & 0x0F0F0F0Fu, x1.x, B);
    A = dp4a_us(w.z & 0xF0F0F0F0u, x1.y, A);
    B = dp4a_us(w.w & 0x0F0F0F0Fu, x1.z, B);
    A = dp4a_us(w.w & 0xF0F0F0F0u, x1.w, A);
}

// Signed 4-bit units (Q4_0): 16 * sum q x over one 16-byte unit.
__device__ __forceinline__ int unit4_signed16(const uint4 w, const uint4 x0, const uint4 x1)
{
    int g = dp4a_ss((w.x << 4) & 0xF0F0F0F0u, x0.x, 0);
    g = dp4a_ss(w.x & 0xF0F0F0F0u, x0.y, g);
    g = dp4a_ss((w.y << 4) & 0xF0F0F0F0u, x0.z, g);
    g = dp4a_ss(w.y & 0xF0F0F0F0u, x0.w, g);
    g = dp4a_ss((w.z << 4) & 0xF0F0F0F0u, x1.x, g);
    g = dp4a_ss(w.z & 0xF0F0F0F0u, x1.y, g);
    g = dp4a_ss((w.w << 4) & 0xF0F0F0F0u, x1.z, g);
    g = dp4a_ss(w.w & 0xF0F0F0F0u, x1.w, g);
    return g;
}

// Weight-only formats on float activations: four weights from the four bytes
// of `b` (each 0..255, the weight plus an offset) as fp32, exactly: the byte
// is placed in the mantissa of 2^23 (PRMT with 0x4B000000 gives 2^23 + byte),
// then 2^23 + offset is subtracted (negb, both halves).  Pairs in f32x2.
__device__ __forceinline__ void byte_floats(uint32_t b, uint64_t negb, uint64_t& q01, uint64_t& q23)
{
    const float f0 = __int_as_float(static_cast<int>(__byte_perm(b, 0x4B000000u, 0x7440)));
    const float f1 = __int_as_float(static_cast<int>(__byte_perm(b, 0x4B000000u, 0x7441)));
    const float f2 = __int_as_float(static_cast<int>(__byte_perm(b, 0x4B000000u, 0x7442)));
    const float f3 = __int_as_float(static_cast<int>(__byte_perm(b, 0x4B000000u, 0x7443)));
    q01 = f2_add(f2_pack(f0, f1), negb);
    q23 = f2_add(f2_pack(f2, f3), negb);
}

// acc2 += q . x for four weights against one float4 of x (f32x2 pairs).
__device__ __forceinline__ uint64_t fma4(uint64_t q01, uint64_t q23, const float4& x, uint64_t acc2)
{
    acc2 = f2_fma(q01, f2_pack(x.x, x.y), acc2);
    return f2_fma(q23, f2_pack(x.z, x.w), acc2);
}

// Barrier of the kThreads threads that run a linear's prologue and
// epilogue: the whole block (kBar = 0), or named barrier kBar when the block
// has further warps (a weight-producer warp) that stay out of it.
template <int kBar, int NT = kThreads>
__device__ __forceinline__ void block_sync()
{
    if constexpr (kBar == 0) {
        __syncthreads();
    } else {
        named_sync(kBar, NT);
    }
}

// Fused prologue for large M*K: a first pass over x for the absmax, a second
// to quantize, each in batches of 16 float4 per thread spread over the
// tokens (all loads of a batch in flight at once).  One block barrier.
template <int MT, bool kCodeSums, int kBar = 0, int NT = kThreads>
__device__ __forceinline__ void fused_prologue_twopass(const GemvArgs& a, float* red_s, float* sx_s, int8_t* xs,
                                                       int (&tsum)[MT])
{
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int M = a.M;
    const int K = a.K;
    const int K4 = K >> 2;
    constexpr int kB = MT >= 16 ? 1 : 16 / MT;        // float4 per token per batch
    float mx[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) mx[m] = 0.0f;
    for (int i0 = 0; i0 < K4; i0 += kB * NT) {
        float4 v[MT][kB];
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            const float4* xr = reinterpret_cast<const float4*>(a.x + static_cast<size_t>(m) * K);
#pragma unroll
            for (int u = 0; u < kB; ++u) {
                const int i = i0 + u * NT + tid;
                v[m][u] = (m < M && i < K4) ? __ldcg(xr + i) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
#pragma unroll
        for (int m = 0; m < MT; ++m)
#pragma unroll
            for (int u = 0; u < kB; ++u)
                mx[m] = fmaxf(mx[m], fmaxf(fmaxf(fabsf(v[m][u].x), fabsf(v[m][u].y)),
                                           fmaxf(fabsf(v[m][u].z), fabsf(v[m][u].w))));
    }
#pragma unroll
    for (int m = 0; m < MT; ++m) {
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) mx[m] = fmaxf(mx[m], __shfl_xor_sync(0xffffffffu, mx[m], off));
        if (lane == 0) red_s[warp * MT + m] = mx[m];
    }
    block_sync<kBar, NT>();
    A8Scale ks[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) {
        float amax = red_s[m];
#pragma unroll
        for (int w = 1; w < (NT / 32); ++w) amax = fmaxf(amax, red_s[w * MT + m]);
        ks[m] = a8_scale(m < M ? amax : 0.0f);
        if (tid == m) {
            sx_s[m] = m < M ? ks[m].s : 0.0f;
            if (m < M && blockIdx.x == 0 && a.sx_out != nullptr) a.sx_out[m] = ks[m].s;
        }
    }
    for (int i0 = 0; i0 < K4; i0 += kB * NT) {
        float4 v[MT][kB];
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            const float4* xr = reinterpret_cast<const float4*>(a.x + static_cast<size_t>(m) * K);
#pragma unroll
            for (int u = 0; u < kB; ++u) {
                const int i = i0 + u * NT + tid;
                v[m][u] = (m < M && i < K4) ? __ldcg(xr + i) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            if (m < M) {
                uint32_t* dst = reinterpret_cast<uint32_t*>(xs + static_cast<size_t>(m) * K);
                uint32_t* gout = (blockIdx.x == 0 && a.qx_out != nullptr)
                                     ? reinterpret_cast<uint32_t*>(a.qx_out + static_cast<size_t>(m) * K)
                                     : nullptr;
                const bool all_exact = a8_needs_exact(ks[m]);
                const uint64_t rr = f2_pack(ks[m].r, ks[m].r);
#pragma unroll
                for (int u = 0; u < kB; ++u) {
                    const int i = i0 + u * NT + tid;
                    if (i < K4) {
                        uint32_t ok = 0xffffffffu;
                        uint32_t q = a8_pack4_fast2(v[m][u], rr, ok);
                        // rare: a possible tie (or a tiny scale): the exact quotient decides
                        if (all_exact || (ok >> 31) == 0u) q = a8_pack4_exact(v[m][u], ks[m]);
                        dst[i] = q;
                        if (gout) gout[i] = q;
                        if constexpr (kCodeSums) tsum[m] += bytesum(q);
                    }
                }
            }
        }
    }
}

// Fused prologue, whole x in registers: NIT float4 per thread and token
// (a compile-time bound, so no predicated-off iterations are issued).
// Loads x, reduces the absmax over the block, and writes the int8 codes to
// shared memory (and, from block 0, to qx_out); tsum gets this thread's code
// sums.  Contains one block barrier; every thread must call it.
//
// kNorm: RMSNorm in front of the quantizer (fusion.cuh).  The norm weight
// does not depend on the previous kernel: it is loaded first and the
// dependency wait (griddepcontrol.wait) is taken here, after those loads are
// in flight and before x is read.  Each token's compensated sum of squares is
// reduced over the block through nrm_s (2 * (NT / 32) * MT floats, free until the
// first merge), then x is normalized in registers.  One more block barrier.
template <int MT, int NIT, bool kCodeSums, bool kNorm = false, int kBar = 0, int NT = kThreads>
__device__ __forceinline__ void fused_prologue_regs(const GemvArgs& a, int nit, float* red_s, float* sx_s,
                                                    int8_t* xs, int (&tsum)[MT], float* nrm_s = nullptr)
{
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int M = a.M;
    const int K = a.K;
    const int K4 = K >> 2;
    float4 gv[kNorm ? NIT : 1];
    if constexpr (kNorm) {
        const float4* gr = reinterpret_cast<const float4*>(a.gamma);
#pragma unroll
        for (int it = 0; it < NIT; ++it) {
            const int i = tid + it * NT;
            gv[it] = (it < nit && i < K4) ? __ldg(gr + i) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        pdl_wait();
    }
    float4 v[MT][NIT];
#pragma unroll
    for (int m = 0; m < MT; ++m) {
        const float4* xr = reinterpret_cast<const float4*>(a.x + static_cast<size_t>(m) * K);
#pragma unroll
        for (int it = 0; it < NIT; ++it) {
            const int i = tid + it * NT;
            v[m][it] = (m < M && it < nit && i < K4) ? __ldcg(xr + i) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
    if constexpr (kNorm) {
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            float hi = 0.0f, lo = 0.0f;
#pragma unroll
            for (int it = 0; it < NIT; ++it) sq_acc4(v[m][it], hi, lo);
            warp_pair_sum(hi, lo);
            if (lane == 0) {
                nrm_s[(warp * MT + m) * 2] = hi;
                nrm_s[(warp * MT + m) * 2 + 1] = lo;
            }
        }
        block_sync<kBar, NT>();
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            float hi = nrm_s[m * 2], lo = nrm_s[m * 2 + 1];
#pragma unroll
            for (int w = 1; w < (NT / 32); ++w) pair_merge(hi, lo, nrm_s[(w * MT + m) * 2], nrm_s[(w * MT + m) * 2 + 1]);
            const float r = rms_scale(hi, lo, K, a.eps);
#pragma unroll
            for (int it = 0; it < NIT; ++it) v[m][it] = rms_apply(v[m][it], r, gv[it]);
        }
    }
#pragma unroll
    for (int m = 0; m < MT; ++m) {
        float mx = 0.0f;
#pragma unroll
        for (int it = 0; it < NIT; ++it)
            mx = fmaxf(mx, fmaxf(fmaxf(fabsf(v[m][it].x), fabsf(v[m][it].y)), fmaxf(fabsf(v[m][it].z), fabsf(v[m][it].w))));
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
        if (lane == 0) red_s[warp * MT + m] = mx;
    }
    block_sync<kBar, NT>();
#pragma unroll
    for (int m = 0; m < MT; ++m) {
        if (m < M) {
            float amax = red_s[m];
#pragma unroll
            for (int w = 1; w < (NT / 32); ++w) amax = fmaxf(amax, red_s[w * MT + m]);
            const A8Scale ks = a8_scale(amax);
            if (tid == m) {
                sx_s[m] = ks.s;
                if (blockIdx.x == 0 && a.sx_out != nullptr) a.sx_out[m] = ks.s;
            }
            uint32_t* dst = reinterpret_cast<uint32_t*>(xs + static_cast<size_t>(m) * K);
            uint32_t* gout = (blockIdx.x == 0 && a.qx_out != nullptr)
                                 ? reinterpret_cast<uint32_t*>(a.qx_out + static_cast<size_t>(m) * K)
                                 : nullptr;
            const uint32_t all_exact = a8_needs_exact(ks) ? 0xffffffffu : 0u;
            const uint64_t rr = f2_pack(ks.r, ks.r);
            // Groups of kG words: the fast codes of a group are straight-line code
            // (independent chains, no branch between them); words with a possible
            // tie (or every word, for a tiny scale) are then redone exactly from
            // the values still in registers.
            constexpr int kG = NIT < 5 ? NIT : 5;
#pragma unroll
            for (int g0 = 0; g0 < NIT; g0 += kG) {
                uint32_t qw[kG];
                uint32_t need = all_exact;
#pragma unroll
                for (int u = 0; u < kG; ++u) {
                    uint32_t ok = 0xffffffffu;
                    if (g0 + u < NIT) qw[u] = a8_pack4_fast2(v[m][g0 + u], rr, ok);
                    need |= ((~ok) >> 31) << u;
                }
                if (need) {
#pragma unroll
                    for (int u = 0; u < kG; ++u)
                        if (g0 + u < NIT && ((need >> u) & 1u)) qw[u] = a8_pack4_exact(v[m][g0 + u], ks);
                }
#pragma unroll
                for (int u = 0; u < kG; ++u) {
                    const int it = g0 + u;
                    const int i = tid + it * NT;
                    if (it < NIT && it < nit && i < K4) {
                        dst[i] = qw[u];
                        if (gout) gout[i] = qw[u];
                        if constexpr (kCodeSums) tsum[m] += bytesum(qw[u]);
                    }
                }
            }
        } else if (tid == m) {
            sx_s[m] = 0.0f;
        }
    }
}

// Tile range of this block in one linear: an even split of the T tiles over
// the grid's clusters of ks blocks (ks = 1 without K splits; the host passes
// T = tq * clusters + tr), processed in rounds of at most RT tiles.
struct BlockRange {
    int t0, ntiles, nrounds;
};

template <int RT, bool KS = false>
__device__ __forceinline__ BlockRange block_range(const GemvArgs& a)
{
    const int ks = KS ? a.ks : 1;                    // K splits share their cluster's range
    const int nb = static_cast<int>(gridDim.x) / ks;
    int b = static_cast<int>(blockIdx.x) / ks + a.rot;
    if (b >= nb) b -= nb;
    const int n = a.tq + (b < a.tr ? 1 : 0);
    return BlockRange{b * a.tq + min(b, a.tr), n, (n + RT - 1) / RT};
}

// Warp w's line range [lo, hi) within a round of nt tiles of C lines: an even
// split, boundaries rounded down to whole 16-line passes.
__device__ __forceinline__ void warp_lines(int warp, int nt, int C, int& lo, int& hi, int nw = kWarps)
{
    const long long nL = static_cast<long long>(nt) * C;
    lo = static_cast<int>((warp * nL / nw) & ~15LL);
    hi = warp == nw - 1 ? static_cast<int>(nL) : static_cast<int>(((warp + 1) * nL / nw) & ~15LL);
}

// One linear per launch, launched with programmatic dependent launch: two
// blocks per SM, so the next GEMV's blocks become resident beside this one's
// and fill their rings before the dependency resolves.
//
// KS: K split over a cluster of P.lin[0].ks blocks (a separate instantiation,
// so the unsplit kernel keeps none of the split's bookkeeping).
template <int FMT, int MT, int XM, bool KS>
__global__ void __launch_bounds__(kThreads, 2) stream_linear_kernel(const __grid_constant__ ChainParams<1> P)
{
    using Acc = typename std::conditional<FMT == FMT_W4, int, float>::type;
    constexpr int kUnit = fmt_unit_bytes(FMT);
    constexpr int kLineBytes = kRows * kUnit;
    constexpr int kSL = fmt_slice_lines(FMT);
    constexpr int kSlotW = fmt_slot_w_bytes(FMT);
    constexpr int kSlot = fmt_slot_bytes(FMT);
    constexpr bool kGroup = fmt_group(FMT);
    constexpr int kHi = fmt_hi_bytes(FMT);           // Q6G32 high-part plane, bytes per unit
    constexpr int kSlotH = fmt_slot_h_bytes(FMT);
    constexpr bool kCodeSums = FMT == FMT_W4;        // activation code sums for the nibble bias
    constexpr int kPassLines = 16;
    constexpr int kPassUnroll = MT == 1 ? kSL / kPassLines : 1;
    constexpr int kRowBufs = 1;                      // per-row parameter buffers
    constexpr int kRowCap = kRowCache;               // rows per buffer
    // up to four tokens take the RMSNorm prologue when a.gamma is set (one
    // kernel for both, so alternating launches share code)
    constexpr bool kNormable = XM == X_FUSED && MT <= 4;

    extern __shared__ __align__(128) uint8_t smem[];
    const int S = P.stages;
    constexpr int RT = kAccWords / MT;               // tiles per round (the host sets P.round_tiles to this)
    constexpr int NL = 1;
    const int M = P.lin[0].M;
    // K split: this block's rank in its cluster and its chunk range [c0, c0 + Cr)
    const int kspl = KS ? P.lin[0].ks : 1;
    const int krank = KS ? static_cast<int>(blockIdx.x) % kspl : 0;
    const int c0 = KS ? static_cast<int>(static_cast<long long>(krank) * P.lin[0].C / kspl) : 0;
    const int Cr = KS ? static_cast<int>(static_cast<long long>(krank + 1) * P.lin[0].C / kspl) - c0 : P.lin[0].C;
    const SmemLayout L = smem_layout(FMT, MT, XM, P.kmax, S, RT, kRowBufs, kRowCap, kspl);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.bars);
    float* sx_s = reinterpret_cast<float*>(smem + L.sx);
    float* red_s = reinterpret_cast<float*>(smem + L.red);
    int* xsum_s = reinterpret_cast<int*>(smem + L.xsum);      // [kWarps][MT] partial code sums (W4)
    float* rowp_s = reinterpret_cast<float*>(smem + L.rowp);  // [kRowBufs][bias | s_w][kRowCache]
    int* meta_s = reinterpret_cast<int*>(smem + L.meta);
    Acc* acc_s = reinterpret_cast<Acc*>(smem + L.acc);
    Acc* bnd_s = reinterpret_cast<Acc*>(smem + L.bnd);
    Acc* mrg_s = reinterpret_cast<Acc*>(smem + L.merge);       // [kspl][MT][RT rows]: own sums, then other ranks'
    uint8_t* ring = smem + L.ring;
    int8_t* xs = reinterpret_cast<int8_t*>(smem + L.xs);

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;

    // ---- per-warp ring of bulk-copy slots
    uint8_t* my_ring = ring + static_cast<size_t>(warp) * S * kSlot;
    const uint32_t my_bars = smem_u32(bars + warp * S);
    if (lane == 0) {
        for (int s = 0; s < S; ++s) mbar_init(my_bars + 8 * s, 1);
        fence_mbar_init();
    }
    __syncwarp();
    pdl_launch_dependents();   // the next kernel may become resident beside this one
    const uint64_t pol = l2_policy_evict_first();

    // Slice cursor over this warp's work: linear, round, line position in the
    // round's range, and (tile, chunk) of that position, advanced without
    // division; the TMA cursor fills the ring ahead of the consumer.
    struct Cursor {
        int lin, round, p, hi, tl, c;
        BlockRange r;
        bool done;
    };
    // (lines of a tile: this block's Cr chunks of it)
    auto enter_round = [&](Cursor& k) {
        warp_lines(warp, min(RT, k.r.ntiles - k.round * RT), Cr, k.p, k.hi);
        k.tl = k.p / Cr;
        k.c = k.p - k.tl * Cr;
    };
    auto cursor_start = [&](Cursor& k) {
        k.lin = 0;
        k.round = 0;
        k.done = false;
        k.r = block_range<RT, KS>(P.lin[0]);
        if (k.r.nrounds > 0) enter_round(k);
    };
    // Next slice of the cursor: linear index, first unit, lines.  False at the end.
    auto cursor_next = [&](Cursor& k, int& lin, size_t& unit0, int& n) -> bool {
        while (!k.done) {
            if (k.round < k.r.nrounds && k.p < k.hi) {
                const int C = P.lin[k.lin].C;
                n = min(min(k.hi - k.p, Cr - k.c), kSL);
                lin = k.lin;
                unit0 = (static_cast<size_t>(k.r.t0 + k.round * RT + k.tl) * C + c0 + k.c) * kRows;
                k.p += n;
                k.c += n;
                if (k.c == Cr) {
                    k.c = 0;
                    ++k.tl;
                }
                return true;
            }
            // next round of this linear, else the next linear with work for this block
            if (k.round < k.r.nrounds) ++k.round;
            while (k.round >= k.r.nrounds) {
                if (++k.lin >= NL) {
                    k.done = true;
                    return false;
                }
                k.r = block_range<RT, KS>(P.lin[k.lin]);
                k.round = 0;
            }
            enter_round(k);
        }
        return false;
    };

    Cursor icur;
    cursor_start(icur);
    int issued = 0, islot = 0;
    auto issue_next = [&]() -> bool {
        int lin, n;
        size_t unit0;
        if (!cursor_next(icur, lin, unit0, n)) return false;
        if (lane == 0) {
            const GemvArgs& ia = P.lin[lin];
            uint8_t* dst = my_ring + static_cast<size_t>(islot) * kSlot;
            const uint32_t bar = my_bars + 8 * islot;
            const uint32_t bw = static_cast<uint32_t>(n * kLineBytes);
            const uint32_t bs = kGroup ? static_cast<uint32_t>(n * kRows * 2) : 0u;
            const uint32_t bh = static_cast<uint32_t>(n * kRows * kHi);
            if (issued >= S) fence_proxy_async_smem();   // the slot was read before
            mbar_arrive_expect_tx(bar, bw + bh + bs);
            bulk_g2s(smem_u32(dst), ia.w + unit0 * kUnit, bw, bar, pol);
            if (kHi > 0) bulk_g2s(smem_u32(dst + kSlotW), ia.whi + unit0 * kHi, bh, bar, pol);
            if (kGroup) bulk_g2s(smem_u32(dst + kSlotW + kSlotH), ia.wscale + unit0, bs, bar, pol);
        }
        ++issued;
        if (++islot == S) islot = 0;
        return true;
    };
    const int ahead = S;
    int consumed = 0;

    // one copy of the issue code (not unrolled): it runs once per launch,
    // before the dependency wait, and its footprint costs instruction fetch
#pragma unroll 1
    for (int s = 0; s < ahead; ++s)
        if (!issue_next()) break;

    // Per-row epilogue parameters of linear li into buffer li % kRowBufs:
    // asynchronous 4-byte copies, complete after cp_async_wait_all().
    auto stage_rows = [&](int li) {
        const GemvArgs& ra = P.lin[li];
        const BlockRange rr = block_range<RT, KS>(ra);
        if (rr.ntiles * kRows > kRowCap) return;
        float* b_s = rowp_s + (li & (kRowBufs - 1)) * 2 * kRowCap;
        float* w_s = b_s + kRowCap;
        const int r0 = rr.t0 * kRows;
        for (int i = tid; i < rr.ntiles * kRows; i += kThreads) {
            const int row = r0 + i;
            const int prow = ra.glu != GLU_NONE ? glu_param_row(row, ra.n_out) : (row < ra.N ? row : -1);
            if (prow >= 0) {
                if (ra.bias != nullptr) cp_async4(b_s + i, ra.bias + prow); else b_s[i] = 0.0f;
                if constexpr (fmt_row_scale(FMT)) cp_async4(w_s + i, ra.s_w + prow);
            }
        }
    };
    stage_rows(0);

    bool dead = false;      // a bounded wait ran out: stop computing, keep the barrier count
    int observed = 0;       // slices whose copy was seen complete
    int cslot = 0;          // consumer position in the ring, and the parity of its phase
    uint32_t cphase = 0;
    int round_count = 0;    // rounds so far over all linears (selects the merge buffers)

    const int h = lane & 1;               // rows 4h .. 4h+3
    const int pl = lane >> 1;             // line within a pass
    const int pp = pl & 3;                // read-order permutation
    const int my_row = 4 * h + pp;        // row held after the tile-end butterfly (lanes < 8)

    for (int li = 0; li < NL; ++li) {
        const GemvArgs& a = P.lin[li];
        const int K = a.K;
        const BlockRange br = block_range<RT, KS>(a);
        const int t0 = br.t0;
        const int ntiles = br.ntiles;
        const int nrounds = br.nrounds;

        // this linear's per-row parameters were staged one linear ahead
        float* bias_s = rowp_s + (li & (kRowBufs - 1)) * 2 * kRowCap;
        float* sw_s = bias_s + kRowCap;
        const int row0 = t0 * kRows;
        const bool rows_cached = ntiles * kRows <= kRowCap;

        // ---- inputs produced by earlier kernels are read only from here on
        // (with the RMSNorm prologue the wait is taken inside it, after the
        // norm weight loads)
        if (!(kNormable && a.gamma != nullptr)) pdl_wait();
        cp_async_wait_all();

        // ---- activation prologue: int8 codes into shared memory (fused: quantize
        // here) and, for W4, per-thread code sums that the epilogue reduces.  All
        // loads of a token are issued before any store, so one memory round trip
        // covers the vector; two block barriers in all.
        const int K4 = K >> 2;
        const int nit = (K4 + kThreads - 1) / kThreads;
        int tsum[MT];
#pragma unroll
        for (int m = 0; m < MT; ++m) tsum[m] = 0;

        bool normed = false;
        if constexpr (kNormable) {
            if (a.gamma != nullptr) {
                // RMSNorm, then the quantizer; x and the norm weight in registers
                // (the host asks for it only when nit <= norm_max_nit(MT))
                constexpr int kIt = norm_max_nit(MT);
                constexpr int kN1 = kIt < 2 ? kIt : 2;
                constexpr int kN2 = kIt < 4 ? kIt : 4;
                float* nrm_s = reinterpret_cast<float*>(acc_s);
                if (nit <= kN1)
                    fused_prologue_regs<MT, kN1, kCodeSums, true>(a, nit, red_s, sx_s, xs, tsum, nrm_s);
                else if (nit <= kN2)
                    fused_prologue_regs<MT, kN2, kCodeSums, true>(a, nit, red_s, sx_s, xs, tsum, nrm_s);
                else
                    fused_prologue_regs<MT, kIt, kCodeSums, true>(a, nit, red_s, sx_s, xs, tsum, nrm_s);
                normed = true;
            }
        }
        if (normed) {
        } else if constexpr (XM == X_F32) {
            // float activations, not quantized: into shared memory with each
            // 32-value chunk's eight float4 XOR-swizzled by (chunk & 7), so the
            // 16 lines of a pass read 8 distinct bank groups
            float4* xs4 = reinterpret_cast<float4*>(xs);
            const float4* xg = reinterpret_cast<const float4*>(a.x);
            const int n4 = M * K4;
            for (int i0 = tid; i0 < n4; i0 += 4 * kThreads) {
                float4 t[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int i = i0 + u * kThreads;
                    t[u] = i < n4 ? __ldcg(xg + i) : make_float4(0.f, 0.f, 0.f, 0.f);
                }
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int i = i0 + u * kThreads;
                    if (i < n4) {
                        const int m = i / K4;
                        const int f = i - m * K4;
                        const int c = f >> 3;
                        xs4[m * K4 + (c << 3) + ((f & 7) ^ (c & 7))] = t[u];
                    }
                }
            }
        } else if constexpr (XM == X_FUSED) {
            constexpr int kRegF4 = 20;                  // float4 of x held per thread
            constexpr int kIt = kRegF4 / MT;            // per token
            constexpr int kB1 = kIt / 5 > 0 ? kIt / 5 : 1;
            constexpr int kB2 = 2 * kIt / 5 > 0 ? 2 * kIt / 5 : 1;
            constexpr int kB3 = 3 * kIt / 5 > 0 ? 3 * kIt / 5 : 1;
            if (nit <= kB1) {
                fused_prologue_regs<MT, kB1, kCodeSums>(a, nit, red_s, sx_s, xs, tsum);
            } else if (nit <= kB2) {
                fused_prologue_regs<MT, kB2, kCodeSums>(a, nit, red_s, sx_s, xs, tsum);
            } else if (nit <= kB3) {
                fused_prologue_regs<MT, kB3, kCodeSums>(a, nit, red_s, sx_s, xs, tsum);
            } else if (nit <= kIt) {
                fused_prologue_regs<MT, kIt, kCodeSums>(a, nit, red_s, sx_s, xs, tsum);
            } else {
                fused_prologue_twopass<MT, kCodeSums>(a, red_s, sx_s, xs, tsum);
            }
        } else {
            if (tid < MT) sx_s[tid] = tid < M ? a.sx_in[tid] : 0.0f;
            // int8 codes from global memory: into shared memory (smem mode), summed for W4
            if (XM == X_SMEM || kCodeSums) {
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    if (m < M) {
                        const uint32_t* qr = reinterpret_cast<const uint32_t*>(a.qx_in + static_cast<size_t>(m) * K);
                        uint32_t* dst = reinterpret_cast<uint32_t*>(xs + static_cast<size_t>(m) * K);
                        for (int i0 = 0; i0 < K4; i0 += 4 * kThreads) {
                            uint32_t b4[4];
#pragma unroll
                            for (int u = 0; u < 4; ++u) {
                                const int i = i0 + u * kThreads + tid;
                                b4[u] = i < K4 ? __ldg(qr + i) : 0u;
                            }
#pragma unroll
                            for (int u = 0; u < 4; ++u) {
                                const int i = i0 + u * kThreads + tid;
                                if (i < K4) {
                                    if constexpr (XM == X_SMEM) dst[i] = b4[u];
                                    if constexpr (kCodeSums) tsum[m] += bytesum(b4[u]);
                                }
                            }
                        }
                    }
                }
            }
        }
        if constexpr (kCodeSums) {
#pragma unroll
            for (int m = 0; m < MT; ++m) {
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) tsum[m] += __shfl_xor_sync(0xffffffffu, tsum[m], off);
                if (lane == 0) xsum_s[warp * MT + m] = tsum[m];
            }
        }
        __syncthreads();

        // Activation chunk (32 int8) of token m at chunk c of this block's K
        // range (the bases start at its first chunk, c0, so the loop keeps no
        // offset of its own).
        const int8_t* xs_k = xs + c0 * 32;
        const int8_t* qg_k = XM == X_GLOBAL ? a.qx_in + c0 * 32 : nullptr;
        auto load_x = [&](int m, int c, uint4& x0, uint4& x1) {
            if constexpr (XM == X_GLOBAL) {
                const uint4* p = reinterpret_cast<const uint4*>(qg_k + static_cast<size_t>(m) * K + c * 32);
                x0 = __ldg(p);
                x1 = __ldg(p + 1);
            } else {
                const uint4* p = reinterpret_cast<const uint4*>(xs_k + static_cast<size_t>(m) * K + c * 32);
                x0 = p[0];
                x1 = p[1];
            }
        };

        // acc[m][j]: row 4h + (j ^ pp) of the current tile, token m (W4: the
        // low-nibble sums; accA the high-nibble sums, folded in at tile end)
        // (up to four tokens; more keep one sum per row and token)
        constexpr bool kSplitAcc = FMT == FMT_W4 && MT <= 4;
        Acc acc[MT][4];
        int accA[kSplitAcc ? MT : 1][4];
#pragma unroll
        for (int m = 0; m < MT; ++m)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                acc[m][j] = Acc(0);
                if constexpr (kSplitAcc) accA[m][j] = 0;
            }

        for (int round = 0; round < nrounds; ++round, ++round_count) {
            const int buf = round_count & 1;
            int lo, hi;
            warp_lines(warp, min(RT, ntiles - round * RT), Cr, lo, hi);
            int* meta = meta_s + (buf * kWarps + warp) * 2;
            if (lane == 0) {
                meta[0] = -1;
                meta[1] = -1;
            }
            __syncwarp();

            int p = lo;
            int tl = lo / Cr;
            int c = lo - tl * Cr;
            while (p < hi) {
                const int n = min(min(hi - p, Cr - c), kSL);
                const int slot = cslot;
                if (!dead) {
                    // a non-blocking test first: the slot has usually landed already
                    bool ok = __all_sync(0xffffffffu, mbar_test_wait(my_bars + 8 * slot, cphase));
                    if (!ok) ok = __all_sync(0xffffffffu, mbar_wait_bounded(my_bars + 8 * slot, cphase, kWaitTimeoutNs));
                    if (ok) {
                        ++observed;
                    } else {
                        dead = true;   // warp-uniform from here on
                        if (lane == 0 && P.err != nullptr) atomicExch(P.err, kErrWaitTimeout);
                    }
                }
                if (!dead) {
                    const uint8_t* sw = my_ring + static_cast<size_t>(slot) * kSlot;
                    const __half* sd = reinterpret_cast<const __half*>(sw + kSlotW + kSlotH);
                    // several tokens: the passes of a slice share one loop body (unrolled,
                    // their bodies outgrow the instruction cache); one token: unrolled
#pragma unroll kPassUnroll
                    for (int pass = 0; pass < kSL / kPassLines; ++pass) {
                        const int line = pass * kPassLines + pl;
                        if (line < n) {
                            // chunk within this block's K range (absolute for the float-x
                            // formats, whose x layout swizzles by chunk; they never split K)
                            const int chunk = (fmt_float_x(FMT) ? c0 : 0) + c + line;
                            const uint8_t* ub = sw + (line * kRows + 4 * h) * kUnit;
                            if constexpr (fmt_float_x(FMT)) {
                                // weight-only on float x: every weight unpacked to fp32 and
                                // multiply-added (the pages' float path), f32x2 pairs
                                const float4* xs4 = reinterpret_cast<const float4*>(xs);
                                const int swz = chunk & 7;
                                uint4 w0[4], w1[4];
#pragma unroll
                                for (int j = 0; j < 4; ++j) {
                                    if constexpr (FMT == FMT_W4F) {
                                        w0[j] = *reinterpret_cast<const uint4*>(ub + ((j ^ pp) << 4));
                                    } else {
                                        const uint8_t* u = ub + ((j ^ pp) << 5);
                                        const uint4 first = *reinterpret_cast<const uint4*>(u + (h << 4));
                                        const uint4 second = *reinterpret_cast<const uint4*>(u + ((h ^ 1) << 4));
                                        w0[j] = h ? second : first;
                                        w1[j] = h ? first : second;
                                    }
                                }
#pragma unroll
                                for (int m = 0; m < MT; ++m) {
                                    if (MT == 1 || m < M) {
                                        float4 xv[8];
                                        const float4* xp = xs4 + static_cast<size_t>(m) * (K >> 2) + chunk * 8;
#pragma unroll
                                        for (int k = 0; k < 8; ++k) xv[k] = xp[k ^ swz];
#pragma unroll
                                        for (int j = 0; j < 4; ++j) {
                                            uint64_t a2 = 0;
                                            uint64_t q01, q23;
                                            if constexpr (FMT == FMT_W4F) {
                                                // byte b of word w: weight 8w+b (low nibble), 8w+4+b (high)
                                                const uint64_t negb = f2_pack(-8388616.0f, -8388616.0f);
                                                const uint32_t wd[4] = {w0[j].x, w0[j].y, w0[j].z, w0[j].w};
#pragma unroll
                                                for (int w = 0; w < 4; ++w) {
                                                    byte_floats(wd[w] & 0x0F0F0F0Fu, negb, q01, q23);
                                                    a2 = fma4(q01, q23, xv[2 * w], a2);
                                                    byte_floats((wd[w] >> 4) & 0x0F0F0F0Fu, negb, q01, q23);
                                                    a2 = fma4(q01, q23, xv[2 * w + 1], a2);
                                                }
                                            } else {
                                                // byte i: weight i as int8; biased by 128 to 1..255
                                                const uint64_t negb = f2_pack(-8388736.0f, -8388736.0f);
                                                const uint32_t wd[8] = {w0[j].x, w0[j].y, w0[j].z, w0[j].w,
                                                                        w1[j].x, w1[j].y, w1[j].z, w1[j].w};
#pragma unroll
                                                for (int k = 0; k < 8; ++k) {
                                                    byte_floats(wd[k] ^ 0x80808080u, negb, q01, q23);
                                                    a2 = fma4(q01, q23, xv[k], a2);
                                                }
                                            }
                                            acc[m][j] = __fadd_rn(acc[m][j], __fadd_rn(__uint_as_float(f2_lo(a2)),
                                                                                       __uint_as_float(f2_hi(a2))));
                                        }
                                    }
                                }
                            } else if constexpr (FMT == FMT_Q6G32) {
                                // n = q + 32 = lo + 16 hi: sum n x from the two planes,
                                // minus 32 sum x, is the exact group sum of q x
                                const uint8_t* hb = sw + kSlotW + (line * kRows + 4 * h) * kHi;
                                uint4 wv[4];
                                uint2 hv[4];
                                float d[4];
#pragma unroll
                                for (int j = 0; j < 4; ++j) {
                                    wv[j] = *reinterpret_cast<const uint4*>(ub + ((j ^ pp) << 4));
                                    hv[j] = *reinterpret_cast<const uint2*>(hb + ((j ^ pp) << 3));
                                    d[j] = __half2float(sd[line * kRows + 4 * h + (j ^ pp)]);
                                }
#pragma unroll
                                for (int m = 0; m < MT; ++m) {
                                    if (MT == 1 || m < M) {
                                        uint4 x0, x1;
                                        load_x(m, chunk, x0, x1);
                                        int xs32 = bytesum(x0.x) + bytesum(x0.y) + bytesum(x0.z) + bytesum(x0.w);
                                        xs32 += bytesum(x1.x) + bytesum(x1.y) + bytesum(x1.z) + bytesum(x1.w);
#pragma unroll
                                        for (int j = 0; j < 4; ++j) {
                                            int B, A;
                                            unit4(wv[j], x0, x1, B, A);
                                            // high part of weight 16w+4s+b: word w, byte b, bits 2s..2s+1
                                            int s0 = dp4a_us(hv[j].x & 0x03030303u, x0.x, 0);
                                            s0 = dp4a_us(hv[j].y & 0x03030303u, x1.x, s0);
                                            int s1 = dp4a_us(hv[j].x & 0x0C0C0C0Cu, x0.y, 0);
                                            s1 = dp4a_us(hv[j].y & 0x0C0C0C0Cu, x1.y, s1);
                                            int s2 = dp4a_us(hv[j].x & 0x30303030u, x0.z, 0);
                                            s2 = dp4a_us(hv[j].y & 0x30303030u, x1.z, s2);
                                            int s3 = dp4a_us(hv[j].x & 0xC0C0C0C0u, x0.w, 0);
                                            s3 = dp4a_us(hv[j].y & 0xC0C0C0C0u, x1.w, s3);
                                            const int hs = s0 + (s1 >> 2) + (s2 >> 4) + (s3 >> 6);
                                            const int g = B + (A >> 4) + 16 * hs - 32 * xs32;
                                            acc[m][j] = __fmaf_rn(d[j], __int2float_rn(g), acc[m][j]);
                                        }
                                    }
                                }
                            } else if constexpr (FMT == FMT_I8G32) {
                                uint4 w0[4], w1[4];
                                float d[4];
#pragma unroll
                                for (int j = 0; j < 4; ++j) {
                                    const uint8_t* u = ub + ((j ^ pp) << 5);
                                    // the two halves are read in a lane-dependent order to spread banks
                                    const uint4 first = *reinterpret_cast<const uint4*>(u + (h << 4));
                                    const uint4 second = *reinterpret_cast<const uint4*>(u + ((h ^ 1) << 4));
                                    w0[j] = h ? second : first;
                                    w1[j] = h ? first : second;
                                    d[j] = __half2float(sd[line * kRows + 4 * h + (j ^ pp)]);
                                }
#pragma unroll
                                for (int m = 0; m < MT; ++m) {
                                    if (MT == 1 || m < M) {
                                        uint4 x0, x1;
                                        load_x(m, chunk, x0, x1);
#pragma unroll
                                        for (int j = 0; j < 4; ++j) {
                                            int g = dp4a_ss(w0[j].x, x0.x, 0);
                                            g = dp4a_ss(w0[j].y, x0.y, g);
                                            g = dp4a_ss(w0[j].z, x0.z, g);
                                            g = dp4a_ss(w0[j].w, x0.w, g);
                                            g = dp4a_ss(w1[j].x, x1.x, g);
                                            g = dp4a_ss(w1[j].y, x1.y, g);
                                            g = dp4a_ss(w1[j].z, x1.z, g);
                                            g = dp4a_ss(w1[j].w, x1.w, g);
                                            acc[m][j] = __fmaf_rn(d[j], __int2float_rn(g), acc[m][j]);
                                        }
                                    }
                                }
                            } else {
                                uint4 wv[4];
                                float d[4];
#pragma unroll
                                for (int j = 0; j < 4; ++j) {
                                    wv[j] = *reinterpret_cast<const uint4*>(ub + ((j ^ pp) << 4));
                                    if constexpr (FMT == FMT_Q4_0)
                                        d[j] = __half2float(sd[line * kRows + 4 * h + (j ^ pp)]);
                                }
#pragma unroll
                                for (int m = 0; m < MT; ++m) {
                                    if (MT == 1 || m < M) {
                                        uint4 x0, x1;
                                        load_x(m, chunk, x0, x1);
#pragma unroll
                                        for (int j = 0; j < 4; ++j) {
                                            if constexpr (kSplitAcc) {
                                                unit4_acc(wv[j], x0, x1, acc[m][j], accA[m][j]);
                                            } else if constexpr (FMT == FMT_W4) {
                                                int B, A;
                                                unit4(wv[j], x0, x1, B, A);
                                                acc[m][j] += B + (A >> 4);
                                            } else {
                                                const int g = unit4_signed16(wv[j], x0, x1) >> 4;
                                                acc[m][j] = __fmaf_rn(d[j], __int2float_rn(g), acc[m][j]);
                                            }
                                        }
                                    }
                                }
                            }
                        }
                    }
                }
                if (++cslot == S) {
                    cslot = 0;
                    cphase ^= 1u;
                }
                ++consumed;
                __syncwarp();
                if (!dead && issued - consumed < ahead) issue_next();   // refill the slot just released

                p += n;
                c += n;
                if (c == Cr || p == hi) {
                    // tile done for this warp: reduce lanes of equal (h, pp), then undo
                    // the read permutation with a two-step butterfly
#pragma unroll
                    for (int m = 0; m < MT; ++m) {
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            if constexpr (FMT == FMT_W4) {
                                if constexpr (kSplitAcc) {
                                    acc[m][j] += accA[m][j] >> 4;
                                    accA[m][j] = 0;
                                }
                                acc[m][j] += __shfl_xor_sync(0xffffffffu, acc[m][j], 8);
                                acc[m][j] += __shfl_xor_sync(0xffffffffu, acc[m][j], 16);
                            } else {
                                acc[m][j] = __fadd_rn(acc[m][j], __shfl_xor_sync(0xffffffffu, acc[m][j], 8));
                                acc[m][j] = __fadd_rn(acc[m][j], __shfl_xor_sync(0xffffffffu, acc[m][j], 16));
                            }
                        }
#pragma unroll
                        for (int j = 0; j < 2; ++j) {
                            const Acc v = __shfl_xor_sync(0xffffffffu, acc[m][j + 2], 4);
                            if constexpr (FMT == FMT_W4) acc[m][j] += v; else acc[m][j] = __fadd_rn(acc[m][j], v);
                        }
                        const Acc v = __shfl_xor_sync(0xffffffffu, acc[m][1], 2);
                        if constexpr (FMT == FMT_W4) acc[m][0] += v; else acc[m][0] = __fadd_rn(acc[m][0], v);
                    }
                    const int tstart = tl * Cr;
                    if (lane < kRows) {
                        const bool full = lo <= tstart && hi >= tstart + Cr;
                        Acc* dst;
                        if (full) {
                            dst = acc_s + (static_cast<size_t>(buf) * RT * kRows + tl * kRows + my_row) * MT;
                        } else {
                            const int which = (lo >= tstart && lo < tstart + Cr) ? 0 : 1;
                            dst = bnd_s + (((buf * kWarps + warp) * 2 + which) * kRows + my_row) * MT;
                            if (lane == 0) meta[which] = tl;
                        }
#pragma unroll
                        for (int m = 0; m < MT; ++m) dst[m] = acc[m][0];
                    }
#pragma unroll
                    for (int m = 0; m < MT; ++m)
#pragma unroll
                        for (int j = 0; j < 4; ++j) acc[m][j] = Acc(0);
                    if (c == Cr) {
                        c = 0;
                        ++tl;
                    }
                }
            }

            __syncthreads();

            // ---- epilogue for this round's rows (coalesced over rows)
            const int rt0 = round * RT;
            const int nrows = min(RT, ntiles - rt0) * kRows;
            const int row_base = (t0 + rt0) * kRows;
            // linear output of round row rl (kernel row `row`), token m
            // this block's sum for round row rl, token m (its warps' tiles merged in order)
            auto own_sum = [&](int m, int rl) -> Acc {
                const int tile = rl >> 3;
                const int rr = rl & 7;
                Acc v = Acc(0);
                bool part = false;
                for (int w = 0; w < kWarps; ++w) {
                    const int* mw = meta_s + (buf * kWarps + w) * 2;
#pragma unroll
                    for (int which = 0; which < 2; ++which) {
                        if (mw[which] == tile) {
                            const Acc pv = bnd_s[(((buf * kWarps + w) * 2 + which) * kRows + rr) * MT + m];
                            if constexpr (FMT == FMT_W4) v += pv; else v = __fadd_rn(v, pv);
                            part = true;
                        }
                    }
                }
                if (!part) v = acc_s[(static_cast<size_t>(buf) * RT * kRows + rl) * MT + m];
                return v;
            };
            // K splits: every rank writes its sums into the leader (rank 0), which adds
            // them in rank order; only the leader writes the outputs.
            constexpr int kRR = RT * kRows;                       // rows of a round, at most
            if constexpr (KS) {
                const uint32_t mrg_u = smem_u32(mrg_s);
                for (int idx = tid; idx < M * nrows; idx += kThreads) {
                    const int m = idx / nrows;
                    const int rl = idx - m * nrows;
                    const Acc v = own_sum(m, rl);
                    const int o = (krank * MT + m) * kRR + rl;
                    if (krank == 0) {
                        mrg_s[o] = v;
                    } else {
                        uint32_t bits;
                        if constexpr (FMT == FMT_W4) bits = static_cast<uint32_t>(v); else bits = __float_as_uint(v);
                        st_cluster_u32(mapa_shared(mrg_u + 4u * static_cast<uint32_t>(o), 0u), bits);
                    }
                }
                cluster_sync();
                if (krank == 0)
                    for (int idx = tid; idx < M * nrows; idx += kThreads) {
                        const int m = idx / nrows;
                        const int rl = idx - m * nrows;
                        Acc v = mrg_s[m * kRR + rl];
                        for (int r = 1; r < kspl; ++r) {
                            const Acc pv = mrg_s[(r * MT + m) * kRR + rl];
                            if constexpr (FMT == FMT_W4) v += pv; else v = __fadd_rn(v, pv);
                        }
                        mrg_s[m * kRR + rl] = v;
                    }
                cluster_sync();                                   // the ranks' buffers are free again
            }
            // linear output of round row rl (kernel row `row`), token m
            auto lin_out = [&](int m, int rl, int row) -> float {
                const Acc v = KS ? mrg_s[m * kRR + rl] : own_sum(m, rl);
                const int ci = row - row0;
                const int prow = a.glu != GLU_NONE ? glu_param_row(row, a.n_out) : row;
                const float b = rows_cached ? bias_s[ci] : (a.bias != nullptr ? a.bias[prow] : 0.0f);
                if constexpr (FMT == FMT_W4) {
                    int xsum = 0;
#pragma unroll
                    for (int w = 0; w < kWarps; ++w) xsum += xsum_s[w * MT + m];
                    const int accv = v - 8 * xsum;          // remove the +8 nibble bias
                    const float swr = rows_cached ? sw_s[ci] : a.s_w[prow];
                    return __fmaf_rn(__fmul_rn(swr, sx_s[m]), __int2float_rn(accv), b);
                } else if constexpr (fmt_row_scale(FMT)) {
                    const float swr = rows_cached ? sw_s[ci] : a.s_w[prow];
                    return __fmaf_rn(swr, v, b);
                } else {
                    return __fmaf_rn(sx_s[m], v, b);
                }
            };
            if (KS && krank != 0) {
                // another rank writes the outputs
            } else if (a.glu == GLU_NONE) {
                for (int idx = tid; idx < M * nrows; idx += kThreads) {
                    const int m = idx / nrows;
                    const int rl = idx - m * nrows;
                    const int row = row_base + rl;
                    if (row >= a.N) continue;
                    float out = lin_out(m, rl, row);
                    const size_t o = static_cast<size_t>(m) * a.N + row;
                    if (a.residual != nullptr) out = __fadd_rn(a.residual[o], out);
                    a.y[o] = out;
                }
            } else {
                // gated: output j pairs gate row 8(j/4) + j%4 with the up row 4 below it
                const int nout = nrows >> 1;
                const int j0 = row_base >> 1;
                for (int idx = tid; idx < M * nout; idx += kThreads) {
                    const int m = idx / nout;
                    const int jo = idx - m * nout;
                    const int j = j0 + jo;
                    if (j >= a.n_out) continue;
                    const int rlg = (jo >> 2) * kRows + (jo & 3);
                    const float g = lin_out(m, rlg, row_base + rlg);
                    const float u = lin_out(m, rlg + 4, row_base + rlg + 4);
                    float out = glu_act_call(a.glu, g, u);
                    const size_t o = static_cast<size_t>(m) * a.n_out + j;
                    if (a.residual != nullptr) out = __fadd_rn(a.residual[o], out);
                    a.y[o] = out;
                }
            }
            // accumulator and merge buffers alternate between rounds: no barrier here
        }
    }

    // ---- after a timeout: wait (bounded) for copies still in flight into this warp's ring
    if (dead) {
        for (int k = observed; k < issued; ++k) {
            const int slot = k % S;
            if (!mbar_wait_bounded(my_bars + 8 * slot, static_cast<uint32_t>(k / S) & 1u, kWaitTimeoutNs)) break;
        }
    }
}

template <int FMT, int MT, int XM, bool KS = false>
cudaError_t launch_gemv_t(const ChainParams<1>& p, int grid, size_t smem, bool pdl, cudaStream_t s)
{
    auto kern = stream_linear_kernel<FMT, MT, XM, KS>;
    static SmemLimit limit;
    cudaError_t e = raise_smem_limit(reinterpret_cast<const void*>(kern), limit, smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    int na = 0;
    if (pdl) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    if (KS) {                            // K splits: clusters of ks blocks
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = static_cast<unsigned>(p.lin[0].ks);
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    cfg.attrs = na ? attr : nullptr;
    cfg.numAttrs = static_cast<unsigned>(na);
    return cudaLaunchKernelEx(&cfg, kern, p);
}

template <int FMT>
cudaError_t launch_gemv_fmt(const ChainParams<1>& p, int MT, int xmode, int grid, size_t smem, bool pdl,
                            cudaStream_t s)
{
#define W4_CASE(mt)                                                                               \
    case mt:                                                                                      \
        return xmode == X_FUSED  ? launch_gemv_t<FMT, mt, X_FUSED>(p, grid, smem, pdl, s)         \
               : xmode == X_SMEM ? launch_gemv_t<FMT, mt, X_SMEM>(p, grid, smem, pdl, s)          \
                                 : launch_gemv_t<FMT, mt, X_GLOBAL>(p, grid, smem, pdl, s);
#define W4_SPLIT_CASE(mt)                                                                         \
    case mt:                                                                                      \
        return xmode == X_FUSED  ? launch_gemv_t<FMT, mt, X_FUSED, true>(p, grid, smem, pdl, s)   \
               : xmode == X_SMEM ? launch_gemv_t<FMT, mt, X_SMEM, true>(p, grid, smem, pdl, s)    \
                                 : launch_gemv_t<FMT, mt, X_GLOBAL, true>(p, grid, smem, pdl, s);
    // K splits: one and two tokens (kMaxSplitTokens)
    if (p.lin[0].ks > 1) {
        switch (MT) {
            W4_SPLIT_CASE(1)
            W4_SPLIT_CASE(2)
            default:
                return cudaErrorInvalidValue;
        }
    }
    switch (MT) {
        W4_CASE(1)
        W4_CASE(2)
        W4_CASE(4)
        W4_CASE(8)
        W4_CASE(16)
        default:
            return cudaErrorInvalidValue;
    }
#undef W4_CASE
#undef W4_SPLIT_CASE
}

}  // namespace w4k
