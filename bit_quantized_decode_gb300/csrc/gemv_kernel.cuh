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
//   * One persistent thread block per SM, 8 warps.  Each block owns a
//     contiguous, balanced range of 8-row tiles; the range is processed in
//     rounds and each round's lines (8 rows x 32 weights) are split evenly
//     among the warps, so every warp streams the same number of bytes.
//   * Every warp runs its own ring of shared-memory slots fed by 1-D bulk
//     (TMA) copies: lane 0 issues `cp.async.bulk` of whole slices of its
//     range with an evict-first L2 policy, the warp waits on the slot's
//     mbarrier (bounded wait), computes, and refills the slot.  The first
//     slices are issued before the dependency wait and the activation
//     prologue, so weight streaming overlaps both.
//   * Activations: either quantized in the prologue from fp32 x into shared
//     memory (each block repeats the absmax and the codes; block 0 also
//     writes them out), or read as int8 codes from global memory through L1.
//   * Inner loop: lane (l & 7) is a row, (l >> 3) a line; a 16-byte unit is
//     32 4-bit weights laid out so that (w << 4) & 0xF0F0F0F0 and
//     w & 0xF0F0F0F0 are four signed bytes each, 16 x the weights, fed
//     straight to DP4A against the matching int8 activations (the sum is a
//     multiple of 16 and is shifted back exactly at the end).  This is the
//     page's "unpack to two int8x4, two DP4A per 8 weights" (§"DP4A 做了什么")
//     with the sign extension folded into the byte position.
//   * Lanes sharing a row are reduced with shuffles; tiles split between
//     warps are merged in shared memory in warp order (deterministic), then
//     the epilogue writes y coalesced.
#pragma once
#include <cuda_fp16.h>

#include <type_traits>

#include "internal.h"
#include "ptx.cuh"

namespace w4k {

constexpr uint64_t kWaitTimeoutNs = 250ull * 1000ull * 1000ull;

template <int FMT, int MT>
struct UnitMath {
    using Acc = typename std::conditional<FMT == FMT_W4, int, float>::type;
};

// Quantize one activation: clip(rint(v / s), -127, 127); s == 0 gives 0.
__device__ __forceinline__ uint32_t quant_a8(float v, float s)
{
    if (s == 0.0f) return 0u;
    int q = __float2int_rn(__fdiv_rn(v, s));
    q = q > 127 ? 127 : (q < -127 ? -127 : q);
    return static_cast<uint32_t>(q) & 0xffu;
}

template <int FMT, int MT, bool FUSED>
__global__ void __launch_bounds__(kThreads, 1) gemv_kernel(const GemvArgs a)
{
    using Acc = typename UnitMath<FMT, MT>::Acc;
    constexpr int kUnit = fmt_unit_bytes(FMT);
    constexpr int kLineBytes = kRows * kUnit;
    constexpr int kSL = fmt_slice_lines(FMT);
    constexpr int kSlotW = fmt_slot_w_bytes(FMT);
    constexpr int kSlot = fmt_slot_bytes(FMT);
    constexpr bool kGroup = fmt_group(FMT);

    extern __shared__ __align__(128) uint8_t smem[];
    const int S = a.stages;
    const int RT = a.round_tiles;
    const SmemLayout L = smem_layout(FMT, MT, FUSED, a.K, S, RT);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.bars);
    float* sx_s = reinterpret_cast<float*>(smem + L.sx);
    float* red_s = reinterpret_cast<float*>(smem + L.red);
    int* meta_s = reinterpret_cast<int*>(smem + L.meta);
    Acc* acc_s = reinterpret_cast<Acc*>(smem + L.acc);
    Acc* bnd_s = reinterpret_cast<Acc*>(smem + L.bnd);
    uint8_t* ring = smem + L.ring;
    int8_t* xs = reinterpret_cast<int8_t*>(smem + L.xs);

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int C = a.C;
    const int M = a.M;
    const int K = a.K;

    // ---- this block's tiles and rounds
    const int G = gridDim.x;
    const int t0 = static_cast<int>((static_cast<long long>(blockIdx.x) * a.T) / G);
    const int t1 = static_cast<int>((static_cast<long long>(blockIdx.x + 1) * a.T) / G);
    const int ntiles = t1 - t0;
    const int nrounds = (ntiles + RT - 1) / RT;

    // Warp w's line range [lo, hi) within a round of nt tiles: an even split,
    // boundaries rounded down to whole passes of 4 lines.
    auto warp_range = [&](int round, int& lo, int& hi) {
        const int nt = min(RT, ntiles - round * RT);
        const int nL = nt * C;
        lo = static_cast<int>((static_cast<long long>(warp) * nL / kWarps) & ~3LL);
        hi = warp == kWarps - 1 ? nL : static_cast<int>((static_cast<long long>(warp + 1) * nL / kWarps) & ~3LL);
    };

    // ---- per-warp ring of bulk-copy slots
    uint8_t* my_ring = ring + static_cast<size_t>(warp) * S * kSlot;
    const uint32_t my_bars = smem_u32(bars + warp * S);
    if (lane == 0) {
        for (int s = 0; s < S; ++s) mbar_init(my_bars + 8 * s, 1);
        fence_mbar_init();
    }
    __syncwarp();
    const uint64_t pol = l2_policy_evict_first();

    // Issue iterator: walks this warp's slices, round by round.
    int is_round = 0, is_p = 0, is_hi = 0;
    if (nrounds > 0) warp_range(0, is_p, is_hi);
    int issued = 0;
    auto issue_next = [&]() -> bool {
        while (is_round < nrounds) {
            if (is_p < is_hi) {
                const int tl = is_p / C;
                const int e = min(min(is_hi, (tl + 1) * C), is_p + kSL);
                const int n = e - is_p;
                const int tile = t0 + is_round * RT + tl;
                const size_t unit0 = (static_cast<size_t>(tile) * C + (is_p - tl * C)) * kRows;
                if (lane == 0) {
                    const int slot = issued % S;
                    uint8_t* dst = my_ring + static_cast<size_t>(slot) * kSlot;
                    const uint32_t bar = my_bars + 8 * slot;
                    const uint32_t bw = static_cast<uint32_t>(n * kLineBytes);
                    const uint32_t bs = kGroup ? static_cast<uint32_t>(n * kRows * 2) : 0u;
                    fence_proxy_async_smem();
                    mbar_arrive_expect_tx(bar, bw + bs);
                    bulk_g2s(smem_u32(dst), a.w + unit0 * kUnit, bw, bar, pol);
                    if (kGroup) bulk_g2s(smem_u32(dst + kSlotW), a.wscale + unit0, bs, bar, pol);
                }
                ++issued;
                is_p = e;
                return true;
            }
            ++is_round;
            if (is_round < nrounds) warp_range(is_round, is_p, is_hi);
        }
        return false;
    };

    for (int s = 0; s < S; ++s)
        if (!issue_next()) break;

    // ---- inputs produced by earlier kernels are read only from here on
    pdl_wait();
    pdl_launch_dependents();

    // ---- activation prologue
    if constexpr (FUSED) {
        float mx[MT];
#pragma unroll
        for (int m = 0; m < MT; ++m) mx[m] = 0.0f;
        const int K4 = K >> 2;
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            if (m < M) {
                const float4* xr = reinterpret_cast<const float4*>(a.x + static_cast<size_t>(m) * K);
                for (int i = tid; i < K4; i += kThreads) {
                    const float4 v = __ldcg(xr + i);
                    mx[m] = fmaxf(mx[m], fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
                }
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) mx[m] = fmaxf(mx[m], __shfl_xor_sync(0xffffffffu, mx[m], off));
            if (lane == 0) red_s[warp * MT + m] = mx[m];
        }
        __syncthreads();
        if (tid < MT) {
            float amax = 0.0f;
            for (int w = 0; w < kWarps; ++w) amax = fmaxf(amax, red_s[w * MT + tid]);
            const float s = tid < M ? __fdiv_rn(amax, 127.0f) : 0.0f;
            sx_s[tid] = s;
            if (blockIdx.x == 0 && tid < M && a.sx_out != nullptr) a.sx_out[tid] = s;
        }
        __syncthreads();
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            uint32_t* dst = reinterpret_cast<uint32_t*>(xs + static_cast<size_t>(m) * K);
            if (m < M) {
                const float s = sx_s[m];
                const float4* xr = reinterpret_cast<const float4*>(a.x + static_cast<size_t>(m) * K);
                uint32_t* gout = (blockIdx.x == 0 && a.qx_out != nullptr)
                                     ? reinterpret_cast<uint32_t*>(a.qx_out + static_cast<size_t>(m) * K)
                                     : nullptr;
                for (int i = tid; i < K4; i += kThreads) {
                    const float4 v = __ldcg(xr + i);
                    const uint32_t q = quant_a8(v.x, s) | (quant_a8(v.y, s) << 8) | (quant_a8(v.z, s) << 16) |
                                       (quant_a8(v.w, s) << 24);
                    dst[i] = q;
                    if (gout) gout[i] = q;
                }
            } else {
                for (int i = tid; i < K4; i += kThreads) dst[i] = 0u;
            }
        }
    } else {
        if (tid < MT) sx_s[tid] = tid < M ? a.sx_in[tid] : 0.0f;
    }
    __syncthreads();

    // Activation chunk (32 int8) of token m at chunk c.
    auto load_x = [&](int m, int c, uint4& x0, uint4& x1) {
        if constexpr (FUSED) {
            const uint4* p = reinterpret_cast<const uint4*>(xs + static_cast<size_t>(m) * K + c * 32);
            x0 = p[0];
            x1 = p[1];
        } else {
            const uint4* p = reinterpret_cast<const uint4*>(a.qx_in + static_cast<size_t>(m) * K + c * 32);
            x0 = __ldg(p);
            x1 = __ldg(p + 1);
        }
    };

    Acc acc[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) acc[m] = Acc(0);

    bool dead = false;      // a bounded wait ran out: stop computing, keep the barrier count
    int consumed = 0;       // slices whose slot has been released
    int observed = 0;       // slices whose copy was seen complete
    const int r = lane & 7;

    for (int round = 0; round < nrounds; ++round) {
        const int buf = round & 1;
        int lo, hi;
        warp_range(round, lo, hi);
        int* meta = meta_s + (buf * kWarps + warp) * 2;
        if (lane == 0) {
            meta[0] = -1;
            meta[1] = -1;
        }
        __syncwarp();

        for (int p = lo; p < hi;) {
            const int tl = p / C;
            const int tend = (tl + 1) * C;
            const int e = min(min(hi, tend), p + kSL);
            const int n = e - p;
            const int c0 = p - tl * C;
            const int slot = consumed % S;
            const uint32_t parity = static_cast<uint32_t>(consumed / S) & 1u;

            if (!dead) {
                const bool ok = mbar_wait_bounded(my_bars + 8 * slot, parity, kWaitTimeoutNs);
                if (__all_sync(0xffffffffu, ok)) {
                    ++observed;
                } else {
                    dead = true;   // warp-uniform from here on
                    if (lane == 0 && a.err != nullptr) atomicExch(a.err, kErrWaitTimeout);
                }
            }
            if (!dead) {
                const uint8_t* sw = my_ring + static_cast<size_t>(slot) * kSlot;
                const __half* sd = reinterpret_cast<const __half*>(sw + kSlotW);
#pragma unroll 2
                for (int line = lane >> 3; line < n; line += 4) {
                    const int u = line * kRows + r;
                    const int chunk = c0 + line;
                    if constexpr (FMT == FMT_I8G32) {
                        const uint4 w0 = *reinterpret_cast<const uint4*>(sw + u * 32);
                        const uint4 w1 = *reinterpret_cast<const uint4*>(sw + u * 32 + 16);
                        const float d = __half2float(sd[u]);
#pragma unroll
                        for (int m = 0; m < MT; ++m) {
                            if (MT == 1 || m < M) {
                                uint4 x0, x1;
                                load_x(m, chunk, x0, x1);
                                int g = dp4a_ss(w0.x, x0.x, 0);
                                g = dp4a_ss(w0.y, x0.y, g);
                                g = dp4a_ss(w0.z, x0.z, g);
                                g = dp4a_ss(w0.w, x0.w, g);
                                g = dp4a_ss(w1.x, x1.x, g);
                                g = dp4a_ss(w1.y, x1.y, g);
                                g = dp4a_ss(w1.z, x1.z, g);
                                g = dp4a_ss(w1.w, x1.w, g);
                                acc[m] = __fmaf_rn(d, __int2float_rn(g), acc[m]);
                            }
                        }
                    } else {
                        const uint4 wv = *reinterpret_cast<const uint4*>(sw + u * 16);
                        // 16 x (weights 8w..8w+3) and 16 x (weights 8w+4..8w+7) as signed bytes
                        const uint32_t l0 = (wv.x << 4) & 0xF0F0F0F0u, h0 = wv.x & 0xF0F0F0F0u;
                        const uint32_t l1 = (wv.y << 4) & 0xF0F0F0F0u, h1 = wv.y & 0xF0F0F0F0u;
                        const uint32_t l2 = (wv.z << 4) & 0xF0F0F0F0u, h2 = wv.z & 0xF0F0F0F0u;
                        const uint32_t l3 = (wv.w << 4) & 0xF0F0F0F0u, h3 = wv.w & 0xF0F0F0F0u;
                        float d = 0.0f;
                        if constexpr (FMT == FMT_Q4_0) d = __half2float(sd[u]);
#pragma unroll
                        for (int m = 0; m < MT; ++m) {
                            if (MT == 1 || m < M) {
                                uint4 x0, x1;
                                load_x(m, chunk, x0, x1);
                                int g = dp4a_ss(l0, x0.x, 0);
                                g = dp4a_ss(h0, x0.y, g);
                                g = dp4a_ss(l1, x0.z, g);
                                g = dp4a_ss(h1, x0.w, g);
                                g = dp4a_ss(l2, x1.x, g);
                                g = dp4a_ss(h2, x1.y, g);
                                g = dp4a_ss(l3, x1.z, g);
                                g = dp4a_ss(h3, x1.w, g);
                                if constexpr (FMT == FMT_W4) {
                                    acc[m] += g;
                                } else {
                                    acc[m] = __fmaf_rn(d, __int2float_rn(g >> 4), acc[m]);
                                }
                            }
                        }
                    }
                }
            }
            ++consumed;
            __syncwarp();
            if (!dead) issue_next();   // refill the slot just released

            if (e == tend || e == hi) {
                // this warp is done with tile tl: reduce lanes of equal row
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    if constexpr (FMT == FMT_W4) {
                        acc[m] += __shfl_xor_sync(0xffffffffu, acc[m], 8);
                        acc[m] += __shfl_xor_sync(0xffffffffu, acc[m], 16);
                    } else {
                        acc[m] = __fadd_rn(acc[m], __shfl_xor_sync(0xffffffffu, acc[m], 8));
                        acc[m] = __fadd_rn(acc[m], __shfl_xor_sync(0xffffffffu, acc[m], 16));
                    }
                }
                if (lane < kRows) {
                    const bool full = lo <= tl * C && hi >= tend;
                    Acc* dst;
                    if (full) {
                        dst = acc_s + (static_cast<size_t>(buf) * RT * kRows + tl * kRows + lane) * MT;
                    } else {
                        const int which = (lo >= tl * C && lo < tend) ? 0 : 1;
                        dst = bnd_s + (((buf * kWarps + warp) * 2 + which) * kRows + lane) * MT;
                        if (lane == 0) meta[which] = tl;
                    }
#pragma unroll
                    for (int m = 0; m < MT; ++m) dst[m] = acc[m];
                }
#pragma unroll
                for (int m = 0; m < MT; ++m) acc[m] = Acc(0);
            }
            p = e;
        }

        __syncthreads();

        // ---- epilogue for this round's rows (coalesced over rows)
        const int rt0 = round * RT;
        const int nrows = min(RT, ntiles - rt0) * kRows;
        const int row_base = (t0 + rt0) * kRows;
        for (int idx = tid; idx < M * nrows; idx += kThreads) {
            const int m = idx / nrows;
            const int rl = idx - m * nrows;
            const int row = row_base + rl;
            if (row >= a.N) continue;
            const int tl = rl >> 3;
            const int rr = rl & 7;
            Acc v = Acc(0);
            bool part = false;
            for (int w = 0; w < kWarps; ++w) {
                const int* mw = meta_s + (buf * kWarps + w) * 2;
#pragma unroll
                for (int which = 0; which < 2; ++which) {
                    if (mw[which] == tl) {
                        const Acc pv = bnd_s[(((buf * kWarps + w) * 2 + which) * kRows + rr) * MT + m];
                        if constexpr (FMT == FMT_W4) v += pv; else v = __fadd_rn(v, pv);
                        part = true;
                    }
                }
            }
            if (!part) v = acc_s[(static_cast<size_t>(buf) * RT * kRows + rl) * MT + m];
            const float b = a.bias != nullptr ? a.bias[row] : 0.0f;
            float out;
            if constexpr (FMT == FMT_W4) {
                out = __fmaf_rn(__fmul_rn(a.s_w[row], sx_s[m]), __int2float_rn(v >> 4), b);
            } else {
                out = __fmaf_rn(sx_s[m], v, b);
            }
            a.y[static_cast<size_t>(m) * a.N + row] = out;
        }
        // accumulator and merge buffers alternate between rounds: no barrier here
    }

    // ---- after a timeout: wait (bounded) for copies still in flight into this warp's ring
    if (dead) {
        for (int k = observed; k < issued; ++k) {
            const int slot = k % S;
            if (!mbar_wait_bounded(my_bars + 8 * slot, static_cast<uint32_t>(k / S) & 1u, kWaitTimeoutNs)) break;
        }
    }
}

template <int FMT, int MT, bool FUSED>
cudaError_t launch_gemv_t(const GemvArgs& a, int grid, size_t smem, bool pdl, cudaStream_t s)
{
    auto kern = gemv_kernel<FMT, MT, FUSED>;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    static int configured[64] = {0};
    if (dev < 64 && configured[dev] < static_cast<int>(smem)) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        configured[dev] = static_cast<int>(smem);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = pdl ? attr : nullptr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, a);
}

template <int FMT>
cudaError_t launch_gemv_fmt(const GemvArgs& a, int MT, bool fused, int grid, size_t smem, bool pdl, cudaStream_t s)
{
#define W4_CASE(mt)                                                                   \
    case mt:                                                                          \
        return fused ? launch_gemv_t<FMT, mt, true>(a, grid, smem, pdl, s)            \
                     : launch_gemv_t<FMT, mt, false>(a, grid, smem, pdl, s);
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
}

}  // namespace w4k
