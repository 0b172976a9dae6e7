// A decode step's chain of per-row INT4 linears in one persistent launch
// (w4a8_linear_chain).  What each linear computes is the fused decode linear
// of "Jetson Orin AGX INT4 推理优化实践", §"从 FP 线性层到 INT4 DP4A 的数学推导":
// per-token INT8 codes of x, exact int32 sums of INT4 x INT8 products on
// DP4A, y = fmaf(s_w s_x, acc, b) -- the same arithmetic, layout and inner
// loop as stream_linear_kernel (gemv_kernel.cuh), so results are identical.
//
// How the launch is organised (GB300 design, not the pages'):
//   * One block per SM, co-resident (cooperative launch): fifteen consumer
//     warps and one producer warp (sixteen warps keep 128 registers a thread).
//     Not eight consumers: the per-slice protocol (wait, vote, release,
//     tile-end reduction) and the loop's dependency chains leave eight warps
//     issuing half the time, and the consumers must outrun HBM by a wide
//     margin for the ring to pay off.
//   * The weights never depend on the activations, so the producer warp
//     streams them for every linear in order -- through the grid barriers
//     between linears and through each linear's activation prologue -- into
//     per-consumer-warp rings of 4 KB slots (1-D bulk copies, evict-first).
//     A slot is refilled once its consumer released it (empty mbarrier).
//     Shared memory holds only about 4 us of streaming per SM, less than the
//     dependency chains of two short linears in a row, so the producer also
//     prefetches a window of the coming slices into L2 (no completion
//     tracked): HBM keeps streaming while the ring is full, and the copies
//     that follow read L2.
//   * The consumers compute linear after linear: grid barrier (atomic count
//     over the blocks), activation quantization into shared memory, DP4A over
//     the ring, merge and epilogue.  Their barriers are a named barrier of
//     the consumer warps; the producer warp never joins one.
//   * Every wait is bounded; a wait that runs out records an error, stops the
//     producer and lets every warp finish without further work.
#include "gemv_kernel.cuh"

namespace w4k {

namespace {

constexpr int kConsumerBar = 1;                  // named barrier of the consumer warps
constexpr int kSliceLines = fmt_slice_lines(FMT_W4);
constexpr int kUnitBytes = fmt_unit_bytes(FMT_W4);
constexpr int kLineBytes = kRows * kUnitBytes;
constexpr int kSlotBytes = fmt_slot_bytes(FMT_W4);
constexpr uint64_t kChainWaitNs = 250ull * 1000ull * 1000ull;

// The slices (runs of at most kSliceLines lines of one tile) that consumer
// warp w takes, in order over the chain's linears and rounds: the consumer
// walks them with its own loop; the producer keeps one cursor per warp.
struct SliceCursor {
    int lin, round, p, hi, tl, c;
    BlockRange r;
    bool done;
};

template <int RT>
__device__ __forceinline__ void cursor_enter_round(SliceCursor& k, const ChainParams<kMaxChain>& P, int w)
{
    const int C = P.lin[k.lin].C;
    warp_lines(w, min(RT, k.r.ntiles - k.round * RT), C, k.p, k.hi, kChainWarps);
    k.tl = k.p / C;
    k.c = k.p - k.tl * C;
}

template <int RT>
__device__ __forceinline__ void cursor_start(SliceCursor& k, const ChainParams<kMaxChain>& P, int w)
{
    k.lin = 0;
    k.round = 0;
    k.done = false;
    k.r = block_range<RT>(P.lin[0]);
    if (k.r.nrounds > 0) cursor_enter_round<RT>(k, P, w);
}

// Next slice of warp w: linear, first unit, lines.  False when none is left.
template <int RT>
__device__ bool cursor_next(SliceCursor& k, const ChainParams<kMaxChain>& P, int w, int& lin, size_t& unit0, int& n)
{
    while (!k.done) {
        if (k.round < k.r.nrounds && k.p < k.hi) {
            const int C = P.lin[k.lin].C;
            n = min(min(k.hi - k.p, C - k.c), kSliceLines);
            lin = k.lin;
            unit0 = (static_cast<size_t>(k.r.t0 + k.round * RT + k.tl) * C + k.c) * kRows;
            k.p += n;
            k.c += n;
            if (k.c == C) {
                k.c = 0;
                ++k.tl;
            }
            return true;
        }
        if (k.round < k.r.nrounds) ++k.round;
        while (k.round >= k.r.nrounds) {
            if (++k.lin >= P.n) {
                k.done = true;
                return false;
            }
            k.r = block_range<RT>(P.lin[k.lin]);
            k.round = 0;
        }
        cursor_enter_round<RT>(k, P, w);
    }
    return false;
}

// The producer warp.  Lane w < kChainWarps streams the ring of consumer warp w, on
// its own: use u of the ring fills slot u % S once the consumer released
// use u - S (its empty barrier).  A second cursor over the same slices runs
// `ahead` slices in front of the copies and prefetches them into L2, so HBM
// keeps streaming while the ring is full -- during a grid barrier and the
// activation prologue, and through the short linears, whose weights take
// less time to stream than their dependency takes to resolve.  The copies
// then read those lines from L2.
template <int MT>
__device__ __noinline__ void chain_producer(const ChainParams<kMaxChain>& P, uint8_t* ring, uint32_t full0,
                                            uint32_t empty0, volatile int* stop_s)
{
    constexpr int RT = kAccWords / MT;
    const int lane = threadIdx.x & 31;
    if (lane >= kChainWarps) return;
    const int w = lane;
    const int S = P.stages;
    const int ahead = P.prefetch_slices;
    const uint64_t pol = l2_policy_evict_first();
    SliceCursor cur, pcur;
    cursor_start<RT>(cur, P, w);
    cursor_start<RT>(pcur, P, w);
    bool more = true;                          // slices left to copy
    bool pmore = ahead > 0;                    // slices left to prefetch
    int issued = 0, islot = 0, iwrap = 0;      // next use: slot, use / S
    int prefetched = 0;
    uint64_t idle_since = 0;
    bool failed = false;
#pragma unroll 1
    while (more) {
        if (*stop_s) break;
        bool progress = false;
        if (pmore && prefetched - issued < ahead) {
            int lin = 0, n = 0;
            size_t unit0 = 0;
            if (cursor_next<RT>(pcur, P, w, lin, unit0, n)) {
                bulk_prefetch_l2(P.lin[lin].w + unit0 * kUnitBytes, static_cast<uint32_t>(n * kLineBytes));
                ++prefetched;
                progress = true;
            } else {
                pmore = false;
            }
        }
        if (iwrap == 0 || mbar_test_wait(empty0 + 8 * (w * S + islot), static_cast<uint32_t>(iwrap - 1) & 1u)) {
            int lin = 0, n = 0;
            size_t unit0 = 0;
            if (cursor_next<RT>(cur, P, w, lin, unit0, n)) {
                const uint32_t bytes = static_cast<uint32_t>(n * kLineBytes);
                const uint32_t bar = full0 + 8 * (w * S + islot);
                if (iwrap > 0) fence_proxy_async_smem();   // the consumer's reads precede the refill
                mbar_arrive_expect_tx(bar, bytes);
                bulk_g2s(smem_u32(ring + static_cast<size_t>(w * S + islot) * kSlotBytes),
                         P.lin[lin].w + unit0 * kUnitBytes, bytes, bar, pol);
                ++issued;
                if (++islot == S) {
                    islot = 0;
                    ++iwrap;
                }
            } else {
                more = false;
            }
            progress = true;
        }
        if (progress) {
            idle_since = 0;
        } else if (idle_since == 0) {
            idle_since = globaltimer_ns();
        } else if (globaltimer_ns() - idle_since > kChainWaitNs) {
            failed = true;                   // the consumer stopped releasing slots
            break;
        }
    }
    if (failed) {
        *stop_s = 1;
        if (P.err != nullptr) atomicExch(P.err, kErrWaitTimeout);
    }
    // copies still in flight land before the block may exit: the last (at
    // most S) uses of the ring, each the latest use of its slot
    for (int u = issued > S ? issued - S : 0; u < issued; ++u)
        if (!mbar_wait_bounded(full0 + 8 * (w * S + u % S), static_cast<uint32_t>(u / S) & 1u, kChainWaitNs)) break;
}

// Grid barrier between linears (every block resident: cooperative launch):
// a block's consumers arrive once per finished linear; before linear li a
// block waits for li * gridDim.x arrivals.  Waits are bounded.
__device__ __forceinline__ void chain_arrive(unsigned* count)
{
    block_sync<kConsumerBar, kChainConsumers>();
    if (threadIdx.x == 0) red_add_release_gpu(count, 1u);
}

__device__ __forceinline__ bool chain_wait(const unsigned* count, unsigned target, unsigned* err, int* flag_s)
{
    if (threadIdx.x == 0) {
        bool ok = true;
        if (ld_acquire_gpu(count) < target) {
            const uint64_t t0 = globaltimer_ns();
            while (ld_acquire_gpu(count) < target) {
                if (globaltimer_ns() - t0 > kChainWaitNs) {
                    ok = false;
                    break;
                }
            }
        }
        __threadfence();
        if (!ok && err != nullptr) atomicExch(err, kErrBarrierTimeout);
        *flag_s = ok ? 1 : 0;
    }
    // thread 0's spin is divergent: reconverge warp 0 before the barrier
    // (bar.sync is the aligned form, which assumes a converged warp)
    __syncwarp();
    block_sync<kConsumerBar, kChainConsumers>();
    return *flag_s != 0;
}

template <int MT>
__global__ void __launch_bounds__(kChainThreads, 1) stream_chain_kernel(const __grid_constant__ ChainParams<kMaxChain> P)
{
    constexpr int RT = kAccWords / MT;              // tiles per round (the host sets P.round_tiles to this)
    constexpr int kRowCap = kRowCache / 2;          // rows per per-row parameter buffer
    constexpr int kPassLines = 16;
    constexpr int kPassUnroll = MT == 1 ? kSliceLines / kPassLines : 1;
    extern __shared__ __align__(128) uint8_t smem[];
    const int S = P.stages;
    const int NL = P.n;
    const int M = P.lin[0].M;
    const ChainLayout L = chain_layout(MT, P.kmax, S, RT);
    const uint32_t full0 = smem_u32(smem + L.full);
    const uint32_t empty0 = smem_u32(smem + L.empty);
    float* sx_s = reinterpret_cast<float*>(smem + L.sx);
    float* red_s = reinterpret_cast<float*>(smem + L.red);
    int* xsum_s = reinterpret_cast<int*>(smem + L.xsum);
    float* rowp_s = reinterpret_cast<float*>(smem + L.rowp);   // [2][bias | s_w][kRowCap]
    int* meta_s = reinterpret_cast<int*>(smem + L.meta);
    int* acc_s = reinterpret_cast<int*>(smem + L.acc);
    int* bnd_s = reinterpret_cast<int*>(smem + L.bnd);
    uint8_t* ring = smem + L.ring;
    int8_t* xs = reinterpret_cast<int8_t*>(smem + L.xs);
    __shared__ int flag_s;
    __shared__ volatile int stop_s;

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    if (tid == 0) {
        for (int i = 0; i < kChainWarps * S; ++i) {
            mbar_init(full0 + 8 * i, 1);
            mbar_init(empty0 + 8 * i, 1);
        }
        fence_mbar_init();
        stop_s = 0;
    }
    __syncthreads();                                // the only barrier of all nine warps
    if (warp == kChainWarps) {
        chain_producer<MT>(P, ring, full0, empty0, &stop_s);
        return;
    }

    // ---- consumer warps (256 threads)
    uint8_t* my_ring = ring + static_cast<size_t>(warp) * S * kSlotBytes;
    const uint32_t my_full = full0 + 8 * warp * S;
    const uint32_t my_empty = empty0 + 8 * warp * S;

    // per-row epilogue parameters of linear li into buffer li & 1 (asynchronous
    // 4-byte copies, complete after cp_async_wait_all())
    auto stage_rows = [&](int li) {
        const GemvArgs& ra = P.lin[li];
        const BlockRange rr = block_range<RT>(ra);
        if (rr.ntiles * kRows > kRowCap) return;
        float* b_s = rowp_s + (li & 1) * 2 * kRowCap;
        float* w_s = b_s + kRowCap;
        const int r0 = rr.t0 * kRows;
        for (int i = tid; i < rr.ntiles * kRows; i += kChainConsumers) {
            const int row = r0 + i;
            if (row < ra.N) {
                if (ra.bias != nullptr) cp_async4(b_s + i, ra.bias + row); else b_s[i] = 0.0f;
                cp_async4(w_s + i, ra.s_w + row);
            }
        }
    };
    stage_rows(0);

    bool dead = false;          // a bounded wait ran out: no more work, barrier arrivals kept
    int cslot = 0;              // consumer position in the ring and the parity of its phase
    uint32_t cphase = 0;
    int round_count = 0;        // rounds over all linears (selects the merge buffers)
    const int h = lane & 1;               // rows 4h .. 4h+3
    const int pl = lane >> 1;             // line within a pass
    const int pp = pl & 3;                // read-order permutation
    const int my_row = 4 * h + pp;        // row held after the tile-end butterfly (lanes < 8)

    for (int li = 0; li < NL; ++li) {
        const GemvArgs& a = P.lin[li];
        const int C = a.C;
        const int K = a.K;
        const BlockRange br = block_range<RT>(a);
        const int t0 = br.t0;
        const int ntiles = br.ntiles;
        const int nrounds = br.nrounds;

        // outputs of the previous linear are written: let the grid know, and
        // read this linear's inputs only once every block has done so
        if (li > 0) {
            chain_arrive(P.barrier);
            if (!chain_wait(P.barrier, static_cast<unsigned>(li) * gridDim.x, P.err, &flag_s) && !dead) {
                dead = true;
                stop_s = 1;
            }
        }
        float* bias_s = rowp_s + (li & 1) * 2 * kRowCap;
        float* sw_s = bias_s + kRowCap;
        const int row0 = t0 * kRows;
        const bool rows_cached = ntiles * kRows <= kRowCap;
        // the next linear's parameters go to the other buffer (its last reader,
        // linear li-1's epilogue, finished before the barrier above)
        cp_async_wait_all();
        if (li + 1 < NL) stage_rows(li + 1);

        // ---- activation prologue: int8 codes into shared memory, code sums
        const int K4 = K >> 2;
        const int nit = (K4 + kChainConsumers - 1) / kChainConsumers;
        int tsum[MT];
#pragma unroll
        for (int m = 0; m < MT; ++m) tsum[m] = 0;
        {
            constexpr int kRegF4 = 10;                  // float4 of x held per thread
            constexpr int kIt = kRegF4 / MT > 0 ? kRegF4 / MT : 1;   // per token
            constexpr int kB1 = kIt / 5 > 0 ? kIt / 5 : 1;
            constexpr int kB3 = 3 * kIt / 5 > 0 ? 3 * kIt / 5 : 1;
            if (nit <= kB1)
                fused_prologue_regs<MT, kB1, true, false, kConsumerBar, kChainConsumers>(a, nit, red_s, sx_s, xs, tsum);
            else if (nit <= kB3)
                fused_prologue_regs<MT, kB3, true, false, kConsumerBar, kChainConsumers>(a, nit, red_s, sx_s, xs, tsum);
            else if (nit <= kIt)
                fused_prologue_regs<MT, kIt, true, false, kConsumerBar, kChainConsumers>(a, nit, red_s, sx_s, xs, tsum);
            else
                fused_prologue_twopass<MT, true, kConsumerBar, kChainConsumers>(a, red_s, sx_s, xs, tsum);
        }
#pragma unroll
        for (int m = 0; m < MT; ++m) {
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) tsum[m] += __shfl_xor_sync(0xffffffffu, tsum[m], off);
            if (lane == 0) xsum_s[warp * MT + m] = tsum[m];
        }
        block_sync<kConsumerBar, kChainConsumers>();

        // acc[m][j]: low-nibble sums of row 4h + (j ^ pp) of the current tile,
        // token m; accA the high-nibble sums, folded in at the tile end
        // (up to four tokens; more keep one sum per row and token)
        constexpr bool kSplitAcc = MT <= 4;
        int acc[MT][4], accA[kSplitAcc ? MT : 1][4];
#pragma unroll
        for (int m = 0; m < MT; ++m)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                acc[m][j] = 0;
                if constexpr (kSplitAcc) accA[m][j] = 0;
            }

        for (int round = 0; round < nrounds; ++round, ++round_count) {
            const int buf = round_count & 1;
            int lo, hi;
            warp_lines(warp, min(RT, ntiles - round * RT), C, lo, hi, kChainWarps);
            int* meta = meta_s + (buf * kChainWarps + warp) * 2;
            if (lane == 0) {
                meta[0] = -1;
                meta[1] = -1;
            }
            __syncwarp();
            int p = lo;
            int tl = lo / C;
            int c = lo - tl * C;
            while (p < hi) {
                const int n = min(min(hi - p, C - c), kSliceLines);
                const int slot = cslot;
                if (!dead && !__all_sync(0xffffffffu, mbar_test_wait(my_full + 8 * slot, cphase))) {
                    const bool ok = mbar_wait_bounded(my_full + 8 * slot, cphase, kChainWaitNs);
                    if (!__all_sync(0xffffffffu, ok)) {
                        dead = true;   // warp-uniform from here on
                        if (lane == 0) {
                            stop_s = 1;
                            if (P.err != nullptr) atomicExch(P.err, kErrWaitTimeout);
                        }
                    }
                }
                if (!dead) {
                    const uint8_t* sw = my_ring + static_cast<size_t>(slot) * kSlotBytes;
#pragma unroll kPassUnroll
                    for (int pass = 0; pass < kSliceLines / kPassLines; ++pass) {
                        const int line = pass * kPassLines + pl;
                        if (line < n) {
                            const int chunk = c + line;
                            const uint8_t* ub = sw + (line * kRows + 4 * h) * kUnitBytes;
                            uint4 wv[4];
#pragma unroll
                            for (int j = 0; j < 4; ++j) wv[j] = *reinterpret_cast<const uint4*>(ub + ((j ^ pp) << 4));
#pragma unroll
                            for (int m = 0; m < MT; ++m) {
                                if (MT == 1 || m < M) {
                                    const uint4* xp = reinterpret_cast<const uint4*>(xs + static_cast<size_t>(m) * K + chunk * 32);
                                    const uint4 x0 = xp[0], x1 = xp[1];
#pragma unroll
                                    for (int j = 0; j < 4; ++j) {
                                        if constexpr (kSplitAcc) {
                                            unit4_acc(wv[j], x0, x1, acc[m][j], accA[m][j]);
                                        } else {
                                            int B, A;
                                            unit4(wv[j], x0, x1, B, A);
                                            acc[m][j] += B + (A >> 4);
                                        }
                                    }
                                }
                            }
                        }
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(my_empty + 8 * slot);      // the slot may be refilled
                }
                if (++cslot == S) {
                    cslot = 0;
                    cphase ^= 1u;
                }
                p += n;
                c += n;
                if (c == C || p == hi) {
                    // tile done for this warp: reduce lanes of equal (h, pp), then undo
                    // the read permutation with a two-step butterfly
#pragma unroll
                    for (int m = 0; m < MT; ++m) {
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            if constexpr (kSplitAcc) {
                                acc[m][j] += accA[m][j] >> 4;
                                accA[m][j] = 0;
                            }
                            acc[m][j] += __shfl_xor_sync(0xffffffffu, acc[m][j], 8);
                            acc[m][j] += __shfl_xor_sync(0xffffffffu, acc[m][j], 16);
                        }
#pragma unroll
                        for (int j = 0; j < 2; ++j) acc[m][j] += __shfl_xor_sync(0xffffffffu, acc[m][j + 2], 4);
                        acc[m][0] += __shfl_xor_sync(0xffffffffu, acc[m][1], 2);
                    }
                    const int tstart = tl * C;
                    if (lane < kRows) {
                        const bool full = lo <= tstart && hi >= tstart + C;
                        int* dst;
                        if (full) {
                            dst = acc_s + (static_cast<size_t>(buf) * RT * kRows + tl * kRows + my_row) * MT;
                        } else {
                            const int which = (lo >= tstart && lo < tstart + C) ? 0 : 1;
                            dst = bnd_s + (((buf * kChainWarps + warp) * 2 + which) * kRows + my_row) * MT;
                            if (lane == 0) meta[which] = tl;
                        }
#pragma unroll
                        for (int m = 0; m < MT; ++m) dst[m] = acc[m][0];
                    }
#pragma unroll
                    for (int m = 0; m < MT; ++m)
#pragma unroll
                        for (int j = 0; j < 4; ++j) acc[m][j] = 0;
                    if (c == C) {
                        c = 0;
                        ++tl;
                    }
                }
            }
            block_sync<kConsumerBar, kChainConsumers>();

            // ---- epilogue for this round's rows (coalesced over rows)
            const int rt0 = round * RT;
            const int nrows = min(RT, ntiles - rt0) * kRows;
            const int row_base = (t0 + rt0) * kRows;
            for (int idx = tid; idx < M * nrows; idx += kChainConsumers) {
                const int m = idx / nrows;
                const int rl = idx - m * nrows;
                const int row = row_base + rl;
                if (row >= a.N) continue;
                const int tile = rl >> 3;
                const int rr = rl & 7;
                int v = 0;
                bool part = false;
                for (int w = 0; w < kChainWarps; ++w) {
                    const int* mw = meta_s + (buf * kChainWarps + w) * 2;
#pragma unroll
                    for (int which = 0; which < 2; ++which) {
                        if (mw[which] == tile) {
                            v += bnd_s[(((buf * kChainWarps + w) * 2 + which) * kRows + rr) * MT + m];
                            part = true;
                        }
                    }
                }
                if (!part) v = acc_s[(static_cast<size_t>(buf) * RT * kRows + rl) * MT + m];
                int xsum = 0;
#pragma unroll
                for (int w = 0; w < kChainWarps; ++w) xsum += xsum_s[w * MT + m];
                const int accv = v - 8 * xsum;           // remove the +8 nibble bias
                const int ci = row - row0;
                const float b = rows_cached ? bias_s[ci] : (a.bias != nullptr ? a.bias[row] : 0.0f);
                const float swr = rows_cached ? sw_s[ci] : a.s_w[row];
                a.y[static_cast<size_t>(m) * a.N + row] = __fmaf_rn(__fmul_rn(swr, sx_s[m]), __int2float_rn(accv), b);
            }
            // accumulator and merge buffers alternate between rounds: no barrier here
        }
    }

    // the final arrival; the block that completes the count resets it for the next launch
    block_sync<kConsumerBar, kChainConsumers>();
    if (threadIdx.x == 0) {
        const unsigned prev = atom_add_release_gpu(P.barrier, 1u);
        if (prev + 1u == static_cast<unsigned>(NL) * gridDim.x) atomicExch(P.barrier, 0u);
    }
}

}  // namespace

cudaError_t launch_chain_w4(const ChainParams<kMaxChain>& p, int MT, int grid, size_t smem, cudaStream_t s)
{
    const void* kern = nullptr;
    switch (MT) {
        case 1: kern = reinterpret_cast<const void*>(stream_chain_kernel<1>); break;
        case 2: kern = reinterpret_cast<const void*>(stream_chain_kernel<2>); break;
        case 4: kern = reinterpret_cast<const void*>(stream_chain_kernel<4>); break;
        case 8: kern = reinterpret_cast<const void*>(stream_chain_kernel<8>); break;
        case 16: kern = reinterpret_cast<const void*>(stream_chain_kernel<16>); break;
        default: return cudaErrorInvalidValue;
    }
    static SmemLimit limits[5];
    const int li = MT == 1 ? 0 : MT == 2 ? 1 : MT == 4 ? 2 : MT == 8 ? 3 : 4;
    cudaError_t e = raise_smem_limit(kern, limits[li], smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(kChainThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    void* args[] = {const_cast<ChainParams<kMaxChain>*>(&p)};
    return cudaLaunchKernelExC(&cfg, kern, args);
}

}  // namespace w4k
