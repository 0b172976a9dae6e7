// Multi-token per-row INT4 decode GEMV on the 5th-generation tensor cores.
//
// What it computes ("Jetson Orin AGX INT4 推理优化实践", §"从 FP 线性层到 INT4 DP4A
// 的数学推导"; the multi-token verify case of "在香橙派上跑 Gemma4", §五):
//   acc[m][j] = sum_i q_w[j][i] qx[m][i]  (exact),
//   y[m][j]   = fmaf(s_w[j] * sx[m], (float)acc[m][j], b[j])
// for M = 3..16 tokens sharing one pass over the weights.  The int8 codes and
// scales come from the activation quantizer launched before this kernel.
//
// How (GB300 design): the product is a GEMM of N x K by K x 16, so it runs on
// tcgen05.mma (kind::f8f6f4, e4m3 operands, M = 128 rows, K = 32 per
// instruction).  e4m3 bytes 0x00..0x0F are exactly n 2^-9 (subnormals below
// 8, the first binade above), so a weight enters as its biased nibble
// n = q + 8 masked into a byte: two masks give eight weights, in order.  An
// int8 code x = 16 h + l is split into h = x >> 4 in [-8, 7] (e4m3
// sign-magnitude) and l = x & 15, both exact, laid side by side in N = 32
// (columns 0-15 the tokens' h, 16-31 their l): one MMA covers 32 K for all
// sixteen tokens.  Products n h 2^-18 and n l 2^-18 are exact and every
// partial sum is a multiple of 2^-18 below 64 in magnitude (|n l| <= 225 and a
// split covers at most 16384 K), so the fp32 accumulators hold the sums
// exactly; the epilogue forms sum n x = 16 S_h + S_l and removes the bias,
// sum q x = sum n x - 8 sum x, with each token's code sum over the split.
//   * One block of ten warps per (128-row group, K split), two blocks per
//     SM.  K splits of a row group form one thread-block cluster: the other
//     splits add their exact integer sums into the leader's shared memory
//     (remote atomics), arrive once on its mbarrier with cluster-scope release
//     and exit; only the leader waits, then writes y.
//   * Packed weights stream through a ring of stages (512 K x 128 rows,
//     32 KB: one 2 KB bulk copy per 8-row tile) issued before the dependency
//     wait; the operand pipeline steps through the stage in two 256-K blocks.
//   * Warps 0-7 form two groups that take alternate K blocks.  Thread t of a
//     group masks row t % 128's nibbles into e4m3 bytes (two LOP3 and a shift
//     per 8 weights, the block's whole 256 K) and stores them into tensor
//     memory as the MMA's A operand (three buffers of 64 columns).  The same
//     threads copy the block's codes (a small cp.async ring), split each code
//     once and write both halves into the activation tile (B, shared memory,
//     K-major, no swizzle): thread t takes token t % 16 in two 16-K groups,
//     so eight consecutive threads store 128 contiguous bytes.
//   * Lane 0 of warp 8 issues a block's eight MMAs into one accumulator (a
//     second one, alternating, made the K loop no faster and doubled the
//     tensor-memory reads at the end) and commits them; warp 9 issues the
//     weight copies.  "Operands written" is a named barrier per buffer (one
//     warp group and warp 8), "operands read" the MMA commit's mbarrier, and
//     the ring has full / empty mbarriers: no block-wide barrier sits in the
//     K loop.  Warp 8 also allocates and frees the tensor memory, so warps
//     0-3 go from the accumulator read straight to the epilogue.
//   * In the K loop the dequantizing warps' per-block chain (shared-memory
//     loads, tensor-memory stores and their wait, the named barrier to the
//     MMA lane, the commit's mbarrier) is the critical path, not the tensor
//     cores' arithmetic: hence K blocks of 256 (half the hand-offs of 128),
//     three operand buffers, two warp groups that overlap their chains, and no
//     division in the loop.  Around the loop, what a launch costs is latency:
//     the set-up (cluster barrier, tensor-memory allocation, row parameters)
//     runs before the dependency wait, and the tail is one tensor-memory read,
//     the split reduction and the epilogue.
#include <cuda_fp16.h>

#include "fusion.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace w4k {
namespace {

constexpr uint64_t kTcWaitNs = 250ull * 1000ull * 1000ull;
constexpr int kTcN = 2 * kTcTok;      // MMA N: each token's high and low code halves
constexpr uint32_t kTcCols = 256;     // tensor-memory columns: A x 3 (64 each), D x 2 (32 each)
constexpr uint32_t kTcColA = 0;
constexpr uint32_t kTcAStride = kTcKb / 4;   // one K block of e4m3 A: 4 bytes per column
constexpr uint32_t kTcColD = kTcColA + kTcBufs * kTcAStride;
constexpr int kTcAccs = 1;            // accumulators (K slice kk into D[kk % kTcAccs])
// Instruction descriptor, kind::f8f6f4: D fp32 (bits 4-5 = 1), A and B e4m3
// (bits 7-12 = 0), both K-major (bits 15, 16 = 0), N >> 3 at bits 17-22,
// M >> 4 at bits 24-28.
constexpr uint32_t kTcIdesc = (1u << 4) | (static_cast<uint32_t>(kTcN >> 3) << 17) |
                              (static_cast<uint32_t>(kTcRows >> 4) << 24);
// B tile: core matrices of 8 columns x 16 K (16 B rows), column groups 128 B
// apart, K groups 512 B apart (four column groups); one MMA's 32 K is 1024 B.
constexpr uint32_t kTcBsbo = 128;
constexpr uint32_t kTcBlbo = 512;

// 32 biased nibbles (n = q + 8) of one row -> 32 e4m3 bytes n 2^-9 in K
// order: byte b of word w holds weight 8w+b (low nibble) and 8w+4+b (high).
__device__ __forceinline__ void tc_unit_e4m3(const uint4 u, uint32_t* h)
{
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        h[2 * i] = w[i] & 0x0F0F0F0Fu;
        h[2 * i + 1] = (w[i] >> 4) & 0x0F0F0F0Fu;
    }
}

// Four int8 codes x -> the e4m3 bytes of h = x >> 4 (sign-magnitude, |h| <= 8)
// and of l = x & 15, each exactly its value times 2^-9.
__device__ __forceinline__ void tc_split4(uint32_t c, uint32_t& hi, uint32_t& lo)
{
    lo = c & 0x0F0F0F0Fu;
    const uint32_t u = (c >> 4) & 0x0F0F0F0Fu;              // h + 16 for negative h
    const uint32_t bm = prmt_sign_bytes(c);                  // 0xFF in the bytes of negative x (so of h)
    const uint32_t m = (u ^ (bm & 0x0F0F0F0Fu)) + (bm & 0x01010101u);   // |h| = 16 - u there
    hi = m | (bm & 0x80808080u);
}

__global__ void __launch_bounds__(kTcThreads, 2) tc_linear_kernel(const __grid_constant__ TcArgs A)
{
    extern __shared__ __align__(128) uint8_t smem[];
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const bool mma_warp = warp == kTcDqWarps;
    const bool producer = warp == kTcDqWarps + 1;
    const int S = A.stages;
    const int ks = A.splits;
    const TcSmem L = tc_smem(S, ks);
    uint8_t* ring = smem + L.ring;
    uint8_t* bbuf = smem + L.bbuf;
    uint8_t* codes = smem + L.codes;
    const uint32_t bars = smem_u32(smem + L.bars);
    const uint32_t full_b = bars;                        // [S]  stage landed (1 arrival + bytes)
    const uint32_t empty_b = bars + 8 * S;               // [S]  stage read by the dequantizing warps
    const uint32_t free_b = bars + 16 * S;               // [kTcBufs]  MMAs reading an operand buffer completed
    const uint32_t red_b = bars + 8 * (2 * S + 2 * kTcBufs);   // the leader's: every other split's sums added
    // operand buffer j written by one group of four dequantizing warps: named
    // barrier 1 + j (that group and the MMA warp)
    constexpr uint32_t kReadyCount = (kTcDqWarps / 2 + 1) * 32;
    auto ready_arrive = [](int j) {
        if (j == 0) named_arrive(1, kReadyCount);
        else if (j == 1) named_arrive(2, kReadyCount);
        else named_arrive(3, kReadyCount);
    };
    auto ready_sync = [](int j) {
        if (j == 0) named_sync(1, kReadyCount);
        else if (j == 1) named_sync(2, kReadyCount);
        else named_sync(3, kReadyCount);
    };
    static_assert(kTcBufs == 3, "one named barrier per operand buffer");
    static_assert(kTcColD + kTcAccs * kTcN <= kTcCols, "tensor-memory columns");
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L.tmem);   // [0] base address, [1] stop flag
    int* xsum_s = reinterpret_cast<int*>(smem + L.xsum);                 // [kTcTok] code sums of the split
    float* sx_s = reinterpret_cast<float*>(smem + L.sx);                 // [kTcTok] token scales
    volatile uint32_t* dead_s = tmem_slot + 1;

    constexpr int kSubs = kTcStageChunks / kTcChunks;      // K blocks per ring stage
    static_assert((kSubs & (kSubs - 1)) == 0, "K blocks per stage: a power of two");
    const int g = blockIdx.x / ks;                         // row group
    const int split = blockIdx.x - g * ks;                 // = rank in the cluster
    const int cb = static_cast<int>(static_cast<long long>(split) * A.C / ks);
    const int ce = static_cast<int>(static_cast<long long>(split + 1) * A.C / ks);
    const int nb = (ce - cb + kTcChunks - 1) / kTcChunks;  // K blocks of this split
    const int nst = (ce - cb + kTcStageChunks - 1) / kTcStageChunks;   // ring stages
    const int tile0 = g * (kTcRows / kRows);
    const int ntl = min(kTcRows / kRows, A.T - tile0);     // 8-row tiles present

    if (tid == 0) {
        for (int n = 0; n < kTcTok; ++n) xsum_s[n] = 0;
        for (int s = 0; s < S; ++s) {
            mbar_init(full_b + 8 * s, 1);
            mbar_init(empty_b + 8 * s, kTcDqWarps);
        }
        for (int j = 0; j < kTcBufs; ++j) {
            mbar_init(free_b + 8 * j, 1);         // the MMA lane's commit
        }
        if (ks > 1 && split == 0) mbar_init(red_b, static_cast<uint32_t>((ks - 1) * kTcRows));
        fence_mbar_init();
        *dead_s = 0u;
    }
    // the leader's K-split sums start at zero: the other splits add into them
    int* red = reinterpret_cast<int*>(smem + L.red);
    if (ks > 1 && split == 0)
        for (int i = tid; i < kTcRows * kTcTok; i += kTcThreads) red[i] = 0;
    __syncthreads();
    pdl_launch_dependents();

    // stage st of the weights into ring slot st % S (copy warp: lane 0 sets
    // the byte count, lane l < 16 copies 8-row tile l: up to 16 chunks, 2 KB)
    const uint64_t pol = l2_policy_evict_first();
    auto issue = [&](int st) {
        const int slot = st % S;
        const int c0 = cb + st * kTcStageChunks;
        const int nch = min(kTcStageChunks, ce - c0);
        const uint32_t bar = full_b + 8 * slot;
        if (lane == 0) {
            if (st >= S) fence_proxy_async_smem();
            mbar_arrive_expect_tx(bar, static_cast<uint32_t>(ntl * nch * kRows * 16));
        }
        __syncwarp();
        if (lane < ntl)
            bulk_g2s(smem_u32(ring + static_cast<size_t>(slot) * kTcStageBytes + lane * kTcStageChunks * kRows * 16),
                     A.w + (static_cast<size_t>(tile0 + lane) * A.C + c0) * kRows * 16,
                     static_cast<uint32_t>(nch * kRows * 16), bar, pol);
    };
    int issued = 0;      // stages whose weights were requested (producer warp)
    if (producer)
        for (; issued < S && issued < nst; ++issued) issue(issued);
    // the leader's zeroed sums and its barrier are visible to the whole cluster
    // (all of this runs before the dependency wait, beside the previous kernel)
    if (ks > 1) cluster_sync();
    // the MMA warp holds the tensor memory (it frees it while warps 0-3 write y)
    if (mma_warp) {
        tmem_alloc(smem_u32(tmem_slot), kTcCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tmem_slot;
    auto fail = [&]() {
        *dead_s = 1u;
        if (A.err != nullptr) atomicExch(A.err, kErrWaitTimeout);
    };
    // this row's output parameters do not depend on the previous kernel
    const bool row_thread = tid < kTcRows;
    const int row = g * kTcRows + tid;
    const int prow = A.glu == GLU_NONE ? (row < A.N ? row : -1) : glu_param_row(row, A.n_out);
    float sw_r = 0.0f, bv_r = 0.0f;
    if (row_thread && split == 0 && prow >= 0) {
        sw_r = A.s_w[prow];
        bv_r = A.bias != nullptr ? A.bias[prow] : 0.0f;
    }

    // Warps 0-7, two groups of four on alternate K blocks (see below): A of a
    // K block, this thread's row (tensor-memory lane t % 128, which warp t / 32
    // reaches as warp (t / 32) % 4 does) over the block's 256 K as e4m3 (the
    // buffer's 64 columns) in two halves of four chunks, sixteen columns per
    // store; the group arrives on the stage's empty barrier once it is read.
    const bool dequant = warp < kTcDqWarps;
    const int row_a = tid & (kTcRows - 1);
    const int grp = warp >> 2;
    const uint32_t tlane = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint8_t* my_units =
        ring + (row_a >> 3) * (kTcStageChunks * kRows * 16) + (grp * kTcChunks) * kRows * 16 + (row_a & 7) * 16;
    auto convert_a = [&](int slot, int j, int nch) {
        const uint8_t* units = my_units + static_cast<size_t>(slot) * kTcStageBytes;
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
            constexpr int kQ = kTcChunks / 2;
            uint4 u[kQ];
#pragma unroll
            for (int e = 0; e < kQ; ++e)
                if (kQ * hf + e < nch) u[e] = *reinterpret_cast<const uint4*>(units + (kQ * hf + e) * kRows * 16);
            if (hf == 1) {
                __syncwarp();
                if (lane == 0) mbar_arrive(empty_b + 8 * slot);   // this group's block of the stage is read
            }
#pragma unroll
            for (int r = 0; r < kQ / 2; ++r) {
                uint32_t h[16];
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    if (kQ * hf + 2 * r + e < nch) {
                        tc_unit_e4m3(u[2 * r + e], &h[e * 8]);
                    } else {
#pragma unroll
                        for (int k = 0; k < 8; ++k) h[e * 8 + k] = 0u;
                    }
                }
                tmem_st16(tbase + tlane + kTcColA + j * kTcAStride + 32 * hf + 16 * r, h);
            }
        }
    };
    // The weights do not depend on the previous kernel: each group converts its
    // first K block (stage 0, operand buffer grp) before the dependency wait.
    // Its loop then skips that block's stage wait and A: once both groups have
    // read stage 0 the copy warp may refill the slot, whose barrier would then
    // be a phase further on.
    bool first_a_done = false;
    if (dequant && grp < nb) {
        bool ok = mbar_wait_bounded(full_b, 0u, kTcWaitNs);
        if (!__all_sync(0xffffffffu, ok)) {
            if (lane == 0 && !*dead_s) fail();
        } else {
            tc_fence_after();
            convert_a(0, grp, min(kTcChunks, ce - (cb + grp * kTcChunks)));
            first_a_done = true;
        }
    }

    // ---- inputs produced by earlier kernels (codes, scales) from here on
    pdl_wait();
    // token scales for the epilogue, fetched while the K loop runs (the MMA
    // warp waits for them before the block barrier that ends the loop)
    if (mma_warp) {
        if (lane < kTcTok) cp_async4(sx_s + lane, lane < A.M ? A.sx + lane : A.sx, lane < A.M ? 4u : 0u);
        cp_async_commit();
    }

    int committed = 0;   // K blocks whose MMAs were committed (MMA warp)
    if (mma_warp) {
        // --------------------------------------------------------- MMA warp
        // Every K block is synchronised (named barrier) and committed even after a
        // failure, so that warps 0-7, which arrive once per block and wait for each
        // buffer's commit in order, never block on a missing step.
        const uint32_t dcol = tbase + kTcColD;
        for (int b = 0; b < nb; ++b) {
            const int j = b % kTcBufs;
            const int nch = min(kTcChunks, ce - (cb + b * kTcChunks));
            ready_sync(j);                           // A[j] and B[j] written by warps 0-7
            if (lane == 0) {
                if (!*dead_s) {
                    // K slice kk (32 K: 8 tensor-memory columns of A, 1024 B of B, which is
                    // 64 in the descriptor's address field and cannot carry) accumulates
                    // into D[kk % kTcAccs]; the first block's first slice per accumulator
                    // overwrites.
                    tc_fence_after();
                    const uint64_t bdesc = smem_desc_noswizzle(smem_u32(bbuf + j * kTcBBytes), kTcBlbo, kTcBsbo);
                    const uint32_t acol = tbase + kTcColA + j * kTcAStride;
                    static_assert((kTcAccs == 1 || kTcAccs == 2) && kTcChunks == 8, "eight MMAs per block");
                    constexpr uint32_t d1 = (1 % kTcAccs) * kTcN;
                    if (nch == kTcChunks && b > 0) {
                        tc_mma_f8_ts_x4(dcol, dcol + d1, dcol, dcol + d1, acol, bdesc, kTcIdesc, 1u);
                        tc_mma_f8_ts_x4(dcol, dcol + d1, dcol, dcol + d1, acol + 32, bdesc + 256, kTcIdesc, 1u);
                    } else {
#pragma unroll
                        for (int kk = 0; kk < kTcChunks; ++kk)
                            if (kk < nch)
                                tc_mma_f8_ts(dcol + (kk % kTcAccs) * kTcN, acol + kk * 8,
                                             bdesc + static_cast<uint64_t>(kk * 64), kTcIdesc,
                                             b > 0 || kk >= kTcAccs ? 1u : 0u);
                    }
                }
                tc_commit(free_b + 8 * j);
            }
            committed = b + 1;
        }
        if (lane == 0) {
            // every committed MMA completes before tensor memory is read or freed
            if (committed > 0) {
                const int last = committed - 1;
                if (!mbar_wait_bounded(free_b + 8 * (last % kTcBufs), static_cast<uint32_t>(last / kTcBufs) & 1u,
                                       kTcWaitNs) && !*dead_s)
                    fail();
            }
            if (committed < nb && !*dead_s) fail();
        }
        // lane 0's wait above is a divergent loop: reconverge the warp before the
        // block barrier (bar.sync is the aligned form, which assumes a converged
        // warp), so the barrier follows the last MMA's completion
        __syncwarp();
        cp_async_wait_group<0>();   // the token scales
    } else if (producer) {
        // ---------------------------------------------------- producer warp
        // refill each stage's slot once warps 0-7 have read it
        for (; issued < nst; ++issued) {
            const int prev = issued - S;
            bool ok = true;
            if (lane == 0)
                ok = !*dead_s && mbar_wait_bounded(empty_b + 8 * (prev % S), static_cast<uint32_t>(prev / S) & 1u, kTcWaitNs);
            if (!__shfl_sync(0xffffffffu, static_cast<int>(ok), 0)) {
                if (lane == 0 && !*dead_s) fail();
                break;
            }
            issue(issued);
        }
        // after a failure: copies still in flight land before the ring is reused or the block exits
        if (lane == 0 && *dead_s)
            for (int k = issued - S > 0 ? issued - S : 0; k < issued; ++k)
                if (!mbar_wait_bounded(full_b + 8 * (k % S), static_cast<uint32_t>(k / S) & 1u, kTcWaitNs)) break;
        __syncwarp();
    } else {
        // ------------------------------------------- warps 0-7: A and B
        // Two warp groups take alternate K blocks: group g = warp / 4 the blocks
        // b = g, g + 2, ..., i.e. sub-block g of every weight stage.  Thread t
        // works on row t % 128 (tensor-memory lane t % 128, which warp t / 32
        // reaches as warp (t / 32) % 4 does) over the whole 256 K of its blocks,
        // and splits the codes of token t % 16 in K groups (t % 128) / 16 and
        // that + 8 (16 K each) into both halves of the activation tile B.  A
        // group's per-block chain (waits, stores, fences, the hand-off) thus has
        // two block periods to run while the other group fills the next buffer.
        static_assert(kSubs == 2 && kTcDqWarps == 8, "two groups of four warps, one K block of a stage each");
        const int cn = row_a & (kTcTok - 1);
        const int kg = row_a >> 4;
        static_assert(kTcThreadCodes == 32 && kTcRows * kTcThreadCodes == kTcTok * kTcKb,
                      "each dequantizing thread copies two 16-K groups of one token per block");
        int xsum = 0;       // this thread's code sum (token cn, its K groups) over the split's K range
        auto fetch_codes = [&](int b, int cs) {
            uint8_t* dst = codes + cs * (kTcDqWarps * 32 * kTcThreadCodes) + tid * kTcThreadCodes;
            const int kbase = (cb + b * kTcChunks) * 32;
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int kofs = kbase + (kg + 8 * e) * 16;
                const bool ok = b < nb && cn < A.M && kofs < ce * 32;
                cp_async16(dst + 16 * e, ok ? A.qx + static_cast<size_t>(cn) * A.K + kofs : A.qx, ok ? 16u : 0u);
            }
            cp_async_commit();
        };
#pragma unroll
        for (int i = 0; i < kTcCodeRing - 1; ++i) fetch_codes(grp + 2 * i, i);
        // ring positions kept as counters (no division in the loop): weight
        // stage slot and its phase, operand buffer j = b % 3 and q = b / 3 (the
        // previous commit on buffer j is that of block b - 3, phase (q - 1) & 1),
        // code-ring slots of this block and of the one fetched
        int slot = 0, j = grp, q = 0, cs = 0, cs_next = kTcCodeRing - 1;
        uint32_t sph = 0u;
        for (int b = grp; b < nb; b += 2) {
            if (b > grp) {
                if (++slot == S) { slot = 0; sph ^= 1u; }
                j += 2;
                if (j >= kTcBufs) { j -= kTcBufs; ++q; }
                if (++cs == kTcCodeRing) cs = 0;
                if (++cs_next == kTcCodeRing) cs_next = 0;
            }
            const int nch = min(kTcChunks, ce - (cb + b * kTcChunks));
            fetch_codes(b + 2 * (kTcCodeRing - 1), cs_next);
            // buffer j is free once the commit of block b - kTcBufs arrived (the MMA
            // lane commits every block, failed or not, so this wait keeps its order)
            const bool a_done = first_a_done && b == grp;
            bool ok = b < kTcBufs || mbar_wait_bounded(free_b + 8 * j, static_cast<uint32_t>(q - 1) & 1u, kTcWaitNs);
            if (ok && !*dead_s && !a_done) ok = mbar_wait_bounded(full_b + 8 * slot, sph, kTcWaitNs);
            if (!__all_sync(0xffffffffu, ok) && lane == 0 && !*dead_s) fail();
            if (*dead_s) {
                // stop working but keep the per-block handshake
                cp_async_wait_group<kTcCodeRing - 1>();
                ready_arrive(j);
                continue;
            }
            tc_fence_after();
            if (!a_done) convert_a(slot, j, nch);
            // B: token cn, K groups kg and kg + 8 of the block: the high halves in
            // column cn, the low halves in column 16 + cn
            cp_async_wait_group<kTcCodeRing - 1>();
            const uint8_t* mc = codes + cs * (kTcDqWarps * 32 * kTcThreadCodes) + tid * kTcThreadCodes;
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const uint4 c = *reinterpret_cast<const uint4*>(mc + 16 * e);
                uint4 hv, lv;
                tc_split4(c.x, hv.x, lv.x);
                tc_split4(c.y, hv.y, lv.y);
                tc_split4(c.z, hv.z, lv.z);
                tc_split4(c.w, hv.w, lv.w);
                uint8_t* bt = bbuf + j * kTcBBytes + (kg + 8 * e) * kTcBlbo + (cn & 7) * 16 + (cn >> 3) * kTcBsbo;
                *reinterpret_cast<uint4*>(bt) = hv;
                *reinterpret_cast<uint4*>(bt + 2 * kTcBsbo) = lv;
                xsum = __dp4a(static_cast<int>(c.x), 0x01010101, xsum);
                xsum = __dp4a(static_cast<int>(c.y), 0x01010101, xsum);
                xsum = __dp4a(static_cast<int>(c.z), 0x01010101, xsum);
                xsum = __dp4a(static_cast<int>(c.w), 0x01010101, xsum);
            }
            fence_proxy_async_smem();
            tmem_wait_st();
            tc_fence_before();
            ready_arrive(j);
        }
        cp_async_wait_group<0>();
        // token cn's code sum: lanes cn and cn + 16 of each of the eight warps
        xsum += __shfl_xor_sync(0xffffffffu, xsum, 16);
        if (lane < kTcTok) atomicAdd(xsum_s + cn, xsum);
        __syncwarp();
    }
    __syncthreads();

    // ---- the accumulator: row tid, tokens 0..15 (warps 0-3)
    const bool dead = *dead_s != 0u;
    int acc[kTcTok];
#pragma unroll
    for (int n = 0; n < kTcTok; ++n) acc[n] = 0;
    if (row_thread && !dead && nb > 0) {
        // the MMA warp saw the last commit complete before the barrier above;
        // each accumulator holds sum n h 2^-18 (columns 0-15) and sum n l 2^-18
        // (16-31) exactly: times 2^18 they are exact integers, and over the
        // accumulators 16 S_h + S_l, less 8 sum x, is the exact sum q x
        tc_fence_after();
        const int used = min(kTcAccs, min(kTcChunks, ce - cb));   // accumulators written at all
        for (int q = 0; q < used; ++q) {
            uint32_t dh[kTcTok], dl[kTcTok];
            const uint32_t da = tbase + (static_cast<uint32_t>(warp * 32) << 16) + kTcColD + q * kTcN;
            tmem_ld16x2(da, dh, da + kTcTok, dl);
#pragma unroll
            for (int n = 0; n < kTcTok; ++n)
                acc[n] += 16 * __float2int_rn(__fmul_rn(__uint_as_float(dh[n]), 262144.0f)) +
                          __float2int_rn(__fmul_rn(__uint_as_float(dl[n]), 262144.0f));
        }
#pragma unroll
        for (int n = 0; n < kTcTok; ++n) acc[n] -= 8 * xsum_s[n];
    }
    tc_fence_before();
    __syncthreads();
    if (mma_warp) {
        tc_fence_after();
        tmem_dealloc(tbase, kTcCols);
    }

    // ---- K splits: every other split adds its exact integer sums into the
    // leader's (red[n][row], integer adds in any order give the same sums),
    // arrives once per row thread on the leader's barrier and exits; only the
    // leader waits, for the last of them.
    if (ks > 1) {
        if (split != 0) {
            if (row_thread) {
                const uint32_t dst = mapa_shared(smem_u32(red + tid), 0);
#pragma unroll
                for (int n = 0; n < kTcTok; ++n)
                    red_add_cluster_u32(dst + 4 * n * kTcRows, static_cast<uint32_t>(acc[n]));
                mbar_arrive_remote_release(mapa_shared(red_b, 0));
            }
            return;
        }
        if (!row_thread) return;
        if (!mbar_wait_cluster_bounded(red_b, 0u, kTcWaitNs) && !dead) fail();
#pragma unroll
        for (int n = 0; n < kTcTok; ++n) acc[n] += red[n * kTcRows + tid];
    }
    if (!row_thread) return;

    // ---- epilogue: y = fmaf(s_w s_x, acc, b), coalesced over rows per token
    // (a partial sum of a dead split makes the row wrong: the error word says so).
    // Every load (token scales, residuals) is issued before the first store: y
    // may alias the residual, so a store between two loads would serialise them.
    const bool dead_out = *dead_s != 0u;
    if (A.glu == GLU_NONE) {
        if (row < A.N && !dead_out) {
            const float sw = sw_r;
            const float bv = bv_r;
            float v[kTcTok];
#pragma unroll
            for (int n = 0; n < kTcTok; ++n)
                v[n] = n < A.M ? __fmaf_rn(__fmul_rn(sw, sx_s[n]), __int2float_rn(acc[n]), bv) : 0.0f;
            if (A.residual != nullptr) {
                float rv[kTcTok];
#pragma unroll
                for (int n = 0; n < kTcTok; ++n)
                    rv[n] = n < A.M ? A.residual[static_cast<size_t>(n) * A.N + row] : 0.0f;
#pragma unroll
                for (int n = 0; n < kTcTok; ++n) v[n] = __fadd_rn(rv[n], v[n]);
            }
#pragma unroll
            for (int n = 0; n < kTcTok; ++n)
                if (n < A.M) A.y[static_cast<size_t>(n) * A.N + row] = v[n];
        }
    } else {
        // gated: this thread's row pairs with the row 4 lanes away (gate rows
        // r % 8 < 4, up rows 4 below them, in the same tile).  The gate lane
        // writes output j for the even tokens, the up lane for the odd ones.
        const bool have = row < A.N && prow >= 0 && !dead_out;
        const bool up = (row & 4) != 0;
        const float sw = have ? sw_r : 0.0f;
        const float bv = have ? bv_r : 0.0f;
        const int j = (row >> 3) * 4 + (row & 3);
        float v[kTcTok];
#pragma unroll
        for (int n = 0; n < kTcTok; ++n)
            v[n] = n < A.M ? __fmaf_rn(__fmul_rn(sw, sx_s[n]), __int2float_rn(acc[n]), bv) : 0.0f;
        constexpr int kHalfTok = kTcTok / 2;
        float gv[kHalfTok], uv[kHalfTok], rv[kHalfTok];
#pragma unroll
        for (int k = 0; k < kHalfTok; ++k) {
            // token 2k + up is this lane's: the partner sends its value there
            const float other = __shfl_xor_sync(0xffffffffu, up ? v[2 * k] : v[2 * k + 1], 4);
            gv[k] = up ? other : v[2 * k];
            uv[k] = up ? v[2 * k + 1] : other;
            const int n = 2 * k + (up ? 1 : 0);
            rv[k] = (have && A.residual != nullptr && n < A.M) ? A.residual[static_cast<size_t>(n) * A.n_out + j] : 0.0f;
        }
        if (have) {
#pragma unroll
            for (int k = 0; k < kHalfTok; ++k) {
                const int n = 2 * k + (up ? 1 : 0);
                if (n < A.M) {
                    float out = glu_act_call(A.glu, gv[k], uv[k]);
                    if (A.residual != nullptr) out = __fadd_rn(rv[k], out);
                    A.y[static_cast<size_t>(n) * A.n_out + j] = out;
                }
            }
        }
    }
}

}  // namespace

cudaError_t launch_gemv_w4_tc(const TcArgs& a, int grid, size_t smem, bool pdl, cudaStream_t s)
{
    auto kern = tc_linear_kernel;
    static SmemLimit limit;
    cudaError_t e = raise_smem_limit(reinterpret_cast<const void*>(kern), limit, smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(kTcThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    int na = 0;
    if (pdl) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    if (a.splits > 1) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = static_cast<unsigned>(a.splits);
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    cfg.attrs = na > 0 ? attr : nullptr;
    cfg.numAttrs = na;
    return cudaLaunchKernelEx(&cfg, kern, a);
}

}  // namespace w4k
