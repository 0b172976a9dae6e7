// Declarations shared by the host API and the kernel translation units.
#pragma once
#include <atomic>
#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

namespace w4k {

// Weight formats.  W4F and W8F are the weight-only paths on float
// activations that "Jetson Orin AGX INT4 推理优化实践" §"为什么 INT4 float
// 解包不快" measures against INT4 DP4A: per-row INT4 in the W4 layout
// unpacked to float, and per-row INT8 (32-byte units, no scale plane).
enum FmtId { FMT_W4 = 0, FMT_Q4_0 = 1, FMT_I8G32 = 2, FMT_Q6G32 = 3, FMT_W4F = 4, FMT_W8F = 5 };

constexpr int kRows = 8;                 // weight rows per tile
constexpr int kWarps = 8;                // warps per GEMV thread block
constexpr int kThreads = kWarps * 32;
constexpr int kMaxStages = 8;            // ring slots per warp, upper bound
constexpr int kAccWords = 64;            // round_tiles * MT, bounds the per-round accumulator
constexpr int kRowCache = 1024;          // rows per block whose s_w / bias are staged in shared memory
constexpr int kMaxSplitTokens = 2;       // DP4A GEMVs split K for at most this many tokens

// Activation source of a GEMV: quantized in the prologue (from x, or from
// RMSNorm(x) when GemvArgs::gamma is set), int8 codes copied into shared
// memory, codes read from global memory in the inner loop, or (the
// weight-only formats) fp32 x copied into shared memory unquantized.
enum XMode { X_FUSED = 0, X_SMEM = 1, X_GLOBAL = 2, X_F32 = 3 };

// Gated MLP activation applied by the epilogue (fusion.cuh).
enum GluKind { GLU_NONE = 0, GLU_SILU = 1, GLU_GELU_TANH = 2 };

// Row pairing of a gated linear: tile t holds gate rows 4t..4t+3 as its rows
// 0-3 and the matching up rows as rows 4-7.  Kernel row R -> row of the
// caller's [gate; up] parameter arrays (n_out = I gate rows), or -1 past I.
__host__ __device__ inline int glu_param_row(int R, int n_out)
{
    const int j = (R >> 3) * 4 + (R & 3);
    if (j >= n_out) return -1;
    return (R & 4) ? n_out + j : j;
}

// Lines (8 rows x one 32-weight chunk) per ring slot and bytes per unit.
// Q6G32 keeps each unit in two planes: 16 bytes of low nibbles and 8 bytes
// of 2-bit high parts (fmt_hi_bytes).
__host__ __device__ constexpr int fmt_unit_bytes(int fmt) { return fmt == FMT_I8G32 || fmt == FMT_W8F ? 32 : 16; }
__host__ __device__ constexpr int fmt_hi_bytes(int fmt) { return fmt == FMT_Q6G32 ? 8 : 0; }
__host__ __device__ constexpr bool fmt_group(int fmt) { return fmt == FMT_Q4_0 || fmt == FMT_I8G32 || fmt == FMT_Q6G32; }
// Formats with one float scale per row (s_w).
__host__ __device__ constexpr bool fmt_row_scale(int fmt) { return fmt == FMT_W4 || fmt == FMT_W4F || fmt == FMT_W8F; }
// Formats on unquantized float activations.
__host__ __device__ constexpr bool fmt_float_x(int fmt) { return fmt == FMT_W4F || fmt == FMT_W8F; }
__host__ __device__ constexpr int fmt_slice_lines(int fmt)
{
    return fmt == FMT_I8G32 || fmt == FMT_Q6G32 || fmt == FMT_W8F ? 16 : 32;
}
__host__ __device__ constexpr int fmt_slot_w_bytes(int fmt) { return fmt_slice_lines(fmt) * kRows * fmt_unit_bytes(fmt); }
__host__ __device__ constexpr int fmt_slot_h_bytes(int fmt) { return fmt_slice_lines(fmt) * kRows * fmt_hi_bytes(fmt); }
__host__ __device__ constexpr int fmt_slot_s_bytes(int fmt) { return fmt_group(fmt) ? fmt_slice_lines(fmt) * kRows * 2 : 0; }
__host__ __device__ constexpr int fmt_slot_bytes(int fmt)
{
    return fmt_slot_w_bytes(fmt) + fmt_slot_h_bytes(fmt) + fmt_slot_s_bytes(fmt);
}

// One linear of a launch.
struct GemvArgs {
    const uint8_t* w;        // repacked units
    const uint16_t* wscale;  // fp16 group-scale plane (Q4_0, I8G32, Q6G32), else null
    const uint8_t* whi;      // high-part plane (Q6G32), else null
    const float* s_w;        // per-row scales (W4), else null
    const float* bias;       // [N] or null
    const float* x;          // fp32 activations [M][K] (fused quantize), else null
    const int8_t* qx_in;     // int8 activations [M][K] (unfused), else null
    const float* sx_in;      // [M] (unfused), else null
    int8_t* qx_out;          // fused: block 0 writes the codes here (may be null)
    float* sx_out;           // fused: block 0 writes the scales here (may be null)
    float* y;                // [M][n_out]
    const float* gamma;      // RMSNorm weight [K] (fused prologue, one to four tokens), else null
    float eps;               // RMSNorm epsilon
    const float* residual;   // [M][n_out] added to the output (may alias y), else null
    int glu;                 // GluKind: rows paired per tile (glu_param_row), n_out = I
    int n_out;               // outputs per token: N, or I for a gated linear
    int M, N, K;             // N: weight rows (a gated linear: 8 ceil(I / 4))
    int C;                   // K / 32
    int T;                   // ceil(N / 8)
    int tq, tr;              // T = tq * grid + tr: block b owns tq (+1 if b < tr) tiles, from b tq + min(b, tr)
    int rot;                 // block b takes the range of block (b + rot) % grid (balances chains over linears)
    int ks;                  // K splits: clusters of ks blocks share a tile range, block rank r
                             // takes chunks [r C / ks, (r + 1) C / ks) (0 or 1: no split)
};

// Kernel parameters: up to NCH linears computed in order by one launch.
constexpr int kMaxChain = 128;
template <int NCH>
struct ChainParams {
    GemvArgs lin[NCH];
    int n;                   // linears in this launch (1..NCH)
    int kmax;                // largest K: sizes the shared-memory activation buffer
    int stages;              // ring slots per warp
    int round_tiles;         // tiles per accumulation round
    unsigned* barrier;       // grid barrier state [2] (chains only)
    unsigned* err;           // device error word
    int prefetch_slices;     // chains: slices per ring prefetched into L2 ahead of the copies
};

struct SmemLayout {
    int bars, sx, red, xsum, rowp, meta, acc, bnd, merge, ring, xs, total;
};

__host__ __device__ inline int align_up(int v, int a) { return (v + a - 1) / a * a; }

__host__ __device__ inline SmemLayout smem_layout(int fmt, int MT, int xmode, int K, int stages, int round_tiles,
                                                  int row_bufs = 1, int row_cap = kRowCache, int ks = 1)
{
    SmemLayout L;
    int o = 0;
    L.bars = o;  o = align_up(o + kWarps * stages * 8, 16);
    L.sx = o;    o = align_up(o + MT * 4, 16);
    L.red = o;   o = align_up(o + kWarps * MT * 4, 16);
    L.xsum = o;  o = align_up(o + kWarps * MT * 4, 16);
    L.rowp = o;  o = align_up(o + row_bufs * 2 * row_cap * 4, 16);
    L.meta = o;  o = align_up(o + 2 * kWarps * 2 * 4, 16);
    L.acc = o;   o = align_up(o + 2 * round_tiles * kRows * MT * 4, 16);
    L.bnd = o;   o = align_up(o + 2 * kWarps * 2 * kRows * MT * 4, 16);
    // K splits: the round's per-row sums of this block, then (in the leader)
    // one buffer per other rank that rank writes through the cluster
    L.merge = o; o = align_up(o + (ks > 1 ? ks * round_tiles * kRows * MT * 4 : 0), 128);
    L.ring = o;  o = align_up(o + kWarps * stages * fmt_slot_bytes(fmt), 128);
    L.xs = o;    o += xmode == X_F32 ? MT * K * 4 : (xmode != X_GLOBAL ? MT * K : 0);
    L.total = o;
    return L;
}

// Persistent chain (gemv_chain.cu): fifteen consumer warps plus one warp
// that streams the weights of every linear in order into the consumers'
// rings.  Shared memory: full and empty barriers per slot, then the
// consumer areas (two per-row parameter buffers), the rings and the codes.
constexpr int kChainWarps = 15;                          // consumer warps (with the producer: 16, 128 registers each)
constexpr int kChainConsumers = kChainWarps * 32;
constexpr int kChainThreads = (kChainWarps + 1) * 32;

struct ChainLayout {
    int full, empty, sx, red, xsum, rowp, meta, acc, bnd, ring, xs, total;
};

__host__ __device__ inline ChainLayout chain_layout(int MT, int K, int stages, int round_tiles)
{
    ChainLayout L;
    int o = 0;
    L.full = o;  o += kChainWarps * stages * 8;
    L.empty = o; o = align_up(o + kChainWarps * stages * 8, 16);
    L.sx = o;    o = align_up(o + MT * 4, 16);
    L.red = o;   o = align_up(o + kChainWarps * MT * 4, 16);
    L.xsum = o;  o = align_up(o + kChainWarps * MT * 4, 16);
    L.rowp = o;  o = align_up(o + 2 * 2 * (kRowCache / 2) * 4, 16);
    L.meta = o;  o = align_up(o + 2 * kChainWarps * 2 * 4, 16);
    L.acc = o;   o = align_up(o + 2 * round_tiles * kRows * MT * 4, 16);
    L.bnd = o;   o = align_up(o + 2 * kChainWarps * 2 * kRows * MT * 4, 128);
    L.ring = o;  o = align_up(o + kChainWarps * stages * fmt_slot_bytes(FMT_W4), 128);
    L.xs = o;    o += MT * K;
    L.total = o;
    return L;
}

// Error codes written to the device error word.
constexpr unsigned kErrWaitTimeout = 0x57414954u;     // "WAIT": an mbarrier wait ran out
constexpr unsigned kErrBarrierTimeout = 0x42415252u;  // "BARR": a grid barrier wait ran out

// Dynamic shared-memory limit set so far for one kernel, per device.
// raise_smem_limit (w4a8_api.cu) raises it under a lock, so host threads
// launching the same kernel concurrently never lower another's setting.
constexpr int kMaxDevices = 64;
struct SmemLimit {
    std::atomic<int> bytes[kMaxDevices];
};
cudaError_t raise_smem_limit(const void* kern, SmemLimit& rec, size_t smem);

// Kernel launchers, one translation unit per format.
cudaError_t launch_gemv_w4(const ChainParams<1>& p, int MT, int xmode, int grid, size_t smem, bool pdl,
                           cudaStream_t s);
cudaError_t launch_gemv_q4_0(const ChainParams<1>& p, int MT, int xmode, int grid, size_t smem, bool pdl,
                             cudaStream_t s);
cudaError_t launch_gemv_i8g32(const ChainParams<1>& p, int MT, int xmode, int grid, size_t smem, bool pdl,
                              cudaStream_t s);
cudaError_t launch_gemv_q6g32(const ChainParams<1>& p, int MT, int xmode, int grid, size_t smem, bool pdl,
                              cudaStream_t s);
// Largest x float4 per thread and token the RMSNorm prologue holds in
// registers (x and the norm weight together).
__host__ __device__ constexpr int norm_max_nit(int MT) { return MT >= 4 ? 4 : 20 / (MT + 1); }
// Weight-only GEMVs on float activations (W4F, W8F; xmode X_F32; MT in {1, 2, 4}).
cudaError_t launch_gemv_a32(int fmt, const ChainParams<1>& p, int MT, int grid, size_t smem, bool pdl,
                            cudaStream_t s);
// Chains of per-row INT4 linears (cooperative launch, fused quantization,
// a producer warp streaming the weights; gemv_chain.cu).
cudaError_t launch_chain_w4(const ChainParams<kMaxChain>& p, int MT, int grid, size_t smem, cudaStream_t s);

// ---------------------------------------------- multi-token tensor-core GEMV
// Per-row INT4 GEMV for 3..16 tokens on the tcgen05 tensor cores
// (gemv_tc.cu): one block of kTcThreads per (128-row group, K split), the
// K splits of a row group forming one thread-block cluster.
constexpr int kTcDqWarps = 8;                    // warps 0-7: A and B, two groups of four on alternate K blocks
constexpr int kTcThreads = (kTcDqWarps + 2) * 32;  // then the MMA warp and the copy warp
constexpr int kTcRows = 128;                     // MMA M: weight rows per block
constexpr int kTcTok = 16;                       // MMA N: tokens (fewer are zero-padded)
constexpr int kTcChunks = 8;                     // 32-weight chunks per K block
constexpr int kTcKb = 32 * kTcChunks;            // K per block: 256
constexpr int kTcStageChunks = 16;              // chunks per weight-ring stage (2 K blocks): 2 KB copies per tile
constexpr int kTcStageBytes = (kTcRows / kRows) * kTcStageChunks * kRows * 16;   // 32 KB of packed weights
constexpr int kTcBBytes = 2 * kTcTok * kTcKb;    // e4m3 activation tile per K block (high and low halves)
constexpr int kTcThreadCodes = kTcKb / 8;        // codes a dequantizing thread copies per K block (its group's)
constexpr int kTcCodeRing = 2;                   // K blocks of int8 codes in flight per warp group
constexpr int kTcBufs = 3;                       // A (tensor memory) / B (shared memory) operand buffers
constexpr int kTcMaxSplit = 8;                   // K splits (cluster size) at most
constexpr int kTcMaxSplitK = 16384;              // K per split at most: |sum n l| <= 225 K stays below 2^24

struct TcArgs {
    const uint8_t* w;       // repacked per-row INT4 (8-row tiles)
    const float* s_w;       // [N] (a gated linear: [2 n_out], gate rows then up rows)
    const float* bias;      // same rows as s_w, or null
    const int8_t* qx;       // [M][K] activation codes
    const float* sx;        // [M]
    float* y;               // [M][n_out]
    const float* residual;  // [M][n_out] added to the output (may alias y), or null
    int glu;                // GluKind
    int n_out;              // outputs per token
    int M, N, K, C, T;      // C = K / 32 chunks, T = row tiles
    int splits;             // K splits per row group (= cluster size)
    int stages;             // weight ring depth (K blocks)
    unsigned* err;
};

struct TcSmem {
    int ring, bbuf, codes, red, bars, tmem, xsum, sx, total;
};

__host__ __device__ inline TcSmem tc_smem(int stages, int splits)
{
    TcSmem L;
    int o = 0;
    L.ring = o;  o += stages * kTcStageBytes;
    L.bbuf = o;  o += kTcBufs * kTcBBytes;
    L.codes = o; o += kTcCodeRing * (kTcDqWarps * 32) * kTcThreadCodes;
    L.red = o;   o += splits > 1 ? kTcRows * kTcTok * 4 : 0;   // the leader's K-split sums
    L.bars = o;  o += (2 * stages + 2 * kTcBufs + 1) * 8;
    L.tmem = o;  o += 16;
    L.xsum = o;  o += kTcTok * 4;
    L.sx = o;    o += kTcTok * 4;
    L.total = o;
    return L;
}

cudaError_t launch_gemv_w4_tc(const TcArgs& a, int grid, size_t smem, bool pdl, cudaStream_t s);

// Pure-read bandwidth probe (hbm_read.cu): one block per SM streams `bytes`
// bytes once and XORs every 32-bit word into *sink (cleared first).
// A bounded wait that nothing completes (hbm_read.cu): it must end and set
// the device error word.
cudaError_t launch_wait_selftest(int cluster, unsigned long long timeout_ns, unsigned* err, cudaStream_t s);
cudaError_t launch_hbm_read(const void* buf, unsigned long long bytes, unsigned* sink, unsigned* err, int sms,
                            cudaStream_t s);

// Load-time and activation kernels (prep_kernels.cu).
constexpr int kMaxShards = 8;
struct ShardTable {
    const void* p[kMaxShards];
    const void* p2[kMaxShards];
    int row0[kMaxShards + 1];
    int n;
    int glu_rows;           // > 0: two shards (gate, up) of this many rows, paired per tile
};

cudaError_t launch_a8_quantize(const float* x, int M, int K, int8_t* qx, float* sx, bool pdl, cudaStream_t s);
// RMSNorm then the activation quantizer (one block per token).
cudaError_t launch_rms_a8_quantize(const float* x, const float* gamma, float eps, int M, int K, int8_t* qx,
                                   float* sx, bool pdl, cudaStream_t s);
// The operators on their own (fp32 out): RMSNorm, gated activation of a
// [M][2I] gate|up output, elementwise add.
cudaError_t launch_rmsnorm(const float* x, const float* gamma, float eps, int M, int K, float* out, bool pdl,
                           cudaStream_t s);
cudaError_t launch_glu(const float* gu, int kind, int M, int I, float* out, bool pdl, cudaStream_t s);
cudaError_t launch_add(const float* a, const float* b, long long n, float* out, bool pdl, cudaStream_t s);
cudaError_t launch_w4_quantize_rows(const float* W, int N, int K, uint32_t* packed, float* s_w, cudaStream_t s);
cudaError_t launch_w8_quantize_rows(const float* W, int N, int K, int8_t* q, float* s_w, cudaStream_t s);
cudaError_t launch_w8_repack(const ShardTable& st, int N, int K, void* out, cudaStream_t s);
cudaError_t launch_q4_0_quantize(const float* W, int N, int K, uint8_t* blocks, cudaStream_t s);
cudaError_t launch_i8g32_quantize(const float* W, int N, int K, int8_t* q, uint16_t* d, cudaStream_t s);
cudaError_t launch_w4_repack(const ShardTable& st, int N, int K, void* out, cudaStream_t s);
cudaError_t launch_q4_0_repack(const ShardTable& st, int N, int K, void* out, cudaStream_t s);
cudaError_t launch_i8g32_repack(const ShardTable& st, int N, int K, void* out, cudaStream_t s);
cudaError_t launch_q6g32_repack(const ShardTable& st, int N, int K, void* out, cudaStream_t s);

}  // namespace w4k
