// C ABI of the decode GEMV library (declared in include/w4a8.h): argument
// checks, launch configuration and dispatch.  No entry point allocates
// memory or synchronises, except the two device-error-word calls.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/w4a8.h"
#include "internal.h"

using namespace w4k;

// Device error word written by kernels whose bounded waits run out.
__device__ unsigned g_w4_error_word;

namespace {

struct DeviceInfo {
    int sms = 0;
    int smem_optin = 0;       // largest dynamic shared memory one block may use
    int smem_per_sm = 0;
    int smem_reserved = 0;    // per-block shared memory the runtime reserves
    unsigned* err = nullptr;
    bool ready = false;
};
DeviceInfo g_dev[kMaxDevices];
// Guards the one-time set-up of g_dev (and of the no-alloc scratch address):
// host threads may call the library concurrently, each on its own stream.
std::mutex g_setup_mutex;
std::atomic<bool> g_dev_ready[kMaxDevices];

// Launch tuning set by w4_set_tuning (0 = automatic).
int g_tune[7] = {0, 0, 0, 0, 0, 0, 0};
// Weight bytes a chain block prefetches into L2 ahead of its ring copies (KB):
// none by default (measured slower: the prefetches slowed the stream they lead).
constexpr int kChainPrefetchKB = 0;

w4_status device_info(DeviceInfo** out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return W4_ERR_CUDA;
    DeviceInfo& d = g_dev[dev];
    if (!g_dev_ready[dev].load(std::memory_order_acquire)) {
        std::lock_guard<std::mutex> lock(g_setup_mutex);
        if (g_dev_ready[dev].load(std::memory_order_relaxed)) {
            *out = &d;
            return W4_OK;
        }
        if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return W4_ERR_CUDA;
        if (cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
            return W4_ERR_CUDA;
        if (cudaDeviceGetAttribute(&d.smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess)
            return W4_ERR_CUDA;
        if (cudaDeviceGetAttribute(&d.smem_reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev) != cudaSuccess)
            return W4_ERR_CUDA;
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_w4_error_word) != cudaSuccess) return W4_ERR_CUDA;
        d.err = static_cast<unsigned*>(p);
        d.ready = true;
        g_dev_ready[dev].store(true, std::memory_order_release);
    }
    *out = &d;
    return W4_OK;
}

}  // namespace

namespace w4k {
cudaError_t raise_smem_limit(const void* kern, SmemLimit& rec, size_t smem)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    const int want = static_cast<int>(smem);
    if (rec.bytes[dev].load(std::memory_order_acquire) >= want) return cudaSuccess;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (rec.bytes[dev].load(std::memory_order_relaxed) >= want) return cudaSuccess;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, want);
    if (e == cudaSuccess) rec.bytes[dev].store(want, std::memory_order_release);
    return e;
}
}  // namespace w4k

namespace {

inline bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

inline w4_status cuda_status(cudaError_t e) { return e == cudaSuccess ? W4_OK : W4_ERR_CUDA; }

inline int round_pow2_tokens(int M) { return M <= 1 ? 1 : M <= 2 ? 2 : M <= 4 ? 4 : M <= 8 ? 8 : 16; }

// A DP4A GEMV of a group format (Q4_0, I8G32, Q6G32) with more than eight
// tokens runs as two launches of the eight-token kernel over the same
// weights, tokens 0-7 and the rest.  Every step of the GEMV is per token (the
// quantize prologue, the epilogue, the residual), so the split changes no
// token's codes or integer group sums.  The sixteen-token inner loop holds
// twice the accumulators and spills.  Measured on GB300 (single GEMVs, weights
// rotated past L2, us, two launches / one launch):
//   I8G32 lm_head 262144x1536   M = 9: 234 / 380    12: 288 / 417    16: 324 / 467
//   Q6G32 lm_head 262144x1536   M = 9: 304 / 557    12: 403 / 666    16: 495 / 847
//   Q4_0 gate/up 12288x1536     M = 9: 19.1 / 23.4  12: 21.4 / 26.2  16: 24.8 / 30.3
//   Q4_0 QKV 2560x1536          M = 9: 10.7 / 13.0  12: 12.0 / 14.2  16: 13.6 / 15.5
//   Q4_0 down 1536x6144         M = 9: 22.4 / 22.3  12: 25.0 / 24.7  16: 28.4 / 28.3
// (the M = 9 lm_head rows and the Q6G32 M = 12 row ran the second launch on its
// own token count's kernel; the second launch now takes the first's kernel
// and shared-memory plan, which took the short GEMVs' split from 13.0 to
// 10.7 us (QKV, 9 tokens) and from 16.6 to 12.0 us (12 tokens): launches of
// one configuration follow each other on an SM without draining it.)
constexpr int kGroupLaunchTokens = 8;

// Tokens in the first (and every full) launch of an M-token call; M for one
// launch.  W4_TUNE_GROUP_LAUNCH_TOKENS = t > 0 sets the limit to t tokens.
inline int launch_tokens(int fmt, int M)
{
    if (fmt == FMT_W4 || fmt_float_x(fmt)) return M;
    const int t = g_tune[W4_TUNE_GROUP_LAUNCH_TOKENS] > 0 ? g_tune[W4_TUNE_GROUP_LAUNCH_TOKENS] : kGroupLaunchTokens;
    return M > t ? t : M;
}

w4_status check_mk(int M, int K)
{
    if (M < 0 || K <= 0) return W4_ERR_INVALID_ARG;
    if (M > W4_MAX_M || K % 32 != 0 || K > W4_MAX_K) return W4_ERR_UNSUPPORTED_SHAPE;
    return W4_OK;
}

w4_status build_shards(const void* const* p, const void* const* p2, const int* rows, int n, ShardTable& st, int& N)
{
    if (n < 1 || n > kMaxShards || p == nullptr || rows == nullptr) return W4_ERR_INVALID_ARG;
    std::memset(&st, 0, sizeof(st));
    long long total = 0;
    st.n = n;
    for (int s = 0; s < n; ++s) {
        if (rows[s] < 0) return W4_ERR_INVALID_ARG;
        if (rows[s] > 0 && p[s] == nullptr) return W4_ERR_INVALID_ARG;
        if (p2 != nullptr && rows[s] > 0 && p2[s] == nullptr) return W4_ERR_INVALID_ARG;
        st.p[s] = p[s];
        st.p2[s] = p2 ? p2[s] : nullptr;
        st.row0[s] = static_cast<int>(total);
        total += rows[s];
        if (total > (1LL << 30)) return W4_ERR_UNSUPPORTED_SHAPE;
    }
    st.row0[n] = static_cast<int>(total);
    N = static_cast<int>(total);
    return W4_OK;
}

size_t tiles(int N) { return (static_cast<size_t>(N) + kRows - 1) / kRows; }

// Launch configuration of one GEMV: activation mode, ring depth, shared memory.
struct Plan {
    int xmode = X_GLOBAL;
    int stages = 0;
    int smem = 0;
};

// Largest ring (at most the cap) whose layout fits `budget`; 0 if fewer than 2 stages fit.
int stages_for(int fmt, int MT, int xmode, int K, int RT, int budget, int ks = 1)
{
    const int cap = g_tune[W4_TUNE_MAX_STAGES] > 0 ? g_tune[W4_TUNE_MAX_STAGES] : kMaxStages;
    int s = cap < kMaxStages ? cap : kMaxStages;
    while (s >= 2 && smem_layout(fmt, MT, xmode, K, s, RT, 1, kRowCache, ks).total > budget) --s;
    return s >= 2 ? s : 0;
}

// Whether a DP4A GEMV of MT tokens over T row tiles runs two of its own
// blocks per SM.  Two tokens: always (see plan_gemv).  One token: for a GEMV
// of at least 64 tiles per SM: measured alone, the lm_head 152064 x 3584 takes
// 42.4 us on 304 blocks against 45.2 us on 152; shorter ones leave the second
// slot to the next linear, which fetches its weights there (the 7B step took
// 0.925 ms with every linear on 304 blocks against 0.876 ms, and 0.899
// against 0.870 ms with the gate/up projection alone on 304: alone it gains
// 1 us, the down projection after it loses its prefetch).
bool two_blocks_per_sm(const DeviceInfo& d, int MT, int T, int ks)
{
    return ks == 1 && (MT == 2 || (MT == 1 && T >= 64 * d.sms));
}

// Shared-memory budget of a DP4A GEMV block.  One token: half an SM when a
// ring of at least two stages fits there (two blocks per SM: this GEMV beside
// the next one in the stream, or, for a long GEMV, two of its own; see
// gemv_grid), else the whole-block budget.  Two tokens (`two_per_sm`): half
// an SM too where the ring fits, the two blocks of the SM this GEMV's own,
// else the whole block (the 7B step: 1.250 ms so, with the K = 18944 down
// projection's fused prologue on the whole block; 1.370 ms with every linear
// on the whole block, 1.653 with half an SM and the second slot left to the
// next linear; the 152064 x 3584 lm_head alone 44.3 against 63.3 us).  More tokens: the whole-block budget (a deeper ring pays
// once the inner loop does M times the DP4A work per weight byte).  `fused`
// asks for the quantize prologue.
bool plan_gemv(const DeviceInfo& d, int fmt, int MT, bool fused, int K, int RT, Plan& p, int ks = 1,
               bool two_per_sm = false)
{
    const int half = d.smem_per_sm / 2 - d.smem_reserved;
    const int whole = d.smem_optin;
    int bps = g_tune[W4_TUNE_BLOCKS_PER_SM];
    if (bps == 0 && MT > 1 && !(two_per_sm && MT <= 2 && ks == 1)) bps = 1;
    int modes[2] = {fused ? X_FUSED : X_SMEM, fused ? -1 : X_GLOBAL};
    if (fmt_float_x(fmt)) {
        modes[0] = X_F32;
        modes[1] = -1;
    }
    for (int pass = 0; pass < 2; ++pass) {
        // pass 0: co-resident budget (unless forced to one block per SM)
        if (pass == 0 && bps == 1) continue;
        if (pass == 1 && bps == 2) break;
        const int budget = pass == 0 ? half : whole;
        for (int mi = 0; mi < 2; ++mi) {
            const int xm = modes[mi];
            if (xm < 0) continue;
            const int s = stages_for(fmt, MT, xm, K, RT, budget, ks);
            if (s >= 2) {
                p.xmode = xm;
                p.stages = s;
                p.smem = smem_layout(fmt, MT, xm, K, s, RT, 1, kRowCache, ks).total;
                return true;
            }
        }
    }
    return false;
}

// Blocks of a DP4A GEMV launch over T row tiles: one per SM (or the tuned
// cap), never more than the tiles; with K splits, clusters of ks blocks each
// take a tile range (grid = clusters * ks).  With `two_per_sm` (see
// two_blocks_per_sm) and blocks that fit two per SM (smem: the planned
// bytes), two per SM.
int gemv_grid(const DeviceInfo& d, int T, int ks = 1, int smem = 0, bool two_per_sm = false)
{
    int grid = d.sms;
    const int half = d.smem_per_sm / 2 - d.smem_reserved;
    if (ks == 1 && two_per_sm && smem > 0 && smem <= half) grid = 2 * d.sms;
    if (g_tune[W4_TUNE_GRID_BLOCKS] > 0) grid = g_tune[W4_TUNE_GRID_BLOCKS];
    int clusters = grid / ks;
    if (clusters < 1) clusters = 1;
    return (T < clusters ? T : clusters) * ks;
}

// K splits of a DP4A GEMV with C chunks per row over T tiles: clusters of ks
// blocks share a tile range, block r taking chunks [r C / ks, (r + 1) C / ks),
// and add their per-row sums in the leader's shared memory (exact integers for
// per-row INT4; fp32 group sums in rank order otherwise).  Measured on GB300
// at one token, every split was slower than none, also where the tiles are
// too few for the SMs (the 512-row GEMV: 2.68 us unsplit, 3.77 / 4.05 us in
// two / four; the Gemma Q4_0 down projection: 4.06 against 5.17 / 5.44 us):
// these GEMVs are latency-bound, and the cluster launch and the merge's two
// cluster barriers per round cost more than the shorter loop saves.  So a
// split is never chosen on its own; W4_TUNE_K_SPLITS forces one where each
// rank keeps at least 16 chunks (one pass) per tile, for one or two tokens.
int choose_splits(const DeviceInfo& d, int fmt, int MT, int T, int C)
{
    (void)T;
    if (fmt_float_x(fmt) || MT > kMaxSplitTokens) return 1;
    int grid = d.sms;
    if (g_tune[W4_TUNE_GRID_BLOCKS] > 0) grid = g_tune[W4_TUNE_GRID_BLOCKS];
    const int forced = g_tune[W4_TUNE_K_SPLITS];
    if (forced > 1 && C / forced >= 16 && grid / forced >= 1) return forced;
    return 1;
}

// One planned DP4A GEMV launch.
struct GemvLaunch {
    ChainParams<1> cp;
    int MT, xmode, grid, smem;
};

// Plan one launch of a.M tokens on the kernel for MT tokens (a.M <= MT; the
// kernel skips the tokens past a.M at run time).
w4_status plan_launch(const DeviceInfo& dev, int fmt, GemvArgs a, bool fused, int MT, GemvLaunch& L)
{
    a.C = a.K / 32;
    a.T = static_cast<int>(tiles(a.N));
    a.ks = choose_splits(dev, fmt, MT, a.T, a.C);
    ChainParams<1>& cp = L.cp;
    std::memset(&cp, 0, sizeof(cp));
    cp.n = 1;
    cp.kmax = a.K;
    cp.round_tiles = kAccWords / MT;
    cp.err = dev.err;
    Plan p;
    if (a.ks > 1 && !plan_gemv(dev, fmt, MT, fused, a.K, cp.round_tiles, p, a.ks)) a.ks = 1;   // no room to merge
    const bool two = two_blocks_per_sm(dev, MT, a.T, a.ks);
    if (!plan_gemv(dev, fmt, MT, fused, a.K, cp.round_tiles, p, a.ks, two)) return W4_ERR_UNSUPPORTED_SHAPE;
    cp.stages = p.stages;
    const int grid = gemv_grid(dev, a.T, a.ks, p.smem, two);
    const int clusters = grid / a.ks;
    a.tq = a.T / clusters;
    a.tr = a.T % clusters;
    cp.lin[0] = a;
    L.MT = MT;
    L.xmode = p.xmode;
    L.grid = grid;
    L.smem = p.smem;
    return W4_OK;
}

// Launch one GEMV: one kernel, or, where launch_tokens splits the tokens, one
// kernel per group of them, each a programmatic dependent of the one before.
// Every launch of a call runs the first launch's kernel and shared-memory
// plan, so the next launch's blocks can take an SM as soon as this one's
// leave it.  Every launch is planned before
// the first is issued, so a failed check launches nothing.
w4_status run_gemv(int fmt, GemvArgs a, bool fused, unsigned flags, cudaStream_t s)
{
    DeviceInfo* dev = nullptr;
    w4_status st = device_info(&dev);
    if (st != W4_OK) return st;
    const int mc = launch_tokens(fmt, a.M);
    const int nl = (a.M + mc - 1) / mc;
    const int MT = round_pow2_tokens(mc);
    GemvLaunch L[W4_MAX_M];
    for (int c = 0; c < nl; ++c) {
        const size_t m0 = static_cast<size_t>(c) * mc;
        GemvArgs t = a;
        t.M = a.M - static_cast<int>(m0) < mc ? a.M - static_cast<int>(m0) : mc;
        const size_t xo = m0 * static_cast<size_t>(a.K), yo = m0 * static_cast<size_t>(a.n_out);
        if (t.x) t.x += xo;
        if (t.qx_in) t.qx_in += xo;
        if (t.sx_in) t.sx_in += m0;
        if (t.qx_out) t.qx_out += xo;
        if (t.sx_out) t.sx_out += m0;
        t.y += yo;
        if (t.residual) t.residual += yo;
        st = plan_launch(*dev, fmt, t, fused, MT, L[c]);
        if (st != W4_OK) return st;
    }
    for (int c = 0; c < nl; ++c) {
        const GemvLaunch& l = L[c];
        const bool pdl = c > 0 || (flags & W4_FLAG_PDL) != 0;
        cudaError_t e;
        if (fmt_float_x(fmt)) e = launch_gemv_a32(fmt, l.cp, l.MT, l.grid, l.smem, pdl, s);
        else if (fmt == FMT_W4) e = launch_gemv_w4(l.cp, l.MT, l.xmode, l.grid, l.smem, pdl, s);
        else if (fmt == FMT_Q4_0) e = launch_gemv_q4_0(l.cp, l.MT, l.xmode, l.grid, l.smem, pdl, s);
        else if (fmt == FMT_I8G32) e = launch_gemv_i8g32(l.cp, l.MT, l.xmode, l.grid, l.smem, pdl, s);
        else e = launch_gemv_q6g32(l.cp, l.MT, l.xmode, l.grid, l.smem, pdl, s);
        if (e != cudaSuccess) return W4_ERR_CUDA;
    }
    return W4_OK;
}

// Chain of per-row INT4 linears in one cooperative launch.
w4_status run_chain(const w4_linear_desc* d, int n, int M, unsigned* barrier, cudaStream_t s)
{
    DeviceInfo* dev = nullptr;
    w4_status st = device_info(&dev);
    if (st != W4_OK) return st;
    const int MT = round_pow2_tokens(M);
    // host staging only, copied into the launch; one per host thread, so
    // threads launching chains on their own streams do not share it
    thread_local ChainParams<kMaxChain> cp;
    std::memset(&cp, 0, sizeof(cp));
    int kmax = 32;
    for (int i = 0; i < n; ++i) {
        GemvArgs& a = cp.lin[i];
        a.w = static_cast<const uint8_t*>(d[i].w);
        a.s_w = d[i].s_w;
        a.bias = d[i].bias;
        a.x = d[i].x;
        a.qx_out = d[i].qx;
        a.sx_out = d[i].sx;
        a.y = d[i].y;
        a.M = M;
        a.N = d[i].N;
        a.n_out = d[i].N;
        a.K = d[i].K;
        a.C = a.K / 32;
        a.T = static_cast<int>(tiles(a.N));
        if (a.K > kmax) kmax = a.K;
    }
    cp.n = n;
    cp.kmax = kmax;
    cp.round_tiles = kAccWords / MT;
    cp.barrier = barrier;
    cp.err = dev->err;
    // one block per SM with the whole shared memory: the x buffer sized for
    // the largest K, then the deepest ring (at most the tuned cap) that fits
    const int cap_s = g_tune[W4_TUNE_MAX_STAGES] > 0 && g_tune[W4_TUNE_MAX_STAGES] < kMaxStages
                          ? g_tune[W4_TUNE_MAX_STAGES] : kMaxStages;
    int S = cap_s;
    while (S >= 2 && chain_layout(MT, kmax, S, cp.round_tiles).total > dev->smem_optin) --S;
    if (S < 2) return W4_ERR_UNSUPPORTED_SHAPE;
    cp.stages = S;
    const int smem = chain_layout(MT, kmax, S, cp.round_tiles).total;
    // L2 lookahead per block, spread over the eight rings in 4 KB slices
    const int la_kb = g_tune[W4_TUNE_CHAIN_PREFETCH_KB] > 0 ? g_tune[W4_TUNE_CHAIN_PREFETCH_KB] : kChainPrefetchKB;
    cp.prefetch_slices = la_kb / (kChainWarps * 4);
    int grid = dev->sms;
    if (g_tune[W4_TUNE_GRID_BLOCKS] > 0 && g_tune[W4_TUNE_GRID_BLOCKS] < grid) grid = g_tune[W4_TUNE_GRID_BLOCKS];
    // the blocks holding a linear's remainder tiles move on from linear to
    // linear, so no block carries an extra tile in every linear of the chain
    int rot = 0;
    for (int i = 0; i < n; ++i) {
        cp.lin[i].tq = cp.lin[i].T / grid;
        cp.lin[i].tr = cp.lin[i].T % grid;
        cp.lin[i].rot = rot;
        rot = (rot + cp.lin[i].tr) % grid;
    }
    return cuda_status(launch_chain_w4(cp, MT, grid, static_cast<size_t>(smem), s));
}

// Would the fused kernel (x quantized into shared memory) fit on device d?
bool fused_fits_on(const DeviceInfo& d, int fmt, int M, int K, bool norm)
{
    const int MT = round_pow2_tokens(launch_tokens(fmt, M));
    if (norm && (MT > 4 || (K / 4 + kThreads - 1) / kThreads > norm_max_nit(MT))) return false;
    Plan p;
    return plan_gemv(d, fmt, MT, true, K, kAccWords / MT, p);
}

bool fused_fits(int fmt, int M, int K, bool norm)
{
    DeviceInfo* dev = nullptr;
    if (device_info(&dev) != W4_OK) return false;
    return fused_fits_on(*dev, fmt, M, K, norm);
}

// Operators fused around one linear (w4_fusion, checked).
struct Fuse {
    const float* gamma = nullptr;
    float eps = 0.0f;
    int glu = GLU_NONE;
    const float* residual = nullptr;
};

w4_status check_fusion(int fmt, const w4_fusion* f, Fuse& z)
{
    z = Fuse();
    if (f == nullptr) return W4_OK;
    if (f->glu < W4_GLU_NONE || f->glu > W4_GLU_GELU_TANH) return W4_ERR_INVALID_ARG;
    if (f->glu != W4_GLU_NONE && fmt != FMT_W4 && fmt != FMT_Q4_0) return W4_ERR_UNSUPPORTED_SHAPE;
    if (f->norm_weight != nullptr) {
        if (!(f->norm_eps > 0.0f) || !(f->norm_eps < 3.0e38f)) return W4_ERR_INVALID_ARG;
        if (!aligned(f->norm_weight, 16)) return W4_ERR_MISALIGNED;
    }
    if (f->residual != nullptr && !aligned(f->residual, 4)) return W4_ERR_MISALIGNED;
    z.gamma = f->norm_weight;
    z.eps = f->norm_weight != nullptr ? f->norm_eps : 0.0f;
    z.glu = f->glu;
    z.residual = f->residual;
    return W4_OK;
}

// Weight rows behind n outputs: a gated linear pairs 4 gate and 4 up rows per tile.
inline int weight_rows(int n, int glu) { return glu != GLU_NONE ? 8 * ((n + 3) / 4) : n; }

// Per-row INT4 with this many tokens runs on the tensor cores (gemv_tc.cu),
// up to kTcMaxSplit K splits of kTcMaxSplitK.
bool use_tc(int fmt, int M, int K)
{
    const int lo = g_tune[W4_TUNE_TC_MIN_M] > 0 ? g_tune[W4_TUNE_TC_MIN_M] : 3;
    return fmt == FMT_W4 && M >= lo && M <= kTcTok && K <= kTcMaxSplit * kTcMaxSplitK;
}

// Tensor-core GEMV on device d: one block per (128-row group, K split);
// enough splits to cover the SMs, rounded down to a power of two (clusters of
// 5 or 6 blocks measured slower), at most kTcMaxSplit, and enough to keep
// every split within kTcMaxSplitK; the deepest weight ring that leaves room
// for a second block per SM.  N: weight rows.
w4_status tc_plan(const DeviceInfo& d, int N, int K, int& ks, int& S)
{
    const int C = K / 32;
    const int G = (N + kTcRows - 1) / kTcRows;
    auto fill = [&](int blocks) {
        int k = (blocks + G - 1) / G;
        if (k > kTcMaxSplit) k = kTcMaxSplit;
        while (k & (k - 1)) --k;                // clusters of 1, 2, 4 or 8 blocks
        return k;
    };
    // Both block slots of every SM when the splits stay long (at least four
    // K blocks each: the 7B down projection, 1-2% faster per step); otherwise
    // one: with shorter splits (QKV, O) the second slot is worth more to the
    // next linear, whose blocks become resident there and fetch their weights.
    ks = fill(d.sms);
    if (G * 2 <= d.sms && C / fill(2 * d.sms) >= 4 * kTcChunks) ks = fill(2 * d.sms);
    const int need = (K + kTcMaxSplitK - 1) / kTcMaxSplitK;
    if (ks < need) ks = need;
    if (ks > C) ks = C;
    if (ks < need || ks > kTcMaxSplit) return W4_ERR_UNSUPPORTED_SHAPE;
    const int half = d.smem_per_sm / 2 - d.smem_reserved;
    S = 4;
    while (S > 2 && tc_smem(S, ks).total > half) --S;
    if (tc_smem(S, ks).total > d.smem_optin) return W4_ERR_UNSUPPORTED_SHAPE;
    return W4_OK;
}

w4_status run_gemv_tc(const void* w, const float* s_w, const float* bias, const int8_t* qx, const float* sx, int M,
                      int N, int K, float* y, bool pdl, cudaStream_t s, int n_out, int glu, const float* residual)
{
    DeviceInfo* dev = nullptr;
    w4_status st = device_info(&dev);
    if (st != W4_OK) return st;
    TcArgs a = {};
    a.w = static_cast<const uint8_t*>(w);
    a.s_w = s_w;
    a.bias = bias;
    a.qx = qx;
    a.sx = sx;
    a.y = y;
    a.residual = residual;
    a.glu = glu;
    a.n_out = n_out;
    a.M = M;
    a.N = N;
    a.K = K;
    a.C = K / 32;
    a.T = static_cast<int>(tiles(N));
    a.err = dev->err;
    const int G = (N + kTcRows - 1) / kTcRows;
    int ks = 0, S = 0;
    st = tc_plan(*dev, N, K, ks, S);
    if (st != W4_OK) return st;
    a.splits = ks;
    a.stages = S;
    return cuda_status(launch_gemv_w4_tc(a, G * ks, static_cast<size_t>(tc_smem(S, ks).total), pdl, s));
}

// One GEMV on int8 codes; N outputs per token (a gated linear: 2N weight
// rows' worth of parameters, rows paired per tile), epilogue fusions in fz.
w4_status gemv_common(int fmt, const void* w, const float* s_w, const float* bias, const int8_t* qx,
                      const float* sx, int M, int N, int K, float* y, cudaStream_t s, bool pdl = false,
                      const Fuse& fz = Fuse())
{
    w4_status st = check_mk(M, K);
    if (st != W4_OK) return st;
    if (N < 0) return W4_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return W4_OK;
    if (!w || !qx || !sx || !y || (fmt == FMT_W4 && !s_w)) return W4_ERR_INVALID_ARG;
    if (!aligned(w, 16) || !aligned(qx, 16) || !aligned(sx, 4) || !aligned(y, 4) || (s_w && !aligned(s_w, 4)) ||
        (bias && !aligned(bias, 4)))
        return W4_ERR_MISALIGNED;
    if (N > (1 << 30) - 8) return W4_ERR_UNSUPPORTED_SHAPE;
    const int Nw = weight_rows(N, fz.glu);
    if (use_tc(fmt, M, K)) return run_gemv_tc(w, s_w, bias, qx, sx, M, Nw, K, y, pdl, s, N, fz.glu, fz.residual);
    GemvArgs a = {};
    a.w = static_cast<const uint8_t*>(w);
    const size_t units = tiles(Nw) * kRows * (K / 32);
    a.whi = fmt_hi_bytes(fmt) > 0 ? a.w + units * static_cast<size_t>(fmt_unit_bytes(fmt)) : nullptr;
    a.wscale = fmt == FMT_W4 ? nullptr
                             : reinterpret_cast<const uint16_t*>(
                                   a.w + units * static_cast<size_t>(fmt_unit_bytes(fmt) + fmt_hi_bytes(fmt)));
    a.s_w = s_w;
    a.bias = bias;
    a.qx_in = qx;
    a.sx_in = sx;
    a.y = y;
    a.glu = fz.glu;
    a.residual = fz.residual;
    a.n_out = N;
    a.M = M;
    a.N = Nw;
    a.K = K;
    return run_gemv(fmt, a, false, pdl ? W4_FLAG_PDL : 0u, s);
}

w4_status linear_common(int fmt, const void* w, const float* s_w, const float* bias, const float* x, int M, int N,
                        int K, float* y, int8_t* qx, float* sx, unsigned flags, cudaStream_t s,
                        const w4_fusion* f = nullptr)
{
    w4_status st = check_mk(M, K);
    if (st != W4_OK) return st;
    if (N < 0 || (flags & ~W4_FLAG_PDL) != 0) return W4_ERR_INVALID_ARG;
    Fuse fz;
    st = check_fusion(fmt, f, fz);
    if (st != W4_OK) return st;
    if (M == 0) return W4_OK;
    if (!x || !qx || !sx) return W4_ERR_INVALID_ARG;
    if (N > 0 && (!w || !y || (fmt == FMT_W4 && !s_w))) return W4_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(qx, 16) || !aligned(sx, 4) || (w && !aligned(w, 16)) || (y && !aligned(y, 4)) ||
        (s_w && !aligned(s_w, 4)) || (bias && !aligned(bias, 4)))
        return W4_ERR_MISALIGNED;
    if (N > (1 << 30) - 8) return W4_ERR_UNSUPPORTED_SHAPE;
    const bool norm = fz.gamma != nullptr;
    const bool pdl = (flags & W4_FLAG_PDL) != 0;
    if (N == 0 || use_tc(fmt, M, K) || !fused_fits(fmt, M, K, norm)) {
        // quantize (normalize first if asked) into the caller's qx/sx once, then
        // the GEMV on int8 codes (tensor cores for many tokens), chained by
        // programmatic dependent launch
        st = cuda_status(norm ? launch_rms_a8_quantize(x, fz.gamma, fz.eps, M, K, qx, sx, pdl, s)
                              : launch_a8_quantize(x, M, K, qx, sx, pdl, s));
        if (st != W4_OK || N == 0) return st;
        return gemv_common(fmt, w, s_w, bias, qx, sx, M, N, K, y, s, true, fz);
    }
    const int Nw = weight_rows(N, fz.glu);
    GemvArgs a = {};
    a.w = static_cast<const uint8_t*>(w);
    const size_t units = tiles(Nw) * kRows * (K / 32);
    a.whi = fmt_hi_bytes(fmt) > 0 ? a.w + units * static_cast<size_t>(fmt_unit_bytes(fmt)) : nullptr;
    a.wscale = fmt == FMT_W4 ? nullptr
                             : reinterpret_cast<const uint16_t*>(
                                   a.w + units * static_cast<size_t>(fmt_unit_bytes(fmt) + fmt_hi_bytes(fmt)));
    a.s_w = s_w;
    a.bias = bias;
    a.x = x;
    a.qx_out = qx;
    a.sx_out = sx;
    a.y = y;
    a.gamma = fz.gamma;
    a.eps = fz.eps;
    a.glu = fz.glu;
    a.residual = fz.residual;
    a.n_out = N;
    a.M = M;
    a.N = Nw;
    a.K = K;
    return run_gemv(fmt, a, true, flags, s);
}

}  // namespace

extern "C" {

const char* w4_status_str(w4_status st)
{
    switch (st) {
        case W4_OK: return "W4_OK";
        case W4_ERR_INVALID_ARG: return "W4_ERR_INVALID_ARG";
        case W4_ERR_UNSUPPORTED_SHAPE: return "W4_ERR_UNSUPPORTED_SHAPE";
        case W4_ERR_MISALIGNED: return "W4_ERR_MISALIGNED";
        case W4_ERR_CUDA: return "W4_ERR_CUDA";
        case W4_ERR_DEVICE_TIMEOUT: return "W4_ERR_DEVICE_TIMEOUT";
    }
    return "W4_ERR_UNKNOWN";
}

int w4_version(void) { return 1; }

static_assert(W4_FMT_W4 == FMT_W4 && W4_FMT_Q4_0 == FMT_Q4_0 && W4_FMT_I8G32 == FMT_I8G32 &&
                  W4_FMT_Q6G32 == FMT_Q6G32,
              "public format codes");

w4_status w4_plan(int fmt, int M, int N, int K, unsigned what, const w4_device_desc* dev, w4_launch_plan* out)
{
    if (!dev || !out || fmt < FMT_W4 || fmt > FMT_Q6G32 ||
        (what & ~(W4_PLAN_LINEAR | W4_PLAN_NORM | W4_PLAN_GLU)) != 0)
        return W4_ERR_INVALID_ARG;
    const bool linear = (what & W4_PLAN_LINEAR) != 0;
    const bool norm = (what & W4_PLAN_NORM) != 0;
    const bool glu = (what & W4_PLAN_GLU) != 0;
    if ((norm && !linear) || (glu && fmt != FMT_W4 && fmt != FMT_Q4_0)) return W4_ERR_INVALID_ARG;
    if (dev->sms <= 0 || dev->smem_per_sm <= 0 || dev->smem_reserved < 0 || dev->smem_optin <= 0)
        return W4_ERR_INVALID_ARG;
    w4_status st = check_mk(M, K);
    if (st != W4_OK) return st;
    if (N < 0) return W4_ERR_INVALID_ARG;
    DeviceInfo d;
    d.sms = dev->sms;
    d.smem_per_sm = dev->smem_per_sm;
    d.smem_reserved = dev->smem_reserved;
    d.smem_optin = dev->smem_optin;
    w4_launch_plan p = {};
    p.k_splits = 1;
    if (M > 0) {
        if (N > (1 << 30) - 8) return W4_ERR_UNSUPPORTED_SHAPE;
        const int Nw = weight_rows(N, glu ? GLU_SILU : GLU_NONE);
        const int T = static_cast<int>(tiles(Nw));
        const bool tc = use_tc(fmt, M, K);
        if (linear && (N == 0 || tc || !fused_fits_on(d, fmt, M, K, norm))) p.quantize_launches = 1;
        if (N > 0) {
            if (tc) {
                int ks = 0, S = 0;
                st = tc_plan(d, Nw, K, ks, S);
                if (st != W4_OK) return st;
                p.path = W4_PATH_TENSOR_CORES;
                p.grid = (Nw + kTcRows - 1) / kTcRows * ks;
                p.threads = kTcThreads;
                p.smem_bytes = tc_smem(S, ks).total;
                p.stages = S;
                p.k_splits = ks;
                p.gemv_launches = 1;
            } else {
                const int mc = launch_tokens(fmt, M);
                const int MT = round_pow2_tokens(mc);
                const int ks = choose_splits(d, fmt, MT, T, K / 32);
                Plan q;
                const bool two = two_blocks_per_sm(d, MT, T, ks);
                if (!plan_gemv(d, fmt, MT, linear && p.quantize_launches == 0, K, kAccWords / MT, q, ks, two))
                    return W4_ERR_UNSUPPORTED_SHAPE;
                p.path = q.xmode == X_FUSED ? W4_PATH_FUSED : q.xmode == X_SMEM ? W4_PATH_CODES_SMEM
                                                                                : W4_PATH_CODES_GLOBAL;
                p.grid = gemv_grid(d, T, ks, q.smem, two);
                p.k_splits = ks;
                p.threads = kThreads;
                p.smem_bytes = q.smem;
                p.stages = q.stages;
                p.gemv_launches = (M + mc - 1) / mc;
            }
        }
    }
    *out = p;
    return W4_OK;
}

w4_status w4_describe_device(w4_device_desc* out)
{
    if (!out) return W4_ERR_INVALID_ARG;
    DeviceInfo* dev = nullptr;
    const w4_status st = device_info(&dev);
    if (st != W4_OK) return st;
    out->sms = dev->sms;
    out->smem_per_sm = dev->smem_per_sm;
    out->smem_reserved = dev->smem_reserved;
    out->smem_optin = dev->smem_optin;
    return W4_OK;
}

w4_status w4_set_tuning(int key, int value)
{
    if (key < 0 || key > W4_TUNE_GROUP_LAUNCH_TOKENS || value < 0) return W4_ERR_INVALID_ARG;
    if (key == W4_TUNE_GROUP_LAUNCH_TOKENS && value > W4_MAX_M) return W4_ERR_INVALID_ARG;
    if (key == W4_TUNE_K_SPLITS && value != 0 && value != 1 && value != 2 && value != 4 && value != 8)
        return W4_ERR_INVALID_ARG;
    if (key == W4_TUNE_CHAIN_PREFETCH_KB && value > 4096) return W4_ERR_INVALID_ARG;
    if (key == W4_TUNE_TC_MIN_M && value > W4_MAX_M + 1) return W4_ERR_INVALID_ARG;
    if (key == W4_TUNE_BLOCKS_PER_SM && value > 2) return W4_ERR_INVALID_ARG;
    if (key == W4_TUNE_MAX_STAGES && value == 1) return W4_ERR_INVALID_ARG;
    g_tune[key] = value;
    return W4_OK;
}

int w4_get_tuning(int key)
{
    if (key < 0 || key > W4_TUNE_GROUP_LAUNCH_TOKENS) return -1;
    return g_tune[key];
}

// ------------------------------------------------------------ quantizers
w4_status w4_quantize_rows(const float* W, int N, int K, uint32_t* packed, float* s_w, w4_stream_t s)
{
    if (N < 0 || K <= 0 || K % 8 != 0) return N < 0 || K <= 0 ? W4_ERR_INVALID_ARG : W4_ERR_UNSUPPORTED_SHAPE;
    if (N == 0) return W4_OK;
    if (!W || !packed || !s_w) return W4_ERR_INVALID_ARG;
    if (!aligned(W, 16) || !aligned(packed, 4) || !aligned(s_w, 4)) return W4_ERR_MISALIGNED;
    return cuda_status(launch_w4_quantize_rows(W, N, K, packed, s_w, reinterpret_cast<cudaStream_t>(s)));
}

w4_status q4_0_quantize(const float* W, int N, int K, uint8_t* blocks, w4_stream_t s)
{
    if (N < 0 || K <= 0) return W4_ERR_INVALID_ARG;
    if (K % 32 != 0) return W4_ERR_UNSUPPORTED_SHAPE;
    if (N == 0) return W4_OK;
    if (!W || !blocks) return W4_ERR_INVALID_ARG;
    if (!aligned(W, 16)) return W4_ERR_MISALIGNED;
    return cuda_status(launch_q4_0_quantize(W, N, K, blocks, reinterpret_cast<cudaStream_t>(s)));
}

w4_status i8g32_quantize(const float* W, int N, int K, int8_t* q, uint16_t* d, w4_stream_t s)
{
    if (N < 0 || K <= 0) return W4_ERR_INVALID_ARG;
    if (K % 32 != 0) return W4_ERR_UNSUPPORTED_SHAPE;
    if (N == 0) return W4_OK;
    if (!W || !q || !d) return W4_ERR_INVALID_ARG;
    if (!aligned(W, 16) || !aligned(q, 16) || !aligned(d, 2)) return W4_ERR_MISALIGNED;
    return cuda_status(launch_i8g32_quantize(W, N, K, q, d, reinterpret_cast<cudaStream_t>(s)));
}

// ---------------------------------------------------------------- repack
size_t w4_repacked_bytes(int N, int K)
{
    if (N < 0 || K <= 0 || K % 32 != 0) return 0;
    return tiles(N) * kRows * static_cast<size_t>(K) / 2;
}

size_t q4_0_repacked_bytes(int N, int K)
{
    if (N < 0 || K <= 0 || K % 32 != 0) return 0;
    return tiles(N) * kRows * (static_cast<size_t>(K) / 2 + static_cast<size_t>(K) / 16);
}

size_t i8g32_repacked_bytes(int N, int K)
{
    if (N < 0 || K <= 0 || K % 32 != 0) return 0;
    return tiles(N) * kRows * (static_cast<size_t>(K) + static_cast<size_t>(K) / 16);
}

size_t q6g32_repacked_bytes(int N, int K)
{
    if (N < 0 || K <= 0 || K % 32 != 0) return 0;
    return tiles(N) * kRows * (static_cast<size_t>(K) / 2 + static_cast<size_t>(K) / 4 + static_cast<size_t>(K) / 16);
}

w4_status w4_repack(const uint32_t* const* shard_packed, const int* shard_rows, int n_shards, int K, void* out,
                    size_t out_bytes, w4_stream_t s)
{
    if (K <= 0) return W4_ERR_INVALID_ARG;
    if (K % 32 != 0 || K > W4_MAX_K) return W4_ERR_UNSUPPORTED_SHAPE;
    ShardTable st;
    int N = 0;
    w4_status r = build_shards(reinterpret_cast<const void* const*>(shard_packed), nullptr, shard_rows, n_shards, st, N);
    if (r != W4_OK) return r;
    if (N == 0) return W4_OK;
    if (!out) return W4_ERR_INVALID_ARG;
    if (out_bytes < w4_repacked_bytes(N, K)) return W4_ERR_UNSUPPORTED_SHAPE;
    if (!aligned(out, 16)) return W4_ERR_MISALIGNED;
    for (int i = 0; i < n_shards; ++i)
        if (st.p[i] && !aligned(st.p[i], 16)) return W4_ERR_MISALIGNED;
    return cuda_status(launch_w4_repack(st, N, K, out, reinterpret_cast<cudaStream_t>(s)));
}

w4_status q4_0_repack(const uint8_t* const* shard_blocks, const int* shard_rows, int n_shards, int K, void* out,
                      size_t out_bytes, w4_stream_t s)
{
    if (K <= 0) return W4_ERR_INVALID_ARG;
    if (K % 32 != 0 || K > W4_MAX_K) return W4_ERR_UNSUPPORTED_SHAPE;
    ShardTable st;
    int N = 0;
    w4_status r = build_shards(reinterpret_cast<const void* const*>(shard_blocks), nullptr, shard_rows, n_shards, st, N);
    if (r != W4_OK) return r;
    if (N == 0) return W4_OK;
    if (!out) return W4_ERR_INVALID_ARG;
    if (out_bytes < q4_0_repacked_bytes(N, K)) return W4_ERR_UNSUPPORTED_SHAPE;
    if (!aligned(out, 16)) return W4_ERR_MISALIGNED;
    return cuda_status(launch_q4_0_repack(st, N, K, out, reinterpret_cast<cudaStream_t>(s)));
}

w4_status i8g32_repack(const int8_t* const* shard_q, const uint16_t* const* shard_d, const int* shard_rows,
                       int n_shards, int K, void* out, size_t out_bytes, w4_stream_t s)
{
    if (K <= 0) return W4_ERR_INVALID_ARG;
    if (K % 32 != 0 || K > W4_MAX_K) return W4_ERR_UNSUPPORTED_SHAPE;
    if (shard_d == nullptr) return W4_ERR_INVALID_ARG;
    ShardTable st;
    int N = 0;
    w4_status r = build_shards(reinterpret_cast<const void* const*>(shard_q), reinterpret_cast<const void* const*>(shard_d),
                               shard_rows, n_shards, st, N);
    if (r != W4_OK) return r;
    if (N == 0) return W4_OK;
    if (!out) return W4_ERR_INVALID_ARG;
    if (out_bytes < i8g32_repacked_bytes(N, K)) return W4_ERR_UNSUPPORTED_SHAPE;
    if (!aligned(out, 16)) return W4_ERR_MISALIGNED;
    for (int i = 0; i < n_shards; ++i) {
        if (st.p[i] && !aligned(st.p[i], 16)) return W4_ERR_MISALIGNED;
        if (st.p2[i] && !aligned(st.p2[i], 2)) return W4_ERR_MISALIGNED;
    }
    return cuda_status(launch_i8g32_repack(st, N, K, out, reinterpret_cast<cudaStream_t>(s)));
}

w4_status q6g32_repack(const int8_t* const* shard_q, const uint16_t* const* shard_d, const int* shard_rows,
                       int n_shards, int K, void* out, size_t out_bytes, w4_stream_t s)
{
    if (K <= 0) return W4_ERR_INVALID_ARG;
    if (K % 32 != 0 || K > W4_MAX_K) return W4_ERR_UNSUPPORTED_SHAPE;
    if (shard_d == nullptr) return W4_ERR_INVALID_ARG;
    ShardTable st;
    int N = 0;
    w4_status r = build_shards(reinterpret_cast<const void* const*>(shard_q), reinterpret_cast<const void* const*>(shard_d),
                               shard_rows, n_shards, st, N);
    if (r != W4_OK) return r;
    if (N == 0) return W4_OK;
    if (!out) return W4_ERR_INVALID_ARG;
    if (out_bytes < q6g32_repacked_bytes(N, K)) return W4_ERR_UNSUPPORTED_SHAPE;
    if (!aligned(out, 16)) return W4_ERR_MISALIGNED;
    for (int i = 0; i < n_shards; ++i)
        if (st.p2[i] && !aligned(st.p2[i], 2)) return W4_ERR_MISALIGNED;
    return cuda_status(launch_q6g32_repack(st, N, K, out, reinterpret_cast<cudaStream_t>(s)));
}

size_t w4_glu_repacked_bytes(int I, int K)
{
    if (I < 0 || I > (1 << 29) || K <= 0 || K % 32 != 0) return 0;
    return w4_repacked_bytes(8 * ((I + 3) / 4), K);
}

size_t q4_0_glu_repacked_bytes(int I, int K)
{
    if (I < 0 || I > (1 << 29) || K <= 0 || K % 32 != 0) return 0;
    return q4_0_repacked_bytes(8 * ((I + 3) / 4), K);
}

namespace {
// Two shards (gate, up) of I rows each, paired per tile by the repack.
w4_status glu_shards(const void* gate, const void* up, int I, int K, ShardTable& st, int& Nw)
{
    if (K <= 0 || I < 0) return W4_ERR_INVALID_ARG;
    if (K % 32 != 0 || K > W4_MAX_K || I > (1 << 29)) return W4_ERR_UNSUPPORTED_SHAPE;
    const void* p[2] = {gate, up};
    const int rows[2] = {I, I};
    int N = 0;
    w4_status r = build_shards(p, nullptr, rows, 2, st, N);
    if (r != W4_OK) return r;
    st.glu_rows = I;
    Nw = I > 0 ? 8 * ((I + 3) / 4) : 0;
    return W4_OK;
}
}  // namespace

w4_status w4_repack_glu(const uint32_t* gate, const uint32_t* up, int I, int K, void* out, size_t out_bytes,
                        w4_stream_t s)
{
    ShardTable st;
    int Nw = 0;
    w4_status r = glu_shards(gate, up, I, K, st, Nw);
    if (r != W4_OK || Nw == 0) return r;
    if (!out) return W4_ERR_INVALID_ARG;
    if (out_bytes < w4_glu_repacked_bytes(I, K)) return W4_ERR_UNSUPPORTED_SHAPE;
    if (!aligned(out, 16) || !aligned(gate, 16) || !aligned(up, 16)) return W4_ERR_MISALIGNED;
    return cuda_status(launch_w4_repack(st, Nw, K, out, reinterpret_cast<cudaStream_t>(s)));
}

w4_status q4_0_repack_glu(const uint8_t* gate, const uint8_t* up, int I, int K, void* out, size_t out_bytes,
                          w4_stream_t s)
{
    ShardTable st;
    int Nw = 0;
    w4_status r = glu_shards(gate, up, I, K, st, Nw);
    if (r != W4_OK || Nw == 0) return r;
    if (!out) return W4_ERR_INVALID_ARG;
    if (out_bytes < q4_0_glu_repacked_bytes(I, K)) return W4_ERR_UNSUPPORTED_SHAPE;
    if (!aligned(out, 16)) return W4_ERR_MISALIGNED;
    return cuda_status(launch_q4_0_repack(st, Nw, K, out, reinterpret_cast<cudaStream_t>(s)));
}

w4_status w4_concat_f32(const float* const* parts, const int* lens, int n_parts, float* out, w4_stream_t s)
{
    if (n_parts < 0 || (n_parts > 0 && (!parts || !lens))) return W4_ERR_INVALID_ARG;
    size_t off = 0;
    for (int i = 0; i < n_parts; ++i) {
        if (lens[i] < 0 || (lens[i] > 0 && (!parts[i] || !out))) return W4_ERR_INVALID_ARG;
        if (lens[i] == 0) continue;
        cudaError_t e = cudaMemcpyAsync(out + off, parts[i], static_cast<size_t>(lens[i]) * sizeof(float),
                                        cudaMemcpyDeviceToDevice, reinterpret_cast<cudaStream_t>(s));
        if (e != cudaSuccess) return W4_ERR_CUDA;
        off += static_cast<size_t>(lens[i]);
    }
    return W4_OK;
}

// ------------------------------------------------------------- per token
w4_status a8_quantize(const float* x, int M, int K, int8_t* qx, float* sx, w4_stream_t s)
{
    w4_status st = check_mk(M, K);
    if (st != W4_OK) return st;
    if (M == 0) return W4_OK;
    if (!x || !qx || !sx) return W4_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(qx, 16) || !aligned(sx, 4)) return W4_ERR_MISALIGNED;
    return cuda_status(launch_a8_quantize(x, M, K, qx, sx, false, reinterpret_cast<cudaStream_t>(s)));
}

w4_status w4a8_gemv(const void* w, const float* s_w, const float* bias, const int8_t* qx, const float* sx, int M,
                    int N, int K, float* y, w4_stream_t s)
{
    return gemv_common(FMT_W4, w, s_w, bias, qx, sx, M, N, K, y, reinterpret_cast<cudaStream_t>(s));
}

w4_status q4_0_gemv(const void* w, const float* bias, const int8_t* qx, const float* sx, int M, int N, int K,
                    float* y, w4_stream_t s)
{
    return gemv_common(FMT_Q4_0, w, nullptr, bias, qx, sx, M, N, K, y, reinterpret_cast<cudaStream_t>(s));
}

w4_status i8g32_gemv(const void* w, const float* bias, const int8_t* qx, const float* sx, int M, int N, int K,
                     float* y, w4_stream_t s)
{
    return gemv_common(FMT_I8G32, w, nullptr, bias, qx, sx, M, N, K, y, reinterpret_cast<cudaStream_t>(s));
}

w4_status q6g32_gemv(const void* w, const float* bias, const int8_t* qx, const float* sx, int M, int N, int K,
                     float* y, w4_stream_t s)
{
    return gemv_common(FMT_Q6G32, w, nullptr, bias, qx, sx, M, N, K, y, reinterpret_cast<cudaStream_t>(s));
}

w4_status q6g32_linear(const void* w, const float* bias, const float* x, int M, int N, int K, float* y, int8_t* qx,
                       float* sx, unsigned flags, w4_stream_t s)
{
    return linear_common(FMT_Q6G32, w, nullptr, bias, x, M, N, K, y, qx, sx, flags,
                         reinterpret_cast<cudaStream_t>(s));
}

w4_status w4a8_linear(const void* w, const float* s_w, const float* bias, const float* x, int M, int N, int K,
                      float* y, int8_t* qx, float* sx, unsigned flags, w4_stream_t s)
{
    return linear_common(FMT_W4, w, s_w, bias, x, M, N, K, y, qx, sx, flags, reinterpret_cast<cudaStream_t>(s));
}

w4_status q4_0_linear(const void* w, const float* bias, const float* x, int M, int N, int K, float* y, int8_t* qx,
                      float* sx, unsigned flags, w4_stream_t s)
{
    return linear_common(FMT_Q4_0, w, nullptr, bias, x, M, N, K, y, qx, sx, flags, reinterpret_cast<cudaStream_t>(s));
}

w4_status i8g32_linear(const void* w, const float* bias, const float* x, int M, int N, int K, float* y, int8_t* qx,
                       float* sx, unsigned flags, w4_stream_t s)
{
    return linear_common(FMT_I8G32, w, nullptr, bias, x, M, N, K, y, qx, sx, flags,
                         reinterpret_cast<cudaStream_t>(s));
}

// ------------------------------------------------ fusions around the linear
w4_status w4a8_linear_fused(const void* w, const float* s_w, const float* bias, const float* x, int M, int N, int K,
                            float* y, int8_t* qx, float* sx, const w4_fusion* f, unsigned flags, w4_stream_t s)
{
    return linear_common(FMT_W4, w, s_w, bias, x, M, N, K, y, qx, sx, flags, reinterpret_cast<cudaStream_t>(s), f);
}

w4_status q4_0_linear_fused(const void* w, const float* bias, const float* x, int M, int N, int K, float* y,
                            int8_t* qx, float* sx, const w4_fusion* f, unsigned flags, w4_stream_t s)
{
    return linear_common(FMT_Q4_0, w, nullptr, bias, x, M, N, K, y, qx, sx, flags,
                         reinterpret_cast<cudaStream_t>(s), f);
}

w4_status i8g32_linear_fused(const void* w, const float* bias, const float* x, int M, int N, int K, float* y,
                             int8_t* qx, float* sx, const w4_fusion* f, unsigned flags, w4_stream_t s)
{
    return linear_common(FMT_I8G32, w, nullptr, bias, x, M, N, K, y, qx, sx, flags,
                         reinterpret_cast<cudaStream_t>(s), f);
}

w4_status q6g32_linear_fused(const void* w, const float* bias, const float* x, int M, int N, int K, float* y,
                             int8_t* qx, float* sx, const w4_fusion* f, unsigned flags, w4_stream_t s)
{
    return linear_common(FMT_Q6G32, w, nullptr, bias, x, M, N, K, y, qx, sx, flags,
                         reinterpret_cast<cudaStream_t>(s), f);
}

namespace {
w4_status check_norm_args(const float* x, const float* g, float eps, int M, int K)
{
    w4_status st = check_mk(M, K);
    if (st != W4_OK) return st;
    if (M == 0) return W4_OK;
    if (!x || !g || !(eps > 0.0f) || !(eps < 3.0e38f)) return W4_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(g, 16)) return W4_ERR_MISALIGNED;
    return W4_OK;
}
}  // namespace

w4_status rms_a8_quantize(const float* x, const float* norm_weight, float eps, int M, int K, int8_t* qx, float* sx,
                          unsigned flags, w4_stream_t s)
{
    if ((flags & ~W4_FLAG_PDL) != 0) return W4_ERR_INVALID_ARG;
    w4_status st = check_norm_args(x, norm_weight, eps, M, K);
    if (st != W4_OK || M == 0) return st;
    if (!qx || !sx) return W4_ERR_INVALID_ARG;
    if (!aligned(qx, 16) || !aligned(sx, 4)) return W4_ERR_MISALIGNED;
    return cuda_status(launch_rms_a8_quantize(x, norm_weight, eps, M, K, qx, sx, (flags & W4_FLAG_PDL) != 0,
                                              reinterpret_cast<cudaStream_t>(s)));
}

w4_status w4_rmsnorm(const float* x, const float* norm_weight, float eps, int M, int K, float* out, unsigned flags,
                     w4_stream_t s)
{
    if ((flags & ~W4_FLAG_PDL) != 0) return W4_ERR_INVALID_ARG;
    w4_status st = check_norm_args(x, norm_weight, eps, M, K);
    if (st != W4_OK || M == 0) return st;
    if (!out) return W4_ERR_INVALID_ARG;
    if (!aligned(out, 16)) return W4_ERR_MISALIGNED;
    return cuda_status(launch_rmsnorm(x, norm_weight, eps, M, K, out, (flags & W4_FLAG_PDL) != 0,
                                      reinterpret_cast<cudaStream_t>(s)));
}

w4_status w4_glu(const float* gu, int kind, int M, int I, float* out, unsigned flags, w4_stream_t s)
{
    if ((flags & ~W4_FLAG_PDL) != 0 || M < 0 || I < 0) return W4_ERR_INVALID_ARG;
    if (kind != W4_GLU_SILU && kind != W4_GLU_GELU_TANH) return W4_ERR_INVALID_ARG;
    if (M > W4_MAX_M || I > (1 << 30)) return W4_ERR_UNSUPPORTED_SHAPE;
    if (M == 0 || I == 0) return W4_OK;
    if (!gu || !out) return W4_ERR_INVALID_ARG;
    if (!aligned(gu, 4) || !aligned(out, 4)) return W4_ERR_MISALIGNED;
    return cuda_status(launch_glu(gu, kind, M, I, out, (flags & W4_FLAG_PDL) != 0, reinterpret_cast<cudaStream_t>(s)));
}

w4_status w4_add(const float* a, const float* b, long long n, float* out, unsigned flags, w4_stream_t s)
{
    if ((flags & ~W4_FLAG_PDL) != 0 || n < 0) return W4_ERR_INVALID_ARG;
    if (n > (1LL << 31) * 255) return W4_ERR_UNSUPPORTED_SHAPE;
    if (n == 0) return W4_OK;
    if (!a || !b || !out) return W4_ERR_INVALID_ARG;
    if (!aligned(a, 4) || !aligned(b, 4) || !aligned(out, 4)) return W4_ERR_MISALIGNED;
    return cuda_status(launch_add(a, b, n, out, (flags & W4_FLAG_PDL) != 0, reinterpret_cast<cudaStream_t>(s)));
}

// ------------------------------------- weight-only paths on float activations
w4_status w8_quantize_rows(const float* W, int N, int K, int8_t* q, float* s_w, w4_stream_t s)
{
    if (N < 0 || K <= 0) return W4_ERR_INVALID_ARG;
    if (K % 4 != 0) return W4_ERR_UNSUPPORTED_SHAPE;
    if (N == 0) return W4_OK;
    if (!W || !q || !s_w) return W4_ERR_INVALID_ARG;
    if (!aligned(W, 16) || !aligned(q, 4) || !aligned(s_w, 4)) return W4_ERR_MISALIGNED;
    return cuda_status(launch_w8_quantize_rows(W, N, K, q, s_w, reinterpret_cast<cudaStream_t>(s)));
}

size_t w8_repacked_bytes(int N, int K)
{
    if (N < 0 || K <= 0 || K % 32 != 0) return 0;
    return tiles(N) * kRows * static_cast<size_t>(K);
}

w4_status w8_repack(const int8_t* const* shard_q, const int* shard_rows, int n_shards, int K, void* out,
                    size_t out_bytes, w4_stream_t s)
{
    if (K <= 0) return W4_ERR_INVALID_ARG;
    if (K % 32 != 0 || K > W4_MAX_K) return W4_ERR_UNSUPPORTED_SHAPE;
    ShardTable st;
    int N = 0;
    w4_status r = build_shards(reinterpret_cast<const void* const*>(shard_q), nullptr, shard_rows, n_shards, st, N);
    if (r != W4_OK) return r;
    if (N == 0) return W4_OK;
    if (!out) return W4_ERR_INVALID_ARG;
    if (out_bytes < w8_repacked_bytes(N, K)) return W4_ERR_UNSUPPORTED_SHAPE;
    if (!aligned(out, 16)) return W4_ERR_MISALIGNED;
    for (int i = 0; i < n_shards; ++i)
        if (st.p[i] && !aligned(st.p[i], 16)) return W4_ERR_MISALIGNED;
    return cuda_status(launch_w8_repack(st, N, K, out, reinterpret_cast<cudaStream_t>(s)));
}

namespace {
w4_status a32_common(int fmt, const void* w, const float* s_w, const float* bias, const float* x, int M, int N,
                     int K, float* y, unsigned flags, cudaStream_t s)
{
    w4_status st = check_mk(M, K);
    if (st != W4_OK) return st;
    if (N < 0 || (flags & ~W4_FLAG_PDL) != 0) return W4_ERR_INVALID_ARG;
    if (M > 4 || N > (1 << 30) - 8) return W4_ERR_UNSUPPORTED_SHAPE;
    if (M == 0 || N == 0) return W4_OK;
    if (!w || !s_w || !x || !y) return W4_ERR_INVALID_ARG;
    if (!aligned(w, 16) || !aligned(x, 16) || !aligned(y, 4) || !aligned(s_w, 4) || (bias && !aligned(bias, 4)))
        return W4_ERR_MISALIGNED;
    GemvArgs a = {};
    a.w = static_cast<const uint8_t*>(w);
    a.s_w = s_w;
    a.bias = bias;
    a.x = x;
    a.y = y;
    a.n_out = N;
    a.M = M;
    a.N = N;
    a.K = K;
    return run_gemv(fmt, a, false, flags, s);
}
}  // namespace

w4_status w4a32_gemv(const void* w, const float* s_w, const float* bias, const float* x, int M, int N, int K,
                     float* y, unsigned flags, w4_stream_t s)
{
    return a32_common(FMT_W4F, w, s_w, bias, x, M, N, K, y, flags, reinterpret_cast<cudaStream_t>(s));
}

w4_status w8a32_gemv(const void* w, const float* s_w, const float* bias, const float* x, int M, int N, int K,
                     float* y, unsigned flags, w4_stream_t s)
{
    return a32_common(FMT_W8F, w, s_w, bias, x, M, N, K, y, flags, reinterpret_cast<cudaStream_t>(s));
}

// The single-linear calls keep nothing between launches: K is never split
// across blocks through global memory, so no call needs a workspace.
size_t w4_workspace_bytes(int M, int N, int K)
{
    (void)M;
    (void)N;
    (void)K;
    return 0;
}

// ----------------------------------------------------------------- chains
size_t w4_chain_workspace_bytes(void) { return 256; }

namespace {
// Checks of a chain's descriptors shared by both chain entry points; W4_OK
// with nothing to launch sets *empty.
w4_status check_chain(const w4_linear_desc* descs, int n, int M, bool* empty)
{
    *empty = false;
    if (n < 0 || M < 0 || (n > 0 && descs == nullptr)) return W4_ERR_INVALID_ARG;
    if (n > W4_MAX_CHAIN || M > W4_MAX_M) return W4_ERR_UNSUPPORTED_SHAPE;
    if (n == 0 || M == 0) {
        *empty = true;
        return W4_OK;
    }
    for (int i = 0; i < n; ++i) {
        const w4_linear_desc& d = descs[i];
        w4_status st = check_mk(M, d.K);
        if (st != W4_OK) return st;
        if (d.N <= 0) return d.N < 0 ? W4_ERR_INVALID_ARG : W4_ERR_UNSUPPORTED_SHAPE;
        if (!d.w || !d.s_w || !d.x || !d.y) return W4_ERR_INVALID_ARG;
        if (!aligned(d.w, 16) || !aligned(d.x, 16) || !aligned(d.y, 4) || !aligned(d.s_w, 4) ||
            (d.bias && !aligned(d.bias, 4)) || (d.qx && !aligned(d.qx, 16)) || (d.sx && !aligned(d.sx, 4)))
            return W4_ERR_MISALIGNED;
    }
    return W4_OK;
}
}  // namespace

w4_status w4a8_linear_chain(const w4_linear_desc* descs, int n, int M, void* workspace, size_t ws_bytes,
                            w4_stream_t s)
{
    bool empty = false;
    w4_status st = check_chain(descs, n, M, &empty);
    if (st != W4_OK || empty) return st;
    if (workspace == nullptr) return W4_ERR_INVALID_ARG;
    if (ws_bytes < w4_chain_workspace_bytes()) return W4_ERR_UNSUPPORTED_SHAPE;
    if (!aligned(workspace, 16)) return W4_ERR_MISALIGNED;
    return run_chain(descs, n, M, static_cast<unsigned*>(workspace), reinterpret_cast<cudaStream_t>(s));
}

// ------------------------------------------- chains without caller memory
// For callers that cannot allocate device memory (see w4a8.h): the chain's
// grid-barrier state lives in this fixed array instead of a caller workspace.
// In host code `g_chain_scratch` is only a host-side stand-in for the symbol;
// the kernel gets the device address from cudaGetSymbolAddress.
constexpr size_t kChainScratchBytes = 256;
static __device__ __align__(256) unsigned char g_chain_scratch[kChainScratchBytes];

namespace {
// Device address of the scratch array per device, looked up once.  The
// look-up runs under the set-up lock, so threads calling at once for the
// first time store the same address once.
std::atomic<unsigned*> g_chain_scratch_ptr[kMaxDevices];

w4_status chain_scratch(unsigned** out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return W4_ERR_CUDA;
    unsigned* p = g_chain_scratch_ptr[dev].load(std::memory_order_acquire);
    if (p == nullptr) {
        std::lock_guard<std::mutex> lock(g_setup_mutex);
        p = g_chain_scratch_ptr[dev].load(std::memory_order_relaxed);
        if (p == nullptr) {
            void* a = nullptr;
            if (cudaGetSymbolAddress(&a, g_chain_scratch) != cudaSuccess || a == nullptr) return W4_ERR_CUDA;
            p = static_cast<unsigned*>(a);
            g_chain_scratch_ptr[dev].store(p, std::memory_order_release);
        }
    }
    *out = p;
    return W4_OK;
}
}  // namespace

size_t w4_chain_noalloc_scratch_bytes(void) { return kChainScratchBytes; }

w4_status w4a8_linear_chain_noalloc(const w4_linear_desc* descs, int n, int M, w4_stream_t s)
{
    if (w4_chain_workspace_bytes() > kChainScratchBytes) return W4_ERR_UNSUPPORTED_SHAPE;
    // every check first: a call that fails them enqueues nothing, not even the clear below
    bool empty = false;
    w4_status st = check_chain(descs, n, M, &empty);
    if (st != W4_OK || empty) return st;
    unsigned* scratch = nullptr;
    st = chain_scratch(&scratch);
    if (st != W4_OK) return st;
    // the array keeps the previous call's contents: the barrier count must start at zero
    if (cudaMemsetAsync(scratch, 0, w4_chain_workspace_bytes(), reinterpret_cast<cudaStream_t>(s)) != cudaSuccess)
        return W4_ERR_CUDA;
    return run_chain(descs, n, M, scratch, reinterpret_cast<cudaStream_t>(s));
}

// ------------------------------------------------------ device error word
w4_status w4_device_error(unsigned* code)
{
    if (!code) return W4_ERR_INVALID_ARG;
    DeviceInfo* dev = nullptr;
    w4_status st = device_info(&dev);
    if (st != W4_OK) return st;
    if (cudaDeviceSynchronize() != cudaSuccess) return W4_ERR_CUDA;
    unsigned v = 0;
    if (cudaMemcpy(&v, dev->err, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return W4_ERR_CUDA;
    *code = v;
    return v ? W4_ERR_DEVICE_TIMEOUT : W4_OK;
}

w4_status w4_last_device_error(unsigned* code) { return w4_device_error(code); }

// ------------------------------------------------------ pure-read probe
w4_status w4_hbm_read(const void* buf, size_t bytes, unsigned* sink, w4_stream_t s)
{
    if (!sink || (bytes > 0 && !buf)) return W4_ERR_INVALID_ARG;
    if (bytes % 16 != 0) return W4_ERR_UNSUPPORTED_SHAPE;
    if (!aligned(sink, 4) || (buf && !aligned(buf, 16))) return W4_ERR_MISALIGNED;
    DeviceInfo* dev = nullptr;
    const w4_status st = device_info(&dev);
    if (st != W4_OK) return st;
    return cuda_status(launch_hbm_read(buf, bytes, sink, dev->err, dev->sms, reinterpret_cast<cudaStream_t>(s)));
}

w4_status w4_selftest_wait_timeout(int cluster, unsigned timeout_us, w4_stream_t s)
{
    if ((cluster != 0 && cluster != 1) || timeout_us == 0 || timeout_us > 1000000u) return W4_ERR_INVALID_ARG;
    DeviceInfo* dev = nullptr;
    const w4_status st = device_info(&dev);
    if (st != W4_OK) return st;
    return cuda_status(launch_wait_selftest(cluster, 1000ull * timeout_us, dev->err, reinterpret_cast<cudaStream_t>(s)));
}

w4_status w4_clear_device_error(void)
{
    DeviceInfo* dev = nullptr;
    w4_status st = device_info(&dev);
    if (st != W4_OK) return st;
    if (cudaMemset(dev->err, 0, sizeof(unsigned)) != cudaSuccess) return W4_ERR_CUDA;
    return cuda_status(cudaDeviceSynchronize());
}

}  // extern "C"
