/*
 * w4a8.h -- C ABI of the GB300 (sm_103a) bit-quantized decode GEMV library.
 *
 * The library computes the batch-1 (and few-token) decode linear layer
 *     y[m][j] = W[j][:] . x[m][:] + b[j]
 * with 4-bit (or 8-bit) weights and per-token INT8 activations, as defined on
 *   [Orin-INT4]   "Jetson Orin AGX INT4 推理优化实践：super 分支从 9 tok/s 到 24 tok/s"
 *   [310B-Gemma4] "在香橙派上跑 Gemma4：vLLM 适配昇腾 310B 的内核开发实录"
 *
 * Conventions for every entry point:
 *   - Pointers are DEVICE pointers unless a parameter says "host".  The caller
 *     allocates and frees every buffer; the library allocates nothing and keeps
 *     no state beyond cached device attributes and one device error word.
 *   - Work is enqueued on the caller's stream `s` and nothing synchronises.
 *   - Arguments are checked on the host before any launch; a failed check
 *     returns an error and launches nothing.  A launch failure returns
 *     W4_ERR_CUDA.  Kernels never trap: a bounded wait that runs out sets the
 *     device error word (see w4_device_error) and the kernel returns.
 *   - M = 0 or N = 0 is a valid empty call (returns W4_OK, launches nothing).
 *   - Shapes: 1 <= M <= 16 tokens, K > 0, K % 32 == 0.
 *   - Alignment: weight buffers, qx and x must be 16-byte aligned; float
 *     arrays 4-byte aligned.  A violation returns W4_ERR_MISALIGNED.
 *
 * Formats ("canonical" = the format a caller stores, before repacking):
 *   W4    per-row symmetric INT4 [Orin-INT4] §"从 FP 线性层到 INT4 DP4A 的数学推导":
 *         uint32 [N][K/8], weight k of a word in bits 4k..4k+3 (two's complement,
 *         §"DP4A 做了什么"), plus float s_w[N].
 *   Q4_0  [310B-Gemma4] §3.1: 18-byte blocks [N][K/32]: fp16 d (little endian),
 *         then 16 nibble bytes; byte i holds element i (low) and i+16 (high);
 *         element value n - 8, weight d*(n - 8).
 *   I8G32 [310B-Gemma4] §3.2 (lm_head widened to int8 with per-group fp16
 *         scales): int8 q [N][K] plus fp16 d [N][K/32]; weight d*q.
 *
 * Device ("repacked") layouts, produced by the *_repack calls and consumed by
 * the GEMVs.  Rows are grouped in tiles of 8 (T = ceil(N/8) tiles; rows past N
 * are zero).  C = K/32 chunks of 32 weights per row.  Unit (t, c, r) is the
 * 32 weights of row 8t+r in chunk c; units are stored in (t, c, r) order:
 *   W4, Q4_0: 16 bytes per unit at ((t*C + c)*8 + r)*16.  Word w (0..3) of the
 *         unit holds weights 32c+8w+b in the low nibble of byte b and
 *         32c+8w+4+b in the high nibble.  W4 stores each nibble biased,
 *         n = q + 8 in 0..15; Q4_0 stores 4-bit two's complement n - 8.
 *         Padded rows are zero bytes and never reach the output.
 *         Q4_0 then has a plane of fp16 d, one per unit, at byte
 *         T*8*C*16 + ((t*C + c)*8 + r)*2.
 *   I8G32: 32 bytes per unit (the 32 int8 in order) at ((t*C + c)*8 + r)*32,
 *         then the fp16 d plane at byte T*8*C*32 + ((t*C + c)*8 + r)*2.
 *   Q6G32 (the I8G32 values, q in [-32, 31], packed in 6 bits; a layout of
 *         this library, [310B-Gemma4] §3.2 widens them to int8 instead):
 *         n = q + 32.  A low plane of 16 bytes per unit at ((t*C + c)*8 + r)*16
 *         holding n & 15 with the W4 nibble places; a high plane of 8 bytes per
 *         unit at T*8*C*16 + ((t*C + c)*8 + r)*8 holding n >> 4, weight
 *         32c+16h+4s+b in bits 2s..2s+1 of byte b of word h; then the fp16 d
 *         plane at T*8*C*24 + ((t*C + c)*8 + r)*2.  0.8125 bytes per weight.
 */
#ifndef W4A8_H
#define W4A8_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* w4_stream_t; /* a cudaStream_t; NULL = legacy default stream */

typedef enum {
    W4_OK = 0,
    W4_ERR_INVALID_ARG = 1,       /* null pointer, negative size, bad shard table */
    W4_ERR_UNSUPPORTED_SHAPE = 2, /* M > 16, K % 32 != 0, K too large, buffer too small */
    W4_ERR_MISALIGNED = 3,        /* a pointer breaks the alignment rule above */
    W4_ERR_CUDA = 4,              /* a CUDA runtime call or launch failed */
    W4_ERR_DEVICE_TIMEOUT = 5     /* a kernel's bounded wait ran out (see w4_device_error) */
} w4_status;

/* Human-readable name of a status.  Never NULL. */
const char* w4_status_str(w4_status st);

/* Library ABI version (increases on incompatible change). */
int w4_version(void);

/* Largest K each GEMV accepts.  Row sums of biased products n * x
 * (|n x| <= 15 * 127) are accumulated in int32, which bounds K near 1.1e6;
 * the library accepts K <= 131072. */
#define W4_MAX_K 131072
#define W4_MAX_M 16
#define W4_MAX_SHARDS 8

/* Flags for the *_linear calls. */
#define W4_FLAG_PDL 1u /* launch as a programmatic dependent of the previous kernel in
                          the stream.  Legal only when the previous kernel does not
                          write this call's weight buffer (weights are prefetched
                          before the dependency wait); inputs x/qx/sx and outputs are
                          touched only after it. */

/* ------------------------------------------------------------------------
 * Launch tuning (process-wide; value 0 restores the automatic choice).
 *   W4_TUNE_BLOCKS_PER_SM  1: one GEMV block per SM with the whole shared
 *                          memory; 2: half of it, so that a GEMV launched with
 *                          W4_FLAG_PDL is resident beside the previous one.
 *                          Default: 2 for one token (when a ring fits), 1 for
 *                          several.
 *   W4_TUNE_MAX_STAGES     cap on the ring depth per warp (>= 2).
 *   W4_TUNE_GRID_BLOCKS    cap on the grid size (default: the SM count).
 *   W4_TUNE_TC_MIN_M       per-row INT4 calls with at least this many tokens
 *                          run on the tensor cores (default 0: 3; 17: never).
 *   W4_TUNE_K_SPLITS       DP4A GEMVs of one or two tokens: K split over a
 *                          cluster of 2, 4 or 8 blocks sharing a tile range
 *                          (where each split keeps at least 16 chunks of 32 K);
 *                          0 or 1: no split, the default (a split measured
 *                          slower on every shape tried).
 *   W4_TUNE_GROUP_LAUNCH_TOKENS  Q4_0 / I8G32 / Q6G32 calls with more tokens
 *                          than this run as launches of at most this many
 *                          tokens (1..16; default 0: 8).
 *   W4_TUNE_CHAIN_PREFETCH_KB  w4a8_linear_chain: weight bytes (KB, at most
 *                          4096) each block prefetches into L2 ahead of the
 *                          weights it copies into shared memory (default
 *                          0: none; below 32 none).
 * Returns W4_ERR_INVALID_ARG for an unknown key or an out-of-range value.
 * Not thread-safe with concurrent launches; set before launching.
 * ------------------------------------------------------------------------ */
#define W4_TUNE_BLOCKS_PER_SM 0
#define W4_TUNE_MAX_STAGES 1
#define W4_TUNE_GRID_BLOCKS 2
#define W4_TUNE_TC_MIN_M 3
#define W4_TUNE_CHAIN_PREFETCH_KB 4
#define W4_TUNE_K_SPLITS 5
#define W4_TUNE_GROUP_LAUNCH_TOKENS 6
w4_status w4_set_tuning(int key, int value);
int w4_get_tuning(int key); /* current value, -1 for an unknown key */

/* ------------------------------------------------------------------------
 * Launch plan: what a GEMV or linear call launches on a device, computed on
 * the host from a description of the device (no CUDA call, so it also runs
 * without a GPU).  The launch path takes its decisions through the same
 * functions, with the current tuning (w4_set_tuning).
 *   fmt:  W4_FMT_W4, W4_FMT_Q4_0, W4_FMT_I8G32 or W4_FMT_Q6G32.
 *   M, N, K: the call's shapes (N outputs; a gated call reads 2N weight rows).
 *   what: 0 for the *_gemv call on int8 codes, or W4_PLAN_LINEAR for the
 *         *_linear call on float x, with W4_PLAN_NORM (RMSNorm fused in, a
 *         *_linear_fused option) and W4_PLAN_GLU (gated, W4 and Q4_0 only).
 *   dev:  host; the device attributes of the same names (SM count, shared
 *         memory per SM, shared memory per block reserved by the system,
 *         opt-in maximum per block).  w4_describe_device fills it for the
 *         current device.
 *   out:  host; path (W4_PATH_*), quantize_launches (1 when a *_linear call
 *         quantizes x in a kernel of its own first, else 0), and the GEMV
 *         launch: grid, threads, smem_bytes (dynamic, per block), stages
 *         (weight-ring depth), k_splits (K splits per tile range, which form
 *         one thread-block cluster: per 128-row group on the tensor cores, per
 *         range of 8-row tiles on DP4A; 1 without a split), gemv_launches
 *         (GEMV kernels per call: 0 without a GEMV; 2 for a Q4_0 / I8G32 /
 *         Q6G32 call of more than 8 tokens, which runs tokens 0-7 and the
 *         rest as two launches of one kernel over the same weights, both
 *         as the fields above describe; otherwise 1).
 * Paths:
 *   W4_PATH_NONE          nothing (M = 0, or N = 0 where only the quantizer
 *                         of a *_linear call runs);
 *   W4_PATH_FUSED         one DP4A GEMV launch with the activation quantizer
 *                         (and the norm) in its prologue;
 *   W4_PATH_CODES_SMEM    DP4A GEMV on int8 codes staged in shared memory;
 *   W4_PATH_CODES_GLOBAL  DP4A GEMV reading the int8 codes from global memory;
 *   W4_PATH_TENSOR_CORES  tensor-core GEMV on int8 codes (per-row INT4).
 * Returns W4_ERR_INVALID_ARG for a null pointer, an unknown fmt or flag, a
 * non-positive device field, W4_PLAN_NORM without W4_PLAN_LINEAR or a GLU on
 * I8G32 / Q6G32, and otherwise the shape status the call would return.
 * ------------------------------------------------------------------------ */
#define W4_FMT_W4 0
#define W4_FMT_Q4_0 1
#define W4_FMT_I8G32 2
#define W4_FMT_Q6G32 3
#define W4_PLAN_LINEAR 1u
#define W4_PLAN_NORM 2u
#define W4_PLAN_GLU 4u
#define W4_PATH_NONE 0
#define W4_PATH_FUSED 1
#define W4_PATH_CODES_SMEM 2
#define W4_PATH_CODES_GLOBAL 3
#define W4_PATH_TENSOR_CORES 4
typedef struct {
    int sms;
    int smem_per_sm;
    int smem_reserved;
    int smem_optin;
} w4_device_desc;
typedef struct {
    int path;
    int quantize_launches;
    int grid;
    int threads;
    int smem_bytes;
    int stages;
    int k_splits;
    int gemv_launches;
} w4_launch_plan;
w4_status w4_plan(int fmt, int M, int N, int K, unsigned what, const w4_device_desc* dev, w4_launch_plan* out);
/* The current device's description (W4_ERR_CUDA without a usable device). */
w4_status w4_describe_device(w4_device_desc* out);

/* ------------------------------------------------------------------------
 * Load time: quantize float weights (device kernels).
 * ------------------------------------------------------------------------ */

/* Per-row symmetric INT4, [Orin-INT4] §"从 FP 线性层到 INT4 DP4A 的数学推导":
 * s_w[j] = max_i |W[j][i]| / 7 (the page leaves s^W open; this maps the row's
 * absmax to the top code, as s^x does for x), q = clip(rint(W / s_w), -8, 7),
 * packed into canonical W4 words.  W: float [N][K] (16-B aligned, row-major);
 * packed: uint32 [N][K/8]; s_w: float [N].  K % 8 == 0. */
w4_status w4_quantize_rows(const float* W, int N, int K, uint32_t* packed, float* s_w, w4_stream_t s);

/* Q4_0 blocks, [310B-Gemma4] §3.1: d = fp16(max|w| / 8) per 32-block,
 * n = clip(rint(w / d), -8, 7) + 8.  W: float [N][K]; blocks: [N][K/32][18]. */
w4_status q4_0_quantize(const float* W, int N, int K, uint8_t* blocks, w4_stream_t s);

/* int8 + fp16 group-32 scales, [310B-Gemma4] §3.2: d = fp16(max|w| / 32),
 * q = clip(rint(w / d), -32, 31).  q: int8 [N][K]; d: fp16 bits [N][K/32]. */
w4_status i8g32_quantize(const float* W, int N, int K, int8_t* q, uint16_t* d, w4_stream_t s);

/* ------------------------------------------------------------------------
 * Load time on the host: the same three quantizers as plain C++ over host
 * memory, for loaders that hold float weights on the host.  Outputs are
 * bit-identical to the device calls above (IEEE fp32 division,
 * round-half-to-even to an integer, fp16 round-to-nearest-even).  All
 * pointers are HOST pointers (no alignment rule); the call is synchronous,
 * makes no CUDA call and keeps no state, so it is safe from any thread.
 * Same shapes and checks as the device calls: N >= 0, K > 0, and K % 8 == 0
 * (w4_quantize_rows_host) or K % 32 == 0 (the group formats).
 * ------------------------------------------------------------------------ */
w4_status w4_quantize_rows_host(const float* W, int N, int K, uint32_t* packed, float* s_w);
w4_status q4_0_quantize_host(const float* W, int N, int K, uint8_t* blocks);
w4_status i8g32_quantize_host(const float* W, int N, int K, int8_t* q, uint16_t* d);

/* ------------------------------------------------------------------------
 * Load time: repack canonical weights into the device layout, fusing shards.
 * [310B-Gemma4] §3.1 (load-time reorder; q/k/v and gate/up concatenated by
 * rows into one matrix, one repack, one matmul per token).
 *
 * shard_* are HOST arrays of n_shards (1..W4_MAX_SHARDS) device pointers;
 * shard_rows is a HOST array of row counts.  The fused matrix has
 * N = sum(shard_rows) rows, shard 0 first.  `out` must hold *_repacked_bytes
 * (N, K) bytes (out_bytes is checked) and must not overlap the shards.
 * ------------------------------------------------------------------------ */
size_t w4_repacked_bytes(int N, int K);
w4_status w4_repack(const uint32_t* const* shard_packed, const int* shard_rows, int n_shards, int K,
                    void* out, size_t out_bytes, w4_stream_t s);

size_t q4_0_repacked_bytes(int N, int K);
w4_status q4_0_repack(const uint8_t* const* shard_blocks, const int* shard_rows, int n_shards, int K,
                      void* out, size_t out_bytes, w4_stream_t s);

size_t i8g32_repacked_bytes(int N, int K);
w4_status i8g32_repack(const int8_t* const* shard_q, const uint16_t* const* shard_d, const int* shard_rows,
                       int n_shards, int K, void* out, size_t out_bytes, w4_stream_t s);

/* Q6G32 from the I8G32 canonical format (codes must lie in [-32, 31], as
 * i8g32_quantize makes them; other codes are packed modulo 64). */
size_t q6g32_repacked_bytes(int N, int K);
w4_status q6g32_repack(const int8_t* const* shard_q, const uint16_t* const* shard_d, const int* shard_rows,
                       int n_shards, int K, void* out, size_t out_bytes, w4_stream_t s);

/* Gate/up weights of a gated MLP, paired for the GLU epilogue of the
 * *_linear_fused calls: row tile t holds gate rows 4t..4t+3 and then up rows
 * 4t..4t+3 (8 ceil(I/4) rows in all, padding past I zero), so one thread
 * block sees both halves of every output.  gate and up: canonical [I][..]
 * device arrays (W4: uint32 [I][K/8]; Q4_0: 18-byte blocks [I][K/32]).
 * out: *_glu_repacked_bytes(I, K) bytes, 16-byte aligned. */
size_t w4_glu_repacked_bytes(int I, int K);
w4_status w4_repack_glu(const uint32_t* gate, const uint32_t* up, int I, int K, void* out, size_t out_bytes,
                        w4_stream_t s);
size_t q4_0_glu_repacked_bytes(int I, int K);
w4_status q4_0_repack_glu(const uint8_t* gate, const uint8_t* up, int I, int K, void* out, size_t out_bytes,
                          w4_stream_t s);

/* Concatenate per-shard float vectors (per-row scales s_w, bias) into `out`
 * in shard order.  parts: HOST array of device pointers; lens: HOST array. */
w4_status w4_concat_f32(const float* const* parts, const int* lens, int n_parts, float* out, w4_stream_t s);

/* ------------------------------------------------------------------------
 * Per token: activation quantization.
 * [Orin-INT4] §"从 FP 线性层到 INT4 DP4A 的数学推导":
 *   sx[m] = max_i |x[m][i]| / 127 (IEEE fp32 division),
 *   qx[m][i] = clip(rint(x[m][i] / sx[m]), -127, 127); an all-zero token gives
 *   sx = 0, qx = 0.  NaN/Inf inputs are undefined behaviour.
 * x: float [M][K]; qx: int8 [M][K]; sx: float [M].
 * ------------------------------------------------------------------------ */
w4_status a8_quantize(const float* x, int M, int K, int8_t* qx, float* sx, w4_stream_t s);

/* ------------------------------------------------------------------------
 * Per token: GEMV on INT8 activations.
 *
 * w4a8_gemv, [Orin-INT4] §"从 FP 线性层到 INT4 DP4A 的数学推导" and §"DP4A 做了什么":
 *   acc[m][j] = sum_i q_w[j][i] * qx[m][i]   (exact int32),
 *   y[m][j]   = fmaf(s_w[j] * sx[m], (float)acc, b[j])   (b = 0 if bias NULL).
 *   Up to two tokens the sums run on DP4A; from three tokens (see
 *   W4_TUNE_TC_MIN_M) on the tensor cores, with exact fp8 products and fp32
 *   partial sums.  y is bit-identical either way.
 * q4_0_gemv / i8g32_gemv / q6g32_gemv, [310B-Gemma4] §3.1 / §3.2:
 *   acc_g = exact int32 sum over 32-block g,
 *   y[m][j] = fmaf(sx[m], sum_g d_g * acc_g, b[j])  (fp32; group order unspecified).
 *   With more than 8 tokens these (and the *_linear calls of these formats)
 *   run as two launches of the eight-token kernel, tokens 0-7 and the rest,
 *   each reading the weights once.  Every step is per token: codes, scales
 *   and integer group sums are those of one launch; y may differ from a call
 *   of other token counts only in the fp32 group-sum order.
 * w: repacked weights; s_w: float [N]; bias: float [N] or NULL; qx: int8 [M][K];
 * sx: float [M]; y: float [M][N] (row m at y + m*N).
 * ------------------------------------------------------------------------ */
w4_status w4a8_gemv(const void* w, const float* s_w, const float* bias, const int8_t* qx, const float* sx,
                    int M, int N, int K, float* y, w4_stream_t s);
/* Device scratch a GEMV or linear call of this shape needs from its caller:
 * always 0.  Where K is split over several blocks (W4_PATH_* plans with
 * k_splits > 1) the partial sums merge on chip, in the shared memory of one
 * thread-block cluster, so no call takes a workspace. */
size_t w4_workspace_bytes(int M, int N, int K);
w4_status q4_0_gemv(const void* w, const float* bias, const int8_t* qx, const float* sx,
                    int M, int N, int K, float* y, w4_stream_t s);
w4_status i8g32_gemv(const void* w, const float* bias, const int8_t* qx, const float* sx,
                     int M, int N, int K, float* y, w4_stream_t s);
w4_status q6g32_gemv(const void* w, const float* bias, const int8_t* qx, const float* sx,
                     int M, int N, int K, float* y, w4_stream_t s);

/* ------------------------------------------------------------------------
 * Per token: the whole decode linear, quantization fused into the GEMV
 * ([Orin-INT4] §"后续还能继续优化什么" item 2 names fusing the activation
 * quantization with a neighbouring operator).  Each thread block quantizes x
 * into its shared memory; block 0 also writes qx and sx (caller buffers, same
 * shapes as a8_quantize) so that the caller sees the codes used.  When M*K
 * does not fit in shared memory the call runs a8_quantize into qx/sx and then
 * the *_gemv kernel; results are identical either way.
 * flags: 0 or W4_FLAG_PDL.
 * ------------------------------------------------------------------------ */
w4_status w4a8_linear(const void* w, const float* s_w, const float* bias, const float* x, int M, int N, int K,
                      float* y, int8_t* qx, float* sx, unsigned flags, w4_stream_t s);
w4_status q4_0_linear(const void* w, const float* bias, const float* x, int M, int N, int K,
                      float* y, int8_t* qx, float* sx, unsigned flags, w4_stream_t s);
w4_status i8g32_linear(const void* w, const float* bias, const float* x, int M, int N, int K,
                       float* y, int8_t* qx, float* sx, unsigned flags, w4_stream_t s);
w4_status q6g32_linear(const void* w, const float* bias, const float* x, int M, int N, int K,
                       float* y, int8_t* qx, float* sx, unsigned flags, w4_stream_t s);

/* ------------------------------------------------------------------------
 * The decode linear with its neighbouring operators fused in.
 * [Orin-INT4] §"后续还能继续优化什么" item 1 names the kernel boundaries
 * between RMSNorm, quantization, linear, SwiGLU and the residual add;
 * [310B-Gemma4] §4.2 names add+rmsnorm and gelu+mul fusions.  With f:
 *   - f->norm_weight != NULL: x is first normalized per token,
 *       r = 1 / sqrt(S / K + eps),  x'_i = (x_i * r) * g_i,
 *     with S = sum_i x_i^2 rounded once to fp32 and every other step an IEEE
 *     fp32 operation; x' is then quantized (qx, sx hold its codes).
 *     norm_weight: float [K], 16-byte aligned; norm_eps > 0 and finite.
 *   - f->glu = W4_GLU_SILU or W4_GLU_GELU_TANH: w comes from *_repack_glu
 *     (I = N gate rows and N up rows); s_w and bias hold 2N values, the gate
 *     rows' then the up rows'; the linear's gate and up outputs g, u (each
 *     exactly as the plain linear makes them) become
 *       SiLU:      y = fl(fl(g / fl(1 + expf(-g))) * u)
 *       GELU tanh: y = (g / 2)(1 + tanhf(sqrt(2/pi)(g + 0.044715 g^3))) u,
 *     y: float [M][N].  Only W4 and Q4_0 take a GLU.
 *   - f->residual != NULL: float [M][N], added last, y = residual + out (fp32);
 *     it may be y itself (the in-place residual update) but must not
 *     otherwise overlap y.
 * f = NULL or all fields zero is exactly the *_linear call.  x must not
 * overlap y.  Many tokens (the tensor-core path) or a long x run the
 * normalize+quantize as its own kernel (rms_a8_quantize) ahead of the GEMV;
 * the results are the same.
 * ------------------------------------------------------------------------ */
#define W4_GLU_NONE 0
#define W4_GLU_SILU 1
#define W4_GLU_GELU_TANH 2
typedef struct {
    const float* norm_weight;
    float norm_eps;
    int glu;
    const float* residual;
} w4_fusion;

w4_status w4a8_linear_fused(const void* w, const float* s_w, const float* bias, const float* x, int M, int N,
                            int K, float* y, int8_t* qx, float* sx, const w4_fusion* f, unsigned flags,
                            w4_stream_t s);
w4_status q4_0_linear_fused(const void* w, const float* bias, const float* x, int M, int N, int K, float* y,
                            int8_t* qx, float* sx, const w4_fusion* f, unsigned flags, w4_stream_t s);
w4_status i8g32_linear_fused(const void* w, const float* bias, const float* x, int M, int N, int K, float* y,
                             int8_t* qx, float* sx, const w4_fusion* f, unsigned flags, w4_stream_t s);
w4_status q6g32_linear_fused(const void* w, const float* bias, const float* x, int M, int N, int K, float* y,
                             int8_t* qx, float* sx, const w4_fusion* f, unsigned flags, w4_stream_t s);

/* RMSNorm (as above) then the activation quantizer, one kernel: qx, sx of
 * the normalized tokens.  x: float [M][K]; norm_weight: float [K]. */
w4_status rms_a8_quantize(const float* x, const float* norm_weight, float eps, int M, int K, int8_t* qx, float* sx,
                          unsigned flags, w4_stream_t s);

/* The same operators as separate kernels (what a decoder runs without the
 * fusions), fp32 in and out, flags 0 or W4_FLAG_PDL:
 *   w4_rmsnorm: out[M][K] = RMSNorm(x) exactly as above (out may not overlap x);
 *   w4_glu:     out[M][I] = act(gu[m][j]) * gu[m][I + j] for a [M][2I] gate|up
 *               output (kind W4_GLU_SILU or W4_GLU_GELU_TANH), as above;
 *   w4_add:     out[i] = a[i] + b[i], i < n (out may be a or b). */
w4_status w4_rmsnorm(const float* x, const float* norm_weight, float eps, int M, int K, float* out, unsigned flags,
                     w4_stream_t s);
w4_status w4_glu(const float* gu, int kind, int M, int I, float* out, unsigned flags, w4_stream_t s);
w4_status w4_add(const float* a, const float* b, long long n, float* out, unsigned flags, w4_stream_t s);

/* ------------------------------------------------------------------------
 * Weight-only paths on float activations: the two paths [Orin-INT4]
 * §"为什么 INT4 float 解包不快" measures INT4 DP4A against (weight-only INT8,
 * and INT4 unpacked to float).  The activations are not quantized:
 *   y[m][j] = fmaf(s_w[j], sum_i q_w[j][i] * x[m][i], b[j]),
 * every weight converted to fp32 and multiply-added in fp32 (summation order
 * unspecified).
 *   w4a32_gemv: per-row INT4 weights in the w4_repack layout (the bytes the
 *     DP4A path reads), unpacked to float.
 *   w8a32_gemv: per-row INT8 weights from w8_quantize_rows (s_w = max|W|/127,
 *     q = clip(rint(W / s_w), -127, 127), int8 [N][K]) in the w8_repack
 *     layout: 32-byte units holding a row's 32 int8 weights of a chunk in
 *     order, in the (t, c, r) order of the other formats, no scale plane.
 * x: float [M][K], 16-byte aligned; 1 <= M <= 4; flags: 0 or W4_FLAG_PDL.
 * x is staged in shared memory as fp32 beside a weight ring of at least two
 * stages, so M*K is limited to about 40000 values (W4_ERR_UNSUPPORTED_SHAPE
 * beyond: K = 18944 takes at most two tokens).
 * ------------------------------------------------------------------------ */
w4_status w8_quantize_rows(const float* W, int N, int K, int8_t* q, float* s_w, w4_stream_t s);
size_t w8_repacked_bytes(int N, int K);
w4_status w8_repack(const int8_t* const* shard_q, const int* shard_rows, int n_shards, int K, void* out,
                    size_t out_bytes, w4_stream_t s);
w4_status w4a32_gemv(const void* w, const float* s_w, const float* bias, const float* x, int M, int N, int K,
                     float* y, unsigned flags, w4_stream_t s);
w4_status w8a32_gemv(const void* w, const float* s_w, const float* bias, const float* x, int M, int N, int K,
                     float* y, unsigned flags, w4_stream_t s);

/* ------------------------------------------------------------------------
 * A chain of per-row INT4 decode linears in one launch (a decode step's
 * linear set).  Linear i computes exactly what w4a8_linear computes for
 * descs[i]; linear i+1 reads its x only after every output of linear i is
 * written, so descs[i+1].x may alias (part of) descs[i].y.  While a linear's
 * activations wait on that dependency, the weights of the following linears
 * keep streaming (one persistent block per SM, cooperative launch).
 *
 * descs: HOST array of n (1..W4_MAX_CHAIN) descriptors, all with the same
 * M tokens.  Per descriptor: w (repacked W4, 16-B aligned), s_w [N], bias [N]
 * or NULL, x [M][K] (16-B aligned), y [M][N], and qx [M][K] / sx [M] to
 * receive the activation codes, or NULL.
 * workspace: device memory of w4_chain_workspace_bytes() bytes, 16-B aligned,
 * zero-filled before its first use; each call leaves it zero again, ready for
 * the next.  Calls that share a workspace must not overlap on the GPU.  After
 * a call that reported W4_ERR_DEVICE_TIMEOUT, zero the workspace again.
 * Host threads may call the chain entry points at the same time, each with
 * its own workspace and stream: the launch parameters are staged per thread.
 * The chain runs its linears on DP4A whatever M is.  Per-row INT4 calls of
 * three or more tokens are faster through the per-linear entry points
 * (w4a8_linear with W4_FLAG_PDL, on the tensor cores), which need the qx / sx
 * buffers the chain may leave out.  On the 7B step the per-linear launches
 * chained with W4_FLAG_PDL are also faster at one token (0.872 against
 * 1.03-1.07 ms); the chain is the single-launch alternative. 
 * ------------------------------------------------------------------------ */
#define W4_MAX_CHAIN 128
typedef struct {
    const void* w;
    const float* s_w;
    const float* bias;
    const float* x;
    float* y;
    int8_t* qx;
    float* sx;
    int N;
    int K;
} w4_linear_desc;

size_t w4_chain_workspace_bytes(void);
w4_status w4a8_linear_chain(const w4_linear_desc* descs, int n, int M, void* workspace, size_t ws_bytes,
                            w4_stream_t s);

/* ------------------------------------------------------------------------
 * w4a8_linear_chain without caller-provided device memory.  The source pages
 * have no counterpart of this entry point: it exists for callers that cannot
 * allocate device memory at the point of the call -- for example code running
 * under an engine whose memory planner owns every device allocation, or code
 * that must not call cudaMalloc while a stream is being captured into a CUDA
 * graph -- and therefore cannot provide the chain's workspace.
 *
 * The grid-barrier state lives in a fixed array of
 * w4_chain_noalloc_scratch_bytes() (256) bytes inside the library; every GPU
 * that loads the library holds it until the process exits.  Each call clears
 * it (cudaMemsetAsync on `s`) and then runs exactly w4a8_linear_chain.  The
 * call allocates nothing and frees nothing.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress); make that first call before any stream capture.
 *   - All calls share the one array: calls that overlap on the GPU (other
 *     streams, other threads) race on it and must be serialised by the caller.
 *   - A workspace need above the array's size is rejected with
 *     W4_ERR_UNSUPPORTED_SHAPE; all other arguments are checked as in
 *     w4a8_linear_chain, before anything is enqueued: a call that fails a
 *     check does not touch the array (no clear), so it cannot disturb a
 *     chain already in flight.
 * ------------------------------------------------------------------------ */
size_t w4_chain_noalloc_scratch_bytes(void);
w4_status w4a8_linear_chain_noalloc(const w4_linear_desc* descs, int n, int M, w4_stream_t s);

/* ------------------------------------------------------------------------
 * Device error word.  Kernels that give up a bounded wait (about 0.25 s on an
 * mbarrier) record a nonzero code here and return early; their outputs are
 * then undefined.  w4_device_error synchronises the current device, reads the
 * word into *code (host pointer) and returns W4_ERR_DEVICE_TIMEOUT if it is
 * nonzero, else W4_OK.  w4_clear_device_error zeroes it (synchronous).
 * ------------------------------------------------------------------------ */
w4_status w4_device_error(unsigned* code);
w4_status w4_last_device_error(unsigned* code); /* the same call under a second name */
w4_status w4_clear_device_error(void);

/* Self-test of the timeout path: launches a kernel whose bounded wait nothing
 * completes (an mbarrier on which no thread arrives), so it gives up after
 * timeout_us microseconds (1..1000000) and sets the device error word to the
 * wait-timeout code (0x57414954, "WAIT"), as a GEMV's waits do.  cluster = 1
 * waits as the K-split leader does (two blocks in a cluster, cluster-scope
 * acquire, the other block leaving); 0 waits as every other ring does.  The
 * kernel always finishes and faults nothing; clear the word afterwards.
 * W4_ERR_INVALID_ARG for other arguments. */
w4_status w4_selftest_wait_timeout(int cluster, unsigned timeout_us, w4_stream_t s);

/* ------------------------------------------------------------------------
 * Pure-read HBM bandwidth probe: the roofline denominator for a kernel that
 * only reads.  [310B-Gemma4] §4.1 measures the device's pure read bandwidth
 * (distinct from a read+write copy) as the bound of a weight-streaming decode;
 * this is the same measurement on this device.  The kernel streams `bytes`
 * bytes of `buf` (16-byte aligned; bytes a multiple of 16) once through the
 * same per-warp bulk-copy rings as the GEMVs (one block per SM, evict-first)
 * and writes the XOR of all its 32-bit words to *sink (device, 4 bytes), so
 * that no read is dead.  bytes = 0 writes 0.  Time it with events on `s`.
 * ------------------------------------------------------------------------ */
w4_status w4_hbm_read(const void* buf, size_t bytes, unsigned* sink, w4_stream_t s);

#ifdef __cplusplus
}
#endif

#endif /* W4A8_H */
