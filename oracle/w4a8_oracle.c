/*
 * CPU oracle for bit-quantized decode GEMV.  TEST INFRASTRUCTURE ONLY.
 *
 * Plain, slow, single-threaded C that states what the decode path computes,
 * one definition per function, written from the two source pages:
 *
 *   [Orin-INT4]   "Jetson Orin AGX INT4 推理优化实践：super 分支从 9 tok/s 到 24 tok/s"
 *                 (jsqmd.com/news/867209)
 *   [310B-Gemma4] "在香橙派上跑 Gemma4：vLLM 适配昇腾 310B 的内核开发实录"
 *                 (hiascend.com forum thread 02200219947507257174)
 *
 * Only the test suite, the smoke check and the benchmark's CPU-baseline leg
 * may call this library.  It shares no code, header or table with the GPU
 * library and includes nothing from it.
 *
 * Precision: quantization decisions (scales, codes) are taken in IEEE fp32,
 * the precision the GPU kernels take them in, so codes must match bit for
 * bit.  Integer dot products are exact (int64, checked to fit int32).
 * Dequantized outputs are formed in fp64.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fno-fast-math (no FMA
 * contraction, IEEE division).
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>

/* status codes */
#define ORC_OK 0
#define ORC_ERR_ARG 1
#define ORC_ERR_INT32_OVERFLOW 2

/* ------------------------------------------------------------------------ */
/* fp16 <-> fp32, written from the IEEE 754 binary16 definition             */
/* ------------------------------------------------------------------------ */

static uint32_t f32_bits(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }
static float bits_f32(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }

/* binary16 -> binary32 (exact). */
float orc_half_to_float(uint16_t h)
{
    uint32_t sign = (uint32_t)(h >> 15) & 1u;
    uint32_t exp = (uint32_t)(h >> 10) & 0x1fu;
    uint32_t man = (uint32_t)h & 0x3ffu;
    double v;
    if (exp == 0x1f) {
        if (man != 0) return bits_f32(0x7fc00000u | (sign << 31));
        return bits_f32((sign << 31) | 0x7f800000u);
    }
    if (exp == 0) v = ldexp((double)man, -24);                 /* subnormal: man * 2^-24 */
    else v = ldexp((double)(man | 0x400u), (int)exp - 25);      /* (1024+man) * 2^(e-25) */
    return (float)(sign ? -v : v);
}

/* binary32 -> binary16, round to nearest, ties to even; overflow -> inf. */
uint16_t orc_float_to_half(float f)
{
    uint32_t u = f32_bits(f);
    uint16_t sign = (uint16_t)((u >> 16) & 0x8000u);
    if (isnan(f)) return (uint16_t)(sign | 0x7e00u);
    double a = fabs((double)f);
    if (isinf(f)) return (uint16_t)(sign | 0x7c00u);
    if (a == 0.0) return sign;
    /* The binary16 value grid: below 2^-14 the spacing is 2^-24 (subnormals);
       in [2^e, 2^(e+1)) with e >= -14 the spacing is 2^(e-10).  Round a to the
       grid point nearest to it, ties to the even multiple. */
    int e;
    frexp(a, &e);           /* a = m * 2^e with m in [0.5, 1): a in [2^(e-1), 2^e) */
    int lead = e - 1;       /* a in [2^lead, 2^(lead+1)) */
    int qexp = lead < -14 ? -24 : lead - 10;
    double scaled = ldexp(a, -qexp);        /* exact: power-of-two scaling */
    double r = nearbyint(scaled);           /* default rounding mode: ties to even */
    double v = ldexp(r, qexp);
    if (v >= 65520.0) return (uint16_t)(sign | 0x7c00u);   /* rounds past max finite */
    if (v > 65504.0) v = 65504.0;
    /* encode v exactly */
    if (v < ldexp(1.0, -14)) {
        uint32_t m = (uint32_t)ldexp(v, 24);
        return (uint16_t)(sign | m);
    }
    int ve;
    frexp(v, &ve);
    int vl = ve - 1;                                   /* v in [2^vl, 2^(vl+1)) */
    uint32_t m = (uint32_t)ldexp(v, 10 - vl) - 1024u; /* 10-bit fraction */
    return (uint16_t)(sign | (uint16_t)((uint32_t)(vl + 15) << 10) | (uint16_t)m);
}

/* ------------------------------------------------------------------------ */
/* Dynamic per-token INT8 activation quantization                            */
/* [Orin-INT4] §"从 FP 线性层到 INT4 DP4A 的数学推导":                         */
/*   s^x = max_i |x_i| / 127,  q^x_i = clip(round(x_i / s^x), -127, 127).    */
/* round = round half to even (rintf); an all-zero token gives s^x = 0 and  */
/* q^x = 0.                                                                  */
/* ------------------------------------------------------------------------ */
int orc_quantize_act_int8(const float* x, int M, int K, int8_t* qx, float* sx)
{
    if (M < 0 || K < 0 || (M * (size_t)K && (!x || !qx)) || (M && !sx)) return ORC_ERR_ARG;
    for (int m = 0; m < M; ++m) {
        const float* xr = x + (size_t)m * K;
        float amax = 0.0f;
        for (int i = 0; i < K; ++i) {
            float a = fabsf(xr[i]);
            if (a > amax) amax = a;
        }
        float s = amax / 127.0f;
        sx[m] = s;
        for (int i = 0; i < K; ++i) {
            int q = 0;
            if (s != 0.0f) {
                float t = xr[i] / s;
                q = (int)rintf(t);
                if (q > 127) q = 127;
                if (q < -127) q = -127;
            }
            qx[(size_t)m * K + i] = (int8_t)q;
        }
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* Per-row symmetric INT4 weight quantization                                */
/* [Orin-INT4] §"从 FP 线性层到 INT4 DP4A 的数学推导":                         */
/*   W_{j,i} ~ s^W_j q^W_{j,i},  q^W = clip(round(W / s^W_j), -8, 7).        */
/* The page leaves s^W_j open; the reading taken here maps the row's        */
/* largest magnitude to the largest positive code, as s^x does for x:       */
/*   s^W_j = max_i |W_{j,i}| / 7.   An all-zero row gives s^W = 0, q = 0.    */
/* q is written unpacked, one int8 per weight, [N][K].                      */
/* ------------------------------------------------------------------------ */
int orc_quantize_rows_int4(const float* W, int N, int K, int8_t* q, float* sw)
{
    if (N < 0 || K < 0 || !W || !q || !sw) return ORC_ERR_ARG;
    for (int j = 0; j < N; ++j) {
        const float* wr = W + (size_t)j * K;
        float amax = 0.0f;
        for (int i = 0; i < K; ++i) {
            float a = fabsf(wr[i]);
            if (a > amax) amax = a;
        }
        float s = amax / 7.0f;
        sw[j] = s;
        for (int i = 0; i < K; ++i) {
            int v = 0;
            if (s != 0.0f) {
                v = (int)rintf(wr[i] / s);
                if (v > 7) v = 7;
                if (v < -8) v = -8;
            }
            q[(size_t)j * K + i] = (int8_t)v;
        }
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* Nibble packing, [Orin-INT4] §"DP4A 做了什么":                               */
/*   uint32 packed = [w7 w6 w5 w4 w3 w2 w1 w0], w0 in the low nibble, so     */
/*   weight k of a word sits in bits 4k..4k+3, as a 4-bit two's-complement  */
/*   value (the page sign-extends it on unpack).                             */
/* q is [N][K] int8 in [-8, 7]; packed is [N][K/8] uint32.  K % 8 == 0.     */
/* ------------------------------------------------------------------------ */
int orc_pack_int4(const int8_t* q, int N, int K, uint32_t* packed)
{
    if (N < 0 || K < 0 || K % 8 != 0 || !q || !packed) return ORC_ERR_ARG;
    for (int j = 0; j < N; ++j)
        for (int w = 0; w < K / 8; ++w) {
            uint32_t word = 0;
            for (int k = 0; k < 8; ++k) {
                int v = q[(size_t)j * K + 8 * w + k];
                if (v < -8 || v > 7) return ORC_ERR_ARG;
                word |= ((uint32_t)v & 0xfu) << (4 * k);
            }
            packed[(size_t)j * (K / 8) + w] = word;
        }
    return ORC_OK;
}

int orc_unpack_int4(const uint32_t* packed, int N, int K, int8_t* q)
{
    if (N < 0 || K < 0 || K % 8 != 0 || !q || !packed) return ORC_ERR_ARG;
    for (int j = 0; j < N; ++j)
        for (int w = 0; w < K / 8; ++w) {
            uint32_t word = packed[(size_t)j * (K / 8) + w];
            for (int k = 0; k < 8; ++k) {
                int nib = (int)((word >> (4 * k)) & 0xfu);
                q[(size_t)j * K + 8 * w + k] = (int8_t)(nib >= 8 ? nib - 16 : nib); /* sign extend */
            }
        }
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* DP4A, [Orin-INT4] §"DP4A 做了什么":                                          */
/*   acc <- acc + a0 b0 + a1 b1 + a2 b2 + a3 b3, a_k and b_k signed int8,   */
/*   byte k of each 32-bit operand.                                          */
/* ------------------------------------------------------------------------ */
int32_t orc_dp4a(uint32_t a, uint32_t b, int32_t c)
{
    int64_t s = c;
    for (int k = 0; k < 4; ++k) {
        int8_t ak = (int8_t)(uint8_t)((a >> (8 * k)) & 0xffu);
        int8_t bk = (int8_t)(uint8_t)((b >> (8 * k)) & 0xffu);
        s += (int64_t)ak * (int64_t)bk;
    }
    return (int32_t)(uint32_t)(uint64_t)s;   /* wraps like the hardware's 32-bit adder */
}

/* ------------------------------------------------------------------------ */
/* Integer dot products, [Orin-INT4] §"从 FP 线性层到 INT4 DP4A 的数学推导":   */
/*   acc_j = sum_i q^W_{j,i} q^x_i, summed exactly (int64) and required to  */
/*   fit int32, the accumulator width the page argues is safe in           */
/*   §"INT32 accumulator 是否安全".                                           */
/* packed: [N][K/8] canonical words; qx: [M][K]; acc: [M][N].               */
/* ------------------------------------------------------------------------ */
int orc_gemv_w4a8_acc(const uint32_t* packed, const int8_t* qx, int M, int N, int K, int32_t* acc)
{
    if (M < 0 || N < 0 || K < 0 || K % 8 != 0 || (M && N && (!packed || !qx || !acc))) return ORC_ERR_ARG;
    int overflow = 0;
    for (int m = 0; m < M; ++m)
        for (int j = 0; j < N; ++j) {
            int64_t s = 0;
            for (int i = 0; i < K; ++i) {
                uint32_t word = packed[(size_t)j * (K / 8) + i / 8];
                int nib = (int)((word >> (4 * (i % 8))) & 0xfu);
                int w = nib >= 8 ? nib - 16 : nib;
                s += (int64_t)w * (int64_t)qx[(size_t)m * K + i];
            }
            if (s > INT32_MAX || s < INT32_MIN) overflow = 1;
            acc[(size_t)m * N + j] = (int32_t)s;
        }
    return overflow ? ORC_ERR_INT32_OVERFLOW : ORC_OK;
}

/* Dequantization, [Orin-INT4] §"从 FP 线性层到 INT4 DP4A 的数学推导":
 *   y_j = s^W_j s^x acc_j + b_j, formed in fp64; bias may be NULL (b = 0). */
int orc_epilogue_w4a8(const int32_t* acc, const float* sw, const float* sx, const float* bias,
                      int M, int N, double* y)
{
    if (M < 0 || N < 0 || (M && N && (!acc || !sw || !sx || !y))) return ORC_ERR_ARG;
    for (int m = 0; m < M; ++m)
        for (int j = 0; j < N; ++j) {
            double b = bias ? (double)bias[j] : 0.0;
            y[(size_t)m * N + j] = (double)sw[j] * (double)sx[m] * (double)acc[(size_t)m * N + j] + b;
        }
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* Q4_0 blocks, [310B-Gemma4] §3.1 "Q4_0 融合反量化+矩阵乘":                    */
/*   32 weights per block = 16 bytes of 4-bit values + one fp16 scale,      */
/*   18 bytes in all.  Block byte layout (GGUF convention): bytes 0..1 the  */
/*   fp16 scale d (little endian), bytes 2..17 the nibbles; byte 2+i holds  */
/*   element i in its low nibble and element i+16 in its high nibble.       */
/*   The value of a nibble n is n - 8; the weight is d * (n - 8).           */
/* Quantization: d = fp16(max|w| / 8); n = clip(round(w / d), -8, 7) + 8,   */
/* with w / d taken against the stored (fp16) d.  d == 0 gives n = 8.       */
/* blocks: [N][K/32][18] bytes.  K % 32 == 0.                               */
/* ------------------------------------------------------------------------ */
#define Q4_0_BLOCK_BYTES 18

int orc_q4_0_block_bytes(void) { return Q4_0_BLOCK_BYTES; }

int orc_quantize_q4_0(const float* W, int N, int K, uint8_t* blocks)
{
    if (N < 0 || K < 0 || K % 32 != 0 || !W || !blocks) return ORC_ERR_ARG;
    for (int j = 0; j < N; ++j)
        for (int g = 0; g < K / 32; ++g) {
            const float* wg = W + (size_t)j * K + 32 * g;
            uint8_t* blk = blocks + ((size_t)j * (K / 32) + g) * Q4_0_BLOCK_BYTES;
            float amax = 0.0f;
            for (int i = 0; i < 32; ++i) {
                float a = fabsf(wg[i]);
                if (a > amax) amax = a;
            }
            uint16_t dh = orc_float_to_half(amax / 8.0f);
            float d = orc_half_to_float(dh);
            blk[0] = (uint8_t)(dh & 0xff);
            blk[1] = (uint8_t)(dh >> 8);
            int n[32];
            for (int i = 0; i < 32; ++i) {
                int v = 0;
                if (d != 0.0f) {
                    v = (int)rintf(wg[i] / d);
                    if (v > 7) v = 7;
                    if (v < -8) v = -8;
                }
                n[i] = v + 8;
            }
            for (int i = 0; i < 16; ++i) blk[2 + i] = (uint8_t)(n[i] | (n[i + 16] << 4));
        }
    return ORC_OK;
}

/* Value (n - 8) of element i of a block, and the block's scale. */
static int q4_0_value(const uint8_t* blk, int i)
{
    uint8_t byte = blk[2 + (i % 16)];
    int n = i < 16 ? (byte & 0xf) : (byte >> 4);
    return n - 8;
}

int orc_dequantize_q4_0(const uint8_t* blocks, int N, int K, double* W)
{
    if (N < 0 || K < 0 || K % 32 != 0 || !blocks || !W) return ORC_ERR_ARG;
    for (int j = 0; j < N; ++j)
        for (int g = 0; g < K / 32; ++g) {
            const uint8_t* blk = blocks + ((size_t)j * (K / 32) + g) * Q4_0_BLOCK_BYTES;
            double d = (double)orc_half_to_float((uint16_t)(blk[0] | (blk[1] << 8)));
            for (int i = 0; i < 32; ++i) W[(size_t)j * K + 32 * g + i] = d * (double)q4_0_value(blk, i);
        }
    return ORC_OK;
}

/* Q4_0 GEMV against per-token INT8 activations.  Per block g of row j:
 *   acc_g = sum_{i in g} (n_i - 8) q^x_i          (exact integer),
 *   y_j   = s^x * sum_g d_g * acc_g + b_j          (fp64).
 * acc_out (nullable): [M][N][K/32] group accumulators.  y: [M][N]. */
int orc_gemv_q4_0(const uint8_t* blocks, const int8_t* qx, const float* sx, const float* bias,
                  int M, int N, int K, int32_t* acc_out, double* y)
{
    if (M < 0 || N < 0 || K < 0 || K % 32 != 0) return ORC_ERR_ARG;
    if (M && N && (!blocks || !qx || !sx || !y)) return ORC_ERR_ARG;
    const int G = K / 32;
    for (int m = 0; m < M; ++m)
        for (int j = 0; j < N; ++j) {
            double sum = 0.0;
            for (int g = 0; g < G; ++g) {
                const uint8_t* blk = blocks + ((size_t)j * G + g) * Q4_0_BLOCK_BYTES;
                int32_t a = 0;
                for (int i = 0; i < 32; ++i) a += q4_0_value(blk, i) * (int32_t)qx[(size_t)m * K + 32 * g + i];
                if (acc_out) acc_out[((size_t)m * N + j) * G + g] = a;
                double d = (double)orc_half_to_float((uint16_t)(blk[0] | (blk[1] << 8)));
                sum += d * (double)a;
            }
            double b = bias ? (double)bias[j] : 0.0;
            y[(size_t)m * N + j] = (double)sx[m] * sum + b;
        }
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* int8 weights with one fp16 scale per group of 32 ("i8g32")              */
/* [310B-Gemma4] §3.2 "Q6_K int8 lm_head": the 6-bit lm_head values are    */
/* widened losslessly to int8 and carry a pre-multiplied fp16 scale per     */
/* group.  Here a group is 32 weights and the values lie in [-32, 31]:      */
/*   d = fp16(max|w| / 32),  q = clip(round(w / d), -32, 31).               */
/* q: [N][K] int8; d: [N][K/32] fp16 bits.                                   */
/* ------------------------------------------------------------------------ */
int orc_quantize_i8g32(const float* W, int N, int K, int8_t* q, uint16_t* d)
{
    if (N < 0 || K < 0 || K % 32 != 0 || !W || !q || !d) return ORC_ERR_ARG;
    for (int j = 0; j < N; ++j)
        for (int g = 0; g < K / 32; ++g) {
            const float* wg = W + (size_t)j * K + 32 * g;
            float amax = 0.0f;
            for (int i = 0; i < 32; ++i) {
                float a = fabsf(wg[i]);
                if (a > amax) amax = a;
            }
            uint16_t dh = orc_float_to_half(amax / 32.0f);
            float df = orc_half_to_float(dh);
            d[(size_t)j * (K / 32) + g] = dh;
            for (int i = 0; i < 32; ++i) {
                int v = 0;
                if (df != 0.0f) {
                    v = (int)rintf(wg[i] / df);
                    if (v > 31) v = 31;
                    if (v < -32) v = -32;
                }
                q[(size_t)j * K + 32 * g + i] = (int8_t)v;
            }
        }
    return ORC_OK;
}

/* y_j = s^x * sum_g d_g * acc_g + b_j, acc_g = sum_{i in g} q_{j,i} q^x_i. */
int orc_gemv_i8g32(const int8_t* q, const uint16_t* d, const int8_t* qx, const float* sx,
                   const float* bias, int M, int N, int K, int32_t* acc_out, double* y)
{
    if (M < 0 || N < 0 || K < 0 || K % 32 != 0) return ORC_ERR_ARG;
    if (M && N && (!q || !d || !qx || !sx || !y)) return ORC_ERR_ARG;
    const int G = K / 32;
    for (int m = 0; m < M; ++m)
        for (int j = 0; j < N; ++j) {
            double sum = 0.0;
            for (int g = 0; g < G; ++g) {
                int32_t a = 0;
                for (int i = 0; i < 32; ++i)
                    a += (int32_t)q[(size_t)j * K + 32 * g + i] * (int32_t)qx[(size_t)m * K + 32 * g + i];
                if (acc_out) acc_out[((size_t)m * N + j) * G + g] = a;
                sum += (double)orc_half_to_float(d[(size_t)j * G + g]) * (double)a;
            }
            double b = bias ? (double)bias[j] : 0.0;
            y[(size_t)m * N + j] = (double)sx[m] * sum + b;
        }
    return ORC_OK;
}

/* Bytes one output row of K weights occupies in each format
 * ([Orin-INT4] table in §"为什么 INT4 float 解包不快": FP16 2 B, INT8 1 B,
 * INT4 0.5 B per weight), with bits in {16, 8, 4}. */
long long orc_row_weight_bytes(int K, int bits)
{
    if (K < 0 || (bits != 16 && bits != 8 && bits != 4)) return -1;
    return (long long)K * bits / 8;
}

/* ------------------------------------------------------------------------ */
/* Operators around the linear.  [Orin-INT4] §"后续还能继续优化什么" item 1    */
/* lists RMSNorm, the activation quantization, the linear, SwiGLU and the    */
/* residual add as the operators with kernel boundaries between them;        */
/* [310B-Gemma4] §4.2 names add+rmsnorm and gelu+mul as the fusions to make. */
/* Neither page writes the operators out; the readings taken here are the    */
/* usual definitions in the models those pages run (Qwen2-architecture      */
/* DeepSeek-R1-Distill-Qwen-7B: RMSNorm and a SiLU-gated MLP; Gemma: a      */
/* GELU(tanh)-gated MLP).                                                    */
/* ------------------------------------------------------------------------ */

/* RMSNorm of each token, every step in IEEE fp32 (the precision in which   */
/* the codes that follow are decided):                                       */
/*   S   = sum_i x_i^2, rounded once to fp32 (accumulated here in fp64, each */
/*         square exact in fp64),                                            */
/*   ms  = S / K,  r = 1 / sqrt(ms + eps),                                   */
/*   out_i = (x_i * r) * g_i.                                                */
/* x, out: [M][K]; g: [K]; eps >= 0 (an all-zero token with eps = 0 gives   */
/* NaN, as the formula does).                                                */
int orc_rmsnorm_f32(const float* x, const float* g, float eps, int M, int K, float* out)
{
    if (M < 0 || K <= 0 || !(eps >= 0.0f) || (M && (!x || !g || !out))) return ORC_ERR_ARG;
    for (int m = 0; m < M; ++m) {
        const float* xr = x + (size_t)m * K;
        double S = 0.0;
        for (int i = 0; i < K; ++i) S += (double)xr[i] * (double)xr[i];
        const float S32 = (float)S;
        const float ms = S32 / (float)K;
        const float r = 1.0f / sqrtf(ms + eps);
        for (int i = 0; i < K; ++i) out[(size_t)m * K + i] = (xr[i] * r) * g[i];
    }
    return ORC_OK;
}

/* Gated activations of the MLP, in fp64: out_i = act(gate_i) * up_i with   */
/*   kind 1 (SwiGLU):    act(v) = v / (1 + exp(-v))          (SiLU),         */
/*   kind 2 (GELU tanh): act(v) = v/2 (1 + tanh(sqrt(2/pi) (v + 0.044715 v^3))). */
int orc_glu(const double* gate, const double* up, int n, int kind, double* out)
{
    if (n < 0 || (kind != 1 && kind != 2) || (n && (!gate || !up || !out))) return ORC_ERR_ARG;
    const double k0 = sqrt(2.0 / 3.14159265358979323846);
    for (int i = 0; i < n; ++i) {
        const double v = gate[i];
        double a;
        if (kind == 1) a = v / (1.0 + exp(-v));
        else a = 0.5 * v * (1.0 + tanh(k0 * (v + 0.044715 * v * v * v)));
        out[i] = a * up[i];
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* The two paths [Orin-INT4] §"为什么 INT4 float 解包不快" measures against    */
/* INT4 DP4A: weight-only INT8 (int8 weights, float activations, float       */
/* multiply-add) and INT4 with float unpacking (each 4-bit weight unpacked,  */
/* sign-extended, converted to float and multiply-added with the float      */
/* activation).  Neither quantizes the activations.                         */
/* ------------------------------------------------------------------------ */

/* Per-row symmetric INT8 weights for the weight-only path.  The page gives  */
/* no formula; the reading mirrors the per-row INT4 one with 127 in place of */
/* 7: s^W_j = max_i |W_{j,i}| / 127, q = clip(round(W / s^W_j), -127, 127), */
/* round half to even.  An all-zero row gives s = 0, q = 0.                  */
int orc_quantize_rows_int8(const float* W, int N, int K, int8_t* q, float* sw)
{
    if (N < 0 || K < 0 || !W || !q || !sw) return ORC_ERR_ARG;
    for (int j = 0; j < N; ++j) {
        const float* wr = W + (size_t)j * K;
        float amax = 0.0f;
        for (int i = 0; i < K; ++i) {
            float a = fabsf(wr[i]);
            if (a > amax) amax = a;
        }
        float s = amax / 127.0f;
        sw[j] = s;
        for (int i = 0; i < K; ++i) {
            int v = 0;
            if (s != 0.0f) {
                v = (int)rintf(wr[i] / s);
                if (v > 127) v = 127;
                if (v < -127) v = -127;
            }
            q[(size_t)j * K + i] = (int8_t)v;
        }
    }
    return ORC_OK;
}

/* Weight-only linear on float activations (both paths above):              */
/*   y[m][j] = s^W_j sum_i q_{j,i} x[m][i] + b_j, formed in fp64.           */
/* q: int8 [N][K] (INT4 codes in [-8, 7] or INT8 codes); x: fp32 [M][K].    */
int orc_gemv_weight_only(const int8_t* q, const float* sw, const float* x, const float* bias, int M, int N, int K,
                         double* y)
{
    if (M < 0 || N < 0 || K < 0 || (M && N && (!q || !sw || !x || !y))) return ORC_ERR_ARG;
    for (int m = 0; m < M; ++m)
        for (int j = 0; j < N; ++j) {
            double s = 0.0;
            for (int i = 0; i < K; ++i) s += (double)q[(size_t)j * K + i] * (double)x[(size_t)m * K + i];
            y[(size_t)m * N + j] = (double)sw[j] * s + (bias ? (double)bias[j] : 0.0);
        }
    return ORC_OK;
}
