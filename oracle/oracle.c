/*
 * oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow CPU reference ("the oracle") for everything the GPU library
 * computes: affine group quantize/pack, unpack and dequantize, the affine
 * quantized matrix-vector product (qmv) and its small-M transposed sibling
 * (qmm_t), and the Q8_0 / Q4_K block-quantized matrix-vector products.
 *
 * Only the test suite, the smoke check and the CPU-baseline leg of the
 * benchmark load this file's library. The GPU path never links, includes or
 * calls it, and this file includes nothing from the GPU path.
 *
 * Every floating-point result is computed in IEEE binary64 by the plain
 * definition of the operation: dequantize each weight exactly, then take a
 * sequential dot product. The only binary32 arithmetic is in quantize, where
 * the chosen codes depend on it (scale = (max-min)/(2^bits-1), the code
 * rint((w-bias)/scale)), and there it is done in binary32 on purpose so that
 * the codes are the ones a binary32 implementation must produce. (The
 * orc_*_f32loop functions at the end are plain binary32 loops kept only as
 * a CPU timing baseline; nothing compares against them.)
 *
 * Sources (page title, then the passage):
 *  - metaltile-std quantized.rs, kernel mt_qmv: the qmv sum
 *    out[n] = sum_g (scale_g * sum_{i in g} q_i x_i + bias_g * sum_{i in g} x_i),
 *    its argument layout (w u32 [N, K*bits/32], scales/biases [N, K/gs],
 *    x [K]) and the low-nibble-first packing of 4-bit codes.
 *  - MLX PR "[Metal] Add staged affine_qmm_t_nax kernels with split-k",
 *    Correctness section: fp32 accumulation, one rounding after the sum;
 *    its reproduction script: quantize(w, group_size=64, bits=4) and
 *    quantized_matmul(x, wq, scales, biases, transpose=True).
 *  - hanzo-kernel quant.rs, dp4a matvecs: int8 activations, exact integer
 *    inner sums (orc_quantize_x_q8, orc_q8_0_gemv_i8).
 *  - hanzo-kernel quant.rs: Q8_0 (one f16 scale + 32 int8 per block; packed
 *    9-word block, scale in the low half of word 0), Q4_K (144-byte super-block
 *    d, dmin, scales[12], qs[128]; get_scale_min_k4; w = d*sc*q - dmin*m).
 *  - hanzo-kernel quant.rs names Q6_K and the 34-byte Q8_0 block without
 *    writing them out; their layouts are read from the GGUF format's
 *    published block definitions (section "GGUF block layouts" below).
 *
 * Where the pages leave a step open, the reading taken is stated at the
 * function that takes it.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ORC_F32 = 0, ORC_F16 = 1, ORC_BF16 = 2 };

enum { ORC_OK = 0, ORC_EINVAL = 1 };

/* ------------------------------------------------------------------------ */
/* Storage formats                                                           */
/* ------------------------------------------------------------------------ */

/* IEEE binary16 bit pattern -> value. Full decode: zero, subnormal, normal,
 * infinity and NaN. (hanzo-kernel quant.rs, Q8_0 packed section, decodes the
 * normal and zero cases only; the full definition is used here.) */
double orc_f16_to_f64(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int m = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24);              /* m * 2^-24 (zero, subnormal) */
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + m), e - 25);  /* (1 + m/1024) * 2^(e-15) */
    return sign ? -v : v;
}

/* bfloat16 bit pattern -> value: the upper half of an IEEE binary32. */
double orc_bf16_to_f64(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Round a finite or non-finite binary32 value to a binary format with
 * `mant` explicit mantissa bits and exponent bias `bias` (all exponent
 * codes 1..2*bias normal, code 2*bias+1 reserved for inf/NaN), round to
 * nearest, ties to even. Returns the bit pattern (1 + ebits + mant bits). */
static uint32_t round_to_format(float f, int mant, int bias)
{
    const int ebits_max = 2 * bias + 1;          /* all-ones exponent code */
    uint32_t sign_bit = signbit(f) ? 0x8000u : 0u; /* both formats are 16 bits wide */
    double a = fabs((double)f);
    if (isnan(f))
        return sign_bit | ((uint32_t)ebits_max << mant) | (1u << (mant - 1));
    if (isinf(f))
        return sign_bit | ((uint32_t)ebits_max << mant);
    const int emin = 1 - bias;                   /* smallest normal exponent */
    int ex;
    frexp(a, &ex);                               /* a = fr * 2^ex, fr in [0.5,1) */
    int E = ex - 1;                              /* a in [2^E, 2^(E+1)) */
    if (a == 0.0 || E < emin) {
        /* subnormal range: quantum 2^(emin - mant); a / quantum is exact */
        double n = rint(ldexp(a, mant - emin));
        return sign_bit | (uint32_t)n;           /* n == 2^mant -> smallest normal */
    }
    double n = rint(ldexp(a, mant - E));         /* in [2^mant, 2^(mant+1)] */
    if (n == ldexp(1.0, mant + 1)) {
        n = ldexp(1.0, mant);
        E += 1;
    }
    if (E + bias >= ebits_max)                   /* overflow -> infinity */
        return sign_bit | ((uint32_t)ebits_max << mant);
    return sign_bit | ((uint32_t)(E + bias) << mant) | ((uint32_t)n - (1u << mant));
}

uint16_t orc_f32_to_f16_rne(float f) { return (uint16_t)round_to_format(f, 10, 15); }
uint16_t orc_f32_to_bf16_rne(float f) { return (uint16_t)round_to_format(f, 7, 127); }

/* value of element i of an array stored in `dtype` */
static double load_t(const void* p, int64_t i, int dtype)
{
    switch (dtype) {
    case ORC_F32: return (double)((const float*)p)[i];
    case ORC_F16: return orc_f16_to_f64(((const uint16_t*)p)[i]);
    default:      return orc_bf16_to_f64(((const uint16_t*)p)[i]);
    }
}

/* round a binary32 value to `dtype`, store it, return the stored value */
static float store_t(void* p, int64_t i, float v, int dtype)
{
    uint16_t h;
    switch (dtype) {
    case ORC_F32:
        ((float*)p)[i] = v;
        return v;
    case ORC_F16:
        h = orc_f32_to_f16_rne(v);
        ((uint16_t*)p)[i] = h;
        return (float)orc_f16_to_f64(h);
    default:
        h = orc_f32_to_bf16_rne(v);
        ((uint16_t*)p)[i] = h;
        return (float)orc_bf16_to_f64(h);
    }
}

static int valid_affine(int bits, int gs, int64_t N, int64_t K)
{
    if (!(bits == 2 || bits == 3 || bits == 4 || bits == 6 || bits == 8)) return 0;
    if (!(gs == 32 || gs == 64 || gs == 128)) return 0;
    if (N < 0 || K <= 0 || K % gs != 0 || (K * bits) % 32 != 0) return 0;
    return 1;
}

/* ------------------------------------------------------------------------ */
/* Packed code stream                                                        */
/* ------------------------------------------------------------------------ */

/* Each row is one little-endian bit stream: bit j of code i sits at stream
 * position p = i*bits + j, i.e. word p/32, bit p%32. For bits=4 this is the
 * low-nibble-first order of metaltile-std quantized.rs (mt_qmv: nibble j of a
 * word is element 8*word + j); for 3 and 6 bits (no layout on the pages) a
 * code may straddle two words. Rows start on a word boundary. */
static unsigned get_code(const uint32_t* row, int64_t i, int bits)
{
    unsigned q = 0;
    for (int j = 0; j < bits; ++j) {
        int64_t p = i * bits + j;
        q |= ((row[p / 32] >> (p % 32)) & 1u) << j;
    }
    return q;
}

static void put_code(uint32_t* row, int64_t i, int bits, unsigned q)
{
    for (int j = 0; j < bits; ++j) {
        int64_t p = i * bits + j;
        if ((q >> j) & 1u) row[p / 32] |= 1u << (p % 32);
    }
}

/* q[n*K + k] = code of element (n, k) */
int orc_unpack(const uint32_t* packed, int bits, int64_t N, int64_t K, uint8_t* q)
{
    if (!(bits == 2 || bits == 3 || bits == 4 || bits == 6 || bits == 8)) return ORC_EINVAL;
    if (N < 0 || K <= 0 || (K * bits) % 32) return ORC_EINVAL;
    const int64_t wpr = K * bits / 32;
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k)
            q[n * K + k] = (uint8_t)get_code(packed + n * wpr, k, bits);
    return ORC_OK;
}

/* packed rows from codes (inverse of orc_unpack) */
int orc_pack(const uint8_t* q, int bits, int64_t N, int64_t K, uint32_t* packed)
{
    if ((K * bits) % 32 || K <= 0 || N < 0) return ORC_EINVAL;
    const int64_t wpr = K * bits / 32;
    memset(packed, 0, (size_t)(N * wpr) * sizeof(uint32_t));
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k)
            put_code(packed + n * wpr, k, bits, q[n * K + k] & ((1u << bits) - 1));
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* Affine quantize                                                           */
/* ------------------------------------------------------------------------ */

/* Affine group quantization of W [N, K] (binary32), groups of `gs`
 * consecutive elements along K within a row. Per group:
 *   mn, mx  = min, max of the group (exact)
 *   s       = (mx - mn) / (2^bits - 1)                 binary32
 *   s', b'  = s and mn rounded to the storage dtype (RNE); stored
 *   q_i     = clamp(rint((w_i - b') / s'), 0, 2^bits - 1)  binary32, RNE
 *             (q_i = 0 for every element when s' == 0)
 * Codes are computed from the stored s', b' so that the round-trip error
 * bound refers to the values a consumer reads. The scale/bias formulas are
 * the quantization the MLX PR's reproduction script requests
 * (mx.quantize(w, group_size, bits): bias = min, scale = (max-min)/(2^b-1)). */
int orc_quantize(const float* W, int64_t N, int64_t K, int bits, int gs, int dtype,
                 uint32_t* packed, void* scales, void* biases)
{
    if (!valid_affine(bits, gs, N, K) || dtype < 0 || dtype > 2) return ORC_EINVAL;
    const unsigned L = (1u << bits) - 1;
    const int64_t G = K / gs, wpr = K * bits / 32;
    memset(packed, 0, (size_t)(N * wpr) * sizeof(uint32_t));
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t g = 0; g < G; ++g) {
            const float* w = W + n * K + g * gs;
            float mn = w[0], mx = w[0];
            for (int i = 1; i < gs; ++i) {
                if (w[i] < mn) mn = w[i];
                if (w[i] > mx) mx = w[i];
            }
            float range = mx - mn;
            float s = range / (float)L;
            float s_st = store_t(scales, n * G + g, s, dtype);
            float b_st = store_t(biases, n * G + g, mn, dtype);
            for (int i = 0; i < gs; ++i) {
                unsigned q = 0;
                if (s_st != 0.0f) {
                    float d = w[i] - b_st;
                    float r = rintf(d / s_st);
                    if (r <= 0.0f) q = 0;
                    else if (r >= (float)L) q = L;
                    else q = (unsigned)r;
                }
                put_code(packed + n * wpr, g * gs + i, bits, q);
            }
        }
    }
    return ORC_OK;
}

/* what[n*K + k] = s'[n, k/gs] * q[n, k] + b'[n, k/gs] in binary64 */
int orc_dequantize(const uint32_t* packed, const void* scales, const void* biases, int dtype,
                   int bits, int gs, int64_t N, int64_t K, double* what)
{
    if (!valid_affine(bits, gs, N, K) || dtype < 0 || dtype > 2) return ORC_EINVAL;
    const int64_t G = K / gs, wpr = K * bits / 32;
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k) {
            double s = load_t(scales, n * G + k / gs, dtype);
            double b = load_t(biases, n * G + k / gs, dtype);
            what[n * K + k] = s * (double)get_code(packed + n * wpr, k, bits) + b;
        }
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* Affine qmv / qmm_t                                                        */
/* ------------------------------------------------------------------------ */

/* out[m, j] = sum_k what[rows[j], k] * x[m, k] (binary64, k ascending), and
 * absdot[m, j] = sum_k |what[rows[j], k] * x[m, k]|, for the listed rows
 * (all N rows when rows == NULL, in which case j == n).
 * W is stored [N, K] and X [M, K], so this is out = X * What^T: the
 * transposed product of the MLX PR (quantized_matmul(..., transpose=True));
 * M == 1 is qmv (metaltile-std quantized.rs, mt_qmv). Output layout
 * [M, nrows] row-major. */
int orc_qmm(const uint32_t* packed, const void* scales, const void* biases, const void* x,
            int dtype, int bits, int gs, int64_t M, int64_t N, int64_t K,
            const int64_t* rows, int64_t nrows, double* out, double* absdot)
{
    if (!valid_affine(bits, gs, N, K) || dtype < 0 || dtype > 2 || M < 0) return ORC_EINVAL;
    if (!rows) nrows = N;
    const int64_t G = K / gs, wpr = K * bits / 32;
    double* what = (double*)malloc((size_t)K * sizeof(double));
    double* xv = (double*)malloc((size_t)(M * K + 1) * sizeof(double));
    if (!what || !xv) { free(what); free(xv); return ORC_EINVAL; }
    for (int64_t i = 0; i < M * K; ++i) xv[i] = load_t(x, i, dtype);
    for (int64_t j = 0; j < nrows; ++j) {
        int64_t n = rows ? rows[j] : j;
        if (n < 0 || n >= N) { free(what); free(xv); return ORC_EINVAL; }
        for (int64_t k = 0; k < K; ++k) {
            double s = load_t(scales, n * G + k / gs, dtype);
            double b = load_t(biases, n * G + k / gs, dtype);
            what[k] = s * (double)get_code(packed + n * wpr, k, bits) + b;
        }
        for (int64_t m = 0; m < M; ++m) {
            double acc = 0.0, aacc = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                double p = what[k] * xv[m * K + k];
                acc += p;
                aacc += fabs(p);
            }
            out[m * nrows + j] = acc;
            if (absdot) absdot[m * nrows + j] = aacc;
        }
    }
    free(what);
    free(xv);
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* Q8_0                                                                      */
/* ------------------------------------------------------------------------ */

/* Packed Q8_0 block (hanzo-kernel quant.rs, Q8_0 PACKED matvec): 9 words;
 * the low 16 bits of word 0 are the f16 scale d (the high 16 bits are not
 * read); words 1..8 hold the 32 signed int8 codes, four per word, byte 0 of
 * word 1 first. w[32b + j] = d_b * q_j. Blocks are [N][K/32][9]. */
int orc_q8_0_dequant_block(const uint32_t* blk, double* w32)
{
    double d = orc_f16_to_f64((uint16_t)(blk[0] & 0xffffu));
    for (int j = 0; j < 32; ++j) {
        unsigned byte = (blk[1 + j / 4] >> (8 * (j % 4))) & 0xffu;
        int q = byte >= 128 ? (int)byte - 256 : (int)byte;   /* two's complement */
        w32[j] = d * (double)q;
    }
    return ORC_OK;
}

/* out[j] = sum_k w[rows[j], k] * x[k] for the Q8_0 matrix (binary64) */
int orc_q8_0_gemv(const uint32_t* blocks, const float* x, int64_t N, int64_t K,
                  const int64_t* rows, int64_t nrows, double* out, double* absdot)
{
    if (N < 0 || K <= 0 || K % 32) return ORC_EINVAL;
    if (!rows) nrows = N;
    const int64_t nb = K / 32;
    double w32[32];
    for (int64_t j = 0; j < nrows; ++j) {
        int64_t n = rows ? rows[j] : j;
        if (n < 0 || n >= N) return ORC_EINVAL;
        double acc = 0.0, aacc = 0.0;
        for (int64_t b = 0; b < nb; ++b) {
            orc_q8_0_dequant_block(blocks + (n * nb + b) * 9, w32);
            for (int i = 0; i < 32; ++i) {
                double p = w32[i] * (double)x[b * 32 + i];
                acc += p;
                aacc += fabs(p);
            }
        }
        out[j] = acc;
        if (absdot) absdot[j] = aacc;
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* Q8_0 with integer activations (hanzo-kernel quant.rs, "dp4a matvec" and    */
/* "PACKED dp4a matvec": int8 weights and int8 activations, the inner sum an  */
/* exact integer dot product, then out[row] = sum_block wd * dot(qw, xq)).     */
/* The activations are quantized per 32-element block: d = amax / 127 and    */
/* q = rint(x / d), both in binary32 (the codes a binary32 implementation     */
/* must produce), q = 0 for an all-zero block; the block's activation scale   */
/* multiplies the weight scale.                                              */
/* ------------------------------------------------------------------------ */

int orc_quantize_x_q8(const float* x, int64_t K, int8_t* xq, float* xd)
{
    if (K <= 0 || K % 32) return ORC_EINVAL;
    for (int64_t b = 0; b < K / 32; ++b) {
        const float* xb = x + 32 * b;
        float amax = 0.0f;
        for (int i = 0; i < 32; ++i) {
            float a = fabsf(xb[i]);
            if (a > amax) amax = a;
        }
        float d = amax / 127.0f;
        xd[b] = d;
        for (int i = 0; i < 32; ++i) {
            int q = 0;
            if (d != 0.0f) {
                float r = rintf(xb[i] / d);
                q = r > 127.0f ? 127 : (r < -127.0f ? -127 : (int)r);
            }
            xq[32 * b + i] = (int8_t)q;
        }
    }
    return ORC_OK;
}

/* the exact integer dot product of one Q8_0 block's codes with 32 int8 codes */
int64_t orc_q8_0_block_dot_i8(const uint32_t* blk, const int8_t* xq32)
{
    int64_t s = 0;
    for (int j = 0; j < 32; ++j) {
        unsigned byte = (blk[1 + j / 4] >> (8 * (j % 4))) & 0xffu;
        int q = byte >= 128 ? (int)byte - 256 : (int)byte;
        s += (int64_t)q * (int64_t)xq32[j];
    }
    return s;
}

/* out[j] = sum_b d_w[rows[j], b] * xd[b] * dot_b (binary64; dot_b exact) */
int orc_q8_0_gemv_i8(const uint32_t* blocks, const int8_t* xq, const float* xd, int64_t N, int64_t K,
                     const int64_t* rows, int64_t nrows, double* out, double* absdot)
{
    if (N < 0 || K <= 0 || K % 32) return ORC_EINVAL;
    if (!rows) nrows = N;
    const int64_t nb = K / 32;
    for (int64_t j = 0; j < nrows; ++j) {
        int64_t n = rows ? rows[j] : j;
        if (n < 0 || n >= N) return ORC_EINVAL;
        double acc = 0.0, aacc = 0.0;
        for (int64_t b = 0; b < nb; ++b) {
            const uint32_t* blk = blocks + (n * nb + b) * 9;
            double dw = orc_f16_to_f64((uint16_t)(blk[0] & 0xffffu));
            double scale = dw * (double)xd[b];
            int64_t dot = orc_q8_0_block_dot_i8(blk, xq + 32 * b);
            int64_t adot = 0;
            for (int i = 0; i < 32; ++i) {
                unsigned byte = (blk[1 + i / 4] >> (8 * (i % 4))) & 0xffu;
                int q = byte >= 128 ? (int)byte - 256 : (int)byte;
                int64_t p = (int64_t)q * (int64_t)xq[32 * b + i];
                adot += p < 0 ? -p : p;
            }
            acc += scale * (double)dot;
            aacc += fabs(scale) * (double)adot;
        }
        out[j] = acc;
        if (absdot) absdot[j] = aacc;
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* Q4_K                                                                      */
/* ------------------------------------------------------------------------ */

/* get_scale_min_k4 (hanzo-kernel quant.rs, q4k_sc / q4k_m): the 12 scale
 * bytes hold eight 6-bit (scale, min) pairs. For j < 4 the scale is the low
 * 6 bits of byte j and the min the low 6 bits of byte j+4; for j >= 4 the
 * scale is the low nibble of byte j+4 plus the top two bits of byte j-4 as
 * bits 4..5, and the min is the high nibble of byte j+4 plus the top two bits
 * of byte j as bits 4..5. */
void orc_q4_k_scale_min(const uint8_t* sc12, int j, int* sc, int* m)
{
    if (j < 4) {
        *sc = sc12[j] & 63;
        *m = sc12[j + 4] & 63;
    } else {
        *sc = (sc12[j + 4] & 15) | ((sc12[j - 4] >> 6) << 4);
        *m = (sc12[j + 4] >> 4) | ((sc12[j] >> 6) << 4);
    }
}

/* 144-byte Q4_K super-block -> 256 weights (hanzo-kernel quant.rs,
 * matvec_q4k): bytes 0..1 d (f16, little-endian), 2..3 dmin (f16),
 * 4..15 the scale bytes, 16..143 qs. For g in 0..3 and i in 0..31, with
 * qb = qs[32g + i]:
 *   w[64g + i]      = d * sc_{2g}   * (qb & 15) - dmin * m_{2g}
 *   w[64g + 32 + i] = d * sc_{2g+1} * (qb >> 4) - dmin * m_{2g+1}       */
int orc_q4_k_dequant_block(const uint8_t* blk, double* w256)
{
    double d = orc_f16_to_f64((uint16_t)(blk[0] | (blk[1] << 8)));
    double dmin = orc_f16_to_f64((uint16_t)(blk[2] | (blk[3] << 8)));
    const uint8_t* sc12 = blk + 4;
    const uint8_t* qs = blk + 16;
    for (int g = 0; g < 4; ++g) {
        int sc_lo, m_lo, sc_hi, m_hi;
        orc_q4_k_scale_min(sc12, 2 * g, &sc_lo, &m_lo);
        orc_q4_k_scale_min(sc12, 2 * g + 1, &sc_hi, &m_hi);
        for (int i = 0; i < 32; ++i) {
            unsigned qb = qs[32 * g + i];
            w256[64 * g + i] = d * sc_lo * (double)(qb & 15u) - dmin * m_lo;
            w256[64 * g + 32 + i] = d * sc_hi * (double)(qb >> 4) - dmin * m_hi;
        }
    }
    return ORC_OK;
}

/* out[j] = sum_k w[rows[j], k] * x[k] for the Q4_K matrix (binary64);
 * blocks are [N][K/256][144] bytes. */
int orc_q4_k_gemv(const uint8_t* blocks, const float* x, int64_t N, int64_t K,
                  const int64_t* rows, int64_t nrows, double* out, double* absdot)
{
    if (N < 0 || K <= 0 || K % 256) return ORC_EINVAL;
    if (!rows) nrows = N;
    const int64_t nb = K / 256;
    double w256[256];
    for (int64_t j = 0; j < nrows; ++j) {
        int64_t n = rows ? rows[j] : j;
        if (n < 0 || n >= N) return ORC_EINVAL;
        double acc = 0.0, aacc = 0.0;
        for (int64_t b = 0; b < nb; ++b) {
            orc_q4_k_dequant_block(blocks + (n * nb + b) * 144, w256);
            for (int i = 0; i < 256; ++i) {
                double p = w256[i] * (double)x[b * 256 + i];
                acc += p;
                aacc += fabs(p);
            }
        }
        out[j] = acc;
        if (absdot) absdot[j] = aacc;
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* GGUF block layouts beyond the pages: the 34-byte Q8_0 block and Q6_K      */
/* ------------------------------------------------------------------------ */
/*
 * hanzo-kernel quant.rs names Q6_K beside Q4_K as following the same shape
 * (a block decode feeding the same contraction) and describes its Q8_0
 * "production layout" as the 34-byte block re-packed into nine 32-bit words.
 * Neither block layout is written out on the pages. Reading taken here: the
 * GGUF file format's published block definitions.
 *  - Q8_0, 34 bytes per 32 weights: bytes 0..1 the scale d (f16,
 *    little-endian), bytes 2..33 the codes q_0..q_31 (int8); w_j = d * q_j.
 *    The same (d, q) as the nine-word block, without the padding.
 *  - Q6_K, 210 bytes per 256 weights: ql[128] (bytes 0..127) the low four
 *    bits of the codes, qh[64] (bytes 128..191) the high two bits, sc[16]
 *    (bytes 192..207) signed 8-bit scales, one per 16 weights, d (bytes
 *    208..209, f16). Element e = 128h + 32c + l (h < 2, c < 4, l < 32):
 *      low  = nibble c/2 (low nibble first) of ql[64h + 32(c%2) + l]
 *      high = bits 2c..2c+1 of qh[32h + l]
 *      q_e  = (low + 16*high) - 32            (in -32..31)
 *      w_e  = d * sc[e/16] * q_e
 *    (e/16 = 8h + 2c + l/16: each 16 consecutive weights share a scale.)
 */

/* 34-byte Q8_0 block -> 32 weights */
int orc_q8_0_34b_dequant_block(const uint8_t* blk, double* w32)
{
    double d = orc_f16_to_f64((uint16_t)(blk[0] | (blk[1] << 8)));
    for (int j = 0; j < 32; ++j) {
        int q = blk[2 + j] >= 128 ? (int)blk[2 + j] - 256 : (int)blk[2 + j];
        w32[j] = d * (double)q;
    }
    return ORC_OK;
}

/* out[j] = sum_k w[rows[j], k] * x[k]; blocks [N][K/32][34] bytes (binary64) */
int orc_q8_0_34b_gemv(const uint8_t* blocks, const float* x, int64_t N, int64_t K,
                      const int64_t* rows, int64_t nrows, double* out, double* absdot)
{
    if (N < 0 || K <= 0 || K % 32) return ORC_EINVAL;
    if (!rows) nrows = N;
    const int64_t nb = K / 32;
    double w32[32];
    for (int64_t j = 0; j < nrows; ++j) {
        int64_t n = rows ? rows[j] : j;
        if (n < 0 || n >= N) return ORC_EINVAL;
        double acc = 0.0, aacc = 0.0;
        for (int64_t b = 0; b < nb; ++b) {
            orc_q8_0_34b_dequant_block(blocks + (n * nb + b) * 34, w32);
            for (int i = 0; i < 32; ++i) {
                double p = w32[i] * (double)x[b * 32 + i];
                acc += p;
                aacc += fabs(p);
            }
        }
        out[j] = acc;
        if (absdot) absdot[j] = aacc;
    }
    return ORC_OK;
}

/* the signed 6-bit code q_e (-32..31) of element e of a Q6_K super-block */
int orc_q6_k_code(const uint8_t* blk, int e)
{
    const uint8_t* ql = blk;
    const uint8_t* qh = blk + 128;
    int h = e / 128, c = (e / 32) % 4, l = e % 32;
    int low = (ql[64 * h + 32 * (c % 2) + l] >> (4 * (c / 2))) & 15;
    int high = (qh[32 * h + l] >> (2 * c)) & 3;
    return low + 16 * high - 32;
}

/* 210-byte Q6_K super-block -> 256 weights */
int orc_q6_k_dequant_block(const uint8_t* blk, double* w256)
{
    const int8_t* sc = (const int8_t*)(blk + 192);
    double d = orc_f16_to_f64((uint16_t)(blk[208] | (blk[209] << 8)));
    for (int e = 0; e < 256; ++e)
        w256[e] = d * (double)sc[e / 16] * (double)orc_q6_k_code(blk, e);
    return ORC_OK;
}

/* out[j] = sum_k w[rows[j], k] * x[k]; blocks [N][K/256][210] bytes (binary64) */
int orc_q6_k_gemv(const uint8_t* blocks, const float* x, int64_t N, int64_t K,
                  const int64_t* rows, int64_t nrows, double* out, double* absdot)
{
    if (N < 0 || K <= 0 || K % 256) return ORC_EINVAL;
    if (!rows) nrows = N;
    const int64_t nb = K / 256;
    double w256[256];
    for (int64_t j = 0; j < nrows; ++j) {
        int64_t n = rows ? rows[j] : j;
        if (n < 0 || n >= N) return ORC_EINVAL;
        double acc = 0.0, aacc = 0.0;
        for (int64_t b = 0; b < nb; ++b) {
            orc_q6_k_dequant_block(blocks + (n * nb + b) * 210, w256);
            for (int i = 0; i < 256; ++i) {
                double p = w256[i] * (double)x[b * 256 + i];
                acc += p;
                aacc += fabs(p);
            }
        }
        out[j] = acc;
        if (absdot) absdot[j] = aacc;
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* Plain binary32 loops: a CPU timing baseline, not a reference              */
/* ------------------------------------------------------------------------ */
/*
 * The same loops as orc_qmm, orc_q8_0_gemv and orc_q4_k_gemv with every
 * value and the accumulator in binary32: what a plain, untuned CPU
 * implementation of these products computes. They exist to be timed beside
 * the binary64 oracle (the "reasonable CPU" number); no test takes them as
 * the expected result.
 */
int orc_qmm_f32loop(const uint32_t* packed, const void* scales, const void* biases, const void* x,
                    int dtype, int bits, int gs, int64_t M, int64_t N, int64_t K,
                    const int64_t* rows, int64_t nrows, float* out)
{
    if (!valid_affine(bits, gs, N, K) || dtype < 0 || dtype > 2 || M < 0) return ORC_EINVAL;
    if (!rows) nrows = N;
    const int64_t G = K / gs, wpr = K * bits / 32;
    float* w = (float*)malloc((size_t)K * sizeof(float));
    float* xv = (float*)malloc((size_t)(M * K + 1) * sizeof(float));
    if (!w || !xv) { free(w); free(xv); return ORC_EINVAL; }
    for (int64_t i = 0; i < M * K; ++i) xv[i] = (float)load_t(x, i, dtype);
    for (int64_t j = 0; j < nrows; ++j) {
        int64_t n = rows ? rows[j] : j;
        if (n < 0 || n >= N) { free(w); free(xv); return ORC_EINVAL; }
        for (int64_t k = 0; k < K; ++k) {
            float s = (float)load_t(scales, n * G + k / gs, dtype);
            float b = (float)load_t(biases, n * G + k / gs, dtype);
            w[k] = s * (float)get_code(packed + n * wpr, k, bits) + b;
        }
        for (int64_t m = 0; m < M; ++m) {
            float acc = 0.0f;
            for (int64_t k = 0; k < K; ++k) acc += w[k] * xv[m * K + k];
            out[m * nrows + j] = acc;
        }
    }
    free(w);
    free(xv);
    return ORC_OK;
}

int orc_q8_0_gemv_f32loop(const uint32_t* blocks, const float* x, int64_t N, int64_t K,
                          const int64_t* rows, int64_t nrows, float* out)
{
    if (N < 0 || K <= 0 || K % 32) return ORC_EINVAL;
    if (!rows) nrows = N;
    const int64_t nb = K / 32;
    for (int64_t j = 0; j < nrows; ++j) {
        int64_t n = rows ? rows[j] : j;
        if (n < 0 || n >= N) return ORC_EINVAL;
        float acc = 0.0f;
        for (int64_t b = 0; b < nb; ++b) {
            const uint32_t* blk = blocks + (n * nb + b) * 9;
            float d = (float)orc_f16_to_f64((uint16_t)(blk[0] & 0xffffu));
            for (int i = 0; i < 32; ++i) {
                unsigned byte = (blk[1 + i / 4] >> (8 * (i % 4))) & 0xffu;
                int q = byte >= 128 ? (int)byte - 256 : (int)byte;
                acc += d * (float)q * x[b * 32 + i];
            }
        }
        out[j] = acc;
    }
    return ORC_OK;
}

int orc_q4_k_gemv_f32loop(const uint8_t* blocks, const float* x, int64_t N, int64_t K,
                          const int64_t* rows, int64_t nrows, float* out)
{
    if (N < 0 || K <= 0 || K % 256) return ORC_EINVAL;
    if (!rows) nrows = N;
    const int64_t nb = K / 256;
    for (int64_t j = 0; j < nrows; ++j) {
        int64_t n = rows ? rows[j] : j;
        if (n < 0 || n >= N) return ORC_EINVAL;
        float acc = 0.0f;
        for (int64_t b = 0; b < nb; ++b) {
            const uint8_t* blk = blocks + (n * nb + b) * 144;
            float d = (float)orc_f16_to_f64((uint16_t)(blk[0] | (blk[1] << 8)));
            float dmin = (float)orc_f16_to_f64((uint16_t)(blk[2] | (blk[3] << 8)));
            for (int g = 0; g < 4; ++g) {
                int sc_lo, m_lo, sc_hi, m_hi;
                orc_q4_k_scale_min(blk + 4, 2 * g, &sc_lo, &m_lo);
                orc_q4_k_scale_min(blk + 4, 2 * g + 1, &sc_hi, &m_hi);
                for (int i = 0; i < 32; ++i) {
                    unsigned qb = blk[16 + 32 * g + i];
                    acc += (d * (float)sc_lo * (float)(qb & 15u) - dmin * (float)m_lo) * x[b * 256 + 64 * g + i];
                    acc += (d * (float)sc_hi * (float)(qb >> 4) - dmin * (float)m_hi) * x[b * 256 + 64 * g + 32 + i];
                }
            }
        }
        out[j] = acc;
    }
    return ORC_OK;
}
