/*
 * moe4_oracle.c -- the oracle for the 4-bit MoE expert-layer numerics.
 *
 * TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT.  Plain, slow, single-threaded C that spells out,
 * step by step, what the CUDA library has to compute.  Only the test suite, the smoke check and
 * the benchmark's CPU-baseline leg may load it.  It shares no source, header, table or constant
 * with the CUDA library and never calls it; the library never calls it either.
 *
 * Floating point.  Every `float` operation below is one IEEE-754 binary32 operation rounded to
 * nearest-even, in the order written.  The file is compiled with -ffp-contract=off and without
 * -ffast-math (oracle/build.py), so no multiply and add are ever fused.  `double` appears only
 * where a step says so, and only where the double result is exact.
 *
 * Sources.  The method is described in prose only, on these pages:
 *   [DEBUT]  "Inkling 2 Small's Native 4-Bit Training: Debut and Doubts" (agihunt.info), the
 *            "Confirmed" list: NVFP4 forward of the expert layers, MXFP8 backward with
 *            requantisation and stochastic rounding; Four Over Six choosing between two scaling
 *            factors; and the post title "per-expert scales".
 *   [LHC]    "4-bit computation from the start of Inkling 2 Small's pretraining" (lhc.media):
 *            the paragraph on fewer bits (four-bit values sharing a scale across sixteen values,
 *            4.5 bits per value); the two paragraphs on the backward pass (dequantise, transpose at
 *            higher precision, requantise into MXFP8 with stochastic rounding that keeps the value
 *            on average); the paragraph on communication (NVFP4 dispatch; a Hadamard transform
 *            spreads out extreme values before the return path is quantised).
 *   [4WEEK]  "Thinking Machines: Nvidia FP4 Up to 6x Faster, Runs Gain 8%" (fourweekmba.com),
 *            "What Thinking Machines Changed" (3.6x fewer bits than BF16).
 * Where the pages are silent the reading taken is stated beside the function that takes it.
 */
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#if defined(__FLT_EVAL_METHOD__) && __FLT_EVAL_METHOD__ != 0
#error "the oracle needs float expressions evaluated in float (FLT_EVAL_METHOD == 0)"
#endif

static uint32_t f2u(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }
static float u2f(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }

/* ============================================================================================
 * Number formats.  The pages name NVFP4 (4-bit values, one scale per 16) and MXFP8 (8-bit
 * values, one scale per 32) but give no bit layouts.  Reading: the element of NVFP4 is E2M1 and
 * its block scale is E4M3 with a binary32 per-tensor scale; MXFP8 is E4M3 elements with an E8M0
 * scale.  Each format is written below as the sorted list of its non-negative values, indexed by
 * the code without its sign bit, so a cast is "nearest list entry".
 * ========================================================================================== */

/* E2M1: sign | 2 exponent bits (bias 1) | 1 mantissa bit.  Values 0, .5, 1, 1.5, 2, 3, 4, 6. */
static double e2m1_grid(int i)
{
    int e = i >> 1, m = i & 1;
    if (e == 0) return m * 0.5;
    return (1.0 + m * 0.5) * ldexp(1.0, e - 1);
}

/* E4M3 (the OCP "E4M3FN" variant): sign | 4 exponent bits (bias 7) | 3 mantissa bits, no
 * infinities, code 0x7F is NaN, so the non-negative finite codes are 0..126 and the largest
 * value is 448. */
static double e4m3_grid(int i)
{
    int e = i >> 3, m = i & 7;
    if (e == 0) return m * ldexp(1.0, -9);
    return (1.0 + m / 8.0) * ldexp(1.0, e - 7);
}

/* Largest index c in [0, n-2] with grid(c) <= a, for 0 <= a < grid(n-1).  Binary search. */
static int grid_floor(double a, double (*grid)(int), int n)
{
    int lo = 0, hi = n - 1; /* grid(lo) <= a < grid(hi) */
    while (hi - lo > 1) {
        int mid = (lo + hi) / 2;
        if (grid(mid) <= a) lo = mid; else hi = mid;
    }
    return lo;
}

/* Round a >= 0 to the nearest grid entry; a tie goes to the even index (the entry whose
 * mantissa's last bit is 0); anything at or above the top entry saturates to it.  2a and
 * lo + hi are exact in double, so the comparison is exact. */
static int grid_rne_sat(double a, double (*grid)(int), int n)
{
    if (a >= grid(n - 1)) return n - 1;
    int c = grid_floor(a, grid, n);
    double two_a = 2.0 * a, sum = grid(c) + grid(c + 1);
    if (two_a < sum) return c;
    if (two_a > sum) return c + 1;
    return (c & 1) ? c + 1 : c;
}

/* binary32 -> E2M1 code (4 bits), nearest-even, saturating at +-6.  The sign is kept, so a small
 * negative value becomes -0 (code 0x8). */
uint32_t orc_e2m1_rne_sat(float v)
{
    uint32_t sign = (f2u(v) >> 31) << 3;
    return sign | (uint32_t)grid_rne_sat(fabs((double)v), e2m1_grid, 8);
}

float orc_e2m1_value(uint32_t code)
{
    float mag = (float)e2m1_grid((int)(code & 7));
    return (code & 8) ? -mag : mag;
}

/* binary32 -> E4M3 code, nearest-even, saturating at +-448 (values at or above 448 in
 * magnitude give 448). */
uint32_t orc_e4m3_rne_sat(float v)
{
    uint32_t sign = (f2u(v) >> 31) << 7;
    return sign | (uint32_t)grid_rne_sat(fabs((double)v), e4m3_grid, 127);
}

float orc_e4m3_value(uint32_t code)
{
    if ((code & 0x7F) == 0x7F) return NAN;
    float mag = (float)e4m3_grid((int)(code & 0x7F));
    return (code & 0x80) ? -mag : mag;
}

/* E8M0 scale byte b means 2^(b-127); 0xFF is never produced. */
float orc_e8m0_value(uint32_t b) { return (float)ldexp(1.0, (int)b - 127); }

/* binary32 -> bfloat16 bits, nearest-even (finite inputs). */
uint32_t orc_bf16_rne(float v)
{
    uint32_t u = f2u(v);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return u >> 16;
}

float orc_bf16_value(uint32_t h) { return u2f((h & 0xFFFFu) << 16); }

/* ============================================================================================
 * Philox4x32-10, from its published description (Salmon, Moraes, Dror and Shaw, "Parallel
 * random numbers: as easy as 1, 2, 3", SC'11): a 4-word counter and a 2-word key; each of the
 * ten rounds multiplies counter words 0 and 2 by the two round multipliers, mixes the high
 * halves with words 1 and 3 and the key, and the key is bumped by the two Weyl constants
 * between rounds.
 * ========================================================================================== */
void orc_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2], uint32_t out[4])
{
    uint32_t c0 = ctr_in[0], c1 = ctr_in[1], c2 = ctr_in[2], c3 = ctr_in[3];
    uint32_t k0 = key_in[0], k1 = key_in[1];
    for (int round = 0; round < 10; ++round) {
        uint64_t p0 = (uint64_t)0xD2511F53u * c0;
        uint64_t p1 = (uint64_t)0xCD9E8D57u * c2;
        uint32_t n0 = (uint32_t)(p1 >> 32) ^ c1 ^ k0;
        uint32_t n1 = (uint32_t)p1;
        uint32_t n2 = (uint32_t)(p0 >> 32) ^ c3 ^ k1;
        uint32_t n3 = (uint32_t)p0;
        c0 = n0; c1 = n1; c2 = n2; c3 = n3;
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* The random number of one element.  The pages ask only that stochastic rounding keep the value
 * on average.  Reading: each element draws a 16-bit number keyed on (seed, element index), idx
 * being the element's linear index in the OUTPUT array.  Philox runs on counter (lo(idx/8),
 * hi(idx/8), stream_id, 0) with key (lo(seed), hi(seed)); the element takes word (idx/2) % 4 of
 * the output, its low 16 bits when idx is even and its high 16 bits when idx is odd.  One Philox
 * call therefore serves eight consecutive elements. */
uint32_t orc_sr_word(uint64_t seed, uint32_t stream_id, uint64_t idx)
{
    uint64_t j = idx >> 3;
    uint32_t ctr[4] = {(uint32_t)j, (uint32_t)(j >> 32), stream_id, 0u};
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    uint32_t out[4];
    orc_philox4x32_10(ctr, key, out);
    uint32_t word = out[(idx >> 1) & 3];
    return (idx & 1) ? (word >> 16) : (word & 0xFFFFu);
}

/* Stochastic rounding of binary32 v to E4M3 [LHC, backward-pass paragraphs: "probabilistically
 * chooses the higher or lower representable value based on their distance"].  lo is the largest
 * E4M3 magnitude <= |v|, hi the next one; frac = (|v| - lo) / (hi - lo) (exact in double); the
 * magnitude rounds up to hi iff r16 < floor(frac * 2^16), r16 being the element's 16-bit number.
 * The probability of rounding up is floor(frac * 2^16) / 2^16: frac less at most 2^-16, so the
 * value is kept on average to within 2^-16 of a gap.  Magnitudes >= 448 give 448.  The sign is
 * applied afterwards. */
uint32_t orc_e4m3_sr(float v, uint32_t r16)
{
    uint32_t sign = (f2u(v) >> 31) << 7;
    double a = fabs((double)v);
    if (a >= 448.0) return sign | 126u;
    int c = grid_floor(a, e4m3_grid, 127);
    double lo = e4m3_grid(c), hi = e4m3_grid(c + 1);
    double frac = (a - lo) / (hi - lo);
    uint32_t threshold = (uint32_t)floor(frac * 65536.0);
    return sign | (uint32_t)(r16 < threshold ? c + 1 : c);
}

/* ============================================================================================
 * NVFP4 quantisation with Four Over Six.
 * [LHC, fewer-bits paragraph]: 4-bit values with a scale shared across sixteen values.
 * [DEBUT, Confirmed]: quantisation chooses between two scaling factors (Four Over Six) and the
 * recipe uses per-expert scales.
 * Readings (the pages give no formula):
 *  - two-level scaling: a binary32 per-tensor encode scale g_enc = 2688 / amax (2688 = 6 * 448,
 *    so the largest block maps to the top of both E2M1 and E4M3), g_enc = 1 when amax = 0 and
 *    FLT_MAX when the division overflows; the stored decode scale is g_dec = 1 / g_enc.  One
 *    per-tensor scale per matrix: per expert for weights, per whole tensor for activations.
 *  - per 16-block of y = x * g_enc: candidate m in {6, 4}: sf_m = E4M3(a / m) with a the block
 *    amax; codes q_i = E2M1(y_i * (1 / sf_m)); error err_m = sum of (y_i - e2m1(q_i) * sf_m)^2
 *    summed as a fixed pairwise tree (offsets 8, 4, 2, 1).  If sf_m is 0 every code is a zero
 *    carrying y_i's sign and d_i = y_i.  Pick m = 4 iff err_4 < err_6 (ties, including all-zero
 *    blocks, keep 6).  With Four Over Six off, m = 6 always.
 *  - the error is measured on y (the g_enc-scaled values): the same choice as in the original
 *    domain up to the constant factor g_enc^2, and it fixes one order of operations.
 *  - sf_4 saturates at 448 for blocks with a > 1792; that candidate is then kept as computed.
 * ========================================================================================== */

/* The global encode/decode scales from the tensor amax. */
void orc_nvfp4_global_scales(float amax, float *g_enc_out, float *g_dec_out)
{
    float g_enc;
    if (amax == 0.0f) {
        g_enc = 1.0f;
    } else {
        g_enc = 2688.0f / amax;
        if (isinf(g_enc)) g_enc = FLT_MAX;
    }
    *g_enc_out = g_enc;
    *g_dec_out = 1.0f / g_enc;
}

/* One candidate of one block: returns err_m, writes the 16 codes and the scale code. */
static float nvfp4_candidate(const float y[16], float a, float m, uint8_t q[16], uint8_t *sf_code)
{
    float t = a / m;
    uint32_t s = orc_e4m3_rne_sat(t);
    float sfv = orc_e4m3_value(s);
    float d[16];
    if (sfv == 0.0f) {
        for (int i = 0; i < 16; ++i) {
            q[i] = (uint8_t)((f2u(y[i]) >> 31) << 3);
            d[i] = y[i];
        }
    } else {
        float rcp = 1.0f / sfv;
        for (int i = 0; i < 16; ++i) {
            float v = y[i] * rcp;
            q[i] = (uint8_t)orc_e2m1_rne_sat(v);
            float back = orc_e2m1_value(q[i]) * sfv; /* exact: at most 6 significant bits */
            d[i] = y[i] - back;
        }
    }
    float s16[16];
    for (int i = 0; i < 16; ++i) s16[i] = d[i] * d[i];
    for (int off = 8; off >= 1; off >>= 1)
        for (int i = 0; i < off; ++i) s16[i] = s16[i] + s16[i + off];
    *sf_code = (uint8_t)s;
    return s16[0];
}

/* Quantise one matrix x[rows, cols] (row stride ld, in elements) of binary32 values.
 * amax_given: NULL to compute the tensor amax here, else the amax to use.
 * codes [rows, cols/2]: element 2j in the low nibble, 2j+1 in the high nibble.
 * sf    [rows, cols/16]: E4M3 block scale codes.
 * choice (may be NULL) [rows, cols/16]: 4 or 6, the candidate kept.
 * Returns 0, or -1 when cols is not a multiple of 16. */
int orc_nvfp4_quantize(const float *x, int64_t rows, int64_t cols, int64_t ld,
                       const float *amax_given, int four_over_six,
                       uint8_t *codes, uint8_t *sf, float *g_dec_out, uint8_t *choice)
{
    if (cols % 16 != 0) return -1;
    float amax = 0.0f;
    if (amax_given) {
        amax = *amax_given;
    } else {
        for (int64_t r = 0; r < rows; ++r)
            for (int64_t c = 0; c < cols; ++c) {
                float a = fabsf(x[r * ld + c]);
                if (a > amax) amax = a;
            }
    }
    float g_enc, g_dec;
    orc_nvfp4_global_scales(amax, &g_enc, &g_dec);
    *g_dec_out = g_dec;

    int64_t nblk = cols / 16;
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t b = 0; b < nblk; ++b) {
            float y[16];
            float a = 0.0f;
            for (int i = 0; i < 16; ++i) {
                y[i] = x[r * ld + b * 16 + i] * g_enc;
                float ay = fabsf(y[i]);
                if (ay > a) a = ay;
            }
            uint8_t q6[16], q4[16], s6, s4;
            float err6 = nvfp4_candidate(y, a, 6.0f, q6, &s6);
            const uint8_t *q = q6;
            uint8_t s = s6, pick = 6;
            if (four_over_six) {
                float err4 = nvfp4_candidate(y, a, 4.0f, q4, &s4);
                if (err4 < err6) { q = q4; s = s4; pick = 4; }
            }
            for (int j = 0; j < 8; ++j)
                codes[r * (cols / 2) + b * 8 + j] = (uint8_t)(q[2 * j] | (q[2 * j + 1] << 4));
            sf[r * nblk + b] = s;
            if (choice) choice[r * nblk + b] = pick;
        }
    }
    return 0;
}

/* Dequantise: x_hat = (e2m1(q) * sf) * g_dec; the first product is exact. */
void orc_nvfp4_dequantize(const uint8_t *codes, const uint8_t *sf, float g_dec,
                          int64_t rows, int64_t cols, float *out)
{
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < cols; ++c) {
            uint8_t byte = codes[r * (cols / 2) + c / 2];
            uint32_t q = (c & 1) ? (byte >> 4) : (byte & 0xF);
            float e = orc_e2m1_value(q);
            float s = orc_e4m3_value(sf[r * (cols / 16) + c / 16]);
            float es = e * s;
            out[r * cols + c] = es * g_dec;
        }
}

/* ============================================================================================
 * MXFP8 quantisation of 32-blocks [LHC, backward-pass paragraphs: requantise "into MXFP8"].
 * Readings:
 *  - the scale exponent of a block with amax A is the smallest integer e with A <= 448 * 2^e,
 *    clamped to [-127, 127] (A = 0 gives -127, byte 0).  With this rule no scaled element exceeds
 *    448, so nothing is clipped and stochastic rounding stays unbiased;
 *  - the stored scale byte is e + 127 (E8M0); the scaled element is v = x * 2^-e;
 *  - elements are rounded to E4M3 stochastically (words from orc_sr_word, keyed on the element's
 *    index in the output array) or to nearest-even.
 * ========================================================================================== */
int orc_mx_scale_exponent(float amax)
{
    double A = (double)amax;
    int e = -127;
    while (e < 127 && A > 448.0 * ldexp(1.0, e)) ++e;
    return e;
}

/* Quantise z[P, Q] (row-major binary32) along Q in 32-blocks.  Element (p, q) has output index
 * idx_base + p*Q + q.  sr != 0: stochastic rounding; else nearest-even.
 * q8 [P, Q] E4M3 codes, e8 [P, Q/32] scale bytes.  Returns -1 when Q % 32 != 0. */
int orc_mxfp8_quantize_rows(const float *z, int64_t P, int64_t Q, int sr, uint64_t seed,
                            uint32_t stream_id, uint64_t idx_base, uint8_t *q8, uint8_t *e8)
{
    if (Q % 32 != 0) return -1;
    for (int64_t p = 0; p < P; ++p) {
        for (int64_t b = 0; b < Q / 32; ++b) {
            const float *blk = z + p * Q + b * 32;
            float A = 0.0f;
            for (int i = 0; i < 32; ++i) {
                float a = fabsf(blk[i]);
                if (a > A) A = a;
            }
            int e = orc_mx_scale_exponent(A);
            float scale = (float)ldexp(1.0, -e); /* an exact power of two (2^-127 is subnormal) */
            e8[p * (Q / 32) + b] = (uint8_t)(e + 127);
            for (int i = 0; i < 32; ++i) {
                float v = blk[i] * scale;
                uint64_t idx = idx_base + (uint64_t)(p * Q + b * 32 + i);
                uint32_t code = sr ? orc_e4m3_sr(v, orc_sr_word(seed, stream_id, idx))
                                   : orc_e4m3_rne_sat(v);
                q8[p * Q + b * 32 + i] = (uint8_t)code;
            }
        }
    }
    return 0;
}

/* Dequantise MXFP8 rows: e4m3(q) * 2^(e8 - 127). */
void orc_mxfp8_dequantize_rows(const uint8_t *q8, const uint8_t *e8, int64_t P, int64_t Q, float *out)
{
    for (int64_t p = 0; p < P; ++p)
        for (int64_t q = 0; q < Q; ++q)
            out[p * Q + q] = orc_e4m3_value(q8[p * Q + q]) * orc_e8m0_value(e8[p * (Q / 32) + q / 32]);
}

/* Dequantise -> transpose at binary32 -> requantise to MXFP8 [LHC, backward-pass paragraphs],
 * for nmat matrices of NVFP4 [rows, cols] (codes, sf and one g_dec each).  Output matrix m is
 * [cols, rows] (q_t) with scales [cols, rows/32] (e8_t); element (m, c, r) has output index
 * m*cols*rows + c*rows + r.  Returns -1 unless rows % 32 == 0 and cols % 16 == 0. */
int orc_mxfp8_requant_transpose(const uint8_t *codes, const uint8_t *sf, const float *g_dec,
                                int64_t nmat, int64_t rows, int64_t cols, int sr, uint64_t seed,
                                uint32_t stream_id, uint8_t *q_t, uint8_t *e8_t)
{
    if (rows % 32 != 0 || cols % 16 != 0) return -1;
    float *xh = (float *)malloc(sizeof(float) * (size_t)(rows * cols));
    float *xt = (float *)malloc(sizeof(float) * (size_t)(rows * cols));
    if (!xh || !xt) { free(xh); free(xt); return -2; }
    for (int64_t m = 0; m < nmat; ++m) {
        orc_nvfp4_dequantize(codes + m * rows * (cols / 2), sf + m * rows * (cols / 16), g_dec[m],
                             rows, cols, xh);
        for (int64_t r = 0; r < rows; ++r)
            for (int64_t c = 0; c < cols; ++c) xt[c * rows + r] = xh[r * cols + c];
        orc_mxfp8_quantize_rows(xt, cols, rows, sr, seed, stream_id, (uint64_t)(m * cols * rows),
                                q_t + m * cols * rows, e8_t + m * cols * (rows / 32));
    }
    free(xh);
    free(xt);
    return 0;
}

/* ============================================================================================
 * Hadamard return-path codec [LHC, communication paragraph: "a Hadamard transform spreads out
 * extreme values before quantization"].  Readings: the transform is the Sylvester-ordered
 * Hadamard matrix of order 128 (no random signs; the pages mention none), applied to every
 * contiguous 128-chunk of each row, normalised by RN(1/sqrt(128)), and it is its own inverse;
 * the rotated values are quantised to NVFP4 (Four Over Six as the caller asks) with their own
 * per-tensor scale.
 * ========================================================================================== */

/* In-place fast Walsh-Hadamard transform of 128 values: butterflies of span 1, 2, 4, ..., 64,
 * (u[i], u[i+h]) <- (u[i] + u[i+h], u[i] - u[i+h]) for i with bit h clear, then every value times
 * RN(1/sqrt(128)). */
void orc_fwht128(float *u)
{
    for (int h = 1; h < 128; h <<= 1)
        for (int i = 0; i < 128; ++i)
            if ((i & h) == 0) {
                float a = u[i], b = u[i + h];
                u[i] = a + b;
                u[i + h] = a - b;
            }
    const float c = (float)(1.0 / sqrt(128.0));
    for (int i = 0; i < 128; ++i) u[i] = u[i] * c;
}

float orc_hadamard_scale(void) { return (float)(1.0 / sqrt(128.0)); }

/* Rotate each 128-chunk of x[rows, cols] (binary32, row-major) into out. */
int orc_hadamard_rotate(const float *x, int64_t rows, int64_t cols, float *out)
{
    if (cols % 128 != 0) return -1;
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c0 = 0; c0 < cols; c0 += 128) {
            float u[128];
            for (int i = 0; i < 128; ++i) u[i] = x[r * cols + c0 + i];
            orc_fwht128(u);
            for (int i = 0; i < 128; ++i) out[r * cols + c0 + i] = u[i];
        }
    return 0;
}

/* hadamard_quant: rotate, then NVFP4-quantise the rotated tensor with its own amax. */
int orc_hadamard_quant(const float *x, int64_t rows, int64_t cols, int four_over_six,
                       uint8_t *codes, uint8_t *sf, float *g_dec_out)
{
    if (cols % 128 != 0) return -1;
    float *rot = (float *)malloc(sizeof(float) * (size_t)(rows * cols));
    if (!rot) return -2;
    orc_hadamard_rotate(x, rows, cols, rot);
    int rc = orc_nvfp4_quantize(rot, rows, cols, cols, NULL, four_over_six, codes, sf, g_dec_out, NULL);
    free(rot);
    return rc;
}

/* hadamard_dequant: NVFP4 dequantise, inverse rotation (the same transform), round to bf16. */
int orc_hadamard_dequant(const uint8_t *codes, const uint8_t *sf, float g_dec, int64_t rows,
                         int64_t cols, uint16_t *out_bf16)
{
    if (cols % 128 != 0) return -1;
    float *xh = (float *)malloc(sizeof(float) * (size_t)(rows * cols));
    float *rot = (float *)malloc(sizeof(float) * (size_t)(rows * cols));
    if (!xh || !rot) { free(xh); free(rot); return -2; }
    orc_nvfp4_dequantize(codes, sf, g_dec, rows, cols, xh);
    orc_hadamard_rotate(xh, rows, cols, rot);
    for (int64_t i = 0; i < rows * cols; ++i) out_bf16[i] = (uint16_t)orc_bf16_rne(rot[i]);
    free(xh);
    free(rot);
    return 0;
}

/* ============================================================================================
 * The 8.25-bit return-path codec [LHC, communication paragraph: after the Hadamard transform the
 * return path is quantised with per-block scales, cutting its payload from sixteen to 8.25 bits
 * per value].  The pages name the element format "S2F6" without defining it.  Reading: 8.25 bits
 * is an 8-bit element plus one 8-bit scale per 32 values, i.e. the MXFP8 layout used elsewhere in
 * the recipe: E4M3 elements, E8M0 scales by the ceiling rule, nearest-even rounding (the return
 * path belongs to the forward pass, for which the pages mention no stochastic rounding).
 * ========================================================================================== */
int orc_hadamard_quant_mx(const float *x, int64_t rows, int64_t cols, uint8_t *q, uint8_t *e8)
{
    if (cols % 128 != 0) return -1;
    float *rot = (float *)malloc(sizeof(float) * (size_t)(rows * cols));
    if (!rot) return -2;
    orc_hadamard_rotate(x, rows, cols, rot);
    int rc = orc_mxfp8_quantize_rows(rot, rows, cols, 0, 0, 0, 0, q, e8);
    free(rot);
    return rc;
}

int orc_hadamard_dequant_mx(const uint8_t *q, const uint8_t *e8, int64_t rows, int64_t cols, uint16_t *out_bf16)
{
    if (cols % 128 != 0) return -1;
    float *xh = (float *)malloc(sizeof(float) * (size_t)(rows * cols));
    float *rot = (float *)malloc(sizeof(float) * (size_t)(rows * cols));
    if (!xh || !rot) { free(xh); free(rot); return -2; }
    orc_mxfp8_dequantize_rows(q, e8, rows, cols, xh);
    orc_hadamard_rotate(xh, rows, cols, rot);
    for (int64_t i = 0; i < rows * cols; ++i) out_bf16[i] = (uint16_t)orc_bf16_rne(rot[i]);
    free(xh);
    free(rot);
    return 0;
}

/* ============================================================================================
 * Array helpers for the cast tests: convert the binary32 bit patterns start .. start+count-1.
 * ========================================================================================== */
void orc_e2m1_rne_sat_range(uint32_t start, uint64_t count, uint8_t *out)
{
    for (uint64_t i = 0; i < count; ++i) out[i] = (uint8_t)orc_e2m1_rne_sat(u2f(start + (uint32_t)i));
}

void orc_e4m3_rne_sat_range(uint32_t start, uint64_t count, uint8_t *out)
{
    for (uint64_t i = 0; i < count; ++i) out[i] = (uint8_t)orc_e4m3_rne_sat(u2f(start + (uint32_t)i));
}

void orc_bf16_rne_array(const float *x, int64_t n, uint16_t *out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = (uint16_t)orc_bf16_rne(x[i]);
}

void orc_sr_words(uint64_t seed, uint32_t stream_id, uint64_t idx_base, int64_t n, uint16_t *out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = (uint16_t)orc_sr_word(seed, stream_id, idx_base + (uint64_t)i);
}

void orc_e4m3_sr_array(const float *v, const uint16_t *r16, int64_t n, uint8_t *out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = (uint8_t)orc_e4m3_sr(v[i], r16[i]);
}

void orc_e4m3_rne_sat_array(const float *v, int64_t n, uint8_t *out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = (uint8_t)orc_e4m3_rne_sat(v[i]);
}

void orc_e2m1_rne_sat_array(const float *v, int64_t n, uint8_t *out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = (uint8_t)orc_e2m1_rne_sat(v[i]);
}
