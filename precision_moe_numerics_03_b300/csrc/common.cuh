// common.cuh -- device helpers shared by the libmoe4 kernels (sm_103a).
//
// Conversions use the hardware's own cvt instructions (inline PTX); every binary32 step that a
// result depends on bit for bit is written with an explicit round-to-nearest intrinsic
// (__fmul_rn, __fadd_rn, ...) so the compiler can neither fuse nor reorder it.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "../../include/moe4.h"

namespace moe4 {

// ------------------------------------------------------------------ host-side helpers
#define MOE4_CHECK_ARG(cond)          \
    do {                              \
        if (!(cond)) return MOE4_ERR_ARG; \
    } while (0)

static inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
static inline bool aligned4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }
static inline cudaStream_t as_stream(void *s) { return reinterpret_cast<cudaStream_t>(s); }
static inline int launch_status() {
    return cudaGetLastError() == cudaSuccess ? MOE4_OK : MOE4_ERR_CUDA;
}
int num_sms();
// The NVFP4 quantiser of binary32 matrices with a given per-matrix amax (quant.cu), skipping the
// matrices m with skip_offs[m + 1] == skip_offs[m] when skip_offs is not null.  Arguments checked
// by the caller.  ctas_per_sm bounds its grid-stride grid (8 fills the GPU; fewer leaves room on
// every SM for a kernel running beside it on another stream, and then selects the quantiser form
// that takes two blocks per iteration within 72 registers).
int quantize_f32_given(const float *x, int64_t nmat, int64_t rows, int64_t cols, const float *amax_in,
                       uint8_t *codes, uint8_t *sf, float *g_dec, const int32_t *skip_offs, bool four_over_six,
                       bool sf_mma, cudaStream_t st, int ctas_per_sm = 8);

// ------------------------------------------------------------------ bf16
__device__ __forceinline__ float bf16_lo(uint32_t pair) { return __uint_as_float(pair << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t pair) { return __uint_as_float(pair & 0xFFFF0000u); }
__device__ __forceinline__ uint16_t f32_to_bf16_bits(float v) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(v));
}
// bf16(lo) | bf16(hi) << 16, both nearest-even.
__device__ __forceinline__ uint32_t bf16x2_rn(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// ------------------------------------------------------------------ FP4 / FP8 conversions
// Eight binary32 values -> eight E2M1 codes packed into a 32-bit word (element i in nibble i),
// nearest-even with saturation at +-6.  The conversion keeps the sign of a result that rounds to
// zero (a small negative value gives -0, code 0x8), which the exhaustive conversion test checks.
__device__ __forceinline__ uint32_t e2m1x8_rn(const float v[8]) {
    uint32_t out;
    asm("{\n"
        ".reg .b8 b0, b1, b2, b3;\n"
        "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n"
        "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n"
        "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n"
        "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n"
        "mov.b32 %0, {b0, b1, b2, b3};\n"
        "}"
        : "=r"(out)
        : "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]));
    return out;
}

// Eight E2M1 codes (nibble i = element i) -> eight exact binary32 values.
__device__ __forceinline__ void e2m1x8_to_f32(uint32_t word, float out[8]) {
    uint32_t h[4];
    asm("{\n"
        ".reg .b8 b0, b1, b2, b3;\n"
        "mov.b32 {b0, b1, b2, b3}, %4;\n"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n"
        "cvt.rn.f16x2.e2m1x2 %1, b1;\n"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\n"
        "cvt.rn.f16x2.e2m1x2 %3, b3;\n"
        "}"
        : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
        : "r"(word));
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&h[i]));
        out[2 * i] = f.x;
        out[2 * i + 1] = f.y;
    }
}

// Non-negative binary32 -> E4M3 code, nearest-even with saturation at 448.
__device__ __forceinline__ uint32_t e4m3_rn(float v) {
    uint16_t out;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(out) : "f"(0.0f), "f"(v));
    return out & 0xFFu;
}

// Four binary32 -> four E4M3 codes (byte i = element i), nearest-even, saturating.
__device__ __forceinline__ uint32_t e4m3x4_rn(float a, float b, float c, float d) {
    uint16_t lo, hi;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(b), "f"(a));
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(d), "f"(c));
    return (uint32_t)lo | ((uint32_t)hi << 16);
}

// E4M3 code -> exact binary32 value (through f16, which holds every E4M3 value exactly).
__device__ __forceinline__ float e4m3_to_f32(uint32_t code) {
    uint32_t h2;
    uint16_t in = (uint16_t)(code & 0xFFu);
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(in));
    return __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFFu)));
}

// ------------------------------------------------------------------ Philox4x32-10
// Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy as 1, 2, 3" (SC'11).
struct Philox4 {
    uint32_t x, y, z, w;
};

// The ten round keys of one (k0, k1) = (lo(seed), hi(seed)): round i uses k0 + i*0x9E3779B9 and
// k1 + i*0xBB67AE85.  Computed on the host and passed by value as a kernel parameter, so each key
// is read from the constant bank as an operand of the round's three-input XOR.
struct PhiloxKeys {
    uint32_t k0[10], k1[10];
};
static inline PhiloxKeys philox_keys(uint64_t seed) {
    PhiloxKeys k;
    uint32_t a = (uint32_t)seed, b = (uint32_t)(seed >> 32);
    for (int i = 0; i < 10; ++i) {
        k.k0[i] = a;
        k.k1[i] = b;
        a += 0x9E3779B9u;
        b += 0xBB67AE85u;
    }
    return k;
}

template <int NR>
__device__ __forceinline__ void philox_rounds(uint32_t &c0, uint32_t &c1, uint32_t &c2, uint32_t &c3,
                                              const PhiloxKeys &K) {
#pragma unroll
    for (int r = 0; r < NR; ++r) {
        // high and low halves as two multiplies (measured cheaper on this GPU than one 64-bit
        // product: ~96 versus ~122 issue slots per call)
        const uint32_t hi0 = __umulhi(c0, 0xD2511F53u), lo0 = c0 * 0xD2511F53u;
        const uint32_t hi1 = __umulhi(c2, 0xCD9E8D57u), lo1 = c2 * 0xCD9E8D57u;
        const uint32_t n0 = hi1 ^ c1 ^ K.k0[r];
        const uint32_t n2 = hi0 ^ c3 ^ K.k1[r];
        c1 = lo1;
        c3 = lo0;
        c0 = n0;
        c2 = n2;
    }
}

__device__ __forceinline__ Philox4 philox4x32_10(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3,
                                                 const PhiloxKeys K) {
    philox_rounds<10>(c0, c1, c2, c3, K);
    return {c0, c1, c2, c3};
}

// The same generator returning the complement of each word.  The last round's XORs absorb the
// complement, and ~(c * M) = c * (2^32 - M) + (2^32 - 1) is one multiply-add, so the complemented
// words cost nothing extra; the rounding below works on ~r.
__device__ __forceinline__ Philox4 philox4x32_10_not(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3,
                                                     const PhiloxKeys K) {
    philox_rounds<9>(c0, c1, c2, c3, K);
    const uint32_t hi0 = __umulhi(c0, 0xD2511F53u), hi1 = __umulhi(c2, 0xCD9E8D57u);
    return {~(hi1 ^ c1 ^ K.k0[9]), c2 * 0x326172A9u + 0xFFFFFFFFu, ~(hi0 ^ c3 ^ K.k1[9]),
            c0 * 0x2DAEE0ADu + 0xFFFFFFFFu};
}

// ------------------------------------------------------------------ stochastic-rounding numbers
// Every element draws a 16-bit number keyed on (seed, its index idx in the output array): the
// eight output indices 8j .. 8j+7 share Philox4x32-10 call j, on counter (lo(j), hi(j),
// stream_id, 0) and key (lo(seed), hi(seed)); element 8j + 2i + h takes half h (0 low, 1 high)
// of output word i.  So the four words of call j, stored in order, are the eight numbers in
// index order (little-endian 16-bit halves).
__device__ __forceinline__ Philox4 sr_words8(uint64_t j, uint32_t stream_id, const PhiloxKeys K) {
    return philox4x32_10((uint32_t)j, (uint32_t)(j >> 32), stream_id, 0u, K);
}
// Their complements; the 32-bit form is for tensors of at most 2^35 values (counter word 1 zero).
__device__ __forceinline__ Philox4 sr_words8_not(uint64_t j, uint32_t stream_id, const PhiloxKeys K) {
    return philox4x32_10_not((uint32_t)j, (uint32_t)(j >> 32), stream_id, 0u, K);
}
__device__ __forceinline__ Philox4 sr_words8_not32(uint32_t j, uint32_t stream_id, const PhiloxKeys K) {
    return philox4x32_10_not(j, 0u, stream_id, 0u, K);
}

// ------------------------------------------------------------------ MXFP8 scale and rounding
// Smallest e with a <= 448 * 2^e, clamped to [-127, 127], from the bits of a >= 0.
__device__ __forceinline__ int mx_scale_exponent(float a) {
    const uint32_t bits = __float_as_uint(a);
    const int field = (int)(bits >> 23);
    if (field == 0) return -127;  // zero or subnormal: every candidate below -127 clamps
    const int p = field - 127;
    const int e = p - 8 + ((bits & 0x7FFFFFu) > 0x600000u ? 1 : 0);
    return e < -127 ? -127 : e;
}

// The same scale as one biased field fs = e + 135, clamped below at 8 (e >= -127), for finite
// a >= 0: adding 0x1FFFFF to the bits carries into the exponent exactly when the mantissa field
// exceeds 0x600000 (a > 1.75 * 2^p, i.e. a > 448 * 2^(p-8)), and zero or subnormal a gives a
// field below 8.  Scale code e + 127 = fs - 8; 2^-e = (262 - fs) << 23.
__device__ __forceinline__ uint32_t mx_scale_fs(float a) {
    return max((__float_as_uint(a) + 0x1FFFFFu) >> 23, 8u);
}
__device__ __forceinline__ float mx_inv_scale_fs(uint32_t fs) { return __uint_as_float((262u - fs) << 23); }

// 2^-e as binary32 for e in [-127, 126].
__device__ __forceinline__ float pow2_neg(int e) { return __uint_as_float((uint32_t)(127 - e) << 23); }

// Stochastic rounding of v (|v| <= 448) to an E4M3 code with the element's 16-bit number r: the
// magnitude goes up to the next E4M3 value iff r < floor(frac * 2^16), frac = distance above the
// value below in units of the gap.  E4M3 normal range (|v| >= 2^-6): the value below keeps v's
// top 3 mantissa bits, so its code is ((bits >> 20) & 0x7FF) - 960 (exponent rebias 127 -> 7, 3
// mantissa bits), the next value is code + 1, and floor(frac * 2^16) is v's low 20 mantissa bits
// shifted right by 4.  Subnormal range (|v| < 2^-6): the gap is 2^-9 and the code floor(|v|*512).
__device__ __forceinline__ uint32_t e4m3_sr_normal(uint32_t bits, uint32_t r) {
    return (((bits >> 20) & 0x7FFu) - 960u + (r < ((bits & 0xFFFFFu) >> 4) ? 1u : 0u)) | ((bits >> 24) & 0x80u);
}
__device__ __forceinline__ bool e4m3_is_normal(uint32_t bits) { return (bits & 0x7FFFFFFFu) >= 0x3C800000u; }
__device__ __forceinline__ uint32_t e4m3_sr_small(uint32_t bits, uint32_t r) {
    const float s = __fmul_rn(__uint_as_float(bits & 0x7FFFFFFFu), 512.0f);
    const uint32_t fl = __float2uint_rz(s);
    const uint32_t thr = __float2uint_rz(__fmul_rn(__fsub_rn(s, __uint2float_rz(fl)), 65536.0f));
    return (fl + (r < thr ? 1u : 0u)) | ((bits >> 24) & 0x80u);
}
// Zero (+-0) needs no arithmetic; the float path for tiny non-zero values is a rarely taken branch.
__device__ __forceinline__ uint32_t e4m3_sr(float v, uint32_t r) {
    const uint32_t bits = __float_as_uint(v);
    if (e4m3_is_normal(bits)) return e4m3_sr_normal(bits, r);
    if ((bits & 0x7FFFFFFFu) == 0u) return (bits >> 24) & 0x80u;
    return e4m3_sr_small(bits, r);
}
// The integer-carry form for a value that is zero or at least 2^-6 in magnitude, with nw = ~word
// (each 16-bit half of nw is 0xFFFF - r of its element).  Adding 16 * (0xFFFF - r) to the binary32
// bits carries into bit 20 exactly when r < (low20 >> 4), the rule above (the low 4 bits of low20
// cannot complete a carry on their own); masking the low 20 bits then leaves the chosen E4M3
// value (|v| <= 448 keeps the carry below the sign bit and the result finite), which the
// nearest-even conversion returns unchanged.
//   low half:  16 * (0xFFFF - r) = nw's low 16 bits inserted at bit 4 (one bfi);
//   high half: nw >> 12 = 16 * (0xFFFF - r) plus a nibble of the low half, added to the bits with
//              their own low nibble cleared, where that nibble cannot carry (one high multiply-add).
__device__ __forceinline__ uint32_t sr_carry_lo(uint32_t bits, uint32_t nw) {
    uint32_t x;
    asm("bfi.b32 %0, %1, %2, 4, 16;" : "=r"(x) : "r"(nw), "r"(0u));
    return (bits + x) & 0xFFF00000u;
}
__device__ __forceinline__ uint32_t sr_carry_hi(uint32_t bits, uint32_t nw) {
    uint32_t t;
    asm("mad.hi.u32 %0, %1, %2, %3;" : "=r"(t) : "r"(nw), "r"(1u << 20), "r"(bits & 0xFFFFFFF0u));
    return t & 0xFFF00000u;
}
// The fast-path test for four values: 2*bits - 2 (mod 2^32) drops the sign and sends +-0 to the
// top, so the minimum is >= 2*0x3C800000 - 2 iff each value is zero or at least 2^-6 in magnitude.
constexpr uint32_t kSrFastMin = 0x78FFFFFEu;
__device__ __forceinline__ uint32_t sr_fast_key4(float v0, float v1, float v2, float v3) {
    return min(min(__float_as_uint(v0) * 2u - 2u, __float_as_uint(v1) * 2u - 2u),
               min(__float_as_uint(v2) * 2u - 2u, __float_as_uint(v3) * 2u - 2u));
}
// Four consecutive elements (byte i = element i) that passed that test, their numbers in the
// complemented words n01 (elements 0, 1) and n23 (elements 2, 3).
__device__ __forceinline__ uint32_t e4m3x4_sr_fast(float v0, float v1, float v2, float v3, uint32_t n01,
                                                   uint32_t n23) {
    return e4m3x4_rn(__uint_as_float(sr_carry_lo(__float_as_uint(v0), n01)),
                     __uint_as_float(sr_carry_hi(__float_as_uint(v1), n01)),
                     __uint_as_float(sr_carry_lo(__float_as_uint(v2), n23)),
                     __uint_as_float(sr_carry_hi(__float_as_uint(v3), n23)));
}
// The same for any four values: the fast path when it applies, else element by element.
__device__ __forceinline__ uint32_t e4m3x4_sr_nw(float v0, float v1, float v2, float v3, uint32_t n01, uint32_t n23) {
    if (sr_fast_key4(v0, v1, v2, v3) >= kSrFastMin) return e4m3x4_sr_fast(v0, v1, v2, v3, n01, n23);
    return e4m3_sr(v0, ~n01 & 0xFFFFu) | (e4m3_sr(v1, ~n01 >> 16) << 8) | (e4m3_sr(v2, ~n23 & 0xFFFFu) << 16) |
           (e4m3_sr(v3, ~n23 >> 16) << 24);
}

// max(|a|, |b|) per 16-bit half (f16 or bf16); the sign bit of each half is the XOR of the
// inputs' signs, so the caller takes the magnitude of the final result.
template <bool kF16>
__device__ __forceinline__ uint32_t max_abs16x2(uint32_t a, uint32_t b) {
    uint32_t r;
    if constexpr (kF16)
        asm("max.xorsign.abs.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    else
        asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// Four E2M1 code pairs (a word) -> four f16x2 (exact).
__device__ __forceinline__ void e2m1x8_to_h2x4(uint32_t w, uint32_t h[4]) {
    asm("{\n"
        ".reg .b8 b0, b1, b2, b3;\n"
        "mov.b32 {b0, b1, b2, b3}, %4;\n"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n"
        "cvt.rn.f16x2.e2m1x2 %1, b1;\n"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\n"
        "cvt.rn.f16x2.e2m1x2 %3, b3;\n"
        "}"
        : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
        : "r"(w));
}

// ------------------------------------------------------------------ packed binary32 pairs
// mul/add/sub.rn.f32x2: two IEEE round-to-nearest operations in one instruction.  The compiler may
// fuse a packed multiply and a following packed add or subtract into one multiply-add (observed:
// one rounding instead of two), so these are used only where a product feeds no add or subtract;
// bit-exact multiply-then-add chains use __fmul_rn / __fadd_rn, which are never fused.
__device__ __forceinline__ uint64_t f2_pack(float a, float b) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float &a, float &b) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t f2_sub(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

// Two E2M1 codes (a byte) -> f16x2, and two E4M3 codes (16 bits) -> f16x2: both exact.
__device__ __forceinline__ uint32_t e2m1x2_to_h2(uint32_t byte_in_low8) {
    uint32_t h;
    asm("{\n"
        ".reg .b8 b0, b1, b2, b3;\n"
        "mov.b32 {b0, b1, b2, b3}, %1;\n"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n"
        "}"
        : "=r"(h)
        : "r"(byte_in_low8));
    return h;
}
__device__ __forceinline__ uint32_t e4m3x2_to_h2(uint32_t two_codes) {
    uint32_t h;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"((uint16_t)two_codes));
    return h;
}

__device__ __forceinline__ float2 h2_bits_to_f2(uint32_t h) {
    return __half22float2(*reinterpret_cast<const __half2 *>(&h));
}

// fma.rn.f32x2: two single-rounding multiply-adds.
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}

// Offset of the scale byte of (row, blk) in the tensor-core tile layout of a matrix with
// `rows` rows and `nblk` blocks per row (nblk % 4 == 0): 512 bytes per 128-row tile and group of
// four blocks, row 32j + i of the tile at 16i + 4j.
__device__ __forceinline__ int64_t sf_mma_offset(int64_t row, int64_t blk, int64_t nblk) {
    const int64_t rt = row >> 7, i = row & 31, j = (row >> 5) & 3;
    const int64_t kg = blk >> 2, kb = blk & 3;
    return (rt * (nblk >> 2) + kg) * 512 + i * 16 + j * 4 + kb;
}
// The same byte in the canonical [rows, nblk] layout or in the tile layout.
__device__ __forceinline__ int64_t sf_offset(int64_t row, int64_t blk, int64_t nblk, bool mma) {
    return mma ? sf_mma_offset(row, blk, nblk) : row * nblk + blk;
}

// d0 = RN(lo(e2) * nsf + y0), d1 = RN(hi(e2) * nsf + y1): binary32 multiply-adds taking the two
// f16 halves of e2 and the f16 nsf as exact operands.
__device__ __forceinline__ void fma2_f16(uint32_t e2, uint16_t nsf, float y0, float y1, float &d0, float &d1) {
    asm("{\n"
        ".reg .b16 lo, hi;\n"
        "mov.b32 {lo, hi}, %2;\n"
        "fma.rn.f32.f16 %0, lo, %3, %4;\n"
        "fma.rn.f32.f16 %1, hi, %3, %5;\n"
        "}"
        : "=f"(d0), "=f"(d1)
        : "r"(e2), "h"(nsf), "f"(y0), "f"(y1));
}

// ------------------------------------------------------------------ misc
__device__ __forceinline__ int warp_id() { return threadIdx.x >> 5; }
__device__ __forceinline__ int lane_id() { return threadIdx.x & 31; }

// ------------------------------------------------------------------ Hadamard(128)
// One thread per 16 consecutive values (an NVFP4 block): 8 consecutive lanes hold one 128-chunk,
// lane l its sub-block l % 8, so a warp covers four chunks.  Butterfly span h pairs element i (bit
// h clear) with i+h: the lower one becomes u[i] + u[i+h], the upper one u[i] - u[i+h], each one
// binary32 rounding, spans in the order 1, 2, ..., 64.  Spans 1..8 are inside a thread; spans
// 16, 32, 64 pair lane l with lane l ^ 1, ^2, ^4, where fma(+-1, own, partner) rounds the exact
// sum or difference once, as the add or subtract would.
__device__ __forceinline__ void fwht128_sub16(float u[16]) {
    // span 1 in scalar form (its inputs may be products, which must not meet a packed add)
#pragma unroll
    for (int i = 0; i < 16; i += 2) {
        const float a = u[i], b = u[i + 1];
        u[i] = __fadd_rn(a, b);
        u[i + 1] = __fsub_rn(a, b);
    }
    // spans 2, 4, 8 two butterflies at a time: elements i, i+1 (i even, bit h clear) against
    // i+h, i+h+1; every input is a sum or difference, so packed add/sub round as the scalar ones
#pragma unroll
    for (int h = 2; h < 16; h <<= 1)
#pragma unroll
        for (int i = 0; i < 16; i += 2)
            if ((i & h) == 0) {
                const uint64_t a = f2_pack(u[i], u[i + 1]), b = f2_pack(u[i + h], u[i + h + 1]);
                f2_unpack(f2_add(a, b), u[i], u[i + 1]);
                f2_unpack(f2_sub(a, b), u[i + h], u[i + h + 1]);
            }
    const int lane = lane_id();
#pragma unroll
    for (int lm = 1; lm < 8; lm <<= 1) {
        const float sgn = (lane & lm) ? -1.0f : 1.0f;
        const uint64_t sg2 = f2_pack(sgn, sgn);
#pragma unroll
        for (int i = 0; i < 16; i += 2) {
            const float p0 = __shfl_xor_sync(0xFFFFFFFFu, u[i], lm), p1 = __shfl_xor_sync(0xFFFFFFFFu, u[i + 1], lm);
            f2_unpack(f2_fma(sg2, f2_pack(u[i], u[i + 1]), f2_pack(p0, p1)), u[i], u[i + 1]);
        }
    }
    const float c = __uint_as_float(0x3DB504F3u);  // nearest binary32 to 1/sqrt(128)
    const uint64_t c2 = f2_pack(c, c);
#pragma unroll
    for (int i = 0; i < 16; i += 2) f2_unpack(f2_mul(f2_pack(u[i], u[i + 1]), c2), u[i], u[i + 1]);
}


}  // namespace moe4
