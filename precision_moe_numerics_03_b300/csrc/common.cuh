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

// ------------------------------------------------------------------ bf16
__device__ __forceinline__ float bf16_lo(uint32_t pair) { return __uint_as_float(pair << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t pair) { return __uint_as_float(pair & 0xFFFF0000u); }
__device__ __forceinline__ uint16_t f32_to_bf16_bits(float v) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(v));
}

// ------------------------------------------------------------------ FP4 / FP8 conversions
// Eight binary32 values -> eight E2M1 codes packed into a 32-bit word (element i in nibble i),
// nearest-even with saturation at +-6.  The sign bit of every code is then forced to the sign of
// its input, so a small negative value is -0 (code 0x8) whatever the hardware does with -0.
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
    uint32_t signs = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) signs |= (__float_as_uint(v[i]) >> 31) << (4 * i + 3);
    return out | signs;
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

__device__ __forceinline__ Philox4 philox4x32_10(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3,
                                                 uint32_t k0, uint32_t k1) {
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        const uint32_t lo0 = 0xD2511F53u * c0, hi0 = __umulhi(0xD2511F53u, c0);
        const uint32_t lo1 = 0xCD9E8D57u * c2, hi1 = __umulhi(0xCD9E8D57u, c2);
        const uint32_t n0 = hi1 ^ c1 ^ k0;
        const uint32_t n2 = hi0 ^ c3 ^ k1;
        c0 = n0;
        c1 = lo1;
        c2 = n2;
        c3 = lo0;
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    return {c0, c1, c2, c3};
}

// The four stochastic-rounding words of output indices 4j .. 4j+3.
__device__ __forceinline__ Philox4 sr_words4(uint64_t j, uint32_t stream_id, uint64_t seed) {
    return philox4x32_10((uint32_t)j, (uint32_t)(j >> 32), stream_id, 0u, (uint32_t)seed,
                         (uint32_t)(seed >> 32));
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

// 2^-e as binary32 for e in [-127, 126].
__device__ __forceinline__ float pow2_neg(int e) { return __uint_as_float((uint32_t)(127 - e) << 23); }

// Stochastic rounding of v (|v| <= 448) to an E4M3 code with random word r: the magnitude goes
// up to the next E4M3 value iff r < floor(frac * 2^32), frac = distance above the value below in
// units of the gap.  E4M3 normal range: the gap is 2^20 units of v's last bit, so the threshold
// is v's low 20 mantissa bits shifted up by 12; subnormal range (below 2^-6): gap 2^-9.
__device__ __forceinline__ uint32_t e4m3_sr(float v, uint32_t r) {
    const uint32_t sign = (__float_as_uint(v) >> 31) << 7;
    const float a = fabsf(v);
    const uint32_t ab = __float_as_uint(a);
    float chosen;
    if (ab >= 0x3C800000u) {  // a >= 2^-6
        const uint32_t thr = (ab & 0xFFFFFu) << 12;
        const uint32_t lo = ab & 0xFFF00000u;
        chosen = __uint_as_float(r < thr ? lo + 0x100000u : lo);
    } else {
        const float s = __fmul_rn(a, 512.0f);
        const float fl = floorf(s);
        const uint32_t thr = __float2uint_rz(__fmul_rn(__fsub_rn(s, fl), 4294967296.0f));
        chosen = __fmul_rn(r < thr ? __fadd_rn(fl, 1.0f) : fl, 0.001953125f);  // * 2^-9, exact
    }
    return e4m3_rn(chosen) | sign;
}

// ------------------------------------------------------------------ misc
__device__ __forceinline__ int warp_id() { return threadIdx.x >> 5; }
__device__ __forceinline__ int lane_id() { return threadIdx.x & 31; }

}  // namespace moe4
