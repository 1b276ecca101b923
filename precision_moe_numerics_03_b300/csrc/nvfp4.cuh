// nvfp4.cuh -- the NVFP4 block quantiser with Four Over Six, shared by the quantisation kernels
// (quant.cu) and the fused quantise + requantise kernel (requant.cu).
//
// Method: "4-bit computation from the start of Inkling 2 Small's pretraining" (lhc.media),
// fewer-bits paragraph: 4-bit values with a scale shared by sixteen values; "Inkling 2 Small's
// Native 4-Bit Training: Debut and Doubts" (agihunt.info, "Confirmed"): Four Over Six chooses
// between two scaling factors per block.
#pragma once

#include <cfloat>

#include "common.cuh"

namespace moe4 {

// ------------------------------------------------------------------ NVFP4 block quantiser
struct GlobalScale {
    float enc, dec;
};

__device__ __forceinline__ GlobalScale global_scale(float amax) {
    float enc = 1.0f;
    if (amax != 0.0f) {
        enc = __fdiv_rn(2688.0f, amax);
        if (isinf(enc)) enc = FLT_MAX;
    }
    return {enc, __fdiv_rn(1.0f, enc)};
}

// One candidate scale (a/m) for a block of 16 scaled values y: codes (two words, nibble i =
// element i), scale code, and the pairwise-tree sum of squared errors.  Every binary32 step is a
// round-to-nearest intrinsic that is never fused into a multiply-add (a fused d*d + s would round
// once and change near-tie choices); the products e2m1 * e4m3 are exact in f16x2.
// tab[code] = (E4M3 value of a scale code, RN(1/value)) for codes 0..127, built per CTA by
// fill_scale_tab with the same conversion and division, so a lookup replaces both.
__device__ __forceinline__ void fill_scale_tab(float2 *tab) {
    for (int i = threadIdx.x; i < 128; i += blockDim.x) {
        const float v = e4m3_to_f32((uint32_t)i);
        tab[i] = make_float2(v, v == 0.0f ? 0.0f : __fdiv_rn(1.0f, v));
    }
    __syncthreads();
}

template <int M>  // the candidate's target for the block amax: 6 or 4
__device__ __forceinline__ float nvfp4_candidate(const float y[16], float a, const float2 *tab, uint32_t &w0,
                                                 uint32_t &w1, uint32_t &scode) {
    // a/4 is a power-of-two scaling: the product by 0.25 rounds the same real number
    const float t = M == 4 ? __fmul_rn(a, 0.25f) : __fdiv_rn(a, (float)M);
    scode = e4m3_rn(t);  // t >= 0 (or NaN): codes 0..0x7F
    const float2 sv = tab[scode];
    const float sfv = sv.x;
    float d[16];
    if (sfv == 0.0f) {
        w0 = w1 = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            w0 |= (__float_as_uint(y[i]) >> 31) << (4 * i + 3);
            w1 |= (__float_as_uint(y[i + 8]) >> 31) << (4 * i + 3);
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) d[i] = y[i];
    } else {
        const float rcp = sv.y;
        float v[16];
        // packed products: they feed only the E2M1 conversion, never an add, so nothing can fuse
        const uint64_t r2 = f2_pack(rcp, rcp);
#pragma unroll
        for (int i = 0; i < 8; ++i) f2_unpack(f2_mul(f2_pack(y[2 * i], y[2 * i + 1]), r2), v[2 * i], v[2 * i + 1]);
        w0 = e2m1x8_rn(v);
        w1 = e2m1x8_rn(v + 8);
        // d = y - e*sf: e*sf has at most 6 significant bits and is exact, so the fused form rounds
        // once, exactly as the subtraction of the exact product does.  e (E2M1) and -sf (E4M3)
        // are exact in f16 and enter the binary32 multiply-add as f16 operands.
        const uint16_t nsf = __half_as_ushort(__float2half_rn(-sfv));
        uint32_t eh[8];
        e2m1x8_to_h2x4(w0, eh);
        e2m1x8_to_h2x4(w1, eh + 4);
#pragma unroll
        for (int i = 0; i < 8; ++i) fma2_f16(eh[i], nsf, y[2 * i], y[2 * i + 1], d[2 * i], d[2 * i + 1]);
    }
    float s[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) s[i] = __fmul_rn(d[i], d[i]);
#pragma unroll
    for (int off = 8; off >= 1; off >>= 1)
#pragma unroll
        for (int i = 0; i < off; ++i) s[i] = __fadd_rn(s[i], s[i + off]);
    return s[0];
}

__device__ __forceinline__ void nvfp4_block(const float y[16], bool four_over_six, const float2 *tab, uint32_t &w0,
                                            uint32_t &w1, uint32_t &scode) {
    float a = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) a = fmaxf(a, fabsf(y[i]));
    const float err6 = nvfp4_candidate<6>(y, a, tab, w0, w1, scode);
    if (four_over_six) {
        uint32_t u0, u1, s4;
        const float err4 = nvfp4_candidate<4>(y, a, tab, u0, u1, s4);
        if (err4 < err6) {
            w0 = u0;
            w1 = u1;
            scode = s4;
        }
    }
}


}  // namespace moe4
