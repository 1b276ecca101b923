// requant.cu -- dequantise -> transpose -> MXFP8 requantisation with stochastic rounding, and the
// MXFP8 quantisation of bf16 tensors (row-wise or transposed).
//
// Method: "4-bit computation from the start of Inkling 2 Small's pretraining" (lhc.media),
// backward-pass paragraphs: the forward operands are dequantised, transposed at higher precision
// and requantised into MXFP8 with stochastic rounding, which picks the upper or lower neighbour
// with probability given by the distance so that the value is kept on average.
//
// Tile: 128 input rows (the output's contiguous dimension) x 64 input columns.  Phase 1: each
// thread reads one row's 32 codes (16 bytes) and two scale bytes, dequantises them to binary32
// and stores them transposed in shared memory (row pitch 132 floats: conflict-free both ways).
// Phase 2: each warp emits one output row segment of 128 values: lane l owns 4 consecutive values
// (one Philox call gives their 4 words), 8 lanes form one 32-block (amax by 3 shuffles).
#include "common.cuh"

namespace moe4 {

constexpr int kTileR = 128;
constexpr int kTileC = 64;
constexpr int kPitch = kTileR + 4;

enum class SrcKind { Nvfp4, Bf16 };

// Output of one warp iteration: the 128 values of output row c (input column c) in this tile.
// Lane l owns values 4l..4l+3; lanes 8b..8b+7 form 32-block b (amax by three shuffles).
template <bool kSR>
__device__ __forceinline__ void emit_row(const float4 x4, int64_t m, int64_t c, int64_t r0, int64_t R, int64_t C,
                                         uint8_t *__restrict__ q_t, uint8_t *__restrict__ e8_t,
                                         const PhiloxKeys keys, uint32_t stream_id) {
    const int lane = lane_id();
    float a = fmaxf(fmaxf(fabsf(x4.x), fabsf(x4.y)), fmaxf(fabsf(x4.z), fabsf(x4.w)));
    a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, 1));
    a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, 2));
    a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, 4));
    const int e = mx_scale_exponent(a);
    const float s = pow2_neg(e);
    float v0, v1, v2, v3;
    f2_unpack(f2_mul(f2_pack(x4.x, x4.y), f2_pack(s, s)), v0, v1);
    f2_unpack(f2_mul(f2_pack(x4.z, x4.w), f2_pack(s, s)), v2, v3);
    const int64_t r = r0 + lane * 4;
    const int64_t idx = (m * C + c) * R + r;
    uint32_t packed;
    if constexpr (kSR) {
        packed = e4m3x4_sr(v0, v1, v2, v3, sr_words4((uint64_t)idx >> 2, stream_id, keys));
    } else {
        packed = e4m3x4_rn(v0, v1, v2, v3);
    }
    if (r < R) {
        *reinterpret_cast<uint32_t *>(q_t + idx) = packed;
        if ((lane & 7) == 0) e8_t[(m * C + c) * (R / 32) + (r >> 5)] = (uint8_t)(e + 127);
    }
}

// The row-wise MXFP8 of the 32 values a thread holds in phase 1 (one block along the row),
// nearest-even: written to q_r [R, C] and e8_r [R, C/32] when the kernel also emits that layout.
__device__ __forceinline__ void emit_rowwise32(const float v[32], int64_t r, int64_t c, int64_t C,
                                               uint8_t *__restrict__ q_r, uint8_t *__restrict__ e8_r) {
    float a = 0.0f;
#pragma unroll
    for (int i = 0; i < 32; ++i) a = fmaxf(a, fabsf(v[i]));
    const int e = mx_scale_exponent(a);
    const float s = pow2_neg(e);
    uint32_t w[8];
#pragma unroll
    for (int j = 0; j < 8; ++j)
        w[j] = e4m3x4_rn(__fmul_rn(v[4 * j], s), __fmul_rn(v[4 * j + 1], s), __fmul_rn(v[4 * j + 2], s),
                         __fmul_rn(v[4 * j + 3], s));
    uint4 *dst = reinterpret_cast<uint4 *>(q_r + r * C + c);
    dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
    dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
    e8_r[r * (C / 32) + c / 32] = (uint8_t)(e + 127);
}

template <SrcKind kind, bool kSR, bool kRow = false>
__global__ void __launch_bounds__(256) requant_transpose_kernel(
    const uint8_t *__restrict__ codes, const uint8_t *__restrict__ sf, const float *__restrict__ g_dec,
    const uint16_t *__restrict__ xbf, int64_t nmat, int64_t R, int64_t C, uint8_t *__restrict__ q_t,
    uint8_t *__restrict__ e8_t, const PhiloxKeys keys, uint32_t stream_id, bool sf_mma,
    uint8_t *__restrict__ q_r = nullptr, uint8_t *__restrict__ e8_r = nullptr) {
    __shared__ __align__(16) float tile[kTileC][kPitch];
    const int64_t n_rt = (R + kTileR - 1) / kTileR;
    const int64_t n_ct = (C + kTileC - 1) / kTileC;
    const int64_t t = blockIdx.x;
    const int64_t rt = t % n_rt;
    const int64_t rest = t / n_rt;
    const int64_t ct = rest % n_ct;
    const int64_t m = rest / n_ct;
    const int64_t r0 = rt * kTileR, c0 = ct * kTileC;

    // phase 1: load, dequantise, transpose into shared memory
    {
        const int rl = threadIdx.x & (kTileR - 1);
        const int half = threadIdx.x >> 7;
        const int64_t r = r0 + rl;
        const int64_t c = c0 + half * 32;
        float v[32];
        if (r < R && c < C) {
            if constexpr (kind == SrcKind::Nvfp4) {
                const uint4 w = __ldg(reinterpret_cast<const uint4 *>(codes + ((m * R + r) * C + c) / 2));
                // the scales of blocks c/16 and c/16 + 1 (c/16 even): adjacent bytes in both layouts
                const int64_t nblk = C / 16, b = c / 16;
                const int64_t soff = sf_mma ? m * R * nblk + ((r >> 7) * (nblk >> 2) + (b >> 2)) * 512 + (r & 31) * 16 +
                                                  ((r >> 5) & 3) * 4 + (b & 3)
                                            : (m * R + r) * nblk + b;
                const uint32_t sf2 = e4m3x2_to_h2(__ldg(reinterpret_cast<const uint16_t *>(sf + soff)));
                const uint32_t sfa2 = __byte_perm(sf2, 0, 0x1010), sfb2 = __byte_perm(sf2, 0, 0x3232);
                const uint64_t g2 = f2_pack(g_dec[m], g_dec[m]);
                const uint32_t words[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const __half2 sfh = *reinterpret_cast<const __half2 *>(q < 2 ? &sfa2 : &sfb2);
#pragma unroll
                    for (int b2 = 0; b2 < 4; ++b2) {
                        // e2m1 * e4m3 has at most 6 significant bits: exact in f16, then exact in f32
                        uint32_t h = e2m1x2_to_h2(words[q] >> (8 * b2));
                        const __half2 es = __hmul2(*reinterpret_cast<const __half2 *>(&h), sfh);
                        const float2 f = __half22float2(es);
                        f2_unpack(f2_mul(f2_pack(f.x, f.y), g2), v[8 * q + 2 * b2], v[8 * q + 2 * b2 + 1]);
                    }
                }
            } else {
                const uint4 *src = reinterpret_cast<const uint4 *>(xbf + (m * R + r) * C + c);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const uint4 w = __ldg(src + q);
                    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        v[8 * q + 2 * i] = bf16_lo(ws[i]);
                        v[8 * q + 2 * i + 1] = bf16_hi(ws[i]);
                    }
                }
                if constexpr (kRow) emit_rowwise32(v, r, c, C, q_r, e8_r);
            }
        } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = 0.0f;
        }
#pragma unroll
        for (int i = 0; i < 32; ++i) tile[half * 32 + i][rl] = v[i];
    }
    __syncthreads();

    // phase 2: two output row segments (128 values each) per warp iteration
    const int lane = lane_id();
#pragma unroll 1
    for (int cl = warp_id(); cl < kTileC; cl += 16) {
        const int64_t ca = c0 + cl, cb = c0 + cl + 8;
        const float4 xa = *reinterpret_cast<const float4 *>(&tile[cl][lane * 4]);
        const float4 xb = *reinterpret_cast<const float4 *>(&tile[cl + 8][lane * 4]);
        if (ca < C) emit_row<kSR>(xa, m, ca, r0, R, C, q_t, e8_t, keys, stream_id);
        if (cb < C) emit_row<kSR>(xb, m, cb, r0, R, C, q_t, e8_t, keys, stream_id);
    }
}

// Row-wise MXFP8 of bf16 x [R, C]: 8 lanes per 32-block along C, 4 values per lane.
__global__ void __launch_bounds__(256) mxfp8_rowwise_kernel(const uint16_t *__restrict__ x, int64_t R, int64_t C,
                                                            uint8_t *__restrict__ q, uint8_t *__restrict__ e8,
                                                            const PhiloxKeys keys, uint32_t stream_id, bool sr) {
    const int64_t groups = R * C / 4;  // one group of 4 values per thread
    for (int64_t gidx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; gidx - (threadIdx.x & 31) < groups;
         gidx += (int64_t)gridDim.x * blockDim.x) {
        const bool live = gidx < groups;
        float x4[4] = {0.f, 0.f, 0.f, 0.f};
        if (live) {
            const uint2 w = __ldg(reinterpret_cast<const uint2 *>(x + gidx * 4));
            x4[0] = bf16_lo(w.x);
            x4[1] = bf16_hi(w.x);
            x4[2] = bf16_lo(w.y);
            x4[3] = bf16_hi(w.y);
        }
        float a = fmaxf(fmaxf(fabsf(x4[0]), fabsf(x4[1])), fmaxf(fabsf(x4[2]), fabsf(x4[3])));
        a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, 1));
        a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, 2));
        a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, 4));
        const int e = mx_scale_exponent(a);
        const float s = pow2_neg(e);
        const float v0 = __fmul_rn(x4[0], s), v1 = __fmul_rn(x4[1], s);
        const float v2 = __fmul_rn(x4[2], s), v3 = __fmul_rn(x4[3], s);
        uint32_t packed;
        if (sr) {
            packed = e4m3x4_sr(v0, v1, v2, v3, sr_words4((uint64_t)gidx, stream_id, keys));
        } else {
            packed = e4m3x4_rn(v0, v1, v2, v3);
        }
        if (!live) continue;
        *reinterpret_cast<uint32_t *>(q + gidx * 4) = packed;
        if ((gidx & 7) == 0) e8[gidx >> 3] = (uint8_t)(e + 127);
    }
}

}  // namespace moe4

using namespace moe4;

extern "C" int mxfp8_requant_transpose_sr(const uint8_t *codes, const uint8_t *sf, const float *g_dec,
                                          int64_t nmat, int64_t rows, int64_t cols, uint8_t *q_t,
                                          uint8_t *e8_t, uint64_t seed, uint32_t stream_id, uint32_t flags,
                                          void *stream) {
    MOE4_CHECK_ARG(nmat >= 1 && rows >= 0 && cols > 0 && rows % 32 == 0 && cols % 32 == 0);
    MOE4_CHECK_ARG(codes && sf && g_dec && q_t && e8_t);
    MOE4_CHECK_ARG(aligned16(codes) && aligned4(q_t) && (reinterpret_cast<uintptr_t>(sf) & 1u) == 0);
    MOE4_CHECK_ARG((flags & ~(MOE4_SR | MOE4_SF_MMA_LAYOUT)) == 0);
    const bool sf_mma = (flags & MOE4_SF_MMA_LAYOUT) != 0;
    MOE4_CHECK_ARG(!sf_mma || (rows % 128 == 0 && cols % 64 == 0));
    const int64_t tiles = nmat * ((rows + kTileR - 1) / kTileR) * ((cols + kTileC - 1) / kTileC);
    if (tiles == 0) return MOE4_OK;
    MOE4_CHECK_ARG(tiles < (int64_t(1) << 31));
    if (flags & MOE4_SR)
        requant_transpose_kernel<SrcKind::Nvfp4, true><<<(unsigned)tiles, 256, 0, as_stream(stream)>>>(
            codes, sf, g_dec, nullptr, nmat, rows, cols, q_t, e8_t, philox_keys(seed), stream_id, sf_mma);
    else
        requant_transpose_kernel<SrcKind::Nvfp4, false><<<(unsigned)tiles, 256, 0, as_stream(stream)>>>(
            codes, sf, g_dec, nullptr, nmat, rows, cols, q_t, e8_t, philox_keys(seed), stream_id, sf_mma);
    return launch_status();
}

extern "C" int mxfp8_quantize(const uint16_t *x, int64_t rows, int64_t cols, uint8_t *q, uint8_t *e8,
                              uint64_t seed, uint32_t stream_id, uint32_t flags, void *stream) {
    MOE4_CHECK_ARG(rows >= 0 && cols > 0 && cols % 32 == 0);
    MOE4_CHECK_ARG(q && e8 && (rows == 0 || x));
    MOE4_CHECK_ARG((flags & ~(MOE4_SR | MOE4_ROWWISE | MOE4_COLWISE)) == 0);
    const bool row = (flags & MOE4_ROWWISE) != 0, col = (flags & MOE4_COLWISE) != 0;
    MOE4_CHECK_ARG(row != col);
    const bool sr = (flags & MOE4_SR) != 0;
    cudaStream_t st = as_stream(stream);
    if (row) {
        MOE4_CHECK_ARG(aligned16(x) && aligned4(q));
        const int64_t groups = rows * cols / 4;
        if (groups == 0) return MOE4_OK;
        int64_t grid = (groups + 255) / 256;
        const int64_t cap = (int64_t)num_sms() * 8;
        if (grid > cap) grid = cap;
        mxfp8_rowwise_kernel<<<(unsigned)grid, 256, 0, st>>>(x, rows, cols, q, e8, philox_keys(seed), stream_id, sr);
    } else {
        MOE4_CHECK_ARG(rows % 32 == 0 && aligned16(x) && aligned4(q));
        const int64_t tiles = ((rows + kTileR - 1) / kTileR) * ((cols + kTileC - 1) / kTileC);
        if (tiles == 0) return MOE4_OK;
        MOE4_CHECK_ARG(tiles < (int64_t(1) << 31));
        if (sr)
            requant_transpose_kernel<SrcKind::Bf16, true><<<(unsigned)tiles, 256, 0, st>>>(
                nullptr, nullptr, nullptr, x, 1, rows, cols, q, e8, philox_keys(seed), stream_id, false);
        else
            requant_transpose_kernel<SrcKind::Bf16, false><<<(unsigned)tiles, 256, 0, st>>>(
                nullptr, nullptr, nullptr, x, 1, rows, cols, q, e8, philox_keys(seed), stream_id, false);
    }
    return launch_status();
}

extern "C" int mxfp8_quantize_rowcol(const uint16_t *x, int64_t rows, int64_t cols, uint8_t *q_row,
                                     uint8_t *e8_row, uint8_t *q_col, uint8_t *e8_col, uint32_t flags,
                                     void *stream) {
    MOE4_CHECK_ARG(rows >= 0 && rows % 32 == 0 && cols > 0 && cols % 32 == 0 && flags == 0);
    MOE4_CHECK_ARG(q_row && e8_row && q_col && e8_col && (rows == 0 || x));
    MOE4_CHECK_ARG(aligned16(x) && aligned16(q_row) && aligned4(q_col));
    const int64_t tiles = ((rows + kTileR - 1) / kTileR) * ((cols + kTileC - 1) / kTileC);
    if (tiles == 0) return MOE4_OK;
    MOE4_CHECK_ARG(tiles < (int64_t(1) << 31));
    requant_transpose_kernel<SrcKind::Bf16, false, true><<<(unsigned)tiles, 256, 0, as_stream(stream)>>>(
        nullptr, nullptr, nullptr, x, 1, rows, cols, q_col, e8_col, philox_keys(0), 0u, false, q_row, e8_row);
    return launch_status();
}
