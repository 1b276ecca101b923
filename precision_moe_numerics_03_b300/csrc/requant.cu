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

template <SrcKind kind>
__global__ void __launch_bounds__(256) requant_transpose_kernel(
    const uint8_t *__restrict__ codes, const uint8_t *__restrict__ sf, const float *__restrict__ g_dec,
    const uint16_t *__restrict__ xbf, int64_t nmat, int64_t R, int64_t C, uint8_t *__restrict__ q_t,
    uint8_t *__restrict__ e8_t, uint64_t seed, uint32_t stream_id, bool sr, bool sf_mma) {
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
                const uint16_t s2 = __ldg(reinterpret_cast<const uint16_t *>(sf + soff));
                const float gd = g_dec[m];
                const float sa = e4m3_to_f32(s2 & 0xFFu), sb = e4m3_to_f32(s2 >> 8);
                e2m1x8_to_f32(w.x, v);
                e2m1x8_to_f32(w.y, v + 8);
                e2m1x8_to_f32(w.z, v + 16);
                e2m1x8_to_f32(w.w, v + 24);
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] = __fmul_rn(__fmul_rn(v[i], i < 16 ? sa : sb), gd);
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
            }
        } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = 0.0f;
        }
#pragma unroll
        for (int i = 0; i < 32; ++i) tile[half * 32 + i][rl] = v[i];
    }
    __syncthreads();

    // phase 2: one output row segment (128 values) per warp iteration
    const int lane = lane_id();
    const int64_t nblk_out = R / 32;
    for (int cl = warp_id(); cl < kTileC; cl += 8) {
        const int64_t c = c0 + cl;
        if (c >= C) break;
        const float4 x4 = *reinterpret_cast<const float4 *>(&tile[cl][lane * 4]);
        float a = fmaxf(fmaxf(fabsf(x4.x), fabsf(x4.y)), fmaxf(fabsf(x4.z), fabsf(x4.w)));
        a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, 1));
        a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, 2));
        a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, 4));
        const int e = mx_scale_exponent(a);
        const float s = pow2_neg(e);
        const float v0 = __fmul_rn(x4.x, s), v1 = __fmul_rn(x4.y, s);
        const float v2 = __fmul_rn(x4.z, s), v3 = __fmul_rn(x4.w, s);
        const int64_t r = r0 + lane * 4;
        const int64_t idx = (m * C + c) * R + r;
        uint32_t packed;
        if (sr) {
            const Philox4 w = sr_words4((uint64_t)idx >> 2, stream_id, seed);
            packed = e4m3_sr(v0, w.x) | (e4m3_sr(v1, w.y) << 8) | (e4m3_sr(v2, w.z) << 16) |
                     (e4m3_sr(v3, w.w) << 24);
        } else {
            packed = e4m3x4_rn(v0, v1, v2, v3);
        }
        if (r < R) {
            *reinterpret_cast<uint32_t *>(q_t + idx) = packed;
            if ((lane & 7) == 0) e8_t[(m * C + c) * nblk_out + (r >> 5)] = (uint8_t)(e + 127);
        }
    }
}

// Row-wise MXFP8 of bf16 x [R, C]: 8 lanes per 32-block along C, 4 values per lane.
__global__ void __launch_bounds__(256) mxfp8_rowwise_kernel(const uint16_t *__restrict__ x, int64_t R, int64_t C,
                                                            uint8_t *__restrict__ q, uint8_t *__restrict__ e8,
                                                            uint64_t seed, uint32_t stream_id, bool sr) {
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
        if (!live) continue;
        const int e = mx_scale_exponent(a);
        const float s = pow2_neg(e);
        const float v0 = __fmul_rn(x4[0], s), v1 = __fmul_rn(x4[1], s);
        const float v2 = __fmul_rn(x4[2], s), v3 = __fmul_rn(x4[3], s);
        uint32_t packed;
        if (sr) {
            const Philox4 w = sr_words4((uint64_t)gidx, stream_id, seed);
            packed = e4m3_sr(v0, w.x) | (e4m3_sr(v1, w.y) << 8) | (e4m3_sr(v2, w.z) << 16) |
                     (e4m3_sr(v3, w.w) << 24);
        } else {
            packed = e4m3x4_rn(v0, v1, v2, v3);
        }
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
    requant_transpose_kernel<SrcKind::Nvfp4><<<(unsigned)tiles, 256, 0, as_stream(stream)>>>(
        codes, sf, g_dec, nullptr, nmat, rows, cols, q_t, e8_t, seed, stream_id, (flags & MOE4_SR) != 0, sf_mma);
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
        mxfp8_rowwise_kernel<<<(unsigned)grid, 256, 0, st>>>(x, rows, cols, q, e8, seed, stream_id, sr);
    } else {
        MOE4_CHECK_ARG(rows % 32 == 0 && aligned16(x) && aligned4(q));
        const int64_t tiles = ((rows + kTileR - 1) / kTileR) * ((cols + kTileC - 1) / kTileC);
        if (tiles == 0) return MOE4_OK;
        requant_transpose_kernel<SrcKind::Bf16><<<(unsigned)tiles, 256, 0, st>>>(
            nullptr, nullptr, nullptr, x, 1, rows, cols, q, e8, seed, stream_id, sr, false);
    }
    return launch_status();
}
