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

// Nvfp4: dequantised NVFP4 codes.  Bf16: a bf16 tensor.  SwigluBwd: the SwiGLU gradient
// dGU [R, 2f] (gate columns, then up columns) formed from the binary32 GU and dH and rounded to
// bf16 exactly as moe4_swiglu_backward does; its tiles pair 32 gate columns with the same 32 up
// columns, so each GU and dH value is read once.
// CombineBwd: the combine's gradient dYhat [R, C] formed on the fly, dispatched row r = token t's
// slot j: bf16(w[t, j] * dy[t]) as moe4_combine_backward computes it (padding rows zero).
enum class SrcKind { Nvfp4, Bf16, SwigluBwd, CombineBwd };

// Output of half a warp: 128 values of output row c (input column c) of this tile.  Lane
// sub = lane % 16 owns values 8*sub .. 8*sub + 7; lanes 4b .. 4b+3 of the half form 32-block b
// (amax by two shuffles).  Every lane takes part in the shuffles; `live` only guards the stores.
template <bool kSR>
__device__ __forceinline__ void emit8(const float x[8], bool live, int64_t m, int64_t c, int64_t r0, int64_t R,
                                      int64_t C, uint8_t *__restrict__ q_t, uint8_t *__restrict__ e8_t,
                                      const PhiloxKeys keys, uint32_t stream_id) {
    const int sub = lane_id() & 15;
    float a = fmaxf(fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3]))),
                    fmaxf(fmaxf(fabsf(x[4]), fabsf(x[5])), fmaxf(fabsf(x[6]), fabsf(x[7]))));
    a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, 1));
    a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, 2));
    const int e = mx_scale_exponent(a);
    const float s = pow2_neg(e);
    const uint64_t s2 = f2_pack(s, s);
    float v[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) f2_unpack(f2_mul(f2_pack(x[2 * i], x[2 * i + 1]), s2), v[2 * i], v[2 * i + 1]);
    const int64_t r = r0 + sub * 8;
    const int64_t idx = (m * C + c) * R + r;
    uint32_t lo, hi;
    if constexpr (kSR) {
        const uint64_t j = (uint64_t)idx >> 2;
        lo = e4m3x4_sr(v[0], v[1], v[2], v[3], sr_words4(j, stream_id, keys));
        hi = e4m3x4_sr(v[4], v[5], v[6], v[7], sr_words4(j + 1, stream_id, keys));
    } else {
        lo = e4m3x4_rn(v[0], v[1], v[2], v[3]);
        hi = e4m3x4_rn(v[4], v[5], v[6], v[7]);
    }
    if (live && r < R) {
        *reinterpret_cast<uint2 *>(q_t + idx) = make_uint2(lo, hi);
        if ((sub & 3) == 0) e8_t[(m * C + c) * (R / 32) + (r >> 5)] = (uint8_t)(e + 127);
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

// Shared tile: 64 input columns x 128 input rows of 16-bit values, transposed (row = input
// column).  An NVFP4 source stores e2m1 * e4m3 as f16 (at most 6 significant bits: exact) and the
// binary32 product with g_dec is formed when the value is read back, the same single rounding;
// a bf16 source stores its bits.
constexpr int kPitch16 = kTileR + 8;

template <SrcKind kind, bool kSR, bool kRow = false>
__global__ void __launch_bounds__(256, (kSR || kind == SrcKind::SwigluBwd || kind == SrcKind::CombineBwd) ? 4 : 5)
requant_transpose_kernel(
    const uint8_t *__restrict__ codes, const uint8_t *__restrict__ sf, const float *__restrict__ g_dec,
    const uint16_t *__restrict__ xbf, int64_t nmat, int64_t R, int64_t C, uint8_t *__restrict__ q_t,
    uint8_t *__restrict__ e8_t, const PhiloxKeys keys, uint32_t stream_id, bool sf_mma,
    uint8_t *__restrict__ q_r = nullptr, uint8_t *__restrict__ e8_r = nullptr, const float *__restrict__ gu = nullptr,
    const float *__restrict__ dh = nullptr, const int32_t *__restrict__ src_of = nullptr,
    const int32_t *__restrict__ row_of = nullptr, const float *__restrict__ wts = nullptr, int topk = 0) {
    constexpr bool kSwb = kind == SrcKind::SwigluBwd;
    __shared__ __align__(16) uint16_t tile[kTileC][kPitch16];
    const int64_t f = C / 2;  // SwigluBwd: C = 2f
    const int64_t n_rt = (R + kTileR - 1) / kTileR;
    const int64_t n_ct = kSwb ? f / 32 : (C + kTileC - 1) / kTileC;
    const int64_t t = blockIdx.x;
    const int64_t rt = t % n_rt;
    const int64_t rest = t / n_rt;
    const int64_t ct = rest % n_ct;
    const int64_t m = rest / n_ct;
    const int64_t r0 = rt * kTileR, c0 = ct * (kSwb ? 32 : kTileC);
    // output column of transposed tile row cl
    auto out_col = [&](int cl) -> int64_t { return kSwb ? (cl < 32 ? c0 + cl : f + c0 + (cl - 32)) : c0 + cl; };

    // phase 1: load, (NVFP4: e2m1 * e4m3 in f16), store transposed
    {
        const int rl = threadIdx.x & (kTileR - 1);
        const int half = threadIdx.x >> 7;
        const int64_t r = r0 + rl;
        const int64_t c = out_col(half * 32);
        uint32_t h[16];  // 32 16-bit values, element 2i in the low half of h[i]
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
                const uint32_t words[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const __half2 sfh = *reinterpret_cast<const __half2 *>(q < 2 ? &sfa2 : &sfb2);
#pragma unroll
                    for (int b2 = 0; b2 < 4; ++b2) {
                        uint32_t e2 = e2m1x2_to_h2(words[q] >> (8 * b2));
                        const __half2 es = __hmul2(*reinterpret_cast<const __half2 *>(&e2), sfh);
                        h[4 * q + b2] = *reinterpret_cast<const uint32_t *>(&es);
                    }
                }
            } else if constexpr (kSwb) {
                // 16 gate/up column pairs per thread (one s per pair): dg = (dh * u) * s * (1 + g *
                // (1 - s)) and du = dh * (g * s), s = 1 / (1 + exp(-g)), each step one binary32
                // rounding, then bf16; dg to tile rows half*16 + i, du to rows 32 + half*16 + i
                const int64_t j0 = c0 + half * 16;
                const float4 *gp = reinterpret_cast<const float4 *>(gu + r * 2 * f + j0);
                const float4 *upp = reinterpret_cast<const float4 *>(gu + r * 2 * f + f + j0);
                const float4 *dp = reinterpret_cast<const float4 *>(dh + r * f + j0);
#pragma unroll 2
                for (int k4 = 0; k4 < 4; ++k4) {
                    const float4 g4 = __ldg(gp + k4), u4 = __ldg(upp + k4), d4 = __ldg(dp + k4);
                    const float gs[4] = {g4.x, g4.y, g4.z, g4.w}, us[4] = {u4.x, u4.y, u4.z, u4.w};
                    const float ds[4] = {d4.x, d4.y, d4.z, d4.w};
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float sg = __fdiv_rn(1.0f, __fadd_rn(1.0f, expf(-gs[i])));
                        const float dsilu = __fmul_rn(sg, __fadd_rn(1.0f, __fmul_rn(gs[i], __fsub_rn(1.0f, sg))));
                        const float dgv = __fmul_rn(__fmul_rn(ds[i], us[i]), dsilu);
                        const float duv = __fmul_rn(ds[i], __fmul_rn(gs[i], sg));
                        tile[half * 16 + 4 * k4 + i][rl] = f32_to_bf16_bits(dgv);
                        tile[32 + half * 16 + 4 * k4 + i][rl] = f32_to_bf16_bits(duv);
                    }
                }
            } else if constexpr (kind == SrcKind::CombineBwd) {
                const int32_t tok = __ldg(src_of + r);
                float wj = 0.0f;
                if (tok >= 0)
                    for (int j = 0; j < topk; ++j)
                        if (__ldg(row_of + (int64_t)tok * topk + j) == (int32_t)r) wj = __ldg(wts + (int64_t)tok * topk + j);
                const uint4 *src = reinterpret_cast<const uint4 *>(xbf + (int64_t)(tok < 0 ? 0 : tok) * C + c);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const uint4 w = tok >= 0 ? __ldg(src + q) : make_uint4(0, 0, 0, 0);
                    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        h[4 * q + i] = (uint32_t)f32_to_bf16_bits(__fmul_rn(wj, bf16_lo(ws[i]))) |
                                       ((uint32_t)f32_to_bf16_bits(__fmul_rn(wj, bf16_hi(ws[i]))) << 16);
                }
                if constexpr (kRow) {
                    float v[32];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        v[2 * i] = bf16_lo(h[i]);
                        v[2 * i + 1] = bf16_hi(h[i]);
                    }
                    emit_rowwise32(v, r, c, C, q_r, e8_r);
                }
            } else {
                const uint4 *src = reinterpret_cast<const uint4 *>(xbf + (m * R + r) * C + c);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const uint4 w = __ldg(src + q);
                    h[4 * q] = w.x;
                    h[4 * q + 1] = w.y;
                    h[4 * q + 2] = w.z;
                    h[4 * q + 3] = w.w;
                }
                if constexpr (kRow) {
                    float v[32];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        v[2 * i] = bf16_lo(h[i]);
                        v[2 * i + 1] = bf16_hi(h[i]);
                    }
                    emit_rowwise32(v, r, c, C, q_r, e8_r);
                }
            }
        } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) h[i] = 0u;
            if constexpr (kSwb) {
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    tile[half * 16 + i][rl] = 0;
                    tile[32 + half * 16 + i][rl] = 0;
                }
            }
        }
        if constexpr (!kSwb) {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                tile[half * 32 + 2 * i][rl] = (uint16_t)(h[i] & 0xFFFFu);
                tile[half * 32 + 2 * i + 1][rl] = (uint16_t)(h[i] >> 16);
            }
        }
    }
    __syncthreads();
    if constexpr (kSwb && kRow) {
        // the row-wise MXFP8 block of row r: gate columns (half 0) or up columns (half 1), read
        // back from one column of the transposed tile
        const int rl = threadIdx.x & (kTileR - 1);
        const int half = threadIdx.x >> 7;
        const int64_t r = r0 + rl;
        if (r < R) {
            float v[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = __uint_as_float((uint32_t)tile[half * 32 + i][rl] << 16);
            emit_rowwise32(v, r, out_col(half * 32), C, q_r, e8_r);
        }
    }

    // phase 2: each warp emits two output rows per iteration (lanes 0-15 and 16-31)
    const float g = (kind == SrcKind::Nvfp4) ? __ldg(g_dec + m) : 1.0f;
    const int lane = lane_id();
    const int sub = lane & 15;
#pragma unroll 1
    for (int i = 0; i < kTileC / 16; ++i) {
        const int cl = warp_id() + 16 * i + 8 * (lane >> 4);
        const uint4 p = *reinterpret_cast<const uint4 *>(&tile[cl][sub * 8]);
        const uint32_t pw[4] = {p.x, p.y, p.z, p.w};
        float x[8];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            if constexpr (kind == SrcKind::Nvfp4) {
                const float2 f = h2_bits_to_f2(pw[k]);
                f2_unpack(f2_mul(f2_pack(f.x, f.y), f2_pack(g, g)), x[2 * k], x[2 * k + 1]);
            } else {
                x[2 * k] = bf16_lo(pw[k]);
                x[2 * k + 1] = bf16_hi(pw[k]);
            }
        }
        const int64_t c = out_col(cl);
        emit8<kSR>(x, c < C, m, c, r0, R, C, q_t, e8_t, keys, stream_id);
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
    MOE4_CHECK_ARG(aligned16(codes) && aligned16(q_t) && (reinterpret_cast<uintptr_t>(sf) & 1u) == 0);
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
        MOE4_CHECK_ARG(rows % 32 == 0 && aligned16(x) && aligned16(q));
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
    MOE4_CHECK_ARG(aligned16(x) && aligned16(q_row) && aligned16(q_col));
    const int64_t tiles = ((rows + kTileR - 1) / kTileR) * ((cols + kTileC - 1) / kTileC);
    if (tiles == 0) return MOE4_OK;
    MOE4_CHECK_ARG(tiles < (int64_t(1) << 31));
    requant_transpose_kernel<SrcKind::Bf16, false, true><<<(unsigned)tiles, 256, 0, as_stream(stream)>>>(
        nullptr, nullptr, nullptr, x, 1, rows, cols, q_col, e8_col, philox_keys(0), 0u, false, q_row, e8_row);
    return launch_status();
}

extern "C" int moe4_swiglu_backward_mxfp8(const float *gu, const float *dh, int64_t rows, int64_t f, uint8_t *q_row,
                                          uint8_t *e8_row, uint8_t *q_col, uint8_t *e8_col, uint32_t flags,
                                          void *stream) {
    MOE4_CHECK_ARG(rows >= 0 && rows % 32 == 0 && f > 0 && f % 32 == 0 && flags == 0);
    MOE4_CHECK_ARG(q_row && e8_row && q_col && e8_col && (rows == 0 || (gu && dh)));
    MOE4_CHECK_ARG(aligned16(gu) && aligned16(dh) && aligned16(q_row) && aligned16(q_col));
    const int64_t tiles = ((rows + kTileR - 1) / kTileR) * (f / 32);
    if (tiles == 0) return MOE4_OK;
    MOE4_CHECK_ARG(tiles < (int64_t(1) << 31));
    requant_transpose_kernel<SrcKind::SwigluBwd, false, true><<<(unsigned)tiles, 256, 0, as_stream(stream)>>>(
        nullptr, nullptr, nullptr, nullptr, 1, rows, 2 * f, q_col, e8_col, philox_keys(0), 0u, false, q_row, e8_row, gu,
        dh);
    return launch_status();
}

extern "C" int moe4_combine_backward_mxfp8(const uint16_t *dy, const int32_t *row_of, const float *w,
                                           const int32_t *src_of, int64_t T, int64_t k, int64_t d, int64_t rows_total,
                                           uint8_t *q_row, uint8_t *e8_row, uint8_t *q_col, uint8_t *e8_col,
                                           uint32_t flags, void *stream) {
    MOE4_CHECK_ARG(T >= 0 && k >= 1 && k <= 32 && d > 0 && d % 32 == 0 && rows_total >= 0 && rows_total % 32 == 0);
    MOE4_CHECK_ARG(flags == 0 && src_of && q_row && e8_row && q_col && e8_col);
    MOE4_CHECK_ARG(T == 0 || (dy && row_of && w && aligned16(dy)));
    MOE4_CHECK_ARG(aligned16(q_row) && aligned16(q_col));
    const int64_t tiles = ((rows_total + kTileR - 1) / kTileR) * ((d + kTileC - 1) / kTileC);
    if (tiles == 0) return MOE4_OK;
    MOE4_CHECK_ARG(tiles < (int64_t(1) << 31));
    requant_transpose_kernel<SrcKind::CombineBwd, false, true><<<(unsigned)tiles, 256, 0, as_stream(stream)>>>(
        nullptr, nullptr, nullptr, dy, 1, rows_total, d, q_col, e8_col, philox_keys(0), 0u, false, q_row, e8_row,
        nullptr, nullptr, src_of, row_of, w, (int)k);
    return launch_status();
}
