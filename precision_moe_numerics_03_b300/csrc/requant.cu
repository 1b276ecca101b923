// requant.cu -- dequantise -> transpose -> MXFP8 requantisation with stochastic rounding, and the
// MXFP8 quantisation of bf16 tensors (row-wise or transposed).
//
// Method: "4-bit computation from the start of Inkling 2 Small's pretraining" (lhc.media),
// backward-pass paragraphs: the forward operands are dequantised, transposed at higher precision
// and requantised into MXFP8 with stochastic rounding, which picks the upper or lower neighbour
// with probability given by the distance so that the value is kept on average.
//
// Tile: 128 input rows (the output's contiguous dimension) x 64 input columns (128 for the
// two-layout quantisers of bf16 sources, and for the stochastic rounding of NVFP4 sources whose
// column count is a multiple of 128: twice the work per barrier and per scale-range reduction).
// Phase 1: each thread reads one row's 32 values (16 code
// bytes and two scale bytes, or 64 bytes of bf16; two such groups on a 128-column tile) and
// stores them as 16 column pairs, one 32-bit word each, in the transposed shared tile.  Phase 2:
// each warp emits two output rows (one column pair) of 128 values: lane l owns 4 consecutive
// values of each (two lanes share the Philox calls that give their 16-bit numbers), 8 lanes form
// one 32-block.
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

// Output of one warp: 128 values of each of the output rows cA and cA + 1 (the input columns of
// one pair-row of the tile, word p = {column cA, column cA + 1} as 16-bit halves).  Lane l owns
// input rows 4l .. 4l+3 of both; lanes 8b .. 8b+7 form 32-block b, whose amax is taken on the
// packed 16-bit pairs (the binary32 values are monotone in them: an NVFP4 source is scaled by
// g > 0 with one rounding, a bf16 source converts exactly).  Every lane takes part in the
// shuffles; `live` only guards the stores.  The scale codes go to e8s[cl], e8s[cl + 1] (the
// tile's 64 output rows x 4 blocks), written out once per tile.
template <SrcKind kind, bool kSR, bool kJ32>
__device__ __forceinline__ void emit_pair(const uint4 p, float g, bool live, int64_t m, int64_t cA, int64_t r0,
                                          int64_t R, int64_t C, uint8_t *__restrict__ q_t, uint8_t (*e8s)[4], int cl,
                                          const PhiloxKeys keys, uint32_t stream_id, bool safe, int64_t mr) {
    constexpr bool kF16 = kind == SrcKind::Nvfp4;
    const int lane = lane_id();
    uint32_t mx = max_abs16x2<kF16>(max_abs16x2<kF16>(p.x, p.y), max_abs16x2<kF16>(p.z, p.w));
    mx = max_abs16x2<kF16>(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 1));
    mx = max_abs16x2<kF16>(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 2));
    mx = max_abs16x2<kF16>(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 4));
    const uint32_t w[4] = {p.x, p.y, p.z, p.w};
    float xa[4], xb[4], aA, aB;
    if constexpr (kF16) {
        const float2 am = h2_bits_to_f2(mx);
        aA = __fmul_rn(fabsf(am.x), g);
        aB = __fmul_rn(fabsf(am.y), g);
        const uint64_t g2 = f2_pack(g, g);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float2 f = h2_bits_to_f2(w[k]);
            f2_unpack(f2_mul(f2_pack(f.x, f.y), g2), xa[k], xb[k]);
        }
    } else {
        aA = fabsf(bf16_lo(mx));
        aB = fabsf(bf16_hi(mx));
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            xa[k] = bf16_lo(w[k]);
            xb[k] = bf16_hi(w[k]);
        }
    }
    const uint32_t fA = mx_scale_fs(aA), fB = mx_scale_fs(aB);
    const uint64_t s2 = f2_pack(mx_inv_scale_fs(fA), mx_inv_scale_fs(fB));
    float va[4], vb[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) f2_unpack(f2_mul(f2_pack(xa[k], xb[k]), s2), va[k], vb[k]);
    const int64_t rowA = m * C + cA;  // output row in the [nmat * C, R] view
    const int64_t idx = rowA * R + r0 + 4 * lane;
    uint32_t qa, qb;
    if constexpr (kSR) {
        // the 16-bit numbers of this lane's values: indices idx .. idx+3 (row A) and idx+R ..
        // idx+R+3 (row B), with idx % 8 = 4 * (lane & 1) (R and r0 are multiples of 32); lanes 2m
        // and 2m+1 share one Philox call per row, so the even lane runs row A's call, the odd lane
        // row B's, and each hands its partner the two words of the partner's half.  The random
        // index counts matrices from mr's origin (mr = m plus the call's matrix base), so a call
        // over a slice of a weight stack draws the numbers of the whole stack's call.
        const bool odd = (lane & 1) != 0;
        const int64_t i8 = (mr * C + cA) * R + r0 + 8 * (lane >> 1) + (odd ? R : 0);
        Philox4 P;
        if constexpr (kJ32)
            P = sr_words8_not32((uint32_t)((uint64_t)i8 >> 3), stream_id, keys);
        else
            P = sr_words8_not((uint64_t)i8 >> 3, stream_id, keys);
        const uint32_t g0 = __shfl_xor_sync(0xFFFFFFFFu, odd ? P.x : P.z, 1);
        const uint32_t g1 = __shfl_xor_sync(0xFFFFFFFFu, odd ? P.y : P.w, 1);
        const uint32_t a01 = odd ? g0 : P.x, a23 = odd ? g1 : P.y;
        const uint32_t b01 = odd ? P.z : g0, b23 = odd ? P.w : g1;
        if (safe) {  // the tile's scales rule out non-zero values below 2^-6 (see the kernel)
            qa = e4m3x4_sr_fast(va[0], va[1], va[2], va[3], a01, a23);
            qb = e4m3x4_sr_fast(vb[0], vb[1], vb[2], vb[3], b01, b23);
        } else if (min(sr_fast_key4(va[0], va[1], va[2], va[3]), sr_fast_key4(vb[0], vb[1], vb[2], vb[3])) >=
                   kSrFastMin) {  // one test for the eight values (the per-element path is rare)
            qa = e4m3x4_sr_fast(va[0], va[1], va[2], va[3], a01, a23);
            qb = e4m3x4_sr_fast(vb[0], vb[1], vb[2], vb[3], b01, b23);
        } else {
            qa = e4m3x4_sr_nw(va[0], va[1], va[2], va[3], a01, a23);
            qb = e4m3x4_sr_nw(vb[0], vb[1], vb[2], vb[3], b01, b23);
        }
    } else {
        qa = e4m3x4_rn(va[0], va[1], va[2], va[3]);
        qb = e4m3x4_rn(vb[0], vb[1], vb[2], vb[3]);
    }
    if (live && r0 + 4 * lane < R) {
        *reinterpret_cast<uint32_t *>(q_t + idx) = qa;
        *reinterpret_cast<uint32_t *>(q_t + idx + R) = qb;
        if ((lane & 7) == 0) {  // the tile's scale codes, stored after the loop
            e8s[cl][lane >> 3] = (uint8_t)(fA - 8u);
            e8s[cl + 1][lane >> 3] = (uint8_t)(fB - 8u);
        }
    }
}

// The row-wise MXFP8 of the 32 bf16 values a thread holds in phase 1 (one block along the row,
// h[i] = elements 2i, 2i+1), nearest-even: written to q_r [R, C] and e8_r [R, C/32] (canonical or
// tile layout) when the kernel also emits that layout.  The amax is taken on the packed pairs.
__device__ __forceinline__ void emit_rowwise32(const uint32_t h[16], int64_t r, int64_t c, int64_t C,
                                               uint8_t *__restrict__ q_r, uint8_t *__restrict__ e8_r, bool e8_mma) {
    uint32_t mx = max_abs16x2<false>(h[0], h[1]);
#pragma unroll
    for (int i = 2; i < 16; ++i) mx = max_abs16x2<false>(mx, h[i]);
    const uint32_t fs = mx_scale_fs(fmaxf(fabsf(bf16_lo(mx)), fabsf(bf16_hi(mx))));
    const float s = mx_inv_scale_fs(fs);
    const uint64_t s2 = f2_pack(s, s);
    uint32_t w[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        float v0, v1, v2, v3;
        f2_unpack(f2_mul(f2_pack(bf16_lo(h[2 * j]), bf16_hi(h[2 * j])), s2), v0, v1);
        f2_unpack(f2_mul(f2_pack(bf16_lo(h[2 * j + 1]), bf16_hi(h[2 * j + 1])), s2), v2, v3);
        w[j] = e4m3x4_rn(v0, v1, v2, v3);
    }
    uint4 *dst = reinterpret_cast<uint4 *>(q_r + r * C + c);
    dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
    dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
    e8_r[sf_offset(r, c / 32, C / 32, e8_mma)] = (uint8_t)(fs - 8u);
}

// Shared tile: 32 pair-rows x 128 input rows of 32-bit words; word [p][r] holds input columns
// 2p (low half) and 2p + 1 (high half) of input row r as 16-bit values.  An NVFP4 source stores
// e2m1 * e4m3 as f16 (at most 6 significant bits: exact) and the binary32 product with g_dec is
// formed when the value is read back, the same single rounding; a bf16 source stores its bits.
// Phase 1 writes one word per pair (consecutive rows across a warp), phase 2 reads 16 bytes per
// lane (512 contiguous bytes per warp): both conflict-free.
constexpr int kPairs = kTileC / 2;

// TC: tile columns, 64, or 128 for the bf16 and combine-gradient sources (each thread then
// holds two 32-column groups of its row, all eight 16-byte loads issued before any is used:
// twice the bytes in flight of the 64-column tile, for kernels that wait on their loads).
template <SrcKind kind, bool kSR, bool kRow = false, bool kJ32 = true, int TC = kTileC>
__global__ void __launch_bounds__(256, (kSR || kind == SrcKind::SwigluBwd || TC == 128) ? 4 : 5)
requant_transpose_kernel(
    const uint8_t *__restrict__ codes, const uint8_t *__restrict__ sf, const float *__restrict__ g_dec,
    const uint16_t *__restrict__ xbf, int64_t nmat, int64_t R, int64_t C, uint8_t *__restrict__ q_t,
    uint8_t *__restrict__ e8_t, const PhiloxKeys keys, uint32_t stream_id, bool sf_mma,
    uint8_t *__restrict__ q_r = nullptr, uint8_t *__restrict__ e8_r = nullptr, const float *__restrict__ gu = nullptr,
    const float *__restrict__ dh = nullptr, const int32_t *__restrict__ src_of = nullptr,
    const int32_t *__restrict__ row_of = nullptr, const float *__restrict__ wts = nullptr, int topk = 0,
    bool e8_mma = false, const int32_t *__restrict__ skip_offs = nullptr, int64_t m_base = 0) {
    constexpr bool kSwb = kind == SrcKind::SwigluBwd;
    static_assert(TC == 64 || (TC == 128 && kind != SrcKind::SwigluBwd),
                  "128-column tiles: NVFP4, bf16 and combine-gradient sources");
    // expert weights: a matrix whose group has no rows (skip_offs[m + 1] == skip_offs[m]) is
    // skipped whole, its outputs left as they are
    if (skip_offs != nullptr && __ldg(skip_offs + blockIdx.z + 1) == __ldg(skip_offs + blockIdx.z)) return;
    __shared__ __align__(16) uint32_t tile[TC / 2][kTileR];
    __shared__ __align__(4) uint8_t e8s[TC][4];
    const int64_t f = C / 2;  // SwigluBwd: C = 2f
    // grid (row tiles, column tiles, matrices): no index division
    const int64_t m = blockIdx.z;
    const int64_t r0 = (int64_t)blockIdx.x * kTileR, c0 = (int64_t)blockIdx.y * (kSwb ? 32 : TC);
    // input column (output row) of tile column cl
    auto out_col = [&](int cl) -> int64_t { return kSwb ? (cl < 32 ? c0 + cl : f + c0 + (cl - 32)) : c0 + cl; };

    // NVFP4 source with stochastic rounding: the smallest non-zero and the largest block scale of
    // the tile (f16 bits), reduced over the CTA (see `safe` below)
    constexpr bool kScaleRange = kSR && kind == SrcKind::Nvfp4;
    __shared__ uint32_t sf_red[2][8];
    uint32_t sf_lo = 0x7C00u, sf_hi = 0u;
    // phase 1: load, (NVFP4: e2m1 * e4m3 in f16), store transposed
    if constexpr (TC == 128) {
        // thread (row rl, half): tile columns 32 * half + 64 * g, g = 0, 1 -> pair-rows
        // 16 * half + 32 * g + i; the values are those of the 64-column path below
        const int rl = threadIdx.x & (kTileR - 1);
        const int half = threadIdx.x >> 7;
        const int64_t r = r0 + rl;
        if constexpr (kind == SrcKind::Nvfp4) {
            // both groups' code words and scale pairs are loaded before either is used
            const int64_t nblk = C / 16;
            uint4 wq[2];
            uint16_t sq[2];
#pragma unroll
            for (int g = 0; g < 2; ++g) {
                const int64_t c = c0 + 32 * half + 64 * g, b = c / 16;
                const bool ld = r < R && c < C;
                const int64_t soff = sf_mma ? m * R * nblk + ((r >> 7) * (nblk >> 2) + (b >> 2)) * 512 +
                                                  (r & 31) * 16 + ((r >> 5) & 3) * 4 + (b & 3)
                                            : (m * R + r) * nblk + b;
                wq[g] = ld ? __ldg(reinterpret_cast<const uint4 *>(codes + ((m * R + r) * C + c) / 2))
                           : make_uint4(0, 0, 0, 0);
                sq[g] = ld ? __ldg(reinterpret_cast<const uint16_t *>(sf + soff)) : (uint16_t)0;
            }
#pragma unroll
            for (int g = 0; g < 2; ++g) {
                const int64_t c = c0 + 32 * half + 64 * g;
                uint32_t h[16];
                if (r < R && c < C) {
                    const uint32_t sf2 = e4m3x2_to_h2(sq[g]);
                    const uint32_t sfa2 = __byte_perm(sf2, 0, 0x1010), sfb2 = __byte_perm(sf2, 0, 0x3232);
                    if constexpr (kScaleRange) {
                        const uint32_t sa = sf2 & 0xFFFFu, sb = sf2 >> 16;
                        sf_lo = min(sf_lo, min(sa ? sa : 0x7C00u, sb ? sb : 0x7C00u));
                        sf_hi = max(sf_hi, max(sa, sb));
                    }
                    const uint32_t words[4] = {wq[g].x, wq[g].y, wq[g].z, wq[g].w};
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const __half2 sfh = *reinterpret_cast<const __half2 *>(q < 2 ? &sfa2 : &sfb2);
                        uint32_t e2[4];
                        e2m1x8_to_h2x4(words[q], e2);
#pragma unroll
                        for (int b2 = 0; b2 < 4; ++b2) {
                            const __half2 es = __hmul2(*reinterpret_cast<const __half2 *>(&e2[b2]), sfh);
                            h[4 * q + b2] = *reinterpret_cast<const uint32_t *>(&es);
                        }
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < 16; ++i) h[i] = 0u;
                }
#pragma unroll
                for (int i = 0; i < 16; ++i) tile[16 * half + 32 * g + i][rl] = h[i];
            }
        } else {
        int32_t tok = 0;
        float wj = 0.0f;
        if constexpr (kind == SrcKind::CombineBwd) {
            if (r < R) {
                tok = __ldg(src_of + r);
                if (tok >= 0) {
                    const int64_t base = (int64_t)tok * topk;
                    const bool vec = (topk & 3) == 0 &&
                                     ((reinterpret_cast<uintptr_t>(row_of) | reinterpret_cast<uintptr_t>(wts)) & 15u) == 0;
                    if (vec) {
                        for (int j = 0; j < topk; j += 4) {
                            const int4 ro = __ldg(reinterpret_cast<const int4 *>(row_of + base + j));
                            const float4 wv = __ldg(reinterpret_cast<const float4 *>(wts + base + j));
                            wj = ro.x == (int32_t)r ? wv.x : wj;
                            wj = ro.y == (int32_t)r ? wv.y : wj;
                            wj = ro.z == (int32_t)r ? wv.z : wj;
                            wj = ro.w == (int32_t)r ? wv.w : wj;
                        }
                    } else {
                        for (int j = 0; j < topk; ++j)
                            if (__ldg(row_of + base + j) == (int32_t)r) wj = __ldg(wts + base + j);
                    }
                }
            }
        }
        uint4 v[2][4];
#pragma unroll
        for (int g = 0; g < 2; ++g) {
            const int64_t c = c0 + 32 * half + 64 * g;
            const bool ld = r < R && c < C && (kind != SrcKind::CombineBwd || tok >= 0);
            const uint4 *src = reinterpret_cast<const uint4 *>(
                kind == SrcKind::CombineBwd ? xbf + (int64_t)(tok < 0 ? 0 : tok) * C + c : xbf + (m * R + r) * C + c);
#pragma unroll
            for (int q = 0; q < 4; ++q) v[g][q] = ld ? __ldg(src + q) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int g = 0; g < 2; ++g) {
            const int64_t c = c0 + 32 * half + 64 * g;
            uint32_t h[16];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const uint32_t ws[4] = {v[g][q].x, v[g][q].y, v[g][q].z, v[g][q].w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    if constexpr (kind == SrcKind::CombineBwd)
                        h[4 * q + i] = (uint32_t)f32_to_bf16_bits(__fmul_rn(wj, bf16_lo(ws[i]))) |
                                       ((uint32_t)f32_to_bf16_bits(__fmul_rn(wj, bf16_hi(ws[i]))) << 16);
                    else
                        h[4 * q + i] = ws[i];
                }
            }
            const bool in = r < R && c < C;
            if (!in) {
#pragma unroll
                for (int i = 0; i < 16; ++i) h[i] = 0u;
            }
            if constexpr (kRow) {
                if (in) emit_rowwise32(h, r, c, C, q_r, e8_r, e8_mma);
            }
#pragma unroll
            for (int i = 0; i < 16; ++i) tile[16 * half + 32 * g + i][rl] = h[i];
        }
        }
    } else {
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
                if constexpr (kScaleRange) {
                    const uint32_t sa = sf2 & 0xFFFFu, sb = sf2 >> 16;
                    sf_lo = min(sa ? sa : 0x7C00u, sb ? sb : 0x7C00u);
                    sf_hi = max(sa, sb);
                }
                const uint32_t words[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const __half2 sfh = *reinterpret_cast<const __half2 *>(q < 2 ? &sfa2 : &sfb2);
                    uint32_t e2[4];
                    e2m1x8_to_h2x4(words[q], e2);
#pragma unroll
                    for (int b2 = 0; b2 < 4; ++b2) {
                        const __half2 es = __hmul2(*reinterpret_cast<const __half2 *>(&e2[b2]), sfh);
                        h[4 * q + b2] = *reinterpret_cast<const uint32_t *>(&es);
                    }
                }
            } else if constexpr (kSwb) {
                // 16 gate/up column pairs per thread (one s per pair): dg = (dh * u) * s * (1 + g *
                // (1 - s)) and du = dh * (g * s), s = 1 / (1 + exp(-g)), each step one binary32
                // rounding, then bf16; gate column c0 + half*16 + i goes to pair-row half*8 + i/2,
                // its up partner to pair-row 16 + half*8 + i/2
                const int64_t j0 = c0 + half * 16;
                const float4 *gp = reinterpret_cast<const float4 *>(gu + r * 2 * f + j0);
                const float4 *upp = reinterpret_cast<const float4 *>(gu + r * 2 * f + f + j0);
                const float4 *dp = reinterpret_cast<const float4 *>(dh + r * f + j0);
#pragma unroll 2
                for (int k4 = 0; k4 < 4; ++k4) {
                    const float4 g4 = __ldg(gp + k4), u4 = __ldg(upp + k4), d4 = __ldg(dp + k4);
                    const float gs[4] = {g4.x, g4.y, g4.z, g4.w}, us[4] = {u4.x, u4.y, u4.z, u4.w};
                    const float ds[4] = {d4.x, d4.y, d4.z, d4.w};
                    uint32_t dgb[4], dub[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float sg = __frcp_rn(__fadd_rn(1.0f, expf(-gs[i])));
                        const float dsilu = __fmul_rn(sg, __fadd_rn(1.0f, __fmul_rn(gs[i], __fsub_rn(1.0f, sg))));
                        const float dgv = __fmul_rn(__fmul_rn(ds[i], us[i]), dsilu);
                        const float duv = __fmul_rn(ds[i], __fmul_rn(gs[i], sg));
                        dgb[i] = f32_to_bf16_bits(dgv);
                        dub[i] = f32_to_bf16_bits(duv);
                    }
                    tile[half * 8 + 2 * k4][rl] = dgb[0] | (dgb[1] << 16);
                    tile[half * 8 + 2 * k4 + 1][rl] = dgb[2] | (dgb[3] << 16);
                    tile[16 + half * 8 + 2 * k4][rl] = dub[0] | (dub[1] << 16);
                    tile[16 + half * 8 + 2 * k4 + 1][rl] = dub[2] | (dub[3] << 16);
                }
            } else if constexpr (kind == SrcKind::CombineBwd) {
                const int32_t tok = __ldg(src_of + r);
                float wj = 0.0f;
                if (tok >= 0) {
                    // the routing slot of row r: its k row indices and weights are loaded together
                    // (16-byte loads when k % 4 == 0 and both arrays are 16-byte aligned), so the
                    // dy loads below wait on src_of only
                    const int64_t base = (int64_t)tok * topk;
                    const bool vec = (topk & 3) == 0 &&
                                     ((reinterpret_cast<uintptr_t>(row_of) | reinterpret_cast<uintptr_t>(wts)) & 15u) == 0;
                    if (vec) {
                        for (int j = 0; j < topk; j += 4) {
                            const int4 ro = __ldg(reinterpret_cast<const int4 *>(row_of + base + j));
                            const float4 wv = __ldg(reinterpret_cast<const float4 *>(wts + base + j));
                            wj = ro.x == (int32_t)r ? wv.x : wj;
                            wj = ro.y == (int32_t)r ? wv.y : wj;
                            wj = ro.z == (int32_t)r ? wv.z : wj;
                            wj = ro.w == (int32_t)r ? wv.w : wj;
                        }
                    } else {
                        for (int j = 0; j < topk; ++j)
                            if (__ldg(row_of + base + j) == (int32_t)r) wj = __ldg(wts + base + j);
                    }
                }
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
                if constexpr (kRow) emit_rowwise32(h, r, c, C, q_r, e8_r, e8_mma);
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
                if constexpr (kRow) emit_rowwise32(h, r, c, C, q_r, e8_r, e8_mma);
            }
        } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) h[i] = 0u;
            if constexpr (kSwb) {
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    tile[half * 8 + i][rl] = 0u;
                    tile[16 + half * 8 + i][rl] = 0u;
                }
            }
        }
        if constexpr (!kSwb) {
#pragma unroll
            for (int i = 0; i < 16; ++i) tile[half * 16 + i][rl] = h[i];
        }
    }
    if constexpr (kScaleRange) {
        sf_lo = __reduce_min_sync(0xFFFFFFFFu, sf_lo);
        sf_hi = __reduce_max_sync(0xFFFFFFFFu, sf_hi);
        if (lane_id() == 0) {
            sf_red[0][warp_id()] = sf_lo;
            sf_red[1][warp_id()] = sf_hi;
        }
    }
    __syncthreads();
    // safe: every non-zero value of the tile reaches at least 2^-6 after the MXFP8 scaling, so
    // the stochastic rounding needs no per-value test.  A non-zero value is e*sf with |e| >= 1/2,
    // and each 32-block's amax is at most 6 * sf_max * g (to within one rounding), so with
    // 2^-e > 224 / amax a value lands at |v| >= (sf_min / sf_max) * (112 / 6) * (1 - 2^-23), which
    // is above 2^-6 for sf_max <= 1024 * sf_min; 0.5 * sf_min * g >= 2^-100 keeps every product
    // normal and the scale exponent unclamped.  An all-zero tile is safe too.
    bool safe = false;
    if constexpr (kScaleRange) {
        const int ln = lane_id();
        const uint32_t lo = __reduce_min_sync(0xFFFFFFFFu, ln < 8 ? sf_red[0][ln] : 0x7C00u);
        const uint32_t hi = __reduce_max_sync(0xFFFFFFFFu, ln < 8 ? sf_red[1][ln] : 0u);
        const float lo_f = __half2float(__ushort_as_half((unsigned short)lo));
        const float hi_f = __half2float(__ushort_as_half((unsigned short)hi));
        const float gd = __ldg(g_dec + m);
        safe = lo == 0x7C00u || (hi_f <= lo_f * 1024.0f && 0.5f * lo_f * gd >= 0x1p-100f);
    }
    if constexpr (kSwb && kRow) {
        // the row-wise MXFP8 block of row r: gate columns (half 0) or up columns (half 1), read
        // back from one column of the transposed tile
        const int rl = threadIdx.x & (kTileR - 1);
        const int half = threadIdx.x >> 7;
        const int64_t r = r0 + rl;
        if (r < R) {
            uint32_t hw[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) hw[i] = tile[half * 16 + i][rl];
            emit_rowwise32(hw, r, out_col(half * 32), C, q_r, e8_r, e8_mma);
        }
    }

    // phase 2: each warp emits one pair-row (two output rows) per iteration
    const float g = (kind == SrcKind::Nvfp4) ? __ldg(g_dec + m) : 1.0f;
#pragma unroll 1
    for (int i = 0; i < TC / 16; ++i) {
        const int cp = warp_id() + 8 * i;
        const uint4 p = *reinterpret_cast<const uint4 *>(&tile[cp][4 * lane_id()]);
        const int64_t cA = out_col(2 * cp);
        emit_pair<kind, kSR, kJ32>(p, g, cA < C, m, cA, r0, R, C, q_t, e8s, 2 * cp, keys, stream_id, safe,
                                   m + m_base);
    }
    // scale codes: one thread per output row, its (up to) four blocks of this tile; the four are
    // adjacent bytes in both layouts (a whole word when R % 128 == 0)
    __syncthreads();
    if (threadIdx.x < TC) {
        const int cl = threadIdx.x;
        const int64_t c = out_col(cl);
        if (c < C) {
            const int64_t row = m * C + c, nkb = R / 32, kb0 = r0 >> 5;
            const int64_t off = sf_offset(row, kb0, nkb, e8_mma);
            const uint32_t word = *reinterpret_cast<const uint32_t *>(e8s[cl]);
            if ((nkb & 3) == 0 && ((reinterpret_cast<uintptr_t>(e8_t) & 3u) == 0)) {
                *reinterpret_cast<uint32_t *>(e8_t + off) = word;
            } else {
                const int nb = nkb - kb0 < 4 ? (int)(nkb - kb0) : 4;
                for (int b = 0; b < nb; ++b) e8_t[off + b] = (uint8_t)(word >> (8 * b));
            }
        }
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
        const uint32_t fs = mx_scale_fs(a);
        const float s = mx_inv_scale_fs(fs);
        const float v0 = __fmul_rn(x4[0], s), v1 = __fmul_rn(x4[1], s);
        const float v2 = __fmul_rn(x4[2], s), v3 = __fmul_rn(x4[3], s);
        uint32_t packed;
        if (sr) {  // indices 4*gidx .. 4*gidx+3: half of Philox call gidx/2 (see sr_words8)
            const Philox4 P = sr_words8_not((uint64_t)gidx >> 1, stream_id, keys);
            packed = (gidx & 1) ? e4m3x4_sr_nw(v0, v1, v2, v3, P.z, P.w) : e4m3x4_sr_nw(v0, v1, v2, v3, P.x, P.y);
        } else {
            packed = e4m3x4_rn(v0, v1, v2, v3);
        }
        if (!live) continue;
        *reinterpret_cast<uint32_t *>(q + gidx * 4) = packed;
        if ((gidx & 7) == 0) e8[gidx >> 3] = (uint8_t)(fs - 8u);
    }
}

// Grid of the transposing kernel: x row tiles, y column tiles, z matrices (rejected beyond the
// launch limits: 2^31 - 1 and 65535).
// tile columns of the two-layout quantisers of bf16 sources (mxfp8_quantize_rowcol and the combine
// gradient): the wide tile, whose threads keep twice the loads in flight
constexpr int kWideTile = 128;

static bool requant_grid(int64_t rows, int64_t col_tiles, int64_t nmat, dim3 &grid) {
    const int64_t rt = (rows + kTileR - 1) / kTileR;
    if (rt >= (int64_t(1) << 31) || col_tiles > 65535 || nmat > 65535) return false;
    grid = dim3((unsigned)rt, (unsigned)col_tiles, (unsigned)nmat);
    return true;
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
    MOE4_CHECK_ARG((flags & ~(MOE4_SR | MOE4_SF_MMA_LAYOUT | MOE4_SF_OUT_MMA)) == 0);
    const bool sf_mma = (flags & MOE4_SF_MMA_LAYOUT) != 0;
    const bool e8_mma = (flags & MOE4_SF_OUT_MMA) != 0;
    MOE4_CHECK_ARG(!sf_mma || (rows % 128 == 0 && cols % 64 == 0));
    MOE4_CHECK_ARG(!e8_mma || (rows % 128 == 0 && cols % 128 == 0));
    dim3 grid;
    MOE4_CHECK_ARG(requant_grid(rows, (cols + kTileC - 1) / kTileC, nmat, grid));
    if (rows == 0) return MOE4_OK;
    // output indices below 2^35: the Philox counter's second word is zero throughout
    const bool j32 = (uint64_t)nmat * (uint64_t)rows * (uint64_t)cols <= (uint64_t(1) << 35);
    const PhiloxKeys keys = philox_keys(seed);
    cudaStream_t st = as_stream(stream);
#define MOE4_REQUANT_ARGS                                                                                        \
    codes, sf, g_dec, nullptr, nmat, rows, cols, q_t, e8_t, keys, stream_id, sf_mma, nullptr, nullptr, nullptr, \
        nullptr, nullptr, nullptr, nullptr, 0, e8_mma
    if ((flags & MOE4_SR) && j32 && cols % 128 == 0) {
        dim3 g128 = grid;  // 128-column tiles: half the column tiles
        g128.y = (unsigned)(cols / 128);
        requant_transpose_kernel<SrcKind::Nvfp4, true, false, true, 128><<<g128, 256, 0, st>>>(MOE4_REQUANT_ARGS);
    } else if ((flags & MOE4_SR) && j32)
        requant_transpose_kernel<SrcKind::Nvfp4, true><<<grid, 256, 0, st>>>(MOE4_REQUANT_ARGS);
    else if (flags & MOE4_SR)
        requant_transpose_kernel<SrcKind::Nvfp4, true, false, false><<<grid, 256, 0, st>>>(MOE4_REQUANT_ARGS);
    else
        requant_transpose_kernel<SrcKind::Nvfp4, false><<<grid, 256, 0, st>>>(MOE4_REQUANT_ARGS);
#undef MOE4_REQUANT_ARGS
    return launch_status();
}

// MOE4_SHARE_SMS: quantiser CTAs per SM (72 registers x 256 threads each), leaving the rest of the
// register file to two requantiser CTAs (56 x 256 on 128-column tiles) launched beside it
constexpr int kShareCtasPerSm = 2;

extern "C" int nvfp4_quantize_f32_requant(const float *x, int64_t nmat, int64_t rows, int64_t cols,
                                          const float *amax_in, uint8_t *codes, uint8_t *sf, float *g_dec,
                                          uint8_t *q_t, uint8_t *e8_t, uint64_t seed, uint32_t stream_id,
                                          int64_t mat_base, const int32_t *group_offs, uint32_t flags, void *stream) {
    MOE4_CHECK_ARG(nmat >= 1 && rows >= 0 && rows % 32 == 0 && cols > 0 && cols % 64 == 0);
    MOE4_CHECK_ARG(mat_base >= 0 && mat_base <= (int64_t(1) << 40));
    MOE4_CHECK_ARG(x && amax_in && codes && sf && g_dec && q_t && e8_t);
    MOE4_CHECK_ARG(aligned16(x) && aligned16(codes) && aligned16(q_t) && (reinterpret_cast<uintptr_t>(sf) & 1u) == 0);
    MOE4_CHECK_ARG((flags & ~(MOE4_FOUR_OVER_SIX | MOE4_SR | MOE4_SF_MMA_LAYOUT | MOE4_SF_OUT_MMA | MOE4_PASS_QUANT |
                              MOE4_PASS_REQUANT | MOE4_SHARE_SMS)) == 0);
    MOE4_CHECK_ARG((flags & (MOE4_PASS_QUANT | MOE4_PASS_REQUANT)) != (MOE4_PASS_QUANT | MOE4_PASS_REQUANT));
    const bool sf_mma = (flags & MOE4_SF_MMA_LAYOUT) != 0;
    const bool e8_mma = (flags & MOE4_SF_OUT_MMA) != 0;
    MOE4_CHECK_ARG(!sf_mma || rows % 128 == 0);
    MOE4_CHECK_ARG(!e8_mma || (rows % 128 == 0 && cols % 128 == 0));
    MOE4_CHECK_ARG(rows * (cols / 16) < (int64_t(1) << 32));
    dim3 grid;
    MOE4_CHECK_ARG(requant_grid(rows, cols / kTileC, nmat, grid));
    if (rows == 0) return MOE4_OK;
    cudaStream_t st = as_stream(stream);
    // two passes over the experts that have rows: the HBM-bound quantiser of the binary32
    // masters, then the issue-bound requantiser of its codes (one fused pass measured slower:
    // its block quantiser and the requantiser share a CTA's issue slots and its barrier)
    if ((flags & MOE4_PASS_REQUANT) == 0) {
        const int rc = quantize_f32_given(x, nmat, rows, cols, amax_in, codes, sf, g_dec, group_offs,
                                          (flags & MOE4_FOUR_OVER_SIX) != 0, sf_mma, st,
                                          (flags & MOE4_SHARE_SMS) ? kShareCtasPerSm : 8);
        if (rc != MOE4_OK) return rc;
        if (flags & MOE4_PASS_QUANT) return MOE4_OK;
    }
    const bool j32 = (uint64_t)(mat_base + nmat) * (uint64_t)rows * (uint64_t)cols <= (uint64_t(1) << 35);
    const PhiloxKeys keys = philox_keys(seed);
#define MOE4_WEIGHT_ARGS                                                                                          \
    codes, sf, g_dec, nullptr, nmat, rows, cols, q_t, e8_t, keys, stream_id, sf_mma, nullptr, nullptr, nullptr, \
        nullptr, nullptr, nullptr, nullptr, 0, e8_mma, group_offs, mat_base
    if ((flags & MOE4_SR) && j32 && cols % 128 == 0) {
        dim3 g128 = grid;  // 128-column tiles: half the column tiles
        g128.y = (unsigned)(cols / 128);
        requant_transpose_kernel<SrcKind::Nvfp4, true, false, true, 128><<<g128, 256, 0, st>>>(MOE4_WEIGHT_ARGS);
    } else if ((flags & MOE4_SR) && j32)
        requant_transpose_kernel<SrcKind::Nvfp4, true><<<grid, 256, 0, st>>>(MOE4_WEIGHT_ARGS);
    else if (flags & MOE4_SR)
        requant_transpose_kernel<SrcKind::Nvfp4, true, false, false><<<grid, 256, 0, st>>>(MOE4_WEIGHT_ARGS);
    else
        requant_transpose_kernel<SrcKind::Nvfp4, false><<<grid, 256, 0, st>>>(MOE4_WEIGHT_ARGS);
#undef MOE4_WEIGHT_ARGS
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
        dim3 grid;
        MOE4_CHECK_ARG(requant_grid(rows, (cols + kTileC - 1) / kTileC, 1, grid));
        if (rows == 0) return MOE4_OK;
        if (sr && (uint64_t)rows * (uint64_t)cols <= (uint64_t(1) << 35))
            requant_transpose_kernel<SrcKind::Bf16, true><<<grid, 256, 0, st>>>(
                nullptr, nullptr, nullptr, x, 1, rows, cols, q, e8, philox_keys(seed), stream_id, false);
        else if (sr)
            requant_transpose_kernel<SrcKind::Bf16, true, false, false><<<grid, 256, 0, st>>>(
                nullptr, nullptr, nullptr, x, 1, rows, cols, q, e8, philox_keys(seed), stream_id, false);
        else
            requant_transpose_kernel<SrcKind::Bf16, false><<<grid, 256, 0, st>>>(
                nullptr, nullptr, nullptr, x, 1, rows, cols, q, e8, philox_keys(seed), stream_id, false);
    }
    return launch_status();
}

extern "C" int mxfp8_quantize_rowcol(const uint16_t *x, int64_t rows, int64_t cols, uint8_t *q_row,
                                     uint8_t *e8_row, uint8_t *q_col, uint8_t *e8_col, uint32_t flags,
                                     void *stream) {
    MOE4_CHECK_ARG(rows >= 0 && rows % 32 == 0 && cols > 0 && cols % 32 == 0 && (flags & ~MOE4_SF_OUT_MMA) == 0);
    MOE4_CHECK_ARG(q_row && e8_row && q_col && e8_col && (rows == 0 || x));
    MOE4_CHECK_ARG(aligned16(x) && aligned16(q_row) && aligned16(q_col));
    const bool e8_mma = (flags & MOE4_SF_OUT_MMA) != 0;
    MOE4_CHECK_ARG(!e8_mma || (rows % 128 == 0 && cols % 128 == 0));
    dim3 grid;
    MOE4_CHECK_ARG(requant_grid(rows, (cols + kWideTile - 1) / kWideTile, 1, grid));
    if (rows == 0) return MOE4_OK;
    requant_transpose_kernel<SrcKind::Bf16, false, true, true, kWideTile><<<grid, 256, 0, as_stream(stream)>>>(
        nullptr, nullptr, nullptr, x, 1, rows, cols, q_col, e8_col, philox_keys(0), 0u, false, q_row, e8_row, nullptr,
        nullptr, nullptr, nullptr, nullptr, 0, e8_mma);
    return launch_status();
}

extern "C" int moe4_swiglu_backward_mxfp8(const float *gu, const float *dh, int64_t rows, int64_t f, uint8_t *q_row,
                                          uint8_t *e8_row, uint8_t *q_col, uint8_t *e8_col, uint32_t flags,
                                          void *stream) {
    MOE4_CHECK_ARG(rows >= 0 && rows % 32 == 0 && f > 0 && f % 32 == 0 && (flags & ~MOE4_SF_OUT_MMA) == 0);
    MOE4_CHECK_ARG(q_row && e8_row && q_col && e8_col && (rows == 0 || (gu && dh)));
    MOE4_CHECK_ARG(aligned16(gu) && aligned16(dh) && aligned16(q_row) && aligned16(q_col));
    const bool e8_mma = (flags & MOE4_SF_OUT_MMA) != 0;
    MOE4_CHECK_ARG(!e8_mma || (rows % 128 == 0 && f % 64 == 0));
    dim3 grid;
    MOE4_CHECK_ARG(requant_grid(rows, f / 32, 1, grid));
    if (rows == 0) return MOE4_OK;
    requant_transpose_kernel<SrcKind::SwigluBwd, false, true><<<grid, 256, 0, as_stream(stream)>>>(
        nullptr, nullptr, nullptr, nullptr, 1, rows, 2 * f, q_col, e8_col, philox_keys(0), 0u, false, q_row, e8_row, gu,
        dh, nullptr, nullptr, nullptr, 0, e8_mma);
    return launch_status();
}

extern "C" int moe4_combine_backward_mxfp8(const uint16_t *dy, const int32_t *row_of, const float *w,
                                           const int32_t *src_of, int64_t T, int64_t k, int64_t d, int64_t rows_total,
                                           uint8_t *q_row, uint8_t *e8_row, uint8_t *q_col, uint8_t *e8_col,
                                           uint32_t flags, void *stream) {
    MOE4_CHECK_ARG(T >= 0 && k >= 1 && k <= 32 && d > 0 && d % 32 == 0 && rows_total >= 0 && rows_total % 32 == 0);
    MOE4_CHECK_ARG((flags & ~MOE4_SF_OUT_MMA) == 0 && src_of && q_row && e8_row && q_col && e8_col);
    MOE4_CHECK_ARG(T == 0 || (dy && row_of && w && aligned16(dy)));
    MOE4_CHECK_ARG(aligned16(q_row) && aligned16(q_col));
    const bool e8_mma = (flags & MOE4_SF_OUT_MMA) != 0;
    MOE4_CHECK_ARG(!e8_mma || (rows_total % 128 == 0 && d % 128 == 0));
    dim3 grid;
    MOE4_CHECK_ARG(requant_grid(rows_total, (d + kWideTile - 1) / kWideTile, 1, grid));
    if (rows_total == 0) return MOE4_OK;
    requant_transpose_kernel<SrcKind::CombineBwd, false, true, true, kWideTile><<<grid, 256, 0, as_stream(stream)>>>(
        nullptr, nullptr, nullptr, dy, 1, rows_total, d, q_col, e8_col, philox_keys(0), 0u, false, q_row, e8_row,
        nullptr, nullptr, src_of, row_of, w, (int)k, e8_mma);
    return launch_status();
}
