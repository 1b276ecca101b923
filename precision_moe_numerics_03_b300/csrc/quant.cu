// quant.cu -- NVFP4 quantisation with Four Over Six, NVFP4 dequantisation, and the Hadamard(128)
// return-path codec.
//
// Method: "4-bit computation from the start of Inkling 2 Small's pretraining" (lhc.media):
// 4-bit values with a scale shared by sixteen values (fewer-bits paragraph); a Hadamard
// transform spreads out extreme values before the return path is quantised (communication
// paragraph).  "Inkling 2 Small's Native 4-Bit Training: Debut and Doubts" (agihunt.info,
// "Confirmed"): Four Over Six chooses between two scaling factors; per-expert scales.
//
// HBM-bound kernels: 16-byte vector loads, one thread per 16-value block (two 16-byte loads, one
// 8-byte code store, one scale byte), grid-stride loops sized to the SM count.
#include <atomic>

#include "common.cuh"

#include <cfloat>

namespace moe4 {

// The current device's SM count, looked up once per device.
int num_sms() {
    static std::atomic<int> cached[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = 0;
    int n = cached[dev].load(std::memory_order_relaxed);
    if (n == 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
        cached[dev].store(n, std::memory_order_relaxed);
    }
    return n;
}

// ------------------------------------------------------------------ amax pass
// Per matrix: max |x| over bf16 values, as binary32 bits (non-negative floats order as unsigned
// integers), folded into amax_bits[m] with one atomicMax per block.
// Eight consecutive values as four bf16 pairs (element 2i in the low half of word i): bf16 input
// as stored, binary32 input rounded to bf16 (nearest-even) first.
template <typename TIn>
__device__ __forceinline__ uint4 load8_bf16(const TIn *p) {
    if constexpr (sizeof(TIn) == 2) {
        return __ldg(reinterpret_cast<const uint4 *>(p));
    } else {
        const float4 a = __ldg(reinterpret_cast<const float4 *>(p)), b = __ldg(reinterpret_cast<const float4 *>(p) + 1);
        return make_uint4(bf16x2_rn(a.x, a.y), bf16x2_rn(a.z, a.w), bf16x2_rn(b.x, b.y), bf16x2_rn(b.z, b.w));
    }
}

template <typename TIn>
__global__ void __launch_bounds__(256) amax_bf16_kernel(const TIn *__restrict__ x, int64_t rows,
                                                        int64_t cols, int64_t ld, int64_t mat_stride,
                                                        unsigned int *__restrict__ amax_bits) {
    const int m = blockIdx.y;
    const TIn *xm = x + (int64_t)m * mat_stride;
    const int64_t vec_per_row = cols / 8;
    const int64_t nvec = rows * vec_per_row;
    uint32_t best = 0;  // two packed bf16 magnitudes
    for (int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; v < nvec;
         v += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = (ld == cols) ? 0 : v / vec_per_row;
        const int64_t c = (ld == cols) ? v * 8 : (v - r * vec_per_row) * 8;
        const uint4 q = load8_bf16(xm + r * ld + c);
        best = __vmaxu2(best, q.x & 0x7FFF7FFFu);
        best = __vmaxu2(best, q.y & 0x7FFF7FFFu);
        best = __vmaxu2(best, q.z & 0x7FFF7FFFu);
        best = __vmaxu2(best, q.w & 0x7FFF7FFFu);
    }
    uint32_t mag = max(best & 0xFFFFu, best >> 16) << 16;
    mag = __reduce_max_sync(0xFFFFFFFFu, mag);
    __shared__ uint32_t part[8];
    if (lane_id() == 0) part[warp_id()] = mag;
    __syncthreads();
    if (threadIdx.x == 0) {
        uint32_t b = 0;
        for (int i = 0; i < (int)(blockDim.x >> 5); ++i) b = max(b, part[i]);
        if (b) atomicMax(amax_bits + m, b);
    }
}

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
        // code 0 has no reciprocal (its blocks take the zero-scale branch); its slot holds -0, the
        // addend of the squared errors' multiply-adds, read from memory so that the compiler
        // cannot drop it (see nvfp4_candidate)
        tab[i] = make_float2(v, v == 0.0f ? -0.0f : __fdiv_rn(1.0f, v));
    }
    __syncthreads();
}

template <int M>  // the candidate's target for the block amax: 6 or 4
__device__ __forceinline__ float nvfp4_candidate(const float y[16], float a, const float2 *tab, uint32_t &w0,
                                                 uint32_t &w1, uint32_t &scode) {
    // a/4 is a power-of-two scaling: the product by 0.25 rounds the same real number.  a/6 is
    // formed by Markstein's correction step (P. Markstein, IBM J. Res. Dev. 34(1), 1990): with
    // y = RN(1/6), q0 = RN(a*y), r = RN(a - 6*q0) in one fma, t = RN(q0 + r*y).  t is not always
    // RN(a/6) (it differs in the last place for about 0.03% of normal a), but its E4M3 code, the
    // only use of t, is that of RN(a/6) for every binary32 a >= 0 (checked exhaustively against
    // the division); a is clamped to FLT_MAX so that +inf keeps the saturated code of inf / 6.
    float t;
    if constexpr (M == 4) {
        t = __fmul_rn(a, 0.25f);
    } else {
        static_assert(M == 6, "candidates 4 and 6");
        const float am = fminf(a, FLT_MAX), y = __uint_as_float(0x3E2AAAABu);
        const float q0 = __fmul_rn(am, y);
        t = __fmaf_rn(__fmaf_rn(-q0, 6.0f, am), y, q0);
    }
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
    // the squared error: s[i] = RN(d[i]^2), then the fixed tree s[i] += s[i + off] for off = 8, 4,
    // 2, 1, as pairs (s[2j], s[2j+1]), each pair step the scalar tree's two operations.  A square
    // is RN(d*d + (-0)), which is RN(d*d): a packed multiply would be fused with the packed add
    // that consumes it, and -0 as a constant would let the compiler turn the multiply-add back
    // into that multiply, so the addend comes from the scale table in shared memory
    const float nz = tab[0].y;
    const uint64_t nz2 = f2_pack(nz, nz);
    uint64_t p2[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const uint64_t dj = f2_pack(d[2 * j], d[2 * j + 1]);
        p2[j] = f2_fma(dj, dj, nz2);
    }
#pragma unroll
    for (int off = 4; off >= 1; off >>= 1)
#pragma unroll
        for (int j = 0; j < off; ++j) p2[j] = f2_add(p2[j], p2[j + off]);
    float s0, s1;
    f2_unpack(p2[0], s0, s1);
    return __fadd_rn(s0, s1);
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


// A block's 16 inputs as loaded (binary32: four float4; bf16: two uint4), kept apart from their
// conversion to bf16 pairs so that two blocks' loads can be issued before either is used.
template <typename TIn>
struct RawBlock;
template <>
struct RawBlock<float> {
    float4 v[4];
};
template <>
struct RawBlock<uint16_t> {
    uint4 v[2];
};
template <typename TIn>
__device__ __forceinline__ void raw_load(RawBlock<TIn> &r, const TIn *p, bool ok) {
    if constexpr (sizeof(TIn) == 4) {
#pragma unroll
        for (int i = 0; i < 4; ++i)
            r.v[i] = ok ? __ldg(reinterpret_cast<const float4 *>(p) + i) : make_float4(0.f, 0.f, 0.f, 0.f);
    } else {
#pragma unroll
        for (int i = 0; i < 2; ++i) r.v[i] = ok ? __ldg(reinterpret_cast<const uint4 *>(p) + i) : make_uint4(0, 0, 0, 0);
    }
}
// Eight bf16 pairs (element 2i in the low half of word i): bf16 input as stored, binary32 input
// rounded to bf16 (nearest-even), as load8_bf16 forms them.
template <typename TIn>
__device__ __forceinline__ void raw_words(const RawBlock<TIn> &r, uint32_t w[8]) {
    if constexpr (sizeof(TIn) == 4) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            w[2 * i] = bf16x2_rn(r.v[i].x, r.v[i].y);
            w[2 * i + 1] = bf16x2_rn(r.v[i].z, r.v[i].w);
        }
    } else {
        const uint32_t a[8] = {r.v[0].x, r.v[0].y, r.v[0].z, r.v[0].w, r.v[1].x, r.v[1].y, r.v[1].z, r.v[1].w};
#pragma unroll
        for (int i = 0; i < 8; ++i) w[i] = a[i];
    }
}

// One thread per 16-value block.  amax per matrix from amax_in (given) or amax_bits (pass 1).  The
// block index b runs over all matrices; with contiguous rows (ld == cols) the input, code and
// canonical-scale offsets are b*16, b*8 and b, and the matrix index only moves forward in the
// grid-stride loop, so no division is needed on that path.  kTwo: two blocks (b and b + stride)
// per iteration, both blocks' loads issued first, so each warp has twice the bytes in flight.
template <typename TIn, bool kTwo>
__device__ __forceinline__ void nvfp4_quant_blocks(
    const TIn *__restrict__ x, int64_t nmat, int64_t rows, int64_t cols, int64_t ld,
    int64_t mat_stride, const float *__restrict__ amax_in, const unsigned int *__restrict__ amax_bits,
    bool four_over_six, bool sf_mma, uint8_t *__restrict__ codes, uint8_t *__restrict__ sf,
    float *__restrict__ g_dec, uint32_t div_m, uint32_t div_s, const int32_t *__restrict__ skip_offs) {
    __shared__ float2 tab[128];
    fill_scale_tab(tab);
    const int64_t nblk = cols / 16;
    const int64_t per_mat = rows * nblk;
    const int64_t total = nmat * per_mat;
    const int64_t gtid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    // matrix m is skipped (no output written) when skip_offs[m + 1] == skip_offs[m]: an expert
    // that received no rows
    auto skipped = [&](int64_t mm) {
        return skip_offs != nullptr && __ldg(skip_offs + mm + 1) == __ldg(skip_offs + mm);
    };
    if (gtid < nmat && !skipped(gtid)) {
        const float am = amax_in ? amax_in[gtid] : __uint_as_float(amax_bits[gtid]);
        g_dec[gtid] = global_scale(am).dec;
    }
    const bool contiguous = (ld == cols);
    // the matrix of a block: index, first block, end, encode scale, skipped
    struct Mat {
        int64_t m, begin, end;
        float g_enc;
        bool skip;
    };
    auto enter = [&](Mat &s, int64_t bb) {
        if (bb >= s.end) {
            s.m = bb / per_mat;
            s.begin = s.m * per_mat;
            s.end = s.begin + per_mat;
            const float am = amax_in ? amax_in[s.m] : __uint_as_float(amax_bits[s.m]);
            s.g_enc = global_scale(am).enc;
            s.skip = skipped(s.m);
        }
    };
    // row and block of bb within its matrix (the tile-layout scale offset and, with strided rows,
    // the input address need them)
    auto locate = [&](const Mat &s, int64_t bb, int64_t &row, int64_t &blk) {
        const int64_t rem = bb - s.begin;
        row = 0;
        blk = 0;
        if (sf_mma) {
            // nblk % 4 == 0 here: rem / nblk = (rem / 4) / (nblk / 4) by multiply and shift
            row = (int64_t)(uint32_t)(((uint64_t)((uint32_t)rem >> 2) * div_m) >> div_s);
            blk = rem - row * nblk;
        } else if (!contiguous) {
            row = (int64_t)((uint32_t)rem / (uint32_t)nblk);
            blk = rem - row * nblk;
        }
    };
    auto source = [&](const Mat &s, int64_t bb, int64_t row, int64_t blk) -> const TIn * {
        return contiguous ? x + bb * 16 : x + s.m * mat_stride + row * ld + blk * 16;
    };
    auto quantise = [&](const Mat &s, int64_t bb, int64_t row, int64_t blk, const uint32_t wv[8]) {
        // packed products: y feeds the amax, a product and the addend of an FMA, never an add
        float y[16];
        const uint64_t g2 = f2_pack(s.g_enc, s.g_enc);
#pragma unroll
        for (int i = 0; i < 8; ++i) f2_unpack(f2_mul(f2_pack(bf16_lo(wv[i]), bf16_hi(wv[i])), g2), y[2 * i], y[2 * i + 1]);
        uint32_t w0, w1, scode;
        nvfp4_block(y, four_over_six, tab, w0, w1, scode);
        *reinterpret_cast<uint2 *>(codes + bb * 8) = make_uint2(w0, w1);
        if (sf_mma)
            sf[s.begin + sf_mma_offset(row, blk, nblk)] = (uint8_t)scode;
        else
            sf[bb] = (uint8_t)scode;
    };
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    Mat s{-1, 0, 0, 1.0f, false};
    if constexpr (!kTwo) {
        for (int64_t b = gtid; b < total; b += stride) {
            enter(s, b);
            if (s.skip) continue;
            int64_t r1, k1;
            locate(s, b, r1, k1);
            RawBlock<TIn> ra;
            raw_load(ra, source(s, b, r1, k1), true);
            uint32_t wa[8];
            raw_words(ra, wa);
            quantise(s, b, r1, k1, wa);
        }
        return;
    }
    for (int64_t b = gtid; b < total; b += 2 * stride) {
        const int64_t b2 = b + stride;
        enter(s, b);
        Mat s2 = s;
        const bool two = b2 < total;
        if (two) enter(s2, b2);
        const bool l1 = !s.skip, l2 = two && !s2.skip;
        int64_t r1, k1, r2, k2;
        locate(s, b, r1, k1);
        locate(s2, b2, r2, k2);
        RawBlock<TIn> ra, rb;
        raw_load(ra, source(s, b, r1, k1), l1);
        raw_load(rb, source(s2, b2, r2, k2), l2);
        uint32_t wa[8], wb[8];
        raw_words(ra, wa);
        raw_words(rb, wb);
        if (l1) quantise(s, b, r1, k1, wa);
        if (l2) quantise(s2, b2, r2, k2, wb);
        s = s2;  // the next b lies past b2: its matrix is found from b2's
    }
}

#define MOE4_QUANT_PARAMS                                                                                         \
    const TIn *__restrict__ x, int64_t nmat, int64_t rows, int64_t cols, int64_t ld, int64_t mat_stride,          \
        const float *__restrict__ amax_in, const unsigned int *__restrict__ amax_bits, bool four_over_six,       \
        bool sf_mma, uint8_t *__restrict__ codes, uint8_t *__restrict__ sf, float *__restrict__ g_dec,           \
        uint32_t div_m, uint32_t div_s, const int32_t *__restrict__ skip_offs = nullptr
#define MOE4_QUANT_ARGS \
    x, nmat, rows, cols, ld, mat_stride, amax_in, amax_bits, four_over_six, sf_mma, codes, sf, g_dec, div_m, div_s, skip_offs
// One block per iteration, at up to four CTAs per SM: the quantiser running alone on the GPU.
template <typename TIn>
__global__ void __launch_bounds__(256) nvfp4_quant_kernel(MOE4_QUANT_PARAMS) {
    nvfp4_quant_blocks<TIn, false>(MOE4_QUANT_ARGS);
}
// Two blocks per iteration and at most 72 registers: two CTAs of it (72 x 256 registers each) and
// two of the requantiser on 128-column tiles (56 x 256) fill an SM's register file, as the weight
// path runs them side by side.
template <typename TIn>
__global__ void __maxnreg__(72) nvfp4_quant_pair_kernel(MOE4_QUANT_PARAMS) {
    nvfp4_quant_blocks<TIn, true>(MOE4_QUANT_ARGS);
}
#undef MOE4_QUANT_PARAMS
#undef MOE4_QUANT_ARGS

// ------------------------------------------------------------------ dequantise
__global__ void __launch_bounds__(256) nvfp4_dequant_kernel(
    const uint8_t *__restrict__ codes, const uint8_t *__restrict__ sf, const float *__restrict__ g_dec,
    int64_t nmat, int64_t rows, int64_t cols, bool out_bf16, void *__restrict__ out) {
    const int64_t nblk = cols / 16;
    const int64_t per_mat = rows * nblk;
    const int64_t total = nmat * per_mat;
    for (int64_t b = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; b < total;
         b += (int64_t)gridDim.x * blockDim.x) {
        const int64_t m = b / per_mat;
        const uint2 w = *reinterpret_cast<const uint2 *>(codes + b * 8);
        const float sfv = e4m3_to_f32(sf[b]);
        const float gd = g_dec[m];
        float e[16], o[16];
        e2m1x8_to_f32(w.x, e);
        e2m1x8_to_f32(w.y, e + 8);
#pragma unroll
        for (int i = 0; i < 16; ++i) o[i] = __fmul_rn(__fmul_rn(e[i], sfv), gd);
        if (out_bf16) {
            uint32_t p[8];
#pragma unroll
            for (int i = 0; i < 8; ++i)
                p[i] = (uint32_t)f32_to_bf16_bits(o[2 * i]) | ((uint32_t)f32_to_bf16_bits(o[2 * i + 1]) << 16);
            uint4 *dst = reinterpret_cast<uint4 *>(static_cast<uint16_t *>(out) + b * 16);
            dst[0] = make_uint4(p[0], p[1], p[2], p[3]);
            dst[1] = make_uint4(p[4], p[5], p[6], p[7]);
        } else {
            float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(out) + b * 16);
#pragma unroll
            for (int i = 0; i < 4; ++i) dst[i] = make_float4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
        }
    }
}

// ------------------------------------------------------------------ Hadamard(128)
// The Hadamard(128) butterflies on 16 values per thread: fwht128_sub16 (common.cuh).

__device__ __forceinline__ void load16_bf16(const uint16_t *p, float u[16]) {
    const uint4 *src = reinterpret_cast<const uint4 *>(p);
    const uint4 q0 = __ldg(src), q1 = __ldg(src + 1);
    const uint32_t w[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        u[2 * i] = bf16_lo(w[i]);
        u[2 * i + 1] = bf16_hi(w[i]);
    }
}

__device__ __forceinline__ void store16_bf16(uint16_t *p, const float u[16]) {
    uint32_t w[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) w[i] = (uint32_t)f32_to_bf16_bits(u[2 * i]) | ((uint32_t)f32_to_bf16_bits(u[2 * i + 1]) << 16);
    uint4 *dst = reinterpret_cast<uint4 *>(p);
    dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
    dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
}

// The grid-stride loops run over warp-sized groups of sub-blocks so that every lane of a warp
// takes part in the shuffles; lanes past the end compute on zeros and store nothing.  `nsub` (the
// number of 16-value sub-blocks) is a multiple of 8, so a chunk is always whole.
#define MOE4_SUB16_LOOP(nsub)                                                                             \
    for (int64_t b0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) & ~int64_t(31); b0 < (nsub);      \
         b0 += (int64_t)gridDim.x * blockDim.x)

__global__ void __launch_bounds__(256) hadamard_amax_kernel(const uint16_t *__restrict__ x, int64_t nsub,
                                                            unsigned int *__restrict__ amax_bits) {
    float best = 0.0f;
    MOE4_SUB16_LOOP(nsub) {
        const int64_t b = b0 + lane_id();
        float u[16];
        if (b < nsub) {
            load16_bf16(x + b * 16, u);
        } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) u[i] = 0.0f;
        }
        fwht128_sub16(u);
#pragma unroll
        for (int i = 0; i < 16; ++i) best = fmaxf(best, fabsf(u[i]));
    }
    uint32_t m = __reduce_max_sync(0xFFFFFFFFu, __float_as_uint(best));
    __shared__ uint32_t part[8];
    if (lane_id() == 0) part[warp_id()] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
        uint32_t v = 0;
        for (int i = 0; i < (int)(blockDim.x >> 5); ++i) v = max(v, part[i]);
        if (v) atomicMax(amax_bits, v);
    }
}

// Rotate, scale by the tensor's g_enc, and quantise each 16-block with the block quantiser.
__global__ void __launch_bounds__(256) hadamard_quant_kernel(const uint16_t *__restrict__ x, int64_t nsub,
                                                             const unsigned int *__restrict__ amax_bits,
                                                             bool four_over_six, uint8_t *__restrict__ codes,
                                                             uint8_t *__restrict__ sf, float *__restrict__ g_dec) {
    __shared__ float2 tab[128];
    fill_scale_tab(tab);
    const GlobalScale gs = global_scale(__uint_as_float(*amax_bits));
    if (blockIdx.x == 0 && threadIdx.x == 0) *g_dec = gs.dec;
    MOE4_SUB16_LOOP(nsub) {
        const int64_t b = b0 + lane_id();
        const bool live = b < nsub;
        float u[16];
        if (live) {
            load16_bf16(x + b * 16, u);
        } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) u[i] = 0.0f;
        }
        fwht128_sub16(u);
#pragma unroll
        for (int i = 0; i < 8; ++i) f2_unpack(f2_mul(f2_pack(u[2 * i], u[2 * i + 1]), f2_pack(gs.enc, gs.enc)), u[2 * i], u[2 * i + 1]);
        uint32_t w0, w1, scode;
        nvfp4_block(u, four_over_six, tab, w0, w1, scode);
        if (live) {
            *reinterpret_cast<uint2 *>(codes + b * 8) = make_uint2(w0, w1);
            sf[b] = (uint8_t)scode;
        }
    }
}

__global__ void __launch_bounds__(256) hadamard_dequant_kernel(const uint8_t *__restrict__ codes,
                                                               const uint8_t *__restrict__ sf,
                                                               const float *__restrict__ g_dec, int64_t nsub,
                                                               uint16_t *__restrict__ out) {
    const float gd = *g_dec;
    MOE4_SUB16_LOOP(nsub) {
        const int64_t b = b0 + lane_id();
        const bool live = b < nsub;
        float u[16];
        if (live) {
            const uint2 w = *reinterpret_cast<const uint2 *>(codes + b * 8);
            const float sfv = e4m3_to_f32(sf[b]);
            float e[16];
            e2m1x8_to_f32(w.x, e);
            e2m1x8_to_f32(w.y, e + 8);
#pragma unroll
            for (int i = 0; i < 16; ++i) u[i] = __fmul_rn(__fmul_rn(e[i], sfv), gd);
        } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) u[i] = 0.0f;
        }
        fwht128_sub16(u);
        if (live) store16_bf16(out + b * 16, u);
    }
}

// The combine straight from the NVFP4-encoded return path (hadamard_dequant then moe4_combine,
// without the decoded rows in memory).  Lane l of a group of eight holds 16 columns of one
// token's 128-column chunk; in slot order each slot's dispatched row is decoded exactly as
// hadamard_dequant_kernel does it (dequantise, rotate, round to bf16) and added, times its routing
// weight, to a binary32 accumulator exactly as combine_kernel does it; then bf16.  Every lane
// takes part in the shuffles of the rotation; lanes past the end compute on zeros.
__global__ void __launch_bounds__(256) combine_hadamard_kernel(const uint8_t *__restrict__ codes,
                                                               const uint8_t *__restrict__ sf,
                                                               const float *__restrict__ g_dec,
                                                               const int32_t *__restrict__ row_of,
                                                               const float *__restrict__ w, int64_t T, int k,
                                                               int64_t d, uint16_t *__restrict__ y) {
    const float gd = *g_dec;
    const uint32_t per_row = (uint32_t)(d / 16);  // 16-value sub-blocks per row
    const int64_t nsub = T * per_row;
    MOE4_SUB16_LOOP(nsub) {
        const int64_t b = b0 + lane_id();
        const bool live = b < nsub;
        const uint32_t t = live ? (uint32_t)b / per_row : 0u;  // nsub < 2^32 (checked on the host)
        const uint32_t sb = live ? (uint32_t)b - t * per_row : 0u;
        float acc[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) acc[i] = 0.0f;
        // slot j's codes and scale are loaded while slot j-1 is decoded (one slot ahead)
        auto load_slot = [&](int j, uint2 &cw, uint32_t &sfc, float &wj) {
            cw = make_uint2(0u, 0u);
            sfc = 0u;
            wj = 0.0f;
            if (live && j < k) {
                const int64_t row = __ldg(row_of + (int64_t)t * k + j);
                wj = __ldg(w + (int64_t)t * k + j);
                const int64_t sub = row * per_row + sb;
                cw = __ldg(reinterpret_cast<const uint2 *>(codes + sub * 8));
                sfc = __ldg(sf + sub);
            }
        };
        uint2 cw;
        uint32_t sfc;
        float wj;
        load_slot(0, cw, sfc, wj);
        for (int j = 0; j < k; ++j) {
            uint2 ncw;
            uint32_t nsfc;
            float nwj;
            load_slot(j + 1, ncw, nsfc, nwj);
            float u[16];
            if (live) {
                const float sfv = e4m3_to_f32(sfc);
                float e[16];
                e2m1x8_to_f32(cw.x, e);
                e2m1x8_to_f32(cw.y, e + 8);
#pragma unroll
                for (int i = 0; i < 16; ++i) u[i] = __fmul_rn(__fmul_rn(e[i], sfv), gd);
            } else {
#pragma unroll
                for (int i = 0; i < 16; ++i) u[i] = 0.0f;
            }
            fwht128_sub16(u);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const float yh = __uint_as_float((uint32_t)f32_to_bf16_bits(u[i]) << 16);
                acc[i] = __fadd_rn(acc[i], __fmul_rn(wj, yh));
            }
            cw = ncw;
            sfc = nsfc;
            wj = nwj;
        }
        if (live) store16_bf16(y + (int64_t)t * d + (int64_t)sb * 16, acc);
    }
}

// The 8.25-bit return-path codec: Hadamard(128), then MXFP8 (E4M3 elements, one E8M0 scale per 32
// by the ceiling rule, nearest-even).  One pass: the scales are per 32-block, which is the
// sub-block pair of lanes 2k and 2k+1 (block amax by one shuffle).
__global__ void __launch_bounds__(256) hadamard_quant_mx_kernel(const uint16_t *__restrict__ x, int64_t nsub,
                                                                uint8_t *__restrict__ q, uint8_t *__restrict__ e8) {
    MOE4_SUB16_LOOP(nsub) {
        const int64_t b = b0 + lane_id();
        const bool live = b < nsub;
        float u[16];
        if (live) {
            load16_bf16(x + b * 16, u);
        } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) u[i] = 0.0f;
        }
        fwht128_sub16(u);
        float a = 0.0f;
#pragma unroll
        for (int i = 0; i < 16; ++i) a = fmaxf(a, fabsf(u[i]));
        a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, 1));
        const int e = mx_scale_exponent(a);
        const float s = pow2_neg(e);
        uint32_t w[4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
            w[j] = e4m3x4_rn(__fmul_rn(u[4 * j], s), __fmul_rn(u[4 * j + 1], s), __fmul_rn(u[4 * j + 2], s),
                             __fmul_rn(u[4 * j + 3], s));
        if (live) {
            *reinterpret_cast<uint4 *>(q + b * 16) = make_uint4(w[0], w[1], w[2], w[3]);
            if ((b & 1) == 0) e8[b >> 1] = (uint8_t)(e + 127);
        }
    }
}

__global__ void __launch_bounds__(256) hadamard_dequant_mx_kernel(const uint8_t *__restrict__ q,
                                                                  const uint8_t *__restrict__ e8, int64_t nsub,
                                                                  uint16_t *__restrict__ out) {
    MOE4_SUB16_LOOP(nsub) {
        const int64_t b = b0 + lane_id();
        const bool live = b < nsub;
        float u[16];
        if (live) {
            const uint4 codes = *reinterpret_cast<const uint4 *>(q + b * 16);
            const uint32_t eb = e8[b >> 1];
            const float scale = __uint_as_float(eb ? (eb << 23) : 0x00400000u);  // 2^(eb-127), exact
            const uint32_t cw[4] = {codes.x, codes.y, codes.z, codes.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float2 lo = h2_bits_to_f2(e4m3x2_to_h2(cw[j] & 0xFFFFu));  // E4M3 -> f16 is exact
                const float2 hi = h2_bits_to_f2(e4m3x2_to_h2(cw[j] >> 16));
                u[4 * j] = __fmul_rn(lo.x, scale);
                u[4 * j + 1] = __fmul_rn(lo.y, scale);
                u[4 * j + 2] = __fmul_rn(hi.x, scale);
                u[4 * j + 3] = __fmul_rn(hi.y, scale);
            }
        } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) u[i] = 0.0f;
        }
        fwht128_sub16(u);
        if (live) store16_bf16(out + b * 16, u);
    }
}
#undef MOE4_SUB16_LOOP

// Division of n < 2^31 by d >= 1 as (n * m) >> s (Granlund and Montgomery, "Division by invariant
// integers using multiplication", PLDI 1994, theorem 4.2): l = ceil(log2 d), s = 31 + l,
// m = ceil(2^s / d), which is below 2^32.
static void div_magic(uint32_t d, uint32_t &m, uint32_t &s) {
    uint32_t l = 0;
    while ((uint64_t(1) << l) < d) ++l;
    s = 31 + l;
    m = (uint32_t)(((uint64_t(1) << s) + d - 1) / d);
}

static int grid_for(int64_t work_items, int threads, int per_sm) {
    const int64_t need = (work_items + threads - 1) / threads;
    const int64_t cap = (int64_t)num_sms() * per_sm;
    return (int)(need < 1 ? 1 : (need < cap ? need : cap));
}

int quantize_f32_given(const float *x, int64_t nmat, int64_t rows, int64_t cols, const float *amax_in,
                       uint8_t *codes, uint8_t *sf, float *g_dec, const int32_t *skip_offs, bool four_over_six,
                       bool sf_mma, cudaStream_t st, int ctas_per_sm) {
    const int64_t total = nmat * rows * (cols / 16);
    const int grid = grid_for(total > nmat ? total : nmat, 256, ctas_per_sm);
    uint32_t div_m = 0, div_s = 0;
    if (sf_mma) div_magic((uint32_t)(cols / 64), div_m, div_s);
    // fewer than eight CTAs per SM: the SMs are shared with the requantiser (MOE4_SHARE_SMS)
    if (ctas_per_sm < 8)
        nvfp4_quant_pair_kernel<float><<<grid, 256, 0, st>>>(x, nmat, rows, cols, cols, rows * cols, amax_in, nullptr,
                                                             four_over_six, sf_mma, codes, sf, g_dec, div_m, div_s,
                                                             skip_offs);
    else
        nvfp4_quant_kernel<float><<<grid, 256, 0, st>>>(x, nmat, rows, cols, cols, rows * cols, amax_in, nullptr,
                                                        four_over_six, sf_mma, codes, sf, g_dec, div_m, div_s, skip_offs);
    return launch_status();
}

}  // namespace moe4

using namespace moe4;

template <typename TIn>
static int nvfp4_quantize_impl(const TIn *x, int64_t nmat, int64_t rows, int64_t cols, int64_t ld, uint8_t *codes,
                               uint8_t *sf, float *g_dec, const float *amax_in, uint32_t flags, void *ws,
                               size_t ws_bytes, void *stream) {
    MOE4_CHECK_ARG(nmat >= 1 && rows >= 0 && cols > 0 && cols % 16 == 0 && ld >= cols &&
                   (ld * (int64_t)sizeof(TIn)) % 16 == 0);
    MOE4_CHECK_ARG(g_dec);
    MOE4_CHECK_ARG(rows == 0 || (x && codes && sf && aligned16(x) && aligned16(codes)));
    MOE4_CHECK_ARG((flags & ~(MOE4_FOUR_OVER_SIX | MOE4_AMAX_GIVEN | MOE4_SF_MMA_LAYOUT)) == 0);
    const bool given = (flags & MOE4_AMAX_GIVEN) != 0;
    const bool sf_mma = (flags & MOE4_SF_MMA_LAYOUT) != 0;
    MOE4_CHECK_ARG(!given || amax_in);
    // the amax pass runs one grid row per matrix (gridDim.y at most 65535)
    MOE4_CHECK_ARG(given || nmat <= 65535);
    MOE4_CHECK_ARG(!sf_mma || (rows % 128 == 0 && cols % 64 == 0));
    MOE4_CHECK_ARG(rows * (cols / 16) < (int64_t(1) << 32));
    cudaStream_t st = as_stream(stream);
    unsigned int *amax_bits = nullptr;
    if (!given) {
        if (!ws || ws_bytes < (size_t)nmat * sizeof(unsigned int)) return MOE4_ERR_WORKSPACE;
        amax_bits = static_cast<unsigned int *>(ws);
        if (cudaMemsetAsync(amax_bits, 0, (size_t)nmat * sizeof(unsigned int), st) != cudaSuccess)
            return MOE4_ERR_CUDA;
        if (rows > 0) {
            const int64_t nvec = rows * (cols / 8);
            int gx = grid_for(nvec, 256, 8 * 1);
            const int64_t per_mat_cap = ((int64_t)num_sms() * 8 + nmat - 1) / nmat;
            if (gx > per_mat_cap) gx = (int)per_mat_cap;
            if (gx < 1) gx = 1;
            amax_bf16_kernel<TIn><<<dim3(gx, (unsigned)nmat), 256, 0, st>>>(x, rows, cols, ld, rows * ld, amax_bits);
        }
    }
    const int64_t total = nmat * rows * (cols / 16);
    const int grid = grid_for(total > nmat ? total : nmat, 256, 8);
    uint32_t div_m = 0, div_s = 0;
    if (sf_mma) div_magic((uint32_t)(cols / 64), div_m, div_s);
    nvfp4_quant_kernel<TIn><<<grid, 256, 0, st>>>(x, nmat, rows, cols, ld, rows * ld, given ? amax_in : nullptr,
                                                  amax_bits, (flags & MOE4_FOUR_OVER_SIX) != 0, sf_mma, codes, sf,
                                                  g_dec, div_m, div_s);
    return launch_status();
}

extern "C" int nvfp4_quantize(const uint16_t *x, int64_t nmat, int64_t rows, int64_t cols, int64_t ld,
                              uint8_t *codes, uint8_t *sf, float *g_dec, const float *amax_in,
                              uint32_t flags, void *ws, size_t ws_bytes, void *stream) {
    return nvfp4_quantize_impl(x, nmat, rows, cols, ld, codes, sf, g_dec, amax_in, flags, ws, ws_bytes, stream);
}

extern "C" int nvfp4_quantize_f32(const float *x, int64_t nmat, int64_t rows, int64_t cols, int64_t ld,
                                  uint8_t *codes, uint8_t *sf, float *g_dec, const float *amax_in,
                                  uint32_t flags, void *ws, size_t ws_bytes, void *stream) {
    return nvfp4_quantize_impl(x, nmat, rows, cols, ld, codes, sf, g_dec, amax_in, flags, ws, ws_bytes, stream);
}

extern "C" int nvfp4_dequantize(const uint8_t *codes, const uint8_t *sf, const float *g_dec, int64_t nmat,
                                int64_t rows, int64_t cols, void *out, uint32_t flags, void *stream) {
    MOE4_CHECK_ARG(nmat >= 1 && rows >= 0 && cols > 0 && cols % 16 == 0);
    MOE4_CHECK_ARG(codes && sf && g_dec && out && aligned16(out) && aligned16(codes));
    MOE4_CHECK_ARG((flags & ~(MOE4_OUT_BF16 | MOE4_OUT_F32)) == 0);
    const bool bf16 = (flags & MOE4_OUT_BF16) != 0;
    MOE4_CHECK_ARG(bf16 != ((flags & MOE4_OUT_F32) != 0));
    const int64_t total = nmat * rows * (cols / 16);
    if (total == 0) return MOE4_OK;
    nvfp4_dequant_kernel<<<grid_for(total, 256, 8), 256, 0, as_stream(stream)>>>(codes, sf, g_dec, nmat, rows,
                                                                                  cols, bf16, out);
    return launch_status();
}

extern "C" int hadamard_quant(const uint16_t *x, int64_t rows, int64_t cols, uint8_t *codes, uint8_t *sf,
                              float *g_dec, uint32_t flags, void *ws, size_t ws_bytes, void *stream) {
    MOE4_CHECK_ARG(rows >= 0 && cols > 0 && cols % 128 == 0);
    if (flags & MOE4_MXFP8) {  // the 8.25-bit codec: codes = E4M3 [rows, cols], sf = E8M0 [rows, cols/32]
        MOE4_CHECK_ARG(flags == MOE4_MXFP8 && codes && sf && (rows == 0 || (x && aligned16(x))) && aligned16(codes));
        const int64_t nsub = rows * (cols / 16);
        if (nsub == 0) return MOE4_OK;
        hadamard_quant_mx_kernel<<<grid_for(nsub, 256, 8), 256, 0, as_stream(stream)>>>(x, nsub, codes, sf);
        return launch_status();
    }
    MOE4_CHECK_ARG(codes && sf && g_dec && aligned16(codes) && (rows == 0 || (x && aligned16(x))));
    MOE4_CHECK_ARG((flags & ~(MOE4_FOUR_OVER_SIX | MOE4_AMAX_GIVEN)) == 0);
    if (!ws || ws_bytes < sizeof(unsigned int) || !aligned4(ws)) return MOE4_ERR_WORKSPACE;
    cudaStream_t st = as_stream(stream);
    unsigned int *amax_bits = static_cast<unsigned int *>(ws);
    const int64_t nsub = rows * (cols / 16);
    const int grid = grid_for(nsub > 1 ? nsub : 1, 256, 8);
    // with MOE4_AMAX_GIVEN, ws already holds the rotated tensor's amax (as the down-projection
    // GEMM's epilogue returns it): no pass of its own
    if (!(flags & MOE4_AMAX_GIVEN)) {
        if (cudaMemsetAsync(amax_bits, 0, sizeof(unsigned int), st) != cudaSuccess) return MOE4_ERR_CUDA;
        if (nsub > 0) hadamard_amax_kernel<<<grid, 256, 0, st>>>(x, nsub, amax_bits);
    }
    hadamard_quant_kernel<<<grid, 256, 0, st>>>(x, nsub, amax_bits, (flags & MOE4_FOUR_OVER_SIX) != 0, codes, sf,
                                                g_dec);
    return launch_status();
}

extern "C" int hadamard_dequant(const uint8_t *codes, const uint8_t *sf, const float *g_dec, int64_t rows,
                                int64_t cols, uint16_t *out_bf16, uint32_t flags, void *stream) {
    MOE4_CHECK_ARG(rows >= 0 && cols > 0 && cols % 128 == 0 && (flags == 0 || flags == MOE4_MXFP8));
    if (flags == MOE4_MXFP8) {
        MOE4_CHECK_ARG(codes && sf && out_bf16 && aligned16(out_bf16) && aligned16(codes));
        const int64_t nsub = rows * (cols / 16);
        if (nsub == 0) return MOE4_OK;
        hadamard_dequant_mx_kernel<<<grid_for(nsub, 256, 8), 256, 0, as_stream(stream)>>>(codes, sf, nsub, out_bf16);
        return launch_status();
    }
    MOE4_CHECK_ARG(codes && sf && g_dec && out_bf16 && aligned16(out_bf16) && aligned16(codes));
    const int64_t nsub = rows * (cols / 16);
    if (nsub == 0) return MOE4_OK;
    hadamard_dequant_kernel<<<grid_for(nsub, 256, 8), 256, 0, as_stream(stream)>>>(codes, sf, g_dec, nsub, out_bf16);
    return launch_status();
}

extern "C" int moe4_combine_hadamard(const uint8_t *codes, const uint8_t *sf, const float *g_dec,
                                     const int32_t *row_of, const float *w, int64_t T, int64_t k, int64_t d,
                                     uint16_t *y, void *stream) {
    MOE4_CHECK_ARG(T >= 0 && k >= 1 && k <= 32 && d > 0 && d % 128 == 0);
    MOE4_CHECK_ARG(T * (d / 16) < (int64_t(1) << 32));
    MOE4_CHECK_ARG(T == 0 || (codes && sf && g_dec && row_of && w && y && aligned16(codes) && aligned16(y)));
    const int64_t nsub = T * (d / 16);
    if (nsub == 0) return MOE4_OK;
    combine_hadamard_kernel<<<grid_for(nsub, 256, 8), 256, 0, as_stream(stream)>>>(codes, sf, g_dec, row_of, w, T,
                                                                                    (int)k, d, y);
    return launch_status();
}

// ------------------------------------------------------------------ allocation-free variant
// nvfp4_quantize needs scratch for the per-matrix amax of its first pass.  This variant keeps
// that scratch in a fixed array in device memory that belongs to the library, for callers that
// cannot allocate device memory themselves (see include/moe4.h).  Host code only sees a
// host-side stand-in for the symbol, so every call looks up the array's device address in the
// current context.  The lookup allocates nothing, and a fresh one per call stays right after the
// context is torn down and created again (cudaDeviceReset), when the array may have moved.
namespace moe4 {
constexpr int64_t kNoAllocMaxMats = 4096;
static __device__ __align__(256) unsigned int g_noalloc_amax[kNoAllocMaxMats];

static unsigned int *noalloc_amax_address() {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_amax) != cudaSuccess) return nullptr;
    return static_cast<unsigned int *>(p);
}
}  // namespace moe4

extern "C" int nvfp4_quantize_noalloc(const uint16_t *x, int64_t nmat, int64_t rows, int64_t cols, int64_t ld,
                                      uint8_t *codes, uint8_t *sf, float *g_dec, uint32_t flags, void *stream) {
    MOE4_CHECK_ARG(nmat >= 1 && nmat <= kNoAllocMaxMats);
    MOE4_CHECK_ARG(rows >= 0 && cols > 0 && cols % 16 == 0 && ld >= cols && ld % 8 == 0);
    MOE4_CHECK_ARG(g_dec);
    MOE4_CHECK_ARG(rows == 0 || (x && codes && sf && aligned16(x) && aligned16(codes)));
    MOE4_CHECK_ARG((flags & ~(MOE4_FOUR_OVER_SIX | MOE4_SF_MMA_LAYOUT)) == 0);
    const bool sf_mma = (flags & MOE4_SF_MMA_LAYOUT) != 0;
    MOE4_CHECK_ARG(!sf_mma || (rows % 128 == 0 && cols % 64 == 0));
    MOE4_CHECK_ARG(rows * (cols / 16) < (int64_t(1) << 32));
    unsigned int *amax_bits = noalloc_amax_address();
    if (!amax_bits) return MOE4_ERR_CUDA;
    cudaStream_t st = as_stream(stream);
    // the array keeps the previous call's maxima: clear the part this call folds into
    if (cudaMemsetAsync(amax_bits, 0, (size_t)nmat * sizeof(unsigned int), st) != cudaSuccess) return MOE4_ERR_CUDA;
    if (rows > 0) {
        const int64_t nvec = rows * (cols / 8);
        int gx = grid_for(nvec, 256, 8);
        const int64_t per_mat_cap = ((int64_t)num_sms() * 8 + nmat - 1) / nmat;
        if (gx > per_mat_cap) gx = (int)per_mat_cap;
        if (gx < 1) gx = 1;
        amax_bf16_kernel<uint16_t><<<dim3(gx, (unsigned)nmat), 256, 0, st>>>(x, rows, cols, ld, rows * ld, amax_bits);
    }
    const int64_t total = nmat * rows * (cols / 16);
    const int grid = grid_for(total > nmat ? total : nmat, 256, 8);
    uint32_t div_m = 0, div_s = 0;
    if (sf_mma) div_magic((uint32_t)(cols / 64), div_m, div_s);
    nvfp4_quant_kernel<uint16_t><<<grid, 256, 0, st>>>(x, nmat, rows, cols, ld, rows * ld, nullptr, amax_bits,
                                             (flags & MOE4_FOUR_OVER_SIX) != 0, sf_mma, codes, sf, g_dec, div_m,
                                             div_s);
    return launch_status();
}
