// moe.cu -- the MoE layer around the expert GEMMs: top-k routing, the dispatch permutation of
// NVFP4 rows, SwiGLU between the two expert GEMMs, the weighted combine of returned rows, and the
// FP32 master-weight update.
//
// Pages: "Thinking Machines: Nvidia FP4 Up to 6x Faster, Runs Gain 8%" (fourweekmba.com,
// model-card update: each token is routed to 8 of 384 experts); "4-bit computation from the start
// of Inkling 2 Small's pretraining" (lhc.media: inputs are dispatched in NVFP4; results are
// combined after the return path; master weights stay in FP32).
#include "common.cuh"

namespace moe4 {

// ------------------------------------------------------------------ top-k routing
// One warp per token.  Round i picks the best (largest logit, then lowest expert index) among the
// experts strictly after the previous pick in that order, so k rounds give the k best in order.
__device__ __forceinline__ bool better(float v1, int e1, float v2, int e2) {
    return v1 > v2 || (v1 == v2 && e1 < e2);
}

__global__ void __launch_bounds__(256) route_topk_kernel(const float *__restrict__ logits, int64_t T, int E, int k,
                                                         int32_t *__restrict__ idx_out, float *__restrict__ w_out) {
    const int lane = lane_id();
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t t = (int64_t)blockIdx.x * (blockDim.x >> 5) + warp_id(); t < T; t += warps) {
        const float *row = logits + t * E;
        float last_v = __int_as_float(0x7F800000);  // +inf: nothing picked yet
        int last_e = -1;
        float my_v = 0.0f;
        int my_e = 0;
        for (int i = 0; i < k; ++i) {
            float bv = -__int_as_float(0x7F800000);
            int be = 0x7FFFFFFF;
            for (int e = lane; e < E; e += 32) {
                const float v = row[e];
                const bool eligible = better(last_v, last_e, v, e);
                if (eligible && better(v, e, bv, be)) {
                    bv = v;
                    be = e;
                }
            }
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1) {
                const float ov = __shfl_xor_sync(0xFFFFFFFFu, bv, off);
                const int oe = __shfl_xor_sync(0xFFFFFFFFu, be, off);
                if (better(ov, oe, bv, be)) {
                    bv = ov;
                    be = oe;
                }
            }
            last_v = bv;
            last_e = be;
            if (lane == i) {
                my_v = bv;
                my_e = be;
            }
        }
        // softmax over the k picks, relative to the largest (pick 0); sum in slot order
        const float top = __shfl_sync(0xFFFFFFFFu, my_v, 0);
        const float ex = lane < k ? expf(__fsub_rn(my_v, top)) : 0.0f;
        float sum = 0.0f;
        for (int j = 0; j < k; ++j) sum = __fadd_rn(sum, __shfl_sync(0xFFFFFFFFu, ex, j));
        if (lane < k) {
            idx_out[t * k + lane] = my_e;
            w_out[t * k + lane] = __fdiv_rn(ex, sum);
        }
    }
}

// ------------------------------------------------------------------ dispatch plan
// Counting sort of the T*k (token, slot) entries by expert, stable in flat order t*k + j.
constexpr int kChunk = 1024;

__global__ void __launch_bounds__(256) plan_count_kernel(const int32_t *__restrict__ idx, int64_t n, int E,
                                                         int32_t *__restrict__ chunk_counts) {
    extern __shared__ int32_t cnt[];
    for (int e = threadIdx.x; e < E; e += blockDim.x) cnt[e] = 0;
    __syncthreads();
    const int64_t base = (int64_t)blockIdx.x * kChunk;
    for (int i = threadIdx.x; i < kChunk; i += blockDim.x) {
        const int64_t f = base + i;
        if (f < n) {
            const int e = idx[f];
            if ((unsigned)e < (unsigned)E) atomicAdd(&cnt[e], 1);  // out-of-range indices are dropped
        }
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) chunk_counts[(int64_t)blockIdx.x * E + e] = cnt[e];
}

// Per expert: exclusive prefix over chunks (in place) and the padded group offsets.
__global__ void __launch_bounds__(1024) plan_scan_kernel(int32_t *__restrict__ chunk_counts, int64_t nchunks, int E,
                                                         int32_t *__restrict__ totals, int32_t *__restrict__ offs) {
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int32_t run = 0;
        for (int64_t c = 0; c < nchunks; ++c) {
            const int32_t v = chunk_counts[c * E + e];
            chunk_counts[c * E + e] = run;
            run += v;
        }
        totals[e] = run;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        int32_t o = 0;
        for (int e = 0; e < E; ++e) {
            offs[e] = o;
            o += (totals[e] + 127) / 128 * 128;
        }
        offs[E] = o;
    }
}

// One warp per chunk, 32 entries at a time in flat order: rank among equal experts by
// __match_any_sync, so the assignment is stable.
__global__ void __launch_bounds__(32) plan_assign_kernel(const int32_t *__restrict__ idx, int64_t n, int k, int E,
                                                         const int32_t *__restrict__ chunk_base,
                                                         const int32_t *__restrict__ offs,
                                                         int32_t *__restrict__ row_of, int32_t *__restrict__ src_of) {
    extern __shared__ int32_t run[];
    const int64_t chunk = blockIdx.x;
    for (int e = threadIdx.x; e < E; e += 32) run[e] = offs[e] + chunk_base[chunk * E + e];
    __syncwarp();
    const int lane = threadIdx.x;
    const unsigned lt = (1u << lane) - 1u;
    for (int s = 0; s < kChunk; s += 32) {
        const int64_t f = chunk * kChunk + s + lane;
        const int ev = f < n ? idx[f] : -1;
        const bool live = (unsigned)ev < (unsigned)E;
        const int e = live ? ev : -1 - lane;  // dead lanes never match a live one
        const unsigned same = __match_any_sync(0xFFFFFFFFu, e);
        int row = 0;
        if (live) row = run[e] + __popc(same & lt);
        __syncwarp();
        if (live && (same & lt) == 0) run[e] += __popc(same);
        __syncwarp();
        if (live) {
            row_of[f] = row;
            src_of[row] = (int32_t)(f / k);
        } else if (f < n) {
            row_of[f] = -1;
        }
    }
}

// ------------------------------------------------------------------ NVFP4 row gather
// One warp per dispatched row: codes in 16-byte pieces, scales in 8-byte pieces (or bytes).
// One warp per dispatched row.  A row is cbytes of codes (NVFP4: cols/2, MXFP8: cols) and sbytes
// of scales (NVFP4: cols/16, MXFP8: cols/32).
__global__ void __launch_bounds__(256) permute_rows_kernel(const uint8_t *__restrict__ codes,
                                                           const uint8_t *__restrict__ sf, int64_t cbytes,
                                                           int64_t sbytes, const int32_t *__restrict__ src_of,
                                                           int64_t rows_total, uint8_t *__restrict__ out_codes,
                                                           uint8_t *__restrict__ out_sf, bool sf_mma) {
    const int lane = lane_id();
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t r = (int64_t)blockIdx.x * (blockDim.x >> 5) + warp_id(); r < rows_total; r += warps) {
        const int32_t src = src_of[r];
        uint4 *dc = reinterpret_cast<uint4 *>(out_codes + r * cbytes);
        const uint4 *sc = reinterpret_cast<const uint4 *>(codes + (int64_t)(src < 0 ? 0 : src) * cbytes);
        for (int64_t i = lane; i < cbytes / 16; i += 32) dc[i] = src < 0 ? make_uint4(0, 0, 0, 0) : __ldg(sc + i);
        if (sf_mma) {
            // 4 consecutive blocks of a row are one 32-bit word in both layouts
            const uint32_t *ss = reinterpret_cast<const uint32_t *>(sf + (int64_t)(src < 0 ? 0 : src) * sbytes);
            for (int64_t kg = lane; kg < sbytes / 4; kg += 32) {
                const int64_t off = ((r >> 7) * (sbytes / 4) + kg) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4;
                *reinterpret_cast<uint32_t *>(out_sf + off) = src < 0 ? 0u : __ldg(ss + kg);
            }
        } else if (sbytes % 8 == 0) {
            uint2 *ds = reinterpret_cast<uint2 *>(out_sf + r * sbytes);
            const uint2 *ss = reinterpret_cast<const uint2 *>(sf + (int64_t)(src < 0 ? 0 : src) * sbytes);
            for (int64_t i = lane; i < sbytes / 8; i += 32) ds[i] = src < 0 ? make_uint2(0, 0) : __ldg(ss + i);
        } else {
            for (int64_t i = lane; i < sbytes; i += 32)
                out_sf[r * sbytes + i] = src < 0 ? 0 : sf[(int64_t)src * sbytes + i];
        }
    }
}

// ------------------------------------------------------------------ SwiGLU
// With kAmax, also the largest |h| of the bf16 results (as binary32 bits, one atomicMax per
// block).  Each instance is held to 32 registers so that eight blocks stay resident per SM.
template <bool kAmax>
__global__ void __launch_bounds__(256, 8) swiglu_kernel(const float *__restrict__ gu, int64_t rows, int64_t f,
                                                        uint16_t *__restrict__ h, unsigned int *__restrict__ amax_bits) {
    const int64_t quads = rows * f / 4;
    uint32_t best = 0;  // two packed bf16 magnitudes
    for (int64_t q = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; q < quads; q += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = (q * 4) / f;
        const int64_t c = q * 4 - r * f;
        const float4 g = __ldg(reinterpret_cast<const float4 *>(gu + r * 2 * f + c));
        const float4 u = __ldg(reinterpret_cast<const float4 *>(gu + r * 2 * f + f + c));
        const float gs[4] = {g.x, g.y, g.z, g.w}, us[4] = {u.x, u.y, u.z, u.w};
        uint32_t out[2] = {0, 0};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float silu = __fdiv_rn(gs[i], __fadd_rn(1.0f, expf(-gs[i])));
            out[i >> 1] |= (uint32_t)f32_to_bf16_bits(__fmul_rn(silu, us[i])) << (16 * (i & 1));
        }
        *reinterpret_cast<uint2 *>(h + r * f + c) = make_uint2(out[0], out[1]);
        if (kAmax) best = __vmaxu2(best, __vmaxu2(out[0] & 0x7FFF7FFFu, out[1] & 0x7FFF7FFFu));
    }
    if (kAmax) {
        __shared__ uint32_t part[8];
        uint32_t mag = max(best & 0xFFFFu, best >> 16) << 16;
        mag = __reduce_max_sync(0xFFFFFFFFu, mag);
        if (lane_id() == 0) part[threadIdx.x >> 5] = mag;
        __syncthreads();
        if (threadIdx.x == 0) {
            uint32_t m = part[0];
            for (int w = 1; w < (int)(blockDim.x >> 5); ++w) m = max(m, part[w]);
            if (m) atomicMax(amax_bits, m);
        }
    }
}

// ------------------------------------------------------------------ SwiGLU backward
// h = silu(g) * u:  du = dh * silu(g),  dg = dh * u * s * (1 + g * (1 - s)) with s = 1/(1+exp(-g)).
__global__ void __launch_bounds__(256) swiglu_bwd_kernel(const float *__restrict__ gu, const float *__restrict__ dh,
                                                         int64_t rows, int64_t f, uint16_t *__restrict__ dgu) {
    const int64_t fq = f / 4;
    for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
        const float *gr = gu + r * 2 * f, *dr = dh + r * f;
        uint16_t *outr = dgu + r * 2 * f;
#pragma unroll 2
        for (int64_t cq = threadIdx.x; cq < fq; cq += blockDim.x) {
            const int64_t c = cq * 4;
            const float4 g = __ldg(reinterpret_cast<const float4 *>(gr + c));
            const float4 u = __ldg(reinterpret_cast<const float4 *>(gr + f + c));
            const float4 d = __ldg(reinterpret_cast<const float4 *>(dr + c));
            const float gs[4] = {g.x, g.y, g.z, g.w}, us[4] = {u.x, u.y, u.z, u.w}, ds[4] = {d.x, d.y, d.z, d.w};
            uint32_t og[2] = {0, 0}, ou[2] = {0, 0};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                // RN(1 / x) by the reciprocal intrinsic: the same correctly rounded value as the
                // division of 1 by x
                const float sg = __frcp_rn(__fadd_rn(1.0f, expf(-gs[i])));
                const float silu = __fmul_rn(gs[i], sg);
                const float dsilu = __fmul_rn(sg, __fadd_rn(1.0f, __fmul_rn(gs[i], __fsub_rn(1.0f, sg))));
                const float dgv = __fmul_rn(__fmul_rn(ds[i], us[i]), dsilu);
                const float duv = __fmul_rn(ds[i], silu);
                og[i >> 1] |= (uint32_t)f32_to_bf16_bits(dgv) << (16 * (i & 1));
                ou[i >> 1] |= (uint32_t)f32_to_bf16_bits(duv) << (16 * (i & 1));
            }
            *reinterpret_cast<uint2 *>(outr + c) = make_uint2(og[0], og[1]);
            *reinterpret_cast<uint2 *>(outr + f + c) = make_uint2(ou[0], ou[1]);
        }
    }
}

// ------------------------------------------------------------------ combine backward
// dyhat[r] = w[t, j] * dy[t] for the dispatched row r of (t, j); padding rows are zero.  One warp
// per dispatched row; the slot j is found among the k rows of token t.
__global__ void __launch_bounds__(256) combine_bwd_kernel(const uint16_t *__restrict__ dy, const int32_t *__restrict__ row_of,
                                                          const float *__restrict__ w, const int32_t *__restrict__ src_of,
                                                          int k, int64_t d, int64_t rows_total,
                                                          uint16_t *__restrict__ dyhat) {
    const int lane = lane_id();
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t r = (int64_t)blockIdx.x * (blockDim.x >> 5) + warp_id(); r < rows_total; r += warps) {
        const int32_t t = src_of[r];
        float wj = 0.0f;
        if (t >= 0) {
            for (int j = 0; j < k; ++j)
                if (row_of[(int64_t)t * k + j] == r) wj = w[(int64_t)t * k + j];
        }
        uint4 *dst = reinterpret_cast<uint4 *>(dyhat + r * d);
        const uint4 *src = reinterpret_cast<const uint4 *>(dy + (int64_t)(t < 0 ? 0 : t) * d);
        for (int64_t i = lane; i < d / 8; i += 32) {
            uint4 o = make_uint4(0, 0, 0, 0);
            if (t >= 0) {
                const uint4 q = __ldg(src + i);
                const uint32_t qs[4] = {q.x, q.y, q.z, q.w};
                uint32_t os[4];
#pragma unroll
                for (int h = 0; h < 4; ++h)
                    os[h] = (uint32_t)f32_to_bf16_bits(__fmul_rn(wj, bf16_lo(qs[h]))) |
                            ((uint32_t)f32_to_bf16_bits(__fmul_rn(wj, bf16_hi(qs[h]))) << 16);
                o = make_uint4(os[0], os[1], os[2], os[3]);
            }
            dst[i] = o;
        }
    }
}

// ------------------------------------------------------------------ combine
// One thread per 8 output columns of one token; slots in order, one RN product and one RN add.
// KC > 0: k == KC, known when compiled, so every slot's row is loaded before the first is added
// (the sum runs in slot order either way); KC == 0: any k.
template <int KC>
__global__ void __launch_bounds__(256) combine_kernel(const uint16_t *__restrict__ yhat, const int32_t *__restrict__ row_of,
                                                      const float *__restrict__ w, int64_t T, int k, int64_t d,
                                                      uint16_t *__restrict__ y) {
    // one token per block iteration, eight columns per thread and step: no index division
    const int64_t per_tok = d / 8;
    for (int64_t t = blockIdx.x; t < T; t += gridDim.x)
    for (int64_t ci = threadIdx.x; ci < per_tok; ci += blockDim.x) {
        const int64_t c = ci * 8;
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        if constexpr (KC > 0) {
            uint4 q[KC];
            float wk[KC];
#pragma unroll
            for (int j = 0; j < KC; ++j) {
                const int64_t row = row_of[t * KC + j];
                wk[j] = w != nullptr ? w[t * KC + j] : 1.0f;
                q[j] = __ldg(reinterpret_cast<const uint4 *>(yhat + row * d + c));
            }
#pragma unroll
            for (int j = 0; j < KC; ++j) {
                const uint32_t ws[4] = {q[j].x, q[j].y, q[j].z, q[j].w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    acc[2 * i] = __fadd_rn(acc[2 * i], __fmul_rn(wk[j], bf16_lo(ws[i])));
                    acc[2 * i + 1] = __fadd_rn(acc[2 * i + 1], __fmul_rn(wk[j], bf16_hi(ws[i])));
                }
            }
        }
        for (int j = 0; KC == 0 && j < k; ++j) {
            const int64_t row = row_of[t * k + j];
            // without weights (the dispatch's gradient) each slot's value is added as it is: the
            // product by 1 is exact
            const float wj = w != nullptr ? w[t * k + j] : 1.0f;
            const uint4 q = __ldg(reinterpret_cast<const uint4 *>(yhat + row * d + c));
            const uint32_t ws[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                acc[2 * i] = __fadd_rn(acc[2 * i], __fmul_rn(wj, bf16_lo(ws[i])));
                acc[2 * i + 1] = __fadd_rn(acc[2 * i + 1], __fmul_rn(wj, bf16_hi(ws[i])));
            }
        }
        uint32_t p[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
            p[i] = (uint32_t)f32_to_bf16_bits(acc[2 * i]) | ((uint32_t)f32_to_bf16_bits(acc[2 * i + 1]) << 16);
        *reinterpret_cast<uint4 *>(y + t * d + c) = make_uint4(p[0], p[1], p[2], p[3]);
    }
}

// ------------------------------------------------------------------ SGD on FP32 master weights
__global__ void __launch_bounds__(256) sgd_kernel(float *__restrict__ w32, const float *__restrict__ dw, int64_t n,
                                                  float lr, uint16_t *__restrict__ wb) {
    for (int64_t q = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; q < n / 4; q += (int64_t)gridDim.x * blockDim.x) {
        float4 w = reinterpret_cast<float4 *>(w32)[q];
        const float4 g = __ldg(reinterpret_cast<const float4 *>(dw) + q);
        w.x = __fsub_rn(w.x, __fmul_rn(lr, g.x));
        w.y = __fsub_rn(w.y, __fmul_rn(lr, g.y));
        w.z = __fsub_rn(w.z, __fmul_rn(lr, g.z));
        w.w = __fsub_rn(w.w, __fmul_rn(lr, g.w));
        reinterpret_cast<float4 *>(w32)[q] = w;
        const uint32_t lo = (uint32_t)f32_to_bf16_bits(w.x) | ((uint32_t)f32_to_bf16_bits(w.y) << 16);
        const uint32_t hi = (uint32_t)f32_to_bf16_bits(w.z) | ((uint32_t)f32_to_bf16_bits(w.w) << 16);
        reinterpret_cast<uint2 *>(wb)[q] = make_uint2(lo, hi);
    }
}

static unsigned grid_cap(int64_t items, int per_block, int per_sm) {
    int64_t g = (items + per_block - 1) / per_block;
    const int64_t cap = (int64_t)num_sms() * per_sm;
    if (g > cap) g = cap;
    return (unsigned)(g < 1 ? 1 : g);
}

}  // namespace moe4

using namespace moe4;

extern "C" int moe4_route_topk(const float *logits, int64_t T, int64_t E, int64_t k, int32_t *idx, float *w,
                               void *stream) {
    MOE4_CHECK_ARG(T >= 0 && E >= 1 && E <= 4096 && k >= 1 && k <= 32 && k <= E);
    MOE4_CHECK_ARG(T == 0 || (logits && idx && w));
    if (T == 0) return MOE4_OK;
    route_topk_kernel<<<grid_cap(T * 32, 256, 16), 256, 0, as_stream(stream)>>>(logits, T, (int)E, (int)k, idx, w);
    return launch_status();
}

extern "C" int moe4_permute_plan(const int32_t *idx, int64_t T, int64_t k, int64_t E, int32_t *offs,
                                 int32_t *row_of, int32_t *src_of, int64_t rows_cap, void *ws, size_t ws_bytes,
                                 void *stream) {
    MOE4_CHECK_ARG(T >= 0 && k >= 1 && E >= 1 && E <= 4096 && offs);
    // row indices and offsets are int32: the padded row count must fit
    MOE4_CHECK_ARG(T <= INT32_MAX && k <= INT32_MAX && T * k + 127 * E <= INT32_MAX);
    MOE4_CHECK_ARG(rows_cap >= T * k + 127 * E);
    MOE4_CHECK_ARG(T == 0 || (idx && row_of && src_of));
    const int64_t n = T * k;
    const int64_t nchunks = (n + kChunk - 1) / kChunk;
    const size_t need = (size_t)(nchunks * E + E) * sizeof(int32_t);
    if (!ws || ws_bytes < need) return MOE4_ERR_WORKSPACE;
    cudaStream_t st = as_stream(stream);
    int32_t *chunk = static_cast<int32_t *>(ws);
    int32_t *totals = chunk + nchunks * E;
    if (src_of && cudaMemsetAsync(src_of, 0xFF, (size_t)rows_cap * sizeof(int32_t), st) != cudaSuccess)
        return MOE4_ERR_CUDA;
    const size_t smem = (size_t)E * sizeof(int32_t);
    if (nchunks > 0) plan_count_kernel<<<(unsigned)nchunks, 256, smem, st>>>(idx, n, (int)E, chunk);
    plan_scan_kernel<<<1, 1024, 0, st>>>(chunk, nchunks, (int)E, totals, offs);
    if (nchunks > 0)
        plan_assign_kernel<<<(unsigned)nchunks, 32, smem, st>>>(idx, n, (int)k, (int)E, chunk, offs, row_of, src_of);
    return launch_status();
}

extern "C" int moe4_permute_nvfp4(const uint8_t *codes, const uint8_t *sf, int64_t T, int64_t cols,
                                  const int32_t *src_of, int64_t rows_total, uint8_t *out_codes, uint8_t *out_sf,
                                  uint32_t flags, void *stream) {
    MOE4_CHECK_ARG(T >= 0 && cols > 0 && cols % 32 == 0 && rows_total >= 0);
    MOE4_CHECK_ARG(src_of && out_codes && out_sf && (T == 0 || (codes && sf)));
    MOE4_CHECK_ARG(aligned16(codes) && aligned16(out_codes) && aligned16(sf) && aligned16(out_sf));
    MOE4_CHECK_ARG(flags == 0 || flags == MOE4_SF_MMA_LAYOUT || flags == MOE4_MXFP8);
    const bool sf_mma = (flags & MOE4_SF_MMA_LAYOUT) != 0;
    const bool mx = (flags & MOE4_MXFP8) != 0;
    MOE4_CHECK_ARG(!sf_mma || (rows_total % 128 == 0 && cols % 64 == 0));
    if (rows_total == 0) return MOE4_OK;
    permute_rows_kernel<<<grid_cap(rows_total * 32, 256, 16), 256, 0, as_stream(stream)>>>(
        codes, sf, mx ? cols : cols / 2, mx ? cols / 32 : cols / 16, src_of, rows_total, out_codes, out_sf, sf_mma);
    return launch_status();
}

extern "C" int moe4_swiglu(const float *gu, int64_t rows, int64_t f, uint16_t *h, void *stream) {
    MOE4_CHECK_ARG(rows >= 0 && f > 0 && f % 4 == 0);
    MOE4_CHECK_ARG(rows == 0 || (gu && h && aligned16(gu) && (reinterpret_cast<uintptr_t>(h) & 7u) == 0));
    if (rows == 0) return MOE4_OK;
    swiglu_kernel<false><<<grid_cap(rows * f / 4, 256, 8), 256, 0, as_stream(stream)>>>(gu, rows, f, h, nullptr);
    return launch_status();
}

extern "C" int moe4_swiglu_amax(const float *gu, int64_t rows, int64_t f, uint16_t *h, float *amax_out,
                                void *stream) {
    MOE4_CHECK_ARG(rows >= 0 && f > 0 && f % 4 == 0 && amax_out && aligned4(amax_out));
    MOE4_CHECK_ARG(rows == 0 || (gu && h && aligned16(gu) && (reinterpret_cast<uintptr_t>(h) & 7u) == 0));
    cudaStream_t st = as_stream(stream);
    if (cudaMemsetAsync(amax_out, 0, sizeof(float), st) != cudaSuccess) return MOE4_ERR_CUDA;
    if (rows == 0) return MOE4_OK;
    swiglu_kernel<true><<<grid_cap(rows * f / 4, 256, 8), 256, 0, st>>>(gu, rows, f, h,
                                                                        reinterpret_cast<unsigned int *>(amax_out));
    return launch_status();
}

extern "C" int moe4_swiglu_backward(const float *gu, const float *dh, int64_t rows, int64_t f, uint16_t *dgu,
                                    void *stream) {
    MOE4_CHECK_ARG(rows >= 0 && f > 0 && f % 4 == 0 && gu && dh && dgu && aligned16(gu) && aligned16(dh) &&
                   (reinterpret_cast<uintptr_t>(dgu) & 7u) == 0);
    if (rows == 0) return MOE4_OK;
    swiglu_bwd_kernel<<<grid_cap(rows * 256, 256, 8), 256, 0, as_stream(stream)>>>(gu, dh, rows, f, dgu);
    return launch_status();
}

extern "C" int moe4_combine_backward(const uint16_t *dy, const int32_t *row_of, const float *w, const int32_t *src_of,
                                     int64_t T, int64_t k, int64_t d, int64_t rows_total, uint16_t *dyhat,
                                     void *stream) {
    MOE4_CHECK_ARG(T >= 0 && k >= 1 && k <= 32 && d > 0 && d % 8 == 0 && rows_total >= 0);
    MOE4_CHECK_ARG(src_of && dyhat && aligned16(dyhat) && (T == 0 || (dy && row_of && w && aligned16(dy))));
    if (rows_total == 0) return MOE4_OK;
    combine_bwd_kernel<<<grid_cap(rows_total * 32, 256, 16), 256, 0, as_stream(stream)>>>(dy, row_of, w, src_of,
                                                                                           (int)k, d, rows_total, dyhat);
    return launch_status();
}

extern "C" int moe4_combine(const uint16_t *yhat, const int32_t *row_of, const float *w, int64_t T, int64_t k,
                            int64_t d, uint16_t *y, void *stream) {
    MOE4_CHECK_ARG(T >= 0 && k >= 1 && k <= 32 && d > 0 && d % 8 == 0);
    MOE4_CHECK_ARG(T == 0 || (yhat && row_of && w && y && aligned16(yhat) && aligned16(y)));
    if (T == 0) return MOE4_OK;
    if (k == 8)
        combine_kernel<8><<<grid_cap(T * 256, 256, 8), 256, 0, as_stream(stream)>>>(yhat, row_of, w, T, (int)k, d, y);
    else
        combine_kernel<0><<<grid_cap(T * 256, 256, 8), 256, 0, as_stream(stream)>>>(yhat, row_of, w, T, (int)k, d, y);
    return launch_status();
}

extern "C" int moe4_dispatch_backward(const uint16_t *dxp, const int32_t *row_of, int64_t T, int64_t k, int64_t d,
                                      uint16_t *dx, void *stream) {
    MOE4_CHECK_ARG(T >= 0 && k >= 1 && k <= 32 && d > 0 && d % 8 == 0);
    MOE4_CHECK_ARG(T == 0 || (dxp && row_of && dx && aligned16(dxp) && aligned16(dx)));
    if (T == 0) return MOE4_OK;
    if (k == 8)
        combine_kernel<8><<<grid_cap(T * 256, 256, 8), 256, 0, as_stream(stream)>>>(dxp, row_of, nullptr, T, (int)k, d, dx);
    else
        combine_kernel<0><<<grid_cap(T * 256, 256, 8), 256, 0, as_stream(stream)>>>(dxp, row_of, nullptr, T, (int)k, d, dx);
    return launch_status();
}

extern "C" int moe4_sgd_update(float *w32, const float *dw, int64_t n, float lr, uint16_t *w_bf16, void *stream) {
    MOE4_CHECK_ARG(n >= 0 && n % 4 == 0);
    MOE4_CHECK_ARG(n == 0 || (w32 && dw && w_bf16 && aligned16(w32) && aligned16(dw) &&
                              (reinterpret_cast<uintptr_t>(w_bf16) & 7u) == 0));
    if (n == 0) return MOE4_OK;
    sgd_kernel<<<grid_cap(n / 4, 256, 8), 256, 0, as_stream(stream)>>>(w32, dw, n, lr, w_bf16);
    return launch_status();
}
