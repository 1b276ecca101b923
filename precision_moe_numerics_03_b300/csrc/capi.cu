// capi.cu -- library-level entry points: version, status, workspace sizes, the device's own
// conversions (for checking them against the definition), and the scale-factor layout change
// that the tensor-core GEMMs read.
#include "common.cuh"

namespace moe4 {

__global__ void __launch_bounds__(256) convert_kernel(int kind, const float *__restrict__ in, int64_t n,
                                                      void *__restrict__ out, const PhiloxKeys keys) {
    for (int64_t q = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; q < n / 4; q += (int64_t)gridDim.x * blockDim.x) {
        const float4 v = __ldg(reinterpret_cast<const float4 *>(in) + q);
        if (kind == 0) {
            const float v8[8] = {v.x, v.y, v.z, v.w, 0.f, 0.f, 0.f, 0.f};
            const uint32_t nib = e2m1x8_rn(v8);
            uint32_t bytes = 0;
#pragma unroll
            for (int i = 0; i < 4; ++i) bytes |= ((nib >> (4 * i)) & 0xFu) << (8 * i);
            reinterpret_cast<uint32_t *>(out)[q] = bytes;
        } else if (kind == 1) {
            reinterpret_cast<uint32_t *>(out)[q] = e4m3x4_rn(v.x, v.y, v.z, v.w);
        } else if (kind == 2) {
            const uint32_t lo = (uint32_t)f32_to_bf16_bits(v.x) | ((uint32_t)f32_to_bf16_bits(v.y) << 16);
            const uint32_t hi = (uint32_t)f32_to_bf16_bits(v.z) | ((uint32_t)f32_to_bf16_bits(v.w) << 16);
            reinterpret_cast<uint2 *>(out)[q] = make_uint2(lo, hi);
        } else {
            // the kernels' four-at-a-time rounding (integer fast path, per-element path otherwise);
            // indices 4q .. 4q+3 are half of Philox call q/2
            const Philox4 P = sr_words8_not((uint64_t)q >> 1, 0u, keys);
            reinterpret_cast<uint32_t *>(out)[q] =
                (q & 1) ? e4m3x4_sr_nw(v.x, v.y, v.z, v.w, P.z, P.w) : e4m3x4_sr_nw(v.x, v.y, v.z, v.w, P.x, P.y);
        }
    }
}

__global__ void __launch_bounds__(256) sr_words_kernel(const PhiloxKeys keys, uint32_t stream_id, uint64_t j0, int64_t nq,
                                                       uint4 *__restrict__ out) {
    for (int64_t q = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; q < nq; q += (int64_t)gridDim.x * blockDim.x) {
        const Philox4 w = sr_words8(j0 + (uint64_t)q, stream_id, keys);  // the numbers of 8 indices
        out[q] = make_uint4(w.x, w.y, w.z, w.w);
    }
}

// Canonical [nmat, rows, nblk] -> tile layout: one 32-bit word (4 consecutive blocks of one row)
// per thread, stored at (tile * nblk/4 + kg) * 512 + 16 * (row % 32) + 4 * ((row / 32) % 4).
__global__ void __launch_bounds__(256) sf_layout_kernel(const uint32_t *__restrict__ in, int64_t nmat, int64_t rows,
                                                        int64_t nblk, uint8_t *__restrict__ out) {
    const int64_t words_per_row = nblk / 4;
    const int64_t total = nmat * rows * words_per_row;
    for (int64_t w = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; w < total; w += (int64_t)gridDim.x * blockDim.x) {
        const int64_t grow = w / words_per_row;
        const int64_t kg = w - grow * words_per_row;
        const int64_t m = grow / rows;
        const int64_t row = grow - m * rows;
        const int64_t off = m * rows * nblk + ((row >> 7) * words_per_row + kg) * 512 + (row & 31) * 16 + ((row >> 5) & 3) * 4;
        *reinterpret_cast<uint32_t *>(out + off) = __ldg(in + w);
    }
}

}  // namespace moe4

using namespace moe4;

extern "C" int moe4_version(void) { return 100; }

extern "C" const char *moe4_status_string(int status) {
    switch (status) {
        case MOE4_OK: return "ok";
        case MOE4_ERR_ARG: return "invalid argument (pointer, size, alignment or flag)";
        case MOE4_ERR_UNSUPPORTED: return "unsupported request";
        case MOE4_ERR_CUDA: return "CUDA error";
        case MOE4_ERR_TIMEOUT: return "a device-side wait timed out";
        case MOE4_ERR_WORKSPACE: return "workspace missing or too small";
        default: return "unknown status";
    }
}

extern "C" size_t moe4_workspace_size(int op, int64_t a, int64_t b, int64_t c) {
    switch (op) {
        case MOE4_OP_NVFP4_QUANTIZE: return (size_t)(a > 0 ? a : 1) * sizeof(unsigned int);
        case MOE4_OP_HADAMARD_QUANT: return sizeof(unsigned int);
        case MOE4_OP_PERMUTE_PLAN: {
            const int64_t n = a * b;
            const int64_t nchunks = (n + 1023) / 1024;
            return (size_t)(nchunks * c + c) * sizeof(int32_t);
        }
        default: return 0;
    }
}

extern "C" size_t moe4_workspace_size_gemm(int kind, int64_t a_rows, int64_t E, int64_t b_rows, int64_t K) {
    const int64_t blk = kind == 0 ? 16 : 32;
    const size_t a = (size_t)(a_rows * (K / blk));
    const size_t b = (size_t)(E * b_rows * (K / blk));
    // MXFP8: room for the contraction-grouped kernels' expert order (up to 4096 experts)
    const size_t order = kind == 1 ? 4096 * sizeof(int32_t) : 0;
    return ((a + 255) / 256 * 256) + ((b + 255) / 256 * 256) + order;
}

extern "C" int moe4_check_group_offsets(const int32_t *offs_host, int64_t E, int64_t total, int64_t align) {
    MOE4_CHECK_ARG(offs_host && E >= 1 && total >= 0 && align >= 1);
    MOE4_CHECK_ARG(offs_host[0] == 0 && (int64_t)offs_host[E] == total);
    for (int64_t e = 0; e < E; ++e) {
        MOE4_CHECK_ARG(offs_host[e + 1] >= offs_host[e]);
        MOE4_CHECK_ARG((int64_t)offs_host[e + 1] % align == 0);
    }
    return MOE4_OK;
}

extern "C" int moe4_convert(int kind, const float *in, int64_t n, void *out, void *stream) {
    MOE4_CHECK_ARG(kind >= 0 && kind <= 3 && n >= 0 && n % 4 == 0 && in && out && aligned16(in) && aligned4(out));
    // bf16 output is stored eight bytes (four values) at a time
    MOE4_CHECK_ARG(kind != 2 || (reinterpret_cast<uintptr_t>(out) & 7u) == 0);
    if (n == 0) return MOE4_OK;
    int64_t grid = (n / 4 + 255) / 256;
    if (grid > (int64_t)num_sms() * 16) grid = (int64_t)num_sms() * 16;
    convert_kernel<<<(unsigned)grid, 256, 0, as_stream(stream)>>>(kind, in, n, out, philox_keys(0));
    return launch_status();
}

extern "C" int moe4_sr_words(uint64_t seed, uint32_t stream_id, uint64_t idx_base, int64_t n, uint16_t *out,
                             void *stream) {
    MOE4_CHECK_ARG(n >= 0 && n % 8 == 0 && idx_base % 8 == 0 && out && aligned16(out));
    if (n == 0) return MOE4_OK;
    int64_t grid = (n / 8 + 255) / 256;
    if (grid > (int64_t)num_sms() * 16) grid = (int64_t)num_sms() * 16;
    sr_words_kernel<<<(unsigned)grid, 256, 0, as_stream(stream)>>>(philox_keys(seed), stream_id, idx_base / 8, n / 8,
                                                                   reinterpret_cast<uint4 *>(out));
    return launch_status();
}

extern "C" int moe4_sf_to_mma_layout(const uint8_t *sf, int64_t nmat, int64_t rows, int64_t nblk, uint8_t *out,
                                     void *stream) {
    MOE4_CHECK_ARG(nmat >= 1 && rows >= 0 && rows % 128 == 0 && nblk > 0 && nblk % 4 == 0);
    MOE4_CHECK_ARG(sf && out && aligned4(sf) && aligned4(out));
    const int64_t words = nmat * rows * nblk / 4;
    if (words == 0) return MOE4_OK;
    int64_t grid = (words + 255) / 256;
    if (grid > (int64_t)num_sms() * 16) grid = (int64_t)num_sms() * 16;
    sf_layout_kernel<<<(unsigned)grid, 256, 0, as_stream(stream)>>>(reinterpret_cast<const uint32_t *>(sf), nmat,
                                                                    rows, nblk, out);
    return launch_status();
}
