// The NVFP4 quantiser's 6-candidate block scale t = a / 6 (csrc/quant.cu, nvfp4_candidate) is
// formed by Markstein's correction step on a clamped to FLT_MAX.  This program evaluates that
// step and the correctly rounded division __fdiv_rn(a, 6) for every binary32 a >= 0 (zero,
// subnormals, normals, +inf) and counts the a whose E4M3 codes (cvt.rn.satfinite) differ, and,
// for information, those whose binary32 quotients differ.  Prints one line; exit 0 unless CUDA
// fails.  Every index is bounded.
#include <cfloat>
#include <cstdint>
#include <cstdio>
__device__ __forceinline__ uint32_t e4m3_code(float v) {
    uint16_t out;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(out) : "f"(0.0f), "f"(v));
    return out & 0xFFu;
}
__global__ void check(unsigned long long *count) {
    const float y = __uint_as_float(0x3E2AAAABu);  // RN(1/6)
    for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i <= 0x7F800000ull;
         i += (uint64_t)gridDim.x * blockDim.x) {
        const float a = __uint_as_float((uint32_t)i);
        const float ref = __fdiv_rn(a, 6.0f);
        const float am = fminf(a, FLT_MAX);
        const float q0 = __fmul_rn(am, y);
        const float t = __fmaf_rn(__fmaf_rn(-q0, 6.0f, am), y, q0);
        if (e4m3_code(t) != e4m3_code(ref)) atomicAdd(count, 1ull);
        if (__float_as_uint(t) != __float_as_uint(ref)) atomicAdd(count + 1, 1ull);
    }
}
int main() {
    unsigned long long *d = nullptr, h[2] = {0, 0};
    if (cudaMalloc(&d, sizeof(h)) != cudaSuccess || cudaMemset(d, 0, sizeof(h)) != cudaSuccess) return 2;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0) != cudaSuccess || sms <= 0) return 2;
    check<<<sms * 16, 256>>>(d);
    if (cudaDeviceSynchronize() != cudaSuccess) return 3;
    if (cudaMemcpy(h, d, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) return 3;
    printf("code_mismatches %llu quotient_mismatches %llu\n", h[0], h[1]);
    return 0;
}
