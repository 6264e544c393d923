// Per-row e4m3 rounding of bf16 weights: the 1-byte weight format of the
// decode GEMVs (an extension of the weight-streaming path; the pages' decoder
// streams bf16 or f32 weights).
//
// Row r gets the scale 2^e, e the smallest integer with max_k |w[r][k]| <=
// 448 * 2^e (448: the largest finite e4m3 value), and code[r][k] = the e4m3
// value nearest w[r][k] / 2^e (ties to even; OCP 8-bit floating point, E4M3:
// exponent bias 7, 3 mantissa bits, subnormals, no infinities).  Scaling by a
// power of two is exact, and value(code) * 2^e has at most 4 significant bits,
// so the rounded weight is exact in bf16: the prompt GEMMs (bf16) and the step
// GEMVs (codes * scale) compute with the same weights.
#include <cuda_fp8.h>

#include "decode.cuh"

namespace dec {
namespace {

constexpr int kQT = 256;              // threads per row

__device__ __forceinline__ float e4m3_value(__nv_fp8_storage_t c) {
    return __half2float(__half(__nv_cvt_fp8_to_halfraw(c, __NV_E4M3)));
}

__global__ void __launch_bounds__(kQT) k_quantize_e4m3_rows(const __nv_bfloat16 *w, int cols, uint8_t *codes,
                                                            float *scales, __nv_bfloat16 *out) {
    __shared__ float red[kQT / 32];
    const size_t base = (size_t)blockIdx.x * cols;
    float m = 0.f;
    for (int k = threadIdx.x; k < cols; k += kQT) m = fmaxf(m, fabsf(__bfloat162float(w[base + k])));
    m = warp_max(m);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    m = 0.f;
#pragma unroll
    for (int i = 0; i < kQT / 32; ++i) m = fmaxf(m, red[i]);
    // smallest e with m <= 448 * 2^e: m / 448 = f * 2^x with f in [0.5, 1)
    int e = 0;
    if (m > 0.f) {
        int x;
        const float f = frexpf(m / 448.f, &x);
        e = f == 0.5f ? x - 1 : x;
    }
    const float scale = ldexpf(1.f, e), inv = ldexpf(1.f, -e);
    if (threadIdx.x == 0) scales[blockIdx.x] = scale;
    for (int k = threadIdx.x; k < cols; k += kQT) {
        const __nv_fp8_storage_t c = __nv_cvt_float_to_fp8(__bfloat162float(w[base + k]) * inv, __NV_SATFINITE,
                                                           __NV_E4M3);
        codes[base + k] = c;
        out[base + k] = __float2bfloat16(e4m3_value(c) * scale);
    }
}

}  // namespace

void launch_quantize_e4m3_rows(const void *w, size_t rows, int cols, uint8_t *codes, float *scales, void *out,
                               cudaStream_t s) {
    if (rows == 0) return;
    k_quantize_e4m3_rows<<<(unsigned)rows, kQT, 0, s>>>(static_cast<const __nv_bfloat16 *>(w), cols, codes, scales,
                                                         static_cast<__nv_bfloat16 *>(out));
}

}  // namespace dec
