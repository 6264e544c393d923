// Shared device helpers and the per-sequence device state of the decoder.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace dec {

constexpr int kMaxBatch = 64;     // sequences per call (compile-time bound for state arrays)
constexpr int kGroupB = 4;        // activation rows one GEMV CTA keeps in shared memory

// ------------------------------------------------------------------ dtypes
template <typename T> struct Vec16;          // 16 bytes of T
template <> struct Vec16<__nv_bfloat16> { static constexpr int N = 8; };
template <> struct Vec16<float> { static constexpr int N = 4; };
template <> struct Vec16<__half> { static constexpr int N = 8; };

__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }
__device__ __forceinline__ float to_f32(__half v) { return __half2float(v); }

template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) {
    return __float2bfloat16_rn(v);
}
template <> __device__ __forceinline__ __half from_f32<__half>(float v) { return __float2half_rn(v); }

// Launch with programmatic stream serialization: the kernel may start while
// its predecessor drains and must call griddepcontrol.wait before it reads
// the predecessor's results or writes anything the predecessor reads.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args... args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Second bf16 plane of an activation: the rounding residual v - bf16(v), so
// that hi + lo carries about 16 mantissa bits (the tensor-core GEMM reads both).
__device__ __forceinline__ void store_planes(__nv_bfloat16 *hi, __nv_bfloat16 *lo, size_t i, float v) {
    const __nv_bfloat16 h = __float2bfloat16_rn(v);
    hi[i] = h;
    if (lo) lo[i] = __float2bfloat16_rn(v - __bfloat162float(h));
}

// Unpack 16 bytes into floats.
__device__ __forceinline__ void unpack16(const uint4 &u, float (&f)[8], const __nv_bfloat16 *) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}
__device__ __forceinline__ void unpack16(const uint4 &u, float (&f)[8], const __half *) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        __half2 h = *reinterpret_cast<const __half2 *>(&w[i]);
        float2 t = __half22float2(h);
        f[2 * i] = t.x;
        f[2 * i + 1] = t.y;
    }
}
__device__ __forceinline__ void unpack16(const uint4 &u, float (&f)[4], const float *) {
    f[0] = __uint_as_float(u.x);
    f[1] = __uint_as_float(u.y);
    f[2] = __uint_as_float(u.z);
    f[3] = __uint_as_float(u.w);
}

__device__ __forceinline__ uint4 ld_stream(const void *p) {
    // weights are read once per step: keep them out of L1
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// Block-wide sum for blockDim.x a multiple of 32 (<= 1024).  `red` has 32 floats.
__device__ __forceinline__ float block_sum(float v, float *red) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    v = warp_sum(v);
    __syncthreads();
    if (lane == 0) red[warp] = v;
    __syncthreads();
    float t = lane < nw ? red[lane] : 0.f;
    t = warp_sum(t);
    return t;
}

// Q/K RMSNorm over head_dim and NeoX RoPE of one head held by one warp, each
// lane owning PL contiguous dims; RoPE partners (i, i + d/2) sit 16 lanes apart.
template <int PL>
__device__ __forceinline__ void norm_rope_lane(float (&v)[PL], const float *w, float eps, int D,
                                               const float2 *rope_row, int lane) {
    float ss = 0.f;
#pragma unroll
    for (int e = 0; e < PL; ++e) ss += v[e] * v[e];
    ss = warp_sum(ss);
    const float r = rsqrtf(ss / (float)D + eps);
#pragma unroll
    for (int e = 0; e < PL; ++e) v[e] = v[e] * r * w[lane * PL + e];
#pragma unroll
    for (int e = 0; e < PL; ++e) {
        const float p = __shfl_xor_sync(0xffffffffu, v[e], 16);
        const float2 cs = rope_row[(lane & 15) * PL + e];
        v[e] = lane < 16 ? (v[e] * cs.x - p * cs.y) : (v[e] * cs.x + p * cs.y);
    }
}

// ------------------------------------------------------------------ state
// Per-sequence decode state, resident in the workspace.  The step kernels
// read it on the device so a captured CUDA graph replays any step.
struct SeqState {
    int32_t cur_tok[kMaxBatch];   // token fed to the next step
    int32_t n_past[kMaxBatch];    // position of the row processed by the next step
    int32_t kv_off[kMaxBatch];    // first KV slot of the sequence in the pool
    int32_t kv_cap[kMaxBatch];    // KV slots of the sequence
    int32_t active[kMaxBatch];    // 1: row takes part in steps
    int32_t done[kMaxBatch];      // 1: EOS, budget or KV full reached
    int32_t gen[kMaxBatch];       // ids generated so far (the prefill's counts)
    int32_t max_new;              // generation budget of the running loop
    int32_t eos_id;
    int32_t n_seq;
    int32_t error;                // first device-side error code (0 = none)
};

// both flags are loaded before either is tested (one memory round trip)
__device__ __forceinline__ bool row_live(const SeqState *st, int b) {
    const int act = st->active[b], dn = st->done[b];
    return act && !dn;
}

}  // namespace dec
