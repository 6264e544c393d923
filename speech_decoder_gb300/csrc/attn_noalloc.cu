// dec_attn_decode_noalloc: the split-KV decode attention for callers that
// cannot allocate device memory.
//
// Some callers have no way to hand the library a scratch buffer: code that
// runs inside a host engine or plugin interface whose device memory belongs
// to someone else and offers no allocator, or a latency-bound loop that must
// not call cudaMalloc (it can synchronise the whole device).  This entry point
// needs no scratch argument: the per-split partials and the arrival counters
// live in one file-scope device array that every call shares.
#include <mutex>

#include "dec.h"
#include "decode.cuh"

namespace {

// 4 MiB of device memory, reserved on every GPU that loads the library and
// held until the process exits.  A call needs B * n_kv_heads * splits *
// n_rep * (head_dim + 2) floats of partials plus B * n_kv_heads counters,
// each rounded up to 256 bytes (attn_op_scratch_bytes); the split count
// falls to 1 once B * n_kv_heads reaches twice the SM count.  For the 1.7B
// shape (8 KV heads, 2 query heads each, head_dim 128) that admits up to 502
// sequences.
constexpr size_t kNoAllocScratchBytes = size_t(4) << 20;
__device__ __align__(256) unsigned char g_attn_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_scratch_ptr[kMaxDevices] = {};   // device address of g_attn_scratch, per device

}  // namespace

extern "C" dec_status dec_attn_decode_noalloc(const float *q, const void *K, const void *V, int32_t kv_dtype,
                                              int32_t slots, const int32_t *kv_off, const int32_t *kv_len,
                                              int32_t B, int32_t n_heads, int32_t n_kv_heads, int32_t head_dim,
                                              float *out, void *stream) {
    if (!q || !K || !V || !kv_off || !kv_len || !out ||
        !dec::attn_op_shape_ok(B, n_heads, n_kv_heads, head_dim, slots, kv_dtype == DEC_F16 || kv_dtype == DEC_F32))
        return DEC_ERR_INVALID_ARG;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return DEC_ERR_CUDA;
    if (dec::attn_op_scratch_bytes(B, n_heads, n_kv_heads, head_dim, sms) > kNoAllocScratchBytes)
        return DEC_ERR_OOM;                      // shape needs more than the fixed 4 MiB
    void *scratch = nullptr;
    {
        // First call on a device: look up the array's device address with that
        // device current.  The host-side name g_attn_scratch is only a stand-in
        // and must never be passed to a kernel.
        std::lock_guard<std::mutex> lock(g_mu);
        if (!g_scratch_ptr[dev]) {
            void *p = nullptr;
            if (cudaGetSymbolAddress(&p, g_attn_scratch) != cudaSuccess || !p) return DEC_ERR_CUDA;
            g_scratch_ptr[dev] = p;
        }
        scratch = g_scratch_ptr[dev];
    }
    // attn_op_launch zeroes the counters (cudaMemsetAsync, no allocation);
    // the partials are fully rewritten by every call before they are read.
    const cudaError_t e = dec::attn_op_launch(q, K, V, kv_dtype == DEC_F16, slots, kv_off, kv_len, B, n_heads,
                                              n_kv_heads, head_dim, out, scratch, sms,
                                              static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? DEC_OK : DEC_ERR_CUDA;
}
