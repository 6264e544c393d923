// Prefill-path kernels: row RMSNorm, CUDA-core GEMM (fp32 debug build and
// reference for the tensor-core GEMM), packed SwiGLU, Q/K-norm + NeoX RoPE +
// KV write, causal GQA attention, and prompt assembly.
//
// Prefill structure (qwen3_asr/decoder.cpp, build_prefill_graph): token rows
// and encoder rows are concatenated (prefix | enc_out | suffix), every block
// runs on all rows with the causal mask of qwen3_asr/model.cpp, run (key c
// visible to query r iff c <= r), the KV of every position is written.
#include <type_traits>
#include "prefill.cuh"

namespace dec {

// ------------------------------------------------------------------ RMSNorm
template <typename TO>
__global__ void __launch_bounds__(256) k_rmsnorm_rows(const float *x, const float *w, float eps, TO *out,
                                                      TO *out_lo, int H) {
    __shared__ float red[32];
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const size_t t = blockIdx.x;
    const float *xr = x + t * H;
    float ss = 0.f;
    for (int k = threadIdx.x; k < H; k += blockDim.x) ss += xr[k] * xr[k];
    ss = block_sum(ss, red);
    const float r = rsqrtf(ss / (float)H + eps);
    for (int k = threadIdx.x; k < H; k += blockDim.x) {
        const float v = xr[k] * r * w[k];
        if constexpr (std::is_same<TO, __half>::value) out[t * H + k] = __float2half_rn(v);
        else if constexpr (sizeof(TO) == 2) store_planes(out, out_lo, t * H + k, v);
        else out[t * H + k] = v;
    }
}

void launch_rmsnorm_rows_f16(const float *x, const float *w, float eps, void *out, int T, int H, cudaStream_t s) {
    if (T <= 0) return;
    launch_pdl(k_rmsnorm_rows<__half>, dim3(T), dim3(256), 0, s, x, w, eps, (__half *)out, (__half *)nullptr, H);
}

void launch_rmsnorm_rows(const float *x, const float *w, float eps, void *out, void *out_lo, bool act_bf16, int T,
                         int H, cudaStream_t s) {
    if (T <= 0) return;
    if (act_bf16)
        launch_pdl(k_rmsnorm_rows<__nv_bfloat16>, dim3(T), dim3(256), 0, s, x, w, eps, (__nv_bfloat16 *)out,
                   (__nv_bfloat16 *)out_lo, H);
    else launch_pdl(k_rmsnorm_rows<float>, dim3(T), dim3(256), 0, s, x, w, eps, (float *)out, (float *)nullptr, H);
}

// ------------------------------------------------------------------ bf16 -> fp16 (weights, once)
__global__ void k_bf16_to_f16(const __nv_bfloat16 *src, __half *dst, size_t n) {
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x)
        dst[i] = __float2half_rn(__bfloat162float(src[i]));
}

void launch_bf16_to_f16(const void *src, void *dst, size_t n, cudaStream_t s) {
    if (n == 0) return;
    const size_t blocks = (n + 255) / 256;
    k_bf16_to_f16<<<(unsigned)(blocks < 65535 * 8 ? blocks : 65535 * 8), 256, 0, s>>>(
        static_cast<const __nv_bfloat16 *>(src), static_cast<__half *>(dst), n);
}

// ------------------------------------------------------------------ two bf16 planes
__global__ void k_split_planes(const float *x, __nv_bfloat16 *hi, __nv_bfloat16 *lo, size_t n) {
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x)
        store_planes(hi, lo, i, x[i]);
}

void launch_split_planes(const float *x, void *hi, void *lo, size_t n, cudaStream_t s) {
    if (n == 0) return;
    const size_t blocks = (n + 255) / 256;
    k_split_planes<<<(unsigned)(blocks < 65535 * 8 ? blocks : 65535 * 8), 256, 0, s>>>(
        x, static_cast<__nv_bfloat16 *>(hi), static_cast<__nv_bfloat16 *>(lo), n);
}

// ------------------------------------------------------------------ SIMT GEMM
// 64x64 output tile per CTA, 16-deep k slices staged through shared memory,
// 4x4 outputs per thread.  K must be a multiple of 16.
template <typename TA, typename TW, int EPI>
__global__ void __launch_bounds__(256) k_gemm_simt(const TA *A, const TW *W, float *C, int ldc, int M, int N,
                                                   int K) {
    __shared__ float As[16][64 + 4];
    __shared__ float Ws[16][64 + 4];
    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
    const int m0 = blockIdx.y * 64, n0 = blockIdx.x * 64;
    const int lr = tid >> 2, lk = (tid & 3) * 4;
    float acc[4][4] = {};
    for (int k0 = 0; k0 < K; k0 += 16) {
        {
            const int m = m0 + lr, n = n0 + lr;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                As[lk + e][lr] = m < M ? to_f32(A[(size_t)m * K + k0 + lk + e]) : 0.f;
                Ws[lk + e][lr] = n < N ? to_f32(W[(size_t)n * K + k0 + lk + e]) : 0.f;
            }
        }
        __syncthreads();
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            float a[4], b[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) a[i] = As[k][ty * 4 + i];
#pragma unroll
            for (int j = 0; j < 4; ++j) b[j] = Ws[k][tx * 4 + j];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int m = m0 + ty * 4 + i;
        if (m >= M) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int n = n0 + tx * 4 + j;
            if (n >= N) continue;
            float *c = C + (size_t)m * ldc + n;
            if (EPI == EPI_STORE_F32) *c = acc[i][j];
            else *c += acc[i][j];
        }
    }
}

template <typename TA, typename TW>
static void gemm_simt_t(const void *A, const void *W, float *C, int ldc, int M, int N, int K, int epi,
                        cudaStream_t s) {
    dim3 grid((N + 63) / 64, (M + 63) / 64);
    if (epi == EPI_STORE_F32)
        k_gemm_simt<TA, TW, EPI_STORE_F32><<<grid, 256, 0, s>>>((const TA *)A, (const TW *)W, C, ldc, M, N, K);
    else
        k_gemm_simt<TA, TW, EPI_RESID_F32><<<grid, 256, 0, s>>>((const TA *)A, (const TW *)W, C, ldc, M, N, K);
}

void launch_gemm_simt(const void *A, bool a_bf16, const void *W, bool w_bf16, float *C, int ldc, int M, int N,
                      int K, int epi, cudaStream_t s) {
    if (M <= 0) return;
    if (a_bf16 && w_bf16) gemm_simt_t<__nv_bfloat16, __nv_bfloat16>(A, W, C, ldc, M, N, K, epi, s);
    else if (!a_bf16 && !w_bf16) gemm_simt_t<float, float>(A, W, C, ldc, M, N, K, epi, s);
    else if (!a_bf16 && w_bf16) gemm_simt_t<float, __nv_bfloat16>(A, W, C, ldc, M, N, K, epi, s);
    else gemm_simt_t<__nv_bfloat16, float>(A, W, C, ldc, M, N, K, epi, s);
}

// ------------------------------------------------------------------ SwiGLU
template <typename TO>
__global__ void k_swiglu(const float *gu, TO *h, TO *h_lo, int T, int F) {
    const size_t n = (size_t)T * F;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
        const size_t t = i / F;
        const int f = (int)(i % F), blk = f >> 7, j = f & 127;
        const float *row = gu + t * 2 * F;
        const float g = row[blk * 256 + j], u = row[blk * 256 + 128 + j];
        const float v = g / (1.f + expf(-g)) * u;
        if constexpr (sizeof(TO) == 2) store_planes(h, h_lo, i, v);
        else h[i] = v;
    }
}

void launch_swiglu(const float *gu, void *h, void *h_lo, bool act_bf16, int T, int F, cudaStream_t s) {
    if (T <= 0) return;
    const size_t n = (size_t)T * F;
    const int grid = (int)((n + 255) / 256 < 65535 * 4 ? (n + 255) / 256 : 65535 * 4);
    if (act_bf16) k_swiglu<__nv_bfloat16><<<grid, 256, 0, s>>>(gu, (__nv_bfloat16 *)h, (__nv_bfloat16 *)h_lo, T, F);
    else k_swiglu<float><<<grid, 256, 0, s>>>(gu, (float *)h, nullptr, T, F);
}

// ------------------------------------------------------------------ Q/K norm + RoPE + KV write
// One warp per (row, head): heads [0, nq) are queries, [nq, nq + nkv) are KV
// heads (the warp also copies that head's V).
template <typename TKV, int D>
__global__ void __launch_bounds__(256) k_qk_rope_kv(RopeKvArgs a) {
    constexpr int PL = D / 32;
    const int lane = threadIdx.x & 31;
    const long long gw = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int nh = a.nq + a.nkv;
    if (gw >= (long long)a.T * nh) return;
    const int t = (int)(gw / nh), hh = (int)(gw % nh);
    const int pos = a.row_pos[t];
    const size_t ldq = (size_t)(a.nq + 2 * a.nkv) * D;
    const float *row = a.qkv + (size_t)t * ldq;
    const float2 *rope_row = a.rope + (size_t)pos * (D / 2);
    float v[PL];
    if (hh < a.nq) {
#pragma unroll
        for (int e = 0; e < PL; ++e) v[e] = row[(size_t)hh * D + lane * PL + e];
        norm_rope_lane<PL>(v, a.qn_w, a.eps, D, rope_row, lane);
        TKV *q = reinterpret_cast<TKV *>(a.q_out) + ((size_t)t * a.nq + hh) * D + lane * PL;
#pragma unroll
        for (int e = 0; e < PL; ++e) q[e] = from_f32<TKV>(v[e]);
    } else {
        const int g = hh - a.nq;
        const size_t slot = ((size_t)g * a.slots + a.row_slot[t]) * D + lane * PL;
#pragma unroll
        for (int e = 0; e < PL; ++e) v[e] = row[(size_t)(a.nq + g) * D + lane * PL + e];
        norm_rope_lane<PL>(v, a.kn_w, a.eps, D, rope_row, lane);
        TKV *K = reinterpret_cast<TKV *>(a.Kc) + slot;
        TKV *V = reinterpret_cast<TKV *>(a.Vc) + slot;
        TKV *vt = a.vt ? reinterpret_cast<TKV *>(a.vt) + (size_t)(g * D + lane * PL) * a.vt_ld + a.row_vtcol[t] : nullptr;
#pragma unroll
        for (int e = 0; e < PL; ++e) {
            K[e] = from_f32<TKV>(v[e]);
            const TKV x = from_f32<TKV>(row[(size_t)(a.nq + a.nkv + g) * D + lane * PL + e]);
            V[e] = x;
            if (vt) vt[(size_t)e * a.vt_ld] = x;
        }
    }
}

void launch_qk_rope_kv(bool kv_f16, const RopeKvArgs &a, cudaStream_t s) {
    if (a.T <= 0) return;
    const long long warps = (long long)a.T * (a.nq + a.nkv);
    const int grid = (int)((warps + 7) / 8);
    if (kv_f16) {
        if (a.d == 128) k_qk_rope_kv<__half, 128><<<grid, 256, 0, s>>>(a);
        else k_qk_rope_kv<__half, 64><<<grid, 256, 0, s>>>(a);
    } else {
        if (a.d == 128) k_qk_rope_kv<float, 128><<<grid, 256, 0, s>>>(a);
        else k_qk_rope_kv<float, 64><<<grid, 256, 0, s>>>(a);
    }
}

// ------------------------------------------------------------------ V^T of cached keys
// vt[(g d + e) vt_ld + vt_col0 + j] = V[g][kv_off + j][e] for j < n_keys: tiles
// of 32 keys x 32 dims through shared memory (reads along dims, writes along keys).
template <int D>
__global__ void __launch_bounds__(256) k_vt_from_pool(const __half *V, __half *vt, int vt_ld, int slots, int kv_off,
                                                      int n_keys, int vt_col0) {
    __shared__ __half tile[32][33];
    const int g = blockIdx.z, j0 = blockIdx.x * 32, e0 = blockIdx.y * 32;
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;        // 8 rows of 32 threads
    for (int i = ty; i < 32; i += 8) {
        const int j = j0 + i;
        tile[i][tx] = j < n_keys ? V[((size_t)g * slots + kv_off + j) * D + e0 + tx] : __float2half(0.f);
    }
    __syncthreads();
    for (int i = ty; i < 32; i += 8) {
        const int j = j0 + tx;
        if (j < n_keys) vt[(size_t)(g * D + e0 + i) * vt_ld + vt_col0 + j] = tile[tx][i];
    }
}

void launch_vt_from_pool(const void *V, void *vt, int vt_ld, int slots, int nkv, int kv_off, int n_keys, int vt_col0,
                         cudaStream_t s) {
    if (n_keys <= 0) return;
    dim3 grid((n_keys + 31) / 32, 128 / 32, nkv);
    k_vt_from_pool<128><<<grid, 256, 0, s>>>(static_cast<const __half *>(V), static_cast<__half *>(vt), vt_ld, slots,
                                             kv_off, n_keys, vt_col0);
}

// ------------------------------------------------------------------ causal attention (CUDA cores)
// One warp per (query row, head); warps of a CTA share the head so that the
// keys they stream are reused from L1.  Online softmax in fp32.
template <typename TKV, typename TO, int D>
__global__ void __launch_bounds__(256) k_attn_prefill_simt(AttnPrefillArgs a, float scale) {
    constexpr int PL = D / 32;
    const int lane = threadIdx.x & 31;
    const long long gw = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
    if (gw >= (long long)a.T * a.nq) return;
    const int h = (int)(gw / a.T), t = (int)(gw % a.T);
    const int g = h / (a.nq / a.nkv);
    const int pos = a.row_pos[t];
    const int slot0 = a.row_slot[t] - pos;          // first slot of this row's sequence
    const TKV *q = reinterpret_cast<const TKV *>(a.q) + ((size_t)t * a.nq + h) * D + lane * PL;
    float qf[PL];
#pragma unroll
    for (int e = 0; e < PL; ++e) qf[e] = to_f32(q[e]);
    const TKV *Kc = reinterpret_cast<const TKV *>(a.Kc) + ((size_t)g * a.slots + slot0) * D + lane * PL;
    const TKV *Vc = reinterpret_cast<const TKV *>(a.Vc) + ((size_t)g * a.slots + slot0) * D + lane * PL;
    float m = -INFINITY, l = 0.f, acc[PL] = {};
    constexpr int KB = 8;                 // keys per batch: all loads issued before use
    for (int jb = 0; jb <= pos; jb += KB) {
        float kf[KB][PL], vf[KB][PL], sc[KB];
#pragma unroll
        for (int k = 0; k < KB; ++k) {
            const int j = jb + k;
#pragma unroll
            for (int e = 0; e < PL; ++e) {
                kf[k][e] = j <= pos ? to_f32(Kc[(size_t)j * D + e]) : 0.f;
                vf[k][e] = j <= pos ? to_f32(Vc[(size_t)j * D + e]) : 0.f;
            }
        }
#pragma unroll
        for (int k = 0; k < KB; ++k) {
            float d = 0.f;
#pragma unroll
            for (int e = 0; e < PL; ++e) d = fmaf(qf[e], kf[k][e], d);
            sc[k] = d;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
#pragma unroll
            for (int k = 0; k < KB; ++k) sc[k] += __shfl_xor_sync(0xffffffffu, sc[k], o);
        float mb = m;
#pragma unroll
        for (int k = 0; k < KB; ++k) {
            sc[k] = jb + k <= pos ? sc[k] * scale : -INFINITY;
            mb = fmaxf(mb, sc[k]);
        }
        const float corr = expf(m - mb);
        float ls = 0.f;
#pragma unroll
        for (int e = 0; e < PL; ++e) acc[e] *= corr;
#pragma unroll
        for (int k = 0; k < KB; ++k) {
            const float p = expf(sc[k] - mb);
            ls += p;
#pragma unroll
            for (int e = 0; e < PL; ++e) acc[e] = fmaf(p, vf[k][e], acc[e]);
        }
        l = l * corr + ls;
        m = mb;
    }
    const size_t oi = (size_t)t * a.nq * D + (size_t)h * D + lane * PL;
    const float inv = 1.f / l;
#pragma unroll
    for (int e = 0; e < PL; ++e) {
        if constexpr (sizeof(TO) == 2)
            store_planes(reinterpret_cast<__nv_bfloat16 *>(a.o), reinterpret_cast<__nv_bfloat16 *>(a.o_lo), oi + e,
                         acc[e] * inv);
        else reinterpret_cast<float *>(a.o)[oi + e] = acc[e] * inv;
    }
}

template <typename TKV, typename TO>
static void attn_prefill_t(const AttnPrefillArgs &a, cudaStream_t s) {
    const long long warps = (long long)a.T * a.nq;
    const int grid = (int)((warps + 7) / 8);
    const float scale = (float)(1.0 / sqrt((double)a.d));
    if (a.d == 128) k_attn_prefill_simt<TKV, TO, 128><<<grid, 256, 0, s>>>(a, scale);
    else k_attn_prefill_simt<TKV, TO, 64><<<grid, 256, 0, s>>>(a, scale);
}

void launch_attn_prefill_simt(bool kv_f16, bool out_bf16, const AttnPrefillArgs &a, cudaStream_t s) {
    if (a.T <= 0) return;
    if (kv_f16 && out_bf16) attn_prefill_t<__half, __nv_bfloat16>(a, s);
    else if (kv_f16) attn_prefill_t<__half, float>(a, s);
    else if (out_bf16) attn_prefill_t<float, __nv_bfloat16>(a, s);
    else attn_prefill_t<float, float>(a, s);
}

// ------------------------------------------------------------------ gathers
__global__ void k_gather_rows(const float *x, const int32_t *idx, float *out, int H) {
    const int b = blockIdx.x;
    const float *src = x + (size_t)idx[b] * H;
    for (int k = threadIdx.x; k < H; k += blockDim.x) out[(size_t)b * H + k] = src[k];
}

void launch_gather_rows(const float *x, const int32_t *idx, float *out, int B, int H, cudaStream_t s) {
    if (B > 0) k_gather_rows<<<B, 256, 0, s>>>(x, idx, out, H);
}

template <typename TW>
__global__ void k_assemble(const TW *embed, const int32_t *ids, const float *audio, float *x, int n_audio,
                           int prefix_len, int H) {
    const int t = blockIdx.x;
    float *dst = x + (size_t)t * H;
    if (t >= prefix_len && t < prefix_len + n_audio) {
        const float *src = audio + (size_t)(t - prefix_len) * H;
        for (int k = threadIdx.x; k < H; k += blockDim.x) dst[k] = src[k];
    } else {
        const int id = ids[t < prefix_len ? t : t - n_audio];
        const TW *src = embed + (size_t)id * H;
        for (int k = threadIdx.x; k < H; k += blockDim.x) dst[k] = to_f32(src[k]);
    }
}

void launch_assemble(const void *embed, bool w_bf16, const int32_t *ids, const float *audio, float *x, int T,
                     int n_audio, int prefix_len, int H, cudaStream_t s) {
    if (T <= 0) return;
    if (w_bf16)
        k_assemble<__nv_bfloat16><<<T, 256, 0, s>>>((const __nv_bfloat16 *)embed, ids, audio, x, n_audio,
                                                    prefix_len, H);
    else k_assemble<float><<<T, 256, 0, s>>>((const float *)embed, ids, audio, x, n_audio, prefix_len, H);
}

}  // namespace dec
