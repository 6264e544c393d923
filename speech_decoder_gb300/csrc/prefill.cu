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

// One warp per row for H = 128 NJ: lane L holds float4 groups L + 32 j of
// the row in registers, so all of a row's loads are in flight together, the
// sum of squares is a shuffle reduction and no block barrier is needed.
template <typename TO, int NJ>
__global__ void __launch_bounds__(256) k_rmsnorm_rows_w(const float *x, const float *w, float eps, TO *out,
                                                        TO *out_lo, int T) {
    constexpr int H = NJ * 128;
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int lane = threadIdx.x & 31;
    const size_t t = (size_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    if (t >= (size_t)T) return;
    const float4 *xr = reinterpret_cast<const float4 *>(x + t * H);
    float4 v[NJ];
#pragma unroll
    for (int j = 0; j < NJ; ++j) v[j] = xr[lane + 32 * j];
    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < NJ; ++j) ss += v[j].x * v[j].x + v[j].y * v[j].y + v[j].z * v[j].z + v[j].w * v[j].w;
    ss = warp_sum(ss);
    const float r = rsqrtf(ss / (float)H + eps);
    const float4 *w4 = reinterpret_cast<const float4 *>(w);
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
        const float4 g = w4[lane + 32 * j];
        const float y0 = v[j].x * r * g.x, y1 = v[j].y * r * g.y, y2 = v[j].z * r * g.z, y3 = v[j].w * r * g.w;
        const size_t o = t * H + 4 * (size_t)(lane + 32 * j);
        if constexpr (std::is_same<TO, __half>::value) {
            __half2 *hp = reinterpret_cast<__half2 *>(out + o);
            hp[0] = __floats2half2_rn(y0, y1);
            hp[1] = __floats2half2_rn(y2, y3);
        } else if constexpr (sizeof(TO) == 2) {
            store_planes(out, out_lo, o, y0);
            store_planes(out, out_lo, o + 1, y1);
            store_planes(out, out_lo, o + 2, y2);
            store_planes(out, out_lo, o + 3, y3);
        } else {
            *reinterpret_cast<float4 *>(out + o) = make_float4(y0, y1, y2, y3);
        }
    }
}

// the warp-per-row form for H in {512, 1024, 2048, 4096} with 16-byte aligned
// rows, from 512 rows (fewer rows, as in a batched step's 32, would occupy a
// handful of SMs: one CTA per row spreads them wider); false: not applicable
template <typename TO>
static bool rmsnorm_rows_w(const float *x, const float *w, float eps, TO *out, TO *out_lo, int T, int H,
                           cudaStream_t s) {
    if (T < 512 || ((uintptr_t)x | (uintptr_t)w | (uintptr_t)out | (uintptr_t)out_lo) % 16) return false;
    const dim3 grid((T + 7) / 8), block(256);
    switch (H) {
    case 512: launch_pdl(k_rmsnorm_rows_w<TO, 4>, grid, block, 0, s, x, w, eps, out, out_lo, T); return true;
    case 1024: launch_pdl(k_rmsnorm_rows_w<TO, 8>, grid, block, 0, s, x, w, eps, out, out_lo, T); return true;
    case 2048: launch_pdl(k_rmsnorm_rows_w<TO, 16>, grid, block, 0, s, x, w, eps, out, out_lo, T); return true;
    case 4096: launch_pdl(k_rmsnorm_rows_w<TO, 32>, grid, block, 0, s, x, w, eps, out, out_lo, T); return true;
    default: return false;
    }
}

void launch_rmsnorm_rows_f16(const float *x, const float *w, float eps, void *out, int T, int H, cudaStream_t s) {
    if (T <= 0) return;
    if (rmsnorm_rows_w(x, w, eps, (__half *)out, (__half *)nullptr, T, H, s)) return;
    launch_pdl(k_rmsnorm_rows<__half>, dim3(T), dim3(256), 0, s, x, w, eps, (__half *)out, (__half *)nullptr, H);
}

void launch_rmsnorm_rows(const float *x, const float *w, float eps, void *out, void *out_lo, bool act_bf16, int T,
                         int H, cudaStream_t s) {
    if (T <= 0) return;
    if (act_bf16 ? rmsnorm_rows_w(x, w, eps, (__nv_bfloat16 *)out, (__nv_bfloat16 *)out_lo, T, H, s)
                 : rmsnorm_rows_w(x, w, eps, (float *)out, (float *)nullptr, T, H, s))
        return;
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
// One CTA per (16 prompt rows, head): heads [0, nq) are queries, [nq, nq + nkv)
// keys, [nq + nkv, nq + 2 nkv) values; warp w takes rows w and w + 8, lane L
// the features L PL .. L PL + PL - 1 of the row's head.  Value heads also
// write V^T: the 16 rows are staged in shared memory and each V^T row gets
// its 16 columns as two 16-byte stores of 8 consecutive columns (one element
// per store would touch a whole 32-byte sector for 2 bytes); 8 rows whose
// columns are not consecutive from a multiple of 8 (a sequence boundary, a
// chunk at an odd position) are written element by element.
constexpr int kRopeRows = 16;

// PL consecutive features: one 16- or 8-byte load, one 8- or 4-byte store
// of fp16 values
template <int PL>
__device__ __forceinline__ void load_lane(const float *src, float (&v)[PL]) {
    if constexpr (PL == 4) {
        const float4 x = *reinterpret_cast<const float4 *>(src);
        v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
    } else if constexpr (PL == 2) {
        const float2 x = *reinterpret_cast<const float2 *>(src);
        v[0] = x.x; v[1] = x.y;
    } else {
#pragma unroll
        for (int e = 0; e < PL; ++e) v[e] = src[e];
    }
}
template <typename TKV, int PL>
__device__ __forceinline__ void store_lane(TKV *dst, const float (&v)[PL]) {
    if constexpr (std::is_same<TKV, __half>::value && PL == 4) {
        const __half2 lo = __floats2half2_rn(v[0], v[1]), hi = __floats2half2_rn(v[2], v[3]);
        uint2 pk;
        pk.x = *reinterpret_cast<const unsigned *>(&lo);
        pk.y = *reinterpret_cast<const unsigned *>(&hi);
        *reinterpret_cast<uint2 *>(dst) = pk;
    } else if constexpr (std::is_same<TKV, __half>::value && PL == 2) {
        *reinterpret_cast<__half2 *>(dst) = __floats2half2_rn(v[0], v[1]);
    } else {
#pragma unroll
        for (int e = 0; e < PL; ++e) dst[e] = from_f32<TKV>(v[e]);
    }
}

template <typename TKV, int D>
__global__ void __launch_bounds__(256) k_qk_rope_kv(RopeKvArgs a) {
    constexpr int PL = D / 32;
    __shared__ TKV tile[kRopeRows][D + 8];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int hh = blockIdx.y, t0 = blockIdx.x * kRopeRows;
    const size_t ldq = (size_t)(a.nq + 2 * a.nkv) * D;
    const bool is_v = hh >= a.nq + a.nkv;
#pragma unroll
    for (int i = 0; i < kRopeRows / 8; ++i) {
        const int tr = warp + 8 * i, t = t0 + tr;
        if (t >= a.T) break;                                   // warp-uniform
        float v[PL];
        load_lane<PL>(a.qkv + (size_t)t * ldq + (size_t)hh * D + lane * PL, v);
        if (!is_v) {
            const bool is_q = hh < a.nq;
            const float2 *rope_row = a.rope + (size_t)a.row_pos[t] * (D / 2);
            norm_rope_lane<PL>(v, is_q ? a.qn_w : a.kn_w, a.eps, D, rope_row, lane);
            TKV *dst = is_q ? reinterpret_cast<TKV *>(a.q_out) + ((size_t)t * a.nq + hh) * D
                            : reinterpret_cast<TKV *>(a.Kc) + ((size_t)(hh - a.nq) * a.slots + a.row_slot[t]) * D;
            store_lane<TKV, PL>(dst + lane * PL, v);
        } else {
            const int g = hh - a.nq - a.nkv;
            store_lane<TKV, PL>(reinterpret_cast<TKV *>(a.Vc) + ((size_t)g * a.slots + a.row_slot[t]) * D + lane * PL, v);
            store_lane<TKV, PL>(&tile[tr][lane * PL], v);
        }
    }
    if (!is_v || !a.vt) return;                                // CTA-uniform
    __syncthreads();
    if (threadIdx.x >= D) return;
    const int e = threadIdx.x, g = hh - a.nq - a.nkv;
    TKV *dst = reinterpret_cast<TKV *>(a.vt) + (size_t)(g * D + e) * a.vt_ld;
#pragma unroll
    for (int h8 = 0; h8 < kRopeRows; h8 += 8) {
        const int tb = t0 + h8;
        if (tb >= a.T) break;
        const int c0 = a.row_vtcol[tb];
        bool vec = sizeof(TKV) == 2 && tb + 7 < a.T && c0 % 8 == 0;
        for (int k = 1; vec && k < 8; ++k) vec = a.row_vtcol[tb + k] == c0 + k;
        if (vec) {
            uint4 pk;
            uint16_t *h = reinterpret_cast<uint16_t *>(&pk);
#pragma unroll
            for (int k = 0; k < 8; ++k) h[k] = *reinterpret_cast<const uint16_t *>(&tile[h8 + k][e]);
            *reinterpret_cast<uint4 *>(dst + c0) = pk;
        } else {
            for (int k = 0; k < 8 && tb + k < a.T; ++k) dst[a.row_vtcol[tb + k]] = tile[h8 + k][e];
        }
    }
}

void launch_qk_rope_kv(bool kv_f16, const RopeKvArgs &a, cudaStream_t s) {
    if (a.T <= 0) return;
    const dim3 grid((a.T + kRopeRows - 1) / kRopeRows, a.nq + 2 * a.nkv);
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
