// Decode-path kernels: weight-streaming GEMVs with fused prologues/epilogues
// and the split-KV GQA attention for one new token per sequence.
//
// Step structure (qwen3_asr/decoder.cpp, build_step_graph; block math from the
// file header of that page):
//   gemv  RMSNorm(x)*w_attn -> q|k|v            (layer 0: x = embed[token])
//   attn  Q/K RMSNorm + NeoX RoPE + KV append at slot n_past + split-KV softmax
//   gemv  x += o W_o^T
//   gemv  RMSNorm(x)*w_ffn -> gate|up
//   gemv  x += (silu(gate) * up) W_down^T
//   gemv  RMSNorm(x)*w_final -> logits = embed . y, argmax (lowest index on ties)
#include "decode.cuh"

namespace dec {

// ============================================================== GEMV
// One CTA owns a contiguous range of weight rows; each warp streams whole
// rows with 16-byte loads and reduces with shuffles.  Up to kGroupB
// activation rows (sequences) share every weight load.
template <typename TW, int IN, int OUT>
__global__ void __launch_bounds__(256) k_gemv(GemvArgs a) {
    extern __shared__ __align__(16) float xs[];      // [kGroupB][K]
    __shared__ float red[32];
    __shared__ float wbest_v[8][kGroupB];
    __shared__ int wbest_i[8][kGroupB];
    __shared__ int live_s[kGroupB];
    __shared__ unsigned ticket_s;

    const int K = a.K, N = a.N;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int b0 = blockIdx.y * kGroupB;
    const int nb = min(kGroupB, a.B - b0);

    // ---------------------------------------------------------- activations
    for (int bi = 0; bi < kGroupB; ++bi) {
        const int b = b0 + bi;
        const bool live = bi < nb && row_live(a.st, b);
        if (tid == 0) live_s[bi] = live;
        if (!live) continue;                               // uniform in the block
        float *xr = xs + (size_t)bi * K;
        if (IN == IN_PLAIN) {
            for (int k = tid; k < K; k += blockDim.x) xr[k] = a.in[(size_t)b * K + k];
        } else if (IN == IN_SWIGLU) {
            // packed gate|up: block j of 256 outputs = 128 gate rows, then 128 up rows
            const float *gu = a.in + (size_t)b * 2 * a.ffn;
            for (int f = tid; f < K; f += blockDim.x) {
                const int blk = f >> 7, j = f & 127;
                const float g = gu[blk * 256 + j], u = gu[blk * 256 + 128 + j];
                xr[f] = g / (1.f + expf(-g)) * u;
            }
        } else {
            float ss = 0.f;
            if (IN == IN_EMBED_NORM) {
                const int tok = a.st->cur_tok[b];
                const TW *er = reinterpret_cast<const TW *>(a.embed) + (size_t)tok * K;
                for (int k = tid; k < K; k += blockDim.x) {
                    const float v = to_f32(er[k]);
                    xr[k] = v;
                    ss += v * v;
                    if (blockIdx.x == 0) a.x_resid[(size_t)b * K + k] = v;
                }
            } else {
                for (int k = tid; k < K; k += blockDim.x) {
                    const float v = a.in[(size_t)b * K + k];
                    xr[k] = v;
                    ss += v * v;
                }
            }
            ss = block_sum(ss, red);
            const float r = rsqrtf(ss / (float)K + a.eps);
            for (int k = tid; k < K; k += blockDim.x) xr[k] = xr[k] * r * a.norm_w[k];
        }
    }
    __syncthreads();
    bool any_live = false;
#pragma unroll
    for (int bi = 0; bi < kGroupB; ++bi) any_live |= live_s[bi] != 0;
    if (!any_live && OUT != OUT_ARGMAX) return;        // finished rows stream no weights

    // ---------------------------------------------------------- rows
    constexpr int VEC = Vec16<TW>::N;
    constexpr int U = 4;
    const int nchunks = K / VEC;
    const int r0 = (int)((long long)N * blockIdx.x / gridDim.x);
    const int r1 = (int)((long long)N * (blockIdx.x + 1) / gridDim.x);
    float best_v[kGroupB];
    int best_i[kGroupB];
#pragma unroll
    for (int bi = 0; bi < kGroupB; ++bi) {
        best_v[bi] = -INFINITY;
        best_i[bi] = 0x7fffffff;
    }

    for (int r = r0 + warp; any_live && r < r1; r += 8) {
        const uint4 *wr = reinterpret_cast<const uint4 *>(reinterpret_cast<const TW *>(a.W) + (size_t)r * K);
        float acc[kGroupB];
#pragma unroll
        for (int bi = 0; bi < kGroupB; ++bi) acc[bi] = 0.f;
        for (int c0 = lane; c0 < nchunks; c0 += 32 * U) {
            uint4 wv[U];
#pragma unroll
            for (int u = 0; u < U; ++u)
                if (c0 + 32 * u < nchunks) wv[u] = ld_stream(wr + c0 + 32 * u);
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int c = c0 + 32 * u;
                if (c < nchunks) {
                    float f[VEC];
                    unpack16(wv[u], f, (const TW *)nullptr);
#pragma unroll
                    for (int bi = 0; bi < kGroupB; ++bi) {
                        if (bi < nb) {
                            const float *xv = xs + (size_t)bi * K + c * VEC;
#pragma unroll
                            for (int e = 0; e < VEC; ++e) acc[bi] = fmaf(f[e], xv[e], acc[bi]);
                        }
                    }
                }
            }
        }
#pragma unroll
        for (int bi = 0; bi < kGroupB; ++bi) acc[bi] = warp_sum(acc[bi]);
        if (lane == 0) {
#pragma unroll
            for (int bi = 0; bi < kGroupB; ++bi) {
                if (bi < nb && live_s[bi]) {
                    const size_t o = (size_t)(b0 + bi) * N + r;
                    if (OUT == OUT_STORE) a.out[o] = acc[bi];
                    if (OUT == OUT_RESID) a.out[o] += acc[bi];
                    if (OUT == OUT_ARGMAX) {
                        if (a.out) a.out[o] = acc[bi];
                        if (acc[bi] > best_v[bi]) {       // rows ascend: strict '>' keeps the lowest index
                            best_v[bi] = acc[bi];
                            best_i[bi] = r;
                        }
                    }
                }
            }
        }
    }
    if (OUT != OUT_ARGMAX) return;

    // ---------------------------------------------------------- argmax
    if (lane == 0) {
#pragma unroll
        for (int bi = 0; bi < kGroupB; ++bi) {
            wbest_v[warp][bi] = best_v[bi];
            wbest_i[warp][bi] = best_i[bi];
        }
    }
    __syncthreads();
    const int G = gridDim.x;
    if (tid < nb && live_s[tid]) {
        float bv = -INFINITY;
        int bix = 0x7fffffff;
        for (int w = 0; w < 8; ++w) {
            const float v = wbest_v[w][tid];
            const int i = wbest_i[w][tid];
            if (v > bv || (v == bv && i < bix)) { bv = v; bix = i; }
        }
        a.part_val[(size_t)(b0 + tid) * G + blockIdx.x] = bv;
        a.part_idx[(size_t)(b0 + tid) * G + blockIdx.x] = bix;
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) ticket_s = atomicAdd(a.counter, 1u);
    __syncthreads();
    if (ticket_s != gridDim.x * gridDim.y - 1) return;
    __threadfence();
    // last CTA: reduce every sequence's partials and advance the state
    __shared__ float rv[8];
    __shared__ int ri[8];
    for (int b = 0; b < a.B; ++b) {
        if (!row_live(a.st, b)) continue;
        float bv = -INFINITY;
        int bix = 0x7fffffff;
        for (int i = tid; i < G; i += blockDim.x) {
            const float v = __ldcg(a.part_val + (size_t)b * G + i);
            const int ix = __ldcg(a.part_idx + (size_t)b * G + i);
            if (v > bv || (v == bv && ix < bix)) { bv = v; bix = ix; }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float v = __shfl_xor_sync(0xffffffffu, bv, o);
            const int ix = __shfl_xor_sync(0xffffffffu, bix, o);
            if (v > bv || (v == bv && ix < bix)) { bv = v; bix = ix; }
        }
        if (lane == 0) { rv[warp] = bv; ri[warp] = bix; }
        __syncthreads();
        if (tid == 0) {
            for (int w = 1; w < 8; ++w)
                if (rv[w] > bv || (rv[w] == bv && ri[w] < bix)) { bv = rv[w]; bix = ri[w]; }
            SeqState *st = a.st;
            if (bix < 0 || bix >= N) {                  // every logit NaN
                if (st->error == 0) st->error = 2;
                bix = 0;
            }
            st->cur_tok[b] = bix;
            const int gcount = st->gen[b];
            if (gcount < a.out_ids_cap) a.out_ids[(size_t)b * a.out_ids_cap + gcount] = bix;
            st->gen[b] = gcount + 1;
            const int np = st->n_past[b] + 1;
            st->n_past[b] = np;
            if (bix == st->eos_id || gcount + 1 >= st->max_new || np + 1 > st->kv_cap[b]) st->done[b] = 1;
        }
        __syncthreads();
    }
    if (tid == 0) *a.counter = 0u;
}

int gemv_grid(int N, int num_sms) {
    const int by_rows = (N + 7) / 8;
    const int cap = num_sms * 4;
    return by_rows < cap ? by_rows : cap;
}

template <typename TW>
static void launch_gemv_t(int in_mode, int out_mode, const GemvArgs &a, int grid_x, cudaStream_t s) {
    const int nb = a.B < kGroupB ? a.B : kGroupB;
    const size_t smem = (size_t)nb * a.K * sizeof(float);
    dim3 grid(grid_x, (a.B + kGroupB - 1) / kGroupB);
#define DEC_GEMV_CASE(I, O)                                 \
    if (in_mode == I && out_mode == O) {                    \
        k_gemv<TW, I, O><<<grid, 256, smem, s>>>(a);        \
        return;                                             \
    }
    DEC_GEMV_CASE(IN_NORM, OUT_STORE)
    DEC_GEMV_CASE(IN_EMBED_NORM, OUT_STORE)
    DEC_GEMV_CASE(IN_PLAIN, OUT_RESID)
    DEC_GEMV_CASE(IN_SWIGLU, OUT_RESID)
    DEC_GEMV_CASE(IN_NORM, OUT_ARGMAX)
#undef DEC_GEMV_CASE
}

template <typename TW>
static void init_gemv_t() {
    const int smem = kGemvMaxSmem;
    cudaFuncSetAttribute(k_gemv<TW, IN_NORM, OUT_STORE>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    cudaFuncSetAttribute(k_gemv<TW, IN_EMBED_NORM, OUT_STORE>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    cudaFuncSetAttribute(k_gemv<TW, IN_PLAIN, OUT_RESID>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    cudaFuncSetAttribute(k_gemv<TW, IN_SWIGLU, OUT_RESID>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    cudaFuncSetAttribute(k_gemv<TW, IN_NORM, OUT_ARGMAX>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
}

void init_gemv_kernels() {
    init_gemv_t<__nv_bfloat16>();
    init_gemv_t<float>();
}

void launch_gemv(int in_mode, int out_mode, bool w_bf16, const GemvArgs &a, int grid_x, cudaStream_t s) {
    if (w_bf16) launch_gemv_t<__nv_bfloat16>(in_mode, out_mode, a, grid_x, s);
    else launch_gemv_t<float>(in_mode, out_mode, a, grid_x, s);
}

// ============================================================== attention
template <typename TKV, int PL>
__device__ __forceinline__ void load_kv(const TKV *p, float (&f)[PL]) {
#pragma unroll
    for (int e = 0; e < PL; ++e) f[e] = to_f32(p[e]);
}

constexpr int kMaxRep = 8;

template <typename TKV, int D, bool STEP>
__global__ void __launch_bounds__(128) k_attn_decode(AttnDecArgs a, float scale) {
    constexpr int PL = D / 32;
    __shared__ float qs[kMaxRep][D];
    __shared__ float wm[4][kMaxRep], wl[4][kMaxRep];
    __shared__ float wacc[4][kMaxRep][D];
    __shared__ unsigned ticket;

    const int g = blockIdx.x, s = blockIdx.y, S = gridDim.y, b = blockIdx.z;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int n_rep = a.nq / a.nkv;
    int pos, len, off;
    if (STEP) {
        if (!row_live(a.st, b)) return;
        pos = a.st->n_past[b];
        len = pos + 1;
        off = a.st->kv_off[b];
    } else {
        len = a.kv_len[b];
        off = a.kv_off[b];
        if (len <= 0 || off < 0 || (long long)off + len > (long long)a.slots) return;   // row skipped
        pos = len - 1;
    }
    const size_t ldq = (size_t)(a.nq + 2 * a.nkv) * D;
    const float *row = STEP ? a.qkv + (size_t)b * ldq : nullptr;
    const float2 *rope_row = STEP ? a.rope + (size_t)pos * (D / 2) : nullptr;
    TKV *Kc = reinterpret_cast<TKV *>(a.Kc);
    TKV *Vc = reinterpret_cast<TKV *>(a.Vc);

    for (int r = warp; r < n_rep; r += 4) {
        float v[PL];
        const float *src = STEP ? row + (size_t)(g * n_rep + r) * D + lane * PL
                                : a.q_plain + ((size_t)b * a.nq + g * n_rep + r) * D + lane * PL;
#pragma unroll
        for (int e = 0; e < PL; ++e) v[e] = src[e];
        if (STEP) norm_rope_lane<PL>(v, a.qn_w, a.eps, D, rope_row, lane);
#pragma unroll
        for (int e = 0; e < PL; ++e) qs[r][lane * PL + e] = v[e];
    }

    const int chunk = (len + S - 1) / S;
    const int j0 = min(len, s * chunk), j1 = min(len, j0 + chunk);
    if (STEP && a.append && j0 <= pos && pos < j1) {
        const size_t slot = ((size_t)g * a.slots + off + pos) * D + lane * PL;
        if (warp == 0) {
            float v[PL];
            const float *src = row + (size_t)(a.nq + g) * D + lane * PL;
#pragma unroll
            for (int e = 0; e < PL; ++e) v[e] = src[e];
            norm_rope_lane<PL>(v, a.kn_w, a.eps, D, rope_row, lane);
#pragma unroll
            for (int e = 0; e < PL; ++e) Kc[slot + e] = from_f32<TKV>(v[e]);
        } else if (warp == 1) {
            const float *src = row + (size_t)(a.nq + a.nkv + g) * D + lane * PL;
#pragma unroll
            for (int e = 0; e < PL; ++e) Vc[slot + e] = from_f32<TKV>(src[e]);
        }
    }
    __syncthreads();

    float m[kMaxRep], l[kMaxRep], acc[kMaxRep][PL];
#pragma unroll
    for (int r = 0; r < kMaxRep; ++r) {
        m[r] = -INFINITY;
        l[r] = 0.f;
#pragma unroll
        for (int e = 0; e < PL; ++e) acc[r][e] = 0.f;
    }
    for (int j = j0 + warp; j < j1; j += 4) {
        const size_t base = ((size_t)g * a.slots + off + j) * D + lane * PL;
        float kf[PL], vf[PL];
        load_kv<TKV, PL>(Kc + base, kf);
        load_kv<TKV, PL>(Vc + base, vf);
#pragma unroll
        for (int r = 0; r < kMaxRep; ++r) {
            if (r < n_rep) {
                float d = 0.f;
#pragma unroll
                for (int e = 0; e < PL; ++e) d = fmaf(qs[r][lane * PL + e], kf[e], d);
                const float sc = warp_sum(d) * scale;
                const float mn = fmaxf(m[r], sc);
                const float corr = expf(m[r] - mn);
                const float p = expf(sc - mn);
                l[r] = l[r] * corr + p;
#pragma unroll
                for (int e = 0; e < PL; ++e) acc[r][e] = fmaf(p, vf[e], acc[r][e] * corr);
                m[r] = mn;
            }
        }
    }
#pragma unroll
    for (int r = 0; r < kMaxRep; ++r) {
        if (r < n_rep) {
            if (lane == 0) { wm[warp][r] = m[r]; wl[warp][r] = l[r]; }
#pragma unroll
            for (int e = 0; e < PL; ++e) wacc[warp][r][lane * PL + e] = acc[r][e];
        }
    }
    __syncthreads();

    const int nkv = a.nkv;
    float *part = a.part + (((size_t)b * nkv + g) * S + s) * n_rep * (D + 2);
    for (int idx = tid; idx < n_rep * D; idx += blockDim.x) {
        const int r = idx / D, i = idx % D;
        float M = -INFINITY;
        for (int w = 0; w < 4; ++w) M = fmaxf(M, wm[w][r]);
        float A = 0.f, L = 0.f;
        if (M != -INFINITY) {
            for (int w = 0; w < 4; ++w) {
                const float f = expf(wm[w][r] - M);
                A += wacc[w][r][i] * f;
                L += wl[w][r] * f;
            }
        }
        float *pr = part + (size_t)r * (D + 2);
        pr[i] = A;
        if (i == 0) { pr[D] = M; pr[D + 1] = L; }
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) ticket = atomicAdd(&a.counter[b * nkv + g], 1u);
    __syncthreads();
    if (ticket != (unsigned)S - 1) return;
    __threadfence();

    // last split of this (sequence, kv head): log-sum-exp combine
    const float *pb = a.part + ((size_t)b * nkv + g) * S * n_rep * (D + 2);
    for (int idx = tid; idx < n_rep * D; idx += blockDim.x) {
        const int r = idx / D, i = idx % D;
        float Mx = -INFINITY;
        for (int t = 0; t < S; ++t) Mx = fmaxf(Mx, __ldcg(pb + ((size_t)t * n_rep + r) * (D + 2) + D));
        float A = 0.f, L = 0.f;
        for (int t = 0; t < S; ++t) {
            const float *pr = pb + ((size_t)t * n_rep + r) * (D + 2);
            const float Mt = __ldcg(pr + D);
            if (Mt == -INFINITY) continue;
            const float f = expf(Mt - Mx);
            A += __ldcg(pr + i) * f;
            L += __ldcg(pr + D + 1) * f;
        }
        a.o[(size_t)b * a.nq * D + (size_t)(g * n_rep + r) * D + i] = A / L;
    }
    if (tid == 0) a.counter[b * nkv + g] = 0u;
}

template <bool STEP>
static void attn_launch(bool kv_f16, const AttnDecArgs &a, int splits, cudaStream_t s) {
    dim3 grid(a.nkv, splits, a.B);
    const float scale = (float)(1.0 / sqrt((double)a.d));
    if (kv_f16) {
        if (a.d == 128) k_attn_decode<__half, 128, STEP><<<grid, 128, 0, s>>>(a, scale);
        else k_attn_decode<__half, 64, STEP><<<grid, 128, 0, s>>>(a, scale);
    } else {
        if (a.d == 128) k_attn_decode<float, 128, STEP><<<grid, 128, 0, s>>>(a, scale);
        else k_attn_decode<float, 64, STEP><<<grid, 128, 0, s>>>(a, scale);
    }
}

void launch_attn_decode(bool kv_f16, const AttnDecArgs &a, int splits, cudaStream_t s) {
    attn_launch<true>(kv_f16, a, splits, s);
}

void launch_attn_decode_plain(bool kv_f16, const AttnDecArgs &a, int splits, cudaStream_t s) {
    attn_launch<false>(kv_f16, a, splits, s);
}

int attn_decode_splits(int B, int nkv, int num_sms) {
    const int want = (2 * num_sms + B * nkv - 1) / (B * nkv);
    return want < 1 ? 1 : (want > kAttnMaxSplits ? kAttnMaxSplits : want);
}

size_t attn_decode_part_floats(int B, int nq, int nkv, int d, int splits) {
    return (size_t)B * nkv * splits * (nq / nkv) * (d + 2);
}

static size_t align256(size_t n) { return (n + 255) & ~size_t(255); }

size_t attn_op_scratch_bytes(int B, int nq, int nkv, int d, int num_sms) {
    const int S = attn_decode_splits(B, nkv, num_sms);
    return align256(attn_decode_part_floats(B, nq, nkv, d, S) * sizeof(float)) +
           align256((size_t)B * nkv * sizeof(unsigned));
}

bool attn_op_shape_ok(int B, int nq, int nkv, int d, int slots, int kv_ok) {
    return B >= 1 && B <= 1 << 16 && nkv >= 1 && nq >= nkv && nq % nkv == 0 && nq / nkv <= kMaxRep &&
           (d == 64 || d == 128) && slots >= 1 && kv_ok;
}

cudaError_t attn_op_launch(const float *q, const void *K, const void *V, bool kv_f16, int slots,
                           const int32_t *kv_off, const int32_t *kv_len, int B, int nq, int nkv, int d, float *out,
                           void *scratch, int num_sms, cudaStream_t s) {
    const int S = attn_decode_splits(B, nkv, num_sms);
    const size_t part_bytes = align256(attn_decode_part_floats(B, nq, nkv, d, S) * sizeof(float));
    unsigned *counter = reinterpret_cast<unsigned *>(static_cast<char *>(scratch) + part_bytes);
    cudaError_t e = cudaMemsetAsync(counter, 0, (size_t)B * nkv * sizeof(unsigned), s);
    if (e != cudaSuccess) return e;
    AttnDecArgs a{};
    a.Kc = const_cast<void *>(K);
    a.Vc = const_cast<void *>(V);
    a.slots = slots;
    a.o = out;
    a.part = static_cast<float *>(scratch);
    a.counter = counter;
    a.nq = nq;
    a.nkv = nkv;
    a.d = d;
    a.B = B;
    a.q_plain = q;
    a.kv_off = kv_off;
    a.kv_len = kv_len;
    launch_attn_decode_plain(kv_f16, a, S, s);
    return cudaGetLastError();
}

}  // namespace dec
