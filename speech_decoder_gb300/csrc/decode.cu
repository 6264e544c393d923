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
#include "ptx.cuh"

namespace dec {

// ============================================================== attention
template <typename TKV, int PL>
__device__ __forceinline__ void load_kv(const TKV *p, float (&f)[PL]) {
#pragma unroll
    for (int e = 0; e < PL; ++e) f[e] = to_f32(p[e]);
}

constexpr int kMaxRep = 8;
constexpr int kKB = 8;     // keys per warp batch in the decode attention

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
    // every CTA waits on the preceding grid before any exit, which keeps the
    // chain of programmatic launches ordered
    ptx::pdl_launch();
    ptx::pdl_wait();
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

    // splits cover at least kAttnMinChunk keys each: short sequences use few
    // splits and the combine reads only the splits that ran
    const int chunk = max(kAttnMinChunk, (len + S - 1) / S);
    const int n_used = (len + chunk - 1) / chunk;
    if (s >= n_used) return;
    const int j0 = s * chunk, j1 = min(len, j0 + chunk);
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
    // keys in batches of kKB per warp: all K/V loads of a batch are issued
    // before any of them is used
    for (int jb = j0 + warp * kKB; jb < j1; jb += 4 * kKB) {
        float kf[kKB][PL], vf[kKB][PL];
#pragma unroll
        for (int k = 0; k < kKB; ++k) {
            const int j = jb + k;
            if (j < j1) {
                const size_t base = ((size_t)g * a.slots + off + j) * D + lane * PL;
                load_kv<TKV, PL>(Kc + base, kf[k]);
                load_kv<TKV, PL>(Vc + base, vf[k]);
            } else {
#pragma unroll
                for (int e = 0; e < PL; ++e) kf[k][e] = vf[k][e] = 0.f;
            }
        }
#pragma unroll
        for (int r = 0; r < kMaxRep; ++r) {
            if (r < n_rep) {
                float sc[kKB];
#pragma unroll
                for (int k = 0; k < kKB; ++k) {
                    float d = 0.f;
#pragma unroll
                    for (int e = 0; e < PL; ++e) d = fmaf(qs[r][lane * PL + e], kf[k][e], d);
                    sc[k] = d;
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1)
#pragma unroll
                    for (int k = 0; k < kKB; ++k) sc[k] += __shfl_xor_sync(0xffffffffu, sc[k], o);
                float mb = m[r];
#pragma unroll
                for (int k = 0; k < kKB; ++k) {
                    sc[k] = jb + k < j1 ? sc[k] * scale : -INFINITY;
                    mb = fmaxf(mb, sc[k]);
                }
                const float corr = expf(m[r] - mb);
                float ls = 0.f;
#pragma unroll
                for (int e = 0; e < PL; ++e) acc[r][e] *= corr;
#pragma unroll
                for (int k = 0; k < kKB; ++k) {
                    const float p = expf(sc[k] - mb);
                    ls += p;
#pragma unroll
                    for (int e = 0; e < PL; ++e) acc[r][e] = fmaf(p, vf[k][e], acc[r][e]);
                }
                l[r] = l[r] * corr + ls;
                m[r] = mb;
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
    if (ticket != (unsigned)n_used - 1) return;
    __threadfence();

    // last split of this (sequence, kv head): log-sum-exp combine.  The
    // per-split maxima and sums are staged in shared memory first, then every
    // output element is a weighted sum over the splits.
    __shared__ float cw[kAttnMaxSplits][kMaxRep], cm[kAttnMaxSplits][kMaxRep];
    const float *pb = a.part + ((size_t)b * nkv + g) * S * n_rep * (D + 2);
    for (int idx = tid; idx < n_used * n_rep; idx += blockDim.x) {
        const int t = idx / n_rep, r = idx % n_rep;
        const float *pr = pb + ((size_t)t * n_rep + r) * (D + 2);
        cm[t][r] = __ldcg(pr + D);
        cw[t][r] = __ldcg(pr + D + 1);
    }
    __syncthreads();
    if (tid < n_rep) {
        const int r = tid;
        float Mx = -INFINITY;
        for (int t = 0; t < n_used; ++t) Mx = fmaxf(Mx, cm[t][r]);
        float L = 0.f;
        for (int t = 0; t < n_used; ++t) {
            const float f = cm[t][r] == -INFINITY ? 0.f : expf(cm[t][r] - Mx);
            cm[t][r] = f;
            L += cw[t][r] * f;
        }
        const float inv = 1.f / L;
        for (int t = 0; t < n_used; ++t) cw[t][r] = cm[t][r] * inv;
    }
    __syncthreads();
    for (int idx = tid; idx < n_rep * D; idx += blockDim.x) {
        const int r = idx / D, i = idx % D;
        float A = 0.f;
#pragma unroll 4
        for (int t = 0; t < n_used; ++t) A = fmaf(__ldcg(pb + ((size_t)t * n_rep + r) * (D + 2) + i), cw[t][r], A);
        const size_t oi = (size_t)b * a.nq * D + (size_t)(g * n_rep + r) * D + i;
        a.o[oi] = A;
        if (a.o_bf16) a.o_bf16[oi] = __float2bfloat16_rn(A);
    }
    if (tid == 0) a.counter[b * nkv + g] = 0u;
}

template <bool STEP>
static void attn_launch(bool kv_f16, const AttnDecArgs &a, int splits, cudaStream_t s) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(a.nkv, splits, a.B);
    cfg.blockDim = dim3(128);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const float scale = (float)(1.0 / sqrt((double)a.d));
    if (kv_f16) {
        if (a.d == 128) cudaLaunchKernelEx(&cfg, k_attn_decode<__half, 128, STEP>, a, scale);
        else cudaLaunchKernelEx(&cfg, k_attn_decode<__half, 64, STEP>, a, scale);
    } else {
        if (a.d == 128) cudaLaunchKernelEx(&cfg, k_attn_decode<float, 128, STEP>, a, scale);
        else cudaLaunchKernelEx(&cfg, k_attn_decode<float, 64, STEP>, a, scale);
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

// ============================================================== batched-step helpers
template <typename TW>
__global__ void k_embed_rows(const TW *embed, SeqState *st, float *x, int H) {
    const int b = blockIdx.x;
    ptx::pdl_launch();
    ptx::pdl_wait();
    if (!row_live(st, b)) return;
    const TW *src = embed + (size_t)st->cur_tok[b] * H;
    for (int k = threadIdx.x; k < H; k += blockDim.x) x[(size_t)b * H + k] = to_f32(src[k]);
}

void launch_embed_rows(const void *embed, bool w_bf16, SeqState *st, float *x, int B, int H, cudaStream_t s) {
    if (w_bf16) k_embed_rows<__nv_bfloat16><<<B, 256, 0, s>>>((const __nv_bfloat16 *)embed, st, x, H);
    else k_embed_rows<float><<<B, 256, 0, s>>>((const float *)embed, st, x, H);
}

// One CTA per row: strict '>' scan per thread over ascending indices, then a
// tie-aware block reduction (lowest index wins), then the greedy-state update.
__global__ void __launch_bounds__(512) k_argmax_rows(const float *logits, int V, SeqState *st, int32_t *out_ids,
                                                     int out_ids_cap) {
    __shared__ float rv[16];
    __shared__ int ri[16];
    const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    ptx::pdl_launch();
    ptx::pdl_wait();
    if (!row_live(st, b)) return;
    const float *row = logits + (size_t)b * V;
    float bv = -INFINITY;
    int bix = 0x7fffffff;
    for (int i = tid; i < V; i += blockDim.x) {
        const float v = __ldcg(row + i);
        if (v > bv) { bv = v; bix = i; }
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
        for (int w = 1; w < (int)(blockDim.x >> 5); ++w)
            if (rv[w] > bv || (rv[w] == bv && ri[w] < bix)) { bv = rv[w]; bix = ri[w]; }
        if (bix < 0 || bix >= V) {
            atomicCAS(&st->error, 0, 2);
            bix = 0;
        }
        st->cur_tok[b] = bix;
        const int gcount = st->gen[b];
        if (gcount < out_ids_cap) out_ids[(size_t)b * out_ids_cap + gcount] = bix;
        st->gen[b] = gcount + 1;
        const int np = st->n_past[b] + 1;
        st->n_past[b] = np;
        if (bix == st->eos_id || gcount + 1 >= st->max_new || np + 1 > st->kv_cap[b]) st->done[b] = 1;
    }
}

void launch_argmax_rows(const float *logits, int B, int V, SeqState *st, int32_t *out_ids, int out_ids_cap,
                        cudaStream_t s) {
    k_argmax_rows<<<B, 512, 0, s>>>(logits, V, st, out_ids, out_ids_cap);
}

}  // namespace dec
