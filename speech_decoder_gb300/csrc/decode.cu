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
#include "attn_step.cuh"

namespace dec {

// ---------------------------------------------------------------- plain mode
// q already normed and roped ([B, nq, d]), keys [0, kv_len) at kv_off; no
// append.  Keys are loaded into registers in batches of kKB per warp.
template <typename TKV, int D>
__global__ void __launch_bounds__(kAW * 32) k_attn_plain(AttnDecArgs a, float scale) {
    constexpr int PL = D / 32;
    __shared__ AttnSmem<D, kAW> sm;
    const int g = blockIdx.x, s = blockIdx.y, S = gridDim.y, b = blockIdx.z;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int n_rep = a.nq / a.nkv;
    // every CTA waits on the preceding grid before any exit, which keeps the
    // chain of programmatic launches ordered
    ptx::pdl_launch();
    ptx::pdl_wait();
    const int len = a.kv_len[b], off = a.kv_off[b];
    if (len <= 0 || off < 0 || (long long)off + len > (long long)a.slots) return;   // row skipped
    const TKV *Kc = reinterpret_cast<const TKV *>(a.Kc);
    const TKV *Vc = reinterpret_cast<const TKV *>(a.Vc);
    int chunk, n_used;
    attn_split(len, S, chunk, n_used);
    if (s >= n_used) return;
    const int j0 = s * chunk, j1 = min(len, j0 + chunk);
    const size_t head_base = ((size_t)g * a.slots + off) * D;
    const int jb0 = j0 + warp * kKB;
    float kf[kKB][PL], vf[kKB][PL];
    load_kv_batch<TKV, PL>(Kc, Vc, head_base, jb0, j1, lane, kf, vf);
    for (int r = warp; r < n_rep; r += kAW) {
        const float *src = a.q_plain + ((size_t)b * a.nq + g * n_rep + r) * D + lane * PL;
#pragma unroll
        for (int e = 0; e < PL; ++e) sm.qs[r][lane * PL + e] = src[e];
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
    for (int jb = jb0; jb < j1; jb += kAW * kKB) {
        if (jb != jb0) load_kv_batch<TKV, PL>(Kc, Vc, head_base, jb, j1, lane, kf, vf);
        attn_batch<PL>(sm.qs, kf, vf, jb, j1, n_rep, scale, lane, m, l, acc);
    }
    attn_park<D, kAW>(sm, m, l, acc, n_rep, warp, lane);
    __syncthreads();
    attn_finish<D, kAW>(a, sm, b, g, s, S, n_used, n_rep);
}

// ---------------------------------------------------------------- step mode
// NREP: query heads per KV head (1 or 2) for the grouped scoring; 0 = any
// n_rep <= kMaxRep with the lane-per-dims scoring (W = kAW warps)
// Two CTA sizes: SMALL = false (one CTA per SM: 16 warps, 256-key tiles) for
// a few sequences; SMALL = true (8 warps, 128-key tiles, about half the shared
// memory, two CTAs per SM) for batched rows, whose many (sequence, head,
// split) CTAs would otherwise run in several waves.
template <bool SMALL, int NREP>
__host__ __device__ constexpr int attn_step_warps() {
    return SMALL ? kAW : (NREP ? kSW : kAW);
}

template <typename TKV, int D, int NREP, bool SMALL>
__global__ void __launch_bounds__(attn_step_warps<SMALL, NREP>() * 32, SMALL ? 2 : 1)
    k_attn_step(AttnDecArgs a, float scale) {
    constexpr int W = attn_step_warps<SMALL, NREP>();
    constexpr int PL = D / 32;
    constexpr int T = attn_tile_keys<TKV, D>() / 2, NBUF = SMALL ? 1 : 2;
    extern __shared__ __align__(128) unsigned char dsm[];
    __shared__ __align__(8) uint64_t bar[NBUF];
    const int lane = threadIdx.x & 31;
    // Q/K norm weights: no dependency on earlier kernels
    float qw[PL], kw[PL];
    load_vec<PL>(a.qn_w + lane * PL, qw);
    load_vec<PL>(a.kn_w + lane * PL, kw);
    if (threadIdx.x == 0) {
        for (int i = 0; i < NBUF; ++i) ptx::mbar_init(&bar[i], 1);
        ptx::fence_mbar_init();
    }
    ptx::pdl_launch();
    ptx::pdl_wait();
    uint32_t phase = 0;
    attn_step_core<TKV, D, NREP, W, T, NBUF>(a, scale, blockIdx.x, blockIdx.y, gridDim.y, blockIdx.z, dsm, bar, phase,
                                             qw, kw, a.min_chunk > 0 ? a.min_chunk : attn_step_min_chunk(SMALL ? kGroupB + 1 : 1));
}

template <typename TKV, int D, int NREP, bool SMALL>
constexpr size_t attn_step_smem() {
    return (SMALL ? 1 : 2) * 2 * (size_t)(attn_tile_keys<TKV, D>() / 2) * D * sizeof(TKV) +
           sizeof(AttnSmem<D, attn_step_warps<SMALL, NREP>()>);
}

template <typename TKV, int D, int NREP, bool SMALL>
static void launch_step_attn(cudaLaunchConfig_t cfg, const AttnDecArgs &a, float scale) {
    cfg.blockDim = dim3(attn_step_warps<SMALL, NREP>() * 32);
    cfg.dynamicSmemBytes = attn_step_smem<TKV, D, NREP, SMALL>();
    cudaLaunchKernelEx(&cfg, k_attn_step<TKV, D, NREP, SMALL>, a, scale);
}

template <typename TKV, int D, bool SMALL>
static void launch_step_attn_rep(cudaLaunchConfig_t cfg, const AttnDecArgs &a, float scale) {
    const int n_rep = a.nq / a.nkv;
    if (n_rep == 1) launch_step_attn<TKV, D, 1, SMALL>(cfg, a, scale);
    else if (n_rep == 2) launch_step_attn<TKV, D, 2, SMALL>(cfg, a, scale);
    else launch_step_attn<TKV, D, 0, SMALL>(cfg, a, scale);
}

template <typename TKV, int D>
static void launch_step_attn_size(cudaLaunchConfig_t cfg, const AttnDecArgs &a, float scale) {
    if (a.B > kGroupB) launch_step_attn_rep<TKV, D, true>(cfg, a, scale);
    else launch_step_attn_rep<TKV, D, false>(cfg, a, scale);
}

template <typename TKV, int D, int NREP>
static void init_step_attn() {
    cudaFuncSetAttribute(k_attn_step<TKV, D, NREP, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)attn_step_smem<TKV, D, NREP, false>());
    cudaFuncSetAttribute(k_attn_step<TKV, D, NREP, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)attn_step_smem<TKV, D, NREP, true>());
}

template <bool STEP>
static void attn_launch(bool kv_f16, const AttnDecArgs &a, int splits, cudaStream_t s) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(a.nkv, splits, a.B);
    cfg.blockDim = dim3(kAW * 32);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const float scale = (float)(1.0 / sqrt((double)a.d));
    if (STEP) {
        if (kv_f16 && a.d == 128) launch_step_attn_size<__half, 128>(cfg, a, scale);
        else if (kv_f16) launch_step_attn_size<__half, 64>(cfg, a, scale);
        else if (a.d == 128) launch_step_attn_size<float, 128>(cfg, a, scale);
        else launch_step_attn_size<float, 64>(cfg, a, scale);
        return;
    }
    if (kv_f16) {
        if (a.d == 128) cudaLaunchKernelEx(&cfg, k_attn_plain<__half, 128>, a, scale);
        else cudaLaunchKernelEx(&cfg, k_attn_plain<__half, 64>, a, scale);
    } else {
        if (a.d == 128) cudaLaunchKernelEx(&cfg, k_attn_plain<float, 128>, a, scale);
        else cudaLaunchKernelEx(&cfg, k_attn_plain<float, 64>, a, scale);
    }
}

void init_attn_kernels() {
    init_step_attn<__half, 128, 0>();
    init_step_attn<__half, 128, 1>();
    init_step_attn<__half, 128, 2>();
    init_step_attn<__half, 64, 0>();
    init_step_attn<__half, 64, 1>();
    init_step_attn<__half, 64, 2>();
    init_step_attn<float, 128, 0>();
    init_step_attn<float, 128, 1>();
    init_step_attn<float, 128, 2>();
    init_step_attn<float, 64, 0>();
    init_step_attn<float, 64, 1>();
    init_step_attn<float, 64, 2>();
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
    if (w_bf16) launch_pdl(k_embed_rows<__nv_bfloat16>, dim3(B), dim3(256), 0, s, (const __nv_bfloat16 *)embed, st, x, H);
    else launch_pdl(k_embed_rows<float>, dim3(B), dim3(256), 0, s, (const float *)embed, st, x, H);
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
    int i0 = 0;
    if ((V & 3) == 0) {
        // float4 loads, eight in flight per thread; each thread still visits
        // its indices in ascending order
        const float4 *r4 = reinterpret_cast<const float4 *>(row);
        const int V4 = V >> 2, nt = (int)blockDim.x;
        for (int base = tid; base < V4; base += 8 * nt) {
            float4 v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int i = base + u * nt;
                v[u] = i < V4 ? __ldcg(r4 + i) : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int i = 4 * (base + u * nt);
                if (v[u].x > bv) { bv = v[u].x; bix = i; }
                if (v[u].y > bv) { bv = v[u].y; bix = i + 1; }
                if (v[u].z > bv) { bv = v[u].z; bix = i + 2; }
                if (v[u].w > bv) { bv = v[u].w; bix = i + 3; }
            }
        }
        i0 = V;
    }
    for (int i = i0 + tid; i < V; i += blockDim.x) {
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
    launch_pdl(k_argmax_rows, dim3(B), dim3(512), 0, s, logits, V, st, out_ids, out_ids_cap);
}

}  // namespace dec
