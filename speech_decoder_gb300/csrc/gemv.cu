// Weight-streaming GEMV of the decode step (one activation row per sequence).
//
// Each CTA owns a contiguous block of weight rows; each of its warps streams
// whole rows in 4 KB slices ("units": 256 chunks of 16 bytes) and reduces them
// against the activation row with shuffles.  Weights never depend on earlier
// kernels, so every warp issues its first slices before waiting on the
// preceding kernel (programmatic dependent launch): the next projection's
// weights stream in while the previous kernel drains.
//
// Bytes in flight come from 16-byte non-allocating loads double-buffered in
// registers.  This kernel serves fp32 weights (the debug build) and, when
// selected, bf16 weights; the default bf16 path is the producer-warp GEMV of
// gemv_stream.cu.
//
// Prologues: RMSNorm(x)*w (the pre-LN norms and the final norm), the embedding
// row of the step's token (layer 0), the plain attention output, or
// silu(gate)*up from the packed gate|up rows.  Epilogues: store, residual add,
// or logits + argmax with the lowest index winning ties and a last-CTA
// reduction that advances the greedy state (qwen3_asr/decoder.cpp,
// build_step_graph: final RMSNorm, tied lm_head, argmax).
#include <cstdlib>
#include <cstring>

#include "decode.cuh"
#include "ptx.cuh"

namespace dec {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kUnit = 8;                    // 16-byte chunks per lane per unit

__device__ __forceinline__ void report(SeqState *st, int code) {
    if (st) atomicCAS(&st->error, 0, code);
}

// Activation element k lives at xs_off(k): for bf16 weights the 8 values of a
// 16-byte weight chunk are split into a low and a high float4 so that lanes
// reading consecutive chunks read consecutive 16-byte words.
template <typename TW>
__device__ __forceinline__ int xs_off(int k, int CPR) {
    if (sizeof(TW) == 4) return k;
    const int c = k >> 3, half = (k >> 2) & 1;
    return ((half * CPR + c) << 2) + (k & 3);
}

// Build the activation rows of this CTA's sequences in shared memory.  All
// threads of the block take part.  Global loads are issued kPro at a time
// before any of them is used.  Returns whether any row is live.
constexpr int kPro = 8;

template <typename TW, int IN>
__device__ bool gemv_prologue(const GemvArgs &a, float *xs, int b0, int nb, int CPR, int *live_s, float *sred) {
    const int K = a.K, tid = threadIdx.x, nt = blockDim.x;
    int any = 0;
    for (int bi = 0; bi < kGroupB; ++bi) {
        const int b = b0 + bi;
        const bool live = bi < nb && row_live(a.st, b);
        any |= live;
        if (tid == 0) live_s[bi] = live;
        if (!live) continue;                                    // uniform in the block
        float *xr = xs + (size_t)bi * K;
        if (IN == IN_SWIGLU) {
            // packed gate|up: block j of 256 outputs = 128 gate rows, then the 128 up rows
            const float *gu = a.in + (size_t)b * 2 * a.ffn;
            for (int f0 = tid; f0 < K; f0 += kPro * nt) {
                float g[kPro], u[kPro];
#pragma unroll
                for (int i = 0; i < kPro; ++i) {
                    const int f = f0 + i * nt, blk = f >> 7, j = f & 127;
                    g[i] = f < K ? gu[blk * 256 + j] : 0.f;
                    u[i] = f < K ? gu[blk * 256 + 128 + j] : 0.f;
                }
#pragma unroll
                for (int i = 0; i < kPro; ++i) {
                    const int f = f0 + i * nt;
                    if (f < K) xr[xs_off<TW>(f, CPR)] = g[i] / (1.f + expf(-g[i])) * u[i];
                }
            }
            continue;
        }
        const float *src = IN == IN_EMBED_NORM ? nullptr : a.in + (size_t)b * K;
        const TW *er = IN == IN_EMBED_NORM ? reinterpret_cast<const TW *>(a.embed) + (size_t)a.st->cur_tok[b] * K
                                           : nullptr;
        float ss = 0.f;
        for (int k0 = tid; k0 < K; k0 += kPro * nt) {
            float v[kPro];
#pragma unroll
            for (int i = 0; i < kPro; ++i) {
                const int k = k0 + i * nt;
                v[i] = k < K ? (IN == IN_EMBED_NORM ? to_f32(er[k]) : src[k]) : 0.f;
            }
#pragma unroll
            for (int i = 0; i < kPro; ++i) {
                const int k = k0 + i * nt;
                if (k < K) {
                    xr[xs_off<TW>(k, CPR)] = v[i];
                    ss += v[i] * v[i];
                    if (IN == IN_EMBED_NORM && blockIdx.x == 0) a.x_resid[(size_t)b * K + k] = v[i];
                }
            }
        }
        if (IN == IN_PLAIN) continue;
        ss = block_sum(ss, sred);
        const float r = rsqrtf(ss / (float)K + a.eps);
        for (int k0 = tid; k0 < K; k0 += kPro * nt) {
            float w[kPro];
#pragma unroll
            for (int i = 0; i < kPro; ++i) {
                const int k = k0 + i * nt;
                w[i] = k < K ? a.norm_w[k] : 0.f;
            }
#pragma unroll
            for (int i = 0; i < kPro; ++i) {
                const int k = k0 + i * nt;
                if (k < K) {
                    const int o = xs_off<TW>(k, CPR);
                    xr[o] = xr[o] * r * w[i];
                }
            }
        }
    }
    return __syncthreads_or(any) != 0;
}

// Dot products of one 16-byte weight chunk against the activation rows.
template <typename TW>
__device__ __forceinline__ void unit_fma(const uint4 &w, int c, int CPR, int K, int nb, const float *xs,
                                         float (&acc)[kGroupB]) {
    constexpr int VEC = Vec16<TW>::N;
    float f[VEC];
    unpack16(w, f, (const TW *)nullptr);
#pragma unroll
    for (int bi = 0; bi < kGroupB; ++bi) {
        if (bi < nb) {
            const float4 *x4 = reinterpret_cast<const float4 *>(xs + (size_t)bi * K);
            const float4 lo = x4[c];
            acc[bi] = fmaf(f[0], lo.x, acc[bi]);
            acc[bi] = fmaf(f[1], lo.y, acc[bi]);
            acc[bi] = fmaf(f[2], lo.z, acc[bi]);
            acc[bi] = fmaf(f[3], lo.w, acc[bi]);
            if (VEC == 8) {
                const float4 hi = x4[CPR + c];
                acc[bi] = fmaf(f[VEC == 8 ? 4 : 0], hi.x, acc[bi]);
                acc[bi] = fmaf(f[VEC == 8 ? 5 : 0], hi.y, acc[bi]);
                acc[bi] = fmaf(f[VEC == 8 ? 6 : 0], hi.z, acc[bi]);
                acc[bi] = fmaf(f[VEC == 8 ? 7 : 0], hi.w, acc[bi]);
            }
        }
    }
}

// Argmax across warps and CTAs; the last CTA to finish advances the greedy
// state of every live sequence.  All threads of the block take part.
__device__ void argmax_finalize(const GemvArgs &a, const float (&best_v)[kGroupB], const int (&best_i)[kGroupB],
                                int b0, int nb, const int *live_s) {
    __shared__ float wbest_v[kWarps][kGroupB];
    __shared__ int wbest_i[kWarps][kGroupB];
    __shared__ unsigned ticket_s;
    __shared__ float rv[kWarps];
    __shared__ int ri[kWarps];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, N = a.N;
#pragma unroll
    for (int bi = 0; bi < kGroupB; ++bi) {
        float bv = best_v[bi];
        int bix = best_i[bi];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float v = __shfl_xor_sync(0xffffffffu, bv, o);
            const int ix = __shfl_xor_sync(0xffffffffu, bix, o);
            if (v > bv || (v == bv && ix < bix)) { bv = v; bix = ix; }
        }
        if (lane == 0) {
            wbest_v[warp][bi] = bv;
            wbest_i[warp][bi] = bix;
        }
    }
    __syncthreads();
    const int G = gridDim.x;
    if (tid < nb && live_s[tid]) {
        float bv = -INFINITY;
        int bix = 0x7fffffff;
        for (int w = 0; w < kWarps; ++w) {
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
            for (int w = 1; w < kWarps; ++w)
                if (rv[w] > bv || (rv[w] == bv && ri[w] < bix)) { bv = rv[w]; bix = ri[w]; }
            SeqState *st = a.st;
            if (bix < 0 || bix >= N) {                       // every logit NaN
                report(st, 2);
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

// Rows of this CTA, cut into units (4 KB slices of a row); unit u covers row
// r0 + u / SEG, slice u % SEG.  Units are dealt round-robin to the warps, so a
// row's slices may land in different warps: each unit's partial dot products
// go to shared memory and are summed per row, in slice order, at the end.
struct Share {
    int r0, r1, SEG, n_units, my_units;
    __device__ Share(int N, int CPR, int warp) {
        r0 = (int)((long long)N * blockIdx.x / gridDim.x);
        r1 = (int)((long long)N * (blockIdx.x + 1) / gridDim.x);
        SEG = (CPR + 32 * kUnit - 1) / (32 * kUnit);
        n_units = (r1 - r0) * SEG;
        my_units = n_units > warp ? (n_units - warp + kWarps - 1) / kWarps : 0;
    }
    __device__ int unit(int k, int warp) const { return warp + k * kWarps; }     // k-th unit of a warp
    __device__ int row(int u) const { return r0 + u / SEG; }
};

// Unit finished: reduce across the warp and park the partial sums.
__device__ __forceinline__ void unit_done(int u, int nb, float *part, float (&acc)[kGroupB]) {
#pragma unroll
    for (int bi = 0; bi < kGroupB; ++bi) acc[bi] = warp_sum(acc[bi]);
    if ((threadIdx.x & 31) == 0) {
#pragma unroll
        for (int bi = 0; bi < kGroupB; ++bi)
            if (bi < nb) part[(size_t)u * kGroupB + bi] = acc[bi];
    }
#pragma unroll
    for (int bi = 0; bi < kGroupB; ++bi) acc[bi] = 0.f;
}

// All units parked: finish the CTA's rows (store, residual add, or argmax
// candidates).  All threads of the block take part.
template <int OUT>
__device__ void rows_epilogue(const GemvArgs &a, const Share &sh, const float *part, int b0, int nb,
                              const int *live_s, float (&best_v)[kGroupB], int (&best_i)[kGroupB]) {
    __syncthreads();
    for (int rr = threadIdx.x; rr < sh.r1 - sh.r0; rr += blockDim.x) {
#pragma unroll
        for (int bi = 0; bi < kGroupB; ++bi) {
            if (bi >= nb || !live_s[bi]) continue;
            float v = 0.f;
            for (int sg = 0; sg < sh.SEG; ++sg) v += part[(size_t)(rr * sh.SEG + sg) * kGroupB + bi];
            const int row = sh.r0 + rr;
            const size_t o = (size_t)(b0 + bi) * a.N + row;
            if (OUT == OUT_STORE) a.out[o] = v;
            if (OUT == OUT_RESID) a.out[o] += v;
            if (OUT == OUT_ARGMAX) {
                if (a.out) a.out[o] = v;
                if (v > best_v[bi]) {            // rows ascend per thread: lowest index on ties
                    best_v[bi] = v;
                    best_i[bi] = row;
                }
            }
        }
    }
}

// ============================================================== register variant
template <typename TW, int IN, int OUT>
__global__ void __launch_bounds__(kThreads, 2) k_gemv_ldg(GemvArgs a) {
    extern __shared__ __align__(16) float xsm[];
    constexpr int VEC = Vec16<TW>::N;
    __shared__ float sred[32];
    __shared__ int live_s[kGroupB];
    const int K = a.K, CPR = K / VEC;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int b0 = blockIdx.y * kGroupB;
    const int nb = min(kGroupB, a.B - b0);
    const Share sh(a.N, CPR, warp);
    const TW *W = reinterpret_cast<const TW *>(a.W);
    float *part = xsm + (((size_t)nb * K + 3) & ~size_t(3));

    auto load_unit = [&](int k, uint4 (&buf)[kUnit]) {
        const int u = sh.unit(k, warp), seg = u % sh.SEG;
        const uint4 *wr = reinterpret_cast<const uint4 *>(W + (size_t)sh.row(u) * K);
#pragma unroll
        for (int j = 0; j < kUnit; ++j) {
            const int c = seg * 32 * kUnit + lane + 32 * j;
            buf[j] = c < CPR ? ld_stream(wr + c) : make_uint4(0, 0, 0, 0);
        }
    };
    auto compute = [&](int k, const uint4 (&buf)[kUnit], float (&acc)[kGroupB]) {
        const int u = sh.unit(k, warp), seg = u % sh.SEG;
#pragma unroll
        for (int j = 0; j < kUnit; ++j) {
            const int c = seg * 32 * kUnit + lane + 32 * j;
            if (c < CPR) unit_fma<TW>(buf[j], c, CPR, K, nb, xsm, acc);
        }
        unit_done(u, nb, part, acc);
    };

    uint4 bufA[kUnit], bufB[kUnit];
    if (sh.my_units > 0) load_unit(0, bufA);               // weights: no dependency on earlier kernels
    ptx::pdl_launch();
    ptx::pdl_wait();
    const bool any_live = gemv_prologue<TW, IN>(a, xsm, b0, nb, CPR, live_s, sred);
    const int n_k = any_live ? sh.my_units : 0;
    float acc[kGroupB], best_v[kGroupB];
    int best_i[kGroupB];
#pragma unroll
    for (int bi = 0; bi < kGroupB; ++bi) {
        acc[bi] = 0.f;
        best_v[bi] = -INFINITY;
        best_i[bi] = 0x7fffffff;
    }
    for (int k = 0; k < n_k; k += 2) {
        if (k + 1 < n_k) load_unit(k + 1, bufB);
        compute(k, bufA, acc);
        if (k + 1 < n_k) {
            if (k + 2 < n_k) load_unit(k + 2, bufA);
            compute(k + 1, bufB, acc);
        }
    }
    if (OUT == OUT_ARGMAX || any_live) rows_epilogue<OUT>(a, sh, part, b0, nb, live_s, best_v, best_i);
    if (OUT == OUT_ARGMAX) argmax_finalize(a, best_v, best_i, b0, nb, live_s);
}

// ------------------------------------------------------------------ host side
// 1: registers (fp32 weights always, bf16 weights when selected),
// 4: producer-warp stream (bf16 weights)
static int g_impl = 0;
void gemv_set_impl(int impl) {
    if (impl == 1 || impl == 4) g_impl = impl;
}
void gemv_reload_env() {
    const char *v = std::getenv("SPEECH_DECODER_GEMV");
    g_impl = v && !std::strcmp(v, "ldg") ? 1 : 4;
    const char *n = std::getenv("SPEECH_DECODER_GEMV_SLOTS");
    gemv_stream_set_slots(n ? std::atoi(n) : 0);
}
int gemv_impl() {
    if (g_impl == 0) gemv_reload_env();
    return g_impl;
}
int gemv_default_ctas_per_sm() { return gemv_impl() == 4 ? 1 : 2; }

int gemv_grid(int N, int num_sms, int ctas_per_sm) {
    const int g = num_sms * ctas_per_sm;
    return N < g ? N : g;
}

GemvPlan gemv_plan(int K, bool w_bf16, int nb, int N, int grid_x) {
    GemvPlan p{};
    const int row_bytes = K * (w_bf16 ? 2 : 4);
    p.n_ring = 0;
    const int seg = (row_bytes / 16 + 32 * kUnit - 1) / (32 * kUnit);
    p.max_units = ((N + grid_x - 1) / grid_x) * seg;
    const size_t xs = ((size_t)nb * K + 3) / 4 * 16;
    const size_t part = (size_t)p.max_units * kGroupB * 4;
    p.smem = xs + part;
    p.ok = (row_bytes % 16 == 0) && p.smem <= (size_t)kGemvMaxSmem;
    return p;
}

template <typename TW, int IN, int OUT>
static void launch_one(const GemvArgs &a, dim3 grid, size_t smem, cudaStream_t s) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaLaunchKernelEx(&cfg, k_gemv_ldg<TW, IN, OUT>, a);
}

template <typename TW>
static void launch_gemv_t(int in_mode, int out_mode, GemvArgs a, int grid_x, cudaStream_t s) {
    if (sizeof(TW) == 2 && gemv_impl() == 4 && launch_gemv_stream(in_mode, out_mode, a, grid_x, s)) return;
    if (a.wscale) return;               // e4m3 codes: only the producer-warp GEMV reads them
    const int nb = a.B < kGroupB ? a.B : kGroupB;
    const GemvPlan p = gemv_plan(a.K, sizeof(TW) == 2, nb, a.N, grid_x);
    a.n_ring = p.n_ring;
    a.max_units = p.max_units;
    dim3 grid(grid_x, (a.B + kGroupB - 1) / kGroupB);
#define DEC_GEMV_CASE(I, O)                            \
    if (in_mode == I && out_mode == O) {               \
        launch_one<TW, I, O>(a, grid, p.smem, s);      \
        return;                                        \
    }
    DEC_GEMV_CASE(IN_NORM, OUT_STORE)
    DEC_GEMV_CASE(IN_EMBED_NORM, OUT_STORE)
    DEC_GEMV_CASE(IN_PLAIN, OUT_RESID)
    DEC_GEMV_CASE(IN_SWIGLU, OUT_RESID)
    DEC_GEMV_CASE(IN_NORM, OUT_ARGMAX)
#undef DEC_GEMV_CASE
}

void launch_gemv(int in_mode, int out_mode, bool w_bf16, const GemvArgs &a, int grid_x, cudaStream_t s) {
    if (w_bf16) launch_gemv_t<__nv_bfloat16>(in_mode, out_mode, a, grid_x, s);
    else launch_gemv_t<float>(in_mode, out_mode, a, grid_x, s);
}

template <typename F>
static void set_attrs(F *fn) {
    cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kGemvMaxSmem);
    // one carveout for every step kernel: no L1/shared reconfiguration between launches
    cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
}

template <typename TW, int IN, int OUT>
static void init_one() {
    set_attrs(k_gemv_ldg<TW, IN, OUT>);
}

template <typename TW>
static void init_t() {
    init_one<TW, IN_NORM, OUT_STORE>();
    init_one<TW, IN_EMBED_NORM, OUT_STORE>();
    init_one<TW, IN_PLAIN, OUT_RESID>();
    init_one<TW, IN_SWIGLU, OUT_RESID>();
    init_one<TW, IN_NORM, OUT_ARGMAX>();
}

void init_gemv_kernels() {
    init_t<__nv_bfloat16>();
    init_t<float>();
    init_gemv_stream_kernels();
    init_attn_kernels();
    init_attn_cluster();
}

}  // namespace dec
