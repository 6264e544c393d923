// Weight-streaming GEMV of the decode step, fed by a producer warp (bf16
// weights, or e4m3 codes with one power-of-two scale per row for a single
// sequence; one activation row per sequence, up to four sequences per CTA).
//
// One CTA per SM owns a contiguous block of weight rows.  Its producer warp
// copies whole rows, as many as fit a 16 KB stage, into a ring of shared-memory
// stages with 1-D bulk copies (TMA) completing on mbarriers; eight consumer
// warps take the stages round-robin (chunk j goes to warp j % 8), each
// finishing its rows itself: dot products against the activation rows held in
// shared memory, a warp reduction, and the epilogue.  Weights never depend on
// earlier kernels, so the ring is filled before the kernel waits for its
// predecessor (programmatic dependent launch), and once the producer has issued
// its last own row it pulls the CTA's share of the NEXT kernel's weights into
// L2: HBM keeps streaming while the launch boundary drains.
//
// Block math (qwen3_asr/decoder.cpp, build_step_graph; the decoder block of the
// page's file header): the prologue builds RMSNorm(x)*w (pre-LN norms, final
// norm), the embedding row of the step's token (layer 0), the plain attention
// output, or silu(gate)*up from the packed gate|up rows; the epilogue stores,
// adds into the residual, or writes logits and takes the argmax with the lowest
// index winning ties, the last CTA advancing the greedy state.
//
// Option (off by default: slower than the separate attention kernel on the
// benchmark shapes): the q|k|v GEMV of a single sequence finishes the step
// attention itself.  Each CTA counts the rows it completed of every KV head's
// q, k and v rows on an acquire-release ticket, and the CTA that completes a
// head's last rows runs that head's attention in its (by then idle) ring
// memory.  No CTA waits for another, and the step loses one kernel boundary
// per layer.
#include <climits>

#include <cuda_fp8.h>

#include "attn_step.cuh"

namespace dec {
namespace {

constexpr int kCW = 8;                        // consumer warps
constexpr int kCT = kCW * 32;                 // consumer threads
constexpr int kTT = kCT + 32;                 // + the producer warp
constexpr int kStage = 16 * 1024;             // bytes per ring stage (whole rows)
constexpr int kMaxStages = 12;
constexpr int kAutoStages = 12;               // 192 KB in flight per SM covers the loaded HBM latency
constexpr uint64_t kWaitNs = 200000000ull;    // every wait gives up after 0.2 s
constexpr int kBarCons = 1;                   // named barrier of the consumer warps
constexpr int kBarProd = 2;                   // consumers arrive, the producer warp waits: prologue published

__device__ __forceinline__ void cons_sync() { ptx::named_bar_sync(kBarCons, kCT); }

__device__ __forceinline__ void report(SeqState *st, int code) {
    if (st) atomicCAS(&st->error, 0, code);
}

// activation element k of a weight row with EPC weights per 16-byte chunk
// (8 bf16 or 16 e4m3 codes) lives at xs_off<EPC>(k): the chunk's values are
// split into float4 parts, part p of chunk c at float4 index p * CPR + c
// (conflict-free reads).  For bf16 rows: the 8 values of
// a 16-byte chunk are split into low/high float4 halves (conflict-free reads)
template <int EPC>
__device__ __forceinline__ int xs_off(int k, int CPR) {
    const int c = k / EPC, part = (k % EPC) >> 2;
    return ((part * CPR + c) << 2) + (k & 3);
}

// whole rows of rb bytes per stage
__host__ __device__ __forceinline__ int rows_per_stage(int rb) {
    return rb >= kStage ? 1 : kStage / rb;
}

// OUT_SWIGLU: (gate, up) row pairs per stage, a power of two so that a chunk
// that starts at a multiple of it never crosses a 128-feature block of the
// packed gate|up layout; 0 = a pair does not fit one stage
__host__ __device__ __forceinline__ int pairs_per_stage(int rb) {
    const int r = rows_per_stage(rb) / 2;
    int p = 0;
    if (r >= 1) {
        p = 1;
        while (p * 2 <= r && p * 2 <= 128) p *= 2;
    }
    return rb > kStage ? 0 : p;
}

// The weights of one 16-byte chunk as floats: 8 bf16 values (WB = 2) or 16
// e4m3 codes (WB = 1; byte i of the chunk is weight i).
__device__ __forceinline__ void unpack_e4m3x16(const uint4 &u, float (&f)[16]) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const __half2 h(__nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w[i] >> (16 * j)), __NV_E4M3));
            const float2 v = __half22float2(h);
            f[4 * i + 2 * j] = v.x;
            f[4 * i + 2 * j + 1] = v.y;
        }
}

template <int WB>
__device__ __forceinline__ void unpack_w(const uint4 &u, float (&f)[16 / WB]) {
    if constexpr (WB == 2) unpack16(u, f, (const __nv_bfloat16 *)nullptr);
    else unpack_e4m3x16(u, f);
}

// acc += the chunk's weights . its activations (Q float4 parts), in order
template <int Q>
__device__ __forceinline__ void fma_chunk(const float (&f)[4 * Q], const float4 (&x)[Q], float &acc) {
#pragma unroll
    for (int q = 0; q < Q; ++q) {
        acc = fmaf(f[4 * q], x[q].x, acc);
        acc = fmaf(f[4 * q + 1], x[q].y, acc);
        acc = fmaf(f[4 * q + 2], x[q].z, acc);
        acc = fmaf(f[4 * q + 3], x[q].w, acc);
    }
}

template <int Q>
__device__ __forceinline__ void load_parts(const float4 *x4, int c, int CPR, float4 (&x)[Q]) {
#pragma unroll
    for (int q = 0; q < Q; ++q) x[q] = x4[q * CPR + c];
}

// Head dims, query heads per KV head and key tile of the fused step attention.
constexpr int kFD = 128;
constexpr int kFRep = 2;
constexpr int kFT = attn_tile_keys<__half, kFD>() / 2, kFBuf = 2;
constexpr size_t kFusedAttnSmem = kFBuf * 2 * (size_t)kFT * kFD * sizeof(__half) + sizeof(AttnSmem<kFD, kTT / 32>);

__host__ __device__ __forceinline__ int range_overlap(int a0, int a1, int b0, int b1) {
    const int lo = a0 > b0 ? a0 : b0, hi = a1 < b1 ? a1 : b1;
    return hi > lo ? hi - lo : 0;
}

// OUT_QKV_ATTN tail (all threads of the CTA, after its rows [r0, r1) of the
// q|k|v row are stored).  Thread g adds the CTA's rows of KV head g (its q, k
// and v rows) to the head's acquire-release ticket; the CTA whose addition
// completes the head's (kFRep + 2) * kFD rows runs its attention.  Every count
// is added before any attention runs, so no head's completion waits behind
// another head's attention.  Shared memory from `smem` on holds the key/value
// tiles; bar points to the tail's two mbarriers (one per tile buffer); mask is
// a shared word.
__device__ void qkv_attn_tail(const GemvArgs &a, int r0, int r1, unsigned char *smem, uint64_t *bar,
                              unsigned *mask) {
    constexpr int W = kTT / 32, PL = kFD / 32;
    const AttnDecArgs &at = a.at;
    const int lane = threadIdx.x & 31;
    const unsigned need = (unsigned)((kFRep + 2) * kFD);
    float qw[PL], kw[PL];
    load_vec<PL>(at.qn_w + lane * PL, qw);
    load_vec<PL>(at.kn_w + lane * PL, kw);
    if (threadIdx.x == 0) *mask = 0u;
    __syncthreads();                                     // every store of the rows precedes the releases
    if (threadIdx.x < at.nkv) {
        const int g = threadIdx.x, qd = at.nq * kFD, kd = at.nkv * kFD;
        const int cnt = range_overlap(r0, r1, g * kFRep * kFD, (g + 1) * kFRep * kFD) +
                        range_overlap(r0, r1, qd + g * kFD, qd + (g + 1) * kFD) +
                        range_overlap(r0, r1, qd + kd + g * kFD, qd + kd + (g + 1) * kFD);
        if (cnt > 0 && atomic_add_acq_rel(&at.counter[g], (unsigned)cnt) + (unsigned)cnt == need) {
            at.counter[g] = 0u;                          // every CTA of the head has added: reset for the next launch
            atomicOr(mask, 1u << g);
        }
    }
    __syncthreads();
    const unsigned m = *mask;
    uint32_t phase = 0;
    for (int g = 0; g < at.nkv; ++g) {
        if (!((m >> g) & 1u)) continue;                  // uniform
        // the ring, the activation rows and an earlier head's tiles were
        // accessed by the generic proxy; the tiles arrive there by bulk copy
        ptx::fence_proxy_async_smem();
        __syncthreads();
        attn_step_core<__half, kFD, kFRep, W, kFT, kFBuf>(at, a.at_scale, g, 0, 1, 0, smem, bar, phase, qw, kw,
                                                         kAttnMinChunk);
    }
}

// Activation rows of this CTA's sequences into shared memory (consumer
// threads).  The rows' loads are issued together with the liveness reads (rows
// that turn out finished are computed and not stored).  RMSNorm inputs are
// stored as x * w and each warp parks its partial sums of x^2 in sred; the
// row's scale r = 1 / sqrt(mean(x^2) + eps) (row_scales, after the kernel's
// barrier that publishes the rows) multiplies the finished dot products.
// The norm weights were loaded into registers (nwr: this thread's first
// kNwRegs elements) before the kernel waited on its predecessor.
constexpr int kNwRegs = 8;                            // K = 2048 over 256 consumer threads

template <int NB, int IN, int EPC>
__device__ void prologue(const GemvArgs &a, float *xs, const float (&nwr)[kNwRegs], int b0, int *live, int CPR,
                         float *sred) {
    const int K = a.K, tid = threadIdx.x;
    // the rows' liveness flags: loaded here, stored to shared memory only after
    // the activation loads are issued (a store through the generic pointer
    // first would hold those loads back by a whole memory round trip)
    const bool lv = tid < kGroupB && tid < NB && b0 + tid < a.B && row_live(a.st, b0 + tid);
    if (IN == IN_EMBED_NORM) {                            // the token ids come from the state
        if (tid < kGroupB) live[tid] = lv;
        cons_sync();
    }
    // loads in flight per thread and row: one pass over K = 2048, and over
    // K = 6144 (down projection inputs) for a single row
    constexpr int P = (IN == IN_SWIGLU || IN == IN_PLAIN) && NB == 1 ? 24 : 8;
    float ss[NB];
#pragma unroll
    for (int bi = 0; bi < NB; ++bi) ss[bi] = 0.f;
    for (int k0 = tid; k0 < K; k0 += P * kCT) {
        float v[NB][P];
#pragma unroll
        for (int bi = 0; bi < NB; ++bi) {
            const int b = b0 + bi;
            const bool ex = b < a.B && (IN != IN_EMBED_NORM || live[bi]);
            if (IN == IN_SWIGLU) {
                // packed gate|up: block j of 256 outputs = 128 gate rows, then the 128 up rows
                const float *gu = a.in + (size_t)b * 2 * a.ffn;
                float g[P], u[P];
#pragma unroll
                for (int i = 0; i < P; ++i) {
                    const int f = k0 + i * kCT, blk = f >> 7, j = f & 127;
                    g[i] = ex && f < K ? gu[blk * 256 + j] : 0.f;
                    u[i] = ex && f < K ? gu[blk * 256 + 128 + j] : 0.f;
                }
#pragma unroll
                for (int i = 0; i < P; ++i) v[bi][i] = g[i] / (1.f + expf(-g[i])) * u[i];
            } else if (IN == IN_EMBED_NORM) {
                const __nv_bfloat16 *er =
                    reinterpret_cast<const __nv_bfloat16 *>(a.embed) + (size_t)(ex ? a.st->cur_tok[b] : 0) * K;
#pragma unroll
                for (int i = 0; i < P; ++i) {
                    const int k = k0 + i * kCT;
                    v[bi][i] = ex && k < K ? __bfloat162float(er[k]) : 0.f;
                }
            } else {
                const float *src = a.in + (size_t)b * K;
#pragma unroll
                for (int i = 0; i < P; ++i) {
                    const int k = k0 + i * kCT;
                    v[bi][i] = ex && k < K ? src[k] : 0.f;
                }
            }
        }
        if (IN != IN_EMBED_NORM && k0 == tid && tid < kGroupB) live[tid] = lv;
        constexpr bool kNorm = IN == IN_NORM || IN == IN_EMBED_NORM;
        static_assert(!kNorm || P <= kNwRegs, "the first pass's norm weights are the registers");
#pragma unroll
        for (int bi = 0; bi < NB; ++bi) {
            float *xr = xs + (size_t)bi * K;
#pragma unroll
            for (int i = 0; i < P; ++i) {
                const int k = k0 + i * kCT;
                if (k < K) {
                    float w = 1.f;
                    if (kNorm) w = k0 == tid ? nwr[i < kNwRegs ? i : 0] : a.norm_w[k];
                    xr[xs_off<EPC>(k, CPR)] = v[bi][i] * w;
                    ss[bi] += v[bi][i] * v[bi][i];
                    if (IN == IN_EMBED_NORM && blockIdx.x == 0 && b0 + bi < a.B && live[bi])
                        a.x_resid[(size_t)(b0 + bi) * K + k] = v[bi][i];
                }
            }
        }
    }
    if constexpr (IN == IN_NORM || IN == IN_EMBED_NORM) {
#pragma unroll
        for (int bi = 0; bi < NB; ++bi) {
            const float t = warp_sum(ss[bi]);
            if ((tid & 31) == 0) sred[(tid >> 5) * NB + bi] = t;
        }
    }
}

// RMSNorm scale of each row from the consumer warps' partial sums (after the
// barrier that publishes them)
template <int NB, int IN>
__device__ __forceinline__ void row_scales(const GemvArgs &a, const float *sred, float (&rs)[NB]) {
    if constexpr (IN == IN_NORM || IN == IN_EMBED_NORM) {
#pragma unroll
        for (int bi = 0; bi < NB; ++bi) {
            float t = 0.f;
#pragma unroll
            for (int w = 0; w < kCW; ++w) t += sred[w * NB + bi];
            rs[bi] = rsqrtf(t / (float)a.K + a.eps);
        }
    }
}

// OUT_RESID: the residual values of the CTA's rows [r0, r0 + n) of each
// sequence, loaded with the activation rows (v[bi * n + row - r0]); v null
// when the CTA holds more rows than the shared array (then read in place)
struct Resid {
    const float *v;
    int r0, n;
};
constexpr int kResidRows = 32;

// Epilogue of one finished row (lane 0 of the warp that computed it).
template <int NB, int OUT>
__device__ __forceinline__ void row_out(const GemvArgs &a, int row, int b0, const int *live, const Resid &rd,
                                        const float (&acc)[NB], float (&best_v)[NB], int (&best_i)[NB]) {
#pragma unroll
    for (int bi = 0; bi < NB; ++bi) {
        if (!live[bi]) continue;
        const size_t o = (size_t)(b0 + bi) * a.N + row;
        if (OUT == OUT_STORE || OUT == OUT_QKV_ATTN) a.out[o] = acc[bi];
        if (OUT == OUT_RESID) a.out[o] = (rd.v ? rd.v[bi * rd.n + row - rd.r0] : a.out[o]) + acc[bi];
        if (OUT == OUT_ARGMAX) {
            if (a.out) a.out[o] = acc[bi];
            if (acc[bi] > best_v[bi]) {                    // rows ascend per warp: lowest index on ties
                best_v[bi] = acc[bi];
                best_i[bi] = row;
            }
        }
    }
}

// Rows [row0, row0 + nr) of one stage; two rows share each activation read.
// WB: bytes per weight (2: bf16; 1: e4m3 codes, the row's scale a.wscale[row]
// multiplies its dot product).
template <int NB, int OUT, int WB>
__device__ __forceinline__ void stage_rows(const GemvArgs &a, const uint4 *stage, int row0, int nr, int CPR, int b0,
                                           const float *xs, const float (&rs)[NB], const int *live, const Resid &rd,
                                           float (&best_v)[NB], int (&best_i)[NB]) {
    constexpr int Q = 4 / WB;                      // float4 activation parts per chunk
    const int lane = threadIdx.x & 31, K = a.K;
    int rr = 0;
    for (; rr + 1 < nr; rr += 2) {
        const uint4 *w0 = stage + (size_t)rr * CPR, *w1 = w0 + CPR;
        const float ws0 = WB == 1 ? __ldg(a.wscale + row0 + rr) : 1.f;
        const float ws1 = WB == 1 ? __ldg(a.wscale + row0 + rr + 1) : 1.f;
        float a0[NB], a1[NB];
#pragma unroll
        for (int b = 0; b < NB; ++b) a0[b] = a1[b] = 0.f;
#pragma unroll 2
        for (int c = lane; c < CPR; c += 32) {
            float f0[16 / WB], f1[16 / WB];
            unpack_w<WB>(w0[c], f0);
            unpack_w<WB>(w1[c], f1);
#pragma unroll
            for (int b = 0; b < NB; ++b) {
                float4 x[Q];
                load_parts<Q>(reinterpret_cast<const float4 *>(xs + (size_t)b * K), c, CPR, x);
                fma_chunk<Q>(f0, x, a0[b]);
                fma_chunk<Q>(f1, x, a1[b]);
            }
        }
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            a0[b] = warp_sum(a0[b]) * rs[b] * ws0;
            a1[b] = warp_sum(a1[b]) * rs[b] * ws1;
        }
        if (lane == 0) {
            row_out<NB, OUT>(a, row0 + rr, b0, live, rd, a0, best_v, best_i);
            row_out<NB, OUT>(a, row0 + rr + 1, b0, live, rd, a1, best_v, best_i);
        }
    }
    if (rr < nr) {
        const uint4 *w0 = stage + (size_t)rr * CPR;
        const float ws0 = WB == 1 ? __ldg(a.wscale + row0 + rr) : 1.f;
        float a0[NB];
#pragma unroll
        for (int b = 0; b < NB; ++b) a0[b] = 0.f;
#pragma unroll 4
        for (int c = lane; c < CPR; c += 32) {
            float f0[16 / WB];
            unpack_w<WB>(w0[c], f0);
#pragma unroll
            for (int b = 0; b < NB; ++b) {
                float4 x[Q];
                load_parts<Q>(reinterpret_cast<const float4 *>(xs + (size_t)b * K), c, CPR, x);
                fma_chunk<Q>(f0, x, a0[b]);
            }
        }
#pragma unroll
        for (int b = 0; b < NB; ++b) a0[b] = warp_sum(a0[b]) * rs[b] * ws0;
        if (lane == 0) row_out<NB, OUT>(a, row0 + rr, b0, live, rd, a0, best_v, best_i);
    }
}

// OUT_SWIGLU: pairs [j0, j0 + n): gate rows first, then the n up rows; each
// warp writes silu(gate) * up per feature.  WB as for stage_rows (feature f's
// gate row is (f / 128) * 256 + f % 128 of the packed matrix, its up row 128
// further).
template <int NB, int WB>
__device__ __forceinline__ void stage_pairs(const GemvArgs &a, const uint4 *stage, int j0, int n, int i0, int i1,
                                            int CPR, int b0, const float *xs, const float (&rs)[NB],
                                            const int *live) {
    constexpr int Q = 4 / WB;
    const int lane = threadIdx.x & 31, K = a.K;
    for (int i = i0; i < i1; ++i) {
        const uint4 *wg = stage + (size_t)i * CPR, *wu = stage + (size_t)(n + i) * CPR;
        const int f = j0 + i, grow = (f >> 7) * 256 + (f & 127);
        const float wsg = WB == 1 ? __ldg(a.wscale + grow) : 1.f;
        const float wsu = WB == 1 ? __ldg(a.wscale + grow + 128) : 1.f;
        float ag[NB], au[NB];
#pragma unroll
        for (int b = 0; b < NB; ++b) ag[b] = au[b] = 0.f;
#pragma unroll 2
        for (int c = lane; c < CPR; c += 32) {
            float f0[16 / WB], f1[16 / WB];
            unpack_w<WB>(wg[c], f0);
            unpack_w<WB>(wu[c], f1);
#pragma unroll
            for (int b = 0; b < NB; ++b) {
                float4 x[Q];
                load_parts<Q>(reinterpret_cast<const float4 *>(xs + (size_t)b * K), c, CPR, x);
                fma_chunk<Q>(f0, x, ag[b]);
                fma_chunk<Q>(f1, x, au[b]);
            }
        }
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            ag[b] = warp_sum(ag[b]) * rs[b] * wsg;
            au[b] = warp_sum(au[b]) * rs[b] * wsu;
        }
        if (lane == 0) {
#pragma unroll
            for (int b = 0; b < NB; ++b)
                if (live[b]) a.out[(size_t)(b0 + b) * a.N + j0 + i] = ag[b] / (1.f + expf(-ag[b])) * au[b];
        }
    }
}

}  // namespace

// WB: bytes per weight, 2 (bf16) or 1 (e4m3 codes with per-row scales a.wscale)
template <int NB, int IN, int OUT, int WB>
__global__ void __launch_bounds__(kTT, OUT == OUT_QKV_ATTN ? 1 : 2) k_gemv_stream(GemvArgs a) {
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ __align__(8) uint64_t full[kMaxStages];
    __shared__ __align__(8) uint64_t empty[kMaxStages];
    __shared__ __align__(8) uint64_t attn_bar[2];
    __shared__ volatile int issued_s, abort_s;
    __shared__ int first_fail_s;
    __shared__ int live_s[kGroupB];
    __shared__ float sred[32];
    __shared__ float wv[kCW * kGroupB];
    __shared__ int wi[kCW * kGroupB];
    __shared__ float rv[kTT / 32];
    __shared__ int ri[kTT / 32];
    __shared__ unsigned ticket_s;
    __shared__ float resid_s[OUT == OUT_RESID ? kGroupB * kResidRows : 1];

    const int NS = a.n_ring;
    const int K = a.K, CPR = K * WB / 16;             // 16-byte chunks per weight row
    const size_t rb = (size_t)K * WB;
    // units: weight rows, or (gate, up) pairs for OUT_SWIGLU (a.N = ffn
    // features; each CTA's range starts at a multiple of R)
    constexpr bool kPair = OUT == OUT_SWIGLU;
    const int R = kPair ? pairs_per_stage((int)rb) : rows_per_stage((int)rb);
    int r0, r1;
    if (kPair) {
        const long long U = (a.N + R - 1) / R;
        r0 = (int)min((long long)a.N, R * (U * blockIdx.x / gridDim.x));
        r1 = (int)min((long long)a.N, R * (U * (blockIdx.x + 1) / gridDim.x));
    } else {
        r0 = (int)((long long)a.N * blockIdx.x / gridDim.x);
        r1 = (int)((long long)a.N * (blockIdx.x + 1) / gridDim.x);
    }
    const int n_chunks = (r1 - r0 + R - 1) / R;
    const int b0 = blockIdx.y * kGroupB;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    float *xs = reinterpret_cast<float *>(smem + (size_t)NS * kStage);
    const unsigned char *W = reinterpret_cast<const unsigned char *>(a.W);
    constexpr bool kNorm = IN == IN_NORM || IN == IN_EMBED_NORM;

    // consumer work units: (gate, up) pairs, or at most two rows of a chunk
    // (two rows share each activation read); every warp takes units round
    // robin, so a CTA's rows spread over all consumer warps
    const int UPC = kPair ? R : (R + 1) / 2;             // units per full chunk
    if (tid == 0) {
        for (int s = 0; s < NS; ++s) {
            ptx::mbar_init(&full[s], 1);
            ptx::mbar_init(&empty[s], UPC);             // one arrival per unit of the chunk
        }
        if (OUT == OUT_QKV_ATTN) {
            ptx::mbar_init(&attn_bar[0], 1);
            ptx::mbar_init(&attn_bar[1], 1);
        }
        issued_s = 0;
        abort_s = 0;
        first_fail_s = INT_MAX;
        ptx::fence_mbar_init();
    }
    __syncthreads();
    ptx::pdl_launch();

    // chunk g (units r0 + g R ...) into stage g % NS; producer lane 0 only
    auto issue = [&](int g) {
        const int slot = g % NS, u = r0 + g * R, n = min(R, r1 - u);
        unsigned char *dst = smem + (size_t)slot * kStage;
        if (kPair) {
            // gate rows of features [u, u + n), then their up rows
            const size_t grow = (size_t)(u >> 7) * 256 + (u & 127);
            const uint32_t half = (uint32_t)(n * rb);
            ptx::mbar_expect_tx(&full[slot], 2 * half);
            ptx::bulk_g2s(dst, W + grow * rb, half, &full[slot]);
            ptx::bulk_g2s(dst + half, W + (grow + 128) * rb, half, &full[slot]);
        } else {
            const uint32_t bytes = (uint32_t)(n * rb);
            ptx::mbar_expect_tx(&full[slot], bytes);
            ptx::bulk_g2s(dst, W + (size_t)u * rb, bytes, &full[slot]);
        }
        __threadfence_block();
        issued_s = g + 1;
    };
    // chunk g's rows into L2 only (no copy to shared memory)
    auto pf_chunk = [&](int g) {
        const int u = r0 + g * R, n = min(R, r1 - u);
        if (kPair) {
            const size_t grow = (size_t)(u >> 7) * 256 + (u & 127);
            const uint32_t half = (uint32_t)(n * rb);
            ptx::bulk_prefetch_l2(W + grow * rb, half);
            ptx::bulk_prefetch_l2(W + (grow + 128) * rb, half);
        } else {
            ptx::bulk_prefetch_l2(W + (size_t)u * rb, (uint32_t)(n * rb));
        }
    };
    // Before the dependency wait only the first a.pre_bulk chunks are copied
    // into the ring; the rest of the ring's first fill goes to L2 and is
    // copied after the consumers' activation loads: bulk copies in flight to
    // this SM would queue those loads behind up to 192 KB of weights.
    const int fill = min(NS, n_chunks);
    const int pre = a.pre_bulk > 0 ? min(a.pre_bulk, fill) : fill;
    if (warp == kCW && lane == 0) {
        for (int g = 0; g < pre; ++g) issue(g);          // weights: no dependency on earlier kernels
        for (int g = pre; g < fill; ++g) pf_chunk(g);
        // this layer's cached keys and values, for the attention that follows:
        // one (sequence, kv head, K or V) range per CTA, pulled into L2.  The
        // state may still be changing (a hint only); ranges are clamped to the pool.
        if (a.kvp_K) {
            const int n_reg = a.B * a.kvp_nkv * 2;
            for (int ri = blockIdx.x; ri < n_reg; ri += gridDim.x) {
                const int b = ri / (2 * a.kvp_nkv), g = (ri >> 1) % a.kvp_nkv;
                const volatile SeqState *st = a.st;
                if (!st->active[b] || st->done[b]) continue;
                const int off = st->kv_off[b];
                int len = st->n_past[b];
                if (off < 0 || off >= a.kvp_slots || len <= 0) continue;
                len = min(len, a.kvp_slots - off);
                const size_t rbk = (size_t)a.kvp_row_bytes;
                const unsigned char *base = reinterpret_cast<const unsigned char *>((ri & 1) ? a.kvp_V : a.kvp_K) +
                                            ((size_t)g * a.kvp_slots + off) * rbk;
                const size_t bytes = (size_t)len * rbk;
                for (size_t o = 0; o < bytes; o += 32768)
                    ptx::bulk_prefetch_l2(base + o, (uint32_t)(bytes - o < 32768 ? bytes - o : 32768));
            }
        }
    }

    float rs[NB];                                         // RMSNorm scale of each row (1: no norm)
#pragma unroll
    for (int b = 0; b < NB; ++b) rs[b] = 1.f;
    if (warp < kCW) {
        float nwr[kNwRegs];                               // weights: no dependency either
#pragma unroll
        for (int i = 0; i < kNwRegs; ++i) {
            const int k = tid + i * kCT;
            nwr[i] = kNorm && k < K ? a.norm_w[k] : 0.f;
        }
        ptx::pdl_wait();
        // OUT_RESID: this CTA's residual values, in flight with the activation rows
        float rv0 = 0.f;
        const int nres = r1 - r0;
        const bool rpre = OUT == OUT_RESID && nres <= kResidRows && tid < NB * nres;
        if (rpre && b0 + tid / nres < a.B) rv0 = a.out[(size_t)(b0 + tid / nres) * a.N + r0 + tid % nres];
        prologue<NB, IN, 16 / WB>(a, xs, nwr, b0, live_s, CPR, sred);
        if (rpre) resid_s[tid] = rv0;
        // rows, partial sums, live_s, resid_s: published to the consumers
        // without waiting for the producer, which may still be issuing copies
        ptx::named_bar_arrive(kBarProd, kTT);
        cons_sync();
    } else {
        ptx::named_bar_sync(kBarProd, kTT);               // the producer needs live_s
    }
    bool any = false;
#pragma unroll
    for (int b = 0; b < NB; ++b) any |= live_s[b] != 0;
    row_scales<NB, IN>(a, sred, rs);

    float best_v[NB];
    int best_i[NB];
#pragma unroll
    for (int b = 0; b < NB; ++b) {
        best_v[b] = -INFINITY;
        best_i[b] = INT_MAX;
    }
    if (warp == kCW) {
        if (lane == 0 && any) {
            for (int g = pre; g < n_chunks; ++g) {
                // chunk g - NS was issued only after chunk g - 2NS had been
                // consumed, so this parity names exactly one phase of the slot
                const int slot = g % NS;
                const uint32_t par = ((g / NS) - 1) & 1;
                bool ok = ptx::mbar_try_wait(&empty[slot], par);
                if (!ok) {
                    const uint64_t t0 = ptx::now_ns();
                    while (!ok && !abort_s && ptx::now_ns() - t0 <= kWaitNs) ok = ptx::mbar_try_wait(&empty[slot], par);
                }
                if (!ok) {
                    if (!abort_s) {
                        report(a.st, 8);
                        abort_s = 1;
                    }
                    break;
                }
                issue(g);
            }
        }
        // own rows all issued: pull this CTA's share of the next kernel's weights into L2
        if (lane == 0 && a.pf) {
            const size_t prb = (size_t)a.pf_K * (a.pf_wb ? a.pf_wb : 2);
            const long long p0 = (long long)a.pf_N * blockIdx.x / gridDim.x;
            const long long p1 = (long long)a.pf_N * (blockIdx.x + 1) / gridDim.x;
            size_t bytes = (size_t)(p1 - p0) * prb;
            if (bytes > (size_t)a.pf_bytes) bytes = (size_t)a.pf_bytes & ~size_t(15);
            const unsigned char *src = reinterpret_cast<const unsigned char *>(a.pf) + (size_t)p0 * prb;
            for (size_t o = 0; o < bytes; o += 32768)
                ptx::bulk_prefetch_l2(src + o, (uint32_t)(bytes - o < 32768 ? bytes - o : 32768));
        }
    } else if (any) {
        const Resid rd{OUT == OUT_RESID && r1 - r0 <= kResidRows ? resid_s : nullptr, r0, r1 - r0};
        // Unit v (chunk v / UPC) goes to warp v % 8.  A warp may run more than
        // one ring lap ahead of the slowest one, so before the parity wait it
        // waits until the producer has ISSUED chunk j: that happens only after
        // chunk j - NS was consumed, hence landed, so the slot is then in chunk
        // j's phase.  The last unit of a short chunk arrives for the units the
        // chunk lacks.
        const int last_n = (r1 - r0) - (n_chunks - 1) * R;
        const int n_units = n_chunks > 0 ? (n_chunks - 1) * UPC + (kPair ? last_n : (last_n + 1) / 2) : 0;
        for (int v = warp; v < n_units; v += kCW) {
            const int j = v / UPC, k = v % UPC;
            const int slot = j % NS;
            bool ok = !abort_s;
            if (ok && issued_s <= j) {
                const uint64_t t0 = ptx::now_ns();
                while (issued_s <= j && !abort_s && ptx::now_ns() - t0 <= kWaitNs) {
                }
                ok = issued_s > j;
            }
            ok = ok && ptx::mbar_wait_ns(&full[slot], (j / NS) & 1, kWaitNs);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) {
                if (lane == 0) {
                    if (!abort_s) {
                        report(a.st, 9);
                        abort_s = 1;
                    }
                    atomicMin(&first_fail_s, j);
                }
                break;
            }
            const int row0 = r0 + j * R, n = min(R, r1 - row0);
            const int units = kPair ? n : (n + 1) / 2;
            const uint4 *stage = reinterpret_cast<const uint4 *>(smem + (size_t)slot * kStage);
            if (kPair) {
                stage_pairs<NB, WB>(a, stage, row0, n, k, k + 1, CPR, b0, xs, rs, live_s);
            } else {
                const int rr = 2 * k, nr = min(2, n - rr);
                stage_rows<NB, OUT, WB>(a, stage + (size_t)rr * CPR, row0 + rr, nr, CPR, b0, xs, rs, live_s, rd,
                                        best_v, best_i);
            }
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive_cnt(&empty[slot], k == units - 1 ? (uint32_t)(UPC - units + 1) : 1u);
        }
    }
    __syncthreads();
    // copies that were issued but not consumed (no live row, or a wait that
    // gave up) must land before the CTA exits
    if (tid == 0 && (!any || abort_s)) {
        const int first = any ? first_fail_s : 0;
        for (int g = first; g < issued_s; ++g) ptx::mbar_wait_ns(&full[g % NS], (g / NS) & 1, kWaitNs);
    }
    if constexpr (OUT == OUT_QKV_ATTN) {
        // a live row whose every chunk was consumed (uniform: shared flags after the barrier)
        if (any && !abort_s) qkv_attn_tail(a, r0, r1, smem, attn_bar, &ticket_s);
        return;
    }
    if (OUT != OUT_ARGMAX) return;

    // ---- argmax across warps and CTAs; the last CTA advances the greedy state
    if (warp < kCW && lane == 0) {
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            wv[warp * kGroupB + b] = best_v[b];
            wi[warp * kGroupB + b] = best_i[b];
        }
    }
    __syncthreads();
    const int G = gridDim.x;
    if (tid < NB && live_s[tid]) {
        float bv = -INFINITY;
        int bix = INT_MAX;
        for (int w = 0; w < kCW; ++w) {
            const float v = wv[w * kGroupB + tid];
            const int ix = wi[w * kGroupB + tid];
            if (v > bv || (v == bv && ix < bix)) {
                bv = v;
                bix = ix;
            }
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
        int bix = INT_MAX;
        for (int i = tid; i < G; i += kTT) {
            const float v = __ldcg(a.part_val + (size_t)b * G + i);
            const int ix = __ldcg(a.part_idx + (size_t)b * G + i);
            if (v > bv || (v == bv && ix < bix)) {
                bv = v;
                bix = ix;
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float v = __shfl_xor_sync(0xffffffffu, bv, o);
            const int ix = __shfl_xor_sync(0xffffffffu, bix, o);
            if (v > bv || (v == bv && ix < bix)) {
                bv = v;
                bix = ix;
            }
        }
        if (lane == 0) {
            rv[warp] = bv;
            ri[warp] = bix;
        }
        __syncthreads();
        if (tid == 0) {
            for (int w = 1; w < kTT / 32; ++w)
                if (rv[w] > bv || (rv[w] == bv && ri[w] < bix)) {
                    bv = rv[w];
                    bix = ri[w];
                }
            SeqState *st = a.st;
            if (bix < 0 || bix >= a.N) {                        // every logit NaN
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

// ------------------------------------------------------------------ host side
static int g_stream_slots = 0;          // 0: as many as keep two CTAs per SM

void gemv_stream_set_slots(int slots) {
    if (slots == 0 || (slots >= 2 && slots <= kMaxStages)) g_stream_slots = slots;
}

GemvPlan gemv_stream_plan(int in_mode, int K, int nb, int N, int grid_x) {
    GemvPlan p{};
    (void)in_mode;
    const size_t xs = ((size_t)nb * K * 4 + 15) / 16 * 16;
    int ns = g_stream_slots ? g_stream_slots : kAutoStages;
    while (ns > 2 && (size_t)ns * kStage + xs > (size_t)kGemvMaxSmem) --ns;
    p.n_ring = ns;
    p.max_units = (N + grid_x - 1) / grid_x;
    p.smem = (size_t)ns * kStage + xs;
    p.ok = K % 8 == 0 && K >= 8 && p.smem <= (size_t)kGemvMaxSmem;
    return p;
}

template <int NB, int IN, int OUT, int WB = 2>
static void launch_nb(const GemvArgs &a, dim3 grid, size_t smem, cudaStream_t s) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kTT);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaLaunchKernelEx(&cfg, k_gemv_stream<NB, IN, OUT, WB>, a);
}

// e4m3 weights (a.wscale set): one sequence, K a multiple of 16
static bool launch_e4m3(int in_mode, int out_mode, GemvArgs a, int grid_x, cudaStream_t s) {
    if (a.B != 1 || a.K % 16) return false;
    const GemvPlan p = gemv_stream_plan(in_mode, a.K, 1, a.N, grid_x);
    if (!p.ok) return false;
    a.n_ring = p.n_ring;
    a.max_units = p.max_units;
    const dim3 grid(grid_x, 1);
#define DEC_E4M3_CASE(I, O)                                 \
    if (in_mode == I && out_mode == O) {                    \
        launch_nb<1, I, O, 1>(a, grid, p.smem, s);           \
        return true;                                         \
    }
    DEC_E4M3_CASE(IN_NORM, OUT_STORE)
    DEC_E4M3_CASE(IN_EMBED_NORM, OUT_STORE)
    DEC_E4M3_CASE(IN_PLAIN, OUT_RESID)
    DEC_E4M3_CASE(IN_SWIGLU, OUT_RESID)
    DEC_E4M3_CASE(IN_NORM, OUT_ARGMAX)
    if (in_mode == IN_NORM && out_mode == OUT_SWIGLU && pairs_per_stage(a.K) > 0) {
        launch_nb<1, IN_NORM, OUT_SWIGLU, 1>(a, grid, p.smem, s);
        return true;
    }
#undef DEC_E4M3_CASE
    return false;
}

template <int IN, int OUT>
static void launch_io(GemvArgs a, int grid_x, cudaStream_t s) {
    const int nb = a.B < kGroupB ? a.B : kGroupB;
    const GemvPlan p = gemv_stream_plan(IN, a.K, nb, a.N, grid_x);
    a.n_ring = p.n_ring;
    a.max_units = p.max_units;
    const dim3 grid(grid_x, (a.B + kGroupB - 1) / kGroupB);
    switch (nb) {
    case 1: launch_nb<1, IN, OUT>(a, grid, p.smem, s); break;
    case 2: launch_nb<2, IN, OUT>(a, grid, p.smem, s); break;
    case 3: launch_nb<3, IN, OUT>(a, grid, p.smem, s); break;
    default: launch_nb<4, IN, OUT>(a, grid, p.smem, s); break;
    }
}

bool gemv_stream_qkv_attn_ok(int K, int grid_x, int nq, int nkv, int d, bool kv_f16) {
    if (d != kFD || !kv_f16 || nkv < 1 || nkv > 32 || nq != kFRep * nkv) return false;
    const GemvPlan p = gemv_stream_plan(IN_NORM, K, 1, (nq + 2 * nkv) * d, grid_x);
    return p.ok && p.smem >= kFusedAttnSmem;
}

bool launch_gemv_stream(int in_mode, int out_mode, const GemvArgs &a, int grid_x, cudaStream_t s) {
    if (a.wscale) return launch_e4m3(in_mode, out_mode, a, grid_x, s);
    const int nb = a.B < kGroupB ? a.B : kGroupB;
    if (!gemv_stream_plan(in_mode, a.K, nb, a.N, grid_x).ok) return false;
    if (out_mode == OUT_QKV_ATTN) {
        if (a.B != 1 || a.N != (a.at.nq + 2 * a.at.nkv) * a.at.d ||
            !gemv_stream_qkv_attn_ok(a.K, grid_x, a.at.nq, a.at.nkv, a.at.d, true))
            return false;
        GemvArgs f = a;
        const GemvPlan p = gemv_stream_plan(in_mode, a.K, 1, a.N, grid_x);
        f.n_ring = p.n_ring;
        f.max_units = p.max_units;
        if (in_mode == IN_NORM) launch_nb<1, IN_NORM, OUT_QKV_ATTN>(f, dim3(grid_x, 1), p.smem, s);
        else if (in_mode == IN_EMBED_NORM) launch_nb<1, IN_EMBED_NORM, OUT_QKV_ATTN>(f, dim3(grid_x, 1), p.smem, s);
        else return false;
        return true;
    }
#define DEC_STREAM_CASE(I, O)            \
    if (in_mode == I && out_mode == O) { \
        launch_io<I, O>(a, grid_x, s);   \
        return true;                     \
    }
    DEC_STREAM_CASE(IN_NORM, OUT_STORE)
    DEC_STREAM_CASE(IN_EMBED_NORM, OUT_STORE)
    DEC_STREAM_CASE(IN_PLAIN, OUT_RESID)
    DEC_STREAM_CASE(IN_SWIGLU, OUT_RESID)
    DEC_STREAM_CASE(IN_NORM, OUT_ARGMAX)
    if (in_mode == IN_NORM && out_mode == OUT_SWIGLU && pairs_per_stage(2 * a.K) > 0) {
        launch_io<IN_NORM, OUT_SWIGLU>(a, grid_x, s);
        return true;
    }
#undef DEC_STREAM_CASE
    return false;
}

template <int NB, int IN, int OUT, int WB = 2>
static void init_nb() {
    auto fn = k_gemv_stream<NB, IN, OUT, WB>;
    cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kGemvMaxSmem);
    cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
}

bool gemv_stream_swiglu_ok(int K, int nb, int ffn, int grid_x) {
    return pairs_per_stage(2 * K) > 0 && gemv_stream_plan(IN_NORM, K, nb, ffn, grid_x).ok;
}

template <int IN, int OUT>
static void init_io() {
    init_nb<1, IN, OUT>();
    init_nb<2, IN, OUT>();
    init_nb<3, IN, OUT>();
    init_nb<4, IN, OUT>();
}

void init_gemv_stream_kernels() {
    init_io<IN_NORM, OUT_STORE>();
    init_io<IN_EMBED_NORM, OUT_STORE>();
    init_io<IN_PLAIN, OUT_RESID>();
    init_io<IN_SWIGLU, OUT_RESID>();
    init_io<IN_NORM, OUT_ARGMAX>();
    init_io<IN_NORM, OUT_SWIGLU>();
    init_nb<1, IN_NORM, OUT_QKV_ATTN>();
    init_nb<1, IN_EMBED_NORM, OUT_QKV_ATTN>();
    init_nb<1, IN_NORM, OUT_STORE, 1>();
    init_nb<1, IN_EMBED_NORM, OUT_STORE, 1>();
    init_nb<1, IN_PLAIN, OUT_RESID, 1>();
    init_nb<1, IN_SWIGLU, OUT_RESID, 1>();
    init_nb<1, IN_NORM, OUT_ARGMAX, 1>();
    init_nb<1, IN_NORM, OUT_SWIGLU, 1>();
}

}  // namespace dec
