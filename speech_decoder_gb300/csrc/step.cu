// Persistent decode step of one sequence: the whole greedy step (every block
// of the model and the head) in ONE cooperative launch, one CTA per SM.
//
// Phases of each block (qwen3_asr/decoder.cpp, build_step_graph; block math
// from the page's file header), separated by grid-wide barriers:
//
//   P1  RMSNorm(x) . Wqkv                    (block 0: x = embed[token])
//   P2  Q/K RMSNorm + NeoX RoPE + KV append + attention: item (KV head g,
//       split s) on CTA g S + s, keys [s c, (s + 1) c), partial softmax sums
//   P3  combine the partials, x += o . Wo
//   P4  RMSNorm(x) . Wgu, h = silu(gate) * up   (packed gate|up rows)
//   P5  x += h . Wd
//   then RMSNorm(x) . embed -> logits, argmax, greedy-state update.
//
// A producer warp streams the CTA's rows of EVERY projection of the step, in
// phase order, through a ring of shared-memory stages (1-D bulk copies on
// mbarriers); it is throttled only by free stages, so the next projection's
// rows are on chip when its phase starts and HBM keeps streaming across the
// barriers.  At the start of each block it also lands the CTA's attention
// item's cached keys and values (TMA, 128-byte swizzle) in their own buffer.
// Sixteen consumer warps do the arithmetic.  Everything a phase needs that
// does not depend on the phase before (norm weights, residual values) is
// loaded before the barrier that opens the phase; after it each CTA reads
// one activation vector and computes.  The barrier is one release-add on a
// counter and an acquire poll by one thread per CTA.  Every wait is bounded;
// a wait that gives up records an error code in the sequence state, and the
// CTA then skips its remaining work while still joining every barrier.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>

#include "attn_step.cuh"
#include "step.cuh"
#include "tc.cuh"

namespace dec {
namespace {

constexpr int kCW = 16;                    // consumer warps
constexpr int kCT = kCW * 32;              // consumer threads
constexpr int kTT = kCT + 32;              // + the producer warp
constexpr int kStage = 16 * 1024;          // bytes per ring stage (whole rows)
constexpr int kMaxStages = 12;
constexpr int kD = 128;                    // head_dim
constexpr int kPL = kD / 32;
constexpr int kMaxRepS = 4;                // query heads per KV head at most
constexpr int kAttnBytes = 2 * 2 * kAttnKeys * 64 * 2;   // K and V tiles [part][key][64 dims] f16
constexpr int kBox = 32;                   // key rows per TMA box
constexpr int kNw = 12;                    // norm weights per consumer thread (K <= 6144)
constexpr int kResid = 64;                 // residual rows per CTA at most
constexpr uint64_t kWaitNs = 200000000ull; // every wait gives up after 0.2 s
constexpr int kBarCons = 1;                // named barrier of the consumer warps

__device__ __forceinline__ void cons_sync() { ptx::named_bar_sync(kBarCons, kCT); }

__device__ __forceinline__ void report(const StepArgs &a, int code) { atomicCAS(&a.st->error, 0, code); }

__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long *p) {
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void red_release_add(unsigned long long *p) {
    asm volatile("red.release.gpu.global.add.u64 [%0], 1;" ::"l"(p) : "memory");
}

// this CTA's contiguous block [r0, r1) of N units
__device__ __forceinline__ void cta_range(int N, int &r0, int &r1) {
    r0 = (int)((long long)N * blockIdx.x / gridDim.x);
    r1 = (int)((long long)N * (blockIdx.x + 1) / gridDim.x);
}

__host__ __device__ __forceinline__ int rows_per_stage(int K) {
    const int rb = K * 2;
    return rb >= kStage ? 1 : kStage / rb;
}
// (gate, up) feature pairs per stage: a power of two, so that a chunk starting
// at a multiple of it stays inside one 128-feature block of the packed layout
__host__ __device__ __forceinline__ int pairs_per_stage(int K) {
    const int r = rows_per_stage(K) / 2;
    int p = 1;
    while (p * 2 <= r && p * 2 <= 128) p *= 2;
    return p;
}

// activation element k of a bf16 weight row: the 8 values of a 16-byte chunk
// sit in a low and a high float4 (conflict-free reads)
__device__ __forceinline__ int xs_off(int k, int CPR) {
    const int c = k >> 3, half = (k >> 2) & 1;
    return ((half * CPR + c) << 2) + (k & 3);
}

// byte offset of dims [8 c, 8 c + 8) of key row `row` in one 64-dim part of a tile
__device__ __forceinline__ uint32_t sw_off(int row, int c) { return (uint32_t)(row * 128 + ((c ^ (row & 7)) << 4)); }

struct Ring {
    unsigned char *base;
    uint64_t *full, *empty;
    int NS;
    volatile int *issued;      // chunks the producer has issued
    volatile int *abort;       // a bounded wait gave up: skip the remaining work, keep joining barriers
    int *first_fail;           // first chunk that was not consumed (for the final drain)
};

// The attention item of this CTA (one sequence): KV head g, split s, keys
// [j0, j1) of the n_past + 1 positions; rows [j0, j0 + ncopy) come from the
// pool, the new key (slot pos) from this step's q|k|v row when `mine`.
struct Item {
    bool has;
    int g, s, j0, j1, ncopy, pos, off;
    bool mine;
};

struct GridBar {
    unsigned long long target = 0;
    // every consumer thread; the phase's global writes precede the release
    __device__ void sync(const StepArgs &a, volatile int *abort) {
        cons_sync();
        target += gridDim.x;
        if (threadIdx.x == 0) {
            red_release_add(a.bar);
            uint64_t t0 = 0;
            int n = 0;
            while (ld_acquire_u64(a.bar) < target) {
                if (++n == 256) {
                    n = 0;
                    const uint64_t t = ptx::now_ns();
                    if (!t0) {
                        t0 = t;
                    } else if (t - t0 > kWaitNs) {
                        report(a, 7);
                        *abort = 1;
                        break;
                    }
                }
            }
        }
        cons_sync();
    }
};

// ------------------------------------------------------------------ producer
__device__ void produce(const StepArgs &a, const Ring &rg, const Item &it, uint64_t *attn_full, uint64_t *attn_empty,
                        unsigned char *tiles) {
    uint32_t g = 0;
    // wait for a free stage for chunk g (chunk g - NS consumed)
    auto slot_free = [&](int slot) -> bool {
        if (g < (uint32_t)rg.NS) return true;
        const uint32_t par = ((g / rg.NS) - 1) & 1;
        if (ptx::mbar_try_wait(&rg.empty[slot], par)) return true;
        const uint64_t t0 = ptx::now_ns();
        for (;;) {
            if (*rg.abort) return false;
            if (ptx::mbar_try_wait(&rg.empty[slot], par)) return true;
            if (ptx::now_ns() - t0 > kWaitNs) {
                report(a, 8);
                *rg.abort = 1;
                return false;
            }
        }
    };
    auto publish = [&]() {
        ++g;
        __threadfence_block();
        *rg.issued = (int)g;
    };
    auto stream_rows = [&](const __nv_bfloat16 *W, int N, int K) -> bool {
        int r0, r1;
        cta_range(N, r0, r1);
        const int R = rows_per_stage(K);
        const size_t rb = (size_t)K * 2;
        for (int r = r0; r < r1; r += R) {
            const int slot = g % rg.NS;
            if (!slot_free(slot)) return false;
            const uint32_t bytes = (uint32_t)(min(R, r1 - r) * rb);
            ptx::mbar_expect_tx(&rg.full[slot], bytes);
            ptx::bulk_g2s(rg.base + (size_t)slot * kStage, reinterpret_cast<const unsigned char *>(W) + r * rb, bytes,
                          &rg.full[slot]);
            publish();
        }
        return true;
    };
    // gate|up packed in blocks of 128 gate rows + the same 128 features' up rows
    auto stream_pairs = [&](const __nv_bfloat16 *W, int F, int K) -> bool {
        const int R = pairs_per_stage(K);
        const int U = (F + R - 1) / R;
        const int f0 = min(F, R * (int)((long long)U * blockIdx.x / gridDim.x));
        const int f1 = min(F, R * (int)((long long)U * (blockIdx.x + 1) / gridDim.x));
        const size_t rb = (size_t)K * 2;
        for (int f = f0; f < f1; f += R) {
            const int slot = g % rg.NS;
            if (!slot_free(slot)) return false;
            const int n = min(R, f1 - f);
            const size_t grow = (size_t)(f >> 7) * 256 + (f & 127);
            const uint32_t half = (uint32_t)(n * rb);
            unsigned char *dst = rg.base + (size_t)slot * kStage;
            ptx::mbar_expect_tx(&rg.full[slot], 2 * half);
            ptx::bulk_g2s(dst, reinterpret_cast<const unsigned char *>(W) + grow * rb, half, &rg.full[slot]);
            ptx::bulk_g2s(dst + half, reinterpret_cast<const unsigned char *>(W) + (grow + 128) * rb, half,
                          &rg.full[slot]);
            publish();
        }
        return true;
    };
    const int H = a.H, F = a.F, nqd = a.nq * kD;
    for (int l = 0; l < a.L; ++l) {
        if (it.has) {
            // the item's cached keys and values of this block, once the
            // previous block's attention has read the buffer
            if (l > 0 && !ptx::mbar_wait_ns(attn_empty, (l - 1) & 1, kWaitNs)) {
                report(a, 13);
                *rg.abort = 1;
                return;
            }
            if (it.ncopy > 0) {
                const CUtensorMap *mk = a.kv_maps + 2 * l, *mv = mk + 1;
                const int nbox = (it.ncopy + kBox - 1) / kBox;
                const int y0 = it.g * a.slots + it.off + it.j0;
                ptx::mbar_expect_tx(attn_full, (uint32_t)(nbox * 4 * kBox * 128));
                for (int i = 0; i < nbox; ++i) {
                    const int y = y0 + i * kBox;
                    unsigned char *kt = tiles + (size_t)i * kBox * 128;
                    unsigned char *vt = tiles + 2 * kAttnKeys * 128 + (size_t)i * kBox * 128;
                    tma_load_2d(kt, mk, 0, y, attn_full);
                    tma_load_2d(kt + kAttnKeys * 128, mk, 64, y, attn_full);
                    tma_load_2d(vt, mv, 0, y, attn_full);
                    tma_load_2d(vt + kAttnKeys * 128, mv, 64, y, attn_full);
                }
            } else {
                ptx::mbar_arrive(attn_full);
            }
        }
        const StepLayer &Ly = a.layers[l];
        if (!stream_rows(Ly.wqkv, a.qkv_n, H)) return;
        if (!stream_rows(Ly.wo, H, nqd)) return;
        if (!stream_pairs(Ly.wgu, F, H)) return;
        if (!stream_rows(Ly.wd, H, F)) return;
    }
    stream_rows(a.embed, a.V, H);
}

// ------------------------------------------------------------------ projection phases (consumers)
enum { P_EMBED = 0, P_NORM = 1, P_PLAIN = 2, P_ATTN = 3 };
enum { E_STORE = 0, E_RESID = 1, E_SWIGLU = 2, E_ARGMAX = 3 };

// chunk g of the ring: wait until issued (the parity then names one phase) and landed
__device__ __forceinline__ bool chunk_ready(const StepArgs &a, const Ring &rg, uint32_t g) {
    const int lane = threadIdx.x & 31;
    bool ok = !*rg.abort;
    if (ok && *rg.issued <= (int)g) {
        const uint64_t t0 = ptx::now_ns();
        while (*rg.issued <= (int)g && !*rg.abort && ptx::now_ns() - t0 <= kWaitNs) {
        }
        ok = *rg.issued > (int)g;
    }
    ok = ok && ptx::mbar_wait_ns(&rg.full[g % rg.NS], (g / rg.NS) & 1, kWaitNs);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok && lane == 0) {
        if (!*rg.abort) report(a, 9);
        *rg.abort = 1;
        atomicMin(rg.first_fail, (int)g);
    }
    return ok;
}

// dot products of rows [0, nr) of a stage with the activation row; two rows
// share each activation read.  acc[i] for row i (lane 0 holds the sums)
__device__ __forceinline__ void dot2(const uint4 *w0, const uint4 *w1, const float *xs, int CPR, float &a0,
                                     float &a1) {
    const int lane = threadIdx.x & 31;
    const float4 *x4 = reinterpret_cast<const float4 *>(xs);
    a0 = a1 = 0.f;
#pragma unroll 2
    for (int c = lane; c < CPR; c += 32) {
        float f0[8], f1[8];
        unpack16(w0[c], f0, (const __nv_bfloat16 *)nullptr);
        unpack16(w1[c], f1, (const __nv_bfloat16 *)nullptr);
        const float4 lo = x4[c], hi = x4[CPR + c];
        a0 = fmaf(f0[0], lo.x, a0); a0 = fmaf(f0[1], lo.y, a0); a0 = fmaf(f0[2], lo.z, a0); a0 = fmaf(f0[3], lo.w, a0);
        a0 = fmaf(f0[4], hi.x, a0); a0 = fmaf(f0[5], hi.y, a0); a0 = fmaf(f0[6], hi.z, a0); a0 = fmaf(f0[7], hi.w, a0);
        a1 = fmaf(f1[0], lo.x, a1); a1 = fmaf(f1[1], lo.y, a1); a1 = fmaf(f1[2], lo.z, a1); a1 = fmaf(f1[3], lo.w, a1);
        a1 = fmaf(f1[4], hi.x, a1); a1 = fmaf(f1[5], hi.y, a1); a1 = fmaf(f1[6], hi.z, a1); a1 = fmaf(f1[7], hi.w, a1);
    }
    a0 = warp_sum(a0);
    a1 = warp_sum(a1);
}
__device__ __forceinline__ float dot1(const uint4 *w0, const float *xs, int CPR) {
    const int lane = threadIdx.x & 31;
    const float4 *x4 = reinterpret_cast<const float4 *>(xs);
    float a0 = 0.f;
#pragma unroll 4
    for (int c = lane; c < CPR; c += 32) {
        float f0[8];
        unpack16(w0[c], f0, (const __nv_bfloat16 *)nullptr);
        const float4 lo = x4[c], hi = x4[CPR + c];
        a0 = fmaf(f0[0], lo.x, a0); a0 = fmaf(f0[1], lo.y, a0); a0 = fmaf(f0[2], lo.z, a0); a0 = fmaf(f0[3], lo.w, a0);
        a0 = fmaf(f0[4], hi.x, a0); a0 = fmaf(f0[5], hi.y, a0); a0 = fmaf(f0[6], hi.z, a0); a0 = fmaf(f0[7], hi.w, a0);
    }
    return warp_sum(a0);
}

struct PhaseIo {
    const float *in;           // P_NORM, P_PLAIN: activation vector [K]
    const float *nw;           // this thread's norm weights (registers), P_NORM / P_EMBED
    const float *resid;        // E_RESID: residual values of the CTA's rows (shared memory)
    float *out;
};

// One projection phase: prologue (activation vector into shared memory; RMS
// scale r of normed inputs, applied to the finished dot products), then the
// CTA's chunks of the ring, chunk j to warp j % 16.
template <int IN, int OUT>
__device__ __noinline__ void gemv_phase(const StepArgs &a, const Ring &rg, uint32_t &gctr, int N, int K,
                                        const PhaseIo &io, float *xs, float *red, float &best_v, int &best_i) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int CPR = K / 8;
    int r0, r1, R;
    if (OUT == E_SWIGLU) {
        R = pairs_per_stage(K);
        const int U = (N + R - 1) / R;
        r0 = min(N, R * (int)((long long)U * blockIdx.x / gridDim.x));
        r1 = min(N, R * (int)((long long)U * (blockIdx.x + 1) / gridDim.x));
    } else {
        R = rows_per_stage(K);
        cta_range(N, r0, r1);
    }
    const int n_chunks = (r1 - r0 + R - 1) / R;

    // ---- prologue
    float ss = 0.f;
    if (IN == P_ATTN) {
        // o = softmax-weighted values of every query head: combine the splits
        const int n_rep = a.nq / a.nkv, S = a.S;
        for (int k = tid; k < K; k += kCT) {
            const int hq = k / kD, i = k % kD, g = hq / n_rep, r = hq % n_rep;
            const float *pb = a.part + ((size_t)g * S * n_rep + r) * (kD + 2);
            float M = -INFINITY;
            for (int s = 0; s < S; ++s) M = fmaxf(M, __ldcg(pb + (size_t)s * n_rep * (kD + 2) + kD));
            float O = 0.f, L = 0.f;
            for (int s = 0; s < S; ++s) {
                const float *ps = pb + (size_t)s * n_rep * (kD + 2);
                const float m = __ldcg(ps + kD);
                const float w = m == -INFINITY ? 0.f : expf(m - M);
                O = fmaf(w, __ldcg(ps + i), O);
                L = fmaf(w, __ldcg(ps + kD + 1), L);
            }
            xs[xs_off(k, CPR)] = O / L;
        }
    } else {
        constexpr int P = kNw;
        float v[P];
        const __nv_bfloat16 *er = IN == P_EMBED ? a.embed + (size_t)a.st->cur_tok[0] * K : nullptr;
#pragma unroll
        for (int i = 0; i < P; ++i) {
            const int k = tid + i * kCT;
            v[i] = k < K ? (IN == P_EMBED ? __bfloat162float(er[k]) : __ldcg(io.in + k)) : 0.f;
        }
#pragma unroll
        for (int i = 0; i < P; ++i) {
            const int k = tid + i * kCT;
            if (k < K) {
                const float w = IN == P_PLAIN ? 1.f : io.nw[i];
                xs[xs_off(k, CPR)] = v[i] * w;
                ss += v[i] * v[i];
                if (IN == P_EMBED && blockIdx.x == 0) a.x[k] = v[i];
            }
        }
    }
    float rs = 1.f;
    if (IN == P_NORM || IN == P_EMBED) {
        ss = warp_sum(ss);
        if (lane == 0) red[warp] = ss;
    }
    cons_sync();                                       // activation rows and partial sums visible
    if (IN == P_NORM || IN == P_EMBED) {
        float t = 0.f;
#pragma unroll
        for (int w = 0; w < kCW; ++w) t += red[w];
        rs = rsqrtf(t / (float)K + a.eps);
    }

    // ---- chunks
    const size_t rb = (size_t)K * 2;
    for (int j = warp; j < n_chunks; j += kCW) {
        const uint32_t g = gctr + j;
        if (!chunk_ready(a, rg, g)) break;
        const unsigned char *stage = rg.base + (size_t)(g % rg.NS) * kStage;
        const int u0 = r0 + j * R, n = min(R, r1 - u0);
        if (OUT == E_SWIGLU) {
            const uint4 *wg = reinterpret_cast<const uint4 *>(stage);
            const uint4 *wu = reinterpret_cast<const uint4 *>(stage + (size_t)n * rb);
            for (int i = 0; i < n; ++i) {
                float ag, au;
                dot2(wg + (size_t)i * CPR, wu + (size_t)i * CPR, xs, CPR, ag, au);
                if (lane == 0) {
                    ag *= rs;
                    au *= rs;
                    io.out[u0 + i] = ag / (1.f + expf(-ag)) * au;
                }
            }
        } else {
            const uint4 *w = reinterpret_cast<const uint4 *>(stage);
            int i = 0;
            for (; i + 1 < n; i += 2) {
                float a0, a1;
                dot2(w + (size_t)i * CPR, w + (size_t)(i + 1) * CPR, xs, CPR, a0, a1);
                if (lane == 0) {
                    const int row = u0 + i;
                    a0 *= rs;
                    a1 *= rs;
                    if (OUT == E_STORE) {
                        io.out[row] = a0;
                        io.out[row + 1] = a1;
                    } else if (OUT == E_RESID) {
                        io.out[row] = io.resid[row - r0] + a0;
                        io.out[row + 1] = io.resid[row + 1 - r0] + a1;
                    } else {
                        io.out[row] = a0;
                        io.out[row + 1] = a1;
                        if (a0 > best_v) { best_v = a0; best_i = row; }          // rows ascend: lowest index on ties
                        if (a1 > best_v) { best_v = a1; best_i = row + 1; }
                    }
                }
            }
            if (i < n) {
                float a0 = dot1(w + (size_t)i * CPR, xs, CPR);
                if (lane == 0) {
                    const int row = u0 + i;
                    a0 *= rs;
                    if (OUT == E_STORE) io.out[row] = a0;
                    else if (OUT == E_RESID) io.out[row] = io.resid[row - r0] + a0;
                    else {
                        io.out[row] = a0;
                        if (a0 > best_v) { best_v = a0; best_i = row; }
                    }
                }
            }
        }
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&rg.empty[g % rg.NS]);
    }
    gctr += n_chunks;
}

// ------------------------------------------------------------------ attention item (consumers)
struct AttnScratch {
    float qs[kMaxRepS][kD];
    float p[kMaxRepS][kAttnKeys];
    float accp[8][kD];                     // [key part][head] x dims, 8 (part, head) slots
    float m[kMaxRepS], l[kMaxRepS];
};

__device__ __noinline__ void attn_item(const StepArgs &a, const StepLayer &Ly, int l, const Item &it,
                                       unsigned char *tiles, AttnScratch &sc, uint64_t *attn_full,
                                       uint64_t *attn_empty, const float (&qw)[kPL], const float (&kw)[kPL],
                                       volatile int *abort) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int n_rep = a.nq / a.nkv;
    const int nk = it.j1 - it.j0;
    // the new row's cos/sin and the step's q/k/v rows (written before the barrier)
    float2 cs[kPL];
    {
        const float2 *rope_row = a.rope + (size_t)it.pos * (kD / 2) + (lane & 15) * kPL;
#pragma unroll
        for (int e = 0; e < kPL; e += 2) {
            const float4 c = *reinterpret_cast<const float4 *>(rope_row + e);
            cs[e] = make_float2(c.x, c.y);
            cs[e + 1] = make_float2(c.z, c.w);
        }
    }
    float v[kPL];
    const bool is_q = warp < n_rep, is_k = warp == n_rep && it.mine, is_v = warp == n_rep + 1 && it.mine;
    if (is_q) load_vec_cg<kPL>(a.qkv + (size_t)(it.g * n_rep + warp) * kD + lane * kPL, v);
    if (is_k) load_vec_cg<kPL>(a.qkv + (size_t)(a.nq + it.g) * kD + lane * kPL, v);
    if (is_v) load_vec_cg<kPL>(a.qkv + (size_t)(a.nq + a.nkv + it.g) * kD + lane * kPL, v);
    if (!ptx::mbar_wait_ns(attn_full, l & 1, kWaitNs) && lane == 0) {
        report(a, 11);
        *abort = 1;
    }
    if (is_q) {
        norm_rope_regs<kPL>(v, qw, cs, a.eps, kD, lane);
#pragma unroll
        for (int e = 0; e < kPL; ++e) sc.qs[warp][lane * kPL + e] = v[e];
    }
    if (is_k || is_v) {
        if (is_k) norm_rope_regs<kPL>(v, kw, cs, a.eps, kD, lane);
        __half *pool = (is_k ? Ly.K : Ly.V) + ((size_t)it.g * a.slots + it.off + it.pos) * kD;
        const int d0 = lane * kPL, part = d0 >> 6, col = d0 & 63, rr = it.pos - it.j0;
        __half *dst = reinterpret_cast<__half *>(tiles + (is_k ? 0 : 2 * kAttnKeys * 128) + part * kAttnKeys * 128 +
                                                 sw_off(rr, col >> 3)) + (col & 7);
#pragma unroll
        for (int e = 0; e < kPL; ++e) {
            const __half q = __float2half_rn(v[e]);
            pool[d0 + e] = q;
            dst[e] = q;
        }
    }
    cons_sync();
    // scores: thread -> key tid % 128 of head tid / 128
    {
        const int kk = tid & (kAttnKeys - 1), r = tid / kAttnKeys;
        if (r < n_rep) {
            float d = 0.f;
            if (kk < nk) {
#pragma unroll
                for (int c = 0; c < kD / 8; ++c) {
                    const uint4 kv =
                        *reinterpret_cast<const uint4 *>(tiles + (c >> 3) * kAttnKeys * 128 + sw_off(kk, c & 7));
                    float f[8];
                    unpack16(kv, f, (const __half *)nullptr);
                    const float4 q0 = *reinterpret_cast<const float4 *>(&sc.qs[r][c * 8]);
                    const float4 q1 = *reinterpret_cast<const float4 *>(&sc.qs[r][c * 8 + 4]);
                    d = fmaf(f[0], q0.x, d); d = fmaf(f[1], q0.y, d); d = fmaf(f[2], q0.z, d); d = fmaf(f[3], q0.w, d);
                    d = fmaf(f[4], q1.x, d); d = fmaf(f[5], q1.y, d); d = fmaf(f[6], q1.z, d); d = fmaf(f[7], q1.w, d);
                }
            }
            sc.p[r][kk] = kk < nk ? d * a.scale : -INFINITY;
        }
    }
    cons_sync();
    if (warp < n_rep) {                          // softmax statistics: warp r owns head r
        float mx = -INFINITY;
#pragma unroll
        for (int i = 0; i < kAttnKeys / 32; ++i) mx = fmaxf(mx, sc.p[warp][lane + 32 * i]);
        mx = warp_max(mx);
        float sum = 0.f;
#pragma unroll
        for (int i = 0; i < kAttnKeys / 32; ++i) {
            const float e = mx == -INFINITY ? 0.f : expf(sc.p[warp][lane + 32 * i] - mx);
            sc.p[warp][lane + 32 * i] = e;
            sum += e;
        }
        sum = warp_sum(sum);
        if (lane == 0) {
            sc.m[warp] = mx;
            sc.l[warp] = sum;
        }
    }
    cons_sync();
    // P V: thread -> (key part kp, head r, dims 2 dp, 2 dp + 1); 8 (part, head) slots
    {
        const int per = n_rep * 64, parts = kCT / per;
        const int kp = tid / per, rem = tid % per, r = rem >> 6, dp = rem & 63;
        const int d0 = 2 * dp, part = d0 >> 6, col = d0 & 63;
        const unsigned char *vb = tiles + 2 * kAttnKeys * 128 + part * kAttnKeys * 128;
        float a0 = 0.f, a1 = 0.f;
        for (int kk = kp; kk < nk; kk += parts) {
            const float2 vf = __half22float2(*reinterpret_cast<const __half2 *>(vb + sw_off(kk, col >> 3) + (col & 7) * 2));
            const float pk = sc.p[r][kk];
            a0 = fmaf(pk, vf.x, a0);
            a1 = fmaf(pk, vf.y, a1);
        }
        sc.accp[kp * n_rep + r][d0] = a0;
        sc.accp[kp * n_rep + r][d0 + 1] = a1;
    }
    cons_sync();
    // the item's partial: sum over key parts, then max and sum of exp
    {
        const int per = n_rep * 64, parts = kCT / per;
        float *pb = a.part + ((size_t)it.g * a.S + it.s) * n_rep * (kD + 2);
        for (int e = tid; e < n_rep * kD; e += kCT) {
            const int r = e / kD, i = e % kD;
            float s = 0.f;
            for (int kp = 0; kp < parts; ++kp) s += sc.accp[kp * n_rep + r][i];
            pb[(size_t)r * (kD + 2) + i] = s;
            if (i == 0) {
                pb[(size_t)r * (kD + 2) + kD] = sc.m[r];
                pb[(size_t)r * (kD + 2) + kD + 1] = sc.l[r];
            }
        }
    }
    cons_sync();                                 // tiles read: the producer may refill them
    if (tid == 0) ptx::mbar_arrive(attn_empty);
}

// bytes of the activation vector area (also the attention item's scratch)
__host__ __device__ __forceinline__ int xs_area(int H, int F, int nqd) {
    int n = H > F ? H : F;
    n = n > nqd ? n : nqd;
    const int b = n * 4 > (int)sizeof(AttnScratch) ? n * 4 : (int)sizeof(AttnScratch);
    return (b + 1023) & ~1023;
}

// ------------------------------------------------------------------ the step kernel
__global__ void __launch_bounds__(kTT, 1) k_decode_step(StepArgs a) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char *base =
        reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ __align__(8) uint64_t full[kMaxStages], empty[kMaxStages];
    __shared__ __align__(8) uint64_t attn_full, attn_empty;
    __shared__ volatile int issued_s, abort_s, prod_done_s;
    __shared__ int first_fail_s;
    __shared__ float red[32];
    __shared__ float resid_s[kResid];
    __shared__ float wv[kCW];
    __shared__ int wi[kCW];
    __shared__ unsigned ticket_s;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // a finished sequence or a recorded error: the step is a no-op (uniform)
    if (!row_live(a.st, 0) || a.st->error) return;

    const int H = a.H, F = a.F, nqd = a.nq * kD;
    const int xs_bytes = xs_area(H, F, nqd);
    unsigned char *tiles = base;
    float *xs = reinterpret_cast<float *>(base + kAttnBytes);
    AttnScratch &sc = *reinterpret_cast<AttnScratch *>(xs);
    Ring rg;
    rg.base = base + kAttnBytes + xs_bytes;
    rg.full = full;
    rg.empty = empty;
    rg.NS = a.ring_stages;
    rg.issued = &issued_s;
    rg.abort = &abort_s;
    rg.first_fail = &first_fail_s;

    Item it{};
    {
        const int pos = a.st->n_past[0], len = pos + 1;
        it.pos = pos;
        it.off = a.st->kv_off[0];
        it.has = (int)blockIdx.x < a.nkv * a.S;
        it.g = blockIdx.x / a.S;
        it.s = blockIdx.x % a.S;
        int chunk = (len + a.S - 1) / a.S;
        if (chunk > kAttnKeys) {                  // the launch sized S for the context capacity: never
            if (tid == 0) report(a, 12);
            chunk = kAttnKeys;
        }
        it.j0 = min(len, it.s * chunk);
        it.j1 = min(len, it.j0 + chunk);
        it.ncopy = max(0, min(it.j1, pos) - it.j0);
        it.mine = pos >= it.j0 && pos < it.j1;
    }

    if (tid == 0) {
        for (int s = 0; s < rg.NS; ++s) {
            ptx::mbar_init(&full[s], 1);
            ptx::mbar_init(&empty[s], 1);
        }
        ptx::mbar_init(&attn_full, 1);
        ptx::mbar_init(&attn_empty, 1);
        issued_s = 0;
        abort_s = 0;
        prod_done_s = 0;
        first_fail_s = 0x7fffffff;
        ptx::fence_mbar_init();
    }
    __syncthreads();

    if (warp == kCW) {                            // producer warp
        if (lane == 0) {
            produce(a, rg, it, &attn_full, &attn_empty, tiles);
            __threadfence_block();
            prod_done_s = 1;
        }
        return;
    }

    GridBar gb;
    uint32_t gctr = 0;
    float best_v = -INFINITY;
    int best_i = 0x7fffffff;
    float nw[kNw];
    auto load_norm = [&](const float *w, int K) {
#pragma unroll
        for (int i = 0; i < kNw; ++i) {
            const int k = tid + i * kCT;
            nw[i] = k < K ? w[k] : 0.f;
        }
    };
    // residual values of this CTA's rows of an H-row projection
    auto load_resid = [&]() {
        int r0, r1;
        cta_range(H, r0, r1);
        if (tid < r1 - r0) resid_s[tid] = __ldcg(a.x + r0 + tid);
    };
    float qw[kPL], kw[kPL];
    load_norm(a.layers[0].attn_norm, H);
    for (int l = 0; l < a.L; ++l) {
        const StepLayer &Ly = a.layers[l];
        PhaseIo io{};
        io.nw = nw;
        io.in = a.x;
        io.out = a.qkv;
        if (l == 0) gemv_phase<P_EMBED, E_STORE>(a, rg, gctr, a.qkv_n, H, io, xs, red, best_v, best_i);
        else gemv_phase<P_NORM, E_STORE>(a, rg, gctr, a.qkv_n, H, io, xs, red, best_v, best_i);
        if (it.has) {
            load_vec<kPL>(Ly.qn + lane * kPL, qw);
            load_vec<kPL>(Ly.kn + lane * kPL, kw);
        }
        gb.sync(a, &abort_s);
        // every consumer thread of an item's CTA enters (the item's named barriers)
        if (it.has) attn_item(a, Ly, l, it, tiles, sc, &attn_full, &attn_empty, qw, kw, &abort_s);
        load_resid();
        gb.sync(a, &abort_s);
        io.resid = resid_s;
        io.out = a.x;
        gemv_phase<P_ATTN, E_RESID>(a, rg, gctr, H, nqd, io, xs, red, best_v, best_i);
        load_norm(Ly.ffn_norm, H);
        gb.sync(a, &abort_s);
        io.in = a.x;
        io.out = a.h;
        gemv_phase<P_NORM, E_SWIGLU>(a, rg, gctr, F, H, io, xs, red, best_v, best_i);
        load_resid();
        gb.sync(a, &abort_s);
        io.in = a.h;
        io.out = a.x;
        gemv_phase<P_PLAIN, E_RESID>(a, rg, gctr, H, F, io, xs, red, best_v, best_i);
        load_norm(l + 1 < a.L ? a.layers[l + 1].attn_norm : a.final_norm, H);
        gb.sync(a, &abort_s);
    }
    {
        PhaseIo io{};
        io.nw = nw;
        io.in = a.x;
        io.out = a.logits;
        gemv_phase<P_NORM, E_ARGMAX>(a, rg, gctr, a.V, H, io, xs, red, best_v, best_i);
    }

    // ---- argmax across warps and CTAs; the last CTA advances the greedy state
    if (lane == 0) {
        wv[warp] = best_v;
        wi[warp] = best_i;
    }
    cons_sync();
    const int G = gridDim.x;
    if (tid == 0) {
        float bv = -INFINITY;
        int bix = 0x7fffffff;
        for (int w = 0; w < kCW; ++w)
            if (wv[w] > bv || (wv[w] == bv && wi[w] < bix)) {
                bv = wv[w];
                bix = wi[w];
            }
        a.am_val[blockIdx.x] = bv;
        a.am_idx[blockIdx.x] = bix;
        __threadfence();
        ticket_s = atomicAdd(a.am_counter, 1u);
    }
    cons_sync();
    if (ticket_s == (unsigned)G - 1) {
        __threadfence();
        float bv = -INFINITY;
        int bix = 0x7fffffff;
        for (int i = tid; i < G; i += kCT) {
            const float v = __ldcg(a.am_val + i);
            const int ix = __ldcg(a.am_idx + i);
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
            wv[warp] = bv;
            wi[warp] = bix;
        }
        cons_sync();
        if (tid == 0) {
            for (int w = 1; w < kCW; ++w)
                if (wv[w] > bv || (wv[w] == bv && wi[w] < bix)) {
                    bv = wv[w];
                    bix = wi[w];
                }
            SeqState *st = a.st;
            if (bix < 0 || bix >= a.V) {          // every logit NaN
                report(a, 2);
                bix = 0;
            }
            st->cur_tok[0] = bix;
            const int gc = st->gen[0];
            if (gc < a.out_ids_cap) a.out_ids[gc] = bix;
            st->gen[0] = gc + 1;
            const int np = st->n_past[0] + 1;
            st->n_past[0] = np;
            if (bix == st->eos_id || gc + 1 >= st->max_new || np + 1 > st->kv_cap[0]) st->done[0] = 1;
            *a.am_counter = 0u;
        }
    }
    // a wait that gave up: once the producer has stopped, drain the copies it
    // issued that nobody consumed, so none lands after the CTA exits
    cons_sync();
    if (tid == 0 && abort_s) {
        const uint64_t t0 = ptx::now_ns();
        while (!prod_done_s && ptx::now_ns() - t0 <= kWaitNs) __nanosleep(64);
        for (int g = first_fail_s; g < issued_s; ++g) ptx::mbar_wait_ns(&full[g % rg.NS], (g / rg.NS) & 1, kWaitNs);
    }
}

PFN_cuTensorMapEncodeTiled_v12000 g_step_encode = nullptr;
int g_optin = 0;

}  // namespace

// ------------------------------------------------------------------ host side
int step_splits(int max_ctx) { return (max_ctx + kAttnKeys - 1) / kAttnKeys; }

static size_t static_smem() {
    cudaFuncAttributes fa{};
    return cudaFuncGetAttributes(&fa, k_decode_step) == cudaSuccess ? fa.sharedSizeBytes : 4096;
}

StepPlan step_plan(int H, int F, int nqd) {
    StepPlan p{};
    int dev = 0, coop = 0;
    if (!g_optin && cudaGetDevice(&dev) == cudaSuccess) {
        cudaDeviceGetAttribute(&g_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev);
        if (!coop) g_optin = -1;
    }
    if (g_optin <= 0) return p;
    const size_t fixed = 1024 + kAttnBytes + (size_t)xs_area(H, F, nqd);   // alignment pad, tiles, activations
    const size_t budget = (size_t)g_optin - static_smem();
    if (budget < fixed + 4 * (size_t)kStage) return p;
    p.ring_stages = (int)std::min<size_t>(kMaxStages, (budget - fixed) / kStage);
    p.smem = fixed + (size_t)p.ring_stages * kStage;
    p.ok = true;
    return p;
}

bool step_kv_maps(CUtensorMap *k_map, CUtensorMap *v_map, const void *K, const void *V, int rows) {
    if (!g_step_encode) {
        cudaDriverEntryPointQueryResult q;
        void *fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !fn) {
            cudaGetLastError();
            return false;
        }
        g_step_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    const cuuint64_t dims[2] = {(cuuint64_t)kD, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)kD * 2};
    const cuuint32_t box[2] = {64, kBox};
    const cuuint32_t es[2] = {1, 1};
    for (int i = 0; i < 2; ++i) {
        if (g_step_encode(i ? v_map : k_map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void *>(i ? V : K), dims,
                          strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return false;
    }
    return true;
}

bool step_supported(int head_dim, int n_rep, int nkv, int H, int F, int max_ctx, int num_sms) {
    if (head_dim != kD || (n_rep != 1 && n_rep != 2 && n_rep != 4) || nkv < 1 || num_sms < 1) return false;
    if (nkv * step_splits(max_ctx) > num_sms) return false;          // one attention item per CTA
    if ((H + num_sms - 1) / num_sms > kResid) return false;          // residual rows per CTA
    if (std::max(H, F) > kNw * kCT || H % 8 || F % 128 || n_rep * nkv * kD > kNw * kCT) return false;
    const StepPlan p = step_plan(H, F, n_rep * nkv * kD);
    if (!p.ok) return false;
    int per_sm = 0;
    if (cudaFuncSetAttribute(k_decode_step, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p.smem) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_decode_step, kTT, p.smem) != cudaSuccess ||
        per_sm < 1) {
        cudaGetLastError();
        return false;
    }
    return true;
}

cudaError_t launch_step(StepArgs a, int num_sms, cudaStream_t s) {
    const StepPlan p = step_plan(a.H, a.F, a.nq * kD);
    if (!p.ok) return cudaErrorInvalidValue;
    a.ring_stages = p.ring_stages;
    cudaError_t e = cudaMemsetAsync(a.bar, 0, sizeof(unsigned long long), s);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(num_sms);
    cfg.blockDim = dim3(kTT);
    cfg.dynamicSmemBytes = p.smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    void *args[] = {&a};
    return cudaLaunchKernelExC(&cfg, reinterpret_cast<void *>(k_decode_step), args);
}

}  // namespace dec
