// Persistent decode step: the whole greedy step (every block of the model and
// the head) in ONE cooperative launch, one CTA per SM.
//
// The step's phases (qwen3_asr/decoder.cpp, build_step_graph; block math from
// the page's file header) run back to back, separated by a grid-wide barrier
// (a counter in global memory, polled with a bounded wait):
//
//   A  RMSNorm(x) . Wqkv            (layer 0: x = embed[token])
//   B  Q/K RMSNorm + NeoX RoPE + KV append + split-KV attention
//   C  x += o . Wo
//   D  RMSNorm(x) . Wgu             (packed gate|up)
//   E  x += (silu(gate) * up) . Wd
//   F  RMSNorm(x) . embed -> logits, argmax, greedy-state update
//
// Weights never depend on the activations, so each CTA runs a producer warp
// that streams the CTA's rows of EVERY projection of the step, in phase
// order, through a ring of shared-memory stages with 1-D bulk copies (TMA),
// completing on mbarriers.  The producer is throttled only by free stages:
// it runs ahead through barriers, prologues and the attention phase, so the
// next projection's rows are already on chip when its phase starts.  Sixteen
// consumer warps do the arithmetic and synchronise with named barriers (the
// producer never joins them).  Every wait is bounded; a wait that gives up
// records an error code in the sequence state.
#include "decode.cuh"
#include "ptx.cuh"
#include "step.cuh"

namespace dec {

constexpr int kCW = 16;                    // consumer warps
constexpr int kCT = kCW * 32;              // consumer threads
constexpr int kTT = kCT + 32;              // + the producer warp
constexpr int kStage = 16 * 1024;          // bytes per ring stage (whole rows)
constexpr int kD = 128;                    // head_dim of this kernel
constexpr int kPL = kD / 32;
constexpr int kRep = 4;                    // max query heads per KV head in this kernel
constexpr int kKB = 4;                     // keys per warp batch
constexpr uint64_t kWaitNs = 200000000ull; // every wait gives up after 0.2 s
constexpr int kBarCons = 1;                // named barrier of the consumer warps

__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long *p) {
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void cons_sync() { ptx::named_bar_sync(kBarCons, kCT); }

__device__ __forceinline__ void report(const StepArgs &a, int code) { atomicCAS(&a.st->error, 0, code); }

// this CTA's contiguous row block of an N-row matrix
__device__ __forceinline__ void cta_rows(int N, int &r0, int &r1) {
    r0 = (int)((long long)N * blockIdx.x / gridDim.x);
    r1 = (int)((long long)N * (blockIdx.x + 1) / gridDim.x);
}

// rows per ring stage: as many whole rows as fit one stage (at least one)
__device__ __host__ __forceinline__ int rows_per_stage(int K) {
    const int rb = K * 2;
    return rb >= kStage ? 1 : kStage / rb;
}

// activation element k of a bf16 weight row lives at xs_off(k): the 8 values of
// a 16-byte chunk are split into low/high float4 halves (conflict-free reads)
__device__ __forceinline__ int xs_off(int k, int CPR) {
    const int c = k >> 3, half = (k >> 2) & 1;
    return ((half * CPR + c) << 2) + (k & 3);
}

// consumer-only block reduction (512 threads)
__device__ __forceinline__ float cons_sum(float v, float *red) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    v = warp_sum(v);
    cons_sync();
    if (lane == 0) red[warp] = v;
    cons_sync();
    float t = lane < kCW ? red[lane] : 0.f;
    return warp_sum(t);
}

struct Ring {
    unsigned char *base;
    uint64_t *full, *empty;
    int NS;
    volatile int *issued;    // chunks the producer has issued so far
    volatile int *abort;     // a bounded wait gave up: skip the remaining work, keep joining barriers
    int *first_fail;         // first chunk that was not consumed (for the final drain)
};

struct Grid {
    unsigned long long target = 0;
    __device__ void sync(const StepArgs &a) {
        cons_sync();
        target += gridDim.x;
        if (threadIdx.x == 0) {
            __threadfence();
            atomicAdd(a.bar, 1ull);
            const uint64_t t0 = ptx::now_ns();
            while (ld_acquire_u64(a.bar) < target) {
                if (ptx::now_ns() - t0 > kWaitNs || *(volatile int *)&a.st->error) {   // never hang
                    report(a, 7);
                    break;
                }
            }
            __threadfence();
        }
        cons_sync();
    }
};

enum { P_NORM = 0, P_EMBED = 1, P_PLAIN = 2, P_SWIGLU = 3 };
enum { E_STORE = 0, E_RESID = 1, E_ARGMAX = 2 };

// ------------------------------------------------------------------ producer
// Streams, in phase order, this CTA's rows of every projection of the step.
__device__ void produce(const StepArgs &a, const Ring &rg, volatile int *issued_s, volatile int *abort_s) {
    const int H = a.H, F = a.F, nqd = a.nq * kD;
    uint32_t g = 0;
    auto stream_rows = [&](const __nv_bfloat16 *W, int N, int K) -> bool {
        int r0, r1;
        cta_rows(N, r0, r1);
        const int R = rows_per_stage(K);
        const size_t rb = (size_t)K * 2;
        for (int r = r0; r < r1; r += R) {
            const int slot = g % rg.NS;
            if (g >= (uint32_t)rg.NS) {
                // chunk g - NS was issued after chunk g - 2NS had been consumed,
                // so this parity names exactly one phase
                bool ok = false;
                const uint64_t t0 = ptx::now_ns();
                while (!ok) {
                    if (*abort_s) return false;
                    ok = ptx::mbar_try_wait(&rg.empty[slot], ((g / rg.NS) - 1) & 1);
                    if (!ok && ptx::now_ns() - t0 > kWaitNs) break;
                }
                if (!ok) {
                    report(a, 8);
                    *abort_s = 1;
                    return false;
                }
            }
            const uint32_t bytes = (uint32_t)(min(R, r1 - r) * rb);
            ptx::mbar_expect_tx(&rg.full[slot], bytes);
            ptx::bulk_g2s(rg.base + (size_t)slot * kStage, reinterpret_cast<const unsigned char *>(W) + r * rb, bytes,
                          &rg.full[slot]);
            ++g;
            __threadfence_block();
            *issued_s = (int)g;
        }
        return true;
    };
    for (int l = 0; l < a.L; ++l) {
        const StepLayer &Ly = a.layers[l];
        if (!stream_rows(Ly.wqkv, a.qkv_n, H)) return;
        if (!stream_rows(Ly.wo, H, nqd)) return;
        if (!stream_rows(Ly.wgu, 2 * F, H)) return;
        if (!stream_rows(Ly.wd, H, F)) return;
    }
    stream_rows(a.embed, a.V, H);
}

// ------------------------------------------------------------------ projection phase (consumers)
template <int NB, int IN, int OUT>
__device__ __noinline__ void gemv_phase(const StepArgs &a, const Ring &rg, uint32_t &gctr, int N, int K,
                                        const float *in, const float *norm_w, float *out, float *xs, float *red,
                                        float *sred, const int *live, float (&best_v)[NB], int (&best_i)[NB]) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int CPR = K / 8;
    const int R = rows_per_stage(K);
    const size_t rb = (size_t)K * 2;
    int r0, r1;
    cta_rows(N, r0, r1);

    // prologue: activation rows into shared memory (the stages keep streaming)
    for (int b = 0; b < NB; ++b) {
        float *xr = xs + (size_t)b * K;
        if (IN == P_SWIGLU) {
            const float *gu = in + (size_t)b * 2 * a.F;
            for (int f0 = tid; f0 < K; f0 += 8 * kCT) {
                float gv[8], uv[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int f = f0 + i * kCT, blk = f >> 7, j = f & 127;
                    gv[i] = f < K ? gu[blk * 256 + j] : 0.f;
                    uv[i] = f < K ? gu[blk * 256 + 128 + j] : 0.f;
                }
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int f = f0 + i * kCT;
                    if (f < K) xr[xs_off(f, CPR)] = gv[i] / (1.f + expf(-gv[i])) * uv[i];
                }
            }
            continue;
        }
        const __nv_bfloat16 *er = IN == P_EMBED ? a.embed + (size_t)a.st->cur_tok[b] * K : nullptr;
        float ss = 0.f;
        for (int k0 = tid; k0 < K; k0 += 8 * kCT) {
            float v[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int k = k0 + i * kCT;
                v[i] = k < K ? (IN == P_EMBED ? __bfloat162float(er[k]) : in[(size_t)b * K + k]) : 0.f;
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int k = k0 + i * kCT;
                if (k < K) {
                    xr[xs_off(k, CPR)] = v[i];
                    ss += v[i] * v[i];
                    if (IN == P_EMBED && blockIdx.x == 0) a.x[(size_t)b * K + k] = v[i];
                }
            }
        }
        if (IN == P_PLAIN) continue;
        ss = cons_sum(ss, sred);
        const float r = rsqrtf(ss / (float)K + a.eps);
        for (int k = tid; k < K; k += kCT) {
            const int o = xs_off(k, CPR);
            xr[o] = xr[o] * r * norm_w[k];
        }
    }

    cons_sync();

    // Stages are dealt round-robin to the consumer warps: warp w consumes the
    // phase's chunks w, w + 16, ...  Each chunk holds whole rows, so a warp
    // finishes its rows itself and warps never wait on each other inside the
    // loop.  A warp may run more than one ring lap ahead of the slowest one, so
    // before the parity wait it waits until the producer has ISSUED chunk g:
    // that happens only after chunk g - NS was consumed, hence landed, so the
    // slot's barrier is then in the phase of chunk g and the parity is
    // unambiguous.  A wait that gives up marks the CTA aborted; every warp then
    // skips the rest of the step's chunks but still reaches every barrier.
    const int n_chunks = (r1 - r0 + R - 1) / R;
    for (int j = warp; j < n_chunks; j += kCW) {
        const uint32_t g = gctr + j;
        const int slot = g % rg.NS;
        const uint32_t par = (g / rg.NS) & 1;
        bool ok = !*rg.abort;
        if (ok && *rg.issued <= (int)g) {
            const uint64_t t0 = ptx::now_ns();
            while (*rg.issued <= (int)g && !*rg.abort && ptx::now_ns() - t0 <= kWaitNs) {
            }
            ok = *rg.issued > (int)g;
        }
        ok = ok && ptx::mbar_wait_ns(&rg.full[slot], par, kWaitNs);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) {
            if (lane == 0) {
                if (!*rg.abort) report(a, 9);
                *rg.abort = 1;
                atomicMin(rg.first_fail, (int)g);
            }
            break;
        }
        const int row0 = r0 + j * R, rows_here = min(R, r1 - row0);
        const unsigned char *stage = rg.base + (size_t)slot * kStage;
        for (int rr = 0; rr < rows_here; ++rr) {
            const uint4 *wr = reinterpret_cast<const uint4 *>(stage + rr * rb);
            float acc[NB];
#pragma unroll
            for (int b = 0; b < NB; ++b) acc[b] = 0.f;
#pragma unroll 4
            for (int c = lane; c < CPR; c += 32) {
                float f[8];
                unpack16(wr[c], f, (const __nv_bfloat16 *)nullptr);
#pragma unroll
                for (int b = 0; b < NB; ++b) {
                    const float4 *x4 = reinterpret_cast<const float4 *>(xs + (size_t)b * K);
                    const float4 lo = x4[c], hi = x4[CPR + c];
                    acc[b] = fmaf(f[0], lo.x, acc[b]);
                    acc[b] = fmaf(f[1], lo.y, acc[b]);
                    acc[b] = fmaf(f[2], lo.z, acc[b]);
                    acc[b] = fmaf(f[3], lo.w, acc[b]);
                    acc[b] = fmaf(f[4], hi.x, acc[b]);
                    acc[b] = fmaf(f[5], hi.y, acc[b]);
                    acc[b] = fmaf(f[6], hi.z, acc[b]);
                    acc[b] = fmaf(f[7], hi.w, acc[b]);
                }
            }
#pragma unroll
            for (int b = 0; b < NB; ++b) acc[b] = warp_sum(acc[b]);
            if (lane == 0) {
                const int row = row0 + rr;
#pragma unroll
                for (int b = 0; b < NB; ++b) {
                    if (!live[b]) continue;
                    const size_t o = (size_t)b * N + row;
                    if (OUT == E_STORE) out[o] = acc[b];
                    if (OUT == E_RESID) out[o] += acc[b];
                    if (OUT == E_ARGMAX) {
                        out[o] = acc[b];
                        if (acc[b] > best_v[b]) {        // rows ascend per warp: lowest index on ties
                            best_v[b] = acc[b];
                            best_i[b] = row;
                        }
                    }
                }
            }
        }
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&rg.empty[slot]);
    }
    gctr += n_chunks;
    cons_sync();
}

// ------------------------------------------------------------------ attention phase (consumers)
__device__ __noinline__ void attn_phase(const StepArgs &a, const StepLayer &Ly, float *smem, const int *live,
                                        unsigned *ticket) {
    float *qs = smem;                                       // [kRep][kD]
    float *wm = qs + kRep * kD;                             // [kCW][kRep]
    float *wl = wm + kCW * kRep;                            // [kCW][kRep]
    float *wacc = wl + kCW * kRep;                          // [kCW][kRep][kD]
    float *cw = wacc + kCW * kRep * kD;                     // [kAttnMaxSplits][kRep]
    float *cm = cw + kAttnMaxSplits * kRep;                 // [kAttnMaxSplits][kRep]
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nq = a.nq, nkv = a.nkv, n_rep = nq / nkv, S = a.splits;
    const int items = a.B * nkv * S;
    for (int it = blockIdx.x; it < items; it += gridDim.x) {
        const int b = it / (nkv * S), g = (it / S) % nkv, s = it % S;
        if (!live[b]) continue;
        const int pos = a.st->n_past[b], len = pos + 1, off = a.st->kv_off[b];
        // one split per 256 keys at least: short contexts run without a combine
        const int chunk = max(256, (len + S - 1) / S);
        const int n_used = (len + chunk - 1) / chunk;
        if (s >= n_used) continue;
        const int j0 = s * chunk, j1 = min(len, j0 + chunk);
        const float *row = a.qkv + (size_t)b * a.qkv_n;
        const float2 *rope_row = a.rope + (size_t)pos * (kD / 2);
        for (int r = warp; r < n_rep; r += kCW) {
            float v[kPL];
#pragma unroll
            for (int e = 0; e < kPL; ++e) v[e] = row[(size_t)(g * n_rep + r) * kD + lane * kPL + e];
            norm_rope_lane<kPL>(v, Ly.qn, a.eps, kD, rope_row, lane);
#pragma unroll
            for (int e = 0; e < kPL; ++e) qs[r * kD + lane * kPL + e] = v[e];
        }
        if (j0 <= pos && pos < j1) {                        // this split owns the new token's slot
            const size_t slot = ((size_t)g * a.slots + off + pos) * kD + lane * kPL;
            if (warp == n_rep) {
                float v[kPL];
#pragma unroll
                for (int e = 0; e < kPL; ++e) v[e] = row[(size_t)(nq + g) * kD + lane * kPL + e];
                norm_rope_lane<kPL>(v, Ly.kn, a.eps, kD, rope_row, lane);
#pragma unroll
                for (int e = 0; e < kPL; ++e) Ly.K[slot + e] = __float2half_rn(v[e]);
            } else if (warp == n_rep + 1) {
#pragma unroll
                for (int e = 0; e < kPL; ++e)
                    Ly.V[slot + e] = __float2half_rn(row[(size_t)(nq + nkv + g) * kD + lane * kPL + e]);
            }
        }
        cons_sync();
        float m[kRep], l[kRep], acc[kRep][kPL];
#pragma unroll
        for (int r = 0; r < kRep; ++r) {
            m[r] = -INFINITY;
            l[r] = 0.f;
#pragma unroll
            for (int e = 0; e < kPL; ++e) acc[r][e] = 0.f;
        }
        for (int jb = j0 + warp * kKB; jb < j1; jb += kCW * kKB) {
            float kf[kKB][kPL], vf[kKB][kPL];
#pragma unroll
            for (int k = 0; k < kKB; ++k) {
                const int j = jb + k;
                const size_t base = ((size_t)g * a.slots + off + j) * kD + lane * kPL;
#pragma unroll
                for (int e = 0; e < kPL; ++e) {
                    kf[k][e] = j < j1 ? __half2float(Ly.K[base + e]) : 0.f;
                    vf[k][e] = j < j1 ? __half2float(Ly.V[base + e]) : 0.f;
                }
            }
#pragma unroll
            for (int r = 0; r < kRep; ++r) {
                if (r < n_rep) {
                    float sc[kKB];
#pragma unroll
                    for (int k = 0; k < kKB; ++k) {
                        float d = 0.f;
#pragma unroll
                        for (int e = 0; e < kPL; ++e) d = fmaf(qs[r * kD + lane * kPL + e], kf[k][e], d);
                        sc[k] = d;
                    }
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1)
#pragma unroll
                        for (int k = 0; k < kKB; ++k) sc[k] += __shfl_xor_sync(0xffffffffu, sc[k], o);
                    float mb = m[r];
#pragma unroll
                    for (int k = 0; k < kKB; ++k) {
                        sc[k] = jb + k < j1 ? sc[k] * a.scale : -INFINITY;
                        mb = fmaxf(mb, sc[k]);
                    }
                    const float corr = expf(m[r] - mb);
                    float ls = 0.f;
#pragma unroll
                    for (int e = 0; e < kPL; ++e) acc[r][e] *= corr;
#pragma unroll
                    for (int k = 0; k < kKB; ++k) {
                        const float p = expf(sc[k] - mb);
                        ls += p;
#pragma unroll
                        for (int e = 0; e < kPL; ++e) acc[r][e] = fmaf(p, vf[k][e], acc[r][e]);
                    }
                    l[r] = l[r] * corr + ls;
                    m[r] = mb;
                }
            }
        }
#pragma unroll
        for (int r = 0; r < kRep; ++r) {
            if (r < n_rep) {
                if (lane == 0) {
                    wm[warp * kRep + r] = m[r];
                    wl[warp * kRep + r] = l[r];
                }
#pragma unroll
                for (int e = 0; e < kPL; ++e) wacc[(warp * kRep + r) * kD + lane * kPL + e] = acc[r][e];
            }
        }
        cons_sync();
        if (n_used == 1) {                                  // whole context in this CTA: normalise and write
            for (int idx = tid; idx < n_rep * kD; idx += kCT) {
                const int r = idx / kD, i = idx % kD;
                float M = -INFINITY;
                for (int w = 0; w < kCW; ++w) M = fmaxf(M, wm[w * kRep + r]);
                float A = 0.f, L = 0.f;
                for (int w = 0; w < kCW; ++w) {
                    const float f = wm[w * kRep + r] == -INFINITY ? 0.f : expf(wm[w * kRep + r] - M);
                    A += wacc[(w * kRep + r) * kD + i] * f;
                    L += wl[w * kRep + r] * f;
                }
                a.o[(size_t)b * nq * kD + (size_t)(g * n_rep + r) * kD + i] = A / L;
            }
            cons_sync();
            continue;
        }
        float *part = a.attn_part + (((size_t)b * nkv + g) * S + s) * n_rep * (kD + 2);
        for (int idx = tid; idx < n_rep * kD; idx += kCT) {
            const int r = idx / kD, i = idx % kD;
            float M = -INFINITY;
            for (int w = 0; w < kCW; ++w) M = fmaxf(M, wm[w * kRep + r]);
            float A = 0.f, L = 0.f;
            if (M != -INFINITY) {
                for (int w = 0; w < kCW; ++w) {
                    const float f = expf(wm[w * kRep + r] - M);
                    A += wacc[(w * kRep + r) * kD + i] * f;
                    L += wl[w * kRep + r] * f;
                }
            }
            float *pr = part + (size_t)r * (kD + 2);
            pr[i] = A;
            if (i == 0) {
                pr[kD] = M;
                pr[kD + 1] = L;
            }
        }
        __threadfence();
        cons_sync();
        if (tid == 0) *ticket = atomicAdd(&a.attn_counter[b * nkv + g], 1u);
        cons_sync();
        if (*ticket == (unsigned)n_used - 1) {
            __threadfence();
            const float *pb = a.attn_part + ((size_t)b * nkv + g) * S * n_rep * (kD + 2);
            for (int idx = tid; idx < n_used * n_rep; idx += kCT) {
                const int t = idx / n_rep, r = idx % n_rep;
                const float *pr = pb + ((size_t)t * n_rep + r) * (kD + 2);
                cm[t * kRep + r] = __ldcg(pr + kD);
                cw[t * kRep + r] = __ldcg(pr + kD + 1);
            }
            cons_sync();
            if (tid < n_rep) {
                const int r = tid;
                float Mx = -INFINITY;
                for (int t = 0; t < n_used; ++t) Mx = fmaxf(Mx, cm[t * kRep + r]);
                float L = 0.f;
                for (int t = 0; t < n_used; ++t) {
                    const float f = cm[t * kRep + r] == -INFINITY ? 0.f : expf(cm[t * kRep + r] - Mx);
                    cm[t * kRep + r] = f;
                    L += cw[t * kRep + r] * f;
                }
                const float inv = 1.f / L;
                for (int t = 0; t < n_used; ++t) cw[t * kRep + r] = cm[t * kRep + r] * inv;
            }
            cons_sync();
            for (int idx = tid; idx < n_rep * kD; idx += kCT) {
                const int r = idx / kD, i = idx % kD;
                float A = 0.f;
#pragma unroll 4
                for (int t = 0; t < n_used; ++t)
                    A = fmaf(__ldcg(pb + ((size_t)t * n_rep + r) * (kD + 2) + i), cw[t * kRep + r], A);
                a.o[(size_t)b * nq * kD + (size_t)(g * n_rep + r) * kD + i] = A;
            }
            if (tid == 0) a.attn_counter[b * nkv + g] = 0u;
        }
        cons_sync();
    }
}

// ------------------------------------------------------------------ head: argmax across CTAs (consumers)
template <int NB>
__device__ __noinline__ void argmax_phase(const StepArgs &a, float (&best_v)[NB], int (&best_i)[NB],
                                          const int *live, float *wv, int *wi, unsigned *ticket) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, V = a.V;
    // candidates sit in lane 0 of the row-owner warps; others hold -inf
#pragma unroll
    for (int b = 0; b < NB; ++b) {
        if (lane == 0) {
            wv[warp * kGroupB + b] = best_v[b];
            wi[warp * kGroupB + b] = best_i[b];
        }
    }
    cons_sync();
    const int G = gridDim.x;
    if (tid < NB && live[tid]) {
        float bv = -INFINITY;
        int bi = 0x7fffffff;
        for (int w = 0; w < kCW; ++w) {
            const float v = wv[w * kGroupB + tid];
            const int ix = wi[w * kGroupB + tid];
            if (v > bv || (v == bv && ix < bi)) { bv = v; bi = ix; }
        }
        a.am_val[(size_t)tid * G + blockIdx.x] = bv;
        a.am_idx[(size_t)tid * G + blockIdx.x] = bi;
    }
    __threadfence();
    cons_sync();
    if (tid == 0) *ticket = atomicAdd(a.am_counter, 1u);
    cons_sync();
    if (*ticket != (unsigned)G - 1) return;
    __threadfence();
    for (int b = 0; b < NB; ++b) {
        if (!live[b]) continue;
        float bv = -INFINITY;
        int bi = 0x7fffffff;
        for (int i = tid; i < G; i += kCT) {
            const float v = __ldcg(a.am_val + (size_t)b * G + i);
            const int ix = __ldcg(a.am_idx + (size_t)b * G + i);
            if (v > bv || (v == bv && ix < bi)) { bv = v; bi = ix; }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float v = __shfl_xor_sync(0xffffffffu, bv, o);
            const int ix = __shfl_xor_sync(0xffffffffu, bi, o);
            if (v > bv || (v == bv && ix < bi)) { bv = v; bi = ix; }
        }
        cons_sync();
        if (lane == 0) {
            wv[warp] = bv;
            wi[warp] = bi;
        }
        cons_sync();
        if (tid == 0) {
            for (int w = 1; w < kCW; ++w)
                if (wv[w] > bv || (wv[w] == bv && wi[w] < bi)) { bv = wv[w]; bi = wi[w]; }
            SeqState *st = a.st;
            if (bi < 0 || bi >= V) {
                atomicCAS(&st->error, 0, 2);
                bi = 0;
            }
            st->cur_tok[b] = bi;
            const int gc = st->gen[b];
            if (gc < a.out_ids_cap) a.out_ids[(size_t)b * a.out_ids_cap + gc] = bi;
            st->gen[b] = gc + 1;
            const int np = st->n_past[b] + 1;
            st->n_past[b] = np;
            if (bi == st->eos_id || gc + 1 >= st->max_new || np + 1 > st->kv_cap[b]) st->done[b] = 1;
        }
    }
    if (tid == 0) *a.am_counter = 0u;
}

// ------------------------------------------------------------------ the step kernel
template <int NB>
__global__ void __launch_bounds__(kTT, 1) k_decode_step(StepArgs a) {
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ float sred[32];
    __shared__ int live[kGroupB];
    __shared__ int any_s;
    __shared__ volatile int issued_s;
    __shared__ int first_fail_s;
    __shared__ volatile int abort_s, prod_done_s;
    __shared__ unsigned ticket_s;
    __shared__ float wv[kCW * kGroupB];
    __shared__ int wi[kCW * kGroupB];

    const int NS = a.ring_stages;
    Ring rg;
    rg.base = smem;
    float *xs = reinterpret_cast<float *>(smem + (size_t)NS * kStage);           // activations / attention
    float *red = xs + a.union_floats;                                            // [2][kCW][kCW][kGroupB]
    rg.full = reinterpret_cast<uint64_t *>(red + 2 * kCW * kCW * kGroupB);
    rg.empty = rg.full + NS;
    rg.NS = NS;
    rg.issued = &issued_s;
    rg.abort = &abort_s;
    rg.first_fail = &first_fail_s;

    // after a recorded error every further step is a no-op
    if (threadIdx.x < kGroupB)
        live[threadIdx.x] = threadIdx.x < NB && row_live(a.st, threadIdx.x) && a.st->error == 0;
    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            ptx::mbar_init(&rg.full[s], 1);
            ptx::mbar_init(&rg.empty[s], 1);
        }
        abort_s = 0;
        prod_done_s = 0;
        issued_s = 0;
        first_fail_s = 0x7fffffff;
        ptx::fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        int any = 0;
        for (int b = 0; b < NB; ++b) any |= live[b];
        any_s = any;
    }
    __syncthreads();
    if (!any_s) return;                                     // finished rows: the step is a no-op

    if (threadIdx.x >= kCT) {                               // producer warp
        if (threadIdx.x == kCT) {
            produce(a, rg, &issued_s, &abort_s);
            __threadfence_block();
            prod_done_s = 1;
        }
        return;
    }

    Grid grid;
    uint32_t gctr = 0;
    const int H = a.H, F = a.F, nqd = a.nq * kD;
    float nb_v[NB];
    int nb_i[NB];
    for (int l = 0; l < a.L; ++l) {
        const StepLayer &Ly = a.layers[l];
        if (l == 0)
            gemv_phase<NB, P_EMBED, E_STORE>(a, rg, gctr, a.qkv_n, H, nullptr, Ly.attn_norm, a.qkv, xs, red, sred,
                                             live, nb_v, nb_i);
        else
            gemv_phase<NB, P_NORM, E_STORE>(a, rg, gctr, a.qkv_n, H, a.x, Ly.attn_norm, a.qkv, xs, red, sred, live,
                                            nb_v, nb_i);
        grid.sync(a);
        attn_phase(a, Ly, xs, live, &ticket_s);
        grid.sync(a);
        gemv_phase<NB, P_PLAIN, E_RESID>(a, rg, gctr, H, nqd, a.o, nullptr, a.x, xs, red, sred, live, nb_v, nb_i);
        grid.sync(a);
        gemv_phase<NB, P_NORM, E_STORE>(a, rg, gctr, 2 * F, H, a.x, Ly.ffn_norm, a.gu, xs, red, sred, live, nb_v,
                                        nb_i);
        grid.sync(a);
        gemv_phase<NB, P_SWIGLU, E_RESID>(a, rg, gctr, H, F, a.gu, nullptr, a.x, xs, red, sred, live, nb_v, nb_i);
        grid.sync(a);
    }
    float best_v[NB];
    int best_i[NB];
#pragma unroll
    for (int b = 0; b < NB; ++b) {
        best_v[b] = -INFINITY;
        best_i[b] = 0x7fffffff;
    }
    gemv_phase<NB, P_NORM, E_ARGMAX>(a, rg, gctr, a.V, H, a.x, a.final_norm, a.logits, xs, red, sred, live, best_v,
                                     best_i);
    argmax_phase<NB>(a, best_v, best_i, live, wv, wi, &ticket_s);
    // a wait that gave up: once the producer has stopped, drain the copies it
    // issued that nobody consumed, so none lands after the CTA exits
    cons_sync();
    if (threadIdx.x == 0 && abort_s) {
        const uint64_t t0 = ptx::now_ns();
        while (!prod_done_s && ptx::now_ns() - t0 <= kWaitNs) __nanosleep(64);
        for (int g = first_fail_s; g < issued_s; ++g) ptx::mbar_wait_ns(&rg.full[g % NS], (g / NS) & 1, kWaitNs);
    }
}

// ------------------------------------------------------------------ host side
static void *step_kernel(int B) {
    switch (B) {
    case 1: return reinterpret_cast<void *>(k_decode_step<1>);
    case 2: return reinterpret_cast<void *>(k_decode_step<2>);
    case 3: return reinterpret_cast<void *>(k_decode_step<3>);
    default: return reinterpret_cast<void *>(k_decode_step<4>);
    }
}

static int g_optin = 0;

StepPlan step_plan(int H, int F, int nqd, int B) {
    StepPlan p{};
    int dev = 0, coop = 0;
    if (!g_optin && cudaGetDevice(&dev) == cudaSuccess) {
        cudaDeviceGetAttribute(&g_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev);
        if (!coop) g_optin = -1;
    }
    if (g_optin <= 0) return p;
    const int max_k = std::max(H, std::max(F, nqd));
    const size_t xs = (size_t)B * max_k * 4;
    const size_t attn = ((size_t)kRep * kD + 2 * kCW * kRep + (size_t)kCW * kRep * kD + 2 * kAttnMaxSplits * kRep) * 4;
    p.union_floats = (int)((std::max(xs, attn) + 15) / 16 * 4);
    const size_t red = (size_t)2 * kCW * kCW * kGroupB * 4;
    const size_t fixed = (size_t)p.union_floats * 4 + red + 1024;            // + barriers and slack
    const size_t static_smem = 2048;
    if ((size_t)g_optin < fixed + static_smem + 2 * (size_t)kStage) return p;
    p.ring_stages = (int)std::min<size_t>(12, ((size_t)g_optin - static_smem - fixed) / kStage);
    p.smem = (size_t)p.ring_stages * kStage + fixed;
    p.ok = p.ring_stages >= 2;
    return p;
}

bool step_supported(int head_dim, int n_rep, int H, int F, int nqd, int max_b) {
    if (head_dim != kD || n_rep < 1 || n_rep > kRep) return false;
    for (int B = 1; B <= max_b && B <= kGroupB; ++B) {
        const StepPlan p = step_plan(H, F, nqd, B);
        if (!p.ok) return false;
        const void *fn = step_kernel(B);
        int per_sm = 0;
        if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p.smem) != cudaSuccess ||
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, kTT, p.smem) != cudaSuccess || per_sm < 1) {
            cudaGetLastError();
            return false;
        }
    }
    return true;
}

cudaError_t launch_step(StepArgs a, int num_sms, cudaStream_t s) {
    const StepPlan p = step_plan(a.H, a.F, a.nq * kD, a.B);
    if (!p.ok) return cudaErrorInvalidValue;
    a.ring_stages = p.ring_stages;
    a.union_floats = p.union_floats;
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
    return cudaLaunchKernelExC(&cfg, step_kernel(a.B), args);
}

}  // namespace dec
