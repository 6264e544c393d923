// Device code of the decode attention shared by the standalone step-attention
// kernel and the q|k|v GEMV that finishes a KV head's attention itself:
// vector loads, per-head Q/K RMSNorm + NeoX RoPE in registers, the online
// softmax over key batches, the split combine, and the step-mode core.
//
// Block math (qwen3_asr/decoder.cpp, build_step_graph; the decoder block of
// the page's file header): q, k normed per head then rotated at the row's
// position, k and v appended at slot n_past, softmax(q k^T / sqrt(d)) v over
// slots [0, n_past] of the sequence, query head h reading KV head h / n_rep.
#pragma once
#include "decode.cuh"
#include "ptx.cuh"

namespace dec {
namespace {

__device__ __forceinline__ unsigned atomic_add_acq_rel(unsigned *p, unsigned v) {
    unsigned old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

// PL contiguous values of one lane in a single vector load (the lane's offset
// is a multiple of PL elements; rows are 256-byte aligned)
template <int PL>
__device__ __forceinline__ void load_vec(const float *p, float (&f)[PL]) {
    static_assert(PL == 2 || PL == 4, "2 or 4 values per lane");
    if (PL == 4) {
        const float4 v = *reinterpret_cast<const float4 *>(p);
        f[0] = v.x; f[1] = v.y; f[PL == 4 ? 2 : 0] = v.z; f[PL == 4 ? 3 : 1] = v.w;
    } else {
        const float2 v = *reinterpret_cast<const float2 *>(p);
        f[0] = v.x; f[1] = v.y;
    }
}

// load_vec through L2 (the values may come from other CTAs of the same kernel)
template <int PL>
__device__ __forceinline__ void load_vec_cg(const float *p, float (&f)[PL]) {
    static_assert(PL == 2 || PL == 4, "2 or 4 values per lane");
    if (PL == 4) {
        const float4 v = __ldcg(reinterpret_cast<const float4 *>(p));
        f[0] = v.x; f[1] = v.y; f[PL == 4 ? 2 : 0] = v.z; f[PL == 4 ? 3 : 1] = v.w;
    } else {
        const float2 v = __ldcg(reinterpret_cast<const float2 *>(p));
        f[0] = v.x; f[1] = v.y;
    }
}

template <typename TKV, int PL>
__device__ __forceinline__ void load_kv(const TKV *p, float (&f)[PL]) {
    if constexpr (sizeof(TKV) == 4) {
        load_vec<PL>(reinterpret_cast<const float *>(p), f);
    } else if constexpr (PL == 4) {
        const uint2 u = *reinterpret_cast<const uint2 *>(p);
        const float2 a = __half22float2(*reinterpret_cast<const __half2 *>(&u.x));
        const float2 b = __half22float2(*reinterpret_cast<const __half2 *>(&u.y));
        f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
    } else {
        const uint32_t u = *reinterpret_cast<const uint32_t *>(p);
        const float2 a = __half22float2(*reinterpret_cast<const __half2 *>(&u));
        f[0] = a.x; f[1] = a.y;
    }
}

// Per-head RMSNorm * w, then NeoX RoPE, with the lane's weights (w) and
// cos/sin pairs (cs, for dims (lane & 15) * PL + e) already in registers; RoPE
// partners (i, i + d/2) sit 16 lanes apart.
template <int PL>
__device__ __forceinline__ void norm_rope_regs(float (&v)[PL], const float (&w)[PL], const float2 (&cs)[PL],
                                               float eps, int D, int lane) {
    float ss = 0.f;
#pragma unroll
    for (int e = 0; e < PL; ++e) ss += v[e] * v[e];
    ss = warp_sum(ss);
    const float r = rsqrtf(ss / (float)D + eps);
#pragma unroll
    for (int e = 0; e < PL; ++e) v[e] = v[e] * r * w[e];
#pragma unroll
    for (int e = 0; e < PL; ++e) {
        const float p = __shfl_xor_sync(0xffffffffu, v[e], 16);
        v[e] = lane < 16 ? (v[e] * cs[e].x - p * cs[e].y) : (v[e] * cs[e].x + p * cs[e].y);
    }
}

constexpr int kMaxRep = 8;
constexpr int kKB = 8;     // keys per warp batch in the decode attention
constexpr int kAW = 8;     // warps per attention CTA

template <typename TKV, int PL>
__device__ __forceinline__ void load_kv_batch(const TKV *Kc, const TKV *Vc, size_t head_base, int jb, int j1, int lane,
                                              float (&kf)[kKB][PL], float (&vf)[kKB][PL]) {
#pragma unroll
    for (int k = 0; k < kKB; ++k) {
        const int j = jb + k;
        if (j < j1) {
            const size_t base = head_base + (size_t)j * (PL * 32) + lane * PL;
            load_kv<TKV, PL>(Kc + base, kf[k]);
            load_kv<TKV, PL>(Vc + base, vf[k]);
        } else {
#pragma unroll
            for (int e = 0; e < PL; ++e) kf[k][e] = vf[k][e] = 0.f;
        }
    }
}

// One batch of kKB keys (registers kf, vf; keys jb + k < j1 are real) for
// every query head of the group: scores, online softmax, weighted values.
template <int PL>
__device__ __forceinline__ void attn_batch(const float (*qs)[PL * 32], const float (&kf)[kKB][PL],
                                           const float (&vf)[kKB][PL], int jb, int j1, int n_rep, float scale,
                                           int lane, float (&m)[kMaxRep], float (&l)[kMaxRep],
                                           float (&acc)[kMaxRep][PL]) {
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

// Shared memory of the attention CTAs (W warps) besides the key/value tiles.
template <int D, int W>
struct AttnSmem {
    float qs[kMaxRep][D];
    float wm[W][kMaxRep], wl[W][kMaxRep];
    float wacc[W][kMaxRep][D];
    float cw[kAttnMaxSplits][kMaxRep], cm[kAttnMaxSplits][kMaxRep];
    unsigned ticket;
};

// Every warp's (m, l, acc) is in shared memory.  One split: normalise and
// write o.  Several: write this split's partial, take an acquire-release
// ticket, and the last split of the (sequence, kv head) combines them with
// log-sum-exp weights.  All threads of the CTA take part.
template <int D, int W>
__device__ void attn_finish(const AttnDecArgs &a, AttnSmem<D, W> &sm, int b, int g, int s, int S, int n_used,
                            int n_rep) {
    const int tid = threadIdx.x, nkv = a.nkv;
    if (n_used == 1) {
        for (int idx = tid; idx < n_rep * D; idx += blockDim.x) {
            const int r = idx / D, i = idx % D;
            float M = -INFINITY;
            for (int w = 0; w < W; ++w) M = fmaxf(M, sm.wm[w][r]);
            float A = 0.f, L = 0.f;
            for (int w = 0; w < W; ++w) {
                const float f = sm.wm[w][r] == -INFINITY ? 0.f : expf(sm.wm[w][r] - M);
                A += sm.wacc[w][r][i] * f;
                L += sm.wl[w][r] * f;
            }
            const size_t oi = (size_t)b * a.nq * D + (size_t)(g * n_rep + r) * D + i;
            a.o[oi] = A / L;
            if (a.o_bf16) store_planes(a.o_bf16, a.o_bf16_lo, oi, A / L);
        }
        return;
    }
    float *part = a.part + (((size_t)b * nkv + g) * S + s) * n_rep * (D + 2);
    for (int idx = tid; idx < n_rep * D; idx += blockDim.x) {
        const int r = idx / D, i = idx % D;
        float M = -INFINITY;
        for (int w = 0; w < W; ++w) M = fmaxf(M, sm.wm[w][r]);
        float A = 0.f, L = 0.f;
        if (M != -INFINITY) {
            for (int w = 0; w < W; ++w) {
                const float f = expf(sm.wm[w][r] - M);
                A += sm.wacc[w][r][i] * f;
                L += sm.wl[w][r] * f;
            }
        }
        float *pr = part + (size_t)r * (D + 2);
        pr[i] = A;
        if (i == 0) { pr[D] = M; pr[D + 1] = L; }
    }
    // the CTA's partial is complete (barrier); one acquire-release ticket per
    // CTA publishes it and, for the last split, makes every other split's visible
    __syncthreads();
    if (tid == 0) sm.ticket = atomic_add_acq_rel(&a.counter[b * nkv + g], 1u);
    __syncthreads();
    if (sm.ticket != (unsigned)n_used - 1) return;

    // last split: the per-split maxima and sums are staged in shared memory
    // first, then every output element is a weighted sum over the splits
    const float *pb = a.part + ((size_t)b * nkv + g) * S * n_rep * (D + 2);
    for (int idx = tid; idx < n_used * n_rep; idx += blockDim.x) {
        const int t = idx / n_rep, r = idx % n_rep;
        const float *pr = pb + ((size_t)t * n_rep + r) * (D + 2);
        sm.cm[t][r] = __ldcg(pr + D);
        sm.cw[t][r] = __ldcg(pr + D + 1);
    }
    __syncthreads();
    if (tid < n_rep) {
        const int r = tid;
        float Mx = -INFINITY;
        for (int t = 0; t < n_used; ++t) Mx = fmaxf(Mx, sm.cm[t][r]);
        float L = 0.f;
        for (int t = 0; t < n_used; ++t) {
            const float f = sm.cm[t][r] == -INFINITY ? 0.f : expf(sm.cm[t][r] - Mx);
            sm.cm[t][r] = f;
            L += sm.cw[t][r] * f;
        }
        const float inv = 1.f / L;
        for (int t = 0; t < n_used; ++t) sm.cw[t][r] = sm.cm[t][r] * inv;
    }
    __syncthreads();
    for (int idx = tid; idx < n_rep * D; idx += blockDim.x) {
        const int r = idx / D, i = idx % D;
        float A = 0.f;
#pragma unroll 4
        for (int t = 0; t < n_used; ++t) A = fmaf(__ldcg(pb + ((size_t)t * n_rep + r) * (D + 2) + i), sm.cw[t][r], A);
        const size_t oi = (size_t)b * a.nq * D + (size_t)(g * n_rep + r) * D + i;
        a.o[oi] = A;
        if (a.o_bf16) store_planes(a.o_bf16, a.o_bf16_lo, oi, A);
    }
    if (tid == 0) a.counter[b * nkv + g] = 0u;
}

template <int D, int W>
__device__ __forceinline__ void attn_park(AttnSmem<D, W> &sm, const float (&m)[kMaxRep], const float (&l)[kMaxRep],
                                          const float (&acc)[kMaxRep][D / 32], int n_rep, int warp, int lane) {
    constexpr int PL = D / 32;
#pragma unroll
    for (int r = 0; r < kMaxRep; ++r) {
        if (r < n_rep) {
            if (lane == 0) { sm.wm[warp][r] = m[r]; sm.wl[warp][r] = l[r]; }
#pragma unroll
            for (int e = 0; e < PL; ++e) sm.wacc[warp][r][lane * PL + e] = acc[r][e];
        }
    }
}


// ---------------------------------------------------------------- step mode
// The step's row: Q/K RMSNorm + NeoX RoPE, K/V append at slot n_past, then the
// split's keys.  The CTA copies its keys and values from the pool into
// shared-memory tiles with two 1-D bulk copies (TMA) per tile: one round trip
// however many keys the split holds, overlapped with the query work.  The
// appended key (slot n_past) is written into the tile from registers.
// Keys are scored by groups of kLG lanes (kLG = 8: each lane holds D / 8 dims
// of the key, the query heads' matching dims in registers), four keys per warp
// at a time: a score needs three shuffle levels, and each group keeps its own
// online softmax over its keys; the groups of a warp are merged once at the end.
constexpr int kLG = 8;
constexpr int kSW = 16;                 // warps of the step attention (n_rep <= 2)

template <int N>
__device__ __forceinline__ void load_seg(const __half *p, float (&f)[N]) {
    static_assert(N % 8 == 0, "whole 16-byte chunks");
#pragma unroll
    for (int c = 0; c < N / 8; ++c) {
        const uint4 u = reinterpret_cast<const uint4 *>(p)[c];
        const __half2 *h = reinterpret_cast<const __half2 *>(&u);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 t = __half22float2(h[i]);
            f[c * 8 + 2 * i] = t.x;
            f[c * 8 + 2 * i + 1] = t.y;
        }
    }
}
template <int N>
__device__ __forceinline__ void load_seg(const float *p, float (&f)[N]) {
    static_assert(N % 4 == 0, "whole 16-byte chunks");
#pragma unroll
    for (int c = 0; c < N / 4; ++c) {
        const float4 u = reinterpret_cast<const float4 *>(p)[c];
        f[4 * c] = u.x;
        f[4 * c + 1] = u.y;
        f[4 * c + 2] = u.z;
        f[4 * c + 3] = u.w;
    }
}

// The lane with index g in its key group holds, of each D-element row, the
// 16-byte chunks c * kLG + g (c < DL / EPC, EPC elements per chunk): the kLG
// lanes of a group read 128 contiguous bytes per load, free of bank
// conflicts.  ildim gives the row element behind local element i.
template <typename TKV>
__host__ __device__ constexpr int il_epc() { return 16 / (int)sizeof(TKV); }
template <typename TKV>
__device__ __forceinline__ int ildim(int i, int g) {
    constexpr int EPC = il_epc<TKV>();
    return ((i / EPC) * kLG + g) * EPC + i % EPC;
}
template <int N>
__device__ __forceinline__ void load_seg_il(const __half *row, int g, float (&f)[N]) {
#pragma unroll
    for (int c = 0; c < N / 8; ++c) {
        const uint4 u = reinterpret_cast<const uint4 *>(row)[c * kLG + g];
        const __half2 *h = reinterpret_cast<const __half2 *>(&u);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 t = __half22float2(h[i]);
            f[c * 8 + 2 * i] = t.x;
            f[c * 8 + 2 * i + 1] = t.y;
        }
    }
}
template <int N>
__device__ __forceinline__ void load_seg_il(const float *row, int g, float (&f)[N]) {
#pragma unroll
    for (int c = 0; c < N / 4; ++c) {
        const float4 u = reinterpret_cast<const float4 *>(row)[c * kLG + g];
        f[4 * c] = u.x;
        f[4 * c + 1] = u.y;
        f[4 * c + 2] = u.z;
        f[4 * c + 3] = u.w;
    }
}

template <typename TKV, int D>
constexpr int attn_tile_keys() {
    return 65536 / (D * (int)sizeof(TKV)) < 256 ? 65536 / (D * (int)sizeof(TKV)) : 256;
}


// One (sequence b, kv head g, split s of S) of the step attention, run by all
// W warps of the CTA once the step's q/k/v row is complete.  dsm holds NBUF
// buffers of key and value tiles (T keys each) followed by AttnSmem<D, W>:
// tile k of the split goes to buffer k % NBUF, the first NBUF tiles are
// requested at once and each later one as soon as its buffer is consumed.
// bar[i] is buffer i's initialised mbarrier, bit i of phase the parity of its
// next phase; qw, kw are this lane's Q/K norm weights; splits hold at least
// min_chunk keys.  The q/k/v row is read through L2: other CTAs of the same
// kernel may have written it.  Rows that are not live and splits without keys
// return at once (uniformly).
template <typename TKV, int D, int NREP, int W, int T, int NBUF>
__device__ void attn_step_core(const AttnDecArgs &a, float scale, int g, int s, int S, int b, unsigned char *dsm,
                               uint64_t *bar, uint32_t &phase, const float (&qw)[D / 32], const float (&kw)[D / 32],
                               int min_chunk) {
    constexpr int PL = D / 32;
    constexpr int DL = D / kLG;
    TKV *Kb = reinterpret_cast<TKV *>(dsm);          // buffer i: keys at Kb + 2 i T D, values T D further
    AttnSmem<D, W> &sm = *reinterpret_cast<AttnSmem<D, W> *>(dsm + (size_t)NBUF * 2 * T * D * sizeof(TKV));
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int n_rep = NREP ? NREP : a.nq / a.nkv;
    // the step's raw q/k/v rows do not depend on the sequence state: issue
    // their loads first (warp r < n_rep takes query head r; warps 0 and 1 the
    // new key and value, used only by the split that appends them)
    const size_t ldq = (size_t)(a.nq + 2 * a.nkv) * D;
    const float *row = a.qkv + (size_t)b * ldq;
    float qv[PL], nv[PL];
    load_vec_cg<PL>(row + (size_t)(g * n_rep + (warp < n_rep ? warp : 0)) * D + lane * PL, qv);
    load_vec_cg<PL>(row + (size_t)(a.nq + (warp == 1 ? a.nkv : 0) + g) * D + lane * PL, nv);
    // the row's position and KV range load together with its liveness flags
    const int pos = a.st->n_past[b], len = pos + 1, off = a.st->kv_off[b];
    if (!row_live(a.st, b)) return;
    int chunk, n_used;
    attn_split(len, S, chunk, n_used, min_chunk);
    if (s >= n_used) return;
    const int j0 = s * chunk, j1 = min(len, j0 + chunk);
    TKV *Kc = reinterpret_cast<TKV *>(a.Kc);
    TKV *Vc = reinterpret_cast<TKV *>(a.Vc);
    const size_t head_base = ((size_t)g * a.slots + off) * D;
    // this position's cos/sin pairs
    float2 cs[PL];
    {
        const float2 *rope_row = a.rope + (size_t)pos * (D / 2) + (lane & 15) * PL;
#pragma unroll
        for (int e = 0; e < PL; e += 2) {
            const float4 c = *reinterpret_cast<const float4 *>(rope_row + e);
            cs[e] = make_float2(c.x, c.y);
            cs[e + 1] = make_float2(c.z, c.w);
        }
    }
    __syncthreads();                                  // the buffers' previous use is over for every thread
    // keys [t0, min(t1, pos)) of tile t0 from the pool (the new key is written from registers)
    auto issue = [&](int t0) {
        const int t1 = min(j1, t0 + T), ncopy = max(0, min(t1, pos) - t0);
        if (ncopy <= 0) return;
        const int i = ((t0 - j0) / T) % NBUF;
        TKV *Ks = Kb + (size_t)i * 2 * T * D;
        const uint32_t bytes = (uint32_t)(ncopy * D * sizeof(TKV));
        ptx::mbar_expect_tx(&bar[i], 2 * bytes);
        ptx::bulk_g2s(Ks, Kc + head_base + (size_t)t0 * D, bytes, &bar[i]);
        ptx::bulk_g2s(Ks + (size_t)T * D, Vc + head_base + (size_t)t0 * D, bytes, &bar[i]);
    };
    if (tid == 0)
        for (int k = 0; k < NBUF && j0 + k * T < j1; ++k) issue(j0 + k * T);

    constexpr int NR = NREP ? NREP : kMaxRep;         // running softmax state per head
    constexpr int AL = NREP ? DL : PL;                // accumulator dims per lane
    float m[NR], l[NR], acc[NR][AL];
#pragma unroll
    for (int r = 0; r < NR; ++r) {
        m[r] = -INFINITY;
        l[r] = 0.f;
#pragma unroll
        for (int e = 0; e < AL; ++e) acc[r][e] = 0.f;
    }
    const int lg = lane % kLG, kslot = lane / kLG;  // grouped scoring: dims (ildim) and key of this lane
    float qr[NREP ? NREP : 1][NREP ? DL : 1];
    bool failed = false;
    for (int t0 = j0; t0 < j1; t0 += T) {
        const int t1 = min(j1, t0 + T);
        const int ncopy = max(0, min(t1, pos) - t0);  // rows from the pool (the new key excluded)
        const int bi = ((t0 - j0) / T) % NBUF;
        TKV *Ks = Kb + (size_t)bi * 2 * T * D;
        TKV *Vs = Ks + (size_t)T * D;
        if (t0 == j0) {
            for (int r = warp; r < n_rep; r += W) {          // n_rep <= W: one head per warp
                float v[PL];
#pragma unroll
                for (int e = 0; e < PL; ++e) v[e] = qv[e];
                norm_rope_regs<PL>(v, qw, cs, a.eps, D, lane);
#pragma unroll
                for (int e = 0; e < PL; ++e) sm.qs[r][lane * PL + e] = v[e];
            }
        }
        if (t0 <= pos && pos < t1 && a.append) {          // the new key and value: pool and tile
            const size_t slot = head_base + (size_t)pos * D + lane * PL;
            const size_t ts = (size_t)(pos - t0) * D + lane * PL;
            if (warp == 0) {
                float v[PL];
#pragma unroll
                for (int e = 0; e < PL; ++e) v[e] = nv[e];
                norm_rope_regs<PL>(v, kw, cs, a.eps, D, lane);
#pragma unroll
                for (int e = 0; e < PL; ++e) {
                    const TKV q = from_f32<TKV>(v[e]);
                    Kc[slot + e] = q;
                    Ks[ts + e] = q;
                }
            } else if (warp == 1) {
#pragma unroll
                for (int e = 0; e < PL; ++e) {
                    const TKV q = from_f32<TKV>(nv[e]);
                    Vc[slot + e] = q;
                    Vs[ts + e] = q;
                }
            }
        }
        if (ncopy > 0) {
            const bool ok = ptx::mbar_wait_ns(&bar[bi], (phase >> bi) & 1u, 200000000ull);
            phase ^= 1u << bi;
            if (!ok && !failed) {
                failed = true;
                if (tid == 0) atomicCAS(&a.st->error, 0, 10);
            }
        }
        __syncthreads();                              // tiles, new key and queries visible
        if constexpr (NREP > 0) {
            if (t0 == j0) {
#pragma unroll
                for (int r = 0; r < NREP; ++r)
#pragma unroll
                    for (int i = 0; i < DL; ++i) qr[r][i] = sm.qs[r][ildim<TKV>(i, lg)];
            }
            for (int jb = t0 + warp * (32 / kLG); jb < t1; jb += W * (32 / kLG)) {
                const int j = jb + kslot;
                const bool valid = j < t1;
                float kk[DL];
                if (valid) {
                    load_seg_il<DL>(Ks + (size_t)(j - t0) * D, lg, kk);
                } else {
#pragma unroll
                    for (int i = 0; i < DL; ++i) kk[i] = 0.f;
                }
                float sc[NREP];
#pragma unroll
                for (int r = 0; r < NREP; ++r) {
                    float d = 0.f;
#pragma unroll
                    for (int i = 0; i < DL; ++i) d = fmaf(qr[r][i], kk[i], d);
#pragma unroll
                    for (int o = 1; o < kLG; o <<= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
                    sc[r] = d * scale;
                }
                if (valid) {
                    float vv[DL];
                    load_seg_il<DL>(Vs + (size_t)(j - t0) * D, lg, vv);
#pragma unroll
                    for (int r = 0; r < NREP; ++r) {
                        const float mb = fmaxf(m[r], sc[r]);
                        const float corr = expf(m[r] - mb), p = expf(sc[r] - mb);
                        l[r] = l[r] * corr + p;
#pragma unroll
                        for (int i = 0; i < DL; ++i) acc[r][i] = fmaf(p, vv[i], acc[r][i] * corr);
                        m[r] = mb;
                    }
                }
            }
        } else {
            for (int jb = t0 + warp * kKB; jb < t1; jb += W * kKB) {
                float kf[kKB][PL], vf[kKB][PL];
#pragma unroll
                for (int k = 0; k < kKB; ++k) {
                    const int j = jb + k;
                    if (j < t1) {
                        load_kv<TKV, PL>(Ks + (size_t)(j - t0) * D + lane * PL, kf[k]);
                        load_kv<TKV, PL>(Vs + (size_t)(j - t0) * D + lane * PL, vf[k]);
                    } else {
#pragma unroll
                        for (int e = 0; e < PL; ++e) kf[k][e] = vf[k][e] = 0.f;
                    }
                }
                attn_batch<PL>(sm.qs, kf, vf, jb, t1, n_rep, scale, lane, m, l, acc);
            }
        }
        __syncthreads();                              // tile consumed before its buffer is refilled
        if (tid == 0 && t0 + NBUF * T < j1) issue(t0 + NBUF * T);
    }
    if constexpr (NREP > 0) {
        // merge the warp's key groups (lanes with equal dims), then park the
        // warp's state: lanes of group 0 hold the dims
#pragma unroll
        for (int r = 0; r < NREP; ++r) {
            float M = m[r];
#pragma unroll
            for (int o = kLG; o < 32; o <<= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
            const float f = m[r] == -INFINITY ? 0.f : expf(m[r] - M);
            float L = l[r] * f;
#pragma unroll
            for (int o = kLG; o < 32; o <<= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
#pragma unroll
            for (int i = 0; i < DL; ++i) {
                float v = acc[r][i] * f;
#pragma unroll
                for (int o = kLG; o < 32; o <<= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
                if (kslot == 0) sm.wacc[warp][r][ildim<TKV>(i, lg)] = v;
            }
            if (lane == 0) {
                sm.wm[warp][r] = M;
                sm.wl[warp][r] = L;
            }
        }
    } else {
        attn_park<D, W>(sm, m, l, acc, n_rep, warp, lane);
    }
    __syncthreads();
    attn_finish<D, W>(a, sm, b, g, s, S, n_used, n_rep);
}

}  // namespace
}  // namespace dec
