// Tensor-core GEMM of the prefill projections on sm_103a: tcgen05.mma with
// TMEM accumulators, operands staged by TMA (cp.async.bulk.tensor, 128-byte
// swizzle), one elected thread issuing the MMAs.
//
// Swapped operands: the weight rows are the MMA's M side (128 features per
// tile) and the prompt rows are its N side (up to 256 tokens per tile), so a
// short prompt (T = 152) fills one N tile with no padding waste.  The
// accumulator tile sits in TMEM with TMEM lane = feature and column = token;
// the epilogue warps read it back with tcgen05.ld and write C[token][feature]
// (consecutive lanes -> consecutive features -> coalesced rows).
//
// Epilogues: store fp32 (q|k|v), add into the fp32 residual (o and down
// projections), or SwiGLU: a gate|up weight block of 256 rows feeds two MMAs
// into two TMEM column ranges, and the epilogue writes silu(gate) * up in bf16
// (model.cpp, load: pack_gate_up; decoder.cpp header: SwiGLU on packed
// gate_up).
//
// Activations in two planes: X = X_hi + X_lo, both bf16 (X_lo the bf16
// rounding of the residual x - X_hi), so the product carries about 16
// mantissa bits of each activation while the weights stay bf16; every K step
// issues one MMA per plane into the same accumulator.  Over 28 blocks a single
// bf16 rounding of every projection input alone moves the logits by about
// 2.4e-2 of their largest magnitude; with both planes the activations add
// next to nothing to the error.
//
// When a GEMM has fewer output tiles than SMs (short prompts), K is split
// across CTAs; each split writes its partial tile to scratch and a second,
// fully parallel kernel sums the splits in split order (deterministic) and
// applies the epilogue.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstdlib>

#include "gemm_tc.cuh"
#include "prefill.cuh"
#include "ptx.cuh"
#include "tc.cuh"

namespace dec {

constexpr int kBK = 64;                 // K elements per stage: one 128-byte swizzle row of bf16
constexpr int kTcThreads = 192;         // warp 0 TMA, warp 1 MMA + TMEM allocation, warps 2-5 epilogue
constexpr uint32_t kTcPolls = 1u << 24; // bounded mbarrier waits

struct TcArgs {
    int n_feat, T, K;
    int groups;                  // 1, or 2 for gate|up blocks
    int planes;                  // activation planes: 1 (X) or 2 (X_hi, X_lo)
    int BN, n_stages, k_tiles, splits, kt_per_split;
    int epi;
    float *C;
    int ldc;
    __nv_bfloat16 *Hout, *Hout_lo;  // SwiGLU output planes (Hout_lo may be null)
    int out_f16;                 // SwiGLU output: one fp16 plane in Hout (operands of an fp16 GEMM)
    int ldh;
    float *part;
    const float *bias;           // EPI_BIAS_F32
    int *err;
    uint32_t idesc, tmem_cols;
};

__device__ __forceinline__ void tc_report(int *err, int code) {
    if (err) atomicCAS(err, 0, code);
}

// ------------------------------------------------------------------ epilogue
// One output element: feature f of this tile (TMEM lane), token t.
__device__ __forceinline__ void epi_store(const TcArgs &a, int f, int t, float v, float up) {
    if (t >= a.T) return;
    if (a.epi == EPI_SWIGLU_BF16) {
        const float h = v / (1.f + expf(-v)) * up;
        if (a.out_f16) {
            reinterpret_cast<__half *>(a.Hout)[(size_t)t * a.ldh + f] = __float2half_rn(h);
            return;
        }
        const __nv_bfloat16 hi = __float2bfloat16_rn(h);
        a.Hout[(size_t)t * a.ldh + f] = hi;
        if (a.Hout_lo) a.Hout_lo[(size_t)t * a.ldh + f] = __float2bfloat16_rn(h - __bfloat162float(hi));
    } else if (f < a.n_feat) {
        float *c = a.C + (size_t)t * a.ldc + f;
        if (a.epi == EPI_STORE_F32) *c = v;
        else if (a.epi == EPI_BIAS_F32) *c = v + a.bias[f];
        else *c += v;
    }
}

// Residual epilogue of one chunk of N tokens [t0, t0 + N): feature row f and,
// with two_rows, row f + 128.  Every residual load is issued before the
// first store.  Written as `*c += v` per element, each load would wait for
// the previous element's store (the compiler cannot rule out that the two
// addresses alias), one memory round trip per element in turn.
template <int N>
__device__ __forceinline__ void resid_load(const TcArgs &a, int f, int t0, bool two_rows, float (&x0)[N],
                                           float (&x1)[N]) {
    const bool in0 = f < a.n_feat, in1 = two_rows && f + 128 < a.n_feat;
#pragma unroll
    for (int j = 0; j < N; ++j) {
        const int t = t0 + j;
        const float *c = a.C + (size_t)t * a.ldc + f;
        x0[j] = t < a.T && in0 ? __ldcg(c) : 0.f;
        x1[j] = t < a.T && in1 ? __ldcg(c + 128) : 0.f;
    }
}
template <int N>
__device__ __forceinline__ void resid_store(const TcArgs &a, int f, int t0, bool two_rows, const float (&x0)[N],
                                            const float (&x1)[N], const float (&v)[N], const float (&u)[N]) {
    const bool in0 = f < a.n_feat, in1 = two_rows && f + 128 < a.n_feat;
#pragma unroll
    for (int j = 0; j < N; ++j) {
        const int t = t0 + j;
        if (t >= a.T) break;
        float *c = a.C + (size_t)t * a.ldc + f;
        if (in0) c[0] = x0[j] + v[j];
        if (in1) c[128] = x1[j] + u[j];
    }
}

// kResid: the residual epilogue of one split (its own instance, so that the
// residual values' registers do not raise the other instances' count: a
// CTA with fewer registers shares its SM with more of the preceding
// kernel's CTAs under programmatic launch)
template <bool kResid>
__global__ void __launch_bounds__(kTcThreads, 1)
    k_gemm_tc(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
              const __grid_constant__ CUtensorMap tmB2, TcArgs a) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem =
        reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int S = a.n_stages;
    const uint32_t a_bytes = (uint32_t)a.groups * 16384u, b_bytes = (uint32_t)a.BN * 128u;
    const uint32_t stage_bytes = a_bytes + (uint32_t)a.planes * b_bytes;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + (size_t)S * stage_bytes);
    uint64_t *empty = full + S;
    uint64_t *done = empty + S;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(done + 1);
    __shared__ int abort_s;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m0 = blockIdx.x * 128 * a.groups;              // first weight row of the tile
    const int n0 = blockIdx.y * a.BN;                        // first token of the tile
    const int kt0 = blockIdx.z * a.kt_per_split;
    const int nk = min(a.k_tiles, kt0 + a.kt_per_split) - kt0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            ptx::mbar_init(&full[s], 1);
            ptx::mbar_init(&empty[s], 1);
        }
        ptx::mbar_init(done, 1);
        abort_s = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         ptx::smem_u32(tmem_slot)),
                     "r"(a.tmem_cols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    // Programmatic dependent launch: the weight tiles (A) do not depend on the
    // preceding kernel, so the first stages' A loads are issued before the
    // dependency wait; activations (B) and every global write come after it.
    ptx::pdl_launch();
    int issued = 0;    // producer: stages issued (for the drain on abort)
    if (warp == 0 && lane == 0) {
        // ---------------------------------------------------------- TMA producer
        const int pre = min(S, nk);
        for (int i = 0; i < pre; ++i) {
            ptx::mbar_expect_tx(&full[i], stage_bytes);
            tma_load_2d(smem + (size_t)i * stage_bytes, &tmA, (kt0 + i) * kBK, m0, &full[i]);
        }
        ptx::pdl_wait();
        for (int i = 0; i < pre; ++i) {
            unsigned char *st = smem + (size_t)i * stage_bytes;
            tma_load_2d(st + a_bytes, &tmB, (kt0 + i) * kBK, n0, &full[i]);
            if (a.planes == 2) tma_load_2d(st + a_bytes + b_bytes, &tmB2, (kt0 + i) * kBK, n0, &full[i]);
        }
        issued = pre;
        for (int i = pre; i < nk; ++i) {
            const int s = i % S;
            if (i >= S && !ptx::mbar_wait_bounded(&empty[s], ((i / S) - 1) & 1, kTcPolls)) {
                tc_report(a.err, 4);
                abort_s = 1;
                break;
            }
            if (*(volatile int *)&abort_s) break;
            ptx::mbar_expect_tx(&full[s], stage_bytes);
            unsigned char *st = smem + (size_t)s * stage_bytes;
            tma_load_2d(st, &tmA, (kt0 + i) * kBK, m0, &full[s]);
            tma_load_2d(st + a_bytes, &tmB, (kt0 + i) * kBK, n0, &full[s]);
            if (a.planes == 2) tma_load_2d(st + a_bytes + b_bytes, &tmB2, (kt0 + i) * kBK, n0, &full[s]);
            issued = i + 1;
        }
    } else if (warp == 1 && lane == 0) {
        // ---------------------------------------------------------- MMA issuer
        for (int i = 0; i < nk; ++i) {
            const int s = i % S;
            if (!ptx::mbar_wait_bounded(&full[s], (i / S) & 1, kTcPolls)) {
                tc_report(a.err, 5);
                abort_s = 1;
                break;
            }
            tc_fence_after();
            const uint32_t abase = ptx::smem_u32(smem + (size_t)s * stage_bytes), bbase = abase + a_bytes;
#pragma unroll
            for (int kk = 0; kk < kBK / 16; ++kk) {
                for (int pl = 0; pl < a.planes; ++pl) {
                    const uint64_t bdesc = sw128_desc(bbase + pl * b_bytes + kk * 32);
                    for (int g = 0; g < a.groups; ++g)
                        mma_f16(tmem + (uint32_t)(g * a.BN), sw128_desc(abase + g * 16384 + kk * 32), bdesc, a.idesc,
                                 (i | kk | pl) != 0);
                }
            }
            mma_commit(&empty[s]);                     // stage free once these MMAs have read it
        }
        mma_commit(done);                               // accumulator final
    } else if (warp >= 2) {
        // ---------------------------------------------------------- epilogue
        ptx::pdl_wait();
        const bool ok = ptx::mbar_wait_bounded(done, 0, kTcPolls);
        if (!ok) tc_report(a.err, 6);
        tc_fence_after();
        const int q = warp & 3;                         // TMEM lane quarter this warp may access
        const int r = 32 * q + lane;                    // feature row within the 128-row MMA tile
        const int f = (a.epi == EPI_SWIGLU_BF16 ? blockIdx.x * 128 : m0) + r;
        const uint32_t tq = tmem + ((uint32_t)(32 * q) << 16);
        const int ncols = a.groups * a.BN;
        // TMEM is read 32 columns per load where the tile allows (one wait per
        // load), 16 for a remainder
        if (a.splits == 1) {
            int c = 0;
            // two groups outside SwiGLU: rows m0 + 128 + r in the second TMEM range
            const bool pair = a.groups == 2 && a.epi != EPI_SWIGLU_BF16;
            if (kResid) {
                // 16 columns at a time: the residual values live next to the
                // accumulator values
                for (; c < a.BN; c += 16) {
                    float v[16], u[16], x0[16], x1[16];
                    resid_load<16>(a, f, n0 + c, pair, x0, x1);
                    tmem_ld16(tq + c, v);
                    if (a.groups == 2) tmem_ld16(tq + a.BN + c, u);
                    resid_store<16>(a, f, n0 + c, pair, x0, x1, v, u);
                }
            }
            for (; c + 32 <= a.BN; c += 32) {
                float v[32], u[32];
                tmem_ld32(tq + c, v);
                if (a.groups == 2) tmem_ld32(tq + a.BN + c, u);
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    epi_store(a, f, n0 + c + j, v[j], a.groups == 2 ? u[j] : 0.f);
                    if (pair) epi_store(a, f + 128, n0 + c + j, u[j], 0.f);
                }
            }
            for (; c < a.BN; c += 16) {
                float v[16], u[16];
                tmem_ld16(tq + c, v);
                if (a.groups == 2) tmem_ld16(tq + a.BN + c, u);
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    epi_store(a, f, n0 + c + j, v[j], a.groups == 2 ? u[j] : 0.f);
                    if (pair) epi_store(a, f + 128, n0 + c + j, u[j], 0.f);
                }
            }
        } else {
            // split-K: park the partial tile; k_splitk_reduce sums the splits
            const int tile = blockIdx.y * gridDim.x + blockIdx.x;
            float *mine = a.part + ((size_t)tile * a.splits + blockIdx.z) * ncols * 128;
            int c = 0;
            for (; c + 32 <= ncols; c += 32) {
                float v[32];
                tmem_ld32(tq + c, v);
#pragma unroll
                for (int j = 0; j < 32; ++j) mine[(size_t)(c + j) * 128 + r] = v[j];
            }
            for (; c < ncols; c += 16) {
                float v[16];
                tmem_ld16(tq + c, v);
#pragma unroll
                for (int j = 0; j < 16; ++j) mine[(size_t)(c + j) * 128 + r] = v[j];
            }
        }
    }
    // the producer drains what it issued if the MMA side gave up
    if (warp == 0 && lane == 0 && abort_s) {
        for (int i = 0; i < issued; ++i) ptx::mbar_wait_bounded(&full[i % S], (i / S) & 1, kTcPolls);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(a.tmem_cols) : "memory");
}

// Per-head Q/K RMSNorm + RoPE + KV write of one prompt row's head (the warp
// holds its 128 values, lane L features 4L .. 4L + 3 of q|k|v head hh):
// queries to r.q_out, keys to the pool, values to the pool and V^T.
__device__ __forceinline__ void rope_kv_head(const RopeKvArgs &r, int t, int hh, float (&v)[4], int lane) {
    constexpr int D = 128, PL = 4;
    const int pos = r.row_pos[t];
    const float2 *rope_row = r.rope + (size_t)pos * (D / 2);
    if (hh < r.nq) {
        norm_rope_lane<PL>(v, r.qn_w, r.eps, D, rope_row, lane);
        __half *q = reinterpret_cast<__half *>(r.q_out) + ((size_t)t * r.nq + hh) * D + lane * PL;
#pragma unroll
        for (int e = 0; e < PL; ++e) q[e] = __float2half_rn(v[e]);
    } else if (hh < r.nq + r.nkv) {
        const int g = hh - r.nq;
        norm_rope_lane<PL>(v, r.kn_w, r.eps, D, rope_row, lane);
        __half *K = reinterpret_cast<__half *>(r.Kc) + ((size_t)g * r.slots + r.row_slot[t]) * D + lane * PL;
#pragma unroll
        for (int e = 0; e < PL; ++e) K[e] = __float2half_rn(v[e]);
    } else {
        const int g = hh - r.nq - r.nkv;
        __half *V = reinterpret_cast<__half *>(r.Vc) + ((size_t)g * r.slots + r.row_slot[t]) * D + lane * PL;
        __half *vt = r.vt ? reinterpret_cast<__half *>(r.vt) + (size_t)(g * D + lane * PL) * r.vt_ld + r.row_vtcol[t]
                          : nullptr;
#pragma unroll
        for (int e = 0; e < PL; ++e) {
            const __half x = __float2half_rn(v[e]);
            V[e] = x;
            if (vt) vt[(size_t)e * r.vt_ld] = x;
        }
    }
}

// Sum the split-K partial tiles in split order and apply the epilogue.  One
// thread per (tile, token column, 4 consecutive features): reads are
// 512-byte coalesced per column and every load of a thread is independent.
// With rope set (128-row tiles = heads), a warp is one (head, row) and applies
// the Q/K norm, RoPE and KV write instead of storing q|k|v.
__global__ void __launch_bounds__(256) k_splitk_reduce(TcArgs a, int mt, RopeKvArgs rk, int rope) {
    ptx::pdl_launch();
    ptx::pdl_wait();
    const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    const int per_tile = a.BN * 32;
    const int tile = (int)(idx / per_tile), rem = (int)(idx % per_tile);
    const int c = rem >> 5, r = (rem & 31) * 4;
    const int tx = tile % mt, ty = tile / mt;
    const int t = ty * a.BN + c;
    if (ty >= (a.T + a.BN - 1) / a.BN || t >= a.T) return;
    const int ncols = a.groups * a.BN;
    const float *base = a.part + (size_t)tile * a.splits * ncols * 128;
    float4 g = make_float4(0.f, 0.f, 0.f, 0.f), u = g;
    for (int s = 0; s < a.splits; ++s) {
        const float4 v = __ldcg(reinterpret_cast<const float4 *>(base + ((size_t)s * ncols + c) * 128 + r));
        g.x += v.x; g.y += v.y; g.z += v.z; g.w += v.w;
        if (a.groups == 2) {
            const float4 w = __ldcg(reinterpret_cast<const float4 *>(base + ((size_t)s * ncols + a.BN + c) * 128 + r));
            u.x += w.x; u.y += w.y; u.z += w.z; u.w += w.w;
        }
    }
    if (rope) {
        float v[4] = {g.x, g.y, g.z, g.w};
        rope_kv_head(rk, t, tx, v, threadIdx.x & 31);
        return;
    }
    const int f = (a.epi == EPI_SWIGLU_BF16 ? tx * 128 : tx * 128 * a.groups) + r;
    epi_store(a, f, t, g.x, u.x);
    epi_store(a, f + 1, t, g.y, u.y);
    epi_store(a, f + 2, t, g.z, u.z);
    epi_store(a, f + 3, t, g.w, u.w);
    if (a.groups == 2 && a.epi != EPI_SWIGLU_BF16) {       // 256-row tile: the second 128 rows
        epi_store(a, f + 128, t, u.x, 0.f);
        epi_store(a, f + 129, t, u.y, 0.f);
        epi_store(a, f + 130, t, u.z, 0.f);
        epi_store(a, f + 131, t, u.w, 0.f);
    }
}

// Split-K sum of a residual projection (o, down) and the RMSNorm of the
// finished rows: one CTA per prompt row, warp w = 128-row weight tile w (lane
// L its features 4L .. 4L + 3).  The residual row is stored, its sum of
// squares reduced over the CTA, and the normalised row written as two bf16
// planes for the next projection.
struct NormArgs {
    const float *w;
    float eps;
    __nv_bfloat16 *hi, *lo;
    int f16;                     // one fp16 plane in hi instead of two bf16 planes
};

__global__ void __launch_bounds__(1024) k_splitk_resid_norm(TcArgs a, NormArgs n) {
    __shared__ float red[32];
    ptx::pdl_launch();
    ptx::pdl_wait();
    const int t = blockIdx.x, w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int H = a.n_feat, f = w * 128 + 4 * lane;
    const float *base = a.part + (size_t)w * a.splits * a.BN * 128 + (size_t)t * 128 + 4 * lane;
    float4 g = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int sp = 0; sp < a.splits; ++sp) {               // in split order
        const float4 v = __ldcg(reinterpret_cast<const float4 *>(base + (size_t)sp * a.BN * 128));
        g.x += v.x; g.y += v.y; g.z += v.z; g.w += v.w;
    }
    float4 *c = reinterpret_cast<float4 *>(a.C + (size_t)t * a.ldc + f);
    float4 x = *c;
    x.x += g.x; x.y += g.y; x.z += g.z; x.w += g.w;
    *c = x;
    const float ss = block_sum(x.x * x.x + x.y * x.y + x.z * x.z + x.w * x.w, red);
    const float r = rsqrtf(ss / (float)H + n.eps);
    const float4 wv = *reinterpret_cast<const float4 *>(n.w + f);
    const size_t o = (size_t)t * H + f;
    if (n.f16) {
        __half2 *hp = reinterpret_cast<__half2 *>(reinterpret_cast<__half *>(n.hi) + o);
        hp[0] = __floats2half2_rn(x.x * r * wv.x, x.y * r * wv.y);
        hp[1] = __floats2half2_rn(x.z * r * wv.z, x.w * r * wv.w);
        return;
    }
    store_planes(n.hi, n.lo, o, x.x * r * wv.x);
    store_planes(n.hi, n.lo, o + 1, x.y * r * wv.y);
    store_planes(n.hi, n.lo, o + 2, x.z * r * wv.z);
    store_planes(n.hi, n.lo, o + 3, x.w * r * wv.w);
}

// ------------------------------------------------------------------ persistent form (long prompts)
// One CTA per SM walks output tiles of 256 weight rows (two 128-row MMA groups:
// gate and up rows for SwiGLU) x BN prompt rows, the tiles of one prompt-row
// block consecutively (its activation panel stays in L2 while the weights
// pass); the TMA producer runs ahead through a ring that spans tile
// boundaries.  Up to BN = 128 the accumulator is double-buffered in TMEM
// (columns 0-255 and 256-511): the epilogue warps drain tile i while the MMA
// warp runs tile i + 1.  With BN = 256 one accumulator fills the 512 columns
// and the MMAs of tile i + 1 start once the epilogue has drained tile i.
constexpr int kPtBN = 128;              // a batch of fewer rows is short: one prompt-row tile of its own size

template <bool kResid>   // the residual epilogue (o, down) as its own instance, as in k_gemm_tc
__global__ void __launch_bounds__(kTcThreads, 1)
    k_gemm_tc_pt(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                 const __grid_constant__ CUtensorMap tmB2, TcArgs a) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem =
        reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int S = a.n_stages;
    const int BN = a.BN;                          // a multiple of 16, at most 256
    constexpr int G = 2;                          // 128-row weight groups per tile (SwiGLU: gate, up)
    const uint32_t a_bytes = (uint32_t)G * 16384u, b_bytes = (uint32_t)BN * 128u;
    const uint32_t stage_bytes = a_bytes + (uint32_t)a.planes * b_bytes;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + (size_t)S * stage_bytes);
    uint64_t *empty = full + S;
    uint64_t *tfull = empty + S;                  // [2] accumulator buffer ready for the epilogue
    uint64_t *tempty = tfull + 2;                 // [2] accumulator buffer drained
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(tempty + 2);
    __shared__ int abort_s;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // 256-row weight tiles; the last may be half outside the matrix (its
    // rows read as zeros, its outputs skipped)
    const int MT = (a.n_feat * (a.epi == EPI_SWIGLU_BF16 ? 2 : 1) + 128 * G - 1) / (128 * G);
    const int NT = (a.T + BN - 1) / BN;
    const int tiles = MT * NT;
    const int KT = a.k_tiles;
    // accumulators that fit TMEM's 512 columns (2 BN columns each): two up to
    // BN = 128 (tile i's epilogue overlaps tile i + 1's MMAs), else one
    const int nbuf = 2 * G * BN <= 512 ? 2 : 1;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            ptx::mbar_init(&full[s], 1);
            ptx::mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(&tfull[b], 1);
            ptx::mbar_init(&tempty[b], 4);           // one arrival per epilogue warp
        }
        abort_s = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         ptx::smem_u32(tmem_slot)),
                     "r"(512)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    ptx::pdl_launch();

    if (warp == 0 && lane == 0) {
        // ---------------------------------------------------------- TMA producer
        int it = 0;
        bool waited = false;
        for (int t = blockIdx.x; t < tiles && !*(volatile int *)&abort_s; t += gridDim.x) {
            const int m0 = (t % MT) * 128 * G, n0 = (t / MT) * BN;
            for (int kt = 0; kt < KT; ++kt, ++it) {
                const int s = it % S;
                if (it >= S && !ptx::mbar_wait_bounded(&empty[s], ((it / S) - 1) & 1, kTcPolls)) {
                    tc_report(a.err, 14);
                    abort_s = 1;
                    break;
                }
                unsigned char *st = smem + (size_t)s * stage_bytes;
                ptx::mbar_expect_tx(&full[s], stage_bytes);
                tma_load_2d(st, &tmA, kt * kBK, m0, &full[s]);           // weights: no dependency
                if (!waited) {
                    ptx::pdl_wait();                                    // activations come from the predecessor
                    waited = true;
                }
                tma_load_2d(st + a_bytes, &tmB, kt * kBK, n0, &full[s]);
                if (a.planes == 2) tma_load_2d(st + a_bytes + b_bytes, &tmB2, kt * kBK, n0, &full[s]);
            }
        }
        // stages issued but not consumed (a wait that gave up) land before the CTA exits
        if (*(volatile int *)&abort_s)
            for (int i = it > S ? it - S : 0; i < it; ++i) ptx::mbar_wait_bounded(&full[i % S], (i / S) & 1, kTcPolls);
    } else if (warp == 1 && lane == 0) {
        // ---------------------------------------------------------- MMA issuer
        int it = 0, tl = 0;
        for (int t = blockIdx.x; t < tiles; t += gridDim.x, ++tl) {
            const int buf = tl % nbuf, use = tl / nbuf;
            if (tl >= nbuf && !ptx::mbar_wait_bounded(&tempty[buf], (use - 1) & 1, kTcPolls)) {
                tc_report(a.err, 15);
                abort_s = 1;
            }
            if (*(volatile int *)&abort_s) break;
            tc_fence_after();
            const uint32_t acc = tmem + (uint32_t)(buf * G * BN);
            for (int kt = 0; kt < KT; ++kt, ++it) {
                const int s = it % S;
                if (!ptx::mbar_wait_bounded(&full[s], (it / S) & 1, kTcPolls)) {
                    tc_report(a.err, 16);
                    abort_s = 1;
                    break;
                }
                tc_fence_after();
                const uint32_t abase = ptx::smem_u32(smem + (size_t)s * stage_bytes), bbase = abase + a_bytes;
#pragma unroll
                for (int kk = 0; kk < kBK / 16; ++kk) {
                    for (int pl = 0; pl < a.planes; ++pl) {
                        const uint64_t bdesc = sw128_desc(bbase + pl * b_bytes + kk * 32);
#pragma unroll
                        for (int g = 0; g < G; ++g)
                            mma_f16(acc + (uint32_t)(g * BN), sw128_desc(abase + g * 16384 + kk * 32), bdesc,
                                    a.idesc, (kt | kk | pl) != 0);
                    }
                }
                mma_commit(&empty[s]);                  // stage free once these MMAs have read it
            }
            if (*(volatile int *)&abort_s) break;
            mma_commit(&tfull[buf]);                    // accumulator buffer final
        }
    } else if (warp >= 2) {
        // ---------------------------------------------------------- epilogue
        ptx::pdl_wait();
        const int q = warp & 3;                         // TMEM lane quarter this warp may access
        const int r = 32 * q + lane;                    // row within a 128-row group
        int tl = 0;
        for (int t = blockIdx.x; t < tiles; t += gridDim.x, ++tl) {
            const int buf = tl % nbuf, use = tl / nbuf;
            const bool ok = ptx::mbar_wait_bounded(&tfull[buf], use & 1, kTcPolls);
            if (!ok && lane == 0) {
                tc_report(a.err, 17);
                abort_s = 1;
            }
            // warp-uniform: the TMEM loads below are warp-collective
            if (__any_sync(0xffffffffu, !ok || *(volatile int *)&abort_s)) break;
            tc_fence_after();
            const int mt = t % MT, n0 = (t / MT) * BN;
            const uint32_t tq = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(buf * G * BN);
            const bool swiglu = a.epi == EPI_SWIGLU_BF16;
            const int f = swiglu ? mt * 128 + r : mt * 128 * G + r;
            const bool two = G == 2;                     // the tile's second 128 rows in columns BN ..
            const bool pair = two && !swiglu;            // ... are rows f + 128 (SwiGLU: the up rows)
            int c = 0;
            if (kResid) {
                // 16 columns at a time (BN is a multiple of 16): the residual
                // values live next to the accumulator values
                for (; c < BN; c += 16) {
                    float v[16], u[16], x0[16], x1[16];
                    resid_load<16>(a, f, n0 + c, pair, x0, x1);
                    tmem_ld16(tq + c, v);
                    if (two) tmem_ld16(tq + BN + c, u);
                    resid_store<16>(a, f, n0 + c, pair, x0, x1, v, u);
                }
            }
            for (; c + 32 <= BN; c += 32) {
                float v[32], u[32];
                tmem_ld32(tq + c, v);
                if (two) tmem_ld32(tq + BN + c, u);
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    epi_store(a, f, n0 + c + j, v[j], two ? u[j] : 0.f);
                    if (pair) epi_store(a, f + 128, n0 + c + j, u[j], 0.f);
                }
            }
            if (c < BN) {                                // a 16-column remainder
                float v[16], u[16];
                tmem_ld16(tq + c, v);
                if (two) tmem_ld16(tq + BN + c, u);
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    epi_store(a, f, n0 + c + j, v[j], two ? u[j] : 0.f);
                    if (pair) epi_store(a, f + 128, n0 + c + j, u[j], 0.f);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&tempty[buf]);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(512) : "memory");
}

// ------------------------------------------------------------------ host side
static PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
static int g_pt_max_smem = 0;
static bool g_tc_ready = false;
static int g_max_dyn_smem = 0;

void init_gemm_tc() {
    if (g_tc_ready) return;
    cudaDriverEntryPointQueryResult q;
    void *fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess && fn) {
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        // the opt-in limit covers static and dynamic shared memory together
        int dev = 0, optin = 0;
        cudaFuncAttributes fa{};
        if (cudaGetDevice(&dev) == cudaSuccess &&
            cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) == cudaSuccess &&
            cudaFuncGetAttributes(&fa, k_gemm_tc<true>) == cudaSuccess) {
            g_max_dyn_smem = optin - (int)fa.sharedSizeBytes;
            if (cudaFuncSetAttribute(k_gemm_tc<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, g_max_dyn_smem) ==
                    cudaSuccess &&
                cudaFuncSetAttribute(k_gemm_tc<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, g_max_dyn_smem) ==
                    cudaSuccess)
                g_tc_ready = true;
            cudaFuncAttributes fp{};
            if (cudaFuncGetAttributes(&fp, k_gemm_tc_pt<true>) == cudaSuccess) {
                g_pt_max_smem = optin - (int)fp.sharedSizeBytes;
                if (cudaFuncSetAttribute(k_gemm_tc_pt<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         g_pt_max_smem) != cudaSuccess ||
                    cudaFuncSetAttribute(k_gemm_tc_pt<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         g_pt_max_smem) != cudaSuccess)
                    g_pt_max_smem = 0;
            }
        }
    }
    cudaGetLastError();
}

bool gemm_tc_ready() { return g_tc_ready; }

// Persistent form: tiles of 256 weight rows x BN prompt rows, ring stages of
// 64 K.  Long prompts take BN = 256 (128 x 256 MMAs: fewer shared-memory
// operand bytes per FLOP than 128 x 128, one accumulator in TMEM) except in
// the gate|up projection, whose SwiGLU epilogue gains more from overlapping
// the next tile's MMAs (BN = 128, two accumulators).  Run-time options, BN a
// multiple of 16 up to 256: SPEECH_DECODER_PT_BN (default 256),
// SPEECH_DECODER_PT_BN_GU (gate|up, default 128) and SPEECH_DECODER_PT_STAGES
// (ring stages at most, 3 to 6; default 6).
static int env_int(const char *name, int dflt, int lo, int hi) {
    const char *e = std::getenv(name);
    const int v = e ? std::atoi(e) : dflt;
    return v < lo ? lo : (v > hi ? hi : v);
}
struct PtShape {
    int BN, stages;
    long long tiles;
    size_t smem;
};
static PtShape pt_shape(int T, int n_feat, int epi, int planes) {
    static const int bn_pr = env_int("SPEECH_DECODER_PT_BN", 256, 16, 256) / 16 * 16;
    static const int bn_gu = env_int("SPEECH_DECODER_PT_BN_GU", 128, 16, 256) / 16 * 16;
    static const int cap = env_int("SPEECH_DECODER_PT_STAGES", 6, 3, 6);
    PtShape p{};
    const int bn = epi == EPI_SWIGLU_BF16 ? bn_gu : bn_pr;
    p.BN = T >= bn ? bn : (T + 15) / 16 * 16;
    const int stage = 2 * 16384 + planes * p.BN * 128;
    p.stages = std::min(cap, (g_pt_max_smem - 1024 - 256) / stage);
    p.tiles = (long long)((n_feat + 255) / 256) * ((T + p.BN - 1) / p.BN);
    p.smem = (size_t)p.stages * stage + 1024 + 256;
    return p;
}

static bool make_map(CUtensorMap *m, const void *ptr, uint64_t rows, uint64_t K, uint32_t box_rows, bool f16 = false) {
    const cuuint64_t dims[2] = {K, rows};
    const cuuint64_t strides[1] = {K * 2};
    const cuuint32_t box[2] = {(cuuint32_t)kBK, box_rows};
    const cuuint32_t es[2] = {1, 1};
    return g_encode(m, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                    const_cast<void *>(ptr), dims, strides, box, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

TcPlan gemm_tc_plan(int T, int n_feat, int K, int groups, int num_sms, size_t scratch_floats, int force_splits,
                    int planes) {
    TcPlan p{};
    p.ok = g_tc_ready && T >= 1 && K % kBK == 0 && n_feat % (128 * groups) == 0 && (planes == 1 || planes == 2);
    if (!p.ok) return p;
    // two activation planes: N tiles of at most 128 tokens keep three or more
    // stages; a prompt of up to 256 rows stays one N tile (the weights, the
    // bytes that bound a short prompt, are then read once)
    const int bn_max = planes == 2 && T > 256 ? 128 : 256;
    const int BN = T <= bn_max ? ((T + 15) / 16) * 16 : bn_max;
    p.BN = BN;
    const size_t stage = (size_t)groups * 16384 + (size_t)planes * BN * 128;
    const size_t budget = (size_t)g_max_dyn_smem - 1024 - 256;     // alignment pad + barriers
    p.n_stages = (int)std::min<size_t>(8, budget / stage);
    if (p.n_stages < 2) {
        p.ok = false;
        return p;
    }
    p.mt = n_feat / (128 * groups);
    p.nt = (T + BN - 1) / BN;
    p.k_tiles = K / kBK;
    const int tiles = p.mt * p.nt;
    // split K so that every SM has a CTA, in ONE wave (a second, partial wave
    // of split CTAs would leave most SMs idle for a whole CTA's time)
    int splits = 1;
    if (tiles < num_sms) splits = std::max(1, std::min(p.k_tiles / 2, num_sms / tiles));
    if (force_splits > 0) splits = std::min(force_splits, p.k_tiles);
    // the scratch for partial tiles bounds the split count
    while (splits > 1 && (size_t)tiles * splits * groups * BN * 128 > scratch_floats) --splits;
    p.kt_per_split = (p.k_tiles + splits - 1) / splits;
    p.splits = (p.k_tiles + p.kt_per_split - 1) / p.kt_per_split;
    int cols = 32;
    while (cols < groups * BN) cols *= 2;
    p.tmem_cols = cols;
    p.smem = (size_t)p.n_stages * stage + 1024 + 256;
    return p;
}

// Long prompts with 256-row weight tiles: the persistent kernel (at least one
// tile per SM, no split-K).
// Persistent kernel: at least one 256-row weight tile per SM, no split-K
// (long prompts; the vocabulary projection of a batch of rows).  SwiGLU
// needs whole 256-row gate|up blocks; otherwise the last tile may be partial.
static bool use_persistent(int T, int n_feat, int K, int groups, int epi, int planes, int num_sms,
                           int force_splits) {
    if (!g_tc_ready || g_pt_max_smem <= 0 || force_splits > 0 || K % kBK || n_feat % 128) return false;
    if (epi == EPI_SWIGLU_BF16 && (groups != 2 || n_feat % 256)) return false;
    const PtShape p = pt_shape(T, n_feat, epi, planes);
    if (p.stages < 3) return false;
    return (T >= 1024 || p.BN < kPtBN) && p.tiles >= num_sms;
}

static bool pt_disabled() {
    static int v = -1;
    if (v < 0) {
        const char *e = std::getenv("SPEECH_DECODER_GEMM_PT");
        v = e && e[0] == '0' ? 1 : 0;
    }
    return v == 1;
}

static cudaError_t launch_tc(const void *X, const void *X_lo, int T, const void *W, int n_feat, int K, int groups,
                             int epi, float *C, int ldc, void *Hout, void *Hout_lo, int ldh, float *scratch,
                             size_t scratch_floats, int *err, int num_sms, cudaStream_t s, int force_splits,
                             const float *bias, const RopeKvArgs *rope, const NormArgs *norm = nullptr,
                             bool f16 = false) {
    // f16: weights and activations both fp16 (one plane; a tcgen05 f16-kind
    // MMA takes A and B of one type), else bf16
    if (epi == EPI_BIAS_F32 && !bias) return cudaErrorInvalidValue;
    const int planes = X_lo ? 2 : 1;
    if (!pt_disabled() && use_persistent(T, n_feat, K, groups, epi, planes, num_sms, force_splits)) {
        if (rope || norm) return cudaErrorNotSupported;
        const PtShape ps = pt_shape(T, n_feat, epi, planes);
        const int BN = ps.BN;
        CUtensorMap mA, mB, mB2;
        if (!make_map(&mA, W, (uint64_t)n_feat, (uint64_t)K, 256u, f16) ||
            !make_map(&mB, X, (uint64_t)T, (uint64_t)K, (uint32_t)BN, f16) ||
            !make_map(&mB2, X_lo ? X_lo : X, (uint64_t)T, (uint64_t)K, (uint32_t)BN, f16))
            return cudaErrorInvalidValue;
        TcArgs a{};
        a.n_feat = epi == EPI_SWIGLU_BF16 ? n_feat / 2 : n_feat;
        a.T = T;
        a.K = K;
        a.groups = 2;
        a.planes = planes;
        a.BN = BN;
        a.n_stages = ps.stages;
        a.k_tiles = K / kBK;
        a.splits = 1;
        a.kt_per_split = a.k_tiles;
        a.epi = epi;
        a.C = C;
        a.ldc = ldc;
        a.Hout = static_cast<__nv_bfloat16 *>(Hout);
        a.Hout_lo = static_cast<__nv_bfloat16 *>(Hout_lo);
        a.ldh = ldh;
        a.bias = bias;
        a.err = err;
        a.idesc = mma_idesc_f16(!f16, 128, BN);
        a.out_f16 = f16;
        a.tmem_cols = 512;
        cudaLaunchConfig_t cfg{};
        cfg.gridDim = dim3((unsigned)std::min<long long>(num_sms, ps.tiles));
        cfg.blockDim = dim3(kTcThreads);
        cfg.dynamicSmemBytes = ps.smem;
        cfg.stream = s;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        const cudaError_t e = epi == EPI_RESID_F32 ? cudaLaunchKernelEx(&cfg, k_gemm_tc_pt<true>, mA, mB, mB2, a)
                                                   : cudaLaunchKernelEx(&cfg, k_gemm_tc_pt<false>, mA, mB, mB2, a);
        return e != cudaSuccess ? e : cudaPeekAtLastError();
    }
    const TcPlan p = gemm_tc_plan(T, n_feat, K, groups, num_sms, scratch_floats, force_splits, planes);
    if (!p.ok) return cudaErrorInvalidValue;
    // the folded rope needs the reduction kernel with one 128-row tile per head
    if (rope && (p.splits < 2 || groups != 1 || p.nt != 1 || rope->d != 128 || n_feat % 128)) return cudaErrorNotSupported;
    if (norm && (p.splits < 2 || groups != 1 || p.nt != 1 || epi != EPI_RESID_F32 || n_feat % 128 ||
                 n_feat > 32 * 128 || ldc % 4 || p.BN < T))
        return cudaErrorNotSupported;
    CUtensorMap mA, mB, mB2;
    if (!make_map(&mA, W, (uint64_t)n_feat, (uint64_t)K, 128u * groups, f16) ||
        !make_map(&mB, X, (uint64_t)T, (uint64_t)K, (uint32_t)p.BN, f16) ||
        !make_map(&mB2, X_lo ? X_lo : X, (uint64_t)T, (uint64_t)K, (uint32_t)p.BN, f16))
        return cudaErrorInvalidValue;
    TcArgs a{};
    a.n_feat = epi == EPI_SWIGLU_BF16 ? n_feat / 2 : n_feat;
    a.T = T;
    a.K = K;
    a.groups = groups;
    a.planes = planes;
    a.BN = p.BN;
    a.n_stages = p.n_stages;
    a.k_tiles = p.k_tiles;
    a.splits = p.splits;
    a.kt_per_split = p.kt_per_split;
    a.epi = epi;
    a.C = C;
    a.ldc = ldc;
    a.Hout = static_cast<__nv_bfloat16 *>(Hout);
    a.Hout_lo = static_cast<__nv_bfloat16 *>(Hout_lo);
    a.ldh = ldh;
    a.part = scratch;
    a.bias = bias;
    a.err = err;
    // instruction descriptor: f32 accumulate, A and B bf16 (or fp16), both K-major, N = BN, M = 128
    a.idesc = mma_idesc_f16(!f16, 128, p.BN);
    a.out_f16 = f16;
    a.tmem_cols = (uint32_t)p.tmem_cols;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(p.mt, p.nt, p.splits);
    cfg.blockDim = dim3(kTcThreads);
    cfg.dynamicSmemBytes = p.smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = epi == EPI_RESID_F32 && p.splits == 1 ? cudaLaunchKernelEx(&cfg, k_gemm_tc<true>, mA, mB, mB2, a)
                                                           : cudaLaunchKernelEx(&cfg, k_gemm_tc<false>, mA, mB, mB2, a);
    if (e == cudaSuccess && norm) {
        cfg.gridDim = dim3((unsigned)T);
        cfg.blockDim = dim3((unsigned)(32 * p.mt));
        cfg.dynamicSmemBytes = 0;
        e = cudaLaunchKernelEx(&cfg, k_splitk_resid_norm, a, *norm);
    } else if (e == cudaSuccess && p.splits > 1) {
        const long long threads = (long long)p.mt * p.nt * p.BN * 32;
        cfg.gridDim = dim3((unsigned)((threads + 255) / 256));
        cfg.blockDim = dim3(256);
        cfg.dynamicSmemBytes = 0;
        e = cudaLaunchKernelEx(&cfg, k_splitk_reduce, a, p.mt, rope ? *rope : RopeKvArgs{}, rope ? 1 : 0);
    }
    return e != cudaSuccess ? e : cudaPeekAtLastError();
}

cudaError_t launch_gemm_tc(const void *X, const void *X_lo, int T, const void *W, int n_feat, int K, int groups,
                           int epi, float *C, int ldc, void *Hout, void *Hout_lo, int ldh, float *scratch,
                           size_t scratch_floats, int *err, int num_sms, cudaStream_t s, int force_splits,
                           const float *bias, bool f16) {
    return launch_tc(X, f16 ? nullptr : X_lo, T, W, n_feat, K, groups, epi, C, ldc, Hout, f16 ? nullptr : Hout_lo, ldh,
                     scratch, scratch_floats, err, num_sms, s, force_splits, bias, nullptr, nullptr, f16);
}

cudaError_t launch_gemm_tc_resid_norm(const void *X, const void *X_lo, int T, const void *W, int n_feat, int K,
                                      float *C, int ldc, const float *norm_w, float eps, void *hi, void *lo,
                                      float *scratch, size_t scratch_floats, int *err, int num_sms, cudaStream_t s,
                                      bool f16) {
    const NormArgs n{norm_w, eps, static_cast<__nv_bfloat16 *>(hi), f16 ? nullptr : static_cast<__nv_bfloat16 *>(lo),
                     f16 ? 1 : 0};
    return launch_tc(X, f16 ? nullptr : X_lo, T, W, n_feat, K, 1, EPI_RESID_F32, C, ldc, nullptr, nullptr, 0, scratch,
                     scratch_floats, err, num_sms, s, 0, nullptr, nullptr, &n, f16);
}

cudaError_t launch_gemm_tc_qkv_rope(const void *X, const void *X_lo, int T, const void *W, int n_feat, int K,
                                    const RopeKvArgs &r, float *scratch, size_t scratch_floats, int *err, int num_sms,
                                    cudaStream_t s, bool f16) {
    return launch_tc(X, f16 ? nullptr : X_lo, T, W, n_feat, K, 1, EPI_STORE_F32, nullptr, 0, nullptr, nullptr, 0,
                     scratch, scratch_floats, err, num_sms, s, 0, nullptr, &r, nullptr, f16);
}

}  // namespace dec
