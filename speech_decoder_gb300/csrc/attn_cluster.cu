// Step attention of a few sequences as one thread-block cluster per
// (sequence, KV head): the cluster's CTAs split the keys, each scores its
// share from shared-memory tiles that TMA lands in the 128-byte-swizzled
// layout (conflict-free rows for one thread per key), and the CTAs combine
// their partial softmax sums through distributed shared memory: no global
// partials, no atomic ticket, no second kernel.
//
// Block math (qwen3_asr/decoder.cpp, build_step_graph; the decoder block of
// the page's file header): q and k RMS-normed per head, then rotated (NeoX
// RoPE) at the row's position; k and v appended at slot n_past; each query
// head h attends, with scale 1/sqrt(d), over slots [0, n_past] of KV head
// h / n_rep.
//
// One CTA of 8 warps per (split s, KV head g, sequence b); the cluster is the
// S splits of one (g, b).  Split s holds keys [s c, min(len, (s + 1) c)) with
// c = ceil(len / S) <= kCT, len = n_past + 1, so one key tile per CTA.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cmath>

#include "attn_step.cuh"
#include "tc.cuh"

namespace dec {
namespace {

constexpr int kCD = 128;               // head_dim
constexpr int kCT = 128;               // keys per CTA at most
constexpr int kCBox = 32;              // key rows per TMA box (64 dims x 32 rows, 4 KB)
constexpr int kCThreads = 256;
constexpr int kCMaxSplits = 8;         // portable cluster size
constexpr uint64_t kCWaitNs = 200000000ull;

template <int NREP>
struct ClSmem {
    // key and value tiles: [part (dims 0-63 | 64-127)][row][64 halfs], 128-byte swizzle
    __half K[2][kCT][64];
    __half V[2][kCT][64];
    float qs[NREP][kCD];               // normed, rotated queries
    float p[NREP][kCT];                // scores, then exp(score - m)
    float accp[2][NREP][kCD];          // P V of the two key halves
    // the cluster's partial results for this CTA's output slice, pushed by
    // every CTA t of the cluster: in_acc[t][j] (sum_k exp(s_k - m_t) v_k for
    // element e0 + j of the slice), in_m[t][r] / in_l[t][r] (CTA t's max score
    // and sum of exp of head r)
    float in_acc[NREP * kCD];
    float in_m[kCMaxSplits][NREP], in_l[kCMaxSplits][NREP];
    uint64_t bar;
};

// byte offset of dims [8 c, 8 c + 8) of key row `row` inside one 64-dim part
__device__ __forceinline__ uint32_t sw_off(int row, int c) {
    return (uint32_t)(row * 128 + ((c ^ (row & 7)) << 4));
}

template <int NREP>
__global__ void __launch_bounds__(kCThreads, 1)
    k_attn_cluster(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV, AttnDecArgs a,
                   float scale) {
    extern __shared__ unsigned char dsm_raw[];
    ClSmem<NREP> &sm =
        *reinterpret_cast<ClSmem<NREP> *>((reinterpret_cast<uintptr_t>(dsm_raw) + 1023) & ~uintptr_t(1023));
    constexpr int PL = kCD / 32;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int S = gridDim.x, g = blockIdx.y, b = blockIdx.z;
    const uint32_t rank = ptx::cluster_rank();
    const int s = (int)rank;
    if (tid == 0) {
        ptx::mbar_init(&sm.bar, 1);
        ptx::fence_mbar_init();
    }
    float qw[PL], kw[PL];                       // Q/K norm weights: no dependency on earlier kernels
    load_vec<PL>(a.qn_w + lane * PL, qw);
    load_vec<PL>(a.kn_w + lane * PL, kw);
    __syncthreads();
    ptx::pdl_launch();
    ptx::pdl_wait();

    // the row's raw projections, in flight with the state: warp r < NREP the
    // query of head g n_rep + r, warps NREP and NREP + 1 the key and value
    // (used by the split that owns slot n_past)
    const size_t ldq = (size_t)(a.nq + 2 * a.nkv) * kCD;
    const float *row = a.qkv + (size_t)b * ldq;
    float raw[PL];
    if (warp < NREP + 2) {
        const int hrow = warp < NREP ? g * NREP + warp : a.nq + (warp == NREP ? 0 : a.nkv) + g;
        load_vec_cg<PL>(row + (size_t)hrow * kCD + lane * PL, raw);
    }
    const int pos = a.st->n_past[b], off = a.st->kv_off[b];
    // a finished row: every CTA of the cluster sees the same state and leaves
    if (!row_live(a.st, b)) return;
    // distributed shared memory may be written only once every CTA of the
    // cluster runs: arrive now, wait just before the first push
    ptx::cluster_arrive_relaxed();
    const int len = pos + 1;
    int chunk = (len + S - 1) / S;
    if (chunk > kCT) {                                      // the launch sized S for the capacity: never
        if (tid == 0) atomicCAS(&a.st->error, 0, 12);
        chunk = kCT;
    }
    const int j0 = min(len, s * chunk), j1 = min(len, j0 + chunk), nk = j1 - j0;
    const int ncopy = max(0, min(j1, pos) - j0);            // rows from the pool (the new key excluded)
    const bool mine = pos >= j0 && pos < j1;                // this split appends the new key
    const int rr = pos - j0;
    const int y0 = g * a.slots + off + j0;
    if (tid == 0 && ncopy > 0) {
        const int nbox = (ncopy + kCBox - 1) / kCBox;
        ptx::mbar_expect_tx(&sm.bar, (uint32_t)(nbox * 4 * kCBox * 128));
        for (int i = 0; i < nbox; ++i) {
            const int y = y0 + i * kCBox;
            tma_load_2d(&sm.K[0][i * kCBox][0], &tmK, 0, y, &sm.bar);
            tma_load_2d(&sm.K[1][i * kCBox][0], &tmK, 64, y, &sm.bar);
            tma_load_2d(&sm.V[0][i * kCBox][0], &tmV, 0, y, &sm.bar);
            tma_load_2d(&sm.V[1][i * kCBox][0], &tmV, 64, y, &sm.bar);
        }
    }

    // queries (warp r: head g n_rep + r) and, in the split that owns slot pos,
    // the new key (warp NREP) and value (warp NREP + 1)
    float2 cs[PL];
    {
        const float2 *rope_row = a.rope + (size_t)pos * (kCD / 2) + (lane & 15) * PL;
#pragma unroll
        for (int e = 0; e < PL; e += 2) {
            const float4 c = *reinterpret_cast<const float4 *>(rope_row + e);
            cs[e] = make_float2(c.x, c.y);
            cs[e + 1] = make_float2(c.z, c.w);
        }
    }
    __half nh[PL];
    if (warp < NREP) {
        norm_rope_regs<PL>(raw, qw, cs, a.eps, kCD, lane);
#pragma unroll
        for (int e = 0; e < PL; ++e) sm.qs[warp][lane * PL + e] = raw[e];
    } else if (mine && warp < NREP + 2) {
        const bool is_k = warp == NREP;
        float (&v)[PL] = raw;
        if (is_k) norm_rope_regs<PL>(v, kw, cs, a.eps, kCD, lane);
        __half *pool = reinterpret_cast<__half *>(is_k ? a.Kc : a.Vc) + ((size_t)g * a.slots + off + pos) * kCD;
#pragma unroll
        for (int e = 0; e < PL; ++e) {
            nh[e] = __float2half_rn(v[e]);
            pool[lane * PL + e] = nh[e];
        }
    }
    if (ncopy > 0 && !ptx::mbar_wait_ns(&sm.bar, 0, kCWaitNs) && tid == 0) atomicCAS(&a.st->error, 0, 11);
    if (mine && (warp == NREP || warp == NREP + 1)) {
        // the new row into the landed tile: dims lane*4 .. lane*4+3
        __half (*T)[kCT][64] = warp == NREP ? sm.K : sm.V;
        const int d0 = lane * PL, part = d0 >> 6, col = d0 & 63;
        __half *dst = reinterpret_cast<__half *>(reinterpret_cast<unsigned char *>(&T[part][0][0]) +
                                                 sw_off(rr, col >> 3)) + (col & 7);
#pragma unroll
        for (int e = 0; e < PL; ++e) dst[e] = nh[e];
    }
    __syncthreads();

    // scores: thread t -> key t % kCT of head t / kCT (and + 2 for four heads)
    {
        const int kk = tid & (kCT - 1);
        for (int r = tid / kCT; r < NREP; r += kCThreads / kCT) {
            float d = 0.f, e = 0.f;                 // two FMA chains
            if (kk < nk) {
#pragma unroll
                for (int c = 0; c < kCD / 8; ++c) {
                    const uint4 kv = *reinterpret_cast<const uint4 *>(
                        reinterpret_cast<const unsigned char *>(&sm.K[c >> 3][0][0]) + sw_off(kk, c & 7));
                    float f[8];
                    unpack16(kv, f, (const __half *)nullptr);
                    const float4 q0 = *reinterpret_cast<const float4 *>(&sm.qs[r][c * 8]);
                    const float4 q1 = *reinterpret_cast<const float4 *>(&sm.qs[r][c * 8 + 4]);
                    d = fmaf(f[0], q0.x, d);
                    d = fmaf(f[1], q0.y, d);
                    d = fmaf(f[2], q0.z, d);
                    d = fmaf(f[3], q0.w, d);
                    e = fmaf(f[4], q1.x, e);
                    e = fmaf(f[5], q1.y, e);
                    e = fmaf(f[6], q1.z, e);
                    e = fmaf(f[7], q1.w, e);
                }
            }
            d += e;
            sm.p[r][kk] = kk < nk ? d * scale : -INFINITY;
        }
    }
    __syncthreads();
    ptx::cluster_wait();
    // softmax statistics of this CTA's keys: warp r owns head r
    if (warp < NREP) {
        float mx = -INFINITY;
#pragma unroll
        for (int i = 0; i < kCT / 32; ++i) mx = fmaxf(mx, sm.p[warp][lane + 32 * i]);
        mx = warp_max(mx);
        float sum = 0.f;
#pragma unroll
        for (int i = 0; i < kCT / 32; ++i) {
            const float e = mx == -INFINITY ? 0.f : expf(sm.p[warp][lane + 32 * i] - mx);
            sm.p[warp][lane + 32 * i] = e;
            sum += e;
        }
        sum = warp_sum(sum);
        // this head's statistics to every CTA of the cluster
        if (lane < S) {
            ptx::st_cluster(&sm.in_m[s][warp], (uint32_t)lane, mx);
            ptx::st_cluster(&sm.in_l[s][warp], (uint32_t)lane, sum);
        }
    }
    __syncthreads();
    // P V: thread -> (key half h, head r, dims 2 dp, 2 dp + 1)
    {
        constexpr int PER = NREP * 64;               // threads per key half
        for (int idx = tid; idx < 2 * PER; idx += kCThreads) {
            const int h = idx / PER, rem = idx % PER, r = rem >> 6, dp = rem & 63;
            const int d0 = 2 * dp, part = d0 >> 6, col = d0 & 63;
            const unsigned char *vb = reinterpret_cast<const unsigned char *>(&sm.V[part][0][0]);
            // keys h, h + 2, ...: two pairs of accumulators, four loads in flight
            float a0 = 0.f, a1 = 0.f, b0 = 0.f, b1 = 0.f;
            const unsigned char *vc = vb + (col & 7) * 2;
            int kk = h;
#pragma unroll 2
            for (; kk + 2 < nk; kk += 4) {
                const float2 v = __half22float2(*reinterpret_cast<const __half2 *>(vc + sw_off(kk, col >> 3)));
                const float2 w = __half22float2(*reinterpret_cast<const __half2 *>(vc + sw_off(kk + 2, col >> 3)));
                const float pk = sm.p[r][kk], pw = sm.p[r][kk + 2];
                a0 = fmaf(pk, v.x, a0);
                a1 = fmaf(pk, v.y, a1);
                b0 = fmaf(pw, w.x, b0);
                b1 = fmaf(pw, w.y, b1);
            }
            if (kk < nk) {
                const float2 v = __half22float2(*reinterpret_cast<const __half2 *>(vc + sw_off(kk, col >> 3)));
                const float pk = sm.p[r][kk];
                a0 = fmaf(pk, v.x, a0);
                a1 = fmaf(pk, v.y, a1);
            }
            sm.accp[h][r][d0] = a0 + b0;
            sm.accp[h][r][d0 + 1] = a1 + b1;
        }
    }
    __syncthreads();
    // CTA t normalises output elements [t E / S, (t + 1) E / S): push this
    // CTA's partial sums of each element to its owner
    constexpr int E = NREP * kCD;
    const int ES = E / S;                          // S divides E (S a power of two up to 8)
    for (int idx = tid; idx < E; idx += kCThreads) {
        const int r = idx / kCD, i = idx % kCD, t = idx / ES;
        ptx::st_cluster(&sm.in_acc[s * ES + (idx - t * ES)], (uint32_t)t, sm.accp[0][r][i] + sm.accp[1][r][i]);
    }
    // every push complete and visible; afterwards no CTA touches another's
    // shared memory, so none has to wait for its peers before leaving
    ptx::cluster_sync();
    for (int j = tid; j < ES; j += kCThreads) {
        const int idx = s * ES + j, r = idx / kCD, i = idx % kCD;
        float M = -INFINITY;
        for (int t = 0; t < S; ++t) M = fmaxf(M, sm.in_m[t][r]);
        float L = 0.f, O = 0.f;
        for (int t = 0; t < S; ++t) {
            const float mt = sm.in_m[t][r];
            const float w = mt == -INFINITY ? 0.f : expf(mt - M);
            L = fmaf(w, sm.in_l[t][r], L);
            O = fmaf(w, sm.in_acc[t * ES + j], O);
        }
        const size_t oi = (size_t)b * a.nq * kCD + (size_t)(g * NREP + r) * kCD + i;
        a.o[oi] = O / L;
        if (a.o_bf16) store_planes(a.o_bf16, a.o_bf16_lo, oi, O / L);
    }
}

PFN_cuTensorMapEncodeTiled_v12000 g_cl_encode = nullptr;
bool g_cl_ready = false;

template <int NREP>
constexpr size_t cl_smem() {
    return sizeof(ClSmem<NREP>) + 1024;
}

bool make_pool_map(CUtensorMap *m, const void *pool, int rows) {
    const cuuint64_t dims[2] = {(cuuint64_t)kCD, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)kCD * 2};
    const cuuint32_t box[2] = {64, kCBox};
    const cuuint32_t es[2] = {1, 1};
    return g_cl_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void *>(pool), dims, strides, box, es,
                       CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                       CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int NREP>
cudaError_t launch_cl(const CUtensorMap &mK, const CUtensorMap &mV, const AttnDecArgs &a, int S, float scale,
                      cudaStream_t s) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(S, a.nkv, a.B);
    cfg.blockDim = dim3(kCThreads);
    cfg.dynamicSmemBytes = cl_smem<NREP>();
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = S;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, k_attn_cluster<NREP>, mK, mV, a, scale);
}

}  // namespace

void init_attn_cluster() {
    if (g_cl_ready) return;
    cudaDriverEntryPointQueryResult q;
    void *fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn) {
        cudaGetLastError();
        return;
    }
    g_cl_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    bool ok = cudaFuncSetAttribute(k_attn_cluster<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   (int)cl_smem<1>()) == cudaSuccess;
    ok = ok && cudaFuncSetAttribute(k_attn_cluster<2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)cl_smem<2>()) == cudaSuccess;
    ok = ok && cudaFuncSetAttribute(k_attn_cluster<4>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)cl_smem<4>()) == cudaSuccess;
    cudaGetLastError();
    g_cl_ready = ok;
}

int attn_cluster_splits(int capacity, int nq, int nkv, int d, bool kv_f16, int B) {
    const int n_rep = nkv > 0 ? nq / nkv : 0;
    if (!g_cl_ready || !kv_f16 || d != kCD || B < 1 || B > kGroupB || nkv < 1 || nq % nkv ||
        (n_rep != 1 && n_rep != 2 && n_rep != 4) || capacity < 1)
        return 0;
    // the smallest cluster with at most kCT / 2 keys per CTA (scores and P V
    // are latency-bound loops over the CTA's keys), at most 8 CTAs, at least
    // enough for the whole context at kCT keys per CTA
    int S = 1;
    while (S * (kCT / 2) < capacity && S < kCMaxSplits) S *= 2;
    while (S * kCT < capacity) S *= 2;
    return S <= kCMaxSplits ? S : 0;
}

cudaError_t launch_attn_cluster(const AttnDecArgs &a, int S, cudaStream_t s) {
    const int n_rep = a.nq / a.nkv;
    if (S < 1 || S > kCMaxSplits || a.d != kCD) return cudaErrorInvalidValue;
    CUtensorMap mK, mV;
    if (!make_pool_map(&mK, a.Kc, a.nkv * a.slots) || !make_pool_map(&mV, a.Vc, a.nkv * a.slots))
        return cudaErrorInvalidValue;
    const float scale = (float)(1.0 / std::sqrt((double)kCD));
    if (n_rep == 1) return launch_cl<1>(mK, mV, a, S, scale, s);
    if (n_rep == 2) return launch_cl<2>(mK, mV, a, S, scale, s);
    if (n_rep == 4) return launch_cl<4>(mK, mV, a, S, scale, s);
    return cudaErrorInvalidValue;
}

}  // namespace dec
