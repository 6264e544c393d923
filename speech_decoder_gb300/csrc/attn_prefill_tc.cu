// Causal GQA attention of the prefill on the tensor cores (tcgen05, TMEM, TMA).
//
// One CTA per (query tile of 128 prompt rows of one sequence, query head).
// For each key tile of 128 keys up to the causal limit:
//   S = Q K^T          tcgen05.mma (fp16 in, fp32 in TMEM columns [0, 128))
//   softmax            four warps, one query row per thread: tcgen05.ld of the
//                      row, causal mask, online max / sum in fp32 (exp2 with
//                      the 1/sqrt(d) * log2(e) scale), P in fp16 written to
//                      shared memory in the 128-byte-swizzled K-major layout,
//                      the running output rescaled in TMEM (ld, scale, st)
//   O += P V           tcgen05.mma into TMEM columns [128, 256); B is V^T
//                      (rows = dims, keys contiguous), written transposed by
//                      the Q/K-norm + RoPE + KV kernel
// Warp 0 issues TMA (Q once, K and V^T double-buffered), warp 1 issues the
// MMAs and owns TMEM, warps 2-5 run the softmax and the epilogue (O / l into
// the two bf16 planes of the attention output).  The mask follows
// qwen3_asr/model.cpp, run: key c is visible to query r iff c <= r; scores
// are q.k / sqrt(d) (the page gives no scale; 1/sqrt(head_dim)).
#include <cuda.h>
#include <cudaTypedefs.h>

#include "prefill.cuh"
#include "ptx.cuh"
#include "tc.cuh"

namespace dec {

namespace {

constexpr int kD = 128;                  // head_dim of this kernel
constexpr int kBQ = 128;                 // query rows per tile (MMA M)
constexpr int kBK = 128;                 // keys per tile
constexpr int kThreads = 192;
constexpr uint32_t kAtom = 128 * 128;    // one 64-wide swizzle atom of a 128-row fp16 tile (bytes)
constexpr uint32_t kTile = 2 * kAtom;    // a 128 x 128 fp16 tile
constexpr uint64_t kWaitNs = 200000000ull;
constexpr uint32_t kTmemCols = 512;      // S of even key tiles, O, S of odd key tiles (one CTA per SM)

constexpr float kLazy = 8.f;             // log2 headroom before the running output is rescaled

struct Smem {                            // offsets into the 1024-aligned dynamic shared memory
    static constexpr uint32_t q = 0;
    static constexpr uint32_t k = q + kTile;           // [2] stages
    static constexpr uint32_t vt = k + 2 * kTile;      // [2] stages
    static constexpr uint32_t p = vt + 2 * kTile;      // [2] buffers
    static constexpr uint32_t bytes = p + 2 * kTile;
};

struct Sync {
    uint64_t q_full, kv_full[2], kv_empty[2], s_full[2], p_ready[2], pv_done[2];
    uint32_t tmem;
    int abort;
};

// 2^x on the special-function unit (max relative error about 2^-22; the
// probabilities are rounded to fp16 right after)
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ bool wait_bar(Sync &sy, uint64_t *bar, uint32_t parity, int *err, int code) {
    if (*(volatile int *)&sy.abort) return false;
    if (ptx::mbar_wait_ns(bar, parity, kWaitNs)) return true;
    *(volatile int *)&sy.abort = 1;
    if (err) atomicCAS(err, 0, code);
    return false;
}

}  // namespace

__global__ void __launch_bounds__(kThreads, 1)
    k_attn_prefill_tc(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmVt, AttnPrefillTcArgs a) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char *sm =
        reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ Sync sy;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int4 tile = a.tiles[blockIdx.y];      // (first global row, first position, rows, item)
    const int h = blockIdx.x, g = h / (a.nq / a.nkv);
    const int row0 = tile.x, pos0 = tile.y, n_rows = tile.z, item = tile.w;
    const int kv_off = a.kv_off[item], vt_col = a.vt_col[item];
    const int n_kt = (pos0 + n_rows + kBK - 1) / kBK;   // key tiles up to the causal limit

    if (threadIdx.x == 0) {
        ptx::mbar_init(&sy.q_full, 1);
        for (int s = 0; s < 2; ++s) {
            ptx::mbar_init(&sy.kv_full[s], 1);
            ptx::mbar_init(&sy.kv_empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(&sy.s_full[b], 1);
            ptx::mbar_init(&sy.p_ready[b], 128);
            ptx::mbar_init(&sy.pv_done[b], 1);
        }
        sy.abort = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 1) tmem_alloc(&sy.tmem, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // TMEM columns: S of even key tiles [0, 128), O [128, 256), S of odd tiles [256, 384)
    const uint32_t tO = sy.tmem + 128;
    auto tS = [&](int j) { return sy.tmem + ((j & 1) ? 256u : 0u); };
    const uint32_t sbase = ptx::smem_u32(sm);

    int issued = 0;                              // producer: key tiles issued (drained on abort)
    if (warp == 0 && lane == 0) {
        // ---------------------------------------------------------- TMA producer
        ptx::mbar_expect_tx(&sy.q_full, kTile);
        for (int at = 0; at < 2; ++at) tma_load_3d(sm + Smem::q + at * kAtom, &tmQ, 64 * at, h, row0, &sy.q_full);
        for (int j = 0; j < n_kt; ++j) {
            const int s = j & 1;
            if (j >= 2 && !wait_bar(sy, &sy.kv_empty[s], ((j >> 1) - 1) & 1, a.err, 21)) break;
            ptx::mbar_expect_tx(&sy.kv_full[s], 2 * kTile);
            for (int at = 0; at < 2; ++at) {
                tma_load_2d(sm + Smem::k + s * kTile + at * kAtom, &tmK, 64 * at, g * a.slots + kv_off + j * kBK,
                            &sy.kv_full[s]);
                tma_load_2d(sm + Smem::vt + s * kTile + at * kAtom, &tmVt, vt_col + j * kBK + 64 * at, g * kD,
                            &sy.kv_full[s]);
            }
            issued = j + 1;
        }
    } else if (warp == 1 && lane == 0) {
        // ---------------------------------------------------------- MMA issuer
        // S of tile j + 1 is issued before P of tile j is awaited, so the tensor
        // core computes the next scores while the softmax warps work on these
        const uint32_t idesc = mma_idesc_f16(false, kBQ, kBK);     // both MMAs are 128 x 128 (x 16)
        auto issue_s = [&](int j) -> bool {
            const int s = j & 1;
            if (!wait_bar(sy, &sy.kv_full[s], (j >> 1) & 1, a.err, 23)) return false;
            tc_fence_after();
            const uint32_t qb = sbase + Smem::q, kb = sbase + Smem::k + s * kTile;
#pragma unroll
            for (int k = 0; k < kD / 16; ++k) {
                const uint32_t off = (k >> 2) * kAtom + (k & 3) * 32;
                mma_f16(tS(j), sw128_desc(qb + off), sw128_desc(kb + off), idesc, k > 0);
            }
            mma_commit(&sy.s_full[s]);
            return true;
        };
        if (wait_bar(sy, &sy.q_full, 0, a.err, 22) && issue_s(0)) {
            for (int j = 0; j < n_kt; ++j) {
                const int s = j & 1;
                if (j + 1 < n_kt && !issue_s(j + 1)) break;
                if (!wait_bar(sy, &sy.p_ready[j & 1], (j >> 1) & 1, a.err, 24)) break;
                tc_fence_after();
                const uint32_t pb = sbase + Smem::p + (j & 1) * kTile, vb = sbase + Smem::vt + s * kTile;
#pragma unroll
                for (int k = 0; k < kBK / 16; ++k) {
                    const uint32_t off = (k >> 2) * kAtom + (k & 3) * 32;
                    mma_f16(tO, sw128_desc(pb + off), sw128_desc(vb + off), idesc, (j | k) != 0);
                }
                mma_commit(&sy.kv_empty[s]);
                mma_commit(&sy.pv_done[j & 1]);
            }
        }
    } else if (warp >= 2) {
        // ---------------------------------------------------------- softmax + epilogue
        const int quarter = warp & 3;                       // TMEM lanes this warp may access
        const int r = 32 * quarter + lane;                  // query row of the tile
        const uint32_t lane_off = (uint32_t)(32 * quarter) << 16;
        const int qpos = pos0 + r;                          // causal limit of this row
        const bool row_ok = r < n_rows;
        const float c2 = a.scale * 1.4426950408889634f;     // scores to log2 units
        // tcgen05.ld / st are warp-collective (.sync.aligned): every decision
        // that guards them is made uniform across the warp.
        // Lazy rescaling: probabilities are exp2(s - m) against a reference
        // max m that moves only when a row's scores exceed it by more than
        // kLazy (then the running output is rescaled once); otherwise P may
        // reach 2^kLazy, exact enough in fp16 and summed in fp32.  P is
        // double-buffered, so tile j + 1's softmax overlaps tile j's P . V.
        float m = -INFINITY, l = 0.f;
        bool ok = true;
        for (int j = 0; j < n_kt && ok; ++j) {
            ok = __all_sync(0xffffffffu, wait_bar(sy, &sy.s_full[j & 1], (j >> 1) & 1, a.err, 25));
            if (!ok) break;
            tc_fence_after();
            float sv[kBK];
            tmem_ld128(tS(j) + lane_off, sv);
            // raw scores; the positive scale is applied to the maximum and
            // folded into the exponent's FMA.  A tile wholly inside every
            // row's causal range (warp-uniform test) needs no mask.
            float mx = -INFINITY;
            if ((j + 1) * kBK - 1 <= pos0 + 32 * quarter && 32 * quarter + 31 < n_rows) {
#pragma unroll
                for (int c = 0; c < kBK; ++c) mx = fmaxf(mx, sv[c]);
            } else {
#pragma unroll
                for (int c = 0; c < kBK; ++c) {
                    const bool vis = row_ok && j * kBK + c <= qpos;
                    sv[c] = vis ? sv[c] : -INFINITY;
                    mx = fmaxf(mx, sv[c]);
                }
            }
            mx *= c2;
            const bool resc = __any_sync(0xffffffffu, mx > m + kLazy);
            float corr = 1.f;
            if (resc) {
                const float m_new = fmaxf(m, mx);
                corr = m == -INFINITY ? 0.f : ex2(m - m_new);
                m = m_new;
            }
            const bool none = m == -INFINITY;
            const float nm = -m;
            float ls4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int c = 0; c < kBK; ++c) {
                sv[c] = none ? 0.f : ex2(fmaf(sv[c], c2, nm));
                ls4[c & 3] += sv[c];
            }
            l = l * corr + ((ls4[0] + ls4[1]) + (ls4[2] + ls4[3]));
            // P buffer j & 1 was last read by P . V of tile j - 2
            if (j >= 2) {
                ok = __all_sync(0xffffffffu,
                                wait_bar(sy, &sy.pv_done[j & 1], ((j >> 1) - 1) & 1, a.err, 26));
                if (!ok) break;
            }
            unsigned char *prow = sm + Smem::p + (j & 1) * kTile;
#pragma unroll
            for (int c8 = 0; c8 < kBK / 8; ++c8) {
                uint32_t w[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const __half2 hp = __floats2half2_rn(sv[8 * c8 + 2 * i], sv[8 * c8 + 2 * i + 1]);
                    w[i] = *reinterpret_cast<const uint32_t *>(&hp);
                }
                const int at = c8 >> 3, ch = c8 & 7;
                *reinterpret_cast<uint4 *>(prow + at * kAtom + sw128_offset(r, ch)) = make_uint4(w[0], w[1], w[2], w[3]);
            }
            if (j > 0 && resc) {                            // rescale the running output (whole warp)
                // every earlier P . V has written O
                ok = __all_sync(0xffffffffu,
                                wait_bar(sy, &sy.pv_done[(j - 1) & 1], ((j - 1) >> 1) & 1, a.err, 28));
                if (!ok) break;
                tc_fence_after();
                float t[kD];
                tmem_ld128(tO + lane_off, t);
#pragma unroll
                for (int i = 0; i < kD; ++i) t[i] *= corr;
                tmem_st128(tO + lane_off, t);
            }
            fence_async_smem();
            tc_fence_before();
            ptx::mbar_arrive(&sy.p_ready[j & 1]);
        }
        if (ok)
            ok = __all_sync(0xffffffffu,
                            wait_bar(sy, &sy.pv_done[(n_kt - 1) & 1], ((n_kt - 1) >> 1) & 1, a.err, 27));
        tc_fence_after();
        if (ok) {                                           // whole warp loads; rows past the tile do not store
            const float inv = row_ok ? 1.f / l : 0.f;
            const size_t base = (size_t)(row0 + r) * a.nq * kD + (size_t)h * kD;
            __nv_bfloat16 *hi = a.o + base, *lo = a.o_lo ? a.o_lo + base : nullptr;
            float o[kD];
            tmem_ld128(tO + lane_off, o);
#pragma unroll
            for (int c = 0; c < kD; c += 16) {
                const float *t = o + c;
                uint32_t wh[8], wl[8];
                if (a.o_f16) {
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const __half2 hh = __floats2half2_rn(t[2 * i] * inv, t[2 * i + 1] * inv);
                        wh[i] = *reinterpret_cast<const uint32_t *>(&hh);
                    }
                    if (!row_ok) continue;
                    uint4 *dh = reinterpret_cast<uint4 *>(hi + c);
                    dh[0] = make_uint4(wh[0], wh[1], wh[2], wh[3]);
                    dh[1] = make_uint4(wh[4], wh[5], wh[6], wh[7]);
                    continue;
                }
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float v0 = t[2 * i] * inv, v1 = t[2 * i + 1] * inv;
                    const __nv_bfloat162 b = __floats2bfloat162_rn(v0, v1);
                    const __nv_bfloat162 d = __floats2bfloat162_rn(v0 - __bfloat162float(b.x),
                                                                   v1 - __bfloat162float(b.y));
                    wh[i] = *reinterpret_cast<const uint32_t *>(&b);
                    wl[i] = *reinterpret_cast<const uint32_t *>(&d);
                }
                if (!row_ok) continue;
                uint4 *dh = reinterpret_cast<uint4 *>(hi + c);
                dh[0] = make_uint4(wh[0], wh[1], wh[2], wh[3]);
                dh[1] = make_uint4(wh[4], wh[5], wh[6], wh[7]);
                if (lo) {
                    uint4 *dl = reinterpret_cast<uint4 *>(lo + c);
                    dl[0] = make_uint4(wl[0], wl[1], wl[2], wl[3]);
                    dl[1] = make_uint4(wl[4], wl[5], wl[6], wl[7]);
                }
            }
        }
    }
    // a wait that gave up: let every issued copy land before the CTA exits
    if (warp == 0 && lane == 0 && *(volatile int *)&sy.abort) {
        ptx::mbar_wait_ns(&sy.q_full, 0, kWaitNs);
        for (int j = 0; j < issued; ++j) ptx::mbar_wait_ns(&sy.kv_full[j & 1], (j >> 1) & 1, kWaitNs);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(sy.tmem, kTmemCols);
}

// ------------------------------------------------------------------ host side
static PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
static bool g_ready = false;

static bool init_encode() {
    if (g_encode) return true;
    cudaDriverEntryPointQueryResult q;
    void *fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess && fn)
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    cudaGetLastError();
    return g_encode != nullptr;
}

void init_attn_prefill_tc() {
    if (g_ready) return;
    if (!init_encode()) return;
    g_ready = cudaFuncSetAttribute(k_attn_prefill_tc, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   (int)(Smem::bytes + 1024)) == cudaSuccess;
    cudaGetLastError();
}

bool attn_prefill_tc_ok(int d, bool kv_f16) { return g_ready && d == kD && kv_f16; }

cudaError_t launch_attn_prefill_tc(const AttnPrefillTcArgs &a, int n_tiles, cudaStream_t s) {
    if (!g_ready || n_tiles <= 0) return n_tiles <= 0 ? cudaSuccess : cudaErrorInvalidValue;
    CUtensorMap mQ, mK, mVt;
    const cuuint32_t es3[3] = {1, 1, 1}, es2[2] = {1, 1};
    {   // q [rows][nq][d] fp16: box = 64 dims of one head over 128 rows
        const cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)a.nq, (cuuint64_t)a.q_rows};
        const cuuint64_t strides[2] = {(cuuint64_t)kD * 2, (cuuint64_t)a.nq * kD * 2};
        const cuuint32_t box[3] = {64, 1, kBQ};
        if (g_encode(&mQ, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void *>(a.q), dims, strides, box, es3,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    {   // K pool [nkv * slots][d] fp16
        const cuuint64_t dims[2] = {(cuuint64_t)kD, (cuuint64_t)a.nkv * a.slots};
        const cuuint64_t strides[1] = {(cuuint64_t)kD * 2};
        const cuuint32_t box[2] = {64, kBK};
        if (g_encode(&mK, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void *>(a.Kc), dims, strides, box, es2,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    {   // V^T [nkv * d][vt_ld] fp16 (keys contiguous)
        const cuuint64_t dims[2] = {(cuuint64_t)a.vt_ld, (cuuint64_t)a.nkv * kD};
        const cuuint64_t strides[1] = {(cuuint64_t)a.vt_ld * 2};
        const cuuint32_t box[2] = {64, kD};
        if (g_encode(&mVt, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void *>(a.vt), dims, strides, box, es2,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    // heads vary fastest: blocks are dispatched in index order, so every
    // head's longest query tiles (the tile list is sorted by causal length)
    // start before any head's short ones and the grid ends on short tiles
    if (n_tiles > 65535) return cudaErrorInvalidValue;
    dim3 grid(a.nq, n_tiles);
    k_attn_prefill_tc<<<grid, kThreads, Smem::bytes + 1024, s>>>(mQ, mK, mVt, a);
    return cudaPeekAtLastError();
}

}  // namespace dec
