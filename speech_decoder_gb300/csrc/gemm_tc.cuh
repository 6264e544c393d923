// Tensor-core (tcgen05 / TMEM / TMA) bf16 GEMM for the prefill projections.
#pragma once
#include <algorithm>

#include "common.cuh"

namespace dec {

// Epilogues of the prefill projections (shared with the CUDA-core GEMM).
enum GemmEpi { EPI_STORE_F32 = 0, EPI_RESID_F32 = 1, EPI_SWIGLU_BF16 = 2, EPI_BIAS_F32 = 3 };

struct RopeKvArgs;

struct TcPlan {
    bool ok;
    int BN, n_stages, mt, nt, k_tiles, splits, kt_per_split, tmem_cols;
    size_t smem;
};

// Y = X W^T for X [T, K] (bf16 rows of the prompt) and W [n_feat, K] (bf16
// weights); with f16 both are fp16 and X_lo / Hout_lo are unused (SwiGLU
// writes one fp16 plane).  X_lo (may be null) is a second bf16 plane of the same shape with
// X + X_lo the activation (the bf16 rounding residual): both planes enter the
// product.  epi: EPI_STORE_F32 writes C[t][f]; EPI_RESID_F32 adds into C;
// EPI_SWIGLU_BF16 (groups = 2, W packed in blocks of 128 gate rows + 128 up
// rows) writes Hout[t][f] = bf16(silu(gate) * up) for f < n_feat / 2 and, if
// Hout_lo is not null, the bf16 rounding residual into Hout_lo.  groups = 2
// with the other epilogues makes each CTA own 256 weight rows (two 128-row
// MMA tiles sharing every activation tile: half the activation traffic per
// FLOP, for long prompts); n_feat must then be a multiple of 256.
// scratch holds split-K partial tiles, summed by a second kernel in split
// order; err receives a device error code if a bounded wait expires.
TcPlan gemm_tc_plan(int T, int n_feat, int K, int groups, int num_sms, size_t scratch_floats,
                    int force_splits = 0, int planes = 1);
// EPI_BIAS_F32 writes C[t][f] = y + bias[f].
cudaError_t launch_gemm_tc(const void *X, const void *X_lo, int T, const void *W, int n_feat, int K, int groups,
                           int epi, float *C, int ldc, void *Hout, void *Hout_lo, int ldh, float *scratch,
                           size_t scratch_floats, int *err, int num_sms, cudaStream_t s, int force_splits = 0,
                           const float *bias = nullptr, bool f16 = false);
// The q|k|v projection of the prompt with the per-head Q/K RMSNorm, RoPE and
// KV write of the rope kernel folded into the split-K reduction (one warp per
// row and head: head_dim 128, fp16 KV).  Returns cudaErrorNotSupported (and
// launches nothing) where the projection would not run split-K in one
// 128-row tile per head; the caller then runs the GEMM and the rope kernel.
// A residual projection of the prompt (o, down: C += X W^T) whose split-K
// reduction also writes the RMSNorm of the finished rows for the next
// projection: hi/lo = two bf16 planes of C[t] * rsqrt(mean(C[t]^2) + eps) * w.
// cudaErrorNotSupported (nothing launched) unless it runs split-K in one
// prompt-row tile with 128-row weight tiles and n_feat <= 4096.
cudaError_t launch_gemm_tc_resid_norm(const void *X, const void *X_lo, int T, const void *W, int n_feat, int K,
                                      float *C, int ldc, const float *norm_w, float eps, void *hi, void *lo,
                                      float *scratch, size_t scratch_floats, int *err, int num_sms, cudaStream_t s,
                                      bool f16 = false);
cudaError_t launch_gemm_tc_qkv_rope(const void *X, const void *X_lo, int T, const void *W, int n_feat, int K,
                                    const RopeKvArgs &r, float *scratch, size_t scratch_floats, int *err, int num_sms,
                                    cudaStream_t s, bool f16 = false);
void init_gemm_tc();
bool gemm_tc_ready();

}  // namespace dec
