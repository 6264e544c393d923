// Tensor-core (tcgen05 / TMEM / TMA) bf16 GEMM for the prefill projections.
#pragma once
#include "common.cuh"

namespace dec {

// C[M, N] (float32, row stride ldc) = or += A[M, K] . W[N, K]^T, A and W bf16.
bool gemm_tc_supported(int M, int N, int K);
void launch_gemm_tc(const void *A, const void *W, float *C, int ldc, int M, int N, int K, int epi,
                    cudaStream_t s);
void init_gemm_tc();

}  // namespace dec
