#include "gemm_tc.cuh"

namespace dec {
bool gemm_tc_supported(int, int, int) { return false; }
void launch_gemm_tc(const void *, const void *, float *, int, int, int, int, int, cudaStream_t) {}
void init_gemm_tc() {}
}  // namespace dec
