// Chooses the GEMM kernel for a W8A8 problem.
#include "gemm.h"
#include "m2_kernels.h"

namespace m2 {

size_t gemm_workspace_bytes(int M, int N, int K) {
  (void)M; (void)N; (void)K;
  return 0;
}

cudaError_t gemm_fp8(const uint8_t* A, const uint8_t* B, uint16_t* y, int M, int N, int K, float scale, void* ws,
                     size_t ws_bytes, cudaStream_t st, int* launches) {
  (void)ws; (void)ws_bytes;
  *launches = (M > 0) ? 1 : 0;
  return launch_gemm_fp8_simt(A, B, y, M, N, K, scale, st);
}

}  // namespace m2
