// Chooses the GEMM kernel for a problem shape: the cluster split-K kernel
// for up to 128 activation rows (decode), the skinny split-K kernel with a
// global reduce for 129 to 256, the persistent tensor-core kernel above that
// (prefill).  Operands are e4m3 codes (W8A8) or
// bf16 values (the W8A16 arm).
#include "gemm.h"
#include "m2_kernels.h"

namespace m2 {

size_t gemm_workspace_bytes(int M, int N, int K) {
  if (M <= kFewRowMax) return 0;
  if (M <= kSkinnyMaxRows) return gemm_tc_skinny_workspace(M, N, K);
  return 0;
}

size_t gemm_workspace_bytes_bf16(int M, int N, int K) {
  if (M <= kFewRowMax) return 0;
  if (M <= kSkinnyMaxRows) return gemm_tc_skinny_workspace(M, N, 2 * K);
  return 0;
}

cudaError_t gemm_fp8(const uint8_t* A, const uint8_t* B, uint16_t* y, int M, int N, int K, float scale, void* ws,
                     size_t ws_bytes, int* err, cudaStream_t st, int* launches, bool w_static) {
  *launches = 0;
  if (M <= 0) return cudaSuccess;
  if (M <= kFewRowMax) {
    *launches = 1;
    return gemm_tc_fewrow(A, B, y, M, N, K, scale, w_static, err, st);
  }
  if (M <= kSkinnyMaxRows) return gemm_tc_skinny(A, B, y, M, N, K, scale, ws, ws_bytes, err, st, launches);
  *launches = 1;
  return gemm_tc_big(A, B, y, M, N, K, scale, w_static, err, st);
}

cudaError_t gemm_bf16(const uint16_t* A, const uint16_t* B, uint16_t* y, int M, int N, int K, float scale, void* ws,
                      size_t ws_bytes, int* err, cudaStream_t st, int* launches, bool w_static) {
  *launches = 0;
  if (M <= 0) return cudaSuccess;
  if (M <= kFewRowMax) {
    *launches = 1;
    return gemm_tc_fewrow_bf16(A, B, y, M, N, K, scale, w_static, err, st);
  }
  if (M <= kSkinnyMaxRows) return gemm_tc_skinny_bf16(A, B, y, M, N, K, scale, ws, ws_bytes, err, st, launches);
  *launches = 1;
  return gemm_tc_big_bf16(A, B, y, M, N, K, scale, w_static, err, st);
}

}  // namespace m2
