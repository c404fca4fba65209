// W8A8 GEMM dispatch: y[M,N] = bf16(scale * A[M,K] . B[N,K]^T), e4m3 operands.
#pragma once
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace m2 {
// Scratch bytes gemm_fp8 needs for this shape (split-K partials).
size_t gemm_workspace_bytes(int M, int N, int K);
// *launches receives the number of kernels launched.
// err: device error word for bounded-wait timeouts (may be null).
cudaError_t gemm_fp8(const uint8_t* A, const uint8_t* B, uint16_t* y, int M, int N, int K, float scale,
                     void* ws, size_t ws_bytes, int* err, cudaStream_t st, int* launches);

// tensor-core kernels (gemm_tc.cu)
size_t gemm_tc_skinny_workspace(int Mtok, int N, int K);
cudaError_t gemm_tc_skinny(const uint8_t* X, const uint8_t* W, uint16_t* y, int Mtok, int N, int K, float scale,
                           void* ws, size_t ws_bytes, int* err, cudaStream_t st, int* launches);
cudaError_t gemm_tc_big(const uint8_t* A, const uint8_t* B, uint16_t* y, int M, int N, int K, float scale, int* err,
                        cudaStream_t st);
constexpr int kSkinnyMaxRows = 256;
}  // namespace m2
