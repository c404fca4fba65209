// GEMM dispatch: y[M,N] = bf16(scale * A[M,K] . B[N,K]^T) on the tensor
// cores, operands e4m3 codes (W8A8) or bf16 values (the W8A16 arm).
#pragma once
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace m2 {
// Scratch bytes gemm_fp8 / gemm_bf16 need for this shape (split-K partials).
size_t gemm_workspace_bytes(int M, int N, int K);
size_t gemm_workspace_bytes_bf16(int M, int N, int K);
// *launches receives the number of kernels launched.
// err: device error word for bounded-wait timeouts (may be null).
// w_static: B (the weights) is never written by a kernel of the stream.
cudaError_t gemm_fp8(const uint8_t* A, const uint8_t* B, uint16_t* y, int M, int N, int K, float scale,
                     void* ws, size_t ws_bytes, int* err, cudaStream_t st, int* launches, bool w_static = false);
cudaError_t gemm_bf16(const uint16_t* A, const uint16_t* B, uint16_t* y, int M, int N, int K, float scale,
                      void* ws, size_t ws_bytes, int* err, cudaStream_t st, int* launches, bool w_static = false);

// tensor-core kernels (gemm_tc.cu); Kbytes = K x operand size
size_t gemm_tc_skinny_workspace(int Mtok, int N, int Kbytes);
cudaError_t gemm_tc_skinny(const uint8_t* X, const uint8_t* W, uint16_t* y, int Mtok, int N, int K, float scale,
                           void* ws, size_t ws_bytes, int* err, cudaStream_t st, int* launches);
cudaError_t gemm_tc_skinny_bf16(const uint16_t* X, const uint16_t* W, uint16_t* y, int Mtok, int N, int K,
                                float scale, void* ws, size_t ws_bytes, int* err, cudaStream_t st, int* launches);
// Up to kFewRowMax rows: K split across a cluster, partials added in
// distributed shared memory (no scratch).  w_static: no kernel of the stream
// writes W (so its first tiles may be fetched before the previous kernel ends).
constexpr int kFewRowMax = 128;
cudaError_t gemm_tc_fewrow(const uint8_t* X, const uint8_t* W, uint16_t* y, int Mtok, int N, int K, float scale,
                           bool w_static, int* err, cudaStream_t st);
cudaError_t gemm_tc_fewrow_bf16(const uint16_t* X, const uint16_t* W, uint16_t* y, int Mtok, int N, int K, float scale,
                                bool w_static, int* err, cudaStream_t st);
// More than 256 rows: the persistent CTA-pair kernel; w_static as above.
cudaError_t gemm_tc_big(const uint8_t* A, const uint8_t* B, uint16_t* y, int M, int N, int K, float scale,
                        bool w_static, int* err, cudaStream_t st);
cudaError_t gemm_tc_big_bf16(const uint16_t* A, const uint16_t* B, uint16_t* y, int M, int N, int K, float scale,
                             bool w_static, int* err, cudaStream_t st);
constexpr int kSkinnyMaxRows = 256;

// Failure-detection self-test: one CTA allocates TMEM, waits with the GEMMs'
// bounded mbarrier wait (limit_ns) on a barrier nothing arrives at, takes
// their abort path (error word, drain, TMEM freed) and returns.
cudaError_t launch_wait_selftest(uint64_t limit_ns, int* err, cudaStream_t st);

// W8A16 weight preparation (dequant.cu): out[i] = bf16(dec(q[i]) * scale),
// the product formed in f32 and rounded to nearest even.
cudaError_t launch_dequant_e4m3_bf16(const uint8_t* q, size_t n, float scale, uint16_t* out, cudaStream_t st);
}  // namespace m2
