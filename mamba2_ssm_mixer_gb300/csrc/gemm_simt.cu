// Plain CUDA-core W8A8 GEMM: y[M,N] = bf16(scale * A[M,K] . B[N,K]^T) with
// e4m3 operands and fp32 accumulation.  This is the simple, obviously-correct
// device GEMM; the tensor-core kernels are measured against it.
#include "m2_kernels.h"

namespace m2 {

namespace {
constexpr int BM = 64, BN = 64, BK = 64;
}

// 256 threads, 4x4 outputs each.  Tiles are staged in shared memory as fp32
// in k-major order so the inner loop reads broadcast-friendly rows.
__global__ void __launch_bounds__(256) k_gemm_fp8_simt(const uint8_t* __restrict__ A, const uint8_t* __restrict__ B,
                                                       uint16_t* __restrict__ y, int M, int N, int K, float scale) {
  __shared__ float As[BK][BM + 4];
  __shared__ float Bs[BK][BN + 4];
  const int tid = threadIdx.x;
  const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN;
  const int tx = tid & 15, ty = tid >> 4;
  float acc[4][4] = {};
  // loader: each thread moves 16 bytes of A and 16 of B per k-tile
  const int lr = tid >> 2;          // row within tile 0..63
  const int lk = (tid & 3) * 16;    // k offset 0,16,32,48
  for (int k0 = 0; k0 < K; k0 += BK) {
    {
      int gm = m0 + lr, gk = k0 + lk;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (gm < M && gk < K) v = *reinterpret_cast<const uint4*>(A + (size_t)gm * K + gk);
      const uint16_t* p = reinterpret_cast<const uint16_t*>(&v);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        float2 f = e4m3x2_to_f2(p[e]);
        As[lk + 2 * e][lr] = f.x;
        As[lk + 2 * e + 1][lr] = f.y;
      }
      int gn = n0 + lr;
      v = make_uint4(0, 0, 0, 0);
      if (gn < N && gk < K) v = *reinterpret_cast<const uint4*>(B + (size_t)gn * K + gk);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        float2 f = e4m3x2_to_f2(p[e]);
        Bs[lk + 2 * e][lr] = f.x;
        Bs[lk + 2 * e + 1][lr] = f.y;
      }
    }
    __syncthreads();
#pragma unroll 8
    for (int k = 0; k < BK; ++k) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[k][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = Bs[k][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    int gm = m0 + ty * 4 + i;
    if (gm >= M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      int gn = n0 + tx * 4 + j;
      if (gn < N) y[(size_t)gm * N + gn] = f2bfbits(acc[i][j] * scale);
    }
  }
}

cudaError_t launch_gemm_fp8_simt(const uint8_t* A, const uint8_t* B, uint16_t* y, int M, int N, int K, float scale,
                                 cudaStream_t st) {
  if (M == 0 || N == 0) return cudaSuccess;
  dim3 grid((N + BN - 1) / BN, (M + BM - 1) / BM);
  k_gemm_fp8_simt<<<grid, 256, 0, st>>>(A, B, y, M, N, K, scale);
  return cudaGetLastError();
}

}  // namespace m2
