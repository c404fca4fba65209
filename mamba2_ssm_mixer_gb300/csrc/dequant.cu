// Weight dequantisation of the W8A16 arm: each e4m3 weight code times the
// tensor's weight_scale, rounded to bf16 once when the handle is created
// (vllm.cpp PR #1289, commit "the FP8 W8A8 seam": the host arm's DenseBf16
// expands the fp8 tower into a bf16 buffer; here that happens once, on the
// device, instead of on every call).
#include "gemm.h"
#include "launch_util.h"
#include "m2_common.cuh"

namespace m2 {

// OCP FP8 E4M3: sign, 4 exponent bits (bias 7), 3 mantissa bits; exponent 0
// is subnormal (m x 2^-9); S.1111.111 is NaN; no infinities.  Every value is
// exact in f32.
__device__ __forceinline__ float e4m3_value(uint32_t c) {
  const uint32_t e = (c >> 3) & 0xFu, m = c & 7u;
  float mag;
  if (e == 0u)
    mag = (float)m * 0x1p-9f;
  else if (e == 15u && m == 7u)
    mag = __uint_as_float(0x7FC00000u);
  else
    mag = __uint_as_float(((e + 120u) << 23) | (m << 20));   // (1 + m/8) 2^(e-7)
  return (c & 0x80u) ? -mag : mag;
}

// 8 codes per thread (one 8-byte load, one 16-byte store); the tail element
// by element.
__global__ void __launch_bounds__(256) k_dequant_e4m3_bf16(const uint8_t* __restrict__ q, size_t n, float scale,
                                                           uint16_t* __restrict__ out) {
  pdl_wait();
  pdl_trigger();
  const size_t n8 = n / 8;
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += stride) {
    const uint2 v = reinterpret_cast<const uint2*>(q)[i];
    const uint32_t w[2] = {v.x, v.y};
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t c0 = (w[j >> 1] >> (16 * (j & 1))) & 0xFFu, c1 = (w[j >> 1] >> (16 * (j & 1) + 8)) & 0xFFu;
      o[j] = (uint32_t)f2bfbits(e4m3_value(c0) * scale) | ((uint32_t)f2bfbits(e4m3_value(c1) * scale) << 16);
    }
    reinterpret_cast<uint4*>(out)[i] = make_uint4(o[0], o[1], o[2], o[3]);
  }
  for (size_t i = n8 * 8 + (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride)
    out[i] = f2bfbits(e4m3_value(q[i]) * scale);
}

cudaError_t launch_dequant_e4m3_bf16(const uint8_t* q, size_t n, float scale, uint16_t* out, cudaStream_t st) {
  if (n == 0) return cudaSuccess;
  if ((uintptr_t)q % 8 || (uintptr_t)out % 16) return cudaErrorInvalidValue;
  size_t blocks = (n / 8 + 255) / 256;
  if (blocks < 1) blocks = 1;
  const size_t cap = (size_t)8 * device_sm_count();
  if (blocks > cap) blocks = cap;
  return launch_pdl(k_dequant_e4m3_bf16, dim3((unsigned)blocks), dim3(256), 0, st, q, n, scale, out);
}

}  // namespace m2
