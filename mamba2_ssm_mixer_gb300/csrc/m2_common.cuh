// Shared device helpers and the compile-time geometry of the mixer block.
#pragma once
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <stdint.h>

namespace m2 {

// NemotronH Mamba2 mixer geometry.
constexpr int kH = 2688;                 // hidden
constexpr int kI = 4096;                 // d_inner
constexpr int kNH = 64;                  // heads
constexpr int kP = 64;                   // head dim
constexpr int kG = 8;                    // groups (B/C sharing and RMSNorm groups)
constexpr int kN = 128;                  // d_state
constexpr int kW = 4;                    // conv width
constexpr int kConv = kI + 2 * kG * kN;  // 6144
constexpr int kZ = kI + kConv + kNH;     // 10304: z | xBC | dt
constexpr int kHPG = kNH / kG;           // heads per group: 8
constexpr int kGroupCh = kI / kG;        // channels per norm group: 512
constexpr int kChunk = 256;              // SSD chunk length
constexpr int kMaxSeq = 256;             // sequences per prefill call

// Column offsets inside one in_proj row.
constexpr int kOffXBC = kI;              // 4096
constexpr int kOffDt = kI + kConv;       // 10240
// Column offsets inside one conv output row (x | B | C).
constexpr int kOffB = kI;                // 4096
constexpr int kOffC = kI + kG * kN;      // 5120

// Device error word bits.
constexpr int kErrSlot = 1;      // a decode row named a slot outside [0, n_slots)
constexpr int kErrTimeout = 2;   // a bounded wait ran out
constexpr int kErrDupSlot = 4;   // two decode rows of one call named the same slot

__device__ __forceinline__ float bf2f(__nv_bfloat16 v) { return __bfloat162float(v); }
__device__ __forceinline__ float bfbits2f(uint16_t b) { return __uint_as_float(((uint32_t)b) << 16); }
__device__ __forceinline__ uint16_t f2bfbits(float v) {
  __nv_bfloat16 h = __float2bfloat16_rn(v);
  return *reinterpret_cast<uint16_t*>(&h);
}
// Two floats to one bf16x2 word (round to nearest even), a in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  uint32_t d;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(b), "f"(a));
  return d;
}
// Round to bf16 and back (storage rounding between ops).
__device__ __forceinline__ float round_bf16(float v) { return bfbits2f(f2bfbits(v)); }

// e4m3 code of fp32(v / scale): IEEE division, then round-to-nearest-even
// with saturation to +-448 (NaN stays NaN).
__device__ __forceinline__ uint8_t quant_e4m3(float v, float scale) {
  float t = __fdiv_rn(v, scale);
  return (uint8_t)__nv_cvt_float_to_fp8(t, __NV_SATFINITE, __NV_E4M3);
}

// Two e4m3 codes (a in the low byte) of fp32(a / scale), fp32(b / scale).
// When inv is nonzero it is exactly 1 / scale (scale a power of two), and
// v * inv is the same correctly rounded quotient as the division.
__device__ __forceinline__ uint16_t quant2_e4m3(float a, float b, float scale, float inv) {
  float2 t;
  if (inv != 0.f) {
    t = make_float2(a * inv, b * inv);
  } else {
    t = make_float2(__fdiv_rn(a, scale), __fdiv_rn(b, scale));
  }
  return (uint16_t)__nv_cvt_float2_to_fp8x2(t, __NV_SATFINITE, __NV_E4M3);
}

__device__ __forceinline__ float silu_f(float v) { return v / (1.0f + expf(-v)); }
// SiLU with the fast exponential and division (a few float ulps; used where
// the result is rounded to bf16 next).
__device__ __forceinline__ float silu_fast(float v) { return __fdividef(v, 1.0f + __expf(-v)); }
__device__ __forceinline__ float softplus_f(float v) { return v > 20.0f ? v : log1pf(expf(v)); }

// Two e4m3 codes (low byte first) to two floats.
__device__ __forceinline__ float2 e4m3x2_to_f2(uint16_t two) {
  __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)two, __NV_E4M3);
  __half2 hh = *reinterpret_cast<__half2*>(&h);
  return __half22float2(hh);
}

// Sequence layout of one prefill call, passed by value to kernels.
struct SeqInfo {
  int nseq;
  int total_tokens;
  int total_chunks;
  int cu_seqlens[kMaxSeq + 1];   // token offsets
  int cu_chunks[kMaxSeq + 1];    // chunk offsets
  uint32_t has_init[kMaxSeq / 32];
};

// Sequence id of a chunk (binary search over cu_chunks).
__device__ __forceinline__ int seq_of_chunk(const SeqInfo& si, int c) {
  int lo = 0, hi = si.nseq - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (si.cu_chunks[mid] <= c) lo = mid; else hi = mid - 1;
  }
  return lo;
}
__device__ __forceinline__ int seq_of_token(const SeqInfo& si, int t) {
  int lo = 0, hi = si.nseq - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (si.cu_seqlens[mid] <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

}  // namespace m2

namespace m2 {
// Programmatic dependent launch: wait for the previous kernel on the stream
// (no-op when launched without the attribute) / let the next one start.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
}  // namespace m2
