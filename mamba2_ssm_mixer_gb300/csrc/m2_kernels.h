// Host-side launchers of the block's kernels (internal to libm2).
#pragma once
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "m2_common.cuh"

namespace m2 {

struct DecodeTaps {
  uint16_t* u;     // bf16 [Bt, 6144]
  float* dt;       // f32 [Bt, 64]
  uint16_t* y;     // bf16 [Bt, 4096]
  uint16_t* o;     // bf16 [Bt, 4096]
};

struct BlockParams {
  const uint16_t* conv_w;   // bf16 [6144, 4]
  const uint16_t* conv_b;   // bf16 [6144] or null
  const float* A_log;       // [64]
  const float* D;           // [64]
  const float* dt_bias;     // [64]
  const uint16_t* norm_w;   // bf16 [4096]
  float eps, s_x, s_y;
};

// elementwise.cu
cudaError_t launch_quant_e4m3(const uint16_t* x, size_t n, float scale, uint8_t* q, cudaStream_t st);
cudaError_t launch_conv_silu_prefill(const uint16_t* zx, const BlockParams& bp, const uint16_t* conv_state,
                                     const SeqInfo& si, uint16_t* u, cudaStream_t st);
cudaError_t launch_conv_state_update(const uint16_t* zx, uint16_t* conv_state, const SeqInfo& si,
                                     cudaStream_t st);
cudaError_t launch_gated_norm_quant(const uint16_t* y, const uint16_t* zx, const BlockParams& bp, int T,
                                    uint8_t* q2, uint16_t* o_tap, cudaStream_t st);
cudaError_t launch_rmsnorm_residual(uint16_t* h, const uint16_t* add, const uint16_t* w, float eps,
                                    uint16_t* normed, int T, int n, cudaStream_t st);

// ssd.cu
// cum: the in-chunk cumulative log-decay as (hi, lo) float pairs.
cudaError_t launch_ssd_cumsum(const uint16_t* zx, const BlockParams& bp, const SeqInfo& si, float* dt, float2* cum,
                              cudaStream_t st);
cudaError_t launch_ssd_state_pass(float* states, const float2* cum, const SeqInfo& si, float* ssm_state,
                                  cudaStream_t st);

// ssd_tc.cu (tensor-core chunk states and chunk scan)
cudaError_t launch_ssd_chunk_state_tc(const uint16_t* u, const float* dt, const float2* cum, const SeqInfo& si,
                                      float* states, int* err, cudaStream_t st);
cudaError_t launch_ssd_chunk_scan_tc(const uint16_t* u, const float* dt, const float2* cum, const float* states,
                                     const BlockParams& bp, const SeqInfo& si, uint16_t* y, int* err,
                                     cudaStream_t st);

// decode_tma.cu (persistent, TMA-streamed state)
cudaError_t launch_decode_stream(const uint16_t* zx, const BlockParams& bp, uint16_t* conv_pool, float* ssm_pool,
                                 int n_slots, const int32_t* slot_idx, int Bt, uint8_t* q2, int* err,
                                 const DecodeTaps& taps, cudaStream_t st);

}  // namespace m2
