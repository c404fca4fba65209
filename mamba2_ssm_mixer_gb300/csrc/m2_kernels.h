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

cudaError_t launch_gated_norm_quant(const uint16_t* y, const uint16_t* zx, const BlockParams& bp, int T,
                                    uint8_t* q2, uint16_t* o_tap, cudaStream_t st);
cudaError_t launch_rmsnorm_residual(uint16_t* h, const uint16_t* add, const uint16_t* w, float eps,
                                    uint16_t* normed, uint8_t* q, float s_q, int T, int n, cudaStream_t st);

// ssd.cu
// Per (chunk, head), for each token s of the chunk: the in-chunk cumulative
// log-decay cum_s as an unevaluated (hi, lo) float pair, dt_s, and the source
// factor colf_s = dt_s exp(cum_e - cum_s) with e the last token of s's
// 32-token block (<= dt_s: cum never increases); zeros past the chunk's end.
// One 4 KB record per (chunk, head), arrays of 256 (vector loads of 4
// consecutive tokens), stored [chunk][head].
struct CumDt {
  float hi[kChunk], lo[kChunk], dt[kChunk], colf[kChunk];
};
static_assert(sizeof(CumDt) == 4096, "one cum/dt record is 4 KB (one bulk copy)");
// Bytes of one (chunk, head) S_in operand image: bf16 high part and remainder
// [2][64 p][128 n] in the MMA's K-major 128-byte-swizzled layout.
constexpr int kSinImageBytes = 2 * 64 * 128 * 2;

// dt_tok (optional, may be null): dt as [T, 64] for the intermediate taps.
cudaError_t launch_ssd_cumsum(const uint16_t* zx, const BlockParams& bp, const SeqInfo& si, CumDt* cumdt,
                              float* dt_tok, cudaStream_t st);
// Reads the chunk states, writes the state entering each chunk as S_in images
// and the final state of each sequence to ssm_state.
// conv_state (may be null): also writes each sequence's new conv window
// (the last 3 raw xBC inputs of zx), after the conv has read the old one.
cudaError_t launch_ssd_state_pass(const float* states, const CumDt* cumdt, const SeqInfo& si, uint8_t* sin_img,
                                  void* ssm_state, bool bf16_state, const uint16_t* zx, uint16_t* conv_state,
                                  cudaStream_t st);

// ssd_recurrent.cu: the whole SSD stage of a prefill whose sequences all have
// at most kRecMaxT tokens, token by token (one CTA per sequence and head):
// writes y, the final states to ssm_state (read first where the sequence has
// initial state), each sequence's new conv window (conv_state may be null)
// and dt as [T, 64] (dt_tok may be null).
constexpr int kRecMaxT = 64;
cudaError_t launch_ssd_recurrent(const uint16_t* zx, const uint16_t* u, const BlockParams& bp, const SeqInfo& si,
                                 uint16_t* y, void* ssm_state, bool bf16_state, uint16_t* conv_state, float* dt_tok,
                                 cudaStream_t st);

// ssd_tc.cu (tensor-core chunk states and chunk scan)
// Chunk states f32 [chunk][head][64][128].
cudaError_t launch_ssd_chunk_state_tc(const uint16_t* u, const CumDt* cumdt, const SeqInfo& si, float* states,
                                      int* err, cudaStream_t st);
cudaError_t launch_ssd_chunk_scan_tc(const uint16_t* u, const CumDt* cumdt, const uint8_t* sin_img,
                                     const BlockParams& bp, const SeqInfo& si, uint16_t* y, int* err,
                                     cudaStream_t st);

// decode_tma.cu: the persistent, TMA-streamed decode kernel (conv window
// update, dt, state update, y, gated norm, quant).  ssm_pool: f32 rows, or
// bf16 rows when bf16_state (widened to f32 when read, rounded to bf16 when
// written back).  l2_prefetch (may be null): l2_prefetch_bytes of a buffer
// the next kernel reads (the out_proj weights), brought into L2 with an
// evict-last policy.  *launches receives the number of kernels launched.
cudaError_t launch_decode_stream(const uint16_t* zx, const BlockParams& bp, uint16_t* conv_pool, void* ssm_pool,
                                 bool bf16_state, int n_slots, const int32_t* slot_idx, int Bt, uint8_t* q2, int* err,
                                 const DecodeTaps& taps, cudaStream_t st, int* launches,
                                 const void* l2_prefetch = nullptr, size_t l2_prefetch_bytes = 0);

}  // namespace m2
