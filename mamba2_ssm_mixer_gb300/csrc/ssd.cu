// Mamba2 SSD chunked scan for prefill (Mamba2ChunkScan of vllm.cpp PR #1288,
// "What it does"): the small stages.  The recurrence
//   S_h <- exp(dt A_h) S_h + dt x_h B_g^T,   y_h = S_h C_g + D_h x_h
// is evaluated blockwise over chunks of 256 tokens (Dao & Gu 2024, SSD
// block decomposition):
//   1. dt = softplus(dt_raw + dt_bias), cum = inclusive cumsum of dt*A in chunk
//   2. chunk state  S_c = sum_t exp(cum_last - cum_t) dt_t x_t B_t^T
//   3. state pass   S_in(c+1) = exp(cum_last(c)) S_in(c) + S_c   (sequential)
//   4. chunk scan   y_t = sum_{s<=t} (C_t.B_s) exp(cum_t - cum_s) dt_s x_s
//                       + exp(cum_t) C_t S_in^T + D x_t
// Chunks never cross a sequence boundary; the last chunk of a sequence is
// partial.  Stages 2 and 4 are tensor-core kernels (ssd_tc.cu).
#include "launch_util.h"
#include "m2_kernels.h"

namespace m2 {

namespace {
struct ChunkPos {
  int seq, t0, n;   // sequence, first token (global), tokens in the chunk
};
__device__ __forceinline__ ChunkPos chunk_pos(const SeqInfo& si, int c) {
  ChunkPos cp;
  cp.seq = seq_of_chunk(si, c);
  int local = c - si.cu_chunks[cp.seq];
  cp.t0 = si.cu_seqlens[cp.seq] + local * kChunk;
  int end = si.cu_seqlens[cp.seq + 1];
  cp.n = min(kChunk, end - cp.t0);
  return cp;
}
}  // namespace

// 1. dt and the in-chunk cumulative log-decay.  One CTA (256 threads) per
// (chunk, head); thread i owns token i of the chunk.  The cumulative sum is
// formed in double and stored as an unevaluated pair of floats (hi, lo):
// within a chunk it reaches |cum| ~ 400 for fast-decaying heads, and the
// decay factors are exponentials of differences of two such sums, which a
// single float would leave with ~1e-4 relative error.
__global__ void __launch_bounds__(256) k_ssd_cumsum(const uint16_t* __restrict__ zx, const float* __restrict__ A_log,
                                                    const float* __restrict__ dt_bias, const SeqInfo si,
                                                    float* __restrict__ dt_out, float2* __restrict__ cum_out) {
  __shared__ double wsum[8];
  pdl_wait();
  pdl_trigger();
  const int c = blockIdx.x, h = blockIdx.y, i = threadIdx.x;
  const ChunkPos cp = chunk_pos(si, c);
  const float A = -expf(A_log[h]);
  float dt = 0.f;
  double a = 0.0;
  if (i < cp.n) {
    dt = softplus_f(bfbits2f(zx[(size_t)(cp.t0 + i) * kZ + kOffDt + h]) + dt_bias[h]);
    a = (double)(dt * A);
  }
  // inclusive block scan in double
  double v = a;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const double n = __shfl_up_sync(0xffffffffu, v, o);
    if ((i & 31) >= o) v += n;
  }
  if ((i & 31) == 31) wsum[i >> 5] = v;
  __syncthreads();
  double pre = 0.0;
  for (int w = 0; w < (i >> 5); ++w) pre += wsum[w];
  v += pre;
  if (i < cp.n) {
    const float hi = (float)v;
    dt_out[(size_t)(cp.t0 + i) * kNH + h] = dt;
    cum_out[(size_t)(cp.t0 + i) * kNH + h] = make_float2(hi, (float)(v - (double)hi));
  }
}

// 3. sequential state passing over the chunks of each sequence.  states[c]
// is replaced in place by the state entering chunk c; the state after the
// last chunk goes to ssm_state (read first if the sequence has initial state).
// Each thread owns 4 consecutive state entries and keeps the loads of up to 8
// chunks in flight before walking the recurrence.
__global__ void __launch_bounds__(256) k_ssd_state_pass(float* __restrict__ states, const float2* __restrict__ cum,
                                                        const SeqInfo si, float* __restrict__ ssm_state) {
  pdl_wait();
  pdl_trigger();
  const int s = blockIdx.x, h = blockIdx.y;
  const int e4 = blockIdx.z * 256 + threadIdx.x;   // float4 index inside [P, N]
  const bool init = (si.has_init[s >> 5] >> (s & 31)) & 1u;
  float4* fin = reinterpret_cast<float4*>(ssm_state + ((size_t)s * kNH + h) * (kP * kN)) + e4;
  float4 run = init ? *fin : make_float4(0.f, 0.f, 0.f, 0.f);
  const int c0 = si.cu_chunks[s], c1 = si.cu_chunks[s + 1];
  const int tbeg = si.cu_seqlens[s], tend = si.cu_seqlens[s + 1];
  for (int cb = c0; cb < c1; cb += 8) {
    float4 sc[8];
    float dec[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int c = cb + k;
      if (c < c1) {
        sc[k] = reinterpret_cast<const float4*>(states + ((size_t)c * kNH + h) * (kP * kN))[e4];
        const int tl = min(tbeg + (c - c0 + 1) * kChunk, tend) - 1;
        const float2 cl = cum[(size_t)tl * kNH + h];
        dec[k] = cl.x + cl.y;
      }
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int c = cb + k;
      if (c < c1) {
        reinterpret_cast<float4*>(states + ((size_t)c * kNH + h) * (kP * kN))[e4] = run;
        const float d = expf(dec[k]);
        run.x = fmaf(d, run.x, sc[k].x);
        run.y = fmaf(d, run.y, sc[k].y);
        run.z = fmaf(d, run.z, sc[k].z);
        run.w = fmaf(d, run.w, sc[k].w);
      }
    }
  }
  *fin = run;
}

cudaError_t launch_ssd_cumsum(const uint16_t* zx, const BlockParams& bp, const SeqInfo& si, float* dt, float2* cum,
                              cudaStream_t st) {
  return launch_pdl(k_ssd_cumsum, dim3(si.total_chunks, kNH), dim3(256), 0, st, zx, bp.A_log, bp.dt_bias, si, dt,
                    cum);
}

cudaError_t launch_ssd_state_pass(float* states, const float2* cum, const SeqInfo& si, float* ssm_state,
                                  cudaStream_t st) {
  return launch_pdl(k_ssd_state_pass, dim3(si.nseq, kNH, (kP * kN) / 4 / 256), dim3(256), 0, st, states, cum, si,
                    ssm_state);
}

}  // namespace m2
