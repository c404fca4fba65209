// Mamba2 SSD chunked scan for prefill (Mamba2ChunkScan of vllm.cpp PR #1288,
// "What it does"), CUDA-core version.  The recurrence
//   S_h <- exp(dt A_h) S_h + dt x_h B_g^T,   y_h = S_h C_g + D_h x_h
// is evaluated blockwise over chunks of 256 tokens (Dao & Gu 2024, SSD
// block decomposition):
//   1. dt = softplus(dt_raw + dt_bias), cum = inclusive cumsum of dt*A in chunk
//   2. chunk state  S_c = sum_t exp(cum_last - cum_t) dt_t x_t B_t^T
//   3. state pass   S_in(c+1) = exp(cum_last(c)) S_in(c) + S_c   (sequential)
//   4. chunk scan   y_t = sum_{s<=t} (C_t.B_s) exp(cum_t - cum_s) dt_s x_s
//                       + exp(cum_t) C_t S_in^T + D x_t
// Chunks never cross a sequence boundary; the last chunk of a sequence is
// partial.
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
// (chunk, head); thread i owns token i of the chunk.
__global__ void __launch_bounds__(256) k_ssd_cumsum(const uint16_t* __restrict__ zx, const float* __restrict__ A_log,
                                                    const float* __restrict__ dt_bias, const SeqInfo si,
                                                    float* __restrict__ dt_out, float* __restrict__ cum_out) {
  __shared__ float wsum[8];
  pdl_wait();
  pdl_trigger();
  const int c = blockIdx.x, h = blockIdx.y, i = threadIdx.x;
  const ChunkPos cp = chunk_pos(si, c);
  const float A = -expf(A_log[h]);
  float dt = 0.f, a = 0.f;
  if (i < cp.n) {
    dt = softplus_f(bfbits2f(zx[(size_t)(cp.t0 + i) * kZ + kOffDt + h]) + dt_bias[h]);
    a = dt * A;
  }
  // inclusive block scan
  float v = a;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    float n = __shfl_up_sync(0xffffffffu, v, o);
    if ((i & 31) >= o) v += n;
  }
  if ((i & 31) == 31) wsum[i >> 5] = v;
  __syncthreads();
  float pre = 0.f;
  for (int w = 0; w < (i >> 5); ++w) pre += wsum[w];
  v += pre;
  if (i < cp.n) {
    dt_out[(size_t)(cp.t0 + i) * kNH + h] = dt;
    cum_out[(size_t)(cp.t0 + i) * kNH + h] = v;
  }
}

// 2. chunk states.  One CTA per (chunk, head); thread -> (p = tid/4,
// n in [32*(tid%4), +32)).  Tokens are staged 32 at a time.
__global__ void __launch_bounds__(256) k_ssd_chunk_state(const uint16_t* __restrict__ u, const float* __restrict__ dt,
                                                         const float* __restrict__ cum, const SeqInfo si,
                                                         float* __restrict__ states) {
  __shared__ float xs[32][kP];
  __shared__ float bs[32][kN];
  const int c = blockIdx.x, h = blockIdx.y, g = h / kHPG, tid = threadIdx.x;
  const ChunkPos cp = chunk_pos(si, c);
  const float cl = cum[(size_t)(cp.t0 + cp.n - 1) * kNH + h];
  const int p = tid >> 2, nb = (tid & 3) * 32;
  float acc[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) acc[j] = 0.f;
  for (int s0 = 0; s0 < cp.n; s0 += 32) {
    // stage x (scaled by exp(cum_last - cum_s) * dt_s) and B for 32 tokens
    for (int e = tid; e < 32 * kP; e += 256) {
      int s = e / kP, pp = e % kP, t = cp.t0 + s0 + s;
      float v = 0.f;
      if (s0 + s < cp.n) {
        float w = expf(cl - cum[(size_t)t * kNH + h]) * dt[(size_t)t * kNH + h];
        v = w * bfbits2f(u[(size_t)t * kConv + h * kP + pp]);
      }
      xs[s][pp] = v;
    }
    for (int e = tid; e < 32 * kN; e += 256) {
      int s = e / kN, nn = e % kN, t = cp.t0 + s0 + s;
      bs[s][nn] = (s0 + s < cp.n) ? bfbits2f(u[(size_t)t * kConv + kOffB + g * kN + nn]) : 0.f;
    }
    __syncthreads();
#pragma unroll 4
    for (int s = 0; s < 32; ++s) {
      float xv = xs[s][p];
#pragma unroll
      for (int j = 0; j < 32; ++j) acc[j] = fmaf(xv, bs[s][nb + j], acc[j]);
    }
    __syncthreads();
  }
  float* out = states + (((size_t)c * kNH + h) * kP + p) * kN + nb;
#pragma unroll
  for (int j = 0; j < 32; j += 4) *reinterpret_cast<float4*>(out + j) = make_float4(acc[j], acc[j + 1], acc[j + 2], acc[j + 3]);
}

// 3. sequential state passing over the chunks of each sequence.  states[c]
// is replaced in place by the state entering chunk c; the state after the
// last chunk goes to ssm_state (read first if the sequence has initial state).
// Each thread owns 4 consecutive state entries and keeps the loads of up to 8
// chunks in flight before walking the recurrence.
__global__ void __launch_bounds__(256) k_ssd_state_pass(float* __restrict__ states, const float* __restrict__ cum,
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
        dec[k] = cum[(size_t)tl * kNH + h];
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

// 4. chunk scan.  One CTA per (chunk, head, 32-row tile); thread ->
// (row r = tid/8, p in [8*(tid%8), +8)).
constexpr int kRT = 32;
__global__ void __launch_bounds__(256) k_ssd_chunk_scan(const uint16_t* __restrict__ u, const float* __restrict__ dt,
                                                        const float* __restrict__ cum, const float* __restrict__ states,
                                                        const float* __restrict__ Dp, const SeqInfo si,
                                                        uint16_t* __restrict__ y) {
  __shared__ float cs[kRT][kN + 1];       // C rows of this tile
  __shared__ float sb[32][kN + 1];        // B rows of the source tile (reused for S_in)
  __shared__ float xsrc[32][kP];          // x rows of the source tile
  __shared__ float cbw[kRT][33];          // weighted C.B for (row, source)
  __shared__ float cum_r[kRT];
  const int c = blockIdx.x, h = blockIdx.y, g = h / kHPG, r0 = blockIdx.z * kRT, tid = threadIdx.x;
  const ChunkPos cp = chunk_pos(si, c);
  if (r0 >= cp.n) return;
  const int r = tid >> 3, pb = (tid & 7) * 8;
  const int rows = min(kRT, cp.n - r0);
  for (int e = tid; e < kRT * kN; e += 256) {
    int rr = e / kN, nn = e % kN;
    cs[rr][nn] = rr < rows ? bfbits2f(u[(size_t)(cp.t0 + r0 + rr) * kConv + kOffC + g * kN + nn]) : 0.f;
  }
  if (tid < kRT) cum_r[tid] = tid < rows ? cum[(size_t)(cp.t0 + r0 + tid) * kNH + h] : 0.f;
  float acc[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) acc[j] = 0.f;
  __syncthreads();

  // off-diagonal: exp(cum_t) * C_t . S_in[p, :], S_in staged 32 p-rows at a time
  const float* Sin = states + ((size_t)c * kNH + h) * (kP * kN);
  for (int pp0 = 0; pp0 < kP; pp0 += 32) {
    for (int e = tid; e < 32 * kN; e += 256) sb[e / kN][e % kN] = Sin[(size_t)(pp0 + e / kN) * kN + e % kN];
    __syncthreads();
    if (pb >= pp0 && pb < pp0 + 32) {
#pragma unroll 2
      for (int j = 0; j < 8; ++j) {
        float s = 0.f;
        for (int nn = 0; nn < kN; ++nn) s = fmaf(cs[r][nn], sb[pb - pp0 + j][nn], s);
        acc[j] = s;
      }
    }
    __syncthreads();
  }
  {
    float d = expf(cum_r[r]);
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[j] *= d;
  }

  // diagonal blocks: sources s < r0 + rows, 32 at a time
  const int send = r0 + rows;
  for (int s0 = 0; s0 < send; s0 += 32) {
    for (int e = tid; e < 32 * kN; e += 256) {
      int ss = e / kN, nn = e % kN;
      sb[ss][nn] = (s0 + ss < cp.n) ? bfbits2f(u[(size_t)(cp.t0 + s0 + ss) * kConv + kOffB + g * kN + nn]) : 0.f;
    }
    for (int e = tid; e < 32 * kP; e += 256) {
      int ss = e / kP, pp = e % kP;
      xsrc[ss][pp] = (s0 + ss < cp.n) ? bfbits2f(u[(size_t)(cp.t0 + s0 + ss) * kConv + h * kP + pp]) : 0.f;
    }
    __syncthreads();
    // weighted CB: 8 threads per row, 4 sources each; masked entries are set
    // to zero without evaluating exp (the masked exponent can overflow)
    {
      const int sj = (tid & 7) * 4;
      const int tr = r0 + r;
#pragma unroll 1
      for (int q = 0; q < 4; ++q) {
        int ss = sj + q, sg = s0 + ss;
        float w = 0.f;
        if (sg <= tr && r < rows && sg < cp.n) {
          float dot = 0.f;
          for (int nn = 0; nn < kN; ++nn) dot = fmaf(cs[r][nn], sb[ss][nn], dot);
          size_t ti = (size_t)(cp.t0 + sg) * kNH + h;
          w = dot * expf(cum_r[r] - cum[ti]) * dt[ti];
        }
        cbw[r][ss] = w;
      }
    }
    __syncthreads();
#pragma unroll 4
    for (int ss = 0; ss < 32; ++ss) {
      float w = cbw[r][ss];
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[j] = fmaf(w, xsrc[ss][pb + j], acc[j]);
    }
    __syncthreads();
  }
  if (r < rows) {
    const int t = cp.t0 + r0 + r;
    const float Dh = Dp[h];
    uint16_t ob[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      float xv = bfbits2f(u[(size_t)t * kConv + h * kP + pb + j]);
      ob[j] = f2bfbits(acc[j] + Dh * xv);
    }
    *reinterpret_cast<uint4*>(y + (size_t)t * kI + h * kP + pb) = *reinterpret_cast<uint4*>(ob);
  }
}

cudaError_t launch_ssd_cumsum(const uint16_t* zx, const BlockParams& bp, const SeqInfo& si, float* dt, float* cum,
                              cudaStream_t st) {
  return launch_pdl(k_ssd_cumsum, dim3(si.total_chunks, kNH), dim3(256), 0, st, zx, bp.A_log, bp.dt_bias, si, dt,
                    cum);
}

cudaError_t launch_ssd_chunk_state(const uint16_t* u, const float* dt, const float* cum, const SeqInfo& si,
                                   float* states, cudaStream_t st) {
  k_ssd_chunk_state<<<dim3(si.total_chunks, kNH), 256, 0, st>>>(u, dt, cum, si, states);
  return cudaGetLastError();
}

cudaError_t launch_ssd_state_pass(float* states, const float* cum, const SeqInfo& si, float* ssm_state,
                                  cudaStream_t st) {
  return launch_pdl(k_ssd_state_pass, dim3(si.nseq, kNH, (kP * kN) / 4 / 256), dim3(256), 0, st, states, cum, si,
                    ssm_state);
}

cudaError_t launch_ssd_chunk_scan(const uint16_t* u, const float* dt, const float* cum, const float* states,
                                  const BlockParams& bp, const SeqInfo& si, uint16_t* y, cudaStream_t st) {
  k_ssd_chunk_scan<<<dim3(si.total_chunks, kNH, kChunk / kRT), 256, 0, st>>>(u, dt, cum, states, bp.D, si, y);
  return cudaGetLastError();
}

}  // namespace m2
