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
// carried as an unevaluated pair of floats (hi, lo) with error-free additions
// (Knuth's two-sum, folded as in double-float arithmetic), ~48 significant
// bits: within a chunk it reaches |cum| ~ 400 for fast-decaying heads, and the
// decay factors are exponentials of differences of two such sums, which a
// single float would leave with ~1e-4 relative error.  (Float pairs rather
// than double: this part's FP64 rate is a small fraction of its FP32 rate.)
namespace {
struct FF {
  float hi, lo;
};
__device__ __forceinline__ FF ff_add(FF a, FF b) {
  const float s = a.hi + b.hi;
  const float bb = s - a.hi;
  const float e = (a.hi - (s - bb)) + (b.hi - bb);   // s + e == a.hi + b.hi exactly
  const float l = e + (a.lo + b.lo);
  const float h = s + l;
  return {h, l - (h - s)};
}
}  // namespace

// Depends only on the in_proj output, so it may run beside the conv.
__global__ void __launch_bounds__(256) k_ssd_cumsum(const uint16_t* __restrict__ zx, const float* __restrict__ A_log,
                                                    const float* __restrict__ dt_bias, const SeqInfo si,
                                                    CumDt* __restrict__ cumdt, float* __restrict__ dt_tok) {
  __shared__ FF wsum[8];
  __shared__ FF cums[kChunk];
  pdl_wait();
  pdl_trigger();
  const int c = blockIdx.x, h = blockIdx.y, i = threadIdx.x;
  const ChunkPos cp = chunk_pos(si, c);
  const float A = -expf(A_log[h]);
  float dt = 0.f;
  FF v = {0.f, 0.f};
  if (i < cp.n) {
    dt = softplus_f(bfbits2f(zx[(size_t)(cp.t0 + i) * kZ + kOffDt + h]) + dt_bias[h]);
    v.hi = dt * A;
  }
  // inclusive block scan
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const FF n = {__shfl_up_sync(0xffffffffu, v.hi, o), __shfl_up_sync(0xffffffffu, v.lo, o)};
    if ((i & 31) >= o) v = ff_add(v, n);
  }
  if ((i & 31) == 31) wsum[i >> 5] = v;
  __syncthreads();
  FF pre = {0.f, 0.f};
  for (int w = 0; w < (i >> 5); ++w) pre = ff_add(pre, wsum[w]);
  v = ff_add(v, pre);
  cums[i] = v;
  __syncthreads();
  CumDt& r = cumdt[(size_t)c * kNH + h];
  float colf = 0.f;
  if (i < cp.n) {
    const FF ce = cums[min(i | 31, cp.n - 1)];            // last token of this 32-token block
    colf = dt * expf((ce.hi - v.hi) + (ce.lo - v.lo));   // exponent <= 0
    if (dt_tok) dt_tok[(size_t)(cp.t0 + i) * kNH + h] = dt;
  } else {
    v = {0.f, 0.f};
  }
  r.hi[i] = v.hi;
  r.lo[i] = v.lo;
  r.dt[i] = dt;
  r.colf[i] = colf;
}

// 3. sequential state passing over the chunks of each sequence: the state
// entering chunk c is written as the scan's S_in image (bf16 high part and
// remainder, K-major 128-byte-swizzled [64 p][128 n] each); the state after
// the last chunk goes to ssm_state (read first if the sequence has initial
// state).  Each thread owns 4 consecutive entries of one row p and keeps the
// loads of up to 8 chunks in flight before walking the recurrence.
__device__ __forceinline__ uint32_t sin_offset(int p, int n) {
  return (uint32_t)((n >> 6) * 8192 + (p >> 3) * 1024 + (p & 7) * 128 + ((((n & 63) >> 3) ^ (p & 7)) << 4) +
                    (n & 7) * 2);
}

// The initial / final state rows: f32, or bf16 (widened when read, rounded
// to nearest even when written).
__device__ __forceinline__ float4 ld_state4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ void st_state4(float* p, float4 v) { *reinterpret_cast<float4*>(p) = v; }
__device__ __forceinline__ float4 ld_state4(const uint16_t* p) {
  const uint2 w = *reinterpret_cast<const uint2*>(p);
  return make_float4(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xFFFF0000u), __uint_as_float(w.y << 16),
                     __uint_as_float(w.y & 0xFFFF0000u));
}
__device__ __forceinline__ void st_state4(uint16_t* p, float4 v) {
  *reinterpret_cast<uint2*>(p) = make_uint2(pack_bf16x2(v.x, v.y), pack_bf16x2(v.z, v.w));
}

// The blocks of slice 0 also hand each sequence's conv window over
// (CausalConv1dFwd's state output): the last 3 raw xBC inputs of [old state,
// x], oldest first, 96 channels per head index.  The conv kernel, which reads
// the old windows, has finished before this kernel starts (stream order).
template <typename SS>
__global__ void __launch_bounds__(256) k_ssd_state_pass(const float* __restrict__ states,
                                                        const CumDt* __restrict__ cumdt, const SeqInfo si,
                                                        uint8_t* __restrict__ sin_img,
                                                        SS* __restrict__ ssm_state, const uint16_t* __restrict__ zx,
                                                        uint16_t* __restrict__ conv_state) {
  pdl_wait();
  pdl_trigger();
  const int s = blockIdx.x, h = blockIdx.y;
  constexpr int kChPerHead = kConv / kNH;   // 96
  if (conv_state && blockIdx.z == 0 && threadIdx.x < kChPerHead) {
    const int ch = h * kChPerHead + threadIdx.x;
    const int T = si.cu_seqlens[s + 1] - si.cu_seqlens[s];
    const int t0 = si.cu_seqlens[s];
    const bool init = (si.has_init[s >> 5] >> (s & 31)) & 1u;
    uint16_t* st = conv_state + ((size_t)s * kConv + ch) * (kW - 1);
    uint16_t old[kW - 1], nw[kW - 1];
#pragma unroll
    for (int k = 0; k < kW - 1; ++k) old[k] = init ? st[k] : (uint16_t)0;
#pragma unroll
    for (int k = 0; k < kW - 1; ++k) {
      const int idx = T + k;   // index into [old(3), x(T)]
      nw[k] = idx < kW - 1 ? old[idx] : zx[(size_t)(t0 + idx - (kW - 1)) * kZ + kOffXBC + ch];
    }
#pragma unroll
    for (int k = 0; k < kW - 1; ++k) st[k] = nw[k];
  }
  const int e4 = blockIdx.z * 256 + threadIdx.x;   // float4 index inside [P, N]
  const int p = (e4 * 4) / kN, n = (e4 * 4) % kN;
  const uint32_t off = sin_offset(p, n);
  const bool init = (si.has_init[s >> 5] >> (s & 31)) & 1u;
  SS* fin = ssm_state + ((size_t)s * kNH + h) * (kP * kN) + 4 * (size_t)e4;
  float4 run = init ? ld_state4(fin) : make_float4(0.f, 0.f, 0.f, 0.f);
  const int c0 = si.cu_chunks[s], c1 = si.cu_chunks[s + 1];
  const int tbeg = si.cu_seqlens[s], tend = si.cu_seqlens[s + 1];
  for (int cb = c0; cb < c1; cb += 8) {
    float4 sc[8];
    float dec[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int c = cb + k;
      sc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
      dec[k] = 0.f;
      if (c < c1) {
        sc[k] = reinterpret_cast<const float4*>(states + ((size_t)c * kNH + h) * (kP * kN))[e4];
        const int nl = min(kChunk, tend - (tbeg + (c - c0) * kChunk));   // tokens in chunk c
        const CumDt& cl = cumdt[(size_t)c * kNH + h];
        dec[k] = cl.hi[nl - 1] + cl.lo[nl - 1];
      }
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int c = cb + k;
      if (c < c1) {
        uint8_t* img = sin_img + ((size_t)c * kNH + h) * kSinImageBytes;
        const float f[4] = {run.x, run.y, run.z, run.w};
        uint16_t hi[4], lo[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          hi[q] = f2bfbits(f[q]);
          lo[q] = f2bfbits(f[q] - bfbits2f(hi[q]));
        }
        *reinterpret_cast<uint2*>(img + off) = *reinterpret_cast<const uint2*>(hi);
        *reinterpret_cast<uint2*>(img + kSinImageBytes / 2 + off) = *reinterpret_cast<const uint2*>(lo);
        const float d = expf(dec[k]);
        run.x = fmaf(d, run.x, sc[k].x);
        run.y = fmaf(d, run.y, sc[k].y);
        run.z = fmaf(d, run.z, sc[k].z);
        run.w = fmaf(d, run.w, sc[k].w);
      }
    }
  }
  st_state4(fin, run);
}

cudaError_t launch_ssd_cumsum(const uint16_t* zx, const BlockParams& bp, const SeqInfo& si, CumDt* cumdt,
                              float* dt_tok, cudaStream_t st) {
  return launch_pdl(k_ssd_cumsum, dim3(si.total_chunks, kNH), dim3(256), 0, st, zx, bp.A_log, bp.dt_bias, si, cumdt,
                    dt_tok);
}

cudaError_t launch_ssd_state_pass(const float* states, const CumDt* cumdt, const SeqInfo& si, uint8_t* sin_img,
                                  void* ssm_state, bool bf16_state, const uint16_t* zx, uint16_t* conv_state,
                                  cudaStream_t st) {
  static_assert(kConv % kNH == 0, "the conv window hand-off splits the channels over the heads");
  const dim3 grid(si.nseq, kNH, (kP * kN) / 4 / 256);
  if (bf16_state)
    return launch_pdl(k_ssd_state_pass<uint16_t>, grid, dim3(256), 0, st, states, cumdt, si, sin_img,
                      static_cast<uint16_t*>(ssm_state), zx, conv_state);
  return launch_pdl(k_ssd_state_pass<float>, grid, dim3(256), 0, st, states, cumdt, si, sin_img,
                    static_cast<float*>(ssm_state), zx, conv_state);
}

}  // namespace m2
