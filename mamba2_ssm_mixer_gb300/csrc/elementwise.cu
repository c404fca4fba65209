// Memory-bound kernels of the mixer block: static e4m3 activation quant,
// causal conv1d + SiLU (prefill) and its state hand-off, gated group RMSNorm
// with the out_proj quant fused into its epilogue, and the residual RMSNorm
// used between stacked blocks.
#include "m2_kernels.h"

namespace m2 {

// ---------------------------------------------------------------------------
// Static per-tensor activation quant (kQuantFp8Static of vllm.cpp PR #988,
// "The Thor finding, measured"): q = e4m3_satfinite_rne(fp32(x) / s).
// 8 bf16 in (16 B), 8 codes out (8 B) per thread; grid-stride.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) k_quant_e4m3_vec(const uint4* __restrict__ x, size_t nvec, float scale,
                                                        uint2* __restrict__ q) {
  size_t stride = (size_t)gridDim.x * blockDim.x;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < nvec; i += stride) {
    uint4 v = x[i];
    uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[2] = {0u, 0u};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint32_t lo = quant_e4m3(bfbits2f((uint16_t)(w[j] & 0xFFFFu)), scale);
      uint32_t hi = quant_e4m3(bfbits2f((uint16_t)(w[j] >> 16)), scale);
      o[j >> 1] |= (lo | (hi << 8)) << ((j & 1) * 16);
    }
    q[i] = make_uint2(o[0], o[1]);
  }
}

__global__ void k_quant_e4m3_scalar(const uint16_t* __restrict__ x, size_t begin, size_t n, float scale,
                                    uint8_t* __restrict__ q) {
  size_t stride = (size_t)gridDim.x * blockDim.x;
  for (size_t i = begin + (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride)
    q[i] = quant_e4m3(bfbits2f(x[i]), scale);
}

cudaError_t launch_quant_e4m3(const uint16_t* x, size_t n, float scale, uint8_t* q, cudaStream_t st) {
  if (n == 0) return cudaSuccess;
  bool aligned = ((uintptr_t)x % 16 == 0) && ((uintptr_t)q % 8 == 0);
  size_t nvec = aligned ? n / 8 : 0;
  if (nvec) {
    size_t blocks = (nvec + 255) / 256;
    if (blocks > 152 * 16) blocks = 152 * 16;
    k_quant_e4m3_vec<<<(unsigned)blocks, 256, 0, st>>>(reinterpret_cast<const uint4*>(x), nvec, scale,
                                                         reinterpret_cast<uint2*>(q));
  }
  size_t rest = n - nvec * 8;
  if (rest) {
    size_t blocks = (rest + 255) / 256;
    if (blocks > 152 * 16) blocks = 152 * 16;
    k_quant_e4m3_scalar<<<(unsigned)blocks, 256, 0, st>>>(x, nvec * 8, n, scale, q);
  }
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Causal depthwise conv1d (width 4) + SiLU over packed sequences
// (CausalConv1dFwd(silu) of PR #1288, "What it does").  The xBC columns are
// read in place from the in_proj row (the split is addressing).  Taps before a
// sequence's first token come from conv_state (has_initial) or are zero.
//   u[t, c] = bf16(silu(b[c] + sum_j w[c, j] * x[t - 3 + j, c]))
// One thread per (token, channel pair).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) k_conv_silu_prefill(const uint16_t* __restrict__ zx,
                                                           const uint16_t* __restrict__ conv_w,
                                                           const uint16_t* __restrict__ conv_b,
                                                           const uint16_t* __restrict__ conv_state,
                                                           const SeqInfo si, uint16_t* __restrict__ u) {
  const int t = blockIdx.y;
  const int c = (blockIdx.x * blockDim.x + threadIdx.x) * 2;
  if (c >= kConv || t >= si.total_tokens) return;
  const int s = seq_of_token(si, t);
  const int tl = t - si.cu_seqlens[s];
  const bool init = (si.has_init[s >> 5] >> (s & 31)) & 1u;
  float xv[2][kW];
#pragma unroll
  for (int j = 0; j < kW; ++j) {
    int tt = tl - (kW - 1) + j;   // local time of tap j
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      float v = 0.f;
      if (tt >= 0) {
        v = bfbits2f(zx[(size_t)(t - (kW - 1) + j) * kZ + kOffXBC + c + e]);
      } else if (init) {
        v = bfbits2f(conv_state[((size_t)s * kConv + c + e) * (kW - 1) + (kW - 1) + tt]);
      }
      xv[e][j] = v;
    }
  }
  uint32_t packed = 0;
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    float acc = conv_b ? bfbits2f(conv_b[c + e]) : 0.f;
#pragma unroll
    for (int j = 0; j < kW; ++j) acc = fmaf(bfbits2f(conv_w[(c + e) * kW + j]), xv[e][j], acc);
    packed |= (uint32_t)f2bfbits(silu_f(acc)) << (16 * e);
  }
  *reinterpret_cast<uint32_t*>(u + (size_t)t * kConv + c) = packed;
}

// New conv window of each sequence: the last 3 raw xBC inputs of
// [old state, x], oldest first.  Runs after the conv so reads of the old
// state never race with this write; one thread owns one channel's 3 taps.
__global__ void __launch_bounds__(256) k_conv_state_update(const uint16_t* __restrict__ zx,
                                                           uint16_t* __restrict__ conv_state, const SeqInfo si) {
  const int s = blockIdx.y;
  const int c = blockIdx.x * blockDim.x + threadIdx.x;
  if (c >= kConv) return;
  const int T = si.cu_seqlens[s + 1] - si.cu_seqlens[s];
  const int t0 = si.cu_seqlens[s];
  const bool init = (si.has_init[s >> 5] >> (s & 31)) & 1u;
  uint16_t* st = conv_state + ((size_t)s * kConv + c) * (kW - 1);
  uint16_t old[kW - 1];
#pragma unroll
  for (int k = 0; k < kW - 1; ++k) old[k] = init ? st[k] : (uint16_t)0;
  uint16_t nw[kW - 1];
#pragma unroll
  for (int k = 0; k < kW - 1; ++k) {
    int idx = T + k;   // index into [old(3), x(T)]
    nw[k] = idx < kW - 1 ? old[idx] : zx[(size_t)(t0 + idx - (kW - 1)) * kZ + kOffXBC + c];
  }
#pragma unroll
  for (int k = 0; k < kW - 1; ++k) st[k] = nw[k];
}

cudaError_t launch_conv_silu_prefill(const uint16_t* zx, const BlockParams& bp, const uint16_t* conv_state,
                                     const SeqInfo& si, uint16_t* u, cudaStream_t st) {
  dim3 grid((kConv / 2 + 255) / 256, si.total_tokens);
  k_conv_silu_prefill<<<grid, 256, 0, st>>>(zx, bp.conv_w, bp.conv_b, conv_state, si, u);
  return cudaGetLastError();
}

cudaError_t launch_conv_state_update(const uint16_t* zx, uint16_t* conv_state, const SeqInfo& si,
                                     cudaStream_t st) {
  dim3 grid((kConv + 255) / 256, si.nseq);
  k_conv_state_update<<<grid, 256, 0, st>>>(zx, conv_state, si);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Gated group RMSNorm (RmsNormGatedGroup(n_groups) of PR #1288) with the
// out_proj activation quant in its epilogue:
//   g = y * silu(z);  o = bf16(g / sqrt(mean_group(g^2) + eps) * w);
//   q2 = e4m3(o / s_y)
// One CTA of 128 threads per (token, group of 512 channels), 4 per thread.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float block_sum_128(float v, float* red) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float s = red[0] + red[1] + red[2] + red[3];
  return s;
}

__global__ void __launch_bounds__(128) k_gated_norm_quant(const uint16_t* __restrict__ y,
                                                          const uint16_t* __restrict__ zx,
                                                          const uint16_t* __restrict__ norm_w, float eps,
                                                          float s_y, uint8_t* __restrict__ q2,
                                                          uint16_t* __restrict__ o_tap) {
  __shared__ float red[4];
  const int t = blockIdx.x, g = blockIdx.y;
  const int c = g * kGroupCh + threadIdx.x * 4;
  uint2 yv = *reinterpret_cast<const uint2*>(y + (size_t)t * kI + c);
  uint2 zv = *reinterpret_cast<const uint2*>(zx + (size_t)t * kZ + c);
  uint2 wv = *reinterpret_cast<const uint2*>(norm_w + c);
  const uint16_t* yb = reinterpret_cast<const uint16_t*>(&yv);
  const uint16_t* zb = reinterpret_cast<const uint16_t*>(&zv);
  const uint16_t* wb = reinterpret_cast<const uint16_t*>(&wv);
  float gv[4];
  float ss = 0.f;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    gv[e] = bfbits2f(yb[e]) * silu_f(bfbits2f(zb[e]));
    ss = fmaf(gv[e], gv[e], ss);
  }
  ss = block_sum_128(ss, red);
  const float r = 1.0f / sqrtf(ss / (float)kGroupCh + eps);
  uint32_t qq = 0;
  uint16_t ob[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    ob[e] = f2bfbits(gv[e] * r * bfbits2f(wb[e]));
    qq |= (uint32_t)quant_e4m3(bfbits2f(ob[e]), s_y) << (8 * e);
  }
  *reinterpret_cast<uint32_t*>(q2 + (size_t)t * kI + c) = qq;
  if (o_tap) *reinterpret_cast<uint2*>(o_tap + (size_t)t * kI + c) = *reinterpret_cast<uint2*>(ob);
}

cudaError_t launch_gated_norm_quant(const uint16_t* y, const uint16_t* zx, const BlockParams& bp, int T,
                                    uint8_t* q2, uint16_t* o_tap, cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  dim3 grid(T, kG);
  k_gated_norm_quant<<<grid, 128, 0, st>>>(y, zx, bp.norm_w, bp.eps, bp.s_y, q2, o_tap);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Residual add + RMSNorm between stacked blocks.  One CTA per row.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) k_rmsnorm_residual(uint16_t* __restrict__ h, const uint16_t* __restrict__ add,
                                                          const uint16_t* __restrict__ w, float eps,
                                                          uint16_t* __restrict__ normed, int n) {
  __shared__ float red[8];
  const int t = blockIdx.x;
  uint16_t* hr = h + (size_t)t * n;
  const int nv = n / 8;
  float ss = 0.f;
  if (!normed) {   // residual add only
    for (int v = threadIdx.x; v < nv; v += blockDim.x) {
      uint4 hv = reinterpret_cast<uint4*>(hr)[v];
      uint16_t* hb = reinterpret_cast<uint16_t*>(&hv);
      uint4 av = reinterpret_cast<const uint4*>(add + (size_t)t * n)[v];
      const uint16_t* ab = reinterpret_cast<const uint16_t*>(&av);
#pragma unroll
      for (int e = 0; e < 8; ++e) hb[e] = f2bfbits(bfbits2f(hb[e]) + bfbits2f(ab[e]));
      reinterpret_cast<uint4*>(hr)[v] = hv;
    }
    return;
  }
  for (int v = threadIdx.x; v < nv; v += blockDim.x) {
    uint4 hv = reinterpret_cast<uint4*>(hr)[v];
    uint16_t* hb = reinterpret_cast<uint16_t*>(&hv);
    if (add) {
      uint4 av = reinterpret_cast<const uint4*>(add + (size_t)t * n)[v];
      const uint16_t* ab = reinterpret_cast<const uint16_t*>(&av);
#pragma unroll
      for (int e = 0; e < 8; ++e) hb[e] = f2bfbits(bfbits2f(hb[e]) + bfbits2f(ab[e]));
      reinterpret_cast<uint4*>(hr)[v] = hv;
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) { float f = bfbits2f(hb[e]); ss = fmaf(f, f, ss); }
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  float tot = 0.f;
  for (int i = 0; i < (int)(blockDim.x >> 5); ++i) tot += red[i];
  const float r = 1.0f / sqrtf(tot / (float)n + eps);
  for (int v = threadIdx.x; v < nv; v += blockDim.x) {
    uint4 hv = reinterpret_cast<uint4*>(hr)[v];
    uint4 wv = reinterpret_cast<const uint4*>(w)[v];
    const uint16_t* hb = reinterpret_cast<const uint16_t*>(&hv);
    const uint16_t* wb = reinterpret_cast<const uint16_t*>(&wv);
    uint4 ov;
    uint16_t* ob = reinterpret_cast<uint16_t*>(&ov);
#pragma unroll
    for (int e = 0; e < 8; ++e) ob[e] = f2bfbits(bfbits2f(hb[e]) * r * bfbits2f(wb[e]));
    reinterpret_cast<uint4*>(normed + (size_t)t * n)[v] = ov;
  }
}

cudaError_t launch_rmsnorm_residual(uint16_t* h, const uint16_t* add, const uint16_t* w, float eps,
                                    uint16_t* normed, int T, int n, cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  k_rmsnorm_residual<<<T, 256, 0, st>>>(h, add, w, eps, normed, n);
  return cudaGetLastError();
}

}  // namespace m2
