// Memory-bound kernels of the mixer block: static e4m3 activation quant,
// causal conv1d + SiLU (prefill; its state hand-off runs in the SSD state
// pass, after every old window has been read), gated group RMSNorm
// with the out_proj quant fused into its epilogue, and the residual RMSNorm
// used between stacked blocks.
#include "launch_util.h"
#include "m2_kernels.h"

namespace m2 {

// ---------------------------------------------------------------------------
// Static per-tensor activation quant (kQuantFp8Static of vllm.cpp PR #988,
// "The Thor finding, measured"): q = e4m3_satfinite_rne(fp32(x) / s).
// 8 bf16 in (16 B), 8 codes out (8 B) per vector; grid-stride, two
// independent vectors in flight per thread.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint2 quant8_e4m3(uint4 v, float scale, float inv) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t o[2] = {0u, 0u};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t two = quant2_e4m3(__uint_as_float(w[j] << 16), __uint_as_float(w[j] & 0xFFFF0000u), scale, inv);
    o[j >> 1] |= two << ((j & 1) * 16);
  }
  return make_uint2(o[0], o[1]);
}

__global__ void __launch_bounds__(256) k_quant_e4m3_vec(const uint4* __restrict__ x, size_t nvec, float scale,
                                                        float inv, uint2* __restrict__ q) {
  pdl_wait();
  pdl_trigger();
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < nvec; i += 2 * stride) {
    const bool two = i + stride < nvec;
    const uint4 a = x[i];
    const uint4 b = two ? x[i + stride] : make_uint4(0, 0, 0, 0);
    q[i] = quant8_e4m3(a, scale, inv);
    if (two) q[i + stride] = quant8_e4m3(b, scale, inv);
  }
}

__global__ void k_quant_e4m3_scalar(const uint16_t* __restrict__ x, size_t begin, size_t n, float scale,
                                    uint8_t* __restrict__ q) {
  pdl_wait();
  pdl_trigger();
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
    cudaError_t e = launch_pdl(k_quant_e4m3_vec, dim3((unsigned)blocks), dim3(256), 0, st,
                               reinterpret_cast<const uint4*>(x), nvec, scale, exact_inverse(scale),
                               reinterpret_cast<uint2*>(q));
    if (e != cudaSuccess) return e;
  }
  size_t rest = n - nvec * 8;
  if (rest) {
    size_t blocks = (rest + 255) / 256;
    if (blocks > 152 * 16) blocks = 152 * 16;
    cudaError_t e = launch_pdl(k_quant_e4m3_scalar, dim3((unsigned)blocks), dim3(256), 0, st, x, nvec * 8, n, scale, q);
    if (e != cudaSuccess) return e;
  }
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Causal depthwise conv1d (width 4) + SiLU over packed sequences
// (CausalConv1dFwd(silu) of PR #1288, "What it does").  The xBC columns are
// read in place from the in_proj row (the split is addressing).  Taps before a
// sequence's first token come from conv_state (has_initial) or are zero.
//   u[t, c] = bf16(silu(b[c] + sum_j w[c, j] * x[t - 3 + j, c]))
// One CTA per tile of 64 tokens x 256 channels: the tile's rows plus the 3
// rows before it are staged in shared memory with 16-byte asynchronous copies
// (all of them in flight at once), then each thread runs one channel pair
// over 32 consecutive tokens with the 3 previous inputs in registers (a
// sliding window reset at sequence starts).
// ---------------------------------------------------------------------------
constexpr int kCvT = 64;                 // tokens per tile
constexpr int kCvC = 256;                // channels per tile
constexpr int kCvRows = kCvT + kW - 1;   // staged rows: 3 before the tile + the tile

__device__ __forceinline__ void cp_async16(void* dst_smem, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                   (uint32_t)__cvta_generic_to_shared(dst_smem)),
               "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

__device__ __forceinline__ float2 bf2_to_f2(uint32_t v) {
  return make_float2(bfbits2f((uint16_t)(v & 0xFFFFu)), bfbits2f((uint16_t)(v >> 16)));
}

// Packed pairs of floats (f32x2 arithmetic of the sm_100 family), element 0
// in the low word: the conv runs a channel pair per thread.
__device__ __forceinline__ uint64_t f2pk(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ uint64_t bf2pk(uint32_t v) {   // bf16 pair -> f32 pair
  return f2pk(__uint_as_float(v << 16), __uint_as_float(v & 0xFFFF0000u));
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ uint64_t mul2f(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t add2f(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
// silu(v) = v / (1 + 2^(-v log2 e)) for a pair, with the hardware's
// approximate base-2 exponential and reciprocal (relative error ~1e-7; the
// result is rounded to bf16 next), packed to a bf16 pair.
__device__ __forceinline__ uint32_t silu2_bf16(uint64_t v) {
  const uint64_t m = mul2f(v, f2pk(-1.4426950408889634f, -1.4426950408889634f));   // -log2(e)
  float m0, m1;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(m0), "=f"(m1) : "l"(m));
  float e0, e1;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e0) : "f"(m0));
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e1) : "f"(m1));
  const uint64_t d = add2f(f2pk(e0, e1), f2pk(1.f, 1.f));
  float d0, d1;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(d0), "=f"(d1) : "l"(d));
  float r0, r1;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r0) : "f"(d0));
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r1) : "f"(d1));
  const uint64_t s = mul2f(v, f2pk(r0, r1));
  float s0, s1;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(s0), "=f"(s1) : "l"(s));
  return pack_bf16x2(s0, s1);
}

// (at most 40 registers: six CTAs per SM, 3.4 waves of the 4 x 2048 prefill
// instead of 4.04 with five)
__global__ void __launch_bounds__(256, 6) k_conv_silu_prefill(const uint16_t* __restrict__ zx,
                                                           const uint16_t* __restrict__ conv_w,
                                                           const uint16_t* __restrict__ conv_b,
                                                           const uint16_t* __restrict__ conv_state,
                                                           const SeqInfo si, uint16_t* __restrict__ u) {
  __shared__ __align__(16) uint16_t tile[kCvRows][kCvC];   // 33.5 KB
  pdl_wait();
  pdl_trigger();
  const int c0 = blockIdx.x * kCvC, t0 = blockIdx.y * kCvT, T = si.total_tokens;
  // rows t0 - 3 .. t0 + 63 (rows outside [0, T) are never read: zero them)
  for (int i = threadIdx.x; i < kCvRows * (kCvC / 8); i += blockDim.x) {
    const int r = i / (kCvC / 8), q = i % (kCvC / 8);
    const int t = t0 - (kW - 1) + r;
    if (t >= 0 && t < T)
      cp_async16(&tile[r][q * 8], zx + (size_t)t * kZ + kOffXBC + c0 + q * 8);
    else
      *reinterpret_cast<uint4*>(&tile[r][q * 8]) = make_uint4(0, 0, 0, 0);
  }
  cp_async_wait_all();
  __syncthreads();

  const int pr = threadIdx.x & (kCvC / 2 - 1), half = threadIdx.x / (kCvC / 2);
  const int c = c0 + 2 * pr;
  const int t_begin = t0 + half * (kCvT / 2);
  if (t_begin >= T) return;
  const int t_end = min(t_begin + kCvT / 2, T);
  // weights and bias of the channel pair, packed per tap
  uint64_t w[kW];
#pragma unroll
  for (int j = 0; j < kW; ++j) w[j] = f2pk(bfbits2f(conv_w[c * kW + j]), bfbits2f(conv_w[(c + 1) * kW + j]));
  const uint64_t bias = conv_b ? f2pk(bfbits2f(conv_b[c]), bfbits2f(conv_b[c + 1])) : f2pk(0.f, 0.f);
  // staged input pair of token t (t0 - 3 <= t < t0 + 64)
  auto row = [&](int t) { return bf2pk(*reinterpret_cast<const uint32_t*>(&tile[t - t0 + kW - 1][2 * pr])); };
  int s = seq_of_token(si, t_begin);
  int seq_start = si.cu_seqlens[s], seq_end = si.cu_seqlens[s + 1];
  // window[k] = input at time t - 3 + k (k = 0, 1, 2) for the next token t
  uint64_t win[kW - 1];
  auto load_window = [&](int t) {
    const bool init = (si.has_init[s >> 5] >> (s & 31)) & 1u;
#pragma unroll
    for (int k = 0; k < kW - 1; ++k) {
      const int tt = t - (kW - 1) + k;
      if (tt >= seq_start) {
        win[k] = row(tt);
      } else if (init) {
        const int tap = (kW - 1) + (tt - seq_start);   // 0..2
        const uint16_t* st = conv_state + ((size_t)s * kConv + c) * (kW - 1);
        win[k] = f2pk(bfbits2f(st[tap]), bfbits2f(st[(kW - 1) + tap]));
      } else {
        win[k] = f2pk(0.f, 0.f);
      }
    }
  };
  load_window(t_begin);
  uint32_t* urow = reinterpret_cast<uint32_t*>(u + (size_t)t_begin * kConv + c);
  int t = t_begin;
  while (t < t_end) {
    if (t == seq_end) {   // first token of the next sequence
      ++s;
      seq_start = seq_end;
      seq_end = si.cu_seqlens[s + 1];
      load_window(t);
    }
    // tokens of one sequence: no boundary test inside
    const int seg_end = min(t_end, seq_end);
#pragma unroll 4
    for (; t < seg_end; ++t) {
      const uint64_t x = row(t);
      const uint64_t acc = fma2(w[3], x, fma2(w[2], win[2], fma2(w[1], win[1], fma2(w[0], win[0], bias))));
      *urow = silu2_bf16(acc);
      urow += kConv / 2;
      win[0] = win[1];
      win[1] = win[2];
      win[2] = x;
    }
  }
}

cudaError_t launch_conv_silu_prefill(const uint16_t* zx, const BlockParams& bp, const uint16_t* conv_state,
                                     const SeqInfo& si, uint16_t* u, cudaStream_t st) {
  static_assert(kConv % kCvC == 0, "conv tiles cover the channels exactly");
  dim3 grid(kConv / kCvC, (si.total_tokens + kCvT - 1) / kCvT);
  return launch_pdl(k_conv_silu_prefill, grid, dim3(kCvC), 0, st, zx, bp.conv_w, bp.conv_b, conv_state, si, u);
}

// ---------------------------------------------------------------------------
// Gated group RMSNorm (RmsNormGatedGroup(n_groups) of PR #1288) with the
// out_proj activation quant in its epilogue:
//   g = y * silu(z);  o = bf16(g / sqrt(mean_group(g^2) + eps) * w);
//   q2 = e4m3(o / s_y)
// One CTA of 8 warps per token; warp g owns group g (512 channels, 16 per
// lane), so the group reduction is a warp shuffle.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) k_gated_norm_quant(const uint16_t* __restrict__ y,
                                                          const uint16_t* __restrict__ zx,
                                                          const uint16_t* __restrict__ norm_w, float eps,
                                                          float s_y, float inv_y, uint8_t* __restrict__ q2,
                                                          uint16_t* __restrict__ o_tap) {
  pdl_wait();
  pdl_trigger();
  const int t = blockIdx.x, g = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = g * kGroupCh + lane * 16;
  const uint4* yp = reinterpret_cast<const uint4*>(y + (size_t)t * kI + c);
  const uint4* zp = reinterpret_cast<const uint4*>(zx + (size_t)t * kZ + c);
  const uint4* wp = reinterpret_cast<const uint4*>(norm_w + c);
  uint4 yv[2] = {yp[0], yp[1]}, zv[2] = {zp[0], zp[1]}, wv[2] = {wp[0], wp[1]};
  const uint16_t* yb = reinterpret_cast<const uint16_t*>(yv);
  const uint16_t* zb = reinterpret_cast<const uint16_t*>(zv);
  const uint16_t* wb = reinterpret_cast<const uint16_t*>(wv);
  float gv[16];
  float ss = 0.f;
#pragma unroll
  for (int e = 0; e < 16; ++e) {
    gv[e] = bfbits2f(yb[e]) * silu_fast(bfbits2f(zb[e]));
    ss = fmaf(gv[e], gv[e], ss);
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  const float r = 1.0f / sqrtf(ss / (float)kGroupCh + eps);
  uint32_t qq[4] = {0u, 0u, 0u, 0u};
  uint16_t ob[16];
#pragma unroll
  for (int e = 0; e < 16; ++e) ob[e] = f2bfbits(gv[e] * r * bfbits2f(wb[e]));
#pragma unroll
  for (int e = 0; e < 16; e += 2)
    qq[e >> 2] |= (uint32_t)quant2_e4m3(bfbits2f(ob[e]), bfbits2f(ob[e + 1]), s_y, inv_y) << (8 * (e & 3));
  *reinterpret_cast<uint4*>(q2 + (size_t)t * kI + c) = make_uint4(qq[0], qq[1], qq[2], qq[3]);
  if (o_tap) {
    uint4* op = reinterpret_cast<uint4*>(o_tap + (size_t)t * kI + c);
    op[0] = reinterpret_cast<const uint4*>(ob)[0];
    op[1] = reinterpret_cast<const uint4*>(ob)[1];
  }
}

cudaError_t launch_gated_norm_quant(const uint16_t* y, const uint16_t* zx, const BlockParams& bp, int T,
                                    uint8_t* q2, uint16_t* o_tap, cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  return launch_pdl(k_gated_norm_quant, dim3(T), dim3(256), 0, st, y, zx, bp.norm_w, bp.eps, bp.s_y,
                    exact_inverse(bp.s_y), q2, o_tap);
}

// ---------------------------------------------------------------------------
// Residual add + RMSNorm between stacked blocks, optionally with the next
// block's static e4m3 activation quant of the normed row (the same bf16
// normed value, then the same code as fp8_quant).  One CTA per row.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) k_rmsnorm_residual(uint16_t* __restrict__ h, const uint16_t* __restrict__ add,
                                                          const uint16_t* __restrict__ w, float eps,
                                                          uint16_t* __restrict__ normed, uint8_t* __restrict__ q,
                                                          float s_q, float inv_q, int n) {
  __shared__ float red[8];
  pdl_wait();
  pdl_trigger();
  const int t = blockIdx.x;
  uint16_t* hr = h + (size_t)t * n;
  const int nv = n / 8;
  float ss = 0.f;
  if (!normed && !q) {   // residual add only
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
    if (normed) reinterpret_cast<uint4*>(normed + (size_t)t * n)[v] = ov;
    if (q) {
      uint32_t c[2] = {0u, 0u};
#pragma unroll
      for (int e = 0; e < 8; e += 2)
        c[e >> 2] |= (uint32_t)quant2_e4m3(bfbits2f(ob[e]), bfbits2f(ob[e + 1]), s_q, inv_q) << (8 * (e & 3));
      reinterpret_cast<uint2*>(q + (size_t)t * n)[v] = make_uint2(c[0], c[1]);
    }
  }
}

cudaError_t launch_rmsnorm_residual(uint16_t* h, const uint16_t* add, const uint16_t* w, float eps,
                                    uint16_t* normed, uint8_t* q, float s_q, int T, int n, cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  return launch_pdl(k_rmsnorm_residual, dim3(T), dim3(256), 0, st, h, add, w, eps, normed, q, s_q,
                    q ? exact_inverse(s_q) : 0.f, n);
}

}  // namespace m2
