// The SSD recurrence of a prefill evaluated token by token, for calls whose
// sequences are all short (Mamba2ChunkScan of vllm.cpp PR #1288, "What it
// does"; the recurrence of Dao & Gu 2024 in its sequential form):
//   dt_t = softplus(dt_raw_t + dt_bias_h),  a_t = exp(dt_t A_h),  A_h = -exp(A_log_h)
//   S_h <- a_t S_h + dt_t x_t B_t^T,        y_t = S_h C_t + D_h x_t
// For a sequence of a few dozen tokens the chunked evaluation (cumsum, chunk
// states, state pass, chunk scan: four dependent launches sized for 256-token
// chunks) is latency, not work.  Here four CTAs per (sequence, head), each
// owning 16 of the head's 64 state rows, stage the sequence's x, B, C rows in
// shared memory, keep their rows of the f32 state in registers (16 threads a
// row, 8 columns each) and walk the tokens, as a decode step does for one
// token.  It also writes the
// final state and hands each sequence's conv window on (the last 3 raw xBC
// inputs), as the state pass does on the chunked path.
#include "launch_util.h"
#include "m2_kernels.h"

namespace m2 {

namespace {

constexpr int kRecThreads = 256;
constexpr int kRecSplit = 4;                          // CTAs per (sequence, head)
constexpr int kRecRows = kP / kRecSplit;              // 16 state rows per CTA
constexpr int kRecTpr = kRecThreads / kRecRows;       // 16 threads per row, 8 columns each

__device__ __forceinline__ void cp_async16_rec(void* dst_smem, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(dst_smem)),
               "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_wait_rec() { asm volatile("cp.async.wait_all;" ::: "memory"); }

__device__ __forceinline__ float4 ld_state4r(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ void st_state4r(float* p, float4 v) { *reinterpret_cast<float4*>(p) = v; }
__device__ __forceinline__ float4 ld_state4r(const uint16_t* p) {
  const uint2 w = *reinterpret_cast<const uint2*>(p);
  return make_float4(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xFFFF0000u), __uint_as_float(w.y << 16),
                     __uint_as_float(w.y & 0xFFFF0000u));
}
__device__ __forceinline__ void st_state4r(uint16_t* p, float4 v) {
  *reinterpret_cast<uint2*>(p) = make_uint2(pack_bf16x2(v.x, v.y), pack_bf16x2(v.z, v.w));
}

}  // namespace

template <typename SS>
__global__ void __launch_bounds__(kRecThreads) k_ssd_recurrent(const uint16_t* __restrict__ zx,
                                                               const uint16_t* __restrict__ u,
                                                               const float* __restrict__ A_log,
                                                               const float* __restrict__ dt_bias,
                                                               const float* __restrict__ Dp, const SeqInfo si,
                                                               uint16_t* __restrict__ y, SS* __restrict__ ssm_state,
                                                               uint16_t* __restrict__ conv_state,
                                                               float* __restrict__ dt_tok) {
  __shared__ __align__(16) uint16_t xs[kRecMaxT][kRecRows];   // this CTA's x rows       2 KB
  __shared__ __align__(16) uint16_t bs[kRecMaxT][kN];         // the group's B rows    16 KB
  __shared__ __align__(16) uint16_t cs[kRecMaxT][kN];         // the group's C rows    16 KB
  __shared__ float2 da[kRecMaxT];                            // (dt, exp(dt A)) per token
  pdl_wait();
  pdl_trigger();
  const int h = blockIdx.x / kRecSplit, rs = blockIdx.x % kRecSplit, s = blockIdx.y;
  const int g = h / kHPG, tid = threadIdx.x, p0 = rs * kRecRows;
  const int t0 = si.cu_seqlens[s], T = si.cu_seqlens[s + 1] - t0;   // 1 <= T <= kRecMaxT (host-checked)
  const bool init = (si.has_init[s >> 5] >> (s & 31)) & 1u;

  // stage this CTA's x rows (2 16-byte pieces a token), B and C (16 each)
  for (int i = tid; i < T * 34; i += kRecThreads) {
    const int t = i / 34, q = i % 34;
    const uint16_t* row = u + (size_t)(t0 + t) * kConv;
    if (q < 2)
      cp_async16_rec(&xs[t][q * 8], row + h * kP + p0 + q * 8);
    else if (q < 18)
      cp_async16_rec(&bs[t][(q - 2) * 8], row + kOffB + g * kN + (q - 2) * 8);
    else
      cp_async16_rec(&cs[t][(q - 18) * 8], row + kOffC + g * kN + (q - 18) * 8);
  }
  if (tid < T) {
    const float dt = softplus_f(bfbits2f(zx[(size_t)(t0 + tid) * kZ + kOffDt + h]) + dt_bias[h]);
    da[tid] = make_float2(dt, expf(dt * -expf(A_log[h])));
    if (dt_tok && rs == 0) dt_tok[(size_t)(t0 + tid) * kNH + h] = dt;
  }
  // the sequence's new conv window: the last 3 raw xBC inputs of [old window,
  // x] (96 channels per head index, the head's first CTA); the conv kernel
  // has read the old one
  if (conv_state && rs == 0 && tid < kConv / kNH) {
    const int ch = h * (kConv / kNH) + tid;
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

  // this thread's 8 state entries: row p0 + r, columns n0 .. n0 + 7; the 16
  // threads of a row are 16 consecutive lanes of one warp
  const int r = tid / kRecTpr, n0 = (tid % kRecTpr) * 8;
  SS* srow = ssm_state + ((size_t)s * kNH + h) * (kP * kN) + (size_t)(p0 + r) * kN + n0;
  float S[8];
  {
    const float4 a = init ? ld_state4r(srow) : make_float4(0.f, 0.f, 0.f, 0.f);
    const float4 b = init ? ld_state4r(srow + 4) : make_float4(0.f, 0.f, 0.f, 0.f);
    S[0] = a.x, S[1] = a.y, S[2] = a.z, S[3] = a.w, S[4] = b.x, S[5] = b.y, S[6] = b.z, S[7] = b.w;
  }
  cp_async_wait_rec();
  __syncthreads();

  const float Dh = Dp[h];
#pragma unroll 2
  for (int t = 0; t < T; ++t) {
    const float2 d = da[t];
    const float xv = bfbits2f(xs[t][r]);
    const float xd = d.x * xv;
    const uint4 bw = *reinterpret_cast<const uint4*>(&bs[t][n0]);
    const uint4 cw = *reinterpret_cast<const uint4*>(&cs[t][n0]);
    const uint32_t bb[4] = {bw.x, bw.y, bw.z, bw.w}, cc[4] = {cw.x, cw.y, cw.z, cw.w};
    float part[2] = {0.f, 0.f};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      S[2 * k] = fmaf(d.y, S[2 * k], xd * __uint_as_float(bb[k] << 16));
      S[2 * k + 1] = fmaf(d.y, S[2 * k + 1], xd * __uint_as_float(bb[k] & 0xFFFF0000u));
      part[k & 1] = fmaf(S[2 * k], __uint_as_float(cc[k] << 16), part[k & 1]);
      part[k & 1] = fmaf(S[2 * k + 1], __uint_as_float(cc[k] & 0xFFFF0000u), part[k & 1]);
    }
    float acc = part[0] + part[1];
    // the row's 16 column groups of C S^T
#pragma unroll
    for (int o = 1; o < kRecTpr; o <<= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (tid % kRecTpr == 0) y[(size_t)(t0 + t) * kI + h * kP + p0 + r] = f2bfbits(acc + Dh * xv);
  }
  st_state4r(srow, make_float4(S[0], S[1], S[2], S[3]));
  st_state4r(srow + 4, make_float4(S[4], S[5], S[6], S[7]));
}

cudaError_t launch_ssd_recurrent(const uint16_t* zx, const uint16_t* u, const BlockParams& bp, const SeqInfo& si,
                                 uint16_t* y, void* ssm_state, bool bf16_state, uint16_t* conv_state, float* dt_tok,
                                 cudaStream_t st) {
  const dim3 grid(kNH * kRecSplit, si.nseq);
  if (bf16_state)
    return launch_pdl(k_ssd_recurrent<uint16_t>, grid, dim3(kRecThreads), 0, st, zx, u, bp.A_log, bp.dt_bias, bp.D,
                      si, y, static_cast<uint16_t*>(ssm_state), conv_state, dt_tok);
  return launch_pdl(k_ssd_recurrent<float>, grid, dim3(kRecThreads), 0, st, zx, u, bp.A_log, bp.dt_bias, bp.D, si, y,
                    static_cast<float*>(ssm_state), conv_state, dt_tok);
}

}  // namespace m2
