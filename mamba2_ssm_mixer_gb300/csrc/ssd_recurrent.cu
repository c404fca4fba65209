// The SSD recurrence of a prefill evaluated token by token, for calls whose
// sequences are all short (Mamba2ChunkScan of vllm.cpp PR #1288, "What it
// does"; the recurrence of Dao & Gu 2024 in its sequential form):
//   dt_t = softplus(dt_raw_t + dt_bias_h),  a_t = exp(dt_t A_h),  A_h = -exp(A_log_h)
//   S_h <- a_t S_h + dt_t x_t B_t^T,        y_t = S_h C_t + D_h x_t
// For a sequence of a few dozen tokens the chunked evaluation (cumsum, chunk
// states, state pass, chunk scan: four dependent launches sized for 256-token
// chunks) is latency, not work.  Here one CTA per (sequence, head) stages the
// sequence's x, B, C rows in shared memory, keeps the head's 64 x 128 f32
// state in registers (thread t: row p = t / 4, columns 32 (t % 4) ..) and
// walks the tokens, as a decode step does for one token.  It also writes the
// final state and hands each sequence's conv window on (the last 3 raw xBC
// inputs), as the state pass does on the chunked path.
#include "launch_util.h"
#include "m2_kernels.h"

namespace m2 {

namespace {

constexpr int kRecThreads = 256;

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
  __shared__ __align__(16) uint16_t xs[kRecMaxT][kP];   // this head's x rows   8 KB
  __shared__ __align__(16) uint16_t bs[kRecMaxT][kN];   // the group's B rows  16 KB
  __shared__ __align__(16) uint16_t cs[kRecMaxT][kN];   // the group's C rows  16 KB
  __shared__ float2 da[kRecMaxT];                      // (dt, exp(dt A)) per token
  pdl_wait();
  pdl_trigger();
  const int h = blockIdx.x, s = blockIdx.y, g = h / kHPG, tid = threadIdx.x;
  const int t0 = si.cu_seqlens[s], T = si.cu_seqlens[s + 1] - t0;   // 1 <= T <= kRecMaxT (host-checked)
  const bool init = (si.has_init[s >> 5] >> (s & 31)) & 1u;

  // stage x (8 16-byte pieces a row), B and C (16 each) of every token
  for (int i = tid; i < T * 40; i += kRecThreads) {
    const int t = i / 40, q = i % 40;
    const uint16_t* row = u + (size_t)(t0 + t) * kConv;
    if (q < 8)
      cp_async16_rec(&xs[t][q * 8], row + h * kP + q * 8);
    else if (q < 24)
      cp_async16_rec(&bs[t][(q - 8) * 8], row + kOffB + g * kN + (q - 8) * 8);
    else
      cp_async16_rec(&cs[t][(q - 24) * 8], row + kOffC + g * kN + (q - 24) * 8);
  }
  if (tid < T) {
    const float dt = softplus_f(bfbits2f(zx[(size_t)(t0 + tid) * kZ + kOffDt + h]) + dt_bias[h]);
    da[tid] = make_float2(dt, expf(dt * -expf(A_log[h])));
    if (dt_tok) dt_tok[(size_t)(t0 + tid) * kNH + h] = dt;
  }
  // the sequence's new conv window: the last 3 raw xBC inputs of [old window,
  // x] (96 channels per head index); the conv kernel has read the old one
  if (conv_state && tid < kConv / kNH) {
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

  // this thread's 32 state entries: row p, columns n0 .. n0 + 31
  const int p = tid >> 2, n0 = (tid & 3) * 32;
  SS* srow = ssm_state + ((size_t)s * kNH + h) * (kP * kN) + (size_t)p * kN + n0;
  float S[32];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const float4 v = init ? ld_state4r(srow + 4 * j) : make_float4(0.f, 0.f, 0.f, 0.f);
    S[4 * j] = v.x, S[4 * j + 1] = v.y, S[4 * j + 2] = v.z, S[4 * j + 3] = v.w;
  }
  cp_async_wait_rec();
  __syncthreads();

  const float Dh = Dp[h];
  for (int t = 0; t < T; ++t) {
    const float2 d = da[t];
    const float xv = bfbits2f(xs[t][p]);
    const float xd = d.x * xv;
    float acc = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint4 bw = *reinterpret_cast<const uint4*>(&bs[t][n0 + 8 * j]);
      const uint4 cw = *reinterpret_cast<const uint4*>(&cs[t][n0 + 8 * j]);
      const uint32_t bb[4] = {bw.x, bw.y, bw.z, bw.w}, cc[4] = {cw.x, cw.y, cw.z, cw.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        float& s0 = S[8 * j + 2 * k];
        float& s1 = S[8 * j + 2 * k + 1];
        s0 = fmaf(d.y, s0, xd * __uint_as_float(bb[k] << 16));
        s1 = fmaf(d.y, s1, xd * __uint_as_float(bb[k] & 0xFFFF0000u));
        acc = fmaf(s0, __uint_as_float(cc[k] << 16), acc);
        acc = fmaf(s1, __uint_as_float(cc[k] & 0xFFFF0000u), acc);
      }
    }
    // the row's four quarters of C S^T
    acc += __shfl_xor_sync(0xffffffffu, acc, 1);
    acc += __shfl_xor_sync(0xffffffffu, acc, 2);
    if ((tid & 3) == 0) y[(size_t)(t0 + t) * kI + h * kP + p] = f2bfbits(acc + Dh * xv);
  }
#pragma unroll
  for (int j = 0; j < 8; ++j)
    st_state4r(srow + 4 * j, make_float4(S[4 * j], S[4 * j + 1], S[4 * j + 2], S[4 * j + 3]));
}

cudaError_t launch_ssd_recurrent(const uint16_t* zx, const uint16_t* u, const BlockParams& bp, const SeqInfo& si,
                                 uint16_t* y, void* ssm_state, bool bf16_state, uint16_t* conv_state, float* dt_tok,
                                 cudaStream_t st) {
  const dim3 grid(kNH, si.nseq);
  if (bf16_state)
    return launch_pdl(k_ssd_recurrent<uint16_t>, grid, dim3(kRecThreads), 0, st, zx, u, bp.A_log, bp.dt_bias, bp.D,
                      si, y, static_cast<uint16_t*>(ssm_state), conv_state, dt_tok);
  return launch_pdl(k_ssd_recurrent<float>, grid, dim3(kRecThreads), 0, st, zx, u, bp.A_log, bp.dt_bias, bp.D, si, y,
                    static_cast<float*>(ssm_state), conv_state, dt_tok);
}

}  // namespace m2
