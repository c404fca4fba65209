// Fused paged decode of the mixer block's middle: for one decode row and one
// group of 8 heads (512 channels), in one CTA:
//   conv window update + SiLU for the group's x, B and C channels,
//   dt = softplus(dt_raw + dt_bias), the single-step state update of the
//   8 heads read from and written back to pool[slot] in place,
//   y = S C + D x, then the gated group RMSNorm over the same 512 channels
//   and the e4m3 quant of its output (out_proj's input).
// The slot-pool gather, advance-in-place and scatter of vllm.cpp PR #1288
// ("What it does": the paged arm advances the gathered rows IN PLACE) become
// addressing through slot_idx; nothing is copied to a working buffer.
// Each CTA owns a disjoint set of conv channels and state rows, so no two
// CTAs touch the same memory (slot ids are unique per call).
#include "m2_kernels.h"

namespace m2 {

constexpr int kDecThreads = 256;

__global__ void __launch_bounds__(kDecThreads) k_decode_fused(
    const uint16_t* __restrict__ zx, const uint16_t* __restrict__ conv_w, const uint16_t* __restrict__ conv_b,
    const float* __restrict__ A_log, const float* __restrict__ Dp, const float* __restrict__ dt_bias,
    const uint16_t* __restrict__ norm_w, float eps, float s_y, uint16_t* __restrict__ conv_pool,
    float* __restrict__ ssm_pool, int n_slots, const int32_t* __restrict__ slot_idx, uint8_t* __restrict__ q2,
    int* __restrict__ err, DecodeTaps taps) {
  __shared__ float ux[kGroupCh];   // conv output, x channels of the group
  __shared__ __align__(16) float ub[kN];   // B of the group (read as float4)
  __shared__ __align__(16) float uc[kN];   // C of the group (read as float4)
  __shared__ float ys[kGroupCh];   // scan output (bf16-rounded)
  __shared__ float dts[kHPG], dAs[kHPG];
  __shared__ float red[kDecThreads / 32];

  const int b = blockIdx.x, g = blockIdx.y, tid = threadIdx.x;
  const int slot = slot_idx[b];
  uint8_t* q2row = q2 + (size_t)b * kI + g * kGroupCh;
  if (slot < 0 || slot >= n_slots) {
    if (slot != -1 && tid == 0) atomicOr(err, kErrSlot);
    for (int i = tid; i < kGroupCh; i += kDecThreads) q2row[i] = 0;
    return;
  }
  const uint16_t* zrow = zx + (size_t)b * kZ;

  // conv window update: 512 x channels + 128 B + 128 C channels
  for (int k = tid; k < kGroupCh + 2 * kN; k += kDecThreads) {
    int c;
    if (k < kGroupCh) c = g * kGroupCh + k;
    else if (k < kGroupCh + kN) c = kOffB + g * kN + (k - kGroupCh);
    else c = kOffC + g * kN + (k - kGroupCh - kN);
    uint16_t* st = conv_pool + ((size_t)slot * kConv + c) * (kW - 1);
    uint16_t t0 = st[0], t1 = st[1], t2 = st[2];
    uint16_t xn = zrow[kOffXBC + c];
    float acc = conv_b ? bfbits2f(conv_b[c]) : 0.f;
    const uint16_t* w = conv_w + c * kW;
    acc = fmaf(bfbits2f(w[0]), bfbits2f(t0), acc);
    acc = fmaf(bfbits2f(w[1]), bfbits2f(t1), acc);
    acc = fmaf(bfbits2f(w[2]), bfbits2f(t2), acc);
    acc = fmaf(bfbits2f(w[3]), bfbits2f(xn), acc);
    st[0] = t1; st[1] = t2; st[2] = xn;
    uint16_t ub16 = f2bfbits(silu_f(acc));
    float uv = bfbits2f(ub16);
    if (k < kGroupCh) ux[k] = uv;
    else if (k < kGroupCh + kN) ub[k - kGroupCh] = uv;
    else uc[k - kGroupCh - kN] = uv;
    if (taps.u) taps.u[(size_t)b * kConv + c] = ub16;
  }
  if (tid < kHPG) {
    int h = g * kHPG + tid;
    float dt = softplus_f(bfbits2f(zrow[kOffDt + h]) + dt_bias[h]);
    dts[tid] = dt;
    dAs[tid] = expf(dt * -expf(A_log[h]));
    if (taps.dt) taps.dt[(size_t)b * kNH + h] = dt;
  }
  __syncthreads();

  // state update: warp w handles rows p = w + 8*i of each head, lane owns
  // 4 consecutive state entries (float4) of the 128
  const int warp = tid >> 5, lane = tid & 31;
  const float4 bv = reinterpret_cast<const float4*>(ub)[lane];
  const float4 cv = reinterpret_cast<const float4*>(uc)[lane];
  for (int hh = 0; hh < kHPG; ++hh) {
    const int h = g * kHPG + hh;
    float4* base = reinterpret_cast<float4*>(ssm_pool + ((size_t)slot * kNH + h) * (kP * kN));
    const float dt = dts[hh], dA = dAs[hh];
    float4 s[kP / 8];
#pragma unroll
    for (int i = 0; i < kP / 8; ++i) s[i] = base[(warp + 8 * i) * (kN / 4) + lane];
    float part[kP / 8];
#pragma unroll
    for (int i = 0; i < kP / 8; ++i) {
      const int p = warp + 8 * i;
      const float xd = dt * ux[hh * kP + p];
      s[i].x = fmaf(dA, s[i].x, xd * bv.x);
      s[i].y = fmaf(dA, s[i].y, xd * bv.y);
      s[i].z = fmaf(dA, s[i].z, xd * bv.z);
      s[i].w = fmaf(dA, s[i].w, xd * bv.w);
      base[p * (kN / 4) + lane] = s[i];
      part[i] = s[i].x * cv.x + s[i].y * cv.y + s[i].z * cv.z + s[i].w * cv.w;
    }
#pragma unroll
    for (int i = 0; i < kP / 8; ++i) {
      float v = part[i];
#pragma unroll
      for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if (lane == 0) {
        const int p = warp + 8 * i;
        ys[hh * kP + p] = round_bf16(v + Dp[h] * ux[hh * kP + p]);
      }
    }
  }
  __syncthreads();

  // gated group RMSNorm + e4m3 quant of the 512 channels
  float gv[kGroupCh / kDecThreads];
  float ss = 0.f;
#pragma unroll
  for (int j = 0; j < kGroupCh / kDecThreads; ++j) {
    const int i = tid + j * kDecThreads;
    gv[j] = ys[i] * silu_f(bfbits2f(zrow[g * kGroupCh + i]));
    ss = fmaf(gv[j], gv[j], ss);
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if (lane == 0) red[warp] = ss;
  __syncthreads();
  float tot = 0.f;
#pragma unroll
  for (int w = 0; w < kDecThreads / 32; ++w) tot += red[w];
  const float r = 1.0f / sqrtf(tot / (float)kGroupCh + eps);
#pragma unroll
  for (int j = 0; j < kGroupCh / kDecThreads; ++j) {
    const int i = tid + j * kDecThreads;
    const int ch = g * kGroupCh + i;
    uint16_t o16 = f2bfbits(gv[j] * r * bfbits2f(norm_w[ch]));
    q2row[i] = quant_e4m3(bfbits2f(o16), s_y);
    if (taps.o) taps.o[(size_t)b * kI + ch] = o16;
    if (taps.y) taps.y[(size_t)b * kI + ch] = f2bfbits(ys[i]);
  }
}

cudaError_t launch_decode_fused(const uint16_t* zx, const BlockParams& bp, uint16_t* conv_pool, float* ssm_pool,
                                int n_slots, const int32_t* slot_idx, int Bt, uint8_t* q2, int* err,
                                const DecodeTaps& taps, cudaStream_t st) {
  dim3 grid(Bt, kG);
  k_decode_fused<<<grid, kDecThreads, 0, st>>>(zx, bp.conv_w, bp.conv_b, bp.A_log, bp.D, bp.dt_bias, bp.norm_w,
                                              bp.eps, bp.s_y, conv_pool, ssm_pool, n_slots, slot_idx, q2, err,
                                              taps);
  return cudaGetLastError();
}

}  // namespace m2
