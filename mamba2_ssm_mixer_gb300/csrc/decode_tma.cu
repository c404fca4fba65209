// Paged decode of the mixer block (conv
// window update + SiLU, dt, the single-step state update of each head read
// from and written back to pool[slot] in place, y = S C + D x, gated group
// RMSNorm and e4m3 quant), organised for HBM bandwidth:
//
//  - persistent CTAs (two per SM, so one streams while the other is in its
//    conv or norm phase) walk the (row, group) work items;
//  - a producer thread streams every head's state (64 x 128, contiguous in the
//    pool: 32 KB in f32, 16 KB in bf16) into a shared-memory ring with
//    cp.async.bulk (TMA, 1-D) several heads ahead, so loads are always in
//    flight;
//  - 8 consumer warps update the state in shared memory, reduce y, and one
//    thread writes the updated 32 KB back with a bulk store;
//  - conv, gate and norm for an item run on the consumer warps while the ring
//    keeps streaming.
// The pool rows are advanced in place through slot_idx: the gather and
// scatter of vllm.cpp PR #1288 ("What it does") are addressing.  Slot ids
// must be unique within a call (two rows advancing one slot would race): a row
// whose slot an earlier row of the call already names is skipped like a bad
// id (output zeroed, nothing touched) and flagged in the error word, so the
// first row naming a slot is the one that advances it.  A bf16 pool
// (the non-f32 state cache of the same section's ssm_dtype term) is widened
// to f32 as it is read, updated and reduced to y in f32, and rounded to bf16
// (nearest even) as it is written back.  Every wait is
// bounded; a wait that runs out sets the device error word and the CTA stops
// issuing work, drains its copies and returns.
#include "m2_kernels.h"
#include "launch_util.h"
#include "tc_ptx.cuh"

namespace m2 {

using namespace tc;

namespace {

constexpr int kRingBytes = 3 * kP * kN * 4;   // 96 KB ring per CTA, 2 CTAs per SM
constexpr int kConsumers = 256;             // 8 warps
constexpr int kThreadsT = kConsumers + 32;  // + producer warp

__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_u32(dst)),
               "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}
__device__ __forceinline__ void bulk_store(void* dst, const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(reinterpret_cast<uint64_t>(dst)),
               "r"(smem_u32(src)), "r"(bytes)
               : "memory");
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void consumers_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kConsumers) : "memory"); }

// True when a row before b names `slot` too (whole warp; every lane gets the
// answer).  Rows are read in strides of 32, so a batch of Bt rows costs each
// lane Bt / 32 cached loads per item.
__device__ __forceinline__ bool slot_named_earlier(const int32_t* __restrict__ slot_idx, int b, int slot, int lane) {
  bool hit = false;
  for (int j = lane; j < b; j += 32) hit |= (slot_idx[j] == slot);
  return __any_sync(0xffffffffu, hit);
}

// Pool element types: 4 consecutive d_state entries as f32.
__device__ __forceinline__ float4 ld4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ void st4(float* p, float4 v) { *reinterpret_cast<float4*>(p) = v; }
__device__ __forceinline__ float4 ld4(const uint16_t* p) {
  const uint2 w = *reinterpret_cast<const uint2*>(p);
  return make_float4(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xFFFF0000u), __uint_as_float(w.y << 16),
                     __uint_as_float(w.y & 0xFFFF0000u));
}
__device__ __forceinline__ void st4(uint16_t* p, float4 v) {
  *reinterpret_cast<uint2*>(p) = make_uint2(pack_bf16x2(v.x, v.y), pack_bf16x2(v.z, v.w));
}

template <typename S>
struct __align__(16) Smem {
  static constexpr int kStages = kRingBytes / (kP * kN * (int)sizeof(S));   // 3 (f32) or 6 (bf16)
  S state[kStages][kP * kN];       // 96 KB ring
  float ux[kGroupCh];
  float4 ub[kN / 4];
  float4 uc[kN / 4];
  float ys[kGroupCh];
  float dts[kHPG], dAs[kHPG];
  float red[kConsumers / 32];
  uint64_t full[kStages], empty[kStages];
  int abort;
};

}  // namespace

template <typename S>
__global__ void __launch_bounds__(kThreadsT, 2)
    k_decode_stream(const uint16_t* __restrict__ zx, const uint16_t* __restrict__ conv_w,
                    const uint16_t* __restrict__ conv_b, const float* __restrict__ A_log, const float* __restrict__ Dp,
                    const float* __restrict__ dt_bias, const uint16_t* __restrict__ norm_w, float eps, float s_y,
                    uint16_t* __restrict__ conv_pool, S* __restrict__ ssm_pool, int n_slots,
                    const int32_t* __restrict__ slot_idx, int Bt, uint8_t* __restrict__ q2, int* __restrict__ err,
                    DecodeTaps taps) {
  constexpr int kStages = Smem<S>::kStages;
  constexpr uint32_t kHeadBytes = kP * kN * sizeof(S);
  extern __shared__ uint8_t smem_raw[];
  Smem<S>& sm = *reinterpret_cast<Smem<S>*>(smem_align<128>(smem_raw));
  volatile int* abort = &sm.abort;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int items = Bt * kG;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], 1);
    }
    sm.abort = 0;
    fence_mbar_init();
  }
  __syncthreads();
  pdl_wait();
  pdl_trigger();

  if (warp == kConsumers / 32) {
    // ------------------------------------------------ producer warp
    // (all lanes walk the items to share the duplicate scan; lane 0 issues)
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    bool issued[kStages];
    uint32_t issued_phase[kStages];
    for (int s = 0; s < kStages; ++s) issued[s] = false, issued_phase[s] = 0;
    for (int it = blockIdx.x; it < items && ok; it += gridDim.x) {
      const int b = it / kG, g = it % kG;
      const int slot = slot_idx[b];
      if (slot < 0 || slot >= n_slots) continue;
      if (slot_named_earlier(slot_idx, b, slot, lane)) continue;
      if (lane == 0) {
        const S* src = ssm_pool + ((size_t)slot * kNH + g * kHPG) * (kP * kN);
        for (int hh = 0; hh < kHPG; ++hh) {
          if (!mbar_wait(&sm.empty[stage], phase ^ 1u, abort)) {
            *abort = 1;
            atomicOr(err, kErrTimeout);
            ok = false;
            break;
          }
          mbar_expect_tx(&sm.full[stage], kHeadBytes);
          bulk_load(sm.state[stage], src + (size_t)hh * (kP * kN), kHeadBytes, &sm.full[stage]);
          issued[stage] = true;
          issued_phase[stage] = phase;
          if (++stage == kStages) stage = 0, phase ^= 1u;
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
    }
    if (lane == 0 && *abort)   // let loads already in flight land before the CTA can exit
      for (int s = 0; s < kStages; ++s)
        if (issued[s]) mbar_wait(&sm.full[s], issued_phase[s], nullptr, 100000000ull);
    return;
  }

  // ------------------------------------------------ consumer warps
  int stage = 0;
  uint32_t phase = 0;
  int prev = -1;   // stage whose bulk store may still be reading shared memory (thread 0)
  // (an abort does not break this loop: every consumer must reach every named
  // barrier; after an abort the waits return at once and nothing is stored)
  for (int it = blockIdx.x; it < items; it += gridDim.x) {
    const int b = it / kG, g = it % kG;
    const int slot = slot_idx[b];
    uint8_t* q2row = q2 + (size_t)b * kI + g * kGroupCh;
    const bool bad = slot < 0 || slot >= n_slots;
    // every consumer warp takes the same decision from the same reads
    const bool dup = !bad && slot_named_earlier(slot_idx, b, slot, lane);
    if (bad || dup) {
      if (tid == 0 && dup) atomicOr(err, kErrDupSlot);
      if (tid == 0 && bad && slot != -1) atomicOr(err, kErrSlot);
      for (int i = tid; i < kGroupCh; i += kConsumers) q2row[i] = 0;
      continue;
    }
    const uint16_t* zrow = zx + (size_t)b * kZ;
    // conv window update of the group's 512 x + 128 B + 128 C channels
    float* ubf = reinterpret_cast<float*>(sm.ub);
    float* ucf = reinterpret_cast<float*>(sm.uc);
    for (int k = tid; k < kGroupCh + 2 * kN; k += kConsumers) {
      int c;
      if (k < kGroupCh) c = g * kGroupCh + k;
      else if (k < kGroupCh + kN) c = kOffB + g * kN + (k - kGroupCh);
      else c = kOffC + g * kN + (k - kGroupCh - kN);
      uint16_t* st = conv_pool + ((size_t)slot * kConv + c) * (kW - 1);
      const uint16_t t0 = st[0], t1 = st[1], t2 = st[2];
      const uint16_t xn = zrow[kOffXBC + c];
      float acc = conv_b ? bfbits2f(conv_b[c]) : 0.f;
      const uint16_t* w = conv_w + c * kW;
      acc = fmaf(bfbits2f(w[0]), bfbits2f(t0), acc);
      acc = fmaf(bfbits2f(w[1]), bfbits2f(t1), acc);
      acc = fmaf(bfbits2f(w[2]), bfbits2f(t2), acc);
      acc = fmaf(bfbits2f(w[3]), bfbits2f(xn), acc);
      st[0] = t1;
      st[1] = t2;
      st[2] = xn;
      const uint16_t u16 = f2bfbits(silu_f(acc));
      const float uv = bfbits2f(u16);
      if (k < kGroupCh) sm.ux[k] = uv;
      else if (k < kGroupCh + kN) ubf[k - kGroupCh] = uv;
      else ucf[k - kGroupCh - kN] = uv;
      if (taps.u) taps.u[(size_t)b * kConv + c] = u16;
    }
    if (tid < kHPG) {
      const int h = g * kHPG + tid;
      const float dt = softplus_f(bfbits2f(zrow[kOffDt + h]) + dt_bias[h]);
      sm.dts[tid] = dt;
      sm.dAs[tid] = expf(dt * -expf(A_log[h]));
      if (taps.dt) taps.dt[(size_t)b * kNH + h] = dt;
    }
    consumers_sync();
    const float4 bv = sm.ub[lane];
    const float4 cv = sm.uc[lane];
    S* dst_base = ssm_pool + ((size_t)slot * kNH + g * kHPG) * (kP * kN);
    for (int hh = 0; hh < kHPG; ++hh) {
      const int h = g * kHPG + hh;
      const bool ok = mbar_wait(&sm.full[stage], phase, abort);
      if (!ok) {
        if (tid == 0) atomicOr(err, kErrTimeout);
        *abort = 1;
      }
      S* St = sm.state[stage];
      const float dt = sm.dts[hh], dA = sm.dAs[hh];
      float part[kP / 8];
#pragma unroll
      for (int i = 0; i < kP / 8; ++i) {
        const int p = warp + 8 * i;
        float4 s = ld4(St + p * kN + 4 * lane);
        const float xd = dt * sm.ux[hh * kP + p];
        s.x = fmaf(dA, s.x, xd * bv.x);
        s.y = fmaf(dA, s.y, xd * bv.y);
        s.z = fmaf(dA, s.z, xd * bv.z);
        s.w = fmaf(dA, s.w, xd * bv.w);
        st4(St + p * kN + 4 * lane, s);   // f32, or rounded to bf16 for a bf16 pool
        part[i] = s.x * cv.x + s.y * cv.y + s.z * cv.z + s.w * cv.w;
      }
#pragma unroll
      for (int i = 0; i < kP / 8; ++i) {
        float v = part[i];
#pragma unroll
        for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == 0) {
          const int p = warp + 8 * i;
          sm.ys[hh * kP + p] = round_bf16(v + Dp[h] * sm.ux[hh * kP + p]);
        }
      }
      fence_async_smem();
      consumers_sync();
      if (tid == 0) {
        // write the head back; release the previous stage once its store has
        // finished reading shared memory (one store stays in flight)
        if (ok) bulk_store(dst_base + (size_t)hh * (kP * kN), sm.state[stage], kHeadBytes);
        else asm volatile("cp.async.bulk.commit_group;" ::: "memory");
        if (prev >= 0) {
          asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
          mbar_arrive(&sm.empty[prev]);
        }
        prev = stage;
      }
      if (++stage == kStages) stage = 0, phase ^= 1u;
    }
    consumers_sync();
    // gated group RMSNorm + e4m3 quant over the 512 channels
    float gv[kGroupCh / kConsumers];
    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < kGroupCh / kConsumers; ++j) {
      const int i = tid + j * kConsumers;
      gv[j] = sm.ys[i] * silu_f(bfbits2f(zrow[g * kGroupCh + i]));
      ss = fmaf(gv[j], gv[j], ss);
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if (lane == 0) sm.red[warp] = ss;
    consumers_sync();
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < kConsumers / 32; ++w) tot += sm.red[w];
    const float r = 1.0f / sqrtf(tot / (float)kGroupCh + eps);
#pragma unroll
    for (int j = 0; j < kGroupCh / kConsumers; ++j) {
      const int i = tid + j * kConsumers;
      const int ch = g * kGroupCh + i;
      const uint16_t o16 = f2bfbits(gv[j] * r * bfbits2f(norm_w[ch]));
      q2row[i] = quant_e4m3(bfbits2f(o16), s_y);
      if (taps.o) taps.o[(size_t)b * kI + ch] = o16;
      if (taps.y) taps.y[(size_t)b * kI + ch] = f2bfbits(sm.ys[i]);
    }
    consumers_sync();   // ys, red, ux reused by the next item
  }
  if (tid == 0) {
    bulk_wait_all();
    if (prev >= 0) mbar_arrive(&sm.empty[prev]);
  }
}

template <typename S>
static cudaError_t launch_decode_t(const uint16_t* zx, const BlockParams& bp, uint16_t* conv_pool, S* ssm_pool,
                                   int n_slots, const int32_t* slot_idx, int Bt, uint8_t* q2, int* err,
                                   const DecodeTaps& taps, cudaStream_t st) {
  auto k = k_decode_stream<S>;
  cudaError_t e = ensure_smem_optin(reinterpret_cast<const void*>(k), (int)(sizeof(Smem<S>) + 128));
  if (e != cudaSuccess) return e;
  const int sms = device_sm_count();
  const int items = Bt * kG;
  const int grid = items < 2 * sms ? items : 2 * sms;
  return launch_pdl(k, dim3(grid), dim3(kThreadsT), sizeof(Smem<S>) + 128, st, zx, bp.conv_w, bp.conv_b, bp.A_log,
                    bp.D, bp.dt_bias, bp.norm_w, bp.eps, bp.s_y, conv_pool, ssm_pool, n_slots, slot_idx, Bt, q2, err,
                    taps);
}

cudaError_t launch_decode_stream(const uint16_t* zx, const BlockParams& bp, uint16_t* conv_pool, void* ssm_pool,
                                 bool bf16_state, int n_slots, const int32_t* slot_idx, int Bt, uint8_t* q2, int* err,
                                 const DecodeTaps& taps, cudaStream_t st) {
  if (bf16_state)
    return launch_decode_t(zx, bp, conv_pool, static_cast<uint16_t*>(ssm_pool), n_slots, slot_idx, Bt, q2, err,
                           taps, st);
  return launch_decode_t(zx, bp, conv_pool, static_cast<float*>(ssm_pool), n_slots, slot_idx, Bt, q2, err, taps, st);
}

}  // namespace m2
