// Paged decode of the mixer block after in_proj, in one kernel organised for
// HBM bandwidth.
// k_decode_stream: per work item, the conv window update + SiLU of its xBC
//   channels and dt, exp(dt A) of its heads (the row's conv window in the pool
//   shifts by one in place), then the single-step state update of each head,
//   read from and written back to pool[slot] in place, y = S C + D x, gated
//   group RMSNorm and e4m3 quant of out_proj's input:
//  - a work item is one (row, group); its 8 heads go to one CTA (HPC = 8,
//    from a few rows up) or, for the smallest batches, to the 8 CTAs of a
//    thread-block cluster, one head each (HPC = 1), so a single row spreads
//    its state traffic over 64 SMs; CTAs (clusters) are persistent (as many
//    as can be resident) and walk the items;
//  - in each CTA a producer thread streams its heads' states (64 x 128,
//    contiguous in the pool: 32 KB in f32, 16 KB in bf16) into a
//    shared-memory ring with cp.async.bulk (TMA, 1-D), items ahead, with an
//    evict-first L2 policy (the rows pass through once), and each item's
//    xBC, gate and dt inputs (of zx) into a small staging ring; the first
//    state loads are issued before waiting on the previous kernel (no earlier
//    kernel of the call writes the pool);
//  - the consumer warps hold the conv windows and conv weights of their next
//    item's channels in registers, loaded one item ahead (the first item's
//    before the wait: in_proj writes neither), run the conv + SiLU in place
//    in the staging slot, then update the state in shared memory; one thread
//    writes it back with a bulk store.  With a cluster, every CTA computes
//    the group's B and C channels (it needs them) and rank 0 writes their
//    windows back after the item's exchange, by which time every rank has
//    read the old ones;
//  - the group's RMSNorm needs the sum of squares over all 8 heads: with a
//    cluster, each CTA stores its partial into every CTA of the cluster
//    (distributed shared memory) and arrives on their barriers; each then
//    adds the partials in rank order (the same total everywhere) and
//    normalises and quantises its own channels.
// The pool rows are advanced in place through slot_idx: the gather and
// scatter of vllm.cpp PR #1288 ("What it does") are addressing.  Slot ids
// must be unique within a call (two rows advancing one slot would race): a row
// whose slot an earlier row of the call already names is skipped like a bad
// id (output zeroed, nothing touched) and flagged in the error word, so the
// first row naming a slot is the one that advances it.  A bf16 pool (the
// non-f32 state cache of the same section's ssm_dtype term) is widened to f32
// as it is read, updated and reduced to y in f32, and rounded to bf16
// (nearest even) as it is written back.  Optionally the state kernel also
// brings a buffer (the out_proj weights) into L2 with an evict-last policy, so
// the next kernel reads it from L2.  Every wait is bounded; a wait that runs
// out sets the device error word and the CTA stops issuing work, drains its
// copies and returns.
#include <map>
#include <mutex>

#include "m2_kernels.h"
#include "launch_util.h"
#include "tc_ptx.cuh"

namespace m2 {

using namespace tc;

namespace {

constexpr int kRingBytes = 3 * kP * kN * 4;   // 96 KB state ring per CTA, 2 CTAs per SM
constexpr int kConsumers = 256;             // 8 warps
constexpr int kThreadsT = kConsumers + 32;  // + producer warp
constexpr int kStg = 4;                     // staging ring depth (items)

__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar)), "l"(pol)
      : "memory");
}
__device__ __forceinline__ void bulk_store(void* dst, const void* src, uint32_t bytes, uint64_t pol) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group.L2::cache_hint [%0], [%1], %2, %3;" ::"l"(
                   reinterpret_cast<uint64_t>(dst)),
               "r"(smem_u32(src)), "r"(bytes), "l"(pol)
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

// One item's inputs as they sit in zx (bulk-copied); the conv replaces the
// xBC inputs with u in place.
template <int HPC>
struct __align__(16) Staging {
  uint16_t xc[kP * HPC];   // x of this CTA's heads: the new xBC inputs, then u (bf16)
  uint16_t bc[kN];         // the group's B: input, then u
  uint16_t cc[kN];         // the group's C: input, then u
  uint16_t z[kP * HPC];    // the gate (z of zx) of this CTA's channels
  uint16_t dtr[kHPG];      // the group's raw dt (dt of zx)
};

// Conv channel pairs of an item: this CTA's x channels, then the group's B
// and C channels (xBC numbering).
template <int HPC>
struct ItemPairs {
  static constexpr int kX = kP * HPC / 2;           // x pairs
  static constexpr int kAll = kX + kN;              // + 64 B pairs + 64 C pairs
  __device__ static int channel(int p, int h0, int g) {
    return p < kX ? h0 * kP + 2 * p : (p < kX + kN / 2 ? kOffB + g * kN + 2 * (p - kX) : kOffC + g * kN + 2 * (p - kX - kN / 2));
  }
};

template <typename S, int HPC>
struct __align__(16) Smem {
  static constexpr int kStages = kRingBytes / (kP * kN * (int)sizeof(S));   // 3 (f32) or 6 (bf16)
  static constexpr int kU = kHPG / HPC;                                      // CTAs per cluster
  S state[kStages][kP * kN];       // 96 KB ring
  Staging<HPC> stg[kStg];
  float2 dtA[HPC];                 // (dt, exp(dt A)) of this CTA's heads, current item
  uint32_t wbc[kU > 1 ? kN : 1][kW - 1];   // rank 0: the group's new B, C windows (pairs), until the exchange
  float ys[kP * HPC];
  float red[kConsumers / 32];
  float part[2][kU];               // the ranks' sums of squares, by item parity
  uint64_t full[kStages], empty[kStages];
  uint64_t sfull[kStg], sempty[kStg];
  uint64_t xb[2];                  // all ranks' partials have arrived, by item parity
  int abort;
};

}  // namespace

// ---------------------------------------------------------------------------
// conv, state update, y, gated norm and quant; cluster of 8 / HPC CTAs per item
// ---------------------------------------------------------------------------
template <typename S, int HPC>
__global__ void __launch_bounds__(kThreadsT, 2)
    k_decode_stream(const uint16_t* __restrict__ zx, const uint16_t* __restrict__ conv_w,
                    const uint16_t* __restrict__ conv_b, const float* __restrict__ A_log,
                    const float* __restrict__ dt_bias, const float* __restrict__ Dp,
                    const uint16_t* __restrict__ norm_w, float eps, float s_y, uint16_t* __restrict__ conv_pool,
                    S* __restrict__ ssm_pool, int n_slots, const int32_t* __restrict__ slot_idx, int Bt,
                    uint8_t* __restrict__ q2, int* __restrict__ err, DecodeTaps taps,
                    const uint8_t* __restrict__ l2_prefetch, uint32_t l2_prefetch_bytes) {
  using Sm = Smem<S, HPC>;
  constexpr int kStages = Sm::kStages;
  constexpr int kU = Sm::kU;
  constexpr uint32_t kHeadBytes = kP * kN * sizeof(S);
  constexpr uint32_t kStgBytes = sizeof(Staging<HPC>);
  constexpr int kCh = kP * HPC;                                  // channels of this CTA
  constexpr int kPer = (kCh + kConsumers - 1) / kConsumers;      // of them per consumer thread
  extern __shared__ uint8_t smem_raw[];
  Sm& sm = *reinterpret_cast<Sm*>(smem_align<128>(smem_raw));
  volatile int* abort = &sm.abort;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int items = Bt * kG;
  const int rank = kU > 1 ? (int)cluster_ctarank() : 0;   // the CTA's heads: rank * HPC .. of the group
  const int cluster = blockIdx.x / kU, nclusters = gridDim.x / kU;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], 1);
    }
    for (int s = 0; s < kStg; ++s) {
      mbar_init(&sm.sfull[s], 1);
      mbar_init(&sm.sempty[s], 1);
    }
    mbar_init(&sm.xb[0], kU);
    mbar_init(&sm.xb[1], kU);
    sm.abort = 0;
    fence_mbar_init();
  }
  __syncwarp();
  if (kU > 1) cluster_sync();   // every CTA's barriers exist before any remote arrive
  else __syncthreads();
  const uint64_t pol_stream = policy_evict_first();

  if (warp == kConsumers / 32) {
    // ------------------------------------------------ producer warp
    // (all lanes walk the items to share the duplicate scan; lane 0 issues)
    int stage = 0, ss = 0, heads = 0;
    uint32_t phase = 0, sphase = 0;
    bool ok = true;
    bool issued[kStages], sissued[kStg];
    uint32_t issued_phase[kStages], sissued_phase[kStg];
    for (int s = 0; s < kStages; ++s) issued[s] = false, issued_phase[s] = 0;
    for (int s = 0; s < kStg; ++s) sissued[s] = false, sissued_phase[s] = 0;
    // the first ring fill of state rows, before waiting on the previous kernel
    // (it writes none of the pool): heads [0, npre) in item order
    int npre = 0;
    for (int it = cluster; it < items && npre < kStages; it += nclusters) {
      const int b = it / kG, g = it % kG;
      const int slot = slot_idx[b];
      if (slot < 0 || slot >= n_slots) continue;
      if (slot_named_earlier(slot_idx, b, slot, lane)) continue;
      for (int hh = 0; hh < HPC && npre < kStages; ++hh, ++npre) {
        if (lane == 0) {
          mbar_expect_tx(&sm.full[npre], kHeadBytes);
          bulk_load(sm.state[npre], ssm_pool + ((size_t)slot * kNH + g * kHPG + rank * HPC + hh) * (kP * kN),
                    kHeadBytes, &sm.full[npre], pol_stream);
          issued[npre] = true;
        }
      }
    }
    pdl_wait();      // u, dt and zx come from the previous kernels
    pdl_trigger();
    for (int it = cluster; it < items && ok; it += nclusters) {
      const int b = it / kG, g = it % kG;
      const int slot = slot_idx[b];
      if (slot < 0 || slot >= n_slots) continue;
      if (slot_named_earlier(slot_idx, b, slot, lane)) continue;
      if (lane == 0) {
        const int h0 = g * kHPG + rank * HPC;
        // the item's inputs
        if (mbar_wait(&sm.sempty[ss], sphase ^ 1u, abort)) {
          Staging<HPC>& st = sm.stg[ss];
          mbar_expect_tx(&sm.sfull[ss], kStgBytes);
          const uint16_t* zr = zx + (size_t)b * kZ;
          bulk_load(st.xc, zr + kOffXBC + h0 * kP, kP * HPC * 2, &sm.sfull[ss], pol_stream);
          bulk_load(st.bc, zr + kOffXBC + kOffB + g * kN, kN * 2, &sm.sfull[ss], pol_stream);
          bulk_load(st.cc, zr + kOffXBC + kOffC + g * kN, kN * 2, &sm.sfull[ss], pol_stream);
          bulk_load(st.z, zr + h0 * kP, kP * HPC * 2, &sm.sfull[ss], pol_stream);
          bulk_load(st.dtr, zr + kOffDt + g * kHPG, kHPG * 2, &sm.sfull[ss], pol_stream);
          sissued[ss] = true;
          sissued_phase[ss] = sphase;
          if (++ss == kStg) ss = 0, sphase ^= 1u;
        } else {
          ok = false;
        }
        // the item's state rows (the first npre heads are already on their way)
        for (int hh = 0; hh < HPC && ok; ++hh, ++heads) {
          if (heads >= npre) {
            if (!mbar_wait(&sm.empty[stage], phase ^ 1u, abort)) {
              ok = false;
              break;
            }
            mbar_expect_tx(&sm.full[stage], kHeadBytes);
            bulk_load(sm.state[stage], ssm_pool + ((size_t)slot * kNH + h0 + hh) * (kP * kN), kHeadBytes,
                      &sm.full[stage], pol_stream);
            issued[stage] = true;
            issued_phase[stage] = phase;
          }
          if (++stage == kStages) stage = 0, phase ^= 1u;
        }
        if (!ok) {
          *abort = 1;
          atomicOr(err, kErrTimeout);
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
    }
    if (lane == 0) {
      // this CTA's share of the buffer the next kernel reads, into L2
      if (l2_prefetch && l2_prefetch_bytes) {
        const uint32_t per = ((l2_prefetch_bytes + gridDim.x - 1) / gridDim.x + 15) & ~15u;
        const uint32_t off = per * blockIdx.x;
        if (off < l2_prefetch_bytes)
          prefetch_l2(l2_prefetch + off, min(per, l2_prefetch_bytes - off), policy_evict_last());
      }
      // let every load issued land before the CTA can exit (state and staging)
      for (int s = 0; s < kStages; ++s)
        if (issued[s]) mbar_wait(&sm.full[s], issued_phase[s], nullptr, 100000000ull);
      for (int s = 0; s < kStg; ++s)
        if (sissued[s]) mbar_wait(&sm.sfull[s], sissued_phase[s], nullptr, 100000000ull);
    }
  } else {
    // ------------------------------------------------ consumer warps
    using IP = ItemPairs<HPC>;
    constexpr int kPPT = (IP::kAll + kConsumers - 1) / kConsumers;   // conv pairs per thread
    // the next item's conv windows (3 words: taps 0-2 of two channels), conv
    // weights and bias of this thread's pairs, loaded one item ahead
    uint32_t win[kPPT][kW - 1], cbv[kPPT];
    uint4 cwv[kPPT];
    auto load_item = [&](int it) {
      if (it >= items) return;
      const int b = it / kG, g = it % kG, slot = slot_idx[b];
      if (slot < 0 || slot >= n_slots) return;   // never read outside the pool
      const int h0 = g * kHPG + rank * HPC;
#pragma unroll
      for (int j = 0; j < kPPT; ++j) {
        const int pp = tid + j * kConsumers;
        if (pp < IP::kAll) {
          const int c = IP::channel(pp, h0, g);
          const uint32_t* tp = reinterpret_cast<const uint32_t*>(conv_pool + ((size_t)slot * kConv + c) * (kW - 1));
#pragma unroll
          for (int k = 0; k < kW - 1; ++k) win[j][k] = tp[k];
          cwv[j] = *reinterpret_cast<const uint4*>(conv_w + (size_t)c * kW);
          cbv[j] = conv_b ? *reinterpret_cast<const uint32_t*>(conv_b + c) : 0u;
        }
      }
    };
    load_item(cluster);   // before the wait: no kernel of the call writes the windows or the weights
    pdl_wait();
    pdl_trigger();
    int stage = 0, ss = 0;
    uint32_t phase = 0, sphase = 0;
    int prev = -1;   // stage whose bulk store may still be reading shared memory (thread 0)
    int k = 0;       // items exchanged so far (the partials' parity)
    // (an abort does not break this loop: every consumer must reach every named
    // barrier; after an abort the waits return at once and nothing is stored)
    for (int it = cluster; it < items; it += nclusters) {
      const int b = it / kG, g = it % kG;
      const int h0 = g * kHPG + rank * HPC;
      const int slot = slot_idx[b];
      uint8_t* q2c = q2 + (size_t)b * kI + h0 * kP;
      const bool bad = slot < 0 || slot >= n_slots;
      // every consumer warp takes the same decision from the same reads (and
      // every CTA of the cluster too: they share the row)
      const bool dup = !bad && slot_named_earlier(slot_idx, b, slot, lane);
      if (bad || dup) {
        if (tid == 0 && rank == 0 && dup) atomicOr(err, kErrDupSlot);
        if (tid == 0 && rank == 0 && bad && slot != -1) atomicOr(err, kErrSlot);
        for (int j = tid; j < kCh; j += kConsumers) q2c[j] = 0;
        load_item(it + nclusters);
        continue;
      }
      if (!mbar_wait(&sm.sfull[ss], sphase, abort)) {
        if (tid == 0) atomicOr(err, kErrTimeout);
        *abort = 1;
      }
      Staging<HPC>& st = sm.stg[ss];
      // conv + SiLU of the item's channel pairs (as the prefill conv: bias,
      // then taps oldest first, then the new input), u in place of the input;
      // the window shifts in (t1, t2, x_new) per channel
#pragma unroll
      for (int j = 0; j < kPPT; ++j) {
        const int pp = tid + j * kConsumers;
        if (pp < IP::kAll) {
          const int c = IP::channel(pp, h0, g);
          uint16_t* xs = pp < IP::kX ? &st.xc[2 * pp]
                                     : (pp < IP::kX + kN / 2 ? &st.bc[2 * (pp - IP::kX)] : &st.cc[2 * (pp - IP::kX - kN / 2)]);
          const uint32_t xn = *reinterpret_cast<const uint32_t*>(xs);
          const uint32_t w0 = win[j][0], w1 = win[j][1], w2 = win[j][2];
          const uint4 cw = cwv[j];
          const uint16_t t0a = w0 & 0xFFFF, t1a = w0 >> 16, t2a = w1 & 0xFFFF;
          const uint16_t t0b = w1 >> 16, t1b = w2 & 0xFFFF, t2b = w2 >> 16;
          const uint16_t xa = xn & 0xFFFF, xb = xn >> 16;
          float acc_a = bfbits2f(cbv[j] & 0xFFFF), acc_b = bfbits2f(cbv[j] >> 16);
          acc_a = fmaf(bfbits2f(cw.x & 0xFFFF), bfbits2f(t0a), acc_a);
          acc_a = fmaf(bfbits2f(cw.x >> 16), bfbits2f(t1a), acc_a);
          acc_a = fmaf(bfbits2f(cw.y & 0xFFFF), bfbits2f(t2a), acc_a);
          acc_a = fmaf(bfbits2f(cw.y >> 16), bfbits2f(xa), acc_a);
          acc_b = fmaf(bfbits2f(cw.z & 0xFFFF), bfbits2f(t0b), acc_b);
          acc_b = fmaf(bfbits2f(cw.z >> 16), bfbits2f(t1b), acc_b);
          acc_b = fmaf(bfbits2f(cw.w & 0xFFFF), bfbits2f(t2b), acc_b);
          acc_b = fmaf(bfbits2f(cw.w >> 16), bfbits2f(xb), acc_b);
          const uint32_t uu = (uint32_t)f2bfbits(silu_f(acc_a)) | ((uint32_t)f2bfbits(silu_f(acc_b)) << 16);
          *reinterpret_cast<uint32_t*>(xs) = uu;
          const uint32_t n0w = (uint32_t)t1a | ((uint32_t)t2a << 16), n1w = (uint32_t)xa | ((uint32_t)t1b << 16),
                         n2w = (uint32_t)t2b | ((uint32_t)xb << 16);
          const bool own = pp < IP::kX || kU == 1;   // x windows, or B/C without a cluster
          if (own) {
            uint32_t* tp = reinterpret_cast<uint32_t*>(conv_pool + ((size_t)slot * kConv + c) * (kW - 1));
            tp[0] = n0w, tp[1] = n1w, tp[2] = n2w;
          } else if (rank == 0) {
            sm.wbc[pp - IP::kX][0] = n0w, sm.wbc[pp - IP::kX][1] = n1w, sm.wbc[pp - IP::kX][2] = n2w;
          }
          if (taps.u && (own || rank == 0)) *reinterpret_cast<uint32_t*>(taps.u + (size_t)b * kConv + c) = uu;
        }
      }
      if (tid < HPC) {
        const int h = h0 + tid;
        const float dt = softplus_f(bfbits2f(st.dtr[rank * HPC + tid]) + dt_bias[h]);
        sm.dtA[tid] = make_float2(dt, expf(dt * -expf(A_log[h])));
        if (taps.dt) taps.dt[(size_t)b * kNH + h] = dt;
      }
      load_item(it + nclusters);
      consumers_sync();   // every u and dt of the item is in shared memory
      const uint2 bw = *reinterpret_cast<const uint2*>(st.bc + 4 * lane);
      const uint2 cw = *reinterpret_cast<const uint2*>(st.cc + 4 * lane);
      const float4 bv = make_float4(__uint_as_float(bw.x << 16), __uint_as_float(bw.x & 0xFFFF0000u),
                                    __uint_as_float(bw.y << 16), __uint_as_float(bw.y & 0xFFFF0000u));
      const float4 cv = make_float4(__uint_as_float(cw.x << 16), __uint_as_float(cw.x & 0xFFFF0000u),
                                    __uint_as_float(cw.y << 16), __uint_as_float(cw.y & 0xFFFF0000u));
      for (int hh = 0; hh < HPC; ++hh) {
        const int h = h0 + hh;
        const bool ok = mbar_wait(&sm.full[stage], phase, abort);
        if (!ok) {
          if (tid == 0) atomicOr(err, kErrTimeout);
          *abort = 1;
        }
        S* St = sm.state[stage];
        const float dt = sm.dtA[hh].x, dA = sm.dtA[hh].y;
        float part[kP / 8];
#pragma unroll
        for (int i = 0; i < kP / 8; ++i) {
          const int p = warp + 8 * i;
          float4 s4 = ld4(St + p * kN + 4 * lane);
          const float xd = dt * bfbits2f(st.xc[hh * kP + p]);
          s4.x = fmaf(dA, s4.x, xd * bv.x);
          s4.y = fmaf(dA, s4.y, xd * bv.y);
          s4.z = fmaf(dA, s4.z, xd * bv.z);
          s4.w = fmaf(dA, s4.w, xd * bv.w);
          st4(St + p * kN + 4 * lane, s4);   // f32, or rounded to bf16 for a bf16 pool
          part[i] = s4.x * cv.x + s4.y * cv.y + s4.z * cv.z + s4.w * cv.w;
        }
#pragma unroll
        for (int i = 0; i < kP / 8; ++i) {
          float v = part[i];
#pragma unroll
          for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
          if (lane == 0) {
            const int p = warp + 8 * i;
            sm.ys[hh * kP + p] = round_bf16(v + Dp[h] * bfbits2f(st.xc[hh * kP + p]));
          }
        }
        fence_async_smem();
        consumers_sync();
        if (tid == 0) {
          // write the head back; release the previous stage once its store has
          // finished reading shared memory (one store stays in flight)
          S* dst = ssm_pool + ((size_t)slot * kNH + h) * (kP * kN);
          if (ok) bulk_store(dst, sm.state[stage], kHeadBytes, pol_stream);
          else asm volatile("cp.async.bulk.commit_group;" ::: "memory");
          if (prev >= 0) {
            asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
            mbar_arrive(&sm.empty[prev]);
          }
          prev = stage;
        }
        if (++stage == kStages) stage = 0, phase ^= 1u;
      }
      // gated group RMSNorm + e4m3 quant: this CTA's 64 HPC channels; the sum
      // of squares over the group's 512 comes from all CTAs of the cluster
      float gv[kPer];
      float ssq = 0.f;
#pragma unroll
      for (int i = 0; i < kPer; ++i) {
        const int j = tid + i * kConsumers;
        gv[i] = j < kCh ? sm.ys[j] * silu_f(bfbits2f(st.z[j])) : 0.f;
        ssq = fmaf(gv[i], gv[i], ssq);
      }
#pragma unroll
      for (int o = 16; o; o >>= 1) ssq += __shfl_xor_sync(0xffffffffu, ssq, o);
      if (lane == 0) sm.red[warp] = ssq;
      consumers_sync();
      float tot = 0.f;
      const int par = k & 1;
      if (kU > 1) {
        if (tid == 0) {
          float mine = 0.f;
#pragma unroll
          for (int w = 0; w < kConsumers / 32; ++w) mine += sm.red[w];
          const uint32_t pa = smem_u32(&sm.part[par][rank]);
          const uint32_t xa = smem_u32(&sm.xb[par]);
          for (int r = 0; r < kU; ++r) st_dsmem_f32(cluster_map(pa, (uint32_t)r), mine);
          for (int r = 0; r < kU; ++r) mbar_arrive_remote(cluster_map(xa, (uint32_t)r));
        }
        if (!mbar_wait_cluster(&sm.xb[par], (uint32_t)(k >> 1) & 1u, abort)) {
          if (tid == 0) atomicOr(err, kErrTimeout);
          *abort = 1;
        }
        // every rank has read the group's old B, C windows (before its own
        // arrival): rank 0 writes the new ones
        if (rank == 0 && tid < kN) {
          const int c = tid < kN / 2 ? kOffB + g * kN + 2 * tid : kOffC + g * kN + 2 * (tid - kN / 2);
          uint32_t* tp = reinterpret_cast<uint32_t*>(conv_pool + ((size_t)slot * kConv + c) * (kW - 1));
          tp[0] = sm.wbc[tid][0], tp[1] = sm.wbc[tid][1], tp[2] = sm.wbc[tid][2];
        }
#pragma unroll
        for (int r = 0; r < kU; ++r) tot += sm.part[par][r];
      } else {
#pragma unroll
        for (int w = 0; w < kConsumers / 32; ++w) tot += sm.red[w];
      }
      const float rn = 1.0f / sqrtf(tot / (float)kGroupCh + eps);
#pragma unroll
      for (int i = 0; i < kPer; ++i) {
        const int j = tid + i * kConsumers;
        if (j < kCh) {
          const int ch = h0 * kP + j;
          const uint16_t o16 = f2bfbits(gv[i] * rn * bfbits2f(norm_w[ch]));
          q2c[j] = quant_e4m3(bfbits2f(o16), s_y);
          if (taps.o) taps.o[(size_t)b * kI + ch] = o16;
          if (taps.y) taps.y[(size_t)b * kI + ch] = f2bfbits(sm.ys[j]);
        }
      }
      ++k;
      consumers_sync();   // ys, red and the staging slot are free for the next item
      if (tid == 0) mbar_arrive(&sm.sempty[ss]);
      if (++ss == kStg) ss = 0, sphase ^= 1u;
    }
    if (tid == 0) {
      bulk_wait_all();
      if (prev >= 0) mbar_arrive(&sm.empty[prev]);
    }
  }
  __syncwarp();
  if (kU > 1) cluster_sync();   // no CTA leaves while another may still write to it
}

namespace {

// Clusters that fit on the device at once for this kernel (cached per
// device and instantiation).
template <typename S, int HPC>
int resident_clusters(size_t smem) {
  constexpr int kU = kHPG / HPC;
  static std::mutex mu;
  static std::map<int, int> by_device;
  int dev = 0;
  cudaGetDevice(&dev);
  std::lock_guard<std::mutex> lock(mu);
  auto it = by_device.find(dev);
  if (it != by_device.end()) return it->second;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(kU * 64);
  cfg.blockDim = dim3(kThreadsT);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kU;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, k_decode_stream<S, HPC>, &cfg) != cudaSuccess || n < 1)
    n = 2 * device_sm_count() / kU;   // two CTAs per SM
  by_device[dev] = n;
  return n;
}

}  // namespace

template <typename S, int HPC>
static cudaError_t launch_state_t(const uint16_t* zx, const BlockParams& bp, uint16_t* conv_pool, S* ssm_pool,
                                  int n_slots, const int32_t* slot_idx, int Bt, uint8_t* q2, int* err,
                                  const DecodeTaps& taps, const void* l2_prefetch, size_t l2_prefetch_bytes,
                                  cudaStream_t st) {
  constexpr int kU = kHPG / HPC;
  auto k = k_decode_stream<S, HPC>;
  const size_t smem = sizeof(Smem<S, HPC>) + 128;
  cudaError_t e = ensure_smem_optin(reinterpret_cast<const void*>(k), (int)smem);
  if (e != cudaSuccess) return e;
  const int items = Bt * kG;
  const int rc = resident_clusters<S, HPC>(smem);
  const int clusters = items < rc ? items : rc;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(clusters * kU);
  cfg.blockDim = dim3(kThreadsT);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = kU;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = kU > 1 ? 2 : 1;
  const uint32_t pf = (l2_prefetch && l2_prefetch_bytes < (1u << 31)) ? (uint32_t)(l2_prefetch_bytes & ~(size_t)15) : 0u;
  return cudaLaunchKernelEx(&cfg, k, zx, bp.conv_w, bp.conv_b, bp.A_log, bp.dt_bias, bp.D, bp.norm_w, bp.eps, bp.s_y,
                            conv_pool, ssm_pool, n_slots, slot_idx, Bt, q2, err, taps,
                            static_cast<const uint8_t*>(pf ? l2_prefetch : nullptr), pf);
}

// Heads per CTA of the state kernel for a batch of Bt rows: one for the
// smallest batches (their few items then use 8 CTAs each), all eight of the
// group otherwise (no exchange: measured faster from a few rows up, where
// the items alone fill the GPU; 2 and 4 heads per CTA were slower at 64 rows).
int decode_heads_per_cta(int Bt) { return Bt <= 2 ? 1 : 8; }

template <typename S>
static cudaError_t launch_state_s(const uint16_t* zx, const BlockParams& bp, uint16_t* conv_pool, S* ssm_pool,
                                  int n_slots, const int32_t* slot_idx, int Bt, uint8_t* q2, int* err,
                                  const DecodeTaps& taps, const void* l2_prefetch, size_t l2_prefetch_bytes,
                                  cudaStream_t st) {
  switch (decode_heads_per_cta(Bt)) {
    case 1:
      return launch_state_t<S, 1>(zx, bp, conv_pool, ssm_pool, n_slots, slot_idx, Bt, q2, err, taps, l2_prefetch,
                                  l2_prefetch_bytes, st);
    default:
      return launch_state_t<S, 8>(zx, bp, conv_pool, ssm_pool, n_slots, slot_idx, Bt, q2, err, taps, l2_prefetch,
                                  l2_prefetch_bytes, st);
  }
}

cudaError_t launch_decode_stream(const uint16_t* zx, const BlockParams& bp, uint16_t* conv_pool, void* ssm_pool,
                                 bool bf16_state, int n_slots, const int32_t* slot_idx, int Bt, uint8_t* q2, int* err,
                                 const DecodeTaps& taps, cudaStream_t st, int* launches, const void* l2_prefetch,
                                 size_t l2_prefetch_bytes) {
  *launches = 0;
  cudaError_t e;
  if (bf16_state)
    e = launch_state_s(zx, bp, conv_pool, static_cast<uint16_t*>(ssm_pool), n_slots, slot_idx, Bt, q2, err, taps,
                       l2_prefetch, l2_prefetch_bytes, st);
  else
    e = launch_state_s(zx, bp, conv_pool, static_cast<float*>(ssm_pool), n_slots, slot_idx, Bt, q2, err, taps,
                       l2_prefetch, l2_prefetch_bytes, st);
  if (e == cudaSuccess) *launches = 1;
  return e;
}

}  // namespace m2
