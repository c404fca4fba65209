// Tensor-core (tcgen05, bf16 operands, f32 accumulation in TMEM) versions of
// the two contraction-heavy SSD stages of the prefill scan (Mamba2ChunkScan of
// vllm.cpp PR #1288, "What it does"; SSD block decomposition of Dao & Gu 2024):
//
// k_ssd_state_tc  one CTA per (chunk, group): for each of the group's 8 heads
//   S_c[n, p] = sum_t B[t, n] * (w_t x[t, p]),  w_t = exp(cum_last - cum_t) dt_t
//   as a 128 x 64 x 256 MMA.  The scaled operand w*x is split into a bf16 high
//   part and a bf16 remainder (two MMAs) so the chunk state keeps ~16 bits.
// k_ssd_scan_tc   one CTA per (chunk, group, 128-row half of the chunk):
//   G = C B^T once for the group (128 x 256 x 128), then per head
//   P[t, s] = G[t, s] exp(cum_t - cum_s) dt_s  (s <= t, else 0),
//   Y_diag = P x (128 x 64 x 256), Y_off = C S_in^T (128 x 64 x 128),
//   y = Y_diag + exp(cum_t) Y_off + D x.
//   P and S_in are split into a bf16 high part and a bf16 remainder (two MMAs
//   each): a single bf16 rounding of P gives y a ~1e-3 relative error, which
//   is enough to flip e4m3 codes of the out_proj input downstream.
// Operands are staged in shared memory in the K-major 128-byte-swizzled layout
// the MMA descriptors describe (transposes are done in registers, 8 x 8 blocks).
#include "m2_kernels.h"
#include "launch_util.h"
#include "tc_ptx.cuh"

namespace m2 {

using namespace tc;

namespace {

constexpr int kThr = 256;   // 8 warps; warps w and w + 4 share TMEM lanes [32 (w % 4), +32)

// Byte offset of the 16-byte chunk holding elements [k8*8, k8*8 + 8) of row r
// in a K-major bf16 operand tile of `rows` rows (64 elements per 128-byte
// swizzle atom; atoms along K are rows*128 bytes apart).
__device__ __forceinline__ uint32_t sw_chunk(int r, int k8, int rows) {
  const int a = k8 >> 3, c = k8 & 7;
  return (uint32_t)(a * rows * 128 + (r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4));
}

__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

__device__ __forceinline__ uint32_t bf2(float a, float b) {
  return (uint32_t)f2bfbits(a) | ((uint32_t)f2bfbits(b) << 16);
}
__device__ __forceinline__ uint16_t h16(const uint4& v, int j) {
  const uint32_t w = (j < 2) ? v.x : (j < 4) ? v.y : (j < 6) ? v.z : v.w;
  return (uint16_t)((j & 1) ? (w >> 16) : (w & 0xFFFFu));
}

// 8 x 8 bf16 transpose: in[i] holds row i (8 values); out[j] holds column j.
__device__ __forceinline__ void transpose8(const uint4 (&in)[8], uint4 (&out)[8]) {
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    uint32_t w[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) w[q] = (uint32_t)h16(in[2 * q], j) | ((uint32_t)h16(in[2 * q + 1], j) << 16);
    out[j] = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

struct ChunkPos {
  int t0, n;
};
__device__ __forceinline__ ChunkPos chunk_of(const SeqInfo& si, int c) {
  const int s = seq_of_chunk(si, c);
  ChunkPos cp;
  cp.t0 = si.cu_seqlens[s] + (c - si.cu_chunks[s]) * kChunk;
  cp.n = min(kChunk, si.cu_seqlens[s + 1] - cp.t0);
  return cp;
}

__device__ __forceinline__ bool wait_or_flag(uint64_t* bar, uint32_t parity, int* err) {
  if (mbar_wait(bar, parity, nullptr)) return true;
  if (err) atomicOr(err, kErrTimeout);
  return false;
}

}  // namespace

// ---------------------------------------------------------------------------
// chunk states
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kThr, 1)
    k_ssd_state_tc(const uint16_t* __restrict__ u, const float* __restrict__ dt, const float2* __restrict__ cum,
                   const SeqInfo si, float* __restrict__ states, int* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sBT = smem;                 // [128 n][256 t]   64 KB
  uint8_t* sWh = sBT + 128 * 256 * 2;  // [64 p][256 t]    32 KB
  uint8_t* sWl = sWh + 64 * 256 * 2;   // [64 p][256 t]    32 KB
  float* wts = reinterpret_cast<float*>(sWl + 64 * 256 * 2);   // [256]
  uint64_t* bar = reinterpret_cast<uint64_t*>(wts + kChunk);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bar + 1);

  const int c = blockIdx.x, g = blockIdx.y, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int quarter = warp & 3, colhalf = warp >> 2;
  const ChunkPos cp = chunk_of(si, c);
  constexpr uint32_t IDESC = idesc_f32acc(128, 64, 1u);   // bf16 x bf16 -> f32, M = 128 (n), N = 64 (p)

  if (tid == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(tslot, 64);
    tc_fence_before();
  }
  pdl_wait();
  pdl_trigger();
  // B^T: rows n, K = t.  8 x 8 blocks: 32 (t) x 16 (n) = 512 blocks.
  for (int blk = tid; blk < 512; blk += kThr) {
    const int tb = blk >> 4, nb = blk & 15;
    uint4 in[8], out[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int t = tb * 8 + i;
      in[i] = t < cp.n ? *reinterpret_cast<const uint4*>(u + (size_t)(cp.t0 + t) * kConv + kOffB + g * kN + nb * 8)
                       : make_uint4(0, 0, 0, 0);
    }
    transpose8(in, out);
#pragma unroll
    for (int j = 0; j < 8; ++j) *reinterpret_cast<uint4*>(sBT + sw_chunk(nb * 8 + j, tb, 128)) = out[j];
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;

  for (int hh = 0; hh < kHPG; ++hh) {
    const int h = g * kHPG + hh;
    const float2 cl = cum[(size_t)(cp.t0 + cp.n - 1) * kNH + h];
    for (int t = tid; t < kChunk; t += kThr) {
      float w = 0.f;
      if (t < cp.n) {
        const float2 ct = cum[(size_t)(cp.t0 + t) * kNH + h];
        w = expf((cl.x - ct.x) + (cl.y - ct.y)) * dt[(size_t)(cp.t0 + t) * kNH + h];
      }
      wts[t] = w;
    }
    __syncthreads();
    // (w x)^T split into hi + lo: rows p, K = t.  32 (t) x 8 (p) blocks.
    for (int blk = tid; blk < 256; blk += kThr) {
      const int tb = blk >> 3, pb = blk & 7;
      uint4 hi_in[8], lo_in[8], hi_out[8], lo_out[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int t = tb * 8 + i;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (t < cp.n) v = *reinterpret_cast<const uint4*>(u + (size_t)(cp.t0 + t) * kConv + h * kP + pb * 8);
        const float w = wts[t];
        uint32_t hw[4], lw[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float a = w * bfbits2f(h16(v, 2 * q)), b = w * bfbits2f(h16(v, 2 * q + 1));
          const uint32_t hp = bf2(a, b);
          const float ah = bfbits2f((uint16_t)(hp & 0xFFFFu)), bh = bfbits2f((uint16_t)(hp >> 16));
          hw[q] = hp;
          lw[q] = bf2(a - ah, b - bh);
        }
        hi_in[i] = make_uint4(hw[0], hw[1], hw[2], hw[3]);
        lo_in[i] = make_uint4(lw[0], lw[1], lw[2], lw[3]);
      }
      transpose8(hi_in, hi_out);
      transpose8(lo_in, lo_out);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        *reinterpret_cast<uint4*>(sWh + sw_chunk(pb * 8 + j, tb, 64)) = hi_out[j];
        *reinterpret_cast<uint4*>(sWl + sw_chunk(pb * 8 + j, tb, 64)) = lo_out[j];
      }
    }
    fence_async_smem();
    __syncthreads();
    if (tid == 0) {
      tc_fence_after();
      const uint32_t a0 = smem_u32(sBT), h0 = smem_u32(sWh), l0 = smem_u32(sWl);
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint64_t ad = desc_kmajor_sw128(a0 + a * 128 * 128) + 2 * j;
          mma_f16(tmem, ad, desc_kmajor_sw128(h0 + a * 64 * 128) + 2 * j, IDESC, (a | j) != 0);
          mma_f16(tmem, ad, desc_kmajor_sw128(l0 + a * 64 * 128) + 2 * j, IDESC, 1u);
        }
      mma_commit(bar);
    }
    __syncwarp();
    const bool ok = wait_or_flag(bar, hh & 1, err);
    tc_fence_after();
    // D[n = 32 quarter + lane][p] -> states[c][h][p][n]; warps 0-3 take p < 32,
    // warps 4-7 p >= 32
    float* out = states + ((size_t)c * kNH + h) * (kP * kN) + quarter * 32 + lane;
    {
      uint32_t r[32];
      tmem_ld_32x32b_x32(tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(colhalf * 32), r);
      tmem_ld_wait();
      if (ok) {
#pragma unroll
        for (int j = 0; j < 32; ++j) out[(size_t)(colhalf * 32 + j) * kN] = __uint_as_float(r[j]);
      }
    }
    tc_fence_before();
    __syncthreads();
  }
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 64);
  }
}

// ---------------------------------------------------------------------------
// chunk scan
// ---------------------------------------------------------------------------
__device__ __forceinline__ void split_bf16(float v, uint16_t& hi, uint16_t& lo) {
  hi = f2bfbits(v);
  lo = f2bfbits(v - bfbits2f(hi));
}

__global__ void __launch_bounds__(kThr, 1)
    k_ssd_scan_tc(const uint16_t* __restrict__ u, const float* __restrict__ dt, const float2* __restrict__ cum,
                  const float* __restrict__ states, const float* __restrict__ Dp, const SeqInfo si,
                  uint16_t* __restrict__ y, int* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sC = smem;                    // [128 t][128 n]   32 KB
  uint8_t* sB = sC + 128 * 128 * 2;      // [KS s][128 n]    64 KB, then P halves:
  uint8_t* sPh = sB;                     //   [128 t][128 s] 32 KB  (high part)
  uint8_t* sPl = sB + 128 * 128 * 2;     //   [128 t][128 s] 32 KB  (remainder)
  uint8_t* sXT = sB + 256 * 128 * 2;     // [64 p][256 s]    32 KB
  uint8_t* sSh = sXT + 64 * 256 * 2;     // [64 p][128 n]    16 KB
  uint8_t* sSl = sSh + 64 * 128 * 2;     // [64 p][128 n]    16 KB
  float2* cums = reinterpret_cast<float2*>(sSl + 64 * 128 * 2);  // [256] (hi, lo)
  float* dts = reinterpret_cast<float*>(cums + kChunk);           // [256]
  uint64_t* bar = reinterpret_cast<uint64_t*>(dts + kChunk);     // [2]
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bar + 2);

  const int c = blockIdx.x, g = blockIdx.y, tb = blockIdx.z, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int quarter = warp & 3, colhalf = warp >> 2;
  const ChunkPos cp = chunk_of(si, c);
  if (tb * 128 >= cp.n) return;
  const int KS = (tb + 1) * 128;           // sources s < KS (causal)
  const int row = quarter * 32 + lane;     // this thread's TMEM lane = row of the tile
  const int tt = tb * 128 + row;           // chunk-local token of that row
  constexpr uint32_t TMEM_COLS = 512;
  constexpr uint32_t COL_G = 0, COL_YD = 256, COL_YO = 320;
  constexpr uint32_t IDESC_Y = idesc_f32acc(128, 64, 1u);

  if (tid == 0) {
    mbar_init(&bar[0], 1);
    mbar_init(&bar[1], 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(tslot, TMEM_COLS);
    tc_fence_before();
  }
  pdl_wait();
  pdl_trigger();
  // C rows of this half and B rows 0..KS-1, natural layout (K = n)
  for (int e = tid; e < 128 * 16; e += kThr) {
    const int r = e >> 4, k8 = e & 15, t = tb * 128 + r;
    uint4 v = t < cp.n ? *reinterpret_cast<const uint4*>(u + (size_t)(cp.t0 + t) * kConv + kOffC + g * kN + k8 * 8)
                       : make_uint4(0, 0, 0, 0);
    *reinterpret_cast<uint4*>(sC + sw_chunk(r, k8, 128)) = v;
  }
  for (int e = tid; e < KS * 16; e += kThr) {
    const int s = e >> 4, k8 = e & 15;
    uint4 v = s < cp.n ? *reinterpret_cast<const uint4*>(u + (size_t)(cp.t0 + s) * kConv + kOffB + g * kN + k8 * 8)
                       : make_uint4(0, 0, 0, 0);
    *reinterpret_cast<uint4*>(sB + sw_chunk(s, k8, KS)) = v;
  }
  fence_async_smem();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
  if (tid == 0) {
    // G[t, s] = sum_n C[t, n] B[s, n]: M = 128, N = KS, K = 128
    const uint32_t idesc = idesc_f32acc(128, KS, 1u);
    const uint32_t c0 = smem_u32(sC), b0 = smem_u32(sB);
#pragma unroll
    for (int a = 0; a < 2; ++a)
#pragma unroll
      for (int j = 0; j < 4; ++j)
        mma_f16(tmem + COL_G, desc_kmajor_sw128(c0 + a * 128 * 128) + 2 * j,
                desc_kmajor_sw128(b0 + a * KS * 128) + 2 * j, idesc, (a | j) != 0);
    mma_commit(&bar[0]);
  }
  __syncwarp();
  bool ok = wait_or_flag(&bar[0], 0, err);   // after this the B tile's memory holds P
  tc_fence_after();
  uint32_t ph = 0;

  for (int hh = 0; hh < kHPG; ++hh) {
    const int h = g * kHPG + hh;
    for (int s = tid; s < KS; s += kThr) {
      cums[s] = s < cp.n ? cum[(size_t)(cp.t0 + s) * kNH + h] : make_float2(0.f, 0.f);
      dts[s] = s < cp.n ? dt[(size_t)(cp.t0 + s) * kNH + h] : 0.f;
    }
    // x^T: rows p, K = s.  (KS/8) x 8 blocks.
    for (int blk = tid; blk < (KS / 8) * 8; blk += kThr) {
      const int sb = blk >> 3, pb = blk & 7;
      uint4 in[8], out[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int s = sb * 8 + i;
        in[i] = s < cp.n ? *reinterpret_cast<const uint4*>(u + (size_t)(cp.t0 + s) * kConv + h * kP + pb * 8)
                         : make_uint4(0, 0, 0, 0);
      }
      transpose8(in, out);
#pragma unroll
      for (int j = 0; j < 8; ++j) *reinterpret_cast<uint4*>(sXT + sw_chunk(pb * 8 + j, sb, 64)) = out[j];
    }
    // S_in (state entering the chunk) as bf16 high + remainder: rows p, K = n
    const float* Sin = states + ((size_t)c * kNH + h) * (kP * kN);
    for (int e = tid; e < 64 * 16; e += kThr) {
      const int p = e >> 4, k8 = e & 15;
      const float4 a = *reinterpret_cast<const float4*>(Sin + p * kN + k8 * 8);
      const float4 b = *reinterpret_cast<const float4*>(Sin + p * kN + k8 * 8 + 4);
      const float f[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
      uint16_t hi[8], lo[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) split_bf16(f[q], hi[q], lo[q]);
      *reinterpret_cast<uint4*>(sSh + sw_chunk(p, k8, 64)) = *reinterpret_cast<const uint4*>(hi);
      *reinterpret_cast<uint4*>(sSl + sw_chunk(p, k8, 64)) = *reinterpret_cast<const uint4*>(lo);
    }
    __syncthreads();
    const float2 cum_t = tt < cp.n ? cums[tt] : make_float2(0.f, 0.f);
    const int tlim = tt < cp.n ? tt : -1;
    for (int half = 0; half < KS / 128; ++half) {
      // P for sources [128 half, +128): warps 0-3 take 32-blocks 0, 1 and
      // warps 4-7 blocks 2, 3 of the half, each for its own row.  For s <= t
      // the exponent cum_t - cum_s is <= 0 (cum never increases), so exp
      // cannot overflow; entries above the diagonal are zero without exp.
#pragma unroll 1
      for (int bb = 0; bb < 2; ++bb) {
        const int sb = colhalf * 2 + bb;            // 32-block inside the half
        const int s0 = half * 128 + sb * 32;
        uint32_t r[32];
        tmem_ld_32x32b_x32(lane_base + COL_G + (uint32_t)s0, r);
        tmem_ld_wait();
        uint16_t hi[32], lo[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const int s = s0 + j;
          const float2 cs = cums[s];
          const float v =
              (s <= tlim) ? __uint_as_float(r[j]) * __expf((cum_t.x - cs.x) + (cum_t.y - cs.y)) * dts[s] : 0.f;
          split_bf16(v, hi[j], lo[j]);
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          *reinterpret_cast<uint4*>(sPh + sw_chunk(row, sb * 4 + q, 128)) = *reinterpret_cast<const uint4*>(hi + 8 * q);
          *reinterpret_cast<uint4*>(sPl + sw_chunk(row, sb * 4 + q, 128)) = *reinterpret_cast<const uint4*>(lo + 8 * q);
        }
      }
      fence_async_smem();
      tc_fence_before();
      __syncthreads();
      if (tid == 0) {
        tc_fence_after();
        const uint32_t ph0 = smem_u32(sPh), pl0 = smem_u32(sPl), x0 = smem_u32(sXT);
#pragma unroll
        for (int a = 0; a < 2; ++a)
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint64_t xd = desc_kmajor_sw128(x0 + (half * 2 + a) * 64 * 128) + 2 * j;
            mma_f16(tmem + COL_YD, desc_kmajor_sw128(ph0 + a * 128 * 128) + 2 * j, xd, IDESC_Y,
                    (half | a | j) != 0);
            mma_f16(tmem + COL_YD, desc_kmajor_sw128(pl0 + a * 128 * 128) + 2 * j, xd, IDESC_Y, 1u);
          }
        if (half == 0) {
          const uint32_t c0 = smem_u32(sC), sh0 = smem_u32(sSh), sl0 = smem_u32(sSl);
#pragma unroll
          for (int a = 0; a < 2; ++a)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const uint64_t cd = desc_kmajor_sw128(c0 + a * 128 * 128) + 2 * j;
              mma_f16(tmem + COL_YO, cd, desc_kmajor_sw128(sh0 + a * 64 * 128) + 2 * j, IDESC_Y, (a | j) != 0);
              mma_f16(tmem + COL_YO, cd, desc_kmajor_sw128(sl0 + a * 64 * 128) + 2 * j, IDESC_Y, 1u);
            }
        }
        mma_commit(&bar[1]);
      }
      __syncwarp();
      ok = wait_or_flag(&bar[1], ph, err) && ok;   // P buffers free again, accumulators final
      ph ^= 1u;
      tc_fence_after();
    }
    // y = Y_diag + exp(cum_t) Y_off + D x; warps 0-3 write p < 32, warps 4-7 p >= 32
    {
      const float et = expf(cum_t.x + cum_t.y);
      const float Dh = Dp[h];
      uint32_t rd[32], ro[32];
      tmem_ld_32x32b_x32(lane_base + COL_YD + (uint32_t)(colhalf * 32), rd);
      tmem_ld_32x32b_x32(lane_base + COL_YO + (uint32_t)(colhalf * 32), ro);
      tmem_ld_wait();
      if (ok && tt < cp.n) {
        const uint16_t* xr = u + (size_t)(cp.t0 + tt) * kConv + h * kP + colhalf * 32;
        uint16_t* yr = y + (size_t)(cp.t0 + tt) * kI + h * kP + colhalf * 32;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint4 xv = *reinterpret_cast<const uint4*>(xr + q * 8);
          uint32_t o[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int j = q * 8 + 2 * e;
            const float a = __uint_as_float(rd[j]) + et * __uint_as_float(ro[j]) + Dh * bfbits2f(h16(xv, 2 * e));
            const float b =
                __uint_as_float(rd[j + 1]) + et * __uint_as_float(ro[j + 1]) + Dh * bfbits2f(h16(xv, 2 * e + 1));
            o[e] = bf2(a, b);
          }
          *reinterpret_cast<uint4*>(yr + q * 8) = make_uint4(o[0], o[1], o[2], o[3]);
        }
      }
    }
    tc_fence_before();
    __syncthreads();
  }
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------
// launchers
// ---------------------------------------------------------------------------
static size_t state_smem() { return 1024 + (128 * 256 + 2 * 64 * 256) * 2 + kChunk * 4 + 64; }
static size_t scan_smem() {
  return 1024 + (128 * 128 + 256 * 128 + 64 * 256 + 2 * 64 * 128) * 2 + 3 * kChunk * 4 + 64;
}

cudaError_t launch_ssd_chunk_state_tc(const uint16_t* u, const float* dt, const float2* cum, const SeqInfo& si,
                                      float* states, int* err, cudaStream_t st) {
  cudaError_t e = ensure_smem_optin(reinterpret_cast<const void*>(k_ssd_state_tc), (int)state_smem());
  if (e != cudaSuccess) return e;
  return launch_pdl(k_ssd_state_tc, dim3(si.total_chunks, kG), dim3(kThr), state_smem(), st, u, dt, cum, si, states,
                    err);
}

cudaError_t launch_ssd_chunk_scan_tc(const uint16_t* u, const float* dt, const float2* cum, const float* states,
                                     const BlockParams& bp, const SeqInfo& si, uint16_t* y, int* err,
                                     cudaStream_t st) {
  cudaError_t e = ensure_smem_optin(reinterpret_cast<const void*>(k_ssd_scan_tc), (int)scan_smem());
  if (e != cudaSuccess) return e;
  return launch_pdl(k_ssd_scan_tc, dim3(si.total_chunks, kG, 2), dim3(kThr), scan_smem(), st, u, dt, cum, states,
                    bp.D, si, y, err);
}

}  // namespace m2
