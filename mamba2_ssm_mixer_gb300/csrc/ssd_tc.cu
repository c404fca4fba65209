// Tensor-core (tcgen05, bf16 operands, f32 accumulation in TMEM) stages of the
// prefill SSD scan (Mamba2ChunkScan of vllm.cpp PR #1288, "What it does"; SSD
// block decomposition of Dao & Gu 2024):
//
// k_ssd_state_tc  one CTA per (chunk, group), 8 warps: for each of the group's
//   8 heads  S_c[n, p] = sum_t B[t, n] (w_t x[t, p]),  w_t = exp(cum_last - cum_t) dt_t,
//   a 128 x 64 x 256 MMA.  w x is split into a bf16 high part and a bf16
//   remainder (two MMAs) so the chunk state keeps ~16 bits.  Staging of head
//   h + 1 overlaps the MMA of head h (double-buffered operands and TMEM).  It
//   also writes each head's x^T tile exactly as the scan's MMA reads it from
//   shared memory, so the scan fetches it with one bulk copy.
// k_ssd_scan_tc   one CTA per (chunk, group, 128-row half of the chunk),
//   warp-specialised: warp 0 loads (TMA for the C and B tiles, bulk copies of
//   the per-head x^T image, S_in image and cum/dt record, one head ahead);
//   warp 1 issues the MMAs; warps 2-9 build P and run the epilogue.
//     G = C B^T                      once per CTA (128 x 256 x 128)
//     P[t, s] = G[t, s] exp(cum_t - cum_s) dt_s   (s <= t, else 0)
//     Y_diag = P x,  Y_off = C S_in^T,  y = Y_diag + exp(cum_t) Y_off + D x
//   P and S_in are split into bf16 high part + remainder (a single bf16
//   rounding of P gives y a ~1e-3 relative error, enough to flip e4m3 codes of
//   the out_proj input downstream).  P is produced in 32-source blocks into a
//   double buffer that the MMA warp consumes; the Y accumulators are
//   double-buffered in TMEM so head h's epilogue overlaps head h+1's MMAs.
// Every wait is bounded; a wait that runs out raises the device error word and
// a CTA-wide abort flag that makes the remaining waits return at once.
#include <cudaTypedefs.h>

#include "launch_util.h"
#include "m2_kernels.h"
#include "tc_ptx.cuh"

namespace m2 {

using namespace tc;

namespace {

// Byte offset of the 16-byte chunk holding elements [k8*8, k8*8 + 8) of row r
// in a K-major bf16 operand tile of `rows` rows (64 elements per 128-byte
// swizzle atom; atoms along K are rows*128 bytes apart).
__device__ __forceinline__ uint32_t sw_chunk(int r, int k8, int rows) {
  const int a = k8 >> 3, c = k8 & 7;
  return (uint32_t)(a * rows * 128 + (r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4));
}

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

// Bounded wait; a wait that runs out flags the device error word and the CTA's
// abort flag, after which every wait returns false at once.
__device__ __forceinline__ bool wait_ab(uint64_t* bar, uint32_t parity, volatile int* abort, int* err) {
  if (mbar_wait(bar, parity, abort)) return true;
  if (!*abort) {
    *abort = 1;
    if (err) atomicOr(err, kErrTimeout);
  }
  return false;
}

__device__ __forceinline__ void split_bf16(float v, uint16_t& hi, uint16_t& lo) {
  hi = f2bfbits(v);
  lo = f2bfbits(v - bfbits2f(hi));
}

}  // namespace

// ---------------------------------------------------------------------------
// chunk states
// ---------------------------------------------------------------------------
constexpr int kStThr = 256;
constexpr int kWBuf = 2 * 64 * 256 * 2;   // one operand buffer: hi + lo [64 p][256 t]

__global__ void __launch_bounds__(kStThr, 1)
    k_ssd_state_tc(const uint16_t* __restrict__ u, const CumDt* __restrict__ cumdt, const SeqInfo si,
                   float* __restrict__ states, uint8_t* __restrict__ xt_img, int* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sBT = smem;                       // [128 n][256 t]   64 KB
  uint8_t* sW = sBT + 128 * 256 * 2;         // [2 buffers] x (hi, lo)   2 x 64 KB
  float* wts = reinterpret_cast<float*>(sW + 2 * kWBuf);    // [2][256]
  uint64_t* bar = reinterpret_cast<uint64_t*>(wts + 2 * kChunk);   // [2]
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bar + 2);
  int* abortp = reinterpret_cast<int*>(tslot + 1);
  volatile int* abort = abortp;

  const int c = blockIdx.x, g = blockIdx.y, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int quarter = warp & 3, side = warp >> 2;
  const ChunkPos cp = chunk_of(si, c);
  constexpr uint32_t IDESC = idesc_f32acc(128, 64, 1u);   // bf16 x bf16 -> f32, M = 128 (n), N = 64 (p)

  if (tid == 0) {
    mbar_init(&bar[0], 1);
    mbar_init(&bar[1], 1);
    *abortp = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(tslot, 128);
    tc_fence_before();
  }
  pdl_wait();
  pdl_trigger();
  // B^T: rows n, K = t.  8 x 8 blocks: 32 (t) x 16 (n) = 512 blocks.
  for (int blk = tid; blk < 512; blk += kStThr) {
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

  // read the accumulator of head hd and write its chunk state
  auto epilogue = [&](int hd) {
    const int k = hd & 1;
    const bool ok = wait_ab(&bar[k], (hd >> 1) & 1, abort, err);
    tc_fence_after();
    // D[n = 32 quarter + lane][p] -> states[c][h][p][n]; warps 0-3 take p < 32,
    // warps 4-7 p >= 32
    float* out = states + ((size_t)c * kNH + g * kHPG + hd) * (kP * kN) + quarter * 32 + lane;
    uint32_t r[32];
    tmem_ld_32x32b_x32(tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(k * 64 + side * 32), r);
    tmem_ld_wait();
    if (ok) {
#pragma unroll
      for (int j = 0; j < 32; ++j) out[(size_t)(side * 32 + j) * kN] = __uint_as_float(r[j]);
    }
    tc_fence_before();
  };

  for (int hh = 0; hh < kHPG; ++hh) {
    const int h = g * kHPG + hh, k = hh & 1;
    uint8_t* sWh = sW + k * kWBuf;
    uint8_t* sWl = sWh + kWBuf / 2;
    float* w = wts + k * kChunk;
    const CumDt* cd = cumdt + ((size_t)c * kNH + h) * kChunk;
    const CumDt cl = cd[cp.n - 1];
    for (int t = tid; t < kChunk; t += kStThr) {
      const CumDt ct = cd[t];
      w[t] = t < cp.n ? expf((cl.hi - ct.hi) + (cl.lo - ct.lo)) * ct.dt : 0.f;
    }
    __syncthreads();
    // x^T (rows p, K = t): written to the scan's image as is, and scaled by w
    // into the hi / lo operands here.  32 (t) x 8 (p) blocks of 8 x 8.
    uint8_t* img = xt_img + ((size_t)c * kNH + h) * kXtImageBytes;
    for (int blk = tid; blk < 256; blk += kStThr) {
      const int tb = blk >> 3, pb = blk & 7;
      uint4 in[8], out[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int t = tb * 8 + i;
        in[i] = t < cp.n ? *reinterpret_cast<const uint4*>(u + (size_t)(cp.t0 + t) * kConv + h * kP + pb * 8)
                         : make_uint4(0, 0, 0, 0);
      }
      transpose8(in, out);
      float wv[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) wv[i] = w[tb * 8 + i];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const uint32_t off = sw_chunk(pb * 8 + j, tb, 64);
        *reinterpret_cast<uint4*>(img + off) = out[j];
        uint16_t hi[8], lo[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) split_bf16(wv[i] * bfbits2f(h16(out[j], i)), hi[i], lo[i]);
        *reinterpret_cast<uint4*>(sWh + off) = *reinterpret_cast<const uint4*>(hi);
        *reinterpret_cast<uint4*>(sWl + off) = *reinterpret_cast<const uint4*>(lo);
      }
    }
    fence_proxy_async_smem();
    __syncthreads();
    if (tid == 0) {
      tc_fence_after();
      const uint32_t a0 = smem_u32(sBT), h0 = smem_u32(sWh), l0 = smem_u32(sWl);
      const uint32_t d = tmem + (uint32_t)(k * 64);
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint64_t ad = desc_kmajor_sw128(a0 + a * 128 * 128) + 2 * j;
          mma_f16(d, ad, desc_kmajor_sw128(h0 + a * 64 * 128) + 2 * j, IDESC, (a | j) != 0);
          mma_f16(d, ad, desc_kmajor_sw128(l0 + a * 64 * 128) + 2 * j, IDESC, 1u);
        }
      mma_commit(&bar[k]);
    }
    __syncwarp();
    if (hh > 0) epilogue(hh - 1);   // overlaps the MMA just issued
  }
  epilogue(kHPG - 1);
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 128);
  }
}

// ---------------------------------------------------------------------------
// chunk scan
// ---------------------------------------------------------------------------
constexpr int kScThr = 320;   // warp 0 loads, warp 1 MMA, warps 2-9 P + epilogue
constexpr int kScP = 256;     // P / epilogue threads

// shared-memory map (bytes from the 1024-aligned base)
constexpr int kSmC = 0;                // C   [128 t][128 n]                 32 KB
constexpr int kSmB = 32 * 1024;        // B   [KS s][128 n] 64 KB; after G: operand buffer 1
constexpr int kSmOp0 = 96 * 1024;      // operand buffer 0: x^T 32 KB + S_in hi/lo 32 KB
constexpr int kSmP = 160 * 1024;       // P   hi atom [128][64] 16 KB + lo atom 16 KB
constexpr int kSmCD = 192 * 1024;      // CumDt [2][256]                     8 KB
constexpr int kSmBar = 200 * 1024;     // barriers
constexpr int kScanSmem = kSmBar + 256 + 1024;

struct ScanBars {
  uint64_t cb, g, drain;
  uint64_t op_full[2], op_empty[2];
  uint64_t p_full[2], p_empty[2];
  uint64_t y_full[2], y_empty[2];
  uint32_t tslot;
  int abort;
};

__global__ void __launch_bounds__(kScThr, 1)
    k_ssd_scan_tc(const __grid_constant__ CUtensorMap tm_u, const uint16_t* __restrict__ u,
                  const CumDt* __restrict__ cumdt, const uint8_t* __restrict__ xt_img,
                  const uint8_t* __restrict__ sin_img, const float* __restrict__ Dp, const SeqInfo si,
                  uint16_t* __restrict__ y, int* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  ScanBars* sb = reinterpret_cast<ScanBars*>(smem + kSmBar);
  volatile int* abort = &sb->abort;

  const int c = blockIdx.x, g = blockIdx.y, tb = blockIdx.z, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const ChunkPos cp = chunk_of(si, c);
  if (tb * 128 >= cp.n) return;
  const int KS = (tb + 1) * 128;       // sources s < KS (causal)
  const int NBLK = KS / 32;            // 32-source P blocks per head
  constexpr uint32_t TMEM_COLS = 512;  // G [0, 256); Y_diag[k] at 256 + 128 k, Y_off[k] at 320 + 128 k
  constexpr uint32_t IDESC_Y = idesc_f32acc(128, 64, 1u);

  if (tid == 0) {
    mbar_init(&sb->cb, 1);
    mbar_init(&sb->g, 1);
    mbar_init(&sb->drain, 1);
    for (int k = 0; k < 2; ++k) {
      mbar_init(&sb->op_full[k], 1);
      mbar_init(&sb->op_empty[k], 2);   // MMA commit + the P side
      mbar_init(&sb->p_full[k], 8);     // one lane per P warp
      mbar_init(&sb->p_empty[k], 1);
      mbar_init(&sb->y_full[k], 1);
      mbar_init(&sb->y_empty[k], 8);
    }
    sb->abort = 0;
    fence_mbar_init();
    tma_prefetch(&tm_u);
  }
  if (warp == 1) {
    tmem_alloc(&sb->tslot, TMEM_COLS);
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sb->tslot;
  pdl_wait();
  pdl_trigger();

  const size_t ch0 = (size_t)c * kNH + g * kHPG;   // (chunk, first head of the group)

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------ loads
      // C (rows of this half) and B (rows 0..KS-1): two 64-column atoms each
      mbar_expect_tx(&sb->cb, (uint32_t)(128 * 128 * 2 + KS * 128 * 2));
      for (int a = 0; a < 2; ++a) {
        tma_load_2d(smem + kSmC + a * 128 * 128, &tm_u, &sb->cb, kOffC + g * kN + a * 64, cp.t0 + tb * 128);
        for (int rb = 0; rb < KS / 128; ++rb)
          tma_load_2d(smem + kSmB + a * KS * 128 + rb * 128 * 128, &tm_u, &sb->cb, kOffB + g * kN + a * 64,
                      cp.t0 + rb * 128);
      }
      const uint32_t xt_bytes = (uint32_t)(KS / 64) * (64 * 128);
      bool issued[2] = {false, false};
      uint32_t issued_par[2] = {0, 0};
      for (int hh = 0; hh < kHPG; ++hh) {
        const int k = hh & 1;
        if (hh == 1 && !wait_ab(&sb->g, 0, abort, err)) break;   // buffer 1 is the B tile's memory
        if (!wait_ab(&sb->op_empty[k], ((hh >> 1) & 1) ^ 1u, abort, err)) break;
        uint8_t* ob = smem + (k == 0 ? kSmOp0 : kSmB);
        mbar_expect_tx(&sb->op_full[k], xt_bytes + (uint32_t)kSinImageBytes + (uint32_t)(kChunk * sizeof(CumDt)));
        bulk_g2s(ob, xt_img + (ch0 + hh) * kXtImageBytes, xt_bytes, &sb->op_full[k]);
        bulk_g2s(ob + 32 * 1024, sin_img + (ch0 + hh) * kSinImageBytes, kSinImageBytes, &sb->op_full[k]);
        bulk_g2s(smem + kSmCD + k * 4096, cumdt + (ch0 + hh) * kChunk, kChunk * sizeof(CumDt), &sb->op_full[k]);
        issued[k] = true;
        issued_par[k] = (hh >> 1) & 1;
      }
      if (*abort) {   // let copies in flight land before the CTA can exit
        mbar_wait(&sb->cb, 0, nullptr, 100000000ull);
        for (int k = 0; k < 2; ++k)
          if (issued[k]) mbar_wait(&sb->op_full[k], issued_par[k], nullptr, 100000000ull);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------ MMA issuer
      if (wait_ab(&sb->cb, 0, abort, err)) {
        tc_fence_after();
        const uint32_t idesc_g = idesc_f32acc(128, KS, 1u);
        const uint32_t c0 = smem_u32(smem + kSmC), b0 = smem_u32(smem + kSmB);
#pragma unroll
        for (int a = 0; a < 2; ++a)
#pragma unroll
          for (int j = 0; j < 4; ++j)
            mma_f16(tmem, desc_kmajor_sw128(c0 + a * 128 * 128) + 2 * j,
                    desc_kmajor_sw128(b0 + a * KS * 128) + 2 * j, idesc_g, (a | j) != 0);
        mma_commit(&sb->g);
      }
      int pb = 0;   // P blocks consumed so far (buffer pb & 1, use pb >> 1)
      for (int hh = 0; hh < kHPG && !*abort; ++hh) {
        const int k = hh & 1;
        if (!wait_ab(&sb->op_full[k], (hh >> 1) & 1, abort, err)) break;
        if (!wait_ab(&sb->y_empty[k], ((hh >> 1) & 1) ^ 1u, abort, err)) break;
        tc_fence_after();
        const uint32_t yd = tmem + 256 + 128 * k, yo = yd + 64;
        uint8_t* ob = smem + (k == 0 ? kSmOp0 : kSmB);
        const uint32_t x0 = smem_u32(ob), sh0 = smem_u32(ob + 32 * 1024), sl0 = sh0 + 16 * 1024;
        const uint32_t c0 = smem_u32(smem + kSmC);
#pragma unroll
        for (int a = 0; a < 2; ++a)
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint64_t cd = desc_kmajor_sw128(c0 + a * 128 * 128) + 2 * j;
            mma_f16(yo, cd, desc_kmajor_sw128(sh0 + a * 64 * 128) + 2 * j, IDESC_Y, (a | j) != 0);
            mma_f16(yo, cd, desc_kmajor_sw128(sl0 + a * 64 * 128) + 2 * j, IDESC_Y, 1u);
          }
        const uint32_t ph0 = smem_u32(smem + kSmP), pl0 = ph0 + 16 * 1024;
        bool ok = true;
        for (int j = 0; j < NBLK; ++j, ++pb) {
          const int b = pb & 1;
          if (!wait_ab(&sb->p_full[b], (pb >> 1) & 1, abort, err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          // block j: sources [32 j, 32 j + 32) = half (j & 1) of x^T atom j / 2;
          // P block b = half b of the P atoms
#pragma unroll
          for (int kk = 0; kk < 2; ++kk) {
            const uint64_t xd = desc_kmajor_sw128(x0 + (j >> 1) * 64 * 128) + (uint64_t)((j & 1) * 4 + kk * 2);
            const uint64_t pofs = (uint64_t)(b * 4 + kk * 2);
            mma_f16(yd, desc_kmajor_sw128(ph0) + pofs, xd, IDESC_Y, (j | kk) != 0);
            mma_f16(yd, desc_kmajor_sw128(pl0) + pofs, xd, IDESC_Y, 1u);
          }
          mma_commit(&sb->p_empty[b]);
        }
        if (!ok) break;
        mma_commit(&sb->op_empty[k]);
        mma_commit(&sb->y_full[k]);
      }
      if (*abort) {
        mma_commit(&sb->drain);
        mbar_wait(&sb->drain, 0, nullptr, 100000000ull);
      }
    }
  } else {
    // ------------------------------------------------ P and epilogue (warps 2..9)
    const int pw = warp - 2;                 // 0..7
    const int quarter = warp & 3;            // TMEM lane quarter this warp may access
    const int side = pw >> 2;                // P: 16-source half of each block; epilogue: 32-column half of p
    const int row = quarter * 32 + lane;     // row of the tile = TMEM lane
    const int tt = tb * 128 + row;           // chunk-local token of that row
    const int tlim = tt < cp.n ? tt : -1;
    const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
    uint8_t* sPh = smem + kSmP;
    uint8_t* sPl = sPh + 16 * 1024;
    bool ok = wait_ab(&sb->g, 0, abort, err);
    tc_fence_after();
    int pb = 0;
    for (int hh = 0; hh < kHPG; ++hh) {
      const int h = g * kHPG + hh, k = hh & 1;
      ok = wait_ab(&sb->op_full[k], (hh >> 1) & 1, abort, err) && ok;
      const CumDt* cd = reinterpret_cast<const CumDt*>(smem + kSmCD + k * 4096);
      const CumDt ct = tt < cp.n ? cd[tt] : CumDt{0.f, 0.f, 0.f, 0.f};
      for (int j = 0; j < NBLK; ++j, ++pb) {
        const int b = pb & 1;
        ok = wait_ab(&sb->p_empty[b], ((pb >> 1) & 1) ^ 1u, abort, err) && ok;
        tc_fence_after();
        const int s0 = j * 32 + side * 16;
        uint32_t r[16];
        tmem_ld_32x32b_x16(lane_base + (uint32_t)s0, r);
        tmem_ld_wait();
        uint16_t hi[16], lo[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int s = s0 + e;
          float v = 0.f;
          if (s <= tlim) {
            const CumDt cs = cd[s];
            v = __uint_as_float(r[e]) * __expf((ct.hi - cs.hi) + (ct.lo - cs.lo)) * cs.dt;
          }
          split_bf16(v, hi[e], lo[e]);
        }
        // 16 sources = two 16-byte chunks: chunk index inside the 64-source
        // atom row is b * 4 + side * 2 (+1)
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const uint32_t off = sw_chunk(row, b * 4 + side * 2 + q, 128);
          *reinterpret_cast<uint4*>(sPh + off) = *reinterpret_cast<const uint4*>(hi + 8 * q);
          *reinterpret_cast<uint4*>(sPl + off) = *reinterpret_cast<const uint4*>(lo + 8 * q);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sb->p_full[b]);
      }
      // epilogue of head hh: y = Y_diag + exp(cum_t) Y_off + D x
      ok = wait_ab(&sb->y_full[k], (hh >> 1) & 1, abort, err) && ok;
      tc_fence_after();
      {
        const float et = expf(ct.hi + ct.lo);
        const float Dh = Dp[h];
        uint32_t rd[32], ro[32];
        tmem_ld_32x32b_x32(lane_base + 256 + 128 * k + (uint32_t)(side * 32), rd);
        tmem_ld_32x32b_x32(lane_base + 320 + 128 * k + (uint32_t)(side * 32), ro);
        tmem_ld_wait();
        if (ok && tt < cp.n) {
          const uint16_t* xr = u + (size_t)(cp.t0 + tt) * kConv + h * kP + side * 32;
          uint16_t* yr = y + (size_t)(cp.t0 + tt) * kI + h * kP + side * 32;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const uint4 xv = *reinterpret_cast<const uint4*>(xr + q * 8);
            uint32_t o[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int jj = q * 8 + 2 * e;
              const float a =
                  __uint_as_float(rd[jj]) + et * __uint_as_float(ro[jj]) + Dh * bfbits2f(h16(xv, 2 * e));
              const float bb = __uint_as_float(rd[jj + 1]) + et * __uint_as_float(ro[jj + 1]) +
                               Dh * bfbits2f(h16(xv, 2 * e + 1));
              o[e] = bf2(a, bb);
            }
            *reinterpret_cast<uint4*>(yr + q * 8) = make_uint4(o[0], o[1], o[2], o[3]);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sb->y_empty[k]);
      // this side no longer reads the operand buffer's cum/dt record
      asm volatile("bar.sync 1, %0;" ::"n"(kScP) : "memory");
      if (pw == 0 && lane == 0) mbar_arrive(&sb->op_empty[k]);
    }
  }
  __syncwarp();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------
// launchers
// ---------------------------------------------------------------------------
static size_t state_smem() { return 1024 + 128 * 256 * 2 + 2 * kWBuf + 2 * kChunk * 4 + 64; }

cudaError_t launch_ssd_chunk_state_tc(const uint16_t* u, const CumDt* cumdt, const SeqInfo& si, float* states,
                                      uint8_t* xt_img, int* err, cudaStream_t st) {
  cudaError_t e = ensure_smem_optin(reinterpret_cast<const void*>(k_ssd_state_tc), (int)state_smem());
  if (e != cudaSuccess) return e;
  return launch_pdl(k_ssd_state_tc, dim3(si.total_chunks, kG), dim3(kStThr), state_smem(), st, u, cumdt, si, states,
                    xt_img, err);
}

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn_ssd() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

cudaError_t launch_ssd_chunk_scan_tc(const uint16_t* u, const CumDt* cumdt, const uint8_t* xt_img,
                                     const uint8_t* sin_img, const BlockParams& bp, const SeqInfo& si, uint16_t* y,
                                     int* err, cudaStream_t st) {
  // u [T, 6144] bf16 as a 2-D tensor: 64-column (128-byte) x 128-row boxes,
  // 128-byte swizzle, rows past T read as zeros
  auto fn = encode_fn_ssd();
  if (!fn) return cudaErrorNotSupported;
  CUtensorMap tm;
  cuuint64_t dims[2] = {(cuuint64_t)kConv, (cuuint64_t)si.total_tokens};
  cuuint64_t strides[1] = {(cuuint64_t)kConv * 2};
  cuuint32_t box[2] = {64, 128};
  cuuint32_t estr[2] = {1, 1};
  if (fn(&tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(u), dims, strides, box, estr,
         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  cudaError_t e = ensure_smem_optin(reinterpret_cast<const void*>(k_ssd_scan_tc), kScanSmem);
  if (e != cudaSuccess) return e;
  return launch_pdl(k_ssd_scan_tc, dim3(si.total_chunks, kG, 2), dim3(kScThr), (size_t)kScanSmem, st, tm, u, cumdt,
                    xt_img, sin_img, bp.D, si, y, err);
}

}  // namespace m2
