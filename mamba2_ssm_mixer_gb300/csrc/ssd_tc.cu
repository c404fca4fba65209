// Tensor-core (tcgen05, bf16 operands, f32 accumulation in TMEM) stages of the
// prefill SSD scan (Mamba2ChunkScan of vllm.cpp PR #1288, "What it does"; SSD
// block decomposition of Dao & Gu 2024):
//
// k_ssd_state_tc  one CTA per (chunk, group): a loader warp brings the B tile
//   and, one head ahead, each head's x tile in by TMA; both stay in the layout
//   TMA writes ([tokens][64 columns], 128-byte swizzle) and feed the MMA as
//   MN-major operands, so nothing is transposed.  For each of the group's 8
//   heads, S_c[n, p] = sum_t B[t, n] (w_t x[t, p]) with
//   w_t = exp(cum_last - cum_t) dt_t is a 128 x 64 x 256 MMA; worker thread t
//   scales its token row by w_t and splits it into a bf16 high part and a bf16
//   remainder (two MMAs) so the chunk state keeps ~16 bits.  A dedicated MMA
//   warp issues each head's MMAs once all worker warps have staged it, so
//   head h's MMAs run during head h+1's staging and head h-1's epilogue.
// k_ssd_scan_tc   one CTA per (128-row half of the chunk, chunk, group),
//   warp-specialised: warp 0 loads (TMA for the C, B and per-head x tiles,
//   bulk copies of the cum/dt record and S_in image, one head ahead); warp 1
//   issues the MMAs; warps 2-9 build P and run the epilogue.
//     G = C B^T                      once per CTA (128 x 256 x 128)
//     P[t, s] = G[t, s] exp(cum_t - cum_s) dt_s  (s < t),  G[t, t] dt_t + D  (s = t),  0  (s > t)
//     Y_diag = P x,  Y_off = C S_in^T,  y = Y_diag + exp(cum_t) Y_off
//   (D x rides on P's diagonal).  P and S_in are split into bf16 high part +
//   remainder (a single bf16 rounding of P gives y a ~1e-3 relative error,
//   enough to flip e4m3 codes of the out_proj input downstream).  P is
//   produced in 32-source blocks into a 4-slot ring that the MMA warp
//   consumes; x is the MMA's N-major operand as TMA wrote it; the Y
//   accumulators are double-buffered in TMEM and each head's epilogue runs
//   after the next head's P blocks, when its MMAs have long finished.
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

__device__ __forceinline__ uint32_t bf2(float a, float b) { return pack_bf16x2(a, b); }

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
  if (mbar_wait_sleep(bar, parity, abort)) return true;
  if (!*abort) {
    *abort = 1;
    if (err) atomicOr(err, kErrTimeout);
  }
  return false;
}

// Packed pairs of floats (the sm_100 family's f32x2 arithmetic): element 0
// in the low word.
__device__ __forceinline__ uint64_t pk2(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
// Two packed floats v -> bf16x2 high parts hi (v truncated to its top 16
// bits) and bf16x2 remainders lo = bf16(v - hi); v - hi is exact, so
// |v - (hi + lo)| <= 2^-9 |v - hi| < 2^-16 |v|.  Element 0 in the low half.
__device__ __forceinline__ void split2t(uint64_t v, uint32_t& hi, uint32_t& lo) {
  uint64_t r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(v), "l"(v & 0xFFFF0000FFFF0000ull));
  uint32_t v0, v1;
  asm("mov.b64 {%0, %1}, %2;" : "=r"(v0), "=r"(v1) : "l"(v));
  asm("prmt.b32 %0, %1, %2, 0x7632;" : "=r"(hi) : "r"(v0), "r"(v1));
  float r0, r1;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r0), "=f"(r1) : "l"(r));
  lo = pack_bf16x2(r0, r1);
}

}  // namespace

// ---------------------------------------------------------------------------
// chunk states
// ---------------------------------------------------------------------------
constexpr int kStWork = 256;             // 8 worker warps; worker thread t owns token row t
constexpr int kStThr = kStWork + 64;     // + a loader warp + an MMA warp
constexpr int kStSmB = 0;                // B [2 slices of 64 n][256 t][64] as TMA writes it    64 KB
constexpr int kStSmX = 64 * 1024;        // x [2 buffers][256 t][64 p] as TMA writes it         64 KB
constexpr int kStSmW = 128 * 1024;       // w x [2 halves of 128 t] x (bf16 high, remainder) [128 t][64 p] 64 KB
constexpr int kStSmBar = 192 * 1024;
constexpr int kStSmem = kStSmBar + 128 + 1024;

struct StateBars {
  uint64_t b_full, x_full[2], x_empty[2], mma[2], drain;
  uint64_t wf[2], we[2];            // operand half staged / read by the MMAs
  uint64_t t_empty[2];              // accumulator k read
  uint32_t tslot;
  int abort;
};

// 16-byte chunk c (0..7) of row r in a 128-byte-swizzled tile with 128-byte
// rows (what TMA writes with CU_TENSOR_MAP_SWIZZLE_128B)
__device__ __forceinline__ uint32_t sw_row_chunk(int r, int c) {
  return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4));
}

// One CTA per (chunk, group): S[h][p][n] = sum_t w_t x_t[p] B_t[n] for the
// group's 8 heads, w_t = exp(cum_last - cum_t) dt_t (zero past the chunk).
// The loader TMA-loads the group's B tile once and each head's x tile into
// one of two buffers, two heads ahead.  Worker thread t scales token row t of
// x by w_t and splits it into a bf16 high part and remainder; the operand
// lives in two halves of 128 tokens, each single-buffered, so the workers of
// half j (warps 4j..4j+3) stage head h+1 there once the MMAs of head h have
// read it.  The MMA warp issues each head's 16 K-steps (two MMAs each, high
// and remainder) into one of two TMEM accumulators, the first 8 from half 0
// and the last 8 from half 1, committing each half as it is read; the
// workers drain accumulator k (head h-1) while head h's MMAs run.
__global__ void __launch_bounds__(kStThr, 1)
    k_ssd_state_tc(const __grid_constant__ CUtensorMap tm_u, const CumDt* __restrict__ cumdt, const SeqInfo si,
                   float* __restrict__ states, int* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_align<1024>(smem_raw);
  StateBars* sb = reinterpret_cast<StateBars*>(smem + kStSmBar);
  volatile int* abort = &sb->abort;
  uint8_t* sB = smem + kStSmB;

  const int c = blockIdx.x, g = blockIdx.y, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const ChunkPos cp = chunk_of(si, c);
  // bf16 x bf16 -> f32, M = 128 (n), N = 64 (p), both operands MN-major
  constexpr uint32_t IDESC = idesc_f32acc_mn(128, 64, 1u, true, true);

  if (tid == 0) {
    mbar_init(&sb->b_full, 1);
    for (int k = 0; k < 2; ++k) {
      mbar_init(&sb->x_full[k], 1);
      mbar_init(&sb->x_empty[k], kStWork / 32);
      mbar_init(&sb->mma[k], 1);
      mbar_init(&sb->wf[k], kStWork / 64);          // the 4 worker warps of a half
      mbar_init(&sb->we[k], 1);
      mbar_init(&sb->t_empty[k], kStWork / 32);
    }
    mbar_init(&sb->drain, 1);
    sb->abort = 0;
    fence_mbar_init();
    tma_prefetch(&tm_u);
  }
  if (warp == 0) {
    tmem_alloc(&sb->tslot, 128);
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sb->tslot;
  pdl_wait();
  pdl_trigger();

  if (warp == kStWork / 32) {
    // ------------------------------------------------ loader
    if (lane == 0) {
      // B: two 64-column slices of 256 rows (rows past the chunk are other
      // tokens or zeros; their products vanish because w = 0 there)
      mbar_expect_tx(&sb->b_full, 256 * 128 * 2);
      for (int a = 0; a < 2; ++a)
        tma_load_2d(sB + a * 256 * 128, &tm_u, &sb->b_full, kOffB + g * kN + a * 64, cp.t0);
      int issued[2] = {-1, -1};   // last head whose x tile went into each buffer
      for (int hh = 0; hh < kHPG; ++hh) {
        const int xb = hh & 1;
        // buffer xb is free once every worker has read head hh-2's rows
        if (!wait_ab(&sb->x_empty[xb], ((hh >> 1) & 1) ^ 1u, abort, err)) break;
        mbar_expect_tx(&sb->x_full[xb], 256 * 64 * 2);
        tma_load_2d(smem + kStSmX + xb * 32 * 1024, &tm_u, &sb->x_full[xb], (g * kHPG + hh) * kP, cp.t0);
        issued[xb] = hh;
      }
      if (*abort) {   // let copies in flight land before the CTA can exit
        mbar_wait(&sb->b_full, 0, nullptr, 100000000ull);
        for (int xb = 0; xb < 2; ++xb)
          if (issued[xb] >= 0) mbar_wait(&sb->x_full[xb], (issued[xb] >> 1) & 1, nullptr, 100000000ull);
      }
    }
  } else if (warp == kStWork / 32 + 1) {
    // ------------------------------------------------ MMA issuer
    if (lane == 0) {
      bool ok = wait_ab(&sb->b_full, 0, abort, err);
      const uint32_t b0 = smem_u32(sB);
      for (int hh = 0; hh < kHPG && ok; ++hh) {
        const int k = hh & 1;
        if (!wait_ab(&sb->t_empty[k], ((hh >> 1) & 1) ^ 1u, abort, err)) break;   // head hh-2 drained
        const uint32_t d = tmem + (uint32_t)(k * 64);
        // S[n, p] += sum_t B[t, n] (w x)[t, p]: 16 K-steps of 16 tokens (2048
        // bytes of each tile), 8 per operand half; B's two 64-column slices
        // are 32 KB apart
        for (int half = 0; half < 2 && ok; ++half) {
          ok = wait_ab(&sb->wf[half], hh & 1, abort, err);
          if (!ok) break;
          tc_fence_after();
          const uint32_t h0 = smem_u32(smem + kStSmW + half * 32 * 1024), l0 = h0 + 16 * 1024;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const int ks = half * 8 + kk;
            const uint64_t ad = desc_mnmajor_sw128(b0 + ks * 2048, 256 * 128);
            mma_f16(d, ad, desc_mnmajor_sw128(h0 + kk * 2048, 1024), IDESC, ks != 0);
            mma_f16(d, ad, desc_mnmajor_sw128(l0 + kk * 2048, 1024), IDESC, 1u);
          }
          mma_commit(&sb->we[half]);   // this half of the operand may be restaged
        }
        if (!ok) break;
        mma_commit(&sb->mma[k]);
      }
      if (*abort) {   // no MMA may still be running when TMEM is freed
        mma_commit(&sb->drain);
        mbar_wait(&sb->drain, 0, nullptr, 100000000ull);
      }
    }
  } else {
    // ------------------------------------------------ workers (8 warps)
    const int quarter = warp & 3, side = warp >> 2;
    const int t = tid, half = t >> 7, tl = t & 127;   // token row t = row tl of operand half `half`
    const CumDt* cd0 = cumdt + (size_t)c * kNH + g * kHPG;
    // this head's cum_t, cum_last and dt_t; the next head's are fetched one head ahead
    float ct_hi = cd0->hi[t], ct_lo = cd0->lo[t], ct_dt = cd0->dt[t];
    float cl_hi = cd0->hi[cp.n - 1], cl_lo = cd0->lo[cp.n - 1];
    bool ok = wait_ab(&sb->b_full, 0, abort, err);
    uint8_t* sWh = smem + kStSmW + half * 32 * 1024;
    uint8_t* sWl = sWh + 16 * 1024;

    auto epilogue = [&](int hd) {
      const int k = hd & 1;
      const bool okm = wait_ab(&sb->mma[k], (hd >> 1) & 1, abort, err);
      tc_fence_after();
      // D[n = 32 quarter + lane][p] -> states[c][h][p][n]; warps 0-3 take p < 32,
      // warps 4-7 p >= 32
      float* out = states + ((size_t)c * kNH + g * kHPG + hd) * (kP * kN) + quarter * 32 + lane;
      uint32_t r[32];
      tmem_ld_32x32b_x32(tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(k * 64 + side * 32), r);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sb->t_empty[k]);   // accumulator k may be overwritten
      if (ok && okm) {
#pragma unroll
        for (int j = 0; j < 32; ++j) out[(size_t)(side * 32 + j) * kN] = __uint_as_float(r[j]);
      }
    };

    for (int hh = 0; hh < kHPG; ++hh) {
      const int xb = hh & 1;
      const uint8_t* sX = smem + kStSmX + xb * 32 * 1024;
      // w_t = exp(cum_last - cum_t) dt_t; zero past the chunk's end
      const float w = t < cp.n ? expf((cl_hi - ct_hi) + (cl_lo - ct_lo)) * ct_dt : 0.f;
      if (hh + 1 < kHPG) {
        const CumDt* nx = cd0 + hh + 1;
        ct_hi = nx->hi[t];
        ct_lo = nx->lo[t];
        ct_dt = nx->dt[t];
        cl_hi = nx->hi[cp.n - 1];
        cl_lo = nx->lo[cp.n - 1];
      }
      ok = wait_ab(&sb->x_full[xb], (hh >> 1) & 1, abort, err) && ok;
      uint4 xv[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) xv[q] = *reinterpret_cast<const uint4*>(sX + sw_row_chunk(t, q));
      __syncwarp();
      if (lane == 0) mbar_arrive(&sb->x_empty[xb]);   // this warp's reads of x buffer xb are done
      // row t of (w x), bf16 high part and remainder, in the x tile's own
      // layout, into operand half `half` once head hh-1's MMAs have read it
      const uint64_t w2 = pk2(w, w);
      uint32_t hi[8][4], lo[8][4];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const uint32_t wd[4] = {xv[q].x, xv[q].y, xv[q].z, xv[q].w};
#pragma unroll
        for (int e = 0; e < 4; ++e)
          split2t(mul2(w2, pk2(__uint_as_float(wd[e] << 16), __uint_as_float(wd[e] & 0xFFFF0000u))), hi[q][e],
                  lo[q][e]);
      }
      ok = wait_ab(&sb->we[half], (hh & 1) ^ 1u, abort, err) && ok;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const uint32_t off = sw_row_chunk(tl, q);
        *reinterpret_cast<uint4*>(sWh + off) = make_uint4(hi[q][0], hi[q][1], hi[q][2], hi[q][3]);
        *reinterpret_cast<uint4*>(sWl + off) = make_uint4(lo[q][0], lo[q][1], lo[q][2], lo[q][3]);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sb->wf[half]);   // this warp's rows of operand half `half` are staged
      // head hh-1's accumulator: its MMAs ran while this head was staged
      if (hh > 0) epilogue(hh - 1);
    }
    epilogue(kHPG - 1);
  }
  __syncwarp();
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
constexpr int kScPW = 8;      // P / epilogue warps
constexpr int kScRing = 4;    // P ring slots (32 sources each)

// shared-memory map (bytes from the 1024-aligned base)
constexpr int kSmC = 0;                 // C [128 t][128 n] K-major, two 64-column atoms   32 KB
constexpr int kSmX0 = 32 * 1024;        // x buffer 0 [256 s][64 p] as TMA writes it       32 KB
constexpr int kSmB = 64 * 1024;         // B [KS s][128 n] (G only); then x buffer 1 + S_in 64 KB
constexpr int kSmX1 = kSmB;             //   x buffer 1                                    32 KB
constexpr int kSmSin = kSmB + 32 * 1024;  // S_in hi, lo [64 p][128 n] K-major each         32 KB
constexpr int kSmP = 128 * 1024;        // P ring: hi atoms [2][128][64], lo atoms [2][128][64] 64 KB
constexpr int kSmCD = 192 * 1024;       // cum/dt records [2]                               8 KB
constexpr int kSmBar = 200 * 1024;      // barriers
constexpr int kScanSmem = kSmBar + 256 + 1024;

struct ScanBars {
  uint64_t cb, g, drain, drain_ld, sin_full, sin_empty;
  uint64_t op_full[2], op_empty[2];
  uint64_t p_full[kScRing], p_empty[kScRing];
  uint64_t y_full[2], y_empty[2];
  uint32_t tslot;
  int abort;
};

__global__ void __launch_bounds__(kScThr, 1)
    k_ssd_scan_tc(const __grid_constant__ CUtensorMap tm_u, const CumDt* __restrict__ cumdt,
                  const uint8_t* __restrict__ sin_img, const float* __restrict__ Dp, const SeqInfo si,
                  uint16_t* __restrict__ y, int* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_align<1024>(smem_raw);
  ScanBars* sb = reinterpret_cast<ScanBars*>(smem + kSmBar);
  volatile int* abort = &sb->abort;

  // the two halves of a (chunk, group) are neighbours in launch order, so the
  // second one's reads of B, x, S_in and cum/dt hit L2
  const int tb = blockIdx.x, c = blockIdx.y, g = blockIdx.z, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const ChunkPos cp = chunk_of(si, c);
  if (tb * 128 >= cp.n) return;
  const int KS = (tb + 1) * 128;       // sources s < KS (causal)
  const int NBLK = KS / 32;            // 32-source P blocks per head
  constexpr uint32_t TMEM_COLS = 512;  // G [0, 256); Y_diag[k] at 256 + 128 k, Y_off[k] at 320 + 128 k
  constexpr uint32_t IDESC_Y = idesc_f32acc(128, 64, 1u);                   // C S_in^T: both K-major
  constexpr uint32_t IDESC_PX = idesc_f32acc_mn(128, 64, 1u, false, true);  // P x: x as TMA writes it

  if (tid == 0) {
    mbar_init(&sb->cb, 1);
    mbar_init(&sb->g, 1);
    mbar_init(&sb->drain, 1);
    mbar_init(&sb->drain_ld, 1);
    mbar_init(&sb->sin_full, 1);
    mbar_init(&sb->sin_empty, 1);
    for (int k = 0; k < 2; ++k) {
      mbar_init(&sb->op_full[k], 1);
      mbar_init(&sb->op_empty[k], 1 + kScPW);   // MMA commit + each P warp
      mbar_init(&sb->y_full[k], 2);           // P x (MMA warp) and C S_in^T (load warp)
      mbar_init(&sb->y_empty[k], kScPW);
    }
    for (int k = 0; k < kScRing; ++k) {
      mbar_init(&sb->p_full[k], kScPW / 2);   // the 4 warps of one side
      mbar_init(&sb->p_empty[k], 1);
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
      int op_issued[2] = {-1, -1}, sin_issued = -1;   // last head whose copies were issued
      bool g_done = false;
      for (int hh = 0; hh < kHPG; ++hh) {
        const int k = hh & 1;
        // x tile and cum/dt record of head hh (buffer 1 is the B tile's memory)
        if (!wait_ab(&sb->op_empty[k], ((hh >> 1) & 1) ^ 1u, abort, err)) break;
        if (k == 1 && !g_done) {
          if (!wait_ab(&sb->g, 0, abort, err)) break;
          g_done = true;
        }
        mbar_expect_tx(&sb->op_full[k], (uint32_t)(KS * 128 + sizeof(CumDt)));
        uint8_t* xb = smem + (k == 0 ? kSmX0 : kSmX1);
        for (int rb = 0; rb < KS / 128; ++rb)
          tma_load_2d(xb + rb * 128 * 128, &tm_u, &sb->op_full[k], (g * kHPG + hh) * kP, cp.t0 + rb * 128);
        bulk_g2s(smem + kSmCD + k * sizeof(CumDt), cumdt + ch0 + hh, (uint32_t)sizeof(CumDt), &sb->op_full[k]);
        op_issued[k] = hh;
        // S_in of head hh: one buffer, free once head hh-1's C S_in^T MMAs are done
        if (hh == 0) {
          if (!g_done) {
            if (!wait_ab(&sb->g, 0, abort, err)) break;
            g_done = true;
          }
        } else if (!wait_ab(&sb->sin_empty, (hh - 1) & 1, abort, err)) {
          break;
        }
        mbar_expect_tx(&sb->sin_full, (uint32_t)kSinImageBytes);
        bulk_g2s(smem + kSmSin, sin_img + (ch0 + hh) * kSinImageBytes, kSinImageBytes, &sb->sin_full);
        sin_issued = hh;
        // Y_off = C S_in^T of head hh (S_in as bf16 high part + remainder),
        // issued from this warp so the MMA warp only issues P x; Y_off[k] is
        // free once head hh-2's epilogue has read it
        if (!wait_ab(&sb->cb, 0, abort, err)) break;
        if (!wait_ab(&sb->sin_full, hh & 1, abort, err)) break;
        if (!wait_ab(&sb->y_empty[k], ((hh >> 1) & 1) ^ 1u, abort, err)) break;
        tc_fence_after();
        {
          const uint64_t c_d = desc_kmajor_sw128(smem_u32(smem + kSmC));
          const uint64_t sh_d = desc_kmajor_sw128(smem_u32(smem + kSmSin));
          const uint64_t sl_d = desc_kmajor_sw128(smem_u32(smem + kSmSin + 16 * 1024));
          const uint32_t yo = tmem + 320 + 128 * k;
          // two 64-column atoms of C (16 KB apart) and of S_in (8 KB apart)
#pragma unroll
          for (int a = 0; a < 2; ++a)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const uint64_t cd = c_d + (uint64_t)(a * 1024 + 2 * j);
              const uint64_t so = (uint64_t)(a * 512 + 2 * j);
              mma_f16(yo, cd, sh_d + so, IDESC_Y, (a | j) != 0);
              mma_f16(yo, cd, sl_d + so, IDESC_Y, 1u);
            }
        }
        mma_commit(&sb->sin_empty);
        mma_commit(&sb->y_full[k]);
      }
      if (*abort) {   // no MMA of this warp may still run when TMEM is freed
        mma_commit(&sb->drain_ld);
        mbar_wait(&sb->drain_ld, 0, nullptr, 100000000ull);
      }
      if (*abort) {   // let copies in flight land before the CTA can exit
        mbar_wait(&sb->cb, 0, nullptr, 100000000ull);
        for (int k = 0; k < 2; ++k)
          if (op_issued[k] >= 0) mbar_wait(&sb->op_full[k], (op_issued[k] >> 1) & 1, nullptr, 100000000ull);
        if (sin_issued >= 0) mbar_wait(&sb->sin_full, sin_issued & 1, nullptr, 100000000ull);
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
      // descriptors: the start-address field counts 16-byte units, so moving
      // within a tile adds (bytes >> 4)
      const uint64_t ph_d = desc_kmajor_sw128(smem_u32(smem + kSmP));
      const uint64_t pl_d = desc_kmajor_sw128(smem_u32(smem + kSmP + 32 * 1024));
      const uint64_t x_d[2] = {desc_mnmajor_sw128(smem_u32(smem + kSmX0), 1024),
                               desc_mnmajor_sw128(smem_u32(smem + kSmX1), 1024)};
      int pb = 0;   // P blocks consumed so far (slot pb % 4, use pb / 4)
      for (int hh = 0; hh < kHPG && !*abort; ++hh) {
        const int k = hh & 1;
        if (!wait_ab(&sb->op_full[k], (hh >> 1) & 1, abort, err)) break;
        if (!wait_ab(&sb->y_empty[k], ((hh >> 1) & 1) ^ 1u, abort, err)) break;
        tc_fence_after();
        const uint32_t yd = tmem + 256 + 128 * k;
        const uint64_t xk = k == 0 ? x_d[0] : x_d[1];
        bool ok = true;
        for (int j = 0; j < NBLK; ++j, ++pb) {
          const int b = pb & (kScRing - 1);
          if (!wait_ab(&sb->p_full[b], (pb >> 2) & 1, abort, err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          // block j: sources [32 j, 32 j + 32) = x rows 32 j.. (4096 bytes per
          // block, 2048 per 16-source K-step); slot b = half (b & 1) of the
          // P atoms b / 2 (16 KB apart), 32 bytes per K-step
          const uint64_t xd = xk + (uint64_t)(j * 256);
          const uint64_t po = (uint64_t)((b >> 1) * 1024 + (b & 1) * 4);
          mma_f16(yd, ph_d + po, xd, IDESC_PX, j != 0);
          mma_f16(yd, pl_d + po, xd, IDESC_PX, 1u);
          mma_f16(yd, ph_d + po + 2, xd + 128, IDESC_PX, 1u);
          mma_f16(yd, pl_d + po + 2, xd + 128, IDESC_PX, 1u);
          mma_commit(&sb->p_empty[b]);
        }
        if (!ok) break;
        mma_commit(&sb->op_empty[k]);   // x(hh) is no longer read once these finish
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
    const int side = pw >> 2;                // P: blocks j = side (mod 2); epilogue: 32-column half of p
    const int row = quarter * 32 + lane;     // row of the tile = TMEM lane
    const int tt = tb * 128 + row;           // chunk-local token of that row
    const int tlim = tt < cp.n ? tt : -1;
    const int rblk = tb * 4 + quarter;       // this warp's 32-token block
    const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
    uint8_t* sPh = smem + kSmP;
    uint8_t* sPl = sPh + 32 * 1024;
    bool ok = wait_ab(&sb->g, 0, abort, err);
    tc_fence_after();
    float prev_cum = 0.f;   // cum_t of the previous head (its epilogue runs one head late)

    // y = Y_diag + exp(cum_t) Y_off for head hd (D x is folded into P's diagonal)
    auto epilogue = [&](int hd, float cum_t) {
      const int k = hd & 1;
      ok = wait_ab(&sb->y_full[k], (hd >> 1) & 1, abort, err) && ok;
      tc_fence_after();
      const float et = expf(cum_t);
      uint32_t rd[32], ro[32];
      tmem_ld_32x32b_x32(lane_base + 256 + 128 * k + (uint32_t)(side * 32), rd);
      tmem_ld_32x32b_x32(lane_base + 320 + 128 * k + (uint32_t)(side * 32), ro);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sb->y_empty[k]);
      if (ok && tt < cp.n) {
        uint16_t* yr = y + (size_t)(cp.t0 + tt) * kI + (g * kHPG + hd) * kP + side * 32;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint32_t o[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int jj = q * 8 + 2 * e;
            o[e] = bf2(__uint_as_float(rd[jj]) + et * __uint_as_float(ro[jj]),
                       __uint_as_float(rd[jj + 1]) + et * __uint_as_float(ro[jj + 1]));
          }
          *reinterpret_cast<uint4*>(yr + q * 8) = make_uint4(o[0], o[1], o[2], o[3]);
        }
      }
    };

    int pb = 0;
    for (int hh = 0; hh < kHPG; ++hh) {
      const int h = g * kHPG + hh, k = hh & 1;
      ok = wait_ab(&sb->op_full[k], (hh >> 1) & 1, abort, err) && ok;
      const CumDt* cd = reinterpret_cast<const CumDt*>(smem + kSmCD + k * sizeof(CumDt));
      const float ct_hi = tt < cp.n ? cd->hi[tt] : 0.f, ct_lo = tt < cp.n ? cd->lo[tt] : 0.f;
      const float Dh = Dp[h];
      // the two sides take alternate 32-source blocks, so each side owns ring
      // slots of one parity (NBLK is even) and 32 sources per warp and block
      for (int j = side; j < NBLK; j += 2) {
        const int pj = pb + j, b = pj & (kScRing - 1);
        ok = wait_ab(&sb->p_empty[b], ((pj >> 2) & 1) ^ 1u, abort, err) && ok;
        tc_fence_after();
        const int s0 = j * 32;
        uint32_t r[32];
        tmem_ld_32x32b_x32(lane_base + (uint32_t)s0, r);
        tmem_ld_wait();
        // The warp's 32 rows are the 32-token block rblk; relative to source
        // block j it is below the diagonal, on it, or above it (all zero).
        // Below: exp(cum_t - cum_s) = exp(cum_t - cum_e) exp(cum_e - cum_s),
        // both factors <= 1 with e the block's last source (the second, times
        // dt_s, is colf_s).  On it: one exp per element, and D on s = t.
        float v[32];
        uint32_t hi[16], lo[16];   // bf16 pairs: sources 2i, 2i+1
        if (j < rblk) {
          const int e = min(j * 32 + 31, cp.n - 1);
          const float rf = tt < cp.n ? __expf((ct_hi - cd->hi[e]) + (ct_lo - cd->lo[e])) : 0.f;
          const uint64_t rf2 = pk2(rf, rf);
          const float4* cf = reinterpret_cast<const float4*>(cd->colf + s0);
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const float4 f = cf[q];
            const uint64_t g01 = pk2(__uint_as_float(r[4 * q]), __uint_as_float(r[4 * q + 1]));
            const uint64_t g23 = pk2(__uint_as_float(r[4 * q + 2]), __uint_as_float(r[4 * q + 3]));
            split2t(mul2(g01, mul2(rf2, pk2(f.x, f.y))), hi[2 * q], lo[2 * q]);
            split2t(mul2(g23, mul2(rf2, pk2(f.z, f.w))), hi[2 * q + 1], lo[2 * q + 1]);
          }
        } else if (j == rblk && (cd->hi[s0] - cd->hi[min(s0 + 31, cp.n - 1)]) +
                                        (cd->lo[s0] - cd->lo[min(s0 + 31, cp.n - 1)]) < 60.f) {
          // On the diagonal, when the block's log-decay span is below 60: the
          // same factorisation as below it, exp(cum_t - cum_s) dt_s =
          // exp(cum_t - cum_e) colf_s, the first factor now >= 1 but at most
          // e^60 (t <= e), the second at least dt_s e^-60; then the causal
          // mask and D on s = t.  (The span is the same for the whole warp.)
          const int e = min(s0 + 31, cp.n - 1);
          const float rf = tt < cp.n ? __expf((ct_hi - cd->hi[e]) + (ct_lo - cd->lo[e])) : 0.f;
          const float4* cf = reinterpret_cast<const float4*>(cd->colf + s0);
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const float4 f = cf[q];
            const float fs[4] = {f.x, f.y, f.z, f.w};
#pragma unroll
            for (int e4 = 0; e4 < 4; ++e4) {
              const int s = s0 + 4 * q + e4;
              const float val = __uint_as_float(r[4 * q + e4]) * (rf * fs[e4]);
              v[4 * q + e4] = s <= tlim ? val + (s == tt ? Dh : 0.f) : 0.f;
            }
          }
#pragma unroll
          for (int e4 = 0; e4 < 16; ++e4) split2t(pk2(v[2 * e4], v[2 * e4 + 1]), hi[e4], lo[e4]);
        } else if (j == rblk) {
          // (a span of 60 or more) one exponential per element; s > t (or a
          // row past the chunk) selects 0, the exponential there may overflow
          // and is discarded by the select
          const float4* h4 = reinterpret_cast<const float4*>(cd->hi + s0);
          const float4* l4 = reinterpret_cast<const float4*>(cd->lo + s0);
          const float4* d4 = reinterpret_cast<const float4*>(cd->dt + s0);
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const float4 hq = h4[q], lq = l4[q], dq = d4[q];
            const float hs[4] = {hq.x, hq.y, hq.z, hq.w}, ls[4] = {lq.x, lq.y, lq.z, lq.w};
            const float ds[4] = {dq.x, dq.y, dq.z, dq.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int s = s0 + 4 * q + e;
              const float val = __uint_as_float(r[4 * q + e]) * __expf((ct_hi - hs[e]) + (ct_lo - ls[e])) * ds[e];
              v[4 * q + e] = s <= tlim ? val + (s == tt ? Dh : 0.f) : 0.f;
            }
          }
#pragma unroll
          for (int e = 0; e < 16; ++e) split2t(pk2(v[2 * e], v[2 * e + 1]), hi[e], lo[e]);
        } else {
#pragma unroll
          for (int e = 0; e < 16; ++e) hi[e] = lo[e] = 0u;
        }
        // 32 sources = the four 16-byte chunks (b & 1) * 4 + q of this row in
        // the P atoms b / 2
        const uint32_t pa = (uint32_t)(b >> 1) * 16 * 1024;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint32_t off = pa + sw_chunk(row, (b & 1) * 4 + q, 128);
          *reinterpret_cast<uint4*>(sPh + off) = make_uint4(hi[4 * q], hi[4 * q + 1], hi[4 * q + 2], hi[4 * q + 3]);
          *reinterpret_cast<uint4*>(sPl + off) = make_uint4(lo[4 * q], lo[4 * q + 1], lo[4 * q + 2], lo[4 * q + 3]);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sb->p_full[b]);
      }
      pb += NBLK;
      // this warp no longer reads head hh's cum/dt record
      __syncwarp();
      if (lane == 0) mbar_arrive(&sb->op_empty[k]);
      // head hh-1's accumulators are complete by now (its MMAs ran during this
      // head's P blocks)
      if (hh > 0) epilogue(hh - 1, prev_cum);
      prev_cum = ct_hi + ct_lo;
    }
    epilogue(kHPG - 1, prev_cum);
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

// u [T, 6144] bf16 as a 2-D tensor: 64-column (128-byte) boxes of box_rows rows,
// 128-byte swizzle, rows past T read as zeros
static cudaError_t make_u_map(CUtensorMap* tm, const uint16_t* u, int total_tokens, int box_rows) {
  auto fn = encode_fn_ssd();
  if (!fn) return cudaErrorNotSupported;
  cuuint64_t dims[2] = {(cuuint64_t)kConv, (cuuint64_t)total_tokens};
  cuuint64_t strides[1] = {(cuuint64_t)kConv * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  if (fn(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(u), dims, strides, box, estr,
         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  return cudaSuccess;
}

cudaError_t launch_ssd_chunk_state_tc(const uint16_t* u, const CumDt* cumdt, const SeqInfo& si, float* states,
                                      int* err, cudaStream_t st) {
  CUtensorMap tm;
  cudaError_t e = make_u_map(&tm, u, si.total_tokens, 256);
  if (e != cudaSuccess) return e;
  e = ensure_smem_optin(reinterpret_cast<const void*>(k_ssd_state_tc), kStSmem);
  if (e != cudaSuccess) return e;
  return launch_pdl(k_ssd_state_tc, dim3(si.total_chunks, kG), dim3(kStThr), (size_t)kStSmem, st, tm, cumdt, si,
                    states, err);
}

cudaError_t launch_ssd_chunk_scan_tc(const uint16_t* u, const CumDt* cumdt, const uint8_t* sin_img,
                                     const BlockParams& bp, const SeqInfo& si, uint16_t* y, int* err,
                                     cudaStream_t st) {
  CUtensorMap tm;
  cudaError_t e = make_u_map(&tm, u, si.total_tokens, 128);
  if (e != cudaSuccess) return e;
  e = ensure_smem_optin(reinterpret_cast<const void*>(k_ssd_scan_tc), kScanSmem);
  if (e != cudaSuccess) return e;
  return launch_pdl(k_ssd_scan_tc, dim3(2, si.total_chunks, kG), dim3(kScThr), (size_t)kScanSmem, st, tm, cumdt,
                    sin_img, bp.D, si, y, err);
}

}  // namespace m2
