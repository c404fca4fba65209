// Tensor-core GEMMs for sm_103a: y = bf16(scale * A . B^T) with operands
// stored K-major ([rows, K] row-major), f32 accumulation in TMEM.  The
// operands are e4m3 codes (W8A8, tcgen05.mma kind::f8f6f4, 32 per MMA) or
// bf16 values (the W8A16 arm, kind::f16, 16 per MMA); either way one MMA
// consumes 32 bytes of each 128-byte swizzled K-slice.
//
// k_gemm_pair (prefill, more than 256 rows): persistent two-CTA clusters,
//   each walking 256 x 256 output tiles with tcgen05.mma.cta_group::2 (each
//   SM stages 128 rows of A and half of B).  Warp roles: warp 0 issues TMA
//   loads of 128-byte-swizzled K-slices into a STAGES-deep shared-memory
//   ring, warp 1 of the even CTA issues the MMAs into one of two TMEM
//   accumulators, warps 2-5 drain the other accumulator (tcgen05.ld), scale,
//   round to bf16 and write 64-column slices through shared memory with TMA
//   stores, so the epilogue of tile i overlaps the MMAs of tile i+1.
// k_gemm_fewrow (decode, up to 128 rows): the weight matrix is the MMA's
//   128-row A operand and the few activation rows are its N operand
//   (D^T = W . X^T); the K dimension is split across the CTAs of a cluster so
//   every SM streams weights, and the partial sums are added in distributed
//   shared memory.
// k_gemm_tc_skinny (129 to 256 rows, and the allocation-free entry point):
//   the same swap-AB tiles with K split across independent CTAs; f32 partials
//   in global scratch are summed by k_splitk_reduce.
// Every mbarrier wait is bounded: a wait that runs out raises the CTA's abort
// flag and the device error word, the roles leave their loops, outstanding
// copies and MMAs are drained with bounded waits, and TMEM is freed.
#include <cudaTypedefs.h>

#include <map>
#include <mutex>

#include "gemm.h"
#include "launch_util.h"
#include "m2_common.cuh"
#include "tc_ptx.cuh"

namespace m2 {

using namespace tc;

namespace {

constexpr int kBM = 128;        // MMA M (rows of the A operand per tile)
constexpr int kBK = 128;        // K bytes per pipeline stage (one 128-byte swizzle row)

// One MMA over 32 bytes of K: 32 e4m3 codes or 16 bf16 values.
template <bool kBf16>
__device__ __forceinline__ void mma_k32b(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  if constexpr (kBf16)
    mma_f16(d_tmem, a, b, idesc, acc);
  else
    mma_f8f6f4(d_tmem, a, b, idesc, acc);
}
constexpr int kThreads = 192;   // 6 warps: producer, MMA, 4 x epilogue

struct __align__(8) Ctl {
  uint64_t full[8];
  uint64_t empty[8];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

__device__ __forceinline__ void raise_abort(Ctl* ctl, int* err) {
  *reinterpret_cast<volatile int*>(&ctl->abort) = 1;
  if (err) atomicOr(err, kErrTimeout);
}

// Output staging of the persistent kernels' epilogue: two buffers per
// epilogue warp, each 32 rows x 64 bf16 (128 bytes a row) in the 128-byte
// swizzle the output tensor map's TMA store reads.
constexpr uint32_t kEpiBuf = 32 * 128;
constexpr uint32_t kEpiBytes = 4 * 2 * kEpiBuf;

// One epilogue warp drains its 32 accumulator lanes (output rows row0 ..
// row0 + 31, this thread row0 + lane) over the tile's BN columns starting
// at TMEM column `tcol` and output column n0: y = bf16(scale * acc).
// With a store map (row stride and base 16-byte aligned) each 64-column
// slice is staged in shared memory and written by one TMA store, full
// 128-byte lines, while the warp converts the next slice; otherwise every
// thread stores its own row.  `buf` alternates the warp's two buffers; a
// buffer is reused only after the store issued from it two slices earlier
// has read it.
template <int BN>
__device__ __forceinline__ void epilogue_rows(uint32_t tcol, uint8_t* bufs, int& buf, const CUtensorMap* tmC,
                                              bool tma_store, uint16_t* __restrict__ C, int M, int N, int row0,
                                              int n0, float scale, int lane) {
  static_assert(BN % 64 == 0, "BN");
  if (tma_store) {
#pragma unroll 1
    for (int c = 0; c < BN; c += 64) {
      // a slice wholly outside the output (and every later one) is neither
      // staged nor stored: each staged buffer is followed by its store, which
      // is what the read wait below counts on (warp-uniform condition)
      if (row0 >= M || n0 + c >= N) break;
      uint32_t r0[32], r1[32];
      tmem_ld_32x32b_x32(tcol + (uint32_t)c, r0);
      tmem_ld_32x32b_x32(tcol + (uint32_t)(c + 32), r1);
      tmem_ld_wait();
      uint8_t* b = bufs + buf * kEpiBuf;
      if (lane == 0) bulk_wait_read<1>();
      __syncwarp();
      const uint32_t row_addr = smem_u32(b) + (uint32_t)lane * 128u;
#pragma unroll
      for (int j = 0; j < 8; ++j) {        // 16-byte chunk j: columns c + 8j .. c + 8j + 7
        const uint32_t* v = j < 4 ? &r0[8 * j] : &r1[8 * (j - 4)];
        st_shared_v4(row_addr + (uint32_t)((j ^ (lane & 7)) << 4),
                     pack_bf16x2(__uint_as_float(v[0]) * scale, __uint_as_float(v[1]) * scale),
                     pack_bf16x2(__uint_as_float(v[2]) * scale, __uint_as_float(v[3]) * scale),
                     pack_bf16x2(__uint_as_float(v[4]) * scale, __uint_as_float(v[5]) * scale),
                     pack_bf16x2(__uint_as_float(v[6]) * scale, __uint_as_float(v[7]) * scale));
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        tma_store_2d(tmC, b, n0 + c, row0);
        bulk_commit();
      }
      buf ^= 1;
    }
    return;
  }
  const int row = row0 + lane;
  uint16_t* crow = C + (size_t)row * N;
  const bool vec_ok = (N % 8) == 0;
#pragma unroll 1
  for (int c = 0; c < BN; c += 32) {
    uint32_t r[32];
    tmem_ld_32x32b_x32(tcol + (uint32_t)c, r);
    tmem_ld_wait();
    const int n = n0 + c;
    if (row < M && n < N) {
      if (vec_ok && n + 32 <= N) {
        uint4* dst = reinterpret_cast<uint4*>(crow + n);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint4 v;
          v.x = pack_bf16x2(__uint_as_float(r[8 * q + 0]) * scale, __uint_as_float(r[8 * q + 1]) * scale);
          v.y = pack_bf16x2(__uint_as_float(r[8 * q + 2]) * scale, __uint_as_float(r[8 * q + 3]) * scale);
          v.z = pack_bf16x2(__uint_as_float(r[8 * q + 4]) * scale, __uint_as_float(r[8 * q + 5]) * scale);
          v.w = pack_bf16x2(__uint_as_float(r[8 * q + 6]) * scale, __uint_as_float(r[8 * q + 7]) * scale);
          dst[q] = v;
        }
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (n + j < N) crow[n + j] = f2bfbits(__uint_as_float(r[j]) * scale);
      }
    }
  }
}

}  // namespace

// ---------------------------------------------------------------------------
// Persistent prefill GEMM on CTA pairs: each cluster of two CTAs computes
// 256 x BN output tiles with one tcgen05.mma.cta_group::2 per 32 bytes of K.
// CTA r of the pair loads rows [128 r, 128 r + 128) of the tile's A block and
// columns [r BN/2, (r+1) BN/2) of its B block into its own shared memory, so
// each SM stages half of B instead of all of it; the even CTA issues the
// MMAs, which read both CTAs' operands and write 128 accumulator lanes into
// each CTA's TMEM.  Barriers: every load of a stage completes on the even
// CTA's full[stage] (expecting both CTAs' bytes); the MMA commits arrive on
// empty[stage] and tfull[acc] of both CTAs (multicast); both CTAs' epilogue
// warps arrive on the even CTA's tempty[acc].  w_static: no kernel of the
// stream writes B (the handle's weights), so the B slices of the first ring
// stages are requested before waiting on the previous kernel (their bytes
// are added to full[stage] then; its arrival comes with the A slice).
// ---------------------------------------------------------------------------
template <int BN, int STAGES, bool kBf16>
__global__ void __launch_bounds__(kThreads, 1)
    k_gemm_pair(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const __grid_constant__ CUtensorMap tmC, int tma_store, uint16_t* __restrict__ C, int M, int N,
                int K, float scale, int w_static, int* err) {
  static_assert(BN % 32 == 0 && BN >= 64 && BN <= 256, "BN");
  static_assert(STAGES <= 8, "STAGES");
  constexpr int kPM = 2 * kBM;                        // rows of a pair tile
  constexpr uint32_t A_BYTES = kBM * kBK;             // this CTA's 128 rows
  constexpr uint32_t B_BYTES = (BN / 2) * kBK;        // this CTA's half of the columns
  constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
  constexpr uint32_t TMEM_COLS = (2 * BN <= 256) ? 256 : 512;
  constexpr uint32_t IDESC = idesc_f32acc(kPM, BN, kBf16 ? 1u : 0u);
  constexpr int ES = kBf16 ? 2 : 1;
  constexpr uint16_t kPair = 0x3;                     // both CTAs of the (two-CTA) cluster

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_align<1024>(smem_raw);
  uint8_t* epi = smem + STAGES * STAGE_BYTES;                           // output staging (kEpiBytes)
  Ctl* ctl = reinterpret_cast<Ctl*>(epi + kEpiBytes);
  volatile int* abort = &ctl->abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();            // 0 issues the MMAs
  const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;
  const int tiles_m = (M + kPM - 1) / kPM, tiles_n = (N + BN - 1) / BN;
  const int num_tiles = tiles_m * tiles_n;
  const int kblocks = (K * ES + kBK - 1) / kBK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&ctl->full[s], 1);
      mbar_init(&ctl->empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&ctl->tfull[i], 1);
      mbar_init(&ctl->tempty[i], 2 * 4);              // one arrival per epilogue warp of both CTAs
    }
    mbar_init(&ctl->drain, 1);
    ctl->abort = 0;
    fence_mbar_init();
    tma_prefetch(&tmA);
    tma_prefetch(&tmB);
    if (tma_store) tma_prefetch(&tmC);
  }
  if (warp == 1) {
    tmem_alloc_pair(&ctl->tmem_base, TMEM_COLS);
    tc_fence_before();
  }
  __syncwarp();
  cluster_sync();                                     // barriers of both CTAs initialised, TMEM allocated
  tc_fence_after();
  const uint32_t tmem_base = ctl->tmem_base;
  // the first tile's B slices of the first ring stages, before the wait
  const int npre = (w_static && pair < num_tiles) ? (kblocks < STAGES ? kblocks : STAGES) : 0;
  if (warp == 0 && lane == 0) {
    const int n0 = (pair / tiles_m) * BN + (int)rank * (BN / 2);
    for (int s = 0; s < npre; ++s) {
      if (rank == 0) mbar_add_tx(&ctl->full[s], 2 * B_BYTES);
      tma_load_2d_pair(smem + s * STAGE_BYTES + A_BYTES, &tmB, cluster_map(smem_u32(&ctl->full[s]), 0),
                       s * (kBK / ES), n0);
    }
  }
  __syncwarp();
  pdl_wait();      // A is produced by the previous kernel
  pdl_trigger();

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer (both CTAs)
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued_phase[STAGES];
      bool issued[STAGES];
      for (int s = 0; s < STAGES; ++s) issued[s] = false, issued_phase[s] = 0;
      bool ok = true;
      int nissued = 0;   // stages whose A slice has been requested
      for (int tile = pair; tile < num_tiles && ok; tile += npairs) {
        const int m0 = (tile % tiles_m) * kPM + (int)rank * kBM;
        const int n0 = (tile / tiles_m) * BN + (int)rank * (BN / 2);
        for (int kb = 0; kb < kblocks; ++kb, ++nissued) {
          const bool pre = nissued < npre;   // its B slice is already on the way
          if (!mbar_wait(&ctl->empty[stage], phase ^ 1u, abort)) {
            raise_abort(ctl, err);
            ok = false;
            break;
          }
          uint8_t* sA = smem + stage * STAGE_BYTES;
          const uint32_t full0 = cluster_map(smem_u32(&ctl->full[stage]), 0);
          if (rank == 0) mbar_expect_tx(&ctl->full[stage], pre ? 2 * A_BYTES : 2 * STAGE_BYTES);
          tma_load_2d_pair(sA, &tmA, full0, kb * (kBK / ES), m0);
          if (!pre) tma_load_2d_pair(sA + A_BYTES, &tmB, full0, kb * (kBK / ES), n0);
          issued[stage] = true;
          issued_phase[stage] = phase;
          if (++stage == STAGES) stage = 0, phase ^= 1u;
        }
      }
      if (*abort) {
        // the even CTA's full barriers count both CTAs' copies: let those in
        // flight land before the pair exits (a stage whose B slice went out
        // before the wait but whose A slice never did gets its arrival here)
        if (rank == 0)
          for (int s = 0; s < STAGES; ++s) {
            if (!issued[s] && s < npre) {
              mbar_arrive(&ctl->full[s]);
              issued[s] = true;
              issued_phase[s] = 0;
            }
            if (issued[s]) mbar_wait(&ctl->full[s], issued_phase[s], nullptr, 100000000ull);
          }
      } else {
        // every stage's last MMA commit has arrived on this CTA's empty
        // barrier before the CTA may exit
        for (int s = 0; s < STAGES; ++s)
          if (issued[s] && !mbar_wait(&ctl->empty[s], issued_phase[s], abort)) {
            raise_abort(ctl, err);
            break;
          }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      // ---------------- MMA issuer (even CTA only)
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int tile = pair; tile < num_tiles && ok; tile += npairs) {
        if (!mbar_wait_cluster(&ctl->tempty[acc], acc_phase ^ 1u, abort)) {
          raise_abort(ctl, err);
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!mbar_wait(&ctl->full[stage], phase, abort)) {
            raise_abort(ctl, err);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(smem + stage * STAGE_BYTES);
          const uint64_t adesc = desc_kmajor_sw128(a_addr);
          const uint64_t bdesc = desc_kmajor_sw128(a_addr + A_BYTES);
#pragma unroll
          for (int k = 0; k < kBK / 32; ++k) {   // 32 bytes of K per MMA: +2 in the address field
            if constexpr (kBf16)
              mma_f16_pair(d_tmem, adesc + 2 * k, bdesc + 2 * k, IDESC, (kb | k) != 0);
            else
              mma_f8f6f4_pair(d_tmem, adesc + 2 * k, bdesc + 2 * k, IDESC, (kb | k) != 0);
          }
          mma_commit_pair(&ctl->empty[stage], kPair);
          if (++stage == STAGES) stage = 0, phase ^= 1u;
        }
        if (!ok) break;
        mma_commit_pair(&ctl->tfull[acc], kPair);
        if (++acc == 2) acc = 0, acc_phase ^= 1u;
      }
      if (*abort) {
        mma_commit_pair(&ctl->drain, kPair);
        mbar_wait(&ctl->drain, 0, nullptr, 100000000ull);
      }
    }
  } else {
    // ---------------- epilogue (both CTAs): warps 2..5 own TMEM lane quarters (warp % 4)
    const int quarter = warp & 3;
    const uint32_t tempty0[2] = {cluster_map(smem_u32(&ctl->tempty[0]), 0),
                                 cluster_map(smem_u32(&ctl->tempty[1]), 0)};
    uint8_t* bufs = epi + quarter * 2 * kEpiBuf;
    int buf = 0;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int tile = pair; tile < num_tiles; tile += npairs) {
      const int m0 = (tile % tiles_m) * kPM + (int)rank * kBM, n0 = (tile / tiles_m) * BN;
      // one decision per warp: the TMEM loads below are warp-collective
      if (!__all_sync(0xffffffffu, mbar_wait(&ctl->tfull[acc], acc_phase, abort))) {
        raise_abort(ctl, err);
        break;
      }
      tc_fence_after();
      epilogue_rows<BN>(tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * BN), bufs, buf, &tmC,
                        tma_store != 0, C, M, N, m0 + quarter * 32, n0, scale, lane);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_remote(tempty0[acc]);
      if (++acc == 2) acc = 0, acc_phase ^= 1u;
    }
    if (lane == 0) bulk_wait<0>();          // this warp's stores are written before the CTA exits
  }
  __syncwarp();
  __syncthreads();
  cluster_sync();                                     // no MMA of the pair still writes either CTA's TMEM
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------
// Skinny (few-row) GEMM, weights as the MMA's A operand, split over K.
//   D^T[n, m] = sum_k W[n, k] X[m, k] for one 128-row block of W and the
//   k-blocks [kb0, kb1) of this split.  splits == 1: bf16 y[m, n] directly;
//   else f32 partial[split][m][n].
// ---------------------------------------------------------------------------
template <int BNT, int STAGES, bool kBf16>
__global__ void __launch_bounds__(kThreads, 1)
    k_gemm_tc_skinny(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                     uint16_t* __restrict__ y, float* __restrict__ partial, int Mtok, int N, int K,
                     int kb_per_split, float scale, int* err) {
  static_assert(BNT % 16 == 0 && BNT >= 16 && BNT <= 256, "BNT");
  constexpr uint32_t A_BYTES = kBM * kBK;
  constexpr uint32_t B_BYTES = BNT * kBK;
  constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
  constexpr uint32_t TMEM_COLS = (BNT <= 32) ? 32 : (BNT <= 64) ? 64 : (BNT <= 128) ? 128 : 256;
  constexpr uint32_t IDESC = idesc_f32acc(kBM, BNT, kBf16 ? 1u : 0u);
  constexpr int ES = kBf16 ? 2 : 1;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_align<1024>(smem_raw);
  Ctl* ctl = reinterpret_cast<Ctl*>(smem + STAGES * STAGE_BYTES);
  volatile int* abort = &ctl->abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * kBM;
  const int split = blockIdx.y;
  const int kblocks = (K * ES + kBK - 1) / kBK;
  const int kb0 = split * kb_per_split;
  const int kb1 = min(kblocks, kb0 + kb_per_split);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&ctl->full[s], 1);
      mbar_init(&ctl->empty[s], 1);
    }
    mbar_init(&ctl->tfull[0], 1);
    mbar_init(&ctl->drain, 1);
    ctl->abort = 0;
    fence_mbar_init();
    tma_prefetch(&tmW);
    tma_prefetch(&tmX);
  }
  if (warp == 1) {
    tmem_alloc(&ctl->tmem_base, TMEM_COLS);
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = ctl->tmem_base;
  pdl_wait();      // operands are produced by the previous kernel
  pdl_trigger();

  if (warp == 0) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool issued[STAGES];
      uint32_t issued_phase[STAGES];
      for (int s = 0; s < STAGES; ++s) issued[s] = false, issued_phase[s] = 0;
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!mbar_wait(&ctl->empty[stage], phase ^ 1u, abort)) {
          raise_abort(ctl, err);
          break;
        }
        uint8_t* sA = smem + stage * STAGE_BYTES;
        mbar_expect_tx(&ctl->full[stage], STAGE_BYTES);
        tma_load_2d(sA, &tmW, &ctl->full[stage], kb * (kBK / ES), n0);
        tma_load_2d(sA + A_BYTES, &tmX, &ctl->full[stage], kb * (kBK / ES), 0);
        issued[stage] = true;
        issued_phase[stage] = phase;
        if (++stage == STAGES) stage = 0, phase ^= 1u;
      }
      if (*abort)
        for (int s = 0; s < STAGES; ++s)
          if (issued[s]) mbar_wait(&ctl->full[s], issued_phase[s], nullptr, 100000000ull);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!mbar_wait(&ctl->full[stage], phase, abort)) {
          raise_abort(ctl, err);
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t a_addr = smem_u32(smem + stage * STAGE_BYTES);
        const uint64_t adesc = desc_kmajor_sw128(a_addr);
        const uint64_t bdesc = desc_kmajor_sw128(a_addr + A_BYTES);
#pragma unroll
        for (int k = 0; k < kBK / 32; ++k)
          mma_k32b<kBf16>(tmem_base, adesc + 2 * k, bdesc + 2 * k, IDESC, (kb != kb0) || (k != 0));
        mma_commit(&ctl->empty[stage]);
        if (++stage == STAGES) stage = 0, phase ^= 1u;
      }
      if (ok) {
        mma_commit(&ctl->tfull[0]);
      } else {
        mma_commit(&ctl->drain);
        mbar_wait(&ctl->drain, 0, nullptr, 100000000ull);
      }
    }
  } else {
    const int quarter = warp & 3;
    if (__all_sync(0xffffffffu, kb1 > kb0 && mbar_wait(&ctl->tfull[0], 0, abort))) {   // warp-uniform: TMEM loads
      tc_fence_after();
      const int n = n0 + quarter * 32 + lane;
#pragma unroll 1
      for (int c = 0; c < BNT; c += 32) {
        uint32_t r[32];
        tmem_ld_32x32b_x32(tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)c, r);
        tmem_ld_wait();
        if (n < N) {
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int m = c + j;
            if (m < Mtok) {
              const float v = __uint_as_float(r[j]);
              if (partial)
                partial[((size_t)split * Mtok + m) * N + n] = v;
              else
                y[(size_t)m * N + n] = f2bfbits(v * scale);
            }
          }
        }
      }
      tc_fence_before();
    } else if (kb1 > kb0) {
      raise_abort(ctl, err);
    }
  }
  __syncwarp();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------
// Few-row GEMM with K split across a thread-block cluster (decode
// projections, Mtok <= 128).  CTA rank r of a cluster of S CTAs (the cluster
// spans grid x; grid y walks the 128-row weight blocks) computes, swap-AB as
// k_gemm_tc_skinny, D^T[n, m] = sum over k-blocks [r K/S, (r+1) K/S) of
// W[n, k] X[m, k].  The partial sums meet in distributed shared memory: each
// CTA copies its accumulator into its own pipeline memory (idle by then),
// the cluster synchronises, and CTA r sums rows [128 r / S, 128 (r+1) / S) of
// the block over the S ranks in rank order (the same order every call),
// scales, rounds to bf16 and stores y.  No global scratch, no second kernel.
// w_static: no kernel of the stream writes the weights (the handle's own
// copies), so the first ring stages of weights are requested before waiting
// on the previous kernel and stream while it finishes.
// Every thread of every CTA reaches both cluster barriers, after an abort
// too (the sums of an aborted call are then wrong and the error word says so).
// ---------------------------------------------------------------------------
template <int BNT, int STAGES, bool kBf16>
__global__ void __launch_bounds__(kThreads, 1)
    k_gemm_fewrow(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                  uint16_t* __restrict__ y, int Mtok, int N, int K, float scale, int w_static, int* err) {
  static_assert(BNT % 16 == 0 && BNT >= 16 && BNT <= 128, "BNT");
  constexpr uint32_t A_BYTES = kBM * kBK;
  constexpr uint32_t B_BYTES = BNT * kBK;
  constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
  constexpr uint32_t TMEM_COLS = BNT <= 32 ? 32 : (BNT <= 64 ? 64 : 128);
  constexpr uint32_t IDESC = idesc_f32acc(kBM, BNT, kBf16 ? 1u : 0u);
  constexpr int ES = kBf16 ? 2 : 1;
  constexpr int RED_LD = BNT + 4;   // floats per exchange row (padding spreads the rows over the banks)
  static_assert(kBM * RED_LD * 4 <= (int)(STAGES * STAGE_BYTES), "the exchange buffer fits in the ring");

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_align<1024>(smem_raw);
  Ctl* ctl = reinterpret_cast<Ctl*>(smem + STAGES * STAGE_BYTES);
  float* red = reinterpret_cast<float*>(smem);   // [128 weight rows][RED_LD], over the ring once it is idle
  volatile int* abort = &ctl->abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = (int)gridDim.x;
  const int rank = (int)cluster_ctarank();
  const int n0 = blockIdx.y * kBM;
  const int kblocks = (K * ES + kBK - 1) / kBK;
  const int kb0 = rank * kblocks / S;
  const int nk = (rank + 1) * kblocks / S - kb0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&ctl->full[s], 1);
      mbar_init(&ctl->empty[s], 1);
    }
    mbar_init(&ctl->tfull[0], 1);
    mbar_init(&ctl->drain, 1);
    ctl->abort = 0;
    fence_mbar_init();
    tma_prefetch(&tmW);
    tma_prefetch(&tmX);
  }
  if (warp == 1) {
    tmem_alloc(&ctl->tmem_base, TMEM_COLS);
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = ctl->tmem_base;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer: ring slot i holds k-block kb0 + i
      const int npre = nk < STAGES ? nk : STAGES;
      if (w_static)
        for (int i = 0; i < npre; ++i) {
          mbar_expect_tx(&ctl->full[i], STAGE_BYTES);
          tma_load_2d(smem + i * STAGE_BYTES, &tmW, &ctl->full[i], (kb0 + i) * (kBK / ES), n0);
        }
      pdl_wait();      // the activations are produced by the previous kernel
      pdl_trigger();
      for (int i = 0; i < npre; ++i) {
        if (!w_static) {
          mbar_expect_tx(&ctl->full[i], STAGE_BYTES);
          tma_load_2d(smem + i * STAGE_BYTES, &tmW, &ctl->full[i], (kb0 + i) * (kBK / ES), n0);
        }
        tma_load_2d(smem + i * STAGE_BYTES + A_BYTES, &tmX, &ctl->full[i], (kb0 + i) * (kBK / ES), 0);
      }
      int issued = npre;
      for (int i = npre; i < nk; ++i) {
        const int stg = i % STAGES;
        const uint32_t use = (uint32_t)(i / STAGES);
        if (!mbar_wait(&ctl->empty[stg], (use & 1u) ^ 1u, abort)) {
          raise_abort(ctl, err);
          break;
        }
        uint8_t* sA = smem + stg * STAGE_BYTES;
        mbar_expect_tx(&ctl->full[stg], STAGE_BYTES);
        tma_load_2d(sA, &tmW, &ctl->full[stg], (kb0 + i) * (kBK / ES), n0);
        tma_load_2d(sA + A_BYTES, &tmX, &ctl->full[stg], (kb0 + i) * (kBK / ES), 0);
        issued = i + 1;
      }
      if (*abort)   // let the copies in flight land before the CTA can exit
        for (int j = issued > STAGES ? issued - STAGES : 0; j < issued; ++j)
          mbar_wait(&ctl->full[j % STAGES], (uint32_t)(j / STAGES) & 1u, nullptr, 100000000ull);
    }
  } else {
    pdl_wait();
    pdl_trigger();
    if (warp == 1) {
      if (lane == 0) {
        // ---------------- MMA issuer
        bool ok = true;
        for (int i = 0; i < nk; ++i) {
          const int stg = i % STAGES;
          if (!mbar_wait(&ctl->full[stg], (uint32_t)(i / STAGES) & 1u, abort)) {
            raise_abort(ctl, err);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(smem + stg * STAGE_BYTES);
          const uint64_t adesc = desc_kmajor_sw128(a_addr);
          const uint64_t bdesc = desc_kmajor_sw128(a_addr + A_BYTES);
#pragma unroll
          for (int k = 0; k < kBK / 32; ++k)
            mma_k32b<kBf16>(tmem_base, adesc + 2 * k, bdesc + 2 * k, IDESC, (i | k) != 0);
          mma_commit(&ctl->empty[stg]);
        }
        if (ok && nk > 0) {
          mma_commit(&ctl->tfull[0]);
        } else {
          mma_commit(&ctl->drain);
          mbar_wait(&ctl->drain, 0, nullptr, 100000000ull);
        }
      }
    } else {
      // ---------------- epilogue warps 2..5: accumulator rows -> own exchange buffer
      const int quarter = warp & 3;
      float* dst = red + (quarter * 32 + lane) * RED_LD;
      if (__all_sync(0xffffffffu, nk > 0 && mbar_wait(&ctl->tfull[0], 0, abort))) {   // warp-uniform: TMEM loads
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < BNT; c += 16) {
          uint32_t r[16];
          tmem_ld_32x32b_x16(tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)c, r);
          tmem_ld_wait();
#pragma unroll
          for (int q = 0; q < 4; ++q)
            *reinterpret_cast<float4*>(dst + c + 4 * q) =
                make_float4(__uint_as_float(r[4 * q]), __uint_as_float(r[4 * q + 1]), __uint_as_float(r[4 * q + 2]),
                            __uint_as_float(r[4 * q + 3]));
        }
        tc_fence_before();
      } else {
        if (nk > 0) raise_abort(ctl, err);
        for (int c = 0; c < BNT; c += 4) *reinterpret_cast<float4*>(dst + c) = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
  }
  __syncwarp();
  cluster_sync();   // every CTA's partial sits in its exchange buffer
  {
    // this CTA's rows of the block, summed over the ranks in rank order;
    // consecutive threads take consecutive weight rows (coalesced stores)
    const int r0 = rank * kBM / S, rows = (rank + 1) * kBM / S - r0;
    const int quads = (Mtok + 3) >> 2;
    const uint32_t red_s = smem_u32(red);
    for (int idx = threadIdx.x; idx < rows * quads; idx += kThreads) {
      const int nl = r0 + idx % rows, m = 4 * (idx / rows);
      const uint32_t off = red_s + (uint32_t)((nl * RED_LD + m) * 4);
      // all ranks' loads first (independent remote reads in flight together),
      // then the sums in rank order
      float4 v[8];
#pragma unroll
      for (int r = 0; r < 8; ++r)
        if (r < S) v[r] = ld_dsmem_f32x4(cluster_map(off, (uint32_t)r));
      float4 acc = v[0];
#pragma unroll
      for (int r = 1; r < 8; ++r)
        if (r < S) acc.x += v[r].x, acc.y += v[r].y, acc.z += v[r].z, acc.w += v[r].w;
      const int n = n0 + nl;
      if (n < N) {
        uint16_t* yc = y + (size_t)m * N + n;
        yc[0] = f2bfbits(acc.x * scale);
        if (m + 1 < Mtok) yc[N] = f2bfbits(acc.y * scale);
        if (m + 2 < Mtok) yc[2 * (size_t)N] = f2bfbits(acc.z * scale);
        if (m + 3 < Mtok) yc[3 * (size_t)N] = f2bfbits(acc.w * scale);
      }
    }
  }
  cluster_sync();   // no CTA leaves while another still reads its buffer
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

// y[m, n] = bf16(scale * sum_s partial[s][m][n]); 4 columns per thread, or
// one when the sizes or y's alignment do not allow vectors.
__global__ void __launch_bounds__(256) k_splitk_reduce(const float* __restrict__ partial, int splits, int Mtok, int N,
                                                       float scale, uint16_t* __restrict__ y, int vec) {
  pdl_wait();
  pdl_trigger();
  const size_t plane = (size_t)Mtok * N;
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  if (vec) {
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < plane / 4; i += stride) {
      float4 acc = reinterpret_cast<const float4*>(partial)[i];
      for (int s = 1; s < splits; ++s) {
        float4 v = reinterpret_cast<const float4*>(partial + s * plane)[i];
        acc.x += v.x, acc.y += v.y, acc.z += v.z, acc.w += v.w;
      }
      uint2 o;
      o.x = pack_bf16x2(acc.x * scale, acc.y * scale);
      o.y = pack_bf16x2(acc.z * scale, acc.w * scale);
      reinterpret_cast<uint2*>(y)[i] = o;
    }
  } else {
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < plane; i += stride) {
      float acc = partial[i];
      for (int s = 1; s < splits; ++s) acc += partial[s * plane + i];
      y[i] = f2bfbits(acc * scale);
    }
  }
}

// ---------------------------------------------------------------------------
// Failure-detection self-test: the abort path of the kernels above, reached
// without breaking anything.  Warp 1's lane 0 (the MMA issuer's role) waits
// on a barrier that no copy or thread ever completes; the wait runs out after
// limit_ns, raises the abort flag and the error word, drains (a commit with
// no MMA outstanding arrives at once) and the CTA frees its TMEM and returns.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(64, 1) k_wait_selftest(uint64_t limit_ns, int* err) {
  __shared__ Ctl ctl;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(&ctl.full[0], 1);
    mbar_init(&ctl.drain, 1);
    ctl.abort = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(&ctl.tmem_base, 32);
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  pdl_wait();
  if (warp == 1 && lane == 0) {
    if (!mbar_wait(&ctl.full[0], 0, &ctl.abort, limit_ns)) raise_abort(&ctl, err);
    if (ctl.abort) {
      mma_commit(&ctl.drain);
      mbar_wait(&ctl.drain, 0, nullptr, 100000000ull);
    }
  }
  __syncwarp();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(ctl.tmem_base, 32);
  }
}

cudaError_t launch_wait_selftest(uint64_t limit_ns, int* err, cudaStream_t st) {
  return launch_pdl(k_wait_selftest, dim3(1), dim3(64), 0, st, limit_ns, err);
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

// Row-major [rows, K] matrix of e4m3 codes (es = 1) or bf16 values (es = 2),
// box of box_rows x 128 bytes, 128B swizzle.
cudaError_t make_map(CUtensorMap* map, const void* base, int rows, int K, int box_rows, int es) {
  auto fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)K * es};
  cuuint32_t box[2] = {(cuuint32_t)(kBK / es), (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  const CUtensorMapDataType dt = es == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8;
  CUresult r = fn(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Output map for the persistent kernels' TMA stores: bf16 [rows, N], box
// 64 columns x 32 rows, 128-byte swizzle.  False when the row stride or the
// base is not 16-byte aligned; the kernels then store per thread.
bool make_store_map(CUtensorMap* map, void* base, int rows, int N) {
  if ((N * 2) % 16 != 0 || (reinterpret_cast<uintptr_t>(base) & 15) != 0) return false;
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)N, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)N * 2};
  cuuint32_t box[2] = {64, 32};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

int num_sms() { return device_sm_count(); }

template <class Kern>
cudaError_t set_smem(Kern k, size_t bytes) {
  return ensure_smem_optin(reinterpret_cast<const void*>(k), (int)bytes);
}

// Two-CTA clusters of k_gemm_pair that fit on the device at once (cached per
// device and instantiation).
template <int BN, int STAGES, bool kBf16>
int pair_clusters(size_t smem) {
  static std::mutex mu;
  static std::map<int, int> by_device;
  int dev = 0;
  cudaGetDevice(&dev);
  std::lock_guard<std::mutex> lock(mu);
  auto it = by_device.find(dev);
  if (it != by_device.end()) return it->second;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * num_sms());
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, k_gemm_pair<BN, STAGES, kBf16>, &cfg) != cudaSuccess || n < 1)
    n = num_sms() / 2;
  by_device[dev] = n;
  return n;
}

template <int BN, int STAGES, bool kBf16>
cudaError_t launch_pair(const void* A, const void* B, uint16_t* y, int M, int N, int K, float scale, bool w_static,
                        int* err, cudaStream_t st) {
  CUtensorMap ta, tb;
  cudaError_t e;
  constexpr int es = kBf16 ? 2 : 1;
  if ((e = make_map(&ta, A, M, K, kBM, es)) != cudaSuccess) return e;
  if ((e = make_map(&tb, B, N, K, BN / 2, es)) != cudaSuccess) return e;
  CUtensorMap tcm = {};
  const int tma_store = make_store_map(&tcm, y, M, N) ? 1 : 0;
  const size_t smem = 1024 + (size_t)STAGES * (kBM + BN / 2) * kBK + kEpiBytes + sizeof(Ctl);
  auto k = k_gemm_pair<BN, STAGES, kBf16>;
  if ((e = set_smem(k, smem)) != cudaSuccess) return e;
  const int tiles = ((M + 2 * kBM - 1) / (2 * kBM)) * ((N + BN - 1) / BN);
  const int cap = pair_clusters<BN, STAGES, kBf16>(smem);
  const int pairs = tiles < cap ? tiles : cap;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * pairs);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = 2;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, k, ta, tb, tcm, tma_store, y, M, N, K, scale, (int)w_static, err);
}

template <int BNT, int STAGES, bool kBf16>
cudaError_t launch_skinny(const void* X, const void* W, uint16_t* y, float* partial, int Mtok, int N, int K,
                          int splits, int kps, float scale, int* err, cudaStream_t st) {
  CUtensorMap tw, tx;
  cudaError_t e;
  constexpr int es = kBf16 ? 2 : 1;
  if ((e = make_map(&tw, W, N, K, kBM, es)) != cudaSuccess) return e;
  if ((e = make_map(&tx, X, Mtok, K, BNT, es)) != cudaSuccess) return e;
  const size_t smem = 1024 + (size_t)STAGES * (kBM + BNT) * kBK + sizeof(Ctl);
  auto k = k_gemm_tc_skinny<BNT, STAGES, kBf16>;
  if ((e = set_smem(k, smem)) != cudaSuccess) return e;
  dim3 grid((N + kBM - 1) / kBM, splits);
  return launch_pdl(k, grid, dim3(kThreads), smem, st, tw, tx, y, splits > 1 ? partial : nullptr, Mtok, N, K, kps,
                    scale, err);
}

// Cluster size of the few-row GEMM: as many K splits as keep every CTA
// resident in one wave (CTAs per SM from the shared-memory footprint, with a
// margin for cluster placement), at most 8 (the portable cluster size), and
// at least two k-blocks per CTA.
int fewrow_splits(int N, int kblocks, size_t smem, int bnt) {
  const int nb = (N + kBM - 1) / kBM;
  int per_sm = (int)((228 * 1024) / (smem + 1024));
  if (per_sm < 1) per_sm = 1;
  int s = (int)(0.9 * per_sm * num_sms() / nb);
  if (s > 8) s = 8;
  if (s > kblocks / 2) s = kblocks / 2;
  // with two CTAs per SM, from 33 rows on, each split's MMAs and exchange
  // grow with the rows and two splits beat more for the 81 weight blocks of
  // in_proj (measured in the decode call of 64 rows with a 4-deep ring: 3
  // splits 80.2 us, 2 splits 78.4, 4 85.8)
  if (bnt >= 64 && nb > 64 && s > 2) s = 2;
  return s < 1 ? 1 : s;
}

template <int BNT, int STAGES, bool kBf16>
cudaError_t launch_fewrow(const void* X, const void* W, uint16_t* y, int Mtok, int N, int K, float scale,
                          bool w_static, int* err, cudaStream_t st) {
  CUtensorMap tw, tx;
  cudaError_t e;
  constexpr int es = kBf16 ? 2 : 1;
  if ((e = make_map(&tw, W, N, K, kBM, es)) != cudaSuccess) return e;
  if ((e = make_map(&tx, X, Mtok, K, BNT, es)) != cudaSuccess) return e;
  const size_t smem = 1024 + (size_t)STAGES * (kBM + BNT) * kBK + sizeof(Ctl);
  auto k = k_gemm_fewrow<BNT, STAGES, kBf16>;
  if ((e = set_smem(k, smem)) != cudaSuccess) return e;
  const int kblocks = (K * es + kBK - 1) / kBK;
  const int S = fewrow_splits(N, kblocks, smem, BNT);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(S, (N + kBM - 1) / kBM);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = S;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, k, tw, tx, y, Mtok, N, K, scale, (int)w_static, err);
}

template <bool kBf16>
cudaError_t fewrow_t(const void* X, const void* W, uint16_t* y, int Mtok, int N, int K, float scale, bool w_static,
                     int* err, cudaStream_t st) {
  const int bnt = (Mtok + 15) / 16 * 16;
  if (bnt <= 16) return launch_fewrow<16, 4, kBf16>(X, W, y, Mtok, N, K, scale, w_static, err, st);
  if (bnt <= 32) return launch_fewrow<32, 4, kBf16>(X, W, y, Mtok, N, K, scale, w_static, err, st);
  // 33-64 rows: an 8-deep ring (192 KB, one CTA per SM), so in_proj's 81
  // weight blocks run unsplit and out_proj's 21 split six ways; paged decode
  // of 64 rows 77.0 -> 74.6 us against a 4-deep ring with 2 and 8 splits
  if (bnt <= 64) return launch_fewrow<64, 8, kBf16>(X, W, y, Mtok, N, K, scale, w_static, err, st);
  // 65-128 rows: a 6-deep ring (192 KB, one CTA per SM); the 23-block stack's
  // decode of 128 rows 2.96 -> 2.85 ms against a 3-deep ring
  if (bnt <= 128) return launch_fewrow<128, 6, kBf16>(X, W, y, Mtok, N, K, scale, w_static, err, st);
  return cudaErrorInvalidValue;
}

}  // namespace

// Split plan of the skinny GEMM for (Mtok, N, Kbytes = K x operand size):
// splits and k-blocks each.  All CTAs fit in one wave (CTAs per SM from the
// shared-memory footprint) and each split streams at least 4 k-blocks, so the
// f32 partials stay small next to the weights.
void skinny_plan(int Mtok, int N, int Kbytes, int* splits, int* kps) {
  const int kblocks = (Kbytes + kBK - 1) / kBK;
  const int nt = (N + kBM - 1) / kBM;
  const int bnt = (Mtok + 15) / 16 * 16;
  const int stages = bnt <= 64 ? 4 : (bnt <= 128 ? 3 : 2);   // 2 CTAs per SM from 32 rows up
  const int smem = 1024 + stages * (kBM + bnt) * kBK + 256;
  int per_sm = (228 * 1024) / (smem + 1024);
  if (per_sm < 1) per_sm = 1;
  int s = (per_sm * num_sms()) / nt;
  if (s > kblocks) s = kblocks;
  if (s < 1) s = 1;
  int per = (kblocks + s - 1) / s;
  if (per < 4) per = kblocks < 4 ? kblocks : 4;
  s = (kblocks + per - 1) / per;
  *splits = s;
  *kps = per;
}

size_t gemm_tc_skinny_workspace(int Mtok, int N, int Kbytes) {
  int s, kps;
  skinny_plan(Mtok, N, Kbytes, &s, &kps);
  return s > 1 ? (size_t)s * Mtok * N * sizeof(float) : 0;
}

namespace {

template <bool kBf16>
cudaError_t skinny_t(const void* X, const void* W, uint16_t* y, int Mtok, int N, int K, float scale, void* ws,
                     size_t ws_bytes, int* err, cudaStream_t st, int* launches) {
  int splits, kps;
  skinny_plan(Mtok, N, K * (kBf16 ? 2 : 1), &splits, &kps);
  float* partial = static_cast<float*>(ws);
  if (splits > 1 && (!ws || ws_bytes < (size_t)splits * Mtok * N * sizeof(float))) return cudaErrorInvalidValue;
  const int bnt = (Mtok + 15) / 16 * 16;
  cudaError_t e;
  if (bnt <= 16) e = launch_skinny<16, 4, kBf16>(X, W, y, partial, Mtok, N, K, splits, kps, scale, err, st);
  else if (bnt <= 32) e = launch_skinny<32, 4, kBf16>(X, W, y, partial, Mtok, N, K, splits, kps, scale, err, st);
  else if (bnt <= 64) e = launch_skinny<64, 4, kBf16>(X, W, y, partial, Mtok, N, K, splits, kps, scale, err, st);
  else if (bnt <= 128) e = launch_skinny<128, 3, kBf16>(X, W, y, partial, Mtok, N, K, splits, kps, scale, err, st);
  else if (bnt <= 256) e = launch_skinny<256, 2, kBf16>(X, W, y, partial, Mtok, N, K, splits, kps, scale, err, st);
  else return cudaErrorInvalidValue;
  if (e != cudaSuccess) return e;
  *launches = 1;
  if (splits > 1) {
    const int vec = (((size_t)Mtok * N) % 4 == 0) && ((uintptr_t)y % 8 == 0) && ((uintptr_t)partial % 16 == 0);
    const size_t items = vec ? (size_t)Mtok * N / 4 : (size_t)Mtok * N;
    int blocks = (int)((items + 255) / 256);
    if (blocks > 4 * num_sms()) blocks = 4 * num_sms();
    e = launch_pdl(k_splitk_reduce, dim3(blocks), dim3(256), 0, st, (const float*)partial, splits, Mtok, N, scale,
                   y, vec);
    *launches = 2;
  }
  return e;
}

template <bool kBf16>
cudaError_t big_t(const void* A, const void* B, uint16_t* y, int M, int N, int K, float scale, bool w_static,
                  int* err, cudaStream_t st) {
  // 256 x 256 tiles on CTA pairs (N = 2688 leaves its last tile half
  // empty, which still beats narrower tiles' extra waves)
  return launch_pair<256, 6, kBf16>(A, B, y, M, N, K, scale, w_static, err, st);
}

}  // namespace

cudaError_t gemm_tc_skinny(const uint8_t* X, const uint8_t* W, uint16_t* y, int Mtok, int N, int K, float scale,
                           void* ws, size_t ws_bytes, int* err, cudaStream_t st, int* launches) {
  return skinny_t<false>(X, W, y, Mtok, N, K, scale, ws, ws_bytes, err, st, launches);
}

cudaError_t gemm_tc_skinny_bf16(const uint16_t* X, const uint16_t* W, uint16_t* y, int Mtok, int N, int K,
                                float scale, void* ws, size_t ws_bytes, int* err, cudaStream_t st, int* launches) {
  return skinny_t<true>(X, W, y, Mtok, N, K, scale, ws, ws_bytes, err, st, launches);
}

cudaError_t gemm_tc_fewrow(const uint8_t* X, const uint8_t* W, uint16_t* y, int Mtok, int N, int K, float scale,
                           bool w_static, int* err, cudaStream_t st) {
  return fewrow_t<false>(X, W, y, Mtok, N, K, scale, w_static, err, st);
}

cudaError_t gemm_tc_fewrow_bf16(const uint16_t* X, const uint16_t* W, uint16_t* y, int Mtok, int N, int K, float scale,
                                bool w_static, int* err, cudaStream_t st) {
  return fewrow_t<true>(X, W, y, Mtok, N, K, scale, w_static, err, st);
}

cudaError_t gemm_tc_big(const uint8_t* A, const uint8_t* B, uint16_t* y, int M, int N, int K, float scale,
                        bool w_static, int* err, cudaStream_t st) {
  return big_t<false>(A, B, y, M, N, K, scale, w_static, err, st);
}

cudaError_t gemm_tc_big_bf16(const uint16_t* A, const uint16_t* B, uint16_t* y, int M, int N, int K, float scale,
                             bool w_static, int* err, cudaStream_t st) {
  return big_t<true>(A, B, y, M, N, K, scale, w_static, err, st);
}

}  // namespace m2
