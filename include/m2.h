/*
 * m2.h — C ABI of a GB300 (sm_103a) implementation of one NemotronH-style
 * Mamba2 mixer block with FP8 W8A8 projections.
 *
 * The block (vllm.cpp PR #1288, "NemotronH's 23 Mamba2 blocks reach the device
 * on the FP8 W8A8 seam", section "What it does"):
 *
 *   in_proj (FP8 W8A8) -> split(z | xBC | dt) -> causal conv1d + SiLU
 *   -> split(x | B | C) -> Mamba2 SSD chunked scan (prefill) or single-step
 *   state update (decode) -> gated group RMSNorm -> out_proj (FP8 W8A8)
 *
 * Conventions for every entry point
 *  - Device pointers are caller-owned, row-major and contiguous.  The library
 *    never frees them.  Host pointers are only read during the call.
 *  - bf16 tensors are passed as uint16_t* (raw bfloat16 bits); e4m3 tensors as
 *    uint8_t* (OCP FP8 E4M3 codes); f32 as float*.
 *  - `stream` is a cudaStream_t (NULL = legacy default stream).  Calls that
 *    launch kernels are asynchronous on that stream; argument validation is
 *    done on the host before anything is launched, so a refused call launches
 *    nothing and writes nothing.
 *  - Every call returns an m2_status; on failure m2_last_error() returns a
 *    thread-local message describing the refusal.
 *
 * Geometry: the kernels are built for the NemotronH mixer geometry
 * (hidden 2688, d_inner 4096, 64 heads of 64, 8 groups, d_state 128, conv
 * width 4, so the in_proj row is 4096 + 6144 + 64 = 10304 wide: PR #1288,
 * opening paragraph, 23 x (10304x2688 + 2688x4096) fp8 elements).  m2_create
 * refuses any other geometry with M2_ESHAPE.
 */
#ifndef M2_H
#define M2_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int m2_status;
enum {
  M2_OK = 0,
  M2_EINVAL = 1,    /* bad argument: null pointer, bad scale, bad slot id    */
  M2_ESHAPE = 2,    /* geometry, size or alignment not supported             */
  M2_ECUDA = 3,     /* a CUDA runtime call failed (message has the error)   */
  M2_ETIMEOUT = 4,  /* a bounded device-side wait ran out (kernel returned) */
  M2_EDEVICE = 5,   /* no usable sm_103 device                              */
  M2_ENOMEM = 6     /* workspace too small or device allocation failed     */
};

enum { M2_DTYPE_F32 = 0, M2_DTYPE_BF16 = 1 };
/* Arithmetic of the two projections (m2_config.arm). */
enum { M2_ARM_W8A8 = 0, M2_ARM_W8A16 = 1 };
enum { M2_LAYOUT_OUT_IN = 0 };   /* weights stored [out, in] (torch Linear) */

/* Model geometry and static per-tensor scales. */
typedef struct m2_config {
  int hidden;       /* 2688 */
  int d_inner;      /* 4096 */
  int nheads;       /* 64 */
  int headdim;      /* 64 */
  int n_groups;     /* 8 (SSM B/C groups and RMSNorm groups) */
  int d_state;      /* 128 */
  int conv_width;   /* 4 */
  int chunk_size;   /* SSD chunk length for prefill: 256 */
  int ssm_dtype;    /* dtype of the recurrent state rows in the caller's pool
                       and prefill state: M2_DTYPE_F32 (PR #1288, "What it
                       does": the ssm_dtype == f32 term) or M2_DTYPE_BF16, a
                       bf16 state cache: rows are widened to f32 when read,
                       updated and reduced to y in f32, and rounded to bf16
                       (nearest even) when written back */
  float eps;        /* gated RMSNorm epsilon (1e-5) */
  float s_x;        /* static input_scale of in_proj's activation (> 0) */
  float s_y;        /* static input_scale of out_proj's activation (> 0) */
  int arm;          /* M2_ARM_W8A8 (0, the device arm: e4m3 activations with
                       the static input_scales above, e4m3 weights) or
                       M2_ARM_W8A16, the host reference arm of PR #1288,
                       section "The comparison is not bit-comparable, and that
                       is the point": input_scale is carried and not applied,
                       so both projections take their bf16 activations as they
                       are (the hidden input and the gated-norm output) against
                       weights dequantised to bf16 once at m2_create,
                       w = bf16(dec(code) * weight_scale), product in f32,
                       round to nearest even (PR #1289, commit "the FP8 W8A8
                       seam": DenseBf16 expands the fp8 tower to bf16).  Both
                       arms accumulate in f32 and round the result to bf16.
                       The W8A16 arm serves m2_prefill and m2_decode only; the
                       pre-quantised and mixed-batch calls refuse it with
                       M2_EINVAL.  The handle then also holds the bf16 weights
                       (2 bytes per weight more). */
} m2_config;

/*
 * Weights of one block.  Pointers may be host or device memory (any pointer
 * cudaMemcpy can read with cudaMemcpyDefault); m2_create copies them into
 * device memory owned by the handle and reads none of them afterwards.
 */
typedef struct m2_weights {
  const uint8_t* in_proj;   /* e4m3 [10304, 2688], [out, in] */
  float s_w1;               /* per-tensor weight_scale of in_proj */
  const uint8_t* out_proj;  /* e4m3 [2688, 4096], [out, in] */
  float s_w2;               /* per-tensor weight_scale of out_proj */
  const uint16_t* conv_w;   /* bf16 [6144, 4]: tap 3 multiplies the current token */
  const uint16_t* conv_b;   /* bf16 [6144] or NULL (no bias) */
  const float* A_log;       /* f32 [64]; A = -exp(A_log) */
  const float* D;           /* f32 [64] skip weight */
  const float* dt_bias;     /* f32 [64] */
  const uint16_t* norm_w;   /* bf16 [4096] gated-norm weight */
  int layout;               /* must be M2_LAYOUT_OUT_IN (PR #950 refuses any
                               other projection orientation) */
} m2_weights;

/* Path counters (PR #1289 thread, GB10 three-leg run: the four kernel
 * counters), plus the bytes this handle uploaded (PR #1288, "Three points
 * where this differs from the spec", point 2). */
typedef struct m2_stats {
  uint64_t bytes_uploaded;
  uint64_t conv_fwd_calls;     /* prefill conv launches */
  uint64_t chunk_scan_calls;   /* prefill SSD scans */
  uint64_t conv_update_rows;   /* decode rows whose conv window advanced */
  uint64_t state_update_rows;  /* decode rows whose SSM state advanced */
  uint64_t prefill_calls;
  uint64_t decode_calls;
  uint64_t kernel_launches;    /* kernels this handle launched */
} m2_stats;

/* Kernel stages of a call, for m2_profile_read(). */
enum {
  M2_STAGE_QUANT_IN = 0,       /* static e4m3 quant of the block input     */
  M2_STAGE_IN_PROJ = 1,        /* W8A8 in_proj GEMM                        */
  M2_STAGE_CONV = 2,           /* prefill causal conv1d + SiLU             */
  M2_STAGE_CONV_STATE = 3,     /* (unused: the hand-off runs in stage 6)   */
  M2_STAGE_SSD_CUMSUM = 4,     /* dt softplus and in-chunk log-decay sums  */
  M2_STAGE_SSD_CHUNK_STATE = 5,
  M2_STAGE_SSD_STATE_PASS = 6,
  M2_STAGE_SSD_CHUNK_SCAN = 7,
  M2_STAGE_NORM_QUANT = 8,     /* gated group RMSNorm + e4m3 quant         */
  M2_STAGE_OUT_PROJ = 9,       /* W8A8 out_proj GEMM                       */
  M2_STAGE_DECODE_FUSED = 10,  /* decode conv + state update + norm + quant */
  M2_STAGE_DEC_QUANT_IN = 11,  /* the same three stages inside m2_decode   */
  M2_STAGE_DEC_IN_PROJ = 12,
  M2_STAGE_DEC_OUT_PROJ = 13,
  M2_NSTAGES = 16
};

/* Optional device buffers that receive intermediates of the next calls
 * (debugging and parity tests).  Any member may be NULL.  Sizes are for a
 * call over T tokens (prefill) or Bt rows (decode).  In the W8A16 arm q is
 * not written (the input is not quantised) and q2 holds codes no stage
 * reads; o is what out_proj consumes. */
typedef struct m2_taps {
  uint8_t* q;      /* e4m3 [T, 2688]  quantised block input            */
  uint16_t* zx;    /* bf16 [T, 10304] in_proj output (z | xBC | dt)    */
  uint16_t* u;     /* bf16 [T, 6144]  conv1d+SiLU output (x | B | C)   */
  float* dt;       /* f32  [T, 64]    softplus(dt + dt_bias)           */
  uint16_t* y;     /* bf16 [T, 4096]  scan output incl. D skip         */
  uint16_t* o;     /* bf16 [T, 4096]  gated group RMSNorm output       */
  uint8_t* q2;     /* e4m3 [T, 4096]  quantised out_proj input         */
} m2_taps;

typedef struct m2_handle m2_handle;

/* Text of the last refusal or CUDA error on this thread ("" if none). */
const char* m2_last_error(void);

/*
 * Create a block: validates the geometry, the orientation and ssm_dtype,
 * copies the weights to the current CUDA device (one allocation per tensor,
 * owned by the handle), synchronises, and counts the uploaded bytes.
 * The handle is tied to the device that was current at creation.
 * Errors: M2_EINVAL (null, non-positive scale, layout), M2_ESHAPE (geometry,
 * chunk size), M2_EDEVICE (no sm_103 device), M2_ECUDA.
 */
m2_status m2_create(const m2_config* cfg, const m2_weights* w, m2_handle** out);

/* Free the handle's device memory (synchronises its device first). NULL ok. */
void m2_destroy(m2_handle* h);

m2_status m2_get_stats(const m2_handle* h, m2_stats* out);

/*
 * Stage timing.  While enabled, every kernel stage of m2_prefill/m2_decode
 * is bracketed by CUDA events recorded on the call's stream.
 * m2_profile_read synchronises those events, adds each stage's elapsed
 * milliseconds and launch count into ms[M2_NSTAGES] / launches[M2_NSTAGES]
 * (either may be NULL) and forgets the records.  Disabling drops pending
 * records.  Not for use inside CUDA graph capture.
 */
m2_status m2_profile_enable(m2_handle* h, int on);
m2_status m2_profile_read(m2_handle* h, double* ms, uint64_t* launches);

/* Install (taps != NULL) or remove (NULL) intermediate taps for later calls. */
m2_status m2_set_taps(m2_handle* h, const m2_taps* taps);

/*
 * Read and clear the handle's device error word (synchronises the device).
 * M2_EINVAL: a decode row named a slot outside [0, n_slots), or a slot an
 * earlier row of the same call already named (that row was skipped, its
 * output zeroed); M2_ETIMEOUT: a bounded wait ran out (the kernel returned
 * early: outputs of that call are incomplete).
 */
m2_status m2_check(m2_handle* h);

/*
 * The same for the standalone entry points (fp8_linear, fp8_linear_bf16,
 * bf16_linear, fp8_linear_noalloc), which have no handle: they share one
 * library-owned error word per device (a file-scope device variable, looked
 * up once per device on the first such call, which should therefore come
 * before any stream capture).  Synchronises the current device, reads and
 * clears its word.  M2_ETIMEOUT: a bounded wait of one of those calls ran
 * out and its y is incomplete.
 */
m2_status m2_check_standalone(void);

/*
 * Self-test of the failure detection (no counterpart on the pages): one
 * kernel allocates tensor memory, waits with the kernels' bounded mbarrier
 * wait on a barrier that nothing ever completes, gives up after limit_us
 * microseconds (1 to 100000), takes the kernels' abort path (sets the error
 * word, drains, frees tensor memory) and returns, leaving the context usable.
 * The error word is the handle's (then m2_check(h) reports M2_ETIMEOUT) or,
 * with h == NULL, the standalone one (m2_check_standalone).  Asynchronous on
 * `stream`.  Errors: M2_EINVAL (limit out of range), M2_EDEVICE, M2_ECUDA.
 */
m2_status m2_selftest_timeout(m2_handle* h, unsigned limit_us, void* stream);

/* Workspace bytes m2_prefill needs for these sequence lengths. */
m2_status m2_prefill_workspace_size(const m2_handle* h, const int32_t* seqlens_host, int nseq,
                                    size_t* bytes);

/*
 * Prefill of nseq packed sequences (varlen).  Chunks of chunk_size tokens
 * never cross a sequence boundary; the last chunk of a sequence is partial.
 * When no sequence has more than 64 tokens the SSD recurrence is evaluated
 * token by token in one kernel instead of chunk-wise (the same results up to
 * f32 rounding order; the workspace size does not change).
 *   hidden       bf16 [sum(T), 2688] device
 *   seqlens_host int32 [nseq] host, each >= 1
 *   has_initial  uint8 [nseq] host or NULL (NULL = every sequence starts from
 *                zero state: the rows are "gathered and zeroed")
 *   conv_state   bf16 [nseq, 6144, 3] device, in/out: read for sequences with
 *                has_initial, always overwritten with the last 3 raw xBC
 *                inputs ([channel][tap], tap 0 oldest)
 *   ssm_state    [nseq, 64, 64, 128] device, f32 or bf16 (the handle's
 *                ssm_dtype), in/out likewise
 *   out          bf16 [sum(T), 2688] device
 *   workspace    device, >= m2_prefill_workspace_size bytes, 256-byte aligned
 * Errors: M2_EINVAL, M2_ESHAPE (nseq > 256 or a length < 1), M2_ENOMEM
 * (workspace too small), M2_ECUDA.
 */
m2_status m2_prefill(m2_handle* h, const uint16_t* hidden, const int32_t* seqlens_host, int nseq,
                     const uint8_t* has_initial, uint16_t* conv_state, void* ssm_state,
                     uint16_t* out, void* workspace, size_t ws_bytes, void* stream);

/*
 * m2_prefill with the block's input already quantised: hidden_q e4m3 [sum(T),
 * 2688] device, 16-byte aligned, holding e4m3(x / s_x) for the handle's s_x
 * (as fp8_quant or m2_rmsnorm_residual_quant write it).  The block's own
 * input quant is skipped; everything else is m2_prefill.
 */
m2_status m2_prefill_q(m2_handle* h, const uint8_t* hidden_q, const int32_t* seqlens_host, int nseq,
                       const uint8_t* has_initial, uint16_t* conv_state, void* ssm_state,
                       uint16_t* out, void* workspace, size_t ws_bytes, void* stream);

/* Workspace bytes m2_decode needs for a batch of Bt rows. */
m2_status m2_decode_workspace_size(const m2_handle* h, int Bt, size_t* bytes);

/*
 * Paged decode: one token per row.  Row b advances pool slot slot_idx[b] in
 * place (PR #1288, "What it does": the paged arm advances the gathered rows
 * IN PLACE).  slot_idx[b] == -1 is a padding row: output zeroed, no state
 * touched.  Slot ids must be unique within a call: a row naming a slot that
 * an earlier row of the call already named is detected on the device, skipped
 * (output zeroed, no state touched; the first row naming the slot advances
 * it) and m2_check() reports M2_EINVAL.  An id outside [-1, n_slots) is
 * detected the same way: that row is skipped, its output zeroed, and
 * m2_check() reports M2_EINVAL.
 *   hidden     bf16 [Bt, 2688] device
 *   conv_pool  bf16 [n_slots, 6144, 3] device
 *   ssm_pool   [n_slots, 64, 64, 128] device, f32 or bf16 (ssm_dtype)
 *   slot_idx   int32 [Bt] device
 *   out        bf16 [Bt, 2688] device
 * Errors: M2_EINVAL, M2_ESHAPE (Bt < 1 or Bt > 4096), M2_ENOMEM, M2_ECUDA.
 */
m2_status m2_decode(m2_handle* h, const uint16_t* hidden, int Bt, uint16_t* conv_pool, void* ssm_pool,
                    int n_slots, const int32_t* slot_idx, uint16_t* out, void* workspace, size_t ws_bytes,
                    void* stream);

/* m2_decode with the input already quantised (hidden_q e4m3 [Bt, 2688], as in
 * m2_prefill_q). */
m2_status m2_decode_q(m2_handle* h, const uint8_t* hidden_q, int Bt, uint16_t* conv_pool, void* ssm_pool,
                      int n_slots, const int32_t* slot_idx, uint16_t* out, void* workspace, size_t ws_bytes,
                      void* stream);

/*
 * A mixed batch in one call (the decode / prefill row classification of
 * vllm.cpp PR #1289's review thread, the correction of the G1(c) arm: a row
 * with one query token and prior state is a decode; batches are ordered
 * decodes first):
 *   hidden  bf16 [Bt + sum(T), 2688]: rows [0, Bt) are decode rows, one token
 *           each, as m2_decode; the rest are the packed prefill sequences,
 *           as m2_prefill (seqlens_host, has_initial, conv_state, ssm_state)
 *   out     bf16 [Bt + sum(T), 2688]
 * The input quant and both projections run once over all rows; the decode
 * rows advance their pool rows in place, the prefill rows run the chunked
 * scan.  Bt = 0 or nseq = 0 is allowed (not both); the decode arguments may
 * be NULL when Bt = 0, the prefill ones when nseq = 0.  Of the intermediate
 * taps this call writes q, zx, y, o and q2 (Bt + sum(T) rows, in batch
 * order); u and dt are not written.  Errors as m2_decode and m2_prefill.
 */
m2_status m2_mixed_workspace_size(const m2_handle* h, int Bt, const int32_t* seqlens_host, int nseq,
                                  size_t* bytes);
m2_status m2_mixed(m2_handle* h, const uint16_t* hidden, int Bt, uint16_t* conv_pool, void* ssm_pool, int n_slots,
                   const int32_t* slot_idx, const int32_t* seqlens_host, int nseq, const uint8_t* has_initial,
                   uint16_t* conv_state, void* ssm_state, uint16_t* out, void* workspace, size_t ws_bytes,
                   void* stream);

/*
 * Standalone static per-tensor activation quantisation (the kQuantFp8Static
 * op of PR #988, section "The Thor finding, measured"):
 *   q[i] = e4m3_satfinite_rne(fp32(x[i]) / scale)   (IEEE fp32 division)
 * Bit-exact.  x bf16 [n] device, q uint8 [n] device.  scale > 0 and finite.
 */
m2_status fp8_quant(const uint16_t* x, size_t n, float scale, uint8_t* q, void* stream);

/* Workspace bytes fp8_linear needs for an M x N x K problem (0 for many). */
m2_status fp8_linear_workspace_size(int M, int N, int K, size_t* bytes);

/*
 * W8A8 linear on pre-quantised activations (MatmulFp8CutlassPreQuantD of
 * PR #972, section "The call-site change"):
 *   y[m, n] = bf16( s_a * s_w * sum_k dec(a_q[m, k]) * dec(w_q[n, k]) )
 * a_q e4m3 [M, K], w_q e4m3 [N, K] ([out, in]), y bf16 [M, N], all device.
 * fp32 accumulation.  K must be a multiple of 16 and all pointers 16-byte
 * aligned.  Errors: M2_EINVAL, M2_ESHAPE, M2_ENOMEM.
 */
m2_status fp8_linear(const uint8_t* a_q, float s_a, const uint8_t* w_q, float s_w, uint16_t* y, int M,
                     int N, int K, void* workspace, size_t ws_bytes, void* stream);

/*
 * fp8_linear for callers that cannot allocate device memory.  The pages have
 * no counterpart to this entry point.
 *
 * Who needs it: code that embeds this library without owning a device
 * allocator (a plain C host with no framework around it), serving loops that
 * forbid allocation after start-up so their memory footprint stays fixed, and
 * code that issues work while a CUDA stream is being captured, where a fresh
 * workspace cannot be allocated on the spot.  fp8_linear needs a caller
 * workspace for its split-K partial sums; this variant instead uses one
 * library-owned scratch array in device memory (a file-scope __device__
 * array of M2_NOALLOC_SCRATCH_BYTES = 16 MiB), so it calls no cudaMalloc,
 * cudaFree or allocating library routine.  The array is part of the library's
 * device code: every GPU on which that code is loaded holds it until the
 * process exits (with the default lazy module loading, the GPUs on which a
 * call of this library has run; with CUDA_MODULE_LOADING=EAGER, every GPU the
 * process initialises, whether or not it calls this entry point).  The
 * device address of the array is cached per device on first use; a
 * cudaDeviceReset() of a device invalidates it, so this entry point must not
 * be called on a device after that device was reset.
 *
 * Same arguments and result as fp8_linear without the workspace.  Only the
 * few-row (decode) form is offered: 1 <= M <= 256, and the split-K partials
 * (splits x M x N floats) must fit the scratch array; larger problems are
 * refused with M2_ESHAPE and a message naming the limit.  The first call on
 * each device looks the array up (cudaGetSymbolAddress) with that device
 * current; make that first call before any stream capture.  All calls share
 * the one array: calls that can overlap on the GPU (different streams, or
 * different host threads) race on it and must be serialised by the caller.
 * Every call overwrites the part of the array it reads, so no clearing is
 * needed between calls.
 */
#define M2_NOALLOC_SCRATCH_BYTES (16u << 20)
m2_status fp8_linear_noalloc(const uint8_t* a_q, float s_a, const uint8_t* w_q, float s_w, uint16_t* y, int M,
                             int N, int K, void* stream);
/* (A bounded wait that runs out inside fp8_linear_noalloc, fp8_linear,
 * fp8_linear_bf16 or bf16_linear is reported by m2_check_standalone().) */

/*
 * The quantise-inside form (MatmulFp8CutlassD of PR #972): x bf16 [M, K] is
 * quantised with s_a (as fp8_quant) into the workspace, then as fp8_linear.
 * Workspace: M*K bytes (rounded up to 256) plus fp8_linear's.
 */
m2_status fp8_linear_bf16(const uint16_t* x, float s_a, const uint8_t* w_q, float s_w, uint16_t* y,
                          int M, int N, int K, void* workspace, size_t ws_bytes, void* stream);

/*
 * Weight dequantisation of the W8A16 arm (what m2_create does to both
 * projections when cfg->arm is M2_ARM_W8A16):
 *   out[i] = bf16( dec(q[i]) * scale )      (product in f32, round to nearest even)
 * q e4m3 [n] (8-byte aligned), out bf16 [n] (16-byte aligned), both device;
 * scale positive and finite.  Bit-exact.  NaN codes give NaN.
 * Errors: M2_EINVAL.
 */
m2_status fp8_dequant(const uint8_t* q, size_t n, float scale, uint16_t* out, void* stream);

/* Workspace bytes bf16_linear needs for an M x N x K problem (0 for many). */
m2_status bf16_linear_workspace_size(int M, int N, int K, size_t* bytes);

/*
 * The W8A16 arm's linear layer (vt::MatmulBT on dequantised weights, PR
 * #1289, GB10 counter-measurement commit):
 *   y[m, n] = bf16( scale * sum_k x[m, k] * w[n, k] )
 * x bf16 [M, K], w bf16 [N, K] ([out, in]), y bf16 [M, N], all device, on the
 * tensor cores with f32 accumulation.  K must be a multiple of 16 and all
 * pointers 16-byte aligned.  Errors: M2_EINVAL, M2_ESHAPE, M2_ENOMEM.
 */
m2_status bf16_linear(const uint16_t* x, const uint16_t* w, float scale, uint16_t* y, int M, int N, int K,
                      void* workspace, size_t ws_bytes, void* stream);

/*
 * Between stacked blocks (pre-norm residual stack):
 *   if add != NULL:     h[t, :] = bf16(h[t, :] + add[t, :])     (in place)
 *   if normed != NULL:  normed[t, :] = bf16( h[t, :] / sqrt(mean(h[t, :]^2) + eps) * w )
 * h bf16 [T, n] in/out, add bf16 [T, n] or NULL, w bf16 [n] (may be NULL when
 * normed is NULL), normed bf16 [T, n] or NULL; all device, 16-byte aligned.
 * n must be a multiple of 8.
 */
m2_status m2_rmsnorm_residual(uint16_t* h, const uint16_t* add, const uint16_t* w, float eps,
                              uint16_t* normed, int T, int n, void* stream);

/*
 * The same step fused with the next block's static activation quant: h (and
 * normed, if not NULL) as m2_rmsnorm_residual, and
 *   q[t, :] = e4m3(normed[t, :] / s_q)        (round to nearest even, saturating)
 * from the bf16 normed value, i.e. exactly the codes fp8_quant would write
 * for it (the static per-tensor quant of PR #988, section "The Thor finding,
 * measured"), so
 * m2_prefill_q / m2_decode_q of the next block see the input m2_prefill /
 * m2_decode would have quantised themselves, one HBM pass fewer.
 * q e4m3 [T, n] device, 8-byte aligned; w is required; s_q > 0.
 */
m2_status m2_rmsnorm_residual_quant(uint16_t* h, const uint16_t* add, const uint16_t* w, float eps, float s_q,
                                    uint16_t* normed, uint8_t* q, int T, int n, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* M2_H */
