// The C ABI of libm2 (declared in include/m2.h): argument validation, the
// handle that owns the block's device weights, workspace carving, and the
// launch sequence of prefill and decode.  All compute runs in the kernels.
#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <vector>

#include "../../include/m2.h"
#include "m2_kernels.h"
#include "gemm.h"

using namespace m2;

namespace {

thread_local std::string g_err;

m2_status fail(m2_status code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_err = buf;
  return code;
}

#define M2_CUDA(call)                                                                          \
  do {                                                                                         \
    cudaError_t e_ = (call);                                                                   \
    if (e_ != cudaSuccess) return fail(M2_ECUDA, "%s: %s", #call, cudaGetErrorString(e_));     \
  } while (0)

// Launch one kernel stage: optional event bracket, error check, launch count.
#define M2_STAGE(h, st, stage, nlaunch, call)                                                  \
  do {                                                                                         \
    cudaEvent_t a_ = nullptr;                                                                  \
    if ((h)->prof_on) {                                                                        \
      a_ = (h)->take_event();                                                                  \
      cudaEventRecord(a_, st);                                                                 \
    }                                                                                          \
    M2_CUDA(call);                                                                             \
    (h)->stats.kernel_launches += (uint64_t)(nlaunch);                                         \
    if (a_) {                                                                                  \
      cudaEvent_t b_ = (h)->take_event();                                                      \
      cudaEventRecord(b_, st);                                                                 \
      (h)->recs.push_back({(stage), (int)(nlaunch), a_, b_});                                  \
    }                                                                                          \
  } while (0)

m2_status check_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return fail(M2_EDEVICE, "no CUDA device");
  int major = 0, minor = 0;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  if (major != 10 || minor != 3)
    return fail(M2_EDEVICE, "device %d is sm_%d%d; libm2 is built for sm_103a only", dev, major, minor);
  return M2_OK;
}

inline size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }

// Bump allocator over a caller-provided workspace.
struct Carve {
  char* base;
  size_t off = 0;
  template <class T>
  T* take(size_t count) {
    T* p = reinterpret_cast<T*>(base ? base + off : nullptr);
    off = align256(off + count * sizeof(T));
    return p;
  }
};

// The error word of the standalone entry points (fp8_linear, fp8_linear_bf16,
// bf16_linear, fp8_linear_noalloc): one file-scope device int per device,
// found once per device; m2_check_standalone reads and clears it.
m2_status standalone_error_word(int** out);

}  // namespace

struct m2_handle {
  int device;
  m2_config cfg;
  uint8_t* in_proj = nullptr;
  uint8_t* out_proj = nullptr;
  float s_w1 = 0, s_w2 = 0;
  // W8A16 arm: both projections dequantised to bf16 at creation
  uint16_t* in_proj_bf16 = nullptr;
  uint16_t* out_proj_bf16 = nullptr;
  bool w8a16() const { return cfg.arm == M2_ARM_W8A16; }
  uint16_t* conv_w = nullptr;
  uint16_t* conv_b = nullptr;
  float* A_log = nullptr;
  float* D = nullptr;
  float* dt_bias = nullptr;
  uint16_t* norm_w = nullptr;
  int* err = nullptr;
  // second stream and fork/join events of m2_mixed (decode rows run beside
  // the prefill rows' scan)
  cudaStream_t side = nullptr;
  cudaEvent_t fork_ev = nullptr, join_ev = nullptr, cum_ev = nullptr;
  m2_stats stats;
  bool taps_on = false;
  m2_taps taps;
  // stage timing
  struct StageRec {
    int stage, launches;
    cudaEvent_t a, b;
  };
  bool prof_on = false;
  std::vector<cudaEvent_t> ev_free;
  std::vector<StageRec> recs;
  cudaEvent_t take_event() {
    if (!ev_free.empty()) {
      cudaEvent_t e = ev_free.back();
      ev_free.pop_back();
      return e;
    }
    cudaEvent_t e = nullptr;
    cudaEventCreate(&e);
    return e;
  }

  BlockParams params() const {
    BlockParams bp;
    bp.conv_w = conv_w;
    bp.conv_b = conv_b;
    bp.A_log = A_log;
    bp.D = D;
    bp.dt_bias = dt_bias;
    bp.norm_w = norm_w;
    bp.eps = cfg.eps;
    bp.s_x = cfg.s_x;
    bp.s_y = cfg.s_y;
    return bp;
  }
};

extern "C" {

const char* m2_last_error(void) { return g_err.c_str(); }

static m2_status upload(m2_handle* h, void** dst, const void* src, size_t bytes) {
  M2_CUDA(cudaMalloc(dst, bytes));
  M2_CUDA(cudaMemcpy(*dst, src, bytes, cudaMemcpyDefault));
  h->stats.bytes_uploaded += bytes;
  return M2_OK;
}

m2_status m2_create(const m2_config* cfg, const m2_weights* w, m2_handle** out) {
  g_err.clear();
  if (!cfg || !w || !out) return fail(M2_EINVAL, "m2_create: null argument");
  *out = nullptr;
  if (cfg->hidden != kH || cfg->d_inner != kI || cfg->nheads != kNH || cfg->headdim != kP ||
      cfg->n_groups != kG || cfg->d_state != kN || cfg->conv_width != kW)
    return fail(M2_ESHAPE,
                "m2_create: geometry (hidden %d, d_inner %d, nheads %d, headdim %d, n_groups %d, d_state %d, "
                "conv %d) is not the supported (2688, 4096, 64, 64, 8, 128, 4)",
                cfg->hidden, cfg->d_inner, cfg->nheads, cfg->headdim, cfg->n_groups, cfg->d_state,
                cfg->conv_width);
  if (cfg->chunk_size != kChunk) return fail(M2_ESHAPE, "m2_create: chunk_size %d is not 256", cfg->chunk_size);
  if (cfg->ssm_dtype != M2_DTYPE_F32 && cfg->ssm_dtype != M2_DTYPE_BF16)
    return fail(M2_EINVAL, "m2_create: ssm_dtype must be M2_DTYPE_F32 or M2_DTYPE_BF16");
  if (cfg->arm != M2_ARM_W8A8 && cfg->arm != M2_ARM_W8A16)
    return fail(M2_EINVAL, "m2_create: arm must be M2_ARM_W8A8 or M2_ARM_W8A16");
  if (!(cfg->eps > 0.f) || !(cfg->s_x > 0.f) || !(cfg->s_y > 0.f) || !(cfg->s_x < 3.0e38f) ||
      !(cfg->s_y < 3.0e38f))
    return fail(M2_EINVAL, "m2_create: eps and activation scales must be positive and finite");
  if (!(w->s_w1 > 0.f) || !(w->s_w2 > 0.f) || !(w->s_w1 < 3.0e38f) || !(w->s_w2 < 3.0e38f))
    return fail(M2_EINVAL, "m2_create: weight scales must be positive and finite");
  if (w->layout != M2_LAYOUT_OUT_IN)
    return fail(M2_EINVAL, "m2_create: projection weights must be stored [out, in]");
  if (!w->in_proj || !w->out_proj || !w->conv_w || !w->A_log || !w->D || !w->dt_bias || !w->norm_w)
    return fail(M2_EINVAL, "m2_create: a required weight pointer is null");
  m2_status st = check_device();
  if (st) return st;

  m2_handle* h = new m2_handle();
  memset(&h->stats, 0, sizeof h->stats);
  memset(&h->taps, 0, sizeof h->taps);
  cudaGetDevice(&h->device);
  h->cfg = *cfg;
  h->s_w1 = w->s_w1;
  h->s_w2 = w->s_w2;
  m2_status s = M2_OK;
  if (!s) s = upload(h, (void**)&h->in_proj, w->in_proj, (size_t)kZ * kH);
  if (!s) s = upload(h, (void**)&h->out_proj, w->out_proj, (size_t)kH * kI);
  if (!s) s = upload(h, (void**)&h->conv_w, w->conv_w, (size_t)kConv * kW * 2);
  if (!s && w->conv_b) s = upload(h, (void**)&h->conv_b, w->conv_b, (size_t)kConv * 2);
  if (!s) s = upload(h, (void**)&h->A_log, w->A_log, kNH * 4);
  if (!s) s = upload(h, (void**)&h->D, w->D, kNH * 4);
  if (!s) s = upload(h, (void**)&h->dt_bias, w->dt_bias, kNH * 4);
  if (!s) s = upload(h, (void**)&h->norm_w, w->norm_w, (size_t)kI * 2);
  if (!s && h->w8a16()) {
    cudaError_t e = cudaMalloc((void**)&h->in_proj_bf16, (size_t)kZ * kH * 2);
    if (e == cudaSuccess) e = cudaMalloc((void**)&h->out_proj_bf16, (size_t)kH * kI * 2);
    if (e == cudaSuccess) e = launch_dequant_e4m3_bf16(h->in_proj, (size_t)kZ * kH, h->s_w1, h->in_proj_bf16, 0);
    if (e == cudaSuccess) e = launch_dequant_e4m3_bf16(h->out_proj, (size_t)kH * kI, h->s_w2, h->out_proj_bf16, 0);
    if (e != cudaSuccess) s = fail(M2_ECUDA, "m2_create: W8A16 weights: %s", cudaGetErrorString(e));
  }
  if (!s) {
    cudaError_t e = cudaMalloc((void**)&h->err, sizeof(int));
    if (e == cudaSuccess) e = cudaMemset(h->err, 0, sizeof(int));
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&h->side, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&h->fork_ev, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&h->join_ev, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&h->cum_ev, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) s = fail(M2_ECUDA, "m2_create: %s", cudaGetErrorString(e));
  }
  if (s) {
    m2_destroy(h);
    return s;
  }
  *out = h;
  return M2_OK;
}

void m2_destroy(m2_handle* h) {
  if (!h) return;
  int prev = 0;
  cudaGetDevice(&prev);
  cudaSetDevice(h->device);
  cudaDeviceSynchronize();
  cudaFree(h->in_proj);
  cudaFree(h->out_proj);
  cudaFree(h->in_proj_bf16);
  cudaFree(h->out_proj_bf16);
  cudaFree(h->conv_w);
  cudaFree(h->conv_b);
  cudaFree(h->A_log);
  cudaFree(h->D);
  cudaFree(h->dt_bias);
  cudaFree(h->norm_w);
  cudaFree(h->err);
  if (h->fork_ev) cudaEventDestroy(h->fork_ev);
  if (h->join_ev) cudaEventDestroy(h->join_ev);
  if (h->cum_ev) cudaEventDestroy(h->cum_ev);
  if (h->side) cudaStreamDestroy(h->side);
  for (auto& r : h->recs) {
    cudaEventDestroy(r.a);
    cudaEventDestroy(r.b);
  }
  for (auto e : h->ev_free) cudaEventDestroy(e);
  cudaSetDevice(prev);
  delete h;
}

m2_status m2_get_stats(const m2_handle* h, m2_stats* out) {
  if (!h || !out) return fail(M2_EINVAL, "m2_get_stats: null argument");
  *out = h->stats;
  return M2_OK;
}

m2_status m2_set_taps(m2_handle* h, const m2_taps* taps) {
  if (!h) return fail(M2_EINVAL, "m2_set_taps: null handle");
  if (taps) {
    h->taps = *taps;
    h->taps_on = true;
  } else {
    memset(&h->taps, 0, sizeof h->taps);
    h->taps_on = false;
  }
  return M2_OK;
}

m2_status m2_profile_enable(m2_handle* h, int on) {
  if (!h) return fail(M2_EINVAL, "m2_profile_enable: null handle");
  h->prof_on = on != 0;
  if (!h->prof_on) {
    for (auto& r : h->recs) {
      h->ev_free.push_back(r.a);
      h->ev_free.push_back(r.b);
    }
    h->recs.clear();
  }
  return M2_OK;
}

m2_status m2_profile_read(m2_handle* h, double* ms, uint64_t* launches) {
  if (!h) return fail(M2_EINVAL, "m2_profile_read: null handle");
  for (auto& r : h->recs) {
    M2_CUDA(cudaEventSynchronize(r.b));
    float t = 0.f;
    M2_CUDA(cudaEventElapsedTime(&t, r.a, r.b));
    if (r.stage >= 0 && r.stage < M2_NSTAGES) {
      if (ms) ms[r.stage] += t;
      if (launches) launches[r.stage] += (uint64_t)r.launches;
    }
    h->ev_free.push_back(r.a);
    h->ev_free.push_back(r.b);
  }
  h->recs.clear();
  return M2_OK;
}

// Status of a device error word's bits (timeouts first: they leave outputs
// incomplete).
static m2_status error_word_status(int v, const char* who) {
  if (v & kErrTimeout) return fail(M2_ETIMEOUT, "%s: a bounded device wait ran out", who);
  if (v & kErrSlot) return fail(M2_EINVAL, "%s: a decode row named a slot outside [0, n_slots)", who);
  if (v & kErrDupSlot)
    return fail(M2_EINVAL, "%s: two decode rows named the same slot (the later rows were skipped)", who);
  return M2_OK;
}

m2_status m2_check(m2_handle* h) {
  if (!h) return fail(M2_EINVAL, "m2_check: null handle");
  int v = 0;
  M2_CUDA(cudaDeviceSynchronize());
  M2_CUDA(cudaMemcpy(&v, h->err, sizeof v, cudaMemcpyDeviceToHost));
  M2_CUDA(cudaMemset(h->err, 0, sizeof(int)));
  return error_word_status(v, "m2_check");
}

m2_status m2_selftest_timeout(m2_handle* h, unsigned limit_us, void* stream) {
  g_err.clear();
  if (limit_us < 1 || limit_us > 100000)
    return fail(M2_EINVAL, "m2_selftest_timeout: limit_us %u not in [1, 100000]", limit_us);
  int* err = nullptr;
  if (h) {
    err = h->err;
  } else {
    m2_status s = check_device();
    if (s) return s;
    if ((s = standalone_error_word(&err))) return s;
  }
  M2_CUDA(launch_wait_selftest((uint64_t)limit_us * 1000ull, err, static_cast<cudaStream_t>(stream)));
  if (h) h->stats.kernel_launches += 1;
  return M2_OK;
}

// ---------------------------------------------------------------- prefill

static m2_status build_seqinfo(const int32_t* seqlens, int nseq, const uint8_t* has_initial, SeqInfo* si) {
  if (nseq < 1 || nseq > kMaxSeq) return fail(M2_ESHAPE, "m2_prefill: nseq %d not in [1, %d]", nseq, kMaxSeq);
  if (!seqlens) return fail(M2_EINVAL, "m2_prefill: seqlens is null");
  memset(si, 0, sizeof *si);
  si->nseq = nseq;
  long long tok = 0, ch = 0;
  for (int s = 0; s < nseq; ++s) {
    if (seqlens[s] < 1) return fail(M2_ESHAPE, "m2_prefill: seqlens[%d] = %d < 1", s, seqlens[s]);
    si->cu_seqlens[s] = (int)tok;
    si->cu_chunks[s] = (int)ch;
    tok += seqlens[s];
    ch += (seqlens[s] + kChunk - 1) / kChunk;
    if (tok > (1 << 24)) return fail(M2_ESHAPE, "m2_prefill: more than 2^24 tokens in one call");
    if (has_initial && has_initial[s]) si->has_init[s >> 5] |= 1u << (s & 31);
  }
  si->cu_seqlens[nseq] = (int)tok;
  si->cu_chunks[nseq] = (int)ch;
  si->total_tokens = (int)tok;
  si->total_chunks = (int)ch;
  return M2_OK;
}

struct PrefillWs {
  uint8_t* q;
  uint16_t* zx;
  uint16_t* u;
  CumDt* cumdt;
  float* states;
  uint8_t* sin_img;
  uint16_t* y;
  uint8_t* q2;
  uint16_t* o;   // W8A16 arm: the gated-norm output, out_proj's bf16 input
  void* gemm_ws;
  size_t gemm_ws_bytes;
  size_t total;
};

static PrefillWs carve_prefill(void* base, int T, int chunks, bool w8a16) {
  Carve c{static_cast<char*>(base)};
  PrefillWs w;
  w.q = w8a16 ? nullptr : c.take<uint8_t>((size_t)T * kH);
  w.zx = c.take<uint16_t>((size_t)T * kZ);
  w.u = c.take<uint16_t>((size_t)T * kConv);
  w.cumdt = c.take<CumDt>((size_t)chunks * kNH);
  w.states = c.take<float>((size_t)chunks * kNH * kP * kN);
  w.sin_img = c.take<uint8_t>((size_t)chunks * kNH * kSinImageBytes);
  w.y = c.take<uint16_t>((size_t)T * kI);
  w.q2 = c.take<uint8_t>((size_t)T * kI);
  w.o = w8a16 ? c.take<uint16_t>((size_t)T * kI) : nullptr;
  size_t g1 = w8a16 ? gemm_workspace_bytes_bf16(T, kZ, kH) : gemm_workspace_bytes(T, kZ, kH);
  size_t g2 = w8a16 ? gemm_workspace_bytes_bf16(T, kH, kI) : gemm_workspace_bytes(T, kH, kI);
  w.gemm_ws_bytes = g1 > g2 ? g1 : g2;
  w.gemm_ws = c.take<char>(w.gemm_ws_bytes);
  w.total = c.off;
  return w;
}

m2_status m2_prefill_workspace_size(const m2_handle* h, const int32_t* seqlens_host, int nseq, size_t* bytes) {
  if (!h || !bytes) return fail(M2_EINVAL, "m2_prefill_workspace_size: null argument");
  SeqInfo si;
  m2_status s = build_seqinfo(seqlens_host, nseq, nullptr, &si);
  if (s) return s;
  *bytes = carve_prefill(nullptr, si.total_tokens, si.total_chunks, h->w8a16()).total;
  return M2_OK;
}

// Longest sequence of a call: at most kRecMaxT tokens takes the token-by-token
// SSD kernel (one launch) instead of the chunked stages (four launches).
static int max_seqlen(const SeqInfo& si) {
  int m = 0;
  for (int i = 0; i < si.nseq; ++i) m = std::max(m, si.cu_seqlens[i + 1] - si.cu_seqlens[i]);
  return m;
}

static m2_status copy_tap(void* dst, const void* src, size_t bytes, cudaStream_t st) {
  if (!dst) return M2_OK;
  M2_CUDA(cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDeviceToDevice, st));
  return M2_OK;
}

// The block's prefill from bf16 hidden (quantised here) or from hidden_q,
// already quantised with the handle's s_x (exactly one of the two given).
static m2_status prefill_impl(m2_handle* h, const uint16_t* hidden, const uint8_t* hidden_q,
                              const int32_t* seqlens_host, int nseq, const uint8_t* has_initial,
                              uint16_t* conv_state, void* ssm_state, uint16_t* out, void* workspace,
                              size_t ws_bytes, void* stream) {
  g_err.clear();
  if (!h || (!hidden && !hidden_q) || !conv_state || !ssm_state || !out || !workspace)
    return fail(M2_EINVAL, "m2_prefill: null argument");
  if ((uintptr_t)workspace % 256) return fail(M2_EINVAL, "m2_prefill: workspace must be 256-byte aligned");
  if ((uintptr_t)hidden % 16 || (uintptr_t)hidden_q % 16 || (uintptr_t)out % 16 || (uintptr_t)ssm_state % 16)
    return fail(M2_EINVAL, "m2_prefill: hidden, out and ssm_state must be 16-byte aligned");
  if (hidden_q && h->w8a16())
    return fail(M2_EINVAL, "m2_prefill_q: the W8A16 arm takes bf16 activations (input_scale is not applied)");
  SeqInfo local;
  m2_status s = build_seqinfo(seqlens_host, nseq, has_initial, &local);
  if (s) return s;
  const int T = local.total_tokens;
  const bool w8a16 = h->w8a16();
  PrefillWs w = carve_prefill(workspace, T, local.total_chunks, w8a16);
  if (ws_bytes < w.total)
    return fail(M2_ENOMEM, "m2_prefill: workspace %zu bytes < %zu needed", ws_bytes, w.total);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const BlockParams bp = h->params();
  const float sc1 = h->cfg.s_x * h->s_w1, sc2 = h->cfg.s_y * h->s_w2;

  int nl = 0;
  const uint8_t* q = hidden_q ? hidden_q : w.q;
  if (w8a16) {
    M2_STAGE(h, st, M2_STAGE_IN_PROJ, nl,
             gemm_bf16(hidden, h->in_proj_bf16, w.zx, T, kZ, kH, 1.0f, w.gemm_ws, w.gemm_ws_bytes, h->err, st, &nl, true));
  } else {
    if (!hidden_q)
      M2_STAGE(h, st, M2_STAGE_QUANT_IN, 1, launch_quant_e4m3(hidden, (size_t)T * kH, h->cfg.s_x, w.q, st));
    M2_STAGE(h, st, M2_STAGE_IN_PROJ, nl,
             gemm_fp8(q, h->in_proj, w.zx, T, kZ, kH, sc1, w.gemm_ws, w.gemm_ws_bytes, h->err, st, &nl, true));
  }
  const bool recur = max_seqlen(local) <= kRecMaxT;
  const bool bf16_state = h->cfg.ssm_dtype == M2_DTYPE_BF16;
  // the cumsum reads only the in_proj output: it runs on the second stream
  // beside the conv (serially while stage profiling)
  float* dt_tap = h->taps_on ? h->taps.dt : nullptr;
  if (!h->prof_on && !recur) {
    M2_CUDA(cudaEventRecord(h->fork_ev, st));
    M2_CUDA(cudaStreamWaitEvent(h->side, h->fork_ev, 0));
    M2_CUDA(launch_ssd_cumsum(w.zx, bp, local, w.cumdt, dt_tap, h->side));
    h->stats.kernel_launches += 1;
    M2_CUDA(cudaEventRecord(h->cum_ev, h->side));
  }
  M2_STAGE(h, st, M2_STAGE_CONV, 1, launch_conv_silu_prefill(w.zx, bp, conv_state, local, w.u, st));
  if (recur) {
    // short sequences: the recurrence token by token (profiled as the scan)
    M2_STAGE(h, st, M2_STAGE_SSD_CHUNK_SCAN, 1,
             launch_ssd_recurrent(w.zx, w.u, bp, local, w.y, ssm_state, bf16_state, conv_state, dt_tap, st));
  } else {
    if (h->prof_on) {
      M2_STAGE(h, st, M2_STAGE_SSD_CUMSUM, 1, launch_ssd_cumsum(w.zx, bp, local, w.cumdt, dt_tap, st));
    } else {
      M2_CUDA(cudaStreamWaitEvent(st, h->cum_ev, 0));
    }
    M2_STAGE(h, st, M2_STAGE_SSD_CHUNK_STATE, 1,
             launch_ssd_chunk_state_tc(w.u, w.cumdt, local, w.states, h->err, st));
    M2_STAGE(h, st, M2_STAGE_SSD_STATE_PASS, 1,
             launch_ssd_state_pass(w.states, w.cumdt, local, w.sin_img, ssm_state, bf16_state, w.zx, conv_state, st));
    M2_STAGE(h, st, M2_STAGE_SSD_CHUNK_SCAN, 1,
             launch_ssd_chunk_scan_tc(w.u, w.cumdt, w.sin_img, bp, local, w.y, h->err, st));
  }
  if (w8a16) {
    // the bf16 normed output feeds out_proj (the e4m3 codes are written too, unused)
    M2_STAGE(h, st, M2_STAGE_NORM_QUANT, 1, launch_gated_norm_quant(w.y, w.zx, bp, T, w.q2, w.o, st));
    M2_STAGE(h, st, M2_STAGE_OUT_PROJ, nl,
             gemm_bf16(w.o, h->out_proj_bf16, out, T, kH, kI, 1.0f, w.gemm_ws, w.gemm_ws_bytes, h->err, st, &nl, true));
  } else {
    M2_STAGE(h, st, M2_STAGE_NORM_QUANT, 1,
             launch_gated_norm_quant(w.y, w.zx, bp, T, w.q2, h->taps_on ? h->taps.o : nullptr, st));
    M2_STAGE(h, st, M2_STAGE_OUT_PROJ, nl,
             gemm_fp8(w.q2, h->out_proj, out, T, kH, kI, sc2, w.gemm_ws, w.gemm_ws_bytes, h->err, st, &nl, true));
  }
  if (h->taps_on) {
    if (w8a16) {
      if ((s = copy_tap(h->taps.o, w.o, (size_t)T * kI * 2, st))) return s;
    } else {
      if ((s = copy_tap(h->taps.q, q, (size_t)T * kH, st))) return s;
    }
    if ((s = copy_tap(h->taps.zx, w.zx, (size_t)T * kZ * 2, st))) return s;
    if ((s = copy_tap(h->taps.u, w.u, (size_t)T * kConv * 2, st))) return s;
    if ((s = copy_tap(h->taps.y, w.y, (size_t)T * kI * 2, st))) return s;
    if ((s = copy_tap(h->taps.q2, w.q2, (size_t)T * kI, st))) return s;
  }
  h->stats.prefill_calls += 1;
  h->stats.conv_fwd_calls += 1;
  h->stats.chunk_scan_calls += 1;
  return M2_OK;
}

m2_status m2_prefill(m2_handle* h, const uint16_t* hidden, const int32_t* seqlens_host, int nseq,
                     const uint8_t* has_initial, uint16_t* conv_state, void* ssm_state, uint16_t* out,
                     void* workspace, size_t ws_bytes, void* stream) {
  if (!hidden) return fail(M2_EINVAL, "m2_prefill: null argument");
  return prefill_impl(h, hidden, nullptr, seqlens_host, nseq, has_initial, conv_state, ssm_state, out, workspace,
                      ws_bytes, stream);
}

m2_status m2_prefill_q(m2_handle* h, const uint8_t* hidden_q, const int32_t* seqlens_host, int nseq,
                       const uint8_t* has_initial, uint16_t* conv_state, void* ssm_state, uint16_t* out,
                       void* workspace, size_t ws_bytes, void* stream) {
  if (!hidden_q) return fail(M2_EINVAL, "m2_prefill_q: null argument");
  return prefill_impl(h, nullptr, hidden_q, seqlens_host, nseq, has_initial, conv_state, ssm_state, out, workspace,
                      ws_bytes, stream);
}

// ---------------------------------------------------------------- decode

struct DecodeWs {
  uint8_t* q;
  uint16_t* zx;
  uint8_t* q2;
  uint16_t* o;   // W8A16 arm: the gated-norm output, out_proj's bf16 input
  void* gemm_ws;
  size_t gemm_ws_bytes;
  size_t total;
};

static DecodeWs carve_decode(void* base, int Bt, bool w8a16) {
  Carve c{static_cast<char*>(base)};
  DecodeWs w;
  w.q = w8a16 ? nullptr : c.take<uint8_t>((size_t)Bt * kH);
  w.zx = c.take<uint16_t>((size_t)Bt * kZ);
  w.q2 = c.take<uint8_t>((size_t)Bt * kI);
  w.o = w8a16 ? c.take<uint16_t>((size_t)Bt * kI) : nullptr;
  size_t g1 = w8a16 ? gemm_workspace_bytes_bf16(Bt, kZ, kH) : gemm_workspace_bytes(Bt, kZ, kH);
  size_t g2 = w8a16 ? gemm_workspace_bytes_bf16(Bt, kH, kI) : gemm_workspace_bytes(Bt, kH, kI);
  w.gemm_ws_bytes = g1 > g2 ? g1 : g2;
  w.gemm_ws = c.take<char>(w.gemm_ws_bytes);
  w.total = c.off;
  return w;
}

m2_status m2_decode_workspace_size(const m2_handle* h, int Bt, size_t* bytes) {
  if (!h || !bytes) return fail(M2_EINVAL, "m2_decode_workspace_size: null argument");
  if (Bt < 1 || Bt > 4096) return fail(M2_ESHAPE, "m2_decode: Bt %d not in [1, 4096]", Bt);
  *bytes = carve_decode(nullptr, Bt, h->w8a16()).total;
  return M2_OK;
}

static m2_status decode_impl(m2_handle* h, const uint16_t* hidden, const uint8_t* hidden_q, int Bt,
                             uint16_t* conv_pool, void* ssm_pool, int n_slots, const int32_t* slot_idx,
                             uint16_t* out, void* workspace, size_t ws_bytes, void* stream) {
  g_err.clear();
  if (!h || (!hidden && !hidden_q) || !conv_pool || !ssm_pool || !slot_idx || !out || !workspace)
    return fail(M2_EINVAL, "m2_decode: null argument");
  if (Bt < 1 || Bt > 4096) return fail(M2_ESHAPE, "m2_decode: Bt %d not in [1, 4096]", Bt);
  if (n_slots < 1) return fail(M2_EINVAL, "m2_decode: n_slots %d < 1", n_slots);
  if ((uintptr_t)workspace % 256) return fail(M2_EINVAL, "m2_decode: workspace must be 256-byte aligned");
  if ((uintptr_t)hidden % 16 || (uintptr_t)hidden_q % 16 || (uintptr_t)out % 16 || (uintptr_t)ssm_pool % 16)
    return fail(M2_EINVAL, "m2_decode: hidden, out and ssm_pool must be 16-byte aligned");
  if (hidden_q && h->w8a16())
    return fail(M2_EINVAL, "m2_decode_q: the W8A16 arm takes bf16 activations (input_scale is not applied)");
  const bool w8a16 = h->w8a16();
  DecodeWs w = carve_decode(workspace, Bt, w8a16);
  if (ws_bytes < w.total) return fail(M2_ENOMEM, "m2_decode: workspace %zu bytes < %zu needed", ws_bytes, w.total);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const BlockParams bp = h->params();
  const float sc1 = h->cfg.s_x * h->s_w1, sc2 = h->cfg.s_y * h->s_w2;
  DecodeTaps dt{};
  if (h->taps_on) {
    dt.u = h->taps.u;
    dt.dt = h->taps.dt;
    dt.y = h->taps.y;
    dt.o = h->taps.o;
  }
  int nl = 0;
  const uint8_t* q = hidden_q ? hidden_q : w.q;
  if (w8a16) {
    M2_STAGE(h, st, M2_STAGE_DEC_IN_PROJ, nl,
             gemm_bf16(hidden, h->in_proj_bf16, w.zx, Bt, kZ, kH, 1.0f, w.gemm_ws, w.gemm_ws_bytes, h->err, st, &nl, true));
    // the kernel writes the bf16 normed rows through its o output, which
    // skips padding rows: those stay zero, so their output rows are zero
    M2_CUDA(cudaMemsetAsync(w.o, 0, (size_t)Bt * kI * 2, st));
    dt.o = w.o;
  } else {
    if (!hidden_q)
      M2_STAGE(h, st, M2_STAGE_DEC_QUANT_IN, 1, launch_quant_e4m3(hidden, (size_t)Bt * kH, h->cfg.s_x, w.q, st));
    M2_STAGE(h, st, M2_STAGE_DEC_IN_PROJ, nl,
             gemm_fp8(q, h->in_proj, w.zx, Bt, kZ, kH, sc1, w.gemm_ws, w.gemm_ws_bytes, h->err, st, &nl, true));
  }
  // the state kernel also brings out_proj's weights into L2 for the next kernel
  const void* w2 = w8a16 ? (const void*)h->out_proj_bf16 : (const void*)h->out_proj;
  const size_t w2_bytes = (size_t)kH * kI * (w8a16 ? 2 : 1);
  M2_STAGE(h, st, M2_STAGE_DECODE_FUSED, nl,
           launch_decode_stream(w.zx, bp, conv_pool, ssm_pool, h->cfg.ssm_dtype == M2_DTYPE_BF16, n_slots, slot_idx,
                                Bt, w.q2, h->err, dt, st, &nl, w2, w2_bytes));
  if (w8a16) {
    M2_STAGE(h, st, M2_STAGE_DEC_OUT_PROJ, nl,
             gemm_bf16(w.o, h->out_proj_bf16, out, Bt, kH, kI, 1.0f, w.gemm_ws, w.gemm_ws_bytes, h->err, st, &nl, true));
  } else {
    M2_STAGE(h, st, M2_STAGE_DEC_OUT_PROJ, nl,
             gemm_fp8(w.q2, h->out_proj, out, Bt, kH, kI, sc2, w.gemm_ws, w.gemm_ws_bytes, h->err, st, &nl, true));
  }
  if (h->taps_on) {
    m2_status s;
    if (w8a16) {
      if ((s = copy_tap(h->taps.o, w.o, (size_t)Bt * kI * 2, st))) return s;
    } else {
      if ((s = copy_tap(h->taps.q, q, (size_t)Bt * kH, st))) return s;
    }
    if ((s = copy_tap(h->taps.zx, w.zx, (size_t)Bt * kZ * 2, st))) return s;
    if ((s = copy_tap(h->taps.q2, w.q2, (size_t)Bt * kI, st))) return s;
  }
  h->stats.decode_calls += 1;
  h->stats.conv_update_rows += (uint64_t)Bt;
  h->stats.state_update_rows += (uint64_t)Bt;
  return M2_OK;
}

m2_status m2_decode(m2_handle* h, const uint16_t* hidden, int Bt, uint16_t* conv_pool, void* ssm_pool,
                    int n_slots, const int32_t* slot_idx, uint16_t* out, void* workspace, size_t ws_bytes,
                    void* stream) {
  if (!hidden) return fail(M2_EINVAL, "m2_decode: null argument");
  return decode_impl(h, hidden, nullptr, Bt, conv_pool, ssm_pool, n_slots, slot_idx, out, workspace, ws_bytes,
                     stream);
}

m2_status m2_decode_q(m2_handle* h, const uint8_t* hidden_q, int Bt, uint16_t* conv_pool, void* ssm_pool,
                      int n_slots, const int32_t* slot_idx, uint16_t* out, void* workspace, size_t ws_bytes,
                      void* stream) {
  if (!hidden_q) return fail(M2_EINVAL, "m2_decode_q: null argument");
  return decode_impl(h, nullptr, hidden_q, Bt, conv_pool, ssm_pool, n_slots, slot_idx, out, workspace, ws_bytes,
                     stream);
}

// ---------------------------------------------------------------- mixed batch

// One call over an ordered batch: Bt decode rows (one token each, state in
// the slot pool) followed by nseq packed prefill sequences.  The input quant
// and both projections run once over all Bt + T rows; the decode rows take
// the paged state kernel, the prefill rows the SSD path.
struct MixedWs {
  PrefillWs pf;   // prefill-only buffers (u, cum/dt, states, S_in, y) of T tokens
  uint8_t* q;     // [Bt + T, 2688]
  uint16_t* zx;   // [Bt + T, 10304]
  uint8_t* q2;    // [Bt + T, 4096]
  void* gemm_ws;
  size_t gemm_ws_bytes;
  size_t total;
};

static MixedWs carve_mixed(void* base, int Bt, int T, int chunks) {
  Carve c{static_cast<char*>(base)};
  MixedWs w;
  const size_t R = (size_t)Bt + T;
  w.q = c.take<uint8_t>(R * kH);
  w.zx = c.take<uint16_t>(R * kZ);
  w.q2 = c.take<uint8_t>(R * kI);
  w.pf = PrefillWs{};
  w.pf.u = c.take<uint16_t>((size_t)T * kConv);
  w.pf.cumdt = c.take<CumDt>((size_t)chunks * kNH);
  w.pf.states = c.take<float>((size_t)chunks * kNH * kP * kN);
  w.pf.sin_img = c.take<uint8_t>((size_t)chunks * kNH * kSinImageBytes);
  w.pf.y = c.take<uint16_t>((size_t)T * kI);
  size_t g1 = gemm_workspace_bytes((int)R, kZ, kH), g2 = gemm_workspace_bytes((int)R, kH, kI);
  w.gemm_ws_bytes = g1 > g2 ? g1 : g2;
  w.gemm_ws = c.take<char>(w.gemm_ws_bytes);
  w.total = c.off;
  return w;
}

m2_status m2_mixed_workspace_size(const m2_handle* h, int Bt, const int32_t* seqlens_host, int nseq,
                                  size_t* bytes) {
  if (!h || !bytes) return fail(M2_EINVAL, "m2_mixed_workspace_size: null argument");
  if (h->w8a16()) return fail(M2_EINVAL, "m2_mixed: not offered for the W8A16 arm (use m2_prefill and m2_decode)");
  if (Bt < 0 || Bt > 4096) return fail(M2_ESHAPE, "m2_mixed: Bt %d not in [0, 4096]", Bt);
  SeqInfo si;
  memset(&si, 0, sizeof si);
  if (nseq > 0) {
    m2_status s = build_seqinfo(seqlens_host, nseq, nullptr, &si);
    if (s) return s;
  } else if (nseq < 0) {
    return fail(M2_ESHAPE, "m2_mixed: nseq %d < 0", nseq);
  }
  if (Bt + si.total_tokens < 1) return fail(M2_ESHAPE, "m2_mixed: empty batch");
  *bytes = carve_mixed(nullptr, Bt, si.total_tokens, si.total_chunks).total;
  return M2_OK;
}

m2_status m2_mixed(m2_handle* h, const uint16_t* hidden, int Bt, uint16_t* conv_pool, void* ssm_pool, int n_slots,
                   const int32_t* slot_idx, const int32_t* seqlens_host, int nseq, const uint8_t* has_initial,
                   uint16_t* conv_state, void* ssm_state, uint16_t* out, void* workspace, size_t ws_bytes,
                   void* stream) {
  g_err.clear();
  if (!h || !hidden || !out || !workspace) return fail(M2_EINVAL, "m2_mixed: null argument");
  if (h->w8a16()) return fail(M2_EINVAL, "m2_mixed: not offered for the W8A16 arm (use m2_prefill and m2_decode)");
  if (Bt < 0 || Bt > 4096) return fail(M2_ESHAPE, "m2_mixed: Bt %d not in [0, 4096]", Bt);
  if (nseq < 0) return fail(M2_ESHAPE, "m2_mixed: nseq %d < 0", nseq);
  if (Bt > 0 && (!conv_pool || !ssm_pool || !slot_idx || n_slots < 1))
    return fail(M2_EINVAL, "m2_mixed: decode rows need conv_pool, ssm_pool, slot_idx and n_slots >= 1");
  if (nseq > 0 && (!conv_state || !ssm_state)) return fail(M2_EINVAL, "m2_mixed: prefill rows need their states");
  if ((uintptr_t)workspace % 256) return fail(M2_EINVAL, "m2_mixed: workspace must be 256-byte aligned");
  if ((uintptr_t)hidden % 16 || (uintptr_t)out % 16 || (uintptr_t)ssm_pool % 16 || (uintptr_t)ssm_state % 16)
    return fail(M2_EINVAL, "m2_mixed: hidden, out and the state rows must be 16-byte aligned");
  SeqInfo local;
  memset(&local, 0, sizeof local);
  if (nseq > 0) {
    m2_status s = build_seqinfo(seqlens_host, nseq, has_initial, &local);
    if (s) return s;
  }
  const int T = local.total_tokens;
  const int R = Bt + T;
  if (R < 1) return fail(M2_ESHAPE, "m2_mixed: empty batch");
  MixedWs w = carve_mixed(workspace, Bt, T, local.total_chunks);
  if (ws_bytes < w.total) return fail(M2_ENOMEM, "m2_mixed: workspace %zu bytes < %zu needed", ws_bytes, w.total);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const BlockParams bp = h->params();
  const float sc1 = h->cfg.s_x * h->s_w1, sc2 = h->cfg.s_y * h->s_w2;
  const bool bf16_state = h->cfg.ssm_dtype == M2_DTYPE_BF16;
  // rows [0, Bt) are the decode rows, [Bt, R) the prefill tokens
  uint16_t* zx_pf = w.zx + (size_t)Bt * kZ;
  uint8_t* q2_pf = w.q2 + (size_t)Bt * kI;
  int nl = 0;
  M2_STAGE(h, st, M2_STAGE_QUANT_IN, 1, launch_quant_e4m3(hidden, (size_t)R * kH, h->cfg.s_x, w.q, st));
  M2_STAGE(h, st, M2_STAGE_IN_PROJ, nl,
           gemm_fp8(w.q, h->in_proj, w.zx, R, kZ, kH, sc1, w.gemm_ws, w.gemm_ws_bytes, h->err, st, &nl, true));
  // A second stream runs the prefill cumsum beside the conv (it reads only
  // the in_proj output), and the decode rows' state kernel beside the chunk
  // scan: that kernel is HBM-bound and the scan latency-bound, while next to
  // the chunk states or the state pass the two contend (the chunk states'
  // 230 KB CTAs wait for SMs the state kernel holds; the state pass is
  // HBM-bound too).  Measured on the mixed step of 64 decode rows and 4 x 2048
  // prefill tokens: started after the cumsum 0.470 ms, after the chunk states
  // 0.473, after the state pass 0.457, after the scan 0.475.  With the
  // token-by-token SSD path it starts at once.  The chunk states wait for the
  // cumsum, the out_proj for the decode rows.  Stage profiling keeps
  // everything on the caller's stream.
  const bool fork = !h->prof_on && T > 0;
  const bool fork_decode = fork && Bt > 0;
  const bool recur = T > 0 && max_seqlen(local) <= kRecMaxT;
  // the decode rows' state kernel on the second stream, after the work that
  // stream is already ordered behind
  auto decode_on_side = [&]() -> cudaError_t {
    DecodeTaps dt{};
    if (h->taps_on) dt.o = h->taps.o, dt.y = h->taps.y;
    int dl = 0;
    cudaError_t e = launch_decode_stream(w.zx, bp, conv_pool, ssm_pool, bf16_state, n_slots, slot_idx, Bt, w.q2,
                                         h->err, dt, h->side, &dl);
    if (e != cudaSuccess) return e;
    h->stats.kernel_launches += (uint64_t)dl;
    return cudaEventRecord(h->join_ev, h->side);
  };
  if (fork) {
    M2_CUDA(cudaEventRecord(h->fork_ev, st));
    M2_CUDA(cudaStreamWaitEvent(h->side, h->fork_ev, 0));
    if (!recur) {
      M2_CUDA(launch_ssd_cumsum(zx_pf, bp, local, w.pf.cumdt, nullptr, h->side));
      M2_CUDA(cudaEventRecord(h->cum_ev, h->side));
      h->stats.kernel_launches += 1;
    } else if (fork_decode) {
      M2_CUDA(decode_on_side());
    }
  }
  if (T > 0) {
    M2_STAGE(h, st, M2_STAGE_CONV, 1, launch_conv_silu_prefill(zx_pf, bp, conv_state, local, w.pf.u, st));
    if (recur) {
      M2_STAGE(h, st, M2_STAGE_SSD_CHUNK_SCAN, 1,
               launch_ssd_recurrent(zx_pf, w.pf.u, bp, local, w.pf.y, ssm_state, bf16_state, conv_state, nullptr,
                                    st));
    } else {
      if (fork) {
        M2_CUDA(cudaStreamWaitEvent(st, h->cum_ev, 0));
      } else {
        M2_STAGE(h, st, M2_STAGE_SSD_CUMSUM, 1, launch_ssd_cumsum(zx_pf, bp, local, w.pf.cumdt, nullptr, st));
      }
      M2_STAGE(h, st, M2_STAGE_SSD_CHUNK_STATE, 1,
               launch_ssd_chunk_state_tc(w.pf.u, w.pf.cumdt, local, w.pf.states, h->err, st));
      M2_STAGE(h, st, M2_STAGE_SSD_STATE_PASS, 1,
               launch_ssd_state_pass(w.pf.states, w.pf.cumdt, local, w.pf.sin_img, ssm_state, bf16_state, zx_pf,
                                     conv_state, st));
      if (fork_decode) {
        M2_CUDA(cudaEventRecord(h->fork_ev, st));
        M2_CUDA(cudaStreamWaitEvent(h->side, h->fork_ev, 0));
        M2_CUDA(decode_on_side());
      }
      M2_STAGE(h, st, M2_STAGE_SSD_CHUNK_SCAN, 1,
               launch_ssd_chunk_scan_tc(w.pf.u, w.pf.cumdt, w.pf.sin_img, bp, local, w.pf.y, h->err, st));
    }
    uint16_t* o_tap = (h->taps_on && h->taps.o) ? h->taps.o + (size_t)Bt * kI : nullptr;
    M2_STAGE(h, st, M2_STAGE_NORM_QUANT, 1, launch_gated_norm_quant(w.pf.y, zx_pf, bp, T, q2_pf, o_tap, st));
  }
  if (fork_decode) {
    M2_CUDA(cudaStreamWaitEvent(st, h->join_ev, 0));
  } else if (Bt > 0) {
    DecodeTaps dt{};
    if (h->taps_on) dt.o = h->taps.o, dt.y = h->taps.y;
    int dl = 0;
    M2_STAGE(h, st, M2_STAGE_DECODE_FUSED, dl,
             launch_decode_stream(w.zx, bp, conv_pool, ssm_pool, bf16_state, n_slots, slot_idx, Bt, w.q2, h->err,
                                  dt, st, &dl));
  }
  M2_STAGE(h, st, M2_STAGE_OUT_PROJ, nl,
           gemm_fp8(w.q2, h->out_proj, out, R, kH, kI, sc2, w.gemm_ws, w.gemm_ws_bytes, h->err, st, &nl, true));
  if (h->taps_on) {   // the row-aligned intermediates, in batch order
    m2_status s;
    if ((s = copy_tap(h->taps.q, w.q, (size_t)R * kH, st))) return s;
    if ((s = copy_tap(h->taps.zx, w.zx, (size_t)R * kZ * 2, st))) return s;
    if ((s = copy_tap(h->taps.q2, w.q2, (size_t)R * kI, st))) return s;
    if (h->taps.y && T > 0 && (s = copy_tap(h->taps.y + (size_t)Bt * kI, w.pf.y, (size_t)T * kI * 2, st))) return s;
  }
  if (T > 0) {
    h->stats.prefill_calls += 1;
    h->stats.conv_fwd_calls += 1;
    h->stats.chunk_scan_calls += 1;
  }
  if (Bt > 0) {
    h->stats.decode_calls += 1;
    h->stats.conv_update_rows += (uint64_t)Bt;
    h->stats.state_update_rows += (uint64_t)Bt;
  }
  return M2_OK;
}

// ---------------------------------------------------------------- standalone ops

m2_status fp8_quant(const uint16_t* x, size_t n, float scale, uint8_t* q, void* stream) {
  g_err.clear();
  if ((!x || !q) && n) return fail(M2_EINVAL, "fp8_quant: null pointer");
  if (!(scale > 0.f) || !(scale < 3.0e38f)) return fail(M2_EINVAL, "fp8_quant: scale must be positive and finite");
  m2_status s = check_device();
  if (s) return s;
  M2_CUDA(launch_quant_e4m3(x, n, scale, q, static_cast<cudaStream_t>(stream)));
  return M2_OK;
}

static m2_status check_linear(const void* a, const uint8_t* w, const uint16_t* y, int M, int N, int K, float s_a,
                              float s_w, const char* who) {
  if (M < 0 || N < 1 || K < 16) return fail(M2_ESHAPE, "%s: M %d, N %d, K %d out of range", who, M, N, K);
  if (K % 16) return fail(M2_ESHAPE, "%s: K %d must be a multiple of 16", who, K);
  if (M && (!a || !w || !y)) return fail(M2_EINVAL, "%s: null pointer", who);
  if ((uintptr_t)a % 16 || (uintptr_t)w % 16 || (uintptr_t)y % 16)
    return fail(M2_EINVAL, "%s: pointers must be 16-byte aligned", who);
  if (!(s_a > 0.f) || !(s_w > 0.f) || !(s_a < 3.0e38f) || !(s_w < 3.0e38f))
    return fail(M2_EINVAL, "%s: scales must be positive and finite", who);
  return check_device();
}

m2_status fp8_linear_workspace_size(int M, int N, int K, size_t* bytes) {
  if (!bytes) return fail(M2_EINVAL, "fp8_linear_workspace_size: null argument");
  if (M < 0 || N < 1 || K < 16 || K % 16) return fail(M2_ESHAPE, "fp8_linear_workspace_size: bad shape");
  *bytes = gemm_workspace_bytes(M, N, K);
  return M2_OK;
}

m2_status fp8_linear(const uint8_t* a_q, float s_a, const uint8_t* w_q, float s_w, uint16_t* y, int M, int N, int K,
                     void* workspace, size_t ws_bytes, void* stream) {
  g_err.clear();
  m2_status s = check_linear(a_q, w_q, y, M, N, K, s_a, s_w, "fp8_linear");
  if (s) return s;
  size_t need = gemm_workspace_bytes(M, N, K);
  if (ws_bytes < need || (need && !workspace))
    return fail(M2_ENOMEM, "fp8_linear: workspace %zu bytes < %zu needed", ws_bytes, need);
  int* err = nullptr;
  if ((s = standalone_error_word(&err))) return s;
  int nl = 0;
  M2_CUDA(gemm_fp8(a_q, w_q, y, M, N, K, s_a * s_w, workspace, ws_bytes, err, static_cast<cudaStream_t>(stream), &nl));
  return M2_OK;
}

m2_status fp8_linear_bf16(const uint16_t* x, float s_a, const uint8_t* w_q, float s_w, uint16_t* y, int M, int N,
                          int K, void* workspace, size_t ws_bytes, void* stream) {
  g_err.clear();
  m2_status s = check_linear(x, w_q, y, M, N, K, s_a, s_w, "fp8_linear_bf16");
  if (s) return s;
  if (!workspace || (uintptr_t)workspace % 256) return fail(M2_EINVAL, "fp8_linear_bf16: workspace must be 256-byte aligned");
  size_t qbytes = align256((size_t)M * K);
  size_t need = qbytes + gemm_workspace_bytes(M, N, K);
  if (ws_bytes < need) return fail(M2_ENOMEM, "fp8_linear_bf16: workspace %zu bytes < %zu needed", ws_bytes, need);
  int* err = nullptr;
  if ((s = standalone_error_word(&err))) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* q = static_cast<uint8_t*>(workspace);
  M2_CUDA(launch_quant_e4m3(x, (size_t)M * K, s_a, q, st));
  int nl = 0;
  M2_CUDA(gemm_fp8(q, w_q, y, M, N, K, s_a * s_w, static_cast<char*>(workspace) + qbytes, ws_bytes - qbytes, err, st, &nl));
  return M2_OK;
}

m2_status fp8_dequant(const uint8_t* q, size_t n, float scale, uint16_t* out, void* stream) {
  g_err.clear();
  if ((!q || !out) && n) return fail(M2_EINVAL, "fp8_dequant: null pointer");
  if ((uintptr_t)q % 8 || (uintptr_t)out % 16)
    return fail(M2_EINVAL, "fp8_dequant: q must be 8-byte and out 16-byte aligned");
  if (!(scale > 0.f) || !(scale < 3.0e38f)) return fail(M2_EINVAL, "fp8_dequant: scale must be positive and finite");
  m2_status s = check_device();
  if (s) return s;
  M2_CUDA(launch_dequant_e4m3_bf16(q, n, scale, out, static_cast<cudaStream_t>(stream)));
  return M2_OK;
}

m2_status bf16_linear_workspace_size(int M, int N, int K, size_t* bytes) {
  if (!bytes) return fail(M2_EINVAL, "bf16_linear_workspace_size: null argument");
  if (M < 0 || N < 1 || K < 16 || K % 16) return fail(M2_ESHAPE, "bf16_linear_workspace_size: bad shape");
  *bytes = gemm_workspace_bytes_bf16(M, N, K);
  return M2_OK;
}

m2_status bf16_linear(const uint16_t* x, const uint16_t* w, float scale, uint16_t* y, int M, int N, int K,
                      void* workspace, size_t ws_bytes, void* stream) {
  g_err.clear();
  if (M < 0 || N < 1 || K < 16) return fail(M2_ESHAPE, "bf16_linear: M %d, N %d, K %d out of range", M, N, K);
  if (K % 16) return fail(M2_ESHAPE, "bf16_linear: K %d must be a multiple of 16", K);
  if (M && (!x || !w || !y)) return fail(M2_EINVAL, "bf16_linear: null pointer");
  if ((uintptr_t)x % 16 || (uintptr_t)w % 16 || (uintptr_t)y % 16)
    return fail(M2_EINVAL, "bf16_linear: pointers must be 16-byte aligned");
  if (!(scale > 0.f) || !(scale < 3.0e38f)) return fail(M2_EINVAL, "bf16_linear: scale must be positive and finite");
  m2_status s = check_device();
  if (s) return s;
  const size_t need = gemm_workspace_bytes_bf16(M, N, K);
  if (ws_bytes < need || (need && !workspace))
    return fail(M2_ENOMEM, "bf16_linear: workspace %zu bytes < %zu needed", ws_bytes, need);
  int* err = nullptr;
  if ((s = standalone_error_word(&err))) return s;
  int nl = 0;
  M2_CUDA(gemm_bf16(x, w, y, M, N, K, scale, workspace, ws_bytes, err, static_cast<cudaStream_t>(stream), &nl));
  return M2_OK;
}

m2_status m2_rmsnorm_residual(uint16_t* h, const uint16_t* add, const uint16_t* w, float eps, uint16_t* normed, int T,
                              int n, void* stream) {
  g_err.clear();
  if (T < 0 || n < 8 || n % 8) return fail(M2_ESHAPE, "m2_rmsnorm_residual: T %d, n %d (n must be a multiple of 8)", T, n);
  if (T && (!h || (normed && !w) || (!normed && !add)))
    return fail(M2_EINVAL, "m2_rmsnorm_residual: null pointer");
  if ((uintptr_t)h % 16 || (uintptr_t)add % 16 || (uintptr_t)w % 16 || (uintptr_t)normed % 16)
    return fail(M2_EINVAL, "m2_rmsnorm_residual: pointers must be 16-byte aligned");
  if (!(eps > 0.f)) return fail(M2_EINVAL, "m2_rmsnorm_residual: eps must be positive");
  m2_status s = check_device();
  if (s) return s;
  M2_CUDA(launch_rmsnorm_residual(h, add, w, eps, normed, nullptr, 1.f, T, n, static_cast<cudaStream_t>(stream)));
  return M2_OK;
}

m2_status m2_rmsnorm_residual_quant(uint16_t* h, const uint16_t* add, const uint16_t* w, float eps, float s_q,
                                    uint16_t* normed, uint8_t* q, int T, int n, void* stream) {
  g_err.clear();
  if (T < 0 || n < 8 || n % 8)
    return fail(M2_ESHAPE, "m2_rmsnorm_residual_quant: T %d, n %d (n must be a multiple of 8)", T, n);
  if (T && (!h || !w || !q)) return fail(M2_EINVAL, "m2_rmsnorm_residual_quant: null pointer");
  if ((uintptr_t)h % 16 || (uintptr_t)add % 16 || (uintptr_t)w % 16 || (uintptr_t)normed % 16 || (uintptr_t)q % 8)
    return fail(M2_EINVAL, "m2_rmsnorm_residual_quant: h, add, w, normed must be 16-byte and q 8-byte aligned");
  if (!(eps > 0.f)) return fail(M2_EINVAL, "m2_rmsnorm_residual_quant: eps must be positive");
  if (!(s_q > 0.f) || !std::isfinite(s_q)) return fail(M2_EINVAL, "m2_rmsnorm_residual_quant: bad scale");
  m2_status s = check_device();
  if (s) return s;
  M2_CUDA(launch_rmsnorm_residual(h, add, w, eps, normed, q, s_q, T, n, static_cast<cudaStream_t>(stream)));
  return M2_OK;
}

// ---------------------------------------------------------------- fp8_linear without allocation

}  // extern "C"

namespace {
// Library-owned scratch for fp8_linear_noalloc: the split-K partial sums.
// Host code must not use this name as an address; it looks the device address
// up once per device (noalloc_scratch below).
__device__ __align__(256) float g_noalloc_scratch[M2_NOALLOC_SCRATCH_BYTES / sizeof(float)];

// The standalone entry points' device error word (bounded-wait timeouts).
__device__ int g_standalone_err;

m2_status standalone_error_word(int** out) {
  static std::mutex mu;
  static std::map<int, int*> by_device;
  int dev = 0;
  M2_CUDA(cudaGetDevice(&dev));
  std::lock_guard<std::mutex> lock(mu);
  auto it = by_device.find(dev);
  if (it != by_device.end()) {
    *out = it->second;
    return M2_OK;
  }
  int* p = nullptr;
  cudaError_t e = cudaGetSymbolAddress(reinterpret_cast<void**>(&p), g_standalone_err);
  if (e != cudaSuccess || !p)
    return fail(M2_ECUDA, "cudaGetSymbolAddress of the standalone error word failed: %s", cudaGetErrorString(e));
  by_device[dev] = p;
  *out = p;
  return M2_OK;
}

m2_status noalloc_scratch(float** out) {
  static std::mutex mu;
  static std::map<int, float*> by_device;
  int dev = 0;
  M2_CUDA(cudaGetDevice(&dev));
  std::lock_guard<std::mutex> lock(mu);
  auto it = by_device.find(dev);
  if (it != by_device.end()) {
    *out = it->second;
    return M2_OK;
  }
  float* p = nullptr;
  cudaError_t e = cudaGetSymbolAddress(reinterpret_cast<void**>(&p), g_noalloc_scratch);
  if (e != cudaSuccess || !p)
    return fail(M2_ECUDA, "fp8_linear_noalloc: cudaGetSymbolAddress of the scratch array failed: %s",
                cudaGetErrorString(e));
  by_device[dev] = p;
  *out = p;
  return M2_OK;
}
}  // namespace

extern "C" m2_status fp8_linear_noalloc(const uint8_t* a_q, float s_a, const uint8_t* w_q, float s_w, uint16_t* y,
                                        int M, int N, int K, void* stream) {
  g_err.clear();
  m2_status s = check_linear(a_q, w_q, y, M, N, K, s_a, s_w, "fp8_linear_noalloc");
  if (s) return s;
  if (M < 1 || M > kSkinnyMaxRows)
    return fail(M2_ESHAPE, "fp8_linear_noalloc: M = %d; this entry point takes 1 <= M <= %d", M, kSkinnyMaxRows);
  const size_t need = gemm_tc_skinny_workspace(M, N, K);
  if (need > (size_t)M2_NOALLOC_SCRATCH_BYTES)
    return fail(M2_ESHAPE, "fp8_linear_noalloc: %d x %d x %d needs %zu bytes of scratch, above the %u-byte array", M,
                N, K, need, (unsigned)M2_NOALLOC_SCRATCH_BYTES);
  float* scratch = nullptr;
  if ((s = noalloc_scratch(&scratch))) return s;
  int* err = nullptr;
  if ((s = standalone_error_word(&err))) return s;
  int nl = 0;
  M2_CUDA(gemm_tc_skinny(a_q, w_q, y, M, N, K, s_a * s_w, scratch, (size_t)M2_NOALLOC_SCRATCH_BYTES, err,
                         static_cast<cudaStream_t>(stream), &nl));
  return M2_OK;
}

extern "C" m2_status m2_check_standalone(void) {
  g_err.clear();
  m2_status s = check_device();
  if (s) return s;
  int* err = nullptr;
  if ((s = standalone_error_word(&err))) return s;
  int v = 0;
  M2_CUDA(cudaDeviceSynchronize());
  M2_CUDA(cudaMemcpy(&v, err, sizeof v, cudaMemcpyDeviceToHost));
  M2_CUDA(cudaMemset(err, 0, sizeof(int)));
  return error_word_status(v, "m2_check_standalone");
}

