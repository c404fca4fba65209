"""Python binding of libm2, a GB300 (sm_103a) Mamba2 mixer block.

Argument marshalling only: every step of the block runs in the CUDA kernels of
libm2.so, reached through its C ABI (include/m2.h).  PyTorch provides device
memory and streams.  There is no fallback: importing this package fails if the
library has not been built (``__graft_entry__.build()`` or
``python mamba2_ssm_mixer_gb300/_build.py``).
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libm2.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is missing: build it with mamba2_ssm_mixer_gb300._build.build() "
                      "(nvcc, sm_103a); there is no CPU or eager fallback")

_lib = ctypes.CDLL(LIB_PATH)

M2_OK, M2_EINVAL, M2_ESHAPE, M2_ECUDA, M2_ETIMEOUT, M2_EDEVICE, M2_ENOMEM = range(7)
M2_DTYPE_F32, M2_DTYPE_BF16 = 0, 1
M2_ARM_W8A8, M2_ARM_W8A16 = 0, 1
M2_LAYOUT_OUT_IN = 0

STATUS_NAMES = {0: "M2_OK", 1: "M2_EINVAL", 2: "M2_ESHAPE", 3: "M2_ECUDA", 4: "M2_ETIMEOUT",
                5: "M2_EDEVICE", 6: "M2_ENOMEM"}

EXPORTED = ["m2_last_error", "m2_create", "m2_destroy", "m2_get_stats", "m2_set_taps", "m2_check",
            "m2_prefill_workspace_size", "m2_prefill", "m2_decode_workspace_size", "m2_decode",
            "fp8_quant", "fp8_linear_workspace_size", "fp8_linear", "fp8_linear_bf16",
            "m2_rmsnorm_residual", "m2_profile_enable", "m2_profile_read", "fp8_linear_noalloc",
            "m2_prefill_q", "m2_decode_q", "m2_rmsnorm_residual_quant", "m2_mixed_workspace_size", "m2_mixed",
            "fp8_dequant", "bf16_linear_workspace_size", "bf16_linear", "m2_check_standalone",
            "m2_selftest_timeout"]

STAGES = ["quant_in", "in_proj", "conv", "conv_state", "ssd_cumsum", "ssd_chunk_state", "ssd_state_pass",
          "ssd_chunk_scan", "norm_quant", "out_proj", "decode_fused", "dec_quant_in", "dec_in_proj",
          "dec_out_proj"]
NSTAGES = 16


class M2Error(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


class m2_config(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int), ("d_inner", ctypes.c_int), ("nheads", ctypes.c_int),
                ("headdim", ctypes.c_int), ("n_groups", ctypes.c_int), ("d_state", ctypes.c_int),
                ("conv_width", ctypes.c_int), ("chunk_size", ctypes.c_int), ("ssm_dtype", ctypes.c_int),
                ("eps", ctypes.c_float), ("s_x", ctypes.c_float), ("s_y", ctypes.c_float), ("arm", ctypes.c_int)]


class m2_weights(ctypes.Structure):
    _fields_ = [("in_proj", ctypes.c_void_p), ("s_w1", ctypes.c_float),
                ("out_proj", ctypes.c_void_p), ("s_w2", ctypes.c_float),
                ("conv_w", ctypes.c_void_p), ("conv_b", ctypes.c_void_p),
                ("A_log", ctypes.c_void_p), ("D", ctypes.c_void_p), ("dt_bias", ctypes.c_void_p),
                ("norm_w", ctypes.c_void_p), ("layout", ctypes.c_int)]


class m2_stats(ctypes.Structure):
    _fields_ = [(n, ctypes.c_uint64) for n in ("bytes_uploaded", "conv_fwd_calls", "chunk_scan_calls",
                                                "conv_update_rows", "state_update_rows", "prefill_calls",
                                                "decode_calls", "kernel_launches")]


class m2_taps(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("q", "zx", "u", "dt", "y", "o", "q2")]


_vp, _i, _f, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
_sigs = {
    "m2_last_error": ([], ctypes.c_char_p),
    "m2_create": ([ctypes.POINTER(m2_config), ctypes.POINTER(m2_weights), ctypes.POINTER(_vp)], _i),
    "m2_destroy": ([_vp], None),
    "m2_get_stats": ([_vp, ctypes.POINTER(m2_stats)], _i),
    "m2_set_taps": ([_vp, ctypes.POINTER(m2_taps)], _i),
    "m2_check": ([_vp], _i),
    "m2_prefill_workspace_size": ([_vp, _vp, _i, ctypes.POINTER(_sz)], _i),
    "m2_prefill": ([_vp, _vp, _vp, _i, _vp, _vp, _vp, _vp, _vp, _sz, _vp], _i),
    "m2_decode_workspace_size": ([_vp, _i, ctypes.POINTER(_sz)], _i),
    "m2_decode": ([_vp, _vp, _i, _vp, _vp, _i, _vp, _vp, _vp, _sz, _vp], _i),
    "fp8_quant": ([_vp, _sz, _f, _vp, _vp], _i),
    "fp8_linear_workspace_size": ([_i, _i, _i, ctypes.POINTER(_sz)], _i),
    "fp8_linear": ([_vp, _f, _vp, _f, _vp, _i, _i, _i, _vp, _sz, _vp], _i),
    "fp8_linear_bf16": ([_vp, _f, _vp, _f, _vp, _i, _i, _i, _vp, _sz, _vp], _i),
    "m2_rmsnorm_residual": ([_vp, _vp, _vp, _f, _vp, _i, _i, _vp], _i),
    "m2_profile_enable": ([_vp, _i], _i),
    "m2_profile_read": ([_vp, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_uint64)], _i),
    "fp8_linear_noalloc": ([_vp, _f, _vp, _f, _vp, _i, _i, _i, _vp], _i),
    "m2_prefill_q": ([_vp, _vp, _vp, _i, _vp, _vp, _vp, _vp, _vp, _sz, _vp], _i),
    "m2_decode_q": ([_vp, _vp, _i, _vp, _vp, _i, _vp, _vp, _vp, _sz, _vp], _i),
    "m2_rmsnorm_residual_quant": ([_vp, _vp, _vp, _f, _f, _vp, _vp, _i, _i, _vp], _i),
    "m2_mixed_workspace_size": ([_vp, _i, _vp, _i, ctypes.POINTER(_sz)], _i),
    "m2_mixed": ([_vp, _vp, _i, _vp, _vp, _i, _vp, _vp, _i, _vp, _vp, _vp, _vp, _vp, _sz, _vp], _i),
    "fp8_dequant": ([_vp, _sz, _f, _vp, _vp], _i),
    "bf16_linear_workspace_size": ([_i, _i, _i, ctypes.POINTER(_sz)], _i),
    "bf16_linear": ([_vp, _vp, _f, _vp, _i, _i, _i, _vp, _sz, _vp], _i),
    "m2_check_standalone": ([], _i),
    "m2_selftest_timeout": ([_vp, ctypes.c_uint, _vp], _i),
}
for _name, (_args, _ret) in _sigs.items():
    _fn = getattr(_lib, _name)
    _fn.argtypes = _args
    _fn.restype = _ret


def last_error() -> str:
    return _lib.m2_last_error().decode()


def _check(status: int):
    if status != M2_OK:
        raise M2Error(status, last_error())


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, torch.Tensor):
        return t.data_ptr()
    return int(t)


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _need(t: torch.Tensor, name: str, dtype, shape=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


HIDDEN, D_INNER, NHEADS, HEADDIM, N_GROUPS, D_STATE, CONV_WIDTH = 2688, 4096, 64, 64, 8, 128, 4
CONV_DIM = D_INNER + 2 * N_GROUPS * D_STATE
ZX_WIDTH = D_INNER + CONV_DIM + NHEADS


def make_config(s_x: float, s_y: float, eps: float = 1e-5, chunk_size: int = 256,
                ssm_dtype: int = M2_DTYPE_F32, arm: int = M2_ARM_W8A8) -> m2_config:
    return m2_config(HIDDEN, D_INNER, NHEADS, HEADDIM, N_GROUPS, D_STATE, CONV_WIDTH, chunk_size, ssm_dtype,
                     eps, s_x, s_y, arm)


class Mamba2Mixer:
    """One mixer block.  ``weights`` maps names to CPU or CUDA tensors:
    in_proj uint8 [10304, 2688], s_w1, out_proj uint8 [2688, 4096], s_w2,
    conv_w bf16 [6144, 4], conv_b bf16 [6144] or None, A_log, D, dt_bias f32 [64],
    norm_w bf16 [4096]; plus s_x, s_y (activation scales) and eps.
    arm: M2_ARM_W8A8 (e4m3 activations) or M2_ARM_W8A16 (bf16 activations
    against weights dequantised to bf16; prefill and decode only)."""

    def __init__(self, weights: dict, device=None, layout: int = M2_LAYOUT_OUT_IN,
                 ssm_dtype: int = M2_DTYPE_F32, chunk_size: int = 256, arm: int = M2_ARM_W8A8):
        self.device = torch.device(device if device is not None else "cuda")
        with torch.cuda.device(self.device):
            keep = {}
            for k in ("in_proj", "out_proj", "conv_w", "conv_b", "A_log", "D", "dt_bias", "norm_w"):
                v = weights.get(k)
                keep[k] = None if v is None else v.contiguous()
            cfg = make_config(weights["s_x"], weights["s_y"], weights.get("eps", 1e-5), chunk_size, ssm_dtype, arm)
            w = m2_weights(_ptr(keep["in_proj"]), weights["s_w1"], _ptr(keep["out_proj"]), weights["s_w2"],
                           _ptr(keep["conv_w"]), _ptr(keep["conv_b"]), _ptr(keep["A_log"]), _ptr(keep["D"]),
                           _ptr(keep["dt_bias"]), _ptr(keep["norm_w"]), layout)
            h = ctypes.c_void_p()
            _check(_lib.m2_create(ctypes.byref(cfg), ctypes.byref(w), ctypes.byref(h)))
        self._h = h
        self._taps = None
        self.s_x = float(weights["s_x"])   # the input quant scale (for pre-quantised inputs)
        self.arm = arm
        # dtype of the SSM state rows this block reads and writes
        self.state_dtype = torch.bfloat16 if ssm_dtype == M2_DTYPE_BF16 else torch.float32

    def close(self):
        if getattr(self, "_h", None):
            _lib.m2_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def handle(self):
        return self._h

    def stats(self) -> dict:
        s = m2_stats()
        _check(_lib.m2_get_stats(self._h, ctypes.byref(s)))
        return {n: getattr(s, n) for n, _ in m2_stats._fields_}

    def set_taps(self, **bufs):
        """Install device buffers for intermediates (q, zx, u, dt, y, o, q2);
        call with no arguments to remove them."""
        if not bufs:
            self._taps = None
            _check(_lib.m2_set_taps(self._h, None))
            return
        t = m2_taps(*[_ptr(bufs.get(n)) for n, _ in m2_taps._fields_])
        self._taps = bufs
        _check(_lib.m2_set_taps(self._h, ctypes.byref(t)))

    def check(self):
        _check(_lib.m2_check(self._h))

    def selftest_timeout(self, limit_us: int = 1000, stream=None):
        """Run the failure-detection self-test on this handle's error word:
        a bounded wait that nothing completes runs out after limit_us; the
        next check() raises M2Error(M2_ETIMEOUT)."""
        _check(_lib.m2_selftest_timeout(self._h, int(limit_us), _stream(stream)))

    def profile(self, on: bool):
        _check(_lib.m2_profile_enable(self._h, int(bool(on))))

    def profile_read(self) -> dict:
        """Per-stage (elapsed ms, launches) since the last read; synchronises."""
        ms = (ctypes.c_double * NSTAGES)()
        n = (ctypes.c_uint64 * NSTAGES)()
        _check(_lib.m2_profile_read(self._h, ms, n))
        return {name: (ms[i], n[i]) for i, name in enumerate(STAGES) if n[i]}

    def prefill_workspace_size(self, seqlens) -> int:
        arr = (ctypes.c_int32 * len(seqlens))(*seqlens)
        n = ctypes.c_size_t()
        _check(_lib.m2_prefill_workspace_size(self._h, arr, len(seqlens), ctypes.byref(n)))
        return n.value

    def decode_workspace_size(self, batch: int) -> int:
        n = ctypes.c_size_t()
        _check(_lib.m2_decode_workspace_size(self._h, batch, ctypes.byref(n)))
        return n.value

    def prefill(self, hidden, seqlens, conv_state, ssm_state, has_initial=None, out=None, workspace=None,
                stream=None):
        """hidden: bf16 [sum(T), 2688], or e4m3 codes (uint8) already quantised
        with this block's s_x (m2_prefill_q)."""
        T = sum(seqlens)
        quantised = hidden.dtype == torch.uint8
        _need(hidden, "hidden", torch.uint8 if quantised else torch.bfloat16, (T, HIDDEN))
        _need(conv_state, "conv_state", torch.bfloat16, (len(seqlens), CONV_DIM, CONV_WIDTH - 1))
        _need(ssm_state, "ssm_state", self.state_dtype, (len(seqlens), NHEADS, HEADDIM, D_STATE))
        if out is None:
            out = torch.empty((T, HIDDEN), dtype=torch.bfloat16, device=hidden.device)
        _need(out, "out", torch.bfloat16, (T, HIDDEN))
        if workspace is None:
            workspace = torch.empty(self.prefill_workspace_size(seqlens), dtype=torch.uint8, device=hidden.device)
        arr = (ctypes.c_int32 * len(seqlens))(*seqlens)
        hi = None if has_initial is None else (ctypes.c_uint8 * len(seqlens))(*[int(bool(v)) for v in has_initial])
        fn = _lib.m2_prefill_q if quantised else _lib.m2_prefill
        _check(fn(self._h, _ptr(hidden), arr, len(seqlens), hi, _ptr(conv_state), _ptr(ssm_state),
                  _ptr(out), _ptr(workspace), workspace.numel(), _stream(stream)))
        return out

    def decode(self, hidden, conv_pool, ssm_pool, slot_idx, out=None, workspace=None, stream=None):
        """hidden: bf16 [Bt, 2688], or e4m3 codes (uint8) already quantised with
        this block's s_x (m2_decode_q)."""
        Bt = hidden.shape[0]
        quantised = hidden.dtype == torch.uint8
        _need(hidden, "hidden", torch.uint8 if quantised else torch.bfloat16, (Bt, HIDDEN))
        n_slots = conv_pool.shape[0]
        _need(conv_pool, "conv_pool", torch.bfloat16, (n_slots, CONV_DIM, CONV_WIDTH - 1))
        _need(ssm_pool, "ssm_pool", self.state_dtype, (n_slots, NHEADS, HEADDIM, D_STATE))
        _need(slot_idx, "slot_idx", torch.int32, (Bt,))
        if out is None:
            out = torch.empty((Bt, HIDDEN), dtype=torch.bfloat16, device=hidden.device)
        _need(out, "out", torch.bfloat16, (Bt, HIDDEN))
        if workspace is None:
            workspace = torch.empty(self.decode_workspace_size(Bt), dtype=torch.uint8, device=hidden.device)
        fn = _lib.m2_decode_q if quantised else _lib.m2_decode
        _check(fn(self._h, _ptr(hidden), Bt, _ptr(conv_pool), _ptr(ssm_pool), n_slots, _ptr(slot_idx),
                  _ptr(out), _ptr(workspace), workspace.numel(), _stream(stream)))
        return out

    def mixed_workspace_size(self, batch: int, seqlens) -> int:
        return _mixed_ws_size(self, batch, list(seqlens))

    def mixed(self, hidden, batch, conv_pool, ssm_pool, slot_idx, seqlens, conv_state, ssm_state,
              has_initial=None, out=None, workspace=None, stream=None):
        """One call over `batch` decode rows (hidden[:batch], states in the
        slot pools) followed by packed prefill sequences (hidden[batch:])."""
        seqlens = list(seqlens)
        R = batch + sum(seqlens)
        _need(hidden, "hidden", torch.bfloat16, (R, HIDDEN))
        if batch:
            n_slots = conv_pool.shape[0]
            _need(conv_pool, "conv_pool", torch.bfloat16, (n_slots, CONV_DIM, CONV_WIDTH - 1))
            _need(ssm_pool, "ssm_pool", self.state_dtype, (n_slots, NHEADS, HEADDIM, D_STATE))
            _need(slot_idx, "slot_idx", torch.int32, (batch,))
        else:
            n_slots = 0
        if seqlens:
            _need(conv_state, "conv_state", torch.bfloat16, (len(seqlens), CONV_DIM, CONV_WIDTH - 1))
            _need(ssm_state, "ssm_state", self.state_dtype, (len(seqlens), NHEADS, HEADDIM, D_STATE))
        if out is None:
            out = torch.empty((R, HIDDEN), dtype=torch.bfloat16, device=hidden.device)
        _need(out, "out", torch.bfloat16, (R, HIDDEN))
        if workspace is None:
            workspace = torch.empty(self.mixed_workspace_size(batch, seqlens), dtype=torch.uint8,
                                    device=hidden.device)
        arr = (ctypes.c_int32 * max(len(seqlens), 1))(*seqlens)
        hi = None if has_initial is None else (ctypes.c_uint8 * len(seqlens))(*[int(bool(v)) for v in has_initial])
        _check(_lib.m2_mixed(self._h, _ptr(hidden), batch, _ptr(conv_pool) if batch else None,
                             _ptr(ssm_pool) if batch else None, n_slots, _ptr(slot_idx) if batch else None,
                             arr, len(seqlens), hi, _ptr(conv_state) if seqlens else None,
                             _ptr(ssm_state) if seqlens else None, _ptr(out), _ptr(workspace), workspace.numel(),
                             _stream(stream)))
        return out


def _mixed_ws_size(blk, Bt, seqlens):
    n = ctypes.c_size_t()
    arr = (ctypes.c_int32 * max(len(seqlens), 1))(*seqlens)
    _check(_lib.m2_mixed_workspace_size(blk._h, Bt, arr, len(seqlens), ctypes.byref(n)))
    return n.value


def check_standalone():
    """Read and clear the standalone entry points' device error word
    (synchronises); raises M2Error(M2_ETIMEOUT) if a bounded wait ran out."""
    _check(_lib.m2_check_standalone())


def selftest_timeout_standalone(limit_us: int = 1000, stream=None):
    """The failure-detection self-test on the standalone error word."""
    _check(_lib.m2_selftest_timeout(None, int(limit_us), _stream(stream)))


def fp8_quant(x: torch.Tensor, scale: float, q: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    _need(x, "x", torch.bfloat16)
    if q is None:
        q = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    _need(q, "q", torch.uint8, tuple(x.shape))
    _check(_lib.fp8_quant(_ptr(x), x.numel(), scale, _ptr(q), _stream(stream)))
    return q


def fp8_linear_workspace_size(M: int, N: int, K: int) -> int:
    n = ctypes.c_size_t()
    _check(_lib.fp8_linear_workspace_size(M, N, K, ctypes.byref(n)))
    return n.value


def fp8_linear(a_q: torch.Tensor, s_a: float, w_q: torch.Tensor, s_w: float, y: torch.Tensor | None = None,
               workspace=None, stream=None) -> torch.Tensor:
    M, K = a_q.shape
    N = w_q.shape[0]
    _need(a_q, "a_q", torch.uint8, (M, K))
    _need(w_q, "w_q", torch.uint8, (N, K))
    if y is None:
        y = torch.empty((M, N), dtype=torch.bfloat16, device=a_q.device)
    _need(y, "y", torch.bfloat16, (M, N))
    if workspace is None:
        workspace = torch.empty(max(fp8_linear_workspace_size(M, N, K), 1), dtype=torch.uint8, device=a_q.device)
    _check(_lib.fp8_linear(_ptr(a_q), s_a, _ptr(w_q), s_w, _ptr(y), M, N, K, _ptr(workspace), workspace.numel(),
                           _stream(stream)))
    return y


def fp8_linear_noalloc(a_q: torch.Tensor, s_a: float, w_q: torch.Tensor, s_w: float, y: torch.Tensor,
                       stream=None) -> torch.Tensor:
    """fp8_linear without a workspace (library-owned scratch; M <= 256)."""
    M, K = a_q.shape
    N = w_q.shape[0]
    _need(a_q, "a_q", torch.uint8, (M, K))
    _need(w_q, "w_q", torch.uint8, (N, K))
    _need(y, "y", torch.bfloat16, (M, N))
    _check(_lib.fp8_linear_noalloc(_ptr(a_q), s_a, _ptr(w_q), s_w, _ptr(y), M, N, K, _stream(stream)))
    return y


def fp8_linear_bf16(x: torch.Tensor, s_a: float, w_q: torch.Tensor, s_w: float, y: torch.Tensor | None = None,
                    workspace=None, stream=None) -> torch.Tensor:
    M, K = x.shape
    N = w_q.shape[0]
    _need(x, "x", torch.bfloat16, (M, K))
    _need(w_q, "w_q", torch.uint8, (N, K))
    if y is None:
        y = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    _need(y, "y", torch.bfloat16, (M, N))
    if workspace is None:
        need = ((M * K + 255) // 256) * 256 + fp8_linear_workspace_size(M, N, K)
        workspace = torch.empty(need, dtype=torch.uint8, device=x.device)
    _check(_lib.fp8_linear_bf16(_ptr(x), s_a, _ptr(w_q), s_w, _ptr(y), M, N, K, _ptr(workspace),
                                workspace.numel(), _stream(stream)))
    return y


def fp8_dequant(q: torch.Tensor, scale: float, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """bf16(dec(q) * scale), the W8A16 arm's weight dequantisation."""
    _need(q, "q", torch.uint8)
    if out is None:
        out = torch.empty(q.shape, dtype=torch.bfloat16, device=q.device)
    _need(out, "out", torch.bfloat16, tuple(q.shape))
    _check(_lib.fp8_dequant(_ptr(q), q.numel(), scale, _ptr(out), _stream(stream)))
    return out


def bf16_linear_workspace_size(M: int, N: int, K: int) -> int:
    n = ctypes.c_size_t()
    _check(_lib.bf16_linear_workspace_size(M, N, K, ctypes.byref(n)))
    return n.value


def bf16_linear(x: torch.Tensor, w: torch.Tensor, scale: float = 1.0, y: torch.Tensor | None = None,
                workspace=None, stream=None) -> torch.Tensor:
    """y = bf16(scale * x @ w^T), bf16 operands on the tensor cores (W8A16 arm)."""
    M, K = x.shape
    N = w.shape[0]
    _need(x, "x", torch.bfloat16, (M, K))
    _need(w, "w", torch.bfloat16, (N, K))
    if y is None:
        y = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    _need(y, "y", torch.bfloat16, (M, N))
    if workspace is None:
        workspace = torch.empty(max(bf16_linear_workspace_size(M, N, K), 1), dtype=torch.uint8, device=x.device)
    _check(_lib.bf16_linear(_ptr(x), _ptr(w), scale, _ptr(y), M, N, K, _ptr(workspace), workspace.numel(),
                            _stream(stream)))
    return y


def m2_rmsnorm_residual(h: torch.Tensor, add: torch.Tensor | None, w: torch.Tensor | None, eps: float,
                        normed: torch.Tensor | None = None, stream=None, norm: bool = True):
    """h += add (if given); returns rmsnorm(h) * w (or None with norm=False)."""
    T, n = h.shape
    _need(h, "h", torch.bfloat16)
    if add is not None:
        _need(add, "add", torch.bfloat16, (T, n))
    if norm:
        _need(w, "w", torch.bfloat16, (n,))
        if normed is None:
            normed = torch.empty_like(h)
    else:
        normed = None
    _check(_lib.m2_rmsnorm_residual(_ptr(h), _ptr(add), _ptr(w), eps, _ptr(normed), T, n, _stream(stream)))
    return normed


def m2_rmsnorm_residual_quant(h: torch.Tensor, add: torch.Tensor | None, w: torch.Tensor, eps: float, s_q: float,
                              q: torch.Tensor | None = None, normed: torch.Tensor | None = None, stream=None):
    """h += add (if given); returns e4m3 codes of rmsnorm(h) * w / s_q (and
    writes the bf16 normed row too when `normed` is given)."""
    T, n = h.shape
    _need(h, "h", torch.bfloat16)
    if add is not None:
        _need(add, "add", torch.bfloat16, (T, n))
    _need(w, "w", torch.bfloat16, (n,))
    if normed is not None:
        _need(normed, "normed", torch.bfloat16, (T, n))
    if q is None:
        q = torch.empty((T, n), dtype=torch.uint8, device=h.device)
    _need(q, "q", torch.uint8, (T, n))
    _check(_lib.m2_rmsnorm_residual_quant(_ptr(h), _ptr(add), _ptr(w), eps, s_q, _ptr(normed), _ptr(q), T, n,
                                          _stream(stream)))
    return q


class Mamba2Stack:
    """Pre-norm residual stack of mixer blocks: for each layer l,
    h <- h + block_l(rmsnorm(h) * norm_w[l]).  Host-side composition of the
    C ABI calls (one rmsnorm_residual and one block call per layer)."""

    def __init__(self, blocks: list, norm_ws: list, eps: float = 1e-5, fused: bool = False):
        """fused: each layer's residual + RMSNorm also writes the next block's
        e4m3 input (m2_rmsnorm_residual_quant), and the blocks run from it
        (m2_prefill_q / m2_decode_q) instead of quantising a bf16 copy."""
        assert len(blocks) == len(norm_ws) and blocks
        self.blocks, self.norm_ws, self.eps, self.fused = blocks, norm_ws, eps, fused

    def _run(self, hidden, call, stream):
        h = hidden.clone()
        out = torch.empty_like(h)
        if self.fused:
            x = torch.empty(h.shape, dtype=torch.uint8, device=h.device)
        else:
            x = torch.empty_like(h)
        for l, blk in enumerate(self.blocks):
            if self.fused:
                m2_rmsnorm_residual_quant(h, out if l else None, self.norm_ws[l], self.eps, blk.s_x, q=x,
                                          stream=stream)
            else:
                m2_rmsnorm_residual(h, out if l else None, self.norm_ws[l], self.eps, x, stream=stream)
            call(l, blk, x, out)
        m2_rmsnorm_residual(h, out, None, self.eps, stream=stream, norm=False)
        return h

    def decode(self, hidden, conv_pools, ssm_pools, slot_idx, workspace=None, stream=None):
        ws = workspace if workspace is not None else torch.empty(
            self.blocks[0].decode_workspace_size(hidden.shape[0]), dtype=torch.uint8, device=hidden.device)
        return self._run(hidden, lambda l, blk, x, out: blk.decode(x, conv_pools[l], ssm_pools[l], slot_idx, out=out,
                                                                    workspace=ws, stream=stream), stream)

    def prefill(self, hidden, seqlens, conv_states, ssm_states, has_initial=None, workspace=None, stream=None):
        ws = workspace if workspace is not None else torch.empty(
            self.blocks[0].prefill_workspace_size(seqlens), dtype=torch.uint8, device=hidden.device)
        return self._run(hidden, lambda l, blk, x, out: blk.prefill(x, seqlens, conv_states[l], ssm_states[l],
                                                                     has_initial=has_initial, out=out, workspace=ws,
                                                                     stream=stream), stream)
