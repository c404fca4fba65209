"""Seeded synthetic inputs for one NemotronH-style Mamba2 mixer block.

This module is the ONLY code shared by the CPU oracle's callers and the CUDA
path's callers (tests and bench).  It draws random numbers and packs them into
the storage formats the block consumes; it contains none of the block's own
arithmetic.  Rounding to bf16 and the per-tensor e4m3 weight encoding of the
generated weights are done by PyTorch's dtype casts (library routines), because
a checkpoint arrives already in those formats.

Every tensor comes from its own counter-based Philox stream, keyed by
``seed = 20261202 + 1000*config + 17*layer + tensor_id`` so that any one tensor
can be regenerated alone.  Values that are bf16 on the device are returned as
numpy float32 arrays holding exactly-bf16 values; e4m3 tensors are uint8 codes.

Distributions (the workload description of the mixer block): projection weights
N(0, 0.02) quantised to e4m3 with a per-tensor fp32 scale amax/448; hidden
N(0, 1) bf16; A_log = log U(1, 16); dt_bias = softplus^-1(d) with
d = exp(U(log 1e-3, log 0.1)); D = 1; conv weights N(0, 0.5); norm weight
1 + N(0, 0.1); prior conv state N(0, 1) bf16; prior SSM state N(0, 0.1) f32.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch

SEED_BASE = 20261202

# tensor ids inside one (config, layer)
T_IN_PROJ, T_OUT_PROJ, T_CONV_W, T_A_LOG, T_DT_BIAS, T_NORM_W = 1, 2, 3, 4, 5, 6
T_HIDDEN, T_CONV_STATE, T_SSM_STATE, T_SLOTS, T_STACK_NORM = 7, 8, 9, 10, 11


@dataclasses.dataclass(frozen=True)
class Geometry:
    """Shape of one mixer block (NemotronH sizes by default)."""
    hidden: int = 2688
    d_inner: int = 4096
    nheads: int = 64
    headdim: int = 64
    n_groups: int = 8
    d_state: int = 128
    conv_width: int = 4

    @property
    def conv_dim(self) -> int:
        return self.d_inner + 2 * self.n_groups * self.d_state

    @property
    def zx_width(self) -> int:
        return self.d_inner + self.conv_dim + self.nheads


NEMOTRON_H = Geometry()

# static per-tensor activation scales (powers of two: the division is exact)
S_X = 1.0 / 64.0
S_Y = 1.0 / 32.0
EPS = 1e-5


def seed_for(config: int, layer: int, tensor_id: int) -> int:
    return SEED_BASE + 1000 * config + 17 * layer + tensor_id


def rng(config: int, layer: int, tensor_id: int) -> np.random.Generator:
    return np.random.Generator(np.random.Philox(key=seed_for(config, layer, tensor_id)))


def as_bf16_values(a: np.ndarray) -> np.ndarray:
    """Round float data to bf16 (PyTorch cast) and return it as float32."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    return t.to(torch.bfloat16).to(torch.float32).numpy()


def quantize_weight_e4m3(w: np.ndarray) -> tuple[np.ndarray, float]:
    """Per-tensor e4m3 encoding of a generated weight (checkpoint format).

    The scale is amax/448 so the largest magnitude lands on the top finite
    e4m3 value; the cast is PyTorch's float8_e4m3fn conversion.
    """
    w = np.ascontiguousarray(w, dtype=np.float32)
    s = float(np.float32(np.abs(w).max()) / np.float32(448.0))
    scaled = torch.from_numpy(w) / torch.tensor(s, dtype=torch.float32)
    scaled = scaled.clamp_(-448.0, 448.0)
    codes = scaled.to(torch.float8_e4m3fn).view(torch.uint8).numpy().copy()
    return codes, s


def make_weights(config: int, layer: int = 0, geo: Geometry = NEMOTRON_H) -> dict:
    """All parameters of one mixer block."""
    g = geo
    w_in = rng(config, layer, T_IN_PROJ).standard_normal((g.zx_width, g.hidden), dtype=np.float32) * 0.02
    in_q, s_w1 = quantize_weight_e4m3(w_in)
    del w_in
    w_out = rng(config, layer, T_OUT_PROJ).standard_normal((g.hidden, g.d_inner), dtype=np.float32) * 0.02
    out_q, s_w2 = quantize_weight_e4m3(w_out)
    del w_out
    conv_w = as_bf16_values(rng(config, layer, T_CONV_W).standard_normal((g.conv_dim, g.conv_width)) * 0.5)
    a_log = as_bf16_values(np.log(rng(config, layer, T_A_LOG).uniform(1.0, 16.0, g.nheads)))
    d_target = np.exp(rng(config, layer, T_DT_BIAS).uniform(math.log(1e-3), math.log(0.1), g.nheads))
    dt_bias = as_bf16_values(np.log(np.expm1(d_target)))
    norm_w = as_bf16_values(1.0 + 0.1 * rng(config, layer, T_NORM_W).standard_normal(g.d_inner))
    return dict(
        in_proj=in_q, s_w1=s_w1, out_proj=out_q, s_w2=s_w2,
        conv_w=conv_w, conv_b=None,
        A_log=a_log.astype(np.float32), D=np.ones(g.nheads, np.float32),
        dt_bias=dt_bias.astype(np.float32), norm_w=norm_w,
        s_x=S_X, s_y=S_Y, eps=EPS, geo=g,
    )


def make_hidden(config: int, tokens: int, geo: Geometry = NEMOTRON_H, layer: int = 0) -> np.ndarray:
    return as_bf16_values(rng(config, layer, T_HIDDEN).standard_normal((tokens, geo.hidden), dtype=np.float32))


def make_conv_state(config: int, rows: int, geo: Geometry = NEMOTRON_H, layer: int = 0) -> np.ndarray:
    a = rng(config, layer, T_CONV_STATE).standard_normal((rows, geo.conv_dim, geo.conv_width - 1), dtype=np.float32)
    return as_bf16_values(a)


def make_ssm_state(config: int, rows: int, geo: Geometry = NEMOTRON_H, layer: int = 0) -> np.ndarray:
    a = rng(config, layer, T_SSM_STATE).standard_normal(
        (rows, geo.nheads, geo.headdim, geo.d_state), dtype=np.float32)
    return a * np.float32(0.1)


def make_slot_idx(config: int, n_slots: int, batch: int) -> np.ndarray:
    perm = rng(config, 0, T_SLOTS).permutation(n_slots)
    return perm[:batch].astype(np.int32)


def make_stack_norm_w(config: int, layer: int, geo: Geometry = NEMOTRON_H) -> np.ndarray:
    return as_bf16_values(1.0 + 0.1 * rng(config, layer, T_STACK_NORM).standard_normal(geo.hidden))


# The five workloads of the mixer block (sizes only; the arrays come from the
# make_* functions above).
WORKLOADS = {
    0: dict(kind="prefill", seqlens=[32], zero_state=True),
    1: dict(kind="decode", batch=1, n_slots=1),
    2: dict(kind="decode", batch=64, n_slots=256),
    3: dict(kind="prefill", seqlens=[2048] * 4, zero_state=True, chunk=256),
    4: dict(kind="stack", layers=23, batch=128, n_slots=512, seqlens=[4096, 1024, 512, 37]),
}


def device_normal(shape, config: int, layer: int, tensor_id: int, std: float, dtype, device):
    """Seeded normal tensor generated on a CUDA device with PyTorch's Philox
    generator (for state pools too large to draw on the host)."""
    g = torch.Generator(device=device)
    g.manual_seed(seed_for(config, layer, tensor_id))
    t = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t.to(dtype)
