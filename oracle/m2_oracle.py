"""CPU oracle for one NemotronH-style Mamba2 mixer block (test infrastructure).

This module is TEST INFRASTRUCTURE.  Only the test suite, the package smoke
check and the benchmark's CPU-baseline leg may import it.  The CUDA library
never calls it and shares no code with it.

It is deliberately plain and slow: numpy in float64, library matmuls as single
steps, and the recurrence run sequentially, token by token.  Values are rounded
to the block's storage dtypes at the points where the op chain hands a tensor
from one op to the next (bf16 for zxbcdt, the conv output, the scan output, the
gated-norm output and the block output; e4m3 codes for both quantised
activations); everything else is float64.

The op chain follows vllm.cpp PR #1288, "NemotronH's 23 Mamba2 blocks reach the
device on the FP8 W8A8 seam", section "What it does":
  in_proj (FP8 W8A8) -> QkvSplit(z | xBC | dt) -> CausalConv1dFwd(silu)
  -> QkvSplit(x | B | C) -> Mamba2ChunkScan -> RmsNormGatedGroup(n_groups)
  -> out_proj (FP8 W8A8).
The pages name the ops but never write their mathematics.  The math used here
is the standard Mamba-2 / SSD selective state-space layer (Dao & Gu, 2024,
"Transformers are SSMs"), which is the plainest reading of the op names; each
reading is listed in the function that takes it.

Parity pins: every function here is pinned by tests/test_oracle_pins.py against
closed forms, brute force, library routines or an independent formulation.
"""
from __future__ import annotations

import numpy as np

# --------------------------------------------------------------------------
# number formats
# --------------------------------------------------------------------------

E4M3_MAX = 448.0


def e4m3_decode(codes) -> np.ndarray:
    """Value of OCP FP8 E4M3 codes (1 sign, 4 exponent bits with bias 7,
    3 mantissa bits; exponent 0 is subnormal; S.1111.111 is NaN; there are no
    infinities).  Returns float64."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    mag = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0))
    out = sign * mag
    return np.where((e == 15) & ((c & 7) == 7), np.nan, out)


# The 127 non-negative finite e4m3 values in code order (monotone increasing).
_E4M3_POS = e4m3_decode(np.arange(0x7F, dtype=np.uint8))


def e4m3_encode(v) -> np.ndarray:
    """Round to the nearest e4m3 value, ties to the even code, saturating.

    Magnitudes at or above 448 (including infinities) become +-448, the
    behaviour of a saturating conversion ("satfinite").  NaN becomes 0x7F.
    The sign of the input (including -0.0) is kept.  Input may be float32 or
    float64; it is used exactly.
    """
    x = np.asarray(v, dtype=np.float64)
    a = np.abs(x)
    lo = np.clip(np.searchsorted(_E4M3_POS, a, side="right") - 1, 0, 125)
    d_lo = a - _E4M3_POS[lo]
    d_hi = _E4M3_POS[lo + 1] - a
    take_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (lo % 2 == 1))
    code = np.where(take_hi, lo + 1, lo)
    code = np.where(a >= E4M3_MAX, 0x7E, code)
    code = code | np.where(np.signbit(x), 0x80, 0)
    code = np.where(np.isnan(x), 0x7F, code)
    return code.astype(np.uint8)


def bf16_round(v) -> np.ndarray:
    """Round float64 values to bfloat16 (8 significant bits, exponent range of
    float32), round-to-nearest-even, directly from the exact input.  Returns
    the rounded values as float64."""
    x = np.asarray(v, dtype=np.float64)
    with np.errstate(over="ignore", invalid="ignore"):
        _, e = np.frexp(x)
        e = np.maximum(e, -125)            # below 2^-126 the quantum stays 2^-133
        r = np.ldexp(np.rint(np.ldexp(x, 8 - e)), e - 8)
        big = np.abs(r) > 3.3895313892515355e38
        r = np.where(big, np.copysign(np.inf, x), r)
    return np.where(np.isfinite(x), r, x)


def f32(v) -> np.ndarray:
    """IEEE round-to-nearest-even to float32, returned as float64."""
    return np.asarray(v, dtype=np.float64).astype(np.float32).astype(np.float64)


# --------------------------------------------------------------------------
# the ops
# --------------------------------------------------------------------------

def quant_static_e4m3(x, scale: float) -> np.ndarray:
    """Static per-tensor activation quantisation: q = e4m3(x / s).

    PR #1288, section "The comparison is not bit-comparable, and that is the
    point": the device arm is W8A8, applying the checkpoint's per-tensor
    input_scale to the activation (the kQuantFp8Static kernel of PR #988,
    section "The Thor finding, measured").  The quotient is formed in float32
    (the kernel's precision for the decision) and then rounded to e4m3.
    """
    q = np.asarray(x, dtype=np.float32) / np.float32(scale)
    return e4m3_encode(q)


def fp8_linear(a_q, s_a: float, w_q, s_w: float) -> np.ndarray:
    """W8A8 linear layer: y = bf16(s_a * s_w * dec(A) @ dec(W)^T).

    A is [M, K] e4m3 codes, W is [N, K] e4m3 codes stored [out, in] (the
    torch-Linear orientation PR #950 requires of every projection), scales are
    per tensor.  PR #972, "the FP8 W8A8 linear path becomes a seam a second
    model can reach", section "The call-site change" (MatmulFp8CutlassPreQuantD
    takes the pre-quantised activation).  Output dtype bf16.
    """
    acc = e4m3_decode(a_q) @ e4m3_decode(w_q).T
    return bf16_round(float(s_a) * float(s_w) * acc)


def dequant_e4m3_bf16(w_q, s_w: float) -> np.ndarray:
    """Weight dequantisation of the W8A16 arm: w = bf16(dec(W) * s_w).

    PR #1289, commit "the FP8 W8A8 seam": the host arm's DenseBf16 expands the
    fp8 weights into a bf16 buffer: each code's value times the tensor's
    per-tensor weight_scale.  The pages do not say in
    what precision the product is formed; the reading taken here: the
    product is rounded to float32 (nearest even), then to bf16 (nearest even).
    dec(W) has at most 4 significant bits and s_w (a float32) 24, so the
    float64 product below is exact before those two roundings.
    """
    return bf16_round(f32(e4m3_decode(w_q) * float(np.float32(s_w))))


def bf16_linear(x, w) -> np.ndarray:
    """W8A16 linear layer: y = bf16(x @ w^T) for bf16 activations x [M, K] and
    dequantised bf16 weights w [N, K] ([out, in]).

    PR #1288, section "The comparison is not bit-comparable, and that is the
    point": the host reference carries input_scale and does not apply it, so
    the activation enters the product as it is; PR #1289, GB10
    counter-measurement commit: the dequantised weights go to a plain matmul
    (vt::MatmulBT).  Exact accumulation (float64), output bf16.
    """
    return bf16_round(np.asarray(x, np.float64) @ np.asarray(w, np.float64).T)


def silu(v):
    v = np.asarray(v, dtype=np.float64)
    return v / (1.0 + np.exp(-v))


def softplus(v):
    """log(1 + e^v); the identity above 20 (where the two agree in float64 to
    ~2e-9 relative)."""
    v = np.asarray(v, dtype=np.float64)
    with np.errstate(over="ignore"):
        return np.where(v > 20.0, v, np.log1p(np.exp(np.minimum(v, 20.0))))


def split_zxbcdt(zx, d_inner: int, conv_dim: int, nheads: int):
    """QkvSplit(z | xBC | dt): head, middle and tail column ranges of the
    in_proj row, widths (d_inner, conv_dim, nheads).  PR #1288, "What it does";
    PR #1289 thread (the split-contract case)."""
    assert zx.shape[-1] == d_inner + conv_dim + nheads
    return zx[..., :d_inner], zx[..., d_inner:d_inner + conv_dim], zx[..., d_inner + conv_dim:]


def split_xbc(u, d_inner: int, n_groups: int, d_state: int):
    """QkvSplit(x | B | C) of the conv output, widths (d_inner, G*N, G*N)."""
    gn = n_groups * d_state
    assert u.shape[-1] == d_inner + 2 * gn
    return u[..., :d_inner], u[..., d_inner:d_inner + gn], u[..., d_inner + gn:]


def causal_conv1d_silu(xbc, w, b, state):
    """CausalConv1dFwd(silu) over one sequence, with carried state.

    Reading (the pages name the op only): depthwise causal convolution of
    width W per channel, u[t, c] = silu(b[c] + sum_j w[c, j] * x[t - (W-1) + j, c]),
    where times before the sequence start are read from ``state`` (the last
    W-1 inputs of the previous call, oldest first; zeros for a fresh sequence).
    The new state is the last W-1 raw (pre-conv) inputs of [state, x]; when
    the call has fewer than W-1 tokens the older state taps shift in.
    xbc: [T, C]; w: [C, W]; b: [C] or None; state: [C, W-1].
    Returns (u rounded to bf16 [T, C], new_state [C, W-1]).
    """
    xbc = np.asarray(xbc, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    T, C = xbc.shape
    W = w.shape[1]
    xp = np.concatenate([np.asarray(state, dtype=np.float64).T, xbc], axis=0)  # [W-1+T, C]
    acc = np.zeros((T, C))
    for j in range(W):
        acc += w[:, j][None, :] * xp[j:j + T]
    if b is not None:
        acc += np.asarray(b, dtype=np.float64)[None, :]
    u = bf16_round(silu(acc))
    new_state = xp[T:].T.copy()   # last W-1 rows of xp
    return u, new_state


def ssd_sequential(x, dt, A, B, C, D, S0):
    """The selective state-space recurrence, one token at a time.

    Reading of Mamba2ChunkScan / the single-step state update (standard
    Mamba-2): per head h with group g(h) = h // (nheads / n_groups),
      S_h <- exp(dt[t,h] * A[h]) * S_h + dt[t,h] * x[t,h,:] (outer) B[t,g,:]
      y[t,h,:] = S_h @ C[t,g,:] + D[h] * x[t,h,:]
    x: [T, nh, P]; dt: [T, nh]; A, D: [nh]; B, C: [T, G, N]; S0: [nh, P, N].
    Returns (y float64 [T, nh, P], S float64 [nh, P, N]).  The chunked form is
    the same function evaluated blockwise; this oracle never uses it.
    """
    x = np.asarray(x, np.float64)
    dt = np.asarray(dt, np.float64)
    A = np.asarray(A, np.float64)
    D = np.asarray(D, np.float64)
    B = np.asarray(B, np.float64)
    C = np.asarray(C, np.float64)
    T, nh, P = x.shape
    G = B.shape[1]
    hpg = nh // G
    S = np.array(S0, dtype=np.float64, copy=True)
    y = np.empty((T, nh, P))
    for t in range(T):
        Bh = np.repeat(B[t], hpg, axis=0)            # [nh, N]
        Ch = np.repeat(C[t], hpg, axis=0)
        decay = np.exp(dt[t] * A)                    # [nh]
        S *= decay[:, None, None]
        S += (dt[t][:, None] * x[t])[:, :, None] * Bh[:, None, :]
        y[t] = np.einsum("hpn,hn->hp", S, Ch) + D[:, None] * x[t]
    return y, S


def _ssd_group_job(args):
    return ssd_sequential(*args)


def ssd_by_group(x, dt, A, B, C, D, S0, map_fn=map):
    """ssd_sequential evaluated group by group: the heads of different groups
    share nothing, so this is the same function; map_fn may be a process
    pool's map to spread the groups over host cores."""
    x = np.asarray(x, np.float64)
    T, nh, P = x.shape
    G = np.asarray(B).shape[1]
    hpg = nh // G
    jobs = []
    for g in range(G):
        hs = slice(g * hpg, (g + 1) * hpg)
        jobs.append((x[:, hs], np.asarray(dt)[:, hs], np.asarray(A)[hs], np.asarray(B)[:, g:g + 1],
                     np.asarray(C)[:, g:g + 1], np.asarray(D)[hs], np.asarray(S0)[hs]))
    res = list(map_fn(_ssd_group_job, jobs))
    y = np.concatenate([r[0] for r in res], axis=1)
    S = np.concatenate([r[1] for r in res], axis=0)
    return y, S


def gated_rmsnorm_group(y, z, w, n_groups: int, eps: float):
    """RmsNormGatedGroup(n_groups).

    Reading: gate first, then normalise each group of d_inner/n_groups
    channels by its own root mean square, then scale by the per-channel
    weight: g = y * silu(z); o = g / sqrt(mean_group(g^2) + eps) * w.
    y, z: [T, I]; w: [I].  Returns o in float64 (unrounded).
    """
    y = np.asarray(y, np.float64)
    T, I = y.shape
    g = y * silu(z)
    gg = g.reshape(T, n_groups, I // n_groups)
    r = 1.0 / np.sqrt(np.mean(gg * gg, axis=-1, keepdims=True) + eps)
    return (gg * r).reshape(T, I) * np.asarray(w, np.float64)[None, :]


def rmsnorm(h, w, eps: float):
    """Plain RMSNorm used between stacked blocks, output bf16."""
    h = np.asarray(h, np.float64)
    r = 1.0 / np.sqrt(np.mean(h * h, axis=-1, keepdims=True) + eps)
    return bf16_round(h * r * np.asarray(w, np.float64)[None, :])


# --------------------------------------------------------------------------
# the block
# --------------------------------------------------------------------------

def _dims(Wt):
    g = Wt["geo"]
    return g.hidden, g.d_inner, g.nheads, g.headdim, g.n_groups, g.d_state, g.conv_width


def block_tokens(Wt, hidden, seqlens, conv_state, ssm_state, keep=False, map_fn=None, arm="w8a8"):
    """Run the mixer block over packed sequences with carried states.

    hidden: [sum(T), H] bf16 values.  conv_state: [nseq, conv_dim, W-1];
    ssm_state: [nseq, nh, P, N] (the states each sequence starts from; zeros
    for a fresh sequence, PR #1288 "What it does": rows are gathered and
    zeroed).  Sequences never share a chunk or a state.
    Returns dict with out [sum(T), H] (bf16 values), conv_state, ssm_state
    (final, per sequence) and, when keep=True, the intermediates.  map_fn, if
    given, runs the recurrence group by group through it (ssd_by_group).
    arm: "w8a8" (the device arm: both projections fp8_linear on e4m3
    activations) or "w8a16" (the host reference arm: bf16 activations
    against dequantised bf16 weights, bf16_linear); everything between the
    projections is the same.
    """
    assert arm in ("w8a8", "w8a16")
    H, I, nh, P, G, N, W = _dims(Wt)
    conv_dim = I + 2 * G * N
    hidden = np.asarray(hidden, np.float64)
    if arm == "w8a16":
        q = None
        zx = bf16_linear(hidden, dequant_e4m3_bf16(Wt["in_proj"], Wt["s_w1"]))
    else:
        q = quant_static_e4m3(hidden, Wt["s_x"])
        zx = fp8_linear(q, Wt["s_x"], Wt["in_proj"], Wt["s_w1"])
    z, xbc, dt_raw = split_zxbcdt(zx, I, conv_dim, nh)
    A = -np.exp(np.asarray(Wt["A_log"], np.float64))
    dt = softplus(dt_raw + np.asarray(Wt["dt_bias"], np.float64)[None, :])

    T_total = hidden.shape[0]
    u = np.empty((T_total, conv_dim))
    y = np.empty((T_total, I))
    conv_out = np.empty_like(np.asarray(conv_state, np.float64))
    ssm_out = np.empty_like(np.asarray(ssm_state, np.float64))
    start = 0
    for s, T in enumerate(seqlens):
        sl = slice(start, start + T)
        u[sl], conv_out[s] = causal_conv1d_silu(xbc[sl], Wt["conv_w"], Wt["conv_b"], conv_state[s])
        xs, Bs, Cs = split_xbc(u[sl], I, G, N)
        args = (xs.reshape(T, nh, P), dt[sl], A, Bs.reshape(T, G, N), Cs.reshape(T, G, N),
                Wt["D"], ssm_state[s])
        if map_fn is None:
            ys, ssm_out[s] = ssd_sequential(*args)
        else:
            ys, ssm_out[s] = ssd_by_group(*args, map_fn=map_fn)
        y[sl] = bf16_round(ys.reshape(T, I))
        start += T
    o = bf16_round(gated_rmsnorm_group(y, z, Wt["norm_w"], G, Wt["eps"]))
    if arm == "w8a16":
        q2 = None
        out = bf16_linear(o, dequant_e4m3_bf16(Wt["out_proj"], Wt["s_w2"]))
    else:
        q2 = quant_static_e4m3(o, Wt["s_y"])
        out = fp8_linear(q2, Wt["s_y"], Wt["out_proj"], Wt["s_w2"])
    res = dict(out=out, conv_state=conv_out, ssm_state=ssm_out)
    if keep:
        res.update(q=q, zx=zx, u=u, dt=dt, y=y, o=o, q2=q2)
    return res


def _store_state(s, state_cache):
    """The state as the caller's cache holds it: f32 rows are returned in full
    precision (the tests compare against the exact value), bf16 rows rounded
    to nearest even (a non-f32 mamba_ssm_cache_dtype, PR #1288 "What it does",
    the ssm_dtype term: the recurrence itself runs in full precision, only
    the stored rows are narrowed)."""
    return bf16_round(s) if state_cache == "bf16" else s


def block_prefill(Wt, hidden, seqlens, conv_state=None, ssm_state=None, keep=False, map_fn=None,
                  state_cache="f32", arm="w8a8"):
    """Prefill of packed sequences; missing states mean fresh sequences.
    state_cache: "f32" or "bf16" (the final ssm states are rounded to bf16);
    arm: "w8a8" or "w8a16" (block_tokens)."""
    H, I, nh, P, G, N, W = _dims(Wt)
    nseq = len(seqlens)
    if conv_state is None:
        conv_state = np.zeros((nseq, I + 2 * G * N, W - 1))
    if ssm_state is None:
        ssm_state = np.zeros((nseq, nh, P, N))
    res = block_tokens(Wt, hidden, seqlens, conv_state, ssm_state, keep=keep, map_fn=map_fn, arm=arm)
    res["ssm_state"] = _store_state(res["ssm_state"], state_cache)
    return res


def block_decode(Wt, hidden, conv_pool, ssm_pool, slot_idx, keep=False, state_cache="f32", arm="w8a8"):
    """One decode token per row, states gathered from a slot pool.

    Row b reads pool[slot_idx[b]] (decode rows always have prior state,
    PR #1288 "What it does": has_initial = true), advances it one token; the
    advanced rows are what the pool holds at those slots afterwards (the
    scatter), every other slot is unchanged.  slot_idx[b] == -1 marks a
    padding row: output zero, no state read or written.
    Returns dict(out [Bt, H], live (row numbers with a slot), conv_rows,
    ssm_rows (the new pool contents at slot_idx[live])).  Inputs are not
    modified.  state_cache "bf16": the pool rows are bf16 values, widened
    exactly when read; y uses the advanced state in full precision, and the
    rows written back are rounded to bf16.  arm: "w8a8" or "w8a16"
    (block_tokens).
    """
    slot_idx = np.asarray(slot_idx)
    live = np.nonzero(slot_idx >= 0)[0]
    H = Wt["geo"].hidden
    out = np.zeros((len(slot_idx), H))
    res = dict(out=out, live=live)
    if len(live):
        rows = slot_idx[live]
        r = block_tokens(Wt, np.asarray(hidden, np.float64)[live], [1] * len(live),
                         np.asarray(conv_pool[rows], np.float64),
                         np.asarray(ssm_pool[rows], np.float64), keep=keep, arm=arm)
        out[live] = r["out"]
        res["conv_rows"] = r["conv_state"]
        res["ssm_rows"] = _store_state(r["ssm_state"], state_cache)
        if keep:
            res.update({k: r[k] for k in ("q", "zx", "u", "dt", "y", "o", "q2")})
    return res


def stack_prefill(layers, norm_ws, hidden, seqlens, eps: float, map_fn=None):
    """Pre-norm residual stack: h <- h + block_l(rmsnorm(h) * w_l), all bf16.
    `layers` may be a list or a callable l -> weights (generated on demand).
    Returns (h_out, final conv states per layer, final ssm states per layer)."""
    h = np.asarray(hidden, np.float64)
    convs, ssms = [], []
    for l, nw in enumerate(norm_ws):
        Wt = layers(l) if callable(layers) else layers[l]
        r = block_prefill(Wt, rmsnorm(h, nw, eps), seqlens, map_fn=map_fn)
        h = bf16_round(h + r["out"])
        convs.append(r["conv_state"])
        ssms.append(r["ssm_state"])
    return h, convs, ssms


def stack_decode(layers, norm_ws, hidden, conv_pools, ssm_pools, slot_idx, eps: float):
    """Decode through the stack; layer l reads its own pools.  Returns
    (h_out, per-layer new conv rows, per-layer new ssm rows) for the live rows."""
    h = np.asarray(hidden, np.float64)
    conv_rows, ssm_rows = [], []
    for Wt, nw, cp, sp in zip(layers, norm_ws, conv_pools, ssm_pools):
        r = block_decode(Wt, rmsnorm(h, nw, eps), cp, sp, slot_idx)
        h = bf16_round(h + r["out"])
        conv_rows.append(r.get("conv_rows"))
        ssm_rows.append(r.get("ssm_rows"))
    return h, conv_rows, ssm_rows
