"""Pins of the CPU oracle against things other than itself.

Each test ties one oracle function to a closed form, a brute-force search, a
library routine, an independent formulation of the same mathematics, or the
numbers the pages print.  None of them re-types the oracle's formula.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")

TINY = synth.Geometry(hidden=32, d_inner=16, nheads=4, headdim=4, n_groups=2, d_state=8, conv_width=4)


# ---------------------------------------------------------------- e4m3 codec

def _golden_e4m3():
    rows = []
    for line in open(os.path.join(GOLDEN, "e4m3_ocp.txt")):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        c, v = line.split()
        rows.append((int(c, 16), float(v)))
    return rows


def test_e4m3_decode_matches_ocp_table():
    for code, val in _golden_e4m3():
        got = oracle.e4m3_decode(np.array([code], np.uint8))[0]
        if math.isnan(val):
            assert math.isnan(got)
        else:
            assert got == val and math.copysign(1, got) == math.copysign(1, val), hex(code)


def test_e4m3_decode_matches_torch_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = oracle.e4m3_decode(codes)
    assert np.array_equal(np.isnan(ref), np.isnan(got))
    fin = ~np.isnan(ref)
    assert np.array_equal(ref[fin], got[fin])
    assert fin.sum() == 254


def _finite_e4m3_table():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)
    vals = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    return codes, vals


def _brute_force_encode(x):
    """Nearest finite e4m3 by exhaustive distance, ties to the even code,
    saturating at 448, NaN -> 0x7F."""
    codes, vals = _finite_e4m3_table()
    x = np.asarray(x, np.float64)
    out = np.empty(x.shape, np.uint8)
    flat, res = x.ravel(), out.ravel()
    for i0 in range(0, flat.size, 4096):
        v = flat[i0:i0 + 4096]
        d = np.abs(v[:, None] - vals[None, :])
        dmin = d.min(axis=1, keepdims=True)
        cand = d == dmin
        # among equal distances prefer even code, and keep the sign of v for zero
        score = np.where(cand, 0, 4) + (codes[None, :] & 1) * 2 + \
            (np.signbit(vals)[None, :] != np.signbit(v)[:, None])
        pick = codes[np.argmin(score, axis=1)]
        sat = np.abs(v) >= 448.0
        pick = np.where(sat, np.where(np.signbit(v), 0xFE, 0x7E), pick)
        pick = np.where(np.isnan(v), 0x7F, pick)
        res[i0:i0 + 4096] = pick
    return out


@pytest.mark.parametrize("scale", [1.0 / 64.0, 1.0, 1.0 / 3.0])
def test_e4m3_encode_all_bf16_patterns_brute_force(scale):
    bits = np.arange(65536, dtype=np.uint32) << 16
    x = bits.view(np.float32)
    q = (x / np.float32(scale)).astype(np.float32)
    got = oracle.e4m3_encode(q)
    ref = _brute_force_encode(q)
    nan = np.isnan(q)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.all(got[nan] & 0x7F == 0x7F)


def test_e4m3_encode_matches_torch_in_range():
    rng = np.random.default_rng(5)
    x = np.concatenate([rng.standard_normal(200000) * 50, rng.standard_normal(50000) * 1e-2,
                        oracle.e4m3_decode(np.arange(0x7E, dtype=np.uint8))]).astype(np.float32)
    # exact midpoints between neighbouring codes: tie cases
    pos = oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    mids = ((pos[:-1] + pos[1:]) / 2).astype(np.float32)
    x = np.concatenate([x, mids, -mids])
    x = x[np.abs(x) < 448]
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(oracle.e4m3_encode(x), ref)


def test_e4m3_encode_saturates():
    x = np.array([448.0, 449.0, 464.0, 500.0, 1e30, np.inf, -np.inf, -1e9], np.float32)
    assert list(oracle.e4m3_encode(x)) == [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0xFE]


def test_e4m3_roundtrip_all_finite_codes():
    codes, vals = _finite_e4m3_table()
    assert np.array_equal(oracle.e4m3_encode(vals), codes)


# ---------------------------------------------------------------- bf16 rounding

def test_bf16_round_matches_torch_on_float32():
    rng = np.random.default_rng(7)
    bits = rng.integers(0, 2 ** 32, 400000, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    x = x[np.isfinite(x)]
    # add exact ties: bf16 value + half a bf16 ulp
    base = (rng.integers(0, 2 ** 16, 20000, dtype=np.uint32) << 16).view(np.float32)
    tie = ((base.view(np.uint32) | 0x8000)).view(np.float32)
    x = np.concatenate([x, tie[np.isfinite(tie)]])
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    got = oracle.bf16_round(x.astype(np.float64))
    assert np.array_equal(ref, got)


def test_bf16_round_no_double_rounding():
    # 1 + 2^-8 + 2^-30 is just above a bf16 tie; via float32 it would hit the tie and round to even (1.0)
    x = np.array([1.0 + 2.0 ** -8 + 2.0 ** -30])
    assert oracle.bf16_round(x)[0] == 1.0 + 2.0 ** -7


# ---------------------------------------------------------------- fp8 linear

def test_fp8_linear_integer_valued_is_exact():
    rng = np.random.default_rng(11)
    ints = np.arange(-8, 9)
    code_of = {int(v): int(oracle.e4m3_encode(np.array([float(v)]))[0]) for v in ints}
    a_i = rng.integers(-8, 9, (9, 2688))
    w_i = rng.integers(-8, 9, (40, 2688))
    a_q = np.vectorize(code_of.get)(a_i).astype(np.uint8)
    w_q = np.vectorize(code_of.get)(w_i).astype(np.uint8)
    exact = a_i.astype(np.int64) @ w_i.astype(np.int64).T
    ref = torch.from_numpy(exact.astype(np.float32)).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.abs(exact).max() < 2 ** 24
    assert np.array_equal(oracle.fp8_linear(a_q, 1.0, w_q, 1.0), ref)


def test_fp8_linear_scales_and_orientation_vs_torch():
    rng = np.random.default_rng(12)
    a_q = rng.integers(0, 256, (5, 64)).astype(np.uint8)
    w_q = rng.integers(0, 256, (7, 64)).astype(np.uint8)
    a_q[(a_q & 0x7F) == 0x7F] = 0
    w_q[(w_q & 0x7F) == 0x7F] = 0
    a = torch.from_numpy(a_q).view(torch.float8_e4m3fn).to(torch.float64)
    w = torch.from_numpy(w_q).view(torch.float8_e4m3fn).to(torch.float64)
    ref = torch.nn.functional.linear(a, w) * (0.25 * 0.003)
    got = oracle.fp8_linear(a_q, 0.25, w_q, 0.003)
    assert got.shape == (5, 7)
    np.testing.assert_allclose(got, ref.numpy(), rtol=2 ** -8, atol=0)


# ---------------------------------------------------------------- elementwise

def test_silu_softplus_vs_torch():
    v = np.linspace(-40, 40, 20001)
    t = torch.from_numpy(v)
    np.testing.assert_allclose(oracle.silu(v), torch.nn.functional.silu(t).numpy(), rtol=1e-14, atol=1e-300)
    np.testing.assert_allclose(oracle.softplus(v), torch.nn.functional.softplus(t).numpy(), rtol=3e-9, atol=0)


# ---------------------------------------------------------------- conv1d

def _conv_brute(x, w, b, state):
    T, C = x.shape
    W = w.shape[1]
    u = np.zeros((T, C))
    for c in range(C):
        hist = list(state[c]) + list(x[:, c])
        for t in range(T):
            acc = 0.0 if b is None else b[c]
            for j in range(W):
                acc += w[c, j] * hist[t + j]
            u[t, c] = acc / (1.0 + math.exp(-acc))
        newst = hist[-(W - 1):]
        state_out = newst
    return u


@pytest.mark.parametrize("T", [1, 2, 3, 7])
def test_conv_brute_force(T):
    rng = np.random.default_rng(T)
    C, W = 5, 4
    x = synth.as_bf16_values(rng.standard_normal((T, C)))
    w = rng.standard_normal((C, W))
    b = rng.standard_normal(C)
    st = rng.standard_normal((C, W - 1))
    u, new_st = oracle.causal_conv1d_silu(x, w, b, st)
    ref = _conv_brute(x, w, b, st)
    np.testing.assert_allclose(u, ref, rtol=2 ** -8, atol=1e-30)
    # new state: the last W-1 raw inputs of [old state, x], oldest first
    for c in range(C):
        hist = list(st[c]) + list(x[:, c])
        assert np.array_equal(new_st[c], np.array(hist[-(W - 1):]))


def test_conv_prefill_equals_single_steps():
    rng = np.random.default_rng(3)
    T, C, W = 9, 6, 4
    x = rng.standard_normal((T, C))
    w = rng.standard_normal((C, W))
    st0 = rng.standard_normal((C, W - 1))
    u_all, st_all = oracle.causal_conv1d_silu(x, w, None, st0)
    st = st0
    for t in range(T):
        u_t, st = oracle.causal_conv1d_silu(x[t:t + 1], w, None, st)
        assert np.array_equal(u_t[0], u_all[t])
    assert np.array_equal(st, st_all)


# ---------------------------------------------------------------- SSD scan

def _ssd_inputs(rng, T, nh=4, P=3, G=2, N=5, init=True):
    x = rng.standard_normal((T, nh, P))
    dt = np.exp(rng.uniform(np.log(1e-3), np.log(0.5), (T, nh)))
    A = -np.exp(rng.uniform(0, np.log(16), nh))
    B = rng.standard_normal((T, G, N))
    C = rng.standard_normal((T, G, N))
    D = rng.standard_normal(nh)
    S0 = rng.standard_normal((nh, P, N)) * (0.3 if init else 0.0)
    return x, dt, A, B, C, D, S0


def _ssd_chunked(x, dt, A, B, C, D, S0, L):
    """Block decomposition of the SSD layer (Dao & Gu 2024, section 6):
    within a chunk the output is the masked quadratic form; chunk states are
    handed across chunk boundaries.  Written independently of the oracle."""
    T, nh, P = x.shape
    G = B.shape[1]
    hpg = nh // G
    S = S0.copy()
    y = np.zeros_like(x)
    for c0 in range(0, T, L):
        c1 = min(T, c0 + L)
        n = c1 - c0
        for h in range(nh):
            g = h // hpg
            a = dt[c0:c1, h] * A[h]
            cum = np.cumsum(a)                                   # [n]
            seg = cum[:, None] - cum[None, :]                    # sum_{k=j+1..i} a_k
            mask = np.tril(np.ones((n, n), bool))
            Lmat = np.where(mask, np.exp(np.where(mask, seg, 0.0)), 0.0)
            CB = C[c0:c1, g] @ B[c0:c1, g].T                     # [n, n]
            Ydiag = (CB * Lmat * dt[c0:c1, h][None, :]) @ x[c0:c1, h]
            Yoff = np.exp(cum)[:, None] * (C[c0:c1, g] @ S[h].T)
            y[c0:c1, h] = Ydiag + Yoff + D[h] * x[c0:c1, h]
            w = np.exp(cum[-1] - cum) * dt[c0:c1, h]             # [n]
            S[h] = np.exp(cum[-1]) * S[h] + (x[c0:c1, h] * w[:, None]).T @ B[c0:c1, g]
    return y, S


@pytest.mark.parametrize("T,L", [(1, 4), (5, 4), (16, 4), (37, 16), (70, 16), (64, 64)])
def test_ssd_sequential_equals_chunked(T, L):
    rng = np.random.default_rng(100 + T)
    args = _ssd_inputs(rng, T)
    y1, S1 = oracle.ssd_sequential(*args)
    y2, S2 = _ssd_chunked(*args, L=L)
    np.testing.assert_allclose(y1, y2, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(S1, S2, rtol=1e-10, atol=1e-12)


def test_ssd_equals_materialised_semiseparable_matrix():
    """y = M x with M[i, j] = C_i . B_j * prod_{k=j+1..i} exp(dt_k A) * dt_j
    (the 'attention-like' dual form) plus the decayed initial state."""
    rng = np.random.default_rng(21)
    T = 11
    x, dt, A, B, C, D, S0 = _ssd_inputs(rng, T)
    nh, P = x.shape[1:]
    G = B.shape[1]
    y_ref = np.zeros_like(x)
    for h in range(nh):
        g = h // (nh // G)
        for i in range(T):
            acc = np.zeros(P)
            for j in range(i + 1):
                dec = 1.0
                for k in range(j + 1, i + 1):
                    dec *= math.exp(dt[k, h] * A[h])
                acc += (C[i, g] @ B[j, g]) * dec * dt[j, h] * x[j, h]
            dec0 = math.exp(sum(dt[k, h] * A[h] for k in range(i + 1)))
            acc += dec0 * (S0[h] @ C[i, g])
            y_ref[i, h] = acc + D[h] * x[i, h]
    y, _ = oracle.ssd_sequential(x, dt, A, B, C, D, S0)
    np.testing.assert_allclose(y, y_ref, rtol=1e-11, atol=1e-12)


def test_ssd_A_zero_closed_form():
    rng = np.random.default_rng(22)
    x, dt, A, B, C, D, S0 = _ssd_inputs(rng, 9)
    A = np.zeros_like(A)
    _, S = oracle.ssd_sequential(x, dt, A, B, C, D, S0)
    nh = x.shape[1]
    hpg = nh // B.shape[1]
    S_ref = S0.copy()
    for h in range(nh):
        S_ref[h] += np.einsum("t,tp,tn->pn", dt[:, h], x[:, h], B[:, h // hpg])
    np.testing.assert_allclose(S, S_ref, rtol=1e-12, atol=1e-12)


def test_ssd_single_token_from_zero_closed_form():
    rng = np.random.default_rng(23)
    x, dt, A, B, C, D, S0 = _ssd_inputs(rng, 1, init=False)
    y, S = oracle.ssd_sequential(x, dt, A, B, C, D, S0)
    nh = x.shape[1]
    hpg = nh // B.shape[1]
    for h in range(nh):
        g = h // hpg
        np.testing.assert_allclose(y[0, h], dt[0, h] * (C[0, g] @ B[0, g]) * x[0, h] + D[h] * x[0, h], rtol=1e-12)


def test_ssd_zero_dt_keeps_state():
    rng = np.random.default_rng(24)
    x, dt, A, B, C, D, S0 = _ssd_inputs(rng, 6)
    dt = np.zeros_like(dt)
    y, S = oracle.ssd_sequential(x, dt, A, B, C, D, S0)
    assert np.array_equal(S, S0)
    hpg = x.shape[1] // B.shape[1]
    for t in range(6):
        for h in range(x.shape[1]):
            np.testing.assert_allclose(y[t, h], S0[h] @ C[t, h // hpg] + D[h] * x[t, h], rtol=1e-12)


def test_ssd_head_group_map_is_contiguous():
    """Heads 0..hpg-1 read group 0: zeroing group 1's B leaves them unchanged."""
    rng = np.random.default_rng(25)
    x, dt, A, B, C, D, S0 = _ssd_inputs(rng, 5, init=False)
    y1, _ = oracle.ssd_sequential(x, dt, A, B, C, D, S0)
    B2 = B.copy()
    B2[:, 1] = 0
    y2, _ = oracle.ssd_sequential(x, dt, A, B2, C, D, S0)
    assert np.array_equal(y1[:, :2], y2[:, :2])
    assert not np.allclose(y1[:, 2:], y2[:, 2:])


# ---------------------------------------------------------------- gated norm

def test_gated_norm_vs_torch_rms_norm():
    rng = np.random.default_rng(31)
    T, I, G = 6, 48, 4
    y = rng.standard_normal((T, I))
    z = rng.standard_normal((T, I))
    w = rng.standard_normal(I)
    g = torch.from_numpy(y) * torch.nn.functional.silu(torch.from_numpy(z))
    ref = torch.cat([torch.nn.functional.rms_norm(g[:, k * 12:(k + 1) * 12], (12,),
                                                  torch.from_numpy(w[k * 12:(k + 1) * 12]), eps=1e-5)
                     for k in range(G)], dim=1).numpy()
    np.testing.assert_allclose(oracle.gated_rmsnorm_group(y, z, w, G, 1e-5), ref, rtol=1e-12, atol=1e-14)


def test_gated_norm_constant_vector_closed_form():
    I, G, eps = 32, 2, 1e-5
    for gval in [0.3, -2.0, 1e-4]:
        zbig = 40.0                                           # silu(40) == 40 to 1e-16
        y = np.full((1, I), gval / zbig * (1 + math.exp(-zbig)))
        z = np.full((1, I), zbig)
        w = np.linspace(0.5, 1.5, I)
        o = oracle.gated_rmsnorm_group(y, z, w, G, eps)
        np.testing.assert_allclose(o[0], w * gval / math.sqrt(gval * gval + eps), rtol=1e-12)


def test_rmsnorm_vs_torch():
    rng = np.random.default_rng(32)
    h = synth.as_bf16_values(rng.standard_normal((5, 64)) * 3)
    w = synth.as_bf16_values(1 + 0.1 * rng.standard_normal(64))
    ref = torch.nn.functional.rms_norm(torch.from_numpy(h.astype(np.float64)), (64,),
                                       torch.from_numpy(w.astype(np.float64)), eps=1e-5)
    ref = ref.to(torch.float32).to(torch.bfloat16).to(torch.float64).numpy()
    got = oracle.rmsnorm(h, w, 1e-5)
    assert np.mean(got != ref) < 1e-3           # only double-rounding ties may differ
    np.testing.assert_allclose(got, ref, rtol=2 ** -7)


# ---------------------------------------------------------------- geometry (pages)

def test_geometry_matches_pages():
    g = json.load(open(os.path.join(GOLDEN, "geometry.json")))
    geo = synth.NEMOTRON_H
    assert geo.zx_width == g["in_proj_out"] == geo.d_inner + geo.conv_dim + geo.nheads
    assert geo.hidden == g["in_proj_in"] == g["out_proj_out"]
    assert geo.d_inner == g["out_proj_in"]
    total = g["n_mamba_blocks"] * (geo.zx_width * geo.hidden + geo.hidden * geo.d_inner)
    assert abs(total - g["fp8_elements_23_blocks_approx"]) / g["fp8_elements_23_blocks_approx"] < 1e-3


def test_split_contract_head_middle_tail():
    geo = synth.NEMOTRON_H
    row = np.arange(geo.zx_width, dtype=np.float64)[None, :]
    z, xbc, dt = oracle.split_zxbcdt(row, geo.d_inner, geo.conv_dim, geo.nheads)
    assert z.shape[-1] == geo.d_inner and xbc.shape[-1] == geo.conv_dim and dt.shape[-1] == geo.nheads
    assert z[0, 0] == 0 and xbc[0, 0] == geo.d_inner and dt[0, 0] == geo.d_inner + geo.conv_dim
    assert dt[0, -1] == geo.zx_width - 1
    x, B, C = oracle.split_xbc(xbc, geo.d_inner, geo.n_groups, geo.d_state)
    assert (x.shape[-1], B.shape[-1], C.shape[-1]) == (4096, 1024, 1024)
    assert B[0, 0] == 2 * geo.d_inner and C[0, -1] == geo.d_inner + geo.conv_dim - 1


# ---------------------------------------------------------------- block level

@pytest.fixture(scope="module")
def tiny_weights():
    return synth.make_weights(90, 0, TINY)


def test_block_decode_after_prefill_equals_longer_prefill(tiny_weights):
    """The carry case: prefill t0 tokens, then decode the rest one at a time
    from the returned states; equals one prefill over all tokens."""
    Wt = tiny_weights
    T, t0 = 12, 5
    h = synth.make_hidden(90, T, TINY)
    full = oracle.block_prefill(Wt, h, [T])
    part = oracle.block_prefill(Wt, h[:t0], [t0])
    conv_pool = part["conv_state"].copy()
    ssm_pool = part["ssm_state"].copy()
    outs = [part["out"]]
    for t in range(t0, T):
        r = oracle.block_decode(Wt, h[t:t + 1], conv_pool, ssm_pool, np.array([0]))
        conv_pool[0], ssm_pool[0] = r["conv_rows"][0], r["ssm_rows"][0]
        outs.append(r["out"])
    np.testing.assert_allclose(np.concatenate(outs), full["out"], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(ssm_pool[0], full["ssm_state"][0], rtol=1e-10, atol=1e-13)
    np.testing.assert_array_equal(conv_pool[0], full["conv_state"][0])


def test_block_dropped_carry_separates(tiny_weights):
    """Zeroed-twin method: restarting from a zero state must change the
    output by far more than rounding noise."""
    Wt = tiny_weights
    T, t0 = 12, 8
    h = synth.make_hidden(91, T, TINY)
    full = oracle.block_prefill(Wt, h, [T])
    fresh = oracle.block_prefill(Wt, h[t0:], [T - t0])
    sep = np.linalg.norm(fresh["out"] - full["out"][t0:]) / np.linalg.norm(full["out"][t0:])
    assert sep > 0.05


def test_block_varlen_equals_separate_calls(tiny_weights):
    Wt = tiny_weights
    lens = [7, 1, 4]
    h = synth.make_hidden(92, sum(lens), TINY)
    packed = oracle.block_prefill(Wt, h, lens)
    s = 0
    for i, n in enumerate(lens):
        r = oracle.block_prefill(Wt, h[s:s + n], [n])
        np.testing.assert_array_equal(packed["out"][s:s + n], r["out"])
        np.testing.assert_array_equal(packed["ssm_state"][i], r["ssm_state"][0])
        s += n


def test_block_decode_padding_and_untouched_slots(tiny_weights):
    Wt = tiny_weights
    rng = np.random.default_rng(93)
    nslots = 6
    conv_pool = synth.as_bf16_values(rng.standard_normal((nslots, TINY.conv_dim, 3)))
    ssm_pool = rng.standard_normal((nslots, TINY.nheads, TINY.headdim, TINY.d_state)) * 0.1
    h = synth.make_hidden(93, 3, TINY)
    r = oracle.block_decode(Wt, h, conv_pool, ssm_pool, np.array([4, -1, 1]))
    assert np.array_equal(r["live"], [0, 2])
    assert np.all(r["out"][1] == 0)
    r1 = oracle.block_decode(Wt, h[2:3], conv_pool, ssm_pool, np.array([1]))
    np.testing.assert_array_equal(r1["out"][0], r["out"][2])
    np.testing.assert_array_equal(r1["ssm_rows"][0], r["ssm_rows"][1])


def test_block_ssm_state_is_float_and_counts(tiny_weights):
    """Element counts asserted against the geometry (a maximum over zero
    elements would also be 0.0)."""
    Wt = tiny_weights
    h = synth.make_hidden(94, 4, TINY)
    r = oracle.block_prefill(Wt, h, [4], keep=True)
    assert r["out"].size == 4 * TINY.hidden
    assert r["zx"].shape == (4, TINY.zx_width)
    assert r["u"].shape == (4, TINY.conv_dim)
    assert r["ssm_state"].shape == (1, TINY.nheads, TINY.headdim, TINY.d_state)
    assert r["ssm_state"].dtype == np.float64
    assert np.count_nonzero(r["ssm_state"]) == r["ssm_state"].size


# ---------------------------------------------------------------- mutations

def test_mutation_wrong_group_map_is_caught(monkeypatch):
    """Plant a transposed head->group map in the oracle; the independent
    chunked form must disagree."""
    rng = np.random.default_rng(41)
    args = _ssd_inputs(rng, 8)
    orig_repeat = np.repeat

    def bad_repeat(a, reps, axis=None):
        if axis == 0 and a.ndim == 2:
            return np.tile(a, (reps, 1))            # h % G instead of h // hpg
        return orig_repeat(a, reps, axis=axis)
    monkeypatch.setattr(oracle.m2_oracle.np, "repeat", bad_repeat)
    y1, _ = oracle.ssd_sequential(*args)
    monkeypatch.undo()
    y2, _ = _ssd_chunked(*args, L=4)
    assert not np.allclose(y1, y2, rtol=1e-6)


def test_mutation_decay_sign_is_caught():
    rng = np.random.default_rng(42)
    x, dt, A, B, C, D, S0 = _ssd_inputs(rng, 8)
    y_bad, _ = oracle.ssd_sequential(x, dt, -A, B, C, D, S0)
    y_ref, _ = _ssd_chunked(x, dt, A, B, C, D, S0, L=4)
    assert not np.allclose(y_bad, y_ref, rtol=1e-6)


def test_ssd_by_group_equals_sequential():
    rng = np.random.default_rng(26)
    args = _ssd_inputs(rng, 13)
    y1, S1 = oracle.ssd_sequential(*args)
    y2, S2 = oracle.ssd_by_group(*args)
    assert np.array_equal(y1, y2) and np.array_equal(S1, S2)


# ---------------------------------------------------------------- bf16 state cache

def test_bf16_state_cache_changes_only_the_stored_rows(tiny_weights):
    """A bf16 state cache holds bf16 values: reading them widens exactly, so
    with a bf16-valued pool the output is the f32-cache output bit for bit and
    the stored rows are those rows rounded to nearest even (torch's cast)."""
    Wt = tiny_weights
    rng = np.random.default_rng(96)
    g = Wt["geo"]
    nslots, Bt = 5, 3
    conv = synth.as_bf16_values(rng.standard_normal((nslots, g.conv_dim, g.conv_width - 1)))
    ssm = synth.as_bf16_values(rng.standard_normal((nslots, g.nheads, g.headdim, g.d_state)) * 0.1)
    h = synth.make_hidden(96, Bt, g)
    slots = np.array([4, 0, 2])
    a = oracle.block_decode(Wt, h, conv, ssm, slots)
    b = oracle.block_decode(Wt, h, conv, ssm, slots, state_cache="bf16")
    np.testing.assert_array_equal(a["out"], b["out"])
    ref = torch.from_numpy(a["ssm_rows"]).to(torch.float32).to(torch.bfloat16).to(torch.float64).numpy()
    # the f64 rows pass through f32 in torch; an f64 -> bf16 rounding and an
    # f64 -> f32 -> bf16 rounding agree except at double-rounding ties
    assert np.mean(b["ssm_rows"] != ref) < 1e-4
    assert np.array_equal(b["ssm_rows"], synth.as_bf16_values(b["ssm_rows"]))


def test_bf16_state_cache_rounds_after_every_step(tiny_weights):
    """Two decode steps through a bf16 cache = step, round, step, round; the
    rounding is not deferred to the end (rows carried in full precision
    differ)."""
    Wt = tiny_weights
    g = Wt["geo"]
    rng = np.random.default_rng(97)
    conv = synth.as_bf16_values(rng.standard_normal((1, g.conv_dim, g.conv_width - 1)))
    ssm = synth.as_bf16_values(rng.standard_normal((1, g.nheads, g.headdim, g.d_state)) * 0.1)
    h = synth.make_hidden(97, 2, g)
    s = np.array([0])
    r1 = oracle.block_decode(Wt, h[:1], conv, ssm, s, state_cache="bf16")
    r2 = oracle.block_decode(Wt, h[1:], r1["conv_rows"], r1["ssm_rows"], s, state_cache="bf16")
    f1 = oracle.block_decode(Wt, h[:1], conv, ssm, s)
    f2 = oracle.block_decode(Wt, h[1:], f1["conv_rows"], f1["ssm_rows"], s)
    np.testing.assert_array_equal(r1["ssm_rows"], oracle.bf16_round(f1["ssm_rows"]))
    assert not np.array_equal(r2["ssm_rows"], oracle.bf16_round(f2["ssm_rows"]))
    rel = np.linalg.norm(r2["ssm_rows"] - f2["ssm_rows"]) / np.linalg.norm(f2["ssm_rows"])
    assert 1e-5 < rel < 1e-2                       # bf16-level, not a different state


def test_bf16_state_cache_prefill_final_state(tiny_weights):
    Wt = tiny_weights
    h = synth.make_hidden(98, 9, Wt["geo"])
    a = oracle.block_prefill(Wt, h, [9])
    b = oracle.block_prefill(Wt, h, [9], state_cache="bf16")
    np.testing.assert_array_equal(a["out"], b["out"])
    np.testing.assert_array_equal(b["ssm_state"], oracle.bf16_round(a["ssm_state"]))


# ---------------------------------------------------------------- W8A16 arm

def test_dequant_power_of_two_scale_is_exact():
    """With a power-of-two weight scale the dequantised weight is the code's
    value (the published OCP table) times the scale, exactly."""
    rows = [(c, v) for c, v in _golden_e4m3() if not math.isnan(v)]
    codes = np.array([c for c, _ in rows], np.uint8)
    vals = np.array([v for _, v in rows])
    for k in (-9, -3, 0, 2):
        got = oracle.dequant_e4m3_bf16(codes, 2.0 ** k)
        assert np.array_equal(got, vals * 2.0 ** k), k


@pytest.mark.parametrize("scale", [0.0123 / 448, 1.7e-4, 3.3, 0.02 / 448 * 3.7])
def test_dequant_matches_torch_float32_product(scale):
    """The reading taken: product in float32, then bf16 (both nearest even).
    torch does the same two roundings with its own kernels."""
    codes = np.arange(256, dtype=np.uint8)
    codes = codes[(codes & 0x7F) != 0x7F]
    t = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float32) * torch.tensor(scale, dtype=torch.float32)
    ref = t.to(torch.bfloat16).to(torch.float64).numpy()
    got = oracle.dequant_e4m3_bf16(codes, scale)
    assert np.array_equal(got, ref)


def test_bf16_linear_integer_valued_is_exact():
    rng = np.random.default_rng(21)
    x_i = rng.integers(-8, 9, (9, 2688))
    w_i = rng.integers(-8, 9, (40, 2688))
    exact = x_i.astype(np.int64) @ w_i.astype(np.int64).T
    ref = torch.from_numpy(exact.astype(np.float32)).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.abs(exact).max() < 2 ** 24
    assert np.array_equal(oracle.bf16_linear(x_i.astype(np.float64), w_i.astype(np.float64)), ref)


def test_bf16_linear_orientation_vs_torch():
    rng = np.random.default_rng(22)
    x = oracle.bf16_round(rng.standard_normal((5, 64)))
    w = oracle.bf16_round(rng.standard_normal((7, 64)) * 0.02)
    ref = torch.nn.functional.linear(torch.from_numpy(x), torch.from_numpy(w)).numpy()
    got = oracle.bf16_linear(x, w)
    assert got.shape == (5, 7)
    np.testing.assert_allclose(got, ref, rtol=2 ** -8, atol=0)


def _pow2_scales(Wt, s_w1=2.0 ** -6, s_w2=2.0 ** -5):
    W = dict(Wt)
    W["s_w1"], W["s_w2"] = s_w1, s_w2
    return W


def test_w8a16_in_proj_on_grid_equals_w8a8(tiny_weights):
    """Activations already on the e4m3 grid (times s_x) and power-of-two
    weight scales: quantising changes nothing and dequantising is exact, so
    the two arms' in_proj outputs are the same bf16 values."""
    Wt = _pow2_scales(tiny_weights)
    rng = np.random.default_rng(94)
    codes = rng.integers(0, 256, (6, TINY.hidden)).astype(np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0
    h = oracle.e4m3_decode(codes) * Wt["s_x"]
    a = oracle.block_prefill(Wt, h, [6], keep=True, arm="w8a8")
    b = oracle.block_prefill(Wt, h, [6], keep=True, arm="w8a16")
    assert np.array_equal(a["zx"], b["zx"])
    assert b["q"] is None and b["q2"] is None


def test_w8a16_activation_is_not_quantised(tiny_weights):
    """A one-hot input row far outside the e4m3 range: the W8A16 in_proj row
    is that value times one dequantised weight column (a single product,
    rounded once to bf16); the W8A8 arm saturates it at 448 s_x instead."""
    Wt = tiny_weights
    k, v = 5, 1000.3 * Wt["s_x"]
    h = np.zeros((1, TINY.hidden))
    h[0, k] = v
    b = oracle.block_prefill(Wt, h, [1], keep=True, arm="w8a16")
    col = oracle.dequant_e4m3_bf16(Wt["in_proj"][:, k], Wt["s_w1"])
    assert np.array_equal(b["zx"][0], oracle.bf16_round(v * col))
    a = oracle.block_prefill(Wt, h, [1], keep=True, arm="w8a8")
    assert np.array_equal(a["zx"][0], oracle.bf16_round(448.0 * Wt["s_x"] * Wt["s_w1"]
                                                       * oracle.e4m3_decode(Wt["in_proj"][:, k])))
    assert not np.array_equal(a["zx"], b["zx"])


def test_w8a16_decode_after_prefill_equals_longer_prefill(tiny_weights):
    Wt = tiny_weights
    T, t0 = 10, 6
    h = synth.make_hidden(95, T, TINY)
    full = oracle.block_prefill(Wt, h, [T], arm="w8a16")
    part = oracle.block_prefill(Wt, h[:t0], [t0], arm="w8a16")
    conv_pool, ssm_pool = part["conv_state"].copy(), part["ssm_state"].copy()
    outs = [part["out"]]
    for t in range(t0, T):
        r = oracle.block_decode(Wt, h[t:t + 1], conv_pool, ssm_pool, np.array([0]), arm="w8a16")
        conv_pool[0], ssm_pool[0] = r["conv_rows"][0], r["ssm_rows"][0]
        outs.append(r["out"])
    np.testing.assert_allclose(np.concatenate(outs), full["out"], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(ssm_pool[0], full["ssm_state"][0], rtol=1e-10, atol=1e-13)


def test_w8a16_and_w8a8_arms_separate_by_the_activation_quant(tiny_weights):
    """The two arms are not bit-comparable: they differ by the e4m3
    activation quantisation (a few percent), and by nothing larger."""
    Wt = tiny_weights
    h = synth.make_hidden(96, 12, TINY)
    a = oracle.block_prefill(Wt, h, [12], arm="w8a8")["out"]
    b = oracle.block_prefill(Wt, h, [12], arm="w8a16")["out"]
    sep = np.linalg.norm(a - b) / np.linalg.norm(b)
    assert 1e-3 < sep < 0.2, sep


def test_dequant_rounds_through_float32_many_scales():
    """Over a million (code, scale) products a few dozen land where rounding
    the product to float32 first moves it onto a bf16 tie; torch's float32
    multiply and bf16 conversion decide those the same way the oracle does."""
    rng = np.random.default_rng(23)
    scales = (10 ** rng.uniform(-5, -1, 4000)).astype(np.float32)
    codes = np.arange(256, dtype=np.uint8)
    codes = codes[(codes & 0x7F) != 0x7F]
    t = (torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float32)[None, :]
         * torch.from_numpy(scales)[:, None])
    ref = t.to(torch.bfloat16).to(torch.float64).numpy()
    got = np.stack([oracle.dequant_e4m3_bf16(codes, float(s)) for s in scales])
    assert np.array_equal(got, ref)


# ---------------------------------------------------------------- the stack

def _tiny_stack(L=3):
    layers = [synth.make_weights(97, l, TINY) for l in range(L)]
    norms = [synth.make_stack_norm_w(97, l, TINY) for l in range(L)]
    return layers, norms


def test_stack_with_silent_blocks_is_the_identity():
    """Blocks whose out_proj weights are all zero add nothing: the residual
    stream passes through unchanged while every layer's states still advance."""
    layers, norms = _tiny_stack()
    for W in layers:
        W["out_proj"] = np.zeros_like(W["out_proj"])
    h = synth.make_hidden(97, 9, TINY)
    out, convs, ssms = oracle.stack_prefill(layers, norms, h, [9], 1e-5)
    assert np.array_equal(out, h)
    assert all(np.abs(s).max() > 0 for s in ssms)


def test_stack_decode_after_prefill_equals_longer_prefill():
    """The carry case through the whole stack: prefill t0 tokens, then decode
    the rest token by token from every layer's returned states."""
    layers, norms = _tiny_stack()
    T, t0 = 9, 5
    h = synth.make_hidden(98, T, TINY)
    full, fconv, fssm = oracle.stack_prefill(layers, norms, h, [T], 1e-5)
    part, convs, ssms = oracle.stack_prefill(layers, norms, h[:t0], [t0], 1e-5)
    convs = [c.copy() for c in convs]
    ssms = [s.copy() for s in ssms]
    outs = [part]
    for t in range(t0, T):
        o, crow, srow = oracle.stack_decode(layers, norms, h[t:t + 1], convs, ssms, np.array([0]), 1e-5)
        for l in range(len(layers)):
            convs[l][0], ssms[l][0] = crow[l][0], srow[l][0]
        outs.append(o)
    np.testing.assert_allclose(np.concatenate(outs), full, rtol=1e-12, atol=1e-12)
    for l in range(len(layers)):
        np.testing.assert_allclose(ssms[l][0], fssm[l][0], rtol=1e-10, atol=1e-13)
        np.testing.assert_array_equal(convs[l][0], fconv[l][0])


# ---------------------------------------------------------------- static quant

def test_f32_rounds_to_nearest_even():
    assert oracle.f32(np.array([1 + 2.0 ** -24]))[0] == 1.0                    # tie: even
    assert oracle.f32(np.array([1 + 3 * 2.0 ** -24]))[0] == 1 + 2.0 ** -22     # tie: even (up)
    assert oracle.f32(np.array([1 + 2.0 ** -24 + 2.0 ** -40]))[0] == 1 + 2.0 ** -23


def test_static_quant_matches_torch_in_range():
    """In range, the static quant equals torch's float32 division followed by
    its e4m3 cast (torch maps out-of-range values to NaN instead of
    saturating, so those are compared with the saturation pin)."""
    rng = np.random.default_rng(31)
    for s in (1 / 64, 1 / 32, 1 / 3, 0.0123):
        x = (rng.standard_normal(100000) * 2).astype(np.float32).astype(np.float64)
        q = oracle.quant_static_e4m3(x, s)
        t = (torch.from_numpy(x.astype(np.float32)) / torch.tensor(s, dtype=torch.float32)).to(
            torch.float8_e4m3fn).view(torch.uint8).numpy()
        inr = np.abs(x / s) < 448
        assert inr.mean() > 0.99
        assert np.array_equal(q[inr], t[inr])
    big = np.array([1000.0, -1e30])
    assert np.array_equal(oracle.quant_static_e4m3(big, 1.0), np.array([0x7E, 0xFE], np.uint8))


def test_static_quant_decides_on_the_float32_quotient():
    """x / s rounded to float32 lands exactly on the e4m3 tie 1.0625 (which
    goes to the even code, 1.0) although the exact quotient lies just above
    it: the decision is taken on the float32 quotient."""
    s = float(np.float32(1 / 3))
    x = float(np.float32(1.0625 * s))
    assert x / s > 1.0625 and np.float32(x) / np.float32(s) == np.float32(1.0625)
    assert oracle.quant_static_e4m3(np.array([x]), s)[0] == oracle.e4m3_encode(np.array([1.0]))[0]


# ---------------------------------------------------------------- block glue: A and dt
#
# The block turns its per-head parameters into the recurrence's inputs
# (vllm.cpp PR #1288, "What it does": the Mamba2 op chain; the reading of
# the standard Mamba-2 parameterisation): A = -exp(A_log) and
# dt = softplus(dt_raw + dt_bias), dt_raw being the in_proj output's tail.
# A block is built whose answers are exact powers of two: in_proj maps the
# first hidden column to dt_raw = 1 in every head and nothing else, so with
# x = B = C = 0 the state only decays, by exp(-a dt) per token.  Choosing
# a = exp(A_log) in {1, 2, 3} and dt_raw + dt_bias in {0, ln 3, ln 7} makes
# dt in {ln 2, ln 4, ln 8} (log(1 + e^v) with e^v in {1, 3, 7}) and the
# per-token decay 2^-(a log2(1 + e^v)); the expected values below are those
# fractions, worked by hand.

GLUE = synth.Geometry(hidden=32, d_inner=32, nheads=8, headdim=4, n_groups=2, d_state=8, conv_width=4)
_LN2, _LN3, _LN7 = math.log(2.0), math.log(3.0), math.log(7.0)
# per head: (A_log, dt_bias, dt = softplus(1 + dt_bias), per-token decay)
GLUE_HEADS = [
    (0.0, -1.0, _LN2, 1 / 2),
    (_LN2, -1.0, _LN2, 1 / 4),
    (0.0, _LN3 - 1.0, 2 * _LN2, 1 / 4),
    (_LN2, _LN3 - 1.0, 2 * _LN2, 1 / 16),
    (_LN3, -1.0, _LN2, 1 / 8),
    (0.0, _LN7 - 1.0, 3 * _LN2, 1 / 8),
    (_LN3, _LN7 - 1.0, 3 * _LN2, 1 / 512),
    (_LN2, _LN7 - 1.0, 3 * _LN2, 1 / 64),
]


def _glue_block(xbc_inputs: bool):
    """Weights of the glue block: in_proj rows of the dt tail read hidden
    column 0 with weight 1 (code 0x38); with xbc_inputs the xBC rows also read
    hidden columns 1.. with random small-integer weights."""
    g = GLUE
    Wt = dict(synth.make_weights(88, 0, g))
    conv_dim = g.d_inner + 2 * g.n_groups * g.d_state
    w = np.zeros((g.zx_width, g.hidden), np.uint8)
    one = oracle.e4m3_encode(np.array([1.0]))[0]
    w[g.d_inner + conv_dim:, 0] = one
    if xbc_inputs:
        rng = np.random.default_rng(88)
        ints = rng.integers(-3, 4, (conv_dim, g.hidden - 1))
        w[g.d_inner:g.d_inner + conv_dim, 1:] = oracle.e4m3_encode(ints.astype(np.float64))
    Wt["in_proj"] = w
    Wt["s_w1"] = 1.0
    Wt["A_log"] = np.array([r[0] for r in GLUE_HEADS], np.float32)
    Wt["dt_bias"] = np.array([r[1] for r in GLUE_HEADS], np.float32)
    Wt["conv_w"] = np.ones_like(Wt["conv_w"])
    return Wt


def test_block_glue_zero_input_decays_by_powers_of_two():
    """x = B = C = 0: the state decays by exp(T dt A); the dt the scan sees and
    the final state are the hand-worked values.  Catches A = -A_log (no decay
    where A_log = 0), a dropped, sign-flipped or misplaced dt_bias, and dt_raw
    dropped or sign-flipped."""
    g = GLUE
    Wt = _glue_block(xbc_inputs=False)
    T = 3
    h = np.zeros((T, g.hidden), np.float32)
    h[:, 0] = 1.0                      # e4m3(1 / s_x) = 64 exactly: dt_raw = s_x * 64 * 1 = 1
    conv_dim = g.d_inner + 2 * g.n_groups * g.d_state
    S0 = np.random.default_rng(89).standard_normal((1, g.nheads, g.headdim, g.d_state)) * 0.1
    r = oracle.block_prefill(Wt, h, [T], np.zeros((1, conv_dim, g.conv_width - 1)), S0, keep=True)
    assert np.all(r["zx"][:, g.d_inner + conv_dim:] == 1.0) and np.all(r["zx"][:, :g.d_inner + conv_dim] == 0)
    dt_ref = np.array([row[2] for row in GLUE_HEADS])
    np.testing.assert_allclose(r["dt"], np.broadcast_to(dt_ref, (T, g.nheads)), rtol=1e-7)
    assert np.all(r["y"] == 0)          # C = 0 and x = 0
    for h_i, row in enumerate(GLUE_HEADS):
        np.testing.assert_allclose(r["ssm_state"][0, h_i], row[3] ** T * S0[0, h_i], rtol=1e-6)


def test_block_glue_first_token_input_carries_the_same_dt():
    """From zero state one token leaves S = dt x (outer) B, with dt the
    hand-worked value of its head (the input term takes the same dt as the
    decay).  x and B are read from the conv output."""
    g = GLUE
    Wt = _glue_block(xbc_inputs=True)
    rng = np.random.default_rng(90)
    h = synth.as_bf16_values(rng.integers(-2, 3, (1, g.hidden)).astype(np.float32) / 8)
    h[0, 0] = 1.0
    conv_dim = g.d_inner + 2 * g.n_groups * g.d_state
    r = oracle.block_prefill(Wt, h, [1], np.zeros((1, conv_dim, g.conv_width - 1)),
                             np.zeros((1, g.nheads, g.headdim, g.d_state)), keep=True)
    x, B, _ = oracle.split_xbc(r["u"][0], g.d_inner, g.n_groups, g.d_state)
    x = x.reshape(g.nheads, g.headdim)
    B = B.reshape(g.n_groups, g.d_state)
    assert np.abs(x).max() > 0.1 and np.abs(B).max() > 0.1
    hpg = g.nheads // g.n_groups
    for h_i, row in enumerate(GLUE_HEADS):
        np.testing.assert_allclose(r["ssm_state"][0, h_i], row[2] * np.outer(x[h_i], B[h_i // hpg]), rtol=1e-7,
                                   atol=1e-12)
