"""The stack glue with the next block's input quant fused into the residual
RMSNorm (m2_rmsnorm_residual_quant) and the blocks run from pre-quantised
input (m2_prefill_q / m2_decode_q).

Every kernel after the quant is shared with the bf16-input path, so the
checks are bit-exact equalities with that path (whose parity with the oracle
the other GPU tests establish), plus the fused codes against the oracle's
RMSNorm and e4m3 encoder.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import assert_e4m3_close, bf16_dev, device_weights, f32_dev, to_np

pytestmark = pytest.mark.gpu

m2 = pytest.importorskip("mamba2_ssm_mixer_gb300")


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.init()


@pytest.mark.parametrize("T", [1, 37, 256])
def test_rmsnorm_residual_quant_equals_norm_then_quant(T):
    rng = np.random.default_rng(T)
    h = synth.as_bf16_values(rng.standard_normal((T, 2688)) * 2)
    a = synth.as_bf16_values(rng.standard_normal((T, 2688)))
    w = bf16_dev(synth.make_stack_norm_w(4, 3))
    s_x = synth.S_X
    h1, h2 = bf16_dev(h), bf16_dev(h)
    normed1 = m2.m2_rmsnorm_residual(h1, bf16_dev(a), w, 1e-5)
    q1 = m2.fp8_quant(normed1, s_x)
    normed2 = torch.empty_like(h2)
    q2 = m2.m2_rmsnorm_residual_quant(h2, bf16_dev(a), w, 1e-5, s_x, normed=normed2)
    torch.cuda.synchronize()
    assert torch.equal(h1, h2)                      # the residual sum
    assert torch.equal(normed1, normed2)            # the bf16 normed row
    assert torch.equal(q1, q2)                      # the codes fp8_quant writes for it
    # against the oracle: RMSNorm in f64 then the e4m3 encoder (the bf16 normed
    # value may differ in its last bit, so a code may differ by one step)
    hs = oracle.bf16_round(h.astype(np.float64) + a)
    ref_normed = oracle.rmsnorm(hs, to_np(w), 1e-5)
    ref = oracle.quant_static_e4m3(ref_normed, s_x)
    assert_e4m3_close(to_np(q2), ref, to_np(normed2), ref_normed, s_x)


def test_rmsnorm_residual_quant_without_add_and_normed():
    rng = np.random.default_rng(5)
    h = synth.as_bf16_values(rng.standard_normal((9, 2688)))
    w = bf16_dev(synth.make_stack_norm_w(4, 0))
    hd = bf16_dev(h)
    q = m2.m2_rmsnorm_residual_quant(hd, None, w, 1e-5, 1 / 64)
    ref = m2.fp8_quant(m2.m2_rmsnorm_residual(bf16_dev(h), None, w, 1e-5), 1 / 64)
    torch.cuda.synchronize()
    assert torch.equal(q, ref)
    assert torch.equal(hd, bf16_dev(h))             # no add: h unchanged


@pytest.fixture(scope="module")
def block0():
    Wt = synth.make_weights(0)
    return Wt, m2.Mamba2Mixer(device_weights(Wt))


def test_prefill_q_equals_prefill(block0):
    Wt, blk = block0
    lens = [37, 300, 1]
    T = sum(lens)
    x = bf16_dev(synth.make_hidden(0, T))
    conv0 = bf16_dev(synth.make_conv_state(0, 3))
    ssm0 = f32_dev(synth.make_ssm_state(0, 3))
    c1, s1, c2, s2 = conv0.clone(), ssm0.clone(), conv0.clone(), ssm0.clone()
    out1 = blk.prefill(x, lens, c1, s1, has_initial=[1, 0, 1])
    out2 = blk.prefill(m2.fp8_quant(x, Wt["s_x"]), lens, c2, s2, has_initial=[1, 0, 1])
    torch.cuda.synchronize()
    blk.check()
    assert torch.equal(out1, out2) and torch.equal(c1, c2) and torch.equal(s1, s2)


def test_decode_q_equals_decode(block0):
    Wt, blk = block0
    n_slots, Bt = 32, 16
    x = bf16_dev(synth.make_hidden(2, Bt))
    conv0 = bf16_dev(synth.make_conv_state(2, n_slots))
    ssm0 = f32_dev(synth.make_ssm_state(2, n_slots))
    slots = torch.from_numpy(synth.make_slot_idx(2, n_slots, Bt)).cuda()
    c1, s1, c2, s2 = conv0.clone(), ssm0.clone(), conv0.clone(), ssm0.clone()
    out1 = blk.decode(x, c1, s1, slots)
    out2 = blk.decode(m2.fp8_quant(x, Wt["s_x"]), c2, s2, slots)
    torch.cuda.synchronize()
    blk.check()
    assert torch.equal(out1, out2) and torch.equal(c1, c2) and torch.equal(s1, s2)


def test_fused_stack_equals_unfused_stack():
    L = 3
    weights = [synth.make_weights(4, l) for l in range(L)]
    blocks = [m2.Mamba2Mixer(device_weights(w)) for w in weights]
    norm_ws = [bf16_dev(synth.make_stack_norm_w(4, l)) for l in range(L)]
    plain = m2.Mamba2Stack(blocks, norm_ws, 1e-5)
    fused = m2.Mamba2Stack(blocks, norm_ws, 1e-5, fused=True)
    # decode: 8 rows of a 24-slot pool per layer
    n_slots, Bt = 24, 8
    x = bf16_dev(synth.make_hidden(4, Bt))
    slots = torch.from_numpy(synth.make_slot_idx(4, n_slots, Bt)).cuda()
    pools = [(bf16_dev(synth.make_conv_state(4, n_slots, layer=l)), f32_dev(synth.make_ssm_state(4, n_slots, layer=l)))
             for l in range(L)]
    a = [(c.clone(), s.clone()) for c, s in pools]
    b = [(c.clone(), s.clone()) for c, s in pools]
    h1 = plain.decode(x, [c for c, _ in a], [s for _, s in a], slots)
    h2 = fused.decode(x, [c for c, _ in b], [s for _, s in b], slots)
    torch.cuda.synchronize()
    assert torch.equal(h1, h2)
    for (c1, s1), (c2, s2) in zip(a, b):
        assert torch.equal(c1, c2) and torch.equal(s1, s2)
    # prefill: two sequences, zero initial state
    lens = [300, 37]
    xp = bf16_dev(synth.make_hidden(4, sum(lens)))
    st1 = [(torch.zeros((2, 6144, 3), dtype=torch.bfloat16, device="cuda"),
            torch.zeros((2, 64, 64, 128), dtype=torch.float32, device="cuda")) for _ in range(L)]
    st2 = [(c.clone(), s.clone()) for c, s in st1]
    p1 = plain.prefill(xp, lens, [c for c, _ in st1], [s for _, s in st1])
    p2 = fused.prefill(xp, lens, [c for c, _ in st2], [s for _, s in st2])
    torch.cuda.synchronize()
    assert torch.equal(p1, p2)
    for (c1, s1), (c2, s2) in zip(st1, st2):
        assert torch.equal(c1, c2) and torch.equal(s1, s2)
    for blk in blocks:
        blk.check()
        blk.close()
