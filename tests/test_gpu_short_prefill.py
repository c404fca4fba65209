"""Prefill calls whose sequences all have at most 64 tokens take the
token-by-token SSD kernel (one launch) instead of the chunked stages; longer
sequences take the chunked path.  Both are checked against the oracle with
the block's checks (exact e4m3 rounding of the device's own input, out_proj
of the device's codes, the decomposed output bound, states, conv windows),
at both sides of the 64-token boundary, with initial states, with a bf16
state cache, carried into decode, and inside a mixed call."""
import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import (assert_bf16_close, assert_block_out, assert_e4m3_close, assert_out_is_gemm, assert_state,
                     bf16_dev, device_weights, f32_dev, gpu_out_proj, q2_tap, rel_l2, to_np)

pytestmark = pytest.mark.gpu

m2 = pytest.importorskip("mamba2_ssm_mixer_gb300")


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.init()


@pytest.fixture(scope="module")
def block0():
    Wt = synth.make_weights(0)
    return Wt, m2.Mamba2Mixer(device_weights(Wt))


def _prefill(blk, h, lens, conv0, ssm0, has, state_dtype=torch.float32):
    T = sum(lens)
    conv = bf16_dev(conv0)
    ssm = torch.from_numpy(np.ascontiguousarray(ssm0, np.float32)).to(state_dtype).cuda()
    taps = dict(q2=torch.empty((T, 4096), dtype=torch.uint8, device="cuda"),
                o=torch.empty((T, 4096), dtype=torch.bfloat16, device="cuda"),
                y=torch.empty((T, 4096), dtype=torch.bfloat16, device="cuda"),
                dt=torch.empty((T, 64), dtype=torch.float32, device="cuda"))
    blk.set_taps(**taps)
    out = blk.prefill(bf16_dev(h), lens, conv, ssm, has_initial=has)
    blk.set_taps()
    torch.cuda.synchronize()
    blk.check()
    return out, conv, ssm, taps


def _check(Wt, out, conv, ssm, taps, ref, state_np=None):
    q2, o = to_np(taps["q2"]), to_np(taps["o"])
    assert rel_l2(to_np(taps["dt"]), ref["dt"]) < 1e-4
    assert rel_l2(to_np(taps["y"]), ref["y"]) < 1e-2
    assert_e4m3_close(q2, ref["q2"], o, ref["o"], Wt["s_y"])
    assert_out_is_gemm(to_np(out), q2, gpu_out_proj(Wt))
    assert_block_out(to_np(out), ref["out"], q2=q2, ref_q2=ref["q2"], Wt=Wt)
    assert_state(to_np(ssm) if state_np is None else state_np, ref["ssm_state"])
    assert_bf16_close(to_np(conv), ref["conv_state"], atol=1e-3, what="conv_state")


@pytest.mark.parametrize("lens,has", [([1, 2, 5, 37, 64, 3], [1, 0, 1, 0, 1, 1]),   # token by token
                                      ([1, 2, 5, 37, 65, 3], [1, 0, 1, 0, 1, 1]),   # chunked (65 > 64)
                                      ([64] * 9, [1, 0, 0, 1, 0, 1, 1, 0, 1])])
def test_short_varlen_prefill_vs_oracle(block0, lens, has):
    Wt, blk = block0
    conv0 = synth.make_conv_state(21, len(lens))
    ssm0 = synth.make_ssm_state(21, len(lens))
    h = synth.make_hidden(21, sum(lens))
    out, conv, ssm, taps = _prefill(blk, h, lens, conv0, ssm0, has)
    mask = np.array(has, np.float64)
    ref = oracle.block_prefill(Wt, h, lens, conv0 * mask[:, None, None], ssm0 * mask[:, None, None, None], keep=True)
    _check(Wt, out, conv, ssm, taps, ref)


def test_token_by_token_and_chunked_paths_agree(block0):
    """The same 48-token sequence alone (token by token) and beside a
    65-token one (chunked): outputs and final states agree to the precision
    of the chunked path's bf16 high/remainder operands."""
    Wt, blk = block0
    h = synth.make_hidden(22, 48 + 65)
    ssm0 = synth.make_ssm_state(22, 2)
    conv0 = synth.make_conv_state(22, 2)
    a_out, a_conv, a_ssm, _ = _prefill(blk, h[:48], [48], conv0[:1], ssm0[:1], [1])
    b_out, b_conv, b_ssm, _ = _prefill(blk, h, [48, 65], conv0, ssm0, [1, 1])
    assert rel_l2(to_np(a_ssm)[0], to_np(b_ssm)[0]) < 1e-4
    # the windows are raw xBC inputs; the two calls' in_proj may split K
    # differently (48 vs 113 rows), so zx may differ in its last bit
    assert_bf16_close(to_np(a_conv)[0], to_np(b_conv)[0], atol=1e-3, what="conv window")
    assert rel_l2(to_np(a_out), to_np(b_out)[:48]) < 1e-2


def test_short_prefill_bf16_state_cache():
    Wt = synth.make_weights(0)
    blk = m2.Mamba2Mixer(device_weights(Wt), ssm_dtype=m2.M2_DTYPE_BF16)
    try:
        lens, has = [7, 64, 1, 30], [1, 1, 0, 1]
        conv0 = synth.make_conv_state(23, len(lens))
        ssm0 = synth.as_bf16_values(synth.make_ssm_state(23, len(lens)))
        h = synth.make_hidden(23, sum(lens))
        out, conv, ssm, taps = _prefill(blk, h, lens, conv0, ssm0, has, state_dtype=torch.bfloat16)
        mask = np.array(has, np.float64)
        ref = oracle.block_prefill(Wt, h, lens, conv0 * mask[:, None, None], ssm0 * mask[:, None, None, None],
                                   state_cache="bf16", keep=True)
        _check(Wt, out, conv, ssm, taps, ref, state_np=ssm.to(torch.float32).cpu().numpy())
    finally:
        blk.close()


def test_short_prefill_then_decode_carry(block0):
    """A 20-token prefill (token by token) then single-token decodes from the
    returned states equals the oracle's prefill over all 26 tokens."""
    Wt, blk = block0
    T, t0 = 26, 20
    h = synth.make_hidden(24, T)
    conv = torch.zeros((1, 6144, 3), dtype=torch.bfloat16, device="cuda")
    ssm = torch.zeros((1, 64, 64, 128), dtype=torch.float32, device="cuda")
    with q2_tap(blk, t0) as q2:
        out = blk.prefill(bf16_dev(h[:t0]), [t0], conv, ssm)
    outs, q2s = [to_np(out)], [to_np(q2)]
    slot = torch.zeros(1, dtype=torch.int32, device="cuda")
    for t in range(t0, T):
        with q2_tap(blk, 1) as q2:
            outs.append(to_np(blk.decode(bf16_dev(h[t:t + 1]), conv, ssm, slot)))
        q2s.append(to_np(q2))
    torch.cuda.synchronize()
    blk.check()
    ref = oracle.block_prefill(Wt, h, [T], keep=True)
    gemm = gpu_out_proj(Wt)
    for o_, q_ in zip(outs, q2s):
        assert_out_is_gemm(o_, q_, gemm)
    assert_block_out(np.concatenate(outs), ref["out"], q2=np.concatenate(q2s), ref_q2=ref["q2"], Wt=Wt)
    assert_state(to_np(ssm), ref["ssm_state"])


def test_mixed_call_with_short_prefill_rows(block0):
    Wt, blk = block0
    n_slots, Bt, lens = 12, 4, [5, 40]
    conv_pool0 = synth.make_conv_state(25, n_slots)
    ssm_pool0 = synth.make_ssm_state(25, n_slots)
    slots = synth.make_slot_idx(25, n_slots, Bt)
    conv_st0 = synth.make_conv_state(26, len(lens))
    ssm_st0 = synth.make_ssm_state(26, len(lens))
    h = np.concatenate([synth.make_hidden(25, Bt), synth.make_hidden(26, sum(lens))])
    cp, sp = bf16_dev(conv_pool0), f32_dev(ssm_pool0)
    cs, ss = bf16_dev(conv_st0), f32_dev(ssm_st0)
    with q2_tap(blk, Bt + sum(lens)) as q2t:
        out = blk.mixed(bf16_dev(h), Bt, cp, sp, torch.from_numpy(slots).cuda(), lens, cs, ss, has_initial=[0, 1])
    torch.cuda.synchronize()
    blk.check()
    rd = oracle.block_decode(Wt, h[:Bt], conv_pool0, ssm_pool0, slots, keep=True)
    mask = np.array([0.0, 1.0])
    rp = oracle.block_prefill(Wt, h[Bt:], lens, conv_st0 * mask[:, None, None], ssm_st0 * mask[:, None, None, None],
                              keep=True)
    o, q2 = to_np(out), to_np(q2t)
    assert_out_is_gemm(o, q2, gpu_out_proj(Wt))
    assert_block_out(o[:Bt], rd["out"], q2=q2[:Bt], ref_q2=rd["q2"], Wt=Wt)
    assert_block_out(o[Bt:], rp["out"], q2=q2[Bt:], ref_q2=rp["q2"], Wt=Wt)
    assert_state(to_np(sp)[slots], rd["ssm_rows"])
    assert_state(to_np(ss), rp["ssm_state"])
    assert_bf16_close(to_np(cs), rp["conv_state"], atol=1e-3, what="conv_state")
