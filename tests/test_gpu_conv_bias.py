"""The conv bias (conv_b of the causal conv1d): the synthetic weights of the
other tests carry none.  With integer-valued in_proj operands every zx entry
is exact, so the conv output u (bias, then the taps, then SiLU, rounded to
bf16) is compared with the oracle's at bf16 resolution: in the prefill conv
(the chunked and the token-by-token SSD paths) and in the decode kernel's
conv step (eight heads per CTA at 64 rows; one head per CTA in clusters of 8
at one row, where rank 0 writes the group's B and C windows back), followed
by the block checks of the output, the states and the conv windows."""
import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import (assert_block_out, assert_out_is_gemm, assert_state, bf16_dev, device_weights, f32_dev,
                     gpu_out_proj, to_np)

pytestmark = pytest.mark.gpu

m2 = pytest.importorskip("mamba2_ssm_mixer_gb300")


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.init()


@pytest.fixture(scope="module")
def biased():
    """Weights with a conv bias and integer in_proj codes in [-2, 2] (s_w1 = 1)."""
    Wt = dict(synth.make_weights(0))
    rng = np.random.default_rng(11)
    lut = oracle.e4m3_encode(np.arange(-2, 3, dtype=np.float64))
    Wt["in_proj"] = lut[rng.integers(-2, 3, (10304, 2688)) + 2]
    Wt["s_w1"] = 1.0
    Wt["conv_b"] = synth.as_bf16_values(rng.standard_normal(6144) * 0.5)
    blk = m2.Mamba2Mixer(device_weights(Wt))
    yield Wt, blk
    blk.close()


def _hidden(seed, T, Wt):
    """Hidden rows whose static e4m3 codes are the integers -3..3."""
    return np.random.default_rng(seed).integers(-3, 4, (T, 2688)).astype(np.float32) * np.float32(Wt["s_x"])


def _assert_u(u, ref):
    """u within one bf16 step of the oracle's (the f32 sum before the
    rounding may differ from the float64 one in its last bit)."""
    err = np.abs(u.astype(np.float64) - ref)
    assert np.all(err <= np.abs(ref) * 2.0 ** -7 + 1e-6), float(err.max())


@pytest.mark.parametrize("lens,has", [([5, 2, 40, 300], [1, 0, 1, 1]),   # chunked SSD path (300 > 64)
                                      ([5, 2, 40], [1, 0, 1])])          # token by token
def test_prefill_conv_bias(biased, lens, has):
    Wt, blk = biased
    T = sum(lens)
    h = _hidden(31, T, Wt)
    conv0 = synth.make_conv_state(31, len(lens))
    ssm0 = synth.make_ssm_state(31, len(lens))
    conv, ssm = bf16_dev(conv0), f32_dev(ssm0)
    taps = dict(u=torch.empty((T, 6144), dtype=torch.bfloat16, device="cuda"),
                zx=torch.empty((T, 10304), dtype=torch.bfloat16, device="cuda"),
                q2=torch.empty((T, 4096), dtype=torch.uint8, device="cuda"))
    blk.set_taps(**taps)
    out = blk.prefill(bf16_dev(h), lens, conv, ssm, has_initial=has)
    blk.set_taps()
    torch.cuda.synchronize()
    blk.check()
    mask = np.array(has, np.float64)
    ref = oracle.block_prefill(Wt, h, lens, conv0 * mask[:, None, None], ssm0 * mask[:, None, None, None], keep=True)
    assert np.array_equal(to_np(taps["zx"]), ref["zx"])
    _assert_u(to_np(taps["u"]), ref["u"])
    q2 = to_np(taps["q2"])
    assert_out_is_gemm(to_np(out), q2, gpu_out_proj(Wt))
    assert_block_out(to_np(out), ref["out"], q2=q2, ref_q2=ref["q2"], Wt=Wt)
    assert_state(to_np(ssm), ref["ssm_state"])
    assert np.array_equal(to_np(conv), ref["conv_state"])   # raw inputs: exact


@pytest.mark.parametrize("Bt,n_slots", [(64, 96), (1, 4)])
def test_decode_conv_bias(biased, Bt, n_slots):
    Wt, blk = biased
    conv0 = synth.make_conv_state(32, n_slots)
    ssm0 = synth.make_ssm_state(32, n_slots)
    slots = synth.make_slot_idx(32, n_slots, Bt)
    h = _hidden(32, Bt, Wt)
    conv, ssm = bf16_dev(conv0), f32_dev(ssm0)
    taps = dict(u=torch.empty((Bt, 6144), dtype=torch.bfloat16, device="cuda"),
                q2=torch.empty((Bt, 4096), dtype=torch.uint8, device="cuda"))
    blk.set_taps(**taps)
    out = blk.decode(bf16_dev(h), conv, ssm, torch.from_numpy(slots).cuda())
    blk.set_taps()
    torch.cuda.synchronize()
    blk.check()
    ref = oracle.block_decode(Wt, h, conv0, ssm0, slots, keep=True)
    _assert_u(to_np(taps["u"]), ref["u"])
    q2 = to_np(taps["q2"])
    assert_out_is_gemm(to_np(out), q2, gpu_out_proj(Wt))
    assert_block_out(to_np(out), ref["out"], q2=q2, ref_q2=ref["q2"], Wt=Wt)
    assert_state(to_np(ssm)[slots], ref["ssm_rows"])
    conv_np = to_np(conv)
    assert np.array_equal(conv_np[slots], ref["conv_rows"])   # shifted raw inputs: exact
    untouched = np.setdiff1d(np.arange(n_slots), slots)
    assert np.array_equal(conv_np[untouched], conv0[untouched])
