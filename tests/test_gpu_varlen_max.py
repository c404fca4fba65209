"""Prefill at the most sequences a call takes (256): every sequence's
has_initial bit (eight 32-bit words), chunk bookkeeping across 256
sequences, and both SSD paths (all sequences of at most 64 tokens take the
token-by-token kernel; one longer sequence sends the call down the chunked
path), against the oracle with the block checks."""
import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import (assert_bf16_close, assert_block_out, assert_e4m3_close, assert_out_is_gemm, assert_state,
                     bf16_dev, device_weights, f32_dev, gpu_out_proj, to_np)

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
    blk = m2.Mamba2Mixer(device_weights(Wt))
    yield Wt, blk
    blk.close()


@pytest.mark.parametrize("long_lens", [[], [70, 257, 300]], ids=["token-by-token", "chunked"])
def test_prefill_256_sequences(block0, long_lens):
    Wt, blk = block0
    rng = np.random.default_rng(41 + len(long_lens))
    lens = [int(v) for v in rng.integers(1, 25, 256 - len(long_lens))] + long_lens
    rng.shuffle(lens)
    has = [int(v) for v in rng.integers(0, 2, 256)]
    T = sum(lens)
    h = synth.make_hidden(41, T)
    conv0 = synth.make_conv_state(41, 256)
    ssm0 = synth.make_ssm_state(41, 256)
    conv, ssm = bf16_dev(conv0), f32_dev(ssm0)
    taps = dict(q2=torch.empty((T, 4096), dtype=torch.uint8, device="cuda"),
                o=torch.empty((T, 4096), dtype=torch.bfloat16, device="cuda"))
    blk.set_taps(**taps)
    out = blk.prefill(bf16_dev(h), lens, conv, ssm, has_initial=has)
    blk.set_taps()
    torch.cuda.synchronize()
    blk.check()
    mask = np.array(has, np.float64)
    ref = oracle.block_prefill(Wt, h, lens, conv0 * mask[:, None, None], ssm0 * mask[:, None, None, None], keep=True)
    q2, o = to_np(taps["q2"]), to_np(taps["o"])
    assert_e4m3_close(q2, ref["q2"], o, ref["o"], Wt["s_y"])
    assert_out_is_gemm(to_np(out), q2, gpu_out_proj(Wt))
    assert_block_out(to_np(out), ref["out"], q2=q2, ref_q2=ref["q2"], Wt=Wt)
    assert_state(to_np(ssm), ref["ssm_state"])
    assert_bf16_close(to_np(conv), ref["conv_state"], atol=1e-3, what="conv_state")
