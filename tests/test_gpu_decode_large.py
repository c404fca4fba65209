"""Paged decode of larger batches: 200 rows (the projections on the split-K
skinny GEMM with its reduce) and 300 rows (on the CTA-pair GEMM), from a
512-slot pool, so the state kernel's persistent CTAs walk several (row,
group) items each with their conv windows loaded one item ahead.  Against
the oracle with the block checks; slots no row names stay byte-identical."""
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


@pytest.mark.parametrize("Bt", [200, 300])
def test_paged_decode_large_batch(block0, Bt):
    Wt, blk = block0
    n_slots = 512
    conv0 = synth.make_conv_state(51, n_slots)
    ssm0 = synth.make_ssm_state(51, n_slots)
    slots = synth.make_slot_idx(51, n_slots, Bt)
    h = synth.make_hidden(51, Bt)
    conv, ssm = bf16_dev(conv0), f32_dev(ssm0)
    taps = dict(q2=torch.empty((Bt, 4096), dtype=torch.uint8, device="cuda"),
                o=torch.empty((Bt, 4096), dtype=torch.bfloat16, device="cuda"))
    blk.set_taps(**taps)
    out = blk.decode(bf16_dev(h), conv, ssm, torch.from_numpy(slots).cuda())
    blk.set_taps()
    torch.cuda.synchronize()
    blk.check()
    ref = oracle.block_decode(Wt, h, conv0, ssm0, slots, keep=True)
    q2, o = to_np(taps["q2"]), to_np(taps["o"])
    assert_e4m3_close(q2, ref["q2"], o, ref["o"], Wt["s_y"])
    assert_out_is_gemm(to_np(out), q2, gpu_out_proj(Wt))
    assert_block_out(to_np(out), ref["out"], q2=q2, ref_q2=ref["q2"], Wt=Wt)
    ssm_np, conv_np = to_np(ssm), to_np(conv)
    assert_state(ssm_np[slots], ref["ssm_rows"])
    untouched = np.setdiff1d(np.arange(n_slots), slots)
    assert np.array_equal(ssm_np[untouched], ssm0[untouched].astype(np.float64))
    assert np.array_equal(conv_np[untouched], conv0[untouched])
    assert np.array_equal(conv_np[slots][:, :, :2], conv0[slots][:, :, 1:])
    assert_bf16_close(conv_np[slots][:, :, 2], ref["conv_rows"][:, :, 2], atol=1e-3, what="conv tap")
