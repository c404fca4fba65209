"""Failure detection and the slot / residency contracts, on the GPU through
the C ABI.

- A bounded device wait that runs out is reported, and the context stays
  usable: the self-test kernel waits on a barrier nothing completes, gives up
  after a millisecond and takes the kernels' abort path; the error word then
  reads M2_ETIMEOUT once, and the next calls compute correct results.  Both
  error words are covered: a handle's (m2_check) and the standalone entry
  points' (m2_check_standalone).
- Slot ids are unique within a decode call: a repeated id is skipped on the
  device (output zeroed, the slot advanced once, by the first row naming it)
  and reported as M2_EINVAL (the pages' reading: two rows advancing one slot
  would race).
- Residency: the handle uploads the block's weights once, at creation, and a
  prefill or decode call uploads nothing (vllm.cpp PR #1288, "Three points
  where this differs from the spec, deliberately", point 2: X bytes on the
  first call, 0 on the second).
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import (assert_block_out, assert_out_is_gemm, assert_state, bf16_dev, device_weights, f32_dev,
                     gpu_out_proj, q2_tap, to_np, u8_dev)

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


def _decode(blk, Wt, cfg, slots, n_slots):
    conv0 = synth.make_conv_state(cfg, n_slots)
    ssm0 = synth.make_ssm_state(cfg, n_slots)
    h = synth.make_hidden(cfg, len(slots))
    conv, ssm = bf16_dev(conv0), f32_dev(ssm0)
    with q2_tap(blk, len(slots)) as q2:
        out = blk.decode(bf16_dev(h), conv, ssm, torch.tensor(slots, dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    return h, conv0, ssm0, conv, ssm, out, to_np(q2)


def test_bounded_wait_runs_out_and_the_context_stays_usable(block0):
    Wt, blk = block0
    blk.check()                                      # clean to begin with
    blk.selftest_timeout(1000)                       # 1 ms
    torch.cuda.synchronize()
    with pytest.raises(m2.M2Error) as e:
        blk.check()
    assert e.value.status == m2.M2_ETIMEOUT
    blk.check()                                      # read once, then cleared
    # the next calls work and are right
    h, conv0, ssm0, conv, ssm, out, q2 = _decode(blk, Wt, 1, [0], 1)
    blk.check()
    ref = oracle.block_decode(Wt, h, conv0, ssm0, np.array([0]), keep=True)
    assert_out_is_gemm(to_np(out), q2, gpu_out_proj(Wt))
    assert_block_out(to_np(out), ref["out"], q2=q2, ref_q2=ref["q2"], Wt=Wt)
    assert_state(ssm.cpu().numpy()[0], ref["ssm_rows"][0])


def test_standalone_error_word_reports_a_timeout_then_clears():
    m2.check_standalone()
    m2.selftest_timeout_standalone(1000)
    torch.cuda.synchronize()
    with pytest.raises(m2.M2Error) as e:
        m2.check_standalone()
    assert e.value.status == m2.M2_ETIMEOUT
    m2.check_standalone()
    # a standalone GEMM afterwards: correct, and its error word stays clean
    rng = np.random.default_rng(3)
    a = oracle.e4m3_encode(rng.integers(-8, 9, (8, 2688)).astype(np.float64))
    w = oracle.e4m3_encode(rng.integers(-8, 9, (300, 2688)).astype(np.float64))
    y = to_np(m2.fp8_linear(u8_dev(a), 1.0, u8_dev(w), 1.0))
    m2.check_standalone()
    assert np.array_equal(y, oracle.fp8_linear(a, 1.0, w, 1.0))


def test_selftest_refuses_limits_out_of_range(block0):
    _, blk = block0
    for lim in (0, 100001):
        assert m2._lib.m2_selftest_timeout(blk.handle, lim, None) == m2.M2_EINVAL
    assert "limit_us" in m2.last_error()


def test_duplicate_slot_ids_are_detected_and_skipped(block0):
    Wt, blk = block0
    n_slots = 8
    slots = [3, 5, 3, 1, 5]
    h, conv0, ssm0, conv, ssm, out, q2 = _decode(blk, Wt, 4, slots, n_slots)
    with pytest.raises(m2.M2Error) as e:
        blk.check()
    assert e.value.status == m2.M2_EINVAL and "same slot" in str(e.value)
    blk.check()
    # the first row naming a slot advances it; the repeats are padding rows
    eff = np.array([3, 5, -1, 1, -1])
    ref = oracle.block_decode(Wt, h, conv0, ssm0, eff, keep=True)
    o = to_np(out)
    assert np.all(o[[2, 4]] == 0) and np.all(q2[[2, 4]] == 0)
    live = ref["live"]
    assert_out_is_gemm(o, q2, gpu_out_proj(Wt))
    assert_block_out(o[live], ref["out"][live], q2=q2[live], ref_q2=ref["q2"], Wt=Wt)
    ssm_np = ssm.cpu().numpy()
    assert_state(ssm_np[[3, 5, 1]], ref["ssm_rows"])
    untouched = [0, 2, 4, 6, 7]
    assert np.array_equal(ssm_np[untouched], ssm0[untouched])
    conv_np = conv.cpu().to(torch.float32).numpy()
    assert np.array_equal(conv_np[untouched], conv0[untouched])
    assert np.array_equal(conv_np[[3, 5, 1]][:, :, :2], conv0[[3, 5, 1]][:, :, 1:])   # shifted once


def test_mixed_call_detects_duplicate_slot_ids(block0):
    Wt, blk = block0
    n_slots = 6
    conv_pool = bf16_dev(synth.make_conv_state(5, n_slots))
    ssm_pool = f32_dev(synth.make_ssm_state(5, n_slots))
    h = bf16_dev(synth.make_hidden(5, 3 + 20))
    conv_st = torch.zeros((1, 6144, 3), dtype=torch.bfloat16, device="cuda")
    ssm_st = torch.zeros((1, 64, 64, 128), dtype=torch.float32, device="cuda")
    out = blk.mixed(h, 3, conv_pool, ssm_pool, torch.tensor([2, 2, 4], dtype=torch.int32, device="cuda"), [20],
                    conv_st, ssm_st)
    torch.cuda.synchronize()
    with pytest.raises(m2.M2Error) as e:
        blk.check()
    assert e.value.status == m2.M2_EINVAL
    assert torch.all(out[1] == 0) and not torch.all(out[0] == 0)


def test_upload_counter_first_call_then_none(block0):
    """m2_create uploads every weight byte once; prefill and decode upload
    nothing; a second handle counts its own upload (residency keyed on the
    owning handle, PR #1288 "Three points", points 1 and 2)."""
    Wt, _ = block0
    expect = (Wt["in_proj"].nbytes + Wt["out_proj"].nbytes + Wt["conv_w"].size * 2 + Wt["A_log"].size * 4
              + Wt["D"].size * 4 + Wt["dt_bias"].size * 4 + Wt["norm_w"].size * 2)
    blk = m2.Mamba2Mixer(device_weights(Wt))
    try:
        assert blk.stats()["bytes_uploaded"] == expect == 38765312
        h = synth.make_hidden(6, 9)
        conv = torch.zeros((1, 6144, 3), dtype=torch.bfloat16, device="cuda")
        ssm = torch.zeros((1, 64, 64, 128), dtype=torch.float32, device="cuda")
        blk.prefill(bf16_dev(h[:8]), [8], conv, ssm)
        blk.decode(bf16_dev(h[8:]), conv, ssm, torch.zeros(1, dtype=torch.int32, device="cuda"))
        torch.cuda.synchronize()
        blk.check()
        st = blk.stats()
        assert st["bytes_uploaded"] == expect                    # 0 bytes on the later calls
        assert st["prefill_calls"] == 1 and st["decode_calls"] == 1
        blk2 = m2.Mamba2Mixer(device_weights(Wt))
        assert blk2.stats()["bytes_uploaded"] == expect
        blk2.close()
    finally:
        blk.close()
