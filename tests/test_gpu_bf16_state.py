"""A bf16 SSM state cache (the handle's ssm_dtype = M2_DTYPE_BF16): rows are
widened to f32 when read, advanced and reduced to y in f32, and rounded to
bf16 when written back (decode) or returned (prefill).  Compared with the
oracle's state_cache="bf16" path; the state bound is the f32 one, the rows
being bf16 on both sides (a row may differ in its last bit where the f32 and
f64 values round differently)."""
import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import assert_block_out, assert_out_is_gemm, assert_state, bf16_dev, device_weights, gpu_out_proj, q2_tap, to_np

pytestmark = pytest.mark.gpu

m2 = pytest.importorskip("mamba2_ssm_mixer_gb300")


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.init()


@pytest.fixture(scope="module")
def block_bf16():
    Wt = synth.make_weights(0)
    return Wt, m2.Mamba2Mixer(device_weights(Wt), ssm_dtype=m2.M2_DTYPE_BF16)


def _bf16_np(t):
    return t.to(torch.float32).cpu().numpy()


def test_paged_decode_bf16_pool_batch64(block_bf16):
    Wt, blk = block_bf16
    n_slots, Bt = 256, 64
    conv0 = synth.make_conv_state(2, n_slots)
    ssm0 = synth.as_bf16_values(synth.make_ssm_state(2, n_slots))
    slots = synth.make_slot_idx(2, n_slots, Bt)
    h = synth.make_hidden(2, Bt)
    conv, ssm = bf16_dev(conv0), bf16_dev(ssm0)
    with q2_tap(blk, Bt) as q2:
        out = blk.decode(bf16_dev(h), conv, ssm, torch.from_numpy(slots).cuda())
    torch.cuda.synchronize()
    blk.check()
    ref = oracle.block_decode(Wt, h, conv0, ssm0, slots, state_cache="bf16", keep=True)
    assert_out_is_gemm(to_np(out), to_np(q2), gpu_out_proj(Wt))
    assert_block_out(to_np(out), ref["out"], q2=to_np(q2), ref_q2=ref["q2"], Wt=Wt)
    ssm_np = _bf16_np(ssm)
    assert_state(ssm_np[slots], ref["ssm_rows"])
    assert np.mean(ssm_np[slots] != ref["ssm_rows"]) < 1e-2      # mostly the same bf16 value
    untouched = np.setdiff1d(np.arange(n_slots), slots)
    assert np.array_equal(ssm_np[untouched], ssm0[untouched])     # byte-identical
    assert np.array_equal(_bf16_np(conv)[slots][:, :, :2], conv0[slots][:, :, 1:])


def test_varlen_prefill_bf16_state(block_bf16):
    Wt, blk = block_bf16
    lens = [37, 300, 1, 256]
    T = sum(lens)
    h = synth.make_hidden(5, T)
    conv0 = synth.make_conv_state(5, len(lens))
    ssm0 = synth.as_bf16_values(synth.make_ssm_state(5, len(lens)))
    has = [1, 0, 1, 1]
    conv, ssm = bf16_dev(conv0), bf16_dev(ssm0)
    with q2_tap(blk, T) as q2:
        out = blk.prefill(bf16_dev(h), lens, conv, ssm, has_initial=has)
    torch.cuda.synchronize()
    blk.check()
    mask = np.array(has, np.float64)
    ref = oracle.block_prefill(Wt, h, lens, conv0 * mask[:, None, None], ssm0 * mask[:, None, None, None],
                               state_cache="bf16", keep=True)
    assert_out_is_gemm(to_np(out), to_np(q2), gpu_out_proj(Wt))
    assert_block_out(to_np(out), ref["out"], q2=to_np(q2), ref_q2=ref["q2"], Wt=Wt)
    assert_state(_bf16_np(ssm), ref["ssm_state"])


def test_decode_after_prefill_carry_bf16_state(block_bf16):
    Wt, blk = block_bf16
    T, t0 = 40, 33
    h = synth.make_hidden(6, T)
    conv = torch.zeros((1, 6144, 3), dtype=torch.bfloat16, device="cuda")
    ssm = torch.zeros((1, 64, 64, 128), dtype=torch.bfloat16, device="cuda")
    with q2_tap(blk, t0) as q2:
        outs = [to_np(blk.prefill(bf16_dev(h[:t0]), [t0], conv, ssm))]
    q2s = [to_np(q2)]
    slot = torch.zeros(1, dtype=torch.int32, device="cuda")
    for t in range(t0, T):
        with q2_tap(blk, 1) as q2:
            outs.append(to_np(blk.decode(bf16_dev(h[t:t + 1]), conv, ssm, slot)))
        q2s.append(to_np(q2))
    torch.cuda.synchronize()
    blk.check()
    r = oracle.block_prefill(Wt, h[:t0], [t0], state_cache="bf16", keep=True)
    rc, rs, ro, rq = r["conv_state"], r["ssm_state"], [r["out"]], [r["q2"]]
    for t in range(t0, T):
        d = oracle.block_decode(Wt, h[t:t + 1], rc, rs, np.array([0]), state_cache="bf16", keep=True)
        rc, rs = d["conv_rows"], d["ssm_rows"]
        ro.append(d["out"])
        rq.append(d["q2"])
    gemm = gpu_out_proj(Wt)
    for o_, q_ in zip(outs, q2s):
        assert_out_is_gemm(o_, q_, gemm)
    assert_block_out(np.concatenate(outs), np.concatenate(ro), q2=np.concatenate(q2s), ref_q2=np.concatenate(rq),
                     Wt=Wt)
    assert_state(_bf16_np(ssm)[0], rs[0])
