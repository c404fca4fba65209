"""m2_mixed: decode rows and prefill sequences in one call (one input quant,
one in_proj and one out_proj over all rows).  Checked against the oracle on a
small batch, against the separate m2_decode / m2_prefill calls at the bench
shape, and bit-exactly against them when only one kind of row is present."""
import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import (assert_bf16_close, assert_block_out, assert_e4m3_close, assert_state, bf16_dev, device_weights,
                     assert_out_is_gemm, f32_dev, gpu_out_proj, q2_tap, rel_l2, to_np)

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


def test_mixed_small_batch_vs_oracle(block0):
    Wt, blk = block0
    n_slots, Bt, lens = 24, 8, [37, 300]
    conv_pool0 = synth.make_conv_state(2, n_slots)
    ssm_pool0 = synth.make_ssm_state(2, n_slots)
    slots = synth.make_slot_idx(2, n_slots, Bt)
    conv_st0 = synth.make_conv_state(5, len(lens))
    ssm_st0 = synth.make_ssm_state(5, len(lens))
    h = np.concatenate([synth.make_hidden(2, Bt), synth.make_hidden(5, sum(lens))])
    cp, sp = bf16_dev(conv_pool0), f32_dev(ssm_pool0)
    cs, ss = bf16_dev(conv_st0), f32_dev(ssm_st0)
    R = Bt + sum(lens)
    q2t = torch.zeros((R, 4096), dtype=torch.uint8, device="cuda")
    o_t = torch.zeros((R, 4096), dtype=torch.bfloat16, device="cuda")
    y_t = torch.zeros((R, 4096), dtype=torch.bfloat16, device="cuda")
    blk.set_taps(q2=q2t, o=o_t, y=y_t)
    out = blk.mixed(bf16_dev(h), Bt, cp, sp, torch.from_numpy(slots).cuda(), lens, cs, ss, has_initial=[1, 0])
    blk.set_taps()
    torch.cuda.synchronize()
    blk.check()
    rd = oracle.block_decode(Wt, h[:Bt], conv_pool0, ssm_pool0, slots, keep=True)
    mask = np.array([1.0, 0.0])
    rp = oracle.block_prefill(Wt, h[Bt:], lens, conv_st0 * mask[:, None, None], ssm_st0 * mask[:, None, None, None],
                              keep=True)
    o, q2 = to_np(out), to_np(q2t)
    assert rel_l2(to_np(y_t), np.concatenate([rd["y"], rp["y"]])) < 1e-3
    assert_e4m3_close(q2, np.concatenate([rd["q2"], rp["q2"]]), to_np(o_t), np.concatenate([rd["o"], rp["o"]]),
                      Wt["s_y"])
    assert_out_is_gemm(o, q2, gpu_out_proj(Wt))
    assert_block_out(o[:Bt], rd["out"], q2=q2[:Bt], ref_q2=rd["q2"], Wt=Wt)
    assert_block_out(o[Bt:], rp["out"], q2=q2[Bt:], ref_q2=rp["q2"], Wt=Wt)
    assert_state(to_np(sp)[slots], rd["ssm_rows"])
    assert_state(to_np(ss), rp["ssm_state"])
    untouched = np.setdiff1d(np.arange(n_slots), slots)
    assert np.array_equal(to_np(sp)[untouched], ssm_pool0[untouched])


def test_mixed_bench_shape_vs_separate_calls(block0):
    Wt, blk = block0
    n_slots, Bt, lens = 256, 64, [2048] * 4
    conv_pool0 = bf16_dev(synth.make_conv_state(2, n_slots))
    ssm_pool0 = f32_dev(synth.make_ssm_state(2, n_slots))
    slots = torch.from_numpy(synth.make_slot_idx(2, n_slots, Bt)).cuda()
    hd = bf16_dev(synth.make_hidden(2, Bt))
    hp = synth.device_normal((sum(lens), 2688), 3, 0, synth.T_HIDDEN, 1.0, torch.bfloat16, "cuda")
    zc = lambda: torch.zeros((4, 6144, 3), dtype=torch.bfloat16, device="cuda")
    zs = lambda: torch.zeros((4, 64, 64, 128), dtype=torch.float32, device="cuda")
    cp1, sp1, cs1, ss1 = conv_pool0.clone(), ssm_pool0.clone(), zc(), zs()
    cp2, sp2, cs2, ss2 = conv_pool0.clone(), ssm_pool0.clone(), zc(), zs()
    with q2_tap(blk, Bt) as qd:
        od = blk.decode(hd, cp1, sp1, slots)
    with q2_tap(blk, sum(lens)) as qp:
        op = blk.prefill(hp, lens, cs1, ss1)
    with q2_tap(blk, Bt + sum(lens)) as qm:
        om = blk.mixed(torch.cat([hd, hp]), Bt, cp2, sp2, slots, lens, cs2, ss2)
    torch.cuda.synchronize()
    blk.check()
    qm = to_np(qm)
    gemm = gpu_out_proj(Wt)
    assert_out_is_gemm(to_np(om), qm, gemm, what="mixed")
    assert_out_is_gemm(to_np(od), to_np(qd), gemm, what="decode")
    assert_out_is_gemm(to_np(op), to_np(qp), gemm, what="prefill")
    assert_block_out(to_np(om[:Bt]), to_np(od), q2=qm[:Bt], ref_q2=to_np(qd), Wt=Wt, what="mixed vs decode")
    assert_block_out(to_np(om[Bt:]), to_np(op), q2=qm[Bt:], ref_q2=to_np(qp), Wt=Wt, what="mixed vs prefill")
    rows = slots.cpu().numpy()
    assert_state(to_np(sp2)[rows], to_np(sp1)[rows])
    assert_state(to_np(ss2), to_np(ss1))
    # the decode rows' zx comes from the big GEMM here and from the split-K
    # GEMM in m2_decode (different summation order), so the raw xBC taps the
    # conv windows carry may differ in their last bit
    assert_bf16_close(to_np(cp2)[rows], to_np(cp1)[rows], atol=1e-3, what="decode conv rows")
    assert_bf16_close(to_np(cs2), to_np(cs1), atol=1e-3, what="prefill conv state")


def test_mixed_with_one_kind_equals_the_plain_call(block0):
    Wt, blk = block0
    lens = [37, 300]
    hp = bf16_dev(synth.make_hidden(5, sum(lens)))
    c1, s1 = torch.zeros((2, 6144, 3), dtype=torch.bfloat16, device="cuda"), torch.zeros(
        (2, 64, 64, 128), dtype=torch.float32, device="cuda")
    c2, s2 = c1.clone(), s1.clone()
    a = blk.prefill(hp, lens, c1, s1)
    b = blk.mixed(hp, 0, None, None, None, lens, c2, s2)
    n_slots, Bt = 16, 5
    cp0, sp0 = bf16_dev(synth.make_conv_state(2, n_slots)), f32_dev(synth.make_ssm_state(2, n_slots))
    slots = torch.from_numpy(synth.make_slot_idx(2, n_slots, Bt)).cuda()
    hd = bf16_dev(synth.make_hidden(2, Bt))
    cp1, sp1, cp2, sp2 = cp0.clone(), sp0.clone(), cp0.clone(), sp0.clone()
    d1 = blk.decode(hd, cp1, sp1, slots)
    d2 = blk.mixed(hd, Bt, cp2, sp2, slots, [], None, None)
    torch.cuda.synchronize()
    blk.check()
    assert torch.equal(a, b) and torch.equal(c1, c2) and torch.equal(s1, s2)
    assert torch.equal(d1, d2) and torch.equal(cp1, cp2) and torch.equal(sp1, sp2)
