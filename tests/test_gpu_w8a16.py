"""The W8A16 arm (m2_config.arm = M2_ARM_W8A16): the host reference arm of
PR #1288, section "The comparison is not bit-comparable, and that is the
point" -- input_scale carried and not applied, so both projections take their
bf16 activations against weights dequantised to bf16.  Compared with the
oracle's arm="w8a16" path; the two arms' separation is measured against the
parity noise floor in the same run, as the pages do for their carry gate."""
import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import (assert_bf16_close, assert_block_out, assert_out_is_gemm, assert_state, bf16_dev, device_weights,
                     f32_dev, gpu_out_proj, rel_l2, to_np, u8_dev)

pytestmark = pytest.mark.gpu

m2 = pytest.importorskip("mamba2_ssm_mixer_gb300")


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.init()


@pytest.fixture(scope="module")
def block_w8a16():
    Wt = synth.make_weights(0)
    return Wt, m2.Mamba2Mixer(device_weights(Wt), arm=m2.M2_ARM_W8A16)


def _bf16_bits(t):
    return t.view(torch.int16).cpu().numpy().astype(np.uint16)


def _oracle_bits(v):
    return torch.from_numpy(np.asarray(v, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().astype(np.uint16)


@pytest.mark.parametrize("scale", [1.0, 2.0 ** -7, 0.0123 / 448, 1.7e-4, 3.3])
def test_fp8_dequant_all_codes_bit_exact(scale):
    """Every code, at n not a multiple of 8 (vector body and scalar tail)."""
    codes = np.tile(np.arange(256, dtype=np.uint8), 41)[:10247]
    got = to_np(m2.fp8_dequant(u8_dev(codes), scale))
    ref = oracle.dequant_e4m3_bf16(codes, scale)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_fp8_dequant_in_proj_weights_bit_exact():
    Wt = synth.make_weights(0)
    got = m2.fp8_dequant(u8_dev(Wt["in_proj"]), Wt["s_w1"])
    torch.cuda.synchronize()
    ref = oracle.dequant_e4m3_bf16(Wt["in_proj"], Wt["s_w1"])
    assert np.array_equal(_bf16_bits(got), _oracle_bits(ref))


@pytest.mark.parametrize("M,N,K", [(1, 10304, 2688), (64, 10304, 2688), (37, 2688, 4096), (300, 200, 160),
                                   (257, 300, 2688), (300, 203, 160), (513, 10304, 2688), (594, 10304, 2688),
                                   (600, 2688, 4096)])
def test_bf16_linear_integer_exact(M, N, K):
    """Integer-valued bf16 operands: every partial sum is an exact integer below
    2^24, so the bf16 result is bit-exact in any summation order.  Covers the
    few-row and split-K kernels (M <= 256), the CTA-pair kernel with TMA
    stores and with per-thread stores (N = 203), and ragged M, N and K."""
    rng = np.random.default_rng(M * 13 + N)
    x = rng.integers(-8, 9, (M, K)).astype(np.float64)
    w = rng.integers(-8, 9, (N, K)).astype(np.float64)
    y = to_np(m2.bf16_linear(bf16_dev(x), bf16_dev(w)))
    assert np.array_equal(y, oracle.bf16_linear(x, w))


@pytest.mark.parametrize("M", [8, 300])
def test_bf16_linear_random_vs_oracle(M):
    Wt = synth.make_weights(0)
    rng = np.random.default_rng(M)
    h = synth.as_bf16_values(rng.standard_normal((M, 2688)))
    wd = oracle.dequant_e4m3_bf16(Wt["in_proj"], Wt["s_w1"])
    y = to_np(m2.bf16_linear(bf16_dev(h), bf16_dev(wd)))
    ref = oracle.bf16_linear(h, wd)
    atol = 2.0 ** -16 * (np.abs(h) @ np.abs(wd).T)       # f32 accumulation bound, as for the e4m3 GEMM
    assert_bf16_close(y, ref, atol=atol, what="bf16_linear")


def test_w8a16_prefill_varlen_and_separation(block_w8a16):
    Wt, blk = block_w8a16
    lens = [37, 300, 1, 256]
    T = sum(lens)
    h = synth.make_hidden(5, T)
    conv0 = synth.make_conv_state(5, len(lens))
    ssm0 = synth.make_ssm_state(5, len(lens))
    has = [1, 0, 1, 1]
    conv, ssm = bf16_dev(conv0), f32_dev(ssm0)
    taps = dict(zx=torch.empty((T, 10304), dtype=torch.bfloat16, device="cuda"),
                o=torch.empty((T, 4096), dtype=torch.bfloat16, device="cuda"))
    blk.set_taps(**taps)
    out = blk.prefill(bf16_dev(h), lens, conv, ssm, has_initial=has)
    blk.set_taps()
    torch.cuda.synchronize()
    blk.check()
    mask = np.array(has, np.float64)
    c0, s0 = conv0 * mask[:, None, None], ssm0 * mask[:, None, None, None]
    ref = oracle.block_prefill(Wt, h, lens, c0, s0, keep=True, arm="w8a16")
    wd = oracle.dequant_e4m3_bf16(Wt["in_proj"], Wt["s_w1"])
    assert_bf16_close(to_np(taps["zx"]), ref["zx"], atol=2.0 ** -16 * (np.abs(h) @ np.abs(wd).T), what="zx")
    assert rel_l2(to_np(taps["o"]), ref["o"]) < 1e-2
    got = to_np(out)
    assert_out_is_gemm(got, to_np(taps["o"]), gpu_out_proj(Wt, "w8a16"))
    _, floor = assert_block_out(got, ref["out"], o=to_np(taps["o"]), ref_o=ref["o"], Wt=Wt)
    assert_state(to_np(ssm), ref["ssm_state"])
    assert_bf16_close(to_np(conv), ref["conv_state"], atol=1e-3, what="conv_state")
    # the W8A8 arm on the same inputs differs by the e4m3 activation quant:
    # measured here against this run's noise floor, and required to exceed
    # twice that floor (the arms are not bit-comparable by construction)
    sep = rel_l2(got, oracle.block_prefill(Wt, h, lens, c0, s0, arm="w8a8")["out"])
    print(f"W8A16 device vs W8A16 oracle (noise floor) {floor:.3e}; vs W8A8 oracle (separation) {sep:.3e}")
    assert sep > 2 * floor


def test_w8a16_paged_decode_with_padding_row(block_w8a16):
    Wt, blk = block_w8a16
    n_slots = 16
    conv0 = synth.make_conv_state(3, n_slots)
    ssm0 = synth.make_ssm_state(3, n_slots)
    slots = np.array([4, 11, -1, 0, 7, 15], np.int32)
    h = synth.make_hidden(3, len(slots))
    conv, ssm = bf16_dev(conv0), f32_dev(ssm0)
    o_tap = torch.zeros((len(slots), 4096), dtype=torch.bfloat16, device="cuda")
    blk.set_taps(o=o_tap)
    out = blk.decode(bf16_dev(h), conv, ssm, torch.from_numpy(slots).cuda())
    blk.set_taps()
    torch.cuda.synchronize()
    blk.check()
    ref = oracle.block_decode(Wt, h, conv0, ssm0, slots, arm="w8a16", keep=True)
    got = to_np(out)
    assert np.all(got[2] == 0)                                  # padding row: output zero
    lv = ref["live"]
    assert_out_is_gemm(got, to_np(o_tap), gpu_out_proj(Wt, "w8a16"))
    assert_block_out(got[lv], ref["out"][lv], o=to_np(o_tap)[lv], ref_o=ref["o"], Wt=Wt)
    live = slots[slots >= 0]
    ssm_np, conv_np = to_np(ssm), to_np(conv)
    assert_state(ssm_np[live], ref["ssm_rows"])
    untouched = np.setdiff1d(np.arange(n_slots), live)
    assert np.array_equal(ssm_np[untouched], ssm0[untouched])
    assert np.array_equal(conv_np[untouched], conv0[untouched])
    assert np.array_equal(conv_np[live][:, :, :2], conv0[live][:, :, 1:])


def test_w8a16_refuses_prequantised_and_mixed_calls(block_w8a16):
    _, blk = block_w8a16
    q = torch.zeros((4, 2688), dtype=torch.uint8, device="cuda")
    conv = torch.zeros((1, 6144, 3), dtype=torch.bfloat16, device="cuda")
    ssm = torch.zeros((1, 64, 64, 128), dtype=torch.float32, device="cuda")
    with pytest.raises(m2.M2Error) as e:
        blk.prefill(q, [4], conv, ssm)
    assert e.value.status == m2.M2_EINVAL and "W8A16" in str(e.value)
    with pytest.raises(m2.M2Error) as e:
        blk.decode(q[:1], conv, ssm, torch.zeros(1, dtype=torch.int32, device="cuda"))
    assert e.value.status == m2.M2_EINVAL and "W8A16" in str(e.value)
    with pytest.raises(m2.M2Error) as e:
        blk.mixed_workspace_size(1, [4])
    assert e.value.status == m2.M2_EINVAL and "W8A16" in str(e.value)


def test_w8a16_with_bf16_state_cache_carry():
    """The two options together: the W8A16 arm over a bf16 state cache, prefill
    then one-token decodes from the returned states (the carry case)."""
    Wt = synth.make_weights(0)
    blk = m2.Mamba2Mixer(device_weights(Wt), arm=m2.M2_ARM_W8A16, ssm_dtype=m2.M2_DTYPE_BF16)
    T, t0 = 40, 33
    h = synth.make_hidden(6, T)
    conv = torch.zeros((1, 6144, 3), dtype=torch.bfloat16, device="cuda")
    ssm = torch.zeros((1, 64, 64, 128), dtype=torch.bfloat16, device="cuda")
    o_tap = torch.zeros((T, 4096), dtype=torch.bfloat16, device="cuda")
    blk.set_taps(o=o_tap[:t0])
    outs = [to_np(blk.prefill(bf16_dev(h[:t0]), [t0], conv, ssm))]
    slot = torch.zeros(1, dtype=torch.int32, device="cuda")
    for t in range(t0, T):
        blk.set_taps(o=o_tap[t:t + 1])
        outs.append(to_np(blk.decode(bf16_dev(h[t:t + 1]), conv, ssm, slot)))
    blk.set_taps()
    torch.cuda.synchronize()
    blk.check()
    r = oracle.block_prefill(Wt, h[:t0], [t0], state_cache="bf16", arm="w8a16", keep=True)
    rc, rs, ro, rso = r["conv_state"], r["ssm_state"], [r["out"]], [r["o"]]
    for t in range(t0, T):
        d = oracle.block_decode(Wt, h[t:t + 1], rc, rs, np.array([0]), state_cache="bf16", arm="w8a16", keep=True)
        rc, rs = d["conv_rows"], d["ssm_rows"]
        ro.append(d["out"])
        rso.append(d["o"])
    gemm, ot = gpu_out_proj(Wt, "w8a16"), to_np(o_tap)
    assert_out_is_gemm(outs[0], ot[:t0], gemm)
    for i, o_ in enumerate(outs[1:]):
        assert_out_is_gemm(o_, ot[t0 + i:t0 + i + 1], gemm)
    assert_block_out(np.concatenate(outs), np.concatenate(ro), o=to_np(o_tap), ref_o=np.concatenate(rso), Wt=Wt)
    assert_state(ssm.to(torch.float32).cpu().numpy()[0], rs[0])
    blk.close()


def test_w8a16_short_prefill_takes_the_few_row_gemm(block_w8a16):
    """A prefill of at most 256 tokens runs both projections on the split-K
    few-row kernel (bf16 operands); checked at the block level with taps."""
    Wt, blk = block_w8a16
    lens = [100, 20]
    T = sum(lens)
    h = synth.make_hidden(8, T)
    conv = torch.zeros((2, 6144, 3), dtype=torch.bfloat16, device="cuda")
    ssm = torch.zeros((2, 64, 64, 128), dtype=torch.float32, device="cuda")
    taps = dict(zx=torch.empty((T, 10304), dtype=torch.bfloat16, device="cuda"),
                o=torch.empty((T, 4096), dtype=torch.bfloat16, device="cuda"))
    blk.set_taps(**taps)
    out = blk.prefill(bf16_dev(h), lens, conv, ssm)
    blk.set_taps()
    torch.cuda.synchronize()
    blk.check()
    ref = oracle.block_prefill(Wt, h, lens, keep=True, arm="w8a16")
    wd = oracle.dequant_e4m3_bf16(Wt["in_proj"], Wt["s_w1"])
    assert_bf16_close(to_np(taps["zx"]), ref["zx"], atol=2.0 ** -16 * (np.abs(h) @ np.abs(wd).T), what="zx")
    assert_out_is_gemm(to_np(out), to_np(taps["o"]), gpu_out_proj(Wt, "w8a16"))
    assert_block_out(to_np(out), ref["out"], o=to_np(taps["o"]), ref_o=ref["o"], Wt=Wt)
    assert_state(to_np(ssm), ref["ssm_state"])
