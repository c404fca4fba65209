"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Bit-exact: the e4m3 activation quant, the in_proj output and the conv
windows when every product and sum is exactly representable, the slot
gather/scatter (untouched slots byte-identical, shifted taps copied exactly).
Tolerance (floating point): block output max abs <= 2e-2 and relative L2 <=
1e-2; f32 SSM state relative L2 <= 1e-3.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import (assert_bf16_close, assert_block_out, assert_e4m3_close, assert_state, bf16_dev,
                     assert_out_is_gemm, device_weights, f32_dev, gemm_atol, gpu_out_proj, max_abs, q2_tap, rel_l2,
                     to_np, u8_dev)

pytestmark = pytest.mark.gpu

m2 = pytest.importorskip("mamba2_ssm_mixer_gb300")


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.init()


# ---------------------------------------------------------------- fp8 quant

@pytest.mark.parametrize("scale", [1.0 / 64.0, 1.0, 1.0 / 3.0, 1e-3])
def test_fp8_quant_bit_exact_all_bf16_patterns(scale):
    bits = (np.arange(65536, dtype=np.uint32) << 16).view(np.float32)
    x = torch.from_numpy(np.arange(65536, dtype=np.int32).astype(np.int16)).view(torch.bfloat16).cuda()
    q = to_np(m2.fp8_quant(x, scale))
    ref = oracle.quant_static_e4m3(bits, scale)
    nan = np.isnan(bits / np.float32(scale))
    assert np.array_equal(q[~nan], ref[~nan])
    assert np.all((q[nan] & 0x7F) == 0x7F)


@pytest.mark.parametrize("n", [1, 7, 8, 9, 4095, 1 << 20])
def test_fp8_quant_ragged_sizes_and_offsets(n):
    rng = np.random.default_rng(n)
    h = synth.as_bf16_values(rng.standard_normal(n + 3) * 4)
    x = bf16_dev(h)
    for off in (0, 1):
        xs = x[off:off + n]
        q = torch.full((n + 1,), 0xAB, dtype=torch.uint8, device="cuda")
        m2.fp8_quant(xs, 1 / 64, q[off:off + n] if off == 0 else q[1:1 + n])
        got = to_np(q)
        ref = oracle.quant_static_e4m3(h[off:off + n], 1 / 64)
        sl = slice(0, n) if off == 0 else slice(1, 1 + n)
        assert np.array_equal(got[sl], ref)
        assert got[n if off == 0 else 0] == 0xAB      # no write past the end


# ---------------------------------------------------------------- fp8 linear

def _int_codes(rng, shape, lo=-8, hi=8):
    """Random integers in [lo, hi] and their (exact) e4m3 codes."""
    ints = rng.integers(lo, hi + 1, shape)
    lut = oracle.e4m3_encode(np.arange(lo, hi + 1, dtype=np.float64))
    return ints, lut[ints - lo]


@pytest.mark.parametrize("M,N,K", [(1, 10304, 2688), (64, 10304, 2688), (37, 2688, 4096), (300, 200, 160),
                                   (128, 2688, 4096), (256, 2688, 4096), (5, 7, 2688), (257, 300, 2688),
                                   (300, 203, 160), (1000, 2688, 4096), (8192, 10304, 2688)])
def test_fp8_linear_integer_exact(M, N, K):
    """Integer-valued e4m3 operands: every partial sum is an exact integer
    below 2^24, so any summation order gives the same f32 value and the bf16
    result must be bit-exact.  Shapes cover the few-row cluster kernel
    (M <= 128), the split-K kernel (129-256), the CTA-pair kernel with TMA
    stores (N % 8 == 0) and with per-thread stores (N = 203), ragged M, N
    and K tails."""
    rng = np.random.default_rng(M * 7 + N)
    _, a = _int_codes(rng, (M, K))
    _, w = _int_codes(rng, (N, K))
    y = to_np(m2.fp8_linear(u8_dev(a), 1.0, u8_dev(w), 1.0))
    ref = oracle.fp8_linear(a, 1.0, w, 1.0)
    assert np.array_equal(y, ref)


def test_fp8_linear_partial_last_tile_repeated():
    """in_proj's width 10304 leaves one 64-column slice in the last 256-wide
    tile and M = 594 a partial last row tile: the epilogue's staged TMA
    stores must skip the empty slices without reusing a buffer a store still
    reads.  Five calls in a row, each bit-exact (integer-valued operands)."""
    M, N, K = 594, 10304, 2688
    rng = np.random.default_rng(594)
    _, a = _int_codes(rng, (M, K))
    _, w = _int_codes(rng, (N, K))
    ref = oracle.fp8_linear(a, 1.0, w, 1.0)
    ad, wd = u8_dev(a), u8_dev(w)
    for _ in range(5):
        y = to_np(m2.fp8_linear(ad, 1.0, wd, 1.0))
        assert np.array_equal(y, ref)


@pytest.mark.parametrize("M", [1, 8, 64, 200])
def test_fp8_linear_random_vs_oracle(M):
    Wt = synth.make_weights(0)
    rng = np.random.default_rng(M)
    h = synth.as_bf16_values(rng.standard_normal((M, 2688)))
    q = oracle.quant_static_e4m3(h, Wt["s_x"])
    y = to_np(m2.fp8_linear(u8_dev(q), Wt["s_x"], u8_dev(Wt["in_proj"]), Wt["s_w1"]))
    ref = oracle.fp8_linear(q, Wt["s_x"], Wt["in_proj"], Wt["s_w1"])
    assert_bf16_close(y, ref, atol=gemm_atol(q, Wt["in_proj"], Wt["s_x"] * Wt["s_w1"]), what="in_proj")
    y2 = to_np(m2.fp8_linear_bf16(bf16_dev(h), Wt["s_x"], u8_dev(Wt["in_proj"]), Wt["s_w1"]))
    assert np.array_equal(y, y2)


# ---------------------------------------------------------------- block

@pytest.fixture(scope="module")
def block0():
    Wt = synth.make_weights(0)
    return Wt, m2.Mamba2Mixer(device_weights(Wt))


def _taps(T):
    return dict(q=torch.empty((T, 2688), dtype=torch.uint8, device="cuda"),
                zx=torch.empty((T, 10304), dtype=torch.bfloat16, device="cuda"),
                u=torch.empty((T, 6144), dtype=torch.bfloat16, device="cuda"),
                dt=torch.empty((T, 64), dtype=torch.float32, device="cuda"),
                y=torch.empty((T, 4096), dtype=torch.bfloat16, device="cuda"),
                o=torch.empty((T, 4096), dtype=torch.bfloat16, device="cuda"),
                q2=torch.empty((T, 4096), dtype=torch.uint8, device="cuda"))


def _run_prefill(blk, h, seqlens, conv0=None, ssm0=None, has_initial=None, taps=False):
    nseq = len(seqlens)
    conv = bf16_dev(conv0) if conv0 is not None else torch.zeros((nseq, 6144, 3), dtype=torch.bfloat16, device="cuda")
    ssm = f32_dev(ssm0) if ssm0 is not None else torch.zeros((nseq, 64, 64, 128), dtype=torch.float32, device="cuda")
    tp = _taps(sum(seqlens)) if taps else None
    if tp:
        blk.set_taps(**tp)
    out = blk.prefill(bf16_dev(h), seqlens, conv, ssm, has_initial=has_initial)
    if tp:
        blk.set_taps()
    torch.cuda.synchronize()
    blk.check()
    return out, conv, ssm, tp


def test_config0_prefill_32_tokens_all_stages(block0):
    Wt, blk = block0
    h = synth.make_hidden(0, 32)
    out, conv, ssm, tp = _run_prefill(blk, h, [32], taps=True)
    ref = oracle.block_prefill(Wt, h, [32], keep=True)
    assert np.array_equal(to_np(tp["q"]), ref["q"])                       # bit-exact quant
    assert_bf16_close(to_np(tp["zx"]), ref["zx"], atol=gemm_atol(ref["q"], Wt["in_proj"], Wt["s_x"] * Wt["s_w1"]),
                      what="zx")
    assert rel_l2(to_np(tp["u"]), ref["u"]) < 1e-3
    assert rel_l2(to_np(tp["dt"]), ref["dt"]) < 1e-4
    assert rel_l2(to_np(tp["y"]), ref["y"]) < 1e-2
    assert rel_l2(to_np(tp["o"]), ref["o"]) < 1e-2
    assert_e4m3_close(to_np(tp["q2"]), ref["q2"], to_np(tp["o"]), ref["o"], Wt["s_y"])
    assert_out_is_gemm(to_np(out), to_np(tp["q2"]), gpu_out_proj(Wt))
    assert_block_out(to_np(out), ref["out"], q2=to_np(tp["q2"]), ref_q2=ref["q2"], Wt=Wt)
    assert_state(to_np(ssm), ref["ssm_state"])
    assert_bf16_close(to_np(conv), ref["conv_state"], atol=1e-3, what="conv_state")


def test_prefill_integer_exact_split_and_conv_state():
    """With integer-valued activations and weights every in_proj sum is exact,
    so zx (the z | xBC | dt row) and the conv windows built from it must be
    bit-exact; the conv output must sit at the right column (index identity)."""
    Wt = dict(synth.make_weights(0))
    rng = np.random.default_rng(5)
    _, Wt["in_proj"] = _int_codes(rng, (10304, 2688), -2, 2)
    Wt["s_w1"] = 1.0
    blk = m2.Mamba2Mixer(device_weights(Wt))
    lens = [5, 2, 40]
    hi = rng.integers(-3, 4, (sum(lens), 2688))
    h = hi.astype(np.float32) * np.float32(Wt["s_x"])
    conv0 = synth.make_conv_state(7, 3)
    out, conv, ssm, tp = _run_prefill(blk, h, lens, conv0=conv0, ssm0=np.zeros((3, 64, 64, 128), np.float32),
                                      has_initial=[1, 1, 0], taps=True)
    ref = oracle.block_prefill(Wt, h, lens, conv0.astype(np.float64) * np.array([1, 1, 0])[:, None, None],
                               np.zeros((3, 64, 64, 128)), keep=True)
    assert np.array_equal(to_np(tp["q"]), ref["q"])
    assert np.array_equal(to_np(tp["zx"]), ref["zx"])
    assert np.array_equal(to_np(conv), ref["conv_state"])
    assert_bf16_close(to_np(tp["u"]), ref["u"], atol=1e-5, what="u")
    assert_out_is_gemm(to_np(out), to_np(tp["q2"]), gpu_out_proj(Wt))
    assert_block_out(to_np(out), ref["out"], q2=to_np(tp["q2"]), ref_q2=ref["q2"], Wt=Wt)
    blk.close()


def test_config1_decode_batch1(block0):
    Wt, blk = block0
    conv0 = synth.make_conv_state(1, 1)
    ssm0 = synth.make_ssm_state(1, 1)
    h = synth.make_hidden(1, 1)
    conv, ssm = bf16_dev(conv0), f32_dev(ssm0)
    tp = _taps(1)
    blk.set_taps(**{k: v for k, v in tp.items()})
    out = blk.decode(bf16_dev(h), conv, ssm, torch.zeros(1, dtype=torch.int32, device="cuda"))
    blk.set_taps()
    torch.cuda.synchronize()
    blk.check()
    ref = oracle.block_decode(Wt, h, conv0, ssm0, np.array([0]), keep=True)
    assert np.array_equal(to_np(tp["q"]), ref["q"])
    assert_bf16_close(to_np(tp["zx"]), ref["zx"], atol=gemm_atol(ref["q"], Wt["in_proj"], Wt["s_x"] * Wt["s_w1"]),
                      what="zx")
    assert rel_l2(to_np(tp["u"]), ref["u"]) < 1e-3
    assert_e4m3_close(to_np(tp["q2"]), ref["q2"], to_np(tp["o"]), ref["o"], Wt["s_y"], max_frac=1e-3)
    assert_out_is_gemm(to_np(out), to_np(tp["q2"]), gpu_out_proj(Wt))
    assert_block_out(to_np(out), ref["out"], q2=to_np(tp["q2"]), ref_q2=ref["q2"], Wt=Wt)
    assert_state(to_np(ssm)[0], ref["ssm_rows"][0])
    c = to_np(conv)[0]
    assert np.array_equal(c[:, :2], conv0[0][:, 1:])                      # shifted taps: exact copies
    assert_bf16_close(c[:, 2], ref["conv_rows"][0][:, 2], atol=1e-3, what="conv tap")


def test_config2_paged_decode_batch64(block0):
    Wt, blk = block0
    n_slots, Bt = 256, 64
    conv0 = synth.make_conv_state(2, n_slots)
    ssm0 = synth.make_ssm_state(2, n_slots)
    slots = synth.make_slot_idx(2, n_slots, Bt)
    h = synth.make_hidden(2, Bt)
    conv, ssm = bf16_dev(conv0), f32_dev(ssm0)
    o_tap = torch.zeros((Bt, 4096), dtype=torch.bfloat16, device="cuda")
    q2 = torch.zeros((Bt, 4096), dtype=torch.uint8, device="cuda")
    blk.set_taps(q2=q2, o=o_tap)
    out = blk.decode(bf16_dev(h), conv, ssm, torch.from_numpy(slots).cuda())
    blk.set_taps()
    torch.cuda.synchronize()
    blk.check()
    ref = oracle.block_decode(Wt, h, conv0, ssm0, slots, keep=True)
    assert_e4m3_close(to_np(q2), ref["q2"], to_np(o_tap), ref["o"], Wt["s_y"])
    assert_out_is_gemm(to_np(out), to_np(q2), gpu_out_proj(Wt))
    assert_block_out(to_np(out), ref["out"], q2=to_np(q2), ref_q2=ref["q2"], Wt=Wt)
    ssm_np = ssm.cpu().numpy()
    conv_np = conv.cpu().to(torch.float32).numpy()
    assert_state(ssm_np[slots], ref["ssm_rows"])
    untouched = np.setdiff1d(np.arange(n_slots), slots)
    assert np.array_equal(ssm_np[untouched], ssm0[untouched])                 # byte-identical
    assert np.array_equal(conv_np[untouched], conv0[untouched])
    assert np.array_equal(conv_np[slots][:, :, :2], conv0[slots][:, :, 1:])
    assert_bf16_close(conv_np[slots][:, :, 2], ref["conv_rows"][:, :, 2], atol=1e-3, what="conv tap")
    st = blk.stats()
    assert st["state_update_rows"] >= Bt and st["decode_calls"] >= 1


def test_decode_padding_row_and_bad_slot_flag(block0):
    Wt, blk = block0
    n_slots = 4
    conv0 = synth.make_conv_state(3, n_slots)
    ssm0 = synth.make_ssm_state(3, n_slots)
    h = synth.make_hidden(3, 3)
    conv, ssm = bf16_dev(conv0), f32_dev(ssm0)
    with q2_tap(blk, 3) as q2:
        out = blk.decode(bf16_dev(h), conv, ssm, torch.tensor([2, -1, 0], dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    blk.check()
    ref = oracle.block_decode(Wt, h, conv0, ssm0, np.array([2, -1, 0]), keep=True)
    o = to_np(out)
    assert np.all(o[1] == 0) and np.all(to_np(q2)[1] == 0)
    live = ref["live"]
    assert_out_is_gemm(o, to_np(q2), gpu_out_proj(Wt))
    assert_block_out(o[live], ref["out"][live], q2=to_np(q2)[live], ref_q2=ref["q2"], Wt=Wt)
    assert np.array_equal(ssm.cpu().numpy()[[1, 3]], ssm0[[1, 3]])
    # an id outside the pool is skipped on the device and reported by m2_check
    before = ssm.clone()
    out = blk.decode(bf16_dev(h[:1]), conv, ssm, torch.tensor([7], dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    with pytest.raises(m2.M2Error) as e:
        blk.check()
    assert e.value.status == m2.M2_EINVAL
    assert torch.equal(before, ssm)
    assert torch.all(out == 0)
    blk.check()                                   # the error word was cleared


def test_varlen_prefill_ragged_with_initial_states(block0):
    Wt, blk = block0
    lens = [37, 300, 1, 256, 513, 2]
    rng_conv = synth.make_conv_state(11, len(lens))
    rng_ssm = synth.make_ssm_state(11, len(lens))
    has = [1, 0, 1, 1, 0, 1]
    h = synth.make_hidden(11, sum(lens))
    out, conv, ssm, tp = _run_prefill(blk, h, lens, rng_conv, rng_ssm, has_initial=has, taps=True)
    mask = np.array(has, np.float64)
    ref = oracle.block_prefill(Wt, h, lens, rng_conv * mask[:, None, None], rng_ssm * mask[:, None, None, None],
                               keep=True)
    assert_e4m3_close(to_np(tp["q2"]), ref["q2"], to_np(tp["o"]), ref["o"], Wt["s_y"])
    assert_out_is_gemm(to_np(out), to_np(tp["q2"]), gpu_out_proj(Wt))
    assert_block_out(to_np(out), ref["out"], q2=to_np(tp["q2"]), ref_q2=ref["q2"], Wt=Wt)
    assert_state(to_np(ssm), ref["ssm_state"])
    assert_bf16_close(to_np(conv), ref["conv_state"], atol=1e-3, what="conv_state")


def test_decode_after_prefill_carry(block0):
    """Prefill t0 tokens, decode the rest from the returned states: equals the
    oracle's single prefill over all tokens (the carry case)."""
    Wt, blk = block0
    T, t0 = 40, 33
    h = synth.make_hidden(12, T)
    out, conv, ssm, tp = _run_prefill(blk, h[:t0], [t0], taps=True)
    outs, q2s = [to_np(out)], [to_np(tp["q2"])]
    slot = torch.zeros(1, dtype=torch.int32, device="cuda")
    for t in range(t0, T):
        with q2_tap(blk, 1) as q2:
            outs.append(to_np(blk.decode(bf16_dev(h[t:t + 1]), conv, ssm, slot)))
        q2s.append(to_np(q2))
    ref = oracle.block_prefill(Wt, h, [T], keep=True)
    gemm = gpu_out_proj(Wt)
    for o_, q_ in zip(outs, q2s):                 # each call's out_proj on its own codes
        assert_out_is_gemm(o_, q_, gemm)
    assert_block_out(np.concatenate(outs), ref["out"], q2=np.concatenate(q2s), ref_q2=ref["q2"], Wt=Wt)
    assert_state(to_np(ssm), ref["ssm_state"])


def test_config3_prefill_4x2048(block0):
    Wt, blk = block0
    lens = [2048] * 4
    h = synth.make_hidden(3, sum(lens))
    out, conv, ssm, tp = _run_prefill(blk, h, lens, taps=True)
    ref = oracle.block_prefill(Wt, h, lens, keep=True)
    assert_e4m3_close(to_np(tp["q2"]), ref["q2"], to_np(tp["o"]), ref["o"], Wt["s_y"])
    assert_out_is_gemm(to_np(out), to_np(tp["q2"]), gpu_out_proj(Wt))
    assert_block_out(to_np(out), ref["out"], q2=to_np(tp["q2"]), ref_q2=ref["q2"], Wt=Wt)
    assert_state(to_np(ssm), ref["ssm_state"])
    assert_bf16_close(to_np(conv), ref["conv_state"], atol=1e-3, what="conv_state")


def test_rmsnorm_residual_vs_oracle():
    rng = np.random.default_rng(9)
    h = synth.as_bf16_values(rng.standard_normal((33, 2688)) * 2)
    a = synth.as_bf16_values(rng.standard_normal((33, 2688)))
    w = synth.make_stack_norm_w(4, 0)
    hd, ad = bf16_dev(h), bf16_dev(a)
    normed = m2.m2_rmsnorm_residual(hd, ad, bf16_dev(w), 1e-5)
    hsum = oracle.bf16_round(h.astype(np.float64) + a)
    assert_bf16_close(to_np(hd), hsum, max_frac=1e-4, what="residual")
    assert_bf16_close(to_np(normed), oracle.rmsnorm(hsum, w, 1e-5), what="rmsnorm")
