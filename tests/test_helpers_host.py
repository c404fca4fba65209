"""Host checks of the comparison helpers the GPU tests rely on."""
import numpy as np
import pytest

import oracle
from helpers import assert_e4m3_close


def _codes(vals):
    return oracle.e4m3_encode(np.asarray(vals, np.float64))



def _quant(o, s):
    return oracle.quant_static_e4m3(o, s)


def test_e4m3_close_accepts_codes_their_inputs_explain():
    rng = np.random.default_rng(0)
    s = 1.0 / 32
    ref_o = oracle.bf16_round(rng.standard_normal(4000))
    got_o = ref_o.copy()
    got_o[10] = oracle.bf16_round(ref_o[10] * (1 + 2.0 ** -7))      # one bf16 step: at most one code
    got_o[20] = ref_o[20] + 0.01                                     # a small value moved by an upstream step
    assert_e4m3_close(_quant(got_o, s), _quant(ref_o, s), got_o, ref_o, s, max_frac=1e-3, o_rel_l2=1e-2)


def test_e4m3_close_rejects_codes_their_inputs_do_not_explain():
    rng = np.random.default_rng(1)
    s = 1.0 / 32
    o = oracle.bf16_round(rng.standard_normal(2000))
    g = _quant(o, s)
    g[5] = g[5] + 2 if (g[5] & 0x7F) < 0x70 else g[5] - 2         # two codes off, same input
    with pytest.raises(AssertionError, match="not the e4m3 rounding"):
        assert_e4m3_close(g, _quant(o, s), o, o, s)


def test_e4m3_close_rejects_too_many_differences():
    s = 1.0
    ref_o = np.full(100, 1.0)
    got_o = np.full(100, 1.125)
    with pytest.raises(AssertionError):
        assert_e4m3_close(_quant(got_o, s), _quant(ref_o, s), got_o, ref_o, s, o_rel_l2=1.0)


def _out_case(seed=0, T=40, H=48, K=256):
    rng = np.random.default_rng(seed)
    w = _codes(rng.standard_normal((H, K)) * 40)
    q2 = _codes(rng.standard_normal((T, K)) * 30)
    Wt = dict(out_proj=w, s_y=1.0 / 32, s_w2=2.0 ** -9)
    return rng, Wt, q2


def test_block_out_admits_exactly_what_code_flips_move():
    from helpers import assert_block_out
    rng, Wt, ref_q2 = _out_case()
    q2 = ref_q2.copy()
    big = np.argsort(-np.abs(oracle.e4m3_decode(q2[3])))[:3]      # flip three large codes of row 3 by one step
    q2[3, big] = np.where(q2[3, big] & 0x80, q2[3, big] - 1, q2[3, big] + 1)
    ref = oracle.fp8_linear(ref_q2, Wt["s_y"], Wt["out_proj"], Wt["s_w2"])
    got = oracle.fp8_linear(q2, Wt["s_y"], Wt["out_proj"], Wt["s_w2"])
    assert np.abs(got - ref).max() > 2e-2 + 0.03                   # beyond the plain bound, in row 3 only
    assert_block_out(got, ref, q2=q2, ref_q2=ref_q2, Wt=Wt)
    with pytest.raises(AssertionError):
        assert_block_out(got, ref)                                  # without the codes: the plain bound


def test_block_out_rejects_an_output_error_outside_flipped_rows():
    from helpers import assert_block_out
    rng, Wt, ref_q2 = _out_case(1)
    q2 = ref_q2.copy()
    q2[3, 0] += 1
    ref = oracle.fp8_linear(ref_q2, Wt["s_y"], Wt["out_proj"], Wt["s_w2"])
    got = oracle.fp8_linear(q2, Wt["s_y"], Wt["out_proj"], Wt["s_w2"]).copy()
    got[7, 5] += 0.1                                                # an epilogue error on a row with no flip
    with pytest.raises(AssertionError):
        assert_block_out(got, ref, q2=q2, ref_q2=ref_q2, Wt=Wt)


def test_out_is_gemm_is_bit_exact():
    from helpers import assert_out_is_gemm
    rng, Wt, q2 = _out_case(2)
    gemm = lambda a: oracle.fp8_linear(a, Wt["s_y"], Wt["out_proj"], Wt["s_w2"])
    got = gemm(q2).copy()
    assert_out_is_gemm(got, q2, gemm)
    got[3, 5] = oracle.bf16_round(got[3, 5] * (1 + 2.0 ** -7))      # one bf16 step off
    with pytest.raises(AssertionError, match="1 elements differ"):
        assert_out_is_gemm(got, q2, gemm)
