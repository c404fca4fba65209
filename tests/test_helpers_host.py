"""Host checks of the comparison helpers the GPU tests rely on."""
import numpy as np
import pytest

import oracle
from helpers import assert_e4m3_close


def _codes(vals):
    return oracle.e4m3_encode(np.asarray(vals, np.float64))


def test_e4m3_close_accepts_adjacent_and_near_zero_codes():
    ref = _codes(np.linspace(-3, 3, 4000))
    got = ref.copy()
    got[10] = ref[10] + 1                                                    # the next magnitude code
    i = int(np.argmin(np.abs(oracle.e4m3_decode(ref))))                      # the code nearest zero
    got[i] = _codes([oracle.e4m3_decode(ref[i:i + 1])[0] + 3 * 2.0 ** -9])[0]  # three uniform steps away
    assert_e4m3_close(got, ref, max_frac=1e-3)


def test_e4m3_close_rejects_two_steps_away_from_zero():
    ref = _codes(np.full(2000, 1.0))
    got = ref.copy()
    got[5] = _codes([1.25])[0]                  # two codes above 1.0 (steps of 0.125)
    with pytest.raises(AssertionError, match="more than one step"):
        assert_e4m3_close(got, ref, max_frac=1e-3)


def test_e4m3_close_rejects_too_many_differences():
    ref = _codes(np.full(100, 1.0))
    got = _codes(np.full(100, 1.125))
    with pytest.raises(AssertionError, match="of codes differ"):
        assert_e4m3_close(got, ref)


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
