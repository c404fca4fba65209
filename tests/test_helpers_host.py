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
