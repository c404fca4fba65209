"""fp8_linear_noalloc: the fp8_linear variant for callers that cannot allocate
device memory (no allocator of their own, a fixed footprint after start-up,
or work issued during a stream capture).  It keeps its split-K partial sums in
one library-owned device array instead of a caller workspace.

Checked through the C ABI against the existing fp8_linear entry point, on two
calls in a row with different shapes (the second call must not see the
first call's leftovers in the shared array), with the tolerance the GEMM
parity tests use.  This file is collected last so that a failure here cannot
hide the other tests' results.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from helpers import assert_bf16_close, gemm_atol, to_np, u8_dev

pytestmark = pytest.mark.gpu

m2 = pytest.importorskip("mamba2_ssm_mixer_gb300")


def _codes(rng, shape):
    c = rng.integers(0, 256, shape).astype(np.uint8)
    c[(c & 0x7F) == 0x7F] = 0x00           # no NaN codes
    c[(c & 0x78) == 0x78] &= 0xF7           # keep magnitudes below 256 (no overflow concerns)
    return c


def _noalloc(a, s_a, w, s_w, y):
    st = m2._lib.fp8_linear_noalloc(a.data_ptr(), s_a, w.data_ptr(), s_w, y.data_ptr(), a.shape[0], w.shape[0],
                                    a.shape[1], torch.cuda.current_stream().cuda_stream)
    return st


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def test_noalloc_matches_fp8_linear_on_two_calls_in_a_row():
    rng = np.random.default_rng(2026)
    cases = [(64, 10304, 2688, 1.0 / 64, 2.5e-4),   # decode in_proj shape
             (37, 2688, 4096, 1.0 / 32, 2.4e-4)]    # then a different split count
    for M, N, K, s_a, s_w in cases:
        a, w = _codes(rng, (M, K)), _codes(rng, (N, K))
        ad, wd = u8_dev(a), u8_dev(w)
        y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        assert _noalloc(ad, s_a, wd, s_w, y) == m2.M2_OK, m2.last_error()
        ref = m2.fp8_linear(ad, s_a, wd, s_w)
        torch.cuda.synchronize()
        got = to_np(y)
        assert np.all(np.isfinite(got))
        assert_bf16_close(got, to_np(ref), atol=gemm_atol(a, w, s_a * s_w), what=f"noalloc {M}x{N}x{K}")
        # and against the oracle directly
        assert_bf16_close(got, oracle.fp8_linear(a, s_a, w, s_w), atol=gemm_atol(a, w, s_a * s_w),
                          what=f"noalloc vs oracle {M}x{N}x{K}")


def test_noalloc_refuses_sizes_beyond_its_scratch():
    a = torch.zeros((300, 2688), dtype=torch.uint8, device="cuda")
    w = torch.zeros((2688, 2688), dtype=torch.uint8, device="cuda")
    y = torch.empty((300, 2688), dtype=torch.bfloat16, device="cuda")
    assert _noalloc(a, 1.0, w, 1.0, y) == m2.M2_ESHAPE
    assert "M = 300" in m2.last_error()
    a = torch.zeros((256, 2688), dtype=torch.uint8, device="cuda")
    w = torch.zeros((10304, 2688), dtype=torch.uint8, device="cuda")
    y = torch.empty((256, 10304), dtype=torch.bfloat16, device="cuda")
    assert _noalloc(a, 1.0, w, 1.0, y) == m2.M2_ESHAPE
    assert "scratch" in m2.last_error()
