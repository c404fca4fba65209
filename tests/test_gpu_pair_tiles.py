"""The persistent CTA-pair GEMM (more than 256 rows) on outputs whose width
uses 44 to 192 columns of the last 256-wide column of tiles (the part past
N is computed on B rows read as zeros and never stored), with ragged M (the
last row of tiles part-filled), more tiles than clusters and fewer.
Integer-valued operands make every partial sum an exact integer below 2^24,
so each result is bit-exact against the oracle in any summation order, for
the e4m3 (fp8_linear) and the bf16 (bf16_linear) operand forms."""
import numpy as np
import pytest
import torch

import oracle
from helpers import bf16_dev, to_np, u8_dev

pytestmark = pytest.mark.gpu

m2 = pytest.importorskip("mamba2_ssm_mixer_gb300")


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.init()


SHAPES = [
    (8192, 2688, 256),    # 128 columns of the last tile column (out_proj's width), more tiles than clusters
    (512, 10304, 128),    # 64 columns of it (in_proj's width)
    (20000, 448, 64),     # 192 columns of it, more tiles than clusters
    (2304, 320, 128),     # 64 columns of it, 9 rows of tiles
    (700, 448, 96),       # 192 columns of it, ragged M
    (520, 300, 64),       # 44 columns of it
    (8256, 10304, 128),   # in_proj's width at the mixed step's rows: 64-row last row of tiles
]


def _codes(rng, shape):
    ints = rng.integers(-8, 9, shape)
    lut = oracle.e4m3_encode(np.arange(-8, 9, dtype=np.float64))
    return ints, lut[ints + 8]


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_pair_gemm_items_fp8_exact(M, N, K):
    rng = np.random.default_rng(M + 3 * N + K)
    _, a = _codes(rng, (M, K))
    _, w = _codes(rng, (N, K))
    ref = oracle.fp8_linear(a, 1.0, w, 1.0)
    ad, wd = u8_dev(a), u8_dev(w)
    for _ in range(2):   # a second call on the same buffers
        y = to_np(m2.fp8_linear(ad, 1.0, wd, 1.0))
        assert np.array_equal(y, ref)


@pytest.mark.parametrize("M,N,K", [SHAPES[0], SHAPES[2], SHAPES[4]])
def test_pair_gemm_items_bf16_exact(M, N, K):
    rng = np.random.default_rng(M + 5 * N + K)
    x = rng.integers(-8, 9, (M, K)).astype(np.float64)
    w = rng.integers(-8, 9, (N, K)).astype(np.float64)
    y = to_np(m2.bf16_linear(bf16_dev(x), bf16_dev(w)))
    assert np.array_equal(y, oracle.bf16_linear(x, w))
