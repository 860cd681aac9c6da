"""The tensor-core accumulation probe computes what it claims: on products of
+-1 and 0 every partial sum is a small integer, exact in any accumulator of
13 or more bits, so the probe must return the exact sums (K = 128, one block,
and K = 4096, 32 blocks accumulated in tensor memory); on random codes it
agrees with the oracle's exact sum to within the 2% the pages report for the
previous generation."""
import numpy as np
import pytest
import torch

import fp8_fine_grained_20_b300 as fg
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


def unit_codes(rng, rows, K):
    c = rng.choice(np.array([0x38, 0xB8, 0x00], np.uint8), size=(rows, K), p=[0.4, 0.4, 0.2])
    return c


@pytest.mark.parametrize("K", [128, 4096])
def test_probe_exact_on_small_integers(orc, K):
    gu.cuda_or_skip()
    rng = np.random.default_rng(K)
    A, B = unit_codes(rng, 128, K), unit_codes(rng, 256, K)
    D = gu.host(fg.fp8_mma_accumulation_probe(gu.dev(A), gu.dev(B))).astype(np.float64)
    ref = orc.gemm_blockscaled(A, np.ones((128, K // 128), np.float32), B, np.ones((K // 128, 2), np.float32))
    assert np.array_equal(D, ref)
    assert fg.fp8_get_device_status(reset=True) == 0


def test_probe_close_on_random_codes(orc):
    gu.cuda_or_skip()
    rng = np.random.default_rng(1)
    K = 4096
    A = rng.integers(0, 0x7E, size=(128, K), dtype=np.uint8) | (rng.integers(0, 2, (128, K), dtype=np.uint8) << 7)
    B = rng.integers(0, 0x7E, size=(256, K), dtype=np.uint8) | (rng.integers(0, 2, (256, K), dtype=np.uint8) << 7)
    D = gu.host(fg.fp8_mma_accumulation_probe(gu.dev(A), gu.dev(B))).astype(np.float64)
    ref = orc.gemm_blockscaled(A, np.ones((128, K // 128), np.float32), B, np.ones((K // 128, 2), np.float32))
    assert np.linalg.norm(D - ref) / np.linalg.norm(ref) < 0.02
    assert fg.fp8_get_device_status(reset=True) == 0
