"""Failure detection on the device without a GPU fault: a bounded wait that
nothing satisfies gives up after its limit, records FP8_ERR_DEVICE_TIMEOUT in
the device status word, and the context stays usable (a GEMM afterwards
still matches the oracle).  The GEMM's own pipeline waits are made to run out
the same way: its TMA producer withholds every K-block after the first, the
MMA issuer's bounded wait gives up, both CTAs of every pair stop, drain what
they issued and free their tensor memory."""
import time

import numpy as np
import pytest
import torch

import fp8_fine_grained_20_b300 as fg
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_reports():
    gu.cuda_or_skip()
    fg.fp8_get_device_status(reset=True)
    t0 = time.perf_counter()
    fg.fp8_selftest_bounded_wait(timeout_ns=2_000_000)       # 2 ms
    assert fg.fp8_get_device_status(reset=True) == 5         # FP8_ERR_DEVICE_TIMEOUT
    assert time.perf_counter() - t0 < 5.0
    assert fg.fp8_get_device_status(reset=True) == 0         # cleared by the read


def test_context_usable_after_timeout(orc):
    gu.cuda_or_skip()
    fg.fp8_selftest_bounded_wait(timeout_ns=1_000_000)
    assert fg.fp8_get_device_status(reset=True) == 5
    rng = np.random.default_rng(3)
    qa = rng.integers(0, 0x7E, size=(128, 256), dtype=np.uint8)
    qb = rng.integers(0, 0x7E, size=(128, 256), dtype=np.uint8)
    sa = np.full((128, 2), 0.5, np.float32)
    sb = np.full((2, 1), 0.25, np.float32)
    C = fg.fp8_gemm_blockscaled(gu.dev(qa), gu.dev(np.ascontiguousarray(sa.T)).t(), gu.dev(qb), gu.dev(sb),
                                fg.FP8_SB_BLOCK128x128)
    torch.cuda.synchronize()
    ref = orc.gemm_blockscaled(qa, sa, qb, sb, orc.SB_BLOCK128x128)
    gu.assert_gemm_close(gu.host_bf16_as_f64(C), ref, "GEMM after a timed-out wait")
    assert fg.fp8_get_device_status(reset=True) == 0


def test_timeout_argument_checked():
    gu.cuda_or_skip()
    with pytest.raises(fg.FP8Error):
        fg.fp8_selftest_bounded_wait(timeout_ns=0)
    with pytest.raises(fg.FP8Error):
        fg.fp8_selftest_bounded_wait(timeout_ns=2_000_000_000)


def _small_gemm_operands(seed):
    rng = np.random.default_rng(seed)
    M, N, K = 128, 256, 256
    qa = rng.integers(0, 0x7E, size=(M, K), dtype=np.uint8)
    qb = rng.integers(0, 0x7E, size=(N, K), dtype=np.uint8)
    sa = np.full((M, K // 128), 0.5, np.float32)
    sb = np.full((K // 128, N // 128), 0.25, np.float32)
    return qa, sa, qb, sb


def test_gemm_pipeline_wait_runs_out_and_reports(orc):
    gu.cuda_or_skip()
    fg.fp8_get_device_status(reset=True)
    qa, sa, qb, sb = _small_gemm_operands(5)
    sA = gu.dev(np.ascontiguousarray(sa.T)).t()
    t0 = time.perf_counter()
    fg.fp8_selftest_gemm_timeout(gu.dev(qa), sA, gu.dev(qb), gu.dev(sb), wait_ns=2_000_000)
    assert fg.fp8_get_device_status(reset=True) == 5          # FP8_ERR_DEVICE_TIMEOUT
    assert time.perf_counter() - t0 < 10.0
    # the context is usable and the same GEMM without withholding is correct, twice
    for _ in range(2):
        C = fg.fp8_gemm_blockscaled(gu.dev(qa), sA, gu.dev(qb), gu.dev(sb), fg.FP8_SB_BLOCK128x128)
        torch.cuda.synchronize()
        ref = orc.gemm_blockscaled(qa, sa, qb, sb, orc.SB_BLOCK128x128)
        gu.assert_gemm_close(gu.host_bf16_as_f64(C), ref, "GEMM after its own wait ran out")
        assert fg.fp8_get_device_status(reset=True) == 0


def test_gemm_timeout_selftest_arguments_checked():
    gu.cuda_or_skip()
    qa, sa, qb, sb = _small_gemm_operands(6)
    sA = gu.dev(np.ascontiguousarray(sa.T)).t()
    with pytest.raises(fg.FP8Error):
        fg.fp8_selftest_gemm_timeout(gu.dev(qa), sA, gu.dev(qb), gu.dev(sb), wait_ns=10)
    with pytest.raises(fg.FP8Error):
        fg.fp8_selftest_gemm_timeout(gu.dev(qa[:, :128]), gu.dev(np.ascontiguousarray(sa[:, :1].T)).t(),
                                     gu.dev(qb[:, :128]), gu.dev(sb[:1]), wait_ns=2_000_000)
