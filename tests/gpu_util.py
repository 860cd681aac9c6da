"""Helpers shared by the GPU parity tests (device transfer and the GEMM
acceptance check).  No method arithmetic lives here."""
import numpy as np
import pytest
import torch

# GEMM acceptance: per element |d| <= 2^-7 |ref| + 1e-4 rms(ref), and a relative
# Frobenius error <= 5e-3 (FP32 promotion per 128-K block, one bf16 rounding of
# the output: its 2^-9 relative error is well inside 2^-7).
REL_TOL = 2.0 ** -7
ABS_TOL_RMS = 1e-4
FROB_TOL = 5e-3


def cuda_or_skip():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    return torch.device("cuda", 0)


def bf16_dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t):
    return t.detach().cpu().numpy()


def host_bf16_as_f64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def assert_gemm_close(got, ref, what=""):
    """got: float64 array from the GPU's bf16 output; ref: the oracle's FP64 values."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape
    assert np.all(np.isfinite(got)), what + ": non-finite output"
    rms = np.sqrt(np.mean(ref ** 2))
    err = np.abs(got - ref)
    bound = REL_TOL * np.abs(ref) + ABS_TOL_RMS * rms
    bad = err > bound
    if bad.any():
        i = np.argmax(err - bound)
        raise AssertionError("%s: %d of %d elements out of tolerance; worst at flat %d: got %r ref %r"
                             % (what, int(bad.sum()), bad.size, i, got.flat[i], ref.flat[i]))
    frob = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300)
    assert frob <= FROB_TOL, "%s: relative Frobenius error %.3g" % (what, frob)


def assert_device_status_clean():
    import fp8_fine_grained_20_b300 as fg
    assert fg.fp8_get_device_status(reset=True) == 0
