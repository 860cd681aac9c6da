"""C-ABI library checks that need no GPU: it builds, loads, exports every
symbol the header declares, and rejects bad arguments on the host before any
CUDA call."""
import ctypes
import os
import re

import pytest

import fp8_fine_grained_20_b300 as fg
from fp8_fine_grained_20_b300 import build as fgbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fp8fg.h")


@pytest.fixture(scope="module")
def lib():
    fgbuild.build()
    return fg.capi()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fp8\w*)\s*\(", text)))


def test_header_declares_the_five_calls():
    names = declared_functions()
    for n in ("fp8_quant_act_1x128", "fp8_quant_w_128x128", "fp8_requant_1x128_to_128x1",
              "fp8_gemm_blockscaled", "fp8_grouped_gemm_blockscaled"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert name in fg._SIGNATURES, name


def test_status_strings(lib):
    for code, name in fg.STATUS_NAMES.items():
        assert fg.fp8_status_string(code).startswith(name)
    assert lib.fp8fg_version() >= 100


NULL = ctypes.c_void_p(0)
A16 = ctypes.c_void_p(0x10000)      # 16-byte aligned fake device addresses: never dereferenced,
A16b = ctypes.c_void_p(0x20000)     # every call below is rejected before any CUDA call
MIS = ctypes.c_void_p(0x10008)


def test_quant_act_rejections(lib):
    f = lib.fp8_quant_act_1x128
    assert f(A16, 4, 100, 100, A16b, 100, A16, 1, 4, NULL) == 3            # K % 128
    assert f(A16, -1, 128, 128, A16b, 128, A16, 1, 4, NULL) == 3           # negative M
    assert f(A16, 0, 128, 128, A16b, 128, A16, 1, 4, NULL) == 0            # empty: nothing launched
    assert f(NULL, 4, 128, 128, A16b, 128, A16, 1, 4, NULL) == 1           # null x
    assert f(A16, 4, 128, 64, A16b, 128, A16, 1, 4, NULL) == 6             # ldx < K
    assert f(MIS, 4, 128, 128, A16b, 128, A16, 1, 4, NULL) == 2            # misaligned x
    assert f(A16, 4, 128, 132, A16b, 128, A16, 1, 4, NULL) == 2            # ldx*2 not multiple of 16


def test_quant_w_rejections(lib):
    f = lib.fp8_quant_w_128x128
    assert f(A16, 256, 200, 200, A16b, 256, 0, A16, 2, 1, NULL) == 3       # N % 128
    assert f(A16, 256, 256, 256, A16b, 256, 7, A16, 2, 1, NULL) == 6       # bad layout
    assert f(A16, 256, 256, 256, NULL, 256, 0, A16, 2, 1, NULL) == 1
    assert f(A16, 256, 256, 256, MIS, 256, 0, A16, 2, 1, NULL) == 2


def test_requant_rejections(lib):
    f = lib.fp8_requant_1x128_to_128x1
    assert f(A16, 200, 128, 128, A16, 1, 200, A16b, 200, A16, 1, 128, NULL) == 3   # M % 128
    assert f(A16, 256, 128, 128, NULL, 1, 256, A16b, 256, A16, 1, 128, NULL) == 1
    assert f(A16, 256, 128, 128, A16, 1, 256, A16b, 128, A16, 1, 128, NULL) == 6   # ldqT < M


def test_gemm_rejections(lib):
    f = lib.fp8_gemm_blockscaled
    ok = [A16, 256, A16, 1, 256, A16b, 256, A16, 2, 1, 0, A16b, 256, 256, 256, 256, NULL]
    bad = list(ok); bad[10] = 5
    assert f(*bad) == 6                                   # sb_kind
    bad = list(ok); bad[13] = 200
    assert f(*bad) == 3                                   # M % 128
    bad = list(ok); bad[15] = 0
    assert f(*bad) == 3                                   # K == 0 with a non-empty output
    bad = list(ok); bad[0] = NULL
    assert f(*bad) == 1
    bad = list(ok); bad[5] = MIS
    assert f(*bad) == 2
    bad = list(ok); bad[1] = 128
    assert f(*bad) == 6                                   # lda < K
    bad = list(ok); bad[13] = 0
    assert f(*bad) == 0                                   # empty output


def test_grouped_gemm_rejections(lib):
    f = lib.fp8_grouped_gemm_blockscaled
    ok = [A16, 256, A16, 1, 256, A16b, A16, A16, 4, 256, 256, 256, A16b, 256, NULL]
    bad = list(ok); bad[8] = 0
    assert f(*bad) == 6                                   # G == 0
    bad = list(ok); bad[8] = 5000
    assert f(*bad) == 6                                   # G too large
    bad = list(ok); bad[7] = NULL
    assert f(*bad) == 1                                   # offsets
    bad = list(ok); bad[9] = 100
    assert f(*bad) == 3                                   # M_total % 128
    bad = list(ok); bad[7] = ctypes.c_void_p(0x10002)
    assert f(*bad) == 2


def test_binding_refuses_cpu_tensors():
    import torch
    x = torch.zeros(4, 128, dtype=torch.bfloat16)
    with pytest.raises(TypeError):
        fg.fp8_quant_act_1x128(x)


def test_batched_weight_quant_rejections(lib):
    f = lib.fp8_quant_w_128x128_batched
    K, N = 256, 384
    ok = [A16, 3, K, N, N, K * N, A16b, K, N * K, 0, A16, 3, 1, 6, NULL]
    bad = list(ok); bad[1] = -1
    assert f(*bad) == 3                                   # negative G
    bad = list(ok); bad[1] = 0
    assert f(*bad) == 0                                   # no experts: nothing launched
    bad = list(ok); bad[5] = K * N - 8
    assert f(*bad) == 6                                   # experts overlap
    bad = list(ok); bad[5] = K * N + 4
    assert f(*bad) == 2                                   # expert stride not a multiple of 16 bytes
    bad = list(ok); bad[6] = NULL
    assert f(*bad) == 1
    bad = list(ok); bad[9] = 7
    assert f(*bad) == 6                                   # layout
    bad = list(ok); bad[2] = 200
    assert f(*bad) == 3                                   # K % 128


def test_quantizing_gemm_rejections(lib):
    f = lib.fp8_gemm_blockscaled_q1x128
    ok = [A16, 256, A16, 1, 256, A16b, 256, A16, 2, 1, 0, A16b, 256, A16, 1, 256, 256, 256, 256, NULL]
    bad = list(ok); bad[11] = NULL
    assert f(*bad) == 1                                   # codes
    bad = list(ok); bad[13] = NULL
    assert f(*bad) == 1                                   # scales
    bad = list(ok); bad[12] = 128
    assert f(*bad) == 6                                   # ldcq < N
    bad = list(ok); bad[12] = 264
    assert f(*bad) == 2                                   # ldcq not a multiple of 16
    bad = list(ok); bad[13] = ctypes.c_void_p(0x10002)
    assert f(*bad) == 2                                   # misaligned scales
    bad = list(ok); bad[17] = 200
    assert f(*bad) == 3                                   # N % 128


def test_probe_and_selftest_rejections(lib):
    probe = lib.fp8_mma_accumulation_probe
    assert probe(A16, A16b, 0, A16, NULL) == 3
    assert probe(A16, A16b, 100, A16, NULL) == 3
    assert probe(NULL, A16b, 128, A16, NULL) == 1
    assert probe(MIS, A16b, 128, A16, NULL) == 2
    wait = lib.fp8_selftest_bounded_wait
    assert wait(0, NULL) == 6
    assert wait(2_000_000_000, NULL) == 6


def test_pow2_quantizer_rejections(lib):
    f = lib.fp8_quant_act_1x128_pow2
    assert f(A16, 4, 100, 100, A16b, 100, A16, 1, 4, NULL) == 3            # K % 128
    assert f(NULL, 4, 128, 128, A16b, 128, A16, 1, 4, NULL) == 1
    assert f(MIS, 4, 128, 128, A16b, 128, A16, 1, 4, NULL) == 2
    assert f(A16, 0, 128, 128, A16b, 128, A16, 1, 4, NULL) == 0            # empty
    w = lib.fp8_quant_w_128x128_pow2
    assert w(A16, 256, 200, 200, A16b, 256, 0, A16, 2, 1, NULL) == 3
    assert w(A16, 256, 256, 256, A16b, 256, 7, A16, 2, 1, NULL) == 6
    wb = lib.fp8_quant_w_128x128_batched_pow2
    assert wb(A16, 2, 256, 384, 384, 256 * 384 - 8, A16b, 256, 384 * 256, 0, A16, 3, 1, 6, NULL) == 6
    r = lib.fp8_requant_1x128_to_128x1_pow2
    assert r(A16, 200, 128, 128, A16, 1, 200, A16b, 200, A16, 1, 128, NULL) == 3
    assert r(A16, 256, 128, 128, NULL, 1, 256, A16b, 256, A16, 1, 128, NULL) == 1


def test_mx_gemm_rejections(lib):
    f = lib.fp8_gemm_blockscaled_mx
    ok = [A16, 256, A16, 1, 256, A16b, 256, A16, 2, 1, 0, A16b, 256, 256, 256, 256, NULL]
    bad = list(ok); bad[10] = 5
    assert f(*bad) == 6                                   # sb_kind
    bad = list(ok); bad[14] = 200
    assert f(*bad) == 3                                   # N % 128
    bad = list(ok); bad[15] = 0
    assert f(*bad) == 3                                   # K == 0 with a non-empty output
    bad = list(ok); bad[11] = NULL
    assert f(*bad) == 1
    bad = list(ok); bad[12] = 100
    assert f(*bad) == 6                                   # ldc < N
    g = lib.fp8_grouped_gemm_blockscaled_mx
    ok = [A16, 256, A16, 1, 256, A16b, A16, A16, 4, 256, 256, 256, A16b, 256, NULL]
    bad = list(ok); bad[8] = 0
    assert g(*bad) == 6
    bad = list(ok); bad[7] = NULL
    assert g(*bad) == 1
    bad = list(ok); bad[11] = 100
    assert g(*bad) == 3


def test_gemm_timeout_selftest_rejections(lib):
    f = lib.fp8_selftest_gemm_timeout
    assert f(A16, A16, A16b, A16, A16b, 128, 256, 256, 10, NULL) == 6          # bound below 1 us
    assert f(A16, A16, A16b, A16, A16b, 128, 256, 256, 2_000_000_000, NULL) == 6
    assert f(A16, A16, A16b, A16, A16b, 128, 256, 128, 2_000_000, NULL) == 3   # K < 256
    assert f(NULL, A16, A16b, A16, A16b, 128, 256, 256, 2_000_000, NULL) == 1


def test_swiglu_quant_rejections(lib):
    f = lib.fp8_swiglu_quant_1x128
    ok = [A16, 512, A16b, 512, 4, 256, A16, 256, A16b, 1, 4, NULL, 0, NULL]
    bad = list(ok); bad[5] = 200
    assert f(*bad) == 3                                   # F % 128
    bad = list(ok); bad[4] = -1
    assert f(*bad) == 3
    bad = list(ok); bad[4] = 0
    assert f(*bad) == 0                                   # empty: nothing launched
    bad = list(ok); bad[2] = NULL
    assert f(*bad) == 1                                   # up
    bad = list(ok); bad[1] = 128
    assert f(*bad) == 6                                   # ldg < F
    bad = list(ok); bad[0] = MIS
    assert f(*bad) == 2
    bad = list(ok); bad[11] = A16; bad[12] = 100
    assert f(*bad) == 6                                   # ldy < F with a y output
    bad = list(ok); bad[11] = MIS; bad[12] = 256
    assert f(*bad) == 2                                   # misaligned y


def test_bounds_checked_build_exports_every_symbol():
    """The debug build with every device write bounds-checked (-DFP8FG_BOUNDS,
    loaded when FP8FG_BOUNDS=1) is the same C ABI."""
    path = fgbuild.build(bounds=True)
    dbg = ctypes.CDLL(path)
    for name in declared_functions():
        assert hasattr(dbg, name), name
    dbg.fp8_status_string.restype = ctypes.c_char_p
    assert dbg.fp8_status_string(10).decode().startswith("FP8_ERR_DEVICE_BOUNDS")
