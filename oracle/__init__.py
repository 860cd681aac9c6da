"""CPU oracle for fine-grained FP8 quantization and the block-scaled FP8 GEMM.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference leg may import this package.  It is a thin
numpy/ctypes wrapper over ``fp8fg_oracle.c`` (plain C, single-threaded, FP64 for
the GEMMs) and shares no code with the CUDA path.

Every array here is a numpy array.  bf16 tensors are passed as their uint16 bit
patterns, FP8 codes as uint8 (OCP E4M3), scales as float32.  The layouts are
the plain logical ones:

* ``quant_act_1x128(x[M,K]) -> (q[M,K], s[M,K/128])``
  (DeepSeek-V3 FP8 excerpt, sunipension.com post 314414, Figure 7(a))
* ``quant_w_128x128(w[K,N]) -> (q[K,N], s[K/128,N/128])`` (same figure)
* ``requant_1x128_to_128x1(q[M,K], s[M,K/128]) -> (qT[K,M], sT[K,M/128])``
  (same page: 1x128 tiles become 128x1 tiles for the backward pass)
* ``swiglu_bf16(gate[M,F], up[M,F]) -> y[M,F]`` bf16 bits of
  g*u/(1+exp(-g)) in FP64, rounded once (why-be.why-be.co.kr post 65900: the
  SwiGLU output is recomputed from its cached inputs)
* the three quantizers take ``pow2=True`` for power-of-two scales, the smallest
  2^e >= amax/448 (why-be.why-be.co.kr post 55081 and sunipension.com post
  314414: scaling factors that are integral powers of 2)
* ``gemm_blockscaled(A[M,K], sA[M,K/128], Bt[N,K], sB, sb_kind) -> C[M,N] float64``
  (why-be.why-be.co.kr post 55081, Figure 7(b): FP32 promotion of partials
  per 128-wide K interval, with the two scales applied there)
* ``grouped_gemm_blockscaled(A, sA, B[G,N,K], sB[G,K/128,N/128], offsets) -> C``
  (xn--jj0bz6z98ct0a29q.com post 362465: MoE activations dispatched in FP8)

Readings of the pages (format E4M3, scale = amax/448 as one fp32 division,
codes by round-to-nearest-even of the fp32 quotient, zero groups give s = 0,
requantization dequantizes with one fp32 multiply) are listed in the C file.
"""
import ctypes
import os

import numpy as np

from . import build as _build

SB_BLOCK128x128 = 0
SB_COL128x1 = 1

_lib = None


def _load():
    global _lib
    if _lib is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        i64, i32, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
        lib.orc_e4m3_decode.restype = ctypes.c_double
        lib.orc_e4m3_decode.argtypes = [ctypes.c_uint8]
        lib.orc_e4m3_encode.restype = ctypes.c_uint8
        lib.orc_e4m3_encode.argtypes = [ctypes.c_float]
        lib.orc_quant_act_1x128.argtypes = [vp, i64, i64, i64, vp, i64, vp]
        lib.orc_quant_w_128x128.argtypes = [vp, i64, i64, i64, vp, i64, vp]
        lib.orc_requant_1x128_to_128x1.argtypes = [vp, vp, i64, i64, i64, vp, i64, vp]
        lib.orc_quant_act_1x128_pow2.argtypes = [vp, i64, i64, i64, vp, i64, vp]
        lib.orc_quant_w_128x128_pow2.argtypes = [vp, i64, i64, i64, vp, i64, vp]
        lib.orc_requant_1x128_to_128x1_pow2.argtypes = [vp, vp, i64, i64, i64, vp, i64, vp]
        lib.orc_gemm_blockscaled.argtypes = [vp, i64, vp, vp, i64, vp, i32, i64, i64, i64, vp]
        lib.orc_swiglu_bf16.argtypes = [vp, i64, vp, i64, i64, i64, vp, i64]
        lib.orc_swiglu_bf16.restype = ctypes.c_int64
        lib.orc_gemm_blockscaled_sample.argtypes = [vp, i64, vp, vp, i64, vp, i32, i64, i64,
                                                    i64, vp, vp, i64, vp]
        lib.orc_grouped_gemm_blockscaled.argtypes = [vp, i64, vp, vp, vp, vp, i32, i64, i64,
                                                     i64, vp]
        lib.orc_grouped_gemm_blockscaled_sample.argtypes = [vp, i64, vp, vp, vp, vp, i32, i64,
                                                            i64, i64, vp, vp, i64, vp]
        for name in ("orc_quant_act_1x128", "orc_quant_w_128x128",
                     "orc_requant_1x128_to_128x1", "orc_quant_act_1x128_pow2",
                     "orc_quant_w_128x128_pow2", "orc_requant_1x128_to_128x1_pow2",
                     "orc_gemm_blockscaled",
                     "orc_gemm_blockscaled_sample", "orc_grouped_gemm_blockscaled",
                     "orc_grouped_gemm_blockscaled_sample"):
            getattr(lib, name).restype = ctypes.c_int
        lib.orc_e4m3_decode(0)      # fills the oracle's magnitude table before any threaded call
        _lib = lib
    return _lib


def _p(a):
    return ctypes.c_void_p(a.ctypes.data)


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a


def _check(rc, what):
    if rc != 0:
        raise ValueError("oracle %s rejected its arguments (rc=%d)" % (what, rc))


def e4m3_decode(code: int) -> float:
    """Value of one E4M3 code (NaN for 0x7F / 0xFF)."""
    return _load().orc_e4m3_decode(int(code) & 0xFF)


def e4m3_encode(y: float) -> int:
    """Round-to-nearest-even, saturating E4M3 code of one fp32 value."""
    return int(_load().orc_e4m3_encode(float(np.float32(y))))


def e4m3_encode_array(y) -> np.ndarray:
    """Elementwise ``e4m3_encode`` over a float32 array (slow: one C call each)."""
    y = np.asarray(y, dtype=np.float32).ravel()
    lib = _load()
    return np.fromiter((lib.orc_e4m3_encode(float(v)) for v in y), dtype=np.uint8,
                       count=y.size)


def _chunks(n, parts, align):
    """Split range(n) into at most `parts` pieces whose bounds are multiples of `align`."""
    units = n // align
    parts = max(1, min(parts, units)) if units else 1
    bounds = [align * (units * i // parts) for i in range(parts)] + [n]
    return [(bounds[i], bounds[i + 1]) for i in range(parts) if bounds[i + 1] > bounds[i]]


def _run_parallel(jobs, threads):
    """Run independent oracle calls; ctypes releases the GIL, so threads run in
    parallel.  Only the work distribution is parallel: every call is the plain
    single-threaded C routine on its own rows."""
    if threads is None or threads <= 1 or len(jobs) <= 1:
        return [j() for j in jobs]
    from concurrent.futures import ThreadPoolExecutor
    with ThreadPoolExecutor(max_workers=threads) as ex:
        return list(ex.map(lambda j: j(), jobs))


def default_threads():
    return max(1, min(32, os.cpu_count() or 1))


def quant_act_1x128(x, threads=None, pow2=False):
    """x: uint16 bf16 bits [M, K] -> (q uint8 [M, K], s float32 [M, K/128]).
    `threads` splits the rows (each 1x128 group lies in one row).  pow2: the
    power-of-two scale reading (smallest 2^e >= amax/448)."""
    x = _c(x, np.uint16)
    M, K = x.shape
    q = np.empty((M, K), np.uint8)
    s = np.empty((M, K // 128), np.float32)
    lib = _load()
    fn = lib.orc_quant_act_1x128_pow2 if pow2 else lib.orc_quant_act_1x128

    def job(r0, r1):
        return lambda: _check(fn(_p(x[r0:]), r1 - r0, K, K, _p(q[r0:]), K, _p(s[r0:])), "quant_act_1x128")
    _run_parallel([job(a, b) for a, b in _chunks(M, threads or 1, 1)] if M else [], threads)
    return q, s


def quant_w_128x128(w, threads=None, pow2=False):
    """w: uint16 bf16 bits [K, N] -> (q uint8 [K, N], s float32 [K/128, N/128]).
    `threads` splits the K rows on 128-row block boundaries.  pow2: the
    power-of-two scale reading."""
    w = _c(w, np.uint16)
    K, N = w.shape
    q = np.empty((K, N), np.uint8)
    s = np.empty((K // 128, N // 128), np.float32)
    lib = _load()
    fn = lib.orc_quant_w_128x128_pow2 if pow2 else lib.orc_quant_w_128x128

    def job(r0, r1):
        return lambda: _check(fn(_p(w[r0:]), r1 - r0, N, N, _p(q[r0:]), N, _p(s[r0 // 128:])),
                              "quant_w_128x128")
    if K % 128 or N % 128:
        _check(-1, "quant_w_128x128")
    _run_parallel([job(a, b) for a, b in _chunks(K, threads or 1, 128)] if K else [], threads)
    return q, s


def requant_1x128_to_128x1(q, s, threads=None, pow2=False):
    """(q uint8 [M, K], s float32 [M, K/128]) -> (qT uint8 [K, M], sT float32 [K, M/128]).
    `threads` splits the channels on 128-channel boundaries.  pow2: power-of-two
    scales for the 128x1 groups."""
    q = _c(q, np.uint8)
    s = _c(s, np.float32)
    M, K = q.shape
    assert s.shape == (M, K // 128)
    qT = np.empty((K, M), np.uint8)
    sT = np.empty((K, M // 128), np.float32)
    lib = _load()
    if M % 128 or K % 128:
        _check(-1, "requant_1x128_to_128x1")

    fn = lib.orc_requant_1x128_to_128x1_pow2 if pow2 else lib.orc_requant_1x128_to_128x1

    def job(k0, k1):
        s_part = np.ascontiguousarray(s[:, k0 // 128:k1 // 128])
        return lambda: _check(fn(_p(q[:, k0:]), _p(s_part), M, k1 - k0, K, _p(qT[k0:]), M, _p(sT[k0:])),
                              "requant_1x128_to_128x1")
    _run_parallel([job(a, b) for a, b in _chunks(K, threads or 1, 128)] if K and M else [], threads)
    return qT, sT


def gemm_blockscaled(A, sA, Bt, sB, sb_kind=SB_BLOCK128x128):
    """Full FP64 block-scaled GEMM.

    A uint8 [M, K], sA float32 [M, K/128]; Bt uint8 [N, K] (B stored K-major);
    sB float32 [K/128, ceil(N/128)] (block) or [K/128, N] (per column).
    Returns float64 [M, N]."""
    A, sA, Bt, sB = _c(A, np.uint8), _c(sA, np.float32), _c(Bt, np.uint8), _c(sB, np.float32)
    M, K = A.shape
    N = Bt.shape[0]
    assert Bt.shape == (N, K) and sA.shape == (M, K // 128)
    C = np.empty((M, N), np.float64)
    _check(_load().orc_gemm_blockscaled(_p(A), K, _p(sA), _p(Bt), K, _p(sB), sb_kind,
                                        M, N, K, _p(C)), "gemm_blockscaled")
    return C


def gemm_blockscaled_sample(A, sA, Bt, sB, sb_kind, ms, ns, threads=None):
    """The FP64 GEMM evaluated only at the positions (ms[i], ns[i])."""
    A, sA, Bt, sB = _c(A, np.uint8), _c(sA, np.float32), _c(Bt, np.uint8), _c(sB, np.float32)
    ms, ns = _c(ms, np.int64), _c(ns, np.int64)
    M, K = A.shape
    N = Bt.shape[0]
    out = np.empty(ms.size, np.float64)
    lib = _load()

    def job(i0, i1):
        return lambda: _check(lib.orc_gemm_blockscaled_sample(_p(A), K, _p(sA), _p(Bt), K, _p(sB), sb_kind,
                                                              M, N, K, _p(ms[i0:]), _p(ns[i0:]), i1 - i0,
                                                              _p(out[i0:])), "gemm_blockscaled_sample")
    _run_parallel([job(a, b) for a, b in _chunks(ms.size, threads or 1, 1)] if ms.size else [], threads)
    return out


def grouped_gemm_blockscaled(A, sA, B, sB, offsets):
    """Grouped FP64 GEMM.  A uint8 [M_total, K]; sA float32 [M_total, K/128];
    B uint8 [G, N, K]; sB float32 [G, K/128, N/128]; offsets int32 [G+1].
    Rows outside every expert come back as NaN."""
    A, sA, B, sB = _c(A, np.uint8), _c(sA, np.float32), _c(B, np.uint8), _c(sB, np.float32)
    offsets = _c(offsets, np.int32)
    M_total, K = A.shape
    G, N, _ = B.shape
    C = np.full((M_total, N), np.nan, np.float64)
    _check(_load().orc_grouped_gemm_blockscaled(_p(A), K, _p(sA), _p(B), _p(sB), _p(offsets),
                                                G, M_total, N, K, _p(C)),
           "grouped_gemm_blockscaled")
    return C


def grouped_gemm_blockscaled_sample(A, sA, B, sB, offsets, ms, ns, threads=None):
    """The grouped GEMM evaluated only at (ms[i], ns[i])."""
    A, sA, B, sB = _c(A, np.uint8), _c(sA, np.float32), _c(B, np.uint8), _c(sB, np.float32)
    offsets = _c(offsets, np.int32)
    ms, ns = _c(ms, np.int64), _c(ns, np.int64)
    M_total, K = A.shape
    G, N, _ = B.shape
    out = np.empty(ms.size, np.float64)
    lib = _load()

    def job(i0, i1):
        return lambda: _check(lib.orc_grouped_gemm_blockscaled_sample(_p(A), K, _p(sA), _p(B), _p(sB),
                                                                      _p(offsets), G, M_total, N, K,
                                                                      _p(ms[i0:]), _p(ns[i0:]), i1 - i0,
                                                                      _p(out[i0:])),
                              "grouped_gemm_blockscaled_sample")
    _run_parallel([job(a, b) for a, b in _chunks(ms.size, threads or 1, 1)] if ms.size else [], threads)
    return out


def swiglu_bf16(gate, up, threads=None):
    """gate, up: uint16 bf16 bits [M, F] -> y uint16 bf16 bits [M, F],
    y = bf16(g * u / (1 + exp(-g))) evaluated in FP64 and rounded once."""
    gate, up = _c(gate, np.uint16), _c(up, np.uint16)
    assert gate.shape == up.shape
    M, F = gate.shape
    y = np.empty((M, F), np.uint16)
    lib = _load()

    def job(r0, r1):
        return lambda: lib.orc_swiglu_bf16(_p(gate[r0:]), F, _p(up[r0:]), F, r1 - r0, F, _p(y[r0:]), F)
    undecided = sum(_run_parallel([job(a, b) for a, b in _chunks(M, threads or 1, 1)] if M else [], threads))
    if undecided:
        raise ValueError("oracle swiglu_bf16: %d roundings could not be decided" % undecided)
    return y


def dequant_dense(q, s, axis_groups):
    """FP64 values of codes q [R, C] with scales s: axis_groups=1 -> s [R, C/128]
    (groups along columns), 0 -> s [R/128, C/128] blocks.  Exact in FP64."""
    lib = _load()
    table = np.array([lib.orc_e4m3_decode(c) for c in range(256)], np.float64)
    v = table[np.asarray(q, np.uint8)]
    s = np.asarray(s, np.float64)
    if axis_groups == 1:
        v *= np.repeat(s, 128, axis=1)
    else:
        v *= np.repeat(np.repeat(s, 128, axis=0), 128, axis=1)
    return v


def gemm_blockscaled_dense(A, sA, Bt, sB, sb_kind=SB_BLOCK128x128):
    """The block-scaled GEMM as the FP64 matrix product of the dequantized
    operands (reading R6: the promotion interval equals the quantization group,
    so the result is exactly that product), with numpy's float64 matmul as the
    summation step.  Same arguments as gemm_blockscaled; the summation order
    differs from it only by FP64 rounding."""
    A, Bt = np.asarray(A, np.uint8), np.asarray(Bt, np.uint8)
    sA, sB = np.asarray(sA, np.float32), np.asarray(sB, np.float32)
    a = dequant_dense(A, sA, 1)
    if sb_kind == SB_COL128x1:
        b = dequant_dense(Bt, np.ascontiguousarray(sB.T), 1)          # sB [K/128, N] -> per row of Bt
    else:
        b = dequant_dense(Bt, np.ascontiguousarray(sB.T), 0)          # sB [K/128, N/128] -> blocks of Bt
    return a @ b.T
