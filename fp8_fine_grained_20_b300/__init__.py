"""Fine-grained FP8 quantization and block-scaled FP8 GEMM for NVIDIA B300.

A thin Python binding over the C ABI of ``libfp8fg.so`` (``include/fp8fg.h``).
Every computation runs in the library's CUDA kernels; this module only
marshals arguments.  PyTorch supplies device memory and streams.  There is no
CPU fallback: the calls raise if the library is missing or a tensor is not on
a CUDA device.

Functions (same names as the C entry points):

* ``fp8_quant_act_1x128(x)`` -- bf16 [M, K] -> (codes uint8 [M, K], scales
  float32 logical [M, K/128])   (1x128 tiles, DeepSeek-V3 FP8 excerpt at
  sunipension.com post 314414, Figure 7(a))
* ``fp8_quant_w_128x128(w)`` -- bf16 [K, N] -> (codes uint8 [N, K] (K-major)
  or [K, N], scales float32 [K/128, N/128])   (128x128 blocks, same figure)
* ``fp8_quant_w_128x128_batched(w)`` -- the same for G weights [G, K, N] in one
  launch (the experts of an MoE layer)
* ``fp8_requant_1x128_to_128x1(q, s)`` -- (uint8 [M, K], [M, K/128]) ->
  (uint8 [K, M], float32 logical [K, M/128])   (backward-pass retiling, same page)
* ``fp8_gemm_blockscaled(A, sA, B, sB, sb_kind)`` -- bf16 [M, N]; FP32
  promotion every 128 K with both scales applied (why-be.why-be.co.kr post
  55081, Figure 7(b))
* ``fp8_gemm_blockscaled_q1x128(A, sA, B, sB, sb_kind)`` -- the same GEMM with
  its bf16 output 1x128-quantized in the epilogue -> (codes, scales)
* ``fp8_grouped_gemm_blockscaled(A, sA, B, sB, offsets)`` -- MoE experts
  (xn--jj0bz6z98ct0a29q.com post 362465: FP8-dispatched activations)
* ``*_pow2`` quantizers -- power-of-two scales (the smallest 2^e >= amax/448;
  why-be.why-be.co.kr post 55081 and sunipension.com post 314414: scaling
  factors that are integral powers of 2), and ``fp8_gemm_blockscaled_mx`` /
  ``fp8_grouped_gemm_blockscaled_mx``, which take such scales and let the
  tensor core apply them (no FP32 promotion)

Scale tensors are logical 2-D tensors with arbitrary strides; the default
outputs are "MN-major" views (stride 1 along the row/column index), the layout
the GEMM kernels read fastest.  All calls are asynchronous on the current
torch stream unless ``stream=`` is given.
"""
import ctypes
import os

import torch

__all__ = [
    "FP8Error", "capi", "library_path",
    "fp8_quant_act_1x128", "fp8_quant_w_128x128", "fp8_quant_w_128x128_batched",
    "fp8_requant_1x128_to_128x1",
    "fp8_gemm_blockscaled", "fp8_gemm_blockscaled_q1x128", "fp8_grouped_gemm_blockscaled",
    "fp8_get_device_status", "fp8_status_string", "fp8_selftest_bounded_wait",
    "fp8_mma_accumulation_probe",
    "fp8_quant_act_1x128_pow2", "fp8_quant_w_128x128_pow2", "fp8_quant_w_128x128_batched_pow2",
    "fp8_requant_1x128_to_128x1_pow2", "fp8_gemm_blockscaled_mx", "fp8_grouped_gemm_blockscaled_mx",
    "fp8_selftest_gemm_timeout", "fp8_swiglu_quant_1x128",
    "FP8_KMAJOR_NK", "FP8_ROWMAJOR_KN", "FP8_SB_BLOCK128x128", "FP8_SB_COL128x1",
]

HERE = os.path.dirname(os.path.abspath(__file__))
# FP8FG_BOUNDS=1 selects the debug build in which every device write is
# bounds-checked (an out-of-tile write is skipped and reported as
# FP8_ERR_DEVICE_BOUNDS in the device status word)
library_path = os.path.join(HERE, "libfp8fg_bounds.so" if os.environ.get("FP8FG_BOUNDS") == "1" else "libfp8fg.so")

FP8_OK = 0
FP8_KMAJOR_NK = 0
FP8_ROWMAJOR_KN = 1
FP8_SB_BLOCK128x128 = 0
FP8_SB_COL128x1 = 1

STATUS_NAMES = {
    0: "FP8_OK", 1: "FP8_ERR_NULL", 2: "FP8_ERR_ALIGN", 3: "FP8_ERR_SHAPE", 4: "FP8_ERR_CUDA",
    5: "FP8_ERR_DEVICE_TIMEOUT", 6: "FP8_ERR_ARG", 7: "FP8_ERR_DEVICE", 8: "FP8_ERR_DEVICE_GROUPS",
    9: "FP8_ERR_DEVICE_SCALES", 10: "FP8_ERR_DEVICE_BOUNDS",
}

# (name, argtypes) of every exported function; restype fp8_status_t (int) unless noted
_i64, _int, _vp = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
_SIGNATURES = {
    "fp8_quant_act_1x128": [_vp, _i64, _i64, _i64, _vp, _i64, _vp, _i64, _i64, _vp],
    "fp8_quant_w_128x128": [_vp, _i64, _i64, _i64, _vp, _i64, _int, _vp, _i64, _i64, _vp],
    "fp8_quant_w_128x128_batched": [_vp, _i64, _i64, _i64, _i64, _i64, _vp, _i64, _i64, _int, _vp, _i64, _i64,
                                    _i64, _vp],
    "fp8_requant_1x128_to_128x1": [_vp, _i64, _i64, _i64, _vp, _i64, _i64, _vp, _i64, _vp, _i64, _i64,
                                   _vp],
    "fp8_gemm_blockscaled": [_vp, _i64, _vp, _i64, _i64, _vp, _i64, _vp, _i64, _i64, _int, _vp, _i64,
                             _i64, _i64, _i64, _vp],
    "fp8_gemm_blockscaled_q1x128": [_vp, _i64, _vp, _i64, _i64, _vp, _i64, _vp, _i64, _i64, _int, _vp, _i64,
                                    _vp, _i64, _i64, _i64, _i64, _i64, _vp],
    "fp8_grouped_gemm_blockscaled": [_vp, _i64, _vp, _i64, _i64, _vp, _vp, _vp, _int, _i64, _i64, _i64,
                                     _vp, _i64, _vp],
    "fp8_quant_act_1x128_pow2": [_vp, _i64, _i64, _i64, _vp, _i64, _vp, _i64, _i64, _vp],
    "fp8_quant_w_128x128_pow2": [_vp, _i64, _i64, _i64, _vp, _i64, _int, _vp, _i64, _i64, _vp],
    "fp8_quant_w_128x128_batched_pow2": [_vp, _i64, _i64, _i64, _i64, _i64, _vp, _i64, _i64, _int, _vp, _i64,
                                         _i64, _i64, _vp],
    "fp8_requant_1x128_to_128x1_pow2": [_vp, _i64, _i64, _i64, _vp, _i64, _i64, _vp, _i64, _vp, _i64, _i64,
                                        _vp],
    "fp8_gemm_blockscaled_mx": [_vp, _i64, _vp, _i64, _i64, _vp, _i64, _vp, _i64, _i64, _int, _vp, _i64,
                                _i64, _i64, _i64, _vp],
    "fp8_grouped_gemm_blockscaled_mx": [_vp, _i64, _vp, _i64, _i64, _vp, _vp, _vp, _int, _i64, _i64, _i64,
                                        _vp, _i64, _vp],
    "fp8_selftest_gemm_timeout": [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, ctypes.c_uint64, _vp],
    "fp8_swiglu_quant_1x128": [_vp, _i64, _vp, _i64, _i64, _i64, _vp, _i64, _vp, _i64, _i64, _vp, _i64, _vp],
    "fp8_get_device_status": [_vp, ctypes.POINTER(ctypes.c_int32), _int],
    "fp8_selftest_bounded_wait": [ctypes.c_uint64, _vp],
    "fp8_mma_accumulation_probe": [_vp, _vp, _i64, _vp, _vp],
    "fp8_status_string": [_int],
    "fp8fg_version": [],
}


class FP8Error(RuntimeError):
    """A non-OK status returned by the library."""

    def __init__(self, status, where):
        self.status = int(status)
        super().__init__("%s: %s" % (where, fp8_status_string(status)))


_capi = None


def capi():
    """The ctypes handle of libfp8fg.so with argument types declared."""
    global _capi
    if _capi is None:
        if not os.path.exists(library_path):
            raise ImportError("libfp8fg.so is not built; run `python -m fp8_fine_grained_20_b300.build`")
        lib = ctypes.CDLL(library_path)
        for name, args in _SIGNATURES.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = ctypes.c_int
        lib.fp8_status_string.restype = ctypes.c_char_p
        _capi = lib
    return _capi


def fp8_status_string(status) -> str:
    return capi().fp8_status_string(int(status)).decode()


def _check(status, where):
    if status != FP8_OK:
        raise FP8Error(status, where)


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _need_cuda(*ts):
    for t in ts:
        if not (isinstance(t, torch.Tensor) and t.is_cuda):
            raise TypeError("fp8fg works on CUDA tensors only (no CPU path)")


def _row_major(t, name):
    if t.dim() != 2 or t.stride(1) != 1:
        raise ValueError("%s must be a 2-D tensor with unit stride along its last dimension" % name)


def _scale_out(rows, cols, layout, device):
    """Logical [rows, cols] float32 scale tensor; 'mn' = stride 1 along rows."""
    if layout == "mn":
        return torch.empty((cols, rows), dtype=torch.float32, device=device).t()
    if layout == "row":
        return torch.empty((rows, cols), dtype=torch.float32, device=device)
    raise ValueError("scale layout must be 'mn' or 'row'")


def fp8_quant_act_1x128(x, q=None, s=None, *, scale_layout="mn", stream=None):
    """1x128 activation quantization.  x: bf16 [M, K] (K % 128 == 0).
    Returns (q uint8 [M, K], s float32 logical [M, K/128])."""
    return _quant_act(x, q, s, scale_layout, stream, "fp8_quant_act_1x128")


def fp8_swiglu_quant_1x128(gate, up=None, q=None, s=None, y=None, *, scale_layout="mn", write_y=False,
                           stream=None):
    """SwiGLU recompute fused with 1x128 quantization.  gate, up: bf16 [M, F]
    (unit inner stride; F % 128 == 0); with up=None, `gate` is the fused
    [M, 2F] gate/up output and is split in halves.  Returns (q uint8 [M, F],
    s float32 logical [M, F/128]) and, with write_y=True or y given, also the
    bf16 SwiGLU values y [M, F]."""
    _need_cuda(gate)
    if up is None:
        F2 = gate.shape[1]
        gate, up = gate[:, :F2 // 2], gate[:, F2 // 2:]
    _need_cuda(up)
    _row_major(gate, "gate")
    _row_major(up, "up")
    if gate.dtype != torch.bfloat16 or up.dtype != torch.bfloat16 or gate.shape != up.shape:
        raise TypeError("gate and up must be bfloat16 tensors of one shape")
    M, F = gate.shape
    if q is None:
        q = torch.empty((M, F), dtype=torch.uint8, device=gate.device)
    if s is None:
        s = _scale_out(M, F // 128, scale_layout, gate.device)
    if y is None and write_y:
        y = torch.empty((M, F), dtype=torch.bfloat16, device=gate.device)
    _need_cuda(q, s)
    _row_major(q, "q")
    if y is not None:
        _need_cuda(y)
        _row_major(y, "y")
    _check(capi().fp8_swiglu_quant_1x128(_ptr(gate), gate.stride(0), _ptr(up), up.stride(0), M, F,
                                         _ptr(q), q.stride(0), _ptr(s), s.stride(0), s.stride(1),
                                         _ptr(y) if y is not None else None, y.stride(0) if y is not None else 0,
                                         _stream(stream)), "fp8_swiglu_quant_1x128")
    return (q, s, y) if y is not None else (q, s)


def fp8_quant_act_1x128_pow2(x, q=None, s=None, *, scale_layout="mn", stream=None):
    """fp8_quant_act_1x128 with power-of-two scales (smallest 2^e >= amax/448)."""
    return _quant_act(x, q, s, scale_layout, stream, "fp8_quant_act_1x128_pow2")


def _quant_act(x, q, s, scale_layout, stream, name):
    _need_cuda(x)
    _row_major(x, "x")
    if x.dtype != torch.bfloat16:
        raise TypeError("x must be bfloat16")
    M, K = x.shape
    if q is None:
        q = torch.empty((M, K), dtype=torch.uint8, device=x.device)
    if s is None:
        s = _scale_out(M, K // 128, scale_layout, x.device)
    _need_cuda(q, s)
    _row_major(q, "q")
    _check(getattr(capi(), name)(_ptr(x), M, K, x.stride(0), _ptr(q), q.stride(0), _ptr(s),
                                 s.stride(0), s.stride(1), _stream(stream)), name)
    return q, s


def fp8_quant_w_128x128(w, q=None, s=None, *, q_layout=FP8_KMAJOR_NK, stream=None):
    """128x128 weight quantization.  w: bf16 [K, N].  Returns (q, s) with q
    uint8 [N, K] for FP8_KMAJOR_NK (default) or [K, N] for FP8_ROWMAJOR_KN and
    s float32 [K/128, N/128]."""
    return _quant_w(w, q, s, q_layout, stream, "fp8_quant_w_128x128")


def fp8_quant_w_128x128_pow2(w, q=None, s=None, *, q_layout=FP8_KMAJOR_NK, stream=None):
    """fp8_quant_w_128x128 with power-of-two scales."""
    return _quant_w(w, q, s, q_layout, stream, "fp8_quant_w_128x128_pow2")


def _quant_w(w, q, s, q_layout, stream, name):
    _need_cuda(w)
    _row_major(w, "w")
    if w.dtype != torch.bfloat16:
        raise TypeError("w must be bfloat16")
    K, N = w.shape
    if q is None:
        shape = (N, K) if q_layout == FP8_KMAJOR_NK else (K, N)
        q = torch.empty(shape, dtype=torch.uint8, device=w.device)
    if s is None:
        s = torch.empty((K // 128, N // 128), dtype=torch.float32, device=w.device)
    _need_cuda(q, s)
    _row_major(q, "q")
    _check(getattr(capi(), name)(_ptr(w), K, N, w.stride(0), _ptr(q), q.stride(0), int(q_layout),
                                 _ptr(s), s.stride(0), s.stride(1), _stream(stream)), name)
    return q, s


def fp8_quant_w_128x128_batched(w, q=None, s=None, *, q_layout=FP8_KMAJOR_NK, stream=None):
    """128x128 quantization of G weights in one launch.  w: bf16 [G, K, N]
    (each weight row-major, any expert stride).  Returns (q, s) with q uint8
    [G, N, K] for FP8_KMAJOR_NK (default) or [G, K, N] for FP8_ROWMAJOR_KN and
    s float32 [G, K/128, N/128]."""
    return _quant_w_batched(w, q, s, q_layout, stream, "fp8_quant_w_128x128_batched")


def fp8_quant_w_128x128_batched_pow2(w, q=None, s=None, *, q_layout=FP8_KMAJOR_NK, stream=None):
    """fp8_quant_w_128x128_batched with power-of-two scales."""
    return _quant_w_batched(w, q, s, q_layout, stream, "fp8_quant_w_128x128_batched_pow2")


def _quant_w_batched(w, q, s, q_layout, stream, name):
    _need_cuda(w)
    if w.dim() != 3 or w.stride(2) != 1:
        raise ValueError("w must be a 3-D tensor with unit stride along its last dimension")
    if w.dtype != torch.bfloat16:
        raise TypeError("w must be bfloat16")
    G, K, N = w.shape
    if q is None:
        shape = (G, N, K) if q_layout == FP8_KMAJOR_NK else (G, K, N)
        q = torch.empty(shape, dtype=torch.uint8, device=w.device)
    if s is None:
        s = torch.empty((G, K // 128, N // 128), dtype=torch.float32, device=w.device)
    _need_cuda(q, s)
    if q.dim() != 3 or q.stride(2) != 1 or s.dim() != 3:
        raise ValueError("q must be 3-D with unit inner stride and s 3-D")
    _check(getattr(capi(), name)(_ptr(w), G, K, N, w.stride(1), w.stride(0), _ptr(q), q.stride(1),
                                 q.stride(0), int(q_layout), _ptr(s), s.stride(1), s.stride(2),
                                 s.stride(0), _stream(stream)), name)
    return q, s


def fp8_requant_1x128_to_128x1(q, s, qT=None, sT=None, *, scale_layout="mn", stream=None):
    """1x128 -> 128x1 requantization.  q uint8 [M, K], s logical [M, K/128].
    Returns (qT uint8 [K, M], sT float32 logical [K, M/128])."""
    return _requant(q, s, qT, sT, scale_layout, stream, "fp8_requant_1x128_to_128x1")


def fp8_requant_1x128_to_128x1_pow2(q, s, qT=None, sT=None, *, scale_layout="mn", stream=None):
    """fp8_requant_1x128_to_128x1 with power-of-two scales for the 128x1 groups."""
    return _requant(q, s, qT, sT, scale_layout, stream, "fp8_requant_1x128_to_128x1_pow2")


def _requant(q, s, qT, sT, scale_layout, stream, name):
    _need_cuda(q, s)
    _row_major(q, "q")
    M, K = q.shape
    if tuple(s.shape) != (M, K // 128):
        raise ValueError("s must have logical shape [M, K/128]")
    if qT is None:
        qT = torch.empty((K, M), dtype=torch.uint8, device=q.device)
    if sT is None:
        sT = _scale_out(K, M // 128, scale_layout, q.device)
    _need_cuda(qT, sT)
    _row_major(qT, "qT")
    _check(getattr(capi(), name)(_ptr(q), M, K, q.stride(0), _ptr(s), s.stride(0), s.stride(1),
                                 _ptr(qT), qT.stride(0), _ptr(sT), sT.stride(0), sT.stride(1),
                                 _stream(stream)), name)
    return qT, sT


def fp8_gemm_blockscaled(A, sA, B, sB, sb_kind=FP8_SB_BLOCK128x128, out=None, *, stream=None):
    """C bf16 [M, N] = block-scaled A [M, K] x B [N, K]^T.
    sA logical [M, K/128]; sB logical [K/128, N/128] (block) or [K/128, N] (per column)."""
    return _gemm(A, sA, B, sB, sb_kind, out, stream, "fp8_gemm_blockscaled")


def fp8_gemm_blockscaled_mx(A, sA, B, sB, sb_kind=FP8_SB_BLOCK128x128, out=None, *, stream=None):
    """fp8_gemm_blockscaled with power-of-two scales applied by the tensor core
    (every scale a power of two, e.g. from the _pow2 quantizers)."""
    return _gemm(A, sA, B, sB, sb_kind, out, stream, "fp8_gemm_blockscaled_mx")


def _gemm(A, sA, B, sB, sb_kind, out, stream, name):
    _need_cuda(A, sA, B, sB)
    _row_major(A, "A")
    _row_major(B, "B")
    M, K = A.shape
    N = B.shape[0]
    if B.shape[1] != K:
        raise ValueError("A and B must share K")
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=A.device)
    _need_cuda(out)
    _row_major(out, "out")
    _check(getattr(capi(), name)(_ptr(A), A.stride(0), _ptr(sA), sA.stride(0), sA.stride(1),
                                 _ptr(B), B.stride(0), _ptr(sB), sB.stride(0), sB.stride(1),
                                 int(sb_kind), _ptr(out), out.stride(0), M, N, K, _stream(stream)), name)
    return out


def fp8_gemm_blockscaled_q1x128(A, sA, B, sB, sb_kind=FP8_SB_BLOCK128x128, q=None, s=None, *,
                                scale_layout="mn", stream=None):
    """fp8_gemm_blockscaled whose bf16 output is 1x128-quantized in the epilogue.
    Returns (q uint8 [M, N], s float32 logical [M, N/128])."""
    _need_cuda(A, sA, B, sB)
    _row_major(A, "A")
    _row_major(B, "B")
    M, K = A.shape
    N = B.shape[0]
    if B.shape[1] != K:
        raise ValueError("A and B must share K")
    if q is None:
        q = torch.empty((M, N), dtype=torch.uint8, device=A.device)
    if s is None:
        s = _scale_out(M, N // 128, scale_layout, A.device)
    _need_cuda(q, s)
    _row_major(q, "q")
    _check(capi().fp8_gemm_blockscaled_q1x128(_ptr(A), A.stride(0), _ptr(sA), sA.stride(0), sA.stride(1),
                                              _ptr(B), B.stride(0), _ptr(sB), sB.stride(0), sB.stride(1),
                                              int(sb_kind), _ptr(q), q.stride(0), _ptr(s), s.stride(0),
                                              s.stride(1), M, N, K, _stream(stream)),
           "fp8_gemm_blockscaled_q1x128")
    return q, s


def fp8_grouped_gemm_blockscaled(A, sA, B, sB, offsets, out=None, *, stream=None):
    """Grouped GEMM.  A uint8 [M_total, K], sA logical [M_total, K/128]; B uint8
    [G, N, K] dense; sB float32 [G, K/128, N/128] dense; offsets int32 CUDA
    [G+1].  Returns C bf16 [M_total, N] (rows outside every expert untouched)."""
    return _grouped(A, sA, B, sB, offsets, out, stream, "fp8_grouped_gemm_blockscaled")


def fp8_grouped_gemm_blockscaled_mx(A, sA, B, sB, offsets, out=None, *, stream=None):
    """fp8_grouped_gemm_blockscaled with power-of-two scales applied by the tensor core."""
    return _grouped(A, sA, B, sB, offsets, out, stream, "fp8_grouped_gemm_blockscaled_mx")


def _grouped(A, sA, B, sB, offsets, out, stream, name):
    _need_cuda(A, sA, B, sB, offsets)
    _row_major(A, "A")
    if not (B.is_contiguous() and sB.is_contiguous() and offsets.is_contiguous()):
        raise ValueError("B, sB and offsets must be contiguous")
    if offsets.dtype != torch.int32:
        raise TypeError("offsets must be int32")
    M_total, K = A.shape
    G, N, Kb = B.shape
    if Kb != K or offsets.numel() != G + 1:
        raise ValueError("shape mismatch")
    if out is None:
        out = torch.empty((M_total, N), dtype=torch.bfloat16, device=A.device)
    _need_cuda(out)
    _row_major(out, "out")
    _check(getattr(capi(), name)(_ptr(A), A.stride(0), _ptr(sA), sA.stride(0), sA.stride(1),
                                 _ptr(B), _ptr(sB), _ptr(offsets), G, M_total, N, K,
                                 _ptr(out), out.stride(0), _stream(stream)), name)
    return out


def fp8_get_device_status(reset=True, stream=None) -> int:
    """Synchronise `stream` and return (and by default clear) the device status word."""
    v = ctypes.c_int32(0)
    _check(capi().fp8_get_device_status(_stream(stream), ctypes.byref(v), 1 if reset else 0),
           "fp8_get_device_status")
    return int(v.value)


def fp8_selftest_bounded_wait(timeout_ns=1000000, stream=None):
    """Run the bounded-wait self-test kernel (a wait that nothing satisfies);
    afterwards the device status word holds FP8_ERR_DEVICE_TIMEOUT (5)."""
    _check(capi().fp8_selftest_bounded_wait(int(timeout_ns), _stream(stream)), "fp8_selftest_bounded_wait")


def fp8_selftest_gemm_timeout(A, sA, B, sB, out=None, *, wait_ns=2000000, stream=None):
    """Run the GEMM failure-path self-test: fp8_gemm_blockscaled on dense A
    uint8 [M, K], sA float32 MN-major view [M, K/128] (sA.stride(0) == 1), B uint8
    [N, K], sB float32 [K/128, N/128], with every pipeline wait bounded by
    wait_ns and all loads after the first K-block withheld.  Afterwards the
    device status word holds FP8_ERR_DEVICE_TIMEOUT (5); `out` is undefined."""
    _need_cuda(A, sA, B, sB)
    M, K = A.shape
    N = B.shape[0]
    if not (A.is_contiguous() and B.is_contiguous() and sB.is_contiguous() and sA.stride(0) == 1
            and sA.stride(1) == M):
        raise ValueError("dense operands and an MN-major sA are required")
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=A.device)
    _check(capi().fp8_selftest_gemm_timeout(_ptr(A), _ptr(sA), _ptr(B), _ptr(sB), _ptr(out), M, N, K,
                                            int(wait_ns), _stream(stream)), "fp8_selftest_gemm_timeout")
    return out


def fp8_mma_accumulation_probe(A, B, out=None, *, stream=None):
    """D fp32 [128, 256] = A [128, K] x B [256, K]^T over E4M3 codes (uint8,
    dense), accumulated over the whole K in tensor memory (no promotion)."""
    _need_cuda(A, B)
    if A.dtype != torch.uint8 or B.dtype != torch.uint8 or not (A.is_contiguous() and B.is_contiguous()):
        raise TypeError("A and B must be contiguous uint8 code matrices")
    if A.shape[0] != 128 or B.shape[0] != 256 or A.shape[1] != B.shape[1]:
        raise ValueError("A must be [128, K] and B [256, K]")
    if out is None:
        out = torch.empty((128, 256), dtype=torch.float32, device=A.device)
    _need_cuda(out)
    _check(capi().fp8_mma_accumulation_probe(_ptr(A), _ptr(B), A.shape[1], _ptr(out), _stream(stream)),
           "fp8_mma_accumulation_probe")
    return out
