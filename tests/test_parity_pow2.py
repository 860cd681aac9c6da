"""GPU parity of the power-of-two path against the CPU oracle.

* The *_pow2 quantizers must match the oracle's power-of-two reading bit for
  bit (every code byte and every scale bit): small tiles with edge values,
  ragged shapes, both weight code layouts, batched experts and the full
  quantizer workload.
* The hardware block-scaled GEMMs (fp8_gemm_blockscaled_mx and the grouped
  form) on operands the ORACLE quantized with power-of-two scales must meet
  the GEMM acceptance bound against the oracle's FP64 result, per element
  |d| <= 2^-7 |ref| + 1e-4 rms(ref) and relative Frobenius <= 5e-3: small
  shapes in full (K = 128, a ragged 128-column N tail, more tiles than SMs,
  K not a multiple of 512), the per-column (weight-gradient) and transposed
  (data-gradient) scale forms, the grouped form with empty experts, and the
  full workloads on sampled outputs.
"""
import numpy as np
import pytest
import torch

import fp8_fine_grained_20_b300 as fg
import synth
from tests import gpu_util as gu
from tests.test_parity_gemm import sample_positions, scales_dev
from tests.test_parity_quant import assert_bits_eq

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _device():
    gu.cuda_or_skip()
    fg.fp8_get_device_status(reset=True)
    yield
    gu.assert_device_status_clean()


@pytest.fixture(scope="module")
def threads(orc):
    return orc.default_threads()


# ------------------------------------------------------------- quantizers --

def check_act_pow2(orc, bits, scale_layout="mn"):
    q_ref, s_ref = orc.quant_act_1x128(bits, pow2=True)
    q, s = fg.fp8_quant_act_1x128_pow2(gu.bf16_dev(bits), scale_layout=scale_layout)
    torch.cuda.synchronize()
    assert_bits_eq(gu.host(s), s_ref, "pow2 scales")
    assert_bits_eq(gu.host(q), q_ref, "pow2 codes")


def test_act_pow2_tiny_config(orc):
    a, _, _ = synth.tiny_end_to_end(seed=1)
    check_act_pow2(orc, a)
    check_act_pow2(orc, a, scale_layout="row")


def test_act_pow2_edge_values(orc):
    rows = []
    tile = np.zeros(128, np.float32)
    tile[:6] = [1.0, -1.0, 0.004150390625, 0.004638671875, 3.814697265625e-06, -0.0078125]
    rows.append(tile)
    for j in (-20, 0, 7):                      # amax exactly 448 * 2^j, and one bf16 step above it
        r = np.zeros(128, np.float32)
        r[0] = 448.0 * 2.0 ** j
        rows.append(r)
        r = r.copy()
        r[0] = synth.f32_from_bf16_bits(synth.bf16_bits_from_f32(r[:1]) + np.uint16(1))[0]
        r[1] = -r[0] / 3
        rows.append(r)
    tiny = np.zeros(128, np.float32)           # the 2^-127 clamp
    tiny[0], tiny[1] = 2.0 ** -131, -(2.0 ** -133)
    rows.append(tiny)
    neg0 = np.zeros(128, np.float32)
    neg0[:64] = -0.0
    rows.append(neg0)                          # all-zero group with signed zeros
    big = np.zeros(128, np.float32)
    big[3] = 3.0e38                            # scale 2^120
    big[4] = -1.0e30
    rows.append(big)
    bits = synth.bf16_bits_from_f32(np.stack(rows))
    check_act_pow2(orc, np.concatenate([bits, bits[::-1]], axis=1))


def test_act_pow2_random_and_ragged(orc):
    x, _ = synth.activation(21, 77, 1024, outlier_frac=0.02)
    check_act_pow2(orc, x)
    w = synth.wgrad_tensor(21, 0, 300, 384)
    check_act_pow2(orc, w)


def test_act_pow2_full_workload(orc, threads):
    x, _ = synth.activation(2, 8192, 7168)
    q_ref, s_ref = orc.quant_act_1x128(x, threads=threads, pow2=True)
    q, s = fg.fp8_quant_act_1x128_pow2(gu.bf16_dev(x))
    torch.cuda.synchronize()
    assert_bits_eq(gu.host(s), s_ref, "pow2 scales, full workload")
    assert_bits_eq(gu.host(q), q_ref, "pow2 codes, full workload")


@pytest.mark.parametrize("layout", ["kmajor", "rowmajor"])
def test_weight_pow2(orc, layout):
    w = synth.weight(22, 384, 640)
    wf = synth.f32_from_bf16_bits(w)
    wf[5, 300] = 3.5                           # an outlier in block (0, 2)
    wf[200:328, 0:128] = 0.0                   # an all-zero block
    w = synth.bf16_bits_from_f32(wf)
    q_ref, s_ref = orc.quant_w_128x128(w, pow2=True)
    ql = fg.FP8_KMAJOR_NK if layout == "kmajor" else fg.FP8_ROWMAJOR_KN
    q, s = fg.fp8_quant_w_128x128_pow2(gu.bf16_dev(w), q_layout=ql)
    torch.cuda.synchronize()
    assert_bits_eq(gu.host(s), s_ref, "pow2 weight scales")
    want = q_ref.T if layout == "kmajor" else q_ref
    assert_bits_eq(gu.host(q), want, "pow2 weight codes")


def test_weight_pow2_batched_and_full(orc, threads):
    we = np.stack([synth.weight(40 + g, 256, 384) for g in range(3)])
    q, s = fg.fp8_quant_w_128x128_batched_pow2(gu.bf16_dev(we))
    torch.cuda.synchronize()
    for g in range(3):
        q_ref, s_ref = orc.quant_w_128x128(we[g], pow2=True)
        assert_bits_eq(gu.host(s[g]), s_ref, "batched pow2 scales %d" % g)
        assert_bits_eq(gu.host(q[g]), q_ref.T, "batched pow2 codes %d" % g)
    w = synth.weight(2, 7168, 18432)
    q_ref, s_ref = orc.quant_w_128x128(w, threads=threads, pow2=True)
    q, s = fg.fp8_quant_w_128x128_pow2(gu.bf16_dev(w))
    torch.cuda.synchronize()
    assert_bits_eq(gu.host(s), s_ref, "pow2 weight scales, full workload")
    assert_bits_eq(gu.host(q), np.ascontiguousarray(q_ref.T), "pow2 weight codes, full workload")


def test_requant_pow2_small_and_full(orc, threads):
    for seed, (M, K) in ((30, (256, 384)), (31, (384, 128))):
        x = synth.wgrad_tensor(seed, 0, M, K)
        q1, s1 = orc.quant_act_1x128(x, pow2=True)
        qT_ref, sT_ref = orc.requant_1x128_to_128x1(q1, s1, pow2=True)
        qT, sT = fg.fp8_requant_1x128_to_128x1_pow2(gu.dev(q1), scales_dev(s1, "mn"))
        torch.cuda.synchronize()
        assert_bits_eq(gu.host(sT), sT_ref, "pow2 requant scales %dx%d" % (M, K))
        assert_bits_eq(gu.host(qT), qT_ref, "pow2 requant codes %dx%d" % (M, K))
    x = synth.wgrad_tensor(4, 1, 8192, 7168)
    q1, s1 = orc.quant_act_1x128(x, threads=threads, pow2=True)
    qT_ref, sT_ref = orc.requant_1x128_to_128x1(q1, s1, threads=threads, pow2=True)
    qT, sT = fg.fp8_requant_1x128_to_128x1_pow2(gu.dev(q1), scales_dev(s1, "mn"))
    torch.cuda.synchronize()
    assert_bits_eq(gu.host(sT), sT_ref, "pow2 requant scales, full workload")
    assert_bits_eq(gu.host(qT), qT_ref, "pow2 requant codes, full workload")


# ----------------------------------------------------------------- GEMMs --

def fprop_pow2(orc, M, N, K, seed, threads=None):
    x, _ = synth.activation(seed, M, K, outlier_frac=0.01)
    w = synth.weight(seed, K, N)
    qa, sa = orc.quant_act_1x128(x, threads=threads, pow2=True)
    qw, sw = orc.quant_w_128x128(w, threads=threads, pow2=True)
    return qa, sa, np.ascontiguousarray(qw.T), sw


def wgrad_pow2(orc, T, Cin, Cout, seed, threads=None):
    x = synth.wgrad_tensor(seed, 0, T, Cin)
    dy = synth.wgrad_tensor(seed, 1, T, Cout)
    qx, sx = orc.quant_act_1x128(x, threads=threads, pow2=True)
    qdy, sdy = orc.quant_act_1x128(dy, threads=threads, pow2=True)
    qxT, sxT = orc.requant_1x128_to_128x1(qx, sx, threads=threads, pow2=True)
    qdyT, sdyT = orc.requant_1x128_to_128x1(qdy, sdy, threads=threads, pow2=True)
    return qxT, sxT, qdyT, np.ascontiguousarray(sdyT.T)


def run_mx(qa, sa, qbt, sb, sb_kind):
    C = fg.fp8_gemm_blockscaled_mx(gu.dev(qa), scales_dev(sa, "mn"), gu.dev(qbt), gu.dev(sb), sb_kind)
    torch.cuda.synchronize()
    return C


def test_mx_tiny_config(orc):
    a, b, _ = synth.tiny_end_to_end(seed=1)
    qa, sa = orc.quant_act_1x128(a, pow2=True)
    qb, sb = orc.quant_w_128x128(b, pow2=True)
    qbt = np.ascontiguousarray(qb.T)
    ref = orc.gemm_blockscaled(qa, sa, qbt, sb, orc.SB_BLOCK128x128)
    C = run_mx(qa, sa, qbt, sb, fg.FP8_SB_BLOCK128x128)
    gu.assert_gemm_close(gu.host_bf16_as_f64(C), ref, "mx tiny config")
    # the same operands through the promoting kernel agree within the bound too
    C2 = fg.fp8_gemm_blockscaled(gu.dev(qa), scales_dev(sa, "mn"), gu.dev(qbt), gu.dev(sb), fg.FP8_SB_BLOCK128x128)
    torch.cuda.synchronize()
    gu.assert_gemm_close(gu.host_bf16_as_f64(C2), ref, "promoting kernel on power-of-two operands")


@pytest.mark.parametrize("M,N,K", [(128, 128, 128), (256, 384, 640), (384, 256, 128), (128, 640, 1152),
                                   (512, 896, 384), (256, 256, 2560)])
def test_mx_forward_shapes(orc, M, N, K):
    qa, sa, qbt, sb = fprop_pow2(orc, M, N, K, seed=M + N + K)
    ref = orc.gemm_blockscaled(qa, sa, qbt, sb, orc.SB_BLOCK128x128)
    C = run_mx(qa, sa, qbt, sb, fg.FP8_SB_BLOCK128x128)
    gu.assert_gemm_close(gu.host_bf16_as_f64(C), ref, "mx forward %dx%dx%d" % (M, N, K))


def test_mx_varied_scales_per_row_and_block(orc):
    """Scales spread over 2^-4 .. 2^4 per row, per K-block and per block (or per
    column), so a scale read from the wrong row, column or K-block changes that
    K-block's share of an output by a factor of 2 or more."""
    M, N, K = 256, 512, 1024
    rng = np.random.default_rng(7)
    codes = np.arange(0x00, 0x7F)
    qa = rng.choice(codes, size=(M, K)).astype(np.uint8) | (rng.integers(0, 2, (M, K)) << 7).astype(np.uint8)
    qbt = rng.choice(codes, size=(N, K)).astype(np.uint8) | (rng.integers(0, 2, (N, K)) << 7).astype(np.uint8)
    sa = (2.0 ** rng.integers(-4, 5, (M, K // 128))).astype(np.float32)
    sb = (2.0 ** rng.integers(-4, 5, (K // 128, N // 128))).astype(np.float32)
    ref = orc.gemm_blockscaled(qa, sa, qbt, sb, orc.SB_BLOCK128x128)
    C = run_mx(qa, sa, qbt, sb, fg.FP8_SB_BLOCK128x128)
    gu.assert_gemm_close(gu.host_bf16_as_f64(C), ref, "mx varied scales")
    sbc = (2.0 ** rng.integers(-4, 5, (K // 128, N))).astype(np.float32)
    ref = orc.gemm_blockscaled(qa, sa, qbt, sbc, orc.SB_COL128x1)
    C = run_mx(qa, sa, qbt, sbc, fg.FP8_SB_COL128x1)
    gu.assert_gemm_close(gu.host_bf16_as_f64(C), ref, "mx varied per-column scales")


def test_mx_more_tiles_than_sms(orc, threads):
    M, N, K = 2048, 4864, 384
    qa, sa, qbt, sb = fprop_pow2(orc, M, N, K, seed=78)
    C = gu.host_bf16_as_f64(run_mx(qa, sa, qbt, sb, fg.FP8_SB_BLOCK128x128))
    ms, ns = sample_positions(M, N, 20000, 6)
    ref = orc.gemm_blockscaled_sample(qa, sa, qbt, sb, orc.SB_BLOCK128x128, ms, ns, threads=threads)
    gu.assert_gemm_close(C[ms, ns], ref, "mx persistent multi-tile")


def test_mx_is_deterministic(orc):
    qa, sa, qbt, sb = fprop_pow2(orc, 256, 512, 1024, seed=4)
    assert torch.equal(run_mx(qa, sa, qbt, sb, fg.FP8_SB_BLOCK128x128),
                       run_mx(qa, sa, qbt, sb, fg.FP8_SB_BLOCK128x128))


@pytest.mark.parametrize("T,Cin,Cout", [(256, 256, 384), (640, 384, 640), (128, 128, 128)])
def test_mx_wgrad_shapes(orc, T, Cin, Cout):
    qa, sa, qbt, sb = wgrad_pow2(orc, T, Cin, Cout, seed=T + Cin)
    ref = orc.gemm_blockscaled(qa, sa, qbt, sb, orc.SB_COL128x1)
    C = run_mx(qa, sa, qbt, sb, fg.FP8_SB_COL128x1)
    gu.assert_gemm_close(gu.host_bf16_as_f64(C), ref, "mx wgrad %dx%dx%d" % (Cin, Cout, T))


def test_mx_dgrad_transposed_scale_view(orc):
    T, Cin, Cout = 384, 256, 1024
    dy = synth.wgrad_tensor(43, 1, T, Cout)
    w = synth.weight(43, Cin, Cout)
    qa, sa = orc.quant_act_1x128(dy, pow2=True)
    qw, sw = orc.quant_w_128x128(w, pow2=True)
    ref = orc.gemm_blockscaled(qa, sa, qw, np.ascontiguousarray(sw.T), orc.SB_BLOCK128x128)
    C = fg.fp8_gemm_blockscaled_mx(gu.dev(qa), scales_dev(sa, "mn"), gu.dev(qw), gu.dev(sw).t(),
                                   fg.FP8_SB_BLOCK128x128)
    torch.cuda.synchronize()
    gu.assert_gemm_close(gu.host_bf16_as_f64(C), ref, "mx dgrad")


def test_mx_end_to_end_with_gpu_pow2_quantizers(orc):
    """Forward and weight gradient as a user runs them: GPU pow2 quantizers feed
    the MX GEMM; against the oracle's chain."""
    M, N, K = 256, 384, 512
    x, _ = synth.activation(44, M, K)
    w = synth.weight(44, K, N)
    qa, sa = fg.fp8_quant_act_1x128_pow2(gu.bf16_dev(x))
    qb, sb = fg.fp8_quant_w_128x128_pow2(gu.bf16_dev(w))
    C = fg.fp8_gemm_blockscaled_mx(qa, sa, qb, sb, fg.FP8_SB_BLOCK128x128)
    torch.cuda.synchronize()
    qa_r, sa_r = orc.quant_act_1x128(x, pow2=True)
    qb_r, sb_r = orc.quant_w_128x128(w, pow2=True)
    ref = orc.gemm_blockscaled(qa_r, sa_r, np.ascontiguousarray(qb_r.T), sb_r, orc.SB_BLOCK128x128)
    gu.assert_gemm_close(gu.host_bf16_as_f64(C), ref, "mx forward end to end")
    T, Cin, Cout = 384, 256, 384
    xw = synth.wgrad_tensor(45, 0, T, Cin)
    dy = synth.wgrad_tensor(45, 1, T, Cout)
    qx, sx = fg.fp8_quant_act_1x128_pow2(gu.bf16_dev(xw))
    qdy, sdy = fg.fp8_quant_act_1x128_pow2(gu.bf16_dev(dy))
    qxT, sxT = fg.fp8_requant_1x128_to_128x1_pow2(qx, sx)
    qdyT, sdyT = fg.fp8_requant_1x128_to_128x1_pow2(qdy, sdy)
    dW = fg.fp8_gemm_blockscaled_mx(qxT, sxT, qdyT, sdyT.t(), fg.FP8_SB_COL128x1)
    torch.cuda.synchronize()
    qa_r, sa_r, qbt_r, sb_r = wgrad_pow2(orc, T, Cin, Cout, seed=45)
    ref = orc.gemm_blockscaled(qa_r, sa_r, qbt_r, sb_r, orc.SB_COL128x1)
    gu.assert_gemm_close(gu.host_bf16_as_f64(dW), ref, "mx wgrad end to end")


def test_mx_non_power_of_two_scale_is_reported(orc):
    qa, sa, qbt, sb = fprop_pow2(orc, 128, 256, 256, seed=46)
    sb = sb.copy()
    sb[1, 0] *= np.float32(1.5)
    run_mx(qa, sa, qbt, sb, fg.FP8_SB_BLOCK128x128)
    assert fg.fp8_get_device_status(reset=True) == 9     # FP8_ERR_DEVICE_SCALES


def test_mx_strided_scale_layouts(orc):
    """Row-major A scales (stride K/128 along the rows) and per-column B scales
    stored transposed (stride K/128 along the columns): the scale copier takes
    one scale per copy instead of four, with the same result."""
    qa, sa, qbt, sb = wgrad_pow2(orc, 384, 256, 384, seed=91)
    assert sb.shape == (3, 384)
    ref = orc.gemm_blockscaled(qa, sa, qbt, sb, orc.SB_COL128x1)
    sa_row = gu.dev(np.ascontiguousarray(sa))              # [M, K/128], row-major
    sb_t = gu.dev(np.ascontiguousarray(sb.T)).t()           # logical [K/128, N], strides (1, K/128)
    C = fg.fp8_gemm_blockscaled_mx(gu.dev(qa), sa_row, gu.dev(qbt), sb_t, fg.FP8_SB_COL128x1)
    torch.cuda.synchronize()
    assert fg.fp8_get_device_status(reset=True) == 0
    gu.assert_gemm_close(gu.host_bf16_as_f64(C), ref, "mx strided scale layouts")


@pytest.mark.parametrize("bad", [1.5, np.inf, -1.0])
def test_mx_invalid_column_scale_is_reported(orc, bad):
    """A per-column scale that is not a power of two (x1.5), infinite or
    negative sets FP8_ERR_DEVICE_SCALES."""
    qa, sa, qbt, sb = wgrad_pow2(orc, 256, 128, 256, seed=47)
    sb = sb.copy()
    sb[1, 77] = np.float32(sb[1, 77] * np.float32(bad))
    run_mx(qa, sa, qbt, sb, fg.FP8_SB_COL128x1)
    assert fg.fp8_get_device_status(reset=True) == 9     # FP8_ERR_DEVICE_SCALES


def test_mx_smallest_power_of_two_scale_is_accepted(orc):
    """2^-127 (the fp32 subnormal 0x00400000, UE8M0 byte 0) is a valid scale
    for A and for a B column."""
    qa, sa, qbt, sb = wgrad_pow2(orc, 256, 128, 256, seed=48)
    sa = sa.copy()
    sb = sb.copy()
    tiny = np.array([0x00400000], np.uint32).view(np.float32)[0]
    sa[3, 0] = tiny
    sb[1, 10] = tiny
    ref = orc.gemm_blockscaled(qa, sa, qbt, sb, orc.SB_COL128x1)
    C = run_mx(qa, sa, qbt, sb, fg.FP8_SB_COL128x1)
    assert fg.fp8_get_device_status(reset=True) == 0
    gu.assert_gemm_close(gu.host_bf16_as_f64(C), ref, "mx scale 2^-127")


def moe_pow2(orc, counts, N, K, seed, threads=None):
    G = len(counts)
    padded = (np.asarray(counts) + 127) // 128 * 128
    offsets = np.zeros(G + 1, np.int32)
    offsets[1:] = np.cumsum(padded)
    x = np.zeros((int(offsets[-1]), K), np.uint16)
    for g in range(G):
        if counts[g]:
            xg, _ = synth.activation(seed + g, int(counts[g]), K, outlier_frac=0.0)
            x[offsets[g]:offsets[g] + counts[g]] = xg
    qa, sa = orc.quant_act_1x128(x, threads=threads, pow2=True)
    qb = np.empty((G, N, K), np.uint8)
    sb = np.empty((G, K // 128, N // 128), np.float32)
    for g in range(G):
        qw, sw = orc.quant_w_128x128(synth.weight(seed * 100 + g, K, N), threads=threads, pow2=True)
        qb[g] = qw.T
        sb[g] = sw
    return qa, sa, qb, sb, offsets


def run_grouped_mx(qa, sa, qb, sb, offsets, M_extra=0):
    M_total, K = qa.shape
    A = torch.zeros((M_total + M_extra, K), dtype=torch.uint8, device="cuda")
    A[:M_total] = gu.dev(qa)
    s_full = np.zeros((M_total + M_extra, K // 128), np.float32)
    s_full[:M_total] = sa
    out = torch.full((M_total + M_extra, qb.shape[1]), float("nan"), dtype=torch.bfloat16, device="cuda")
    C = fg.fp8_grouped_gemm_blockscaled_mx(A, scales_dev(s_full, "mn"), gu.dev(qb), gu.dev(sb),
                                           gu.dev(offsets), out=out)
    torch.cuda.synchronize()
    return C


def test_mx_grouped_small_with_empty_experts(orc):
    counts = [200, 0, 128, 37, 0, 300]
    qa, sa, qb, sb, offsets = moe_pow2(orc, counts, N=384, K=640, seed=32)
    ref = orc.grouped_gemm_blockscaled(qa, sa, qb, sb, offsets)
    C = run_grouped_mx(qa, sa, qb, sb, offsets, M_extra=256)
    got = gu.host_bf16_as_f64(C)
    M_total = qa.shape[0]
    gu.assert_gemm_close(got[:M_total], ref, "mx grouped small")
    assert np.all(np.isnan(got[M_total:])), "rows beyond the last expert must stay untouched"
    for g in range(len(counts)):
        assert np.all(got[offsets[g] + counts[g]:offsets[g + 1]] == 0.0)


def test_mx_grouped_all_experts_empty(orc):
    """Every expert empty: no tile, no scale group (the copier and converter
    warps have nothing to do) and the output is not written."""
    gu.cuda_or_skip()
    qa = np.zeros((128, 256), np.uint8)
    sa = np.zeros((128, 2), np.float32)
    qb = np.zeros((3, 256, 256), np.uint8)
    sb = np.ones((3, 2, 2), np.float32)
    out = torch.full((128, 256), 7.0, dtype=torch.bfloat16, device="cuda")
    fg.fp8_grouped_gemm_blockscaled_mx(gu.dev(qa), scales_dev(sa, "mn"), gu.dev(qb), gu.dev(sb),
                                       gu.dev(np.zeros(4, np.int32)), out=out)
    torch.cuda.synchronize()
    assert bool((out == 7.0).all())
    assert fg.fp8_get_device_status(reset=True) == 0


def test_mx_grouped_bad_offsets_report_device_status(orc):
    counts = [128, 128]
    qa, sa, qb, sb, offsets = moe_pow2(orc, counts, N=256, K=128, seed=5)
    bad = offsets.copy()
    bad[1] = 100                                   # not a multiple of 128
    run_grouped_mx(qa, sa, qb, sb, bad)
    assert fg.fp8_get_device_status(reset=True) == 8


# ----------------------------------------------------------- full workloads --

def test_mx_forward_full_workload_sampled(orc, threads):
    M, N, K = 8192, 18432, 7168
    qa, sa, qbt, sb = fprop_pow2(orc, M, N, K, seed=3, threads=threads)
    C = run_mx(qa, sa, qbt, sb, fg.FP8_SB_BLOCK128x128)
    ms, ns = sample_positions(M, N, 4096, 21)
    got = gu.host_bf16_as_f64(C[torch.from_numpy(ms).cuda(), torch.from_numpy(ns).cuda()])
    ref = orc.gemm_blockscaled_sample(qa, sa, qbt, sb, orc.SB_BLOCK128x128, ms, ns, threads=threads)
    gu.assert_gemm_close(got, ref, "mx forward full workload")


def test_mx_wgrad_full_workload_sampled(orc, threads):
    T, Cin, Cout = 8192, 7168, 18432
    qa, sa, qbt, sb = wgrad_pow2(orc, T, Cin, Cout, seed=4, threads=threads)
    C = run_mx(qa, sa, qbt, sb, fg.FP8_SB_COL128x1)
    ms, ns = sample_positions(Cin, Cout, 4096, 22)
    got = gu.host_bf16_as_f64(C[torch.from_numpy(ms).cuda(), torch.from_numpy(ns).cuda()])
    ref = orc.gemm_blockscaled_sample(qa, sa, qbt, sb, orc.SB_COL128x1, ms, ns, threads=threads)
    gu.assert_gemm_close(got, ref, "mx wgrad full workload")


def test_mx_moe_full_workload_sampled(orc, threads):
    inp = synth.moe_inputs(seed=5)
    G, K, N = inp.w.shape
    qa, sa = orc.quant_act_1x128(inp.x, threads=threads, pow2=True)
    qb = np.empty((G, N, K), np.uint8)
    sb = np.empty((G, K // 128, N // 128), np.float32)
    for g in range(G):
        qw, sw = orc.quant_w_128x128(inp.w[g], threads=threads, pow2=True)
        qb[g] = qw.T
        sb[g] = sw
    C = run_grouped_mx(qa, sa, qb, sb, inp.offsets)
    rng = np.random.default_rng(23)
    ms, ns = [], []
    for g in range(G):
        r0, n_g = int(inp.offsets[g]), int(inp.counts[g])
        if n_g:
            ms += list(r0 + rng.integers(0, n_g, 96))
            ns += list(rng.integers(0, N, 96))
    ms, ns = np.array(ms, np.int64), np.array(ns, np.int64)
    got = gu.host_bf16_as_f64(C[torch.from_numpy(ms).cuda(), torch.from_numpy(ns).cuda()])
    ref = orc.grouped_gemm_blockscaled_sample(qa, sa, qb, sb, inp.offsets, ms, ns, threads=threads)
    gu.assert_gemm_close(got, ref, "mx MoE full workload")
    for g in range(G):
        pad0, pad1 = int(inp.offsets[g] + inp.counts[g]), int(inp.offsets[g + 1])
        if pad1 > pad0:
            assert float(C[pad0:pad1].float().abs().max()) == 0.0
