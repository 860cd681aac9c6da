"""GPU parity of the block-scaled FP8 GEMMs against the oracle's FP64 result.

Inputs are bf16 tensors from the seeded generators, quantized by the ORACLE, so
the GEMM kernels are tested in isolation.  Acceptance (per element):
|got - ref| <= 2^-7 |ref| + 1e-4 rms(ref), and relative Frobenius <= 5e-3.
Small shapes are compared in full (several tiles, a ragged 128-column N tail,
K = 128, more tiles than SMs); the full workloads on sampled outputs.
"""
import numpy as np
import pytest
import torch

import fp8_fine_grained_20_b300 as fg
import synth
from tests import gpu_util as gu

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


def scales_dev(s, layout):
    """Logical [R, C] scales on the device, MN-major ('mn') or row-major ('row')."""
    if layout == "mn":
        return gu.dev(np.ascontiguousarray(s.T)).t()
    return gu.dev(s)


def run_gemm(qa, sa, qbt, sb, sb_kind, sa_layout="mn"):
    A = gu.dev(qa)
    B = gu.dev(qbt)
    C = fg.fp8_gemm_blockscaled(A, scales_dev(sa, sa_layout), B, gu.dev(sb), sb_kind)
    torch.cuda.synchronize()
    return C


def fprop_operands(orc, M, N, K, seed, threads=None):
    x, _ = synth.activation(seed, M, K, outlier_frac=0.01)
    w = synth.weight(seed, K, N)
    qa, sa = orc.quant_act_1x128(x, threads=threads)
    qw, sw = orc.quant_w_128x128(w, threads=threads)
    return qa, sa, np.ascontiguousarray(qw.T), sw


def sample_positions(M, N, count, seed, tile_m=128, tile_n=256):
    """Random positions plus the four corners of every tile row/column band."""
    rng = np.random.default_rng(seed)
    ms = list(rng.integers(0, M, count))
    ns = list(rng.integers(0, N, count))
    for m in range(0, M, tile_m * max(1, M // tile_m // 16)):
        for n in range(0, N, tile_n * max(1, N // tile_n // 16)):
            for dm, dn in ((0, 0), (tile_m - 1, 0), (0, min(tile_n, N - n) - 1),
                           (tile_m - 1, min(tile_n, N - n) - 1)):
                if m + dm < M and n + dn < N:
                    ms.append(m + dm)
                    ns.append(n + dn)
    return np.array(ms, np.int64), np.array(ns, np.int64)


def test_gemm_tiny_end_to_end_config(orc):
    a, b, _ = synth.tiny_end_to_end(seed=1)
    qa, sa = orc.quant_act_1x128(a)
    qb, sb = orc.quant_w_128x128(b)
    qbt = np.ascontiguousarray(qb.T)
    ref = orc.gemm_blockscaled(qa, sa, qbt, sb, orc.SB_BLOCK128x128)
    C = run_gemm(qa, sa, qbt, sb, fg.FP8_SB_BLOCK128x128)
    gu.assert_gemm_close(gu.host_bf16_as_f64(C), ref, "tiny config")
    C2 = run_gemm(qa, sa, qbt, sb, fg.FP8_SB_BLOCK128x128, sa_layout="row")
    assert torch.equal(C, C2)


@pytest.mark.parametrize("M,N,K", [(128, 128, 128), (256, 384, 640), (384, 256, 128), (128, 640, 1024),
                                   (512, 896, 384)])
def test_gemm_forward_shapes(orc, M, N, K):
    qa, sa, qbt, sb = fprop_operands(orc, M, N, K, seed=M + N + K)
    ref = orc.gemm_blockscaled(qa, sa, qbt, sb, orc.SB_BLOCK128x128)
    C = run_gemm(qa, sa, qbt, sb, fg.FP8_SB_BLOCK128x128)
    gu.assert_gemm_close(gu.host_bf16_as_f64(C), ref, "forward %dx%dx%d" % (M, N, K))


def test_gemm_more_tiles_than_sms(orc, threads):
    M, N, K = 2048, 4864, 384                    # 16 x 19 = 304 tiles, last N tile ragged
    qa, sa, qbt, sb = fprop_operands(orc, M, N, K, seed=77)
    C = gu.host_bf16_as_f64(run_gemm(qa, sa, qbt, sb, fg.FP8_SB_BLOCK128x128))
    ms, ns = sample_positions(M, N, 20000, 5)
    ref = orc.gemm_blockscaled_sample(qa, sa, qbt, sb, orc.SB_BLOCK128x128, ms, ns, threads=threads)
    gu.assert_gemm_close(C[ms, ns], ref, "persistent multi-tile")


def test_gemm_is_deterministic(orc):
    qa, sa, qbt, sb = fprop_operands(orc, 256, 512, 1024, seed=3)
    C1 = run_gemm(qa, sa, qbt, sb, fg.FP8_SB_BLOCK128x128)
    C2 = run_gemm(qa, sa, qbt, sb, fg.FP8_SB_BLOCK128x128)
    assert torch.equal(C1, C2)


def wgrad_operands(orc, T, Cin, Cout, seed, threads=None):
    """dW[Cin, Cout] = X^T dY with both operands 128x1-quantized along tokens:
    X, dY bf16 are 1x128-quantized, then requantized to 128x1 (transposed)."""
    x = synth.wgrad_tensor(seed, 0, T, Cin)
    dy = synth.wgrad_tensor(seed, 1, T, Cout)
    qx, sx = orc.quant_act_1x128(x, threads=threads)
    qdy, sdy = orc.quant_act_1x128(dy, threads=threads)
    qxT, sxT = orc.requant_1x128_to_128x1(qx, sx, threads=threads)      # [Cin, T], [Cin, T/128]
    qdyT, sdyT = orc.requant_1x128_to_128x1(qdy, sdy, threads=threads)  # [Cout, T], [Cout, T/128]
    return qxT, sxT, qdyT, np.ascontiguousarray(sdyT.T)                # sB logical [T/128, Cout]


@pytest.mark.parametrize("T,Cin,Cout", [(256, 256, 384), (512, 384, 640), (128, 128, 128)])
def test_gemm_wgrad_shapes(orc, T, Cin, Cout):
    qa, sa, qbt, sb = wgrad_operands(orc, T, Cin, Cout, seed=T + Cin)
    ref = orc.gemm_blockscaled(qa, sa, qbt, sb, orc.SB_COL128x1)
    C = run_gemm(qa, sa, qbt, sb, fg.FP8_SB_COL128x1)
    gu.assert_gemm_close(gu.host_bf16_as_f64(C), ref, "wgrad %dx%dx%d" % (Cin, Cout, T))


def test_gemm_block_scales_strided(orc):
    # sB given column-major (stride 1 along kb) must give the same result
    qa, sa, qbt, sb = fprop_operands(orc, 256, 512, 384, seed=9)
    A, B = gu.dev(qa), gu.dev(qbt)
    sA = scales_dev(sa, "mn")
    C1 = fg.fp8_gemm_blockscaled(A, sA, B, gu.dev(sb), fg.FP8_SB_BLOCK128x128)
    C2 = fg.fp8_gemm_blockscaled(A, sA, B, gu.dev(np.ascontiguousarray(sb.T)).t(), fg.FP8_SB_BLOCK128x128)
    torch.cuda.synchronize()
    assert torch.equal(C1, C2)


def dgrad_operands(orc, T, Cin, Cout, seed, threads=None):
    """dX[T, Cin] = dY W^T: dY 1x128-quantized along Cout (the reduction), W
    128x128-quantized in its forward layout [Cin, Cout], which is already the
    K-major B operand of this GEMM; the 128x128 scale grid is read transposed."""
    dy = synth.wgrad_tensor(seed, 1, T, Cout)
    w = synth.weight(seed, Cin, Cout)
    qdy, sdy = orc.quant_act_1x128(dy, threads=threads)
    qw, sw = orc.quant_w_128x128(w, threads=threads)          # [Cin, Cout], [Cin/128, Cout/128]
    return qdy, sdy, qw, sw


@pytest.mark.parametrize("T,Cin,Cout", [(256, 384, 512), (128, 128, 128), (384, 256, 1024)])
def test_gemm_dgrad_shapes(orc, T, Cin, Cout):
    qa, sa, qw, sw = dgrad_operands(orc, T, Cin, Cout, seed=T + Cout)
    ref = orc.gemm_blockscaled(qa, sa, qw, np.ascontiguousarray(sw.T), orc.SB_BLOCK128x128)
    C = fg.fp8_gemm_blockscaled(gu.dev(qa), scales_dev(sa, "mn"), gu.dev(qw), gu.dev(sw).t(),
                                fg.FP8_SB_BLOCK128x128)
    torch.cuda.synchronize()
    gu.assert_gemm_close(gu.host_bf16_as_f64(C), ref, "dgrad %dx%dx%d" % (T, Cin, Cout))


def test_dgrad_end_to_end_with_gpu_quantizers(orc):
    """The backward-data path as a user runs it: dY 1x128 and W 128x128 (row-major
    codes) quantized on the GPU, then the GEMM; against the oracle's chain."""
    T, Cin, Cout = 256, 384, 640
    dy = synth.wgrad_tensor(41, 1, T, Cout)
    w = synth.weight(41, Cin, Cout)
    qdy, sdy = fg.fp8_quant_act_1x128(gu.bf16_dev(dy))
    qw, sw = fg.fp8_quant_w_128x128(gu.bf16_dev(w), q_layout=fg.FP8_ROWMAJOR_KN)
    C = fg.fp8_gemm_blockscaled(qdy, sdy, qw, sw.t(), fg.FP8_SB_BLOCK128x128)
    torch.cuda.synchronize()
    qa_r, sa_r, qw_r, sw_r = dgrad_operands(orc, T, Cin, Cout, seed=41)
    ref = orc.gemm_blockscaled(qa_r, sa_r, qw_r, np.ascontiguousarray(sw_r.T), orc.SB_BLOCK128x128)
    gu.assert_gemm_close(gu.host_bf16_as_f64(C), ref, "dgrad end to end")


# ---------------------------------------------------------------- grouped --

def moe_operands(orc, counts, N, K, seed, threads=None):
    """Per-expert activations (pad rows zero) and weights, quantized by the oracle."""
    G = len(counts)
    padded = (np.asarray(counts) + 127) // 128 * 128
    offsets = np.zeros(G + 1, np.int32)
    offsets[1:] = np.cumsum(padded)
    M_total = int(offsets[-1])
    x = np.zeros((M_total, K), np.uint16)
    for g in range(G):
        if counts[g]:
            xg, _ = synth.activation(seed + g, int(counts[g]), K, outlier_frac=0.0)
            x[offsets[g]:offsets[g] + counts[g]] = xg
    qa, sa = orc.quant_act_1x128(x, threads=threads)
    qb = np.empty((G, N, K), np.uint8)
    sb = np.empty((G, K // 128, N // 128), np.float32)
    for g in range(G):
        qw, sw = orc.quant_w_128x128(synth.weight(seed * 100 + g, K, N), threads=threads)
        qb[g] = qw.T
        sb[g] = sw
    return qa, sa, qb, sb, offsets


def run_grouped(qa, sa, qb, sb, offsets, M_extra=0, fill=None):
    M_total, K = qa.shape
    A = torch.zeros((M_total + M_extra, K), dtype=torch.uint8, device="cuda")
    A[:M_total] = gu.dev(qa)
    s_full = np.zeros((M_total + M_extra, K // 128), np.float32)
    s_full[:M_total] = sa
    out = torch.full((M_total + M_extra, qb.shape[1]), float("nan") if fill is None else fill,
                     dtype=torch.bfloat16, device="cuda")
    C = fg.fp8_grouped_gemm_blockscaled(A, scales_dev(s_full, "mn"), gu.dev(qb), gu.dev(sb),
                                        gu.dev(offsets), out=out)
    torch.cuda.synchronize()
    return C


def test_grouped_small_with_empty_and_exact_experts(orc):
    counts = [200, 0, 128, 37, 0, 300]            # empty experts, one of exactly 128 rows
    qa, sa, qb, sb, offsets = moe_operands(orc, counts, N=384, K=256, seed=31)
    ref = orc.grouped_gemm_blockscaled(qa, sa, qb, sb, offsets)
    C = run_grouped(qa, sa, qb, sb, offsets, M_extra=256)
    got = gu.host_bf16_as_f64(C)
    M_total = qa.shape[0]
    gu.assert_gemm_close(got[:M_total], ref, "grouped small")
    assert np.all(np.isnan(got[M_total:])), "rows beyond the last expert must stay untouched"
    # pad rows (zero codes, zero scales) give exact zeros
    for g in range(len(counts)):
        r0 = offsets[g] + counts[g]
        assert np.all(got[r0:offsets[g + 1]] == 0.0)


def test_grouped_single_expert(orc):
    qa, sa, qb, sb, offsets = moe_operands(orc, [300], N=256, K=384, seed=51)
    ref = orc.grouped_gemm_blockscaled(qa, sa, qb, sb, offsets)
    C = run_grouped(qa, sa, qb, sb, offsets)
    gu.assert_gemm_close(gu.host_bf16_as_f64(C[:300]), ref[:300], "single expert")
    assert float(C[300:].float().abs().max()) == 0.0          # pad rows


def test_grouped_all_experts_empty(orc):
    """Every expert empty: no tile is computed and the output is not written."""
    gu.cuda_or_skip()
    qa = np.zeros((128, 256), np.uint8)
    sa = np.zeros((128, 2), np.float32)
    qb = np.zeros((3, 256, 256), np.uint8)
    sb = np.ones((3, 2, 2), np.float32)
    C = run_grouped(qa, sa, qb, sb, np.zeros(4, np.int32), fill=7.0)
    assert bool((C == 7.0).all())
    assert fg.fp8_get_device_status(reset=True) == 0


def test_grouped_bad_offsets_report_device_status(orc):
    qa, sa, qb, sb, offsets = moe_operands(orc, [128, 128], N=256, K=128, seed=5)
    bad = offsets.copy()
    bad[1] = 100                                   # not a multiple of 128
    run_grouped(qa, sa, qb, sb, bad, fill=1.0)
    assert fg.fp8_get_device_status(reset=True) == 8


# ----------------------------------------------------------- full workloads --

def test_forward_full_workload_sampled(orc, threads):
    M, N, K = 8192, 18432, 7168
    x, _ = synth.activation(3, M, K, outlier_frac=0.0)
    w = synth.weight(3, K, N)
    qa, sa = orc.quant_act_1x128(x, threads=threads)
    qw, sw = orc.quant_w_128x128(w, threads=threads)
    qbt = np.ascontiguousarray(qw.T)
    del x, w, qw
    C = run_gemm(qa, sa, qbt, sw, fg.FP8_SB_BLOCK128x128)
    ms, ns = sample_positions(M, N, 4096, 11)
    got = gu.host_bf16_as_f64(C[torch.from_numpy(ms).cuda(), torch.from_numpy(ns).cuda()])
    ref = orc.gemm_blockscaled_sample(qa, sa, qbt, sw, orc.SB_BLOCK128x128, ms, ns, threads=threads)
    gu.assert_gemm_close(got, ref, "forward full workload")


def test_wgrad_full_workload_sampled(orc, threads):
    T, Cin, Cout = 8192, 7168, 18432
    qa, sa, qbt, sb = wgrad_operands(orc, T, Cin, Cout, seed=4, threads=threads)
    C = run_gemm(qa, sa, qbt, sb, fg.FP8_SB_COL128x1)
    ms, ns = sample_positions(Cin, Cout, 4096, 12)
    got = gu.host_bf16_as_f64(C[torch.from_numpy(ms).cuda(), torch.from_numpy(ns).cuda()])
    ref = orc.gemm_blockscaled_sample(qa, sa, qbt, sb, orc.SB_COL128x1, ms, ns, threads=threads)
    gu.assert_gemm_close(got, ref, "wgrad full workload")


def test_dgrad_full_workload_sampled(orc, threads):
    T, Cin, Cout = 8192, 7168, 18432
    qa, sa, qw, sw = dgrad_operands(orc, T, Cin, Cout, seed=6, threads=threads)
    C = fg.fp8_gemm_blockscaled(gu.dev(qa), scales_dev(sa, "mn"), gu.dev(qw), gu.dev(sw).t(),
                                fg.FP8_SB_BLOCK128x128)
    torch.cuda.synchronize()
    ms, ns = sample_positions(T, Cin, 4096, 14)
    got = gu.host_bf16_as_f64(C[torch.from_numpy(ms).cuda(), torch.from_numpy(ns).cuda()])
    sbT = np.ascontiguousarray(sw.T)
    ref = orc.gemm_blockscaled_sample(qa, sa, qw, sbT, orc.SB_BLOCK128x128, ms, ns, threads=threads)
    gu.assert_gemm_close(got, ref, "dgrad full workload")


def test_moe_full_workload_sampled(orc, threads):
    inp = synth.moe_inputs(seed=5)
    G, K, N = inp.w.shape
    qa, sa = orc.quant_act_1x128(inp.x, threads=threads)
    qb = np.empty((G, N, K), np.uint8)
    sb = np.empty((G, K // 128, N // 128), np.float32)
    for g in range(G):
        qw, sw = orc.quant_w_128x128(inp.w[g], threads=threads)
        qb[g] = qw.T
        sb[g] = sw
    C = run_grouped(qa, sa, qb, sb, inp.offsets)
    rng = np.random.default_rng(13)
    ms, ns = [], []
    for g in range(G):                             # routed rows of every expert, plus pad rows
        r0, n_g = int(inp.offsets[g]), int(inp.counts[g])
        if n_g:
            ms += list(r0 + rng.integers(0, n_g, 96))
            ns += list(rng.integers(0, N, 96))
    ms, ns = np.array(ms, np.int64), np.array(ns, np.int64)
    got = gu.host_bf16_as_f64(C[torch.from_numpy(ms).cuda(), torch.from_numpy(ns).cuda()])
    ref = orc.grouped_gemm_blockscaled_sample(qa, sa, qb, sb, inp.offsets, ms, ns, threads=threads)
    gu.assert_gemm_close(got, ref, "MoE full workload")
    for g in range(G):
        pad0, pad1 = int(inp.offsets[g] + inp.counts[g]), int(inp.offsets[g + 1])
        if pad1 > pad0:
            assert float(C[pad0:pad1].float().abs().max()) == 0.0


# ------------------------------------------------------ quantizing epilogue --

def _bf16_bits(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("kind,M,N,K", [("block", 256, 512, 384), ("block", 384, 384, 1024),
                                         ("col", 256, 384, 256), ("block", 128, 128, 128)])
def test_gemm_q1x128_epilogue_matches_oracle_quantizer(orc, kind, M, N, K):
    """Codes and scales of the quantizing epilogue equal the oracle's 1x128
    quantization of the same GEMM's bf16 output, bit for bit; the bf16 GEMM
    itself is checked against the FP64 oracle."""
    if kind == "block":
        qa, sa, qbt, sb = fprop_operands(orc, M, N, K, seed=M + N + K)
        sb_kind, osk = fg.FP8_SB_BLOCK128x128, orc.SB_BLOCK128x128
    else:
        qa, sa, qbt, sb = wgrad_operands(orc, K, M, N, seed=M + N + K)
        sb_kind, osk = fg.FP8_SB_COL128x1, orc.SB_COL128x1
    A, B, sA, sB = gu.dev(qa), gu.dev(qbt), scales_dev(sa, "mn"), gu.dev(sb)
    C = fg.fp8_gemm_blockscaled(A, sA, B, sB, sb_kind)
    q, s = fg.fp8_gemm_blockscaled_q1x128(A, sA, B, sB, sb_kind)
    torch.cuda.synchronize()
    gu.assert_gemm_close(gu.host_bf16_as_f64(C), orc.gemm_blockscaled(qa, sa, qbt, sb, osk), "bf16 GEMM")
    q_ref, s_ref = orc.quant_act_1x128(_bf16_bits(C))
    assert np.array_equal(gu.host(q), q_ref)
    assert np.array_equal(gu.host(s).view(np.uint32), s_ref.view(np.uint32))


def test_gemm_q1x128_epilogue_full_workload_matches_unfused():
    """Forward GEMM at full size: the fused epilogue equals GEMM -> 1x128
    quantizer on the GPU, every code and scale."""
    gu.cuda_or_skip()
    M, N, K = 8192, 18432, 7168
    g = torch.Generator(device="cuda")
    g.manual_seed(5)
    x = torch.randn((M, K), generator=g, device="cuda").to(torch.bfloat16)
    w = (torch.randn((K, N), generator=g, device="cuda") * 0.02).to(torch.bfloat16)
    qa, sa = fg.fp8_quant_act_1x128(x)
    qb, sb = fg.fp8_quant_w_128x128(w)
    del x, w
    C = fg.fp8_gemm_blockscaled(qa, sa, qb, sb)
    q_ref, s_ref = fg.fp8_quant_act_1x128(C)
    del C
    q, s = fg.fp8_gemm_blockscaled_q1x128(qa, sa, qb, sb)
    torch.cuda.synchronize()
    assert torch.equal(q, q_ref)
    assert torch.equal(s.contiguous().view(torch.int32), s_ref.contiguous().view(torch.int32))
    assert fg.fp8_get_device_status(reset=True) == 0
