"""GPU parity of the three quantizers against the CPU oracle: every code byte
and every scale bit must match, at small sizes with edge values and ragged
shapes and at the full quantizer workload ([8192, 7168] activation,
[7168, 18432] weight)."""
import numpy as np
import pytest
import torch

import fp8_fine_grained_20_b300 as fg
import synth
from tests import gpu_util as gu
from tests.test_oracle_pins import adversarial_pairs, load_worked_tile

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _device():
    gu.cuda_or_skip()
    fg.fp8_get_device_status(reset=True)
    yield
    gu.assert_device_status_clean()


def bits_eq(a, b):
    a = np.ascontiguousarray(a)
    b = np.ascontiguousarray(b)
    if a.dtype == np.float32:
        a, b = a.view(np.uint32), np.ascontiguousarray(b, np.float32).view(np.uint32)
    return a.shape == b.shape and np.array_equal(a, b)


def assert_bits_eq(got, want, what):
    got = np.ascontiguousarray(got)
    want = np.ascontiguousarray(want)
    assert got.shape == want.shape, (what, got.shape, want.shape)
    if got.dtype == np.float32:
        gv, wv = got.view(np.uint32), want.astype(np.float32).view(np.uint32)
    else:
        gv, wv = got, want
    if not np.array_equal(gv, wv):
        idx = np.argwhere(gv != wv)
        i = tuple(idx[0])
        raise AssertionError("%s: %d mismatches, first at %s: got %r want %r"
                             % (what, len(idx), i, got[i], want[i]))


def run_act(bits, scale_layout="mn", ldx_pad=0, ldq_pad=0):
    M, K = bits.shape
    xpad = np.zeros((M, K + ldx_pad), np.uint16)
    xpad[:, :K] = bits
    x = gu.bf16_dev(xpad)[:, :K]
    q = torch.empty((M, K + ldq_pad), dtype=torch.uint8, device="cuda")[:, :K]
    qg, sg = fg.fp8_quant_act_1x128(x, q=q, scale_layout=scale_layout)
    torch.cuda.synchronize()
    return gu.host(qg), gu.host(sg)


def check_act(orc, bits, **kw):
    q_ref, s_ref = orc.quant_act_1x128(bits)
    q, s = run_act(bits, **kw)
    assert_bits_eq(s, s_ref, "scales")
    assert_bits_eq(q, q_ref, "codes")


def test_act_tiny_end_to_end_config(orc):
    a, _, _ = synth.tiny_end_to_end(seed=1)
    check_act(orc, a, scale_layout="mn")
    check_act(orc, a, scale_layout="row")


def edge_tiles():
    """128-wide groups that exercise every special case of the quantizer."""
    tiles = []
    # the hand-worked tile (s = 1) and the same tile x 2^-10
    t = np.zeros(128, np.float32)
    for pos, val, _ in load_worked_tile():
        t[pos] = val
    tiles += [t, t * np.float32(2.0 ** -10)]
    # all zero, negative zeros, single outlier, ties at several scales
    tiles.append(np.zeros(128, np.float32))
    tiles.append(np.full(128, -0.0, np.float32))
    z = np.zeros(128, np.float32)
    z[77] = -3.5
    tiles.append(z)
    ramp = np.linspace(-448, 448, 128).astype(np.float32)
    tiles += [ramp, ramp * np.float32(2.0 ** 20), ramp * np.float32(2.0 ** -30)]
    # bf16 subnormals: amax subnormal -> fp32-subnormal scale (exact-quotient path)
    sub = (np.arange(128, dtype=np.float32) - 64) * np.float32(2.0 ** -133)
    tiles.append(sub)
    sub2 = sub.copy()
    sub2[0] = np.float32(2.0 ** -118)          # s ~ 2^-127: subnormal scale, normal values
    tiles.append(sub2)
    # largest bf16 magnitude, and tiny values next to it (quotients underflow)
    big = np.zeros(128, np.float32)
    big[0] = np.float32(3.3895314e38)
    big[1:] = np.float32(1e-30) * np.arange(1, 128, dtype=np.float32)
    big[2] = -np.float32(1e-30)
    tiles.append(big)
    # adversarial (x, amax) pairs where RN(x/s) differs from RN(x * RN(1/s))
    for x, amax in adversarial_pairs():
        r = np.zeros(128, np.float32)
        r[0], r[1], r[2], r[3] = amax, x, -x, -amax
        tiles.append(r)
    return np.stack(tiles).astype(np.float32)


def test_act_edge_values(orc):
    tiles = edge_tiles()
    bits = synth.bf16_bits_from_f32(tiles)
    # one group per row, and the same groups packed 3 per row
    check_act(orc, bits)
    n = tiles.shape[0] // 3 * 3
    check_act(orc, bits[:n].reshape(n // 3, 384), scale_layout="row")


def test_act_codec_sweep_all_bf16_magnitudes(orc):
    # every finite bf16 with |x| <= 448, in groups whose amax is 448 (s = 1):
    # the GPU's E4M3 rounding of every such value against the oracle's
    mags = np.arange(0x0000, 0x43E1, dtype=np.uint16)          # +0 .. 448
    vals = np.concatenate([mags, mags | np.uint16(0x8000)])
    pad = (-len(vals)) % 127
    vals = np.concatenate([vals, np.zeros(pad, np.uint16)]).reshape(-1, 127)
    groups = np.concatenate([np.full((vals.shape[0], 1), 0x43E0, np.uint16), vals], axis=1)
    check_act(orc, groups)


def exhaustive_ratio_groups(amax_exp):
    """Groups covering every bf16 (amax, x) significand pair with x = amax * 2^-d
    scaled, d = 0..21, both signs: element 0 of each group is amax (exponent
    `amax_exp`), the others are the x values (|x| <= amax), zero padded.  The
    quotient x / s depends only on the significands and d, so this covers
    every ratio a bf16 group can produce at this scale."""
    groups = []
    for ma in range(128):
        amax_bits = ((amax_exp + 127) << 7) | ma
        xs = []
        for d in range(22):
            e = amax_exp + 127 - d
            if e <= 0:
                break
            for mx in range(128):
                if d == 0 and mx > ma:
                    continue
                b = (e << 7) | mx
                xs += [b, b | 0x8000]
        xs = np.array(xs, np.uint16)
        pad = (-len(xs)) % 127
        xs = np.concatenate([xs, np.zeros(pad, np.uint16)]).reshape(-1, 127)
        groups.append(np.concatenate([np.full((xs.shape[0], 1), amax_bits, np.uint16), xs], axis=1))
    return np.concatenate(groups)


@pytest.mark.parametrize("amax_exp", [0, 60, -60])
def test_act_exhaustive_bf16_ratios(orc, amax_exp):
    # every significand pair and exponent gap: the reciprocal-and-correction
    # quotient must equal the oracle's IEEE division in every case
    groups = exhaustive_ratio_groups(amax_exp)
    check_act(orc, groups)
    n = groups.shape[0] // 4 * 4
    check_act(orc, groups[:n].reshape(n // 4, 512), scale_layout="row")


@pytest.mark.parametrize("M,K", [(1, 128), (3, 256), (77, 384), (1000, 1024)])
def test_act_ragged_rows_and_strides(orc, M, K):
    x, _ = synth.activation(13, M, K, outlier_frac=0.02)
    check_act(orc, x, ldx_pad=64, ldq_pad=16)
    check_act(orc, x, scale_layout="row")


def test_act_full_quantizer_workload(orc):
    x, _ = synth.activation(2, 8192, 7168)
    check_act(orc, x)


def test_act_is_deterministic():
    x, _ = synth.activation(3, 512, 2048)
    q1, s1 = run_act(x)
    q2, s2 = run_act(x)
    assert np.array_equal(q1, q2) and bits_eq(s1, s2)


# ------------------------------------------------------------------ weights --

def run_w(bits, q_layout):
    w = gu.bf16_dev(bits)
    q, s = fg.fp8_quant_w_128x128(w, q_layout=q_layout)
    torch.cuda.synchronize()
    return gu.host(q), gu.host(s)


def check_w(orc, bits):
    q_ref, s_ref = orc.quant_w_128x128(bits)
    q, s = run_w(bits, fg.FP8_KMAJOR_NK)
    assert_bits_eq(s, s_ref, "weight scales")
    assert_bits_eq(q, q_ref.T, "weight codes (K-major)")
    q2, s2 = run_w(bits, fg.FP8_ROWMAJOR_KN)
    assert_bits_eq(s2, s_ref, "weight scales")
    assert_bits_eq(q2, q_ref, "weight codes (row-major)")


def test_weight_tiny_config(orc):
    _, b, _ = synth.tiny_end_to_end(seed=1)
    check_w(orc, b)


def test_weight_edge_blocks(orc):
    K, N = 256, 384
    w = synth.f32_from_bf16_bits(synth.weight(21, K, N)).copy()
    w[:128, :128] = 0.0                                          # zero block
    w[:128, 128:256] = (np.arange(128 * 128, dtype=np.float32).reshape(128, 128) % 7 - 3) * np.float32(2.0 ** -133)
    w[128:, :128] *= np.float32(2.0 ** 100)                      # large block
    w[128:, 256:] = 0.0
    w[200, 300] = -448.0                                         # single value block
    check_w(orc, synth.bf16_bits_from_f32(w))


def test_weight_full_quantizer_workload(orc):
    check_w(orc, synth.weight(2, 7168, 18432))


def test_weight_padded_rows(orc):
    """Row strides larger than the row (ldw = N + 64, ldq padded) in both layouts."""
    K, N = 256, 384
    bits = synth.weight(22, K, N)
    q_ref, s_ref = orc.quant_w_128x128(bits)
    wpad = np.zeros((K, N + 64), np.uint16)
    wpad[:, :N] = bits
    w = gu.bf16_dev(wpad)[:, :N]
    qk = torch.full((N, K + 32), 0xAB, dtype=torch.uint8, device="cuda")
    q, s = fg.fp8_quant_w_128x128(w, q=qk[:, :K])
    torch.cuda.synchronize()
    assert_bits_eq(gu.host(q), q_ref.T, "weight codes (K-major, padded)")
    assert_bits_eq(gu.host(s), s_ref, "weight scales (padded)")
    assert np.all(gu.host(qk)[:, K:] == 0xAB), "write outside the code rows"
    qr = torch.full((K, N + 16), 0xAB, dtype=torch.uint8, device="cuda")
    q2, _ = fg.fp8_quant_w_128x128(w, q=qr[:, :N], q_layout=fg.FP8_ROWMAJOR_KN)
    torch.cuda.synchronize()
    assert_bits_eq(gu.host(q2), q_ref, "weight codes (row-major, padded)")
    assert np.all(gu.host(qr)[:, N:] == 0xAB), "write outside the code rows"


@pytest.mark.parametrize("q_layout", [0, 1])
def test_weight_batched_matches_oracle_per_expert(orc, q_layout):
    """One launch over G experts with a padded expert stride; every expert's
    codes and scales equal the oracle's for that expert alone."""
    G, K, N = 3, 256, 384
    experts = [synth.weight(30 + g, K, N) for g in range(G)]
    experts[1] = np.zeros((K, N), np.uint16)          # an all-zero expert
    wbuf = np.zeros((G, K + 128, N), np.uint16)
    for g in range(G):
        wbuf[g, :K] = experts[g]
    w = gu.bf16_dev(wbuf)[:, :K, :]
    q, s = fg.fp8_quant_w_128x128_batched(w, q_layout=q_layout)
    torch.cuda.synchronize()
    q, s = gu.host(q), gu.host(s)
    for g in range(G):
        q_ref, s_ref = orc.quant_w_128x128(experts[g])
        assert_bits_eq(s[g], s_ref, "expert %d scales" % g)
        assert_bits_eq(q[g], q_ref.T if q_layout == 0 else q_ref, "expert %d codes" % g)


def test_weight_batched_moe_experts(orc):
    """The MoE expert weights of the benchmark step (32 x [7168, 2048]), spot-
    checked on four experts."""
    moe = synth.moe_inputs(seed=5, with_weights=True)
    w = gu.bf16_dev(moe.w)
    q, s = fg.fp8_quant_w_128x128_batched(w)
    torch.cuda.synchronize()
    for g in (0, 7, 19, 31):
        q_ref, s_ref = orc.quant_w_128x128(moe.w[g])
        assert_bits_eq(gu.host(s[g]), s_ref, "expert %d scales" % g)
        assert_bits_eq(gu.host(q[g]), q_ref.T, "expert %d codes" % g)


# ---------------------------------------------------------------- requant --

def run_requant(q_np, s_np, s_layout_in="mn"):
    M, K = q_np.shape
    q = gu.dev(q_np)
    if s_layout_in == "mn":
        s = gu.dev(np.ascontiguousarray(s_np.T)).t()
    else:
        s = gu.dev(s_np)
    qT, sT = fg.fp8_requant_1x128_to_128x1(q, s)
    torch.cuda.synchronize()
    return gu.host(qT), gu.host(sT)


def check_requant(orc, bits, **kw):
    q, s = orc.quant_act_1x128(bits)
    qT_ref, sT_ref = orc.requant_1x128_to_128x1(q, s)
    qT, sT = run_requant(q, s, **kw)
    assert_bits_eq(sT, sT_ref, "requant scales")
    assert_bits_eq(qT, qT_ref, "requant codes")


def test_requant_small(orc):
    check_requant(orc, synth.wgrad_tensor(4, 0, 256, 384))
    check_requant(orc, synth.wgrad_tensor(4, 1, 384, 256), s_layout_in="row")


def test_requant_edge_scales(orc):
    rng = np.random.default_rng(8)
    M, K = 256, 256
    q = rng.integers(0, 256, size=(M, K), dtype=np.uint8)
    q[(q & 0x7F) == 0x7F] = 0x01
    q[:, 5] = 0x00                                   # an all-zero channel
    s = np.exp2(rng.uniform(-140, 100, size=(M, K // 128))).astype(np.float32)  # incl. fp32 subnormals
    s[:128, 1] = 0.0                                 # zero-scale groups
    qT_ref, sT_ref = orc.requant_1x128_to_128x1(q, s)
    qT, sT = run_requant(q, s)
    assert_bits_eq(sT, sT_ref, "requant scales")
    assert_bits_eq(qT, qT_ref, "requant codes")


def test_requant_padded_strides(orc):
    """ldq > K, ldqT > M and row-major input scales."""
    bits = synth.wgrad_tensor(4, 1, 256, 384)
    q, s = orc.quant_act_1x128(bits)
    qT_ref, sT_ref = orc.requant_1x128_to_128x1(q, s)
    M, K = q.shape
    qpad = np.zeros((M, K + 48), np.uint8)
    qpad[:, :K] = q
    qd = gu.dev(qpad)[:, :K]
    qTbuf = torch.full((K, M + 16), 0xAB, dtype=torch.uint8, device="cuda")
    qT, sT = fg.fp8_requant_1x128_to_128x1(qd, gu.dev(s), qT=qTbuf[:, :M], scale_layout="row")
    torch.cuda.synchronize()
    assert_bits_eq(gu.host(sT), sT_ref, "requant scales")
    assert_bits_eq(gu.host(qT), qT_ref, "requant codes")
    assert np.all(gu.host(qTbuf)[:, M:] == 0xAB), "write outside the code rows"


@pytest.mark.parametrize("M,K", [(128 * 600, 128), (128, 128 * 700)])
def test_requant_more_blocks_than_ctas_along_one_axis(orc, M, K):
    """One channel block and 600 token blocks, or one token block and 700
    channel blocks: the persistent CTAs (four per SM) take several blocks each,
    stepping along a single axis of the block grid."""
    check_requant(orc, synth.wgrad_tensor(4, 2, M, K))


def test_requant_full_quantizer_workload(orc):
    x, _ = synth.activation(2, 8192, 7168)
    check_requant(orc, x)
