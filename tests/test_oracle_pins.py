"""Pins of the CPU oracle against facts that do not come from the oracle itself.

* E4M3 codec: every one of the 256 codes against torch's float8_e4m3fn (an
  independent library) and against closed-form values; rounding at every
  midpoint and one fp32 ulp either side; saturation.
* Quantizers: a hand-worked tile (tests/golden/worked_tile_s1.txt); exact
  round trip of E4M3-representable tiles; scale covariance under 2^k; zero
  tiles; brute force against exact rational arithmetic (tests/exact_ref.py),
  including inputs chosen where dividing by s and multiplying by 1/s (or by
  448/amax) give different codes.
* GEMMs: numpy float64 matmul of the dequantized operands, an exact integer
  case, linearity in one K-block's scale, the per-column scale mode, and the
  grouped form against per-expert products.
"""
import os

import numpy as np
import pytest
import torch

import synth
from tests import exact_ref

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def torch_e4m3_codes(y):
    """E4M3 codes of float32 values via torch (valid for |y| <= 448)."""
    t = torch.from_numpy(np.ascontiguousarray(y, np.float32))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def e4m3_table():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    return codes.view(torch.float8_e4m3fn).to(torch.float32).numpy()


# ------------------------------------------------------------------ codec --

def test_decode_all_codes_match_torch(orc):
    ref = e4m3_table()
    for c in range(256):
        v = orc.e4m3_decode(c)
        if (c & 0x7F) == 0x7F:
            assert np.isnan(v) and np.isnan(ref[c])
        else:
            assert v == ref[c], hex(c)
            assert np.signbit(v) == bool(c & 0x80)


def test_decode_closed_form_values(orc):
    assert orc.e4m3_decode(0x7E) == 448.0
    assert orc.e4m3_decode(0xFE) == -448.0
    assert orc.e4m3_decode(0x01) == 2.0 ** -9
    assert orc.e4m3_decode(0x07) == 7 * 2.0 ** -9
    assert orc.e4m3_decode(0x08) == 2.0 ** -6
    assert orc.e4m3_decode(0x38) == 1.0
    assert orc.e4m3_decode(0x3F) == 1.875
    assert orc.e4m3_decode(0x40) == 2.0
    assert orc.e4m3_decode(0x00) == 0.0 and not np.signbit(orc.e4m3_decode(0x00))
    assert orc.e4m3_decode(0x80) == 0.0 and np.signbit(orc.e4m3_decode(0x80))


def test_encode_midpoints_and_neighbours(orc):
    tab = e4m3_table()
    mags = tab[:0x7F]          # 0x00..0x7E, increasing
    for c in range(0x7E):
        lo, hi = np.float64(mags[c]), np.float64(mags[c + 1])
        mid = np.float32((lo + hi) / 2)
        assert np.float64(mid) == (lo + hi) / 2       # midpoints are fp32-exact
        want_tie = c if c % 2 == 0 else c + 1
        below = np.nextafter(mid, np.float32(0))
        above = np.nextafter(mid, np.float32(1000))
        for sgn in (1, -1):
            sb = 0x80 if sgn < 0 else 0
            assert orc.e4m3_encode(sgn * mid) == sb | want_tie
            assert orc.e4m3_encode(sgn * below) == sb | c
            assert orc.e4m3_encode(sgn * above) == sb | (c + 1)
            assert orc.e4m3_encode(sgn * np.float32(lo)) == sb | c
    # same decisions through torch for the positive side
    mids = np.float32((mags[:-1].astype(np.float64) + mags[1:]) / 2)
    assert np.array_equal(orc.e4m3_encode_array(mids), torch_e4m3_codes(mids))


def test_encode_random_matches_torch(orc):
    rng = np.random.default_rng(11)
    n = 200_000
    mag = np.exp2(rng.uniform(-16, np.log2(448.0), n)).astype(np.float32)
    y = np.where(rng.random(n) < 0.5, -mag, mag).astype(np.float32)
    y[:10] = [0.0, -0.0, 448.0, -448.0, 1e-30, -1e-30, 2 ** -10, 2 ** -9, 3 * 2 ** -10, 464.0 - 1]
    keep = np.abs(y) <= 448
    got = orc.e4m3_encode_array(y[keep])
    assert np.array_equal(got, torch_e4m3_codes(y[keep]))


def test_encode_saturates(orc):
    for v in (448.0, 448.0001, 463.9, 464.0, 465.0, 1e6, 3.0e38):
        assert orc.e4m3_encode(v) == 0x7E
        assert orc.e4m3_encode(-v) == 0xFE


# ------------------------------------------------------------ quantizers --

def load_worked_tile():
    rows = []
    with open(os.path.join(GOLDEN, "worked_tile_s1.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            pos, val, code = line.split()[:3]
            rows.append((int(pos), float(val), int(code, 16)))
    return rows


def test_worked_tile_s1(orc):
    rows = load_worked_tile()
    tile = np.zeros(128, np.float32)
    want = np.zeros(128, np.uint8)
    for pos, val, code in rows:
        tile[pos] = np.float32(val)
        want[pos] = code
    bits = synth.bf16_bits_from_f32(tile)
    assert np.array_equal(synth.f32_from_bf16_bits(bits), tile), "golden values must be bf16-exact"
    # the worked tile is group 1 of a row; group 0 is all zero, group 2 is the tile x 2^-10
    row = np.concatenate([np.zeros(128, np.float32), tile, tile * np.float32(2.0 ** -10)])
    x = synth.bf16_bits_from_f32(row[None, :])
    q, s = orc.quant_act_1x128(x)
    assert s.shape == (1, 3)
    assert s[0, 0] == 0.0 and np.all(q[0, :128] == 0)
    assert s[0, 1] == 1.0
    assert np.array_equal(q[0, 128:256], want)
    assert s[0, 2] == np.float32(2.0 ** -10)
    assert np.array_equal(q[0, 256:], want)


def test_scale_of_unit_amax_is_rounded_quotient(orc):
    # amax = 1: s = RN32(1/448).  1/448 = 2^-9 * 8/7 and 8/7 = 1.001001...b, so
    # the 23 fraction bits are 00100100100100100100100|1001... -> round up
    # -> 0x124925 with biased exponent 118: bit pattern 0x3B124925.
    row = np.zeros((1, 128), np.float32)
    row[0, 5] = 1.0
    row[0, 6] = -0.5
    q, s = orc.quant_act_1x128(synth.bf16_bits_from_f32(row))
    assert s.view(np.uint32)[0, 0] == 0x3B124925
    assert q[0, 5] == 0x7E            # 1/s rounds to 448 in E4M3
    assert q[0, 6] == 0xF6            # -0.5/s -> -224 = -(1.75 * 2^7): e=14, m=6


def e4m3_grid():
    tab = e4m3_table()
    finite = np.array([c for c in range(256) if (c & 0x7F) != 0x7F])
    return finite, tab[finite]


@pytest.mark.parametrize("j", [-12, -3, 0, 5, 20])
def test_exact_round_trip_of_representable_tiles(orc, j):
    rng = np.random.default_rng(100 + j)
    codes_all, vals_all = e4m3_grid()
    M, K = 4, 384
    idx = rng.integers(0, len(codes_all), size=(M, K))
    codes = codes_all[idx].astype(np.uint8)
    codes[:, ::128] = 0x7E                    # each group holds +448 ...
    codes[:, 1::128] = 0xFE                   # ... and -448
    x = (vals_all[idx].astype(np.float64) * 2.0 ** j).astype(np.float32)
    x[:, ::128] = 448 * 2.0 ** j
    x[:, 1::128] = -448 * 2.0 ** j
    bits = synth.bf16_bits_from_f32(x)
    assert np.array_equal(synth.f32_from_bf16_bits(bits), x)
    q, s = orc.quant_act_1x128(bits)
    assert np.all(s == np.float32(2.0 ** j))
    assert np.array_equal(q, codes)


def test_scale_covariance_power_of_two(orc):
    xa, _, _ = synth.tiny_end_to_end(seed=7, M=8, K=512, N=128)
    q0, s0 = orc.quant_act_1x128(xa)
    x = synth.f32_from_bf16_bits(xa)
    for k in range(-20, 21, 4):
        xk = (x.astype(np.float64) * 2.0 ** k).astype(np.float32)
        qk, sk = orc.quant_act_1x128(synth.bf16_bits_from_f32(xk))
        assert np.array_equal(qk, q0), k
        assert np.array_equal(sk, (s0.astype(np.float64) * 2.0 ** k).astype(np.float32)), k
    w = synth.weight(7, 256, 256)
    qw0, sw0 = orc.quant_w_128x128(w)
    wk = synth.bf16_bits_from_f32(synth.f32_from_bf16_bits(w) * np.float32(2.0 ** 9))
    qwk, swk = orc.quant_w_128x128(wk)
    assert np.array_equal(qwk, qw0)
    assert np.array_equal(swk, sw0 * np.float32(2.0 ** 9))


def test_zero_tiles(orc):
    x = np.zeros((3, 256), np.float32)
    x[1, :128] = -0.0
    x[2, 128:] = np.linspace(-1, 1, 128, dtype=np.float32)
    q, s = orc.quant_act_1x128(synth.bf16_bits_from_f32(x))
    assert np.all(q[:2] == 0) and np.all(s[:2] == 0)
    assert np.all(q[2, :128] == 0) and s[2, 0] == 0 and s[2, 1] > 0
    w = np.zeros((128, 256), np.uint16)
    w[:, :128] = 0x8000                     # -0.0 everywhere in block 0
    qw, sw = orc.quant_w_128x128(w)
    assert np.all(qw == 0) and np.all(sw == 0)


def adversarial_pairs(n_amax=300, seed=0):
    """bf16 (x, amax) pairs where RN(x/s), RN(x*RN(1/s)) and RN(x*RN(448/amax))
    fall on different sides of an E4M3 rounding boundary.  Found by search; the
    expected codes come from the exact reference, not from this search."""
    rng = np.random.default_rng(seed)
    bits = np.arange(0x3B80, 0x4380, dtype=np.uint16)
    xs = synth.f32_from_bf16_bits(bits)
    out = []
    for ab in rng.choice(bits, n_amax):
        amax = synth.f32_from_bf16_bits(np.array([ab]))[0]
        x = xs[xs <= amax]
        s = np.float32(amax) / np.float32(448)
        c1 = torch_e4m3_codes(x / s)
        c2 = torch_e4m3_codes(x * (np.float32(1) / s))
        c3 = torch_e4m3_codes(x * (np.float32(448) / np.float32(amax)))
        for i in np.nonzero((c1 != c2) | (c1 != c3))[0][:2]:
            out.append((x[i], amax))
    return out


def test_quant_act_matches_exact_reference(orc):
    pairs = adversarial_pairs()
    assert len(pairs) >= 10
    rows = []
    for x, amax in pairs:
        r = np.zeros(128, np.float32)
        r[0] = amax
        r[1] = x
        r[2] = -x
        rows.append(r)
    xa, _, _ = synth.tiny_end_to_end(seed=3, M=6, K=256, N=128)
    rand = synth.f32_from_bf16_bits(xa).reshape(-1, 128)
    rand[0, 7] = -3e-38                     # quotient far below the E4M3 grid
    tiles = np.concatenate([np.stack(rows), rand]).astype(np.float32)
    bits = synth.bf16_bits_from_f32(tiles)
    q, s = orc.quant_act_1x128(bits)
    vals = synth.f32_from_bf16_bits(bits)
    for i in range(tiles.shape[0]):
        s_ref, codes = exact_ref.quant_group(vals[i])
        assert s[i, 0] == s_ref, i
        assert np.array_equal(q[i], np.array(codes, np.uint8)), i


def test_quant_w_matches_exact_reference(orc):
    K, N = 128, 256
    w = synth.weight(5, K, N)
    wf = synth.f32_from_bf16_bits(w)
    wf[3, 200] = np.float32(2.5)            # an outlier in block (0, 1)
    w = synth.bf16_bits_from_f32(wf)
    q, s = orc.quant_w_128x128(w)
    for nb in range(2):
        blk = synth.f32_from_bf16_bits(w[:, nb * 128:(nb + 1) * 128])
        s_ref, codes = exact_ref.quant_group(blk.ravel())
        assert s[0, nb] == s_ref
        assert np.array_equal(q[:, nb * 128:(nb + 1) * 128].ravel(), np.array(codes, np.uint8))


def test_requant_matches_exact_reference(orc):
    M, K = 256, 128                          # M != K: a transposition slip shows
    xa = synth.wgrad_tensor(9, 0, M, K)
    q, s = orc.quant_act_1x128(xa)
    qT, sT = orc.requant_1x128_to_128x1(q, s)
    assert qT.shape == (K, M) and sT.shape == (K, M // 128)
    for k in (0, 1, 17, 64, 127):
        for mb in range(M // 128):
            col = np.array([exact_ref.dequant_f32(int(q[m, k]), s[m, k // 128])
                            for m in range(mb * 128, (mb + 1) * 128)], np.float32)
            s_ref, codes = exact_ref.quant_group(col)
            assert sT[k, mb] == s_ref, (k, mb)
            assert np.array_equal(qT[k, mb * 128:(mb + 1) * 128], np.array(codes, np.uint8))


def test_requant_of_power_of_two_scaled_grid_is_exact(orc):
    # Every 1x128 scale is a power of two and every dequantized value is an E4M3
    # value x 2^j with +-448*2^j in each 128-token column group, so the 128x1
    # requantization must reproduce the codes (transposed) and the scale 2^j.
    rng = np.random.default_rng(4)
    codes_all, _ = e4m3_grid()
    M, K = 256, 256
    q = codes_all[rng.integers(0, len(codes_all), size=(M, K))].astype(np.uint8)
    q[0::128, :] = 0x7E
    q[1::128, :] = 0xFE
    s = np.full((M, K // 128), np.float32(2.0 ** -5))
    qT, sT = orc.requant_1x128_to_128x1(q, s)
    assert np.all(sT == np.float32(2.0 ** -5))
    assert np.array_equal(qT, q.T)


# ------------------------------------------------------------------ GEMMs --

def dequant_rows(q, s, group_axis_len=128):
    tab = e4m3_table().astype(np.float64)
    v = tab[q]
    return v * np.repeat(s.astype(np.float64), group_axis_len, axis=1)


def test_gemm_matches_numpy_on_tiny_config(orc):
    a_bits, b_bits, _ = synth.tiny_end_to_end(seed=1)
    qa, sa = orc.quant_act_1x128(a_bits)                 # [256,512], [256,4]
    qb, sb = orc.quant_w_128x128(b_bits)                 # [512,256], [4,2]
    C = orc.gemm_blockscaled(qa, sa, qb.T.copy(), sb, orc.SB_BLOCK128x128)
    A = dequant_rows(qa, sa)
    tab = e4m3_table().astype(np.float64)
    B = tab[qb] * np.kron(sb.astype(np.float64), np.ones((128, 128)))
    ref = A @ B
    assert np.max(np.abs(C - ref)) <= 1e-12 * np.max(np.abs(ref))
    # and the FP8 path stays close to the unquantized product
    exact = synth.f32_from_bf16_bits(a_bits).astype(np.float64) @ \
        synth.f32_from_bf16_bits(b_bits).astype(np.float64)
    assert np.linalg.norm(C - exact) / np.linalg.norm(exact) < 0.05


def test_gemm_integer_special_case_is_exact(orc):
    rng = np.random.default_rng(2)
    M, N, K = 64, 48, 128
    ints = np.arange(-8, 9)
    A = rng.choice(ints, size=(M, K))
    B = rng.choice(ints, size=(K, N))
    enc = {int(v): orc.e4m3_encode(float(v)) for v in ints}
    qa = np.vectorize(enc.get)(A).astype(np.uint8)
    qbt = np.vectorize(enc.get)(B.T).astype(np.uint8)
    C = orc.gemm_blockscaled(qa, np.ones((M, 1), np.float32), qbt,
                             np.ones((1, 1), np.float32), orc.SB_BLOCK128x128)
    assert np.array_equal(C, (A @ B).astype(np.float64))


def test_gemm_linearity_in_one_block_scale(orc):
    rng = np.random.default_rng(3)
    M, N, K = 32, 40, 384
    qa = rng.integers(0, 0x7E, size=(M, K), dtype=np.uint8)
    qbt = rng.integers(0, 0x7E, size=(N, K), dtype=np.uint8) | \
        (rng.integers(0, 2, size=(N, K), dtype=np.uint8) << 7)
    sa = rng.uniform(0.5, 2, size=(M, 3)).astype(np.float32)
    sb = rng.uniform(0.5, 2, size=(3, 1)).astype(np.float32)
    C0 = orc.gemm_blockscaled(qa, sa, qbt, sb, orc.SB_BLOCK128x128)
    sa2 = sa.copy()
    sa2[:, 1] *= 2
    C2 = orc.gemm_blockscaled(qa, sa2, qbt, sb, orc.SB_BLOCK128x128)
    only1 = sa.copy()
    only1[:, [0, 2]] = 0
    C1 = orc.gemm_blockscaled(qa, only1, qbt, sb, orc.SB_BLOCK128x128)
    assert np.allclose(C2 - C0, C1, rtol=1e-12, atol=1e-9 * np.abs(C0).max())


def test_gemm_per_column_scales_match_numpy(orc):
    rng = np.random.default_rng(5)
    M, N, K = 40, 72, 256
    qa = rng.integers(0, 256, size=(M, K), dtype=np.uint8)
    qa[(qa & 0x7F) == 0x7F] = 0x10
    qbt = rng.integers(0, 256, size=(N, K), dtype=np.uint8)
    qbt[(qbt & 0x7F) == 0x7F] = 0x22
    sa = rng.uniform(0.1, 3, size=(M, 2)).astype(np.float32)
    sb = rng.uniform(0.1, 3, size=(2, N)).astype(np.float32)
    C = orc.gemm_blockscaled(qa, sa, qbt, sb, orc.SB_COL128x1)
    tab = e4m3_table().astype(np.float64)
    A = tab[qa] * np.repeat(sa.astype(np.float64), 128, axis=1)
    B = tab[qbt].T * np.repeat(sb.astype(np.float64), 128, axis=0)
    ref = A @ B
    assert np.max(np.abs(C - ref)) <= 1e-12 * np.max(np.abs(ref))
    ms = rng.integers(0, M, 50)
    ns = rng.integers(0, N, 50)
    smp = orc.gemm_blockscaled_sample(qa, sa, qbt, sb, orc.SB_COL128x1, ms, ns)
    assert np.array_equal(smp, C[ms, ns])


def test_grouped_gemm_matches_per_expert_numpy(orc):
    rng = np.random.default_rng(6)
    G, N, K = 4, 256, 256
    offsets = np.array([0, 128, 128, 384, 512], np.int32)   # expert 1 is empty
    M_total = 640                                           # rows 512.. belong to nobody
    qa = rng.integers(0, 0x7E, size=(M_total, K), dtype=np.uint8)
    sa = rng.uniform(0.5, 2, size=(M_total, K // 128)).astype(np.float32)
    qb = rng.integers(0, 0x7E, size=(G, N, K), dtype=np.uint8)
    sb = rng.uniform(0.5, 2, size=(G, K // 128, N // 128)).astype(np.float32)
    C = orc.grouped_gemm_blockscaled(qa, sa, qb, sb, offsets)
    tab = e4m3_table().astype(np.float64)
    A = tab[qa] * np.repeat(sa.astype(np.float64), 128, axis=1)
    for g in range(G):
        r0, r1 = offsets[g], offsets[g + 1]
        B = tab[qb[g]].T * np.kron(sb[g].astype(np.float64), np.ones((128, 128)))
        ref = A[r0:r1] @ B
        if r1 > r0:
            assert np.max(np.abs(C[r0:r1] - ref)) <= 1e-12 * np.max(np.abs(ref))
    assert np.all(np.isnan(C[512:]))
    ms = np.array([0, 130, 383, 400, 600])
    ns = np.array([0, 5, 255, 128, 1])
    smp = orc.grouped_gemm_blockscaled_sample(qa, sa, qb, sb, offsets, ms, ns)
    assert np.array_equal(smp[:4], C[ms[:4], ns[:4]]) and np.isnan(smp[4])


def test_dense_gemm_form_matches_elementwise_oracle(orc):
    """The dense FP64 form used for full-size acceptance equals the plain
    element-wise oracle up to FP64 summation order, for both scale kinds."""
    a, b, _ = synth.tiny_end_to_end(seed=1)
    qa, sa = orc.quant_act_1x128(a)
    qb, sb = orc.quant_w_128x128(b)
    qbt = np.ascontiguousarray(qb.T)
    ref = orc.gemm_blockscaled(qa, sa, qbt, sb, orc.SB_BLOCK128x128)
    got = orc.gemm_blockscaled_dense(qa, sa, qbt, sb, orc.SB_BLOCK128x128)
    assert np.max(np.abs(got - ref)) <= 1e-12 * np.max(np.abs(ref))
    x = synth.wgrad_tensor(3, 0, 256, 128)
    dy = synth.wgrad_tensor(3, 1, 256, 256)
    qx, sx = orc.requant_1x128_to_128x1(*orc.quant_act_1x128(x))
    qd, sd = orc.requant_1x128_to_128x1(*orc.quant_act_1x128(dy))
    sb_col = np.ascontiguousarray(sd.T)
    ref = orc.gemm_blockscaled(qx, sx, qd, sb_col, orc.SB_COL128x1)
    got = orc.gemm_blockscaled_dense(qx, sx, qd, sb_col, orc.SB_COL128x1)
    assert np.max(np.abs(got - ref)) <= 1e-12 * np.max(np.abs(ref))
