"""Pins of the oracle's power-of-two scale reading against facts that do not
come from the oracle itself.

Reading: the scale of a group is the smallest power of two s with
amax / s <= 448 (the exact 2^ceil(log2(amax/448))), never below 2^-127 (the
smallest value of an 8-bit exponent scale), and s = 0 for an all-zero group;
codes are the E4M3 round-to-nearest-even of the exact quotient x / s.  The
pages give the scales of some activations as integral powers of 2
(why-be.why-be.co.kr post 55081; sunipension.com post 314414).

* a hand-worked tile (tests/golden/worked_tile_pow2.txt);
* exact round trip of E4M3-representable tiles times 2^j;
* covariance of scale and codes under x -> x 2^k;
* bounds: 224 < amax / s <= 448 for every group away from the clamp, and no
  code saturates;
* the clamp at 2^-127 for tiny groups, worked by hand;
* brute force against exact rational arithmetic (tests/exact_ref.py) for the
  three quantizers.
"""
import os

import numpy as np
import pytest
import torch

import synth
from tests import exact_ref

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def e4m3_table():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    return codes.view(torch.float8_e4m3fn).to(torch.float32).numpy()


def e4m3_grid():
    tab = e4m3_table()
    finite = np.array([c for c in range(256) if (c & 0x7F) != 0x7F])
    return finite, tab[finite]


def load_tile(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            pos, val, code = line.split()[:3]
            rows.append((int(pos), float(val), int(code, 16)))
    return rows


def test_worked_tile_pow2(orc):
    tile = np.zeros(128, np.float32)
    want = np.zeros(128, np.uint8)
    for pos, val, code in load_tile("worked_tile_pow2.txt"):
        tile[pos] = np.float32(val)
        want[pos] = code
    bits = synth.bf16_bits_from_f32(tile)
    assert np.array_equal(synth.f32_from_bf16_bits(bits), tile), "golden values must be bf16-exact"
    # group 0: the tile; group 1: the tile x 2^6 (s = 2^-2, same codes); group 2: zeros
    row = np.concatenate([tile, tile * np.float32(64.0), np.zeros(128, np.float32)])
    q, s = orc.quant_act_1x128(synth.bf16_bits_from_f32(row[None, :]), pow2=True)
    assert s[0, 0] == np.float32(2.0 ** -8)
    assert s[0, 1] == np.float32(2.0 ** -2)
    assert s[0, 2] == 0.0 and np.all(q[0, 256:] == 0)
    assert np.array_equal(q[0, :128], want)
    assert np.array_equal(q[0, 128:256], want)


def test_pow2_scale_at_power_of_two_boundaries(orc):
    # amax = 448 * 2^j exactly gives s = 2^j; the next bf16 value above it gives 2^(j+1)
    for j in (-20, -9, 0, 7):
        a = np.float32(448.0 * 2.0 ** j)
        above = synth.f32_from_bf16_bits(synth.bf16_bits_from_f32(np.array([a])) + np.uint16(1))[0]
        x = np.zeros((2, 128), np.float32)
        x[0, 3] = a
        x[1, 3] = -above
        q, s = orc.quant_act_1x128(synth.bf16_bits_from_f32(x), pow2=True)
        assert s[0, 0] == np.float32(2.0 ** j) and q[0, 3] == 0x7E
        assert s[1, 0] == np.float32(2.0 ** (j + 1))
        # above = 450 * 2^j, so above / 2^(j+1) = 225: between 224 (0x76) and 240 (0x77), nearer 224
        assert q[1, 3] == 0xF6


@pytest.mark.parametrize("j", [-12, -3, 0, 5, 20])
def test_pow2_exact_round_trip(orc, j):
    rng = np.random.default_rng(300 + j)
    codes_all, vals_all = e4m3_grid()
    M, K = 4, 384
    idx = rng.integers(0, len(codes_all), size=(M, K))
    codes = codes_all[idx].astype(np.uint8)
    codes[:, ::128] = 0x7E
    codes[:, 1::128] = 0xFE
    x = (vals_all[idx].astype(np.float64) * 2.0 ** j).astype(np.float32)
    x[:, ::128] = 448 * 2.0 ** j
    x[:, 1::128] = -448 * 2.0 ** j
    bits = synth.bf16_bits_from_f32(x)
    q, s = orc.quant_act_1x128(bits, pow2=True)
    assert np.all(s == np.float32(2.0 ** j))
    assert np.array_equal(q, codes)
    # weights: one 128x128 block holding the same kind of values
    wq, ws = orc.quant_w_128x128(bits[:, :128].repeat(32, axis=0), pow2=True)
    assert np.all(ws == np.float32(2.0 ** j))
    assert np.array_equal(wq, codes[:, :128].repeat(32, axis=0))


def test_pow2_covariance(orc):
    xa, _, _ = synth.tiny_end_to_end(seed=8, M=8, K=512, N=128)
    q0, s0 = orc.quant_act_1x128(xa, pow2=True)
    x = synth.f32_from_bf16_bits(xa)
    for k in range(-20, 21, 5):
        xk = (x.astype(np.float64) * 2.0 ** k).astype(np.float32)
        qk, sk = orc.quant_act_1x128(synth.bf16_bits_from_f32(xk), pow2=True)
        assert np.array_equal(qk, q0), k
        assert np.array_equal(sk, (s0.astype(np.float64) * 2.0 ** k).astype(np.float32)), k


def test_pow2_bounds_and_no_saturation(orc):
    x, _ = synth.activation(9, 64, 1024, outlier_frac=0.02)
    q, s = orc.quant_act_1x128(x, pow2=True)
    amax = np.abs(synth.f32_from_bf16_bits(x).astype(np.float64)).reshape(64, 8, 128).max(axis=2)
    ratio = amax / s.astype(np.float64)
    assert np.all(ratio <= 448.0) and np.all(ratio > 224.0)
    mant = s.view(np.uint32) & 0x7FFFFF
    assert np.all(mant == 0), "scales must be powers of two"
    # codes never exceed the group's amax code, which is below or at 448
    tab = e4m3_table()
    assert np.all(np.abs(tab[q]) <= 448.0)
    # the non-power-of-two scale never exceeds the power-of-two one, and is more than half of it
    _, s_ref = orc.quant_act_1x128(x)
    assert np.all(s_ref <= s) and np.all(s_ref > s / 2)


def test_pow2_clamp_for_tiny_groups(orc):
    # amax = 2^-131 (a bf16 subnormal): 2^ceil(log2(amax/448)) = 2^-139 is below
    # the smallest 8-bit exponent scale, so s = 2^-127.  x / s = 2^-4 for the
    # largest element: E4M3 e = -4 + 7 = 3, m = 0 -> 0x18.  x = -2^-133 (the
    # smallest bf16 subnormal): x / s = -2^-6, the smallest normal -> 0x88.
    x = np.zeros((1, 128), np.float32)
    x[0, 0] = np.float32(2.0 ** -131)
    x[0, 1] = np.float32(-(2.0 ** -133))
    bits = synth.bf16_bits_from_f32(x)
    assert np.array_equal(synth.f32_from_bf16_bits(bits), x)
    q, s = orc.quant_act_1x128(bits, pow2=True)
    assert s[0, 0] == np.float32(2.0 ** -127)
    assert q[0, 0] == 0x18 and q[0, 1] == 0x88
    assert np.all(q[0, 2:] == 0)


def test_pow2_quant_act_matches_exact_reference(orc):
    xa, _, _ = synth.tiny_end_to_end(seed=11, M=6, K=256, N=128)
    rand = synth.f32_from_bf16_bits(xa).reshape(-1, 128)
    rand[0, 7] = -3e-38
    rand[1] *= np.float32(2.0 ** -100)
    bits = synth.bf16_bits_from_f32(rand)
    q, s = orc.quant_act_1x128(bits, pow2=True)
    vals = synth.f32_from_bf16_bits(bits)
    for i in range(vals.shape[0]):
        s_ref, codes = exact_ref.quant_group_pow2(vals[i])
        assert s[i, 0] == s_ref, i
        assert np.array_equal(q[i], np.array(codes, np.uint8)), i


def test_pow2_quant_w_matches_exact_reference(orc):
    w = synth.weight(12, 128, 256)
    q, s = orc.quant_w_128x128(w, pow2=True)
    for nb in range(2):
        blk = synth.f32_from_bf16_bits(w[:, nb * 128:(nb + 1) * 128])
        s_ref, codes = exact_ref.quant_group_pow2(blk.ravel())
        assert s[0, nb] == s_ref
        assert np.array_equal(q[:, nb * 128:(nb + 1) * 128].ravel(), np.array(codes, np.uint8))


def test_pow2_requant_matches_exact_reference(orc):
    M, K = 256, 128
    xa = synth.wgrad_tensor(13, 0, M, K)
    q, s = orc.quant_act_1x128(xa, pow2=True)
    qT, sT = orc.requant_1x128_to_128x1(q, s, pow2=True)
    assert qT.shape == (K, M) and sT.shape == (K, M // 128)
    for k in (0, 5, 63, 127):
        for mb in range(M // 128):
            col = np.array([exact_ref.dequant_f32(int(q[m, k]), s[m, k // 128])
                            for m in range(mb * 128, (mb + 1) * 128)], np.float32)
            s_ref, codes = exact_ref.quant_group_pow2(col)
            assert sT[k, mb] == s_ref, (k, mb)
            assert np.array_equal(qT[k, mb * 128:(mb + 1) * 128], np.array(codes, np.uint8))
