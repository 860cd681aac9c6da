"""Pins of the oracle's SwiGLU recompute (reading: y = bf16(g * u / (1 + e^-g))
in FP64, rounded once; why-be.why-be.co.kr post 65900, the SwiGLU output is
recomputed from its cached inputs) against facts that do not come from the
oracle itself:

* a 60-digit decimal evaluation (Python's decimal exp is correctly rounded)
  followed by exact-rational bf16 rounding, on random bf16 pairs over many
  binades and on hand-picked specials;
* closed forms: g = 0 gives a signed zero; u = 0 gives a signed zero; a large
  positive gate gives bf16(g u); the sign of y is that of g * u.
"""
import numpy as np

import synth
from tests import exact_ref


def bits(vals):
    return synth.bf16_bits_from_f32(np.asarray(vals, np.float32))


def test_swiglu_matches_high_precision_reference(orc):
    rng = np.random.default_rng(0)
    n = 3000
    g = (rng.standard_normal(n) * 2.0 ** rng.integers(-6, 6, n)).astype(np.float32)
    u = (rng.standard_normal(n) * 2.0 ** rng.integers(-20, 20, n)).astype(np.float32)
    g[:8] = [0.0, -0.0, 100.0, -100.0, 88.0, -88.0, 1e-30, -1e-30]
    gb, ub = bits(g)[None, :], bits(u)[None, :]
    y = orc.swiglu_bf16(gb, ub)[0]
    want = np.array([exact_ref.swiglu_bf16_exact(int(a), int(b)) for a, b in zip(gb[0], ub[0])], np.uint16)
    bad = np.nonzero(y != want)[0]
    assert bad.size == 0, [(hex(gb[0, i]), hex(ub[0, i]), hex(y[i]), hex(want[i])) for i in bad[:5]]


def test_swiglu_closed_forms(orc):
    g = np.array([[0.0, -0.0, 0.0, 64.0, 64.0, 3.0, -3.0, 200.0]], np.float32)
    u = np.array([[5.0, 5.0, -5.0, 1.5, -0.75, 0.0, -0.0, 3.0]], np.float32)
    y = orc.swiglu_bf16(bits(g), bits(u))[0]
    assert y[0] == 0x0000 and y[1] == 0x8000 and y[2] == 0x8000      # 0 * u / 2 keeps the product's sign
    assert y[3] == bits([96.0])[0]                                   # sigmoid(64) = 1 - 1.6e-28: y = 96
    assert y[4] == bits([-48.0])[0]
    assert y[5] == 0x0000 and y[6] == 0x0000                          # u = 0: (+0) and (-3 * -0) = +0
    assert y[7] == bits([600.0])[0]                                   # 600 is bf16-exact


def test_swiglu_sign_and_monotone_gate(orc):
    # for u = 1 the output silu(g) is increasing for g > -1.28 and negative for g < 0
    g = np.linspace(-1.2, 8.0, 128, dtype=np.float32)[None, :]
    gb = bits(g)
    y = synth.f32_from_bf16_bits(orc.swiglu_bf16(gb, bits(np.ones_like(g))))[0]
    gv = synth.f32_from_bf16_bits(gb)[0]
    assert np.all(np.diff(y) >= 0)
    assert np.all((y < 0) == (gv < 0))


def test_swiglu_products_on_bf16_midpoints(orc):
    """g * u exactly on a bf16 rounding midpoint with sigma(g) within 2^-52 of 1
    (g >= 36): FP64 alone would round the tie; the true value lies just below
    the midpoint in magnitude, and the decimal reference says so."""
    rng = np.random.default_rng(1)
    ub = rng.integers(0x3C00, 0x4300, 40000).astype(np.uint16)
    ub = np.concatenate([ub, ub | 0x8000])
    uv = synth.f32_from_bf16_bits(ub).astype(np.float64)
    gs, us = [], []
    for g in (36.0, 40.0, 48.0, 64.0, 100.0, 1000.0, -3.0, -0.75):
        prod = g * uv
        # a midpoint has exactly 9 significant bits with the last one set
        m, e = np.frexp(np.abs(prod))
        scaled = m * 2.0 ** 9
        on_mid = (scaled == np.floor(scaled)) & (np.floor(scaled) % 2 == 1)
        sel = np.nonzero(on_mid)[0][:60]
        gs += [g] * len(sel)
        us += list(ub[sel])
    assert len(gs) >= 200
    gb = bits(np.array(gs, np.float32))[None, :]
    ubs = np.array(us, np.uint16)[None, :]
    y = orc.swiglu_bf16(gb, ubs)[0]
    want = np.array([exact_ref.swiglu_bf16_exact(int(a), int(b)) for a, b in zip(gb[0], ubs[0])], np.uint16)
    bad = np.nonzero(y != want)[0]
    assert bad.size == 0, [(hex(gb[0, i]), hex(ubs[0, i]), hex(y[i]), hex(want[i])) for i in bad[:5]]
