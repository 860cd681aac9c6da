"""Exact rational arithmetic used to pin the oracle (tests only).

Everything here works on ``fractions.Fraction`` values, so each rounding the
method specifies happens exactly once, where the definition puts it:

* ``f32_round``: IEEE binary32 round-to-nearest-even of an exact rational
  (gradual underflow kept, no flush to zero);
* ``e4m3_round``: OCP E4M3 round-to-nearest-even with saturation at +-448;
* ``quant_group``: amax -> s = RN32(amax / 448) -> code = E4M3(RN32(x / s)).

It is deliberately a different mechanism from the C oracle (which bisects a
decode table in double precision), so that an implementation slip in either
one shows up as a disagreement.
"""
import math
import struct
from fractions import Fraction

import numpy as np

E4M3_MAX = Fraction(448)


def f32_bits_to_fraction(bits: int):
    """(sign, |value| as Fraction) of a finite binary32 bit pattern."""
    sign = (bits >> 31) & 1
    e = (bits >> 23) & 0xFF
    m = bits & 0x7FFFFF
    assert e != 0xFF, "finite inputs only"
    if e == 0:
        mag = Fraction(m, 1 << 149)
    else:
        mag = Fraction((1 << 23) | m) * Fraction(2) ** (e - 150)
    return sign, mag


def float_to_fraction(x: float):
    bits = struct.unpack("<I", struct.pack("<f", np.float32(x)))[0]
    return f32_bits_to_fraction(bits)


def _round_half_even(q: Fraction) -> int:
    fl = math.floor(q)
    r = q - fl
    if r > Fraction(1, 2):
        return fl + 1
    if r < Fraction(1, 2):
        return fl
    return fl if fl % 2 == 0 else fl + 1


def _exponent(mag: Fraction) -> int:
    """floor(log2(mag)) for mag > 0, exactly."""
    e = mag.numerator.bit_length() - mag.denominator.bit_length()
    if Fraction(2) ** e > mag:
        e -= 1
    while Fraction(2) ** (e + 1) <= mag:
        e += 1
    return e


def f32_round(mag: Fraction) -> Fraction:
    """Round a non-negative exact value to binary32, nearest-even, subnormals kept."""
    if mag == 0:
        return Fraction(0)
    e = max(_exponent(mag), -126)
    ulp = Fraction(2) ** (e - 23)
    n = _round_half_even(mag / ulp)
    out = n * ulp
    assert out < Fraction(2) ** 128, "overflow is outside the contract"
    return out


def e4m3_round(mag: Fraction) -> Fraction:
    """Round a non-negative exact value to E4M3 (nearest-even), saturating at 448."""
    if mag == 0:
        return Fraction(0)
    e = max(_exponent(mag), -6)
    ulp = Fraction(2) ** (e - 3)
    out = _round_half_even(mag / ulp) * ulp
    return min(out, E4M3_MAX)


def e4m3_code_of(sign: int, mag: Fraction) -> int:
    """Bit pattern of an E4M3 value given exactly (mag must be representable)."""
    if mag == 0:
        return sign << 7
    e = _exponent(mag)
    if e < -6:      # subnormal: mag = m * 2^-9
        m = mag / Fraction(2) ** -9
        assert m.denominator == 1 and 0 < m < 8
        return (sign << 7) | int(m)
    frac = mag / Fraction(2) ** e - 1
    m = frac * 8
    assert m.denominator == 1 and 0 <= m < 8
    code = (sign << 7) | ((e + 7) << 3) | int(m)
    assert (code & 0x7F) != 0x7F
    return code


def quant_group(values_f32):
    """Exact reference of one quantization group.  values_f32: float32 array.
    Returns (scale as float32, list of codes)."""
    vals = [float_to_fraction(v) for v in np.asarray(values_f32, np.float32).ravel()]
    amax = max((mag for _, mag in vals), default=Fraction(0))
    s = f32_round(amax / E4M3_MAX)
    codes = []
    for sign, mag in vals:
        if amax == 0:
            codes.append(0)
            continue
        y = f32_round(mag / s)
        codes.append(e4m3_code_of(sign, e4m3_round(y)))
    return np.float32(float(s)), codes


def dequant_f32(code: int, s: np.float32) -> np.float32:
    """RN32(decode(code) * s), exactly (decode from the bit fields)."""
    sign = (code >> 7) & 1
    e = (code >> 3) & 0xF
    m = code & 7
    assert (code & 0x7F) != 0x7F
    mag = Fraction(m, 512) if e == 0 else (1 + Fraction(m, 8)) * Fraction(2) ** (e - 7)
    _, smag = float_to_fraction(s)
    v = float(f32_round(mag * smag))
    if sign:
        v = -v
    return np.float32(v)


def pow2_scale(amax: Fraction) -> Fraction:
    """The power-of-two scale of a group (reading R12): the smallest 2^e with
    amax <= 448 * 2^e, e >= -127; 0 for an all-zero group."""
    if amax == 0:
        return Fraction(0)
    e = -127
    while E4M3_MAX * Fraction(2) ** e < amax:
        e += 1
    return Fraction(2) ** e


def quant_group_pow2(values_f32):
    """Exact reference of one group with a power-of-two scale: s = pow2_scale(amax),
    code = E4M3(RN32(x / s)).  Returns (scale as float32, list of codes)."""
    vals = [float_to_fraction(v) for v in np.asarray(values_f32, np.float32).ravel()]
    amax = max((mag for _, mag in vals), default=Fraction(0))
    s = pow2_scale(amax)
    codes = []
    for sign, mag in vals:
        if amax == 0:
            codes.append(0)
            continue
        codes.append(e4m3_code_of(sign, e4m3_round(f32_round(mag / s))))
    return np.float32(float(s)), codes


def bf16_round(mag: Fraction) -> Fraction:
    """Round a non-negative exact value to bf16 (8 significant bits),
    nearest-even, subnormals (quantum 2^-133) kept."""
    if mag == 0:
        return Fraction(0)
    e = max(_exponent(mag), -126)
    ulp = Fraction(2) ** (e - 7)
    out = _round_half_even(mag / ulp) * ulp
    assert out < Fraction(2) ** 128, "overflow is outside the contract"
    return out


def bf16_bits_of(sign: int, mag: Fraction) -> int:
    """Bit pattern of a bf16 value given exactly (mag must be representable)."""
    if mag == 0:
        return sign << 15
    f = np.float32(float(mag))
    assert Fraction(float(f)) == mag
    return (sign << 15) | (int(f.view(np.uint32)) >> 16)


def swiglu_bf16_exact(g_bits: int, u_bits: int, digits: int = 60) -> int:
    """bf16 bits of y = g * u * sigma(g), sigma(g) = 1 / (1 + e^-g), rounded
    once.  The sigmoid factor is evaluated with `digits` significant decimal
    digits (decimal's exp is correctly rounded at that precision) in a form
    that keeps its relative precision for any g: for g >= 0, y = g u (1 - t)
    with t = 1 / (1 + e^g); for g < 0, y = g u e^g / (1 + e^g).  The rest is
    exact rational arithmetic."""
    import decimal
    ctx = decimal.Context(prec=digits, Emin=-10 ** 9, Emax=10 ** 9)
    sg, mg = f32_bits_to_fraction(int(g_bits) << 16)
    su, mu = f32_bits_to_fraction(int(u_bits) << 16)
    prod = mg * mu
    sign = sg ^ su
    if prod == 0:
        return sign << 15
    gd = ctx.divide(decimal.Decimal(mg.numerator), decimal.Decimal(mg.denominator))   # |g|
    e = ctx.exp(gd)                                  # e^|g|
    t = Fraction(ctx.divide(decimal.Decimal(1), ctx.add(decimal.Decimal(1), e)))     # 1 / (1 + e^|g|)
    if sg == 0:
        y = prod * (1 - t)                           # g >= 0: sigma(g) = 1 - 1/(1 + e^g)
    else:
        y = prod * t                                 # g < 0: sigma(g) = 1/(1 + e^|g|)
    return bf16_bits_of(sign, bf16_round(y))
