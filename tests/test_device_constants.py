"""The floating-point constants of the device helpers against their
mathematical values (CPU). The "fp32" SiLU' policy forms e^-p as 2^a e^dl with
dl = -p - a ln 2 from a two-float split of ln 2; a slip in the low part would
move its results by ~1e-8 relative, well inside the GPU tests' 5e-7 gradient
tolerance, so the constants are checked here directly."""
import decimal
import os
import re

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "varlen_causal_depthwise_gb300", "csrc", "vcd_device.cuh")

decimal.getcontext().prec = 40
LN2 = decimal.Decimal(2).ln()
LOG2E = 1 / LN2


def _constants():
    text = open(SRC).read()
    found = dict(re.findall(r"constexpr float (k\w+) = ([-+0-9.eE]+)f;", text))
    return {k: np.float32(float(v)) for k, v in found.items()}


def test_log2e_is_the_nearest_float():
    k = _constants()
    assert k["kLog2e"] == np.float32(float(LOG2E))


def test_ln2_split_is_exact_to_double_precision():
    k = _constants()
    hi, lo = k["kLn2Hi"], k["kLn2Lo"]
    assert hi == np.float32(float(LN2))                        # the nearest float
    assert float(hi) == 0.693147182464599609375                # exactly representable as written
    residual = LN2 - decimal.Decimal(float(hi))
    # the low part is the rounded residual: hi + lo equals ln 2 to float64 precision
    assert abs(decimal.Decimal(float(lo)) - residual) <= abs(residual) * decimal.Decimal(2.0 ** -23)
    assert abs(float(decimal.Decimal(float(hi)) + decimal.Decimal(float(lo)) - LN2)) < 1e-16


DF_SRC = os.path.join(ROOT, "varlen_causal_depthwise_gb300", "csrc", "vcd_dfloat.cuh")


def _hex_float(tok):
    tok = tok.rstrip("f")
    return float(tok) if "x" not in tok else float.fromhex(tok)


_NUM = r"(-?0x[0-9a-fp.+-]+f|-?[0-9.]+f)"


def test_double_float_inverse_factorials():
    """The (hi, lo) pairs of 1/n! used by the double-float exp: hi the nearest
    float, hi + lo within 2^-49 of 1/n! relative (the exp's own truncation is
    below 2^-52)."""
    from fractions import Fraction
    import math
    text = open(DF_SRC).read()
    pairs = dict((int(n), (_hex_float(h), _hex_float(l))) for n, h, l in
                 re.findall(r"case (\d+): return \{" + _NUM + ", " + _NUM + r"\};", text))
    pairs[12] = tuple(_hex_float(t) for t in
                      re.search(r"default: return \{" + _NUM + ", " + _NUM + r"\};", text).groups())
    assert sorted(pairs) == list(range(1, 13))     # "case 0: case 1:" share 1/1!
    for n, (hi, lo) in pairs.items():
        exact = Fraction(1, math.factorial(n))
        assert np.float32(hi) == np.float32(float(exact))
        err = abs(Fraction(hi) + Fraction(lo) - exact) / exact
        assert err < Fraction(1, 2 ** 49), (n, float(err))


def test_double_float_ln2_parts():
    """ln 2 in three floats: the first with at most 17 significant bits (so k
    times it is exact for |k| < 128), the three summing to ln 2 within 2^-65."""
    from fractions import Fraction
    text = open(DF_SRC).read()
    parts = [_hex_float(t) for t in re.findall(r"constexpr float kDfLn2[ABC] = (0x[0-9a-fp.+-]+f);", text)]
    assert len(parts) == 3
    a = parts[0]
    m, _ = np.frexp(a)
    assert float(m * 2 ** 17).is_integer()
    err = abs(Fraction(parts[0]) + Fraction(parts[1]) + Fraction(parts[2]) - Fraction(LN2))
    assert err < Fraction(1, 2 ** 65)
    inv = _hex_float(re.search(r"constexpr float kDfInvLn2 = (0x[0-9a-fp.+-]+f);", text).group(1))
    assert np.float32(inv) == np.float32(float(1 / LN2))
