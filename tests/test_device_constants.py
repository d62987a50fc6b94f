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
