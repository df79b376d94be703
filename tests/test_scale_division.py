"""The quantizers' scales are IEEE quotients fl(absmax / 127) and
fl((max - min) / 15).  The kernels form them without a division, as
fma(x, zh, fl(x * zl)) with zh = fl(1/y), zl = fl(1/y - zh) (Brisebarre,
Muller and Raina, IEEE Trans. Computers 53(8), 2004).  This checks, for every
binary32 significand, that the form equals the IEEE quotient, and that the
constants in the kernel source are those two roundings.  Rounding is
scale-invariant while the quotient and x * zl stay normal, so this covers
every x >= 2^-98 (smaller x keep the division in the kernels)."""
import os
import re
from fractions import Fraction

import numpy as np
import pytest

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                   "quantized_reduce_rmsnorm_gb300", "csrc", "device.cuh")


def _split_reciprocal(y):
    zh = np.float32(1.0 / y)                      # fl(1/y): binary64 1/y is within 2^-53, no tie
    zl = np.float32(float(Fraction(1, int(y)) - Fraction(float(zh))))
    return zh, zl


@pytest.mark.parametrize("y,name", [(15, "kInv15"), (127, "kInv127")])
def test_constants_match_source(y, name):
    src = open(SRC).read()
    hi = int(re.search(name + r"Hi = (0x[0-9A-Fa-f]+)u", src).group(1), 16)
    lo = int(re.search(name + r"Lo = (0x[0-9A-Fa-f]+)u", src).group(1), 16)
    zh, zl = _split_reciprocal(y)
    assert int(zh.view(np.uint32)) == hi and int(zl.view(np.uint32)) == lo


@pytest.mark.skipif(np.finfo(np.longdouble).nmant < 60, reason="needs an extended long double")
@pytest.mark.parametrize("y", [15, 127])
def test_fma_quotient_is_correctly_rounded_for_every_significand(y):
    m = np.arange(1 << 23, 1 << 24, dtype=np.int64)
    x = (m.astype(np.float64) * 2.0 ** -23).astype(np.float32)  # every significand, in [1, 2)
    zh, zl = _split_reciprocal(y)
    ref = x / np.float32(y)                                      # IEEE binary32 quotient
    t = x * zl                                                   # fl(x * zl)
    # x * zh (48 bits) + t is exact in the 64-bit extended format; one rounding to binary32
    q = (x.astype(np.longdouble) * np.longdouble(zh) + t.astype(np.longdouble)).astype(np.float32)
    assert np.count_nonzero(q != ref) == 0
