"""The softmax's polynomial 2^x (sm100.cuh: ex2_poly / ex2_poly2), checked on
the CPU from the constants in the source: the same fp32 steps (round to the
nearest integer by the 1.5 * 2^23 shift, the cubic for 2^f on [-1/2, 1/2],
the integer added to the exponent field) against numpy's exp2 in fp64.

Its relative error has to stay far below a bf16 half-ulp (2^-9), since P is
rounded to bf16 for the P.V product right after; and -inf (masked scores)
must give exactly 0, as the SFU's ex2.approx.ftz does."""
import os
import re

import numpy as np

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                   "context_packed_sequence_thd_gb300", "csrc", "sm100.cuh")


def _coeffs():
    src = open(SRC).read()
    body = src[src.index("float ex2_poly(float x)"):]
    body = body[:body.index("}")]
    hexes = re.findall(r"(0x1\.[0-9a-f]+p-?\d+)f", body)
    assert len(hexes) == 3, hexes
    c3, c2, c1 = (np.float32(float.fromhex(h)) for h in hexes)
    return c1, c2, c3


def _ex2_poly(x):
    c1, c2, c3 = _coeffs()
    x = np.maximum(np.asarray(x, np.float32), np.float32(-127.0))
    magic = np.float32(12582912.0)
    t = (x + magic).astype(np.float32)
    f = (x - (t - magic).astype(np.float32)).astype(np.float32)

    def fma(a, b, c):   # single rounding, as the GPU's FFMA
        return (a.astype(np.float64) * b + c).astype(np.float32)

    p = fma(f, np.float32(c3), np.float32(c2))
    p = fma(p, f, np.float32(c1))
    p = fma(p, f, np.float32(1.0))
    bits = (p.view(np.int32).astype(np.int64) + (t.view(np.int32).astype(np.int64) << 23))
    return (bits & 0xFFFFFFFF).astype(np.uint32).view(np.float32)


def test_relative_error_far_below_bf16():
    x = np.linspace(-126.0, 8.0, 2_000_001, dtype=np.float32)
    got = _ex2_poly(x).astype(np.float64)
    rel = np.abs(got / np.exp2(x.astype(np.float64)) - 1.0)
    assert rel.max() < 1.2e-4
    assert rel.max() < 2.0 ** -9 / 16


def test_integers_and_half_integers():
    for j in range(-126, 9):
        assert _ex2_poly(np.float32(j)) == np.float32(2.0 ** j)      # p(0) = 1 exactly
        v = float(_ex2_poly(np.float32(j + 0.5)))
        assert abs(v / 2.0 ** (j + 0.5) - 1) < 1.2e-4


def test_masked_scores_give_exact_zero():
    for x in (-np.inf, -1e30, -200.0, -127.0):
        v = _ex2_poly(np.float32(x))
        assert v == 0.0 and not np.signbit(v)
    # between -127 and -126 the result is tiny and non-negative
    v = _ex2_poly(np.linspace(-127.0, -126.0, 101, dtype=np.float32))
    assert np.all(v >= 0) and np.all(v < 2.0 ** -125)
