"""The V-code arithmetic of the FP8 prologue, checked as a method (CPU).

The Vᵀ kernel forms x / scale = 448 x / amax without a division: with
amax = d 2^E, d in [1, 2), it takes a = 448 (2^-E x) (exact for a bf16 x),
q0 = a rcp(d), and Markstein's correction q = q0 + (a - q0 d) rcp(d), with
the residual exact by FMA, then copies the sign of x onto q.  Here that
sequence runs in fp32 (numpy; an FMA as the exact product plus one fp32
rounding) for every bf16 x <= amax and a spread of bf16 amax values from the
smallest subnormal to the largest finite one, and its E4M3 code must equal
the oracle's code of the exact quotient, ties included.
"""
import numpy as np

import oracle


def _fma32(a, b, c):
    return (np.asarray(a, np.float64) * np.asarray(b, np.float64) + np.asarray(c, np.float64)).astype(np.float32)


def _codes(x, amax):
    den = np.float32(amax)
    pre = np.float32(16777216.0) if den < np.float32(1.17549435e-38) else np.float32(1.0)
    den = np.float32(den * pre)
    ex = int((den.view(np.uint32) >> 23) & 0xFF) - 127
    dm = np.uint32((den.view(np.uint32) & 0x007FFFFF) | 0x3F800000).view(np.float32)
    s2 = np.float32(np.ldexp(1.0, -ex))
    y = np.float32(np.float32(1.0) / dm)
    with np.errstate(all="ignore"):
        a = (((x * pre).astype(np.float32) * s2).astype(np.float32) * np.float32(448)).astype(np.float32)
        q0 = (a * y).astype(np.float32)
        q = np.copysign(_fma32(_fma32(-q0, dm, a), y, q0), x)
    return oracle.e4m3_encode(q.astype(np.float64))


def test_v_codes_equal_the_exact_quotients():
    bits = np.arange(1, 0x7F80, dtype=np.uint32)
    allx = (bits << 16).view(np.float32)
    rng = np.random.default_rng(7)
    picks = np.concatenate([rng.choice(bits, 40), np.array([1, 2, 0x7F, 0x80, 0x81, 0x7F7F], np.uint32)])
    amaxes = list((picks << 16).view(np.float32)) + [np.float32(v) for v in (30.5, 24.5, 29.875, 448.0, 1.0)]
    for am in amaxes:
        x = allx[allx <= am]
        x = np.concatenate([x, -x])
        want = oracle.e4m3_encode(448.0 * x.astype(np.float64) / float(am))
        got = _codes(x, am)
        bad = np.nonzero(got != want)[0]
        assert bad.size == 0, "amax %r: %d codes differ, e.g. x = %r" % (float(am), bad.size, float(x[bad[0]]))


def test_the_plain_product_misses_ties():
    """The shortcut the kernel avoids: x times a rounded 448 / amax.  With
    amax = 24.5, x = 203/4096 gives x / scale = 0.90625, halfway between 0.875
    (even code) and 0.9375; fl(448 / 24.5) is a little large, so the product
    lands above the tie and rounds to the odd code."""
    am = np.float32(24.5)
    x = np.array([203.0 / 4096, -203.0 / 4096], np.float32)
    exact = oracle.e4m3_encode(448.0 * x.astype(np.float64) / 24.5)
    prod = (x * np.float32(np.float32(448.0) / am)).astype(np.float32)
    assert np.all(oracle.e4m3_encode(prod.astype(np.float64)) != exact)
    assert np.all(_codes(x, am) == exact)
