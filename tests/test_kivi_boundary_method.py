"""The fp16 code-boundary method of the 2-bit KIVI kernels, restated on the CPU and checked
against the oracle (no GPU).

The 2-bit flush and pack decide an element's code by fp16 compares against three per-group
boundaries: for each threshold t of the threshold form (code >= k iff RN32(x - gmin) >= t_k), the
smallest fp16 value X with RN32(X - gmin) >= t.  This module restates that selection in float32
numpy -- the guess fp16(gmin + t), its neighbours, a bisection over the fp16 order keys -- and
checks that counting the boundaries each element reaches gives the oracle's codes for every fp16
value of the same thirteen groups the GPU sweep uses.  It pins the method itself; the GPU tests
pin the kernels to the oracle.
"""
from fractions import Fraction

import numpy as np
import pytest

from oracle import kivi as ok

f32 = np.float32
_ALL = np.arange(65536, dtype=np.uint32).astype(np.uint16).view(np.float16)
_FINITE = np.sort(_ALL[np.isfinite(_ALL)].astype(np.float32), kind="stable").astype(np.float16)
KEY_NEG_INF, KEY_POS_INF, NEVER = 0x03FF, 0xFC00, 0x7FFF


def _key(b):
    return b ^ (0xFFFF if b & 0x8000 else 0x8000)


def _bits(k):
    return k ^ (0x8000 if k & 0x8000 else 0xFFFF)


def _h2f(b):
    return np.array([b], np.uint16).view(np.float16)[0].astype(np.float32)


def _f2h(x):
    with np.errstate(over="ignore"):
        return int(np.array([x], np.float32).astype(np.float16).view(np.uint16)[0])


def _reaches(k, z, t):
    with np.errstate(all="ignore"):
        return f32(_h2f(_bits(k)) - z) >= t


def first_reaching(z, t):
    """fp16 bits of the smallest non-NaN fp16 X with RN32(X - z) >= t, or NEVER."""
    with np.errstate(all="ignore"):
        k = _key(_f2h(f32(z + t)))
    k = min(max(k, KEY_NEG_INF + 1), KEY_POS_INF)
    if _reaches(k, z, t):
        if not _reaches(k - 1, z, t):
            return _bits(k)
        lo, hi = KEY_NEG_INF, k - 1
    else:
        if k == KEY_POS_INF:
            return NEVER
        if _reaches(k + 1, z, t):
            return _bits(k + 1)
        if not _reaches(KEY_POS_INF, z, t):
            return NEVER
        lo, hi = k + 1, KEY_POS_INF
    while hi - lo > 1:
        m = (lo + hi) >> 1
        if _reaches(m, z, t):
            hi = m
        else:
            lo = m
    return _bits(hi)


def _fma_ru(a, b, c):
    """float32 fma rounded toward +inf, from the exact rational value."""
    e = Fraction(float(a)) * Fraction(float(b)) + Fraction(float(c))
    r = f32(float(e))
    if Fraction(float(r)) < e:
        r = np.nextafter(r, f32(np.inf))
    elif Fraction(float(r)) - e >= Fraction(float(np.spacing(r))):
        r = np.nextafter(r, f32(-np.inf))
    return r


def thresholds(scale):
    """t1, t2, t3 of the threshold form: code >= k iff RN32(x - gmin) >= t_k."""
    if scale == 0:
        return [f32(np.inf)] * 3
    return [_fma_ru(scale, f32(0.5), f32(scale * f32(2.0 ** -25))),
            _fma_ru(scale, f32(1.5), -f32(scale * f32(2.0 ** -24))),
            _fma_ru(scale, f32(2.5), f32(scale * f32(2.0 ** -23)))]


CASES = [(-1.0, 1.0, 1e-8), (-1000.0, 1000.0, 1e-8), (-65504.0, 65504.0, 1e-8),
         (-2.0 ** -14, 2.0 ** -14, 1e-8), (0.0, 2.25, 1e-8), (-3.0, -1.0, 1e-8),
         (5.0, 5.0078125, 1e-8), (-0.0, 3 * 2.0 ** -24, 1e-8), (-0.001, 3000.0, 1e-8),
         (60000.0, 65504.0, 1e-8), (-65504.0, -60000.0, 1e-8), (-0.5, 0.75, 1e-3),
         (-1e-4, 1e-4, 1e-3)]


@pytest.mark.parametrize("mn,mx,eps", CASES)
def test_boundary_counts_equal_the_oracle_codes(mn, mx, eps):
    lo16, hi16 = np.float16(mn), np.float16(mx)
    vals = _FINITE[(_FINITE >= lo16) & (_FINITE <= hi16)]
    z = f32(lo16)
    scale = max(f32(f32(f32(hi16) - z) / f32(3)), f32(eps))
    cuts = [first_reaching(z, t) for t in thresholds(scale)]
    x = vals.astype(np.float32)
    codes = np.zeros(len(vals), np.int64)
    for b in cuts:
        if b != NEVER:
            codes += x >= _h2f(b)          # fp16 values compare exactly as float32
    recon = np.array([np.float16(f32(f32(c) * scale) + z) for c in range(4)])
    group = np.concatenate([[lo16, hi16], vals]).astype(np.float16)
    want = ok.quant_dequant_along(group[None, :], -1, len(group), 3, eps)[0][2:]
    assert np.array_equal(recon[codes].view(np.uint16), want.view(np.uint16))


def test_the_bisection_runs_where_fp16_values_share_a_difference():
    """Around zero the fp16 spacing falls far below the ulp of x - gmin: there the guess and its
    neighbours do not settle and the bisection decides (the symmetric groups' middle boundary)."""
    z = f32(np.float16(-1000.0))
    t = thresholds(max(f32(f32(2000.0) / f32(3)), f32(1e-8)))[1]
    b = first_reaching(z, t)
    k = _key(b)
    assert _reaches(k, z, t) and not _reaches(k - 1, z, t)
    guess = _key(_f2h(f32(z + t)))
    assert abs(guess - k) > 1
