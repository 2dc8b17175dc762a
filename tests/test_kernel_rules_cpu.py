"""Exhaustive CPU checks of the arithmetic shortcuts the CUDA kernels take in
place of a literal formula (no GPU). Each check emulates the kernel's steps in
exact (long double) arithmetic and compares the outcome with the oracle's
definition over every input that can reach it.

NVFP4 codes of bf16 values (rope_quant_insert_nvfp4, NoPE elements): the
kernel decides the E2M1 code of RN(x / s) from RN(x*yh + RN(x*yl)) with
yh = RD(1/s), yl = RN((1 - s*yh) * yh).
"""
import numpy as np
import pytest

import oracle

LD = np.longdouble


def _bf16_values():
    bits = np.arange(65536, dtype=np.uint32)
    x = (bits << 16).view(np.float32)
    return x[~np.isnan(x) & (x != 0)]


def _two_term(s):
    yh = np.float32(LD(1) / LD(s))
    if LD(yh) > LD(1) / LD(s):
        yh = np.nextafter(yh, np.float32(0))
    r_exact = LD(1) - LD(s) * LD(yh)
    r = np.float32(r_exact)
    assert LD(r) == r_exact and r >= 0          # the kernel's fma gives it exactly
    return yh, np.float32(r * yh)


@pytest.mark.skipif(np.finfo(LD).nmant < 63, reason="needs 64-bit long double mantissa")
def test_nvfp4_two_term_reciprocal_decides_every_code():
    x = _bf16_values()
    finite = np.isfinite(x)
    for sb in range(1, 127):
        s = np.float32(oracle.e4m3_decode(np.array([sb], np.uint8))[0])
        yh, yl = _two_term(s)
        assert yl >= 0 and (yl > 0 or LD(yh) * LD(s) == 1)
        with np.errstate(all="ignore"):
            want = oracle.e2m1_code((x / s).astype(np.float32))
            t = (x * yl).astype(np.float32)
            q = (x.astype(LD) * LD(yh) + t.astype(LD)).astype(np.float32)  # one rounding
        got = oracle.e2m1_code(q)
        got = np.where(np.signbit(q) & (got == 0), 8, got)  # the GPU cvt keeps -0's sign
        # infinite values only meet s = 448 (an infinite amax clamps there)
        sel = finite if s != 448 else np.ones_like(finite)
        bad = np.nonzero((got != want) & sel)[0]
        assert bad.size == 0, (sb, x[bad[:3]], want[bad[:3]], got[bad[:3]])


def test_nvfp4_plain_reciprocal_is_not_enough():
    """Why two terms: RN(x * RN(1/s)) alone mis-rounds midpoint ties for the
    scales with significand 1.875 (e.g. s = 0.9375, x = 1.171875)."""
    s = np.float32(0.9375)
    x = np.float32(1.171875)                    # x / s = 1.25, a tie that goes down
    assert oracle.e2m1_code(np.array([x / s], np.float32))[0] == 2
    y = np.float32(1) / s
    assert oracle.e2m1_code(np.array([x * y], np.float32))[0] == 3
