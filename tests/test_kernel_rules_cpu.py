"""Exhaustive CPU checks of the arithmetic shortcuts the CUDA kernels take in
place of a literal formula (no GPU). Each check emulates the kernel's steps in
exact (long double) arithmetic and compares the outcome with the oracle's
definition over every input that can reach it.

NVFP4 codes of bf16 values (rope_quant_insert_nvfp4, NoPE elements): the
kernel decides the E2M1 code of RN(x / s) from RN(x*yh + RN(x*yl)) with
yh = RD(1/s), yl = RN((1 - s*yh) * yh).
"""
import math

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


# ---------------------------------------------------------------------------
# Plain fp8 rows: the library's per-scale choice of quotient rule
# (kvq_plain_fp8_quotient_mode), against an independent numpy restatement.

def _e4m3_codes(q: np.ndarray) -> np.ndarray:
    """E4M3 bytes of binary32 values: nearest even on a 3-bit fraction
    (subnormal step 2^-9), NaN -> 0x7F, magnitudes >= 448 -> +-448."""
    q64 = q.astype(np.float64)
    sign = np.signbit(q64).astype(np.int64) << 7
    a = np.abs(q64)
    with np.errstate(all="ignore"):
        _, ex = np.frexp(np.where(a > 0, a, 1.0))
        e = ex - 1
        m = np.rint(np.ldexp(a, 3 - e))
        bump = m == 16
        e = np.where(bump, e + 1, e)
        m = np.where(bump, 8, m)
        normal = ((e + 7) << 3) | (m.astype(np.int64) - 8)
        sub = np.rint(a * 512.0).astype(np.int64)
    codes = np.where(a < 2.0 ** -6, sub, normal)
    codes = np.where(a >= 448.0, 0x7E, codes) | sign
    return np.where(np.isnan(q64), 0x7F, codes)


def _expected_mode(scale: float) -> int:
    s = np.float32(scale)
    frac, ex = math.frexp(float(s))
    if frac == 0.5 and -124 <= ex <= 127:
        return 2
    yh = np.float32(1.0) / s
    if np.float64(1.0) - np.float64(s) * np.float64(yh) < 0:
        yh = np.nextafter(yh, np.float32(0))
    yl = np.float32(np.float32(np.float64(1.0) - np.float64(s) * np.float64(yh)) * yh)
    x = _bf16_values_all()
    with np.errstate(all="ignore"):
        q = x / s
        t = (x * yl).astype(np.float32)
        fast = (x.astype(np.float64) * np.float64(yh) + t.astype(np.float64)).astype(np.float32)
    return 1 if np.array_equal(_e4m3_codes(q), _e4m3_codes(fast)) else 0


def _bf16_values_all() -> np.ndarray:
    return (np.arange(65536, dtype=np.uint32) << 16).view(np.float32)


def test_e4m3_restatement_on_known_bytes():
    vals = np.array([0.0, -0.0, 448.0, 464.0, 1e9, np.inf, -np.inf, np.nan, 2.0 ** -9,
                     2.0 ** -10, 3 * 2.0 ** -11, 1.0, 1.0625, 1.1875, 240.0, -0.75],
                    np.float32)
    # 2^-10 is half the subnormal step (tie to 0), 3*2^-11 three quarters
    # of it (rounds to 1), 1.0625 and 1.1875 ties to the even fraction
    want = [0x00, 0x80, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0x7F, 0x01,
            0x00, 0x01, 0x38, 0x38, 0x3A, 0x77, 0xB4]
    assert _e4m3_codes(vals).tolist() == want


@pytest.mark.parametrize("scale", [1.0, 0.5, 4.0, 2.0 ** -126, 0.0125, 0.1, 0.9375, 3.7, 1e-3,
                                   1e-30, 1.5e-38, 1e38, 3.0e38])
def test_plain_fp8_quotient_mode_matches_an_independent_check(scale):
    import fp8_quantized_paged_store_gb300 as kvq
    assert kvq.lib().kvq_plain_fp8_quotient_mode(scale) == _expected_mode(scale)


def test_plain_fp8_quotient_mode_rejects_bad_scales():
    import fp8_quantized_paged_store_gb300 as kvq
    for bad in (0.0, -1.0, float("nan"), float("inf")):
        assert kvq.lib().kvq_plain_fp8_quotient_mode(bad) == -1


# ---------------------------------------------------------------------------
# NVFP4 codes of binary32 rotary values (rope_quant_insert_nvfp4, elements
# 448..511): the kernel decides the E2M1 code of RN(r / s) from
# q = RN(r*yh + RN(r*yl)) + 0.0 with the same two-term reciprocal, for any
# binary32 r (no range check, no division).

_MIDPOINTS = (0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0)


def _rotary_codes_kernel(r, yh, yl):
    """The kernel's steps: t = RN(r*yl), q = RN(r*yh + t) (one rounding of the
    exact sum), q + 0.0; then the GPU conversion, whose code for -0 is 8."""
    with np.errstate(all="ignore"):
        t = (r * yl).astype(np.float32)
        q = (r.astype(LD) * LD(yh) + t.astype(LD)).astype(np.float32)
        q = (q + np.float32(0)).astype(np.float32)
    got = oracle.e2m1_code(q)
    return np.where(np.signbit(q) & (got == 0), 8, got)


def _rotary_codes_oracle(r, s):
    with np.errstate(all="ignore"):
        return oracle.e2m1_code((r / s).astype(np.float32))


def _around(v, k=3):
    """The binary32 values nearest the real v (given in long double), k on
    each side of RN(v), both signs."""
    f = np.float32(v)
    vals = [f]
    lo = hi = f
    for _ in range(k):
        lo = np.nextafter(lo, np.float32(-np.inf))
        hi = np.nextafter(hi, np.float32(np.inf))
        vals += [lo, hi]
    a = np.array(vals, np.float32)
    return np.concatenate([a, -a])


@pytest.mark.skipif(np.finfo(LD).nmant < 63, reason="needs 64-bit long double mantissa")
def test_nvfp4_rotary_two_term_decides_every_code_near_every_midpoint():
    """For every positive E4M3 scale s and every E2M1 midpoint M, the binary32
    r closest to M*s and to B*s for both binary32 rounding boundaries B next
    to M (the only places where a one-unit difference between q and RN(r/s)
    could change the code): codes equal. The r closest to B*s keep r/s more
    than 2**-28 (relative) from B (the minimum over all cases is 2**-27.9),
    while q's sum is within 2**-44 of r/s: no r anywhere can land between."""
    min_margin = 1.0
    for sb in range(1, 127):
        s = np.float32(oracle.e4m3_decode(np.array([sb], np.uint8))[0])
        yh, yl = _two_term(s)
        for m in _MIDPOINTS:
            mf = np.float32(m)
            up = LD(np.nextafter(mf, np.float32(np.inf))) - LD(mf)
            down = LD(mf) - LD(np.nextafter(mf, np.float32(0)))
            for b in (LD(mf), LD(mf) + up / 2, LD(mf) - down / 2):
                r = _around(b * LD(s))
                want = _rotary_codes_oracle(r, s)
                got = _rotary_codes_kernel(r, yh, yl)
                bad = np.nonzero(got != want)[0]
                assert bad.size == 0, (sb, m, r[bad[:3]], want[bad[:3]], got[bad[:3]])
                if b != LD(mf):
                    rel = np.abs(r.astype(LD) / LD(s) - b * np.sign(r.astype(LD))) / b
                    min_margin = min(min_margin, float(rel.min()))
    assert min_margin > 2.0 ** -28, min_margin


@pytest.mark.skipif(np.finfo(LD).nmant < 63, reason="needs 64-bit long double mantissa")
def test_nvfp4_rotary_two_term_random_and_special_values():
    """Random binary32 values over the codes' whole range at every scale,
    plus zeros of both signs, quotients that underflow to -0, subnormals,
    huge values and (with s = 448, the only scale an infinite tile reaches)
    infinities."""
    rng = np.random.default_rng(11)
    special = np.array([0.0, -0.0, 2.0 ** -149, -2.0 ** -149, -2.0 ** -140, 1e-38, -1e-38,
                        3e38, -3e38, 2.0 ** 100, -2.0 ** 100], np.float32)
    for sb in range(1, 127):
        s = np.float32(oracle.e4m3_decode(np.array([sb], np.uint8))[0])
        yh, yl = _two_term(s)
        r = (rng.uniform(-8, 8, 20_000) * s).astype(np.float32)
        wide = (rng.standard_normal(2_000) * np.exp2(rng.uniform(-140, 120, 2_000)))
        r = np.concatenate([r, wide.astype(np.float32), special])
        if s == np.float32(448):
            r = np.concatenate([r, np.array([np.inf, -np.inf], np.float32)])
        bad = np.nonzero(_rotary_codes_kernel(r, yh, yl) != _rotary_codes_oracle(r, s))[0]
        assert bad.size == 0, (sb, r[bad[:3]])
