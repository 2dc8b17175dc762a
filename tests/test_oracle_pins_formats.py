"""Pins of the oracle's format primitives against what the pages and the
format definitions fix (CPU only).

Pages: 'vllm.v1.attention.ops.mxfp4_mla.store' (module docstring,
_ceil_pow2_exponent, _quantize_e2m1); PR 60321 'Add an mxfp4_mla KV cache for
rope-free sparse MLA' (Overview, Claims, Details, review thread);
'vllm.models.deepseek_v41.common.ops.fused_compress_quant_cache' (the two
V4.1 insert kernels).
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
from tests import _independent as ind


def _all_bf16_bits():
    return np.arange(65536, dtype=np.uint32).astype(np.uint16)


def test_format_constants(golden_dir):
    with open(os.path.join(golden_dir, "format_constants.json")) as f:
        g = json.load(f)
    assert oracle.row_bytes(g["latent"], g["group"]) == g["row_bytes_512"]
    assert round(g["bf16_row_bytes_512"] / g["row_bytes_512"], 2) == g["capacity_ratio_2dp"]
    # Power-of-two ranks >= 128 give a pitch that is a multiple of 4.
    for d in (128, 256, 512, 1024, 2048):
        assert oracle.row_bytes(d, 32) % 4 == 0
    # MXFP8 and NVFP4 record widths add up to the dispatcher's keys.
    r8, r4 = g["mxfp8_record"], g["nvfp4_record"]
    assert r8["value_bytes"] + r8["scale_bytes"] == g["record_bytes"]["v41_mxfp8"]
    assert r4["code_bytes"] + r4["scale_bytes"] == g["record_bytes"]["v41_nvfp4"]
    assert 512 // r8["group"] == r8["scale_bytes"] and 512 // r4["group"] == r4["scale_bytes"]
    # The E2M1 value set and its midpoints.
    vals = oracle.e2m1_value(np.arange(16, dtype=np.uint8))
    mags = np.array(g["e2m1_magnitudes"], dtype=np.float32)
    assert np.array_equal(vals[:8], mags)
    assert np.array_equal(vals[8:], -mags) and all(np.signbit(vals[8:]))
    mids = (mags[:-1] + mags[1:]) / 2
    assert np.array_equal(mids, np.array(g["e2m1_midpoints"], dtype=np.float32))
    assert mags.max() == g["e2m1_max"]
    assert float(oracle.e4m3_decode(np.array([0x7E], np.uint8))[0]) == g["e4m3_max"]
    assert float(oracle.e4m3_decode(np.array([0x01], np.uint8))[0]) == g["nvfp4_scale_min"]


def test_e2m1_value_matches_bitfield_definition():
    got = oracle.e2m1_value(np.arange(16, dtype=np.uint8))
    want = np.array([ind.e2m1_decode_from_bits(c) for c in range(16)], dtype=np.float32)
    assert np.array_equal(got, want)
    assert np.array_equal(np.signbit(got), np.signbit(want))


def test_e2m1_midpoints_golden(golden_dir):
    xs, want = [], []
    with open(os.path.join(golden_dir, "e2m1_midpoints.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                a, b = line.split()
                xs.append(float(a))
                want.append(int(b))
    got = oracle.e2m1_code(np.array(xs, dtype=np.float32))
    assert got.tolist() == want


def test_e2m1_special_inputs():
    x = np.array([0.0, -0.0, np.nan, -np.nan, np.inf, -np.inf, 1e-45, -1e-45], np.float32)
    # -0.0 and NaN do not compare below zero; +-inf saturate; a negative
    # subnormal still compares below zero.
    assert oracle.e2m1_code(x).tolist() == [0, 0, 0, 0, 7, 15, 0, 8]


def test_e2m1_brute_force_every_bf16_at_every_scale():
    """Every bf16 pattern x and every exponent e in [-126, 126]: the code of
    x * 2**-e equals the nearest-value search (65,536 x 253 cases)."""
    x = ind.bf16_bits_to_f32(_all_bf16_bits())
    for e in range(-126, 127):
        with np.errstate(over="ignore", invalid="ignore"):
            normalized = x * np.float32(2.0 ** -e)
        got = oracle.e2m1_code(normalized)
        want = ind.e2m1_nearest_code(normalized)
        bad = np.nonzero(got != want)[0]
        assert bad.size == 0, (e, bad[:5], normalized[bad[:5]], got[bad[:5]], want[bad[:5]])


def test_e2m1_brute_force_random_binary32():
    rng = np.random.default_rng(1)
    bits = rng.integers(0, 2 ** 32, size=2_000_000, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    x = np.concatenate([x, rng.uniform(-7, 7, 1_000_000).astype(np.float32)])
    assert np.array_equal(oracle.e2m1_code(x), ind.e2m1_nearest_code(x))


def test_ceil_pow2_exponent_is_exact_ceil_log2():
    rng = np.random.default_rng(2)
    # normal binary32: random patterns plus every power of two and its neighbours
    bits = rng.integers(0x00800000, 0x7F800000, size=1_000_000, dtype=np.uint64).astype(np.uint32)
    p = (np.arange(1, 255, dtype=np.uint32) << 23)
    bits = np.concatenate([bits, p, p + 1, p - 1])
    bits = bits[(bits >= 0x00800000) & (bits < 0x7F800000)]
    v = bits.view(np.float32)
    got = oracle.ceil_pow2_exponent(v)
    assert np.array_equal(got, ind.smallest_pow2_exponent_at_least(v))
    # The bit rule read literally: subnormals give -126, +inf gives 128.
    sub = np.array([1, 2, 0x7FFFFF, 0x400000], np.uint32).view(np.float32)
    assert oracle.ceil_pow2_exponent(sub).tolist() == [-126] * 4
    assert oracle.ceil_pow2_exponent(np.array([np.inf], np.float32)).tolist() == [128]


def _positive_finite_bf16():
    b = np.arange(1, 0x7F80, dtype=np.uint32).astype(np.uint16)
    return ind.bf16_bits_to_f32(b)


def test_mxfp4_scale_never_clamps_and_is_minimal():
    """For every positive finite bf16 amax: amax <= 6 * 2**e (no value clamps),
    and e is the smallest such integer wherever amax/6 is a normal binary32.
    Where amax/6 is subnormal the bit rule gives e = -126 (byte 1)."""
    amax = _positive_finite_bf16()
    e = oracle.mxfp4_scale_exponent(amax).astype(np.int64)
    a64 = amax.astype(np.float64)
    assert np.all(a64 <= 6.0 * np.exp2(e.astype(np.float64)))  # exact in float64
    normal = a64 >= 6.0 * 2.0 ** -126
    assert np.all(a64[normal] > 6.0 * np.exp2(e[normal].astype(np.float64) - 1.0))
    assert np.all(e[~normal] == -126)
    assert e.min() == -126 and e.max() == 126


def test_mxfp4_scale_power_of_two_times_six_lands_on_six():
    k = np.arange(-126, 126)
    amax = (6.0 * np.exp2(k.astype(np.float64))).astype(np.float32)
    e = oracle.mxfp4_scale_exponent(amax)
    assert np.array_equal(e, k)
    # ... so the amax element normalizes to exactly 6 and takes code 7.
    normalized = amax * np.exp2(-e.astype(np.float64)).astype(np.float32)
    assert np.all(normalized == 6.0)
    assert np.all(oracle.e2m1_code(normalized) == 7)


def test_mxfp4_scale_division_and_reciprocal_readings_agree():
    """RN32(amax / 6) and RN32(amax * fl32(1/6)) give the same exponent for
    every positive finite bf16 amax, so the two possible readings of the
    unprinted scale formula coincide."""
    amax = _positive_finite_bf16()
    by_div = oracle.ceil_pow2_exponent(amax / np.float32(6.0))
    by_mul = oracle.ceil_pow2_exponent(amax * np.float32(1.0 / 6.0))
    assert np.array_equal(by_div, by_mul)
    assert np.array_equal(oracle.mxfp4_scale_exponent(amax), by_div)


def test_mxfp4_zero_group_scale_is_127():
    assert oracle.mxfp4_scale_exponent(np.zeros(1, np.float32)).tolist() == [0]


def test_e4m3_decode_matches_bitfield_definition():
    got = oracle.e4m3_decode(np.arange(256, dtype=np.uint8)).astype(np.float64)
    want = ind.E4M3_TABLE
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan) and nan.sum() == 2
    assert np.array_equal(got[~nan], want[~nan])


def test_e4m3_encode_brute_force():
    pos = ind.E4M3_TABLE[:127]
    mids = (pos[:-1] + pos[1:]) / 2
    pts = np.concatenate([pos, mids]).astype(np.float32)  # midpoints are exact
    b = pts.view(np.uint32)
    near = np.concatenate([b, b + 1, b - 1, b + 2, b - 2]).view(np.float32)
    rng = np.random.default_rng(3)
    rand = np.concatenate([rng.uniform(-448, 448, 500_000),
                           rng.uniform(-0.02, 0.02, 500_000),
                           np.exp2(rng.uniform(-14, 8.8, 500_000))]).astype(np.float32)
    y = np.concatenate([near, -near, rand, [0.0, -0.0, 448.0, -448.0]]).astype(np.float32)
    y = y[np.isfinite(y) & (np.abs(y) <= 448.0)]
    got = oracle.e4m3_encode(y)
    want = ind.e4m3_nearest(y)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, (y[bad[:5]], got[bad[:5]], want[bad[:5]])


def test_e4m3_named_values():
    y = np.array([448.0, -448.0, 1.0, 2.0 ** -9, 2.0 ** -6, -0.0, 0.0, np.nan, 2.0 ** -10,
                  3 * 2.0 ** -11, 240.0, 0.1], np.float32)
    want = [0x7E, 0xFE, 0x38, 0x01, 0x08, 0x80, 0x00, 0x7F, 0x00, 0x01, 0x77, 0x1D]
    assert oracle.e4m3_encode(y).tolist() == want
