"""Pins of the oracle's RMSNorm ahead of the MXFP4 store (CPU only).

Pages: 'vllm.v1.attention.ops.mxfp4_mla.store' (store_mxfp4_mla takes the
post-RMSNorm latent) and 'vllm.models.deepseek_v41.common.ops.
fused_compress_quant_cache' (fused_save_compress_norm: bf16 [512] weight, fp32
epsilon, bf16 latent out). The pages fix no summation order: the library fixes
one as part of its interface (block k = elements 8k..8k+7 then
256+8k..256+8k+7, summed left to right; the 32 block sums added as a balanced
pairwise tree). The pins below check the formula against float64, against
cases where the result is exact whatever the order, and the order itself
against a hand-derived row on which three different orders give three
different outputs (tests/golden/rmsnorm_order_worked.json).
"""
import json
import os

import numpy as np

import oracle
import workloads
from tests import _independent as ind


def _bf16(a):
    return workloads.f32_to_bf16_bits(np.asarray(a, np.float32))


def _ulp_distance(a_bits, b_bits):
    """Distance in bf16 units in the last place (same-sign values)."""
    a = a_bits.astype(np.int32)
    b = b_bits.astype(np.int32)
    a = np.where(a & 0x8000, -(a & 0x7FFF), a)
    b = np.where(b & 0x8000, -(b & 0x7FFF), b)
    return np.abs(a - b)


def test_rmsnorm_matches_float64_within_one_ulp():
    rng = np.random.default_rng(3)
    x = _bf16(rng.standard_normal((300, 512)) * np.exp2(rng.uniform(-20, 20, (300, 1))))
    w = _bf16(rng.uniform(0.5, 1.5, 512))
    eps = np.float32(1e-6)
    got = oracle.rmsnorm_rows(x, w, float(eps))
    xf = ind.bf16_bits_to_f32(x).astype(np.float64)
    r = 1.0 / np.sqrt(np.mean(xf * xf, axis=1, keepdims=True) + float(eps))
    y = _bf16((xf * r).astype(np.float32))
    want = _bf16(ind.bf16_bits_to_f32(y).astype(np.float64) * ind.bf16_bits_to_f32(w))
    d = _ulp_distance(got, want)
    assert d.max() <= 1
    assert np.mean(d == 0) > 0.999


def test_rmsnorm_constant_row_is_exactly_one():
    x = np.full((2, 512), 0x4040, np.uint16)   # 3.0
    x[1] = 0xC040                              # -3.0
    w = np.full(512, 0x3F80, np.uint16)
    got = oracle.rmsnorm_rows(x, w, 0.0)
    assert np.all(got[0] == 0x3F80) and np.all(got[1] == 0xBF80)


def test_rmsnorm_scale_invariance_without_eps():
    rng = np.random.default_rng(4)
    x = _bf16(rng.standard_normal((64, 512)))
    w = _bf16(rng.uniform(0.5, 1.5, 512))
    xf = ind.bf16_bits_to_f32(x)
    for k in (-8, 2, 10):
        x2 = _bf16(xf * np.float32(2.0 ** k))           # exact power-of-two scaling
        assert np.array_equal(oracle.rmsnorm_rows(x2, w, 0.0), oracle.rmsnorm_rows(x, w, 0.0))


def test_rmsnorm_weight_power_of_two_scales_exactly():
    rng = np.random.default_rng(5)
    x = _bf16(rng.standard_normal((64, 512)))
    ones = np.full(512, 0x3F80, np.uint16)
    twos = np.full(512, 0x4000, np.uint16)
    z1 = ind.bf16_bits_to_f32(oracle.rmsnorm_rows(x, ones, 1e-6))
    z2 = ind.bf16_bits_to_f32(oracle.rmsnorm_rows(x, twos, 1e-6))
    assert np.array_equal(z2, z1 * np.float32(2.0))


def test_rmsnorm_eps_sits_inside_the_root():
    """All-zero row: mean 0, r = 1/sqrt(eps); a row of tiny values c with
    c*c << eps normalises to c / sqrt(eps)."""
    x = np.zeros((1, 512), np.uint16)
    x[0, 0] = 0x2F80                            # 2**-32, square 2**-64 << eps
    w = np.full(512, 0x3F80, np.uint16)
    got = ind.bf16_bits_to_f32(oracle.rmsnorm_rows(x, w, 2.0 ** -20))
    assert got[0, 0] == np.float32(2.0 ** -32 * 2.0 ** 10) and np.all(got[0, 1:] == 0)


def test_fused_store_equals_rmsnorm_then_store():
    rng = np.random.default_rng(6)
    T = 100
    x = _bf16(rng.standard_normal((T, 512)) * 3)
    w = _bf16(rng.uniform(0.5, 1.5, 512))
    slots = rng.permutation(128)[:T].astype(np.int64)
    slots[::9] = -1
    a = np.full(128 * 272, 0xAA, np.uint8)
    b = a.copy()
    oracle.mxfp4_mla_rmsnorm_store(x, w, 1e-5, slots, a, 1, 128, 128)
    oracle.mxfp4_mla_store(oracle.rmsnorm_rows(x, w, 1e-5), slots, b, 1, 128, 128)
    assert np.array_equal(a, b)


GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "rmsnorm_order_worked.json")


def _order_row():
    g = json.load(open(GOLDEN))
    x = np.full(512, 0x3F80, np.uint16)                     # ones
    x[6:8] = 0
    x[256:264] = 0
    for j, v in g["row"]["values"].items():
        x[int(j)] = _bf16(np.float32([v]))[0]
    eps = float(np.array([int(g["row"]["eps_f32_hex"], 16)], np.uint32).view(np.float32)[0])
    return g, x, eps


def _expected(spec):
    want = np.full(512, int(spec["ones"], 16), np.uint16)
    want[6:8] = int(spec["zeros"], 16)
    want[256:264] = int(spec["zeros"], 16)
    for j in range(6):
        want[j] = int(spec[str(j)], 16)
    return want


def test_rmsnorm_summation_order_golden():
    """The library's order (blocks of 8k..8k+7, 256+8k..256+8k+7, then a
    pairwise tree) gives the hand-derived row; the run-of-16 order and a
    left-to-right sum would give other rows."""
    g, x, eps = _order_row()
    assert eps == np.float32(1e-6)
    w = np.full(512, 0x3F80, np.uint16)
    rows = {k: _expected(v) for k, v in g["expected_bf16_hex"].items()}
    assert not np.array_equal(rows["contract"], rows["run16"])
    assert not np.array_equal(rows["run16"], rows["sequential"])
    assert not np.array_equal(rows["contract"], rows["sequential"])
    got = oracle.rmsnorm_rows(x[None, :], w, eps)[0]
    assert np.array_equal(got, rows["contract"]), [
        (j, hex(got[j]), hex(rows["contract"][j])) for j in np.nonzero(got != rows["contract"])[0]]


def test_rmsnorm_order_golden_row_is_what_the_derivation_says():
    """The fixture's own arithmetic, checked with exact integers: the three
    sums of squares and the fact that eps vanishes next to S/512."""
    g, x, eps = _order_row()
    v = ind.bf16_bits_to_f32(x).astype(np.float64)
    assert np.sum(v != 0) == 502 and np.sum(v == 1.0) == 496
    exact = int(np.sum(v * v))
    assert exact == 2 ** 24 + 213344 + 496
    assert eps < 2.0 ** -9   # below half the binary32 spacing at S/512 ~ 33185
