"""Pins of the sparse-attention oracle (CPU only): closed forms and invariances
that hold whatever the implementation, plus a brute-force loop on a tiny case.

Page: PR 60321 "Add an mxfp4_mla KV cache dtype..." (Read path: gather the
top-k rows, unpack to bf16, two dots; Claims: attention over the packed cache
equals attention over the dequantized bf16 values).
"""
import math

import numpy as np
import pytest

import oracle
import workloads
from oracle.attention import mxfp4_mla_sparse_attention as attn


def _cache(rows_f32, num_slots=None):
    """Store fp32 rows (rounded to bf16) into a flat MXFP4 cache, row i in slot i."""
    lat = workloads.f32_to_bf16_bits(np.asarray(rows_f32, np.float32))
    n = lat.shape[0] if num_slots is None else num_slots
    cache = np.zeros(n * 272, np.uint8)
    oracle.mxfp4_mla_store(lat, np.arange(lat.shape[0], dtype=np.int64), cache, 1, n, n)
    deq = oracle.mxfp4_mla_gather_dequant(cache, 1, n, n, np.arange(n, dtype=np.int64))
    return cache, (deq.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _q(rows_f32):
    return workloads.f32_to_bf16_bits(np.asarray(rows_f32, np.float32))


def _bf(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def test_single_valid_key_returns_its_row():
    rng = np.random.default_rng(1)
    cache, k = _cache(rng.standard_normal((8, 512)))
    q = _q(rng.standard_normal((1, 4, 512)))
    idx = np.array([[-1, 5, -1, 99]], np.int64)          # 99 is past the 8 slots
    out, lse, mass = attn(q, cache, 1, 8, 8, idx, 0.1)
    assert np.array_equal(out[0], np.broadcast_to(k[5], (4, 512)))
    assert np.array_equal(mass[0], np.broadcast_to(np.abs(k[5]), (4, 512)))
    np.testing.assert_allclose(lse[0], 0.1 * (_bf(q[0]) @ k[5]), rtol=1e-15)


def test_zero_scale_is_the_mean_of_the_valid_rows():
    rng = np.random.default_rng(2)
    cache, k = _cache(rng.standard_normal((16, 512)))
    q = _q(rng.standard_normal((2, 3, 512)))
    idx = np.array([[0, 3, 7, -1, 15, 3], [2, -5, 4, 6, 8, 10]], np.int64)
    out, lse, _ = attn(q, cache, 1, 16, 16, idx, 0.0)
    # a repeated index counts twice: it is two entries of the softmax
    np.testing.assert_allclose(out[0], np.broadcast_to(k[[0, 3, 7, 15, 3]].mean(0), (3, 512)),
                               rtol=1e-13, atol=1e-300)
    np.testing.assert_allclose(out[1], np.broadcast_to(k[[2, 4, 6, 8, 10]].mean(0), (3, 512)),
                               rtol=1e-13, atol=1e-300)
    np.testing.assert_allclose(lse, [[math.log(5)] * 3] * 2, rtol=1e-15)


def test_two_keys_give_the_logistic_weights():
    """Rows a and b with q.a - q.b known exactly: out = w a + (1 - w) b with
    w = 1 / (1 + exp(-scale * (q.a - q.b)))."""
    a = np.zeros(512); a[0] = 1.0; a[100] = -2.0
    b = np.zeros(512); b[1] = 1.5; b[300] = 0.5
    cache, k = _cache(np.stack([a, b]))
    assert np.array_equal(k[0], a) and np.array_equal(k[1], b)   # exact in MXFP4
    q = np.zeros((1, 2, 512)); q[0, 0, 0] = 3.0; q[0, 1, 1] = 2.0
    qb = _q(q)
    out, lse, _ = attn(qb, cache, 1, 2, 2, np.array([[0, 1]], np.int64), 0.5)
    for h, (sa, sb) in enumerate([(3.0, 0.0), (0.0, 3.0)]):
        w = 1.0 / (1.0 + math.exp(-0.5 * (sa - sb)))
        np.testing.assert_allclose(out[0, h], w * a + (1 - w) * b, rtol=1e-14, atol=1e-300)
        np.testing.assert_allclose(lse[0, h], math.log(math.exp(0.5 * sa) + math.exp(0.5 * sb)),
                                   rtol=1e-14)


def test_identical_rows_give_that_row():
    rng = np.random.default_rng(3)
    row = rng.standard_normal(512)
    cache, k = _cache(np.tile(row, (6, 1)))
    q = _q(rng.standard_normal((1, 5, 512)) * 10)
    out, _, _ = attn(q, cache, 1, 6, 6, np.arange(6, dtype=np.int64)[None], 1.0)
    np.testing.assert_allclose(out[0], np.broadcast_to(k[0], (5, 512)), rtol=1e-13, atol=1e-300)


def test_pads_are_dropped_and_order_does_not_matter():
    rng = np.random.default_rng(4)
    cache, _ = _cache(rng.standard_normal((64, 512)))
    q = _q(rng.standard_normal((1, 4, 512)))
    base = rng.permutation(64)[:20].astype(np.int64)
    padded = np.concatenate([base, [-1, -7, 64, 1000]])
    rng.shuffle(padded)
    o1, l1, _ = attn(q, cache, 1, 64, 64, base[None], 0.07)
    o2, l2, _ = attn(q, cache, 1, 64, 64, padded[None], 0.07)
    np.testing.assert_allclose(o2, o1, rtol=1e-12, atol=1e-300)
    np.testing.assert_allclose(l2, l1, rtol=1e-14)


def test_no_valid_index_gives_zero_and_minus_infinity():
    rng = np.random.default_rng(5)
    cache, _ = _cache(rng.standard_normal((4, 512)))
    q = _q(rng.standard_normal((2, 2, 512)))
    out, lse, mass = attn(q, cache, 1, 4, 4, np.array([[-1, -1], [4, 9]], np.int64), 1.0)
    assert np.all(out == 0) and np.all(mass == 0) and np.all(np.isneginf(lse))


def test_large_scores_stay_finite_and_pick_the_best_key():
    rng = np.random.default_rng(6)
    cache, k = _cache(rng.standard_normal((10, 512)))
    q = _q(k[3][None, None, :] * 1.0)                    # q = row 3: q.k3 is the largest
    out, lse, _ = attn(q, cache, 1, 10, 10, np.arange(10, dtype=np.int64)[None], 50.0)
    assert np.all(np.isfinite(out)) and np.isfinite(lse).all()
    scores = 50.0 * (k @ _bf(q[0, 0]))
    assert np.argmax(scores) == 3 and scores[3] - np.sort(scores)[-2] > 100
    np.testing.assert_allclose(out[0, 0], k[3], rtol=1e-12, atol=1e-30)


def test_brute_force_loops_on_a_tiny_case():
    """Independent evaluation with Python loops and math.exp (no matrix
    products, running max and sum taken term by term)."""
    rng = np.random.default_rng(7)
    cache, k = _cache(rng.standard_normal((12, 512)) * 0.5)
    qf = rng.standard_normal((2, 3, 512))
    q = _q(qf)
    idx = np.array([[11, 0, -1, 5, 5, 7], [3, 2, 1, 40, -2, 9]], np.int64)
    scale = 0.08
    out, lse, _ = attn(q, cache, 1, 12, 12, idx, scale)
    qd = _bf(q)
    for n in range(2):
        for h in range(3):
            js = [int(j) for j in idx[n] if 0 <= j < 12]
            s = []
            for j in js:
                acc = 0.0
                for d in range(512):
                    acc += qd[n, h, d] * k[j, d]
                s.append(scale * acc)
            m = max(s)
            w = [math.exp(v - m) for v in s]
            tot = sum(w)
            for d in range(0, 512, 37):
                want = sum(w[i] * k[js[i], d] for i in range(len(js))) / tot
                assert out[n, h, d] == pytest.approx(want, rel=1e-12, abs=1e-300)
            assert lse[n, h] == pytest.approx(m + math.log(tot), rel=1e-13)


def test_queries_are_independent():
    rng = np.random.default_rng(8)
    cache, _ = _cache(rng.standard_normal((32, 512)))
    q = _q(rng.standard_normal((3, 2, 512)))
    idx = rng.integers(-2, 32, size=(3, 9)).astype(np.int64)
    out, lse, _ = attn(q, cache, 1, 32, 32, idx, 0.2)
    for n in range(3):
        o1, l1, _ = attn(q[n:n + 1], cache, 1, 32, 32, idx[n:n + 1], 0.2)
        np.testing.assert_array_equal(o1[0], out[n])
        np.testing.assert_array_equal(l1[0], lse[n])
