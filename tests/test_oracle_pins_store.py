"""Pins of the oracle's MXFP4 store and gather (CPU only).

Pages: 'vllm.v1.attention.ops.mxfp4_mla.store' (store_mxfp4_mla: PAD_SLOT_ID
skip, paged view with block stride, flat view); PR 60321 'Add an mxfp4_mla KV
cache for rope-free sparse MLA' (Details: row layout, low nibble = lower index,
round-up scale with no clamp; Read path: unpack to bf16; Claims: the
dequantized values are what attention sees).
"""
import json
import os

import numpy as np

import oracle
import workloads
from tests import _independent as ind

ROW = 272


def _hex(s):
    return np.array([int(b, 16) for b in s.split()], dtype=np.uint8)


def _worked_row(golden_dir):
    with open(os.path.join(golden_dir, "mxfp4_row_worked.json")) as f:
        g = json.load(f)
    row = np.zeros(512, dtype=np.uint16)
    for name, vals in g["latent_bf16_hex"].items():
        if vals == "zeros":
            continue
        k = int(name[1:])
        row[32 * k:32 * k + len(vals)] = [int(v, 16) for v in vals]
    want = np.zeros(ROW, dtype=np.uint8)
    for name, hexs in g["expected_code_bytes_hex"].items():
        k = int(name[1:])
        want[16 * k:16 * k + 16] = _hex(hexs)
    want[256:] = _hex(g["expected_scale_bytes_hex"])
    return row, want


def test_store_worked_row(golden_dir):
    row, want = _worked_row(golden_dir)
    cache = np.full(ROW, 0xAA, dtype=np.uint8)
    oracle.mxfp4_mla_store(row[None, :], np.array([0]), cache, 1, 1, 1)
    assert cache.tolist() == want.tolist()


def test_store_low_nibble_holds_lower_index():
    row = np.zeros(512, dtype=np.uint16)
    row[0] = 0x3F00  # 0.5 -> code 1 (amax 6 in the group pins e = 0)
    row[1] = 0x3F80  # 1.0 -> code 2
    row[2] = 0x40C0  # 6.0 -> code 7
    cache = np.zeros(ROW, dtype=np.uint8)
    oracle.mxfp4_mla_store(row[None, :], np.array([0]), cache, 1, 1, 1)
    assert cache[0] == 0x21 and cache[1] == 0x07 and cache[256] == 127


def test_store_matches_brute_force_rows():
    """Random rows in the normal range against a reference that finds the
    scale by exact comparison and the codes by nearest-value search."""
    d = workloads.store_paged(seed=11, num_tokens=400, num_blocks=8, block_size=64,
                              block_stride_rows=64, layer_row_offset=0)
    lat = d["latent"]
    # add rows at extreme but normal scales
    rng = np.random.default_rng(5)
    extra = (rng.standard_normal((64, 512)) * np.exp2(rng.uniform(-100, 100, (64, 1))))
    lat = np.concatenate([lat, workloads.f32_to_bf16_bits(extra.astype(np.float32))])
    T = lat.shape[0]
    cache = np.zeros(T * ROW, dtype=np.uint8)
    oracle.mxfp4_mla_store(lat, np.arange(T), cache, 1, T, T)
    got = cache.reshape(T, ROW)
    for t in range(T):
        want = ind.mxfp4_row_reference(lat[t])
        assert np.array_equal(got[t], want), t


def test_store_round_trip_within_half_step():
    d = workloads.store_paged(seed=12, num_tokens=300, num_blocks=8, block_size=64,
                              block_stride_rows=64, layer_row_offset=0)
    lat = d["latent"]
    T = lat.shape[0]
    cache = np.zeros(T * ROW, dtype=np.uint8)
    oracle.mxfp4_mla_store(lat, np.arange(T), cache, 1, T, T)
    rows = cache.reshape(T, ROW)
    mags = ind.E2M1_MAGNITUDES
    for t in range(T):
        x = ind.bf16_bits_to_f32(lat[t]).astype(np.float64)
        deq = ind.e2m1_row_decode(rows[t])
        scale = np.exp2(np.repeat(rows[t, 256:].astype(np.float64), 32) - 127.0)
        a = np.abs(x) / scale
        assert np.all(a <= 6.0)  # no value clamps
        k = np.clip(np.searchsorted(mags, a, side="right") - 1, 0, 6)
        half_step = (mags[k + 1] - mags[k]) / 2 * scale
        assert np.all(np.abs(deq - x) <= half_step)


def test_store_skips_pads_and_out_of_range_and_keeps_poison():
    d = workloads.store_small(seed=0)
    lat, slots = d["latent"], d["slot_mapping"].copy()
    slots[0] = 128            # == num_slots: outside the cache, skipped
    slots[1] = 10 ** 12       # far outside
    cache = d["cache"].copy()
    oracle.mxfp4_mla_store(lat, slots, cache, 1, 128, 128)
    rows = cache.reshape(128, ROW)
    written = set(int(s) for s in slots if 0 <= s < 128)
    for s in range(128):
        if s in written:
            t = int(np.nonzero(slots == s)[0][0])
            assert np.array_equal(rows[s], ind.mxfp4_row_reference(lat[t]))
        else:
            assert np.all(rows[s] == 0xAA), s
    assert len(written) == int(np.sum((slots >= 0) & (slots < 128))) <= 64 - 8


def test_store_paged_addressing_with_block_stride():
    """Block size 4, block stride 6 rows, layer offset 1 row: slot s goes to
    buffer row 1 + (s // 4) * 6 + s % 4; every other row keeps its poison."""
    rng = np.random.default_rng(7)
    lat = workloads.f32_to_bf16_bits(rng.standard_normal((5, 512)).astype(np.float32))
    slots = np.array([5, 0, 11, -1, 7])
    buf = np.full(20 * ROW, 0x5A, dtype=np.uint8)
    oracle.mxfp4_mla_store(lat, slots, buf, num_blocks=3, block_size=4, block_stride_rows=6,
                           cache_offset=1 * ROW)
    rows = buf.reshape(20, ROW)
    target = {1 + 6 * 1 + 1: 0, 1 + 0: 1, 1 + 6 * 2 + 3: 2, 1 + 6 * 1 + 3: 4}
    for r in range(20):
        if r in target:
            assert np.array_equal(rows[r], ind.mxfp4_row_reference(lat[target[r]])), r
        else:
            assert np.all(rows[r] == 0x5A), r


def test_store_config1_injected_groups():
    d = workloads.store_small(seed=0)
    lat, slots = d["latent"], d["slot_mapping"]
    cache = d["cache"].copy()
    oracle.mxfp4_mla_store(lat, slots, cache, 1, 128, 128)
    rows = cache.reshape(128, ROW)
    x = ind.bf16_bits_to_f32(lat).astype(np.float64)
    checked = 0
    for t in range(64):
        s = int(slots[t])
        if s < 0:
            continue
        for g in range(16):
            xs = x[t, 32 * g:32 * g + 32]
            amax = np.max(np.abs(xs))
            byte = int(rows[s, 256 + g])
            if amax == 0:
                assert byte == 127 and not np.any(rows[s, 16 * g:16 * g + 16])
                checked += 1
                continue
            m, E = np.frexp(amax / 6.0)
            if m == 0.5:  # amax == 6 * 2**k exactly
                k = E - 1
                assert byte == 127 + k
                j = int(np.argmax(np.abs(xs)))
                code = (rows[s, 16 * g + j // 2] >> (4 * (j % 2))) & 0xF
                assert code == (15 if xs[j] < 0 else 7)
                checked += 1
    assert checked >= 6


def test_gather_equals_independent_decode():
    d = workloads.store_paged(seed=13, num_tokens=256, num_blocks=8, block_size=64,
                              block_stride_rows=96, layer_row_offset=16)
    cache = d["cache"].copy()
    oracle.mxfp4_mla_store(d["latent"], d["slot_mapping"], cache, d["num_blocks"],
                           d["block_size"], d["block_stride_rows"], cache_offset=d["cache_offset"])
    rng = np.random.default_rng(3)
    idx = rng.integers(-3, 512, size=300)
    idx[:5] = [-1, 511, 512, 0, 10 ** 9]   # pad, last slot, out of range, first, far out
    out = oracle.mxfp4_mla_gather_dequant(cache, d["num_blocks"], d["block_size"],
                                          d["block_stride_rows"], idx,
                                          cache_offset=d["cache_offset"])
    base = d["cache_offset"]
    for k, s in enumerate(idx):
        if s < 0 or s >= 512:
            assert np.all(out[k] == 0)
            continue
        r = (s // 64) * 96 + s % 64
        row = cache[base + r * ROW: base + (r + 1) * ROW]
        vals = ind.e2m1_row_decode(row).astype(np.float32)  # exact
        want = (vals.view(np.uint32) >> 16).astype(np.uint16)  # exact: low half is zero
        assert np.all((vals.view(np.uint32) & 0xFFFF) == 0)
        assert np.array_equal(out[k], want), k


def test_gather_of_store_is_the_quantized_value():
    """Store then gather gives, bit for bit, bf16(E2M1 value x 2**e) of each
    element: the values attention over the packed cache computes with."""
    rng = np.random.default_rng(21)
    x = (rng.standard_normal((16, 512)) * 3).astype(np.float32)
    lat = workloads.f32_to_bf16_bits(x)
    cache = np.zeros(16 * ROW, dtype=np.uint8)
    oracle.mxfp4_mla_store(lat, np.arange(16), cache, 1, 16, 16)
    out = oracle.mxfp4_mla_gather_dequant(cache, 1, 16, 16, np.arange(16))
    xf = ind.bf16_bits_to_f32(lat).astype(np.float64)
    got = ind.bf16_bits_to_f32(out).astype(np.float64)
    # the gathered value is the nearest E2M1 grid point of x at the group scale
    for t in range(16):
        for g in range(16):
            xs = xf[t, 32 * g:32 * g + 32]
            amax = np.max(np.abs(xs))
            e = int(ind.smallest_pow2_exponent_at_least(amax / 6.0)) if amax else 0
            grid = np.concatenate([-ind.E2M1_MAGNITUDES[::-1], ind.E2M1_MAGNITUDES]) * 2.0 ** e
            near = grid[np.argmin(np.abs(xs[:, None] - grid[None, :]), axis=1)]
            gs = got[t, 32 * g:32 * g + 32]
            assert np.all(np.abs(gs - xs) <= np.abs(near - xs) + 0.0)


def test_gather_special_scale_bytes():
    row = np.zeros(ROW, dtype=np.uint8)
    row[:256] = 0x8F                 # codes 15 (-6) then 8 (-0)
    row[256:] = 127
    row[256 + 1] = 255               # E8M0 NaN group
    row[256 + 2] = 0                 # 2**-127
    row[256 + 3] = 254               # 2**127: -6 * 2**127 overflows
    out = oracle.mxfp4_mla_gather_dequant(row, 1, 1, 1, np.array([0]))[0]
    assert out[0] == 0xC0C0 and out[1] == 0x8000          # -6.0, -0.0
    assert np.all(out[32:64] == 0x7FC0)                    # NaN group
    assert out[64] == 0x8140 and out[65] == 0x8000        # -6 * 2**-127 = -1.5 * 2**-125
    assert out[96] == 0xFF80 and out[97] == 0x8000        # -inf
