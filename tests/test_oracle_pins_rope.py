"""Pins of the oracle's V4.1 RoPE-then-quantize inserts (CPU only).

Page: 'vllm.models.deepseek_v41.common.ops.fused_compress_quant_cache'
(_rope_quant_insert_mxfp8_kernel, _rope_quant_insert_nvfp4_kernel,
rope_quant_insert): slot and compress-ratio gates, GPT-J interleaved rotation
of pairs 224..255 from a table row of 32 cos then 32 sin, optional NaN
sanitising, MXFP8 (E4M3 + E8M0 per 32) and NVFP4 (E2M1 + E4M3 per 16) records
in segregated page layouts.
"""
import json
import os

import numpy as np
import pytest

import oracle
import workloads
from tests import _independent as ind

CB = 4  # slots per page in these small cases


def _hex(s):
    return [int(b, 16) for b in s.split()]


def _identity_table(rows=16):
    t = np.zeros((rows, 64), np.float32)
    t[:, :32] = 1.0
    return t


def _run(record, latent, positions, table, slots, num_pages, R=1, sanitize=False, fill=0xAA):
    width = {"mxfp8": 528, "nvfp4": 288}[record]
    cache = np.full(num_pages * CB * width, fill, np.uint8)
    fn = {"mxfp8": oracle.rope_quant_insert_mxfp8, "nvfp4": oracle.rope_quant_insert_nvfp4}[record]
    fn(latent, np.asarray(positions, np.int64), table, cache, np.asarray(slots, np.int64),
       num_pages, CB, CB * width, R, sanitize)
    return cache


def _mxfp8_slot(cache, slot):
    page = cache[(slot // CB) * CB * 528:(slot // CB + 1) * CB * 528]
    j = slot % CB
    return page[j * 512:(j + 1) * 512], page[CB * 512 + j * 16:CB * 512 + (j + 1) * 16]


def _nvfp4_slot(cache, slot):
    page = cache[(slot // CB) * CB * 288:(slot // CB + 1) * CB * 288]
    j = slot % CB
    return page[j * 256:(j + 1) * 256], page[CB * 256 + j * 32:CB * 256 + (j + 1) * 32]


def _mxfp8_expected(rot, sanitize=False):
    vals, scales = [], []
    for g in range(16):
        v, s = ind.mxfp8_group_reference(rot[32 * g:32 * g + 32], sanitize)
        vals.append(v)
        scales.append(s)
    return np.concatenate(vals), np.array(scales, np.uint8)


def _nvfp4_expected(rot):
    codes, scales = [], []
    for g in range(32):
        c, s = ind.nvfp4_tile_reference(rot[16 * g:16 * g + 16])
        codes.append(c)
        scales.append(s)
    c = np.concatenate(codes)
    return (c[0::2] | (c[1::2] << 4)).astype(np.uint8), np.array(scales, np.uint8)


def test_worked_records(golden_dir):
    with open(os.path.join(golden_dir, "v41_records_worked.json")) as f:
        g = json.load(f)
    table = workloads.rope_cos_sin_table(rows=4)  # row 0: cos 1, sin 0
    assert np.all(table[0, :32] == 1) and np.all(table[0, 32:] == 0)
    m = g["mxfp8"]
    row = np.zeros(512, np.uint16)
    for name, vals in m["latent_bf16_hex"].items():
        k = int(name[1:])
        row[32 * k:32 * k + len(vals)] = [int(v, 16) for v in vals]
    cache = _run("mxfp8", row[None], [0], table, [5], num_pages=2)
    vals, scales = _mxfp8_slot(cache, 5)
    for name in m["latent_bf16_hex"]:
        k = int(name[1:])
        assert vals[32 * k:32 * k + 4].tolist() == _hex(m["expected_value_bytes_hex"][name])
        assert [scales[k]] == _hex(m["expected_scale_bytes_hex"][name])
    n = g["nvfp4"]
    row = np.zeros(512, np.uint16)
    for name, vals in n["latent_bf16_hex"].items():
        k = int(name[1:])
        row[16 * k:16 * k + len(vals)] = [int(v, 16) for v in vals]
    cache = _run("nvfp4", row[None], [0], table, [6], num_pages=2)
    codes, scales = _nvfp4_slot(cache, 6)
    for name in n["latent_bf16_hex"]:
        k = int(name[1:])
        assert codes[8 * k:8 * k + 2].tolist() == _hex(n["expected_code_bytes_hex"][name])
        assert [scales[k]] == _hex(n["expected_scale_bytes_hex"][name])


def _random_rows(seed, T, spread=6.0):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((T, 512)) * np.exp2(rng.uniform(-spread, spread, (T, 1)))
    return workloads.f32_to_bf16_bits(x.astype(np.float32))


@pytest.mark.parametrize("record", ["mxfp8", "nvfp4"])
def test_identity_rotation_matches_brute_force(record):
    lat = _random_rows(31, 24, spread=20.0)
    T = lat.shape[0]
    cache = _run(record, lat, np.zeros(T), _identity_table(), np.arange(T), num_pages=T // CB)
    for t in range(T):
        x = ind.bf16_bits_to_f32(lat[t])
        if record == "mxfp8":
            v, s = _mxfp8_slot(cache, t)
            ev, es = _mxfp8_expected(x)
        else:
            v, s = _nvfp4_slot(cache, t)
            ev, es = _nvfp4_expected(x)
        assert np.array_equal(v, ev) and np.array_equal(s, es), t


def _quarter_turn_expected(x, pairs=range(224, 256)):
    """cos 0, sin 1: (even, odd) -> (-odd, even) exactly for non-zero inputs."""
    y = x.copy()
    for i in pairs:
        y[2 * i], y[2 * i + 1] = -x[2 * i + 1], x[2 * i]
    return y


@pytest.mark.parametrize("record", ["mxfp8", "nvfp4"])
def test_quarter_and_half_turns(record):
    lat = _random_rows(32, 8)
    x = ind.bf16_bits_to_f32(lat)
    assert np.all(x != 0)
    table = _identity_table(rows=8)
    table[3, :32], table[3, 32:] = 0.0, 1.0      # quarter turn on row 3
    table[5, :32], table[5, 32:] = -1.0, 0.0     # half turn on row 5
    # one distinct pair: only rotary pair 7 (elements 462, 463) turns on row 6
    table[6, 7], table[6, 32 + 7] = 0.0, 1.0
    positions = [3, 5, 6, 0, 3, 5, 6, 0]
    cache = _run(record, lat, positions, table, np.arange(8), num_pages=2)
    for t, p in enumerate(positions):
        if p == 3:
            rot = _quarter_turn_expected(x[t])
        elif p == 5:
            rot = x[t].copy()
            rot[448:] = -x[t, 448:]
        elif p == 6:
            rot = _quarter_turn_expected(x[t], pairs=[224 + 7])
        else:
            rot = x[t]
        if record == "mxfp8":
            v, s = _mxfp8_slot(cache, t)
            ev, es = _mxfp8_expected(rot)
        else:
            v, s = _nvfp4_slot(cache, t)
            ev, es = _nvfp4_expected(rot)
        assert np.array_equal(v, ev) and np.array_equal(s, es), (t, p)


@pytest.mark.parametrize("record", ["mxfp8", "nvfp4"])
def test_slot_and_ratio_gates_and_table_row(record):
    """R = 4: only positions with (pos + 1) % 4 == 0 write, using table row
    (pos // 4) * 4; slot -1 and slots past the cache never write."""
    lat = _random_rows(33, 8)
    x = ind.bf16_bits_to_f32(lat)
    table = _identity_table(rows=32)
    table[8, :32], table[8, 32:] = 0.0, 1.0      # only row 8 turns
    positions = [11, 8, 15, 3, 11, 7, 9, 23]
    slots = [0, 1, 2, 3, -1, 5, 6, 8]            # slot 8 == 2 pages * 4: outside
    cache = _run(record, lat, positions, table, slots, num_pages=2, R=4)
    writes = {0: ("turn", 0), 2: ("id", 2), 3: ("id", 3), 5: ("id", 5)}
    for slot in range(8):
        if record == "mxfp8":
            v, s = _mxfp8_slot(cache, slot)
        else:
            v, s = _nvfp4_slot(cache, slot)
        if slot not in writes:
            assert np.all(v == 0xAA) and np.all(s == 0xAA), slot
            continue
        kind, t = writes[slot]
        rot = _quarter_turn_expected(x[t]) if kind == "turn" else x[t]
        ev, es = _mxfp8_expected(rot) if record == "mxfp8" else _nvfp4_expected(rot)
        assert np.array_equal(v, ev) and np.array_equal(s, es), slot
    # and the gaps between records of other pages stay untouched
    assert cache.size == 2 * CB * (528 if record == "mxfp8" else 288)


def test_nope_pairs_follow_the_literal_formula():
    """On pairs with cos 1, sin 0 the literal formula spreads a NaN to the pair
    partner (x * 0 = NaN) and turns (-0, negative) into (+0, ...)."""
    row = np.full(512, 0x3F80, np.uint16)   # 1.0
    row[4] = 0x7FC0                          # NaN at pair 2, even
    row[40], row[41] = 0x8000, 0xBF80        # (-0, -1) at pair 20
    row[42], row[43] = 0x8000, 0x3F80        # (-0, +1) at pair 21
    table = _identity_table(rows=2)
    for sanitize in (False, True):
        cache = _run("mxfp8", row[None], [0], table, [0], num_pages=1, sanitize=sanitize)
        v, s = _mxfp8_slot(cache, 0)
        nanb = 0x00 if sanitize else 0x7F
        assert v[4] == nanb and v[5] == nanb          # partner poisoned too
        assert v[40] == 0x00                          # -0 - (-1 * 0) = +0
        assert v[42] == 0x80                          # -0 - (+1 * 0) = -0
        assert s[0] == s[1]                           # NaN ignored by amax
    cache = _run("nvfp4", row[None], [0], table, [0], num_pages=1, sanitize=False)
    c, s = _nvfp4_slot(cache, 0)
    assert c[2] == 0x00                               # NaN pair -> codes 0, 0


def test_mxfp8_scale_cap_depends_on_sanitising():
    """An infinite input makes amax inf: e = 128, byte clamp(255) -> 254 with
    sanitising, 255 without; inf clamps to 448 (0x7E)."""
    row = np.full(512, 0x3F80, np.uint16)
    row[0] = 0x7F80                                   # +inf, partner 1.0 -> NaN
    table = _identity_table(rows=2)
    for sanitize, cap in ((False, 255), (True, 254)):
        cache = _run("mxfp8", row[None], [0], table, [0], num_pages=1, sanitize=sanitize)
        v, s = _mxfp8_slot(cache, 0)
        assert s[0] == cap and v[0] == 0x7E
        assert v[1] == (0x00 if sanitize else 0x7F)
        assert np.all(v[2:32] == 0x00)                # 1.0 * 2**-128 -> 0
        assert s[1] == 127 - 8                        # amax 1 -> 1/448 -> e -8


def test_nvfp4_division_ties():
    """Values that land exactly on E2M1 midpoints after the division round to
    the even code, which only a correctly rounded division guarantees."""
    table = _identity_table(rows=2)
    row = np.zeros(512, np.uint16)
    # tile 0: amax 5 -> s = E4M3(5 * fl32(1/6)) = 0.8125; members m * 0.8125
    mids = [5.0, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, -0.25, -0.75, -1.25, -1.75, -2.5, -3.5]
    vals = np.array([m * 0.8125 for m in mids], np.float32)
    vals[0] = 5.0
    row[:14] = workloads.f32_to_bf16_bits(vals)
    assert np.array_equal(ind.bf16_bits_to_f32(row[:14]), vals)   # exact in bf16
    # tile 1: amax 5.625 -> s = 0.9375 (E4M3 0x37), a scale where multiplying
    # by a rounded reciprocal instead of dividing moves the 1.25, 2.5 and 5.0
    # ties up by one code
    ties = [5.625] + [m * 0.9375 for m in (1.25, 2.5, 5.0, -1.25, -2.5, -5.0)]
    vals1 = np.array(ties, np.float32)
    row[16:16 + 7] = workloads.f32_to_bf16_bits(vals1)
    assert np.array_equal(ind.bf16_bits_to_f32(row[16:23]), vals1)
    cache = _run("nvfp4", row[None], [0], table, [0], num_pages=1)
    c, s = _nvfp4_slot(cache, 0)
    assert s[0] == 0x35 and s[1] == 0x37
    codes = np.empty(32, np.uint8)
    codes[0::2], codes[1::2] = c[:16] & 0xF, c[:16] >> 4
    assert codes[:14].tolist() == [7, 0, 2, 2, 4, 4, 6, 6, 8, 10, 10, 12, 12, 14]
    assert codes[16:23].tolist() == [7, 2, 4, 6, 10, 12, 14]


def test_nvfp4_scale_clamps_to_448():
    """A tile whose amax * fl32(1/6) exceeds 448 takes the largest E4M3 scale,
    448 (byte 0x7E): with amax 6144 a member 896 is 896 / 448 = 2 exactly
    (code 4), and the amax itself saturates at 6 (code 7)."""
    table = _identity_table(rows=2)
    row = np.zeros(512, np.uint16)
    vals = np.array([6144.0, 896.0, -896.0, 224.0], np.float32)
    row[:4] = workloads.f32_to_bf16_bits(vals)
    assert np.array_equal(ind.bf16_bits_to_f32(row[:4]), vals)   # exact in bf16
    cache = _run("nvfp4", row[None], [0], table, [0], num_pages=1)
    c, s = _nvfp4_slot(cache, 0)
    assert s[0] == 0x7E
    codes = np.empty(32, np.uint8)
    codes[0::2], codes[1::2] = c[:16] & 0xF, c[:16] >> 4
    # 224 / 448 = 0.5 (code 1); the other twelve members are +0 (code 0)
    assert codes[:16].tolist() == [7, 4, 12, 1] + [0] * 12
