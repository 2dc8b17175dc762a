"""Pins of the oracle's remaining insert layouts (CPU only).

Page: 'vllm.models.deepseek_v41.common.ops.fused_compress_quant_cache'
(rope_quant_insert docstring: plain [448 NoPE | 64 RoPE] bf16 and fp8 rows,
the 584-byte V4 record with eight segregated UE8M0 scale bytes including one
zero padding scale; save_ring_rows: fp32 [kv, score] rows to ring slots,
slot -1 skipped). The kernels behind these are not printed; the readings are
stated in kvq_oracle.c and each pin below checks one of them by an
independent route.
"""
import numpy as np

import oracle
import workloads
from tests import _independent as ind

CB = 4


def _bf(a):
    return workloads.f32_to_bf16_bits(np.asarray(a, np.float32))


def _table(rows=8, cos=1.0, sin=0.0):
    t = np.zeros((rows, 64), np.float32)
    t[:, :32] = cos
    t[:, 32:] = sin
    return t


def _plain(latent, positions, table, slots, pages, fp8=False, scale=1.0, R=1, page_stride=None,
           slot_stride=512, fill=0xAA):
    esize = 1 if fp8 else 2
    page_stride = page_stride or CB * slot_stride
    cache = np.full(pages * page_stride * esize, fill, np.uint8)
    oracle.rope_plain_insert(latent, np.asarray(positions, np.int64), table, cache,
                             np.asarray(slots, np.int64), pages, CB, page_stride, slot_stride,
                             R, fp8, scale)
    return cache


def _plain_row(cache, slot, fp8=False, page_stride=CB * 512, slot_stride=512):
    esize = 1 if fp8 else 2
    off = ((slot // CB) * page_stride + (slot % CB) * slot_stride) * esize
    raw = cache[off:off + 512 * esize]
    return raw if fp8 else raw.view(np.uint16)


# ------------------------------------------------------------ save_ring_rows

def test_ring_rows_copied_bit_for_bit_pads_skipped_slack_untouched():
    rng = np.random.default_rng(1)
    nb, sb, row_stride_state, block_stride = 3, 5, 1100, 6000   # gaps between rows and blocks
    rows = rng.standard_normal((12, 1030)).astype(np.float32)
    rows.view(np.uint32)[0, 7] = 0x7FA00001                     # a NaN payload survives the copy
    slots = np.array([0, 14, -1, 3, 9, 15, 2, -7, 11, 1, 20, 5], np.int64)   # 15, 20: outside
    state = np.full(nb * block_stride + 2 * block_stride, np.nan, np.float32)
    state.view(np.uint32)[:] = 0x7FBADBAD
    oracle.save_ring_rows(rows[:, :1024], slots, state, nb, sb, block_stride, row_stride_state)
    seen = np.zeros(state.size, bool)
    for t, s in enumerate(slots):
        if 0 <= s < nb * sb:
            off = (s // sb) * block_stride + (s % sb) * row_stride_state
            assert np.array_equal(state[off:off + 1024].view(np.uint32),
                                  rows[t, :1024].view(np.uint32))
            seen[off:off + 1024] = True
    assert np.all(state.view(np.uint32)[~seen] == 0x7FBADBAD)


# ------------------------------------------------------------- plain rows

def test_plain_bf16_copies_nope_bits_and_rounds_rotary_values():
    rng = np.random.default_rng(2)
    lat = _bf(rng.standard_normal((4, 512)))
    lat[0, 0] = 0x7FA1          # NaN payload in a NoPE pair
    lat[0, 2:4] = [0x8000, 0xBF80]   # (-0, -1): the rotation formula would give (+0, -1)
    cache = _plain(lat, [0, 1, 2, 3], _table(), [0, 5, 2, 7], 2)
    for t, s in enumerate([0, 5, 2, 7]):
        row = _plain_row(cache, s)
        assert np.array_equal(row[:448], lat[t, :448])
        assert np.array_equal(row[448:], lat[t, 448:])   # identity table: rotary values are exact


def test_plain_bf16_quarter_turn_is_exact():
    rng = np.random.default_rng(3)
    lat = _bf(rng.standard_normal((1, 512)))
    cache = _plain(lat, [0], _table(cos=0.0, sin=1.0), [1], 1)
    row = _plain_row(cache, 1)
    x = ind.bf16_bits_to_f32(lat[0, 448:])
    want = np.empty(64, np.float32)
    want[0::2] = -x[1::2]
    want[1::2] = x[0::2]
    assert np.array_equal(ind.bf16_bits_to_f32(row[448:]), want)
    assert np.array_equal(row[:448], lat[0, :448])


def test_plain_fp8_is_e4m3_of_the_scaled_value():
    rng = np.random.default_rng(4)
    lat = _bf(rng.standard_normal((3, 512)) * np.array([[1.0], [40.0], [0.01]]))
    for scale in (1.0, 0.25, 8.0):
        cache = _plain(lat, [0, 1, 2], _table(), [0, 1, 2], 1, fp8=True, scale=scale)
        for t in range(3):
            x = ind.bf16_bits_to_f32(lat[t]).astype(np.float64) / scale   # exact: power of two
            want = ind.e4m3_nearest(np.clip(x, -448, 448).astype(np.float32))
            assert np.array_equal(_plain_row(cache, t, fp8=True), want)


def test_plain_fp8_divides_by_the_scale():
    """Rotated values x = M*s (cos = M*s, sin = 0 on pairs (1, 0)) with M an
    E4M3 midpoint and s = 0.9375: x / s is the tie M exactly and rounds to
    the even code, while x * RN(1/s) lands above M and would round up."""
    s = np.float32(0.9375)
    mids = np.float32(1.0) + (2 * np.arange(8, dtype=np.float32) + 1) / np.float32(16)
    cosv = (mids * s).astype(np.float32)                 # exact: 5 x 4 significant bits
    assert np.array_equal((cosv / s).astype(np.float32), mids)
    recip = (cosv * (np.float32(1) / s)).astype(np.float32)
    assert not np.array_equal(ind.e4m3_nearest(recip), ind.e4m3_nearest(mids))
    table = np.zeros((1, 64), np.float32)
    table[0, :8] = cosv
    table[0, 8:32] = 1.0
    lat = np.zeros((1, 512), np.uint16)
    lat[0, 448:464:2] = 0x3F80                            # pairs 224..231 = (1, 0)
    cache = _plain(lat, [0], table, [0], 1, fp8=True, scale=float(s))
    row = _plain_row(cache, 0, fp8=True)
    assert np.array_equal(row[448:464:2], ind.e4m3_nearest(mids))
    assert np.all(row[449:464:2] == 0)


def test_plain_strides_gates_and_poison():
    rng = np.random.default_rng(5)
    lat = _bf(rng.standard_normal((6, 512)))
    pos = [3, 4, 7, 0, 11, 5]          # R = 4: positions 3, 7, 11 write, at table rows 0, 4, 8
    slots = [0, 1, 6, 2, 9, -1]        # 9 is past 2 pages of 4
    ps, ss = 4 * 520 + 16, 520
    cache = _plain(lat, pos, _table(rows=12), slots, 2, R=4, page_stride=ps, slot_stride=ss)
    written = {0: 0, 6: 2}
    u16 = cache.view(np.uint16)
    mask = np.zeros(u16.size, bool)
    for s, t in written.items():
        off = (s // CB) * ps + (s % CB) * ss
        assert np.array_equal(u16[off:off + 512], lat[t])
        mask[off:off + 512] = True
    assert np.all(cache.reshape(-1, 2)[~mask] == 0xAA)


# -------------------------------------------------------------- V4 record

def _v4(latent, positions, table, slots, pages, sanitize=False, R=1):
    cache = np.full(pages * CB * 584, 0xAA, np.uint8)
    oracle.rope_quant_insert_v4(latent, np.asarray(positions, np.int64), table, cache,
                                np.asarray(slots, np.int64), pages, CB, CB * 584, R, sanitize)
    return cache


def _v4_slot(cache, slot):
    page = cache[(slot // CB) * CB * 584:(slot // CB + 1) * CB * 584]
    j = slot % CB
    return page[j * 576:(j + 1) * 576], page[CB * 576 + j * 8:CB * 576 + (j + 1) * 8]


def test_v4_record_layout_and_values():
    rng = np.random.default_rng(6)
    lat = _bf(rng.standard_normal((3, 512)) * np.exp2(rng.uniform(-6, 6, (3, 1))))
    lat[1, 64:128] = _bf(rng.standard_normal(64) * 1e-6)      # a tile under the 1e-4 amax floor
    lat[2, 130] = _bf([3000.0])[0]                              # one tile with a large amax
    cache = _v4(lat, [0, 1, 2], _table(), [0, 3, 5], 2)
    for t, s in enumerate([0, 3, 5]):
        vals, scales = _v4_slot(cache, s)
        x = ind.bf16_bits_to_f32(lat[t])
        for g in range(7):
            v, sc = ind.mxfp8_group_reference(x[64 * g:64 * g + 64], False)
            assert np.array_equal(vals[64 * g:64 * g + 64], v), (t, g)
            assert scales[g] == sc
        assert scales[7] == 0
        assert np.array_equal(vals[448:].view(np.uint16), lat[t, 448:])


def test_v4_tiles_are_64_wide():
    """A large value in the second half of a 64-wide tile raises the scale of
    the whole tile (a 32-wide tile would leave the first half alone)."""
    lat = np.zeros((1, 512), np.uint16)
    lat[0, :32] = _bf(np.full(32, 0.5))
    lat[0, 40] = _bf([200.0])[0]
    cache = _v4(lat, [0], _table(), [0], 1)
    vals, scales = _v4_slot(cache, 0)
    v, sc = ind.mxfp8_group_reference(ind.bf16_bits_to_f32(lat[0, :64]), False)
    assert scales[0] == sc and np.array_equal(vals[:64], v)
    v32, sc32 = ind.mxfp8_group_reference(ind.bf16_bits_to_f32(lat[0, :32]), False)
    assert sc32 != sc


def test_v4_sanitising_and_cap():
    lat = np.zeros((2, 512), np.uint16)
    lat[:, 0] = 0x7F80            # +inf: amax inf, e = 128
    lat[:, 450] = 0x7FC0          # NaN in a rotary value
    c0 = _v4(lat, [0, 1], _table(), [0, 1], 1, sanitize=False)
    c1 = _v4(lat, [0, 1], _table(), [0, 1], 1, sanitize=True)
    assert _v4_slot(c0, 0)[1][0] == 255 and _v4_slot(c1, 0)[1][0] == 254
    rot0 = _v4_slot(c0, 0)[0][448:].view(np.uint16)
    rot1 = _v4_slot(c1, 0)[0][448:].view(np.uint16)
    # element 450 is the even half of rotary pair 225: both halves become NaN
    assert np.all((rot0[2:4] & 0x7FFF) > 0x7F80) and np.all(rot1[2:4] == 0)


def test_rotated_nan_is_stored_as_the_canonical_bf16_nan():
    """A NaN that the rotation produces is stored as 0x7FC0 whatever the
    input NaN's sign or payload, and so is the NaN of inf * 0 (negative on
    x86, positive on Arm and CUDA); finite neighbours are untouched."""
    lat = np.zeros((1, 512), np.uint16)
    lat[0, 448] = 0xFFC1            # negative NaN with a payload: pair 224 -> both NaN
    lat[0, 450] = 0x7F80            # +inf with sin 0: inf * 0 in the odd half of pair 225
    lat[0, 452:454] = _bf([1.5, -2.0])
    cache = _plain(lat, [0], _table(), [0], 1)
    rot = _plain_row(cache, 0)[448:]
    assert list(rot[:4]) == [0x7FC0, 0x7FC0, 0x7F80, 0x7FC0]
    assert list(rot[4:6]) == list(_bf([1.5, -2.0]))
    v4 = _v4(lat, [0], _table(), [0], 1)
    assert list(_v4_slot(v4, 0)[0][448:].view(np.uint16)[:4]) == [0x7FC0, 0x7FC0, 0x7F80, 0x7FC0]
