"""GPU parity of mxfp4_mla_store against the CPU oracle, byte for byte over
whole cache buffers (written rows, pad slots, unused slots and the poisoned
pages of other layers alike)."""
import numpy as np
import pytest
import torch

import __graft_entry__
import fp8_quantized_paged_store_gb300 as kvq
import oracle
import workloads
from tests import _gpu as G
from tests import _independent as ind

pytestmark = pytest.mark.gpu

ROW = 272


@pytest.fixture(scope="module", autouse=True)
def _built():
    __graft_entry__.build()


def _store_both(lat, slots, buf, offset, nb, bs, bsr, threads=1):
    want = buf.copy()
    oracle.mxfp4_mla_store(lat, slots, want, nb, bs, bsr, cache_offset=offset, threads=threads)
    if np.any((slots >= 0) & (slots < nb * bs)):
        assert not np.array_equal(want, buf), "the oracle wrote nothing"
    dbuf, view = G.paged_cache_dev(buf, offset, nb, bs, bsr)
    kvq.mxfp4_mla_store(G.latent_dev(lat), G.to_dev(slots), view)
    torch.cuda.synchronize()
    return G.u8_host(dbuf), want


def test_store_small_64_tokens():
    w = workloads.store_small(seed=0)
    got, want = _store_both(w["latent"], w["slot_mapping"], w["cache"], 0, 1, 128, 128)
    assert G.first_diff(got, want) is None, G.first_diff(got, want)


def test_store_paged_16384_tokens_block_stride_192():
    w = workloads.store_paged(seed=0)
    got, want = _store_both(w["latent"], w["slot_mapping"], w["cache"], w["cache_offset"],
                            w["num_blocks"], w["block_size"], w["block_stride_rows"])
    assert G.first_diff(got, want) is None, G.first_diff(got, want)


def test_store_large_4300000_tokens_stride_576():
    """Full size: 4.3M tokens read through a 576-element row stride (2.48e9
    source elements, past 2**31), 8,388,608-slot cache, 1% pads. Compared on
    every byte of the 2.28 GB cache."""
    w = workloads.store_large(seed=0)
    assert w["latent_full"].shape[0] * w["latent_full"].shape[1] > 2 ** 31
    got, want = _store_both(w["latent"], w["slot_mapping"], w["cache"], 0, 1, w["num_slots"],
                            w["num_slots"], threads=oracle.default_threads())
    assert G.first_diff(got, want) is None, G.first_diff(got, want)


def _group_rows(groups: np.ndarray) -> np.ndarray:
    """[G, 32] uint16 groups -> [ceil(G/16), 512] rows (tail padded with +0)."""
    n = -(-groups.shape[0] // 16) * 16
    g = np.zeros((n, 32), dtype=np.uint16)
    g[:groups.shape[0]] = groups
    return g.reshape(-1, 512)


def _flat_store(lat):
    T = lat.shape[0]
    slots = np.arange(T, dtype=np.int64)
    buf = np.full(T * ROW, 0xAA, dtype=np.uint8)
    return _store_both(lat, slots, buf, 0, 1, T, T, threads=oracle.default_threads())


def test_store_every_positive_bf16_amax():
    """One group per positive bf16 amax (0x0001..0x7F80, subnormals and +inf
    included), the other 31 values random with magnitude <= amax."""
    rng = np.random.default_rng(41)
    amax_bits = np.arange(1, 0x7F81, dtype=np.uint32)
    amax = ind.bf16_bits_to_f32(amax_bits).astype(np.float64)
    frac = rng.uniform(-1.0, 1.0, size=(amax.size, 31))
    with np.errstate(invalid="ignore", over="ignore"):
        others = np.where(np.isinf(amax)[:, None], frac * 1e38, frac * amax[:, None])
    groups = np.empty((amax.size, 32), dtype=np.uint16)
    groups[:, 0] = amax_bits
    groups[:, 1:] = workloads.f32_to_bf16_bits(others.astype(np.float32))
    got, want = _flat_store(_group_rows(rng.permuted(groups, axis=1)))
    assert G.first_diff(got, want) is None, G.first_diff(got, want)


def test_store_every_bf16_at_every_exponent():
    """For every group exponent e in [-126, 126] (pinned by an amax element of
    exactly 6 * 2**e, bf16 max for e = 126), every bf16 pattern whose magnitude
    is at most the pin, plus NaNs and -0.0, is quantized at that exponent."""
    all_bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    mag = ind.bf16_bits_to_f32(all_bits).astype(np.float64)
    nan_bits = all_bits[np.isnan(mag)][::509]
    groups = []
    for e in range(-126, 127):
        pin = 6.0 * 2.0 ** e if e < 126 else float(ind.bf16_bits_to_f32(np.array([0x7F7F]))[0])
        pin_bits = int(workloads.f32_to_bf16_bits(np.array([pin], np.float32))[0])
        members = all_bits[np.abs(mag) <= pin]
        members = np.concatenate([members, nan_bits])
        k = -(-members.size // 31)
        padded = np.zeros(k * 31, dtype=np.uint16)
        padded[:members.size] = members
        g = np.empty((k, 32), dtype=np.uint16)
        g[:, 0] = pin_bits
        g[:, 1:] = padded.reshape(k, 31)
        groups.append(g)
    groups = np.concatenate(groups)
    got, want = _flat_store(_group_rows(groups))
    assert G.first_diff(got, want) is None, G.first_diff(got, want)


def test_store_underflow_and_special_values():
    """Large groups (e >= 17) holding tiny negatives whose scaled value rounds
    to -0.0, infinities, NaN groups, -0.0 groups, subnormal-only groups."""
    rows = np.zeros((8, 512), dtype=np.uint16)
    rows[0, :32] = 0x4900              # 2**19 * 1.0 -> e = 17
    rows[0, 1:32:2] = 0x8001           # -2**-133
    rows[1, :32] = 0x7F80              # +inf group
    rows[1, 5] = 0xBF80
    rows[2, :32] = 0x7FC0              # all-NaN group
    rows[2, 32:64] = 0xFFC0            # all -NaN group
    rows[2, 64] = 0x3F80               # NaN with one number
    rows[2, 65:96] = 0x7FC0
    rows[3, :] = 0x8000                # -0.0 row
    rows[4, :] = 0x8001                # -2**-133 row (subnormal amax)
    rows[4, 32:64] = 0x0001
    rows[5, :32] = 0xFF80              # -inf
    rows[5, 32:64] = 0x7F7F            # bf16 max
    rows[5, 64:96] = 0xFF7F
    rows[6, :] = np.arange(512, dtype=np.uint16) * 127   # assorted patterns
    rows[7, :] = np.arange(512, dtype=np.uint16) * 127 + 0x8000
    got, want = _flat_store(rows)
    assert G.first_diff(got, want) is None, G.first_diff(got, want)


@pytest.mark.parametrize("T", [1, 2, 31, 32, 33, 63, 65, 257, 1000])
def test_store_ragged_token_counts_and_pads(T):
    rng = np.random.default_rng(T)
    lat = workloads.f32_to_bf16_bits(
        (rng.standard_normal((T, 512)) * np.exp2(rng.uniform(-8, 8, (T, 1)))).astype(np.float32))
    nslots = 2 * T + 3
    slots = rng.choice(nslots, T, replace=False).astype(np.int64)
    slots[rng.random(T) < 0.2] = -1
    slots[rng.random(T) < 0.05] = nslots + 7       # outside the cache: skipped
    buf = np.full(nslots * ROW, 0xAA, dtype=np.uint8)
    got, want = _store_both(lat, slots, buf, 0, 1, nslots, nslots)
    assert G.first_diff(got, want) is None, G.first_diff(got, want)


def test_store_all_pads_and_empty():
    lat = np.zeros((40, 512), dtype=np.uint16)
    buf = np.full(64 * ROW, 0xAA, dtype=np.uint8)
    got, want = _store_both(lat, np.full(40, -1, np.int64), buf, 0, 1, 64, 64)
    assert np.all(got == 0xAA) and np.array_equal(got, want)
    d = G.to_dev(buf)
    kvq.mxfp4_mla_store(G.bf16_dev(lat[:0]), G.to_dev(np.zeros(0, np.int64)), d)
    torch.cuda.synchronize()
    assert np.all(G.u8_host(d) == 0xAA)


@pytest.mark.parametrize("bs,bsr,offset_rows,nb", [(4, 6, 1, 7), (64, 64, 0, 5), (3, 11, 2, 9),
                                                   (16, 17, 16, 4)])
def test_store_paged_layouts(bs, bsr, offset_rows, nb):
    rng = np.random.default_rng(bs * 100 + bsr)
    num_slots = nb * bs
    T = num_slots - 3
    lat = workloads.f32_to_bf16_bits(rng.standard_normal((T, 512)).astype(np.float32))
    slots = rng.permutation(num_slots)[:T].astype(np.int64)
    slots[::7] = -1
    rows = offset_rows + (nb - 1) * bsr + bs + 2
    buf = np.full(rows * ROW, 0x5A, dtype=np.uint8)
    got, want = _store_both(lat, slots, buf, offset_rows * ROW, nb, bs, bsr)
    assert G.first_diff(got, want) is None, G.first_diff(got, want)


def test_store_source_row_stride_with_poisoned_tail():
    rng = np.random.default_rng(77)
    T, stride = 300, 520
    full = np.full((T, stride), workloads.BF16_MAX_BITS, dtype=np.uint16)
    full[:, :512] = workloads.f32_to_bf16_bits(rng.standard_normal((T, 512)).astype(np.float32))
    slots = rng.permutation(T).astype(np.int64)
    buf = np.full(T * ROW, 0xAA, dtype=np.uint8)
    got, want = _store_both(full[:, :512], slots, buf, 0, 1, T, T)
    assert G.first_diff(got, want) is None, G.first_diff(got, want)


def test_store_rejects_bad_arguments():
    lat = G.bf16_dev(np.zeros((4, 512), np.uint16))
    slots = G.to_dev(np.arange(4, dtype=np.int64))
    cache = G.to_dev(np.zeros(4 * ROW, np.uint8))
    L = kvq.lib()
    s = torch.cuda.current_stream().cuda_stream
    assert L.mxfp4_mla_store(lat.data_ptr(), 4, 256, 512, slots.data_ptr(), cache.data_ptr(),
                             1, 4, 4, 32, s) == kvq.KVQ_EINVAL
    assert L.mxfp4_mla_store(lat.data_ptr() + 2, 4, 512, 512, slots.data_ptr(),
                             cache.data_ptr(), 1, 4, 4, 32, s) == kvq.KVQ_EINVAL
    assert L.mxfp4_mla_store(lat.data_ptr(), 4, 512, 512, slots.data_ptr(), cache.data_ptr(),
                             2, 4, 3, 32, s) == kvq.KVQ_EINVAL
    with pytest.raises((kvq.KvqError, ValueError)):
        kvq.mxfp4_mla_store(lat, slots, cache, group=16)
    torch.cuda.synchronize()
    assert np.all(G.u8_host(cache) == 0)
