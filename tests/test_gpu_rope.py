"""GPU parity of rope_quant_insert_mxfp8 / rope_quant_insert_nvfp4 against the
CPU oracle, byte for byte over the whole paged cache."""
import numpy as np
import pytest
import torch

import __graft_entry__
import fp8_quantized_paged_store_gb300 as kvq
import oracle
import workloads
from tests import _gpu as G

pytestmark = pytest.mark.gpu

FNS = {"mxfp8": (oracle.rope_quant_insert_mxfp8, kvq.rope_quant_insert_mxfp8, 528),
       "nvfp4": (oracle.rope_quant_insert_nvfp4, kvq.rope_quant_insert_nvfp4, 288)}


@pytest.fixture(scope="module", autouse=True)
def _built():
    __graft_entry__.build()


def _insert_both(record, lat, positions, table, cache, slots, num_pages, cache_block, ratio,
                 sanitize, page_stride=None, threads=1):
    fo, fk, width = FNS[record]
    page_stride = page_stride or cache_block * width
    want = cache.copy()
    fo(lat, positions, table, want, slots, num_pages, cache_block, page_stride, ratio, sanitize,
       threads=threads)
    writers = (slots >= 0) & (slots < num_pages * cache_block) & (positions >= 0) & \
        ((positions + 1) % ratio == 0) & (positions - ratio < table.shape[0])
    if np.any(writers):
        assert not np.array_equal(want, cache), "the oracle wrote nothing"
    d = G.to_dev(cache)
    view = d.as_strided((num_pages, cache_block, width), (page_stride, width, 1))
    fk(G.latent_dev(lat), G.to_dev(positions), G.to_dev(table), view, G.to_dev(slots), ratio,
       sanitize_nans=sanitize)
    torch.cuda.synchronize()
    return G.u8_host(d), want


@pytest.mark.parametrize("record", ["mxfp8", "nvfp4"])
@pytest.mark.parametrize("sanitize", [False, True])
def test_insert_65536_tokens_R4_with_nans(record, sanitize):
    w = workloads.rope_insert(seed=0, record=record)
    got, want = _insert_both(record, w["latent"], w["positions"], w["cos_sin"], w["cache"],
                             w["cache_slots"], w["num_pages"], w["cache_block"],
                             w["compress_ratio"], sanitize, threads=oracle.default_threads())
    assert G.first_diff(got, want) is None, G.first_diff(got, want)


@pytest.mark.parametrize("record", ["mxfp8", "nvfp4"])
def test_insert_large_4194304_tokens(record):
    """The scaled variant used for bandwidth: 4,194,304 tokens into 65,536
    pages of 64 slots, same generator; every byte compared."""
    w = workloads.rope_insert(seed=0, num_tokens=4_194_304, num_pages=65_536, record=record)
    got, want = _insert_both(record, w["latent"], w["positions"], w["cos_sin"], w["cache"],
                             w["cache_slots"], w["num_pages"], w["cache_block"],
                             w["compress_ratio"], False, threads=oracle.default_threads())
    assert G.first_diff(got, want) is None, G.first_diff(got, want)


@pytest.mark.parametrize("record", ["mxfp8", "nvfp4"])
@pytest.mark.parametrize("sanitize", [False, True])
def test_insert_special_values(record, sanitize):
    """inf, -inf, NaN, -0.0, subnormals, bf16 max (the rotation can overflow),
    in NoPE and rotary positions; every writer."""
    rng = np.random.default_rng(5)
    T = 96
    specials = np.array([0x7F80, 0xFF80, 0x7FC0, 0xFFC0, 0x8000, 0x0000, 0x0001, 0x8001, 0x7F7F,
                         0xFF7F, 0x0080, 0x8080], dtype=np.uint16)
    lat = workloads.f32_to_bf16_bits(rng.standard_normal((T, 512)).astype(np.float32))
    mask = rng.random((T, 512)) < 0.1
    lat[mask] = rng.choice(specials, size=int(mask.sum()))
    lat[0, :] = 0x8000
    lat[1, 448:] = 0x7F7F
    lat[2, ::2] = 0x7F80
    table = workloads.rope_cos_sin_table(rows=64)
    table[5] = 0.0                              # cos 0 and sin 0: everything rotates to 0
    positions = np.arange(T, dtype=np.int64) % 64
    slots = rng.permutation(T).astype(np.int64)
    cache = np.full(2 * 64 * FNS[record][2], 0xAA, dtype=np.uint8)
    got, want = _insert_both(record, lat, positions, table, cache, slots, 2, 64, 1, sanitize)
    assert G.first_diff(got, want) is None, G.first_diff(got, want)


@pytest.mark.parametrize("record", ["mxfp8", "nvfp4"])
@pytest.mark.parametrize("ratio", [1, 2, 3, 4, 7])
def test_insert_gates_pads_and_ratios(record, ratio):
    rng = np.random.default_rng(ratio)
    T, rows, pages, cb = 333, 200, 3, 64
    lat = workloads.f32_to_bf16_bits(
        (rng.standard_normal((T, 512)) * np.exp2(rng.uniform(-10, 10, (T, 1)))).astype(np.float32))
    positions = rng.integers(0, rows + 10, size=T, dtype=np.int64)
    positions[:4] = [-1, -5, 2 ** 62, np.iinfo(np.int64).max]
    slots = rng.integers(0, pages * cb, size=T).astype(np.int64)
    slots = np.unique(slots)[:T]
    slots = np.concatenate([slots, np.full(T - slots.size, -1)])
    rng.shuffle(slots)
    slots[5] = pages * cb                        # outside the cache
    table = workloads.rope_cos_sin_table(rows=rows)
    cache = np.full(pages * cb * FNS[record][2], 0xAA, dtype=np.uint8)
    got, want = _insert_both(record, lat, positions, table, cache, slots, pages, cb, ratio, False)
    assert G.first_diff(got, want) is None, G.first_diff(got, want)


@pytest.mark.parametrize("record", ["mxfp8", "nvfp4"])
def test_insert_strided_table_and_page_gaps(record):
    """cos_sin row stride 68 floats, page stride larger than the page (gaps
    between pages keep their poison), latent row stride 520."""
    rng = np.random.default_rng(9)
    T, pages, cb = 200, 5, 16
    width = FNS[record][2]
    full = np.full((T, 520), workloads.BF16_MAX_BITS, dtype=np.uint16)
    full[:, :512] = workloads.f32_to_bf16_bits(rng.standard_normal((T, 512)).astype(np.float32))
    base = workloads.rope_cos_sin_table(rows=300)
    table = np.full((300, 68), 7.0, dtype=np.float32)
    table[:, :64] = base
    positions = rng.integers(0, 300, size=T, dtype=np.int64)
    slots = np.concatenate([rng.permutation(pages * cb), np.full(T - pages * cb, -1)])
    rng.shuffle(slots)
    page_stride = cb * width + 48
    cache = np.full(pages * page_stride, 0x5A, dtype=np.uint8)
    fo, fk, _ = FNS[record]
    want = cache.copy()
    fo(full[:, :512], positions, table, want, slots.astype(np.int64), pages, cb, page_stride, 2,
       False)
    d = G.to_dev(cache)
    view = d.as_strided((pages, cb, width), (page_stride, width, 1))
    fk(G.latent_dev(full[:, :512]), G.to_dev(positions), G.to_dev(table), view,
       G.to_dev(slots.astype(np.int64)), 2)
    torch.cuda.synchronize()
    got = G.u8_host(d)
    assert G.first_diff(got, want) is None, G.first_diff(got, want)


def test_nvfp4_division_ties_on_gpu():
    """Quotients that land exactly on E2M1 midpoints (and the scale 0.9375
    where a reciprocal multiply would move them) through the kernel."""
    table = np.zeros((2, 64), np.float32)
    table[:, :32] = 1.0
    row = np.zeros(512, np.uint16)
    mids = [5.0] + [m * 0.8125 for m in (0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, -0.25, -0.75,
                                          -1.25, -1.75, -2.5, -3.5)]
    row[:14] = workloads.f32_to_bf16_bits(np.array(mids, np.float32))
    ties = [5.625] + [m * 0.9375 for m in (1.25, 2.5, 5.0, -1.25, -2.5, -5.0)]
    row[16:23] = workloads.f32_to_bf16_bits(np.array(ties, np.float32))
    lat = np.tile(row, (4, 1))
    cache = np.full(64 * 288, 0xAA, dtype=np.uint8)
    got, want = _insert_both("nvfp4", lat, np.zeros(4, np.int64), table, cache,
                             np.arange(4, dtype=np.int64), 1, 64, 1, False)
    assert G.first_diff(got, want) is None, G.first_diff(got, want)


def _every_scale_tiles():
    """[N, 16] bf16 tiles: for every positive E4M3 scale s, the tile amax 6*s
    followed by every bf16 value of magnitude up to 6*s, both signs."""
    tiles = []
    for sb in range(1, 127):
        s = float(oracle.e4m3_decode(np.array([sb], np.uint8))[0])
        a = int(workloads.f32_to_bf16_bits(np.array([6.0 * s], np.float32))[0])
        mags = np.arange(0, a + 1, dtype=np.uint16)
        vals = np.concatenate([mags, mags | np.uint16(0x8000)])
        vals = np.concatenate([vals, np.zeros((-vals.size) % 15, np.uint16)]).reshape(-1, 15)
        tiles.append(np.concatenate([np.full((vals.shape[0], 1), a, np.uint16), vals], axis=1))
    return np.concatenate(tiles)


def test_nvfp4_every_scale_and_bf16_value():
    """Every positive E4M3 tile scale with every finite bf16 value up to the
    tile amax, in NoPE tiles (the kernel's code rule for bf16 numbers) and in
    rotary tiles under an identity table (its corrected quotient): codes and
    scales against the oracle's division, over about four million values."""
    tiles = _every_scale_tiles()
    tiles = np.concatenate([tiles, np.zeros(((-tiles.shape[0]) % 32, 16), np.uint16)])
    lat = tiles.reshape(-1, 512)
    T = lat.shape[0]
    pages = -(-T // 64)
    table = np.zeros((1, 64), np.float32)
    table[0, :32] = 1.0
    slots = np.random.default_rng(11).permutation(pages * 64)[:T].astype(np.int64)
    cache = np.full(pages * 64 * 288, 0xAA, dtype=np.uint8)
    got, want = _insert_both("nvfp4", lat, np.zeros(T, np.int64), table, cache, slots, pages, 64,
                             1, False, threads=oracle.default_threads())
    assert G.first_diff(got, want) is None, G.first_diff(got, want)


def test_insert_rejects_bad_arguments():
    L = kvq.lib()
    lat = G.bf16_dev(np.zeros((4, 512), np.uint16))
    pos = G.to_dev(np.zeros(4, np.int64))
    tab = G.to_dev(np.zeros((4, 64), np.float32))
    cache = G.to_dev(np.zeros(64 * 528, np.uint8))
    s = torch.cuda.current_stream().cuda_stream
    args = [lat.data_ptr(), 4, 512, pos.data_ptr(), tab.data_ptr(), 64, 4, cache.data_ptr(),
            pos.data_ptr(), 1, 64, 64 * 528, 1, 0, s]
    assert L.rope_quant_insert_mxfp8(*args) == kvq.KVQ_OK
    bad = list(args); bad[11] = 64 * 528 - 16                  # page too small
    assert L.rope_quant_insert_mxfp8(*bad) == kvq.KVQ_EINVAL
    bad = list(args); bad[5] = 60                              # cos stride < 64
    assert L.rope_quant_insert_mxfp8(*bad) == kvq.KVQ_EINVAL
    bad = list(args); bad[12] = 0                              # ratio 0
    assert L.rope_quant_insert_nvfp4(*bad) == kvq.KVQ_EINVAL
    bad = list(args); bad[13] = 2                              # sanitize not 0/1
    assert L.rope_quant_insert_nvfp4(*bad) == kvq.KVQ_EINVAL
    bad = list(args); bad[4] = tab.data_ptr() + 4              # misaligned table
    assert L.rope_quant_insert_nvfp4(*bad) == kvq.KVQ_EINVAL
    torch.cuda.synchronize()
