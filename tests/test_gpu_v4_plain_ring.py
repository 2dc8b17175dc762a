"""GPU parity of rope_quant_insert_v4, rope_plain_insert (bf16 and fp8 rows)
and save_ring_rows against the CPU oracle, byte for byte over the whole
cache or state."""
import numpy as np
import pytest
import torch

import __graft_entry__
import fp8_quantized_paged_store_gb300 as kvq
import oracle
import workloads
from tests import _gpu as G

pytestmark = pytest.mark.gpu

LAYOUTS = ["v4", "bf16", "fp8"]


@pytest.fixture(scope="module", autouse=True)
def _built():
    __graft_entry__.build()


def _run(layout, lat, positions, table, cache, slots, num_pages, cb, ratio, sanitize=False,
         page_stride=None, slot_stride=512, fp8_scale=workloads.PLAIN_FP8_SCALE, threads=1):
    """Oracle and kernel on copies of `cache` (uint8); returns (got, want).
    page_stride is in bytes for the V4 record and in elements for plain rows."""
    positions = np.asarray(positions, np.int64)
    slots = np.asarray(slots, np.int64)
    want = cache.copy()
    d = G.to_dev(cache)
    if layout == "v4":
        page_stride = page_stride or cb * workloads.RECORD_BYTES_V4
        oracle.rope_quant_insert_v4(lat, positions, table, want, slots, num_pages, cb,
                                    page_stride, ratio, sanitize, threads=threads)
        view = d.as_strided((num_pages, cb, workloads.RECORD_BYTES_V4), (page_stride, 584, 1))
        kvq.rope_quant_insert_v4(G.latent_dev(lat), G.to_dev(positions), G.to_dev(table), view,
                                 G.to_dev(slots), ratio, sanitize_nans=sanitize)
    else:
        fp8 = layout == "fp8"
        page_stride = page_stride or cb * slot_stride
        oracle.rope_plain_insert(lat, positions, table, want, slots, num_pages, cb, page_stride,
                                 slot_stride, ratio, fp8, fp8_scale, threads=threads)
        typed = d.view(torch.float8_e4m3fn if fp8 else torch.bfloat16)
        view = typed.as_strided((num_pages, cb, 512), (page_stride, slot_stride, 1))
        kvq.rope_plain_insert(G.latent_dev(lat), G.to_dev(positions), G.to_dev(table), view,
                              G.to_dev(slots), ratio, fp8_scale=fp8_scale if fp8 else None)
    torch.cuda.synchronize()
    return G.u8_host(d), want


def _workload(layout, **kw):
    return workloads.rope_insert(seed=0, record=layout, **kw)


@pytest.mark.parametrize("layout,sanitize", [("v4", False), ("v4", True), ("bf16", False),
                                             ("fp8", False)])
def test_65536_tokens_R4_with_nans(layout, sanitize):
    w = _workload(layout)
    got, want = _run(layout, w["latent"], w["positions"], w["cos_sin"], w["cache"],
                     w["cache_slots"], w["num_pages"], w["cache_block"], w["compress_ratio"],
                     sanitize, threads=oracle.default_threads())
    assert not np.array_equal(want, w["cache"])
    assert G.first_diff(got, want) is None, G.first_diff(got, want)


@pytest.mark.parametrize("layout", LAYOUTS)
def test_large_4194304_tokens(layout):
    """The bandwidth case: 4,194,304 tokens into 65,536 pages of 64 slots."""
    w = _workload(layout, num_tokens=4_194_304, num_pages=65_536)
    got, want = _run(layout, w["latent"], w["positions"], w["cos_sin"], w["cache"],
                     w["cache_slots"], w["num_pages"], w["cache_block"], w["compress_ratio"],
                     False, threads=oracle.default_threads())
    assert G.first_diff(got, want) is None, G.first_diff(got, want)


@pytest.mark.parametrize("layout,sanitize", [("v4", False), ("v4", True), ("bf16", False),
                                             ("fp8", False)])
def test_special_values(layout, sanitize):
    """inf, -inf, NaN of both signs with payloads, -0.0, subnormals, bf16 max
    (the rotation can overflow), in NoPE and rotary positions; a table row of
    zeros; every token writes."""
    rng = np.random.default_rng(15)
    T = 96
    specials = np.array([0x7F80, 0xFF80, 0x7FC0, 0xFFC0, 0x7F81, 0xFFA5, 0x8000, 0x0000, 0x0001,
                         0x8001, 0x7F7F, 0xFF7F, 0x0080, 0x8080], dtype=np.uint16)
    lat = workloads.f32_to_bf16_bits(rng.standard_normal((T, 512)).astype(np.float32))
    mask = rng.random((T, 512)) < 0.1
    lat[mask] = rng.choice(specials, size=int(mask.sum()))
    lat[0, :] = 0x8000
    lat[1, 448:] = 0x7F7F
    lat[2, ::2] = 0x7F80
    lat[3, 64:128] = workloads.f32_to_bf16_bits(rng.standard_normal(64).astype(np.float32) * 1e-7)
    table = workloads.rope_cos_sin_table(rows=64)
    table[5] = 0.0
    positions = np.arange(T, dtype=np.int64) % 64
    slots = rng.permutation(T).astype(np.int64)
    width = {"v4": 584, "bf16": 1024, "fp8": 512}[layout]
    cache = np.full(2 * 64 * width, 0xAA, dtype=np.uint8)
    got, want = _run(layout, lat, positions, table, cache, slots, 2, 64, 1, sanitize)
    assert G.first_diff(got, want) is None, G.first_diff(got, want)


@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("ratio", [1, 3, 4])
def test_gates_pads_and_ratios(layout, ratio):
    rng = np.random.default_rng(100 + ratio)
    T, rows, pages, cb = 333, 200, 3, 64
    lat = workloads.f32_to_bf16_bits(
        (rng.standard_normal((T, 512)) * np.exp2(rng.uniform(-10, 10, (T, 1)))).astype(np.float32))
    positions = rng.integers(0, rows + 10, size=T, dtype=np.int64)
    positions[:4] = [-1, -5, 2 ** 62, np.iinfo(np.int64).max]
    slots = np.unique(rng.integers(0, pages * cb, size=T))[:T].astype(np.int64)
    slots = np.concatenate([slots, np.full(T - slots.size, -1)])
    rng.shuffle(slots)
    slots[5] = pages * cb
    table = workloads.rope_cos_sin_table(rows=rows)
    width = {"v4": 584, "bf16": 1024, "fp8": 512}[layout]
    cache = np.full(pages * cb * width, 0xAA, dtype=np.uint8)
    got, want = _run(layout, lat, positions, table, cache, slots, pages, cb, ratio)
    assert G.first_diff(got, want) is None, G.first_diff(got, want)


@pytest.mark.parametrize("layout", LAYOUTS)
def test_strided_rows_table_and_page_gaps(layout):
    """Latent row stride 520, cos_sin row stride 68 floats, pages with gaps
    (and plain rows with a slot stride of 520 elements): the gaps keep their
    poison."""
    rng = np.random.default_rng(19)
    T, pages, cb = 200, 5, 16
    full = np.full((T, 520), workloads.BF16_MAX_BITS, dtype=np.uint16)
    full[:, :512] = workloads.f32_to_bf16_bits(rng.standard_normal((T, 512)).astype(np.float32))
    table = np.full((300, 68), 7.0, dtype=np.float32)
    table[:, :64] = workloads.rope_cos_sin_table(rows=300)
    positions = rng.integers(0, 300, size=T, dtype=np.int64)
    slots = np.concatenate([rng.permutation(pages * cb), np.full(T - pages * cb, -1)])
    rng.shuffle(slots)
    if layout == "v4":
        page_stride, slot_stride = cb * 584 + 48, 512
        nbytes = pages * page_stride
    else:
        slot_stride = 520
        page_stride = cb * slot_stride + 16
        nbytes = pages * page_stride * (2 if layout == "bf16" else 1)
    cache = np.full(nbytes, 0x5A, dtype=np.uint8)
    got, want = _run(layout, full[:, :512], positions, table, cache, slots, pages, cb, 2,
                     page_stride=page_stride, slot_stride=slot_stride)
    assert G.first_diff(got, want) is None, G.first_diff(got, want)


@pytest.mark.parametrize("scale", [1.0, 0.0125, 0.9375, 3.7, 1e-3, 1e-30])
def test_fp8_scales(scale):
    """Per-tensor scales: a power of two, non-powers of two, one that
    saturates most values at +-448 and one whose quotients overflow to inf
    before the clamp."""
    rng = np.random.default_rng(23)
    T = 128
    lat = workloads.f32_to_bf16_bits(
        (rng.standard_normal((T, 512)) * np.exp2(rng.uniform(-6, 6, (T, 1)))).astype(np.float32))
    table = workloads.rope_cos_sin_table(rows=T)
    cache = np.full(2 * 64 * 512, 0xAA, dtype=np.uint8)
    got, want = _run("fp8", lat, np.arange(T), table, cache, rng.permutation(T), 2, 64, 1,
                     fp8_scale=scale)
    assert G.first_diff(got, want) is None, G.first_diff(got, want)


@pytest.mark.parametrize("scale", [0.0125, 0.9375, 0.5, 2.0 ** -126, 3.0e38])
def test_fp8_every_bf16_nope_value(scale):
    """All 65,536 bf16 patterns (NaN, infinities, zeros, subnormals included)
    as NoPE values at scales that take each way of forming the quotient: the
    two-term reciprocal (0.0125, 0.9375; verified for every pattern at the
    scale), the exact product by a power of two (0.5), and the division (a
    power of two whose reciprocal is not normal, and 3e38 with a subnormal
    reciprocal)."""
    rows = -(-65536 // 448)
    nope = np.zeros(rows * 448, np.uint16)
    nope[:65536] = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    lat = np.zeros((rows, 512), np.uint16)
    lat[:, :448] = nope.reshape(rows, 448)
    lat[:, 448:] = 0x3F80
    table = workloads.rope_cos_sin_table(rows=rows)
    cache = np.full(3 * 64 * 512, 0xAA, dtype=np.uint8)
    got, want = _run("fp8", lat, np.arange(rows), table, cache, np.arange(rows), 3, 64, 1,
                     fp8_scale=scale)
    assert G.first_diff(got, want) is None, G.first_diff(got, want)


def test_fp8_division_ties():
    """Rotated values x = M*s with M an E4M3 midpoint: x / s is the tie M and
    rounds to the even code, where x * RN(1/s) would round up."""
    s = np.float32(0.9375)
    mids = np.float32(1.0) + (2 * np.arange(8, dtype=np.float32) + 1) / np.float32(16)
    table = np.zeros((1, 64), np.float32)
    table[0, :8] = (mids * s).astype(np.float32)
    table[0, 8:32] = 1.0
    lat = np.zeros((32, 512), np.uint16)
    lat[:, 448:512:2] = 0x3F80
    cache = np.full(64 * 512, 0xAA, dtype=np.uint8)
    got, want = _run("fp8", lat, np.zeros(32, np.int64), table, cache, np.arange(32), 1, 64, 1,
                     fp8_scale=float(s))
    assert G.first_diff(got, want) is None, G.first_diff(got, want)


def test_empty_batch_writes_nothing():
    lat = torch.zeros((0, 512), dtype=torch.bfloat16, device=G.DEV)
    none = torch.zeros(0, dtype=torch.int64, device=G.DEV)
    table = G.to_dev(workloads.rope_cos_sin_table(4))
    v4 = torch.full((1, 64, 584), 0xAA, dtype=torch.uint8, device=G.DEV)
    bf = torch.full((1, 64, 512), 2.0, dtype=torch.bfloat16, device=G.DEV)
    f8 = torch.full((1, 64, 512), 0xAA, dtype=torch.uint8, device=G.DEV)
    kvq.rope_quant_insert_v4(lat, none, table, v4, none, 1)
    kvq.rope_plain_insert(lat, none, table, bf, none, 1)
    kvq.rope_plain_insert(lat, none, table, f8.view(torch.float8_e4m3fn), none, 1, fp8_scale=1.0)
    torch.cuda.synchronize()
    assert bool((v4 == 0xAA).all()) and bool((bf == 2.0).all()) and bool((f8 == 0xAA).all())


# --------------------------------------------------------------- ring rows

def _ring(rows, slots, state, nb, sb, state_stride, row_stride):
    """rows: contiguous [N, 1024]; state: flat float32 buffer, seen by the
    kernel as [nb, sb, 1024] with the given strides (floats)."""
    want = state.copy()
    oracle.save_ring_rows(rows, slots, want, nb, sb, state_stride, row_stride)
    d = G.to_dev(state)
    view = d.as_strided((nb, sb, 1024), (state_stride, row_stride, 1))
    kvq.save_ring_rows(G.to_dev(rows), G.to_dev(np.asarray(slots, np.int64)), view)
    torch.cuda.synchronize()
    return d.cpu().numpy().view(np.uint32), want.view(np.uint32)


def test_ring_rows_65536():
    w = workloads.ring_rows(seed=0)
    st = w["state"].reshape(-1)
    got, want = _ring(w["rows"], w["slot_mapping"], st, w["num_blocks"], w["state_block"],
                      w["state_block"] * 1024, 1024)
    assert not np.array_equal(want, st.view(np.uint32))
    assert G.first_diff(got, want) is None, G.first_diff(got, want)


def test_ring_rows_large_1048576():
    """The bandwidth case: 1,048,576 rows (4 GiB) into 8,192 blocks of 128."""
    w = workloads.ring_rows(seed=1, num_rows=1_048_576, num_blocks=8192, state_block=128)
    st = w["state"].reshape(-1)
    got, want = _ring(w["rows"], w["slot_mapping"], st, w["num_blocks"], w["state_block"],
                      w["state_block"] * 1024, 1024)
    assert G.first_diff(got, want) is None, G.first_diff(got, want)


def test_ring_rows_strides_pads_and_payloads():
    """Rows of a wider array (stride 1032), ring rows 1028 floats apart and
    blocks with a gap; NaN payloads and -0.0 survive; slots -1, -7 and past
    the state are skipped."""
    rng = np.random.default_rng(29)
    N, nb, sb = 300, 3, 64
    wide = rng.standard_normal((N, 1032)).astype(np.float32)
    wide.view(np.uint32)[0, :8] = [0x7FA00001, 0xFFC00000, 0x80000000, 0x00000001, 0x7F800000,
                                   0xFF800000, 0x7F7FFFFF, 0x7FFFFFFF]
    rows = wide[:, :1024]
    slots = np.concatenate([rng.permutation(nb * sb), np.full(N - nb * sb, -1)]).astype(np.int64)
    rng.shuffle(slots)
    neg = np.nonzero(slots == -1)[0]
    slots[neg[:3]] = [-7, nb * sb, nb * sb + 5]
    row_stride, state_stride = 1028, 64 * 1028 + 36
    state = np.empty(nb * state_stride, np.float32)
    state.view(np.uint32)[:] = workloads.RING_POISON_BITS
    want = state.copy()
    oracle.save_ring_rows(rows, slots, want, nb, sb, state_stride, row_stride)
    d = G.to_dev(state)
    view = d.as_strided((nb, sb, 1024), (state_stride, row_stride, 1))
    kvq.save_ring_rows(G.to_dev(wide)[:, :1024], G.to_dev(slots), view)
    torch.cuda.synchronize()
    got = d.cpu().numpy().view(np.uint32)
    assert G.first_diff(got, want.view(np.uint32)) is None


def test_ring_rows_empty():
    state = torch.full((2, 4, 1024), 3.0, device=G.DEV)
    kvq.save_ring_rows(torch.zeros((0, 1024), device=G.DEV),
                       torch.zeros(0, dtype=torch.int64, device=G.DEV), state)
    torch.cuda.synchronize()
    assert bool((state == 3.0).all())
