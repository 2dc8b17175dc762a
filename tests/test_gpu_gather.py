"""GPU parity of mxfp4_mla_gather_dequant against the CPU oracle, element for
element (bf16 bit patterns)."""
import numpy as np
import pytest
import torch

import __graft_entry__
import fp8_quantized_paged_store_gb300 as kvq
import oracle
import workloads
from tests import _gpu as G

pytestmark = pytest.mark.gpu
ROW = 272


@pytest.fixture(scope="module", autouse=True)
def _built():
    __graft_entry__.build()


def _gather_both(buf, offset, nb, bs, bsr, idx, out_stride=512, threads=1):
    want = oracle.mxfp4_mla_gather_dequant(buf, nb, bs, bsr, idx.reshape(-1),
                                           cache_offset=offset, threads=threads)
    dbuf, view = G.paged_cache_dev(buf, offset, nb, bs, bsr)
    n = idx.size
    out_full = torch.full((n, out_stride), -1, dtype=torch.int16, device=G.DEV)
    out = out_full.view(torch.bfloat16)[:, :512]
    kvq.mxfp4_mla_gather_dequant(view, G.to_dev(idx.reshape(-1)), out=out)
    torch.cuda.synchronize()
    got_full = G.u16_host(out_full.view(torch.bfloat16))
    if out_stride > 512:
        assert np.all(got_full[:, 512:] == 0xFFFF), "gather wrote past the row"
    return got_full[:, :512], want


def test_gather_1048576_slot_cache_128x2048():
    """Full size: 1,048,576-slot packed cache (filled by the oracle store from
    Student-t rows), 128 queries x 2048 distinct indices with trailing pads."""
    w = workloads.gather(seed=0)
    nthreads = oracle.default_threads()
    buf = np.zeros(w["num_slots"] * ROW, dtype=np.uint8)
    oracle.mxfp4_mla_store(w["fill_latent"], w["fill_slots"], buf, 1, w["num_slots"],
                           w["num_slots"], threads=nthreads)
    got, want = _gather_both(buf, 0, 1, w["num_slots"], w["num_slots"], w["indices"],
                             threads=nthreads)
    assert G.first_diff(got, want) is None, G.first_diff(got, want)


def test_gather_every_code_at_every_scale_byte():
    """16 rows x 16 groups cover all 256 scale bytes (including 0, 1, 253, 254
    and the E8M0 NaN 255); each group holds all 16 codes twice."""
    buf = np.zeros((16, ROW), dtype=np.uint8)
    codes = np.tile(np.arange(16, dtype=np.uint8), 32)           # 512 codes
    packed = codes[0::2] | (codes[1::2] << 4)
    rng = np.random.default_rng(1)
    for r in range(16):
        buf[r, :256] = rng.permutation(packed.reshape(16, 16), axis=1).reshape(-1) if r else packed
        buf[r, 256:] = np.arange(16 * r, 16 * r + 16, dtype=np.uint8)
    idx = np.concatenate([np.arange(16), np.arange(16)[::-1], [-1, 3]]).astype(np.int64)
    got, want = _gather_both(buf.reshape(-1), 0, 1, 16, 16, idx)
    assert G.first_diff(got, want) is None, G.first_diff(got, want)


@pytest.mark.parametrize("n", [1, 2, 31, 33, 100])
def test_gather_pads_out_of_range_paged_and_strided_out(n):
    rng = np.random.default_rng(n)
    nb, bs, bsr, off = 6, 8, 11, 3
    rows = off + (nb - 1) * bsr + bs
    buf = rng.integers(0, 256, size=rows * ROW, dtype=np.uint8)
    buf.reshape(rows, ROW)[:, 256:] = rng.integers(100, 150, size=(rows, 16))
    idx = rng.integers(-2, nb * bs + 3, size=n).astype(np.int64)
    idx[0] = -1
    got, want = _gather_both(buf, off * ROW, nb, bs, bsr, idx, out_stride=520)
    assert G.first_diff(got, want) is None, G.first_diff(got, want)


def test_gather_of_gpu_store_round_trip():
    """store then gather on the GPU equals the oracle's store then gather."""
    w = workloads.store_paged(seed=3, num_tokens=4096, num_blocks=128, block_size=64,
                              block_stride_rows=96, layer_row_offset=16)
    dbuf, view = G.paged_cache_dev(w["cache"], w["cache_offset"], w["num_blocks"],
                                   w["block_size"], w["block_stride_rows"])
    kvq.mxfp4_mla_store(G.latent_dev(w["latent"]), G.to_dev(w["slot_mapping"]), view)
    idx = w["slot_mapping"].copy()
    out = kvq.mxfp4_mla_gather_dequant(view, G.to_dev(idx))
    torch.cuda.synchronize()
    want_cache = w["cache"].copy()
    oracle.mxfp4_mla_store(w["latent"], w["slot_mapping"], want_cache, w["num_blocks"],
                           w["block_size"], w["block_stride_rows"], cache_offset=w["cache_offset"])
    want = oracle.mxfp4_mla_gather_dequant(want_cache, w["num_blocks"], w["block_size"],
                                           w["block_stride_rows"], idx,
                                           cache_offset=w["cache_offset"])
    got = G.u16_host(out)
    assert G.first_diff(got, want) is None, G.first_diff(got, want)
