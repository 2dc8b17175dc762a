"""GPU parity of mxfp4_mla_rmsnorm_store (RMSNorm, then the MXFP4 store, in
one pass) against the CPU oracle, byte for byte over whole cache buffers."""
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


def _prenorm(rng, T):
    """Pre-norm latent: N(0,1) x per-token scale 2**U(-6,6) x per-channel
    scale U(0.25, 4), as bf16."""
    x = rng.standard_normal((T, 512)) * np.exp2(rng.uniform(-6, 6, (T, 1))) * \
        rng.uniform(0.25, 4.0, (1, 512))
    return workloads.f32_to_bf16_bits(x.astype(np.float32))


def _both(lat, w, eps, slots, buf, offset, nb, bs, bsr, threads=1):
    want = buf.copy()
    oracle.mxfp4_mla_rmsnorm_store(lat, w, eps, slots, want, nb, bs, bsr, cache_offset=offset,
                                   threads=threads)
    dbuf, view = G.paged_cache_dev(buf, offset, nb, bs, bsr)
    kvq.mxfp4_mla_rmsnorm_store(G.latent_dev(lat), G.bf16_dev(w), eps, G.to_dev(slots), view)
    torch.cuda.synchronize()
    return G.u8_host(dbuf), want


def test_rmsnorm_store_paged_16384_tokens():
    rng = np.random.default_rng(20)
    w_ = workloads.store_paged(seed=20)
    lat = _prenorm(rng, 16384)
    wt = workloads.f32_to_bf16_bits(rng.uniform(0.5, 1.5, 512).astype(np.float32))
    got, want = _both(lat, wt, 1e-6, w_["slot_mapping"], w_["cache"], w_["cache_offset"],
                      w_["num_blocks"], w_["block_size"], w_["block_stride_rows"])
    assert G.first_diff(got, want) is None, G.first_diff(got, want)


def test_rmsnorm_store_large_strided():
    """4.3M tokens through a 576-element row stride into 8,388,608 slots."""
    rng = np.random.default_rng(21)
    d = workloads.store_large(seed=0)
    wt = workloads.f32_to_bf16_bits(rng.uniform(0.5, 1.5, 512).astype(np.float32))
    got, want = _both(d["latent"], wt, 1e-5, d["slot_mapping"], d["cache"], 0, 1, d["num_slots"],
                      d["num_slots"], threads=oracle.default_threads())
    assert G.first_diff(got, want) is None, G.first_diff(got, want)


@pytest.mark.parametrize("eps", [0.0, 1e-6, 0.5])
def test_rmsnorm_store_degenerate_rows(eps):
    """All-zero rows (with eps 0 the scale is 1/0 and every value NaN), rows
    of NaN, infinities, subnormals, huge values, single spikes."""
    rng = np.random.default_rng(22)
    rows = _prenorm(rng, 12)
    rows[0] = 0
    rows[1] = 0x8000
    rows[2, ::7] = 0x7FC0
    rows[3, 5] = 0x7F80
    rows[4] = 0x0001
    rows[4, ::2] = 0x8003
    rows[5] = 0x7F00
    rows[6] = 0
    rows[6, 300] = 0x4000
    rows[7] = 0x3F80
    wt = workloads.f32_to_bf16_bits(rng.uniform(0.5, 1.5, 512).astype(np.float32))
    wt[::5] = 0x0000
    wt[1::11] = 0x8000 | wt[1::11]
    slots = np.arange(12, dtype=np.int64)
    buf = np.full(12 * ROW, 0xAA, np.uint8)
    got, want = _both(rows, wt, eps, slots, buf, 0, 1, 12, 12)
    assert G.first_diff(got, want) is None, G.first_diff(got, want)


@pytest.mark.parametrize("T", [1, 33, 1000])
def test_rmsnorm_store_ragged_and_pads(T):
    rng = np.random.default_rng(23 + T)
    lat = _prenorm(rng, T)
    wt = workloads.f32_to_bf16_bits(rng.uniform(0.5, 1.5, 512).astype(np.float32))
    n = 2 * T + 1
    slots = rng.choice(n, T, replace=False).astype(np.int64)
    slots[rng.random(T) < 0.2] = -1
    buf = np.full(n * ROW, 0xAA, np.uint8)
    got, want = _both(lat, wt, 1e-6, slots, buf, 0, 1, n, n)
    assert G.first_diff(got, want) is None, G.first_diff(got, want)
