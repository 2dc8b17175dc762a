"""Entry points on pinned HOST buffers: the kernels read their inputs from,
and write their rows into, page-locked host memory that the device addresses
at the same pointer, with no copy before or after the call. Compared byte for
byte with the CPU oracle (store) or with the same call on device buffers."""
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


def _pinned(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).pin_memory()


def test_pointer_kind():
    L = kvq.lib()
    d = torch.zeros(64, device=G.DEV)
    h = torch.zeros(64).pin_memory()
    pageable = torch.zeros(64)
    assert L.kvq_pointer_kind(d.data_ptr()) == kvq.KVQ_PTR_DEVICE
    assert L.kvq_pointer_kind(d[17:].data_ptr()) == kvq.KVQ_PTR_DEVICE
    assert L.kvq_pointer_kind(h.data_ptr()) == kvq.KVQ_PTR_HOST_MAPPED
    assert L.kvq_pointer_kind(h[17:].data_ptr()) == kvq.KVQ_PTR_HOST_MAPPED
    assert L.kvq_pointer_kind(pageable.data_ptr()) == 0
    assert L.kvq_pointer_kind(None) == kvq.KVQ_EINVAL


def test_pageable_host_tensor_is_refused():
    lat = torch.zeros((4, 512), dtype=torch.bfloat16)
    slots = torch.zeros(4, dtype=torch.int64, device=G.DEV)
    cache = torch.zeros(8 * ROW, dtype=torch.uint8, device=G.DEV)
    with pytest.raises(TypeError):
        kvq.mxfp4_mla_store(lat, slots, cache)


@pytest.mark.parametrize("where", ["all_host", "host_inputs", "host_cache"])
def test_store_paged_on_host_buffers(where):
    """The paged workload (16,384 tokens, block stride 192 rows with other
    layers' rows poisoned, 5% pads): latent, slots and cache on the host in
    any mix with the device."""
    w = workloads.store_paged(seed=7)
    nb, bs, bsr, off = w["num_blocks"], w["block_size"], w["block_stride_rows"], w["cache_offset"]
    want = w["cache"].copy()
    oracle.mxfp4_mla_store(w["latent"], w["slot_mapping"], want, nb, bs, bsr, cache_offset=off)
    host_in = where in ("all_host", "host_inputs")
    host_out = where in ("all_host", "host_cache")
    lat = (_pinned(w["latent"].view(np.int16)) if host_in
           else G.to_dev(w["latent"].view(np.int16))).view(torch.bfloat16)
    slots = _pinned(w["slot_mapping"]) if host_in else G.to_dev(w["slot_mapping"])
    buf = _pinned(w["cache"]) if host_out else G.to_dev(w["cache"])
    view = buf[off:].as_strided((nb, bs, ROW), (bsr * ROW, ROW, 1))
    kvq.mxfp4_mla_store(lat, slots, view)
    torch.cuda.synchronize()
    got = buf.numpy() if host_out else buf.cpu().numpy()
    assert G.first_diff(got, want) is None, G.first_diff(got, want)


def test_store_strided_latent_from_host():
    """200,000 tokens read through a 576-element row stride from pinned host
    memory into a pinned host cache of 400,000 slots (1% pads)."""
    lat_full = workloads.store_large_latent(seed=3, num_tokens=200_000, row_stride=576)
    slots = workloads.store_large_slots(seed=3, num_tokens=200_000, num_slots=400_000)
    want = np.full(400_000 * ROW, 0xAA, dtype=np.uint8)
    oracle.mxfp4_mla_store(lat_full[:, :512], slots, want, 1, 400_000, 400_000,
                           threads=oracle.default_threads())
    lat_h = _pinned(lat_full.view(np.int16)).view(torch.bfloat16)[:, :512]
    cache_h = _pinned(np.full(400_000 * ROW, 0xAA, dtype=np.uint8))
    kvq.mxfp4_mla_store(lat_h, _pinned(slots), cache_h)
    torch.cuda.synchronize()
    assert G.first_diff(cache_h.numpy(), want) is None, G.first_diff(cache_h.numpy(), want)


def test_gather_into_host_output():
    """The gather reads a device cache and writes its bf16 rows into pinned
    host memory; the indices come from the host too. Same bits as the gather
    into device memory."""
    w = workloads.gather(seed=2, num_slots=65_536, num_queries=16, topk=512)
    cache = torch.zeros(65_536 * ROW, dtype=torch.uint8, device=G.DEV)
    kvq.mxfp4_mla_store(G.bf16_dev(w["fill_latent"]), G.to_dev(w["fill_slots"]), cache)
    idx_d = G.to_dev(w["indices"])
    dev_out = kvq.mxfp4_mla_gather_dequant(cache, idx_d)
    host_out = kvq.mxfp4_mla_gather_dequant(cache, _pinned(w["indices"]))
    torch.cuda.synchronize()
    assert not host_out.is_cuda and host_out.is_pinned()
    assert torch.equal(host_out.view(torch.int16), dev_out.view(torch.int16).cpu())


@pytest.mark.parametrize("record", ["mxfp8", "nvfp4"])
def test_rope_insert_on_host_buffers(record):
    """A V4.1 insert (65,536 tokens, R = 4, 0.05% NaN) with the latent,
    positions, cos/sin table, slots and paged cache all in pinned host
    memory: byte for byte the oracle's cache."""
    fo, fk, width = {"mxfp8": (oracle.rope_quant_insert_mxfp8, kvq.rope_quant_insert_mxfp8, 528),
                     "nvfp4": (oracle.rope_quant_insert_nvfp4, kvq.rope_quant_insert_nvfp4,
                               288)}[record]
    w = workloads.rope_insert(seed=11, record=record)
    np_, cb = w["num_pages"], w["cache_block"]
    want = w["cache"].copy()
    fo(w["latent"], w["positions"], w["cos_sin"], want, w["cache_slots"], np_, cb, cb * width,
       w["compress_ratio"], False)
    cache_h = _pinned(w["cache"])
    view = cache_h.as_strided((np_, cb, width), (cb * width, width, 1))
    fk(_pinned(w["latent"].view(np.int16)).view(torch.bfloat16), _pinned(w["positions"]),
       _pinned(w["cos_sin"]), view, _pinned(w["cache_slots"]), w["compress_ratio"])
    torch.cuda.synchronize()
    assert G.first_diff(cache_h.numpy(), want) is None, G.first_diff(cache_h.numpy(), want)


def test_ring_rows_into_host_state():
    """save_ring_rows from pinned host rows into a pinned host ring state:
    bit copies, pads skipped, the rest of the state untouched."""
    w = workloads.ring_rows(seed=5, num_rows=4096, num_blocks=64, state_block=128)
    want = w["state"].copy()
    nb, sb = want.shape[0], want.shape[1]
    oracle.save_ring_rows(w["rows"], w["slot_mapping"], want, nb, sb, sb * 1024, 1024)
    state_h = _pinned(w["state"])
    kvq.save_ring_rows(_pinned(w["rows"]), _pinned(w["slot_mapping"]), state_h)
    torch.cuda.synchronize()
    assert np.array_equal(state_h.numpy().view(np.uint32), want.view(np.uint32))


@pytest.mark.parametrize("heads", [128, 48])
def test_attention_query_and_output_on_host(heads):
    """Sparse attention with the queries read from and the output and lse
    written to pinned host memory (packed cache and indices on the device):
    the same bits as with every buffer on the device. A host-mapped query
    is copied in 16-byte pieces that zero the rows past num_heads
    themselves; a device one arrives by tensor-map boxes whose out-of-range
    rows read as zeros: 48 heads compare the two."""
    w = workloads.sparse_attention(seed=3, num_queries=8, num_heads=heads, topk=256,
                                   num_slots=16_384)
    cache = torch.zeros(16_384 * ROW, dtype=torch.uint8, device=G.DEV)
    kvq.mxfp4_mla_store(G.bf16_dev(w["fill_latent"]), G.to_dev(w["fill_slots"]), cache)
    idx = G.to_dev(w["indices"])
    q_np = w["q"].reshape(8, heads, 512)
    status = torch.zeros(1, dtype=torch.int32, device=G.DEV)
    lse_d = torch.empty((8, heads), dtype=torch.float32, device=G.DEV)
    out_d, _ = kvq.mxfp4_mla_sparse_attention(G.bf16_dev(q_np), cache, idx, w["sm_scale"],
                                              lse=lse_d, status=status)
    q_h = _pinned(q_np.view(np.int16)).view(torch.bfloat16)
    lse_h = torch.empty((8, heads), dtype=torch.float32).pin_memory()
    out_h, _ = kvq.mxfp4_mla_sparse_attention(q_h, cache, idx, w["sm_scale"], lse=lse_h,
                                              status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0, "a kernel wait timed out"
    assert not out_h.is_cuda
    assert torch.equal(out_h.view(torch.int16), out_d.view(torch.int16).cpu())
    assert torch.equal(lse_h, lse_d.cpu())


def test_rmsnorm_store_on_host_buffers():
    """The RMSNorm-fused store with the latent, weight, slots and paged cache
    in pinned host memory: byte for byte the oracle's cache."""
    w = workloads.store_paged(seed=8)
    nb, bs, bsr, off = w["num_blocks"], w["block_size"], w["block_stride_rows"], w["cache_offset"]
    rng = np.random.default_rng(8)
    weight = workloads.f32_to_bf16_bits(rng.uniform(0.5, 1.5, 512).astype(np.float32))
    want = w["cache"].copy()
    oracle.mxfp4_mla_rmsnorm_store(w["latent"], weight, 1e-6, w["slot_mapping"], want, nb, bs,
                                   bsr, cache_offset=off)
    buf = _pinned(w["cache"])
    view = buf[off:].as_strided((nb, bs, ROW), (bsr * ROW, ROW, 1))
    kvq.mxfp4_mla_rmsnorm_store(_pinned(w["latent"].view(np.int16)).view(torch.bfloat16),
                                _pinned(weight.view(np.int16)).view(torch.bfloat16), 1e-6,
                                _pinned(w["slot_mapping"]), view)
    torch.cuda.synchronize()
    assert G.first_diff(buf.numpy(), want) is None, G.first_diff(buf.numpy(), want)


def test_compressor_on_host_buffers():
    """fused_save_compress_norm with every argument in pinned host memory
    gives the same latent rows and ring state, bit for bit, as with every
    argument on the device."""
    w = workloads.compress(seed=3, compress_ratio=2, num_reqs=64, max_chunk=100)
    T = w["slot_mapping"].size
    args = [w["kv_score"], w["positions"], w["state"], w["slot_mapping"], w["query_start_loc"],
            w["token_to_req"]]
    outs = []
    for where in ("device", "host"):
        put = G.to_dev if where == "device" else _pinned
        kv, pos, st, sl, qsl, t2r = (put(a) for a in args)
        wt = put(w["weight"].view(np.int16)).view(torch.bfloat16)
        out = (torch.zeros((T, 512), dtype=torch.int16, device=G.DEV) if where == "device"
               else torch.zeros((T, 512), dtype=torch.int16).pin_memory())
        kvq.fused_save_compress_norm(kv, pos, st, sl, qsl, t2r, wt, w["eps"], 2,
                                     out.view(torch.bfloat16))
        torch.cuda.synchronize()
        outs.append((out.cpu().numpy(), st.cpu().numpy().view(np.uint32)))
    assert np.array_equal(outs[0][0], outs[1][0])
    assert np.array_equal(outs[0][1], outs[1][1])
    assert np.any(outs[0][0] != 0)
