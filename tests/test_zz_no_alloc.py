"""mxfp4_mla_sparse_attention_noalloc: the sparse attention for callers that
must not allocate device memory (a framework that owns all device memory
through its own pool and gives a library no allocator; a latency-critical
loop that cannot pay for cudaMalloc's possible device synchronisation). It
takes the split schedule's scratch from an array inside the library.

Called here through the C ABI, twice in a row on different inputs (the second
call finds the first call's partial results still in the shared array), and
compared with the existing entry point given a workspace of its own: the
results must lie within the attention tests' bound of the float64 oracle,
and, being the same kernels on the same schedule, they are expected to be
identical bit for bit. Kept in a file that pytest collects last.
"""
import ctypes

import numpy as np
import pytest
import torch

import __graft_entry__
import fp8_quantized_paged_store_gb300 as kvq
import oracle
import workloads
from oracle.attention import mxfp4_mla_sparse_attention as attn_oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    __graft_entry__.build()


def _inputs(seed, nq, nh, topk, num_slots):
    rng = np.random.default_rng(seed)
    lat = workloads.f32_to_bf16_bits((rng.standard_t(4, (num_slots, 512)) * 0.5)
                                     .astype(np.float32))
    cache = np.zeros(num_slots * 272, np.uint8)
    oracle.mxfp4_mla_store(lat, np.arange(num_slots, dtype=np.int64), cache, 1, num_slots,
                           num_slots, threads=oracle.default_threads())
    q = workloads.f32_to_bf16_bits(rng.standard_normal((nq, nh, 512)).astype(np.float32))
    idx = np.stack([rng.integers(-1, num_slots, topk) for _ in range(nq)]).astype(np.int64)
    idx[:, 0] = rng.integers(0, num_slots, nq)
    return q, cache, idx


def _noalloc(qd, cd, idd, sm_scale, num_slots, out, lse, status):
    """One call of the C entry point through ctypes, on torch's current stream."""
    nq, nh, _ = qd.shape
    rc = kvq.lib().mxfp4_mla_sparse_attention_noalloc(
        qd.data_ptr(), nq, nh, qd.stride(0), qd.stride(1), cd.data_ptr(), 1, num_slots,
        num_slots, idd.data_ptr(), idd.shape[1], ctypes.c_float(sm_scale), out.data_ptr(),
        out.stride(0), out.stride(1), lse.data_ptr(), status.data_ptr(),
        torch.cuda.current_stream().cuda_stream)
    assert rc == kvq.KVQ_OK, kvq.lib().kvq_strerror(rc)


@pytest.mark.parametrize("shapes", [(3, 128, 4096, 16_384), (40, 64, 700, 8_192)])
def test_noalloc_matches_the_workspace_entry_point_on_two_calls(shapes):
    nq, nh, topk, num_slots = shapes
    dev = torch.device("cuda", 0)
    sm_scale = 1 / np.sqrt(512)
    for call, seed in enumerate((31, 32)):
        q, cache, idx = _inputs(seed + nq, nq, nh, topk, num_slots)
        qd = torch.from_numpy(q.view(np.int16)).to(dev).view(torch.bfloat16)
        cd = torch.from_numpy(cache).to(dev)
        idd = torch.from_numpy(idx).to(dev)
        status = torch.zeros(1, dtype=torch.int32, device=dev)
        out_a = torch.empty((nq, nh, 512), dtype=torch.bfloat16, device=dev)
        lse_a = torch.empty((nq, nh), dtype=torch.float32, device=dev)
        _noalloc(qd, cd, idd, sm_scale, num_slots, out_a, lse_a, status)
        lse_b = torch.empty((nq, nh), dtype=torch.float32, device=dev)
        out_b, _ = kvq.mxfp4_mla_sparse_attention(qd, cd, idd, sm_scale, lse=lse_b,
                                                  status=status, workspace=True)
        torch.cuda.synchronize()
        assert int(status.item()) == 0, "a kernel wait timed out"
        a = out_a.float().cpu().numpy().astype(np.float64)
        b = out_b.float().cpu().numpy().astype(np.float64)
        want, want_lse, mass = attn_oracle(q, cache, 1, num_slots, num_slots, idx, sm_scale)
        bound = 2.0 ** -7 * (mass + np.abs(want)) + 2.0 ** -100
        assert np.all(np.abs(a - want) <= bound), f"call {call}: no-alloc output beyond the bound"
        assert np.all(np.abs(b - want) <= bound), f"call {call}: workspace output beyond the bound"
        fin = np.isfinite(want_lse)
        la = lse_a.cpu().numpy().astype(np.float64)
        np.testing.assert_allclose(la[fin], want_lse[fin], rtol=0, atol=2e-3)
        assert torch.equal(out_a.view(torch.int16), out_b.view(torch.int16)), f"call {call}"
        assert torch.equal(lse_a, lse_b), f"call {call}"


def test_noalloc_refuses_shapes_beyond_its_scratch_and_bad_arguments():
    """Rejections happen on the host, before any launch: 129 heads is an
    invalid shape (KVQ_EINVAL); the built-in array is sized for the split
    schedule of 128 heads on this GPU, so a valid shape never exceeds it
    here, and the size query says so."""
    L = kvq.lib()
    need = L.mxfp4_mla_sparse_attention_workspace_size(1, 128, 8192)
    assert 0 < need <= 40 << 20
    dev = torch.device("cuda", 0)
    q = torch.zeros((2, 129, 512), dtype=torch.bfloat16, device=dev)
    cache = torch.zeros(64 * 272, dtype=torch.uint8, device=dev)
    idx = torch.zeros((2, 4), dtype=torch.int64, device=dev)
    out = torch.empty((2, 129, 512), dtype=torch.bfloat16, device=dev)
    rc = L.mxfp4_mla_sparse_attention_noalloc(
        q.data_ptr(), 2, 129, q.stride(0), q.stride(1), cache.data_ptr(), 1, 64, 64,
        idx.data_ptr(), 4, ctypes.c_float(0.1), out.data_ptr(), out.stride(0), out.stride(1),
        None, None, None)
    assert rc == kvq.KVQ_EINVAL
