"""GPU parity of mxfp4_mla_sparse_attention against the float64 oracle.

The kernel rounds the probabilities to bf16 for the p.v product and the
output to bf16, and accumulates in fp32 on the tensor cores, so outputs are
compared with a bound derived from that arithmetic rather than bit for bit:
  |out - exact| <= 2**-7 * (sum_j softmax_j |k_j[d]| + |exact|) + 2**-100
per element (the bf16 rounding of P contributes at most 2**-9 of the first
term, the final rounding 2**-9 of the second, fp32 score and exp2 errors well
under 2**-12; 2**-7 leaves a margin of about four). The absolute 2**-100
covers the fp32 floor: exp2 flushes probabilities below 2**-126 of the
running maximum to zero, and at most 2**11 keys with |k| < 2**14 can lose
less than 2**-101 that way (an exact output of 6e-50 comes out as 0).
lse: |lse - exact| <= 2e-3.
Both schedules are checked: key tiles split evenly over the SMs (pieces of a
(query, value half) cut between CTAs merged by log-sum-exp; the default), and
one CTA per (query, value half). The bound holds for both: a split piece's
output (normalised by its own softmax sum) is rounded to bf16, which adds
at most 2**-9 of the first term, and the merge rounds to bf16 once more.
The packed cache is written by the oracle's store, never by the CUDA path.
"""
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


def _fill_cache(num_slots, seed, num_blocks=1, block_size=None, block_stride_rows=None):
    block_size = block_size or num_slots
    block_stride_rows = block_stride_rows or block_size
    rng = np.random.default_rng(seed)
    lat = workloads.f32_to_bf16_bits(
        (rng.standard_t(4, (num_slots, 512)) * 0.5).astype(np.float32))
    rows = (num_blocks - 1) * block_stride_rows + block_size
    cache = np.full(rows * 272, 0x5A, np.uint8)
    oracle.mxfp4_mla_store(lat, np.arange(num_slots, dtype=np.int64), cache, num_blocks,
                           block_size, block_stride_rows, threads=oracle.default_threads())
    return cache


def _run(q, cache, idx, sm_scale, num_blocks, block_size, block_stride_rows, q_full=None,
         split=True):
    """Kernel on the GPU; q_full (optional) is a wider buffer q is a view of."""
    dev = torch.device("cuda", 0)
    src = q if q_full is None else q_full
    qd = torch.from_numpy(np.ascontiguousarray(src).view(np.int16)).to(dev).view(torch.bfloat16)
    if q_full is not None:
        qd = qd[:, :q.shape[1], :512]
    cd = torch.from_numpy(cache).to(dev)
    if num_blocks > 1:
        cd = cd.as_strided((num_blocks, block_size, 272), (block_stride_rows * 272, 272, 1))
    else:
        cd = cd[:num_blocks * block_size * 272]
    idd = torch.from_numpy(np.ascontiguousarray(idx)).to(dev)
    lse = torch.empty((q.shape[0], q.shape[1]), dtype=torch.float32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    out, _ = kvq.mxfp4_mla_sparse_attention(qd, cd, idd, sm_scale, lse=lse, status=status,
                                            workspace=split)
    torch.cuda.synchronize()
    assert int(status.item()) == 0, "a kernel wait timed out"
    o = out.float().cpu().numpy().astype(np.float64)
    return o, lse.cpu().numpy().astype(np.float64)


def _check(q, cache, idx, sm_scale, num_blocks, block_size, block_stride_rows, q_full=None,
           split=True):
    out, lse = _run(q, cache, idx, sm_scale, num_blocks, block_size, block_stride_rows, q_full,
                    split)
    want, want_lse, mass = attn_oracle(q, cache, num_blocks, block_size, block_stride_rows, idx,
                                       sm_scale)
    err = np.abs(out - want)
    bound = 2.0 ** -7 * (mass + np.abs(want)) + 2.0 ** -100
    bad = np.argwhere(err > bound)
    assert bad.size == 0, (bad[:5], out[tuple(bad[0])], want[tuple(bad[0])],
                           mass[tuple(bad[0])])
    fin = np.isfinite(want_lse)
    assert np.array_equal(np.isfinite(lse), fin)
    assert np.all(np.isneginf(lse[~fin]))
    np.testing.assert_allclose(lse[fin], want_lse[fin], rtol=0, atol=2e-3)
    assert np.all(out[~fin] == 0)
    return out, want


def _queries(seed, nq, nh, scale=1.0):
    rng = np.random.default_rng(seed)
    return workloads.f32_to_bf16_bits((rng.standard_normal((nq, nh, 512)) * scale)
                                      .astype(np.float32))


@pytest.mark.parametrize("split", [True, False])
def test_small_two_tiles_with_pads(split):
    cache = _fill_cache(4096, seed=1)
    q = _queries(2, 3, 128)
    rng = np.random.default_rng(3)
    idx = np.stack([rng.permutation(4096)[:64] for _ in range(3)]).astype(np.int64)
    idx[0, 60:] = -1
    idx[1, 5] = 4096                         # outside the cache: dropped
    idx[2, ::7] = -1
    _check(q, cache, idx, 1 / np.sqrt(512), 1, 4096, 4096, split=split)


@pytest.mark.parametrize("heads", [1, 64, 127, 128])
@pytest.mark.parametrize("topk", [1, 31, 33, 100, 161])
def test_ragged_heads_and_topk(heads, topk):
    cache = _fill_cache(2048, seed=4)
    q = _queries(5 + heads, 2, heads)
    rng = np.random.default_rng(topk)
    idx = np.stack([rng.integers(-1, 2048, topk) for _ in range(2)]).astype(np.int64)
    idx[:, 0] = rng.integers(0, 2048, 2)     # at least one valid key per query
    _check(q, cache, idx, 0.05, 1, 2048, 2048)


def test_paged_cache_with_block_stride_and_strided_query():
    nb, bs, bsr = 40, 64, 96
    cache = _fill_cache(nb * bs, seed=6, num_blocks=nb, block_size=bs, block_stride_rows=bsr)
    rng = np.random.default_rng(7)
    q_full = workloads.f32_to_bf16_bits(rng.standard_normal((4, 130, 576)).astype(np.float32))
    q = np.ascontiguousarray(q_full[:, :128, :512])
    idx = np.stack([rng.permutation(nb * bs)[:256] for _ in range(4)]).astype(np.int64)
    _check(q, cache, idx, 0.04, nb, bs, bsr, q_full=q_full)
    _check(q, cache, idx, 0.04, nb, bs, bsr, q_full=q_full, split=False)


def test_queries_without_valid_keys_and_empty_topk():
    cache = _fill_cache(256, seed=8)
    q = _queries(9, 3, 128)
    idx = np.array([[-1] * 40, [300] * 40, list(range(40))], np.int64)
    out, _ = _check(q, cache, idx, 0.05, 1, 256, 256)
    assert np.all(out[:2] == 0)
    for split in (True, False):
        out0, lse0 = _run(q, cache, np.zeros((3, 0), np.int64), 0.05, 1, 256, 256, split=split)
        assert np.all(out0 == 0) and np.all(np.isneginf(lse0))


def test_growing_scores_exercise_the_output_rescale():
    """Keys ordered by increasing score with a large scale: the running max
    grows by more than the kernel's rescale threshold (32 log2 units) from
    tile to tile: at least once for 99 of the 128 heads, three times for
    head 0."""
    cache = _fill_cache(1024, seed=10)
    q = _queries(11, 1, 128)
    rows = oracle.mxfp4_mla_gather_dequant(cache, 1, 1024, 1024, np.arange(1024, dtype=np.int64))
    k = (rows.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    qd = (q.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    order = np.argsort(k @ qd[0, 0])           # ascending for head 0
    idx = order[None, -512:].astype(np.int64)
    _check(q, cache, idx, 2.0, 1, 1024, 1024)
    _check(q, cache, idx, 2.0, 1, 1024, 1024, split=False)


def test_scale_bytes_outside_the_permute_range():
    """Scale bytes 0, 1, 253 and 254 (results subnormal, or within a factor 4
    of the bf16 maximum) take the arithmetic decode instead of the byte
    permutes. About a third of the rows get byte 0 or 1 in half their groups.
    Rows 7, 135, 263 and 391 get byte 253 or 254 in four groups each (disjoint
    between them), with codes limited to magnitudes up to 1.5 so that every
    decoded value stays finite; each query's top-k holds one of them, and the
    query (near 2**-112, which keeps q.k in range) has the signs of that
    row's large values in its dims. Its logit then exceeds every other key's
    by at least 61 (log2 units), more than the kernel's rescale threshold of
    32, so it sets the running max when it arrives and the unnormalised p.v
    sums stay below the fp32 maximum: the output in its dims is its decoded
    values."""
    rng = np.random.default_rng(20)
    cache = _fill_cache(512, seed=21).reshape(512, 272)
    for r in range(0, 512, 3):
        groups = rng.choice(16, 8, replace=False)
        cache[r, 256 + groups] = rng.integers(0, 2, 8)
    huge = [7, 135, 263, 391]
    for i, r in enumerate(huge):
        for g in range(4 * i, 4 * i + 4):
            cache[r, 256 + g] = 253 + (g & 1)
            cache[r, 16 * g:16 * g + 16] &= 0xBB   # nibble magnitude index <= 3
    cache = cache.reshape(-1)
    z = np.abs(rng.standard_normal((4, 128, 512)))
    z = np.maximum(z, 2.0 ** -10) * 2.0 ** -112 * rng.choice([-1.0, 1.0], (4, 128, 512))
    for i, r in enumerate(huge):
        codes = cache[r * 272 + 64 * i:r * 272 + 64 * i + 64]
        nib = np.stack([codes & 15, codes >> 4], 1).reshape(-1)
        z[i, :, 128 * i:128 * i + 128] = np.abs(z[i, :, 128 * i:128 * i + 128]) * np.where(
            nib & 8, -1.0, 1.0)
    q = workloads.f32_to_bf16_bits(z.astype(np.float32))
    rest = np.setdiff1d(np.arange(512), huge)
    idx = np.stack([rng.permutation(rest)[:150] for _ in range(4)]).astype(np.int64)
    idx[0, 40], idx[1, 100], idx[2, 149], idx[3, 3] = huge
    idx[1, ::37] = -1
    for split in (True, False):
        out, want = _check(q, cache, idx, 4e-5, 1, 512, 512, split=split)
        assert np.all(np.isfinite(out)) and np.abs(want).max() > 2.0 ** 100


@pytest.mark.parametrize("split", [True, False])
def test_full_workload_128_queries_2048_keys(split):
    """The benchmark workload: 1,048,576-slot cache, 128 queries x 128 heads x
    2048 top-k indices with trailing pads; every output compared."""
    w = workloads.sparse_attention(seed=0)
    cache = np.zeros(w["num_slots"] * 272, np.uint8)
    oracle.mxfp4_mla_store(w["fill_latent"], w["fill_slots"], cache, 1, w["num_slots"],
                           w["num_slots"], threads=oracle.default_threads())
    _check(w["q"], cache, w["indices"], w["sm_scale"], 1, w["num_slots"], w["num_slots"],
           split=split)


@pytest.mark.parametrize("nq,topk,heads", [(1, 4096, 128), (1, 8192, 64), (5, 2048, 128),
                                           (3, 333, 128), (77, 64, 16), (200, 96, 128)])
def test_split_schedules(nq, topk, heads):
    """Shapes whose units are cut into many chunks (one query: each value
    half cut into 32 or 64 chunks, merged through the merge's parallel-weight
    path; five queries: ~15 chunks each), into a few (three queries of 333
    keys: two chunks, the per-thread path), or not at all (more units than
    SMs, or few tiles per unit), with ragged top-k and pads; both schedules
    against the oracle."""
    cache = _fill_cache(8192, seed=20 + nq)
    q = _queries(21 + topk, nq, heads)
    rng = np.random.default_rng(22 + heads)
    idx = np.stack([rng.integers(-1, 8192, topk) for _ in range(nq)]).astype(np.int64)
    idx[:, :3] = rng.integers(0, 8192, (nq, 3))
    _check(q, cache, idx, 0.06, 1, 8192, 8192)
    _check(q, cache, idx, 0.06, 1, 8192, 8192, split=False)


def test_split_workspace_too_small_is_refused():
    dev = torch.device("cuda", 0)
    q = torch.zeros((2, 128, 512), dtype=torch.bfloat16, device=dev)
    cache = torch.zeros(64 * 272, dtype=torch.uint8, device=dev)
    idx = torch.zeros((2, 2048), dtype=torch.int64, device=dev)
    need = kvq.attention_workspace_size(2, 128, 2048)
    assert need > 0
    ws = torch.empty(need - 256, dtype=torch.uint8, device=dev)
    with pytest.raises(kvq.KvqError):
        kvq.mxfp4_mla_sparse_attention(q, cache, idx, 0.1, workspace=ws)


def test_rejects_bad_arguments_on_gpu():
    dev = torch.device("cuda", 0)
    q = torch.zeros((2, 129, 512), dtype=torch.bfloat16, device=dev)
    cache = torch.zeros(64 * 272, dtype=torch.uint8, device=dev)
    idx = torch.zeros((2, 4), dtype=torch.int64, device=dev)
    with pytest.raises(kvq.KvqError):
        kvq.mxfp4_mla_sparse_attention(q, cache, idx, 0.1)    # 129 heads
    with pytest.raises(kvq.KvqError):
        kvq.mxfp4_mla_sparse_attention(q[:, :4], cache, idx, float("nan"))


def test_one_query_broadcast_with_query_stride_zero():
    """Every query the same row of memory (query stride 0: a view made by
    expand): the tensor map of Q then has a zero stride, or, if it cannot be
    made, Q is copied in 16-byte pieces; each query's output must match the
    oracle on its own indices, and equal ones for equal index rows."""
    dev = torch.device("cuda", 0)
    cache_np = _fill_cache(2048, seed=40)
    cache = torch.from_numpy(cache_np).to(dev)
    rng = np.random.default_rng(41)
    idx_np = np.stack([rng.permutation(2048)[:300] for _ in range(3)]).astype(np.int64)
    idx_np = np.concatenate([idx_np, idx_np[:1]])  # query 3 repeats query 0's indices
    q1 = _queries(42, 1, 96)
    qd = torch.from_numpy(q1.view(np.int16)).to(dev).view(torch.bfloat16).expand(4, 96, 512)
    assert qd.stride(0) == 0
    for split in (True, False):
        lse = torch.empty((4, 96), dtype=torch.float32, device=dev)
        status = torch.zeros(1, dtype=torch.int32, device=dev)
        out, _ = kvq.mxfp4_mla_sparse_attention(qd, cache, torch.from_numpy(idx_np).to(dev), 0.05,
                                                lse=lse, status=status, workspace=split)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        o = out.float().cpu().numpy().astype(np.float64)
        want, want_lse, mass = attn_oracle(np.repeat(q1, 4, axis=0), cache_np, 1, 2048, 2048,
                                           idx_np, 0.05)
        assert np.all(np.abs(o - want) <= 2.0 ** -7 * (mass + np.abs(want)) + 2.0 ** -100)
        np.testing.assert_allclose(lse.cpu().numpy(), want_lse, rtol=0, atol=2e-3)
        assert torch.equal(out[3].view(torch.int16), out[0].view(torch.int16))


def test_split_and_unsplit_replay_in_a_cuda_graph():
    """Both schedules captured in a CUDA graph (the split one is two
    launches, the merge a programmatic dependent of the attention grid; Q is
    read through a tensor map passed by value) replay to the eager bits, and
    follow the query buffer when it is overwritten in place."""
    dev = torch.device("cuda", 0)
    cache = torch.from_numpy(_fill_cache(4096, seed=30)).to(dev)
    rng = np.random.default_rng(31)
    idx = torch.from_numpy(np.stack([rng.permutation(4096)[:2048] for _ in range(4)])).to(dev)
    q = torch.from_numpy(_queries(32, 4, 128).view(np.int16)).to(dev).view(torch.bfloat16)
    q2 = torch.from_numpy(_queries(33, 4, 128).view(np.int16)).to(dev).view(torch.bfloat16)
    ws = torch.empty(kvq.attention_workspace_size(4, 128, 2048), dtype=torch.uint8, device=dev)
    assert ws.numel() > 0  # 4 queries x 2048 keys split
    for w in (ws, False):
        out = torch.empty((4, 128, 512), dtype=torch.bfloat16, device=dev)
        lse = torch.empty((4, 128), dtype=torch.float32, device=dev)
        status = torch.zeros(1, dtype=torch.int32, device=dev)

        def call():
            kvq.mxfp4_mla_sparse_attention(q, cache, idx, 0.05, out=out, lse=lse, status=status,
                                           workspace=w)

        call()
        torch.cuda.synchronize()
        want_o, want_l = out.clone(), lse.clone()
        q_saved = q.clone()
        q.copy_(q2)
        call()
        torch.cuda.synchronize()
        want_o2, want_l2 = out.clone(), lse.clone()
        q.copy_(q_saved)
        stream = torch.cuda.Stream()
        stream.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(stream):
            call()  # warm-up on the capture stream
        torch.cuda.current_stream().wait_stream(stream)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            call()
        out.zero_()
        lse.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), want_o.view(torch.int16))
        assert torch.equal(lse, want_l)
        q.copy_(q2)
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), want_o2.view(torch.int16))
        assert torch.equal(lse, want_l2)
        assert int(status.item()) == 0
        q.copy_(q_saved)


def _check_ragged(q, cache, runs, sm_scale, num_slots, first_offset=0, extra_tail=0):
    """Ragged runs against the oracle on the same runs padded with -1 into
    [num_queries, longest run]: pads are dropped, so the two are the same
    attention."""
    dev = torch.device("cuda", 0)
    nq = len(runs)
    lens = [len(r) for r in runs]
    flat = np.concatenate([np.full(first_offset, 7, np.int64)] + [np.asarray(r, np.int64)
                                                                    for r in runs]
                          + [np.full(extra_tail, 7, np.int64)])
    offsets = first_offset + np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    width = max(1, max(lens))
    padded = np.full((nq, width), -1, np.int64)
    for n, r in enumerate(runs):
        padded[n, :len(r)] = r
    want, want_lse, mass = attn_oracle(q, cache, 1, num_slots, num_slots, padded, sm_scale)
    qd = torch.from_numpy(np.ascontiguousarray(q).view(np.int16)).to(dev).view(torch.bfloat16)
    cd = torch.from_numpy(cache).to(dev)
    lse = torch.empty((nq, q.shape[1]), dtype=torch.float32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    out, _ = kvq.mxfp4_mla_sparse_attention_ragged(qd, cd, torch.from_numpy(flat).to(dev),
                                                   torch.from_numpy(offsets).to(dev), sm_scale,
                                                   lse=lse, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0, "a kernel wait timed out"
    got = out.float().cpu().numpy().astype(np.float64)
    bound = 2.0 ** -7 * (mass + np.abs(want)) + 2.0 ** -100
    bad = np.argwhere(np.abs(got - want) > bound)
    assert bad.size == 0, bad[:5]
    l = lse.cpu().numpy().astype(np.float64)
    fin = np.isfinite(want_lse)
    assert np.array_equal(np.isfinite(l), fin) and np.all(np.isneginf(l[~fin]))
    np.testing.assert_allclose(l[fin], want_lse[fin], rtol=0, atol=2e-3)
    return got


@pytest.mark.parametrize("heads", [128, 48])
def test_ragged_runs_of_every_length(heads):
    """Sparse prefill: one flat index array cut into runs of 0, 1, 31, 32,
    33, 65, 150, 220, 300, 700 and 2048 indices (with pads and out-of-range
    entries): 0 to 64 tiles, odd counts above one among them (3, 5, 7: the
    last tile's q.k unpaired, the producer groups' shares unequal); an empty
    run gives out = 0 and lse = -inf."""
    cache = _fill_cache(8192, seed=40)
    rng = np.random.default_rng(41)
    lens = [0, 1, 31, 32, 33, 65, 150, 220, 300, 700, 2048, 5]
    runs = []
    for L in lens:
        r = rng.integers(-1, 8192, L)
        if L:
            r[0] = rng.integers(0, 8192)
        if L > 10:
            r[3] = 9000                          # outside the cache: dropped
        runs.append(r)
    q = _queries(42 + heads, len(runs), heads)
    got = _check_ragged(q, cache, runs, 1 / np.sqrt(512), 8192)
    assert np.all(got[0] == 0)


def test_ragged_offsets_are_clamped_to_the_index_array():
    """A run may start past index 0; a last offset past the array's end is
    clamped to it, and an end below its start is an empty run."""
    cache = _fill_cache(4096, seed=43)
    rng = np.random.default_rng(44)
    runs = [rng.integers(0, 4096, 64), rng.integers(0, 4096, 40)]
    q = _queries(45, 2, 128)
    _check_ragged(q, cache, runs, 0.05, 4096, first_offset=5, extra_tail=3)
    dev = torch.device("cuda", 0)
    qd = torch.from_numpy(q.view(np.int16)).to(dev).view(torch.bfloat16)
    cd = torch.from_numpy(cache).to(dev)
    flat = torch.from_numpy(np.concatenate(runs).astype(np.int64)).to(dev)
    off = torch.tensor([0, 64, 10_000], dtype=torch.int64, device=dev)  # run 1 clamped to 40
    a, _ = kvq.mxfp4_mla_sparse_attention_ragged(qd, cd, flat, off, 0.05)
    b, _ = kvq.mxfp4_mla_sparse_attention_ragged(
        qd, cd, flat, torch.tensor([0, 64, 104], dtype=torch.int64, device=dev), 0.05)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    c, _ = kvq.mxfp4_mla_sparse_attention_ragged(
        qd, cd, flat, torch.tensor([50, 20, 104], dtype=torch.int64, device=dev), 0.05)
    assert torch.all(c[0].float() == 0)          # end below start: empty
