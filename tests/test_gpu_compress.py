"""GPU parity of fused_save_compress_norm against the float64 oracle.

The latent is compared per element within the bound the kernel's fp32
arithmetic allows (include/kvq.h):
    |got - exact| <= 2^-7 |exact| + 2^-18 mass + 2^-120
where ``mass`` is the oracle's r * |w| * sum_i w_i |kv_i|; NaN exactly where
the oracle has NaN. Rows that close no group must keep their poison, and the
ring state must match the oracle's bit for bit.
"""
import numpy as np
import pytest
import torch

import __graft_entry__
import fp8_quantized_paged_store_gb300 as kvq
import workloads
from oracle.compress import fused_save_compress_norm as oracle_fscn
from tests import _gpu as G

pytestmark = pytest.mark.gpu

POISON_BF16 = 0x7F81          # a NaN pattern the kernel never writes
POISON_I16 = int(np.array([POISON_BF16], np.uint16).view(np.int16)[0])


@pytest.fixture(scope="module", autouse=True)
def _built():
    __graft_entry__.build()


def _bf16_bits_to_f64(u16):
    return (u16.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _check_latent(got_bits, written, exact, mass):
    assert np.all(got_bits[~written] == POISON_BF16), "a row that closes no group was written"
    g = _bf16_bits_to_f64(got_bits[written])
    e, m = exact[written], mass[written]
    nan_e, nan_g = np.isnan(e), np.isnan(g)
    assert np.array_equal(nan_e, nan_g), f"NaN mismatch at {np.argwhere(nan_e != nan_g)[:5]}"
    ok = ~nan_e
    err = np.abs(g[ok] - e[ok])
    bound = 2.0 ** -7 * np.abs(e[ok]) + 2.0 ** -18 * m[ok] + 2.0 ** -120
    worst = np.max(err / bound) if err.size else 0.0
    assert worst <= 1.0, f"error {worst:.3f} x the bound"
    return worst


def _run(w, prev=False, row_stride=None, out_stride=512, state_row_stride=None, eps=None):
    """Oracle and kernel on the same batch; returns (worst error ratio,
    written count). The state is compared bit for bit."""
    R = w["compress_ratio"]
    eps = w["eps"] if eps is None else eps
    T = w["slot_mapping"].size
    rows = w["kv_score"]
    state_h = None if w["state"] is None else w["state"].copy()
    kw = {}
    if prev:
        kw = dict(prev_rows=w["prev_rows"], prev_row_indices=w["prev_row_indices"])
    written, exact, mass = oracle_fscn(rows, w["positions"], state_h, w["slot_mapping"],
                                       w["query_start_loc"], w["token_to_req"], w["weight"],
                                       eps, R, **kw)
    # device buffers, optionally with wider rows
    width = 512 * R
    if row_stride and row_stride != width:
        wide = np.full((rows.shape[0], row_stride), np.nan, np.float32)
        wide[:, :width] = rows
        kv_d = G.to_dev(wide)[:, :width]
    else:
        kv_d = G.to_dev(rows)
    out = torch.full((T, out_stride), POISON_I16, dtype=torch.int16, device=G.DEV)
    out_bf = out.view(torch.bfloat16)[:, :512]
    st_d = None
    if R == 2:
        st0 = w["state"]
        if state_row_stride and state_row_stride != 1024:
            nb, cap = st0.shape[0], st0.shape[1]
            big = np.full((nb, cap, state_row_stride), -7.0, np.float32)
            big[:, :, :1024] = st0
            st_full = G.to_dev(big)
            st_d = st_full[:, :, :1024]
        else:
            st_full = G.to_dev(st0)
            st_d = st_full
    pr = pi = None
    if prev:
        pr, pi = G.to_dev(w["prev_rows"]), G.to_dev(w["prev_row_indices"])
    kvq.fused_save_compress_norm(
        kv_d, G.to_dev(w["positions"]), st_d, G.to_dev(w["slot_mapping"]),
        G.to_dev(w["query_start_loc"]) if R == 2 else None,
        G.to_dev(w["token_to_req"]) if R == 2 else None,
        G.bf16_dev(w["weight"]), eps, R, out_bf, prev_rows=pr, prev_row_indices=pi)
    torch.cuda.synchronize()
    got = out.cpu().numpy().view(np.uint16)
    assert np.all(got[:, 512:] == POISON_BF16), "the kernel wrote past 512 columns"
    worst = _check_latent(got[:, :512], written, exact, mass)
    if R == 2:
        got_state = st_full.cpu().numpy()
        if state_row_stride and state_row_stride != 1024:
            assert np.all(got_state[:, :, 1024:] == -7.0), "the ring save wrote past 1024 floats"
            got_state = got_state[:, :, :1024]
        assert np.array_equal(got_state.view(np.uint32), state_h.view(np.uint32)), \
            "ring state differs from the oracle"
    return worst, int(written.sum())


@pytest.mark.parametrize("R", [1, 2])
def test_batch_mix(R):
    w = workloads.compress(seed=0, compress_ratio=R)
    worst, n = _run(w)
    assert n > 1000


def test_cr2_prev_rows():
    w = workloads.compress(seed=1, compress_ratio=2, prev_rows=True)
    _run(w, prev=True)


def test_cr2_decode_batch():
    """4096 requests of one token each: every group is a chunk-first group
    (half of them at odd positions, reading the ring), every token saved."""
    w = workloads.compress(seed=2, compress_ratio=2, num_reqs=4096, decode_fraction=1.0,
                           capacity=2, pad_tokens=5)
    _run(w)


def test_cr2_capacity_one_and_long_chunks():
    w = workloads.compress(seed=3, compress_ratio=2, num_reqs=16, max_chunk=3000,
                           decode_fraction=0.0, capacity=1)
    _run(w)


@pytest.mark.parametrize("R", [1, 2])
def test_strides(R):
    """kv rows 1028 floats apart (R = 2) or 516 (R = 1), latent rows 520
    elements apart, ring rows 1032 floats apart with the slack poisoned."""
    w = workloads.compress(seed=4, compress_ratio=R, num_reqs=40, max_chunk=100)
    _run(w, row_stride=1028 if R == 2 else 516, out_stride=520,
         state_row_stride=1032 if R == 2 else None)


@pytest.mark.parametrize("R", [1, 2])
def test_special_values(R):
    """NaN and +-inf in kv and scores, score gaps large enough to underflow
    exp, an all-zero row with eps 0 (0 * inf = NaN), small and large rows
    (squares stay inside binary32: |x| in [2^-63, 2^63])."""
    w = workloads.compress(seed=5, compress_ratio=R, num_reqs=64, max_chunk=20)
    rows = w["kv_score"]
    rng = np.random.default_rng(5)
    T = rows.shape[0]
    flat = rows.reshape(-1)
    idx = rng.choice(flat.size, 40, replace=False)
    flat[idx[:20]] = np.nan
    flat[idx[20:30]] = np.inf
    flat[idx[30:]] = -np.inf
    if R == 2:
        rows[3, 512:] = -200.0
        rows[4, 512:] = 150.0
    rows[7] = 0.0
    rows[8, :512] *= 1e-10
    rows[9, :512] *= 1e15
    w["kv_score"] = rows
    _run(w)
    _run(w, eps=0.0)


def test_large_sampled():
    """The benchmark batch (2048 requests, ~1M tokens, R = 2): the whole
    launch on the GPU; the oracle on 64 requests taken out as a batch of
    their own (requests are independent), compared row for row, plus their
    ring blocks."""
    w = workloads.compress(seed=0, compress_ratio=2, num_reqs=2048, max_chunk=1023,
                           decode_fraction=0.0, capacity=4, pad_tokens=0)
    T = w["slot_mapping"].size
    out = torch.full((T, 512), POISON_I16, dtype=torch.int16, device=G.DEV)
    st_d = G.to_dev(w["state"])
    kvq.fused_save_compress_norm(
        G.to_dev(w["kv_score"]), G.to_dev(w["positions"]), st_d, G.to_dev(w["slot_mapping"]),
        G.to_dev(w["query_start_loc"]), G.to_dev(w["token_to_req"]), G.bf16_dev(w["weight"]),
        w["eps"], 2, out.view(torch.bfloat16))
    torch.cuda.synchronize()
    got = out.cpu().numpy().view(np.uint16)
    got_state = st_d.cpu().numpy()
    rng = np.random.default_rng(9)
    reqs = np.sort(rng.choice(2048, 64, replace=False))
    qsl = w["query_start_loc"]
    tok = np.concatenate([np.arange(qsl[k], qsl[k + 1]) for k in reqs])
    sub_qsl = np.concatenate([[0], np.cumsum(qsl[reqs + 1] - qsl[reqs])])
    sub_t2r = np.repeat(np.arange(64), qsl[reqs + 1] - qsl[reqs])
    state = w["state"].copy()
    written, exact, mass = oracle_fscn(w["kv_score"][tok], w["positions"][tok], state,
                                       w["slot_mapping"][tok], sub_qsl, sub_t2r, w["weight"],
                                       w["eps"], 2)
    _check_latent(got[tok], written, exact, mass)
    blocks = np.unique(w["slot_mapping"][tok] // 4)
    assert np.array_equal(got_state[blocks].view(np.uint32), state[blocks].view(np.uint32))


def test_empty_batch():
    out = torch.zeros((4, 512), dtype=torch.bfloat16, device=G.DEV)
    z = torch.zeros(0, dtype=torch.int64, device=G.DEV)
    kvq.fused_save_compress_norm(torch.zeros((0, 1024), device=G.DEV), z, torch.zeros(
        (2, 2, 1024), device=G.DEV), z, torch.zeros(1, dtype=torch.int64, device=G.DEV), z,
        torch.ones(512, dtype=torch.bfloat16, device=G.DEV), 1e-6, 2, out[:0])
    torch.cuda.synchronize()
    assert bool((out == 0).all())


def test_cr2_inconsistent_inputs_are_skipped_like_the_oracle():
    """Request indices outside [0, num_reqs), an empty chunk, a token outside
    its request's chunk, chunk bounds outside the batch, a prev_rows index
    past the rows given, a ring slot past the state, padding tokens: the
    kernel skips what the oracle skips and writes the same rows and ring
    state."""
    w = workloads.compress(seed=6, compress_ratio=2, num_reqs=12, max_chunk=9,
                           decode_fraction=0.2, capacity=2, pad_tokens=6, prev_rows=True)
    qsl = w["query_start_loc"].copy()
    t2r = w["token_to_req"].copy()
    slots = w["slot_mapping"].copy()
    qsl[0] = -4                              # a chunk start below 0 (reads as 0)
    qsl[5] = qsl[4]                          # request 4 becomes empty (its tokens now belong nowhere)
    qsl[-1] = 10 ** 6                        # a chunk end past the batch
    t2r[0] = 99                              # a request index past num_reqs
    t2r[w["num_real"]:] = -3                 # padding tokens with a negative request index
    slots[2] = w["state"].shape[0] * 2 + 1   # a ring slot past the state
    idx = w["prev_row_indices"].copy()
    idx[7] = 10 ** 6                         # a prev_rows index past the rows given
    w.update(query_start_loc=qsl, token_to_req=t2r, slot_mapping=slots, prev_row_indices=idx)
    _run(w, prev=True)
    _run(w)
