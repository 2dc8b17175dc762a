"""Pins of the fused_save_compress_norm oracle (CPU only).

Page: 'vllm.models.deepseek_v41.common.ops.fused_compress_quant_cache'
(fused_save_compress_norm: closed groups of R in {1, 2} positions pooled
into an RMS-normalised bf16 latent; the R = 2 ring of per-request rows,
position p in row p % capacity; chunk-first tokens read their predecessor
from the ring or from prev_rows; the chunk's last capacity rows saved unless
prev_rows is given). The pooling is read as a per-channel softmax of the
scores over the group; each pin checks the oracle by a route of its own:
closed forms, a token-by-token streaming model of the compressor, and the
invariance of the result under splitting the requests into chunks.
"""
import math

import numpy as np
import pytest

import workloads
from oracle.compress import fused_save_compress_norm as fscn

L = 512
ONE = np.full(L, 0x3F80, np.uint16)          # bf16 1.0 weights


def _bf(a):
    return workloads.f32_to_bf16_bits(np.asarray(a, np.float32))


def _cr1(rows, eps=1e-6, weight=ONE, slots=None, positions=None):
    rows = np.asarray(rows, np.float32)
    T = rows.shape[0]
    slots = np.arange(T) if slots is None else np.asarray(slots)
    positions = np.arange(T) if positions is None else np.asarray(positions)
    return fscn(rows, positions, None, slots, None, None, weight, eps, 1)


def test_cr1_constant_row_closed_form():
    for c in (1.0, -3.5, 1e-3):
        for eps in (0.0, 1e-6, 0.25):
            written, lat, _ = _cr1(np.full((1, L), c), eps=eps)
            assert written[0]
            c32 = float(np.float32(c))
            want = c32 / math.sqrt(c32 * c32 + float(np.float32(eps)))
            assert np.allclose(lat[0], want, rtol=1e-15, atol=0)


def test_cr1_weight_and_alternating_signs():
    a = 2.0
    row = np.where(np.arange(L) % 2 == 0, a, -a)
    w = _bf(np.linspace(0.5, 2.0, L))
    _, lat, mass = _cr1(row[None, :], eps=0.0, weight=w)
    wf = (w.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    assert np.allclose(lat[0], np.sign(row) * wf, rtol=1e-15, atol=0)
    assert np.allclose(mass[0], np.abs(wf), rtol=1e-15)


def test_cr1_gates():
    rows = np.ones((5, L), np.float32)
    written, lat, _ = _cr1(rows, slots=[0, -1, 3, 9, -5], positions=[0, 1, -1, 3, 4])
    assert list(written) == [True, False, False, True, False]
    assert np.all(lat[~written] == 0)


# ------------------------------------------------------------------ CR2

def _pair_call(kv0, s0, kv1, s1, eps=0.0, weight=ONE):
    """One request, two tokens at positions 0 and 1 of one chunk."""
    rows = np.zeros((2, 2 * L), np.float32)
    rows[0, :L], rows[0, L:] = kv0, s0
    rows[1, :L], rows[1, L:] = kv1, s1
    state = np.zeros((1, 2, 2 * L), np.float32)
    return fscn(rows, [0, 1], state, [0, 1], [0, 2], [0, 0], weight, eps, 2)


def test_cr2_equal_scores_average_the_rows():
    written, lat, _ = _pair_call(3.0, 0.7, 5.0, 0.7)
    assert list(written) == [False, True]
    assert np.allclose(lat[1], 1.0, rtol=1e-15)      # pooled 4 everywhere, normalised to 1
    rng = np.random.default_rng(1)
    a, b = rng.standard_normal(L), rng.standard_normal(L)
    _, lat, _ = _pair_call(a, 0.0, b, 0.0)
    m = (a.astype(np.float32).astype(np.float64) + b.astype(np.float32)) / 2
    assert np.allclose(lat[1], m / np.sqrt(np.mean(m * m)), rtol=1e-12)


def test_cr2_score_gap_sets_the_weights():
    """Gap ln 3 in favour of the first row: weights 3/4 and 1/4 (rows 4 and
    0 pool to 3); a gap of 1000 gives weight exactly 1 to the larger score,
    whichever row holds it."""
    s0 = np.float32(math.log(3.0))
    _, lat, _ = _pair_call(4.0, s0, 0.0, 0.0, eps=7.0)
    w = math.exp(float(s0)) / (math.exp(float(s0)) + 1.0)        # 3/4 up to fp32(ln 3)
    p = 4.0 * w
    assert np.allclose(lat[1], p / math.sqrt(p * p + 7.0), rtol=1e-12)
    rng = np.random.default_rng(2)
    a, b = rng.standard_normal(L).astype(np.float32), rng.standard_normal(L).astype(np.float32)
    _, lat_a, _ = _pair_call(a, 0.0, b, -1000.0)
    _, lat_b, _ = _pair_call(a, -1000.0, b, 0.0)
    ra = a.astype(np.float64) / np.sqrt(np.mean(a.astype(np.float64) ** 2))
    rb = b.astype(np.float64) / np.sqrt(np.mean(b.astype(np.float64) ** 2))
    assert np.allclose(lat_a[1], ra, rtol=1e-12) and np.allclose(lat_b[1], rb, rtol=1e-12)


def test_cr2_scores_are_per_channel():
    """Channel d of the score picks channel d of the rows: scores favouring
    row 0 on even channels and row 1 on odd ones."""
    kv0, kv1 = np.full(L, 2.0), np.full(L, -2.0)
    s0 = np.where(np.arange(L) % 2 == 0, 0.0, -1000.0)
    s1 = np.where(np.arange(L) % 2 == 0, -1000.0, 0.0)
    _, lat, _ = _pair_call(kv0, s0, kv1, s1)
    assert np.allclose(lat[1], np.where(np.arange(L) % 2 == 0, 1.0, -1.0), rtol=1e-15)


def _stream_model(seq_rows, start, ring_row, weight, eps):
    """Token-by-token model of the compressor for one request: remember the
    last row; at every odd position pool it with the current row (two-term
    softmax per channel, math.exp) and normalise. The row before `start`
    is ring_row. Pure Python loops: tiny cases only."""
    wf = [float(v) for v in (weight.astype(np.uint32) << 16).view(np.float32)]
    out = {}
    last = [float(v) for v in ring_row]
    for k, row in enumerate(seq_rows):
        p = start + k
        cur = [float(v) for v in row]
        if p % 2 == 1:
            pooled = []
            for d in range(L):
                a, b = last[L + d], cur[L + d]
                m = max(a, b)
                ea, eb = math.exp(a - m), math.exp(b - m)
                pooled.append((ea * last[d] + eb * cur[d]) / (ea + eb))
            ms = sum(v * v for v in pooled) / L
            r = 1.0 / math.sqrt(ms + eps)
            out[p] = [pooled[d] * r * wf[d] for d in range(L)]
        last = cur
    return out


def _requests(seed):
    """Three requests (start position, length); request 1 starts at an odd
    position, so its first group needs the ring row before it."""
    rng = np.random.default_rng(seed)
    spec = [(4, 9), (7, 6), (10, 7)]
    seqs = [rng.standard_normal((n, 2 * L)).astype(np.float32) for _, n in spec]
    ring0 = rng.standard_normal((3, 2 * L)).astype(np.float32)   # row before each start
    return spec, seqs, ring0


def _run_chunks(spec, seqs, ring0, cap, splits, weight, eps):
    """Feed the requests through the oracle in calls; call c takes the c-th
    piece of every request (pieces from `splits`), tokens packed request by
    request. Request k owns ring block k. Returns {(k, position): latent row}
    and the final ring."""
    state = np.full((3, cap, 2 * L), np.nan, np.float32)
    for k, (start, _) in enumerate(spec):
        state[k, (start - 1) % cap] = ring0[k]
    done = [0, 0, 0]
    out = {}
    for c in range(max(len(s) for s in splits)):
        rows, pos, slots, qsl, t2r, owner = [], [], [], [0], [], []
        for k, (start, _) in enumerate(spec):
            n = splits[k][c] if c < len(splits[k]) else 0
            for i in range(done[k], done[k] + n):
                p = start + i
                rows.append(seqs[k][i])
                pos.append(p)
                slots.append(k * cap + p % cap)
                t2r.append(k)
                owner.append((k, p))
            done[k] += n
            qsl.append(len(rows))
        if not rows:
            continue
        written, lat, _ = fscn(np.array(rows), np.array(pos), state, np.array(slots),
                               np.array(qsl), np.array(t2r), weight, eps, 2)
        for i in np.nonzero(written)[0]:
            out[owner[i]] = lat[i]
    return out, state


def test_cr2_equals_streaming_model_and_is_invariant_to_chunking():
    spec, seqs, ring0 = _requests(3)
    w = _bf(np.random.default_rng(4).uniform(0.5, 1.5, L))
    eps = float(np.float32(1e-6))
    whole, ring_whole = _run_chunks(spec, seqs, ring0, 2, [[9], [6], [7]], w, eps)
    pieces, ring_pieces = _run_chunks(spec, seqs, ring0, 2, [[4, 5], [1, 2, 3], [2, 1, 4]], w,
                                      eps)
    assert whole.keys() == pieces.keys()
    for key in whole:
        assert np.array_equal(whole[key], pieces[key]), key
    assert np.array_equal(ring_whole, ring_pieces)
    for k, (start, n) in enumerate(spec):
        model = _stream_model(seqs[k], start, ring0[k], w, eps)
        got = {p: v for (kk, p), v in whole.items() if kk == k}
        assert sorted(got) == sorted(model)
        for p in model:
            assert np.allclose(got[p], model[p], rtol=1e-12, atol=1e-14), (k, p)


def test_cr2_capacity_four_and_chunk_tails():
    """capacity 4: a piece shorter than the capacity keeps older rows of
    the ring; the result still matches the streaming model."""
    spec, seqs, ring0 = _requests(5)
    eps = 0.5
    got, ring = _run_chunks(spec, seqs, ring0, 4, [[1, 1, 1, 6], [3, 3], [5, 1, 1]], ONE, eps)
    for k, (start, n) in enumerate(spec):
        model = _stream_model(seqs[k], start, ring0[k], ONE, eps)
        for p in model:
            assert np.allclose(got[(k, p)], model[p], rtol=1e-12, atol=1e-14)
        # the ring holds the request's last min(4, n) rows at p % 4
        for i in range(max(0, n - 4), n):
            assert np.array_equal(ring[k, (start + i) % 4], seqs[k][i])


def test_ring_save_takes_only_the_last_capacity_rows_and_skips_with_prev_rows():
    rng = np.random.default_rng(6)
    rows = rng.standard_normal((5, 2 * L)).astype(np.float32)
    pos = np.arange(10, 15)
    cap = 2
    state = np.full((1, cap, 2 * L), 9.0, np.float32)
    slots = np.array([p % cap for p in pos])
    fscn(rows, pos, state, slots, [0, 5], [0] * 5, ONE, 0.0, 2)
    assert np.array_equal(state[0, 14 % 2], rows[4]) and np.array_equal(state[0, 13 % 2], rows[3])
    state2 = np.full((1, cap, 2 * L), 9.0, np.float32)
    prev = rng.standard_normal((2, 2 * L)).astype(np.float32)
    fscn(rows, pos, state2, slots, [0, 5], [0] * 5, ONE, 0.0, 2, prev_rows=prev,
         prev_row_indices=np.array([1]))
    assert np.all(state2 == 9.0)


@pytest.mark.parametrize("idx", [1, -1, 5])
def test_prev_rows_select_the_predecessor(idx):
    """A chunk starting at an odd position: prev_rows[idx] is its first
    group's predecessor; -1 reads the ring row; an index past the rows skips
    the group."""
    rng = np.random.default_rng(7)
    rows = rng.standard_normal((2, 2 * L)).astype(np.float32)
    prev = rng.standard_normal((3, 2 * L)).astype(np.float32)
    ring = rng.standard_normal((1, 2, 2 * L)).astype(np.float32)
    state = ring.copy()
    written, lat, _ = fscn(rows, [5, 6], state, [5 % 2, 6 % 2], [0, 2], [0, 0], ONE, 0.0, 2,
                           prev_rows=prev, prev_row_indices=np.array([idx]))
    if idx >= 3:
        assert not written.any()
        return
    pred = prev[idx] if idx >= 0 else ring[0, 4 % 2]
    model = _stream_model(rows[:1], 5, pred, ONE, 0.0)
    assert list(written) == [True, False]
    assert np.allclose(lat[0], model[5], rtol=1e-12, atol=1e-14)


def test_cr2_gates_and_inconsistent_requests():
    rng = np.random.default_rng(8)
    rows = rng.standard_normal((6, 2 * L)).astype(np.float32)
    pos = np.array([1, 2, 3, 4, 5, -1])
    state = np.zeros((2, 2, 2 * L), np.float32)
    # token 0: slot -1; token 2: request index out of range; token 4: outside
    # its request's chunk; token 5: negative position
    slots = np.array([-1, 2 % 2, 3 % 2, 4 % 2, 5 % 2, 1])
    t2r = np.array([0, 0, 7, 0, 1, 0])
    written, _, _ = fscn(rows, pos, state, slots, [0, 4, 4], t2r, ONE, 0.0, 2)
    assert not written.any()
    slots_oob = np.array([0, 1, 4, 1, 0, 1])           # 4 = blocks * capacity: outside the ring
    written, _, _ = fscn(rows[:4], pos[:4], state, slots_oob[:4], [0, 4], [0] * 4, ONE, 0.0, 2)
    assert list(written) == [True, False, False, False]


def test_cr2_chunk_bounds_are_cut_to_the_batch():
    """A chunk given as [-3, 9) over a 4-token batch is the chunk [0, 4):
    same rows written, same latent, same ring."""
    rng = np.random.default_rng(9)
    rows = rng.standard_normal((4, 2 * L)).astype(np.float32)
    pos = np.array([3, 4, 5, 6])
    ring0 = rng.standard_normal((1, 2, 2 * L)).astype(np.float32)
    out = []
    for qsl in ([0, 4], [-3, 4], [0, 9], [-3, 9]):
        state = ring0.copy()
        written, lat, _ = fscn(rows, pos, state, pos % 2, qsl, [0] * 4, ONE, 1e-6, 2)
        out.append((written, lat, state))
    assert list(out[0][0]) == [True, False, True, False]
    # the last two tokens (positions 5 and 6) land in ring rows 1 and 0
    assert np.array_equal(out[0][2][0, 1], rows[2]) and np.array_equal(out[0][2][0, 0], rows[3])
    for written, lat, state in out[1:]:
        assert np.array_equal(written, out[0][0])
        assert np.array_equal(lat, out[0][1])
        assert np.array_equal(state, out[0][2])
