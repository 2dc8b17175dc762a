"""Seeded synthetic inputs for the paged KV-cache store, the V4.1 inserts and
the gather read path.

This module holds none of the quantization arithmetic. It draws random
numbers (numpy PCG64), rounds the drawn fp32 values to bf16 (input
preparation), builds slot maps, positions, the rotary cos/sin table and
poison fills, and says how big each buffer is. Both the CUDA path and the CPU
oracle are fed from these arrays, so they see identical bytes.

Large arrays are drawn in fixed-size row chunks, each from its own child of
``SeedSequence(seed)``, so the bytes do not depend on how many threads drew
them.

Workloads (sizes of the published configurations; ``scaled`` variants keep
the recipe and shrink the counts for fast tests):
  store_small   64 tokens, contiguous 128-slot cache, injected edge groups
  store_paged   16,384 tokens, 2048 blocks x 64 slots, block stride 192 rows
  store_large   4,300,000 tokens, source row stride 576, 8,388,608 slots
  rope_insert   65,536 tokens (or 4,194,304 for the large variant), R = 4;
                records mxfp8 / nvfp4 / v4, or plain bf16 / fp8 rows
  ring_rows     fp32 [kv | score] rows of 1024 values into a paged ring state
  compress      fused_save_compress_norm batches: packed request chunks of
                fp32 [kv | score] rows (R = 2) or kv rows (R = 1)
  gather        1,048,576-slot packed cache, 128 queries x 2048 indices
  sparse_attention  the gather's cache and indices + 128 heads of bf16 queries
"""
import math
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

LATENT = 512
ROW_BYTES_MXFP4 = 272          # 512/2 code bytes + 512/32 scale bytes
RECORD_BYTES_MXFP8 = 528       # 512 value bytes + 16 scale bytes
RECORD_BYTES_NVFP4 = 288       # 256 code bytes + 32 scale bytes
RECORD_BYTES_V4 = 584          # 576 value bytes + 8 scale bytes
PLAIN_FP8_SCALE = 0.0125       # per-tensor scale of the plain fp8 rows (not a power of two)
RING_ROW = 1024                # fp32 values per compressor row ([kv | score])
RING_POISON_BITS = 0x7FBADBAD  # fill of the ring state before a save (a NaN pattern)
POISON = 0xAA                  # fill of this layer's cache rows before a store
OTHER_LAYER_POISON = 0x5A      # fill of interleaved pages of other layers
BF16_MAX_BITS = 0x7F7F         # fill of source columns past the latent
BF16_QNAN_BITS = 0x7FC0
CHUNK_ROWS = 16384


def _threads() -> int:
    return max(1, min(32, len(os.sched_getaffinity(0))))


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (nearest even) and return the uint16 bit patterns.
    Inputs here are finite draws; NaN is injected later as explicit bits."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32)
    t = u >> 16
    t &= 1
    t += 0x7FFF
    t += u
    t >>= 16
    return t.astype(np.uint16)


def _draw_rows(seed: int, num_rows: int, width: int, fill, out: np.ndarray,
               col0: int = 0, tag: int = 0) -> None:
    """Fill out[:, col0:col0+width] (uint16) chunk by chunk; ``fill(rng, n)``
    returns n fp32 values. Chunks draw from independent child seeds."""
    n_chunks = max(1, math.ceil(num_rows / CHUNK_ROWS))
    children = np.random.SeedSequence([seed, tag]).spawn(n_chunks)

    def one(c):
        lo = c * CHUNK_ROWS
        hi = min(num_rows, lo + CHUNK_ROWS)
        rng = np.random.default_rng(children[c])
        vals = fill(rng, (hi - lo) * width).reshape(hi - lo, width)
        out[lo:hi, col0:col0 + width] = f32_to_bf16_bits(vals)

    if n_chunks == 1:
        one(0)
    else:
        with ThreadPoolExecutor(_threads()) as ex:
            list(ex.map(one, range(n_chunks)))


def _normal(rng, n):
    return rng.standard_normal(n, dtype=np.float32)


def _student_t_outliers(rng, n):
    """Student-t(nu=4) x 0.5, with 0.1% of the elements multiplied by 64."""
    x = (rng.standard_t(4, n) * 0.5).astype(np.float32)
    k = max(1, n // 1000)
    x[rng.choice(n, k, replace=False)] *= 64.0
    return x


def _slots_with_pads(rng, num_slots: int, num_tokens: int, pad_count: int) -> np.ndarray:
    slots = rng.choice(num_slots, num_tokens, replace=False).astype(np.int64)
    if pad_count:
        slots[rng.choice(num_tokens, pad_count, replace=False)] = -1
    return slots


# ------------------------------------------------------------ store_small ---

E2M1_MIDPOINTS = (0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0)


def store_small(seed: int = 0) -> dict:
    """64 tokens of N(0,1) x 2**U(-4,4) (per token), with injected groups:
    one all-zero group, groups whose amax is exactly 6 * 2**k, and groups whose
    members sit exactly on E2M1 midpoints times 2**k. Contiguous cache of 128
    slots pre-filled with 0xAA; 64 distinct random slots, 8 of them -1."""
    rng = np.random.default_rng(seed)
    T = 64
    x = rng.standard_normal((T, LATENT))
    x *= np.exp2(rng.uniform(-4.0, 4.0, size=T))[:, None]
    g = 32
    # all-zero group (+0.0)
    x[0, 3 * g:4 * g] = 0.0
    # groups with amax exactly +-6 * 2**k, others strictly inside
    for i, (t, grp) in enumerate([(1, 0), (2, 5), (3, 15), (4, 7), (5, 9), (6, 11)]):
        k = int(rng.integers(-8, 9))
        vals = rng.uniform(-0.99, 0.99, size=g) * 6.0 * 2.0 ** k
        vals[int(rng.integers(0, g))] = (-1.0 if i % 2 else 1.0) * 6.0 * 2.0 ** k
        x[t, grp * g:(grp + 1) * g] = vals
    # groups on exact midpoints: amax 6 * 2**k pins the scale at 2**k
    mids = np.array(E2M1_MIDPOINTS + (0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0))
    for t, grp in [(7, 1), (8, 2), (9, 4), (10, 6), (11, 8), (12, 14)]:
        k = int(rng.integers(-6, 7))
        vals = np.concatenate([mids, -mids, [0.25, -0.25, 0.125, -0.125]])[:g] * 2.0 ** k
        vals[0] = 6.0 * 2.0 ** k
        x[t, grp * g:(grp + 1) * g] = rng.permutation(vals)
    latent = f32_to_bf16_bits(x.astype(np.float32))
    slots = _slots_with_pads(rng, 128, T, 8)
    cache = np.full(128 * ROW_BYTES_MXFP4, POISON, dtype=np.uint8)
    return dict(latent=latent, slot_mapping=slots, cache=cache, num_blocks=1, block_size=128,
                block_stride_rows=128, cache_offset=0)


# ------------------------------------------------------------ store_paged ---

def store_paged(seed: int = 0, num_tokens: int = 16384, num_blocks: int = 2048,
                block_size: int = 64, block_stride_rows: int = 192, layer_row_offset: int = 64,
                pad_fraction: float = 0.05) -> dict:
    """Student-t(4) x 0.5 latent with 0.1% outliers x 64. The buffer holds
    num_blocks groups of block_stride_rows rows; this layer's block b is rows
    [b*stride + offset, b*stride + offset + block_size), the rows around it
    belong to other layers and carry a different poison."""
    rng = np.random.default_rng(seed)
    latent = np.empty((num_tokens, LATENT), dtype=np.uint16)
    _draw_rows(seed, num_tokens, LATENT, _student_t_outliers, latent, tag=2)
    num_slots = num_blocks * block_size
    slots = _slots_with_pads(rng, num_slots, num_tokens, int(round(pad_fraction * num_tokens)))
    rows = num_blocks * block_stride_rows
    cache = np.full((rows, ROW_BYTES_MXFP4), OTHER_LAYER_POISON, dtype=np.uint8)
    mine = (np.arange(num_blocks)[:, None] * block_stride_rows + layer_row_offset
            + np.arange(block_size)[None, :]).reshape(-1)
    cache[mine] = POISON
    return dict(latent=latent, slot_mapping=slots, cache=cache.reshape(-1), num_blocks=num_blocks,
                block_size=block_size, block_stride_rows=block_stride_rows,
                cache_offset=layer_row_offset * ROW_BYTES_MXFP4)


# ------------------------------------------------------------ store_large ---

def store_large_slots(seed: int = 0, num_tokens: int = 4_300_000, num_slots: int = 8_388_608,
                      pad_fraction: float = 0.01) -> np.ndarray:
    rng = np.random.default_rng(seed)
    return _slots_with_pads(rng, num_slots, num_tokens, int(round(pad_fraction * num_tokens)))


def store_large_latent(seed: int = 0, num_tokens: int = 4_300_000, row_stride: int = 576,
                       out: np.ndarray = None) -> np.ndarray:
    """[num_tokens, row_stride] uint16: N(0,1) bf16 in the first 512 columns,
    bf16 max in the rest (to show any read past the latent)."""
    if out is None:
        out = np.empty((num_tokens, row_stride), dtype=np.uint16)
    if row_stride > LATENT:
        out[:, LATENT:] = BF16_MAX_BITS
    _draw_rows(seed, num_tokens, LATENT, _normal, out, tag=3)
    return out


def store_large(seed: int = 0, num_tokens: int = 4_300_000, row_stride: int = 576,
                num_slots: int = 8_388_608, pad_fraction: float = 0.01,
                with_cache: bool = True) -> dict:
    latent = store_large_latent(seed, num_tokens, row_stride)
    slots = store_large_slots(seed, num_tokens, num_slots, pad_fraction)
    d = dict(latent=latent[:, :LATENT], latent_full=latent, slot_mapping=slots,
             num_blocks=1, block_size=num_slots, block_stride_rows=num_slots, cache_offset=0,
             num_slots=num_slots)
    if with_cache:
        d["cache"] = np.full(num_slots * ROW_BYTES_MXFP4, POISON, dtype=np.uint8)
    return d


# ------------------------------------------------------------ rope_insert ---

def rope_cos_sin_table(rows: int = 131072, rotary_dim: int = 64, base: float = 10000.0):
    """fp32 [rows, rotary_dim]: cos(p * base**(-2i/rotary_dim)) for i < rotary_dim/2,
    then the matching sines, evaluated in fp64 and rounded to fp32."""
    half = rotary_dim // 2
    inv_freq = base ** (-np.arange(half, dtype=np.float64) * 2.0 / rotary_dim)
    ang = np.arange(rows, dtype=np.float64)[:, None] * inv_freq[None, :]
    return np.concatenate([np.cos(ang), np.sin(ang)], axis=1).astype(np.float32)


def rope_insert(seed: int = 0, num_tokens: int = 65536, num_pages: int = 1024,
                cache_block: int = 64, nan_fraction: float = 0.0005, table_rows: int = 131072,
                compress_ratio: int = 4, record: str = "mxfp8", pad_count: int = 0) -> dict:
    """N(0,1) bf16 latent with ``nan_fraction`` of the elements set to NaN
    (0x7FC0); positions uniform in [0, table_rows); slots a random injection
    into num_pages * cache_block slots (a permutation when the counts match);
    optionally ``pad_count`` slots set to -1. Cache pre-filled with 0xAA."""
    rng = np.random.default_rng(seed)
    latent = np.empty((num_tokens, LATENT), dtype=np.uint16)
    _draw_rows(seed, num_tokens, LATENT, _normal, latent, tag=4)
    n_nan = int(round(nan_fraction * num_tokens * LATENT))
    if n_nan:
        flat = latent.reshape(-1)
        flat[rng.choice(flat.size, n_nan, replace=False)] = BF16_QNAN_BITS
    positions = rng.integers(0, table_rows, size=num_tokens, dtype=np.int64)
    num_slots = num_pages * cache_block
    slots = _slots_with_pads(rng, num_slots, num_tokens, pad_count)
    if record in ("bf16", "fp8"):
        # plain [pages, cache_block, 512] rows; strides in elements
        esize = 2 if record == "bf16" else 1
        page_elems = cache_block * LATENT
        cache = np.full(num_pages * page_elems * esize, POISON, dtype=np.uint8)
        return dict(latent=latent, positions=positions, cos_sin=rope_cos_sin_table(table_rows),
                    cache=cache, cache_slots=slots, num_pages=num_pages,
                    cache_block=cache_block, page_stride_elems=page_elems,
                    slot_stride_elems=LATENT, compress_ratio=compress_ratio, record=record,
                    fp8=record == "fp8", fp8_scale=PLAIN_FP8_SCALE)
    record_bytes = {"mxfp8": RECORD_BYTES_MXFP8, "nvfp4": RECORD_BYTES_NVFP4,
                    "v4": RECORD_BYTES_V4}[record]
    page_stride = cache_block * record_bytes
    cache = np.full(num_pages * page_stride, POISON, dtype=np.uint8)
    return dict(latent=latent, positions=positions, cos_sin=rope_cos_sin_table(table_rows),
                cache=cache, cache_slots=slots, num_pages=num_pages, cache_block=cache_block,
                page_stride_bytes=page_stride, compress_ratio=compress_ratio, record=record)


# -------------------------------------------------------------- ring_rows ---

def ring_rows(seed: int = 0, num_rows: int = 65536, num_blocks: int = 512,
              state_block: int = 128, pad_fraction: float = 0.05) -> dict:
    """fp32 rows [num_rows, 1024] ~N(0,1) (the [kv | score] halves drawn
    alike); slots a random injection into num_blocks * state_block ring rows
    with ``pad_fraction`` set to -1; the state [num_blocks, state_block, 1024]
    filled with the RING_POISON_BITS pattern."""
    rng = np.random.default_rng([seed, 7])
    rows = np.empty((num_rows, RING_ROW), dtype=np.float32)
    n_chunks = max(1, math.ceil(num_rows / CHUNK_ROWS))
    children = np.random.SeedSequence([seed, 8]).spawn(n_chunks)

    def one(c):
        lo, hi = c * CHUNK_ROWS, min(num_rows, (c + 1) * CHUNK_ROWS)
        rows[lo:hi] = np.random.default_rng(children[c]).standard_normal(
            (hi - lo, RING_ROW), dtype=np.float32)

    with ThreadPoolExecutor(_threads()) as ex:
        list(ex.map(one, range(n_chunks)))
    slots = _slots_with_pads(rng, num_blocks * state_block, num_rows,
                             int(round(pad_fraction * num_rows)))
    state = np.empty((num_blocks, state_block, RING_ROW), dtype=np.float32)
    state.view(np.uint32)[...] = RING_POISON_BITS
    return dict(rows=rows, slot_mapping=slots, state=state, num_blocks=num_blocks,
                state_block=state_block)


# ----------------------------------------------------------------- gather ---

def gather(seed: int = 0, num_slots: int = 1_048_576, num_queries: int = 128, topk: int = 2048,
           max_pad: int = 64) -> dict:
    """Rows to fill every slot of a packed cache (Student-t(4) x 0.5 with 0.1%
    outliers x 64, slot i <- row i), and per query ``topk`` distinct random slot
    indices whose last U{0..max_pad} entries are -1 pads."""
    rng = np.random.default_rng(seed)
    fill_latent = np.empty((num_slots, LATENT), dtype=np.uint16)
    _draw_rows(seed, num_slots, LATENT, _student_t_outliers, fill_latent, tag=5)
    fill_slots = np.arange(num_slots, dtype=np.int64)
    idx = np.empty((num_queries, topk), dtype=np.int64)
    for q in range(num_queries):
        idx[q] = rng.choice(num_slots, topk, replace=False)
        p = int(rng.integers(0, max_pad + 1))
        if p:
            idx[q, topk - p:] = -1
    return dict(fill_latent=fill_latent, fill_slots=fill_slots, indices=idx, num_blocks=1,
                block_size=num_slots, block_stride_rows=num_slots, num_slots=num_slots)


# ------------------------------------------------------- sparse attention ---

def attention_queries(seed: int = 0, num_queries: int = 128, num_heads: int = 128) -> np.ndarray:
    """Decode queries: bf16 N(0, 1) [num_queries, num_heads, 512] (absorbed
    NoPE queries in the latent space)."""
    q = np.empty((num_queries * num_heads, LATENT), dtype=np.uint16)
    _draw_rows(seed, num_queries * num_heads, LATENT, _normal, q, tag=7)
    return q.reshape(num_queries, num_heads, LATENT)


def sparse_attention(seed: int = 0, num_queries: int = 128, num_heads: int = 128,
                     topk: int = 2048, num_slots: int = 1_048_576, max_pad: int = 64) -> dict:
    """The gather workload's cache fill and top-k indices, plus the decode
    queries of attention_queries, and sm_scale = 1/sqrt(512)."""
    d = gather(seed, num_slots, num_queries, topk, max_pad)
    d["q"] = attention_queries(seed, num_queries, num_heads)
    d["sm_scale"] = 1.0 / math.sqrt(LATENT)
    return d


# --------------------------------------------------------------- compress ---

def compress(seed: int = 0, compress_ratio: int = 2, num_reqs: int = 256, max_chunk: int = 511,
             decode_fraction: float = 0.25, capacity: int = 4, pad_tokens: int = 16,
             prev_rows: bool = False) -> dict:
    """A packed batch for fused_save_compress_norm. Each request's chunk has
    length 1 with probability ``decode_fraction``, else U{2..max_chunk}, and
    starts at a position U[0, 100000) (either parity); its tokens are
    consecutive positions, packed request after request, then ``pad_tokens``
    padding tokens (slot -1). Rows: kv ~N(0,1), scores ~N(0,1) x 2 (fp32).
    R = 2: request k owns ring block perm[k] of num_reqs + 8 blocks of
    ``capacity`` rows, slot = block * capacity + p % capacity; the ring holds
    N(0,1) rows (the predecessors of chunks that start at odd positions).
    R = 1: slots are distinct random values in [0, 2T), 5% of them -1.
    prev_rows (R = 2): [num_reqs, 1024] N(0,1) rows, prev_row_indices a
    permutation with a quarter of the entries -1. Weight bf16 U(0.5, 1.5),
    eps 1e-6."""
    rng = np.random.default_rng([seed, 11, compress_ratio])
    lens = np.where(rng.random(num_reqs) < decode_fraction, 1,
                    rng.integers(2, max_chunk + 1, size=num_reqs))
    starts = rng.integers(0, 100_000, size=num_reqs)
    qsl = np.zeros(num_reqs + 1, np.int64)
    qsl[1:] = np.cumsum(lens)
    n_real = int(qsl[-1])
    T = n_real + pad_tokens
    t2r = np.zeros(T, np.int64)
    t2r[:n_real] = np.repeat(np.arange(num_reqs), lens)
    positions = np.zeros(T, np.int64)
    positions[:n_real] = starts[t2r[:n_real]] + (np.arange(n_real) - qsl[t2r[:n_real]])
    width = LATENT * compress_ratio
    rows = np.empty((T, width), np.float32)
    n_chunks = max(1, math.ceil(T / CHUNK_ROWS))
    children = np.random.SeedSequence([seed, 12, compress_ratio]).spawn(n_chunks)

    def one(c):
        lo, hi = c * CHUNK_ROWS, min(T, (c + 1) * CHUNK_ROWS)
        g = np.random.default_rng(children[c])
        rows[lo:hi] = g.standard_normal((hi - lo, width), dtype=np.float32)
        if compress_ratio == 2:
            rows[lo:hi, LATENT:] *= 2.0

    with ThreadPoolExecutor(_threads()) as ex:
        list(ex.map(one, range(n_chunks)))
    weight = f32_to_bf16_bits(rng.uniform(0.5, 1.5, LATENT).astype(np.float32))
    out = dict(kv_score=rows, positions=positions, query_start_loc=qsl, token_to_req=t2r,
               weight=weight, eps=1e-6, compress_ratio=compress_ratio, num_reqs=num_reqs,
               num_real=n_real)
    if compress_ratio == 1:
        slots = _slots_with_pads(rng, 2 * T, T, int(round(0.05 * T)))
        slots[n_real:] = -1
        out.update(slot_mapping=slots, state=None)
        return out
    blocks = rng.permutation(num_reqs + 8)[:num_reqs]
    slots = np.full(T, -1, np.int64)
    slots[:n_real] = blocks[t2r[:n_real]] * capacity + positions[:n_real] % capacity
    state = rng.standard_normal((num_reqs + 8, capacity, 2 * LATENT), dtype=np.float32)
    out.update(slot_mapping=slots, state=state, capacity=capacity)
    if prev_rows:
        idx = rng.permutation(num_reqs).astype(np.int64)
        idx[rng.random(num_reqs) < 0.25] = -1
        out.update(prev_rows=rng.standard_normal((num_reqs, 2 * LATENT), dtype=np.float32),
                   prev_row_indices=idx)
    return out
