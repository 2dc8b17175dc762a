"""CPU oracle for sparse MLA attention over the packed MXFP4 cache.

TEST INFRASTRUCTURE ONLY (see the package docstring): the tests and the
benchmark's CPU leg use it; the product never imports it.

PR 60321 "Add an mxfp4_mla KV cache dtype..." (Read path; Claims): the ragged
sparse-attention kernel gathers each query's top-k rows, unpacks them to bf16
and feeds both dots (scores = q.k, output = softmax(scores).v); attention over
the packed cache equals attention over the same dequantized values stored as
bf16. For the rope-free (NoPE) latent the key and the value of a token are
the same 512-wide row.

This module writes that definition out in float64: the rows come from the
oracle's gather-and-dequantize (exact bf16 values), then

    s_j = sm_scale * sum_d q[h, d] * k_j[d]         over the valid indices j
    p_j = exp(s_j - max s),  l = sum p_j
    out[h, d] = sum_j p_j k_j[d] / l,   lse[h] = max s + log l

An index that is negative (padding) or not below num_slots is not part of the
softmax. A query with no valid index gets out = 0 and lse = -inf (the pages do
not say; this is the reading). ``mass[h, d] = sum_j p_j |k_j[d]| / l`` is
returned alongside as the scale of the rounding error a finite-precision
kernel can make on out[h, d].
"""
import numpy as np

from . import mxfp4_mla_gather_dequant

LATENT = 512


def _bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def mxfp4_mla_sparse_attention(q: np.ndarray, cache: np.ndarray, num_blocks: int,
                               block_size: int, block_stride_rows: int, indices: np.ndarray,
                               sm_scale: float, cache_offset: int = 0):
    """q: uint16 bf16 bits [num_queries, num_heads, 512]; indices: int64
    [num_queries, topk]. Returns (out, lse, mass) in float64:
    [num_queries, num_heads, 512], [num_queries, num_heads], like out."""
    assert q.dtype == np.uint16 and q.ndim == 3 and q.shape[2] == LATENT
    idx = np.ascontiguousarray(indices, dtype=np.int64)
    assert idx.ndim == 2 and idx.shape[0] == q.shape[0]
    nq, nh, _ = q.shape
    num_slots = num_blocks * block_size
    out = np.zeros((nq, nh, LATENT))
    mass = np.zeros((nq, nh, LATENT))
    lse = np.full((nq, nh), -np.inf)
    for n in range(nq):
        valid = idx[n][(idx[n] >= 0) & (idx[n] < num_slots)]
        if valid.size == 0:
            continue
        rows = mxfp4_mla_gather_dequant(cache, num_blocks, block_size, block_stride_rows, valid,
                                        latent_dim=LATENT, cache_offset=cache_offset)
        k = _bf16_to_f64(rows)                                   # [nv, 512], exact
        s = float(sm_scale) * (_bf16_to_f64(q[n]) @ k.T)         # [nh, nv]
        m = s.max(axis=1, keepdims=True)
        p = np.exp(s - m)
        l = p.sum(axis=1, keepdims=True)
        out[n] = (p @ k) / l
        mass[n] = (p @ np.abs(k)) / l
        lse[n] = m[:, 0] + np.log(l[:, 0])
    return out, lse, mass
