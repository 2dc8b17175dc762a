"""CPU oracle for fused_save_compress_norm: pool each closed group of
compressor rows into an RMS-normalised bf16 latent, and save ring rows.

TEST INFRASTRUCTURE ONLY (see the package docstring): the tests and the
benchmark's CPU leg use it; the product never imports it.

Follows "vllm.models.deepseek_v41.common.ops.fused_compress_quant_cache"
(fused_save_compress_norm: docstring and Args). What the page fixes: fp32
[kv | score] rows (512 kv values, then 512 scores; CR1 rows hold kv only);
groups of compress_ratio R in {1, 2} consecutive positions, closed at
positions p with (p + 1) % R == 0; a bf16 [512] RMSNorm weight and an fp32
epsilon; a bf16 latent written only at valid group boundaries; for R = 2 a
ring of fp32 rows per request, position p in row p % capacity of the
request's block, slot_mapping = block * capacity + p % capacity; a chunk's
first token closes its group with the predecessor's ring row, or with
prev_rows[prev_row_indices[req]] when that index is set (-1 reads the ring);
then the chunk's last ``capacity`` rows are stored to the ring, unless
prev_rows is given (the ring is then left to save_ring_rows). For R = 1
there is no ring and slot_mapping only marks valid tokens.

Readings where the page is silent (the kernel itself is not printed):
  * pooling: per channel d, the group's scores go through a softmax over the
    group's rows and weight its kv values:
        w_i[d] = exp(s_i[d] - max_j s_j[d]) / sum_j exp(s_j[d] - max_j s_j[d])
        pooled[d] = sum_i w_i[d] * kv_i[d]
    (for R = 1 pooled = kv);
  * RMSNorm of the pooled row: y[d] = pooled[d] * w[d] / sqrt(mean_d pooled^2 + eps);
  * the latent row written is the closing token's row; a token is valid when
    its slot is >= 0 (and, for R = 2, its ring slot lies inside the state)
    and its position is >= 0; a token whose request index or chunk range is
    inconsistent is skipped, as is a prev_rows index past the rows given;
  * a request's chunk is query_start_loc[k] .. query_start_loc[k + 1] cut to
    the batch's rows [0, T): a start below 0 reads as 0, an end past T as T;
  * the ring rows saved are bit copies of the tokens' 1024 floats.

Written out here in float64 (the exact value of the definition before the
final bf16 rounding). ``mass[t, d] = r * |w[d]| * sum_i w_i[d] |kv_i[d]|`` is
returned with it as the scale of the rounding error an fp32 kernel can make.
"""
import numpy as np

LATENT = 512


def _bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(
        np.float64)


def fused_save_compress_norm(kv_score: np.ndarray, positions: np.ndarray, state,
                             slot_mapping: np.ndarray, query_start_loc, token_to_req,
                             weight_bits: np.ndarray, eps: float, compress_ratio: int,
                             prev_rows=None, prev_row_indices=None):
    """kv_score: float32 [>= T, 512 * R]; state: float32 [blocks, capacity,
    >= 1024] (R = 2; modified in place by the ring save); T =
    len(slot_mapping). Returns (written bool [T], latent float64 [T, 512],
    mass float64 [T, 512]); rows not written are 0."""
    R = int(compress_ratio)
    assert R in (1, 2)
    slot = np.asarray(slot_mapping, np.int64)
    T = slot.size
    pos = np.asarray(positions, np.int64)[:T]
    kv_score = np.asarray(kv_score, np.float32)
    assert kv_score.shape[1] == LATENT * R
    rows = kv_score[:T].astype(np.float64)
    eps = float(np.float32(eps))
    w = _bf16_to_f64(weight_bits)

    written = (slot >= 0) & (pos >= 0) & ((pos + 1) % R == 0)
    pooled = np.zeros((T, LATENT))
    pool_mass = np.zeros((T, LATENT))
    if R == 1:
        pooled[written] = rows[written]
        pool_mass[written] = np.abs(rows[written])
    else:
        blocks, cap = state.shape[0], state.shape[1]
        qsl = np.asarray(query_start_loc, np.int64)
        num_reqs = qsl.size - 1
        req = np.asarray(token_to_req, np.int64)[:T]
        t = np.arange(T)
        req_ok = (req >= 0) & (req < num_reqs)
        r_safe = np.where(req_ok, req, 0)
        qs_t = np.maximum(qsl[r_safe], 0)
        in_chunk = req_ok & (qs_t <= t) & (t < qsl[r_safe + 1])
        written &= in_chunk & (slot < blocks * cap)
        first = t == qs_t
        # the predecessor row of each written token's group
        pred = np.full((T, 2 * LATENT), np.nan)
        inner = written & ~first
        pred[inner] = kv_score[np.nonzero(inner)[0] - 1].astype(np.float64)
        for i in np.nonzero(written & first)[0]:
            k = int(req[i])
            if prev_rows is not None and int(prev_row_indices[k]) >= 0:
                j = int(prev_row_indices[k])
                if j >= prev_rows.shape[0]:
                    written[i] = False
                    continue
                pred[i] = prev_rows[j, :2 * LATENT].astype(np.float64)
            else:
                s = int(slot[i])
                pred[i] = state[s // cap, (int(pos[i]) - 1) % cap, :2 * LATENT].astype(np.float64)
        kv0, s0 = pred[:, :LATENT], pred[:, LATENT:]
        kv1, s1 = rows[:, :LATENT], rows[:, LATENT:]
        with np.errstate(invalid="ignore", over="ignore"):
            m = np.maximum(s0, s1)
            e0, e1 = np.exp(s0 - m), np.exp(s1 - m)
            w0, w1 = e0 / (e0 + e1), e1 / (e0 + e1)
            pooled[written] = (w0 * kv0 + w1 * kv1)[written]
            pool_mass[written] = (w0 * np.abs(kv0) + w1 * np.abs(kv1))[written]

    with np.errstate(invalid="ignore", divide="ignore", over="ignore"):
        r = 1.0 / np.sqrt(np.mean(pooled * pooled, axis=1) + eps)
        latent = pooled * r[:, None] * w[None, :]
        mass = pool_mass * r[:, None] * np.abs(w)[None, :]
    latent[~written] = 0.0
    mass[~written] = 0.0

    if R == 2 and prev_rows is None:
        for k in range(num_reqs):
            qs, qe = max(int(qsl[k]), 0), min(int(qsl[k + 1]), T)
            for i in range(max(qs, qe - cap), qe):
                s = int(slot[i])
                if 0 <= s < blocks * cap:
                    state[s // cap, s % cap, :2 * LATENT] = kv_score[i, :2 * LATENT]
    return written, latent, mass
