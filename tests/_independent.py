"""Independent references used only to pin the oracle.

Each routine here reaches the formats by a different method from the oracle:
nearest-value search over a decoded code table instead of threshold counting,
exponents from float64 frexp or exact comparisons instead of binary32 bit
fields, decoders built from the OCP bit-field definitions. A mistake in the
oracle's arithmetic (a wrong tie direction, a dropped sign, a transposed
nibble, an off-by-one exponent) therefore shows up as a disagreement.
"""
import numpy as np

E2M1_MAGNITUDES = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], dtype=np.float64)


def bf16_bits_to_f32(bits) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint32) << 16).view(np.float32)


def e2m1_decode_from_bits(code: int) -> float:
    """OCP E2M1: sign bit 3, exponent bits 2..1 (bias 1), mantissa bit 0."""
    s = -1.0 if code & 8 else 1.0
    e = (code >> 1) & 3
    m = code & 1
    mag = 0.5 * m if e == 0 else 2.0 ** (e - 1) * (1.0 + 0.5 * m)
    return s * mag


def e2m1_nearest_code(normalized) -> np.ndarray:
    """Brute force: nearest of the eight magnitudes, ties to the even code,
    anything beyond 6 (including +inf) to code 7; sign bit when the binary32
    value compares below zero; NaN -> 0."""
    x = np.asarray(normalized, dtype=np.float32)
    a = np.abs(x).astype(np.float64)
    out = np.zeros(x.shape, dtype=np.uint8)
    finite = np.isfinite(a)
    dist = np.abs(a[..., None] - E2M1_MAGNITUDES)  # [..., 8]
    best = np.argmin(dist, axis=-1)
    # argmin takes the first of equal distances (the odd-lower or even-lower
    # neighbour); move ties onto the even code.
    bd = np.take_along_axis(dist, best[..., None], -1)[..., 0]
    nxt = np.minimum(best + 1, 7)
    tie = (np.take_along_axis(dist, nxt[..., None], -1)[..., 0] == bd) & (nxt != best)
    best = np.where(tie & (best % 2 == 1), nxt, best)
    out[finite] = best[finite].astype(np.uint8)
    out[a > 6.0] = 7  # saturation (also where float64 distances lose precision)
    sign = (x < 0).astype(np.uint8) * 8
    out = out | sign
    out[np.isnan(x)] = 0
    return out


def e4m3_decode_from_bits(b: int) -> float:
    """OCP FP8 E4M3 (fn): bias 7, 3 mantissa bits, subnormals, S.1111.111 NaN."""
    s = -1.0 if b & 0x80 else 1.0
    e = (b >> 3) & 0xF
    m = b & 7
    if e == 0xF and m == 7:
        return float("nan")
    if e == 0:
        return s * (m / 8.0) * 2.0 ** -6
    return s * (1.0 + m / 8.0) * 2.0 ** (e - 7)


E4M3_TABLE = np.array([e4m3_decode_from_bits(b) for b in range(256)], dtype=np.float64)


def e4m3_nearest(y) -> np.ndarray:
    """Brute force round-to-nearest-even onto the finite E4M3 values, for
    |y| <= 448; sign kept on zero; NaN -> 0x7F."""
    y = np.asarray(y, dtype=np.float32)
    a = np.abs(y).astype(np.float64)
    pos = E4M3_TABLE[:127]  # codes 0x00..0x7E, increasing
    dist = np.abs(a[..., None] - pos)
    best = np.argmin(dist, axis=-1)
    bd = np.take_along_axis(dist, best[..., None], -1)[..., 0]
    nxt = np.minimum(best + 1, 126)
    tie = (np.take_along_axis(dist, nxt[..., None], -1)[..., 0] == bd) & (nxt != best)
    best = np.where(tie & (best % 2 == 1), nxt, best)
    out = best.astype(np.uint8) | (np.signbit(y).astype(np.uint8) << 7)
    out[np.isnan(y)] = 0x7F
    return out


def smallest_pow2_exponent_at_least(v) -> np.ndarray:
    """Smallest integer e with 2**e >= v for positive finite v, from frexp:
    v = m * 2**E with m in [0.5, 1), so e = E - 1 when m == 0.5, else E."""
    m, E = np.frexp(np.asarray(v, dtype=np.float64))
    return np.where(m == 0.5, E - 1, E).astype(np.int64)


def mxfp4_row_reference(row_bits: np.ndarray, group: int = 32) -> np.ndarray:
    """Packed MXFP4 row (d/2 code bytes + d/group scale bytes) for a row whose
    finite group maxima make amax/6 a normal binary32 (amax >= 6 * 2**-126),
    or are zero. The scale exponent is the smallest e with amax <= 6 * 2**e,
    found by exact float64 comparison."""
    x = bf16_bits_to_f32(row_bits)
    d = x.shape[0]
    codes = np.zeros(d, dtype=np.uint8)
    scales = np.zeros(d // group, dtype=np.uint8)
    for g in range(d // group):
        xs = x[g * group:(g + 1) * group]
        amax = float(np.max(np.abs(xs.astype(np.float64))))
        if amax == 0.0:
            e = 0
        else:
            assert amax >= 6.0 * 2.0 ** -126, "outside this reference's range"
            e = int(np.floor(np.log2(amax / 6.0))) - 2
            while 6.0 * 2.0 ** e < amax:
                e += 1
        scales[g] = e + 127
        normalized = (xs.astype(np.float64) * 2.0 ** -e).astype(np.float32)  # exact
        codes[g * group:(g + 1) * group] = e2m1_nearest_code(normalized)
    packed = (codes[0::2] | (codes[1::2] << 4)).astype(np.uint8)
    return np.concatenate([packed, scales])


def e2m1_row_decode(row: np.ndarray, d: int = 512, group: int = 32) -> np.ndarray:
    """Decode a packed MXFP4 row to float64 values: E2M1 value * 2**(byte-127)."""
    codes = np.empty(d, dtype=np.uint8)
    codes[0::2] = row[:d // 2] & 0xF
    codes[1::2] = row[:d // 2] >> 4
    vals = np.array([e2m1_decode_from_bits(int(c)) for c in range(16)])[codes]
    scale = np.repeat(row[d // 2:d // 2 + d // group].astype(np.int64), group)
    return vals * np.exp2(scale.astype(np.float64) - 127.0)


def mxfp8_group_reference(r: np.ndarray, sanitize: bool):
    """One MXFP8 group of 32 rotated binary32 values -> (32 value bytes, scale
    byte). Exponent from frexp, values from exact float64 scaling, E4M3 by
    nearest-value search."""
    r = np.asarray(r, dtype=np.float32)
    finite_abs = np.abs(r[~np.isnan(r)])
    amax = np.float32(finite_abs.max()) if finite_abs.size else np.float32(0.0)
    amax = max(amax, np.float32(1e-4))
    v = np.float32(amax) * np.float32(1.0 / 448.0)
    if np.isinf(v):
        e = 128
    else:
        e = int(smallest_pow2_exponent_at_least(v))
    with np.errstate(invalid="ignore", over="ignore"):
        y = (r.astype(np.float64) * 2.0 ** -e).astype(np.float32)
    y = np.where(np.isnan(y), y, np.clip(y, -448.0, 448.0)).astype(np.float32)
    vals = e4m3_nearest(y)
    scale = min(max(e + 127, 0), 254 if sanitize else 255)
    return vals, scale


def nvfp4_tile_reference(r: np.ndarray):
    """One NVFP4 tile of 16 rotated binary32 values -> (16 codes, scale byte).
    q = r / s is formed as a float64 quotient rounded to binary32, which is
    the correctly rounded binary32 quotient here: s has at most 4 significant
    bits, so r / s cannot fall within 2**-53 of a binary32 midpoint without
    being one."""
    r = np.asarray(r, dtype=np.float32)
    finite_abs = np.abs(r[~np.isnan(r)])
    amax = np.float32(finite_abs.max()) if finite_abs.size else np.float32(0.0)
    target = np.float32(amax) * np.float32(1.0 / 6.0)
    target = np.float32(min(max(target, np.float32(0.001953125)), np.float32(448.0)))
    sbyte = int(e4m3_nearest(np.array([target], np.float32))[0])
    s = E4M3_TABLE[sbyte]
    with np.errstate(invalid="ignore"):
        q = (r.astype(np.float64) / s).astype(np.float32)
    return e2m1_nearest_code(q), sbyte
