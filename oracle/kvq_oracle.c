/*
 * kvq_oracle.c — CPU oracle for the MXFP4 / MXFP8 / NVFP4 paged KV-cache store.
 *
 * TEST INFRASTRUCTURE ONLY. This file is the slow, plain, single-threaded
 * reference that the CUDA library is checked against. Only the test suite,
 * the smoke check and the benchmark's CPU-baseline leg may load it; the
 * product path never does. It shares no code, header, table or helper with
 * the CUDA library (fp8_quantized_paged_store_gb300/csrc).
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fno-fast-math -fPIC -shared.
 * All floating point is IEEE binary32 with round-to-nearest-even, gradual
 * underflow (no flush-to-zero) and no fused multiply-add: every product,
 * quotient, sum and difference is rounded on its own, as the pages' Triton
 * code computes in fp32.
 *
 * Pages followed (cited by title and section):
 *   [store]  "vllm.v1.attention.ops.mxfp4_mla.store" (vLLM API docs):
 *            module docstring (row layout), _ceil_pow2_exponent,
 *            _quantize_e2m1, store_mxfp4_mla (argument checks, paged view).
 *   [v41]    "vllm.models.deepseek_v41.common.ops.fused_compress_quant_cache"
 *            (vLLM API docs): _rope_quant_insert_mxfp8_kernel,
 *            _rope_quant_insert_nvfp4_kernel, rope_quant_insert.
 *   [pr]     "[ROCm][Attention] Add an mxfp4_mla KV cache for rope-free sparse
 *            MLA (read/write path)" (vLLM pull request 60321): Overview,
 *            Claims, Details (format and write path; read path), and the
 *            review thread (E2M1 midpoints, zero-group scale byte 127).
 *
 * Readings where the pages are silent are stated beside the code that takes
 * them. Parity status of each function is listed in its comment; the NaN
 * handling of the V4.1 inserts is pinned only by the reading stated here.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* Bit-level helpers (binary32 and bfloat16)                                 */
/* ------------------------------------------------------------------------ */

static uint32_t f32_bits(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return u;
}

static float f32_from_bits(uint32_t u) {
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* bfloat16 is the top half of a binary32, so widening is exact. */
static float bf16_to_f32(uint16_t h) { return f32_from_bits((uint32_t)h << 16); }

/* binary32 -> bfloat16, round to nearest even; every NaN becomes the quiet
 * NaN 0x7FC0. The sign and payload of a NaN that arithmetic produced are not
 * the same on every processor (x86's default NaN is negative, Arm's and
 * CUDA's positive), so a stored NaN carries neither; 0x7FC0 is also what
 * PyTorch's float -> bfloat16 conversion gives for any NaN. */
static uint16_t f32_to_bf16_rne(float f) {
    uint32_t u = f32_bits(f);
    if ((u & 0x7FFFFFFFu) > 0x7F800000u) return 0x7FC0u;
    uint32_t lower = u & 0xFFFFu;
    uint32_t upper = u >> 16;
    if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u))) upper += 1u;
    return (uint16_t)upper;
}

/* Exact 2**k for the k this file needs (-149 <= k <= 127), built from bits so
 * that no library routine is involved. */
static float pow2f(int k) {
    if (k >= -126) return f32_from_bits((uint32_t)(k + 127) << 23);
    return f32_from_bits(1u << (k + 149)); /* subnormal powers of two */
}

/* ------------------------------------------------------------------------ */
/* Format definitions                                                         */
/* ------------------------------------------------------------------------ */

/* [store] module docstring and [pr] Overview: a packed row holds d/2 bytes of
 * two-per-byte E2M1 codes followed by one E8M0 scale byte per group. */
int64_t oracle_row_bytes(int64_t d, int64_t group) { return d / 2 + d / group; }

/* [store] _ceil_pow2_exponent: the smallest integer e with 2**e >= v, read off
 * the binary32 fields of a positive v. With v = m * 2**E, m in [1, 2), the
 * biased exponent field holds E + 127 and the fraction field is zero exactly
 * when v is a power of two, so the answer is E, or E + 1 when the fraction is
 * non-zero. Applied literally to every positive v, including subnormals (field
 * 0, so the result is -126) and +inf (field 255, result 128). */
int32_t oracle_ceil_pow2_exponent(float v) {
    uint32_t u = f32_bits(v);
    int32_t biased = (int32_t)((u >> 23) & 0xFFu);
    uint32_t fraction = u & 0x7FFFFFu;
    int32_t e = biased - 127;
    if (fraction != 0u) e += 1;
    return e;
}

/* The eight E2M1 magnitudes (OCP MX FP4: 1 sign, 2 exponent, 1 mantissa bit,
 * exponent bias 1). Code k (0..7) holds magnitude index k; bit 3 is the sign.
 * [pr] review thread lists the seven midpoints between neighbours. */
static const float kE2M1Magnitude[8] = {0.0f, 0.5f, 1.0f, 1.5f, 2.0f, 3.0f, 4.0f, 6.0f};

float oracle_e2m1_value(uint8_t code) {
    float m = kE2M1Magnitude[code & 7u];
    return (code & 8u) ? -m : m;
}

/* [store] _quantize_e2m1: a binary32 value already divided by its group scale
 * becomes a 4-bit code. The magnitude index is the number of midpoints the
 * magnitude has passed. A value exactly on a midpoint rounds to the neighbour
 * with the even code (round half to even), so the midpoint below an even code
 * is passed when reached (>=) and the one below an odd code only when exceeded
 * (>). Values beyond 6 keep index 7 (saturation). The sign bit is set when the
 * value compares below zero, so a small negative that rounds to magnitude 0
 * encodes as code 8, while -0.0 and NaN (which do not compare below zero)
 * encode with sign 0; NaN also passes no midpoint, giving code 0. */
uint8_t oracle_e2m1_code(float normalized) {
    float a = fabsf(normalized);
    uint8_t index = 0;
    for (int k = 0; k < 7; ++k) {
        float midpoint = 0.5f * (kE2M1Magnitude[k] + kE2M1Magnitude[k + 1]); /* exact */
        int upper_is_even = ((k + 1) % 2) == 0;
        int passed = upper_is_even ? (a >= midpoint) : (a > midpoint);
        index = (uint8_t)(index + (passed ? 1 : 0));
    }
    uint8_t sign = (normalized < 0.0f) ? 8u : 0u;
    return (uint8_t)(index | sign);
}

/* OCP FP8 E4M3 ("e4m3fn", Triton's float8e4nv): 1 sign, 4 exponent bits with
 * bias 7, 3 mantissa bits, subnormals, no infinities, NaN = S.1111.111.
 * Largest finite magnitude 448, smallest subnormal 2**-9. */
float oracle_e4m3_decode(uint8_t b) {
    int sign = (b >> 7) & 1;
    int exp_field = (b >> 3) & 0xF;
    int mant = b & 7;
    float mag;
    if (exp_field == 0xF && mant == 7) {
        mag = NAN;
    } else if (exp_field == 0) {
        mag = (float)mant * pow2f(-9); /* mant/8 * 2**(1-7) */
    } else {
        mag = (float)(8 + mant) * pow2f(exp_field - 7 - 3);
    }
    return sign ? -mag : mag;
}

/* Round a non-negative binary32 holding at most 2**24 to an integer, ties to
 * even. The subtraction q - floor(q) is exact in that range. */
static float round_half_even(float q) {
    float lower = floorf(q);
    float frac = q - lower;
    if (frac > 0.5f) return lower + 1.0f;
    if (frac < 0.5f) return lower;
    return (fmodf(lower, 2.0f) == 0.0f) ? lower : lower + 1.0f;
}

/* binary32 -> E4M3 with round to nearest even, gradual underflow, sign kept
 * on zero (-0 -> 0x80). NaN -> 0x7F. The callers clamp to [-448, 448] first
 * ([v41] both inserts clamp before converting), so magnitudes above 448 never
 * arrive; should one arrive it is treated as overflow and becomes NaN, the
 * non-saturating E4M3 behaviour.
 * Construction: below 2**-6 the grid is the subnormal step 2**-9, so the code
 * is round(a * 2**9) (a result of 8 is the smallest normal, code 8). At or
 * above 2**-6, with a in [2**E, 2**(E+1)), the grid step is 2**(E-3):
 * m = round(a * 2**(3-E)) lies in [8, 16] and the code is (E+7)*8 + (m-8),
 * where m == 16 carries into the next binade by itself. */
uint8_t oracle_e4m3_encode(float y) {
    if (isnan(y)) return 0x7Fu;
    uint8_t sign = signbit(y) ? 0x80u : 0x00u;
    float a = fabsf(y);
    if (a > 448.0f) return (uint8_t)(sign | 0x7Fu);
    int code;
    if (a < pow2f(-6)) {
        code = (int)round_half_even(a * pow2f(9));
    } else {
        int E = (int)((f32_bits(a) >> 23) & 0xFFu) - 127; /* a is normal here */
        float m = round_half_even(a * pow2f(3 - E));
        code = (E + 7) * 8 + ((int)m - 8);
    }
    return (uint8_t)(sign | (uint8_t)code);
}

/* ------------------------------------------------------------------------ */
/* Paged addressing                                                           */
/* ------------------------------------------------------------------------ */

/* [store] store_mxfp4_mla: the layer's cache is a [num_blocks, block_size,
 * row_bytes] view whose block stride may exceed block_size rows (other layers'
 * pages sit between blocks); a flat cache is one block. Slot s lives in block
 * s / block_size at row s % block_size. Returns the row's byte offset. */
static int64_t paged_row_offset(int64_t slot, int64_t block_size, int64_t block_stride_rows,
                                int64_t row_bytes) {
    int64_t block = slot / block_size;
    int64_t row_in_block = slot % block_size;
    return (block * block_stride_rows + row_in_block) * row_bytes;
}

/* ------------------------------------------------------------------------ */
/* MXFP4 group scale and store                                                */
/* ------------------------------------------------------------------------ */

/* [pr] Details, format and write path: the E8M0 scale uses the round-up
 * exponent so that no value clamps; [store] _ceil_pow2_exponent gives that
 * exponent exactly; [pr] review thread: an all-zero group gets scale byte 127.
 * Reading: e = ceil_pow2_exponent(RN32(amax / 6)), 6 being the largest E2M1
 * magnitude, and e = 0 for amax == 0. */
int32_t oracle_mxfp4_scale_exponent(float amax) {
    if (amax == 0.0f) return 0;
    float v = amax / 6.0f;
    return oracle_ceil_pow2_exponent(v);
}

/* Largest magnitude of a group, ignoring NaN (a NaN never compares greater),
 * starting from +0. */
static float group_amax(const float* x, int n) {
    float amax = 0.0f;
    for (int j = 0; j < n; ++j) {
        float a = fabsf(x[j]);
        if (a > amax) amax = a;
    }
    return amax;
}

/* Quantize one latent row (d bf16 values) into a packed MXFP4 row of
 * d/2 + d/group bytes. [store] module docstring, [pr] Details: codes first,
 * two per byte with the lower index in the low nibble, then the scale bytes. */
static void mxfp4_quantize_row(const uint16_t* src, int64_t d, int32_t group, uint8_t* row) {
    float x[1024];
    for (int64_t g0 = 0; g0 < d; g0 += group) {
        for (int j = 0; j < group; ++j) x[j] = bf16_to_f32(src[g0 + j]);
        float amax = group_amax(x, group);
        int32_t e = oracle_mxfp4_scale_exponent(amax);
        row[d / 2 + g0 / group] = (uint8_t)(e + 127);
        /* "fp32 values pre-divided by their group scale": x * 2**-e, one
         * rounding (exact unless the result is subnormal). */
        float inv_scale = pow2f(-e);
        for (int j = 0; j < group; j += 2) {
            uint8_t lo = oracle_e2m1_code(x[j] * inv_scale);
            uint8_t hi = oracle_e2m1_code(x[j + 1] * inv_scale);
            row[(g0 + j) / 2] = (uint8_t)(lo | (uint8_t)(hi << 4));
        }
    }
}

/* [store] store_mxfp4_mla. For each token t: read slot_mapping[t]; skip it if
 * negative (PAD_SLOT_ID) or, reading the passed num_slots as a bound, if it is
 * >= num_blocks * block_size; otherwise quantize row t (row_stride elements
 * apart) and write its row_bytes(d, group) bytes at the slot's paged offset.
 * All other cache bytes are left as they were. Requires group even,
 * d % group == 0 and group <= 1024. */
void oracle_mxfp4_mla_store(const uint16_t* latent, int64_t num_tokens, int64_t latent_dim,
                            int64_t row_stride, const int64_t* slot_mapping, uint8_t* cache,
                            int64_t num_blocks, int64_t block_size, int64_t block_stride_rows,
                            int32_t group) {
    int64_t row_bytes = oracle_row_bytes(latent_dim, group);
    int64_t num_slots = num_blocks * block_size;
    for (int64_t t = 0; t < num_tokens; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0 || slot >= num_slots) continue;
        uint8_t* row = cache + paged_row_offset(slot, block_size, block_stride_rows, row_bytes);
        mxfp4_quantize_row(latent + t * row_stride, latent_dim, group, row);
    }
}

/* ------------------------------------------------------------------------ */
/* MXFP4 gather and dequantize (read path)                                    */
/* ------------------------------------------------------------------------ */

/* [pr] Details, read path: a gathered packed row is unpacked to bf16, each
 * value being the E2M1 code's value times 2**(scale_byte - 127); [pr] Claims:
 * attention over the packed cache equals attention over those values stored
 * as bf16. The product has at most two significant bits, so it is exact in
 * binary32 and in bf16 (down to 2**-128), except that byte 254 with the larger
 * codes overflows to +-inf. Reading (pages silent): scale byte 255, the E8M0
 * NaN, gives bf16 NaN 0x7FC0 for the whole group; an index that is negative
 * (padding) or >= num_slots gives a row of +0.0. */
void oracle_mxfp4_mla_gather_dequant(const uint8_t* cache, int64_t num_blocks, int64_t block_size,
                                     int64_t block_stride_rows, int64_t latent_dim, int32_t group,
                                     const int64_t* indices, int64_t num_indices, uint16_t* out,
                                     int64_t out_row_stride) {
    int64_t row_bytes = oracle_row_bytes(latent_dim, group);
    int64_t num_slots = num_blocks * block_size;
    for (int64_t k = 0; k < num_indices; ++k) {
        uint16_t* dst = out + k * out_row_stride;
        int64_t slot = indices[k];
        if (slot < 0 || slot >= num_slots) {
            for (int64_t j = 0; j < latent_dim; ++j) dst[j] = 0x0000u;
            continue;
        }
        const uint8_t* row = cache + paged_row_offset(slot, block_size, block_stride_rows, row_bytes);
        for (int64_t j = 0; j < latent_dim; ++j) {
            uint8_t byte = row[j / 2];
            uint8_t code = (j % 2 == 0) ? (uint8_t)(byte & 0xFu) : (uint8_t)(byte >> 4);
            uint8_t scale_byte = row[latent_dim / 2 + j / group];
            if (scale_byte == 255u) {
                dst[j] = 0x7FC0u;
                continue;
            }
            float value = oracle_e2m1_value(code) * pow2f((int)scale_byte - 127);
            dst[j] = f32_to_bf16_rne(value);
        }
    }
}

/* ------------------------------------------------------------------------ */
/* V4.1 RoPE-then-quantize inserts                                            */
/* ------------------------------------------------------------------------ */

/* [v41] both insert kernels: the token is skipped when its cache slot is
 * negative, and otherwise unless (position + 1) is a multiple of the compress
 * ratio R. Readings added for inputs the pages leave undefined: a slot at or
 * beyond num_pages * cache_block, a negative position, or a table row
 * (position // R) * R at or beyond cos_sin_rows also skips the token.
 * Returns the table row to use, or -1 to skip. */
static int64_t rope_gate(int64_t slot, int64_t position, int64_t num_pages, int64_t cache_block,
                         int32_t compress_ratio, int64_t cos_sin_rows) {
    if (slot < 0 || slot >= num_pages * cache_block) return -1;
    if (position < 0) return -1;
    /* A table row is at least position - (R - 1), so position - R >= rows can
     * only give a row past the table; testing it first keeps position + 1
     * from overflowing and changes no result. */
    if (position - compress_ratio >= cos_sin_rows) return -1;
    if ((position + 1) % compress_ratio != 0) return -1;
    int64_t table_row = (position / compress_ratio) * compress_ratio;
    if (table_row >= cos_sin_rows) return -1;
    return table_row;
}

/* [v41] GPT-J (interleaved) rotary embedding on a 512-wide row: pair i holds
 * elements 2i (even) and 2i+1 (odd). Pairs 224..255 (the last 64 elements)
 * use cos = cs[i - 224] and sin = cs[32 + i - 224] from the table row; every
 * other pair uses cos 1, sin 0. The rotated pair is
 *   (even*cos - odd*sin, odd*cos + even*sin),
 * evaluated literally for all 256 pairs in binary32, each product and each
 * sum rounded separately (no fused multiply-add). With cos 1, sin 0 this is
 * the identity for finite inputs; a NaN or infinite partner still spreads NaN
 * (x * 0), and (-0, negative) becomes (+0, ...), as the literal formula gives.
 * With sanitize set, NaN results are replaced by +0.0. */
static void rope_rotate_row(const uint16_t* src, const float* cs, int32_t sanitize, float* out) {
    for (int i = 0; i < 256; ++i) {
        float even = bf16_to_f32(src[2 * i]);
        float odd = bf16_to_f32(src[2 * i + 1]);
        float c = 1.0f, s = 0.0f;
        if (i >= 224) {
            c = cs[i - 224];
            s = cs[32 + (i - 224)];
        }
        float ec = even * c;
        float os = odd * s;
        float oc = odd * c;
        float es = even * s;
        float r_even = ec - os;
        float r_odd = oc + es;
        if (sanitize) {
            if (isnan(r_even)) r_even = 0.0f;
            if (isnan(r_odd)) r_odd = 0.0f;
        }
        out[2 * i] = r_even;
        out[2 * i + 1] = r_odd;
    }
}

/* One MXFP8 tile of n rotated values (the rule the comment below states):
 * n E4M3 value bytes and the E8M0 scale byte. */
static void mxfp8_tile(const float* x, int n, int32_t sanitize, uint8_t* values,
                       uint8_t* scale_byte) {
    const float kMinAmax = 1e-4f;
    const float kInv448 = 1.0f / 448.0f;
    float amax = group_amax(x, n);
    if (!(amax >= kMinAmax)) amax = kMinAmax;
    float v = amax * kInv448;
    int32_t e = oracle_ceil_pow2_exponent(v);
    float inv_scale = pow2f(-e);
    for (int j = 0; j < n; ++j) {
        float y = x[j] * inv_scale;
        if (y > 448.0f) y = 448.0f;
        if (y < -448.0f) y = -448.0f;
        values[j] = oracle_e4m3_encode(y);
    }
    int32_t encoded = e + 127;
    int32_t cap = sanitize ? 254 : 255;
    if (encoded < 0) encoded = 0;
    if (encoded > cap) encoded = cap;
    *scale_byte = (uint8_t)encoded;
}

/* [v41] _rope_quant_insert_mxfp8_kernel: the 528-byte V4.1 record. Per group
 * of 32 rotated values:
 *   amax  = max(largest |value| (NaN ignored), fl32(1e-4))
 *   e     = ceil(log2(amax * fl32(1/448)))  -- taken exactly from the bits of
 *           the rounded product (the product is always a normal binary32);
 *           reading: the pages' log2/ceil is meant as the exact ceiling
 *   value = E4M3(clamp(x * 2**-e, -448, 448)), round to nearest even; NaN
 *           passes the clamp and encodes as 0x7F (reading)
 *   scale = clamp(e + 127, 0, sanitize ? 254 : 255)
 * Page layout for CACHE_BLOCK slots: CACHE_BLOCK * 512 value bytes, then
 * CACHE_BLOCK * 16 scale bytes; slot s is row s % CACHE_BLOCK of page
 * s / CACHE_BLOCK, pages page_stride_bytes apart. */
void oracle_rope_quant_insert_mxfp8(const uint16_t* latent, int64_t num_tokens, int64_t row_stride,
                                    const int64_t* positions, const float* cos_sin,
                                    int64_t cos_stride, int64_t cos_sin_rows, uint8_t* cache,
                                    const int64_t* cache_slots, int64_t num_pages,
                                    int64_t cache_block, int64_t page_stride_bytes,
                                    int32_t compress_ratio, int32_t sanitize) {
    float rotated[512];
    for (int64_t t = 0; t < num_tokens; ++t) {
        int64_t slot = cache_slots[t];
        int64_t table_row = rope_gate(slot, positions[t], num_pages, cache_block, compress_ratio,
                                      cos_sin_rows);
        if (table_row < 0) continue;
        rope_rotate_row(latent + t * row_stride, cos_sin + table_row * cos_stride, sanitize,
                        rotated);
        uint8_t* page = cache + (slot / cache_block) * page_stride_bytes;
        uint8_t* values = page + (slot % cache_block) * 512;
        uint8_t* scales = page + cache_block * 512 + (slot % cache_block) * 16;
        for (int g = 0; g < 16; ++g) mxfp8_tile(rotated + 32 * g, 32, sanitize, values + 32 * g,
                                                scales + g);
    }
}

/* [v41] _rope_quant_insert_nvfp4_kernel: the 288-byte V4.1 NVFP4 record. Per
 * tile of 16 rotated values:
 *   amax  = largest |value| (NaN ignored, from +0)
 *   s     = E4M3(clamp(amax * fl32(1/6), 2**-9, 448)), round to nearest even
 *   q     = x / s, correctly rounded binary32 division (the page insists on a
 *           round-to-nearest division because e2m1 ties must land right)
 *   code  = the same E2M1 threshold rule as the MXFP4 store (saturating)
 * Codes pair up two per byte, even element in the low nibble (reading, as in
 * the MXFP4 row). Page layout: CACHE_BLOCK * 256 code bytes, then
 * CACHE_BLOCK * 32 scale bytes (the E4M3 bits of s). */
void oracle_rope_quant_insert_nvfp4(const uint16_t* latent, int64_t num_tokens, int64_t row_stride,
                                    const int64_t* positions, const float* cos_sin,
                                    int64_t cos_stride, int64_t cos_sin_rows, uint8_t* cache,
                                    const int64_t* cache_slots, int64_t num_pages,
                                    int64_t cache_block, int64_t page_stride_bytes,
                                    int32_t compress_ratio, int32_t sanitize) {
    const float kInv6 = 1.0f / 6.0f;
    const float kMinScale = 0.001953125f; /* 2**-9 */
    const float kMaxScale = 448.0f;
    float rotated[512];
    for (int64_t t = 0; t < num_tokens; ++t) {
        int64_t slot = cache_slots[t];
        int64_t table_row = rope_gate(slot, positions[t], num_pages, cache_block, compress_ratio,
                                      cos_sin_rows);
        if (table_row < 0) continue;
        rope_rotate_row(latent + t * row_stride, cos_sin + table_row * cos_stride, sanitize,
                        rotated);
        uint8_t* page = cache + (slot / cache_block) * page_stride_bytes;
        uint8_t* codes = page + (slot % cache_block) * 256;
        uint8_t* scales = page + cache_block * 256 + (slot % cache_block) * 32;
        for (int g = 0; g < 32; ++g) {
            const float* x = rotated + 16 * g;
            float amax = group_amax(x, 16);
            float target = amax * kInv6;
            if (target < kMinScale) target = kMinScale;
            if (target > kMaxScale) target = kMaxScale;
            uint8_t scale_byte = oracle_e4m3_encode(target);
            float s = oracle_e4m3_decode(scale_byte);
            for (int j = 0; j < 16; j += 2) {
                uint8_t lo = oracle_e2m1_code(x[j] / s);
                uint8_t hi = oracle_e2m1_code(x[j + 1] / s);
                codes[(16 * g + j) / 2] = (uint8_t)(lo | (uint8_t)(hi << 4));
            }
            scales[g] = scale_byte;
        }
    }
}

/* ------------------------------------------------------------------------ */
/* RMSNorm ahead of the MXFP4 store                                           */
/* ------------------------------------------------------------------------ */

/* [store] store_mxfp4_mla takes "the post-RMSNorm latent"; the V4.1 page's
 * fused_save_compress_norm normalises with a bf16 [512] weight and an fp32
 * epsilon into a bf16 latent. The pages fix neither the order of the sum of
 * squares nor how the reciprocal square root is formed. This library fixes
 * both as part of its interface, in element terms:
 *   blocks: the 512 elements form 32 blocks of sixteen; block k holds
 *     elements 8k, 8k+1, ..., 8k+7 followed by 256+8k, ..., 256+8k+7;
 *   B[k] = the squares of block k's elements added left to right in that
 *     listed order, from +0 (every square and every sum rounded to binary32);
 *   S = a balanced pairwise tree over B[0..31] in block order: B[0]+B[1],
 *     B[2]+B[3], ..., then neighbouring results added pairwise again, five
 *     levels in all;
 *   r = RN(1 / RN(sqrt(RN(S / 512 + eps)))),      (S / 512 is exact scaling)
 *   y = bf16(RN(x * r)),   z = bf16(y * w)        (y * w is exact in binary32).
 * The row is normalised when latent_dim is 512; z is then quantized exactly
 * as by oracle_mxfp4_mla_store. */
static int rmsnorm_block_element(int k, int i) { return i < 8 ? 8 * k + i : 256 + 8 * k + (i - 8); }

static float rmsnorm_sum_of_squares(const uint16_t* x) {
    float sums[32];
    for (int k = 0; k < 32; ++k) {
        float acc = 0.0f;
        for (int i = 0; i < 16; ++i) {
            float v = bf16_to_f32(x[rmsnorm_block_element(k, i)]);
            acc = acc + v * v;
        }
        sums[k] = acc;
    }
    for (int n = 32; n > 1; n /= 2)
        for (int k = 0; k < n / 2; ++k) sums[k] = sums[2 * k] + sums[2 * k + 1];
    return sums[0];
}

static void rmsnorm_row_512(const uint16_t* x, const uint16_t* w, float eps, uint16_t* z) {
    float mean = rmsnorm_sum_of_squares(x) / 512.0f;
    float var = mean + eps;
    float root = sqrtf(var);
    float r = 1.0f / root;
    for (int j = 0; j < 512; ++j) {
        float xr = bf16_to_f32(x[j]) * r;
        uint16_t y = f32_to_bf16_rne(xr);
        float yw = bf16_to_f32(y) * bf16_to_f32(w[j]);
        z[j] = f32_to_bf16_rne(yw);
    }
}

void oracle_rmsnorm_rows(const uint16_t* x, int64_t num_rows, int64_t row_stride,
                         const uint16_t* weight, float eps, uint16_t* out) {
    for (int64_t t = 0; t < num_rows; ++t) rmsnorm_row_512(x + t * row_stride, weight, eps, out + t * 512);
}

/* RMSNorm, then the MXFP4 store of the normalised row (latent_dim 512). */
void oracle_mxfp4_mla_rmsnorm_store(const uint16_t* latent, int64_t num_tokens, int64_t row_stride,
                                    const uint16_t* weight, float eps,
                                    const int64_t* slot_mapping, uint8_t* cache,
                                    int64_t num_blocks, int64_t block_size,
                                    int64_t block_stride_rows) {
    /* By definition: normalise the token's row, then store it as a one-token
     * batch (the store applies the slot rules). */
    uint16_t z[512];
    for (int64_t t = 0; t < num_tokens; ++t) {
        rmsnorm_row_512(latent + t * row_stride, weight, eps, z);
        oracle_mxfp4_mla_store(z, 1, 512, 512, slot_mapping + t, cache, num_blocks, block_size,
                               block_stride_rows, 32);
    }
}

/* ------------------------------------------------------------------------ */
/* The other rope_quant_insert layouts, and save_ring_rows                    */
/* ------------------------------------------------------------------------ */

/* [v41] rope_quant_insert, docstring: a bfloat16 or float8_e4m3fn cache holds
 * the plain [448 NoPE | 64 RoPE] rows read by FlashInfer, the fp8 one scaled
 * by the per-tensor fp8_scale; the cache is [pages, CACHE_BLOCK, 512] with its
 * own page and row strides and unit element stride. The kernel
 * (_rope_plain_insert_kernel) is not printed. Readings: the gates and table
 * row of the paged records (rope_gate); elements 0..447 are the latent's own
 * values (copied bit for bit into the bf16 cache), elements 448..511 the
 * rotated pairs (binary32 as rope_rotate_row, no sanitising) rounded to bf16,
 * nearest even. The fp8 cache stores E4M3(clamp(RN(x / fp8_scale), -448,
 * 448)) of each element x (the latent's value, or the rotated binary32
 * value): a quotient, as the scale is the dequantizing factor; NaN as 0x7F.
 * Strides are in elements (2 bytes for bf16, 1 for fp8). */
void oracle_rope_plain_insert(const uint16_t* latent, int64_t num_tokens, int64_t row_stride,
                              const int64_t* positions, const float* cos_sin, int64_t cos_stride,
                              int64_t cos_sin_rows, uint8_t* cache, const int64_t* cache_slots,
                              int64_t num_pages, int64_t cache_block, int64_t page_stride,
                              int64_t slot_stride, int32_t compress_ratio, int32_t fp8,
                              float fp8_scale) {
    float rotated[512];
    for (int64_t t = 0; t < num_tokens; ++t) {
        int64_t slot = cache_slots[t];
        int64_t table_row = rope_gate(slot, positions[t], num_pages, cache_block, compress_ratio,
                                      cos_sin_rows);
        if (table_row < 0) continue;
        const uint16_t* src = latent + t * row_stride;
        rope_rotate_row(src, cos_sin + table_row * cos_stride, 0, rotated);
        int64_t base = (slot / cache_block) * page_stride + (slot % cache_block) * slot_stride;
        for (int j = 0; j < 512; ++j) {
            if (!fp8) {
                uint16_t h = j < 448 ? src[j] : f32_to_bf16_rne(rotated[j]);
                uint8_t* dst = cache + 2 * (base + j);
                dst[0] = (uint8_t)(h & 0xFF);
                dst[1] = (uint8_t)(h >> 8);
            } else {
                float x = j < 448 ? bf16_to_f32(src[j]) : rotated[j];
                float y = x / fp8_scale;
                if (y > 448.0f) y = 448.0f;
                if (y < -448.0f) y = -448.0f;
                cache[base + j] = oracle_e4m3_encode(y);
            }
        }
    }
}

/* [v41] rope_quant_insert, docstring: the 584-byte V4 record holds 576 value
 * bytes and eight segregated UE8M0 scale bytes, one of them a zero padding
 * scale. The kernel (_rope_quant_insert_kernel) is not printed. Reading (the
 * split 584 = 448 + 2 * 64 + 8 implies): value bytes 0..447 are the 448 NoPE
 * values as E4M3 in seven tiles of 64, each tile under the V4.1 MXFP8 rule
 * (amax floor 1e-4, e = ceil(log2(amax * (1/448))), values
 * E4M3(clamp(x * 2**-e, -448, 448)), scale byte clamp(e + 127, 0,
 * sanitize ? 254 : 255)); value bytes 448..575 are the 64 rotated values as
 * bf16 (nearest even, little-endian); scale bytes 0..6 belong to the tiles and
 * byte 7 is 0. All 512 values go through rope_rotate_row (identity formula on
 * the NoPE pairs, sanitising as asked), as in the V4.1 records of the same
 * page. Page layout as those records: CACHE_BLOCK * 576 value bytes, then
 * CACHE_BLOCK * 8 scale bytes. */
void oracle_rope_quant_insert_v4(const uint16_t* latent, int64_t num_tokens, int64_t row_stride,
                                 const int64_t* positions, const float* cos_sin,
                                 int64_t cos_stride, int64_t cos_sin_rows, uint8_t* cache,
                                 const int64_t* cache_slots, int64_t num_pages,
                                 int64_t cache_block, int64_t page_stride_bytes,
                                 int32_t compress_ratio, int32_t sanitize) {
    const int kTile = 64;
    float rotated[512];
    for (int64_t t = 0; t < num_tokens; ++t) {
        int64_t slot = cache_slots[t];
        int64_t table_row = rope_gate(slot, positions[t], num_pages, cache_block, compress_ratio,
                                      cos_sin_rows);
        if (table_row < 0) continue;
        rope_rotate_row(latent + t * row_stride, cos_sin + table_row * cos_stride, sanitize,
                        rotated);
        uint8_t* page = cache + (slot / cache_block) * page_stride_bytes;
        uint8_t* values = page + (slot % cache_block) * 576;
        uint8_t* scales = page + cache_block * 576 + (slot % cache_block) * 8;
        for (int g = 0; g < 7; ++g) mxfp8_tile(rotated + kTile * g, kTile, sanitize,
                                               values + kTile * g, scales + g);
        scales[7] = 0;
        for (int j = 0; j < 64; ++j) {
            uint16_t h = f32_to_bf16_rne(rotated[448 + j]);
            values[448 + 2 * j] = (uint8_t)(h & 0xFF);
            values[448 + 2 * j + 1] = (uint8_t)(h >> 8);
        }
    }
}

/* [v41] save_ring_rows: store fp32 [kv, score] rows of 1024 values to their
 * ring slots, skipping slot -1. Reading: slot s goes to row s % STATE_BLOCK of
 * block s / STATE_BLOCK (strides in floats); a slot < 0 or >= num_blocks *
 * STATE_BLOCK is skipped; the row is copied bit for bit. */
void oracle_save_ring_rows(const float* rows, int64_t num_rows, int64_t row_stride,
                           const int64_t* slot_mapping, float* state, int64_t num_blocks,
                           int64_t state_block, int64_t state_stride, int64_t state_row_stride) {
    for (int64_t t = 0; t < num_rows; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0 || slot >= num_blocks * state_block) continue;
        float* dst = state + (slot / state_block) * state_stride + (slot % state_block) * state_row_stride;
        memcpy(dst, rows + t * row_stride, 1024 * sizeof(float));
    }
}

/* ------------------------------------------------------------------------ */
/* Element-wise entry points used by the pin tests                            */
/* ------------------------------------------------------------------------ */

void oracle_e2m1_code_array(const float* in, uint8_t* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_e2m1_code(in[i]);
}

void oracle_ceil_pow2_exponent_array(const float* in, int32_t* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_ceil_pow2_exponent(in[i]);
}

void oracle_mxfp4_scale_exponent_array(const float* amax, int32_t* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_mxfp4_scale_exponent(amax[i]);
}

void oracle_e4m3_encode_array(const float* in, uint8_t* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m3_encode(in[i]);
}

void oracle_e4m3_decode_array(const uint8_t* in, float* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m3_decode(in[i]);
}

void oracle_e2m1_value_array(const uint8_t* in, float* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_e2m1_value(in[i]);
}
