/*
 * kvq.h — C ABI of the GB300 (sm_103a) quantize-and-scatter library for a
 * paged MLA KV cache: MXFP4 store, RoPE-then-quantize inserts (V4.1 MXFP8
 * and NVFP4 records, the V4 record, plain bf16 / fp8 rows), the compressor's
 * ring-state save, the compressor's pooling + RMSNorm step, the MXFP4
 * gather-and-dequantize read and sparse MLA attention on the packed cache.
 *
 * Pages this interface follows (cited by title and section):
 *   [store] "vllm.v1.attention.ops.mxfp4_mla.store" (vLLM API docs):
 *           module docstring, _ceil_pow2_exponent, _quantize_e2m1,
 *           store_mxfp4_mla.
 *   [v41]   "vllm.models.deepseek_v41.common.ops.fused_compress_quant_cache"
 *           (vLLM API docs): _rope_quant_insert_mxfp8_kernel,
 *           _rope_quant_insert_nvfp4_kernel, rope_quant_insert (and its
 *           docstring on the V4 record and the plain rows), save_ring_rows,
 *           fused_save_compress_norm.
 *   [pr]    "[ROCm][Attention] Add an mxfp4_mla KV cache for rope-free sparse
 *           MLA (read/write path)", vLLM pull request 60321: Overview, Claims,
 *           Details (format and write path; read path).
 *
 * Conventions shared by every entry point
 *   - All pointers are DEVICE pointers owned by the caller (cudaMalloc'd, or
 *     any memory the GPU can address). The library allocates nothing, keeps
 *     no pointer past the call, and never synchronises: work is enqueued on
 *     `stream` (0 = the legacy default stream) and the call returns.
 *     Page-locked host memory that the device addresses under the same
 *     pointer (cudaHostAlloc / cudaMallocHost under unified addressing;
 *     kvq_pointer_kind() tells) is such memory: the kernels then read their
 *     inputs from, and write their rows into, host memory over the
 *     host-device link (NVLink-C2C on a GB300 node), with no copy before or
 *     after the call; the call is then bound by the link's bandwidth.
 *   - bf16 data is passed as raw 16-bit patterns (`const void*`).
 *   - Status: 0 (KVQ_OK) on success; KVQ_EINVAL (-1) when an argument is
 *     rejected before anything is launched (nothing is written); KVQ_ECUDA
 *     (-2) when the launch itself failed (cudaGetLastError after the launch).
 *     kvq_strerror() names every status.
 *   - num_tokens / num_indices == 0 returns KVQ_OK without a launch, after
 *     the shape arguments have been checked ([store] store_mxfp4_mla returns
 *     early for an empty batch).
 *   - Device-side conditions that the host cannot see (a slot or index
 *     outside the cache, a position outside the table) never fault: the
 *     affected token is skipped, or for the gather its row is written as
 *     zeros. Two tokens that name the same slot race (last writer unknown),
 *     as in any scatter.
 *   - Alignment: bf16 row bases and row pitches must be multiples of 16
 *     bytes (row strides multiples of 8 elements); cache and output bases
 *     must be 16-byte aligned; int64 arrays 8-byte aligned; the cos/sin table
 *     base 16-byte aligned with a row stride that is a multiple of 4 floats.
 *     Misalignment is KVQ_EINVAL.
 */
#ifndef KVQ_H
#define KVQ_H

#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define KVQ_OK 0
#define KVQ_EINVAL (-1)
#define KVQ_ECUDA (-2)
#define KVQ_ESCRATCH (-3) /* the shapes need more scratch than the built-in array */

/* Short English description of a status code (static storage). */
const char* kvq_strerror(int status);

/* Bytes of one packed MXFP4 row: latent_dim/2 code bytes + latent_dim/group
 * scale bytes ([store] module docstring: row_bytes(d) = d//2 + d//32).
 * kvq_row_bytes(512, 32) == 272. Returns -1 unless latent_dim > 0,
 * group > 0, group even and latent_dim a multiple of group. */
int64_t kvq_row_bytes(int64_t latent_dim, int64_t group);

#define KVQ_PTR_UNADDRESSABLE 0
#define KVQ_PTR_DEVICE 1
#define KVQ_PTR_HOST_MAPPED 2

/* Where `ptr` lives, for a kernel launched on the current device under that
 * same address (a helper of this library; the pages have no counterpart):
 *   KVQ_PTR_DEVICE          memory of the current device, or managed memory;
 *   KVQ_PTR_HOST_MAPPED     page-locked host memory mapped into the device's
 *                           address space at the same address;
 *   KVQ_PTR_UNADDRESSABLE   anything else (pageable host memory, another
 *                           device's memory, host memory registered at a
 *                           different device address): not to be passed;
 *   KVQ_EINVAL for a null pointer, KVQ_ECUDA when the CUDA runtime cannot
 *   answer (no device). Host-only: launches nothing, never synchronises. */
int kvq_pointer_kind(const void* ptr);

/*
 * mxfp4_mla_store — quantize MLA latent rows to MXFP4 and scatter them into a
 * paged cache. [store] store_mxfp4_mla, _ceil_pow2_exponent, _quantize_e2m1;
 * [pr] Details (format and write path).
 *
 * For each token t in [0, num_tokens) with s = slot_mapping[t]:
 *   - s < 0 (padding) or s >= num_blocks*block_size: skipped, nothing read.
 *   - otherwise row t (latent_dim bf16 values starting at
 *     latent_bf16 + t*row_stride_elems) is split into groups of `group`;
 *     each group gets the E8M0 exponent e = ceil(log2(amax/6)) taken from the
 *     binary32 bits of RN(amax/6) (0 for an all-zero group; NaN is ignored by
 *     amax), and every value becomes the E2M1 code of x * 2**-e, rounded to
 *     nearest with ties to the even code, sign bit set when x * 2**-e < 0.
 *     The 272-byte row [256 code bytes, low nibble = lower index | 16 scale
 *     bytes e+127] is written at byte offset
 *       ((s / block_size) * block_stride_rows + s % block_size) * 272
 *     of `cache`. Nothing else in the cache is touched.
 *
 * latent_bf16        bf16 [num_tokens, row_stride_elems], first latent_dim used
 * num_tokens         >= 0
 * latent_dim         must be 512
 * row_stride_elems   >= latent_dim, multiple of 8
 * slot_mapping       int64 [num_tokens]
 * cache              uint8, this layer's view: block b starts at row
 *                    b*block_stride_rows (rows of 272 bytes)
 * num_blocks         >= 1
 * block_size         >= 1 slots per block
 * block_stride_rows  >= block_size (larger when other layers' pages sit
 *                    between this layer's blocks); a flat cache of N rows is
 *                    num_blocks = 1, block_size = block_stride_rows = N
 * group              must be 32 (the OCP MX block size)
 */
int mxfp4_mla_store(const void* latent_bf16, int64_t num_tokens, int64_t latent_dim,
                    int64_t row_stride_elems, const int64_t* slot_mapping, uint8_t* cache,
                    int64_t num_blocks, int64_t block_size, int64_t block_stride_rows,
                    int32_t group, cudaStream_t stream);

/*
 * mxfp4_mla_rmsnorm_store — RMSNorm of the pre-norm latent, then the MXFP4
 * store, in one pass (the latent is never written back as bf16).
 * "vllm.v1.attention.ops.mxfp4_mla.store" (store_mxfp4_mla stores the
 * post-RMSNorm latent) and
 * "vllm.models.deepseek_v41.common.ops.fused_compress_quant_cache"
 * (fused_save_compress_norm: bf16 [512] weight, fp32 epsilon, bf16 latent).
 *
 * Per token with a valid slot: the RMSNorm below, then exactly what
 * mxfp4_mla_store does with the normalised bf16 row. The pages fix neither
 * the summation order nor the reciprocal square root. This library fixes
 * both as part of its interface, in element terms, so the result is
 * reproducible bit for bit by any implementation:
 *   blocks     block k (k = 0..31) = elements 8k..8k+7 followed by
 *              256+8k..256+8k+7,
 *   B_k        = the squares of block k's elements added left to right in
 *              that order (every square and every sum rounded to binary32),
 *   S          = balanced pairwise tree over B_0..B_31 in block order
 *              ((B_0+B_1), (B_2+B_3), ..., then neighbouring pairs of those,
 *              five levels),
 *   r          = RN(1 / RN(sqrt(RN(S / 512 + eps)))),
 *   y          = bf16(RN(x * r)),   z = bf16(y * w).
 * Any other order changes some outputs: a row on which this order, sixteen
 * consecutive elements per block, and a plain left-to-right sum give three
 * different results is among the library's tests.
 *
 * weight_bf16  bf16 [512], 16-byte aligned
 * eps          >= 0 and finite
 * Other arguments, layout, ownership and errors as mxfp4_mla_store.
 */
int mxfp4_mla_rmsnorm_store(const void* latent_bf16, int64_t num_tokens, int64_t latent_dim,
                            int64_t row_stride_elems, const void* weight_bf16, float eps,
                            const int64_t* slot_mapping, uint8_t* cache, int64_t num_blocks,
                            int64_t block_size, int64_t block_stride_rows, int32_t group,
                            cudaStream_t stream);

/*
 * rope_quant_insert_mxfp8 — V4.1 528-byte record: GPT-J RoPE, then MXFP8.
 * [v41] _rope_quant_insert_mxfp8_kernel, rope_quant_insert.
 *
 * For each token t with slot s = cache_slots[t] and position p = positions[t]:
 *   - skipped if s < 0, s >= num_pages*cache_block, p < 0,
 *     (p + 1) % compress_ratio != 0, or the table row
 *     r = (p / compress_ratio) * compress_ratio is >= cos_sin_rows.
 *   - otherwise the 512 bf16 values are widened to binary32 and pair i
 *     (elements 2i, 2i+1) is rotated to (e*c - o*s, o*c + e*s), each product
 *     and sum rounded separately (no fused multiply-add), with
 *     c = cos_sin[r*cos_stride + i-224], s = cos_sin[r*cos_stride + 32 + i-224]
 *     for i >= 224 and c = 1, s = 0 for i < 224. If sanitize_nans, NaN
 *     results become +0.0.
 *   - per group of 32: amax = max(largest |x| ignoring NaN, 1e-4f),
 *     e = ceil(log2(amax * (1/448.f))) exactly, values E4M3(x * 2**-e)
 *     clamped to +-448 and rounded to nearest even (NaN -> 0x7F), scale byte
 *     clamp(e + 127, 0, sanitize_nans ? 254 : 255).
 *   - page P = s / cache_block starts at cache + P*page_stride_bytes; the 512
 *     value bytes go to page + (s % cache_block)*512 and the 16 scale bytes to
 *     page + cache_block*512 + (s % cache_block)*16.
 *
 * latent_bf16       bf16 [num_tokens, row_stride_elems], 512 used
 * positions         int64 [num_tokens]
 * cos_sin           float32 [cos_sin_rows, cos_stride], 32 cos then 32 sin
 * cos_stride        >= 64, multiple of 4
 * cache             uint8, num_pages pages of page_stride_bytes
 * cache_slots       int64 [num_tokens]
 * cache_block       >= 1 slots per page
 * page_stride_bytes >= cache_block*528, multiple of 16
 * compress_ratio    >= 1
 * sanitize_nans     0 or 1
 */
int rope_quant_insert_mxfp8(const void* latent_bf16, int64_t num_tokens, int64_t row_stride_elems,
                            const int64_t* positions, const float* cos_sin, int64_t cos_stride,
                            int64_t cos_sin_rows, uint8_t* cache, const int64_t* cache_slots,
                            int64_t num_pages, int64_t cache_block, int64_t page_stride_bytes,
                            int32_t compress_ratio, int32_t sanitize_nans, cudaStream_t stream);

/*
 * rope_quant_insert_nvfp4 — V4.1 288-byte NVFP4 record: GPT-J RoPE, then E2M1
 * with one E4M3 scale per 16 values. [v41] _rope_quant_insert_nvfp4_kernel.
 *
 * Gates, rotation and sanitising as rope_quant_insert_mxfp8. Per tile of 16:
 * amax = largest |x| ignoring NaN; sc = E4M3(clamp(amax * (1/6.f), 2**-9,
 * 448)) rounded to nearest even; each value becomes the E2M1 code (same rule
 * as mxfp4_mla_store) of the correctly rounded binary32 quotient x / sc. Codes
 * pack two per byte, even element in the low nibble: 256 code bytes at
 * page + (s % cache_block)*256, then the 32 E4M3 scale bytes at
 * page + cache_block*256 + (s % cache_block)*32.
 * page_stride_bytes must be >= cache_block*288 and a multiple of 16.
 */
int rope_quant_insert_nvfp4(const void* latent_bf16, int64_t num_tokens, int64_t row_stride_elems,
                            const int64_t* positions, const float* cos_sin, int64_t cos_stride,
                            int64_t cos_sin_rows, uint8_t* cache, const int64_t* cache_slots,
                            int64_t num_pages, int64_t cache_block, int64_t page_stride_bytes,
                            int32_t compress_ratio, int32_t sanitize_nans, cudaStream_t stream);

/*
 * rope_quant_insert_v4 — the V4 584-byte record: GPT-J RoPE, then 448 E4M3
 * values in seven tiles of 64 and 64 bf16 rotary values. [v41]
 * rope_quant_insert (docstring: 576 value bytes, eight UE8M0 scale bytes of
 * which one is a zero pad; the kernel itself is not printed).
 *
 * Gates, rotation and sanitising as rope_quant_insert_mxfp8. Elements
 * 0..447 form tiles g = 0..6 of 64 quantized by the MXFP8 rule of
 * rope_quant_insert_mxfp8 (1e-4 amax floor, scale byte capped at 254 when
 * sanitising, 255 otherwise); elements 448..511 (the rotated pairs) are
 * stored as bf16, nearest even, every NaN as 0x7FC0. Page P = s / cache_block
 * at cache + P*page_stride_bytes: value bytes at page + (s % cache_block)*576
 * ([448 E4M3 | 64 bf16 little-endian]), scale bytes at
 * page + cache_block*576 + (s % cache_block)*8 (bytes 0..6 the tiles', byte 7
 * always 0).
 * page_stride_bytes must be >= cache_block*584 and a multiple of 16; other
 * arguments as rope_quant_insert_mxfp8.
 */
int rope_quant_insert_v4(const void* latent_bf16, int64_t num_tokens, int64_t row_stride_elems,
                         const int64_t* positions, const float* cos_sin, int64_t cos_stride,
                         int64_t cos_sin_rows, uint8_t* cache, const int64_t* cache_slots,
                         int64_t num_pages, int64_t cache_block, int64_t page_stride_bytes,
                         int32_t compress_ratio, int32_t sanitize_nans, cudaStream_t stream);

/*
 * rope_plain_insert — a plain [448 NoPE | 64 RoPE] row of bf16, or of E4M3
 * with a per-tensor scale, for readers that take unquantized rows. [v41]
 * rope_quant_insert (docstring: bfloat16 and float8_e4m3fn caches of shape
 * [pages, CACHE_BLOCK, 512] with their own strides; the kernel is not
 * printed).
 *
 * Gates and table row as rope_quant_insert_mxfp8 (no sanitising). Rotary
 * pairs i = 224..255 (elements 448..511) are rotated in binary32 as there.
 *   fp8 == 0: elements 0..447 are the latent's bf16 patterns copied bit for
 *             bit; 448..511 are the rotated values rounded to bf16 (nearest
 *             even, every NaN as 0x7FC0).
 *   fp8 == 1: every element x (the latent's value, or the rotated value)
 *             becomes E4M3(clamp(RN(x / fp8_scale), -448, 448)), nearest
 *             even, NaN -> 0x7F.
 * Element j of slot s sits at element
 *   (s / cache_block)*page_stride_elems + (s % cache_block)*slot_stride_elems + j
 * of `cache` (2-byte elements for bf16, 1-byte for fp8).
 *
 * cache              bf16 or E4M3, 16-byte aligned
 * page_stride_elems  multiple of 8, >= (cache_block-1)*slot_stride_elems + 512
 * slot_stride_elems  multiple of 8, >= 512
 * fp8                0 (bf16 cache) or 1 (E4M3 cache)
 * fp8_scale          fp8 == 1 only: finite and > 0 (the dequantizing factor)
 * Other arguments as rope_quant_insert_mxfp8.
 */
int rope_plain_insert(const void* latent_bf16, int64_t num_tokens, int64_t row_stride_elems,
                      const int64_t* positions, const float* cos_sin, int64_t cos_stride,
                      int64_t cos_sin_rows, void* cache, const int64_t* cache_slots,
                      int64_t num_pages, int64_t cache_block, int64_t page_stride_elems,
                      int64_t slot_stride_elems, int32_t compress_ratio, int32_t fp8,
                      float fp8_scale, cudaStream_t stream);

/* How rope_plain_insert forms the E4M3 code of RN(x / fp8_scale) for an fp8
 * cache at this scale (a query of this library; the pages have no
 * counterpart). The codes are those of the correctly rounded quotient in
 * every mode; only the arithmetic differs:
 *   0  every value by a correctly rounded division;
 *   1  the bf16 NoPE values by RN(x*yh + RN(x*yl)), yh = RD(1/scale) and
 *      yl = RN((1 - scale*yh) * yh), because an exhaustive host check found
 *      that rule giving the division's code for all 65,536 bf16 patterns at
 *      this scale; the binary32 rotary values by division;
 *   2  scale a power of two with a normal reciprocal: every value by
 *      RN(x * (1/scale)), the same rounding of the same exact quotient.
 * The check (65,536 host iterations on the calling thread) runs once per
 * distinct scale: the answers for the last 8 distinct scales are kept, so
 * up to 8 layers with different scales each pay it once. KVQ_EINVAL unless
 * 0 < fp8_scale <= 3e38. Host-only: launches nothing. */
int kvq_plain_fp8_quotient_mode(float fp8_scale);

/* Number of those exhaustive host checks run so far in this process (by
 * kvq_plain_fp8_quotient_mode or rope_plain_insert). A diagnostic of this
 * library; the pages have no counterpart. */
int64_t kvq_plain_fp8_checks_run(void);

/*
 * save_ring_rows — store the compressor's fp32 [kv | score] rows of 1024
 * values into their slots of the paged ring state. [v41] save_ring_rows.
 *
 * For each row t with s = slot_mapping[t]: if 0 <= s < num_blocks*state_block
 * the 1024 floats at rows + t*row_stride_elems are copied bit for bit to
 *   state + (s / state_block)*state_stride_elems + (s % state_block)*state_row_stride_elems;
 * otherwise (-1, or outside the state) the row is skipped.
 *
 * rows                    fp32 [num_rows, row_stride_elems], 16-byte aligned
 * row_stride_elems        >= 1024, multiple of 4
 * slot_mapping            int64 [num_rows]
 * state                   fp32, 16-byte aligned
 * num_blocks, state_block >= 1
 * state_row_stride_elems  >= 1024, multiple of 4
 * state_stride_elems      multiple of 4,
 *                         >= (state_block-1)*state_row_stride_elems + 1024
 */
int save_ring_rows(const float* rows, int64_t num_rows, int64_t row_stride_elems,
                   const int64_t* slot_mapping, float* state, int64_t num_blocks,
                   int64_t state_block, int64_t state_stride_elems,
                   int64_t state_row_stride_elems, cudaStream_t stream);

/*
 * fused_save_compress_norm — pool each closed group of compressor rows into
 * an RMS-normalised bf16 latent, and keep the ring rows the next chunk needs.
 * [v41] fused_save_compress_norm (docstring and Args; its kernel is not
 * printed, so the pooling below is this library's reading).
 *
 * A group is compress_ratio (R, 1 or 2) consecutive positions and closes at
 * the token t with position p >= 0, (p + 1) % R == 0 and slot s =
 * slot_mapping[t] >= 0. Only closing tokens write latent row t.
 *   R = 1: kv_score rows are 512 kv values; pooled = the row.
 *   R = 2: rows are [512 kv | 512 score]. Token t (request k =
 *          token_to_req_indices[t], 0 <= k < num_reqs, with
 *          query_start_loc[k] <= t < query_start_loc[k+1] and
 *          s < num_blocks*capacity; otherwise skipped) closes the group
 *          (predecessor, t): the predecessor is row t-1 if t is not its
 *          chunk's first token; else prev_rows[prev_row_indices[k]] when
 *          prev_rows is given and that index is >= 0 (an index >=
 *          num_prev_rows skips the group); else the ring row
 *          (p - 1) % capacity of block s / capacity. Per channel d:
 *            m = max(s0[d], s1[d]),  e_i = exp(s_i[d] - m),
 *            pooled[d] = (e0*kv0[d] + e1*kv1[d]) / (e0 + e1).
 *          After the groups, unless prev_rows is given, each request's
 *          last min(capacity, chunk length) tokens with a slot in
 *          [0, num_blocks*capacity) are copied (1024 floats, bit for bit)
 *          to ring row s % capacity of block s / capacity. Ring rows are
 *          read as they were before the call.
 *   latent[t][d] = bf16(pooled[d] * w[d] / sqrt(mean(pooled^2) + eps)),
 *   computed in fp32 (exp by expf, correctly rounded sqrt, reciprocal and
 *   division, the final bf16 rounding to nearest even): |latent - exact| <=
 *   2^-7 |exact| + 2^-18 * r * |w[d]| * sum_i w_i |kv_i[d]| (r the exact
 *   1/sqrt(mean + eps)). A row whose pooled values overflow binary32 when
 *   squared (|x| >= 2^63) is outside that bound.
 *
 * kv_score               fp32 [num_tokens, row_stride_elems], 512*R used,
 *                        16-byte aligned; row_stride_elems multiple of 4
 * positions, slot_mapping int64 [num_tokens]
 * query_start_loc        R = 2: int64 [num_reqs + 1], non-decreasing; a
 *                        chunk is cut to [0, num_tokens) (a start below 0
 *                        reads as 0, an end past num_tokens as num_tokens)
 * token_to_req_indices   R = 2: int64 [num_tokens]
 * state                  R = 2: fp32 [num_blocks, capacity, >= 1024], block
 *                        stride state_stride_elems, row stride
 *                        state_row_stride_elems (multiples of 4, rows >= 1024
 *                        apart, blocks not overlapping); each request owns
 *                        its block (two requests sharing one race)
 * weight_bf16            bf16 [512], 8-byte aligned; eps finite, >= 0
 * prev_rows              R = 2, optional: fp32 [num_prev_rows, >= 1024],
 *                        row stride prev_row_stride_elems (multiple of 4);
 *                        prev_row_indices int64 [num_reqs] (both or neither)
 * latent_out_bf16        bf16 [num_tokens, out_row_stride_elems] (>= 512,
 *                        multiple of 8), 16-byte aligned; rows of tokens
 *                        that close no group are not written
 * For R = 1 the request, ring and prev_rows arguments are ignored.
 */
int fused_save_compress_norm(const float* kv_score, int64_t num_tokens, int64_t row_stride_elems,
                             const int64_t* positions, const int64_t* slot_mapping,
                             int32_t compress_ratio, const int64_t* query_start_loc,
                             const int64_t* token_to_req_indices, int64_t num_reqs, float* state,
                             int64_t num_blocks, int64_t capacity, int64_t state_stride_elems,
                             int64_t state_row_stride_elems, const void* weight_bf16, float eps,
                             const float* prev_rows, int64_t num_prev_rows,
                             int64_t prev_row_stride_elems, const int64_t* prev_row_indices,
                             void* latent_out_bf16, int64_t out_row_stride_elems,
                             cudaStream_t stream);

/*
 * mxfp4_mla_gather_dequant — read packed MXFP4 rows back to bf16.
 * [pr] Details (read path: gathered rows are unpacked to bf16 before use);
 * [pr] Claims (attention over the packed cache equals attention over these
 * dequantized values stored as bf16).
 *
 * For each k in [0, num_indices) with s = indices[k]: if 0 <= s <
 * num_blocks*block_size, the 272-byte row of slot s (addressed as in
 * mxfp4_mla_store) becomes 512 bf16 values
 *   out[k*out_row_stride_elems + j] = E2M1(code_j) * 2**(scale_byte - 127),
 * exact in bf16 (byte 254 with magnitude >= 2 gives +-inf; byte 255, the
 * E8M0 NaN, gives 0x7FC0 for the whole group). Otherwise (a -1 pad, or an
 * index outside the cache) the output row is 512 x +0.0.
 *
 * latent_dim must be 512; out_row_stride_elems >= 512, multiple of 8.
 */
int mxfp4_mla_gather_dequant(const uint8_t* cache, int64_t num_blocks, int64_t block_size,
                             int64_t block_stride_rows, int64_t latent_dim, const int64_t* indices,
                             int64_t num_indices, void* out_bf16, int64_t out_row_stride_elems,
                             cudaStream_t stream);

/*
 * mxfp4_mla_sparse_attention — sparse MLA decode attention computed directly
 * on the packed MXFP4 cache. [pr] Details (read path: the top-k rows of each
 * query are gathered, unpacked to bf16 and feed both dots, q.k and p.v);
 * [pr] Claims (attention over the packed cache equals attention over the
 * dequantized bf16 values). For the rope-free latent a token's key and value
 * are the same 512-wide row.
 *
 * For query n and head h (h < num_heads), over the valid indices j of row n
 * of `indices` (0 <= s < num_blocks*block_size; pads and out-of-range
 * entries are dropped, repeats count as separate entries):
 *   s_j   = sm_scale * sum_d q[n,h,d] * k_j[d],   k_j = the dequantized row
 *   out[n,h,:] = sum_j softmax(s)_j * k_j          (bf16)
 *   lse[n,h]   = log(sum_j exp(s_j))               (natural log, fp32)
 * A query with no valid index gets out = 0 and lse = -inf.
 * Arithmetic: bf16 inputs, fp32 accumulation on the tensor cores, fp32
 * softmax with exp2, probabilities rounded to bf16 for the p.v product, the
 * output rounded to bf16 once: |out - exact| is within about 2**-8 of
 * sum_j softmax(s)_j |k_j[d]| plus the final bf16 rounding. Range: the
 * softmax rescales its output accumulator only when a head's running max
 * grows by more than 32 (log2 units), so the unnormalised fp32 sums reach
 * (number of valid keys) x 2**32 x max|k|: the result is exact in the sense
 * above while that stays below 2**128: for 2048 keys, |k| < 2**85, which
 * every row whose scale bytes are at most 209 meets (a dequantized value is
 * at most 6 x 2**(scale byte - 127)).
 *
 * q_bf16           bf16; head h of query n at element
 *                  n*q_query_stride + h*q_head_stride (both multiples of 8,
 *                  q_head_stride >= 512), 16-byte aligned base
 * num_queries      >= 0; num_heads in [1, 128]
 * cache            as mxfp4_mla_store (272-byte rows, block stride in rows)
 * indices          int64 [num_queries, topk], row-major; topk >= 0
 * sm_scale         finite, >= 0
 * out_bf16         bf16; head h of query n at element
 *                  n*out_query_stride + h*out_head_stride (multiples of 8,
 *                  out_head_stride >= 512), 16-byte aligned base
 * lse              fp32 [num_queries, num_heads] or NULL
 * status           device int32 or NULL: set to a nonzero value if an
 *                  internal wait of the kernel timed out (the output is then
 *                  undefined); never written otherwise. Without a status
 *                  word such a timeout is reported nowhere and the output
 *                  is undefined: pass one to be told.
 * workspace        device memory of at least workspace_bytes >=
 *                  mxfp4_mla_sparse_attention_workspace_size(num_queries,
 *                  num_heads, topk) bytes, 256-byte aligned, or NULL.
 *                  With a workspace, when there are too few (query, value
 *                  half) units to fill the SMs, every unit's key tiles are
 *                  cut into equal chunks of at least four 32-key tiles, one
 *                  CTA each, so that the grid fills the SMs (the split-K of
 *                  the read path [pr]: a ragged sparse-attention kernel plus
 *                  a split-K partial kernel): each chunk's output
 *                  normalised by its own softmax sum (bf16, a partial) and
 *                  that sum's log-sum-exp are written there and merged by a
 *                  second kernel launched on the same stream (a
 *                  programmatic dependent launch: it overlaps the first
 *                  grid's tail and waits for all of it). A partial's
 *                  rounding adds at most 2**-9 of the softmax-weighted
 *                  magnitudes to the bound above. Its contents
 *                  need no initialisation and are garbage afterwards; two
 *                  calls in flight at once must not share it. Without one,
 *                  or when the units already fill the SMs, one CTA takes
 *                  each unit whole (no second kernel). Both give results
 *                  within the bound above; they may differ in the last bits.
 *                  KVQ_EINVAL if the workspace is too small or misaligned.
 * The library allocates nothing and keeps no pointer after the call.
 */
int mxfp4_mla_sparse_attention(const void* q_bf16, int64_t num_queries, int64_t num_heads,
                               int64_t q_query_stride, int64_t q_head_stride,
                               const uint8_t* cache, int64_t num_blocks, int64_t block_size,
                               int64_t block_stride_rows, const int64_t* indices, int64_t topk,
                               float sm_scale, void* out_bf16, int64_t out_query_stride,
                               int64_t out_head_stride, float* lse, int32_t* status,
                               void* workspace, int64_t workspace_bytes,
                               cudaStream_t stream);

/*
 * mxfp4_mla_sparse_attention_ragged — the same attention for ragged index
 * runs, as sparse prefill produces them: [pr] Details, read path (one
 * sparse-attention kernel serves sparse prefill and decode). Query n attends
 * over indices[key_offsets[n] .. key_offsets[n + 1]) of one flat int64
 * array instead of a padded [num_queries, topk] row; the runs may have any
 * lengths, including 0 (out = 0, lse = -inf).
 *
 * indices      int64 [num_indices], 8-byte aligned (-1 entries and indices
 *              outside the cache are dropped, as above)
 * key_offsets  int64 [num_queries + 1] in device memory, 8-byte aligned:
 *              query n's run starts at key_offsets[n] and ends at
 *              key_offsets[n + 1]; each bound is clamped to [0, num_indices]
 *              and an end below its start gives an empty run, so no offset
 *              makes the kernel read outside `indices`
 * Other arguments, results, arithmetic and errors as
 * mxfp4_mla_sparse_attention without a workspace: one CTA per (query, value
 * half); the number of key tiles of each CTA comes from its run.
 */
int mxfp4_mla_sparse_attention_ragged(const void* q_bf16, int64_t num_queries, int64_t num_heads,
                                      int64_t q_query_stride, int64_t q_head_stride,
                                      const uint8_t* cache, int64_t num_blocks,
                                      int64_t block_size, int64_t block_stride_rows,
                                      const int64_t* indices, int64_t num_indices,
                                      const int64_t* key_offsets, float sm_scale, void* out_bf16,
                                      int64_t out_query_stride, int64_t out_head_stride,
                                      float* lse, int32_t* status, cudaStream_t stream);

/*
 * mxfp4_mla_sparse_attention_workspace_size — bytes of workspace that
 * mxfp4_mla_sparse_attention needs to split these shapes over the current
 * device's SMs: CTAs x num_heads x (256 x 2 + 4), CTAs = units x chunks with
 * units = 2 x num_queries, chunks = min(floor(SMs / units),
 * floor(ceil(topk / 32) / 4)) reduced so that no chunk is empty; 0 when
 * nothing is split (chunks below 2: the units fill the SMs, or topk is
 * short), KVQ_EINVAL for shapes the attention rejects.
 * No page counterpart: a host query of this library.
 */
int64_t mxfp4_mla_sparse_attention_workspace_size(int64_t num_queries, int64_t num_heads,
                                                  int64_t topk);

/*
 * mxfp4_mla_sparse_attention_noalloc — mxfp4_mla_sparse_attention with the
 * split schedule's scratch taken from an array inside this library, for
 * callers that must not allocate device memory: code embedded in a host
 * framework that owns all device memory through its own pool and passes no
 * allocator down (memory allocated behind its back is neither counted nor
 * limited by it), and latency-critical loops that cannot afford cudaMalloc,
 * which may synchronise the device. The pages have no counterpart: this is a
 * convenience of this library. The caller still passes every input and
 * output; arguments, layouts, results and errors are those of
 * mxfp4_mla_sparse_attention with a workspace, plus:
 *   - The scratch is one 40 MiB (41,943,040-byte) __device__ array, enough
 *     for 128 heads split over up to 635 SMs. Every GPU that loads the
 *     library's attention code holds it until the process exits.
 *   - Shapes whose split schedule needs more than that (see
 *     mxfp4_mla_sparse_attention_workspace_size) return KVQ_ESCRATCH and
 *     launch nothing.
 *   - The first call on a device looks the array's device address up
 *     (cudaGetSymbolAddress, with that device current) and keeps it; make
 *     that first call before any stream capture on the device.
 *   - Nothing in the array needs to start at zero. Every call shares it and
 *     it keeps the last call's contents: calls whose kernels may overlap on
 *     the GPU (other streams, other host threads, one device) race on it,
 *     and the caller must order them.
 */
int mxfp4_mla_sparse_attention_noalloc(const void* q_bf16, int64_t num_queries,
                                       int64_t num_heads, int64_t q_query_stride,
                                       int64_t q_head_stride, const uint8_t* cache,
                                       int64_t num_blocks, int64_t block_size,
                                       int64_t block_stride_rows, const int64_t* indices,
                                       int64_t topk, float sm_scale, void* out_bf16,
                                       int64_t out_query_stride, int64_t out_head_stride,
                                       float* lse, int32_t* status, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* KVQ_H */
