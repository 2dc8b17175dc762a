// rope_insert.cu — rope_quant_insert_mxfp8 / rope_quant_insert_nvfp4: the
// V4.1 compressed-cache inserts. GPT-J RoPE on the last 64 elements, then
// MXFP8 (E4M3 values, E8M0 scale per 32) or NVFP4 (E2M1 codes, E4M3 scale per
// 16) into a page layout with the scales segregated after the values.
//
// Follows "vllm.models.deepseek_v41.common.ops.fused_compress_quant_cache"
// (_rope_quant_insert_mxfp8_kernel, _rope_quant_insert_nvfp4_kernel,
// rope_quant_insert).
//
// Work decomposition mirrors the MXFP4 store: a warp owns 32 tokens at a
// time, lane i evaluates token i's gates (slot range, (pos+1) % R == 0,
// table row in range) and addresses once, a ballot lists the writers, and
// each writer row is held as lane l: elements 8l..8l+7 (half 0) and
// 256+8l..256+8l+7 (half 1). Rotary pairs 224..255 are elements 448..511,
// i.e. half 1 of lanes 24..31, which alone read the table row (lane l reads
// cos and sin 4(l-24)..4(l-24)+3 as two 16-byte loads).
//
// The pages evaluate the rotation formula on all 256 pairs, with cos 1 and
// sin 0 outside the rotary range. There it is the identity except for NaN,
// infinities and signed zeros: even' = even - odd*0 and odd' = odd + even*0.
// That is computed exactly, two elements per instruction, as one bf16x2 fma
// of the half-swapped word with (-0, +0) added to the word: the products are
// exact, and each sum is the element itself, a zero, or NaN, so no rounding
// happens and the result equals the binary32 formula bit for bit. Rotary
// pairs use the binary32 formula with every product and sum rounded
// separately (no fused multiply-add).
#include <cstdint>

#include "kvq.h"
#include "kvq_device.cuh"
#include "kvq_host.h"

namespace kvq {
namespace {

constexpr int kRopeWarps = 4;
constexpr int kRopeThreads = 32 * kRopeWarps;

struct RopeParams {
  const uint8_t* latent;  // row t at latent + t * row_pitch
  int64_t row_pitch;      // bytes
  int64_t num_tokens;
  const int64_t* positions;
  const float* cos_sin;
  int64_t cos_stride;  // floats
  int64_t cos_rows;
  uint8_t* cache;
  const int64_t* slots;
  int64_t num_slots;  // num_pages * cache_block
  int64_t cache_block;
  int64_t page_stride;  // bytes
  int64_t ratio;
};

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// (even, odd) -> (even - odd*0, odd + even*0), exactly, for one bf16x2 word.
__device__ __forceinline__ uint32_t nope_pair(uint32_t w) {
  const uint32_t swapped = prmt(w, w, 0x1032);
  uint32_t d;
  asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(swapped), "r"(0x00008000u), "r"(w));
  return d;
}

__device__ __forceinline__ void widen8(uint4 w, float f[8]) {
  f[0] = bf16_lo(w.x); f[1] = bf16_hi(w.x);
  f[2] = bf16_lo(w.y); f[3] = bf16_hi(w.y);
  f[4] = bf16_lo(w.z); f[5] = bf16_hi(w.z);
  f[6] = bf16_lo(w.w); f[7] = bf16_hi(w.w);
}

// Rotated (or identity) binary32 values of the lane's two halves.
__device__ __forceinline__ void rotate_row(uint4 x0, uint4 x1, float4 c, float4 s, int lane,
                                           float f0[8], float f1[8]) {
  x0.x = nope_pair(x0.x);
  x0.y = nope_pair(x0.y);
  x0.z = nope_pair(x0.z);
  x0.w = nope_pair(x0.w);
  widen8(x0, f0);
  if (lane < 24) {
    x1.x = nope_pair(x1.x);
    x1.y = nope_pair(x1.y);
    x1.z = nope_pair(x1.z);
    x1.w = nope_pair(x1.w);
    widen8(x1, f1);
  } else {
    float v[8];
    widen8(x1, v);
    const float cc[4] = {c.x, c.y, c.z, c.w};
    const float ss[4] = {s.x, s.y, s.z, s.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float e = v[2 * k], o = v[2 * k + 1];
      f1[2 * k] = __fsub_rn(__fmul_rn(e, cc[k]), __fmul_rn(o, ss[k]));
      f1[2 * k + 1] = __fadd_rn(__fmul_rn(o, cc[k]), __fmul_rn(e, ss[k]));
    }
  }
}

__device__ __forceinline__ void nan_to_zero(float f[8]) {
#pragma unroll
  for (int k = 0; k < 8; ++k) f[k] = (f[k] == f[k]) ? f[k] : 0.0f;
}

__device__ __forceinline__ float abs_max8(const float f[8]) {
  float m = 0.0f;  // fmaxf ignores NaN
#pragma unroll
  for (int k = 0; k < 8; ++k) m = fmaxf(m, fabsf(f[k]));
  return m;
}

// ------------------------------------------------------------------ MXFP8 ---

template <bool kSanitize>
__device__ __forceinline__ void mxfp8_half(const float f[8], uint8_t* values, uint8_t* scales,
                                           int lane) {
  float amax = abs_max8(f);
  amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
  amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 2));
  amax = fmaxf(amax, 1e-4f);
  const int e = ceil_pow2_exponent(__fmul_rn(amax, 1.0f / 448.0f));  // -22..128
  const float inv = exp2_neg(e);
  // clamp to +-448 and E4M3 rounding are exactly cvt.rn.satfinite; NaN -> 0x7F
  const uint32_t a = cvt_e4m3x2(__fmul_rn(f[0], inv), __fmul_rn(f[1], inv)) |
                     (cvt_e4m3x2(__fmul_rn(f[2], inv), __fmul_rn(f[3], inv)) << 16);
  const uint32_t b = cvt_e4m3x2(__fmul_rn(f[4], inv), __fmul_rn(f[5], inv)) |
                     (cvt_e4m3x2(__fmul_rn(f[6], inv), __fmul_rn(f[7], inv)) << 16);
  st_v2(values + 8 * lane, a, b);
  if ((lane & 3) == 0) {
    const int cap = kSanitize ? 254 : 255;
    const int enc = e + 127;  // >= 105
    st_u8(scales + (lane >> 2), (uint32_t)(enc < cap ? enc : cap));
  }
}

// ------------------------------------------------------------------ NVFP4 ---

// Positive E4M3 code (<= 0x7E) -> its exact binary32 value.
__device__ __forceinline__ float e4m3_value(uint32_t b) {
  const uint32_t ex = b >> 3, man = b & 7u;
  return ex ? __uint_as_float(((ex + 120u) << 23) | (man << 20))
            : __uint_as_float(0x3B000000u) * (float)man;  // man * 2**-9, exact
}

// Correctly rounded binary32 x / s for a tile's E4M3 scale s, given
// y = RN(1/s): the product q0 = RN(x * y) is corrected once,
// q1 = RN(q0 + (x - q0 * s) * y) with both steps fused (Markstein's
// correction). A GB300 check over every E4M3 significand and every binary32
// significand of x, both signs, found q1 == RN(x / s) in all 2**29 cases.
// Scaling x or s by powers of two scales every step exactly while all
// intermediates stay normal, which |q0| in [2**-60, 2**61) ensures for
// s in [2**-9, 448] (the remainder is then >= 2**-115); outside that range
// (and for zero, infinite or NaN q0) the IEEE division is used.
__device__ __forceinline__ float div_by_scale(float x, float s, float y) {
  const float q0 = __fmul_rn(x, y);
  const uint32_t ex = (__float_as_uint(q0) >> 23) & 0xFFu;
  if (ex - 67u > 120u) return __fdiv_rn(x, s);
  const float r = __fmaf_rn(-q0, s, x);
  return __fmaf_rn(r, y, q0);
}

// NaN in an NVFP4 record always ends as code 0 (the code rule gives NaN code
// 0, and amax ignores NaN), so sanitising changes nothing here: callers pass
// values with NaN already turned into +0.0. The +0.0 added to the quotient
// turns -0.0 (x = -0.0, or a tiny negative quotient that underflows) into
// +0.0, which the code rule also codes 0.
__device__ __forceinline__ void nvfp4_half(const float f[8], uint8_t* codes, uint8_t* scales,
                                           int lane) {
  float amax = abs_max8(f);
  amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
  float target = __fmul_rn(amax, 1.0f / 6.0f);
  target = fminf(fmaxf(target, 0.001953125f), 448.0f);
  const uint32_t sbyte = cvt_e4m3x2(target, 0.0f) & 0xFFu;
  const float s = e4m3_value(sbyte);
  const float y = __frcp_rn(s);
  float q[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) q[k] = __fadd_rn(div_by_scale(f[k], s, y), 0.0f);
  st_u32(codes + 4 * lane, cvt_e2m1x8(q[0], q[1], q[2], q[3], q[4], q[5], q[6], q[7]));
  if ((lane & 1) == 0) st_u8(scales + (lane >> 1), sbyte);
}

// ------------------------------------------------------------------ kernel ---

// Ring stage of one writer: latent row (1024 B), its table row's 32 cos and
// 32 sin (256 B), then the destination (page byte offset, slot in page).
constexpr int kRopePrefetch = 4;  // writers per warp in flight
constexpr int kRopeStages = kRopePrefetch + 1;
constexpr int kStageTable = 1024;
constexpr int kStageMeta = 1280;
constexpr int kRopeStageBytes = 1296;
constexpr size_t kRopeSmem = (size_t)kRopeWarps * kRopeStages * kRopeStageBytes;

__device__ __forceinline__ float4 lds_f4(const void* p) {
  const uint4 v = lds_v4(static_cast<const uint4*>(p));
  return make_float4(__uint_as_float(v.x), __uint_as_float(v.y), __uint_as_float(v.z),
                     __uint_as_float(v.w));
}

__device__ __forceinline__ int64_t lds_i64(const void* p) {
  int64_t r;
  const uint32_t a = (uint32_t)__cvta_generic_to_shared(p);
  asm volatile("ld.shared.s64 %0, [%1];" : "=l"(r) : "r"(a) : "memory");
  return r;
}

__device__ __forceinline__ void sts_i64x2(void* p, int64_t a, int64_t b) {
  const uint32_t d = (uint32_t)__cvta_generic_to_shared(p);
  asm volatile("st.shared.v2.s64 [%0], {%1, %2};" ::"r"(d), "l"(a), "l"(b) : "memory");
}

// The writers of a warp's token range, found 32 tokens at a time. Lane i
// evaluates token base+i (slot range, (pos+1) % R == 0, table row in range)
// and keeps its destination and table offsets; `mask` lists the writers not
// yet issued. The raw slot and position of the following window are loaded
// one window early to hide their latency.
struct WriterCursor {
  int64_t base, end;
  uint32_t mask;
  int64_t page_off, in_page, table_off;
  int64_t next_slot, next_pos;

  __device__ __forceinline__ void fetch_raw(const RopeParams& p, int64_t b, int lane) {
    next_slot = -1;
    next_pos = -1;
    if (b + lane < end) {
      next_slot = ld_once_i64(p.slots + b + lane);
      next_pos = ld_once_i64(p.positions + b + lane);
    }
  }

  __device__ __forceinline__ void open(const RopeParams& p, int lane) {
    const int64_t s = next_slot, pos = next_pos;
    page_off = -1;
    in_page = 0;
    table_off = 0;
    // pos - R >= cos_rows puts the table row past the table whatever the
    // remainder; testing it first also keeps pos + 1 from overflowing.
    if (s >= 0 && s < p.num_slots && pos >= 0 && pos - p.ratio < p.cos_rows) {
      int64_t q, r;
      divmod_pos(pos + 1, p.ratio, q, r);
      const int64_t row = pos + 1 - p.ratio;  // (pos // R) * R when R divides pos + 1
      if (r == 0 && row < p.cos_rows) {
        int64_t page;
        divmod_pos(s, p.cache_block, page, in_page);
        page_off = page * p.page_stride;
        table_off = row * p.cos_stride;
      }
    }
    mask = __ballot_sync(0xFFFFFFFFu, page_off >= 0);
    fetch_raw(p, base + 32, lane);
  }

  // Issue the next writer's copies into `stage`; false when the range is done.
  __device__ __forceinline__ bool issue_next(const RopeParams& p, uint8_t* stage, int lane) {
    while (mask == 0) {
      base += 32;
      if (base >= end) return false;
      open(p, lane);
    }
    const int src = __ffs(mask) - 1;
    mask &= mask - 1;
    const int64_t pg = __shfl_sync(0xFFFFFFFFu, page_off, src);
    const int64_t sp = __shfl_sync(0xFFFFFFFFu, in_page, src);
    const int64_t tab = __shfl_sync(0xFFFFFFFFu, table_off, src);
    const uint8_t* row = p.latent + (base + src) * p.row_pitch + 16 * lane;
    cp_async_16(stage + 16 * lane, row);
    cp_async_16(stage + 512 + 16 * lane, row + 512);
    if (lane >= 24) {
      const float* cs = p.cos_sin + tab + 4 * (lane - 24);
      cp_async_16(stage + kStageTable + 16 * (lane - 24), cs);
      cp_async_16(stage + kStageTable + 128 + 16 * (lane - 24), cs + 32);
    }
    if (lane == 0) sts_i64x2(stage + kStageMeta, pg, sp);
    return true;
  }
};

// Each warp owns a contiguous token range. The cursor issues writers into a
// per-warp shared-memory ring kRopePrefetch writers ahead of the one being
// quantized (non-writers cost no row traffic and no pipeline slot). Every
// iteration commits exactly one cp.async group, so writer c is in group c.
// __syncwarp before a refill (the stage was read by all lanes last
// iteration) and after the wait (other lanes' copies and lane 0's metadata
// become visible).
template <bool kNvfp4, bool kSanitize>
__global__ void __launch_bounds__(kRopeThreads) rope_insert_kernel(RopeParams p) {
  extern __shared__ uint4 smem[];
  const int lane = threadIdx.x & 31;
  const int warp_in_block = threadIdx.x >> 5;
  uint8_t* ring =
      reinterpret_cast<uint8_t*>(smem) + warp_in_block * (kRopeStages * kRopeStageBytes);
  const int64_t warp = (int64_t)blockIdx.x * kRopeWarps + warp_in_block;
  const int64_t num_warps = (int64_t)gridDim.x * kRopeWarps;
  WriterCursor cur;
  cur.base = p.num_tokens * warp / num_warps;
  cur.end = p.num_tokens * (warp + 1) / num_warps;
  if (cur.base >= cur.end) return;
  cur.fetch_raw(p, cur.base, lane);
  cur.open(p, lane);

  const int64_t value_bytes = kNvfp4 ? 256 : 512;
  const int64_t scale_bytes = kNvfp4 ? 32 : 16;
  int64_t issued = 0;
  bool more = true;
#pragma unroll
  for (int d = 0; d < kRopePrefetch; ++d) {
    if (more) {
      more = cur.issue_next(p, ring + (int)(issued % kRopeStages) * kRopeStageBytes, lane);
      issued += more ? 1 : 0;
    }
    cp_async_commit();
  }
  for (int64_t c = 0; c < issued; ++c) {
    __syncwarp();
    if (more) {
      more = cur.issue_next(p, ring + (int)(issued % kRopeStages) * kRopeStageBytes, lane);
      issued += more ? 1 : 0;
    }
    cp_async_commit();
    cp_async_wait<kRopePrefetch>();
    __syncwarp();
    const uint8_t* st = ring + (int)(c % kRopeStages) * kRopeStageBytes;
    const uint4 x0 = lds_v4(reinterpret_cast<const uint4*>(st + 16 * lane));
    const uint4 x1 = lds_v4(reinterpret_cast<const uint4*>(st + 512 + 16 * lane));
    float4 cs = make_float4(1.f, 1.f, 1.f, 1.f), sn = make_float4(0.f, 0.f, 0.f, 0.f);
    if (lane >= 24) {
      cs = lds_f4(st + kStageTable + 16 * (lane - 24));
      sn = lds_f4(st + kStageTable + 128 + 16 * (lane - 24));
    }
    const int64_t pg = lds_i64(st + kStageMeta);
    const int64_t slot_in_page = lds_i64(st + kStageMeta + 8);
    float f0[8], f1[8];
    rotate_row(x0, x1, cs, sn, lane, f0, f1);
    if (kSanitize || kNvfp4) {
      nan_to_zero(f0);
      nan_to_zero(f1);
    }
    uint8_t* page = p.cache + pg;
    uint8_t* values = page + slot_in_page * value_bytes;
    uint8_t* scales = page + p.cache_block * value_bytes + slot_in_page * scale_bytes;
    if (kNvfp4) {
      nvfp4_half(f0, values, scales, lane);
      nvfp4_half(f1, values + 128, scales + 16, lane);
    } else {
      mxfp8_half<kSanitize>(f0, values, scales, lane);
      mxfp8_half<kSanitize>(f1, values + 256, scales + 8, lane);
    }
  }
  cp_async_wait<0>();
}

int g_rope_occupancy[4][64];

template <bool kNvfp4, bool kSanitize>
int launch(const RopeParams& p, cudaStream_t stream) {
  auto k = rope_insert_kernel<kNvfp4, kSanitize>;
  const int64_t work_blocks = (p.num_tokens + 32 * kRopeWarps - 1) / (32 * kRopeWarps);
  const unsigned grid = grid_for(
      work_blocks,
      resident_blocks_per_sm(k, kRopeThreads, kRopeSmem, g_rope_occupancy[2 * kNvfp4 + kSanitize]));
  k<<<grid, kRopeThreads, kRopeSmem, stream>>>(p);
  return launch_status();
}

int rope_insert(bool nvfp4, const void* latent_bf16, int64_t num_tokens, int64_t row_stride_elems,
                const int64_t* positions, const float* cos_sin, int64_t cos_stride,
                int64_t cos_sin_rows, uint8_t* cache, const int64_t* cache_slots,
                int64_t num_pages, int64_t cache_block, int64_t page_stride_bytes,
                int32_t compress_ratio, int32_t sanitize_nans, cudaStream_t stream) {
  const int64_t record = nvfp4 ? kNvfp4Record : kMxfp8Record;
  if (num_tokens < 0 || row_stride_elems < kLatent || row_stride_elems % 8 != 0) return KVQ_EINVAL;
  if (cos_stride < 64 || cos_stride % 4 != 0 || cos_sin_rows < 1) return KVQ_EINVAL;
  if (num_pages < 1 || cache_block < 1 || compress_ratio < 1) return KVQ_EINVAL;
  if (sanitize_nans != 0 && sanitize_nans != 1) return KVQ_EINVAL;
  if (cache_block > INT64_MAX / record || page_stride_bytes < cache_block * record ||
      page_stride_bytes % 16 != 0)
    return KVQ_EINVAL;
  if (num_pages > INT64_MAX / page_stride_bytes || num_pages > INT64_MAX / cache_block)
    return KVQ_EINVAL;
  if (cos_sin_rows > INT64_MAX / cos_stride) return KVQ_EINVAL;
  if (num_tokens > INT64_MAX / 2 / row_stride_elems) return KVQ_EINVAL;
  if (num_tokens == 0) return KVQ_OK;
  if (!latent_bf16 || !positions || !cos_sin || !cache || !cache_slots) return KVQ_EINVAL;
  if (!aligned(latent_bf16, 16) || !aligned(cos_sin, 16) || !aligned(cache, 16) ||
      !aligned(positions, 8) || !aligned(cache_slots, 8))
    return KVQ_EINVAL;

  RopeParams p;
  p.latent = static_cast<const uint8_t*>(latent_bf16);
  p.row_pitch = row_stride_elems * 2;
  p.num_tokens = num_tokens;
  p.positions = positions;
  p.cos_sin = cos_sin;
  p.cos_stride = cos_stride;
  p.cos_rows = cos_sin_rows;
  p.cache = cache;
  p.slots = cache_slots;
  p.num_slots = num_pages * cache_block;
  p.cache_block = cache_block;
  p.page_stride = page_stride_bytes;
  p.ratio = compress_ratio;
  if (nvfp4) return sanitize_nans ? launch<true, true>(p, stream) : launch<true, false>(p, stream);
  return sanitize_nans ? launch<false, true>(p, stream) : launch<false, false>(p, stream);
}

}  // namespace
}  // namespace kvq

extern "C" int rope_quant_insert_mxfp8(const void* latent_bf16, int64_t num_tokens,
                                       int64_t row_stride_elems, const int64_t* positions,
                                       const float* cos_sin, int64_t cos_stride,
                                       int64_t cos_sin_rows, uint8_t* cache,
                                       const int64_t* cache_slots, int64_t num_pages,
                                       int64_t cache_block, int64_t page_stride_bytes,
                                       int32_t compress_ratio, int32_t sanitize_nans,
                                       cudaStream_t stream) {
  return kvq::rope_insert(false, latent_bf16, num_tokens, row_stride_elems, positions, cos_sin,
                          cos_stride, cos_sin_rows, cache, cache_slots, num_pages, cache_block,
                          page_stride_bytes, compress_ratio, sanitize_nans, stream);
}

extern "C" int rope_quant_insert_nvfp4(const void* latent_bf16, int64_t num_tokens,
                                       int64_t row_stride_elems, const int64_t* positions,
                                       const float* cos_sin, int64_t cos_stride,
                                       int64_t cos_sin_rows, uint8_t* cache,
                                       const int64_t* cache_slots, int64_t num_pages,
                                       int64_t cache_block, int64_t page_stride_bytes,
                                       int32_t compress_ratio, int32_t sanitize_nans,
                                       cudaStream_t stream) {
  return kvq::rope_insert(true, latent_bf16, num_tokens, row_stride_elems, positions, cos_sin,
                          cos_stride, cos_sin_rows, cache, cache_slots, num_pages, cache_block,
                          page_stride_bytes, compress_ratio, sanitize_nans, stream);
}
