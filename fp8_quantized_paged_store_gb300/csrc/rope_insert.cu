// rope_insert.cu — rope_quant_insert_mxfp8 / rope_quant_insert_nvfp4: the
// V4.1 compressed-cache inserts. GPT-J RoPE on the last 64 elements, then
// MXFP8 (E4M3 values, E8M0 scale per 32) or NVFP4 (E2M1 codes, E4M3 scale per
// 16) into a page layout with the scales segregated after the values.
//
// Follows "vllm.models.deepseek_v41.common.ops.fused_compress_quant_cache"
// (_rope_quant_insert_mxfp8_kernel, _rope_quant_insert_nvfp4_kernel,
// rope_quant_insert).
//
// Work decomposition: a warp owns 32 tokens at a time (grid-stride over
// chunks); lane i evaluates token i's gates (slot range, (pos+1) % R == 0,
// table row in range) and addresses once, and a ballot lists the writers, so
// non-writers cost no row traffic. Writers are taken two at a time with both
// rows' loads (and their table rows) issued before either is quantized. A
// writer row is held as lane l: elements 8l..8l+7 (half 0) and
// 256+8l..256+8l+7 (half 1), each 16-byte load of the warp covering 512
// contiguous bytes. Rotary pairs 224..255 are elements 448..511, i.e. half 1
// of lanes 24..31, which alone read the table row (lane l reads cos and sin
// 4(l-24)..4(l-24)+3 as two 16-byte loads). With at most two writers per
// warp in flight and 32 warps per SM, loads stay in flight while other warps
// compute; a shared-memory cp.async ring measured slower here, the gate and
// ballot work per window then sitting on the critical path.
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

constexpr int kRopeWarps = 8;
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

// Rotated (or identity) binary32 values of the lane's two halves. With
// kZeroNan, NaN results become +0.0 (the sanitising step): on NoPE words by a
// bf16x2 mask (the NoPE formula's result is already exact in bf16), on the
// rotary values by a binary32 select.
template <bool kZeroNan>
__device__ __forceinline__ void rotate_row(uint4 x0, uint4 x1, float4 c, float4 s, int lane,
                                           float f0[8], float f1[8]) {
  auto nope = [](uint32_t w) {
    const uint32_t r = nope_pair(w);
    return kZeroNan ? (r & bf16x2_number_mask(r)) : r;
  };
  x0.x = nope(x0.x);
  x0.y = nope(x0.y);
  x0.z = nope(x0.z);
  x0.w = nope(x0.w);
  widen8(x0, f0);
  if (lane < 24) {
    x1.x = nope(x1.x);
    x1.y = nope(x1.y);
    x1.z = nope(x1.z);
    x1.w = nope(x1.w);
    widen8(x1, f1);
  } else {
    float v[8];
    widen8(x1, v);
    const float cc[4] = {c.x, c.y, c.z, c.w};
    const float ss[4] = {s.x, s.y, s.z, s.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float e = v[2 * k], o = v[2 * k + 1];
      float re = __fsub_rn(__fmul_rn(e, cc[k]), __fmul_rn(o, ss[k]));
      float ro = __fadd_rn(__fmul_rn(o, cc[k]), __fmul_rn(e, ss[k]));
      if (kZeroNan) {
        re = (re == re) ? re : 0.0f;
        ro = (ro == ro) ? ro : 0.0f;
      }
      f1[2 * k] = re;
      f1[2 * k + 1] = ro;
    }
  }
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
// q1 = RN(q0 + (x - q0 * s) * y), both steps fused (Markstein's correction).
// A GB300 check over every E4M3 significand and every binary32 significand
// of x, both signs, found q1 == RN(x / s) in all 2**29 cases. Scaling x or s
// by powers of two scales every step exactly while all intermediates stay
// normal, which |q0| in [2**-60, 2**61) ensures for s in [2**-9, 448] (the
// remainder is then >= 2**-115). The upper bound is checked once per tile
// (amax * y < 2**61, which also excludes infinite or NaN amax); the lower
// one per value. Elsewhere (tiny, zero or infinite values) the IEEE division
// is used, followed by +0.0 to turn a -0.0 quotient into +0.0.
//
// NaN in an NVFP4 record always ends as code 0 (the code rule gives NaN code
// 0, and amax ignores NaN), so sanitising changes nothing here: callers pass
// values with NaN already turned into +0.0. The corrected quotient is never
// -0.0 (x = +-0 takes the IEEE branch), and -0.0 would be code 8 where the
// rule gives 0.
// The rare branch of the quotient, kept out of line so that the eight values
// of a tile share one copy of the division code.
__device__ __noinline__ float nvfp4_quotient_ieee(float x, float s) {
  return __fadd_rn(__fdiv_rn(x, s), 0.0f);
}

// `sy` holds (s, RN(1/s)) for every positive E4M3 code (built once per block).
__device__ __forceinline__ void nvfp4_half(const float f[8], uint8_t* codes, uint8_t* scales,
                                           int lane, const float2* sy) {
  float amax = abs_max8(f);
  amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
  float target = __fmul_rn(amax, 1.0f / 6.0f);
  target = fminf(fmaxf(target, 0.001953125f), 448.0f);
  const uint32_t sbyte = cvt_e4m3x2(target, 0.0f) & 0xFFu;  // 0x01..0x7E
  const float2 t = sy[sbyte];
  const float s = t.x, y = t.y;
  const bool tile_ok = __fmul_rn(amax, y) < 0x1p61f;
  float q[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const float q0 = __fmul_rn(f[k], y);
    if (tile_ok && fabsf(q0) >= 0x1p-60f) {
      q[k] = __fmaf_rn(__fmaf_rn(-q0, s, f[k]), y, q0);
    } else {
      q[k] = nvfp4_quotient_ieee(f[k], s);
    }
  }
  st_u32(codes + 4 * lane, cvt_e2m1x8(q[0], q[1], q[2], q[3], q[4], q[5], q[6], q[7]));
  if ((lane & 1) == 0) st_u8(scales + (lane >> 1), sbyte);
}

// ------------------------------------------------------------------ kernel ---

template <bool kNvfp4, bool kSanitize>
__global__ void __launch_bounds__(kRopeThreads) rope_insert_kernel(RopeParams p) {
  __shared__ float2 scale_table[kNvfp4 ? 128 : 1];
  if (kNvfp4) {
    if (threadIdx.x < 128) {
      const float sv = e4m3_value(threadIdx.x);
      scale_table[threadIdx.x] = make_float2(sv, __frcp_rn(sv));
    }
    __syncthreads();
  }
  const int lane = threadIdx.x & 31;
  const int64_t warp = ((int64_t)blockIdx.x * kRopeThreads + threadIdx.x) >> 5;
  const int64_t num_warps = ((int64_t)gridDim.x * kRopeThreads) >> 5;
  const int64_t value_bytes = kNvfp4 ? 256 : 512;
  const int64_t scale_bytes = kNvfp4 ? 32 : 16;

  for (int64_t base = warp * 32; base < p.num_tokens; base += num_warps * 32) {
    // Lane i: gates and addresses of token base+i.
    int64_t page_off = -1, table_off = 0;
    int64_t in_page = 0;
    if (base + lane < p.num_tokens) {
      const int64_t s = ld_once_i64(p.slots + base + lane);
      if (s >= 0 && s < p.num_slots) {
        const int64_t pos = ld_once_i64(p.positions + base + lane);
        // pos - R >= cos_rows puts the table row past the table whatever the
        // remainder; testing it first also keeps pos + 1 from overflowing.
        if (pos >= 0 && pos - p.ratio < p.cos_rows) {
          int64_t q, r;
          divmod_pos(pos + 1, p.ratio, q, r);
          // (pos+1) % R == 0 makes (pos // R) * R equal to pos + 1 - R.
          const int64_t row = pos + 1 - p.ratio;
          if (r == 0 && row < p.cos_rows) {
            int64_t page;
            divmod_pos(s, p.cache_block, page, in_page);
            page_off = page * p.page_stride;
            table_off = row * p.cos_stride;
          }
        }
      }
    }
    uint32_t todo = __ballot_sync(0xFFFFFFFFu, page_off >= 0);
    while (todo) {
      const int ia = __ffs(todo) - 1;
      todo &= todo - 1;
      const int ib = todo ? __ffs(todo) - 1 : -1;
      if (todo) todo &= todo - 1;
      const uint8_t* sa = p.latent + (base + ia) * p.row_pitch;
      const uint4 xa0 = ld_once_v4(sa + 16 * lane);
      const uint4 xa1 = ld_once_v4(sa + 512 + 16 * lane);
      uint4 xb0 = make_uint4(0, 0, 0, 0), xb1 = xb0;
      if (ib >= 0) {
        const uint8_t* sb = p.latent + (base + ib) * p.row_pitch;
        xb0 = ld_once_v4(sb + 16 * lane);
        xb1 = ld_once_v4(sb + 512 + 16 * lane);
      }
      const int64_t ta = __shfl_sync(0xFFFFFFFFu, table_off, ia);
      const int64_t tb = __shfl_sync(0xFFFFFFFFu, table_off, ib < 0 ? ia : ib);
      float4 ca = make_float4(1.f, 1.f, 1.f, 1.f), sna = make_float4(0.f, 0.f, 0.f, 0.f);
      float4 cb = ca, snb = sna;
      if (lane >= 24) {
        const float* csa = p.cos_sin + ta + 4 * (lane - 24);
        ca = ld_f4(csa);
        sna = ld_f4(csa + 32);
        if (ib >= 0) {
          const float* csb = p.cos_sin + tb + 4 * (lane - 24);
          cb = ld_f4(csb);
          snb = ld_f4(csb + 32);
        }
      }
#pragma unroll
      for (int w = 0; w < 2; ++w) {
        const int i = w ? ib : ia;
        if (i < 0) break;
        const int64_t pg = __shfl_sync(0xFFFFFFFFu, page_off, i);
        const int64_t slot_in_page = __shfl_sync(0xFFFFFFFFu, in_page, i);
        float f0[8], f1[8];
        rotate_row<kSanitize || kNvfp4>(w ? xb0 : xa0, w ? xb1 : xa1, w ? cb : ca, w ? snb : sna,
                                         lane, f0, f1);
        uint8_t* page = p.cache + pg;
        uint8_t* values = page + slot_in_page * value_bytes;
        uint8_t* scales = page + p.cache_block * value_bytes + slot_in_page * scale_bytes;
        if (kNvfp4) {
          nvfp4_half(f0, values, scales, lane, scale_table);
          nvfp4_half(f1, values + 128, scales + 16, lane, scale_table);
        } else {
          mxfp8_half<kSanitize>(f0, values, scales, lane);
          mxfp8_half<kSanitize>(f1, values + 256, scales + 8, lane);
        }
      }
    }
  }
}

int g_rope_occupancy[4][64];

template <bool kNvfp4, bool kSanitize>
int launch(const RopeParams& p, cudaStream_t stream) {
  auto k = rope_insert_kernel<kNvfp4, kSanitize>;
  const int64_t chunks = (p.num_tokens + 31) / 32;
  const int64_t work_blocks = (chunks + kRopeWarps - 1) / kRopeWarps;
  const unsigned grid = grid_for(
      work_blocks, resident_blocks_per_sm(k, kRopeThreads, 0, g_rope_occupancy[2 * kNvfp4 + kSanitize]));
  k<<<grid, kRopeThreads, 0, stream>>>(p);
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
