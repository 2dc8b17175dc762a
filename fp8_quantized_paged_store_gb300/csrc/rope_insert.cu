// rope_insert.cu — rope_quant_insert_mxfp8 / rope_quant_insert_nvfp4: the
// V4.1 compressed-cache inserts. GPT-J RoPE on the last 64 elements, then
// MXFP8 (E4M3 values, E8M0 scale per 32) or NVFP4 (E2M1 codes, E4M3 scale per
// 16) into a page layout with the scales segregated after the values.
//
// Follows "vllm.models.deepseek_v41.common.ops.fused_compress_quant_cache"
// (_rope_quant_insert_mxfp8_kernel, _rope_quant_insert_nvfp4_kernel,
// rope_quant_insert).
//
// Work decomposition (both kernels): a warp owns 32 tokens at a time
// (grid-stride over chunks); lane i evaluates token i's gates (slot range,
// (pos+1) % R == 0, table row in range) and addresses once, and a ballot lists
// the writers, so non-writers cost no row traffic. Writers are taken two at a
// time with both rows' loads (and their table rows) issued before either is
// quantized: with two writers in flight per warp and 40 warps per SM, loads
// stay in flight while other warps compute (a shared-memory cp.async ring
// measured slower here, the gate and ballot work per window then sitting on
// the critical path). A row is held as lane l: elements 8l..8l+7 (half 0) and
// 256+8l..256+8l+7 (half 1), each 16-byte load of the warp covering 512
// contiguous bytes. Rotary pairs 224..255 are elements 448..511.
//
// MXFP8: the rotary elements are half 1 of lanes 24..31, which alone read the
// table row (lane l: cos and sin 4(l-24)..4(l-24)+3, two 16-byte loads).
//
// NVFP4: lanes 0..23 load half 1 as above, and every lane j loads rotary pair
// j (4 bytes) with its own cos and sin, so the rotation and the exact quotient
// of the 64 rotated values are spread over the whole warp instead of 8 lanes.
// The other 448 values are bf16 numbers and take the cheaper exact code rule
// of nvfp4_code_value (two fused products, no ALU work).
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

// Per E4M3 byte b (0..127), built once per block: s = value(b), y = RN(1/s)
// for the corrected quotient, and the two-term reciprocal yh = RD(1/s),
// yl = RN((1 - s*yh) * yh) >= 0 for nvfp4_code_value.
struct ScaleEntry {
  float s, y, yh, yl;
};

__device__ __forceinline__ ScaleEntry make_scale_entry(uint32_t b) {
  ScaleEntry e;
  e.s = e4m3_value(b);
  e.y = __frcp_rn(e.s);
  e.yh = __frcp_rd(e.s);
  e.yl = __fmul_rn(__fmaf_rn(-e.s, e.yh, 1.0f), e.yh);  // 1 - s*yh is exact
  return e;
}

// The NVFP4 tile scale from the tile's |amax| (NaN-free): the E4M3 byte of
// clamp(amax * RN(1/6), 2**-9, 448) and its table entry.
__device__ __forceinline__ uint32_t nvfp4_scale(float amax, const float4* table, ScaleEntry& e) {
  float target = __fmul_rn(amax, 1.0f / 6.0f);
  target = fminf(fmaxf(target, 0.001953125f), 448.0f);
  const uint32_t sbyte = cvt_e4m3x2(target, 0.0f) & 0xFFu;  // 0x01..0x7E
  const float4 t = table[sbyte];
  e.s = t.x;
  e.y = t.y;
  e.yh = t.z;
  e.yl = t.w;
  return sbyte;
}

// Code-deciding stand-in for RN(x / s) when x is a bf16 number other than
// -0 and NaN (at most 8 significant bits): RN(x*yh + RN(x*yl)).
// A midpoint M between neighbouring E2M1 values (0.25, 0.75, ..., 5) has at
// most 3 significant bits and s at most 4, so M*s is a bf16 number: either
// x = M*s and x/s is M exactly, or x differs from M*s by at least one bf16
// step, putting x/s at least 2**-9 (relative) away from every midpoint.
// yh + yl equals 1/s to about 2**-47 (relative), so the fused sum is x/s to
// about 2**-45 before its one rounding: an exact midpoint rounds to M itself
// and every other value stays on its side of every midpoint. The sign is
// x's (|x/s| >= 2**-142 for a nonzero bf16 x, so RN(x/s) is never zero), and
// +0 gives +0. yh is rounded down so that yl >= 0: an infinite x (only in a
// tile with infinite amax, s = 448, yl > 0) gives x*yh and x*yl of one sign
// and an infinite quotient rather than NaN. An exhaustive check over all 126
// positive scales and every non-NaN bf16 x (both infinities with s = 448)
// found the E2M1 codes equal to those of RN(x / s) everywhere.
__device__ __forceinline__ float nvfp4_code_value(float x, const ScaleEntry& e) {
  return __fmaf_rn(x, e.yh, __fmul_rn(x, e.yl));
}

// Correctly rounded binary32 x / s for a tile's E4M3 scale s, given
// y = RN(1/s): the product q0 = RN(x * y) is corrected once,
// q1 = RN(q0 + (x - q0 * s) * y), both steps fused (Markstein's correction).
// A GB300 check over every E4M3 significand and every binary32 significand
// of x, both signs, found q1 == RN(x / s) in all 2**29 cases. Scaling x or s
// by powers of two scales every step exactly while all intermediates stay
// normal, which |q0| in [2**-60, 2**61) ensures for s in [2**-9, 448] (the
// remainder is then >= 2**-115). x = +-0 gives q0 = +-0 and q1 = +0. Values
// outside that range (tiny nonzero, or a tile whose amax * y reaches 2**61,
// which includes infinite amax) make the whole warp take the IEEE division,
// followed by +0.0 to turn a -0.0 quotient into +0.0.
__device__ __noinline__ float nvfp4_quotient_ieee(float x, float s) {
  return __fadd_rn(__fdiv_rn(x, s), 0.0f);
}

__device__ __forceinline__ bool markstein_ok(float x, float q0) {
  return fabsf(q0) >= 0x1p-60f || x == 0.0f;
}

// Eight bf16-exact values of one NoPE half (four bf16x2 words): the NoPE
// formula, NaN and -0.0 to +0.0 (both encode as code 0 and NaN never raises
// the amax), the tile amax over this lane and its partner, then the codes by
// nvfp4_code_value. Lanes with `store` false compute but write nothing.
__device__ __forceinline__ void nvfp4_nope_half(uint4 w, uint8_t* codes, uint8_t* scales, int lane,
                                                const float4* table, bool store) {
  auto clean = [](uint32_t v) {
    const uint32_t r = nope_pair(v);
    return r & bf16x2_nonzero_number_mask(r);
  };
  w.x = clean(w.x);
  w.y = clean(w.y);
  w.z = clean(w.z);
  w.w = clean(w.w);
  const uint32_t m = bf16x2_maxabs(bf16x2_maxabs(w.x, w.y), bf16x2_maxabs(w.z, w.w));
  float amax = fmaxf(fabsf(bf16_lo(m)), fabsf(bf16_hi(m)));
  amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
  ScaleEntry e;
  const uint32_t sbyte = nvfp4_scale(amax, table, e);
  const uint32_t c = cvt_e2m1x8(
      nvfp4_code_value(bf16_lo(w.x), e), nvfp4_code_value(bf16_hi(w.x), e),
      nvfp4_code_value(bf16_lo(w.y), e), nvfp4_code_value(bf16_hi(w.y), e),
      nvfp4_code_value(bf16_lo(w.z), e), nvfp4_code_value(bf16_hi(w.z), e),
      nvfp4_code_value(bf16_lo(w.w), e), nvfp4_code_value(bf16_hi(w.w), e));
  if (store) {
    st_u32(codes + 4 * lane, c);
    if ((lane & 1) == 0) st_u8(scales + (lane >> 1), sbyte);
  }
}

// Rotary pair 224 + lane (elements 448 + 2*lane and 449 + 2*lane) with its
// cos and sin: the binary32 rotation, NaN to +0.0, the amax of tile
// 28 + lane/8 over its eight lanes, and the two codes by the corrected
// quotient. `codes` and `scales` point at the record's first code and scale
// byte.
__device__ __forceinline__ void nvfp4_rotary_pair(uint32_t xr, float c, float sn, uint8_t* codes,
                                                  uint8_t* scales, int lane, const float4* table) {
  const float e = bf16_lo(xr), o = bf16_hi(xr);
  float re = __fsub_rn(__fmul_rn(e, c), __fmul_rn(o, sn));
  float ro = __fadd_rn(__fmul_rn(o, c), __fmul_rn(e, sn));
  re = (re == re) ? re : 0.0f;
  ro = (ro == ro) ? ro : 0.0f;
  float amax = fmaxf(fabsf(re), fabsf(ro));
  amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
  amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 2));
  amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 4));
  ScaleEntry sc;
  const uint32_t sbyte = nvfp4_scale(amax, table, sc);
  const float s = sc.s, y = sc.y;
  const float qe0 = __fmul_rn(re, y), qo0 = __fmul_rn(ro, y);
  const bool ok = __fmul_rn(amax, y) < 0x1p61f && markstein_ok(re, qe0) && markstein_ok(ro, qo0);
  float qe, qo;
  if (__all_sync(0xFFFFFFFFu, ok)) {
    qe = __fmaf_rn(__fmaf_rn(-qe0, s, re), y, qe0);
    qo = __fmaf_rn(__fmaf_rn(-qo0, s, ro), y, qo0);
  } else {
    qe = nvfp4_quotient_ieee(re, s);
    qo = nvfp4_quotient_ieee(ro, s);
  }
  st_u8(codes + 224 + lane, cvt_e2m1x2(qe, qo));
  if ((lane & 7) == 0) st_u8(scales + 28 + (lane >> 3), sbyte);
}

// ------------------------------------------------------------------ gates ---

// Gates and addresses of token `t` (one lane's token): `page_off` >= 0 (byte
// offset of its page) when it writes, with `in_page` its slot in the page and
// `table_off` the offset (floats) of its cos/sin row; -1 otherwise.
__device__ __forceinline__ void token_gates(const RopeParams& p, int64_t t, int64_t& page_off,
                                            int64_t& table_off, int64_t& in_page) {
  page_off = -1;
  table_off = 0;
  in_page = 0;
  if (t >= p.num_tokens) return;
  const int64_t s = ld_once_i64(p.slots + t);
  if (s < 0 || s >= p.num_slots) return;
  const int64_t pos = ld_once_i64(p.positions + t);
  // pos - R >= cos_rows puts the table row past the table whatever the
  // remainder; testing it first also keeps pos + 1 from overflowing.
  if (pos < 0 || pos - p.ratio >= p.cos_rows) return;
  int64_t q, r;
  divmod_pos(pos + 1, p.ratio, q, r);
  // (pos+1) % R == 0 makes (pos // R) * R equal to pos + 1 - R.
  const int64_t row = pos + 1 - p.ratio;
  if (r != 0 || row >= p.cos_rows) return;
  int64_t page;
  divmod_pos(s, p.cache_block, page, in_page);
  page_off = page * p.page_stride;
  table_off = row * p.cos_stride;
}

// ---------------------------------------------------------------- kernels ---

// Five resident blocks (40 warps) per SM: the 48-register cap costs a few
// spilled words in the MXFP8 kernel, but the extra writers in flight lifted it
// by 7 % (4,194,304-token insert: 5292 -> 5680 GB/s; six blocks at 40
// registers lose it again).
template <bool kSanitize>
__global__ void __launch_bounds__(kRopeThreads, 5) mxfp8_insert_kernel(RopeParams p) {
  const int lane = threadIdx.x & 31;
  const int64_t warp = ((int64_t)blockIdx.x * kRopeThreads + threadIdx.x) >> 5;
  const int64_t num_warps = ((int64_t)gridDim.x * kRopeThreads) >> 5;

  for (int64_t base = warp * 32; base < p.num_tokens; base += num_warps * 32) {
    int64_t page_off, table_off, in_page;
    token_gates(p, base + lane, page_off, table_off, in_page);
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
        rotate_row<kSanitize>(w ? xb0 : xa0, w ? xb1 : xa1, w ? cb : ca, w ? snb : sna, lane, f0,
                              f1);
        uint8_t* page = p.cache + pg;
        uint8_t* values = page + slot_in_page * 512;
        uint8_t* scales = page + p.cache_block * 512 + slot_in_page * 16;
        mxfp8_half<kSanitize>(f0, values, scales, lane);
        mxfp8_half<kSanitize>(f1, values + 256, scales + 8, lane);
      }
    }
  }
}

// NaN ends as code 0 in an NVFP4 record with or without sanitising (the code
// rule gives NaN code 0 and the amax ignores it), so one kernel serves both.
__global__ void __launch_bounds__(kRopeThreads, 5) nvfp4_insert_kernel(RopeParams p) {
  __shared__ float4 scale_table[128];  // ScaleEntry of every E4M3 byte 0..127
  if (threadIdx.x < 128) {
    const ScaleEntry e = make_scale_entry(threadIdx.x);
    scale_table[threadIdx.x] = make_float4(e.s, e.y, e.yh, e.yl);
  }
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const int64_t warp = ((int64_t)blockIdx.x * kRopeThreads + threadIdx.x) >> 5;
  const int64_t num_warps = ((int64_t)gridDim.x * kRopeThreads) >> 5;

  for (int64_t base = warp * 32; base < p.num_tokens; base += num_warps * 32) {
    int64_t page_off, table_off, in_page;
    token_gates(p, base + lane, page_off, table_off, in_page);
    uint32_t todo = __ballot_sync(0xFFFFFFFFu, page_off >= 0);
    while (todo) {
      const int ia = __ffs(todo) - 1;
      todo &= todo - 1;
      const int ib = todo ? __ffs(todo) - 1 : -1;
      if (todo) todo &= todo - 1;
      const uint8_t* sa = p.latent + (base + ia) * p.row_pitch;
      const int64_t ta = __shfl_sync(0xFFFFFFFFu, table_off, ia);
      const uint4 xa0 = ld_once_v4(sa + 16 * lane);
      uint4 xa1 = make_uint4(0, 0, 0, 0);
      if (lane < 24) xa1 = ld_once_v4(sa + 512 + 16 * lane);
      const uint32_t ra = ld_once_u32(sa + 896 + 4 * lane);
      const float ca = ld_f32(p.cos_sin + ta + lane);
      const float sna = ld_f32(p.cos_sin + ta + 32 + lane);
      uint4 xb0 = make_uint4(0, 0, 0, 0), xb1 = xb0;
      uint32_t rb = 0;
      float cb = 1.0f, snb = 0.0f;
      if (ib >= 0) {
        const uint8_t* sb = p.latent + (base + ib) * p.row_pitch;
        const int64_t tb = __shfl_sync(0xFFFFFFFFu, table_off, ib);
        xb0 = ld_once_v4(sb + 16 * lane);
        if (lane < 24) xb1 = ld_once_v4(sb + 512 + 16 * lane);
        rb = ld_once_u32(sb + 896 + 4 * lane);
        cb = ld_f32(p.cos_sin + tb + lane);
        snb = ld_f32(p.cos_sin + tb + 32 + lane);
      }
#pragma unroll
      for (int w = 0; w < 2; ++w) {
        const int i = w ? ib : ia;
        if (i < 0) break;
        const int64_t pg = __shfl_sync(0xFFFFFFFFu, page_off, i);
        const int64_t slot_in_page = __shfl_sync(0xFFFFFFFFu, in_page, i);
        uint8_t* page = p.cache + pg;
        uint8_t* codes = page + slot_in_page * 256;
        uint8_t* scales = page + p.cache_block * 256 + slot_in_page * 32;
        nvfp4_nope_half(w ? xb0 : xa0, codes, scales, lane, scale_table, true);
        nvfp4_nope_half(w ? xb1 : xa1, codes + 128, scales + 16, lane, scale_table, lane < 24);
        nvfp4_rotary_pair(w ? rb : ra, w ? cb : ca, w ? snb : sna, codes, scales, lane,
                          scale_table);
      }
    }
  }
}

int g_rope_occupancy[3][64];

template <typename Kernel>
int launch(Kernel k, int* occupancy, const RopeParams& p, cudaStream_t stream) {
  const int64_t chunks = (p.num_tokens + 31) / 32;
  const int64_t work_blocks = (chunks + kRopeWarps - 1) / kRopeWarps;
  const unsigned grid =
      grid_for(work_blocks, resident_blocks_per_sm(k, kRopeThreads, 0, occupancy));
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
  if (nvfp4) return launch(nvfp4_insert_kernel, g_rope_occupancy[2], p, stream);
  return sanitize_nans ? launch(mxfp8_insert_kernel<true>, g_rope_occupancy[1], p, stream)
                       : launch(mxfp8_insert_kernel<false>, g_rope_occupancy[0], p, stream);
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
