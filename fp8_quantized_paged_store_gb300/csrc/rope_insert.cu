// rope_insert.cu — the V4.1 and V4 compressed-cache inserts:
// rope_quant_insert_mxfp8 / _nvfp4 / _v4 and rope_plain_insert. GPT-J RoPE on
// the last 64 elements, then one of five layouts: MXFP8 (E4M3 values, E8M0
// scale per 32; 528-byte record), NVFP4 (E2M1 codes, E4M3 scale per 16;
// 288-byte record), the V4 584-byte record (448 E4M3 values in tiles of 64
// with E8M0 scales, 64 bf16 rotary values, 8 scale bytes of which the last
// is 0), or a plain [448 | 64] row of bf16 or per-tensor-scaled E4M3. The
// records keep their scales segregated after the values in each page.
//
// Follows "vllm.models.deepseek_v41.common.ops.fused_compress_quant_cache"
// (_rope_quant_insert_mxfp8_kernel, _rope_quant_insert_nvfp4_kernel,
// rope_quant_insert: its docstring describes the V4 record and the plain
// rows, whose kernels the page does not print).
//
// Work decomposition (all kernels): a warp owns 32 tokens at a time
// (grid-stride over chunks); lane i evaluates token i's gates (slot range,
// (pos+1) % R == 0, table row in range) and addresses once, and a ballot lists
// the writers, so non-writers cost no row traffic. Writers are taken two at a
// time with both rows' loads (and their table rows) issued before either is
// quantized: with two writers in flight per warp and 40 warps per SM, loads
// stay in flight while other warps compute (a shared-memory cp.async ring
// measured slower here, the gate and ballot work per window then sitting on
// the critical path). Rotary pairs 224..255 are elements 448..511.
//
// The records (MXFP8, NVFP4, V4): lane l < 28 holds a run of 16 NoPE
// elements, 16l..16l+15 (two 16-byte loads at bytes 32l and 32l+16; the
// second hits the sectors the first brought into L1), and every lane j
// rotates rotary pair j with its own cos and sin (4 bytes of the row, one
// cos and one sin). An NVFP4 tile is one lane's run (no amax shuffle), an
// MXFP8 tile of 32 two (one shuffle), a V4 tile of 64 four (two); a run's
// E4M3 values leave in one 16-byte store, its E2M1 codes in one 8-byte
// store. Against holding elements 8l..8l+7 and 256+8l..256+8l+7 (two
// half-row passes, every tile shared by more lanes) this measured 0.345 ->
// 0.310 ms (NVFP4), 0.351 -> 0.329 ms (MXFP8) and 0.379 -> 0.375 ms (V4) on
// 4,194,304 tokens, and removed the spills those kernels had at 48
// registers. The rotary values are spread over the whole warp: the NVFP4
// exact quotients, the MXFP8 tiles 14 and 15 (16 lanes each) and the V4 bf16
// values all run one pair per lane. The 448 NVFP4 NoPE values are bf16
// numbers and take the cheaper exact code rule of nvfp4_code_value2 (two
// fused products, no ALU work).
//
// Plain fp8 rows use the run mapping too (their rotary quotients then run
// two per lane). Plain bf16 rows keep the half-row mapping, which measured
// faster for them (0.389 against 0.397 ms with runs: their NoPE part is a
// plain copy, best done as fully coalesced 512-byte warp stores): lane l
// holds elements 8l..8l+7 (half 0) and 256+8l..256+8l+7 (half 1), and the
// rotary elements are half 1 of lanes 24..31, which alone read the table row
// (cos and sin 4(l-24)..4(l-24)+3, two 16-byte loads each).
//
// The pages evaluate the rotation formula on all 256 pairs, with cos 1 and
// sin 0 outside the rotary range. There it is the identity except for NaN,
// infinities and signed zeros: even' = even - odd*0 and odd' = odd + even*0.
// That is computed exactly, two elements per instruction, as one bf16x2 fma
// of the half-swapped word with (-0, +0) added to the word: the products are
// exact, and each sum is the element itself, a zero, or NaN, so no rounding
// happens and the result equals the binary32 formula bit for bit. Rotary
// pairs use the binary32 formula with every product and sum rounded
// separately (no fused multiply-add). Plain rows take the 448 NoPE values as
// they are (bit for bit in bf16, divided by the scale in fp8).
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>

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
  int64_t slot_pitch;   // plain rows: bytes between the rows of a page
  float fp8_scale;      // plain fp8 rows: the per-tensor scale
  int32_t fp8_mode;     // plain fp8 rows: how x / fp8_scale is formed (Fp8Quotient)
  float fp8_yh, fp8_yl;  // plain fp8 rows: RD(1/scale) and RN((1 - scale*yh) * yh)
};

// How the plain fp8 rows form the E4M3 code of RN(x / scale):
//   kDivide   every value by a correctly rounded division;
//   kTwoTerm  the bf16 NoPE values by RN(x*yh + RN(x*yl)), a two-term
//             reciprocal that the host found to give the division's code for
//             every one of the 65,536 bf16 patterns at this scale; the binary32
//             rotary values by division;
//   kProduct  scale a power of two with a normal reciprocal: every value by
//             RN(x * yh), the same rounding of the same exact quotient.
enum Fp8Quotient : int32_t { kDivide = 0, kTwoTerm = 1, kProduct = 2 };

// Layouts besides NVFP4: the MXFP8 and V4 records and the plain fp8 rows
// (record_run_insert_kernel), the plain bf16 rows (fp8_family_insert_kernel).
enum class Layout { kMxfp8, kV4, kPlainBf16, kPlainFp8 };
constexpr int kV4Record = 584;   // 576 value bytes (448 E4M3 + 64 bf16) + 8 scale bytes

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

// ------------------------------------------------------------------ MXFP8 ---

// Eight values times the power of two `inv` as E4M3 (clamped to +-448,
// NaN -> 0x7F), two per packed product; a product by a power of two is exact
// unless it leaves the normal range, where it rounds like the scalar one.
__device__ __forceinline__ uint2 e4m3x8_scaled(const float f[8], float inv) {
  const float2 i2 = make_float2(inv, inv);
  const float2 p0 = mul2_rn(make_float2(f[0], f[1]), i2), p1 = mul2_rn(make_float2(f[2], f[3]), i2);
  const float2 p2 = mul2_rn(make_float2(f[4], f[5]), i2), p3 = mul2_rn(make_float2(f[6], f[7]), i2);
  return make_uint2(cvt_e4m3x2(p0.x, p0.y) | (cvt_e4m3x2(p1.x, p1.y) << 16),
                    cvt_e4m3x2(p2.x, p2.y) | (cvt_e4m3x2(p3.x, p3.y) << 16));
}


// ------------------------------------------------------------ V4 and plain ---

__device__ __forceinline__ uint32_t bf16x2_rn(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}

// Two binary32 values rounded to bf16 (nearest even) with every NaN stored
// as the quiet NaN 0x7FC0: the sign of a NaN that arithmetic produced is not
// portable, so a stored one carries none.
__device__ __forceinline__ uint32_t bf16x2_rn_nan(float lo, float hi) {
  uint32_t d = bf16x2_rn(lo, hi);
  if (lo != lo) d = (d & 0xFFFF0000u) | 0x7FC0u;
  if (hi != hi) d = (d & 0x0000FFFFu) | 0x7FC00000u;
  return d;
}

// Eight binary32 values as bf16 (bf16x2_rn_nan), 16 bytes.
__device__ __forceinline__ uint4 bf16x8_rn(const float f[8]) {
  return make_uint4(bf16x2_rn_nan(f[0], f[1]), bf16x2_rn_nan(f[2], f[3]),
                    bf16x2_rn_nan(f[4], f[5]), bf16x2_rn_nan(f[6], f[7]));
}

// Eight values as E4M3 of RN(x / scale), clamped to +-448 (NaN -> 0x7F).
__device__ __forceinline__ uint2 e4m3x8_div(const float f[8], float scale) {
  uint32_t w[2];
#pragma unroll
  for (int h = 0; h < 2; ++h)
    w[h] = cvt_e4m3x2(__fdiv_rn(f[4 * h], scale), __fdiv_rn(f[4 * h + 1], scale)) |
           (cvt_e4m3x2(__fdiv_rn(f[4 * h + 2], scale), __fdiv_rn(f[4 * h + 3], scale)) << 16);
  return make_uint2(w[0], w[1]);
}

// Eight values as E4M3 of RN(x*yh + RN(x*yl)) (kTwoTerm) or of RN(x*yh)
// (kProduct, yl unused), two per packed instruction. The product feeds only
// the fused multiply-add's addend, which no instruction can absorb.
template <bool kTwoTerm>
__device__ __forceinline__ uint2 e4m3x8_recip(const float f[8], float yh, float yl) {
  const float2 h2 = make_float2(yh, yh), l2 = make_float2(yl, yl);
  uint32_t c[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float2 x = make_float2(f[2 * k], f[2 * k + 1]);
    const float2 q = kTwoTerm ? fma2_rn(x, h2, mul2_rn(x, l2)) : mul2_rn(x, h2);
    c[k] = cvt_e4m3x2(q.x, q.y);
  }
  return make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
}

// The rotary values of the lane's half 1 (lanes 24..31), binary32 formula
// without contraction and without sanitising.
__device__ __forceinline__ void rotate_pairs(uint4 x1, float4 c, float4 s, float f[8]) {
  float v[8];
  widen8(x1, v);
  const float cc[4] = {c.x, c.y, c.z, c.w};
  const float ss[4] = {s.x, s.y, s.z, s.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float e = v[2 * k], o = v[2 * k + 1];
    f[2 * k] = __fsub_rn(__fmul_rn(e, cc[k]), __fmul_rn(o, ss[k]));
    f[2 * k + 1] = __fadd_rn(__fmul_rn(o, cc[k]), __fmul_rn(e, ss[k]));
  }
}

// One writer row of the plain bf16 layout. `page` points at the slot's page,
// `slot_in_page` is its row there.
template <Layout kL>
__device__ __forceinline__ void write_plain(const RopeParams& p, uint4 x0, uint4 x1, float4 c,
                                            float4 s, uint8_t* page, int64_t slot_in_page,
                                            int lane) {
  static_assert(kL == Layout::kPlainBf16, "plain bf16 rows only");
  {
    uint8_t* row = page + slot_in_page * p.slot_pitch;
    st_v4(row + 16 * lane, x0);
    if (lane < 24) {
      st_v4(row + 512 + 16 * lane, x1);
    } else {
      float f1[8];
      rotate_pairs(x1, c, s, f1);
      st_v4(row + 512 + 16 * lane, bf16x8_rn(f1));
    }
  }
}

// ------------------------------------------------------------------ NVFP4 ---

// Positive E4M3 code (<= 0x7E) -> its exact binary32 value.
__device__ __forceinline__ float e4m3_value(uint32_t b) {
  const uint32_t ex = b >> 3, man = b & 7u;
  return ex ? __uint_as_float(((ex + 120u) << 23) | (man << 20))
            : __uint_as_float(0x3B000000u) * (float)man;  // man * 2**-9, exact
}

// Per E4M3 byte b (0..127), built once per block: s = value(b) and the
// two-term reciprocal yh = RD(1/s), yl = RN((1 - s*yh) * yh) >= 0 that
// nvfp4_code_value2 and nvfp4_rotary_code_value2 divide by.
struct ScaleEntry {
  float s, yh, yl;
};

__device__ __forceinline__ ScaleEntry make_scale_entry(uint32_t b) {
  ScaleEntry e;
  e.s = e4m3_value(b);
  e.yh = __frcp_rd(e.s);
  e.yl = __fmul_rn(__fmaf_rn(-e.s, e.yh, 1.0f), e.yh);  // 1 - s*yh is exact
  return e;
}

// The NVFP4 tile scale from the tile's |amax| (NaN-free): the E4M3 byte of
// clamp(amax * RN(1/6), 2**-9, 448) and its table entry.
__device__ __forceinline__ uint32_t nvfp4_scale(float amax, const float4* table, ScaleEntry& e) {
  // the conversion saturates: targets above 448 (or infinite) give 448
  const float target = fmaxf(__fmul_rn(amax, 1.0f / 6.0f), 0.001953125f);
  const uint32_t sbyte = cvt_e4m3x2(target, 0.0f) & 0xFFu;  // 0x01..0x7E
  const float4 t = table[sbyte];
  e.s = t.x;
  e.yh = t.y;
  e.yl = t.z;
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
// Both bf16 halves of `w` (low element first) go through one packed pair of
// these steps.
__device__ __forceinline__ float2 nvfp4_code_value2(uint32_t w, const ScaleEntry& e) {
  const float2 x = make_float2(bf16_lo(w), bf16_hi(w));
  return fma2_rn(x, make_float2(e.yh, e.yh), mul2_rn(x, make_float2(e.yl, e.yl)));
}

// Code-deciding stand-in for RN(r / s) when r is a binary32 rotary value
// (NaN already cleared): q = RN(r*yh + RN(r*yl)) + 0.0, with yh and yl the
// two-term reciprocal of nvfp4_code_value2. The E2M1 code of a quotient
// depends only on which side of each midpoint M (0.25, 0.75, ..., 5) it lies
// and on ties at M itself; q and RN(r / s) can differ only if r / s lies
// within about 2**-44 (relative) of a binary32 rounding boundary, and can
// then change the code only if that boundary is next to some M. A boundary
// B next to M has 25 significant bits with an odd last one, and s at most 4,
// so B*s is never a binary32 value: the binary32 r nearest B*s keeps r / s
// more than 2**-28 (relative) away from B, far outside the 2**-44 above. Where r /
// s is exactly M, r*yh + RN(r*yl) is within 2**-44 of M and rounds to M. Far
// from the midpoints (tiny, huge, or infinite r, the last only with s = 448
// where yl > 0) the two agree on the code without any range check. The
// final +0.0 turns a -0.0 result (from r = -0 or a quotient that underflows)
// into +0.0, whose code is 0 as the oracle's sign rule gives. A CPU check
// over every E4M3 scale, every midpoint and the binary32 values around each
// adjacent boundary confirms the codes and the margin.
__device__ __forceinline__ float2 nvfp4_rotary_code_value2(float2 r, const ScaleEntry& e) {
  const float2 t = mul2_rn(r, make_float2(e.yl, e.yl));
  return add2_rn(fma2_rn(r, make_float2(e.yh, e.yh), t), make_float2(0.0f, 0.0f));
}

// One NoPE tile of the record (16 bf16-exact values, elements 16*lane ..
// 16*lane+15, two 16-byte words held by this lane): the NoPE formula, NaN and
// -0.0 to +0.0, the tile amax, then eight code bytes by nvfp4_code_value2 and
// the tile's scale byte. Lanes with `store` false compute but write nothing.
__device__ __forceinline__ void nvfp4_nope_tile(uint4 a, uint4 b, uint8_t* codes,
                                                uint8_t* scales, int lane, const float4* table,
                                                bool store) {
  // Fast path, taken when no lane's tile holds a NaN or an infinity (the
  // NaN-propagating |max| of the raw values is finite): the NoPE formula
  // (e*1 - o*0, o*1 + e*0) then changes nothing but signs of zeros, and the
  // clean-up below maps every zero to +0.0, so masking the zeros does both.
  const uint32_t mr =
      bf16x2_maxabs_nan(bf16x2_maxabs_nan(bf16x2_maxabs_nan(a.x, a.y), bf16x2_maxabs_nan(a.z, a.w)),
                        bf16x2_maxabs_nan(bf16x2_maxabs_nan(b.x, b.y), bf16x2_maxabs_nan(b.z, b.w)));
  const bool special = (mr & 0x7F80u) == 0x7F80u || (mr & 0x7F800000u) == 0x7F800000u;
  float amax;
  if (!__any_sync(0xFFFFFFFFu, special)) {
    auto zero = [](uint32_t v) { return v & bf16x2_nonzero_number_mask(v); };
    a = make_uint4(zero(a.x), zero(a.y), zero(a.z), zero(a.w));
    b = make_uint4(zero(b.x), zero(b.y), zero(b.z), zero(b.w));
    amax = fmaxf(fabsf(bf16_lo(mr)), fabsf(bf16_hi(mr)));
  } else {
    auto clean = [](uint32_t v) {
      const uint32_t r = nope_pair(v);
      return r & bf16x2_nonzero_number_mask(r);
    };
    a = make_uint4(clean(a.x), clean(a.y), clean(a.z), clean(a.w));
    b = make_uint4(clean(b.x), clean(b.y), clean(b.z), clean(b.w));
    const uint32_t m =
        bf16x2_maxabs(bf16x2_maxabs(bf16x2_maxabs(a.x, a.y), bf16x2_maxabs(a.z, a.w)),
                      bf16x2_maxabs(bf16x2_maxabs(b.x, b.y), bf16x2_maxabs(b.z, b.w)));
    amax = fmaxf(fabsf(bf16_lo(m)), fabsf(bf16_hi(m)));
  }
  ScaleEntry e;
  const uint32_t sbyte = nvfp4_scale(amax, table, e);
  const float2 q0 = nvfp4_code_value2(a.x, e), q1 = nvfp4_code_value2(a.y, e);
  const float2 q2 = nvfp4_code_value2(a.z, e), q3 = nvfp4_code_value2(a.w, e);
  const float2 q4 = nvfp4_code_value2(b.x, e), q5 = nvfp4_code_value2(b.y, e);
  const float2 q6 = nvfp4_code_value2(b.z, e), q7 = nvfp4_code_value2(b.w, e);
  const uint32_t c0 = cvt_e2m1x8(q0.x, q0.y, q1.x, q1.y, q2.x, q2.y, q3.x, q3.y);
  const uint32_t c1 = cvt_e2m1x8(q4.x, q4.y, q5.x, q5.y, q6.x, q6.y, q7.x, q7.y);
  if (store) {
    st_v2(codes + 8 * lane, c0, c1);
    st_u8(scales + lane, sbyte);
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
  const float2 q = nvfp4_rotary_code_value2(make_float2(re, ro), sc);
  const float qe = q.x, qo = q.y;
  st_u8(codes + 224 + lane, cvt_e2m1x2(qe, qo));
  if ((lane & 7) == 0) st_u8(scales + 28 + (lane >> 3), sbyte);
}

// ------------------------------------------------------------------ gates ---

// Gates and addresses of token `t` (one lane's token): `page_off` >= 0 (byte
// offset of its page) when it writes, with `in_page` its slot in the page and
// `table_off` the offset (floats) of its cos/sin row; -1 otherwise.
// Slot and position of token t (-1, -1 past the batch), loaded where the
// call stands, so that a loop can fetch them a chunk ahead.
struct TokenIds {
  int64_t slot, pos;
};

__device__ __forceinline__ int64_t ld_ahead_i64(const int64_t* p) {
  int64_t r;
  asm volatile("ld.global.nc.L1::no_allocate.s64 %0, [%1];" : "=l"(r) : "l"(p));
  return r;
}

__device__ __forceinline__ TokenIds token_ids(const RopeParams& p, int64_t t) {
  TokenIds r{-1, -1};
  if (t < p.num_tokens) {
    r.slot = ld_ahead_i64(p.slots + t);
    r.pos = ld_ahead_i64(p.positions + t);
  }
  return r;
}

__device__ __forceinline__ void token_gates(const RopeParams& p, TokenIds id, int64_t& page_off,
                                            int64_t& table_off, int64_t& in_page) {
  page_off = -1;
  table_off = 0;
  in_page = 0;
  const int64_t s = id.slot;
  if (s < 0 || s >= p.num_slots) return;
  const int64_t pos = id.pos;
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

// The plain bf16 rows. Five resident blocks (40 warps) per SM: the
// 48-register cap costs a few spilled words, but the extra writers in flight
// lifted the inserts by 7 % when measured on the MXFP8 record (4,194,304
// tokens: 5292 -> 5680 GB/s; six blocks at 40 registers lose it again).
template <Layout kL, bool kSanitize>
__global__ void __launch_bounds__(kRopeThreads, 5) fp8_family_insert_kernel(RopeParams p) {
  const int lane = threadIdx.x & 31;
  const int64_t warp = ((int64_t)blockIdx.x * kRopeThreads + threadIdx.x) >> 5;
  const int64_t num_warps = ((int64_t)gridDim.x * kRopeThreads) >> 5;

  for (int64_t base = warp * 32; base < p.num_tokens; base += num_warps * 32) {
    int64_t page_off, table_off, in_page;
    // (fetching the next chunk's ids a chunk ahead, as the NVFP4 kernel
    // does, costs these kernels spills at 48 registers and measured slower)
    token_gates(p, token_ids(p, base + lane), page_off, table_off, in_page);
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
        write_plain<kL>(p, w ? xb0 : xa0, w ? xb1 : xa1, w ? cb : ca, w ? snb : sna,
                        p.cache + pg, slot_in_page, lane);
      }
    }
  }
}

__device__ __forceinline__ void st_u16(void* p, uint32_t v) {
  asm volatile("st.global.u16 [%0], %1;" ::"l"(p), "h"((unsigned short)v) : "memory");
}

// One writer of the MXFP8 or V4 record, one run per lane: lane l < 28 holds
// NoPE elements 16l..16l+15 (`a`, `b`), and every lane rotates rotary pair l
// (`xr`, with its own cos `c` and sin `sn`). An MXFP8 tile of 32 is two
// lanes' runs (one xor-shuffle), a V4 tile of 64 four (two); the NoPE run
// leaves as one 16-byte store. The MXFP8 rotary tiles 14 and 15 are 16 lanes
// each (four xor-shuffles, two code bytes per lane); the V4 rotary values
// are bf16, four bytes per lane.
template <Layout kL, bool kSanitize>
__device__ __forceinline__ void record_run(const RopeParams& p, uint4 a, uint4 b, uint32_t xr,
                                           float c, float sn, uint8_t* page,
                                           int64_t slot_in_page, int lane) {
  if constexpr (kL == Layout::kPlainFp8) {
    // plain fp8 row: E4M3 of x / scale, the quotient formed as the host chose
    uint8_t* row = page + slot_in_page * p.slot_pitch;
    float f[8];
    uint2 lo, hi;
    widen8(a, f);
    if (p.fp8_mode == kTwoTerm) {
      lo = e4m3x8_recip<true>(f, p.fp8_yh, p.fp8_yl);
      widen8(b, f);
      hi = e4m3x8_recip<true>(f, p.fp8_yh, p.fp8_yl);
    } else if (p.fp8_mode == kProduct) {
      lo = e4m3x8_recip<false>(f, p.fp8_yh, 0.0f);
      widen8(b, f);
      hi = e4m3x8_recip<false>(f, p.fp8_yh, 0.0f);
    } else {
      lo = e4m3x8_div(f, p.fp8_scale);
      widen8(b, f);
      hi = e4m3x8_div(f, p.fp8_scale);
    }
    if (lane < 28) {  // rows are 8-byte aligned
      st_v2(row + 16 * lane, lo.x, lo.y);
      st_v2(row + 16 * lane + 8, hi.x, hi.y);
    }
    const float ev = bf16_lo(xr), od = bf16_hi(xr);
    const float re = __fsub_rn(__fmul_rn(ev, c), __fmul_rn(od, sn));
    const float ro = __fadd_rn(__fmul_rn(od, c), __fmul_rn(ev, sn));
    const uint32_t two = p.fp8_mode == kProduct
                             ? cvt_e4m3x2(__fmul_rn(re, p.fp8_yh), __fmul_rn(ro, p.fp8_yh))
                             : cvt_e4m3x2(__fdiv_rn(re, p.fp8_scale), __fdiv_rn(ro, p.fp8_scale));
    st_u16(row + 448 + 2 * lane, two);
    return;
  }
  constexpr int kValueBytes = kL == Layout::kV4 ? 576 : 512;
  constexpr int kScaleBytes = kL == Layout::kV4 ? 8 : 16;
  constexpr int kCap = kSanitize ? 254 : 255;
  uint8_t* values = page + slot_in_page * kValueBytes;
  uint8_t* scales = page + p.cache_block * kValueBytes + slot_in_page * kScaleBytes;
  auto nope = [](uint32_t w) {
    const uint32_t r = nope_pair(w);
    return kSanitize ? (r & bf16x2_number_mask(r)) : r;
  };
  a.x = nope(a.x);
  a.y = nope(a.y);
  a.z = nope(a.z);
  a.w = nope(a.w);
  b.x = nope(b.x);
  b.y = nope(b.y);
  b.z = nope(b.z);
  b.w = nope(b.w);
  // NaN is ignored by the maxima (a tile of NaN alone ends at the 1e-4 floor)
  const uint32_t m = bf16x2_maxabs(bf16x2_maxabs(bf16x2_maxabs(a.x, a.y), bf16x2_maxabs(a.z, a.w)),
                                   bf16x2_maxabs(bf16x2_maxabs(b.x, b.y), bf16x2_maxabs(b.z, b.w)));
  float amax = fmaxf(fabsf(bf16_lo(m)), fabsf(bf16_hi(m)));
  amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
  if (kL == Layout::kV4) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 2));
  amax = fmaxf(amax, 1e-4f);
  const int e = ceil_pow2_exponent(__fmul_rn(amax, 1.0f / 448.0f));
  const float inv = exp2_neg(e);
  float f[8];
  widen8(a, f);
  const uint2 lo = e4m3x8_scaled(f, inv);
  widen8(b, f);
  const uint2 hi = e4m3x8_scaled(f, inv);
  if (lane < 28) {
    st_v4(values + 16 * lane, make_uint4(lo.x, lo.y, hi.x, hi.y));
    const int enc = e + 127;
    if (kL == Layout::kV4 ? (lane & 3) == 0 : (lane & 1) == 0)
      st_u8(scales + (kL == Layout::kV4 ? lane >> 2 : lane >> 1),
            (uint32_t)(enc < kCap ? enc : kCap));
  }
  // rotary pair `lane`: elements 448 + 2*lane and 449 + 2*lane
  const float ev = bf16_lo(xr), od = bf16_hi(xr);
  float re = __fsub_rn(__fmul_rn(ev, c), __fmul_rn(od, sn));
  float ro = __fadd_rn(__fmul_rn(od, c), __fmul_rn(ev, sn));
  if (kSanitize) {
    re = (re == re) ? re : 0.0f;
    ro = (ro == ro) ? ro : 0.0f;
  }
  if constexpr (kL == Layout::kV4) {
    st_u32(values + 448 + 4 * lane, bf16x2_rn_nan(re, ro));
    if (lane == 0) st_u8(scales + 7, 0u);
  } else {
    float ramax = fmaxf(fmaxf(fabsf(re), fabsf(ro)), 0.0f);
    ramax = fmaxf(ramax, __shfl_xor_sync(0xFFFFFFFFu, ramax, 1));
    ramax = fmaxf(ramax, __shfl_xor_sync(0xFFFFFFFFu, ramax, 2));
    ramax = fmaxf(ramax, __shfl_xor_sync(0xFFFFFFFFu, ramax, 4));
    ramax = fmaxf(ramax, __shfl_xor_sync(0xFFFFFFFFu, ramax, 8));
    ramax = fmaxf(ramax, 1e-4f);
    const int er = ceil_pow2_exponent(__fmul_rn(ramax, 1.0f / 448.0f));
    const float rinv = exp2_neg(er);
    st_u16(values + 448 + 2 * lane, cvt_e4m3x2(__fmul_rn(re, rinv), __fmul_rn(ro, rinv)));
    if ((lane & 15) == 0) {
      const int enc = er + 127;
      st_u8(scales + 14 + (lane >> 4), (uint32_t)(enc < kCap ? enc : kCap));
    }
  }
}

// The MXFP8 and V4 records (record_run per writer), with the token loop of
// the NVFP4 kernel: the next chunk's slots and positions in flight while
// this chunk's writers are stored.
template <Layout kL, bool kSanitize>
__global__ void __launch_bounds__(kRopeThreads, 5) record_run_insert_kernel(RopeParams p) {
  const int lane = threadIdx.x & 31;
  const int64_t warp = ((int64_t)blockIdx.x * kRopeThreads + threadIdx.x) >> 5;
  const int64_t num_warps = ((int64_t)gridDim.x * kRopeThreads) >> 5;

  TokenIds ids = token_ids(p, warp * 32 + lane);
  for (int64_t base = warp * 32; base < p.num_tokens; base += num_warps * 32) {
    int64_t page_off, table_off, in_page;
    token_gates(p, ids, page_off, table_off, in_page);
    ids = token_ids(p, base + num_warps * 32 + lane);
    uint32_t todo = __ballot_sync(0xFFFFFFFFu, page_off >= 0);
    while (todo) {
      const int ia = __ffs(todo) - 1;
      todo &= todo - 1;
      const int ib = todo ? __ffs(todo) - 1 : -1;
      if (todo) todo &= todo - 1;
      const uint8_t* sa = p.latent + (base + ia) * p.row_pitch;
      const int64_t ta = __shfl_sync(0xFFFFFFFFu, table_off, ia);
      uint4 xa0 = make_uint4(0, 0, 0, 0), xa1 = xa0;
      if (lane < 28) {
        xa0 = ld_nc_v4(sa + 32 * lane);
        xa1 = ld_nc_v4(sa + 32 * lane + 16);
      }
      const uint32_t ra = ld_once_u32(sa + 896 + 4 * lane);
      const float ca = ld_f32(p.cos_sin + ta + lane);
      const float sna = ld_f32(p.cos_sin + ta + 32 + lane);
      uint4 xb0 = make_uint4(0, 0, 0, 0), xb1 = xb0;
      uint32_t rb = 0;
      float cb = 1.0f, snb = 0.0f;
      if (ib >= 0) {
        const uint8_t* sb = p.latent + (base + ib) * p.row_pitch;
        const int64_t tb = __shfl_sync(0xFFFFFFFFu, table_off, ib);
        if (lane < 28) {
          xb0 = ld_nc_v4(sb + 32 * lane);
          xb1 = ld_nc_v4(sb + 32 * lane + 16);
        }
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
        record_run<kL, kSanitize>(p, w ? xb0 : xa0, w ? xb1 : xa1, w ? rb : ra, w ? cb : ca,
                                  w ? snb : sna, p.cache + pg, slot_in_page, lane);
      }
    }
  }
}

// NaN ends as code 0 in an NVFP4 record with or without sanitising (the code
// rule gives NaN code 0 and the amax ignores it), so one kernel serves both.
// The next chunk's slots and positions are fetched a chunk ahead (the gates
// and ballot of a chunk otherwise wait for two dependent loads: 0.395 ms ->
// 0.364 ms on the 4,194,304-token insert). Loading the next pair of rows
// before quantizing the current one measured slower: at 64 registers the
// kernel loses a fifth of its warps, at 48 it spills.
__global__ void __launch_bounds__(kRopeThreads, 5) nvfp4_insert_kernel(RopeParams p) {
  __shared__ float4 scale_table[128];  // ScaleEntry of every E4M3 byte 0..127
  if (threadIdx.x < 128) {
    const ScaleEntry e = make_scale_entry(threadIdx.x);
    scale_table[threadIdx.x] = make_float4(e.s, e.yh, e.yl, 0.0f);
  }
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const int64_t warp = ((int64_t)blockIdx.x * kRopeThreads + threadIdx.x) >> 5;
  const int64_t num_warps = ((int64_t)gridDim.x * kRopeThreads) >> 5;

  TokenIds ids = token_ids(p, warp * 32 + lane);
  for (int64_t base = warp * 32; base < p.num_tokens; base += num_warps * 32) {
    int64_t page_off, table_off, in_page;
    token_gates(p, ids, page_off, table_off, in_page);
    ids = token_ids(p, base + num_warps * 32 + lane);  // the next chunk's, in flight meanwhile
    uint32_t todo = __ballot_sync(0xFFFFFFFFu, page_off >= 0);
    while (todo) {
      const int ia = __ffs(todo) - 1;
      todo &= todo - 1;
      const int ib = todo ? __ffs(todo) - 1 : -1;
      if (todo) todo &= todo - 1;
      const uint8_t* sa = p.latent + (base + ia) * p.row_pitch;
      const int64_t ta = __shfl_sync(0xFFFFFFFFu, table_off, ia);
      uint4 xa0 = make_uint4(0, 0, 0, 0), xa1 = xa0;
      if (lane < 28) {
        xa0 = ld_nc_v4(sa + 32 * lane);
        xa1 = ld_nc_v4(sa + 32 * lane + 16);
      }
      const uint32_t ra = ld_once_u32(sa + 896 + 4 * lane);
      const float ca = ld_f32(p.cos_sin + ta + lane);
      const float sna = ld_f32(p.cos_sin + ta + 32 + lane);
      uint4 xb0 = make_uint4(0, 0, 0, 0), xb1 = xb0;
      uint32_t rb = 0;
      float cb = 1.0f, snb = 0.0f;
      if (ib >= 0) {
        const uint8_t* sb = p.latent + (base + ib) * p.row_pitch;
        const int64_t tb = __shfl_sync(0xFFFFFFFFu, table_off, ib);
        if (lane < 28) {
          xb0 = ld_nc_v4(sb + 32 * lane);
          xb1 = ld_nc_v4(sb + 32 * lane + 16);
        }
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
        nvfp4_nope_tile(w ? xb0 : xa0, w ? xb1 : xa1, codes, scales, lane, scale_table, lane < 28);
        nvfp4_rotary_pair(w ? rb : ra, w ? cb : ca, w ? snb : sna, codes, scales, lane,
                          scale_table);
      }
    }
  }
}

int g_rope_occupancy[8][64];

template <typename Kernel>
int launch(Kernel k, int* occupancy, const RopeParams& p, cudaStream_t stream) {
  const int64_t chunks = (p.num_tokens + 31) / 32;
  const int64_t work_blocks = (chunks + kRopeWarps - 1) / kRopeWarps;
  const unsigned grid =
      grid_for(work_blocks, resident_blocks_per_sm(k, kRopeThreads, 0, occupancy));
  k<<<grid, kRopeThreads, 0, stream>>>(p);
  return launch_status();
}

enum class Kind { kMxfp8, kNvfp4, kV4, kPlainBf16, kPlainFp8 };

// E4M3 byte of a binary32 value as the satfinite conversion gives it: round
// to nearest even on a 3-bit fraction (subnormal step 2^-9), NaN -> 0x7F,
// magnitudes that reach 448 or beyond (infinities included) -> +-448.
inline uint32_t host_e4m3(float f) {
  if (f != f) return 0x7Fu;
  const uint32_t sign = std::signbit(f) ? 0x80u : 0u;
  const double a = std::fabs((double)f);
  if (a >= 448.0) return sign | 0x7Eu;
  if (a < 0.015625) return sign | (uint32_t)std::nearbyint(a * 512.0);  // 0..8
  int ex = 0;
  std::frexp(a, &ex);
  int e = ex - 1;                                      // a in [2^e, 2^(e+1))
  double m = std::nearbyint(std::ldexp(a, 3 - e));     // 8..16
  if (m == 16.0) {
    m = 8.0;
    e += 1;
  }
  return sign | (uint32_t)(((e + 7) << 3) | ((int)m - 8));
}

// How the plain fp8 rows divide by `scale` (Fp8Quotient), with yh and yl set
// for the product modes. A power of two with a normal reciprocal takes the
// product. Otherwise yh = RD(1/scale), yl = RN((1 - scale*yh) * yh) (the
// residual is exact), and the two-term rule is used only if it gives the
// division's E4M3 code for every bf16 pattern: an exhaustive check (65,536
// host iterations), run once per distinct scale. The answers for the last
// kFp8Cached distinct scales are kept (one word each: (scale bits << 2) |
// (mode + 1), replaced round robin), so that layers with different scales do
// not repeat the check on every call. Concurrent callers at worst repeat a
// check; every word they read is a complete answer.
constexpr int kFp8Cached = 8;
std::atomic<uint64_t> g_fp8_modes[kFp8Cached];
std::atomic<uint32_t> g_fp8_next{0};
std::atomic<int64_t> g_fp8_checks{0};

inline int32_t fp8_quotient_mode(float scale, float& yh, float& yl) {
  int ex = 0;
  if (std::frexp(scale, &ex) == 0.5f && ex >= -124 && ex <= 127) {
    yh = std::ldexp(1.0f, 1 - ex);
    yl = 0.0f;
    return kProduct;
  }
  yh = 1.0f / scale;
  if (std::fmaf(-scale, yh, 1.0f) < 0.0f) yh = std::nextafterf(yh, 0.0f);
  yl = std::fmaf(-scale, yh, 1.0f) * yh;
  uint32_t bits = 0;
  std::memcpy(&bits, &scale, 4);
  for (int k = 0; k < kFp8Cached; ++k) {
    const uint64_t seen = g_fp8_modes[k].load(std::memory_order_relaxed);
    if (seen != 0 && (seen >> 2) == bits) return (int32_t)(seen & 3u) - 1;
  }
  g_fp8_checks.fetch_add(1, std::memory_order_relaxed);
  int32_t mode = kTwoTerm;
  for (uint32_t b = 0; b < 65536u && mode == kTwoTerm; ++b) {
    const uint32_t w = b << 16;
    float x = 0.0f;
    std::memcpy(&x, &w, 4);
    const float q = x / scale;
    volatile float t = x * yl;
    if (host_e4m3(q) != host_e4m3(std::fmaf(x, yh, t))) mode = kDivide;
  }
  const uint32_t k = g_fp8_next.fetch_add(1, std::memory_order_relaxed) % kFp8Cached;
  g_fp8_modes[k].store(((uint64_t)bits << 2) | (uint64_t)(mode + 1), std::memory_order_relaxed);
  return mode;
}

// Checks shared by every insert; fills the fields of `p` that do not depend
// on the cache layout. KVQ_OK, or KVQ_EINVAL.
int common_args(const void* latent_bf16, int64_t num_tokens, int64_t row_stride_elems,
                const int64_t* positions, const float* cos_sin, int64_t cos_stride,
                int64_t cos_sin_rows, const void* cache, const int64_t* cache_slots,
                int64_t num_pages, int64_t cache_block, int32_t compress_ratio, RopeParams& p) {
  if (num_tokens < 0 || row_stride_elems < kLatent || row_stride_elems % 8 != 0) return KVQ_EINVAL;
  if (cos_stride < 64 || cos_stride % 4 != 0 || cos_sin_rows < 1) return KVQ_EINVAL;
  if (num_pages < 1 || cache_block < 1 || compress_ratio < 1) return KVQ_EINVAL;
  if (num_pages > INT64_MAX / cache_block) return KVQ_EINVAL;
  if (cos_sin_rows > INT64_MAX / cos_stride) return KVQ_EINVAL;
  if (num_tokens > INT64_MAX / 2 / row_stride_elems) return KVQ_EINVAL;
  if (num_tokens > 0) {
    if (!latent_bf16 || !positions || !cos_sin || !cache || !cache_slots) return KVQ_EINVAL;
    if (!aligned(latent_bf16, 16) || !aligned(cos_sin, 16) || !aligned(cache, 16) ||
        !aligned(positions, 8) || !aligned(cache_slots, 8))
      return KVQ_EINVAL;
  }
  p.latent = static_cast<const uint8_t*>(latent_bf16);
  p.row_pitch = row_stride_elems * 2;
  p.num_tokens = num_tokens;
  p.positions = positions;
  p.cos_sin = cos_sin;
  p.cos_stride = cos_stride;
  p.cos_rows = cos_sin_rows;
  p.cache = static_cast<uint8_t*>(const_cast<void*>(cache));
  p.slots = cache_slots;
  p.num_slots = num_pages * cache_block;
  p.cache_block = cache_block;
  p.ratio = compress_ratio;
  p.slot_pitch = 0;
  p.fp8_scale = 1.0f;
  p.fp8_mode = kDivide;
  p.fp8_yh = 1.0f;
  p.fp8_yl = 0.0f;
  return KVQ_OK;
}

int dispatch(Kind kind, bool sanitize, const RopeParams& p, cudaStream_t stream) {
  if (p.num_tokens == 0) return KVQ_OK;
  switch (kind) {
    case Kind::kNvfp4:
      return launch(nvfp4_insert_kernel, g_rope_occupancy[2], p, stream);
    case Kind::kMxfp8:
      return sanitize
                 ? launch(record_run_insert_kernel<Layout::kMxfp8, true>, g_rope_occupancy[1], p,
                          stream)
                 : launch(record_run_insert_kernel<Layout::kMxfp8, false>, g_rope_occupancy[0], p,
                          stream);
    case Kind::kV4:
      return sanitize
                 ? launch(record_run_insert_kernel<Layout::kV4, true>, g_rope_occupancy[4], p,
                          stream)
                 : launch(record_run_insert_kernel<Layout::kV4, false>, g_rope_occupancy[3], p,
                          stream);
    case Kind::kPlainBf16:
      return launch(fp8_family_insert_kernel<Layout::kPlainBf16, false>, g_rope_occupancy[5], p,
                    stream);
    default:
      return launch(record_run_insert_kernel<Layout::kPlainFp8, false>, g_rope_occupancy[6], p,
                    stream);
  }
}

// The paged records (MXFP8 528 B, NVFP4 288 B, V4 584 B): value bytes of the
// page's slots, then their scale bytes; pages page_stride_bytes apart.
int record_insert(Kind kind, const void* latent_bf16, int64_t num_tokens, int64_t row_stride_elems,
                  const int64_t* positions, const float* cos_sin, int64_t cos_stride,
                  int64_t cos_sin_rows, uint8_t* cache, const int64_t* cache_slots,
                  int64_t num_pages, int64_t cache_block, int64_t page_stride_bytes,
                  int32_t compress_ratio, int32_t sanitize_nans, cudaStream_t stream) {
  const int64_t record =
      kind == Kind::kNvfp4 ? kNvfp4Record : (kind == Kind::kV4 ? kV4Record : kMxfp8Record);
  RopeParams p;
  int st = common_args(latent_bf16, num_tokens, row_stride_elems, positions, cos_sin, cos_stride,
                       cos_sin_rows, cache, cache_slots, num_pages, cache_block, compress_ratio, p);
  if (st != KVQ_OK) return st;
  if (sanitize_nans != 0 && sanitize_nans != 1) return KVQ_EINVAL;
  if (cache_block > INT64_MAX / record || page_stride_bytes < cache_block * record ||
      page_stride_bytes % 16 != 0)
    return KVQ_EINVAL;
  if (num_pages > INT64_MAX / page_stride_bytes) return KVQ_EINVAL;
  p.page_stride = page_stride_bytes;
  return dispatch(kind, sanitize_nans != 0, p, stream);
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
  return kvq::record_insert(kvq::Kind::kMxfp8, latent_bf16, num_tokens, row_stride_elems,
                            positions, cos_sin, cos_stride, cos_sin_rows, cache, cache_slots,
                            num_pages, cache_block, page_stride_bytes, compress_ratio,
                            sanitize_nans, stream);
}

extern "C" int rope_quant_insert_nvfp4(const void* latent_bf16, int64_t num_tokens,
                                       int64_t row_stride_elems, const int64_t* positions,
                                       const float* cos_sin, int64_t cos_stride,
                                       int64_t cos_sin_rows, uint8_t* cache,
                                       const int64_t* cache_slots, int64_t num_pages,
                                       int64_t cache_block, int64_t page_stride_bytes,
                                       int32_t compress_ratio, int32_t sanitize_nans,
                                       cudaStream_t stream) {
  return kvq::record_insert(kvq::Kind::kNvfp4, latent_bf16, num_tokens, row_stride_elems,
                            positions, cos_sin, cos_stride, cos_sin_rows, cache, cache_slots,
                            num_pages, cache_block, page_stride_bytes, compress_ratio,
                            sanitize_nans, stream);
}

extern "C" int rope_quant_insert_v4(const void* latent_bf16, int64_t num_tokens,
                                    int64_t row_stride_elems, const int64_t* positions,
                                    const float* cos_sin, int64_t cos_stride, int64_t cos_sin_rows,
                                    uint8_t* cache, const int64_t* cache_slots, int64_t num_pages,
                                    int64_t cache_block, int64_t page_stride_bytes,
                                    int32_t compress_ratio, int32_t sanitize_nans,
                                    cudaStream_t stream) {
  return kvq::record_insert(kvq::Kind::kV4, latent_bf16, num_tokens, row_stride_elems, positions,
                            cos_sin, cos_stride, cos_sin_rows, cache, cache_slots, num_pages,
                            cache_block, page_stride_bytes, compress_ratio, sanitize_nans, stream);
}

extern "C" int kvq_plain_fp8_quotient_mode(float fp8_scale) {
  using namespace kvq;
  if (!(fp8_scale > 0.0f && fp8_scale <= 3.0e38f)) return KVQ_EINVAL;
  float yh = 1.0f, yl = 0.0f;
  return fp8_quotient_mode(fp8_scale, yh, yl);
}

extern "C" int64_t kvq_plain_fp8_checks_run(void) {
  return kvq::g_fp8_checks.load(std::memory_order_relaxed);
}

extern "C" int rope_plain_insert(const void* latent_bf16, int64_t num_tokens,
                                 int64_t row_stride_elems, const int64_t* positions,
                                 const float* cos_sin, int64_t cos_stride, int64_t cos_sin_rows,
                                 void* cache, const int64_t* cache_slots, int64_t num_pages,
                                 int64_t cache_block, int64_t page_stride_elems,
                                 int64_t slot_stride_elems, int32_t compress_ratio, int32_t fp8,
                                 float fp8_scale, cudaStream_t stream) {
  using namespace kvq;
  RopeParams p;
  int st = common_args(latent_bf16, num_tokens, row_stride_elems, positions, cos_sin, cos_stride,
                       cos_sin_rows, cache, cache_slots, num_pages, cache_block, compress_ratio, p);
  if (st != KVQ_OK) return st;
  if (fp8 != 0 && fp8 != 1) return KVQ_EINVAL;
  if (fp8 && !(fp8_scale > 0.0f && fp8_scale <= 3.0e38f)) return KVQ_EINVAL;
  const int64_t es = fp8 ? 1 : 2;  // bytes per element
  if (slot_stride_elems < kLatent || slot_stride_elems % 8 != 0 || page_stride_elems % 8 != 0)
    return KVQ_EINVAL;
  if (cache_block - 1 > (INT64_MAX / 4 - kLatent) / slot_stride_elems) return KVQ_EINVAL;
  if (page_stride_elems < (cache_block - 1) * slot_stride_elems + kLatent) return KVQ_EINVAL;
  if (num_pages > INT64_MAX / 4 / page_stride_elems) return KVQ_EINVAL;
  p.page_stride = page_stride_elems * es;
  p.slot_pitch = slot_stride_elems * es;
  p.fp8_scale = fp8 ? fp8_scale : 1.0f;
  if (fp8) p.fp8_mode = fp8_quotient_mode(fp8_scale, p.fp8_yh, p.fp8_yl);
  return dispatch(fp8 ? Kind::kPlainFp8 : Kind::kPlainBf16, false, p, stream);
}
