// kvq_device.cuh — device helpers shared by the sm_103a kernels.
//
// Conversions use the Blackwell cvt.rn.satfinite.{e2m1x2,e4m3x2}.f32
// instructions. Their behaviour was checked exhaustively over all 2**32
// binary32 inputs on a GB300:
//   * e4m3x2: identical to clamp(x, -448, 448) followed by round-to-nearest-
//     even onto E4M3 with gradual underflow; the sign of zero is kept; every
//     NaN becomes 0x7F. This is exactly the MXFP8 record's value rule.
//   * e2m1x2: identical to the E2M1 midpoint rule (ties to the even code,
//     saturation above 6) with the sign taken from the sign bit, so -0.0
//     gives code 8 and every NaN gives code 7. The MXFP4/NVFP4 rule sets the
//     sign only for values that compare below zero and gives NaN code 0, so
//     callers remove -0.0 and NaN before converting (see the kernels).
//   * In both, the first source operand lands in the high nibble / byte.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace kvq {

constexpr int kLatent = 512;
constexpr int kMxfp4RowBytes = 272;  // 512/2 code bytes + 16 scale bytes
constexpr int kMxfp8Record = 528;    // 512 value bytes + 16 scale bytes
constexpr int kNvfp4Record = 288;    // 256 code bytes + 32 scale bytes

// ---------------------------------------------------------------- memory ---

// 16-byte load of data read exactly once (latent rows): bypass L1.
__device__ __forceinline__ uint4 ld_once_v4(const void* p) {
  uint4 r;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
      : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
      : "l"(p));
  return r;
}

// Read-only 16-byte load that allocates in L1: for sectors that the next
// load of the same warp touches again.
__device__ __forceinline__ uint4 ld_nc_v4(const void* p) {
  uint4 r;
  asm("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
      : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
      : "l"(p));
  return r;
}

__device__ __forceinline__ int64_t ld_once_i64(const int64_t* p) {
  int64_t r;
  asm("ld.global.nc.L1::no_allocate.s64 %0, [%1];" : "=l"(r) : "l"(p));
  return r;
}

__device__ __forceinline__ uint32_t ld_once_u32(const void* p) {
  uint32_t r;
  asm("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(r) : "l"(p));
  return r;
}

__device__ __forceinline__ float ld_f32(const float* p) {
  float r;
  asm("ld.global.nc.f32 %0, [%1];" : "=f"(r) : "l"(p));
  return r;
}

__device__ __forceinline__ uint32_t ld_u32(const void* p) {
  uint32_t r;
  asm("ld.global.nc.u32 %0, [%1];" : "=r"(r) : "l"(p));
  return r;
}

__device__ __forceinline__ uint32_t ld_u8(const void* p) {
  uint32_t r;
  asm("ld.global.nc.u8 %0, [%1];" : "=r"(r) : "l"(p));
  return r;
}

__device__ __forceinline__ float4 ld_f4(const float* p) {
  float4 r;
  asm("ld.global.nc.v4.f32 {%0, %1, %2, %3}, [%4];"
      : "=f"(r.x), "=f"(r.y), "=f"(r.z), "=f"(r.w)
      : "l"(p));
  return r;
}

__device__ __forceinline__ void st_u32(void* p, uint32_t v) {
  asm volatile("st.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ void st_v2(void* p, uint32_t a, uint32_t b) {
  asm volatile("st.global.v2.u32 [%0], {%1, %2};" ::"l"(p), "r"(a), "r"(b) : "memory");
}

__device__ __forceinline__ void st_v4(void* p, uint4 v) {
  asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}

__device__ __forceinline__ void st_u8(void* p, uint32_t v) {
  asm volatile("st.global.u8 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// ------------------------------------------------------------- cp.async ---

// 16-byte asynchronous global -> shared copy, L2 only. Completion is tracked
// per thread with commit groups, so a thread that later reads back only the
// bytes it copied needs no barrier besides cp.async.wait_group.
__device__ __forceinline__ void cp_async_16(void* smem_dst, const void* gmem_src) {
  const uint32_t d = (uint32_t)__cvta_generic_to_shared(smem_dst);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(gmem_src) : "memory");
}

__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}

// Wait until at most n of this thread's most recent commit groups are pending.
template <int n>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(n) : "memory");
}

__device__ __forceinline__ uint4 lds_v4(const uint4* p) {
  uint4 r;
  const uint32_t a = (uint32_t)__cvta_generic_to_shared(p);
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "r"(a)
               : "memory");
  return r;
}

__device__ __forceinline__ uint32_t lds_u32(const void* p) {
  uint32_t r;
  const uint32_t a = (uint32_t)__cvta_generic_to_shared(p);
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(r) : "r"(a) : "memory");
  return r;
}

__device__ __forceinline__ uint32_t lds_u8(const void* p) {
  uint32_t r;
  const uint32_t a = (uint32_t)__cvta_generic_to_shared(p);
  asm volatile("ld.shared.u8 %0, [%1];" : "=r"(r) : "r"(a) : "memory");
  return r;
}

// ------------------------------------------------------------ bf16 words ---

// Low / high bf16 of a bf16x2 word widened to binary32 (exact).
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Packed binary32 pairs: one instruction rounds two IEEE products or fused
// multiply-adds to nearest, each result equal to the scalar one. Only for
// products that no later addition consumes: the compiler may fuse a packed
// product into a packed sum, which the scalar __fmul_rn never allows.
__device__ __forceinline__ float2 mul2_rn(float2 a, float2 b) {
  float2 d;
  asm("{\n .reg .b64 a, b, d;\n mov.b64 a, {%2, %3};\n mov.b64 b, {%4, %5};\n"
      " mul.rn.f32x2 d, a, b;\n mov.b64 {%0, %1}, d;\n}"
      : "=f"(d.x), "=f"(d.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}
__device__ __forceinline__ float2 add2_rn(float2 a, float2 b) {
  float2 d;
  asm("{\n .reg .b64 a, b, d;\n mov.b64 a, {%2, %3};\n mov.b64 b, {%4, %5};\n"
      " add.rn.f32x2 d, a, b;\n mov.b64 {%0, %1}, d;\n}"
      : "=f"(d.x), "=f"(d.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}
__device__ __forceinline__ float2 fma2_rn(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{\n .reg .b64 a, b, c, d;\n mov.b64 a, {%2, %3};\n mov.b64 b, {%4, %5};\n"
      " mov.b64 c, {%6, %7};\n fma.rn.f32x2 d, a, b, c;\n mov.b64 {%0, %1}, d;\n}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}

// Per-half max of |a|, |b| (NaN ignored unless both are NaN); the sign bits of
// the result are the XOR of the inputs' and carry no meaning here.
__device__ __forceinline__ uint32_t bf16x2_maxabs(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// As bf16x2_maxabs, but NaN-propagating: a half is NaN if either input is.
__device__ __forceinline__ uint32_t bf16x2_maxabs_nan(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.NaN.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

__device__ __forceinline__ uint32_t bf16x2_max(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// Per half: 0xFFFF where the value is a number other than +-0, else 0. AND-ing
// a word with it turns NaN and -0.0 into +0.0 and leaves every other value.
__device__ __forceinline__ uint32_t bf16x2_nonzero_number_mask(uint32_t w) {
  uint32_t m;
  asm("set.ne.u32.bf16x2 %0, %1, %2;" : "=r"(m) : "r"(w), "r"(0u));
  return m;
}

// Per half: 0xFFFF where the value is not NaN. AND-ing a word with it turns
// NaN into +0.0 and leaves every other value (including -0.0).
__device__ __forceinline__ uint32_t bf16x2_number_mask(uint32_t w) {
  uint32_t m;
  asm("set.num.u32.bf16x2 %0, %1, %1;" : "=r"(m) : "r"(w));
  return m;
}

// ----------------------------------------------------------- conversions ---

// Two binary32 -> one byte of two E2M1 codes, `lo` in bits 3:0.
__device__ __forceinline__ uint32_t cvt_e2m1x2(float lo, float hi) {
  uint32_t r;
  asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u32.u8 %0, t;\n\t}"
      : "=r"(r)
      : "f"(hi), "f"(lo));
  return r;
}

// Eight binary32 -> 32 bits of E2M1 codes, element k in bits 4k+3:4k.
__device__ __forceinline__ uint32_t cvt_e2m1x8(float f0, float f1, float f2, float f3, float f4,
                                               float f5, float f6, float f7) {
  uint32_t r;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
      "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
      : "=r"(r)
      : "f"(f0), "f"(f1), "f"(f2), "f"(f3), "f"(f4), "f"(f5), "f"(f6), "f"(f7));
  return r;
}

// Two binary32 -> 16 bits of E4M3 (saturating, NaN -> 0x7F), `lo` in 7:0.
__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// ------------------------------------------------------------- exponents ---

// Exact 2**-e as binary32 for -126 <= e <= 128 (2**-127 and 2**-128 are
// subnormal powers of two).
__device__ __forceinline__ float exp2_neg(int e) {
  return e <= 126 ? __uint_as_float((uint32_t)(127 - e) << 23)
                  : __uint_as_float(0x00400000u >> (e - 127));
}

// Smallest e with 2**e >= v, from the binary32 fields of v > 0: the unbiased
// exponent, plus one when the fraction is non-zero (field 0 gives -126).
__device__ __forceinline__ int ceil_pow2_exponent(float v) {
  uint32_t u = __float_as_uint(v);
  return (int)((u >> 23) & 0xFFu) - 127 + ((u & 0x7FFFFFu) != 0u ? 1 : 0);
}

// MXFP4 group exponent from the bf16 bits of the group's |amax|:
// ceil(log2(RN32(amax/6))) read off the binary32 bits, without dividing.
// amax = (1 + m/128) * 2**E; amax/6 = ((1 + m/128)/1.5) * 2**(E-2). The
// factor is below 1 when m < 64, exactly 1 when m == 64, above 1 (but below
// 4/3, and never rounded down to 1) when m > 64. Hence e = E - 2 + (m > 64)
// while amax/6 is a normal binary32, and -126 (fraction field non-zero,
// exponent field 0) below that, so e = max(E - 2 + (m > 64), -126), which
// also covers bf16 subnormal amax. 0 for amax == 0 (zero group), 128 for +inf
// (inf/6 = inf has field 255 and fraction 0), 0 for NaN (all-NaN group: NaN is
// ignored, so amax folds to 0).
__device__ __forceinline__ int mxfp4_group_exponent(uint32_t amax_bits) {
  uint32_t a = amax_bits & 0x7FFFu;
  if (a == 0u || a > 0x7F80u) return 0;
  if (a == 0x7F80u) return 128;
  int e = (int)(a >> 7) - 129 + ((a & 0x7Fu) > 0x40u ? 1 : 0);
  return e < -126 ? -126 : e;
}

// 64-bit quotient and remainder by a positive divisor, through 32-bit
// division when both operands fit (much cheaper on the GPU).
__device__ __forceinline__ void divmod_pos(int64_t n, int64_t d, int64_t& q, int64_t& r) {
  if (((uint64_t)n | (uint64_t)d) <= 0xFFFFFFFFull) {
    uint32_t q32 = (uint32_t)n / (uint32_t)d;
    q = q32;
    r = (int64_t)((uint32_t)n - q32 * (uint32_t)d);
  } else {
    q = n / d;
    r = n - q * d;
  }
}

}  // namespace kvq
