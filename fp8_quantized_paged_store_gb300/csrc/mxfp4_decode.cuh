// mxfp4_decode.cuh — MXFP4 row decode to bf16 by byte permutes, shared by the
// gather and the attention kernels.
//
// Every decoded value E2M1(code) * 2**(byte-127) has at most two significant
// bits, so it is exact in bf16 and can be assembled from bits: the bf16
// pattern of magnitude index i (1..7) is 0x3F00 + 64*i (0x3F00 for i = 1),
// and the scale adds (byte-127) << 7 to it while the result stays a normal
// bf16, i.e. for 2 <= byte <= 252. Per group the eight scaled patterns are
// packed into byte tables, and the codes themselves (masked to three bits)
// select from them with byte permutes: four values per pair of prmt. The
// code's sign bit is bit 3 of a nibble; prmt's sign-replicate mode copies a
// byte's top bit, so the signs of odd codes come straight from the code
// bytes and those of even codes from the code word shifted left by 4.
// Scale bytes 0, 1, 253, 254 (subnormal or overflowing results) and 255 (the
// E8M0 NaN, decoded as bf16 NaN 0x7FC0 for the whole group) take an
// arithmetic path.
#pragma once

#include <cstdint>

#include "kvq_device.cuh"

namespace kvq {
namespace {

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

struct ByteTables {
  uint32_t lo_a, lo_b, hi_a, hi_b;  // low / high bytes of scaled patterns 0..3, 4..7
};

// Scaled bf16 magnitude patterns for a scale byte in [2, 252].
__device__ __forceinline__ ByteTables make_tables(uint32_t scale_byte) {
  const uint32_t off = (uint32_t)(((int)scale_byte - 127) << 7);
  const uint32_t off2 = off * 0x00010001u;  // the same offset in both halves
  const uint32_t p01 = (0x3F00u + off) << 16;  // index 0 stays +0
  const uint32_t p23 = 0x3FC03F80u + off2;
  const uint32_t p45 = 0x40404000u + off2;
  const uint32_t p67 = 0x40C04080u + off2;
  ByteTables t;
  t.lo_a = prmt(p01, p23, 0x6420);
  t.hi_a = prmt(p01, p23, 0x7531);
  t.lo_b = prmt(p45, p67, 0x6420);
  t.hi_b = prmt(p45, p67, 0x7531);
  return t;
}

// Four codes (bits 16k..16k+15 of `c`) -> two bf16x2 words.
template <int k>
__device__ __forceinline__ void decode4(uint32_t c, uint32_t c_shl4, const ByteTables& t,
                                        uint32_t& w0, uint32_t& w1) {
  const uint32_t sel = (c >> (16 * k)) & 0x7777u;
  const uint32_t lo4 = prmt(t.lo_a, t.lo_b, sel);
  const uint32_t hi4 = prmt(t.hi_a, t.hi_b, sel);
  w0 = prmt(lo4, hi4, 0x5140);
  w1 = prmt(lo4, hi4, 0x7362);
  // byte 2k of c holds codes 4k (low nibble) and 4k+1; byte 2k+1 codes 4k+2, 4k+3.
  constexpr uint32_t s0 = ((8u | (2 * k)) << 12) | ((8u | (4 + 2 * k)) << 4);
  constexpr uint32_t s1 = ((8u | (2 * k + 1)) << 12) | ((8u | (4 + 2 * k + 1)) << 4);
  w0 |= prmt(c, c_shl4, s0) & 0x80008000u;
  w1 |= prmt(c, c_shl4, s1) & 0x80008000u;
}

// Arithmetic decode of one code for any scale byte.
__device__ __forceinline__ uint32_t decode_one_slow(uint32_t code, uint32_t scale_byte) {
  if (scale_byte == 255u) return 0x7FC0u;
  const uint32_t i = code & 7u;
  const uint64_t pats = 0x40C0408040404000ull;  // patterns of indices 7..4
  const uint64_t pats_lo = 0x3FC03F803F000000ull;  // indices 3..0
  const uint32_t mag_bits =
      (uint32_t)(((i < 4 ? pats_lo : pats) >> (16 * (i & 3))) & 0xFFFFu);
  const int k = (int)scale_byte - 127;  // -127..127
  const float pow2 = k >= -126 ? __uint_as_float((uint32_t)(k + 127) << 23)
                               : __uint_as_float(0x00400000u);
  const float v = __fmul_rn(__uint_as_float(mag_bits << 16), pow2);  // exact or +inf
  return (__float_as_uint(v) >> 16) | ((code & 8u) << 12);
}

__device__ __noinline__ uint4 decode8_slow(uint32_t c, uint32_t scale_byte) {
  uint32_t h[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) h[j] = decode_one_slow((c >> (4 * j)) & 0xFu, scale_byte);
  return make_uint4(h[0] | (h[1] << 16), h[2] | (h[3] << 16), h[4] | (h[5] << 16),
                    h[6] | (h[7] << 16));
}

// Eight codes of one group -> 16 bytes of bf16. `lut` holds make_tables(b)
// for every scale byte b in [2, 252] (built once per block).
__device__ __forceinline__ uint4 decode8(uint32_t c, uint32_t scale_byte, const uint4* lut) {
  if (scale_byte - 2u > 250u) return decode8_slow(c, scale_byte);
  const uint4 v = lds_v4(lut + scale_byte);
  ByteTables t;
  t.lo_a = v.x;
  t.hi_a = v.y;
  t.lo_b = v.z;
  t.hi_b = v.w;
  const uint32_t c4 = c << 4;
  uint4 r;
  decode4<0>(c, c4, t, r.x, r.y);
  decode4<1>(c, c4, t, r.z, r.w);
  return r;
}

// Eight codes of one group -> 16 bytes of bf16, by byte tables built in
// registers (no table in memory); for a scale byte in [2, 252] only, which
// the caller checks once per group.
__device__ __forceinline__ uint4 decode8_fast(uint32_t c, const ByteTables& t) {
  const uint32_t c4 = c << 4;
  uint4 r;
  decode4<0>(c, c4, t, r.x, r.y);
  decode4<1>(c, c4, t, r.z, r.w);
  return r;
}

}  // namespace
}  // namespace kvq
