// mxfp4_store.cu — mxfp4_mla_store: quantize bf16 MLA latent rows to MXFP4
// and scatter them into a paged cache of 272-byte rows.
//
// Follows "vllm.v1.attention.ops.mxfp4_mla.store" (store_mxfp4_mla,
// _ceil_pow2_exponent, _quantize_e2m1) and PR 60321 "Add an mxfp4_mla KV cache
// for rope-free sparse MLA" (Details: format and write path).
//
// Work decomposition (GB300: 152 SMs, HBM-bound streaming codec):
//   * one wave of 256-thread blocks; each warp owns a contiguous token range;
//   * lane i reads slot_mapping of token i of a 32-token window once and turns
//     it into the row's byte offset (one division per lane per window);
//   * rows stream through a per-warp shared-memory ring filled by cp.async
//     three rows ahead of the row being quantized (pad tokens issue no copy);
//     with 32 KiB of ring per block, six blocks (48 warps, ~144 KiB of loads
//     in flight) fit an SM, which measured faster than four rows ahead with
//     five blocks, or two rows ahead;
//   * one row is 1 KiB; in the store lane l holds the run of elements
//     16l..16l+15 (two 16-byte copies, bytes 32l and 32l+16), so a group of
//     32 is two lanes' runs; the RMSNorm-fused store holds elements 8l..8l+7
//     (half 0, groups 0..7) and 256+8l..256+8l+7 (half 1, groups 8..15),
//     the order its sum of squares is defined in, a group over four lanes;
//   * group amax: bf16x2 max-of-magnitudes (NaN ignored) within the lane, then
//     one xor-shuffle (runs) or two across four lanes with both halves packed
//     in one word (halves);
//   * the E8M0 exponent comes from the amax bits without a division;
//   * values are scaled by the exact power 2**-e in binary32 and converted
//     by cvt.rn.satfinite.e2m1x2.f32 (NaN and -0.0 are cleared first);
//   * each lane stores its eight code bytes in one store and every other lane
//     its group's scale byte (runs), or two 4-byte code words and every
//     fourth lane two scale bytes (halves).
#include <cmath>
#include <cstdint>

#include "kvq.h"
#include "kvq_device.cuh"
#include "kvq_host.h"

namespace kvq {
namespace {

constexpr int kStoreWarps = 8;
constexpr int kStoreThreads = 32 * kStoreWarps;

struct StoreParams {
  const uint8_t* latent;    // row t starts at latent + t * row_pitch
  int64_t row_pitch;        // bytes
  int64_t num_tokens;
  const int64_t* slots;
  uint8_t* cache;           // this layer's view
  int64_t num_slots;        // num_blocks * block_size
  int64_t block_size;
  int64_t block_stride_rows;
  const uint8_t* weight;  // RMSNorm weight, bf16 [512] (fused variant only)
  float eps;
  // warp w's tokens: per_warp, plus one for w < extra (set at launch, so
  // that no warp divides 64-bit numbers: a runtime call that costs the
  // kernel ~1.5% through its registers)
  int64_t per_warp, extra;
};

// Eight bf16 (one 16-byte load) of a group with scale 2**e -> eight E2M1
// codes, element k in bits 4k+3:4k.
//
// The conversion takes the sign from the sign bit (-0.0 -> code 8) and maps
// NaN to code 7, where the E2M1 rule gives both code 0. Fast path (the row
// holds no NaN or infinity and every group exponent is <= 16): the scaled
// value is fma(x, 2**-e, +0.0), which equals RN(x * 2**-e) except that -0.0
// becomes +0.0; a product of a non-zero bf16 (magnitude >= 2**-133) and
// 2**-e >= 2**-16 never underflows to zero, so no other -0.0 can appear.
// Special path: NaN and -0.0 inputs are cleared to +0.0 first, the product is
// rounded on its own and then +0.0 is added, which turns an underflowed
// -0.0 (possible when e >= 17) into +0.0 and changes nothing else.
template <bool kSpecial, bool kPacked>
__device__ __forceinline__ uint32_t encode8(uint4 w, float inv_scale) {
  if (kSpecial) {
    w.x &= bf16x2_nonzero_number_mask(w.x);
    w.y &= bf16x2_nonzero_number_mask(w.y);
    w.z &= bf16x2_nonzero_number_mask(w.z);
    w.w &= bf16x2_nonzero_number_mask(w.w);
  }
  float f[8] = {bf16_lo(w.x), bf16_hi(w.x), bf16_lo(w.y), bf16_hi(w.y),
                bf16_lo(w.z), bf16_hi(w.z), bf16_lo(w.w), bf16_hi(w.w)};
  if (kSpecial) {
#pragma unroll
    for (int k = 0; k < 8; ++k) f[k] = __fadd_rn(__fmul_rn(f[k], inv_scale), 0.0f);
  } else if (!kPacked) {
#pragma unroll
    for (int k = 0; k < 8; ++k) f[k] = __fmaf_rn(f[k], inv_scale, 0.0f);
  } else {
    const float2 i2 = make_float2(inv_scale, inv_scale), z2 = make_float2(0.0f, 0.0f);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 q = fma2_rn(make_float2(f[2 * k], f[2 * k + 1]), i2, z2);
      f[2 * k] = q.x;
      f[2 * k + 1] = q.y;
    }
  }
  return cvt_e2m1x8(f[0], f[1], f[2], f[3], f[4], f[5], f[6], f[7]);
}

// Per-lane |amax| of a half row as bf16 bits, in the low (half 0) and high
// (half 1) 16 bits, folded over the four lanes of each group.
template <bool kNanPropagating>
__device__ __forceinline__ uint32_t group_amax2(uint4 x0, uint4 x1) {
  auto mx = [](uint32_t a, uint32_t b) {
    return kNanPropagating ? bf16x2_maxabs_nan(a, b) : bf16x2_maxabs(a, b);
  };
  const uint32_t m0 = mx(mx(x0.x, x0.y), mx(x0.z, x0.w));
  const uint32_t m1 = mx(mx(x1.x, x1.y), mx(x1.z, x1.w));
  uint32_t g = mx(__byte_perm(m0, m1, 0x5410), __byte_perm(m0, m1, 0x7632));
  g &= 0x7FFF7FFFu;
  auto mg = [](uint32_t a, uint32_t b) {
    return kNanPropagating ? bf16x2_maxabs_nan(a, b) : bf16x2_max(a, b);
  };
  g = mg(g, __shfl_xor_sync(0xFFFFFFFFu, g, 1));
  g = mg(g, __shfl_xor_sync(0xFFFFFFFFu, g, 2));
  return g & 0x7FFF7FFFu;
}

// |amax| of this lane's group as bf16 bits (low 16 bits) when the lane holds a
// run of 16 consecutive values (x0, x1) and a group of 32 is two lanes' runs:
// the maximum over the run, then one xor-shuffle.
template <bool kNanPropagating>
__device__ __forceinline__ uint32_t run_group_amax(uint4 x0, uint4 x1) {
  auto mx = [](uint32_t a, uint32_t b) {
    return kNanPropagating ? bf16x2_maxabs_nan(a, b) : bf16x2_maxabs(a, b);
  };
  uint32_t m = mx(mx(mx(x0.x, x0.y), mx(x0.z, x0.w)), mx(mx(x1.x, x1.y), mx(x1.z, x1.w)));
  m = mx(m, __byte_perm(m, m, 0x1032)) & 0x7FFF7FFFu;
  auto mg = [](uint32_t a, uint32_t b) {
    return kNanPropagating ? bf16x2_maxabs_nan(a, b) : bf16x2_max(a, b);
  };
  m = mg(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
  return m & 0x7FFFu;
}

// Group exponent for a finite amax (bf16 bits a < 0x7F80): the closed form of
// mxfp4_group_exponent without its NaN and infinity cases. (a + 0x3F) >> 7
// adds 1 to the exponent field exactly when the 7-bit mantissa exceeds 0x40.
__device__ __forceinline__ int finite_group_exponent(uint32_t a) {
  const int e = (int)((a + 0x3Fu) >> 7) - 129;
  return a == 0u ? 0 : (e < -126 ? -126 : e);
}

// Quantize one row held by the warp as halves (x0: half 0, x1: half 1; the
// RMSNorm-fused store) and write its 272 bytes at dst.
__device__ __forceinline__ void quantize_store_row(uint4 x0, uint4 x1, uint8_t* dst, int lane) {
  const uint32_t g = group_amax2<true>(x0, x1);
  const uint32_t a0 = g & 0xFFFFu, a1 = g >> 16;
  int e0 = finite_group_exponent(a0);  // group lane/4
  int e1 = finite_group_exponent(a1);  // group 8 + lane/4
  uint32_t c0, c1;
  const bool special = (a0 >= 0x7F80u) | (a1 >= 0x7F80u) | (e0 > 16) | (e1 > 16);
  if (__any_sync(0xFFFFFFFFu, special)) {
    const uint32_t gi = group_amax2<false>(x0, x1);  // NaN ignored
    e0 = mxfp4_group_exponent(gi & 0xFFFFu);
    e1 = mxfp4_group_exponent(gi >> 16);
    c0 = encode8<true, false>(x0, exp2_neg(e0));
    c1 = encode8<true, false>(x1, exp2_neg(e1));
  } else {
    c0 = encode8<false, false>(x0, __uint_as_float((uint32_t)(127 - e0) << 23));
    c1 = encode8<false, false>(x1, __uint_as_float((uint32_t)(127 - e1) << 23));
  }
  st_u32(dst + 4 * lane, c0);
  st_u32(dst + 128 + 4 * lane, c1);
  if ((lane & 3) == 0) {
    st_u8(dst + 256 + (lane >> 2), (uint32_t)(e0 + 127));
    st_u8(dst + 264 + (lane >> 2), (uint32_t)(e1 + 127));
  }
}

// Quantize one row held by the warp as runs (lane l: elements 16l..16l+15 in
// x0, x1; group l/2) and write its 272 bytes at dst: eight code bytes per
// lane in one store, one scale byte per even lane. The fast path scales two
// values per packed fused multiply-add. Against the halves mapping (a group
// over four lanes, two shuffles, two code stores per lane; scalar products)
// this measured 1.082 -> 1.065 ms (packed products) and 1.040 -> 1.017 ms
// (runs) on 4,300,000 rows; the RMSNorm-fused store measured slower with
// packed products (1.086 -> 1.115 ms) and keeps the halves, the order its
// sum of squares is defined in.
__device__ __forceinline__ void quantize_store_run(uint4 x0, uint4 x1, uint8_t* dst, int lane) {
  const uint32_t a = run_group_amax<true>(x0, x1);
  int e = finite_group_exponent(a);
  uint32_t c0, c1;
  if (__any_sync(0xFFFFFFFFu, (a >= 0x7F80u) | (e > 16))) {
    e = mxfp4_group_exponent(run_group_amax<false>(x0, x1));  // NaN ignored
    const float inv = exp2_neg(e);
    c0 = encode8<true, false>(x0, inv);
    c1 = encode8<true, false>(x1, inv);
  } else {
    const float inv = __uint_as_float((uint32_t)(127 - e) << 23);
    c0 = encode8<false, true>(x0, inv);
    c1 = encode8<false, true>(x1, inv);
  }
  st_v2(dst + 8 * lane, c0, c1);
  if ((lane & 1) == 0) st_u8(dst + 256 + (lane >> 1), (uint32_t)(e + 127));
}

// RMSNorm of one row held by the warp (fused variant), in the order the
// library's interface fixes: block k = elements 8k..8k+7 then
// 256+8k..256+8k+7, its squares summed left to right, then a balanced
// pairwise tree over the 32 block sums in block order; every square and sum
// rounded to binary32. Here block k is exactly lane k's two 16-byte pieces,
// and the xor-butterfly over strides 1, 2, 4, 8, 16 adds the same operands
// as that tree (each step's two addends are the sums of neighbouring
// subtrees, and the addition commutes, so every lane ends with the tree's
// bits). Then r = RN(1 / RN(sqrt(S / 512 + eps))) with correctly rounded
// square root and reciprocal, y = bf16(x * r) and z = bf16(y * w). A bf16
// product is exact in binary32, so mul.rn.bf16x2 rounds it once.
__device__ __forceinline__ uint32_t bf16x2_from_f32(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}

__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

__device__ __forceinline__ void rmsnorm_row(uint4& x0, uint4& x1, const uint4& w0, const uint4& w1,
                                            float eps) {
  const uint32_t xw[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
  float v[16];
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    v[2 * k] = bf16_lo(xw[k]);
    v[2 * k + 1] = bf16_hi(xw[k]);
  }
  float acc = 0.0f;
#pragma unroll
  for (int k = 0; k < 16; ++k) acc = __fadd_rn(acc, __fmul_rn(v[k], v[k]));
#pragma unroll
  for (int stride = 1; stride < 32; stride *= 2)
    acc = __fadd_rn(acc, __shfl_xor_sync(0xFFFFFFFFu, acc, stride));
  const float r = __frcp_rn(__fsqrt_rn(__fadd_rn(__fmul_rn(acc, 0x1p-9f), eps)));
  const uint32_t ww[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
  uint32_t z[8];
#pragma unroll
  for (int k = 0; k < 8; ++k)
    z[k] = bf16x2_mul(bf16x2_from_f32(__fmul_rn(v[2 * k], r), __fmul_rn(v[2 * k + 1], r)), ww[k]);
  x0 = make_uint4(z[0], z[1], z[2], z[3]);
  x1 = make_uint4(z[4], z[5], z[6], z[7]);
}

// Prefetch distance (rows per warp in flight) and ring stages: one more stage
// than the distance, so the copy issued at the top of an iteration never
// lands in the stage being read in that iteration.
constexpr int kPrefetch = 3;
constexpr int kStages = kPrefetch + 1;
constexpr int kStageVecs = 64;  // one 1 KiB row = 64 x 16 bytes
constexpr size_t kStoreSmem = (size_t)kStoreWarps * kStages * kStageVecs * sizeof(uint4);

// Cache row index of token t (rows of 272 bytes from the view's base), or
// 0xFFFFFFFF to skip it (pad, outside the cache, or past the warp's range).
// The host guarantees that row indices fit in 32 bits.
template <bool kFlat>
__device__ __forceinline__ uint32_t row_index(const StoreParams& p, int64_t t, int64_t t_end) {
  if (t >= t_end) return 0xFFFFFFFFu;
  const int64_t s = ld_once_i64(p.slots + t);
  if (s < 0 || s >= p.num_slots) return 0xFFFFFFFFu;
  if (kFlat) return (uint32_t)s;
  int64_t blk, in_blk;
  divmod_pos(s, p.block_size, blk, in_blk);
  return (uint32_t)(blk * p.block_stride_rows + in_blk);
}

// Each warp owns a contiguous token range and streams its rows through a
// per-warp shared-memory ring with cp.async, kPrefetch rows ahead of the row
// it quantizes. Lane l copies, and later reads back, only its own bytes of
// each row (32l..32l+31 for runs; 16l..16l+15 and 512+16l..512+16l+15 for
// halves), so the per-thread commit groups alone order the ring: no barrier
// and no spin-wait. Row indices come 32 tokens at
// a time (lane i holds token base+i); the window after the current one is
// loaded early so that prefetches crossing into it find their indices ready.
// The loop is unrolled over the ring's stages so that stage offsets are
// constants.
template <bool kFlat, bool kNorm>
__global__ void __launch_bounds__(kStoreThreads) mxfp4_store_kernel(StoreParams p) {
  extern __shared__ uint4 smem[];
  const int lane = threadIdx.x & 31;
  const int warp_in_block = threadIdx.x >> 5;
  // the plain store holds runs (lane l: bytes 32l..32l+31 of a row); the
  // RMSNorm-fused one halves (bytes 16l..16l+15 and 512+16l..512+16l+15), the
  // order its sum of squares is defined in
  constexpr bool kRuns = !kNorm;
  uint4* ring = smem + warp_in_block * (kStages * kStageVecs) + (kRuns ? 2 * lane : lane);
  const int64_t warp = (int64_t)blockIdx.x * kStoreWarps + warp_in_block;
  const int64_t t_begin = warp * p.per_warp + (warp < p.extra ? warp : p.extra);
  const int64_t t_end = t_begin + p.per_warp + (warp < p.extra ? 1 : 0);
  const int n = (int)(t_end - t_begin);  // < 2**31, checked at launch
  if (n <= 0) return;
  const uint8_t* src = p.latent + t_begin * p.row_pitch + (kRuns ? 32 : 16) * lane;
  const uint32_t pitch = (uint32_t)p.row_pitch;
  uint4 wt0 = make_uint4(0, 0, 0, 0), wt1 = wt0;  // the lane's RMSNorm weights
  if (kNorm) {
    wt0 = ld_once_v4(p.weight + 16 * lane);
    wt1 = ld_once_v4(p.weight + 512 + 16 * lane);
  }

  uint32_t w0 = row_index<kFlat>(p, t_begin + lane, t_end);       // tokens [0, 32)
  uint32_t w1 = row_index<kFlat>(p, t_begin + 32 + lane, t_end);  // tokens [32, 64)

  auto issue = [&](int i, int stage, uint32_t row) {
    if (row != 0xFFFFFFFFu) {
      const uint8_t* s = src + (size_t)i * pitch;
      cp_async_16(ring + stage * kStageVecs, s);
      cp_async_16(ring + stage * kStageVecs + (kRuns ? 1 : 32), s + (kRuns ? 16 : 512));
    }
    cp_async_commit();
  };
#pragma unroll
  for (int d = 0; d < kPrefetch; ++d) issue(d, d, __shfl_sync(0xFFFFFFFFu, w0, d));

  for (int i0 = 0; i0 < n; i0 += kStages) {
#pragma unroll
    for (int u = 0; u < kStages; ++u) {
      const int i = i0 + u;
      if (i < n) {
        const int k = i & 31;
        if (k == 0 && i > 0) {  // next window of 32 tokens
          w0 = w1;
          w1 = row_index<kFlat>(p, t_begin + i + 32 + lane, t_end);
        }
        // prefetch row i + kPrefetch into the stage read kPrefetch rows later
        const int kp = k + kPrefetch;
        const uint32_t rp = __shfl_sync(0xFFFFFFFFu, kp < 32 ? w0 : w1, kp & 31);
        issue(i + kPrefetch, (u + kPrefetch) % kStages,
              i + kPrefetch < n ? rp : 0xFFFFFFFFu);
        cp_async_wait<kPrefetch>();  // row i has landed
        const uint32_t row = __shfl_sync(0xFFFFFFFFu, w0, k);
        if (row != 0xFFFFFFFFu) {
          uint4 x0 = lds_v4(ring + u * kStageVecs);
          uint4 x1 = lds_v4(ring + u * kStageVecs + (kRuns ? 1 : 32));
          if (kNorm) rmsnorm_row(x0, x1, wt0, wt1, p.eps);
          if (kRuns)
            quantize_store_run(x0, x1, p.cache + (size_t)row * kMxfp4RowBytes, lane);
          else
            quantize_store_row(x0, x1, p.cache + (size_t)row * kMxfp4RowBytes, lane);
        }
      }
    }
  }
  cp_async_wait<0>();
}

int g_store_occupancy[4][64];

}  // namespace
}  // namespace kvq

namespace kvq {
namespace {

int store_entry(const void* latent_bf16, int64_t num_tokens, int64_t latent_dim,
                int64_t row_stride_elems, const void* weight_bf16, float eps, bool norm,
                const int64_t* slot_mapping, uint8_t* cache, int64_t num_blocks, int64_t block_size,
                int64_t block_stride_rows, int32_t group, cudaStream_t stream) {
  if (latent_dim != kLatent || group != 32) return KVQ_EINVAL;
  if (num_tokens < 0 || num_blocks < 1 || block_size < 1 || block_stride_rows < block_size)
    return KVQ_EINVAL;
  if (row_stride_elems < latent_dim || row_stride_elems % 8 != 0) return KVQ_EINVAL;
  // The cache view must be addressable without int64 overflow.
  if (num_blocks > INT64_MAX / block_stride_rows / kMxfp4RowBytes) return KVQ_EINVAL;
  if (num_blocks > INT64_MAX / block_size) return KVQ_EINVAL;
  if (num_tokens > INT64_MAX / 2 / row_stride_elems) return KVQ_EINVAL;
  // cache rows are addressed with 32-bit indices (2**32 rows would be 1.1 TB)
  if ((num_blocks - 1) * block_stride_rows + block_size > (int64_t)0xFFFFFFFE) return KVQ_EINVAL;
  if (row_stride_elems * 2 > (int64_t)0xFFFFFFFF) return KVQ_EINVAL;
  if (norm && !(eps >= 0.0f && eps < INFINITY)) return KVQ_EINVAL;
  if (num_tokens == 0) return KVQ_OK;
  if (!latent_bf16 || !slot_mapping || !cache || (norm && !weight_bf16)) return KVQ_EINVAL;
  if (!aligned(latent_bf16, 16) || !aligned(cache, 16) || !aligned(slot_mapping, 8))
    return KVQ_EINVAL;
  if (norm && !aligned(weight_bf16, 16)) return KVQ_EINVAL;

  StoreParams p;
  p.latent = static_cast<const uint8_t*>(latent_bf16);
  p.row_pitch = row_stride_elems * 2;
  p.num_tokens = num_tokens;
  p.slots = slot_mapping;
  p.cache = cache;
  p.num_slots = num_blocks * block_size;
  p.block_size = block_size;
  p.block_stride_rows = block_stride_rows;
  p.weight = static_cast<const uint8_t*>(weight_bf16);
  p.eps = eps;

  const bool flat = (num_blocks == 1) || (block_stride_rows == block_size);
  // at least 32 tokens per warp on average, at most one wave of blocks
  const int64_t work_blocks = (num_tokens + 32 * kStoreWarps - 1) / (32 * kStoreWarps);
  auto k = norm ? (flat ? mxfp4_store_kernel<true, true> : mxfp4_store_kernel<false, true>)
                : (flat ? mxfp4_store_kernel<true, false> : mxfp4_store_kernel<false, false>);
  const unsigned grid =
      grid_for(work_blocks, resident_blocks_per_sm(k, kStoreThreads, kStoreSmem,
                                                   g_store_occupancy[2 * norm + flat]));
  // each warp's token count must fit the kernel's 32-bit loop counter
  if (num_tokens / ((int64_t)grid * kStoreWarps) >= (int64_t)0x7FFFFFFF) return KVQ_EINVAL;
  p.per_warp = num_tokens / ((int64_t)grid * kStoreWarps);
  p.extra = num_tokens - p.per_warp * ((int64_t)grid * kStoreWarps);
  k<<<grid, kStoreThreads, kStoreSmem, stream>>>(p);
  return launch_status();
}

}  // namespace
}  // namespace kvq

extern "C" int mxfp4_mla_store(const void* latent_bf16, int64_t num_tokens, int64_t latent_dim,
                               int64_t row_stride_elems, const int64_t* slot_mapping,
                               uint8_t* cache, int64_t num_blocks, int64_t block_size,
                               int64_t block_stride_rows, int32_t group, cudaStream_t stream) {
  return kvq::store_entry(latent_bf16, num_tokens, latent_dim, row_stride_elems, nullptr, 0.0f,
                          false, slot_mapping, cache, num_blocks, block_size, block_stride_rows,
                          group, stream);
}

extern "C" int mxfp4_mla_rmsnorm_store(const void* latent_bf16, int64_t num_tokens,
                                       int64_t latent_dim, int64_t row_stride_elems,
                                       const void* weight_bf16, float eps,
                                       const int64_t* slot_mapping, uint8_t* cache,
                                       int64_t num_blocks, int64_t block_size,
                                       int64_t block_stride_rows, int32_t group,
                                       cudaStream_t stream) {
  return kvq::store_entry(latent_bf16, num_tokens, latent_dim, row_stride_elems, weight_bf16, eps,
                          true, slot_mapping, cache, num_blocks, block_size, block_stride_rows,
                          group, stream);
}
