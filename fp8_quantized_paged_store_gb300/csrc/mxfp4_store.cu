// mxfp4_store.cu — mxfp4_mla_store: quantize bf16 MLA latent rows to MXFP4
// and scatter them into a paged cache of 272-byte rows.
//
// Follows "vllm.v1.attention.ops.mxfp4_mla.store" (store_mxfp4_mla,
// _ceil_pow2_exponent, _quantize_e2m1) and PR 60321 "Add an mxfp4_mla KV cache
// for rope-free sparse MLA" (Details: format and write path).
//
// Work decomposition (GB300: 152 SMs, HBM-bound streaming codec):
//   * one warp owns 32 consecutive tokens at a time (grid-stride over chunks);
//     lane i loads slot_mapping of token i once and turns it into the row's
//     byte offset (one division per lane per chunk, not per row);
//   * a ballot lists the chunk's valid tokens, so pads cost no row traffic;
//   * rows are processed two at a time, both rows' loads issued first; one
//     row is 1 KiB read as two fully coalesced 512-byte warp loads: lane l
//     holds elements 8l..8l+7 (half 0, groups 0..7) and 256+8l..256+8l+7
//     (half 1, groups 8..15), so a 32-element group spans four lanes;
//   * group amax: bf16x2 max-of-magnitudes (NaN ignored) within the lane, then
//     two xor-shuffles across the four lanes, both halves packed in one word;
//   * the E8M0 exponent comes from the amax bits without a division;
//   * values are scaled by the exact power 2**-e in binary32 and converted
//     by cvt.rn.satfinite.e2m1x2.f32 (NaN and -0.0 are cleared first);
//   * each lane stores two 4-byte code words (two coalesced 128-byte warp
//     stores) and four lanes store the two scale bytes of their groups.
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
};

// Eight bf16 (one 16-byte load) of a group with scale 2**e -> eight E2M1
// codes. NaN and -0.0 are turned into +0.0 first: the conversion would give
// them codes 7 and 8, the E2M1 rule gives both code 0. A product can only
// underflow to -0.0 (which the rule also codes 0) when e >= 17, since the
// smallest bf16 magnitude is 2**-133; kGuard adds +0.0 after the product for
// that case, turning -0.0 into +0.0 and changing nothing else.
template <bool kGuard>
__device__ __forceinline__ uint32_t encode8(uint4 w, float inv_scale) {
  w.x &= bf16x2_nonzero_number_mask(w.x);
  w.y &= bf16x2_nonzero_number_mask(w.y);
  w.z &= bf16x2_nonzero_number_mask(w.z);
  w.w &= bf16x2_nonzero_number_mask(w.w);
  float f[8] = {bf16_lo(w.x), bf16_hi(w.x), bf16_lo(w.y), bf16_hi(w.y),
                bf16_lo(w.z), bf16_hi(w.z), bf16_lo(w.w), bf16_hi(w.w)};
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    f[k] = __fmul_rn(f[k], inv_scale);
    if (kGuard) f[k] = __fadd_rn(f[k], 0.0f);
  }
  return cvt_e2m1x8(f[0], f[1], f[2], f[3], f[4], f[5], f[6], f[7]);
}

// Quantize one row held by the warp (x0: half 0, x1: half 1) and write its 272
// bytes at dst.
__device__ __forceinline__ void quantize_store_row(uint4 x0, uint4 x1, uint8_t* dst, int lane) {
  uint32_t m0 = bf16x2_maxabs(bf16x2_maxabs(x0.x, x0.y), bf16x2_maxabs(x0.z, x0.w));
  uint32_t m1 = bf16x2_maxabs(bf16x2_maxabs(x1.x, x1.y), bf16x2_maxabs(x1.z, x1.w));
  // [half 0 | half 1] in the low / high 16 bits, then fold even and odd.
  uint32_t g = bf16x2_maxabs(__byte_perm(m0, m1, 0x5410), __byte_perm(m0, m1, 0x7632));
  g &= 0x7FFF7FFFu;
  g = bf16x2_max(g, __shfl_xor_sync(0xFFFFFFFFu, g, 1));
  g = bf16x2_max(g, __shfl_xor_sync(0xFFFFFFFFu, g, 2));
  const int e0 = mxfp4_group_exponent(g & 0xFFFFu);  // group lane/4
  const int e1 = mxfp4_group_exponent(g >> 16);      // group 8 + lane/4
  const float s0 = exp2_neg(e0), s1 = exp2_neg(e1);
  uint32_t c0, c1;
  if (__any_sync(0xFFFFFFFFu, (e0 > 16) | (e1 > 16))) {
    c0 = encode8<true>(x0, s0);
    c1 = encode8<true>(x1, s1);
  } else {
    c0 = encode8<false>(x0, s0);
    c1 = encode8<false>(x1, s1);
  }
  st_u32(dst + 4 * lane, c0);
  st_u32(dst + 128 + 4 * lane, c1);
  if ((lane & 3) == 0) {
    st_u8(dst + 256 + (lane >> 2), (uint32_t)(e0 + 127));
    st_u8(dst + 264 + (lane >> 2), (uint32_t)(e1 + 127));
  }
}

template <bool kFlat>
__global__ void __launch_bounds__(kStoreThreads) mxfp4_store_kernel(StoreParams p) {
  const int lane = threadIdx.x & 31;
  const int64_t warp = ((int64_t)blockIdx.x * kStoreThreads + threadIdx.x) >> 5;
  const int64_t num_warps = ((int64_t)gridDim.x * kStoreThreads) >> 5;

  for (int64_t base = warp * 32; base < p.num_tokens; base += num_warps * 32) {
    // Lane i: token base+i -> byte offset of its cache row, or -1 to skip.
    int64_t dst_off = -1;
    if (base + lane < p.num_tokens) {
      const int64_t s = ld_once_i64(p.slots + base + lane);
      if (s >= 0 && s < p.num_slots) {
        if (kFlat) {
          dst_off = s * kMxfp4RowBytes;
        } else {
          int64_t blk, in_blk;
          divmod_pos(s, p.block_size, blk, in_blk);
          dst_off = (blk * p.block_stride_rows + in_blk) * kMxfp4RowBytes;
        }
      }
    }
    uint32_t todo = __ballot_sync(0xFFFFFFFFu, dst_off >= 0);
    while (todo) {
      const int i0 = __ffs(todo) - 1;
      todo &= todo - 1;
      const int i1 = todo ? __ffs(todo) - 1 : -1;
      if (todo) todo &= todo - 1;

      const uint8_t* r0 = p.latent + (base + i0) * p.row_pitch;
      const uint4 x00 = ld_once_v4(r0 + 16 * lane);
      const uint4 x01 = ld_once_v4(r0 + 512 + 16 * lane);
      uint4 x10 = make_uint4(0, 0, 0, 0), x11 = make_uint4(0, 0, 0, 0);
      if (i1 >= 0) {
        const uint8_t* r1 = p.latent + (base + i1) * p.row_pitch;
        x10 = ld_once_v4(r1 + 16 * lane);
        x11 = ld_once_v4(r1 + 512 + 16 * lane);
      }
      const int64_t d0 = __shfl_sync(0xFFFFFFFFu, dst_off, i0);
      quantize_store_row(x00, x01, p.cache + d0, lane);
      if (i1 >= 0) {
        const int64_t d1 = __shfl_sync(0xFFFFFFFFu, dst_off, i1);
        quantize_store_row(x10, x11, p.cache + d1, lane);
      }
    }
  }
}

int g_store_occupancy[2][64];

}  // namespace
}  // namespace kvq

extern "C" int mxfp4_mla_store(const void* latent_bf16, int64_t num_tokens, int64_t latent_dim,
                               int64_t row_stride_elems, const int64_t* slot_mapping,
                               uint8_t* cache, int64_t num_blocks, int64_t block_size,
                               int64_t block_stride_rows, int32_t group, cudaStream_t stream) {
  using namespace kvq;
  if (latent_dim != kLatent || group != 32) return KVQ_EINVAL;
  if (num_tokens < 0 || num_blocks < 1 || block_size < 1 || block_stride_rows < block_size)
    return KVQ_EINVAL;
  if (row_stride_elems < latent_dim || row_stride_elems % 8 != 0) return KVQ_EINVAL;
  // The cache view must be addressable without int64 overflow.
  if (num_blocks > INT64_MAX / block_stride_rows / kMxfp4RowBytes) return KVQ_EINVAL;
  if (num_blocks > INT64_MAX / block_size) return KVQ_EINVAL;
  if (num_tokens > INT64_MAX / 2 / row_stride_elems) return KVQ_EINVAL;
  if (num_tokens == 0) return KVQ_OK;
  if (!latent_bf16 || !slot_mapping || !cache) return KVQ_EINVAL;
  if (!aligned(latent_bf16, 16) || !aligned(cache, 16) || !aligned(slot_mapping, 8))
    return KVQ_EINVAL;

  StoreParams p;
  p.latent = static_cast<const uint8_t*>(latent_bf16);
  p.row_pitch = row_stride_elems * 2;
  p.num_tokens = num_tokens;
  p.slots = slot_mapping;
  p.cache = cache;
  p.num_slots = num_blocks * block_size;
  p.block_size = block_size;
  p.block_stride_rows = block_stride_rows;

  const bool flat = (num_blocks == 1) || (block_stride_rows == block_size);
  const int64_t chunks = (num_tokens + 31) / 32;
  const int64_t work_blocks = (chunks + kStoreWarps - 1) / kStoreWarps;
  if (flat) {
    auto k = mxfp4_store_kernel<true>;
    const unsigned grid =
        grid_for(work_blocks, resident_blocks_per_sm(k, kStoreThreads, g_store_occupancy[1]));
    k<<<grid, kStoreThreads, 0, stream>>>(p);
  } else {
    auto k = mxfp4_store_kernel<false>;
    const unsigned grid =
        grid_for(work_blocks, resident_blocks_per_sm(k, kStoreThreads, g_store_occupancy[0]));
    k<<<grid, kStoreThreads, 0, stream>>>(p);
  }
  return launch_status();
}
