// mxfp4_gather.cu — mxfp4_mla_gather_dequant: gather packed 272-byte MXFP4
// rows by slot index and write them out as bf16.
//
// Follows PR 60321 "Add an mxfp4_mla KV cache for rope-free sparse MLA"
// (Details, read path: gathered rows are unpacked to bf16 before use; Claims:
// attention over the packed cache equals attention over those bf16 values).
//
// Values are decoded by byte permutes from per-group tables of the eight
// scaled bf16 patterns (mxfp4_decode.cuh), built once per block for every
// scale byte in [2, 252]; other scale bytes take an arithmetic path.
//
// Work decomposition: one wave of 256-thread blocks, each warp a contiguous
// range of output rows; indices 32 at a time (lane i loads index i and turns
// it into a source row once); packed rows staged through a per-warp
// cp.async ring seven rows ahead. Lane l decodes code bytes 4l..4l+3 and
// 128+4l..128+4l+3 with the scale bytes of groups l/4 and 8+l/4, and writes
// 16 bytes at elements 8l and 256+8l (two coalesced 512-byte stores). Pads
// and out-of-range indices write zeros.
#include <cstdint>

#include "kvq.h"
#include "kvq_device.cuh"
#include "kvq_host.h"
#include "mxfp4_decode.cuh"

namespace kvq {
namespace {

constexpr int kGatherWarps = 8;
constexpr int kGatherThreads = 32 * kGatherWarps;

struct GatherParams {
  const uint8_t* cache;
  int64_t num_slots;
  int64_t block_size;
  int64_t block_stride_rows;
  const int64_t* indices;
  int64_t num_indices;
  uint8_t* out;        // row k starts at out + k * out_pitch
  int64_t out_pitch;   // bytes
  int64_t per_warp, extra;  // warp w's rows: per_warp, plus one for w < extra
};

constexpr int kGatherPrefetch = 7;  // rows per warp in flight
constexpr int kGatherStages = 8;    // a power of two: stage = row & 7
constexpr int kStagePitch = 288;    // 272-byte row, 16-byte multiple
constexpr int kLutBytes = 256 * 16;
constexpr size_t kGatherSmem =
    (size_t)kLutBytes + (size_t)kGatherWarps * kGatherStages * kStagePitch;

// Row index (272-byte rows from the view's base) of output row k, or
// 0xFFFFFFFF for a zero row (pad, outside the cache, past the range). The
// host guarantees that row indices fit in 32 bits.
template <bool kFlat>
__device__ __forceinline__ uint32_t src_row(const GatherParams& p, int64_t k, int64_t k_end) {
  if (k >= k_end) return 0xFFFFFFFFu;
  const int64_t s = ld_once_i64(p.indices + k);
  if (s < 0 || s >= p.num_slots) return 0xFFFFFFFFu;
  if (kFlat) return (uint32_t)s;
  int64_t blk, in_blk;
  divmod_pos(s, p.block_size, blk, in_blk);
  return (uint32_t)(blk * p.block_stride_rows + in_blk);
}

// Each warp owns a contiguous range of output rows. Packed rows stream
// through a per-warp shared-memory ring: lanes 0..16 copy the 272 bytes of
// the row kGatherPrefetch ahead (17 x 16-byte cp.async); after its own copies
// land, __syncwarp makes the other lanes' bytes visible, and a second
// __syncwarp before each refill keeps a stage from being overwritten while a
// lane still reads it. The block first fills the table of byte-permute
// tables, one 16-byte entry per scale byte (the one block-wide barrier).
template <bool kFlat>
__global__ void __launch_bounds__(kGatherThreads) mxfp4_gather_kernel(GatherParams p) {
  extern __shared__ uint4 smem[];
  uint4* lut = smem;
  if (threadIdx.x >= 2 && threadIdx.x <= 252) {
    const ByteTables t = make_tables(threadIdx.x);
    lut[threadIdx.x] = make_uint4(t.lo_a, t.hi_a, t.lo_b, t.hi_b);
  }
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const int warp_in_block = threadIdx.x >> 5;
  uint8_t* ring = reinterpret_cast<uint8_t*>(smem) + kLutBytes +
                  warp_in_block * (kGatherStages * kStagePitch);
  const int64_t warp = (int64_t)blockIdx.x * kGatherWarps + warp_in_block;
  const int64_t k_begin = warp * p.per_warp + (warp < p.extra ? warp : p.extra);
  const int64_t k_end = k_begin + p.per_warp + (warp < p.extra ? 1 : 0);
  const int n = (int)(k_end - k_begin);  // < 2**31, checked at launch
  if (n <= 0) return;
  const uint4 zero = make_uint4(0, 0, 0, 0);
  uint8_t* out_base = p.out + k_begin * p.out_pitch + 16 * lane;
  const uint32_t pitch = (uint32_t)p.out_pitch;
  const uint8_t* cache_lane = p.cache + 16 * lane;

  auto issue = [&](int i, uint32_t row) {
    if (row != 0xFFFFFFFFu && lane < 17)
      cp_async_16(ring + (i & (kGatherStages - 1)) * kStagePitch + 16 * lane,
                  cache_lane + (size_t)row * kMxfp4RowBytes);
    cp_async_commit();
  };

  uint32_t w0 = src_row<kFlat>(p, k_begin + lane, k_end);
  uint32_t w1 = src_row<kFlat>(p, k_begin + 32 + lane, k_end);
#pragma unroll
  for (int d = 0; d < kGatherPrefetch; ++d) issue(d, __shfl_sync(0xFFFFFFFFu, w0, d));

  for (int i = 0; i < n; ++i) {
    const int k = i & 31;
    if (k == 0 && i > 0) {
      w0 = w1;
      w1 = src_row<kFlat>(p, k_begin + i + 32 + lane, k_end);
    }
    const int kp = k + kGatherPrefetch;
    const uint32_t rp = __shfl_sync(0xFFFFFFFFu, kp < 32 ? w0 : w1, kp & 31);
    __syncwarp();  // every lane is done with the stage about to be refilled
    issue(i + kGatherPrefetch, i + kGatherPrefetch < n ? rp : 0xFFFFFFFFu);
    cp_async_wait<kGatherPrefetch>();
    __syncwarp();  // row i's bytes from all 17 copying lanes are visible
    const uint32_t row = __shfl_sync(0xFFFFFFFFu, w0, k);
    uint8_t* out = out_base + (size_t)i * pitch;
    if (row != 0xFFFFFFFFu) {
      const uint8_t* r = ring + (i & (kGatherStages - 1)) * kStagePitch;
      const uint32_t c0 = lds_u32(r + 4 * lane);
      const uint32_t c1 = lds_u32(r + 128 + 4 * lane);
      const uint32_t b0 = lds_u8(r + 256 + (lane >> 2));
      const uint32_t b1 = lds_u8(r + 264 + (lane >> 2));
      st_v4(out, decode8(c0, b0, lut));
      st_v4(out + 512, decode8(c1, b1, lut));
    } else {
      st_v4(out, zero);
      st_v4(out + 512, zero);
    }
  }
  cp_async_wait<0>();
}

int g_gather_occupancy[2][64];

}  // namespace
}  // namespace kvq

extern "C" int mxfp4_mla_gather_dequant(const uint8_t* cache, int64_t num_blocks,
                                        int64_t block_size, int64_t block_stride_rows,
                                        int64_t latent_dim, const int64_t* indices,
                                        int64_t num_indices, void* out_bf16,
                                        int64_t out_row_stride_elems, cudaStream_t stream) {
  using namespace kvq;
  if (latent_dim != kLatent) return KVQ_EINVAL;
  if (num_indices < 0 || num_blocks < 1 || block_size < 1 || block_stride_rows < block_size)
    return KVQ_EINVAL;
  if (out_row_stride_elems < latent_dim || out_row_stride_elems % 8 != 0) return KVQ_EINVAL;
  if (num_blocks > INT64_MAX / block_stride_rows / kMxfp4RowBytes) return KVQ_EINVAL;
  if (num_blocks > INT64_MAX / block_size) return KVQ_EINVAL;
  if (num_indices > INT64_MAX / 2 / out_row_stride_elems) return KVQ_EINVAL;
  // cache rows are addressed with 32-bit indices (2**32 rows would be 1.1 TB)
  if ((num_blocks - 1) * block_stride_rows + block_size > (int64_t)0xFFFFFFFE) return KVQ_EINVAL;
  if (out_row_stride_elems * 2 > (int64_t)0xFFFFFFFF) return KVQ_EINVAL;
  if (num_indices == 0) return KVQ_OK;
  if (!cache || !indices || !out_bf16) return KVQ_EINVAL;
  if (!aligned(cache, 16) || !aligned(out_bf16, 16) || !aligned(indices, 8)) return KVQ_EINVAL;

  GatherParams p;
  p.cache = cache;
  p.num_slots = num_blocks * block_size;
  p.block_size = block_size;
  p.block_stride_rows = block_stride_rows;
  p.indices = indices;
  p.num_indices = num_indices;
  p.out = static_cast<uint8_t*>(out_bf16);
  p.out_pitch = out_row_stride_elems * 2;

  const bool flat = (num_blocks == 1) || (block_stride_rows == block_size);
  const int64_t work_blocks = (num_indices + 32 * kGatherWarps - 1) / (32 * kGatherWarps);
  auto k = flat ? mxfp4_gather_kernel<true> : mxfp4_gather_kernel<false>;
  const unsigned grid = grid_for(
      work_blocks, resident_blocks_per_sm(k, kGatherThreads, kGatherSmem, g_gather_occupancy[flat]));
  // each warp's row count must fit the kernel's 32-bit loop counter
  if (num_indices / ((int64_t)grid * kGatherWarps) >= (int64_t)0x7FFFFFFF) return KVQ_EINVAL;
  p.per_warp = num_indices / ((int64_t)grid * kGatherWarps);
  p.extra = num_indices - p.per_warp * ((int64_t)grid * kGatherWarps);
  k<<<grid, kGatherThreads, kGatherSmem, stream>>>(p);
  return launch_status();
}
