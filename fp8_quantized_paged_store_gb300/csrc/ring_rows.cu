// ring_rows.cu — save_ring_rows: copy 1024-float compressor rows into the
// slots of a paged ring state.
//
// Follows "vllm.models.deepseek_v41.common.ops.fused_compress_quant_cache"
// (save_ring_rows: each token's fp32 [kv | score] row of 1024 values goes to
// its slot of the ring-state cache; slot -1 marks a token that is not saved).
//
// Pure data movement, so the roofline is HBM: 4096 bytes read and 4096 bytes
// written per saved row. Work decomposition: a warp owns 32 rows at a time
// (grid-stride over chunks of 32); lane i loads the slot of row i of the
// chunk and turns it into a state offset once, and a ballot lists the rows
// that are saved. A saved row is moved as 256 16-byte words, lane l taking
// words l, l+32, ..., l+224, so every warp-wide access covers 512 contiguous
// bytes; all eight loads are issued before the first store.
#include <cstdint>

#include "kvq.h"
#include "kvq_device.cuh"
#include "kvq_host.h"

namespace kvq {
namespace {

constexpr int kRingWarps = 8;
constexpr int kRingThreads = 32 * kRingWarps;
constexpr int kRingRow = 1024;  // floats per row

struct RingParams {
  const float* rows;
  int64_t row_stride;  // floats
  int64_t num_rows;
  const int64_t* slots;
  float* state;
  int64_t num_slots;        // num_blocks * state_block
  int64_t state_block;
  int64_t state_stride;     // floats between blocks
  int64_t state_row_stride; // floats between rows of a block
};

__global__ void __launch_bounds__(kRingThreads) save_ring_rows_kernel(RingParams p) {
  const int lane = threadIdx.x & 31;
  const int64_t warp = (int64_t)blockIdx.x * kRingWarps + (threadIdx.x >> 5);
  const int64_t warps = (int64_t)gridDim.x * kRingWarps;
  const int64_t chunks = (p.num_rows + 31) / 32;
  for (int64_t c = warp; c < chunks; c += warps) {
    const int64_t t = c * 32 + lane;
    int64_t dst = 0;
    bool saved = false;
    if (t < p.num_rows) {
      const int64_t slot = ld_once_i64(p.slots + t);
      if (slot >= 0 && slot < p.num_slots) {
        int64_t b, r;
        divmod_pos(slot, p.state_block, b, r);
        dst = b * p.state_stride + r * p.state_row_stride;
        saved = true;
      }
    }
    unsigned todo = __ballot_sync(0xFFFFFFFFu, saved);
    while (todo) {
      const int i = __ffs(todo) - 1;
      todo &= todo - 1;
      const int64_t off = __shfl_sync(0xFFFFFFFFu, dst, i);
      const float* src = p.rows + (c * 32 + i) * p.row_stride;
      float* out = p.state + off;
      uint4 w[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) w[k] = ld_once_v4(src + 4 * (lane + 32 * k));
#pragma unroll
      for (int k = 0; k < 8; ++k) st_v4(out + 4 * (lane + 32 * k), w[k]);
    }
  }
}

int g_ring_occupancy[64];

}  // namespace
}  // namespace kvq

extern "C" int save_ring_rows(const float* rows, int64_t num_rows, int64_t row_stride_elems,
                              const int64_t* slot_mapping, float* state, int64_t num_blocks,
                              int64_t state_block, int64_t state_stride_elems,
                              int64_t state_row_stride_elems, cudaStream_t stream) {
  using namespace kvq;
  if (num_rows < 0 || row_stride_elems < kRingRow || row_stride_elems % 4 != 0) return KVQ_EINVAL;
  if (num_blocks < 1 || state_block < 1) return KVQ_EINVAL;
  if (state_row_stride_elems < kRingRow || state_row_stride_elems % 4 != 0 ||
      state_stride_elems % 4 != 0)
    return KVQ_EINVAL;
  if (num_blocks > INT64_MAX / state_block) return KVQ_EINVAL;
  if (state_block - 1 > (INT64_MAX / 8 - kRingRow) / state_row_stride_elems) return KVQ_EINVAL;
  if (state_stride_elems < (state_block - 1) * state_row_stride_elems + kRingRow)
    return KVQ_EINVAL;
  if (num_blocks > INT64_MAX / 8 / state_stride_elems) return KVQ_EINVAL;
  if (num_rows > INT64_MAX / 8 / row_stride_elems) return KVQ_EINVAL;
  if (num_rows == 0) return KVQ_OK;
  if (!rows || !slot_mapping || !state) return KVQ_EINVAL;
  if (!aligned(rows, 16) || !aligned(state, 16) || !aligned(slot_mapping, 8)) return KVQ_EINVAL;
  RingParams p;
  p.rows = rows;
  p.row_stride = row_stride_elems;
  p.num_rows = num_rows;
  p.slots = slot_mapping;
  p.state = state;
  p.num_slots = num_blocks * state_block;
  p.state_block = state_block;
  p.state_stride = state_stride_elems;
  p.state_row_stride = state_row_stride_elems;
  const int64_t chunks = (num_rows + 31) / 32;
  const int64_t work_blocks = (chunks + kRingWarps - 1) / kRingWarps;
  const unsigned grid = grid_for(
      work_blocks, resident_blocks_per_sm(save_ring_rows_kernel, kRingThreads, 0, g_ring_occupancy));
  save_ring_rows_kernel<<<grid, kRingThreads, 0, stream>>>(p);
  return launch_status();
}
