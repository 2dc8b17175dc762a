// compress_norm.cu — fused_save_compress_norm: pool each closed group of
// compressor rows into an RMS-normalised bf16 latent, and save the ring rows
// the next chunk needs.
//
// Follows "vllm.models.deepseek_v41.common.ops.fused_compress_quant_cache"
// (fused_save_compress_norm: docstring and Args). Groups of R in {1, 2}
// consecutive positions close at (p + 1) % R == 0. For R = 2 a row is
// [512 kv | 512 score] in fp32 and the group is pooled per channel by a
// softmax of the two scores; for R = 1 the row is 512 kv values and the
// pooled row is the row itself. The pooled row is RMS-normalised with a bf16
// weight and an fp32 epsilon and written as bf16 at the closing token. The
// first token of a request's chunk closes its group with the predecessor in
// the ring (row (p - 1) % capacity of the request's block) or in prev_rows;
// the chunk's last `capacity` rows are then copied into the ring, unless
// prev_rows is given.
//
// Arithmetic (fp32): m = max(s0, s1); e_i = expf(s_i - m);
// pooled = RN((e0*kv0 + e1*kv1) / (e0 + e1)) with the products and the sum
// rounded separately; sum of squares per lane in a fixed order, then an xor
// butterfly over the warp; r = RN(1 / RN(sqrt(RN(RN(S / 512) + eps))));
// latent = bf16(RN(RN(pooled * r) * w)).
//
// Work decomposition. Two roles in one launch: the first `token_blocks`
// blocks own chunks of 32 tokens (grid-stride); lane i decides whether token
// i closes a group whose rows are both in the batch (every group of R = 1;
// for R = 2 a closing token that is not its chunk's first), a ballot lists
// them, and the warp handles them one by one: lane l holds float4 words
// l + 32k (k = 0..3) of each 512-float half, so every warp-wide access
// covers 512 contiguous bytes. The remaining blocks (R = 2 only) give one
// warp to each request: it handles the group its chunk's first token closes
// with the ring or prev_rows, then copies the chunk's last `capacity` rows
// into the ring. The same warp reads the ring row and later writes ring rows,
// each float4 word by the same lane, so the read sees the ring as it was
// before the call; no other warp touches that request's ring block, and the
// token role never reads the ring. Ring reads use coherent loads (the state
// is written by the same launch); the batch rows, prev_rows and the weight
// are read-only and go through the non-coherent path.
#include <cstdint>

#include "kvq.h"
#include "kvq_device.cuh"
#include "kvq_host.h"

namespace kvq {
namespace {

constexpr int kCompressWarps = 8;
constexpr int kCompressThreads = 32 * kCompressWarps;

struct CompressParams {
  const float* rows;   // token t at rows + t * row_stride
  int64_t row_stride;  // floats
  int64_t num_tokens;
  const int64_t* positions;
  const int64_t* slots;
  const int64_t* qsl;   // [num_reqs + 1]
  const int64_t* t2r;   // [num_tokens]
  int64_t num_reqs;
  float* state;
  int64_t num_state_slots;  // blocks * capacity
  int64_t capacity;
  int64_t state_stride;      // floats between blocks
  int64_t state_row_stride;  // floats between the rows of a block
  const uint8_t* weight;     // bf16 [512]
  float eps;
  const float* prev_rows;  // null: read the ring and save it
  int64_t prev_stride;
  int64_t num_prev;
  const int64_t* prev_idx;
  uint8_t* out;        // bf16 row t at out + t * out_pitch
  int64_t out_pitch;   // bytes
  int ratio;
  unsigned token_blocks;
};

// Coherent 16-byte load (data the same launch writes).
__device__ __forceinline__ float4 ld_f4_coherent(const float* p) {
  float4 r;
  asm volatile("ld.global.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(r.x), "=f"(r.y), "=f"(r.z), "=f"(r.w)
               : "l"(p)
               : "memory");
  return r;
}

// Read-only 16-byte load that is not kept in L1.
__device__ __forceinline__ float4 ld_f4_once(const float* p) {
  const uint4 u = ld_once_v4(p);
  return make_float4(__uint_as_float(u.x), __uint_as_float(u.y), __uint_as_float(u.z),
                     __uint_as_float(u.w));
}

__device__ __forceinline__ void st_f4(float* p, float4 v) {
  st_v4(p, make_uint4(__float_as_uint(v.x), __float_as_uint(v.y), __float_as_uint(v.z),
                      __float_as_uint(v.w)));
}

__device__ __forceinline__ uint32_t bf16x2_pack(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}

__device__ __forceinline__ float pool1(float kv0, float s0, float kv1, float s1) {
  const float m = fmaxf(s0, s1);
  const float e0 = expf(__fsub_rn(s0, m));
  const float e1 = expf(__fsub_rn(s1, m));
  return __fdiv_rn(__fadd_rn(__fmul_rn(e0, kv0), __fmul_rn(e1, kv1)), __fadd_rn(e0, e1));
}

__device__ __forceinline__ float4 pool4(float4 kv0, float4 s0, float4 kv1, float4 s1) {
  return make_float4(pool1(kv0.x, s0.x, kv1.x, s1.x), pool1(kv0.y, s0.y, kv1.y, s1.y),
                     pool1(kv0.z, s0.z, kv1.z, s1.z), pool1(kv0.w, s0.w, kv1.w, s1.w));
}

// RMSNorm of the warp's pooled row (lane l: float4 words l + 32k) and the
// bf16 store of the latent row.
__device__ __forceinline__ void norm_store(const CompressParams& p, const float4 x[4],
                                           const float4 w[4], int64_t t, int lane) {
  float acc = 0.f;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    acc = __fadd_rn(acc, __fmul_rn(x[k].x, x[k].x));
    acc = __fadd_rn(acc, __fmul_rn(x[k].y, x[k].y));
    acc = __fadd_rn(acc, __fmul_rn(x[k].z, x[k].z));
    acc = __fadd_rn(acc, __fmul_rn(x[k].w, x[k].w));
  }
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) acc = __fadd_rn(acc, __shfl_xor_sync(0xFFFFFFFFu, acc, o));
  const float r = __frcp_rn(__fsqrt_rn(__fadd_rn(__fmul_rn(acc, 1.0f / 512.0f), p.eps)));
  uint8_t* dst = p.out + t * p.out_pitch;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float y0 = __fmul_rn(__fmul_rn(x[k].x, r), w[k].x);
    const float y1 = __fmul_rn(__fmul_rn(x[k].y, r), w[k].y);
    const float y2 = __fmul_rn(__fmul_rn(x[k].z, r), w[k].z);
    const float y3 = __fmul_rn(__fmul_rn(x[k].w, r), w[k].w);
    st_v2(dst + 8 * (lane + 32 * k), bf16x2_pack(y0, y1), bf16x2_pack(y2, y3));
  }
}

// One group whose predecessor row is `pred` (its kv at pred, scores at
// pred + 512) and whose closing row is `own`; pred_coherent selects the
// load path of the predecessor (ring rows are written by this launch).
template <bool kPredCoherent>
__device__ __forceinline__ void group2(const CompressParams& p, const float* pred,
                                       const float* own, const float4 w[4], int64_t t,
                                       int lane) {
  float4 kv0[4], s0[4], kv1[4], s1[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int j = 4 * (lane + 32 * k);
    if (kPredCoherent) {
      kv0[k] = ld_f4_coherent(pred + j);
      s0[k] = ld_f4_coherent(pred + 512 + j);
    } else {
      kv0[k] = ld_f4_once(pred + j);
      s0[k] = ld_f4_once(pred + 512 + j);
    }
    kv1[k] = ld_f4_once(own + j);
    s1[k] = ld_f4_once(own + 512 + j);
  }
  float4 x[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) x[k] = pool4(kv0[k], s0[k], kv1[k], s1[k]);
  norm_store(p, x, w, t, lane);
}

__device__ __forceinline__ void load_weight(const CompressParams& p, int lane, float4 w[4]) {
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const uint8_t* src = p.weight + 8 * (lane + 32 * k);
    const uint32_t a = ld_u32(src), b = ld_u32(src + 4);
    w[k] = make_float4(bf16_lo(a), bf16_hi(a), bf16_lo(b), bf16_hi(b));
  }
}

__device__ __forceinline__ int64_t ld_i64(const int64_t* p) {
  int64_t r;
  asm("ld.global.nc.s64 %0, [%1];" : "=l"(r) : "l"(p));
  return r;
}

__global__ void __launch_bounds__(kCompressThreads) compress_norm_kernel(CompressParams p) {
  const int lane = threadIdx.x & 31;
  float4 w[4];
  load_weight(p, lane, w);

  if (blockIdx.x < p.token_blocks) {
    // token role: groups whose rows are both in the batch
    const int64_t warp = (int64_t)blockIdx.x * kCompressWarps + (threadIdx.x >> 5);
    const int64_t warps = (int64_t)p.token_blocks * kCompressWarps;
    for (int64_t base = warp * 32; base < p.num_tokens; base += warps * 32) {
      const int64_t t = base + lane;
      bool closes = false;
      if (t < p.num_tokens) {
        const int64_t s = ld_once_i64(p.slots + t);
        const int64_t pos = ld_once_i64(p.positions + t);
        closes = s >= 0 && pos >= 0 && (pos + 1) % p.ratio == 0;
        if (closes && p.ratio == 2) {
          const int64_t req = ld_once_i64(p.t2r + t);
          closes = req >= 0 && req < p.num_reqs && s < p.num_state_slots;
          if (closes) {
            const int64_t qs = ld_i64(p.qsl + req), qe = ld_i64(p.qsl + req + 1);
            // the chunk's first token (a start below 0 reads as 0) is the request role's
            closes = (qs > 0 ? qs : 0) < t && t < qe;
          }
        }
      }
      unsigned todo = __ballot_sync(0xFFFFFFFFu, closes);
      while (todo) {
        const int i = __ffs(todo) - 1;
        todo &= todo - 1;
        const int64_t tt = base + i;
        const float* own = p.rows + tt * p.row_stride;
        if (p.ratio == 1) {
          float4 x[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) x[k] = ld_f4_once(own + 4 * (lane + 32 * k));
          norm_store(p, x, w, tt, lane);
        } else {
          group2<false>(p, own - p.row_stride, own, w, tt, lane);
        }
      }
    }
    return;
  }

  // request role (R = 2): the chunk-first group, then the ring save
  const int64_t warp = (int64_t)(blockIdx.x - p.token_blocks) * kCompressWarps + (threadIdx.x >> 5);
  const int64_t warps = (int64_t)(gridDim.x - p.token_blocks) * kCompressWarps;
  for (int64_t k = warp; k < p.num_reqs; k += warps) {
    int64_t qs = ld_i64(p.qsl + k);
    int64_t qe = ld_i64(p.qsl + k + 1);
    if (qs < 0) qs = 0;
    if (qe > p.num_tokens) qe = p.num_tokens;
    if (qs >= qe) continue;
    const int64_t s = ld_once_i64(p.slots + qs);
    const int64_t pos = ld_once_i64(p.positions + qs);
    const int64_t req = ld_once_i64(p.t2r + qs);
    if (req == k && s >= 0 && s < p.num_state_slots && pos >= 0 && (pos & 1) == 1) {
      const float* own = p.rows + qs * p.row_stride;
      const int64_t j = p.prev_rows ? ld_once_i64(p.prev_idx + k) : -1;
      if (j >= 0) {
        if (j < p.num_prev) group2<false>(p, p.prev_rows + j * p.prev_stride, own, w, qs, lane);
      } else {
        const int64_t blk = s / p.capacity;
        const float* pred = p.state + blk * p.state_stride + ((pos - 1) % p.capacity) * p.state_row_stride;
        group2<true>(p, pred, own, w, qs, lane);
      }
    }
    if (p.prev_rows) continue;
    __syncwarp();
    const int64_t first = qe - p.capacity > qs ? qe - p.capacity : qs;
    for (int64_t t = first; t < qe; ++t) {
      const int64_t st = ld_once_i64(p.slots + t);
      if (st < 0 || st >= p.num_state_slots) continue;
      const float* src = p.rows + t * p.row_stride;
      float* dst = p.state + (st / p.capacity) * p.state_stride + (st % p.capacity) * p.state_row_stride;
      float4 v[8];
#pragma unroll
      for (int c = 0; c < 8; ++c) v[c] = ld_f4_once(src + 4 * (lane + 32 * c));
#pragma unroll
      for (int c = 0; c < 8; ++c) st_f4(dst + 4 * (lane + 32 * c), v[c]);
    }
  }
}

int g_compress_occupancy[64];

}  // namespace
}  // namespace kvq

extern "C" int fused_save_compress_norm(
    const float* kv_score, int64_t num_tokens, int64_t row_stride_elems, const int64_t* positions,
    const int64_t* slot_mapping, int32_t compress_ratio, const int64_t* query_start_loc,
    const int64_t* token_to_req_indices, int64_t num_reqs, float* state, int64_t num_blocks,
    int64_t capacity, int64_t state_stride_elems, int64_t state_row_stride_elems,
    const void* weight_bf16, float eps, const float* prev_rows, int64_t num_prev_rows,
    int64_t prev_row_stride_elems, const int64_t* prev_row_indices, void* latent_out_bf16,
    int64_t out_row_stride_elems, cudaStream_t stream) {
  using namespace kvq;
  if (compress_ratio != 1 && compress_ratio != 2) return KVQ_EINVAL;
  const int64_t width = 512 * (int64_t)compress_ratio;
  if (num_tokens < 0 || row_stride_elems < width || row_stride_elems % 4 != 0) return KVQ_EINVAL;
  if (out_row_stride_elems < 512 || out_row_stride_elems % 8 != 0) return KVQ_EINVAL;
  if (!(eps >= 0.0f && eps <= 3.0e38f)) return KVQ_EINVAL;
  if (num_tokens > INT64_MAX / 8 / row_stride_elems) return KVQ_EINVAL;
  if (num_tokens > INT64_MAX / 4 / out_row_stride_elems) return KVQ_EINVAL;
  CompressParams p{};
  if (compress_ratio == 2) {
    if (num_reqs < 0 || num_blocks < 1 || capacity < 1) return KVQ_EINVAL;
    if (state_row_stride_elems < 1024 || state_row_stride_elems % 4 != 0 ||
        state_stride_elems % 4 != 0)
      return KVQ_EINVAL;
    if (capacity - 1 > (INT64_MAX / 8 - 1024) / state_row_stride_elems) return KVQ_EINVAL;
    if (state_stride_elems < (capacity - 1) * state_row_stride_elems + 1024) return KVQ_EINVAL;
    if (num_blocks > INT64_MAX / 8 / state_stride_elems) return KVQ_EINVAL;
    if ((prev_rows == nullptr) != (prev_row_indices == nullptr)) return KVQ_EINVAL;
    if (prev_rows) {
      if (num_prev_rows < 0 || prev_row_stride_elems < 1024 || prev_row_stride_elems % 4 != 0)
        return KVQ_EINVAL;
      if (num_prev_rows > INT64_MAX / 8 / prev_row_stride_elems) return KVQ_EINVAL;
    }
  }
  if (num_tokens == 0) return KVQ_OK;
  if (!kv_score || !positions || !slot_mapping || !weight_bf16 || !latent_out_bf16)
    return KVQ_EINVAL;
  if (!aligned(kv_score, 16) || !aligned(positions, 8) || !aligned(slot_mapping, 8) ||
      !aligned(weight_bf16, 8) || !aligned(latent_out_bf16, 16))
    return KVQ_EINVAL;
  if (compress_ratio == 2) {
    if (!query_start_loc || !token_to_req_indices || !state) return KVQ_EINVAL;
    if (!aligned(query_start_loc, 8) || !aligned(token_to_req_indices, 8) || !aligned(state, 16))
      return KVQ_EINVAL;
    if (prev_rows && (!aligned(prev_rows, 16) || !aligned(prev_row_indices, 8))) return KVQ_EINVAL;
  }
  p.rows = kv_score;
  p.row_stride = row_stride_elems;
  p.num_tokens = num_tokens;
  p.positions = positions;
  p.slots = slot_mapping;
  p.ratio = compress_ratio;
  p.weight = static_cast<const uint8_t*>(weight_bf16);
  p.eps = eps;
  p.out = static_cast<uint8_t*>(latent_out_bf16);
  p.out_pitch = out_row_stride_elems * 2;
  if (compress_ratio == 2) {
    p.qsl = query_start_loc;
    p.t2r = token_to_req_indices;
    p.num_reqs = num_reqs;
    p.state = state;
    p.capacity = capacity;
    p.num_state_slots = num_blocks * capacity;
    p.state_stride = state_stride_elems;
    p.state_row_stride = state_row_stride_elems;
    p.prev_rows = prev_rows;
    p.prev_stride = prev_row_stride_elems;
    p.num_prev = num_prev_rows;
    p.prev_idx = prev_row_indices;
  }
  const int per_sm = resident_blocks_per_sm(compress_norm_kernel, kCompressThreads, 0,
                                            g_compress_occupancy);
  const int64_t chunks = (num_tokens + 31) / 32;
  const unsigned token_blocks = grid_for((chunks + kCompressWarps - 1) / kCompressWarps, per_sm);
  const unsigned req_blocks =
      (compress_ratio == 2 && num_reqs > 0)
          ? grid_for((num_reqs + kCompressWarps - 1) / kCompressWarps, per_sm)
          : 0u;
  p.token_blocks = token_blocks;
  compress_norm_kernel<<<token_blocks + req_blocks, kCompressThreads, 0, stream>>>(p);
  return launch_status();
}
