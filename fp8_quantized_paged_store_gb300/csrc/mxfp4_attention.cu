// mxfp4_attention.cu — mxfp4_mla_sparse_attention: sparse MLA decode attention
// that reads the packed MXFP4 cache directly, on the tcgen05 tensor cores.
//
// Follows PR 60321 "Add an mxfp4_mla KV cache for rope-free sparse MLA"
// (Read path: each query's top-k rows are gathered and unpacked to bf16 and
// feed both dots, q.k and p.v; Claims: attention over the packed cache equals
// attention over the dequantized bf16 values). For the rope-free latent the
// key and the value of a token are the same 512-wide row.
//
// Work decomposition. One CTA (128 threads, one TMEM lane and one head per
// thread) per (query, half of the 512 value columns): the two CTAs of a query
// both form the full scores q.k (512-deep) and each accumulates 256 output
// columns, so the output accumulator (128 heads x 256 fp32 = 256 TMEM
// columns) and two 32-key score buffers fit the 512 TMEM columns. Keys go in
// tiles of 32:
//   - warp 0 stages the packed rows of tile t+2 with cp.async (17 x 16 bytes
//     per key; pads and out-of-range indices copy nothing and get a -inf
//     score bias);
//   - all threads dequantize tile t+1 into bf16 (byte-permute decode) in the
//     128-byte-swizzled K-major layout the tensor core reads, zero rows for
//     pads; thread 0 then issues S(t+1) = Q K^T (M 128, N 32, K 512) into
//     the free score buffer;
//   - meanwhile all threads take the scores of tile t from TMEM, run the
//     online softmax in fp32 (exp2, running max with a rescale of the output
//     only when the max grows by more than 2**8), and write P (bf16) to
//     shared memory; thread 0 issues O += P V (M 128, N 256, K 32), reading
//     the same dequantized key tile as an MN-major operand.
// MMA completion is tracked with tcgen05.commit on mbarriers; every wait is
// bounded and a timeout ends the CTA with a status code instead of hanging.
//
// Numerics: scores and the output accumulate in fp32 on the tensor core from
// exact bf16 inputs (the dequantized rows are exact); the probabilities are
// rounded to bf16 for the p.v product while the normaliser sums them
// unrounded; the output is rounded to bf16 once at the end.
#include <cstdint>

#include "kvq.h"
#include "kvq_device.cuh"
#include "kvq_host.h"
#include "mxfp4_decode.cuh"

namespace kvq {
namespace {

constexpr int kHeads = 128;     // MMA M: rows = heads of one query
constexpr int kDim = 512;       // latent width (score depth)
constexpr int kTileKeys = 32;   // MMA N of q.k, K of p.v
constexpr int kHalf = 256;      // output columns per CTA
constexpr int kThreads = 128;
constexpr int kRow = 272;       // packed row bytes

constexpr uint32_t kQBytes = kHeads * kDim * 2;          // 8 K-blocks x 128 rows x 128 B
constexpr uint32_t kKBytes = kTileKeys * kDim * 2;       // 8 K-blocks x 32 rows x 128 B
constexpr uint32_t kPBytes = kHeads * kTileKeys * 2;     // 16 row groups x 4 core matrices
constexpr uint32_t kStageBytes = kTileKeys * kRow;
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffK = kOffQ + kQBytes;              // two buffers
constexpr uint32_t kOffP = kOffK + 2 * kKBytes;          // two buffers
constexpr uint32_t kOffStage = kOffP + 2 * kPBytes;      // two buffers
constexpr uint32_t kOffBias = kOffStage + 2 * kStageBytes;  // four tiles x 32 floats
constexpr uint32_t kOffBar = kOffBias + 4 * kTileKeys * 4;  // three mbarriers
constexpr uint32_t kOffTmemSlot = kOffBar + 32;
constexpr uint32_t kSmemUsed = kOffTmemSlot + 16;
constexpr size_t kSmemBytes = kSmemUsed + 1024;  // room to align the base to 1024

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 0;     // 256 columns
constexpr uint32_t kColS = 256;   // two buffers of 32 columns

constexpr uint32_t kWaitPolls = 1u << 22;

struct AttnParams {
  const uint8_t* q;      // head h of query n at q + n * q_qstride + h * q_hstride (bytes)
  int64_t q_qstride, q_hstride;
  int64_t num_heads;
  const uint8_t* cache;
  int64_t num_slots, block_size, block_stride_rows;
  const int64_t* indices;  // [num_queries, topk]
  int64_t topk;
  float scale_log2;        // sm_scale * log2(e)
  uint8_t* out;            // bf16, head h of query n at out + n * o_qstride + h * o_hstride
  int64_t o_qstride, o_hstride;
  float* lse;              // [num_queries, num_heads] or null
  int32_t* status;         // or null
};

// ------------------------------------------------------------------ PTX ---

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void sts_v4(uint32_t a, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}

__device__ __forceinline__ uint4 lds_v4a(uint32_t a) {
  uint4 r;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "r"(a)
               : "memory");
  return r;
}

__device__ __forceinline__ uint32_t lds_u32a(uint32_t a) {
  uint32_t r;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(r) : "r"(a) : "memory");
  return r;
}

__device__ __forceinline__ void cp_async_16a(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}

// Bounded wait for the completion of the phase with the given parity.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  for (uint32_t i = 0; i < kWaitPolls; ++i)
    if (mbar_test(bar, parity)) return true;
  return false;
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tmem_alloc(uint32_t slot, uint32_t cols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot),
               "r"(cols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t cols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(cols)
               : "memory");
}

// D[tmem] (+)= A[smem] * B[smem], bf16 inputs, fp32 accumulate; one thread.
__device__ __forceinline__ void mma_bf16(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive on `bar` once every MMA issued so far by this thread has completed.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

// 32 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(taddr)
      : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
      "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(
          taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
      "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
      "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}

// Shared-memory matrix descriptor: start address, leading / stride byte
// offsets, the fixed 0b001 at bits 46-48, swizzle mode at bits 61-63
// (0 none, 2 128-byte).
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo,
                                              uint32_t swizzle) {
  return (uint64_t)((addr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | ((uint64_t)swizzle << 61);
}

// Instruction descriptor, kind::f16: fp32 accumulator, bf16 A and B, A
// K-major, B K-major or MN-major, N >> 3 at bit 17, M >> 4 at bit 24.
constexpr uint32_t instr_desc(int m, int n, bool b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((b_mn_major ? 1u : 0u) << 16) |
         ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

constexpr uint32_t kIdescQK = instr_desc(kHeads, kTileKeys, false);
constexpr uint32_t kIdescPV = instr_desc(kHeads, kHalf, true);

// ---------------------------------------------------------------- stages ---

// Warp 0: cp.async the packed rows of tile t into staging buffer t & 1 and
// write the tile's score bias (0 valid, -inf pad or out of range) to bias
// buffer t & 3. Always commits one group (empty past the last tile).
__device__ __forceinline__ void stage_tile(const AttnParams& p, const int64_t* idx_row, int64_t t,
                                           int64_t num_tiles, uint32_t stage_base, float* bias,
                                           int lane) {
  if (t < num_tiles) {
    const int64_t k = t * kTileKeys + lane;
    int64_t s = -1;
    if (k < p.topk) s = ld_once_i64(idx_row + k);
    const bool valid = s >= 0 && s < p.num_slots;
    bias[(t & 3) * kTileKeys + lane] = valid ? 0.0f : -__int_as_float(0x7F800000);
    if (valid) {
      int64_t blk, in_blk;
      divmod_pos(s, p.block_size, blk, in_blk);
      const uint8_t* src = p.cache + (blk * p.block_stride_rows + in_blk) * kRow;
      const uint32_t dst = stage_base + (uint32_t)(t & 1) * kStageBytes + (uint32_t)lane * kRow;
#pragma unroll
      for (int c = 0; c < kRow / 16; ++c) cp_async_16a(dst + 16 * c, src + 16 * c);
    }
  }
  cp_async_commit();
}

// All threads: dequantize tile t (staging buffer t & 1) into key buffer t & 1
// in the 128-byte-swizzled K-major layout: element (key j, dim d) at
// kb*4096 + j*128 + ((c ^ (j & 7)) << 4) + 2*(d & 7), kb = d / 64,
// c = (d % 64) / 8. Thread (j, q) = (tid / 4, tid % 4) does dims
// [128q, 128q + 128) of key j; pad keys become zero rows.
__device__ __forceinline__ void dequant_tile(int64_t t, uint32_t stage_base, uint32_t k_base,
                                             const float* bias, int tid) {
  const int j = tid >> 2, q = tid & 3;
  const uint32_t kdst = k_base + (uint32_t)(t & 1) * kKBytes + (uint32_t)j * 128;
  const uint32_t swz = (uint32_t)(j & 7);
  if (bias[(t & 3) * kTileKeys + j] != 0.0f) {
    const uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int i = 0; i < 16; ++i)
      sts_v4(kdst + (uint32_t)(2 * q + (i >> 3)) * 4096 + ((((uint32_t)i & 7) ^ swz) << 4), z);
    return;
  }
  const uint32_t src = stage_base + (uint32_t)(t & 1) * kStageBytes + (uint32_t)j * kRow;
  const uint32_t sw = lds_u32a(src + 256 + 4 * q);
#pragma unroll
  for (int g = 0; g < 4; ++g) {
    const uint4 c = lds_v4a(src + 64 * q + 16 * g);  // codes of dims 128q + 32g .. +31
    const uint32_t sb = (sw >> (8 * g)) & 0xFFu;
    const ByteTables tb = make_tables(sb);
    const uint32_t words[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = 4 * g + u;  // chunk of 8 dims within the thread's 128
      const uint4 v = decode8_direct(words[u], sb, tb);
      sts_v4(kdst + (uint32_t)(2 * q + (i >> 3)) * 4096 + ((((uint32_t)i & 7) ^ swz) << 4), v);
    }
  }
}

// Thread 0: S(t) = Q K(t)^T into score buffer t & 1.
__device__ __forceinline__ void issue_qk(int64_t t, uint32_t q_base, uint32_t k_base,
                                         uint32_t tmem) {
  const uint32_t kb_base = k_base + (uint32_t)(t & 1) * kKBytes;
  const uint32_t d = tmem + kColS + (uint32_t)(t & 1) * kTileKeys;
#pragma unroll
  for (int kb = 0; kb < 8; ++kb) {
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
      const uint64_t a = smem_desc(q_base + kb * (kHeads * 128) + ks * 32, 16, 1024, 2);
      const uint64_t b = smem_desc(kb_base + kb * (kTileKeys * 128) + ks * 32, 16, 1024, 2);
      mma_bf16(d, a, b, kIdescQK, (kb | ks) != 0);
    }
  }
}

// Thread 0: O (+)= P(t) V(t), V = key buffer t & 1 read MN-major from column
// block 4v (LBO: next 64 columns, SBO: next 8 keys), P K-major without swizzle
// (8x16-byte core matrices; LBO: next 8 keys, SBO: next 8 heads).
__device__ __forceinline__ void issue_pv(int64_t t, int v, uint32_t p_base, uint32_t k_base,
                                         uint32_t tmem) {
  const uint32_t pb = p_base + (uint32_t)(t & 1) * kPBytes;
  const uint32_t vb = k_base + (uint32_t)(t & 1) * kKBytes + (uint32_t)v * 4 * (kTileKeys * 128);
#pragma unroll
  for (int ks = 0; ks < kTileKeys / 16; ++ks) {
    const uint64_t a = smem_desc(pb + ks * 256, 128, 512, 0);
    const uint64_t b = smem_desc(vb + ks * 2048, kTileKeys * 128, 1024, 2);
    mma_bf16(tmem + kColO, a, b, kIdescPV, (t | ks) != 0);
  }
}

// ---------------------------------------------------------------- kernel ---

__global__ void __launch_bounds__(kThreads, 1) mxfp4_attention_kernel(AttnParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* sm = smem_raw + (base - raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t n = blockIdx.x >> 1;
  const int v = blockIdx.x & 1;
  const uint32_t q_base = base + kOffQ, k_base = base + kOffK, p_base = base + kOffP;
  const uint32_t stage_base = base + kOffStage;
  float* bias = reinterpret_cast<float*>(sm + kOffBias);
  const uint32_t bar_s0 = base + kOffBar, bar_s1 = bar_s0 + 8, bar_o = bar_s0 + 16;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + kOffTmemSlot);
  const int64_t num_tiles = (p.topk + kTileKeys - 1) / kTileKeys;
  const int64_t* idx_row = p.indices + n * p.topk;

  if (warp == 0) tmem_alloc(smem_addr(tmem_slot), kTmemCols);
  if (tid == 0) {
    mbar_init(bar_s0, 1);
    mbar_init(bar_s1, 1);
    mbar_init(bar_o, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  // Q: head r of this query into the swizzled K-major layout (zero rows past
  // num_heads), 16 bytes per cp.async.
  const uint8_t* qn = p.q + n * p.q_qstride;
  for (int i = 0; i < kHeads * kDim / 8 / kThreads; ++i) {
    const int id = i * kThreads + tid;
    const int r = id >> 6, c64 = id & 63;
    const uint32_t dst = q_base + (uint32_t)(c64 >> 3) * (kHeads * 128) + (uint32_t)r * 128 +
                         ((((uint32_t)c64 & 7) ^ ((uint32_t)r & 7)) << 4);
    if (r < p.num_heads)
      cp_async_16a(dst, qn + r * p.q_hstride + c64 * 16);
    else
      sts_v4(dst, make_uint4(0, 0, 0, 0));
  }
  cp_async_commit();
  if (warp == 0) {
    stage_tile(p, idx_row, 0, num_tiles, stage_base, bias, lane);
    stage_tile(p, idx_row, 1, num_tiles, stage_base, bias, lane);
    cp_async_wait<1>();  // Q and tile 0 have landed
  } else {
    cp_async_wait<0>();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);

  bool ok = true;
  if (num_tiles > 0) {
    dequant_tile(0, stage_base, k_base, bias, tid);
    fence_proxy_async();
  }
  __syncthreads();
  if (tid == 0 && num_tiles > 0) {
    tc_fence_after();
    issue_qk(0, q_base, k_base, tmem);
    mma_commit(bar_s0);
  }

  float m_ref = -__int_as_float(0x7F800000);  // reference max (log2 units)
  float l = 0.0f;                              // sum of p against m_ref
  for (int64_t t = 0; t < num_tiles; ++t) {
    // A: stage t+2, dequantize t+1 into the key buffer PV(t-1) has released,
    // and start S(t+1) on the tensor core.
    if (warp == 0) stage_tile(p, idx_row, t + 2, num_tiles, stage_base, bias, lane);
    bool good = t == 0 || mbar_wait(bar_o, (uint32_t)((t - 1) & 1));
    if (warp == 0) cp_async_wait<1>();  // tile t+1 staged
    if (__syncthreads_or(!good)) {
      ok = false;
      break;
    }
    if (t + 1 < num_tiles) {
      dequant_tile(t + 1, stage_base, k_base, bias, tid);
      fence_proxy_async();
    }
    __syncthreads();
    if (tid == 0 && t + 1 < num_tiles) {
      tc_fence_after();
      issue_qk(t + 1, q_base, k_base, tmem);
      mma_commit(((t + 1) & 1) ? bar_s1 : bar_s0);
    }
    // B: scores of tile t -> probabilities -> P(t); then O += P(t) V(t).
    good = mbar_wait((t & 1) ? bar_s1 : bar_s0, (uint32_t)((t >> 1) & 1));
    if (__syncthreads_or(!good)) {
      ok = false;
      break;
    }
    tc_fence_after();
    uint32_t sr[32];
    tmem_ld32(lane_base + kColS + (uint32_t)(t & 1) * kTileKeys, sr);
    const float* bt = bias + (t & 3) * kTileKeys;
    float s[32];
    float mt = -__int_as_float(0x7F800000);
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      s[j] = __fmaf_rn(__uint_as_float(sr[j]), p.scale_log2, bt[j]);
      mt = fmaxf(mt, s[j]);
    }
    const bool need = mt > m_ref + 8.0f;
    if (__any_sync(0xFFFFFFFFu, need)) {
      const float f = need ? ex2(m_ref - mt) : 1.0f;  // ex2(-inf) = 0
      if (t > 0) {
#pragma unroll 1
        for (int c = 0; c < kHalf / 32; ++c) {
          uint32_t o[32];
          tmem_ld32(lane_base + kColO + 32 * c, o);
#pragma unroll
          for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * f);
          tmem_st32(lane_base + kColO + 32 * c, o);
        }
      }
      l *= f;
      if (need) m_ref = mt;
    }
    const float mu = m_ref == -__int_as_float(0x7F800000) ? 0.0f : m_ref;
    uint32_t pk[16];
    float lsum = 0.0f;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const float p0 = ex2(s[2 * j] - mu), p1 = ex2(s[2 * j + 1] - mu);
      lsum += p0;
      lsum += p1;
      pk[j] = pack_bf16x2(p0, p1);
    }
    l += lsum;
    const uint32_t prow = p_base + (uint32_t)(t & 1) * kPBytes + (uint32_t)(tid >> 3) * 512 +
                          (uint32_t)(tid & 7) * 16;
#pragma unroll
    for (int c = 0; c < 4; ++c)
      sts_v4(prow + 128 * c, make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]));
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {
      tc_fence_after();
      issue_pv(t, v, p_base, k_base, tmem);
      mma_commit(bar_o);
    }
  }
  if (ok && num_tiles > 0) {
    const bool good = mbar_wait(bar_o, (uint32_t)((num_tiles - 1) & 1));
    if (__syncthreads_or(!good)) ok = false;
  }
  if (!ok) {
    if (tid == 0 && p.status) atomicExch(p.status, 1);
  } else {
    tc_fence_after();
    const int h = tid;
    const bool store = h < p.num_heads;
    uint8_t* orow = p.out + n * p.o_qstride + (int64_t)h * p.o_hstride + (int64_t)v * kHalf * 2;
    const float inv = l > 0.0f ? 1.0f / l : 0.0f;
#pragma unroll 1
    for (int c = 0; c < kHalf / 32; ++c) {
      uint32_t o[32];
      if (num_tiles > 0) {
        tmem_ld32(lane_base + kColO + 32 * c, o);
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) o[j] = 0;
      }
      uint32_t w[16];
#pragma unroll
      for (int j = 0; j < 16; ++j)
        w[j] = l > 0.0f ? pack_bf16x2(__uint_as_float(o[2 * j]) * inv,
                                      __uint_as_float(o[2 * j + 1]) * inv)
                        : 0u;
      if (store) {
#pragma unroll
        for (int u = 0; u < 4; ++u)
          st_v4(orow + 64 * c + 16 * u, make_uint4(w[4 * u], w[4 * u + 1], w[4 * u + 2],
                                                    w[4 * u + 3]));
      }
    }
    if (v == 0 && store && p.lse)
      p.lse[n * p.num_heads + h] =
          l > 0.0f ? (m_ref + __log2f(l)) * 0.69314718055994531f : -__int_as_float(0x7F800000);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace
}  // namespace kvq

extern "C" int mxfp4_mla_sparse_attention(const void* q_bf16, int64_t num_queries,
                                          int64_t num_heads, int64_t q_query_stride,
                                          int64_t q_head_stride, const uint8_t* cache,
                                          int64_t num_blocks, int64_t block_size,
                                          int64_t block_stride_rows, const int64_t* indices,
                                          int64_t topk, float sm_scale, void* out_bf16,
                                          int64_t out_query_stride, int64_t out_head_stride,
                                          float* lse, int32_t* status, cudaStream_t stream) {
  using namespace kvq;
  if (num_queries < 0 || num_heads < 1 || num_heads > kHeads || topk < 0) return KVQ_EINVAL;
  if (num_blocks < 1 || block_size < 1 || block_stride_rows < block_size) return KVQ_EINVAL;
  if (num_blocks > INT64_MAX / block_size) return KVQ_EINVAL;
  if (!(sm_scale == sm_scale) || sm_scale < 0.0f || sm_scale > 3.0e38f) return KVQ_EINVAL;
  if (q_head_stride < kDim || q_head_stride % 8 || q_query_stride % 8) return KVQ_EINVAL;
  if (out_head_stride < kDim || out_head_stride % 8 || out_query_stride % 8) return KVQ_EINVAL;
  if (num_queries > INT64_MAX / 2 / (topk > 0 ? topk : 1)) return KVQ_EINVAL;
  if (num_queries == 0) return KVQ_OK;
  if (!q_bf16 || !cache || !out_bf16 || (topk > 0 && !indices)) return KVQ_EINVAL;
  if (!aligned(q_bf16, 16) || !aligned(cache, 16) || !aligned(out_bf16, 16) ||
      !aligned(indices, 8) || (lse && !aligned(lse, 4)) || (status && !aligned(status, 4)))
    return KVQ_EINVAL;
  if (num_queries > 0x7FFFFFFF / 2) return KVQ_EINVAL;

  static int attr_done[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return KVQ_ECUDA;
  if (!attr_done[dev]) {
    if (cudaFuncSetAttribute(mxfp4_attention_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kSmemBytes) != cudaSuccess)
      return KVQ_ECUDA;
    attr_done[dev] = 1;
  }
  AttnParams p;
  p.q = static_cast<const uint8_t*>(q_bf16);
  p.q_qstride = q_query_stride * 2;
  p.q_hstride = q_head_stride * 2;
  p.num_heads = num_heads;
  p.cache = cache;
  p.num_slots = num_blocks * block_size;
  p.block_size = block_size;
  p.block_stride_rows = block_stride_rows;
  p.indices = indices;
  p.topk = topk;
  p.scale_log2 = sm_scale * 1.4426950408889634f;
  p.out = static_cast<uint8_t*>(out_bf16);
  p.o_qstride = out_query_stride * 2;
  p.o_hstride = out_head_stride * 2;
  p.lse = lse;
  p.status = status;
  mxfp4_attention_kernel<<<(unsigned)(2 * num_queries), kThreads, kSmemBytes, stream>>>(p);
  return launch_status();
}
