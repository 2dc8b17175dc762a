// mxfp4_attention.cu — mxfp4_mla_sparse_attention: sparse MLA decode attention
// that reads the packed MXFP4 cache directly, on the tcgen05 tensor cores.
//
// Follows PR 60321 "Add an mxfp4_mla KV cache for rope-free sparse MLA"
// (Read path: each query's top-k rows are gathered and unpacked to bf16 and
// feed both dots, q.k and p.v; Claims: attention over the packed cache equals
// attention over the dequantized bf16 values). For the rope-free latent the
// key and the value of a token are the same 512-wide row.
//
// Work decomposition. One CTA per (query, half of the 512 value columns): the
// two CTAs of a query both form the full scores q.k (512-deep) and each
// accumulates 256 output columns. Tensor memory (512 columns x 128 lanes,
// lane = head) holds the output accumulator (256 columns), two 64-key score
// buffers (128) and the first 256 dims of Q as bf16 pairs (128): the q.k
// products over those dims take Q from tensor memory and read only the key
// tile from shared memory, which halves their shared-memory traffic (a
// 128 x 64 x 16 product that reads both operands from shared memory is bound
// by it). The other 256 dims of Q stay in shared memory. Keys go in tiles of
// 64, and three groups of warps run as a pipeline through mbarriers:
//   - producers (warps 4-11, lane = key, two warps per quarter of the row):
//     load the packed rows two tiles ahead into registers (pads and
//     out-of-range indices load nothing and decode to zero rows),
//     dequantize them with byte permutes into a 128-byte-swizzled K-major
//     bf16 key tile (two buffers), and arrive on its "full" barrier;
//   - the issuer (warp 12, one thread): S(t) = Q K^T (M 128, N 64, K 512)
//     into one of two score buffers once the tile and the buffer are free,
//     then O += P(t-1) V(t-1) (M 128, N 256, K 64; V is the same key tile read
//     MN-major) once softmax has written P; tcgen05.commit on mbarriers
//     tracks completion;
//   - softmax (warps 0-3, one head per thread): read S(t), release its
//     buffer, run the online softmax in fp32 (exp2, running max with a
//     rescale of the output only when the max grows by more than 2**8), and
//     write P (bf16, two buffers) to shared memory.
// Every wait is bounded; a timeout sets a CTA-wide abort flag that ends the
// other roles' waits, and the CTA reports through an optional status word.
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
constexpr int kTileKeys = 64;   // MMA N of q.k, K of p.v
constexpr int kHalf = 256;      // output columns per CTA
constexpr int kThreads = 416;   // softmax warps 0-3, producers 4-11, issuer 12
constexpr int kIssuerWarp = 12;
constexpr int kRow = 272;       // packed row bytes
constexpr int kDepth = 2;       // tiles a producer has in flight

constexpr uint32_t kQhiBytes = kHeads * 256 * 2;         // dims 256..511: 4 K-blocks x 128 rows
constexpr uint32_t kKBytes = kTileKeys * kDim * 2;       // 8 K-blocks x 64 rows x 128 B
constexpr uint32_t kKBlock = kTileKeys * 128;            // bytes of one K-block of a key tile
constexpr uint32_t kPBytes = kHeads * kTileKeys * 2;     // 16 row groups x 8 core matrices
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffK = kOffQ + kQhiBytes;            // two buffers
constexpr uint32_t kOffP = kOffK + 2 * kKBytes;          // two buffers
constexpr uint32_t kOffBar = kOffP + 2 * kPBytes;        // ten mbarriers
constexpr uint32_t kOffTmemSlot = kOffBar + 128;
constexpr uint32_t kOffAbort = kOffTmemSlot + 16;
constexpr uint32_t kSmemUsed = kOffAbort + 16;
constexpr size_t kSmemBytes = kSmemUsed + 1024;  // room to align the base to 1024

// mbarriers, two of each (buffer t & 1)
constexpr uint32_t kBarKFull = 0, kBarSFull = 16, kBarSEmpty = 32, kBarPFull = 48, kBarPvDone = 64;

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 0;     // 256 columns
constexpr uint32_t kColS = 256;   // two buffers of 64 columns
constexpr uint32_t kColQ = 384;   // Q dims 0..255 as 128 columns of bf16 pairs

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

__device__ __forceinline__ void cp_async_16a(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

// Global loads issued where they stand (asm volatile): a producer's prefetch
// of packed rows must not be moved down to its first use a tile later.
__device__ __forceinline__ uint4 ld_issue_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

__device__ __forceinline__ uint32_t ld_issue_u32(const void* p) {
  uint32_t r;
  asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(r) : "l"(p));
  return r;
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

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Bounded wait for the completion of the phase with the given parity. Gives
// up when another role of the CTA has raised the abort flag, or after
// kWaitPolls polls (then raises it itself).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort) {
  for (uint32_t i = 0; i < kWaitPolls; ++i) {
    if (mbar_test(bar, parity)) return true;
    if ((i & 31u) == 31u && *abort) return false;
  }
  *abort = 1;
  return false;
}

// mbar_wait with one outcome for the whole warp (the softmax warps follow it
// with warp-collective TMEM loads).
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort) {
  return __all_sync(0xFFFFFFFFu, mbar_wait(bar, parity, abort));
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

// As mma_bf16 with A (M x 16, lane = row, 8 columns of bf16 pairs) in TMEM.
__device__ __forceinline__ void mma_bf16_ta(uint32_t d, uint32_t a_tmem, uint64_t b,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(accumulate)
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

// --------------------------------------------------------------- producer ---

// One producer thread's share of a key row: the 64 code bytes of dims
// [128q, 128q + 128) and the four scale bytes of those groups. A pad or an
// out-of-range index loads nothing: zero codes decode to +0.0 under any
// scale byte in [2, 252].
struct Packed {
  uint4 c[4];
  uint32_t s;
};

__device__ __forceinline__ int64_t key_index(const AttnParams& p, const int64_t* idx_row,
                                             int64_t k) {
  return k < p.topk ? ld_once_i64(idx_row + k) : -1;
}

__device__ __forceinline__ Packed load_packed(const AttnParams& p, int64_t s, int q) {
  Packed r;
  if (s >= 0 && s < p.num_slots) {
    int64_t blk, in_blk;
    divmod_pos(s, p.block_size, blk, in_blk);
    const uint8_t* row = p.cache + (blk * p.block_stride_rows + in_blk) * kRow;
#pragma unroll
    for (int g = 0; g < 4; ++g) r.c[g] = ld_issue_v4(row + 64 * q + 16 * g);
    r.s = ld_issue_u32(row + 256 + 4 * q);
  } else {
#pragma unroll
    for (int g = 0; g < 4; ++g) r.c[g] = make_uint4(0, 0, 0, 0);
    r.s = 0x7F7F7F7Fu;
  }
  return r;
}

// Dims [128q, 128q + 128) of key j into key buffer `kbuf`, 128-byte-swizzled
// K-major: element (key j, dim d) at kb*kKBlock + j*128 + ((c ^ (j & 7)) << 4)
// + 2*(d & 7), kb = d / 64, c = (d % 64) / 8. With lane = key, each 8-lane
// phase of a 16-byte store covers eight keys and all eight bank groups.
__device__ __forceinline__ void dequant_share(const Packed& x, uint32_t kbuf, int j, int q) {
  const uint32_t kdst = kbuf + (uint32_t)j * 128;
  const uint32_t swz = (uint32_t)(j & 7);
#pragma unroll
  for (int g = 0; g < 4; ++g) {
    const uint32_t sb = (x.s >> (8 * g)) & 0xFFu;
    const ByteTables tb = make_tables(sb);
    const uint32_t words[4] = {x.c[g].x, x.c[g].y, x.c[g].z, x.c[g].w};
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = 4 * g + u;  // chunk of 8 dims within the thread's 128
      const uint4 v = decode8_direct(words[u], sb, tb);
      sts_v4(kdst + (uint32_t)(2 * q + (i >> 3)) * kKBlock + ((((uint32_t)i & 7) ^ swz) << 4),
             v);
    }
  }
}

// --------------------------------------------------------------- issuer ---

// S(t) = Q K(t)^T into score buffer t & 1: dims 0..255 with Q from TMEM
// (16 steps of 8 columns), dims 256..511 with Q from shared memory.
__device__ __forceinline__ void issue_qk(int64_t t, uint32_t q_base, uint32_t k_base,
                                         uint32_t tmem) {
  const uint32_t kb_base = k_base + (uint32_t)(t & 1) * kKBytes;
  const uint32_t d = tmem + kColS + (uint32_t)(t & 1) * kTileKeys;
#pragma unroll
  for (int kb = 0; kb < 4; ++kb) {
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
      const uint64_t b = smem_desc(kb_base + kb * kKBlock + ks * 32, 16, 1024, 2);
      mma_bf16_ta(d, tmem + kColQ + (uint32_t)(8 * (4 * kb + ks)), b, kIdescQK, (kb | ks) != 0);
    }
  }
#pragma unroll
  for (int kb = 4; kb < 8; ++kb) {
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
      const uint64_t a = smem_desc(q_base + (kb - 4) * (kHeads * 128) + ks * 32, 16, 1024, 2);
      const uint64_t b = smem_desc(kb_base + kb * kKBlock + ks * 32, 16, 1024, 2);
      mma_bf16(d, a, b, kIdescQK, 1);
    }
  }
}

// O (+)= P(t) V(t), V = key buffer t & 1 read MN-major from column block 4v
// (LBO: next 64 columns, SBO: next 8 keys), P K-major without swizzle
// (8x16-byte core matrices; LBO: next 8 keys, SBO: next 8 heads).
__device__ __forceinline__ void issue_pv(int64_t t, int v, uint32_t p_base, uint32_t k_base,
                                         uint32_t tmem) {
  const uint32_t pb = p_base + (uint32_t)(t & 1) * kPBytes;
  const uint32_t vb = k_base + (uint32_t)(t & 1) * kKBytes + (uint32_t)v * 4 * kKBlock;
#pragma unroll
  for (int ks = 0; ks < kTileKeys / 16; ++ks) {
    const uint64_t a = smem_desc(pb + ks * 256, 128, 1024, 0);
    const uint64_t b = smem_desc(vb + ks * 2048, kKBlock, 1024, 2);
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
  const uint32_t bars = base + kOffBar;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + kOffTmemSlot);
  volatile int* abort = reinterpret_cast<volatile int*>(sm + kOffAbort);
  const int64_t num_tiles = (p.topk + kTileKeys - 1) / kTileKeys;
  const int64_t* idx_row = p.indices + n * p.topk;

  if (warp == kIssuerWarp) tmem_alloc(smem_addr(tmem_slot), kTmemCols);
  if (tid == 0) {
#pragma unroll
    for (int b = 0; b < 2; ++b) {
      mbar_init(bars + kBarKFull + 8 * b, 256);
      mbar_init(bars + kBarSFull + 8 * b, 1);
      mbar_init(bars + kBarSEmpty + 8 * b, 128);
      mbar_init(bars + kBarPFull + 8 * b, 128);
      mbar_init(bars + kBarPvDone + 8 * b, 1);
    }
    *abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  // Q dims 256..511 of head r into the swizzled K-major layout (zero rows past
  // num_heads), 16 bytes per cp.async.
  const uint8_t* qn = p.q + n * p.q_qstride;
  for (int id = tid; id < kHeads * 32; id += kThreads) {
    const int r = id >> 5, c32 = id & 31;
    const uint32_t dst = q_base + (uint32_t)(c32 >> 3) * (kHeads * 128) + (uint32_t)r * 128 +
                         ((((uint32_t)c32 & 7) ^ ((uint32_t)r & 7)) << 4);
    if (r < p.num_heads)
      cp_async_16a(dst, qn + r * p.q_hstride + 512 + c32 * 16);
    else
      sts_v4(dst, make_uint4(0, 0, 0, 0));
  }
  cp_async_commit();
  cp_async_wait<0>();
  fence_proxy_async();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (warp < 4) {
    // Q dims 0..255 of head `tid` into TMEM lane `tid`, columns kColQ.. as
    // bf16 pairs (the A operand of the first 16 q.k steps).
    const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
    const uint8_t* qrow = qn + (int64_t)tid * p.q_hstride;
#pragma unroll 1
    for (int c = 0; c < 4; ++c) {
      uint32_t w[32];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const uint4 x = tid < p.num_heads ? ld_once_v4(qrow + 128 * c + 16 * k)
                                          : make_uint4(0, 0, 0, 0);
        w[4 * k] = x.x;
        w[4 * k + 1] = x.y;
        w[4 * k + 2] = x.z;
        w[4 * k + 3] = x.w;
      }
      tmem_st32(lane_base + kColQ + 32 * c, w);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  if (warp >= 4 && warp < kIssuerWarp) {
    // ------------------------------------------------------------ producers
    const int j = lane + 32 * (warp & 1), q = (warp - 4) >> 1;
    Packed buf[kDepth];
#pragma unroll
    for (int u = 0; u < kDepth; ++u)
      buf[u] = load_packed(p, key_index(p, idx_row, (int64_t)u * kTileKeys + j), q);
    int64_t s_next = key_index(p, idx_row, (int64_t)kDepth * kTileKeys + j);
    bool live = true;
    for (int64_t t0 = 0; t0 < num_tiles && live; t0 += kDepth) {
#pragma unroll
      for (int u = 0; u < kDepth; ++u) {
        const int64_t t = t0 + u;
        if (t < num_tiles && live) {
          const Packed cur = buf[u];
          buf[u] = load_packed(p, s_next, q);  // tile t + kDepth
          s_next = key_index(p, idx_row, (t + kDepth + 1) * kTileKeys + j);
          // key buffer t & 1 is free once PV(t-2) has completed
          if (t >= 2 && !mbar_wait(bars + kBarPvDone + 8 * (t & 1), (uint32_t)(((t - 2) >> 1) & 1),
                                   abort)) {
            live = false;
          } else {
            dequant_share(cur, k_base + (uint32_t)(t & 1) * kKBytes, j, q);
            fence_proxy_async();
            mbar_arrive(bars + kBarKFull + 8 * (t & 1));
          }
        }
      }
    }
  } else if (warp == kIssuerWarp) {
    // --------------------------------------------------------------- issuer
    if (lane == 0) {
      for (int64_t t = 0; t <= num_tiles; ++t) {
        if (t < num_tiles) {
          if (!mbar_wait(bars + kBarKFull + 8 * (t & 1), (uint32_t)((t >> 1) & 1), abort)) break;
          if (t >= 2 && !mbar_wait(bars + kBarSEmpty + 8 * (t & 1),
                                   (uint32_t)(((t - 2) >> 1) & 1), abort))
            break;
          tc_fence_after();
          issue_qk(t, q_base, k_base, tmem);
          mma_commit(bars + kBarSFull + 8 * (t & 1));
        }
        if (t >= 1) {
          const int64_t u = t - 1;
          if (!mbar_wait(bars + kBarPFull + 8 * (u & 1), (uint32_t)((u >> 1) & 1), abort)) break;
          tc_fence_after();
          issue_pv(u, v, p_base, k_base, tmem);
          mma_commit(bars + kBarPvDone + 8 * (u & 1));
        }
      }
    }
    __syncwarp();
  } else {
    // -------------------------------------------------------------- softmax
    const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
    float m_ref = -__int_as_float(0x7F800000);  // reference max (log2 units)
    float l = 0.0f;                              // sum of p against m_ref
    bool live = true;
    int64_t s_lo = key_index(p, idx_row, lane), s_hi = key_index(p, idx_row, 32 + lane);
    for (int64_t t = 0; t < num_tiles && live; ++t) {
      const uint32_t mask_lo = __ballot_sync(0xFFFFFFFFu, s_lo >= 0 && s_lo < p.num_slots);
      const uint32_t mask_hi = __ballot_sync(0xFFFFFFFFu, s_hi >= 0 && s_hi < p.num_slots);
      s_lo = key_index(p, idx_row, (t + 1) * kTileKeys + lane);
      s_hi = key_index(p, idx_row, (t + 1) * kTileKeys + 32 + lane);
      if (!warp_wait(bars + kBarSFull + 8 * (t & 1), (uint32_t)((t >> 1) & 1), abort)) {
        live = false;
        break;
      }
      tc_fence_after();
      const uint32_t scol = lane_base + kColS + (uint32_t)(t & 1) * kTileKeys;
      // Pass 1: the tile max (scores in log2 units, -inf for dropped keys).
      float mt = -__int_as_float(0x7F800000);
#pragma unroll 1
      for (int hf = 0; hf < 2; ++hf) {
        uint32_t sr[32];
        tmem_ld32(scol + 32 * hf, sr);
        const uint32_t m = hf ? mask_hi : mask_lo;
#pragma unroll
        for (int k = 0; k < 32; ++k)
          if ((m >> k) & 1u) mt = fmaxf(mt, __fmul_rn(__uint_as_float(sr[k]), p.scale_log2));
      }
      const bool need = mt > m_ref + 8.0f;
      if (__any_sync(0xFFFFFFFFu, need)) {
        const float f = need ? ex2(m_ref - mt) : 1.0f;  // ex2(-inf) = 0
        if (t > 0) {
          // O may be touched only once PV(t-1) has completed
          if (!warp_wait(bars + kBarPvDone + 8 * ((t - 1) & 1), (uint32_t)(((t - 1) >> 1) & 1),
                         abort)) {
            live = false;
            break;
          }
          tc_fence_after();
#pragma unroll 1
          for (int c = 0; c < kHalf / 32; ++c) {
            uint32_t o[32];
            tmem_ld32(lane_base + kColO + 32 * c, o);
#pragma unroll
            for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * f);
            tmem_st32(lane_base + kColO + 32 * c, o);
          }
        }
        l *= f;
        if (need) m_ref = mt;
      }
      const float mu = m_ref == -__int_as_float(0x7F800000) ? 0.0f : m_ref;
      // P buffer t & 1 is free once PV(t-2) has completed
      if (t >= 2 && !warp_wait(bars + kBarPvDone + 8 * (t & 1), (uint32_t)(((t - 2) >> 1) & 1),
                               abort)) {
        live = false;
        break;
      }
      // Pass 2: probabilities, their sum, and P (bf16) for this head's row.
      const uint32_t prow = p_base + (uint32_t)(t & 1) * kPBytes + (uint32_t)(tid >> 3) * 1024 +
                            (uint32_t)(tid & 7) * 16;
      float lsum0 = 0.0f, lsum1 = 0.0f;
#pragma unroll 1
      for (int hf = 0; hf < 2; ++hf) {
        uint32_t sr[32];
        tmem_ld32(scol + 32 * hf, sr);
        const uint32_t m = hf ? mask_hi : mask_lo;
        uint32_t pk[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const float x0 = ((m >> (2 * k)) & 1u)
                               ? __fmul_rn(__uint_as_float(sr[2 * k]), p.scale_log2)
                               : -__int_as_float(0x7F800000);
          const float x1 = ((m >> (2 * k + 1)) & 1u)
                               ? __fmul_rn(__uint_as_float(sr[2 * k + 1]), p.scale_log2)
                               : -__int_as_float(0x7F800000);
          const float p0 = ex2(x0 - mu), p1 = ex2(x1 - mu);
          lsum0 += p0;
          lsum1 += p1;
          pk[k] = pack_bf16x2(p0, p1);
        }
#pragma unroll
        for (int c = 0; c < 4; ++c)
          sts_v4(prow + 128 * (4 * hf + c),
                 make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]));
      }
      l += lsum0 + lsum1;
      tc_fence_before();
      mbar_arrive(bars + kBarSEmpty + 8 * (t & 1));
      fence_proxy_async();
      tc_fence_before();
      mbar_arrive(bars + kBarPFull + 8 * (t & 1));
    }
    if (live && num_tiles > 0 &&
        !warp_wait(bars + kBarPvDone + 8 * ((num_tiles - 1) & 1),
                   (uint32_t)(((num_tiles - 1) >> 1) & 1), abort))
      live = false;
    live = __all_sync(0xFFFFFFFFu, live && !*abort);
    if (live) {
      tc_fence_after();
      const int h = tid;
      const bool store = h < p.num_heads;
      uint8_t* orow =
          p.out + n * p.o_qstride + (int64_t)h * p.o_hstride + (int64_t)v * kHalf * 2;
      const float inv = l > 0.0f ? 1.0f / l : 0.0f;
#pragma unroll 1
      for (int c = 0; c < kHalf / 32; ++c) {
        uint32_t o[32];
        if (num_tiles > 0) {
          tmem_ld32(lane_base + kColO + 32 * c, o);
        } else {
#pragma unroll
          for (int k = 0; k < 32; ++k) o[k] = 0;
        }
        uint32_t w[16];
#pragma unroll
        for (int k = 0; k < 16; ++k)
          w[k] = l > 0.0f ? pack_bf16x2(__uint_as_float(o[2 * k]) * inv,
                                        __uint_as_float(o[2 * k + 1]) * inv)
                          : 0u;
        if (store) {
#pragma unroll
          for (int u = 0; u < 4; ++u)
            st_v4(orow + 64 * c + 16 * u, make_uint4(w[4 * u], w[4 * u + 1], w[4 * u + 2],
                                                      w[4 * u + 3]));
        }
      }
      if (v == 0 && store && p.lse)
        p.lse[n * p.num_heads + h] = l > 0.0f ? (m_ref + __log2f(l)) * 0.69314718055994531f
                                              : -__int_as_float(0x7F800000);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (tid == 0 && *abort && p.status) atomicExch(p.status, 1);
  if (warp == kIssuerWarp) {
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
