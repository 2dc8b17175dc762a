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
// lane = head) holds the output accumulator (256 columns), four 32-key score
// buffers (128; softmax writes the bf16 probabilities P back over the scores
// of the same buffer, and p.v takes P from there as its A operand) and the
// first 256 dims of Q as bf16 pairs (128): the q.k products over those dims
// take Q from tensor memory and read only the key tile from shared memory.
// The other 256 dims of Q stay in shared memory next to four 32 KB key tiles
// of 32 keys (a ring of four stages). Three groups of warps run as a
// pipeline through mbarriers:
//   - producers (warps 4-11, lane = key, warp 4+e = dims [64e, 64e + 64)):
//     load the packed rows three tiles ahead into registers (pads and
//     out-of-range indices load nothing and decode to zero rows),
//     dequantize them with byte permutes into a 128-byte-swizzled K-major
//     bf16 key tile, and arrive on its "full" barrier; a stage is reused once
//     the p.v that last read it has completed;
//   - the issuer (warp 12, one thread), event-driven: O += P(u) V(u)
//     (M 128, N 256, K 32; V is the key tile read MN-major) as soon as
//     softmax has written P(u), else S = Q K^T over two tiles at once
//     (M 128, N 64, K 512: the ring is laid out K-block-major, so the same
//     K-block of two neighbouring stages is one 64-row operand) once both
//     are written and the p.v that last read their tensor-memory columns has
//     been issued (MMAs from one thread run in order); tcgen05.commit on
//     mbarriers tracks completion;
//   - softmax (warps 0-3, one head per thread): read S(t), run the online
//     softmax in fp32 (exp2, running max with a rescale of the output only
//     when the max grows by more than 2**8), and store P (bf16 pairs) into
//     tensor memory.
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
constexpr int kTileKeys = 32;   // MMA N of q.k, K of p.v
constexpr int kStages = 4;      // key tiles (and score / probability buffers) in the ring
constexpr int kHalf = 256;      // output columns per CTA
constexpr int kThreads = 416;   // softmax warps 0-3, producers 4-11, issuer 12
constexpr int kIssuerWarp = 12;
constexpr int kRow = 272;       // packed row bytes
constexpr int kDepth = 3;       // tiles a producer has in flight

constexpr uint32_t kQhiBytes = kHeads * 256 * 2;         // dims 256..511: 4 K-blocks x 128 rows
constexpr uint32_t kKBytes = kTileKeys * kDim * 2;       // 8 K-blocks x 32 rows x 128 B
constexpr uint32_t kKBlock = kTileKeys * 128;            // bytes of one K-block of a key tile
// The ring is laid out K-block-major: K-block kb of stage s at
// (kb * kStages + s) * kKBlock, so the same K-block of stages s and s + 1
// (s even) is one 64-row block and q.k runs at N = 64 over a pair of stages.
constexpr uint32_t kKBlockStride = kStages * kKBlock;
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffK = kOffQ + kQhiBytes;            // kStages buffers
constexpr uint32_t kOffBar = kOffK + kStages * kKBytes;  // sixteen mbarriers
constexpr uint32_t kOffTmemSlot = kOffBar + 128;
constexpr uint32_t kOffAbort = kOffTmemSlot + 16;
constexpr uint32_t kSmemUsed = kOffAbort + 16;
constexpr size_t kSmemBytes = kSmemUsed + 1024;  // room to align the base to 1024

// mbarriers, one of each per stage (tile t uses stage t % kStages)
constexpr uint32_t kBarKFull = 0, kBarSFull = 32, kBarPFull = 64, kBarPvDone = 96;

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 0;     // 256 columns
constexpr uint32_t kColS = 256;   // kStages buffers of 32 columns: scores, then P over them
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

// 16 consecutive 32-bit columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15])
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

constexpr uint32_t kIdescQK = instr_desc(kHeads, 2 * kTileKeys, false);
constexpr uint32_t kIdescPV = instr_desc(kHeads, kHalf, true);

// --------------------------------------------------------------- producer ---

// One producer thread's share of a key row: the 32 code bytes of dims
// [64e, 64e + 64) and the two scale bytes of those groups (low 16 bits of s).
// A pad or an out-of-range index loads nothing: zero codes decode to +0.0
// under any scale byte in [2, 252].
struct Packed {
  uint4 c[2];
  uint32_t s;
};

__device__ __forceinline__ int64_t key_index(const AttnParams& p, const int64_t* idx_row,
                                             int64_t k) {
  return k < p.topk ? ld_once_i64(idx_row + k) : -1;
}

__device__ __forceinline__ uint32_t ld_issue_u16(const void* p) {
  uint16_t r;
  asm volatile("ld.global.nc.L1::no_allocate.u16 %0, [%1];" : "=h"(r) : "l"(p));
  return r;
}

__device__ __forceinline__ Packed load_packed(const AttnParams& p, int64_t s, int e) {
  Packed r;
  if (s >= 0 && s < p.num_slots) {
    // blocks laid end to end (stride = block size): the row is the slot
    int64_t row_index = s;
    if (p.block_stride_rows != p.block_size) {
      int64_t blk, in_blk;
      divmod_pos(s, p.block_size, blk, in_blk);
      row_index = blk * p.block_stride_rows + in_blk;
    }
    const uint8_t* row = p.cache + row_index * kRow;
    r.c[0] = ld_issue_v4(row + 32 * e);
    r.c[1] = ld_issue_v4(row + 32 * e + 16);
    r.s = ld_issue_u16(row + 256 + 2 * e);
  } else {
    r.c[0] = make_uint4(0, 0, 0, 0);
    r.c[1] = r.c[0];
    r.s = 0x7F7Fu;
  }
  return r;
}

// Dims [64e, 64e + 64) (K-block e) of key j into the stage whose K-block 0
// is at `kbuf`, 128-byte-swizzled K-major: element (key j, dim d) at
// kb*kKBlockStride + j*128 + ((c ^ (j & 7)) << 4) + 2*(d & 7), kb = d / 64,
// c = (d % 64) / 8. With lane = key, each 8-lane phase of a 16-byte store
// covers eight keys and all eight bank groups.
__device__ __forceinline__ void dequant_share(const Packed& x, uint32_t kbuf, int j, int e) {
  const uint32_t row = kbuf + (uint32_t)e * kKBlockStride + (uint32_t)j * 128;
  const uint32_t swz = (uint32_t)(j & 7);
#pragma unroll
  for (int g = 0; g < 2; ++g) {
    const uint32_t sb = (x.s >> (8 * g)) & 0xFFu;
    const ByteTables tb = make_tables(sb);
    const uint32_t words[4] = {x.c[g].x, x.c[g].y, x.c[g].z, x.c[g].w};
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const uint32_t c = (uint32_t)(4 * g + u);  // chunk of 8 dims within the K-block
      sts_v4(row + ((c ^ swz) << 4), decode8_direct(words[u], sb, tb));
    }
  }
}

// --------------------------------------------------------------- issuer ---

// Descriptors are built once per tile: a descriptor's start address field
// holds address >> 4 in its low 14 bits, and shared-memory addresses stay
// below 2**18, so adding a byte offset / 16 to a base descriptor moves the
// start without carrying into the other fields (fewer instructions in the
// issuing thread, which shares its SMSP with busy warps).
__device__ __forceinline__ uint64_t desc_at(uint64_t base_desc, uint32_t byte_offset) {
  return base_desc + (uint64_t)(byte_offset >> 4);
}

// S(t), S(t+1) = Q K^T over the pair of stages t % kStages (even) and the
// next, into their score columns (N = 64): dims 0..255 with Q from TMEM (16
// steps of 8 columns), dims 256..511 with Q from shared memory. When t is the
// last tile, the second half computes scores of a stage no tile reads.
__device__ __forceinline__ void issue_qk(int64_t t, uint64_t q_desc, uint32_t k_base,
                                         uint32_t tmem) {
  const uint32_t st = (uint32_t)(t % kStages);
  const uint64_t k_desc = smem_desc(k_base + st * kKBlock, 16, 1024, 2);
  const uint32_t d = tmem + kColS + st * kTileKeys;
#pragma unroll
  for (int kb = 0; kb < 4; ++kb) {
#pragma unroll
    for (int ks = 0; ks < 4; ++ks)
      mma_bf16_ta(d, tmem + kColQ + (uint32_t)(8 * (4 * kb + ks)),
                  desc_at(k_desc, kb * kKBlockStride + ks * 32), kIdescQK, (kb | ks) != 0);
  }
#pragma unroll
  for (int kb = 4; kb < 8; ++kb) {
#pragma unroll
    for (int ks = 0; ks < 4; ++ks)
      mma_bf16(d, desc_at(q_desc, (kb - 4) * (kHeads * 128) + ks * 32),
               desc_at(k_desc, kb * kKBlockStride + ks * 32), kIdescQK, 1);
  }
}

// O (+)= P(t) V(t): P (bf16 pairs, written by softmax over the score
// columns of stage t % kStages) is the TMEM A operand, 8 columns per step of
// 16 keys; V is the stage's key rows read MN-major from column block 4v
// (LBO: the stage's next K-block, SBO: next 8 keys).
__device__ __forceinline__ void issue_pv(int64_t t, int v, uint32_t k_base, uint32_t tmem) {
  const uint32_t st = (uint32_t)(t % kStages);
  const uint64_t v_desc = smem_desc(k_base + ((uint32_t)v * 4 * kStages + st) * kKBlock,
                                    kKBlockStride, 1024, 2);
  const uint32_t pa = tmem + kColS + st * kTileKeys;
#pragma unroll
  for (int ks = 0; ks < kTileKeys / 16; ++ks)
    mma_bf16_ta(tmem + kColO, pa + 8 * ks, desc_at(v_desc, ks * 2048), kIdescPV, (t | ks) != 0);
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
  const uint32_t q_base = base + kOffQ, k_base = base + kOffK;
  const uint32_t bars = base + kOffBar;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + kOffTmemSlot);
  volatile int* abort = reinterpret_cast<volatile int*>(sm + kOffAbort);
  const int64_t num_tiles = (p.topk + kTileKeys - 1) / kTileKeys;
  const int64_t* idx_row = p.indices + n * p.topk;

  if (warp == kIssuerWarp) tmem_alloc(smem_addr(tmem_slot), kTmemCols);
  if (tid == 0) {
#pragma unroll
    for (int b = 0; b < kStages; ++b) {
      mbar_init(bars + kBarKFull + 8 * b, 256);
      mbar_init(bars + kBarSFull + 8 * b, 1);
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
    // Lane = key of the tile, warp 4 + e = dims [64e, 64e + 64). Key buffer
    // t % kStages is free once PV(t - kStages) has completed.
    const int e = warp - 4, j = lane;
    Packed buf[kDepth];
#pragma unroll
    for (int u = 0; u < kDepth; ++u)
      buf[u] = load_packed(p, key_index(p, idx_row, (int64_t)u * kTileKeys + j), e);
    int64_t s_next = key_index(p, idx_row, (int64_t)kDepth * kTileKeys + j);
    bool live = true;
    for (int64_t t0 = 0; t0 < num_tiles && live; t0 += kDepth) {
#pragma unroll
      for (int u = 0; u < kDepth; ++u) {
        const int64_t t = t0 + u;
        if (t < num_tiles && live) {
          const Packed cur = buf[u];
          buf[u] = load_packed(p, s_next, e);  // tile t + kDepth
          s_next = key_index(p, idx_row, (t + kDepth + 1) * kTileKeys + j);
          const uint32_t st = (uint32_t)(t % kStages);
          if (t >= kStages &&
              !mbar_wait(bars + kBarPvDone + 8 * st, (uint32_t)(((t / kStages) - 1) & 1), abort)) {
            live = false;
          } else {
            dequant_share(cur, k_base + st * kKBlock, j, e);
            fence_proxy_async();
            mbar_arrive(bars + kBarKFull + 8 * st);
          }
        }
      }
    }
  } else if (warp == kIssuerWarp) {
    // --------------------------------------------------------------- issuer
    if (lane == 0) {
      const uint64_t q_desc = smem_desc(q_base, 16, 1024, 2);
      // Event-driven: O += P(u) V(u) as soon as softmax has written P(u) (it
      // frees key stage u % kStages, so it goes first), else q.k over the
      // pair of tiles t, t + 1 (t even) once both are written and PV(t - 3),
      // the last reader of their TMEM columns, has been issued (MMAs from
      // this thread run in order). Polls without progress are bounded.
      int64_t t = 0, u = 0;
      uint32_t idle = 0;
      while (u < num_tiles) {
        if (u < t && mbar_test(bars + kBarPFull + 8 * (uint32_t)(u % kStages),
                               (uint32_t)((u / kStages) & 1))) {
          tc_fence_after();
          issue_pv(u, v, k_base, tmem);
          mma_commit(bars + kBarPvDone + 8 * (uint32_t)(u % kStages));
          ++u;
          idle = 0;
        } else if (t < num_tiles && t + 1 - u < kStages &&
                   mbar_test(bars + kBarKFull + 8 * (uint32_t)(t % kStages),
                             (uint32_t)((t / kStages) & 1)) &&
                   (t + 1 >= num_tiles ||
                    mbar_test(bars + kBarKFull + 8 * (uint32_t)((t + 1) % kStages),
                              (uint32_t)(((t + 1) / kStages) & 1)))) {
          tc_fence_after();
          issue_qk(t, q_desc, k_base, tmem);
          mma_commit(bars + kBarSFull + 8 * (uint32_t)(t % kStages));
          if (t + 1 < num_tiles) mma_commit(bars + kBarSFull + 8 * (uint32_t)((t + 1) % kStages));
          t += 2;
          idle = 0;
        } else if (++idle >= kWaitPolls) {
          *abort = 1;
          break;
        } else if ((idle & 31u) == 31u && *abort) {
          break;
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
    int64_t s_key = key_index(p, idx_row, lane);
    for (int64_t t = 0; t < num_tiles && live; ++t) {
      const uint32_t mask = __ballot_sync(0xFFFFFFFFu, s_key >= 0 && s_key < p.num_slots);
      s_key = key_index(p, idx_row, (t + 1) * kTileKeys + lane);
      const uint32_t st = (uint32_t)(t % kStages);
      if (!warp_wait(bars + kBarSFull + 8 * st, (uint32_t)((t / kStages) & 1), abort)) {
        live = false;
        break;
      }
      tc_fence_after();
      const uint32_t scol = lane_base + kColS + st * kTileKeys;
      uint32_t sr[32];
      tmem_ld32(scol, sr);
      // the tile max (log2 units, -inf for dropped keys), four chains
      float mc[4] = {-__int_as_float(0x7F800000), -__int_as_float(0x7F800000),
                     -__int_as_float(0x7F800000), -__int_as_float(0x7F800000)};
#pragma unroll
      for (int k = 0; k < 32; ++k)
        if ((mask >> k) & 1u)
          mc[k & 3] = fmaxf(mc[k & 3], __fmul_rn(__uint_as_float(sr[k]), p.scale_log2));
      const float mt = fmaxf(fmaxf(mc[0], mc[1]), fmaxf(mc[2], mc[3]));
      const bool need = mt > m_ref + 8.0f;
      if (__any_sync(0xFFFFFFFFu, need)) {
        const float f = need ? ex2(m_ref - mt) : 1.0f;  // ex2(-inf) = 0
        if (t > 0) {
          // O may be touched only once PV(t-1) has completed
          const int64_t w = t - 1;
          if (!warp_wait(bars + kBarPvDone + 8 * (uint32_t)(w % kStages),
                         (uint32_t)((w / kStages) & 1), abort)) {
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
      // probabilities, their sum, and P (bf16 pairs) over the score columns
      float lsum0 = 0.0f, lsum1 = 0.0f;
      uint32_t pk[16];
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        const float x0 = ((mask >> (2 * k)) & 1u)
                             ? __fmul_rn(__uint_as_float(sr[2 * k]), p.scale_log2)
                             : -__int_as_float(0x7F800000);
        const float x1 = ((mask >> (2 * k + 1)) & 1u)
                             ? __fmul_rn(__uint_as_float(sr[2 * k + 1]), p.scale_log2)
                             : -__int_as_float(0x7F800000);
        const float p0 = ex2(x0 - mu), p1 = ex2(x1 - mu);
        lsum0 += p0;
        lsum1 += p1;
        pk[k] = pack_bf16x2(p0, p1);
      }
      tmem_st16(scol, pk);
      l += lsum0 + lsum1;
      tc_fence_before();
      mbar_arrive(bars + kBarPFull + 8 * st);
    }
    if (live && num_tiles > 0 &&
        !warp_wait(bars + kBarPvDone + 8 * (uint32_t)((num_tiles - 1) % kStages),
                   (uint32_t)(((num_tiles - 1) / kStages) & 1), abort))
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
