// mxfp4_attention.cu — mxfp4_mla_sparse_attention: sparse MLA decode attention
// that reads the packed MXFP4 cache directly, on the tcgen05 tensor cores.
//
// Follows PR 60321 "Add an mxfp4_mla KV cache for rope-free sparse MLA"
// (Read path: each query's top-k rows are gathered and unpacked to bf16 and
// feed both dots, q.k and p.v; Claims: attention over the packed cache equals
// attention over the dequantized bf16 values). For the rope-free latent the
// key and the value of a token are the same 512-wide row.
//
// Work decomposition. A unit of work is (query, half of the 512 value
// columns): the two units of a query both form the full scores q.k
// (512-deep) and each accumulates 256 output columns. A unit is a run of
// 32-key tiles. Without a workspace each unit is one CTA (query n's halves
// on CTAs 2n and 2n + 1), which writes its output. With one (the split-K of
// the read path, for few queries), every unit is cut into `chunks` runs of
// at most `chunk_tiles` tiles, one CTA each (unit u's chunks on CTAs
// u * chunks ..): the CTA writes a bf16 partial, the output of its chunk
// normalised by the chunk's own softmax sum and that sum's log-sum-exp,
// into the caller's workspace, and a second, small kernel combines each
// unit's partials by their log-sum-exps (launched as a programmatic
// dependent of the first, so its launch overlaps the first grid's tail). A
// CTA's work is one contiguous run of one unit either way.
//
// Start-up: one thread loads Q with eight tensor-map boxes (TMA) into the
// two swizzled operand layouts, while the producers issue their first row
// loads; the first half of Q is staged in the still empty key ring and
// moved to tensor memory by the softmax warps.
//
// Each CTA: tensor memory (512 columns x 128 lanes,
// lane = head) holds the output accumulator (256 columns), four 32-key score
// buffers (128; softmax writes the bf16 probabilities P back over the scores
// of the same buffer, and p.v takes P from there as its A operand) and the
// first 256 dims of Q as bf16 pairs (128): the q.k products over those dims
// take Q from tensor memory and read only the key tile from shared memory.
// The other 256 dims of Q stay in shared memory next to four 32 KB key tiles
// of 32 keys (a ring of four stages). Four roles run as a pipeline through
// mbarriers:
//   - producers (warps 4-19, two groups of 8: warps 4-11 take the even
//     tiles, 12-19 the odd ones, so that each warp has two tile periods
//     for a tile's work; a lane takes one key of the tile and one 64-dim
//     K-block, a warp 8 keys x 4 K-blocks):
//     load the packed rows one of its tiles ahead into registers (pads and
//     out-of-range indices load nothing and decode to zero rows),
//     dequantize them with byte permutes into a 128-byte-swizzled K-major
//     bf16 key tile, and arrive on its "full" barrier; a stage is reused once
//     the p.v that last read it has completed;
//   - the q.k issuer (warp 20, one thread): S = Q K^T over two tiles at once
//     (M 128, N 64, K 512: the ring is laid out K-block-major, so the same
//     K-block of two neighbouring stages is one 64-row operand) once both
//     are written; a stage's keys are rewritten only after the p.v of the
//     tile four back has completed, so the score columns it overwrites are
//     free;
//   - the p.v issuer (warp 21, one thread): O += P(u) V(u) (M 128, N 256,
//     K 32; V is the key tile read MN-major) as soon as softmax has written
//     P(u). Two issuers, so that a p.v never waits behind the 32 MMAs of a
//     q.k pair (one thread issuing both took ~1K cycles to react to P);
//     tcgen05.commit on mbarriers tracks completion;
//   - softmax (warps 0-3, one head per thread): read S(t), run the online
//     softmax in fp32 (exp2, running max with a rescale of the output only
//     when the max grows by more than 2**32), and store P (bf16 pairs) into
//     tensor memory; after the last tile, read O out of tensor memory and
//     write the result (the bf16 output, or a chunk's bf16 partial).
// Every wait is bounded; a timeout sets a CTA-wide abort flag that ends the
// other roles' waits, and the CTA reports through an optional status word.
// Before tensor memory is released, each issuing thread waits (bounded, abort
// or not) for every MMA it issued, so that none writes released tensor
// memory or arrives on a released barrier.
//
// Numerics: scores and the output accumulate in fp32 on the tensor core from
// exact bf16 inputs (the dequantized rows are exact); the probabilities are
// rounded to bf16 for the p.v product while the normaliser sums them
// unrounded; the output is rounded to bf16 once at the end.
#include <cuda.h>

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
// softmax warps 0-3, producers 4-19 (two groups), q.k issuer 20, p.v issuer 21
constexpr int kThreads = 704;
constexpr int kIssuerWarp = 20;
constexpr int kPvWarp = 21;
constexpr int kRow = 272;       // packed row bytes
// row loads a producer keeps in flight, in tiles of its group (every other
// tile): one covers two tile periods (two: 1.5% slower, three: spills)
constexpr int kDepth = 1;

constexpr uint32_t kQhiBytes = kHeads * 256 * 2;         // dims 256..511: 4 K-blocks x 128 rows
constexpr uint32_t kKBytes = kTileKeys * kDim * 2;       // 8 K-blocks x 32 rows x 128 B
constexpr uint32_t kKBlock = kTileKeys * 128;            // bytes of one K-block of a key tile
// The ring is laid out K-block-major: K-block kb of stage s at
// (kb * kStages + s) * kKBlock, so the same K-block of stages s and s + 1
// (s even) is one 64-row block and q.k runs at N = 64 over a pair of stages.
constexpr uint32_t kKBlockStride = kStages * kKBlock;
constexpr uint32_t kOffQ = 0;
// dims 0..255 of Q are staged in the ring before the first tile arrives
static_assert(kHeads * 256 * 2 <= kStages * kKBytes, "Q staging exceeds the key ring");
constexpr uint32_t kOffK = kOffQ + kQhiBytes;            // kStages buffers
constexpr uint32_t kOffBar = kOffK + kStages * kKBytes;  // eighteen mbarriers
constexpr uint32_t kOffTmemSlot = kOffBar + 160;
constexpr uint32_t kOffAbort = kOffTmemSlot + 16;
constexpr uint32_t kSmemUsed = kOffAbort + 16;
constexpr size_t kSmemBytes = kSmemUsed + 1024;  // room to align the base to 1024

// mbarriers, one of each per stage (the CTA's i-th tile uses stage i % kStages),
// then one per issuer that it commits its last MMAs to before tensor memory
// is released, and Q's
constexpr uint32_t kBarKFull = 0, kBarSFull = 32, kBarPFull = 64, kBarPvDone = 96;
constexpr uint32_t kBarDrain = 128;   // the q.k issuer's drain
constexpr uint32_t kBarQ = 136;       // Q's eight tensor-map boxes landed
constexpr uint32_t kBarDrain2 = 144;  // the p.v issuer's drain
static_assert(kBarDrain2 + 8 <= kOffTmemSlot - kOffBar, "mbarriers overlap the TMEM slot");

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 0;     // 256 columns
constexpr uint32_t kColS = 256;   // kStages buffers of 32 columns: scores, then P over them
constexpr uint32_t kColQ = 384;   // Q dims 0..255 as 128 columns of bf16 pairs

constexpr uint32_t kWaitPolls = 1u << 22;

// The softmax keeps a reference max per head and rescales the output only
// when a tile's max exceeds it by more than this (log2 units): until then
// the probabilities are taken against the stale reference, up to 2**32.
// Each rescale waits for the previous p.v and rewrites 256 columns of tensor
// memory, and on heavy-tailed latents (Student-t with outliers) a threshold
// of 8 rescaled a warp on a quarter of the tiles (this one: about one per
// CTA; 0.190 -> 0.164 ms on 128 queries x 2048 keys). The rounding is the
// same (bf16 P, fp32 sums) at any magnitude, and exp2 still flushes only
// probabilities below 2**-126 of the true max. The cost is headroom: the
// unnormalised fp32 sums stay finite while n keys x 2**32 x max|v| < 2**128,
// i.e. |v| < 2**85 for 2048 keys.
constexpr float kRescaleLog2 = 32.0f;

struct AttnParams {
  // Q as a [queries][num_heads][512] bf16 tensor map (boxes of 64 dims x 128
  // heads, 128-byte swizzle, heads past num_heads read as zeros), valid when
  // q_tma is set: Q in device memory and the map encoded. Otherwise Q is
  // copied in 16-byte pieces.
  CUtensorMap qmap;
  int q_tma;
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
  // Schedule: unit u = (query u / 2, value half u % 2) is `tiles` tiles of
  // 32 keys, cut into `chunks` runs of `chunk_tiles` tiles (the last may be
  // shorter), CTA b taking chunk b % chunks of unit b / chunks.
  int64_t tiles, units;
  int64_t nq;  // queries
  int64_t chunks, chunk_tiles;
  int64_t grid;  // units * chunks
  // Partial results (null when every unit is one chunk): CTA b's
  // [num_heads][256] bf16 output of its chunk normalised by the chunk's
  // softmax sum at part_o + b * num_heads * 512 bytes, and that sum's
  // log-sum-exp in log2 units (-inf for a chunk without valid keys) at
  // part_lse + b * num_heads.
  uint8_t* part_o;
  float* part_lse;
  // Ragged index runs (one chunk per unit only): query n's indices are
  // indices[key_offsets[n] .. key_offsets[n + 1]), each bound clamped to
  // [0, num_indices]; null for the fixed [num_queries, topk] layout.
  const int64_t* key_offsets;
  int64_t num_indices;
};

// ------------------------------------------------------------------ PTX ---

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ uint4 lds_v4_at(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(a)
               : "memory");
  return v;
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
// of packed rows must not be moved down to its first use a tile later. They
// allocate in L1: a lane's two 16-byte loads fall in one 32-byte sector, and
// the eight producer warps all read each row's scale sector (without L1 the
// CTA sent ~2.9x the rows' sectors to L2 and ran 10% slower).
__device__ __forceinline__ uint4 ld_issue_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
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

// arrive once and expect `bytes` from asynchronous copies in this phase
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

// one box of a 3-D tensor map into shared memory, completing on `bar`
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            int z, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
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

// 16 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
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
constexpr uint32_t kIdescQK1 = instr_desc(kHeads, kTileKeys, false);
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

// Slot index of key j of tile t of the CTA's run of indices
// [key_off, key_off + key_len) (its chunk of a row of the fixed layout, or a
// ragged run), or -1 past the run.
__device__ __forceinline__ int64_t key_index(const AttnParams& p, int64_t t, int j,
                                             int64_t key_off, int64_t key_len) {
  const int64_t k = t * kTileKeys + j;
  return k < key_len ? ld_once_i64(p.indices + key_off + k) : -1;
}

__device__ __forceinline__ uint32_t ld_issue_u16(const void* p) {
  uint16_t r;
  asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(r) : "l"(p));
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
// c = (d % 64) / 8. The eight lanes of a 16-byte store phase hold eight
// consecutive keys of one K-block, so they cover all eight bank groups.
// The range check of the two scale bytes is made once, so that the common
// case is one branch-free run of sixteen independent permute chains.
__device__ __forceinline__ void dequant_share(const Packed& x, uint32_t kbuf, int j, int e) {
  const uint32_t row = kbuf + (uint32_t)e * kKBlockStride + (uint32_t)j * 128;
  const uint32_t swz = (uint32_t)(j & 7);
  const uint32_t sb0 = x.s & 0xFFu, sb1 = (x.s >> 8) & 0xFFu;
  if (sb0 - 2u <= 250u && sb1 - 2u <= 250u) {
    const ByteTables t0 = make_tables(sb0), t1 = make_tables(sb1);
    const uint32_t words[8] = {x.c[0].x, x.c[0].y, x.c[0].z, x.c[0].w,
                               x.c[1].x, x.c[1].y, x.c[1].z, x.c[1].w};
#pragma unroll
    for (int c = 0; c < 8; ++c)  // chunk of 8 dims within the K-block
      sts_v4(row + (((uint32_t)c ^ swz) << 4), decode8_fast(words[c], c < 4 ? t0 : t1));
  } else {
    const uint32_t words[8] = {x.c[0].x, x.c[0].y, x.c[0].z, x.c[0].w,
                               x.c[1].x, x.c[1].y, x.c[1].z, x.c[1].w};
#pragma unroll 1
    for (int c = 0; c < 8; ++c) {
      const uint32_t sb = c < 4 ? sb0 : sb1;
      sts_v4(row + (((uint32_t)c ^ swz) << 4),
             sb - 2u <= 250u ? decode8_fast(words[c], make_tables(sb))
                             : decode8_slow(words[c], sb));
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

// S = Q K^T into the score columns of stage `st` (N = 32), or of the pair of
// stages st (even) and st + 1 (N = 64: the ring is K-block-major, so the
// same K-block of the two stages is one 64-row operand): dims 0..255 with Q
// from TMEM (16 steps of 8 columns), dims 256..511 with Q from shared memory.
template <bool kPair>
__device__ __forceinline__ void issue_qk(uint32_t st, uint64_t q_desc, uint32_t k_base,
                                         uint32_t tmem) {
  constexpr uint32_t idesc = kPair ? kIdescQK : kIdescQK1;
  const uint64_t k_desc = smem_desc(k_base + st * kKBlock, 16, 1024, 2);
  const uint32_t d = tmem + kColS + st * kTileKeys;
#pragma unroll
  for (int kb = 0; kb < 4; ++kb) {
#pragma unroll
    for (int ks = 0; ks < 4; ++ks)
      mma_bf16_ta(d, tmem + kColQ + (uint32_t)(8 * (4 * kb + ks)),
                  desc_at(k_desc, kb * kKBlockStride + ks * 32), idesc, (kb | ks) != 0);
  }
#pragma unroll
  for (int kb = 4; kb < 8; ++kb) {
#pragma unroll
    for (int ks = 0; ks < 4; ++ks)
      mma_bf16(d, desc_at(q_desc, (kb - 4) * (kHeads * 128) + ks * 32),
               desc_at(k_desc, kb * kKBlockStride + ks * 32), idesc, 1);
  }
}

// O (+)= P V of the tile in stage `st`: P (bf16 pairs, written by softmax
// over the stage's score columns) is the TMEM A operand, 8 columns per step
// of 16 keys; V is the stage's key rows read MN-major from column block 4v
// (LBO: the stage's next K-block, SBO: next 8 keys). `first` starts a new
// accumulation (the CTA's first tile).
__device__ __forceinline__ void issue_pv(uint32_t st, int v, bool first, uint32_t k_base,
                                         uint32_t tmem) {
  const uint64_t v_desc = smem_desc(k_base + ((uint32_t)v * 4 * kStages + st) * kKBlock,
                                    kKBlockStride, 1024, 2);
  const uint32_t pa = tmem + kColS + st * kTileKeys;
#pragma unroll
  for (int ks = 0; ks < kTileKeys / 16; ++ks)
    mma_bf16_ta(tmem + kColO, pa + 8 * ks, desc_at(v_desc, ks * 2048), kIdescPV,
                !(first && ks == 0));
}

// ---------------------------------------------------------------- kernel ---

// Q of query n into the operand buffers, once per CTA. Both halves take
// the layout of the A operand of q.k, 128-byte-swizzled K-major: 64-dim
// K-block kb of head r at base + kb * 16384 + r * 128, 16-byte chunk c of
// that row at ((c ^ (r & 7)) << 4); dims 256..511 at q_base (read by the
// MMAs), dims 0..255 staged at `stage` in the still empty key ring and
// moved to tensor memory by the softmax threads (below). Eight tensor-map
// boxes issued by one thread when Q is in device memory (they do not queue
// behind the SM's outstanding-miss limit, as 8,192 separate 16-byte copies
// do); otherwise load_q_smem: the same bytes by threads [0, nthreads), 16
// bytes per cp.async, zero rows past num_heads. Neither is inlined: they run
// once, and kept out of line they leave the roles' loops their registers.
__device__ __noinline__ void load_q_boxes(const AttnParams& p, int64_t n, uint32_t q_base,
                                          uint32_t stage, uint32_t bar) {
  mbar_expect_tx(bar, 8 * kHeads * 128);
#pragma unroll 1
  for (int kb = 0; kb < 8; ++kb)
    tma_load_3d((kb < 4 ? stage : q_base) + (uint32_t)(kb & 3) * (kHeads * 128), &p.qmap, 64 * kb,
                0, (int)n, bar);
}

__device__ __noinline__ void load_q_smem(const AttnParams& p, int64_t n, uint32_t q_base,
                                         uint32_t stage, int tid, int nthreads) {
  const uint8_t* qn = p.q + n * p.q_qstride;
  for (int id = tid; id < kHeads * 64; id += nthreads) {
    const int r = (id >> 5) & (kHeads - 1), c32 = id & 31;
    const bool hi = id >= kHeads * 32;
    const uint32_t dst = (hi ? q_base : stage) + (uint32_t)(c32 >> 3) * (kHeads * 128) +
                         (uint32_t)r * 128 + ((((uint32_t)c32 & 7) ^ ((uint32_t)r & 7)) << 4);
    if (r < p.num_heads)
      cp_async_16a(dst, qn + r * p.q_hstride + (hi ? 512 : 0) + c32 * 16);
    else
      sts_v4(dst, make_uint4(0, 0, 0, 0));
  }
  cp_async_commit();
  cp_async_wait<0>();
  fence_proxy_async();
}

// By the 128 softmax threads (warps 0-3, head = thread): the staged dims
// 0..255 into TMEM lane `head`, columns kColQ.. as bf16 pairs (the A operand
// of the first 16 q.k steps). The eight lanes of a 16-byte load phase read
// eight rows at eight different chunk positions: no bank conflicts.
__device__ __noinline__ void load_q_tmem(uint32_t stage, uint32_t tmem, int tid) {
  const uint32_t lane_base = tmem + ((uint32_t)((tid >> 5) * 32) << 16);
  const uint32_t row = stage + (uint32_t)tid * 128, swz = (uint32_t)(tid & 7);
#pragma unroll 1
  for (int c = 0; c < 4; ++c) {
    uint32_t w[32];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const uint4 x = lds_v4_at(row + (uint32_t)c * (kHeads * 128) + (((uint32_t)k ^ swz) << 4));
      w[4 * k] = x.x;
      w[4 * k + 1] = x.y;
      w[4 * k + 2] = x.z;
      w[4 * k + 3] = x.w;
    }
    tmem_st32(lane_base + kColQ + 32 * c, w);
  }
}

// Bounded wait for the completion of every MMA issued so far by the calling
// thread (commit to the drain barrier, then poll it): runs whether or not
// the CTA is aborting, so that no MMA still writes tensor memory or arrives
// on an mbarrier once the CTA releases them.
__device__ __forceinline__ bool drain_mmas(uint32_t bar) {
  mma_commit(bar);
  for (uint32_t i = 0; i < kWaitPolls; ++i)
    if (mbar_test(bar, 0)) return true;
  return false;
}

// One head's result (thread = head, O in TMEM lanes of this warp): the bf16
// output row half or, for a chunk of a split unit (kPiece), the bf16 output
// normalised by the chunk's softmax sum (a partial) and that sum's
// log-sum-exp (log2 units) in CTA b's partial slot. O is read out 16
// columns at a time, which keeps the softmax loop's live state in registers
// around it, and goes straight to memory (32 bytes per read).
template <bool kPiece>
__device__ __forceinline__ void write_result(const AttnParams& p, int64_t n, int v, int64_t b,
                                             uint32_t lane_base, int h, float m_ref, float l) {
  const float inv = l > 0.0f ? 1.0f / l : 0.0f;
  const bool store = h < p.num_heads;
  uint8_t* orow = kPiece ? p.part_o + (b * p.num_heads + h) * (kHalf * 2)
                         : p.out + n * p.o_qstride + (int64_t)h * p.o_hstride +
                               (int64_t)v * kHalf * 2;
#pragma unroll 1
  for (int c = 0; c < kHalf / 16; ++c) {
    uint32_t o[16];
    tmem_ld16(lane_base + kColO + 16 * c, o);
    uint32_t w[8];
#pragma unroll
    for (int k = 0; k < 8; ++k)
      w[k] = l > 0.0f ? pack_bf16x2(__uint_as_float(o[2 * k]) * inv,
                                    __uint_as_float(o[2 * k + 1]) * inv)
                      : 0u;
    if (store) {
#pragma unroll
      for (int u = 0; u < 2; ++u)
        st_v4(orow + 32 * c + 16 * u, make_uint4(w[4 * u], w[4 * u + 1], w[4 * u + 2],
                                                  w[4 * u + 3]));
    }
  }
  if (!store) return;
  const float lse2 = l > 0.0f ? m_ref + log2f(l) : -__int_as_float(0x7F800000);
  if (kPiece)
    p.part_lse[b * p.num_heads + h] = lse2;
  else if (v == 0 && p.lse)
    p.lse[n * p.num_heads + h] = l > 0.0f ? lse2 * 0.69314718055994531f : lse2;
}

// kPiece: a chunk of a split unit, written as a bf16 partial; otherwise a
// whole unit, written as the bf16 output (the same kernel otherwise).
template <bool kPiece>
__global__ void __launch_bounds__(kThreads, 1)
    mxfp4_attention_kernel(const __grid_constant__ AttnParams p) {
  extern __shared__ uint8_t smem_raw[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t b = blockIdx.x;
  // the merge (launched as this grid's programmatic dependent) may be
  // scheduled once every CTA of this grid has started; it waits for the
  // whole grid before it reads a partial
  if constexpr (kPiece) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // this CTA's unit (query n, value half v) and run of indices: chunk
  // b % chunks of a row of the fixed layout, or the query's ragged run. The
  // grid and the chunk count fit 32 bits (a 64-bit division here, a runtime
  // call, cost the whole kernel 10% in registers and time).
  const uint32_t chunks32 = (uint32_t)p.chunks;
  const uint32_t unit32 = (uint32_t)blockIdx.x / chunks32;
  const int64_t chunk = (int64_t)((uint32_t)blockIdx.x - unit32 * chunks32);
  const int64_t n = unit32 >> 1;
  const int v = (int)(unit32 & 1u);
  int64_t key_off, key_len;
  if (p.key_offsets) {
    int64_t lo = ld_once_i64(p.key_offsets + n), hi = ld_once_i64(p.key_offsets + n + 1);
    lo = lo < 0 ? 0 : (lo > p.num_indices ? p.num_indices : lo);
    hi = hi < lo ? lo : (hi > p.num_indices ? p.num_indices : hi);
    key_off = lo;
    key_len = hi - lo;
  } else {
    const int64_t first = chunk * p.chunk_tiles * kTileKeys;
    const int64_t rest = p.topk - first;
    const int64_t span = p.chunk_tiles * kTileKeys;
    key_off = n * p.topk + first;
    key_len = rest < 0 ? 0 : (rest < span ? rest : span);
  }
  const int64_t n_tiles = (key_len + kTileKeys - 1) / kTileKeys;
  if (n_tiles == 0) {
    // no keys at all: every output row is zero and every log-sum-exp -inf
    // (an empty partial for a chunk)
    if constexpr (kPiece) {
      for (int id = tid; id < p.num_heads * 32; id += kThreads)
        st_v4(p.part_o + (b * p.num_heads + (id >> 5)) * (kHalf * 2) + (id & 31) * 16,
              make_uint4(0, 0, 0, 0));
      for (int h = tid; h < p.num_heads; h += kThreads)
        p.part_lse[b * p.num_heads + h] = -__int_as_float(0x7F800000);
      return;
    } else {
      for (int id = tid; id < p.num_heads * 32; id += kThreads)
        st_v4(p.out + n * p.o_qstride + (int64_t)(id >> 5) * p.o_hstride + v * kHalf * 2 +
                  (id & 31) * 16,
              make_uint4(0, 0, 0, 0));
      if (v == 0 && p.lse)
        for (int h = tid; h < p.num_heads; h += kThreads)
          p.lse[n * p.num_heads + h] = -__int_as_float(0x7F800000);
      return;
    }
  }
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* sm = smem_raw + (base - raw);
  const uint32_t q_base = base + kOffQ, k_base = base + kOffK;
  const uint32_t bars = base + kOffBar;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + kOffTmemSlot);
  volatile int* abort = reinterpret_cast<volatile int*>(sm + kOffAbort);

  if (warp == kIssuerWarp) tmem_alloc(smem_addr(tmem_slot), kTmemCols);
  if (tid == 0) {
#pragma unroll
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bars + kBarKFull + 8 * s, 256);
      mbar_init(bars + kBarSFull + 8 * s, 1);
      mbar_init(bars + kBarPFull + 8 * s, 128);
      mbar_init(bars + kBarPvDone + 8 * s, 1);
    }
    mbar_init(bars + kBarDrain, 1);
    mbar_init(bars + kBarQ, 1);
    mbar_init(bars + kBarDrain2, 1);
    *abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    if (p.q_tma) load_q_boxes(p, n, q_base, k_base, bars + kBarQ);
  }
  // The producers issue their first kDepth tiles of row loads at once while
  // Q is on its way (the tensor-map boxes issued above, or, for a
  // host-mapped Q, the copies of the softmax and q.k issuer warps' 160
  // threads):
  // the two start-up latencies overlap.
  const bool producer = warp >= 4 && warp < kIssuerWarp;
  // producer lane: key j of the tile, dims [64e, 64e + 64); warp 4 + 8 g + w
  // (group g: tiles of parity g) takes keys 8 (w % 4) .. + 7 and K-blocks
  // 4 (w / 4) .. + 3, so that a 16-byte load instruction touches 8 rows
  // (not 32) and a store phase 8 keys
  const int grp = ((warp - 4) >> 3) & 1, pw = (warp - 4) & 7;
  const int e = 4 * (pw >> 2) + (lane >> 3), j = 8 * (pw & 3) + (lane & 7);
  Packed buf[kDepth];
  int64_t s_next = -1;
  if (producer) {
#pragma unroll
    for (int u = 0; u < kDepth; ++u) {
      const int64_t t = grp + 2 * u;  // the group's u-th tile
      buf[u] = load_packed(p, t < n_tiles ? key_index(p, t, j, key_off, key_len) : -1, e);
    }
    const int64_t t = grp + 2 * kDepth;
    s_next = t < n_tiles ? key_index(p, t, j, key_off, key_len) : -1;
  } else if (!p.q_tma) {
    // dims 0..255 staged in the key ring, which the producers fill only
    // after the second barrier below
    load_q_smem(p, n, q_base, k_base, tid < 128 ? tid : tid - 512, 160);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (warp < 4 && (!p.q_tma || warp_wait(bars + kBarQ, 0, abort))) load_q_tmem(k_base, tmem, tid);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  if (producer) {
    // ------------------------------------------------------------ producers
    // Lane = key j of the tile, dims [64e, 64e + 64); group grp takes
    // tiles grp, grp + 2, ... The CTA's i-th tile goes to stage
    // i % kStages, free once the p.v of tile i - kStages has completed; rows
    // are loaded kDepth of the group's tiles ahead.
    bool live = true;
    for (int64_t i0 = grp; i0 < n_tiles && live; i0 += 2 * kDepth) {
#pragma unroll
      for (int u = 0; u < kDepth; ++u) {
        const int64_t i = i0 + 2 * u;
        if (i < n_tiles && live) {
          const Packed cur = buf[u];
          buf[u] = load_packed(p, s_next, e);  // tile i + 2 kDepth
          const int64_t t = i + 2 * kDepth + 2;
          s_next = t < n_tiles ? key_index(p, t, j, key_off, key_len) : -1;
          const uint32_t st = (uint32_t)(i % kStages);
          if (i >= kStages &&
              !mbar_wait(bars + kBarPvDone + 8 * st, (uint32_t)(((i / kStages) - 1) & 1), abort)) {
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
    // ------------------------------------------------------- q.k issuer
    // S = Q K^T of tile qi (with tile qi + 1 when qi's stage is even) once
    // its keys are written. A stage's keys are rewritten only after the p.v
    // of the tile four back has completed, so its score columns are free.
    if (lane == 0 && (!p.q_tma || mbar_wait(bars + kBarQ, 0, abort))) {
      const uint64_t q_desc = smem_desc(q_base, 16, 1024, 2);
      for (int64_t qi = 0; qi < n_tiles;) {
        const uint32_t st = (uint32_t)(qi % kStages);
        const bool pair = (st & 1u) == 0 && qi + 1 < n_tiles;
        if (!mbar_wait(bars + kBarKFull + 8 * st, (uint32_t)((qi / kStages) & 1), abort)) break;
        if (pair && !mbar_wait(bars + kBarKFull + 8 * (st + 1),
                               (uint32_t)(((qi + 1) / kStages) & 1), abort))
          break;
        tc_fence_after();
        if (pair) {
          issue_qk<true>(st, q_desc, k_base, tmem);
          mma_commit(bars + kBarSFull + 8 * st);
          mma_commit(bars + kBarSFull + 8 * (st + 1));
          qi += 2;
        } else {
          issue_qk<false>(st, q_desc, k_base, tmem);
          mma_commit(bars + kBarSFull + 8 * st);
          qi += 1;
        }
      }
      if (!drain_mmas(bars + kBarDrain)) *abort = 1;
    }
    __syncwarp();
  } else if (warp == kPvWarp) {
    // ------------------------------------------------------- p.v issuer
    // O += P(pi) V(pi) as soon as softmax has written P(pi).
    if (lane == 0) {
      for (int64_t pi = 0; pi < n_tiles; ++pi) {
        const uint32_t st = (uint32_t)(pi % kStages);
        if (!mbar_wait(bars + kBarPFull + 8 * st, (uint32_t)((pi / kStages) & 1), abort)) break;
        tc_fence_after();
        issue_pv(st, v, pi == 0, k_base, tmem);
        mma_commit(bars + kBarPvDone + 8 * st);
      }
      if (!drain_mmas(bars + kBarDrain2)) *abort = 1;
    }
    __syncwarp();
  } else {
    // -------------------------------------------------------------- softmax
    const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
    const float kNegInf = -__int_as_float(0x7F800000);
    float m_ref = kNegInf;  // reference max (log2 units)
    float l = 0.0f;         // sum of p against m_ref
    int64_t s_key = key_index(p, 0, lane, key_off, key_len);
    for (int64_t i = 0; i < n_tiles; ++i) {
      const uint32_t mask = __ballot_sync(0xFFFFFFFFu, s_key >= 0 && s_key < p.num_slots);
      s_key = i + 1 < n_tiles ? key_index(p, i + 1, lane, key_off, key_len) : -1;
      const uint32_t st = (uint32_t)(i % kStages);
      if (!warp_wait(bars + kBarSFull + 8 * st, (uint32_t)((i / kStages) & 1), abort)) break;
      tc_fence_after();
      const uint32_t scol = lane_base + kColS + st * kTileKeys;
      uint32_t sr[32];
      tmem_ld32(scol, sr);
      // the tile max (log2 units, -inf for dropped keys), four chains
      float mc[4] = {kNegInf, kNegInf, kNegInf, kNegInf};
#pragma unroll
      for (int k = 0; k < 32; ++k)
        if ((mask >> k) & 1u)
          mc[k & 3] = fmaxf(mc[k & 3], __fmul_rn(__uint_as_float(sr[k]), p.scale_log2));
      const float mt = fmaxf(fmaxf(mc[0], mc[1]), fmaxf(mc[2], mc[3]));
      const bool need = mt > m_ref + kRescaleLog2;
      if (__any_sync(0xFFFFFFFFu, need)) {
        const float f = need ? ex2(m_ref - mt) : 1.0f;  // ex2(-inf) = 0
        if (i > 0) {
          // O may be touched only once the p.v of tile i - 1 has completed
          const int64_t w = i - 1;
          if (!warp_wait(bars + kBarPvDone + 8 * (uint32_t)(w % kStages),
                         (uint32_t)((w / kStages) & 1), abort))
            break;
          tc_fence_after();
#pragma unroll 1
          for (int cc = 0; cc < kHalf / 32; ++cc) {
            uint32_t o[32];
            tmem_ld32(lane_base + kColO + 32 * cc, o);
#pragma unroll
            for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * f);
            tmem_st32(lane_base + kColO + 32 * cc, o);
          }
        }
        l *= f;
        if (need) m_ref = mt;
      }
      const float mu = m_ref == kNegInf ? 0.0f : m_ref;
      // probabilities, their sum, and P (bf16 pairs) over the score columns
      float lsum0 = 0.0f, lsum1 = 0.0f;
      uint32_t pk[16];
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        const float x0 = ((mask >> (2 * k)) & 1u)
                             ? __fmul_rn(__uint_as_float(sr[2 * k]), p.scale_log2)
                             : kNegInf;
        const float x1 = ((mask >> (2 * k + 1)) & 1u)
                             ? __fmul_rn(__uint_as_float(sr[2 * k + 1]), p.scale_log2)
                             : kNegInf;
        const float p0 = ex2(x0 - mu), p1 = ex2(x1 - mu);
        lsum0 += p0;
        lsum1 += p1;
        pk[k] = pack_bf16x2(p0, p1);
      }
      tmem_st16(scol, pk);
      l += lsum0 + lsum1;
      tc_fence_before();
      mbar_arrive(bars + kBarPFull + 8 * st);
      if (i == n_tiles - 1) {
        // the result: wait for the last p.v, then read O out
        if (!warp_wait(bars + kBarPvDone + 8 * st, (uint32_t)((i / kStages) & 1), abort)) break;
        tc_fence_after();
        write_result<kPiece>(p, n, v, b, lane_base, tid, m_ref, l);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (tid == 0 && p.q_tma) {
    // the Q boxes have landed unless a wait for them timed out: then wait
    // (bounded) for them before the CTA's shared memory is released
    for (uint32_t i = 0; i < kWaitPolls && !mbar_test(bars + kBarQ, 0); ++i) {
    }
  }
  if (tid == 0 && *abort && p.status) atomicExch(p.status, 1);
  if (warp == kIssuerWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// Combines the partials of every split unit. Block (u, g) takes unit u and
// heads 8g..8g+7, over the partials of CTAs u * chunks .. u * chunks +
// chunks - 1: out = sum_b 2**(lse_b - L) o_b / sum_b 2**(lse_b - L),
// L = max_b lse_b, and the unit's log-sum-exp L + log2(sum) (in natural log
// units, half 0 only). A unit without any valid key gets zeros and -inf.
// 64 threads take a head, four columns each. Up to kMergeFew partials are
// summed by each thread on its own; beyond that (the launch then gives the
// block dynamic shared memory for kMergeHeads x chunks weights), every
// (head, partial) weight is first worked out in parallel, and the sums keep
// several loads in flight.
constexpr int kMergeHeads = 8;  // heads per block (64 threads each)

// Four consecutive bf16 columns of a partial as fp32.
__device__ __forceinline__ float4 partial4(const uint8_t* at) {
  const uint2 x = *reinterpret_cast<const uint2*>(at);
  return make_float4(__uint_as_float(x.x << 16), __uint_as_float(x.x & 0xFFFF0000u),
                     __uint_as_float(x.y << 16), __uint_as_float(x.y & 0xFFFF0000u));
}
constexpr int kMergeFew = 4;

__global__ void __launch_bounds__(64 * kMergeHeads, 4) mxfp4_attention_merge_kernel(AttnParams p) {
  __shared__ float head_l[kMergeHeads][2], head_w[kMergeHeads][2];
  extern __shared__ float merge_dyn[];  // [kMergeHeads][chunks]: log-sum-exp, then weight
  // launched as the split grid's programmatic dependent: the block may be
  // resident while that grid still runs, and waits here for all of it (and
  // its memory) to complete; a no-op for an ordinary launch
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int64_t unit = blockIdx.x;
  const int pieces = (int)p.chunks;
  const int64_t b0 = unit * p.chunks;  // the unit's first CTA
  const int64_t H = p.num_heads;
  const float kNegInf = -__int_as_float(0x7F800000);
  const int64_t n = unit >> 1;
  const int v = (int)(unit & 1);
  uint32_t dyn_bytes;
  asm("mov.u32 %0, %%dynamic_smem_size;" : "=r"(dyn_bytes));
  if (pieces <= kMergeFew || dyn_bytes < (uint32_t)(kMergeHeads * pieces) * 4u) {
    const int64_t h = (int64_t)blockIdx.y * kMergeHeads + (threadIdx.x >> 6);
    if (h >= H) return;
    const int c4 = threadIdx.x & 63;
    float L = kNegInf;
#pragma unroll 4
    for (int k = 0; k < pieces; ++k) L = fmaxf(L, p.part_lse[(b0 + k) * H + h]);
    float W = 0.0f;
    float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    if (L != kNegInf) {
#pragma unroll 4
      for (int k = 0; k < pieces; ++k) {
        const int64_t row = (b0 + k) * H + h;
        const float w = exp2f(p.part_lse[row] - L);
        const float4 o = partial4(p.part_o + row * (kHalf * 2) + 8 * c4);
        W += w;
        acc.x += w * o.x;
        acc.y += w * o.y;
        acc.z += w * o.z;
        acc.w += w * o.w;
      }
    }
    const float inv = W > 0.0f ? 1.0f / W : 0.0f;
    st_v2(p.out + n * p.o_qstride + h * p.o_hstride + (int64_t)(v * kHalf + 4 * c4) * 2,
          pack_bf16x2(acc.x * inv, acc.y * inv), pack_bf16x2(acc.z * inv, acc.w * inv));
    if (v == 0 && p.lse && c4 == 0)
      p.lse[n * H + h] = W > 0.0f ? (L + log2f(W)) * 0.69314718055994531f : kNegInf;
    return;
  }
  for (int t = threadIdx.x; t < kMergeHeads * pieces; t += blockDim.x) {
    const int hh = t / pieces, k = t - hh * pieces;
    const int64_t h = (int64_t)blockIdx.y * kMergeHeads + hh;
    merge_dyn[hh * pieces + k] = h < H ? p.part_lse[(b0 + k) * H + h] : kNegInf;
  }
  __syncthreads();
  const int hh = threadIdx.x >> 6, c4 = threadIdx.x & 63, half = c4 >> 5;
  // L: the head's largest log-sum-exp (64 threads, two warps)
  float L = kNegInf;
  for (int k = c4; k < pieces; k += 64) L = fmaxf(L, merge_dyn[hh * pieces + k]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) L = fmaxf(L, __shfl_xor_sync(0xFFFFFFFFu, L, o));
  if ((c4 & 31) == 0) head_l[hh][half] = L;
  __syncthreads();
  L = fmaxf(head_l[hh][0], head_l[hh][1]);
  // weights 2**(lse_b - L) (0 for a partial without valid keys) and their sum
  float W = 0.0f;
  for (int k = c4; k < pieces; k += 64) {
    const float w = L != kNegInf ? exp2f(merge_dyn[hh * pieces + k] - L) : 0.0f;
    merge_dyn[hh * pieces + k] = w;
    W += w;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) W += __shfl_xor_sync(0xFFFFFFFFu, W, o);
  if ((c4 & 31) == 0) head_w[hh][half] = W;
  __syncthreads();
  W = head_w[hh][0] + head_w[hh][1];
  const int64_t h = (int64_t)blockIdx.y * kMergeHeads + hh;
  if (h >= H) return;
  float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
  if (W > 0.0f) {
#pragma unroll 8
    for (int k = 0; k < pieces; ++k) {
      const float w = merge_dyn[hh * pieces + k];
      const float4 o = partial4(p.part_o + ((b0 + k) * H + h) * (kHalf * 2) + 8 * c4);
      acc.x += w * o.x;
      acc.y += w * o.y;
      acc.z += w * o.z;
      acc.w += w * o.w;
    }
  }
  const float inv = W > 0.0f ? 1.0f / W : 0.0f;
  st_v2(p.out + n * p.o_qstride + h * p.o_hstride + (int64_t)(v * kHalf + 4 * c4) * 2,
        pack_bf16x2(acc.x * inv, acc.y * inv), pack_bf16x2(acc.z * inv, acc.w * inv));
  if (v == 0 && p.lse && c4 == 0)
    p.lse[n * H + h] = W > 0.0f ? (L + log2f(W)) * 0.69314718055994531f : kNegInf;
}

}  // namespace
}  // namespace kvq

namespace {

// Chunks per unit of the split schedule: as many as fill the SMs with one
// CTA each (every CTA holds all of tensor memory), of at least
// kMinSplitTiles tiles (a CTA's start-up, its partial's write and the merge
// cost a few tiles' time), and none empty; 1 means no split.
constexpr int64_t kMinSplitTiles = 4;
int64_t split_chunks(int64_t units, int64_t tiles) {
  if (units <= 0 || tiles <= 0) return 1;
  int64_t c = kvq::sm_count() / units;
  if (c > tiles / kMinSplitTiles) c = tiles / kMinSplitTiles;
  if (c < 2) return 1;
  const int64_t per = (tiles + c - 1) / c;
  return (tiles + per - 1) / per;
}

// Checks shared by the entry points; fills `p` (without workspace).
int attention_params(const void* q_bf16, int64_t num_queries, int64_t num_heads,
                     int64_t q_query_stride, int64_t q_head_stride, const uint8_t* cache,
                     int64_t num_blocks, int64_t block_size, int64_t block_stride_rows,
                     const int64_t* indices, int64_t topk, float sm_scale, void* out_bf16,
                     int64_t out_query_stride, int64_t out_head_stride, float* lse,
                     int32_t* status, kvq::AttnParams& p) {
  using namespace kvq;
  if (num_queries < 0 || num_heads < 1 || num_heads > kHeads || topk < 0) return KVQ_EINVAL;
  if (num_blocks < 1 || block_size < 1 || block_stride_rows < block_size) return KVQ_EINVAL;
  if (num_blocks > INT64_MAX / block_size) return KVQ_EINVAL;
  if (num_blocks > INT64_MAX / block_stride_rows / kRow) return KVQ_EINVAL;
  if (!(sm_scale == sm_scale) || sm_scale < 0.0f || sm_scale > 3.0e38f) return KVQ_EINVAL;
  if (q_head_stride < kDim || q_head_stride % 8 || q_query_stride % 8) return KVQ_EINVAL;
  if (out_head_stride < kDim || out_head_stride % 8 || out_query_stride % 8) return KVQ_EINVAL;
  if (num_queries > INT64_MAX / 2 / (topk > 0 ? topk : 1)) return KVQ_EINVAL;
  if (num_queries > 0x7FFFFFFF / 2) return KVQ_EINVAL;
  const int64_t tiles = (topk + kTileKeys - 1) / kTileKeys;
  // the schedule's products total * (grid + 1) stay in range
  if (tiles > 0 && 2 * num_queries > INT64_MAX / 1024 / tiles) return KVQ_EINVAL;
  if (num_queries == 0) return KVQ_OK;
  if (!q_bf16 || !cache || !out_bf16 || (topk > 0 && !indices)) return KVQ_EINVAL;
  if (!aligned(q_bf16, 16) || !aligned(cache, 16) || !aligned(out_bf16, 16) ||
      !aligned(indices, 8) || (lse && !aligned(lse, 4)) || (status && !aligned(status, 4)))
    return KVQ_EINVAL;
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
  p.tiles = tiles;
  p.units = 2 * num_queries;
  p.nq = num_queries;
  p.chunks = 1;  // one CTA per unit unless split
  p.chunk_tiles = tiles;
  p.grid = p.units;
  p.part_o = nullptr;
  p.part_lse = nullptr;
  p.key_offsets = nullptr;
  p.num_indices = 0;
  return KVQ_OK;
}

// Bytes of the split schedule's partial results: one per CTA.
int64_t split_bytes(int64_t grid, int64_t num_heads) {
  return grid * num_heads * (int64_t)(kvq::kHalf * 2 + 4);
}

// Cuts every unit into `chunks` runs and lays the partial results out in
// `ws` (256-byte aligned).
void split_layout(kvq::AttnParams& p, int64_t chunks, void* ws) {
  p.chunks = chunks;
  p.chunk_tiles = (p.tiles + chunks - 1) / chunks;
  p.grid = p.units * chunks;
  p.part_o = static_cast<uint8_t*>(ws);
  p.part_lse = reinterpret_cast<float*>(p.part_o + p.grid * p.num_heads * kvq::kHalf * 2);
}

// cuTensorMapEncodeTiled through the runtime (no link to the driver
// library), looked up once; null when the driver does not provide it.
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled() {
  static const EncodeTiledFn fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult found;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &found) != cudaSuccess ||
        found != cudaDriverEntryPointSuccess) {
      cudaGetLastError();
      f = nullptr;
    }
    return reinterpret_cast<EncodeTiledFn>(f);
  }();
  return fn;
}

// Q's tensor map: [queries][num_heads][512] bf16 with the caller's strides,
// boxes of 64 dims x 128 heads x 1 query, 128-byte swizzle, out-of-range
// heads read as zeros. Only for Q in device memory (a host-mapped Q keeps
// the 16-byte copies); false when the map cannot be made.
bool encode_q_map(kvq::AttnParams& p) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p.q) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  const EncodeTiledFn fn = encode_tiled();
  if (a.type != cudaMemoryTypeDevice || !fn) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)kvq::kDim, (cuuint64_t)p.num_heads, (cuuint64_t)p.nq};
  const cuuint64_t strides[2] = {(cuuint64_t)p.q_hstride, (cuuint64_t)p.q_qstride};
  const cuuint32_t box[3] = {64, (cuuint32_t)kvq::kHeads, 1};
  const cuuint32_t unit[3] = {1, 1, 1};
  return fn(&p.qmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
            const_cast<void*>(static_cast<const void*>(p.q)), dims, strides, box, unit,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int launch_attention(const kvq::AttnParams& params, cudaStream_t stream) {
  using namespace kvq;
  AttnParams p = params;
  p.q_tma = encode_q_map(p) ? 1 : 0;
  static int attr_done[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return KVQ_ECUDA;
  if (!attr_done[dev]) {
    if (cudaFuncSetAttribute(mxfp4_attention_kernel<true>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kSmemBytes) != cudaSuccess ||
        cudaFuncSetAttribute(mxfp4_attention_kernel<false>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kSmemBytes) != cudaSuccess)
      return KVQ_ECUDA;
    attr_done[dev] = 1;
  }
  if (p.part_o)
    mxfp4_attention_kernel<true><<<(unsigned)p.grid, kThreads, kSmemBytes, stream>>>(p);
  else
    mxfp4_attention_kernel<false><<<(unsigned)p.grid, kThreads, kSmemBytes, stream>>>(p);
  int rc = launch_status();
  if (rc != KVQ_OK || !p.part_o) return rc;
  const dim3 mgrid((unsigned)p.units, (unsigned)((p.num_heads + kMergeHeads - 1) / kMergeHeads));
  const size_t dyn = p.chunks > kMergeFew ? (size_t)kMergeHeads * (size_t)p.chunks * 4 : 0;
  // a programmatic dependent launch: the merge's launch latency overlaps the
  // attention grid's tail (every attention CTA is resident from the start: a
  // split grid has at most one CTA per SM)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = mgrid;
  cfg.blockDim = dim3(64 * kMergeHeads);
  cfg.dynamicSmemBytes = dyn;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, mxfp4_attention_merge_kernel, p) != cudaSuccess) {
    cudaGetLastError();
    return KVQ_ECUDA;
  }
  return launch_status();
}

}  // namespace

extern "C" int mxfp4_mla_sparse_attention_ragged(
    const void* q_bf16, int64_t num_queries, int64_t num_heads, int64_t q_query_stride,
    int64_t q_head_stride, const uint8_t* cache, int64_t num_blocks, int64_t block_size,
    int64_t block_stride_rows, const int64_t* indices, int64_t num_indices,
    const int64_t* key_offsets, float sm_scale, void* out_bf16, int64_t out_query_stride,
    int64_t out_head_stride, float* lse, int32_t* status, cudaStream_t stream) {
  using namespace kvq;
  if (num_indices < 0) return KVQ_EINVAL;
  AttnParams p;
  int rc = attention_params(q_bf16, num_queries, num_heads, q_query_stride, q_head_stride, cache,
                            num_blocks, block_size, block_stride_rows, indices, 0, sm_scale,
                            out_bf16, out_query_stride, out_head_stride, lse, status, p);
  if (rc != KVQ_OK || num_queries == 0) return rc;
  if (!key_offsets || !aligned(key_offsets, 8) || (num_indices > 0 && !indices)) return KVQ_EINVAL;
  p.key_offsets = key_offsets;
  p.num_indices = num_indices;
  return launch_attention(p, stream);  // one CTA per (query, value half), tiles from its run
}

extern "C" int64_t mxfp4_mla_sparse_attention_workspace_size(int64_t num_queries,
                                                             int64_t num_heads, int64_t topk) {
  if (num_queries < 0 || num_heads < 1 || num_heads > kvq::kHeads || topk < 0) return KVQ_EINVAL;
  if (num_queries > 0x7FFFFFFF / 2 || num_queries > INT64_MAX / 2 / (topk > 0 ? topk : 1))
    return KVQ_EINVAL;
  const int64_t tiles = (topk + kvq::kTileKeys - 1) / kvq::kTileKeys;
  if (tiles > 0 && 2 * num_queries > INT64_MAX / 1024 / tiles) return KVQ_EINVAL;
  if (tiles == 0 || num_queries == 0) return 0;
  const int64_t chunks = split_chunks(2 * num_queries, tiles);
  return chunks > 1 ? split_bytes(2 * num_queries * chunks, num_heads) : 0;
}

extern "C" int mxfp4_mla_sparse_attention(const void* q_bf16, int64_t num_queries,
                                          int64_t num_heads, int64_t q_query_stride,
                                          int64_t q_head_stride, const uint8_t* cache,
                                          int64_t num_blocks, int64_t block_size,
                                          int64_t block_stride_rows, const int64_t* indices,
                                          int64_t topk, float sm_scale, void* out_bf16,
                                          int64_t out_query_stride, int64_t out_head_stride,
                                          float* lse, int32_t* status, void* workspace,
                                          int64_t workspace_bytes, cudaStream_t stream) {
  using namespace kvq;
  AttnParams p;
  int rc = attention_params(q_bf16, num_queries, num_heads, q_query_stride, q_head_stride, cache,
                            num_blocks, block_size, block_stride_rows, indices, topk, sm_scale,
                            out_bf16, out_query_stride, out_head_stride, lse, status, p);
  if (rc != KVQ_OK || num_queries == 0) return rc;
  if (workspace) {
    const int64_t chunks = split_chunks(p.units, p.tiles);
    const int64_t need = chunks > 1 ? split_bytes(p.units * chunks, num_heads) : 0;
    if (workspace_bytes < need || !aligned(workspace, 256)) return KVQ_EINVAL;
    if (chunks > 1) split_layout(p, chunks, workspace);
  }
  return launch_attention(p, stream);
}

// ------------------------------------------------- built-in scratch variant ---
//
// For callers that must not allocate device memory themselves: code embedded
// in a host framework that owns every byte of device memory through its own
// pool and hands a library no allocator (an allocation behind its back is
// memory it neither counts nor limits), and latency-critical loops that
// cannot afford cudaMalloc, which may synchronise the device. Such callers
// can still pass their inputs and outputs; this entry point takes the split
// schedule's scratch from an array in this library's own device memory
// instead of from a workspace argument.
//
// The array is a file-scope __device__ object of kScratchBytes (40 MiB: the
// split schedule of 128 heads over up to 635 SMs). Every GPU that loads this
// library's attention code holds it until the process exits. Host code only
// has a host-side stand-in for its name, so the device address is looked up
// with cudaGetSymbolAddress once per device, with that device current, on
// the first call made on it. Nothing in it needs to start at zero: each call
// writes every piece it later reads. All calls share it and it keeps the last
// call's contents, so two calls whose kernels overlap on the GPU (different
// streams, or different host threads, on one device) race on it and must be
// ordered by the caller.
constexpr int64_t kScratchBytes = 40ll << 20;
__device__ __align__(256) unsigned char g_attention_scratch[kScratchBytes];

int scratch_address(void** out) {
  static void* addr[64] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return KVQ_ECUDA;
  if (!addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_attention_scratch) != cudaSuccess || !p) {
      cudaGetLastError();
      return KVQ_ECUDA;
    }
    addr[dev] = p;
  }
  *out = addr[dev];
  return KVQ_OK;
}

extern "C" int mxfp4_mla_sparse_attention_noalloc(
    const void* q_bf16, int64_t num_queries, int64_t num_heads, int64_t q_query_stride,
    int64_t q_head_stride, const uint8_t* cache, int64_t num_blocks, int64_t block_size,
    int64_t block_stride_rows, const int64_t* indices, int64_t topk, float sm_scale,
    void* out_bf16, int64_t out_query_stride, int64_t out_head_stride, float* lse,
    int32_t* status, cudaStream_t stream) {
  using namespace kvq;
  AttnParams p;
  int rc = attention_params(q_bf16, num_queries, num_heads, q_query_stride, q_head_stride, cache,
                            num_blocks, block_size, block_stride_rows, indices, topk, sm_scale,
                            out_bf16, out_query_stride, out_head_stride, lse, status, p);
  if (rc != KVQ_OK || num_queries == 0) return rc;
  const int64_t chunks = split_chunks(p.units, p.tiles);
  if (chunks > 1) {
    if (split_bytes(p.units * chunks, num_heads) > kScratchBytes) return KVQ_ESCRATCH;
    void* scratch = nullptr;
    rc = scratch_address(&scratch);
    if (rc != KVQ_OK) return rc;
    split_layout(p, chunks, scratch);
  }
  return launch_attention(p, stream);
}
