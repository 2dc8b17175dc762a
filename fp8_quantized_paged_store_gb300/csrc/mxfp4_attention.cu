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
// 32-key tiles; the units' tiles laid end to end (query-major, half 0 before
// half 1) are cut into one contiguous range per CTA of a grid of one CTA per
// SM, so that every SM gets the same number of tiles whatever the number of
// units (the split-K of the read path). A CTA walks its range as segments,
// one per unit it touches: a segment that covers its whole unit writes the
// output; one that covers part of a unit writes an fp32 partial (the output
// normalised by the piece's own softmax sum, and that sum's log-sum-exp)
// into a caller-provided workspace, and a second, small kernel combines the
// pieces of each split unit by their log-sum-exps. Between segments the CTA
// reads the output accumulator out and, when the query changes, reloads Q;
// the producers keep streaming the next segment's keys meanwhile. Without a
// workspace the grid has one CTA per unit and nothing is split.
//
// Each CTA: tensor memory (512 columns x 128 lanes,
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
// Before tensor memory is released, the issuing thread waits (bounded, abort
// or not) for every MMA it issued, so that none writes released tensor
// memory or arrives on a released barrier.
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
constexpr uint32_t kOffBar = kOffK + kStages * kKBytes;  // eighteen mbarriers
constexpr uint32_t kOffTmemSlot = kOffBar + 160;
constexpr uint32_t kOffAbort = kOffTmemSlot + 16;
constexpr uint32_t kSmemUsed = kOffAbort + 16;
constexpr size_t kSmemBytes = kSmemUsed + 1024;  // room to align the base to 1024

// mbarriers, one of each per stage (the CTA's i-th tile uses stage i % kStages),
// then one that softmax completes at every segment boundary (the output
// accumulator has been read out and, for a new query, Q reloaded), and one
// the issuer commits its last MMAs to before tensor memory is released
constexpr uint32_t kBarKFull = 0, kBarSFull = 32, kBarPFull = 64, kBarPvDone = 96;
constexpr uint32_t kBarSeg = 128, kBarDrain = 136;

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
  // Schedule: unit k = (query k / 2, value half k % 2) is `tiles` tiles of
  // 32 keys; the units' tiles laid end to end (`total` of them) are split
  // into `grid` contiguous ranges, CTA b taking [total*b/grid,
  // total*(b+1)/grid).
  int64_t tiles, units, total;
  int64_t nq;  // queries
  int64_t grid;
  // Partial results of units split between CTAs (null when grid is one CTA
  // per unit, so that nothing is split): piece slot 2b (CTA b's first
  // segment) or 2b + 1 (its last), [2 * grid][num_heads][256] fp32 outputs
  // normalised by the piece's softmax sum, and [2 * grid][num_heads] that
  // sum's log-sum-exp in log2 units (-inf for a piece without valid keys).
  float* part_o;
  float* part_lse;
  // Ragged index runs (one CTA per unit only): query n's indices are
  // indices[key_offsets[n] .. key_offsets[n + 1]), each bound clamped to
  // [0, num_indices]; null for the fixed [num_queries, topk] layout.
  const int64_t* key_offsets;
  int64_t num_indices;
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

// Position in a CTA's run of tiles: query n, value half v, and tile t within
// the unit (n, v); next() says whether it entered a new unit. The split schedule orders units half-major (every query's half 0,
// then every query's half 1), so that the two halves of a query run at the
// same time on different CTAs and read the same packed rows through L2.
// Unsplit (one CTA per unit), a CTA's tiles never leave its unit.
template <bool kSplit>
struct Cursor {
  int64_t n, t;
  int32_t v;
  __device__ __forceinline__ bool next(const AttnParams& p) {
    ++t;
    if (kSplit && t == p.tiles) {
      t = 0;
      if (++n == p.nq) {
        n = 0;
        ++v;
      }
      return true;
    }
    return false;
  }
};

// Slot index of key j of the cursor's tile, or -1 past the query's indices.
// Split: query c.n's row of the [num_queries, topk] indices. One CTA per
// unit: the CTA's own run [key_off, key_off + key_len) (a row of the fixed
// layout, or a ragged run).
template <bool kSplit>
__device__ __forceinline__ int64_t key_index(const AttnParams& p, const Cursor<kSplit>& c, int j,
                                             int64_t key_off, int64_t key_len) {
  const int64_t k = c.t * kTileKeys + j;
  if (kSplit) return k < p.topk ? ld_once_i64(p.indices + c.n * p.topk + k) : -1;
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
// accumulation (the first tile of a segment).
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

// Q of query n into the operand buffers (not inlined: they run once per query
// change, and inlined into the softmax loop they made its live state spill):
// dims 256..511 of head r into the
// swizzled K-major shared-memory layout (zero rows past num_heads), 16 bytes
// per cp.async by threads [0, nthreads); then, by the 128 softmax threads
// only (warps 0-3, head = thread), dims 0..255 into TMEM lane `head`,
// columns kColQ.. as bf16 pairs (the A operand of the first 16 q.k steps).
__device__ __noinline__ void load_q_smem(const AttnParams& p, int64_t n, uint32_t q_base,
                                            int tid, int nthreads) {
  const uint8_t* qn = p.q + n * p.q_qstride;
  for (int id = tid; id < kHeads * 32; id += nthreads) {
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
}

__device__ __noinline__ void load_q_tmem(const AttnParams& p, int64_t n, uint32_t tmem,
                                         int tid) {
  const uint32_t lane_base = tmem + ((uint32_t)((tid >> 5) * 32) << 16);
  const uint8_t* qrow = p.q + n * p.q_qstride + (int64_t)tid * p.q_hstride;
#pragma unroll 1
  for (int c = 0; c < 4; ++c) {
    uint32_t w[32];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const uint4 x =
          tid < p.num_heads ? ld_once_v4(qrow + 128 * c + 16 * k) : make_uint4(0, 0, 0, 0);
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

// One head's result for the segment just finished (thread = head, O in TMEM
// lanes of this warp): the bf16 output row half, or for a unit split between
// CTAs the fp32 output normalised by this piece's softmax sum and that sum's
// log-sum-exp (log2 units) in piece slot `slot`.
// Reads O out 16 columns at a time, which keeps the softmax loop's live
// state in registers around it.
template <bool kSplit>
__device__ __forceinline__ void write_segment(const AttnParams& p, int64_t n, int v, bool whole,
                                              int64_t slot, uint32_t lane_base, int h,
                                              float m_ref, float l) {
  if (!kSplit) whole = true;
  const bool store = h < p.num_heads;
  const float inv = l > 0.0f ? 1.0f / l : 0.0f;
  uint8_t* orow = p.out + n * p.o_qstride + (int64_t)h * p.o_hstride + (int64_t)v * kHalf * 2;
  float* prow = whole ? nullptr : p.part_o + (slot * p.num_heads + h) * kHalf;
#pragma unroll 1
  for (int c = 0; c < kHalf / 16; ++c) {
    uint32_t o[16];
    tmem_ld16(lane_base + kColO + 16 * c, o);
    if (whole) {
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
    } else if (store) {
#pragma unroll
      for (int u = 0; u < 4; ++u)
        st_v4(prow + 16 * c + 4 * u,
              make_uint4(__float_as_uint(__uint_as_float(o[4 * u]) * inv),
                         __float_as_uint(__uint_as_float(o[4 * u + 1]) * inv),
                         __float_as_uint(__uint_as_float(o[4 * u + 2]) * inv),
                         __float_as_uint(__uint_as_float(o[4 * u + 3]) * inv)));
    }
  }
  if (!store) return;
  const float lse2 = l > 0.0f ? m_ref + log2f(l) : -__int_as_float(0x7F800000);
  if (!whole)
    p.part_lse[slot * p.num_heads + h] = lse2;
  else if (v == 0 && p.lse)
    p.lse[n * p.num_heads + h] =
        l > 0.0f ? lse2 * 0.69314718055994531f : -__int_as_float(0x7F800000);
}

// First tile of CTA b's range. One CTA per unit: the unit's tiles; split
// (at most 1023 CTAs, total * 1024 in range): total * b / grid.
__device__ __forceinline__ int64_t range_begin(const AttnParams& p, int64_t b) {
  return p.grid == p.units ? b * p.tiles : p.total * b / p.grid;
}

// kSplit: the split schedule (ranges of tiles over units, pieces, Q reloads
// between segments); otherwise one CTA per unit, which compiles without any
// of that.
template <bool kSplit>
__global__ void __launch_bounds__(kThreads, 1) mxfp4_attention_kernel(AttnParams p) {
  extern __shared__ uint8_t smem_raw[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t b = blockIdx.x;
  // One CTA per unit: this CTA's run of indices (a row of the fixed layout,
  // or its query's ragged run) and its number of tiles.
  int64_t key_off = 0, key_len = p.topk;
  if (!kSplit) {
    const int64_t n0 = b >> 1;
    if (p.key_offsets) {
      int64_t lo = ld_once_i64(p.key_offsets + n0), hi = ld_once_i64(p.key_offsets + n0 + 1);
      lo = lo < 0 ? 0 : (lo > p.num_indices ? p.num_indices : lo);
      hi = hi < lo ? lo : (hi > p.num_indices ? p.num_indices : hi);
      key_off = lo;
      key_len = hi - lo;
    } else {
      key_off = n0 * p.topk;
    }
  }
  const int64_t unit_tiles = kSplit ? p.tiles : (key_len + kTileKeys - 1) / kTileKeys;
  if (unit_tiles == 0) {
    // no keys at all: every output row is zero and every log-sum-exp -inf
    // (one CTA per unit)
    const int64_t n = b >> 1;
    const int v = (int)(b & 1);
    for (int id = tid; id < p.num_heads * 32; id += kThreads)
      st_v4(p.out + n * p.o_qstride + (int64_t)(id >> 5) * p.o_hstride + v * kHalf * 2 +
                (id & 31) * 16,
            make_uint4(0, 0, 0, 0));
    if (v == 0 && p.lse)
      for (int h = tid; h < p.num_heads; h += kThreads)
        p.lse[n * p.num_heads + h] = -__int_as_float(0x7F800000);
    return;
  }
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* sm = smem_raw + (base - raw);
  const uint32_t q_base = base + kOffQ, k_base = base + kOffK;
  const uint32_t bars = base + kOffBar;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + kOffTmemSlot);
  volatile int* abort = reinterpret_cast<volatile int*>(sm + kOffAbort);
  // this CTA's run of tiles [g0, g1) and where it starts
  const int64_t g0 = kSplit ? range_begin(p, b) : 0;
  const int64_t n_tiles = kSplit ? range_begin(p, b + 1) - g0 : unit_tiles;  // >= 1
  const int64_t u_first = kSplit ? g0 / p.tiles : b;
  Cursor<kSplit> start;
  start.t = kSplit ? g0 - u_first * p.tiles : 0;
  start.n = kSplit ? u_first % p.nq : b >> 1;
  start.v = (int32_t)(kSplit ? u_first / p.nq : b & 1);

  if (warp == kIssuerWarp) tmem_alloc(smem_addr(tmem_slot), kTmemCols);
  if (tid == 0) {
#pragma unroll
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bars + kBarKFull + 8 * s, 256);
      mbar_init(bars + kBarSFull + 8 * s, 1);
      mbar_init(bars + kBarPFull + 8 * s, 128);
      mbar_init(bars + kBarPvDone + 8 * s, 1);
    }
    mbar_init(bars + kBarSeg, 128);
    mbar_init(bars + kBarDrain, 1);
    *abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  // The producers issue their first kDepth tiles of row loads at once, while
  // the softmax and issuer warps (160 threads) load Q: the two start-up
  // latencies overlap.
  const bool producer = warp >= 4 && warp < kIssuerWarp;
  const int e = warp - 4, j = lane;
  Cursor<kSplit> cl = start;  // a producer's next tile to load
  Packed buf[kDepth];
  int64_t s_next = -1;
  if (producer) {
#pragma unroll
    for (int u = 0; u < kDepth; ++u) {
      buf[u] = load_packed(p, u < n_tiles ? key_index(p, cl, j, key_off, key_len) : -1, e);
      cl.next(p);
    }
    s_next = kDepth < n_tiles ? key_index(p, cl, j, key_off, key_len) : -1;
  } else {
    load_q_smem(p, start.n, q_base, tid < 128 ? tid : tid - 256, 160);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (warp < 4) load_q_tmem(p, start.n, tmem, tid);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  if (producer) {
    // ------------------------------------------------------------ producers
    // Lane = key of the tile, warp 4 + e = dims [64e, 64e + 64). The CTA's
    // i-th tile goes to stage i % kStages, free once the p.v of tile
    // i - kStages has completed; rows are loaded kDepth tiles ahead.
    bool live = true;
    for (int64_t i0 = 0; i0 < n_tiles && live; i0 += kDepth) {
#pragma unroll
      for (int u = 0; u < kDepth; ++u) {
        const int64_t i = i0 + u;
        if (i < n_tiles && live) {
          const Packed cur = buf[u];
          buf[u] = load_packed(p, s_next, e);  // tile i + kDepth
          cl.next(p);
          s_next = i + kDepth + 1 < n_tiles ? key_index(p, cl, j, key_off, key_len) : -1;
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
    // --------------------------------------------------------------- issuer
    if (lane == 0) {
      const uint64_t q_desc = smem_desc(q_base, 16, 1024, 2);
      // Event-driven over the CTA's tiles: O += P(pi) V(pi) as soon as
      // softmax has written P(pi) (it frees a key stage, so it goes first);
      // else q.k of tile qi (with tile qi + 1 when qi's stage is even and
      // both tiles belong to the same query) once its keys are written and
      // the p.v that last read its tensor-memory columns has been issued
      // (MMAs from this thread run in order). The first p.v of a segment
      // waits for softmax to have read out the previous segment's output;
      // the first q.k of a new query waits for softmax to have loaded its Q.
      // Segment boundaries are observed one at a time, in order.
      Cursor<kSplit> cq = start, cp = start;
      int64_t qi = 0, pi = 0, seen = 0;
      int32_t qseg = 0, pseg = 0;  // segments of the next q.k and p.v tiles
      uint32_t idle = 0;
      auto seg_ready = [&](int64_t k) -> bool {
        if constexpr (kSplit) {
          while (seen < k) {
            if (!mbar_test(bars + kBarSeg, (uint32_t)(seen & 1))) return false;
            ++seen;
          }
        }
        return true;
      };
      while (pi < n_tiles) {
        bool progress = false;
        if (pi < qi && mbar_test(bars + kBarPFull + 8 * (uint32_t)(pi % kStages),
                                 (uint32_t)((pi / kStages) & 1))) {
          const bool first = pi == 0 || (kSplit && cp.t == 0);
          if (!first || pi == 0 || seg_ready(pseg)) {
            tc_fence_after();
            issue_pv((uint32_t)(pi % kStages), cp.v, first, k_base, tmem);
            mma_commit(bars + kBarPvDone + 8 * (uint32_t)(pi % kStages));
            ++pi;
            pseg += cp.next(p) ? 1 : 0;
            progress = true;
          }
        }
        if (!progress && qi < n_tiles) {
          const uint32_t st = (uint32_t)(qi % kStages);
          Cursor<kSplit> c2 = cq;
          const int32_t qseg2 = qseg + (c2.next(p) ? 1 : 0);
          // pairs stay within a unit (its next tile is not a unit's first)
          const bool pair = (st & 1u) == 0 && qi + 1 < n_tiles && (!kSplit || c2.t != 0);
          if (qi + (pair ? 1 : 0) - pi < kStages &&
              mbar_test(bars + kBarKFull + 8 * st, (uint32_t)((qi / kStages) & 1)) &&
              (!pair || mbar_test(bars + kBarKFull + 8 * (st + 1),
                                  (uint32_t)(((qi + 1) / kStages) & 1))) &&
              seg_ready(qseg)) {
            tc_fence_after();
            if (pair) {
              issue_qk<true>(st, q_desc, k_base, tmem);
              mma_commit(bars + kBarSFull + 8 * st);
              mma_commit(bars + kBarSFull + 8 * (st + 1));
              qi += 2;
              cq = c2;
              qseg = qseg2 + (cq.next(p) ? 1 : 0);
            } else {
              issue_qk<false>(st, q_desc, k_base, tmem);
              mma_commit(bars + kBarSFull + 8 * st);
              qi += 1;
              cq = c2;
              qseg = qseg2;
            }
            progress = true;
          }
        }
        if (progress) {
          idle = 0;
        } else if (++idle >= kWaitPolls) {
          *abort = 1;
          break;
        } else if ((idle & 31u) == 31u && *abort) {
          break;
        }
      }
      if (!drain_mmas(bars + kBarDrain)) *abort = 1;
    }
    __syncwarp();
  } else {
    // -------------------------------------------------------------- softmax
    const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
    const float kNegInf = -__int_as_float(0x7F800000);
    float m_ref = kNegInf;  // reference max of the segment (log2 units)
    float l = 0.0f;         // sum of p against m_ref
    bool live = true;
    Cursor<kSplit> c = start;
    bool first_seg = true;  // in the CTA's first segment
    int64_t s_key = key_index(p, c, lane, key_off, key_len);
    for (int64_t i = 0; i < n_tiles && live; ++i) {
      const bool seg_first = i == 0 || (kSplit && c.t == 0);
      const bool seg_last = i == n_tiles - 1 || (kSplit && c.t == p.tiles - 1);
      if (seg_first) {
        m_ref = kNegInf;
        l = 0.0f;
      }
      const uint32_t mask = __ballot_sync(0xFFFFFFFFu, s_key >= 0 && s_key < p.num_slots);
      Cursor<kSplit> cn = c;
      const bool new_unit = cn.next(p);
      s_key = i + 1 < n_tiles ? key_index(p, cn, lane, key_off, key_len) : -1;
      const uint32_t st = (uint32_t)(i % kStages);
      if (!warp_wait(bars + kBarSFull + 8 * st, (uint32_t)((i / kStages) & 1), abort)) {
        live = false;
        break;
      }
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
      const bool need = mt > m_ref + 8.0f;
      if (__any_sync(0xFFFFFFFFu, need)) {
        const float f = need ? ex2(m_ref - mt) : 1.0f;  // ex2(-inf) = 0
        if (!seg_first) {
          // O may be touched only once the p.v of tile i - 1 has completed
          const int64_t w = i - 1;
          if (!warp_wait(bars + kBarPvDone + 8 * (uint32_t)(w % kStages),
                         (uint32_t)((w / kStages) & 1), abort)) {
            live = false;
            break;
          }
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
      if (seg_last) {
        // the segment's output: wait for its last p.v, read O out, then (if
        // another segment follows) load Q of a new query and release O
        if (!warp_wait(bars + kBarPvDone + 8 * st, (uint32_t)((i / kStages) & 1), abort)) {
          live = false;
          break;
        }
        tc_fence_after();
        // whole: the segment runs from the unit's first tile to its last
        // (recomputed here rather than kept live through the loop)
        const int64_t cta = blockIdx.x;
        const bool whole = c.t + 1 == p.tiles &&
                           (!first_seg || (kSplit ? range_begin(p, cta) % p.tiles : 0) == 0);
        write_segment<kSplit>(p, c.n, c.v, whole, 2 * cta + (first_seg ? 0 : 1), lane_base, tid,
                              m_ref, l);
        if (kSplit && i + 1 < n_tiles) {
          if (cn.n != c.n) {
            load_q_smem(p, cn.n, q_base, tid, 128);
            load_q_tmem(p, cn.n, tmem, tid);
          }
          tc_fence_before();
          mbar_arrive(bars + kBarSeg);
        }
      }
      c = cn;
      if (new_unit) first_seg = false;
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

// Combines the pieces of every unit split between CTAs. Block (j, g) looks at
// the boundary between CTAs j and j + 1 and heads 8g..8g+7; the unit the
// boundary falls inside (if any) is merged by the blocks of its first
// boundary, over the pieces of CTAs b_first..b_last:
// out = sum_b 2**(lse_b - L) o_b / sum_b 2**(lse_b - L), L = max_b lse_b, and
// the unit's log-sum-exp L + log2(sum) (in natural log units, half 0 only).
// A unit without any valid key gets zeros and -inf. The pieces' slots are
// worked out in parallel into shared memory; 64 threads take a head, four
// columns each. A unit of up to kMergeFew pieces is summed by each thread
// on its own; beyond that (the launch then gives the block dynamic shared
// memory for kMergeHeads x pieces weights), every (head, piece) weight is
// first worked out in parallel, and the sums keep several loads in flight.
constexpr int kMergeMaxPieces = 1024;  // grid <= 1023
constexpr int kMergeHeads = 8;         // heads per block (64 threads each)
constexpr int kMergeFew = 4;

__global__ void __launch_bounds__(64 * kMergeHeads, 4) mxfp4_attention_merge_kernel(AttnParams p) {
  __shared__ int32_t piece_slot[kMergeMaxPieces];
  __shared__ float head_l[kMergeHeads][2], head_w[kMergeHeads][2];
  extern __shared__ float merge_dyn[];  // [kMergeHeads][pieces]: log-sum-exp, then weight
  const int64_t j = blockIdx.x;
  const int64_t gb = p.total * (j + 1) / p.grid;
  const int64_t unit = gb / p.tiles;
  if (gb == unit * p.tiles) return;  // the boundary lies between units
  const int64_t g0 = p.total * j / p.grid;
  if (g0 > unit * p.tiles) return;   // merged by the blocks of an earlier boundary
  const int64_t b_last = ((unit + 1) * p.tiles * p.grid - 1) / p.total;
  const int pieces = (int)(b_last - j + 1);
  for (int k = threadIdx.x; k < pieces; k += blockDim.x) {
    const int64_t bb = j + k;
    piece_slot[k] = (int32_t)(2 * bb + ((p.total * bb / p.grid) / p.tiles == unit ? 0 : 1));
  }
  __syncthreads();
  const int64_t H = p.num_heads;
  const float kNegInf = -__int_as_float(0x7F800000);
  const int64_t n = unit % p.nq;  // half-major unit order
  const int v = (int)(unit / p.nq);
  uint32_t dyn_bytes;
  asm("mov.u32 %0, %%dynamic_smem_size;" : "=r"(dyn_bytes));
  if (pieces <= kMergeFew || dyn_bytes < (uint32_t)(kMergeHeads * pieces) * 4u) {
    const int64_t h = (int64_t)blockIdx.y * kMergeHeads + (threadIdx.x >> 6);
    if (h >= H) return;
    const int c4 = threadIdx.x & 63;
    float L = kNegInf;
#pragma unroll 4
    for (int k = 0; k < pieces; ++k) L = fmaxf(L, p.part_lse[piece_slot[k] * H + h]);
    float W = 0.0f;
    float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    if (L != kNegInf) {
#pragma unroll 4
      for (int k = 0; k < pieces; ++k) {
        const int64_t row = piece_slot[k] * H + h;
        const float w = exp2f(p.part_lse[row] - L);
        const float4 o = *reinterpret_cast<const float4*>(p.part_o + row * kHalf + 4 * c4);
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
    merge_dyn[hh * pieces + k] = h < H ? p.part_lse[piece_slot[k] * H + h] : kNegInf;
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
  // weights 2**(lse_b - L) (0 for a piece without valid keys) and their sum
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
      const float4 o =
          *reinterpret_cast<const float4*>(p.part_o + (piece_slot[k] * H + h) * kHalf + 4 * c4);
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

// CTAs of the split schedule: one per SM (each holds all of tensor memory),
// with at least kMinSplitTiles tiles each (a CTA's start-up and its piece's
// write and merge cost a few tiles' time).
constexpr int64_t kMinSplitTiles = 4;
int64_t split_grid(int64_t total) {
  int64_t sms = kvq::sm_count();
  if (sms > 1023) sms = 1023;
  const int64_t want = total / kMinSplitTiles > 1 ? total / kMinSplitTiles : 1;
  return want < sms ? want : sms;
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
  p.total = 2 * num_queries * tiles;
  p.grid = 2 * num_queries;  // one CTA per unit unless split
  p.part_o = nullptr;
  p.part_lse = nullptr;
  p.key_offsets = nullptr;
  p.num_indices = 0;
  return KVQ_OK;
}

// Bytes of the split schedule's partial results (0 without keys).
int64_t split_bytes(int64_t grid, int64_t num_heads) {
  return 2 * grid * num_heads * (int64_t)(kvq::kHalf * 4 + 4);
}

// Lays the partial results out in `ws` (256-byte aligned) for `grid` CTAs.
void split_layout(kvq::AttnParams& p, int64_t grid, void* ws) {
  p.grid = grid;
  p.part_o = static_cast<float*>(ws);
  p.part_lse = p.part_o + 2 * grid * p.num_heads * kvq::kHalf;
}

int launch_attention(const kvq::AttnParams& p, cudaStream_t stream) {
  using namespace kvq;
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
  if (rc != KVQ_OK || !p.part_o || p.grid < 2) return rc;
  const dim3 mgrid((unsigned)(p.grid - 1), (unsigned)((p.num_heads + kMergeHeads - 1) / kMergeHeads));
  // the most pieces a unit can have: every CTA takes at least total / grid tiles
  const int64_t per_cta = p.total / p.grid;
  const int64_t most = p.tiles / (per_cta > 0 ? per_cta : 1) + 2;
  const size_t dyn = most > kMergeFew
                         ? (size_t)kMergeHeads * (size_t)(most < kMergeMaxPieces ? most : kMergeMaxPieces) * 4
                         : 0;
  mxfp4_attention_merge_kernel<<<mgrid, 64 * kMergeHeads, dyn, stream>>>(p);
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
  p.tiles = 1;  // per CTA from its run; one CTA per (query, value half)
  p.total = p.units;
  return launch_attention(p, stream);
}

extern "C" int64_t mxfp4_mla_sparse_attention_workspace_size(int64_t num_queries,
                                                             int64_t num_heads, int64_t topk) {
  if (num_queries < 0 || num_heads < 1 || num_heads > kvq::kHeads || topk < 0) return KVQ_EINVAL;
  if (num_queries > 0x7FFFFFFF / 2 || num_queries > INT64_MAX / 2 / (topk > 0 ? topk : 1))
    return KVQ_EINVAL;
  const int64_t tiles = (topk + kvq::kTileKeys - 1) / kvq::kTileKeys;
  if (tiles > 0 && 2 * num_queries > INT64_MAX / 1024 / tiles) return KVQ_EINVAL;
  if (tiles == 0 || num_queries == 0) return 0;
  return split_bytes(split_grid(2 * num_queries * tiles), num_heads);
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
  if (workspace && p.tiles > 0) {
    const int64_t grid = split_grid(p.total);
    if (workspace_bytes < split_bytes(grid, num_heads) || !aligned(workspace, 256))
      return KVQ_EINVAL;
    split_layout(p, grid, workspace);
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
// split schedule of 128 heads over up to 159 SMs). Every GPU that loads this
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
  if (p.tiles > 0) {
    const int64_t grid = split_grid(p.total);
    if (split_bytes(grid, num_heads) > kScratchBytes) return KVQ_ESCRATCH;
    void* scratch = nullptr;
    rc = scratch_address(&scratch);
    if (rc != KVQ_OK) return rc;
    split_layout(p, grid, scratch);
  }
  return launch_attention(p, stream);
}
