// Paged GQA decode attention (koas-w, "errors and solutions", section
// "自写 Triton Kernel", Decode_Paged_GQAAttention_Kernel: the kernel walks the
// block_table itself, keeps an online softmax and serves all query heads of
// a GQA group from one K/V read; no gather into contiguous memory) with
// flash-decoding split-K partials merged inside the kernel.
//
// Work partition.  The blocks of all sequences, in order, form one list of
// N blocks; CTA c of S takes blocks [floor(cN/S), floor((c+1)N/S)).  Every
// CTA moves the same number of bytes however skewed the lengths are, and
// consecutive sequences flow through one CTA's pipeline without draining it.
// A "piece" is the run of one sequence's blocks inside one CTA.  A piece
// that is the whole sequence writes the output rows.  A cut piece writes a
// partial (o normalised over its keys, natural-log sum-exp) to the
// workspace and bumps the sequence's arrival counter; the CTA that brings
// the counter to the piece count merges all partials of that sequence
// (log-sum-exp) and writes its rows, then resets the counter to zero.  Only
// a CTA's first piece (cut at its head) and its final piece (cut at its
// tail) can be cut.  Every piece but the final one is handed to the epilogue
// warp: the consumer warps drop their rows into one of two shared buffers and
// stream on, while the epilogue warp combines them, writes the output rows or
// the partial and publishes a cut piece.  The consumers combine and publish
// the final piece themselves, and merge when it arrives last, with their own
// rows taken from shared memory and the others' brought in by bulk copies.
//
// CTA layout (352 threads).  Warps 0 and 1 are producers, filling alternate
// stages of a ring of NST stages guarded by full/empty mbarriers: per
// physical block they issue TMA box loads of K and V (16 tokens x 2 kv heads
// x 64 dims each, 128-byte swizzle; 4 boxes per block at Hkv <= 2), plus a
// bulk copy of the sequence's q rows into each of the first NPH stages of a
// piece.  Two producers overlap the per-stage issue latency of one thread.
// Warp 2 is the epilogue warp.  Warps 3..10 consume: warp (g, ph) handles kv
// head g of the stages whose index is ph modulo NPH = 8 / Hkv, and visits no
// other stage: it takes its q rows from its own first stage of each piece.
// NST is a multiple of NPH, so every slot of the ring holds stages of one
// phase and its Hkv warps wait on each round of it in order.  All consumer
// warps meet at every piece end to combine.
//
// Arithmetic per (block, kv head) on the tensor cores (mma.sync m16n8k16,
// bf16 in, fp32 accumulate), with the G query heads of the group as the
// N = 8 dimension:
//   S^T[16 tokens][8 heads] = K[16 x 128] . Q^T[128 x 8]      (8 MMAs)
//   online softmax over the 16 tokens per head column (fp32, base 2; the
//   reference max moves only by more than 8, so O is rescaled rarely)
//   O^T[128][8]  += V^T[128 x 16] . P^T[16 x 8]                (8 MMAs x 2)
// P is split into bf16 hi + lo parts (two MMAs per tile) so the product
// keeps ~16 bits of the fp32 weights.  K fragments come from ldmatrix on the
// swizzled tiles, V fragments from ldmatrix.trans, P^T from movmatrix.trans
// of the score fragment.
//
// Variants share this code.  Fused store (pa_store_decode*): the CTA that
// stages a sequence's last block patches the new token's K/V rows into its
// tiles and writes them to the pool, so a decode step is one launch.
// Rotary embedding (ROPE, pa_rope_store_decode, with the fused store): the
// cos and sin rows of each sequence's position travel with its q rows, the
// consumers rotate their q fragments in registers and the patch rotates the
// new K row, with the arithmetic of pa_rope_store_kv (rope_rotate8).
// FP8 pools (F8): E4M3 codes with per-kv-head scales; K pages keep the
// token-major layout, V pages are dim-major inside a block and come in one
// bulk copy; codes widen exactly to f16 and the MMAs run in f16, with a
// token order of the score rows that makes every V operand register one
// 32-bit load, K rows read as 16-byte chunks (a dim order per fragment
// column shared with q), and P as one f16 term (see the F8 branches).
// Early K/V requests (p.early_kv, a
// launch flag): the producers issue the first ring stages' pages before the
// wait for the previous kernel.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>

#include <type_traits>

#include "pa_common.cuh"

namespace pa {

struct DecodeParams {
  void *out;
  int out_f32;
  const uint16_t *q;  // [B][HQ][128]
  long long num_blocks;
  const int32_t *block_tables;
  long long bt_stride;
  const int32_t *context_lens;
  int batch;
  float qk_scale_log2;  // softmax scale * log2(e): exponentials are base 2
  int num_splits;
  float *part_o;      // [2][S][HQ][128] (slot-major: a sequence's slot-0 rows are consecutive)
  float *part_lse;    // [2][S][HQ], natural log
  int32_t *counters;  // [S] arrival counters, zero between calls
  int32_t *err;
  const float *k_scale;  // FP8 pools only: per kv head, value = code * scale
  const float *v_scale;
  const uint8_t *v_pool;  // FP8 pools only: V, [num_blocks][Hkv][128][16] bytes
  // Fused store (bf16 pools; new_k == nullptr: none).  Sequence b's new
  // token (position context_lens[b] - 1) has K/V rows new_k / new_v + b *
  // new_tok + h * 128; it goes to pool slot slot_mapping[b] (< 0: none) and,
  // in shared memory, into the staged tile of the sequence's last block.
  const uint16_t *new_k;
  const uint16_t *new_v;
  long long new_k_tok, new_v_tok;
  const int32_t *slot_mapping;
  uint16_t *k_pool;
  uint16_t *v_pool16;
  uint8_t *k_pool8;  // FP8 pools, fused store
  uint8_t *v_pool8;
  // Nonzero: the K/V pages of the first ring stages are requested before the
  // previous kernel in the stream completes (the caller guarantees that
  // kernel does not write the pools).
  int early_kv;
  // Rotary embedding inside the fused store (ROPE kernels): sequence b's new
  // token sits at position positions[b]; its q rows and its new K row are
  // rotated with row positions[b] of the float32 tables [max_position][64]
  // before they are used or stored.
  const int32_t *positions;
  const float *cos_table;
  const float *sin_table;
  long long max_position;
};

// Waits for the previous kernel in the stream to complete, then signals that
// the next kernel may begin (programmatic dependent launch; both no-ops
// without it).
__device__ __forceinline__ void wait_prev_then_release() {
  griddep_wait();
  griddep_launch_dependents();
}

constexpr int kDecodeProducerWarps = 2;
constexpr int kDecodeEpilogueWarp = 2;       // warp index of the epilogue warp
constexpr int kDecodeFirstConsumerWarp = 3;  // consumers are warps 3 .. 3 + CW - 1
constexpr int kDecodeConsumerWarps = 8;
constexpr int kDecodeWarps = kDecodeFirstConsumerWarp + kDecodeConsumerWarps;
constexpr int kDecodeThreads = 32 * kDecodeWarps;
constexpr int kDecodeSmemBudget = 227 * 1024;  // dynamic shared memory of one CTA per SM
// K/V stages requested before the wait for the previous kernel (early K/V):
// six of the eight ring stages at the headline shape measured 0.2 us faster
// per chained step than all eight (the burst of every CTA's early requests
// lands in the previous kernel's tail) and than four or two.
constexpr int kDecodeEarlyStages = 6;
constexpr int kTileBytes = kBlockSize * 64 * 2;  // 16 tokens x 64 dims bf16 = 2 KB per head

__host__ __device__ constexpr int align_up(int x, int a) { return (x + a - 1) / a * a; }

// F8: the pools hold E4M3 codes (one byte per element) with per-kv-head
// scales; K pages keep the token-major layout, V pages are dim-major inside a
// block ([Hkv][128 dims][16 tokens]).
template <int G, int HKV, bool F8 = false, bool ROPE = false>
struct DecodeShape {
  static constexpr int HQ = G * HKV;
  static constexpr int CW = kDecodeConsumerWarps;
  static constexpr int NPH = CW / HKV;  // stage phases = warps per kv head
  // one TMA box = 16 tokens x HB heads x 64 dims; a page of K (or V) takes
  // NPAIR * 2 boxes (head groups x dim halves)
  static constexpr int HB = HKV >= 2 ? 2 : 1;
  static constexpr int NPAIR = HKV / HB;
  // bf16: 16 tokens x HB heads x 64 dims (two boxes per head pair);
  // F8: K 16 tokens x HB heads x 128 dims, V HB heads x 128 dims x 16 tokens
  // (one box each per head pair); 2 KB per head either way
  static constexpr int BOX_BYTES = HB * kTileBytes;
  static constexpr int KV_BYTES = HKV * (F8 ? 1 : 2) * kTileBytes;  // one block of K (or V)
  static constexpr int Q_BYTES = HQ * kHeadDim * 2;
  // ROPE: the cos and sin rows of the sequence's position follow the q rows
  static constexpr int ROPE_BYTES = ROPE ? 2 * (kHeadDim / 2) * 4 : 0;
  static constexpr int STAGE_BYTES = align_up(2 * KV_BYTES + Q_BYTES + ROPE_BYTES, 1024);
  // per consumer warp and query head of its group: o[128], m, l (rows of
  // 132 floats keep the o vectors 16-byte aligned)
  static constexpr int RED_FLOATS_PER_HEAD = kHeadDim + 4;
  static constexpr int RED_M = kHeadDim, RED_L = kHeadDim + 1;
  // two buffers: the epilogue warp combines piece i from one while the
  // consumers already fill the other at the end of piece i + 1
  static constexpr int RED_ONE_FLOATS = align_up(CW * G * RED_FLOATS_PER_HEAD, 256);
  static constexpr int RED_BYTES = NPH > 1 ? 2 * RED_ONE_FLOATS * 4 : 0;
  static constexpr int CTL_BYTES = 512;
  // Prefetched merges: while the consumers stream the CTA's final piece, the
  // epilogue warp brings the other pieces' partials of its sequence into the
  // red buffer nobody uses any more; up to PF_PIECES pieces' rows fit there.
  // The prefetched lse values sit in the merge scratch at PF_W.  A merge the
  // CTA owes besides its final one (a piece the epilogue warp published
  // arrived last) runs beside it, with its weights at DEF_W.
  static constexpr int PF_PIECES = NPH > 1 ? RED_ONE_FLOATS / (HQ * kHeadDim) : 0;
  static constexpr bool PF_LSE_COPY = HQ % 4 == 0;  // lse rows are 16-byte runs
  static constexpr int PF_W = 1024, DEF_W = 1536;
  static constexpr int DEF_MAX_PIECES = 512 / HQ - 1;  // weights room of the owed merge
  // the epilogue warp's combine weights: NPH per query head (NPH * HQ = CW * G)
  static constexpr int EWW_BYTES = 256;
  // merge scratch: one weight per (piece, query head), up to MERGE_MAX_PIECES
  static constexpr int MERGE_FLOATS = 2048;
  static constexpr int MERGE_MAX_PIECES = MERGE_FLOATS / HQ - 1;  // + one row of 1 / sums
  static constexpr int MERGE_BYTES = MERGE_FLOATS * 4;
  static constexpr int NST_FIT =
      (kDecodeSmemBudget - 1024 - RED_BYTES - MERGE_BYTES - CTL_BYTES - EWW_BYTES) /
      (STAGE_BYTES + 16);
  static constexpr int NST_CAP = NST_FIT > 12 ? 12 : NST_FIT;
  // The ring is a multiple of 2 (each slot is always filled by the same one
  // of the two producer warps) and of NPH (each slot always holds stages of
  // the same phase, so the Hkv consumer warps of that phase wait on every
  // round of the slot in order: a parity wait never skips a phase).
  static constexpr int RING_MULT = NPH > 2 ? NPH : 2;
  static constexpr int NST = NST_CAP - NST_CAP % RING_MULT;
  // +1024: the dynamic smem base is realigned to 1024 bytes for the swizzle
  static constexpr int SMEM =
      1024 + NST * STAGE_BYTES + RED_BYTES + MERGE_BYTES + NST * 16 + CTL_BYTES + EWW_BYTES;
  static_assert(NST >= RING_MULT && NST % RING_MULT == 0, "stage ring does not fit");
  static_assert(CW % HKV == 0, "unsupported kv head count");
  static_assert(SMEM <= kDecodeSmemBudget, "shared memory over budget");
  // a final cut piece keeps its own rows (o, lse) in the ring
  static_assert(HQ * (kHeadDim + 1) * 4 <= NST * STAGE_BYTES, "own rows do not fit the ring");
  static_assert(G >= 1 && G <= 8, "group size must fit the N = 8 MMA dimension");
  // combine weights (NPH per query head) and lse live in the merge scratch
  static_assert((NPH + 1) * HQ <= MERGE_FLOATS, "combine weights do not fit");
  static_assert(CW * G * 4 <= EWW_BYTES, "epilogue warp weights do not fit");
  static_assert(!(F8 && ROPE), "rotary embedding is fused for bf16 pools only");
  static_assert(PF_W + (PF_PIECES + 1) * HQ <= DEF_W && DEF_W + 512 <= MERGE_FLOATS,
                "prefetched lse and owed-merge weights do not fit the merge scratch");
  static_assert(DEF_MAX_PIECES >= 1, "owed-merge weights do not fit");
};

// A piece handed to the epilogue warp (one per red buffer).
struct PieceDesc {
  long long slot_row;  // first workspace row of a cut piece's partial
  long long cs0, cs1;  // splits holding the sequence's blocks
  int b;               // sequence
  int kind;            // kPieceWhole, kPieceCut or kPieceEnd
  int pieces;          // non-empty pieces of the sequence
  int pad;
};
constexpr int kPieceWhole = 0;  // write the sequence's output rows
constexpr int kPieceCut = 1;    // write a partial, publish it (the merge if it comes last)
constexpr int kPieceEnd = 2;    // no further piece: the epilogue warp exits

struct DecodeCtl {
  unsigned long long red_full[2];   // mbarriers: red buffer k holds a piece (CW arrivals)
  unsigned long long red_empty[2];  // mbarriers: the epilogue warp is done with buffer k
  unsigned long long merge_bar;     // mbarrier: the final merge's bulk copies
  unsigned long long merge_bar2;    // mbarrier: the deferred merge's bulk copies
  unsigned long long ew_done;       // mbarrier: the epilogue warp has finished
  unsigned long long seen_bar;      // mbarrier: every other piece of the final one arrived
  unsigned long long pf_bar;        // mbarrier: the final piece's prefetched partials
  unsigned long long pub_done;      // mbarrier: the epilogue warp has published every piece
  PieceDesc desc[2];
  // a cut piece the epilogue warp published last: the consumers merge its
  // sequence at their end (def_pending = 1)
  long long def_cs0, def_cs1;
  int def_b, def_pending;
  // the CTA's final piece, cut: its sequence's counter and piece count, for
  // the epilogue warp to watch (fin_valid = 1 once written)
  long long fin_cs0, fin_cs1;
  int fin_pieces, fin_valid;
  int fin_npe;  // pieces handed to the epilogue warp before the final one
  // the epilogue warp prefetched the final piece's other partials (written
  // before it completes seen_bar); use_pf: the consumers' merge reads them
  // (decided once, by consumer thread 0)
  int pf_ready, use_pf;
  int owed_now;  // an owed merge runs beside the final one (consumer thread 0 decides)
  long long first_prefix;    // global index of block 0 of first_b
  int first_b;               // sequence holding this CTA's first block
  int abort;                 // set by a wait that gave up
  int last;                  // this CTA merges the current cut sequence
  // the current piece's sequence: splits pc_cs0..pc_cs1 hold its blocks, in
  // pc_pieces non-empty pieces (consumer thread 0 works them out at the
  // piece start, off the epilogue's path)
  long long pc_cs0, pc_cs1;
  int pc_pieces;
  // consumer thread 0 has decided how the final piece ends (the epilogue
  // warp stops watching the counter)
  int decided;
};
static_assert(sizeof(DecodeCtl) <= 512, "control words do not fit their 512 bytes");

__device__ __forceinline__ int seq_blocks(const int32_t *ctx, int b) {
  const int n = __ldg(ctx + b);
  return n > 0 ? ceil_div_blocks(n) : 0;
}

// Warp-cooperative walk over the CTA's block list.  The walk position is
// (b, ctx, j): block j of sequence b, whose context length is ctx.  One call
// describes the next `count` <= 32 blocks (count <= remaining): lane L gets
// the sequence, block index and context length of block L of the chunk.
// Context lengths of up to 32 following sequences are loaded in parallel
// and placed with a warp scan, so a chunk costs one round of loads however
// many sequences it crosses.  The position then moves past the chunk.  All
// 32 lanes must call it with the same position (the result is uniform).
__device__ __forceinline__ int walk_chunk(const int32_t *ctx_arr, int batch, int &b, int &ctx,
                                          int &j, long long remaining, int lane, int &lb,
                                          int &lj, int &lctx) {
  while (j >= (ctx > 0 ? ceil_div_blocks(ctx) : 0)) {  // leave finished / empty sequences
    if (b + 1 >= batch) return 0;  // inconsistent with the block count: stop the walk
    ++b;
    ctx = __ldg(ctx_arr + b);
    j = 0;
  }
  const int rem = ceil_div_blocks(ctx) - j;  // blocks left in b (>= 1)
  int count = remaining < 32 ? (int)remaining : 32;
  int nctx = 0, nn = 0;
  if (rem < count) {
    const int bb = b + 1 + lane;
    nctx = bb < batch ? __ldg(ctx_arr + bb) : 0;
    nn = nctx > 0 ? ceil_div_blocks(nctx) : 0;
  }
  int incl = nn;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += y;
  }
  // k = number of following sequences that end at or before this lane's block
  int k = 0;
#pragma unroll 4
  for (int kk = 0; kk < 32; ++kk) k += (rem + __shfl_sync(0xffffffffu, incl, kk) <= lane) ? 1 : 0;
  const int ks = k < 32 ? k : 31;
  const int excl_k = __shfl_sync(0xffffffffu, incl - nn, ks);
  const int ctx_k = __shfl_sync(0xffffffffu, nctx, ks);
  bool resolved = true;
  if (lane < rem) {
    lb = b;
    lj = j + lane;
    lctx = ctx;
  } else {
    lb = b + 1 + k;
    lj = lane - rem - excl_k;
    lctx = ctx_k;
    resolved = k < 32;  // beyond 32 following sequences: left for the next chunk
  }
  const unsigned unres = __ballot_sync(0xffffffffu, !resolved);
  if (unres) count = min(count, __ffs(unres) - 1);
  const int last = count - 1;
  b = __shfl_sync(0xffffffffu, lb, last);
  j = __shfl_sync(0xffffffffu, lj, last) + 1;
  ctx = __shfl_sync(0xffffffffu, lctx, last);
  return count;
}

// ---- tensor-core and TMA helpers -------------------------------------------

// 3-D tile load (dims: dim, kv head, token slot) completing on an mbarrier.
// Executed by a whole converged warp with warp-uniform operands (a role
// branch the compiler can see is uniform); one lane, picked by elect.sync,
// issues the copy.  This is the issue pattern the tensor-core MMAs need to
// run at full rate; for these copies it measured neutral.
__device__ __forceinline__ void tma_load_box(uint32_t dst, const CUtensorMap *map, int x, int y,
                                             int z, uint32_t bar, uint64_t policy) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;\n\t}" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar), "l"(policy)
      : "memory");
}

// bulk_load by one elected lane of a converged warp (as tma_load_box).
__device__ __forceinline__ void bulk_load_elect(uint32_t dst, const void *src, uint32_t bytes,
                                                uint32_t bar, uint64_t policy) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;\n\t}" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                        uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr)
               : "memory");
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1,
                                          uint32_t &r2, uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr)
               : "memory");
}

__device__ __forceinline__ uint32_t movm_t(uint32_t x) {
  uint32_t y;
  asm("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

// d += A(16x16, row) . B(16x8, col), bf16 operands, fp32 accumulators.
__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
      "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// d += A(16x16, row) . B(16x8, col), f16 operands, fp32 accumulators.
__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                        uint32_t a3, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, "
      "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Two E4M3 codes (low byte first) to two f16 values (low half first); every
// E4M3 value is exact in f16.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t codes) {
  uint32_t r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"((unsigned short)(codes & 0xFFFFu)));
  return r;
}

// Round two floats to f16 (nearest even, saturated to +-65504), lo in the
// low half.
__device__ __forceinline__ uint32_t float2_to_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ float2 f16x2_to_float2(uint32_t w) {
  float lo, hi;
  asm("{\n\t.reg .f16 a, b;\n\tmov.b32 {a, b}, %2;\n\tcvt.f32.f16 %0, a;\n\t"
      "cvt.f32.f16 %1, b;\n\t}"
      : "=f"(lo), "=f"(hi)
      : "r"(w));
  return make_float2(lo, hi);
}

// Two floats to two E4M3 codes (lo in the low byte): nearest even, saturated
// to +-448 (the same rounding as the FP8 store kernel).
__device__ __forceinline__ uint32_t float2_to_e4m3x2_sat(float lo, float hi) {
  unsigned short r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}

// Byte offset of (row, 16-byte chunk) in a tile written by TMA with the
// 128-byte swizzle: the chunk index is XORed with the row index mod 8.
__device__ __forceinline__ uint32_t swz(int row, int chunk) {
  return row * 128 + ((chunk ^ (row & 7)) << 4);
}

// FP8 K rows: the 16-byte chunk (16 dims) that fragment column qd reads for
// k-steps 4h .. 4h + 3.  The eight threads of a quarter warp read rows r and
// r + HB (score rows gid and gid + 1), so the chunks of the four columns
// must differ from their own set XOR HB for a conflict-free vector load:
// {0, 1, 4, 5} then {2, 3, 6, 7} for HB = 2, {0, 2, 4, 6} then {1, 3, 5, 7}
// for HB = 1.
template <int HB>
__device__ __forceinline__ int f8_k_chunk(int qd, int h) {
  if constexpr (HB == 2) return ((qd & 1) | ((qd & 2) << 1)) + 2 * h;
  else return 2 * qd + h;
}

__device__ __forceinline__ int ld_acquire_gpu(const int *ptr) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(ptr) : "memory");
  return v;
}

__device__ __forceinline__ void fence_acq_rel_gpu() {
  asm volatile("fence.acq_rel.gpu;" ::: "memory");
}

// A cut sequence's counter word holds two counts: the pieces that have
// arrived (low 16 bits) and the pieces whose partial rows are published
// (high 16 bits).  A piece arrives first with a relaxed add (kArrive) and
// publishes afterwards with a release add (kPublish) unless it arrived
// last: the last arrival merges, so it needs only to see every other piece
// published and never publishes its own rows.  Piece counts stay below 2^16
// (at most PA_DECODE_MAX_SPLITS).
constexpr int kArrive = 1, kPublish = 1 << 16;
__device__ __forceinline__ int arrived_count(int w) { return w & 0xFFFF; }
__device__ __forceinline__ int published_count(int w) { return (int)((unsigned)w >> 16); }

// Add with release semantics at GPU scope: the partial rows written before
// it (by this thread, or by the threads a CTA or warp barrier ordered
// before it) are visible to whoever observes the new word with an acquire.
// Returns the old word.
__device__ __forceinline__ int atom_add_release_gpu(int32_t *ptr, int v) {
  int old;
  asm volatile("atom.release.gpu.global.add.s32 %0, [%1], %2;"
               : "=r"(old)
               : "l"(ptr), "r"(v)
               : "memory");
  return old;
}

// Relaxed add (an arrival that publishes nothing); returns the old word.
__device__ __forceinline__ int atom_add_relaxed_gpu(int32_t *ptr, int v) {
  int old;
  asm volatile("atom.relaxed.gpu.global.add.s32 %0, [%1], %2;"
               : "=r"(old)
               : "l"(ptr), "r"(v)
               : "memory");
  return old;
}

// Waits (bounded) until `want` pieces are published on the counter word,
// with acquire semantics: their partial rows are then visible to this
// thread.  The pieces it waits for have arrived, so their CTAs are past
// their blocks and publish without waiting for anything.  On timeout it sets
// *abort, reports PA_DEVERR_WAIT_TIMEOUT and returns false.
__device__ __forceinline__ bool wait_published(const int32_t *ptr, int want, volatile int *abort,
                                               int32_t *err) {
  const long long t0 = clock64();
  while (published_count(ld_acquire_gpu(ptr)) < want) {
    if (*abort) return false;
    if (clock64() - t0 > kWaitTimeoutCycles) {
      *abort = 1;
      report(err, PA_DEVERR_WAIT_TIMEOUT);
      return false;
    }
    __nanosleep(32);
  }
  return true;
}

// ---- output writers ---------------------------------------------------------

__device__ __forceinline__ void store_out1(void *out, int out_f32, long long idx, float a) {
  if (out_f32)
    static_cast<float *>(out)[idx] = a;
  else
    static_cast<__nv_bfloat16 *>(out)[idx] = __float2bfloat16_rn(a);
}

__device__ __forceinline__ void store_out2(void *out, int out_f32, long long idx, float a,
                                           float b) {
  if (out_f32)
    *reinterpret_cast<float2 *>(static_cast<float *>(out) + idx) = make_float2(a, b);
  else
    *reinterpret_cast<uint32_t *>(static_cast<uint16_t *>(out) + idx) = float2_to_bf16x2(a, b);
}

__device__ __forceinline__ void store_out4(void *out, int out_f32, long long idx, float4 v) {
  if (out_f32) {
    *reinterpret_cast<float4 *>(static_cast<float *>(out) + idx) = v;
  } else {
    uint2 w;
    w.x = float2_to_bf16x2(v.x, v.y);
    w.y = float2_to_bf16x2(v.z, v.w);
    *reinterpret_cast<uint2 *>(static_cast<uint16_t *>(out) + idx) = w;
  }
}

// Log-sum-exp merge of one output row (sequence b, query head h) from the
// split-K partials of splits c0..c1 (slot 1 of c0, slot 0 of the others;
// partials are [slot][split][head][dim]),
// by one warp; lane l owns dims 4l..4l+3.  Partials are read through L2
// (written by other CTAs).  When N >= S every split holds at least one
// block; otherwise empty splits are skipped.  Each lane walks the pieces in
// split order with the same arithmetic as merge_sequence_bulk (weights
// e_i = exp(lse_i - M) summed in order, sum of e_i o_i in order, one scale
// by the reciprocal of the first sum), so the row has the same bits
// whichever path merges it.
__device__ __forceinline__ void merge_row(const float *part_o, const float *part_lse, void *out,
                                          int out_f32, long long out_row, int HQ, int h,
                                          long long c0, long long c1, long long S, long long N,
                                          int lane) {
  const bool dense = N >= S;
  auto piece = [&](long long cc) -> bool {
    return dense || cc == c0 || split_begin(cc, S, N) < split_begin(cc + 1, S, N);
  };
  auto row_of = [&](long long cc) -> long long { return ((cc == c0 ? 1 : 0) * S + cc) * HQ + h; };
  float M = -INFINITY;
  for (long long base = c0; base <= c1; base += 32) {
    const long long cc = base + lane;
    if (cc <= c1 && piece(cc)) M = fmaxf(M, __ldcg(part_lse + row_of(cc)));
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  // eight pieces' loads in flight at a time; the sums stay in split order
  float W = 0.f;
  for (long long base = c0; base <= c1; base += 8) {
    float lv[8];
#pragma unroll
    for (int u = 0; u < 8; ++u)
      lv[u] = base + u <= c1 && piece(base + u) ? __ldcg(part_lse + row_of(base + u)) : -INFINITY;
#pragma unroll
    for (int u = 0; u < 8; ++u)
      if (base + u <= c1 && piece(base + u)) W += lv[u] == -INFINITY ? 0.f : __expf(lv[u] - M);
  }
  const float inv = W > 0.f ? 1.f / W : 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (long long base = c0; base <= c1; base += 8) {
    float lv[8];
    float4 v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const bool in = base + u <= c1 && piece(base + u);
      lv[u] = in ? __ldcg(part_lse + row_of(base + u)) : -INFINITY;
      v[u] = in ? __ldcg(reinterpret_cast<const float4 *>(part_o + row_of(base + u) * kHeadDim) +
                         lane)
                : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      if (!(base + u <= c1 && piece(base + u))) continue;
      const float wi = lv[u] == -INFINITY ? 0.f : __expf(lv[u] - M);
      acc.x = fmaf(wi, v[u].x, acc.x);
      acc.y = fmaf(wi, v[u].y, acc.y);
      acc.z = fmaf(wi, v[u].z, acc.z);
      acc.w = fmaf(wi, v[u].w, acc.w);
    }
  }
  store_out4(out, out_f32, out_row * kHeadDim + lane * 4,
             make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv));
}

// Bulk copies of the partial rows of pieces i0 .. i1 - 1 of a sequence whose
// first split is c0 (piece i at row block i - i0 of `buf`), skipping piece
// own_i; with `lse`, also their lse values (piece i's HQ values at
// lse + i * HQ, own piece included: its entries are overwritten after the
// copies land).  One thread issues them; arms `mbar` with their bytes.
// Pieces 1 .. k - 1 are slot-0 rows of consecutive splits, so a run of them
// that skips the own piece is one copy (at most 32 KB each).
template <int HQ>
__device__ void issue_piece_copies(const DecodeParams &p, long long c0, long long S, int i0,
                                   int i1, int own_i, float *buf, float *lse, uint32_t mbar) {
  constexpr int ROW_FLOATS = HQ * kHeadDim;
  constexpr int RUN = (32 * 1024) / (ROW_FLOATS * 4) > 0 ? (32 * 1024) / (ROW_FLOATS * 4) : 1;
  auto row0 = [&](int i) -> long long { return ((i == 0 ? 1 : 0) * S + (c0 + i)) * HQ; };
  const bool own_in = own_i >= i0 && own_i < i1;
  uint32_t bytes = (uint32_t)((i1 - i0 - (own_in ? 1 : 0)) * ROW_FLOATS * 4);
  if (lse) bytes += (uint32_t)((i1 - i0) * HQ * 4);
  mbar_arrive_expect_tx(mbar, bytes);
  const uint64_t pol = l2_policy_evict_first();
  for (int i = i0; i < i1;) {
    if (i == own_i) {
      ++i;
      continue;
    }
    int j = i + 1;
    if (i > 0)
      while (j < i1 && j != own_i && j - i < RUN) ++j;
    bulk_load(smem_addr(buf + (long long)(i - i0) * ROW_FLOATS), p.part_o + row0(i) * kHeadDim,
              (uint32_t)((j - i) * ROW_FLOATS * 4), mbar, pol);
    i = j;
  }
  if (lse) {
    // piece i0 (slot 1 when i0 = 0), then pieces i0 + 1 .. i1 - 1 (slot 0, consecutive)
    bulk_load(smem_addr(lse + i0 * HQ), p.part_lse + row0(i0), HQ * 4, mbar, pol);
    if (i1 > i0 + 1)
      bulk_load(smem_addr(lse + (i0 + 1) * HQ), p.part_lse + row0(i0 + 1),
                (uint32_t)((i1 - i0 - 1) * HQ * 4), mbar, pol);
  }
}

// Log-sum-exp merge of all partials of sequence b by the NT threads
// (thread index ct, named barrier bar_id) of one CTA (needs every split of
// c0..c1 non-empty, N >= S, and k = c1 - c0 + 1 <= MAXP; else returns false
// having done nothing).  One round of loads brings every (piece, head) lse
// into `w`, where each head's terms e_i = exp(lse_i - M) and the reciprocal
// of their sum are formed.  The pieces' partial rows come into shared
// memory (`buf`, 16-byte aligned, `buf_bytes` long; piece i of a batch at
// row block i - i0) by bulk copies, as many pieces per batch as `buf` holds
// (all of them for the common few-piece case: one round trip).  Each thread
// keeps the weighted sums of its (head, 4 dims) items in registers across
// pieces and batches.  The piece of split c_own is read from own_o /
// own_lse (c_own = -1: every piece comes from the workspace).  With
// `prefetched`, every other piece's rows and all lse values were already
// requested by issue_piece_copies into buf / w on `mbar` (phase 0, one
// batch): the merge only waits for them.
template <int HQ, int MAXP, int NT>
__device__ bool merge_sequence_bulk(const DecodeParams &p, int b, long long c0, long long c1,
                                    long long S, long long N, float *w, int ct, int bar_id,
                                    long long c_own, const float *own_o, const float *own_lse,
                                    float *buf, long long buf_bytes, uint32_t mbar,
                                    volatile int *abort_flag, bool prefetched = false) {
  constexpr int ROW_FLOATS = HQ * kHeadDim;  // one piece: HQ rows of o
  constexpr int ITEMS = HQ * (kHeadDim / 4);
  constexpr int IPT = (ITEMS + NT - 1) / NT;  // items per thread
  // many items per thread (a one-warp merge): items outer; when the pieces
  // take several batches, the running sums wait in the last row block of buf
  constexpr bool ITEMS_OUTER = IPT > 4;
  const long long k = c1 - c0 + 1;
  long long per_batch = buf_bytes / (ROW_FLOATS * 4);
  if (ITEMS_OUTER && per_batch < k) --per_batch;  // one row block for the sums
  if (N < S || k > MAXP || per_batch < 1 || (prefetched && per_batch < k)) return false;
  const int kk = (int)k, kb = (int)(per_batch < k ? per_batch : k);
  const int own_i = (int)(c_own - c0);  // outside [0, kk) when c_own = -1
  if (prefetched) {
    // the rows and lse values are (being) copied in; the own piece's lse
    // entries are written once the copies have landed
    __all_sync(0xffffffffu, mbar_wait(mbar, 0, abort_flag, p.err));
    if (own_i >= 0 && own_i < kk)
      for (int h = ct; h < HQ; h += NT) w[own_i * HQ + h] = own_lse[h];
  } else {
    if (ct == 0) {
      // the ring was last read through the generic proxy, and the partials
      // were acquired through it; the copies go through the async proxy
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      asm volatile("fence.proxy.async.global;" ::: "memory");
      issue_piece_copies<HQ>(p, c0, S, 0, kb, own_i, buf, nullptr, mbar);
    }
    for (int e = ct; e < kk * HQ; e += NT)
      w[e] = e / HQ == own_i ? own_lse[e % HQ]
                             : __ldcg(p.part_lse + ((e < HQ ? 1 : 0) * S + c0 + e / HQ) * HQ +
                                      e % HQ);
  }
  named_barrier(bar_id, NT);
  // per head: e_i = exp(lse_i - M) in w (summed in split order) and the
  // reciprocal of the sum in winv; up to 16 pieces in registers
  float *winv = w + kk * HQ;
  for (int h = ct; h < HQ; h += NT) {
    float W = 0.f;
    if (kk <= 16) {
      float lv[16];
      float M = -INFINITY;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        lv[i] = i < kk ? w[i * HQ + h] : -INFINITY;
        M = fmaxf(M, lv[i]);
      }
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        if (i < kk) {
          const float e = lv[i] == -INFINITY ? 0.f : __expf(lv[i] - M);
          w[i * HQ + h] = e;
          W += e;
        }
      }
    } else {
      float M = -INFINITY;
      for (int i = 0; i < kk; ++i) M = fmaxf(M, w[i * HQ + h]);
      for (int i = 0; i < kk; ++i) {
        const float lse = w[i * HQ + h];
        const float e = lse == -INFINITY ? 0.f : __expf(lse - M);
        w[i * HQ + h] = e;
        W += e;
      }
    }
    winv[h] = W > 0.f ? 1.f / W : 0.f;
  }
  named_barrier(bar_id, NT);
  if constexpr (ITEMS_OUTER) {
    // each thread's items in turn, the pieces of the batch in split order;
    // between batches an item's running sum waits in `sums` (its own slot:
    // no other thread reads it)
    float4 *sums = reinterpret_cast<float4 *>(buf + (long long)kb * ROW_FLOATS);
    for (int i0 = 0, batch = 0; i0 < kk; i0 += kb, ++batch) {
      if (!prefetched) __all_sync(0xffffffffu, mbar_wait(mbar, batch & 1, abort_flag, p.err));
      const int i1 = i0 + kb < kk ? i0 + kb : kk;
      for (int item = ct; item < ITEMS; item += NT) {
        const int h = item / (kHeadDim / 4), d = (item % (kHeadDim / 4)) * 4;
        float4 a = i0 == 0 ? make_float4(0.f, 0.f, 0.f, 0.f) : sums[item];
        for (int i = i0; i < i1; ++i) {
          const float *rowp = i == own_i ? own_o : buf + (long long)(i - i0) * ROW_FLOATS;
          const float wi = w[i * HQ + h];
          const float4 v = *reinterpret_cast<const float4 *>(rowp + h * kHeadDim + d);
          a.x = fmaf(wi, v.x, a.x);
          a.y = fmaf(wi, v.y, a.y);
          a.z = fmaf(wi, v.z, a.z);
          a.w = fmaf(wi, v.w, a.w);
        }
        if (i1 < kk) {
          sums[item] = a;
        } else {
          const float inv = winv[h];
          store_out4(p.out, p.out_f32, ((long long)b * HQ + h) * kHeadDim + d,
                     make_float4(a.x * inv, a.y * inv, a.z * inv, a.w * inv));
        }
      }
      if (i1 < kk) {
        // the next batch reuses the rows once every thread is done with them
        named_barrier(bar_id, NT);
        if (ct == 0) {
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          const int i2 = i1 + kb < kk ? i1 + kb : kk;
          issue_piece_copies<HQ>(p, c0, S, i1, i2, own_i, buf, nullptr, mbar);
        }
      }
    }
    return true;
  }
  // this thread's items: head and dim offset of each
  int hh[IPT], dd[IPT];
#pragma unroll
  for (int t = 0; t < IPT; ++t) {
    const int item = ct + t * NT;
    hh[t] = item < ITEMS ? item / (kHeadDim / 4) : 0;
    dd[t] = (item % (kHeadDim / 4)) * 4;
  }
  float4 acc[IPT];
#pragma unroll
  for (int t = 0; t < IPT; ++t) acc[t] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int i0 = 0, batch = 0; i0 < kk; i0 += kb, ++batch) {
    // every thread waits for the batch (warp-uniform; bounded)
    if (!prefetched) __all_sync(0xffffffffu, mbar_wait(mbar, batch & 1, abort_flag, p.err));
    const int i1 = i0 + kb < kk ? i0 + kb : kk;
    // pieces in split order whichever CTA merges: the sums are the same
    // bits run to run (merge_row keeps the same order and arithmetic)
#pragma unroll 2
    for (int i = i0; i < i1; ++i) {
      const float *rowp = i == own_i ? own_o : buf + (long long)(i - i0) * ROW_FLOATS;
#pragma unroll
      for (int t = 0; t < IPT; ++t) {
        if (ct + t * NT < ITEMS) {
          const float wi = w[i * HQ + hh[t]];
          const float4 v = *reinterpret_cast<const float4 *>(rowp + hh[t] * kHeadDim + dd[t]);
          acc[t].x = fmaf(wi, v.x, acc[t].x);
          acc[t].y = fmaf(wi, v.y, acc[t].y);
          acc[t].z = fmaf(wi, v.z, acc[t].z);
          acc[t].w = fmaf(wi, v.w, acc[t].w);
        }
      }
    }
    if (i1 < kk) {
      // the next batch reuses the buffer once every thread is done with it
      named_barrier(bar_id, NT);
      if (ct == 0) {
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        const int i2 = i1 + kb < kk ? i1 + kb : kk;
        issue_piece_copies<HQ>(p, c0, S, i1, i2, own_i, buf, nullptr, mbar);
      }
    }
  }
#pragma unroll
  for (int t = 0; t < IPT; ++t) {
    if (ct + t * NT < ITEMS) {
      const float inv = winv[hh[t]];
      store_out4(p.out, p.out_f32, ((long long)b * HQ + hh[t]) * kHeadDim + dd[t],
                 make_float4(acc[t].x * inv, acc[t].y * inv, acc[t].z * inv, acc[t].w * inv));
    }
  }
  return true;
}

// SPLIT_MERGE: cut pieces only write their partials; merge_kernel, launched
// behind this kernel, merges them (no counters, no merges in this kernel).
template <int G, int HKV, bool F8 = false, bool ROPE = false, bool SPLIT_MERGE = false>
__global__ void __launch_bounds__(kDecodeThreads, 1)
    decode_kernel(const __grid_constant__ CUtensorMap tmap_k,
                  const __grid_constant__ CUtensorMap tmap_v, const DecodeParams p) {
  using S = DecodeShape<G, HKV, F8, ROPE>;
  extern __shared__ uint8_t smem_raw[];
  // realign to 1024 bytes: the 128-byte swizzle pattern repeats every 1 KB
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  float *red = reinterpret_cast<float *>(smem + S::NST * S::STAGE_BYTES);
  float *mw = reinterpret_cast<float *>(smem + S::NST * S::STAGE_BYTES + S::RED_BYTES);
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + S::NST * S::STAGE_BYTES + S::RED_BYTES +
                                                S::MERGE_BYTES);
  uint64_t *empty = full + S::NST;
  DecodeCtl *ctl = reinterpret_cast<DecodeCtl *>(empty + S::NST);
  float *eww = reinterpret_cast<float *>(reinterpret_cast<uint8_t *>(ctl) + S::CTL_BYTES);
  volatile int *abort_flag = &ctl->abort;

  const int tid = threadIdx.x;
  // broadcast from lane 0: the compiler then knows every role branch below
  // is warp-uniform
  const int warp = __shfl_sync(0xffffffffu, tid >> 5, 0);
  const int lane = tid & 31;
  const long long nsplit = p.num_splits;
  const long long c = blockIdx.x;

  // ---- 1. block counts of all sequences: the total N, this CTA's block range
  //         [lo, hi) and the sequence that holds block lo.  One block-wide
  //         inclusive scan over the counts gives both when the batch fits one
  //         pass (one round of context-length loads, two barriers); larger
  //         batches take a pass for N, then a pass for the search.
  __shared__ long long warp_tot[kDecodeWarps];
  if (tid == 0) {
    ctl->first_b = -1;
    ctl->first_prefix = 0;
    ctl->abort = 0;
    ctl->last = 0;
  }
  long long N = 0;
  {
    const int nw = (int)(blockDim.x >> 5);
    long long running = 0;
    for (int base = 0; base < p.batch; base += blockDim.x) {
      const int b = base + tid;
      const int n = b < p.batch ? seq_blocks(p.context_lens, b) : 0;
      long long incl = n;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const long long y = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += y;
      }
      if (lane == 31) warp_tot[warp] = incl;
      __syncthreads();
      long long before = running, chunk_total = 0;
      for (int w = 0; w < nw; ++w) {
        const long long t = warp_tot[w];
        if (w < warp) before += t;
        chunk_total += t;
      }
      running += chunk_total;
      if (base + (int)blockDim.x >= p.batch) {
        // last pass: N is known, and (one-pass batches) so is this
        // sequence's first block
        N = running;
        if (base == 0 && b < p.batch && n > 0) {
          const long long lo1 = split_begin(c, nsplit, N), hi1 = split_begin(c + 1, nsplit, N);
          const long long prefix = before + incl - n;
          if (prefix <= lo1 && lo1 < prefix + n && lo1 < hi1) {
            ctl->first_b = b;
            ctl->first_prefix = prefix;
          }
        }
      }
      __syncthreads();
    }
  }
  const long long lo = N ? split_begin(c, nsplit, N) : 0;
  const long long hi = N ? split_begin(c + 1, nsplit, N) : 0;
  if (p.batch > (int)blockDim.x) {
    // second pass over the prefix sums (batches larger than one pass)
    long long running = 0;
    for (int base = 0; base < p.batch; base += blockDim.x) {
      const int b = base + tid;
      const int n = b < p.batch ? seq_blocks(p.context_lens, b) : 0;
      long long incl = n;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const long long y = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += y;
      }
      if (lane == 31) warp_tot[warp] = incl;
      __syncthreads();
      long long before = running, chunk_total = 0;
      for (int w = 0; w < (int)(blockDim.x >> 5); ++w) {
        const long long t = warp_tot[w];
        if (w < warp) before += t;
        chunk_total += t;
      }
      const long long prefix = before + incl - n;  // global index of block 0 of b
      if (b < p.batch && n > 0 && prefix <= lo && lo < prefix + n && lo < hi) {
        ctl->first_b = b;
        ctl->first_prefix = prefix;
      }
      running += chunk_total;
      __syncthreads();
    }
  }
  // ---- 2b. Under a programmatic dependent launch the previous kernel in the
  //          stream may still be running.  Context lengths and block tables
  //          may be read before the wait for it; so may the K/V pages of the
  //          first ring stages when p.early_kv is set.  q, the new rows, the
  //          workspace and every write come after it.  Each thread lets the
  //          next kernel begin only once it has passed that wait
  //          (wait_prev_then_release), so a kernel that starts early behind
  //          this one finds every kernel before this one complete.
  // rows of empty sequences: sequence b is zeroed by CTA b mod S, by threads
  // t0, t0 + nt, ...
  auto zero_empty_rows = [&](int t0, int nt) {
    for (long long b = c; b < p.batch; b += nsplit)
      if (__ldg(p.context_lens + b) <= 0)
        for (int i = 2 * t0; i < S::HQ * kHeadDim; i += 2 * nt)
          store_out2(p.out, p.out_f32, b * S::HQ * kHeadDim + i, 0.f, 0.f);
  };
  if (lo >= hi || ctl->first_b < 0) {
    // no block for this CTA (N < S), or inconsistent input (never walk from
    // b = -1): only the empty rows and the error bit remain
    wait_prev_then_release();
    zero_empty_rows(tid, blockDim.x);
    if (lo < hi && tid == 0) report(p.err, PA_DEVERR_SHAPE);
    return;
  }

  // ---- 3. pipeline barriers -------------------------------------------------
  const uint32_t stage0 = smem_addr(smem);
  const uint32_t full0 = smem_addr(full);
  const uint32_t empty0 = smem_addr(empty);
  if (tid == 0) {
    for (int i = 0; i < S::NST; ++i) {
      mbar_init(full0 + 8 * i, 1);
      mbar_init(empty0 + 8 * i, HKV);  // the Hkv consumer warps of the slot's phase
    }
    for (int k = 0; k < 2; ++k) {
      mbar_init(smem_addr(&ctl->red_full[k]), S::CW);
      mbar_init(smem_addr(&ctl->red_empty[k]), 1);
    }
    mbar_init(smem_addr(&ctl->merge_bar), 1);
    mbar_init(smem_addr(&ctl->merge_bar2), 1);
    mbar_init(smem_addr(&ctl->ew_done), 1);
    mbar_init(smem_addr(&ctl->seen_bar), 1);
    mbar_init(smem_addr(&ctl->pf_bar), 1);
    mbar_init(smem_addr(&ctl->pub_done), 1);
    ctl->def_pending = 0;
    ctl->fin_valid = 0;
    ctl->pf_ready = 0;
    ctl->decided = 0;
    fence_barrier_init();
  }
  __syncthreads();
  const int first_b = ctl->first_b;
  const long long first_prefix = ctl->first_prefix;

  if (warp < kDecodeProducerWarps) {
    // ---- 4. producer warps: block descriptors 32 at a time; warp pw issues
    //         the stages with index = pw (mod 2), lane 0 of it issuing ----
    const int pw = warp;
    if (lane == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_k))
                   : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_v))
                   : "memory");
    }
    const uint64_t pol_kv = l2_policy_evict_first();
    const uint64_t pol_q = l2_policy_evict_last();
    // the q base in a register before the wait (the copies after it are on
    // the critical path of the first stage)
    const uint16_t *q_base;
    asm volatile("mov.b64 %0, %1;" : "=l"(q_base) : "l"(p.q));
    // The K and V pages of physical block ph into ring slot st, completing
    // on the slot's full barrier (warp-uniform arguments; nothing for an
    // entry outside the pool, which the caller reports).  arm: lane 0 first
    // adds the pages' bytes to the barrier's expected count, without arriving.
    auto issue_kv_stage = [&](int st, long long ph, bool arm) {
      if (!(ph >= 0 && ph < p.num_blocks)) return;
      const uint32_t dst = stage0 + st * S::STAGE_BYTES;
      const uint32_t bar = full0 + 8 * st;
      if (arm) {
        if (lane == 0) mbar_expect_tx(bar, 2u * S::KV_BYTES);
        __syncwarp();
      }
      const int z = (int)(ph * kBlockSize);
      if constexpr (F8) {
        // K: (128 dims, head, slot) box of each head pair, 128-byte
        // swizzle; V: the block's dim-major page is one contiguous run
        // (Hkv x 2 KB): one bulk copy (a tensor box would move 16-byte rows)
#pragma unroll
        for (int pr = 0; pr < S::NPAIR; ++pr)
          tma_load_box(dst + pr * S::BOX_BYTES, &tmap_k, 0, pr * S::HB, z, bar, pol_kv);
        bulk_load_elect(dst + S::KV_BYTES, p.v_pool + ph * S::KV_BYTES, S::KV_BYTES, bar,
                        pol_kv);
      } else {
#pragma unroll
        for (int pr = 0; pr < S::NPAIR; ++pr) {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const uint32_t off = (pr * 2 + h) * S::BOX_BYTES;
            tma_load_box(dst + off, &tmap_k, h * 64, pr * S::HB, z, bar, pol_kv);
            tma_load_box(dst + S::KV_BYTES + off, &tmap_v, h * 64, pr * S::HB, z, bar, pol_kv);
          }
        }
      }
    };
    int b = first_b;
    int ctx = __ldg(p.context_lens + b);
    int j = (int)(lo - first_prefix);
    long long gb = lo, issued = 0;
    bool stop = false;
    bool waited = false;
    while (gb < hi && !stop) {
      int lb, lj, lctx;
      const int count = walk_chunk(p.context_lens, p.batch, b, ctx, j, hi - gb, lane, lb, lj, lctx);
      if (count == 0) {
        wait_prev_then_release();
        if (lane == 0) report(p.err, PA_DEVERR_SHAPE);
        break;
      }
      // all block-table entries of the chunk in one round of loads
      const bool in_row = lane < count && lj < p.bt_stride;
      const long long phys = in_row ? __ldg(p.block_tables + (long long)lb * p.bt_stride + lj) : -1;
      int n_early = 0;  // stages of this chunk whose K/V pages went out before the wait
      if (!waited) {
        // the first chunk's descriptors are ready.  With p.early_kv the K/V
        // pages of the first ring stages go out now (issued == 0 here, so
        // stage i of the chunk is ring slot i and needs no empty wait): lane
        // 0 raises the slot's expected bytes without arriving, so the stage
        // cannot complete before its arrival (with the q copy) below.  The
        // rest waits for the previous kernel, which may write q, the new
        // rows and the workspace.
        if (p.early_kv) {
          n_early = min(count, min(S::NST, kDecodeEarlyStages));
          for (int i = pw; i < n_early; i += kDecodeProducerWarps)
            issue_kv_stage(i, __shfl_sync(0xffffffffu, phys, i), true);
        }
        wait_prev_then_release();
        waited = true;
      }
      // the q rows go with the first NPH stages of every piece: each consumer
      // warp reads them from its own first stage of the piece
      const bool with_q = min(gb + lane - lo, (long long)lj) < S::NPH;
      for (int i = 0; i < count; ++i, ++issued) {
        if ((int)(issued % kDecodeProducerWarps) != pw) continue;
        const int st = (int)(issued % S::NST);
        const int round = (int)(issued / S::NST);
        if (round > 0 &&
            !__all_sync(0xffffffffu,
                        mbar_wait(empty0 + 8 * st, (round - 1) & 1, abort_flag, p.err))) {
          stop = true;
          break;
        }
        const long long ph_i = __shfl_sync(0xffffffffu, phys, i);
        const int b_i = __shfl_sync(0xffffffffu, lb, i);
        const bool q_i = __shfl_sync(0xffffffffu, with_q ? 1 : 0, i) != 0;
        const bool row_i = __shfl_sync(0xffffffffu, in_row ? 1 : 0, i) != 0;
        // every value here is warp-uniform (shuffled from lane i); lane 0
        // arms the barrier, then the warp issues the copies (elect.sync)
        const bool ok = ph_i >= 0 && ph_i < p.num_blocks;
        const uint32_t dst = stage0 + st * S::STAGE_BYTES;
        const uint32_t bar = full0 + 8 * st;
        const bool pre = i < n_early;  // K/V already requested and counted
        if (lane == 0) {
          mbar_arrive_expect_tx(bar, (ok && !pre ? 2u * S::KV_BYTES : 0u) +
                                         (q_i ? S::Q_BYTES + S::ROPE_BYTES : 0u));
          // a context longer than the table row (caller error) or an entry
          // outside the pool: reported, not read
          if (!ok) report(p.err, row_i ? PA_DEVERR_BLOCK_INDEX : PA_DEVERR_SHAPE);
        }
        __syncwarp();
        if (!pre) issue_kv_stage(st, ph_i, false);
        if (q_i) {
          bulk_load_elect(dst + 2 * S::KV_BYTES, q_base + (long long)b_i * S::HQ * kHeadDim,
                          S::Q_BYTES, bar, pol_q);
          if constexpr (ROPE) {
            // the cos and sin rows of the new token's position (row 0 for a
            // position outside the tables: reported, and the new row is
            // then neither stored nor patched)
            long long pos = __ldg(p.positions + b_i);
            if (pos < 0 || pos >= p.max_position) {
              if (lane == 0) report(p.err, PA_DEVERR_POSITION);
              pos = 0;
            }
            const uint32_t rd = dst + 2 * S::KV_BYTES + S::Q_BYTES;
            bulk_load_elect(rd, p.cos_table + pos * (kHeadDim / 2), S::ROPE_BYTES / 2, bar, pol_q);
            bulk_load_elect(rd + S::ROPE_BYTES / 2, p.sin_table + pos * (kHeadDim / 2),
                            S::ROPE_BYTES / 2, bar, pol_q);
          }
        }
      }
      gb += count;
    }
    if (lane == 0 && *abort_flag) {
      // Drain: copies this warp still has in flight must land before the
      // CTA's shared memory is released.  Bounded, independent of the abort
      // flag.
      volatile int never = 0;
      const long long from = issued > S::NST ? issued - S::NST : 0;
      for (long long i = from; i < issued; ++i)
        if ((int)(i % kDecodeProducerWarps) == pw)
          mbar_wait(full0 + 8 * (int)(i % S::NST), (int)((i / S::NST) & 1), &never, nullptr);
    }
    return;
  }

  if (warp == kDecodeEpilogueWarp) {
    // ---- 5a. epilogue warp: takes every piece that ends before the CTA's
    //          final one, in order, from red buffer (piece index mod 2).  With
    //          several warps per kv head it combines their rows and writes
    //          the output rows (whole sequence) or the partial (cut piece);
    //          with one warp per kv head the consumers wrote the rows already.
    //          A cut piece arrives on its sequence's counter when the warp
    //          takes it, before the combine, and publishes its rows after
    //          writing them, unless it arrived last: then its CTA owes the
    //          merge.  The consumers never wait for this, except to reuse a
    //          buffer two pieces later.
    wait_prev_then_release();
    zero_empty_rows(lane, 32);
    // While it waits for the next piece, lane 0 watches the arrival counter
    // of the CTA's final piece (once the consumers have named it): when every
    // other piece of that sequence has arrived it completes seen_bar, and the
    // consumers merge at once, without publishing their own piece.  Before
    // it does, it requests the other pieces' partials (rows and lse) into the
    // red buffer nobody uses any more, when they fit (pf_ready), so that the
    // consumers' merge finds them in shared memory.
    int snoop = 0;  // 0: final piece not named yet, 1: watching, 2: done
    long long fin_cs0 = 0, fin_cs1 = 0;
    int fin_pieces = 0;
    bool pf_issued = false;
    // lane 0: every other piece of the final one has arrived?  Then (with
    // room) request their partials into free_buf, and complete seen_bar.
    auto snoop_final = [&](float *free_buf) {
      if (snoop == 0) {
        if (!*reinterpret_cast<volatile int *>(&ctl->fin_valid)) return;
        __threadfence_block();
        fin_cs0 = ctl->fin_cs0;
        fin_cs1 = ctl->fin_cs1;
        fin_pieces = ctl->fin_pieces;
        snoop = 1;
      }
      int cw_word = 0;
      if (snoop == 1 && arrived_count(cw_word = ld_acquire_gpu(p.counters + fin_cs1)) ==
                            fin_pieces - 1 &&
          published_count(cw_word) == fin_pieces - 1) {
        if constexpr (S::PF_PIECES > 0 && S::PF_LSE_COPY) {
          if (free_buf != nullptr && fin_pieces <= S::PF_PIECES && N >= nsplit &&
              !*reinterpret_cast<volatile int *>(&ctl->def_pending)) {
            asm volatile("fence.proxy.async.global;" ::: "memory");
            issue_piece_copies<S::HQ>(p, fin_cs0, nsplit, 0, fin_pieces, (int)(c - fin_cs0),
                                      free_buf, mw + S::PF_W, smem_addr(&ctl->pf_bar));
            *reinterpret_cast<volatile int *>(&ctl->pf_ready) = 1;
            pf_issued = true;
          }
        }
        mbar_arrive(smem_addr(&ctl->seen_bar));
        snoop = 2;
      }
    };
    auto wait_full = [&](uint32_t bar, int parity, float *free_buf, int npe) -> bool {
      const long long t0 = clock64();
      while (true) {
        int done = lane == 0 ? (int)mbar_test_wait(bar, parity) : 0;
        // waiting for the final piece itself (named, and handed over after
        // npe others): free_buf, the previous piece's buffer, is free for
        // good (a non-final piece may still be in the consumers' hands when
        // the final one is named)
        int fin = 0;
        if (lane == 0 && *reinterpret_cast<volatile int *>(&ctl->fin_valid)) {
          __threadfence_block();
          fin = ctl->fin_npe == npe;
        }
        fin = __shfl_sync(0xffffffffu, fin, 0);
        if (lane == 0 && !done && snoop < 2) snoop_final(fin ? free_buf : nullptr);
        if (__shfl_sync(0xffffffffu, done, 0)) {
          __syncwarp();  // the other lanes are ordered after lane 0's observation
          return true;
        }
        if (*abort_flag) return false;
        if (clock64() - t0 > kWaitTimeoutCycles) {
          if (lane == 0) {
            *abort_flag = 1;
            report(p.err, PA_DEVERR_WAIT_TIMEOUT);
          }
          return false;
        }
        __nanosleep(256);
      }
    };
    for (int npe = 0;; ++npe) {
      const int k = npe & 1;
      // the buffer of the previous piece: once this warp waits for the final
      // piece, nobody writes it again
      float *const other_buf = S::NPH > 1 ? red + (k ^ 1) * S::RED_ONE_FLOATS : nullptr;
      const bool got = wait_full(smem_addr(&ctl->red_full[k]), (npe >> 1) & 1, other_buf, npe);
      const PieceDesc d = ctl->desc[k];
      if (!got || d.kind == kPieceEnd) {
        // every piece handed to this warp is published, and a merge it owes
        // is recorded (def_pending)
        if (lane == 0) mbar_arrive(smem_addr(&ctl->pub_done));
        // The end mark comes when the final piece's blocks are done.  While
        // the consumers combine that piece, lane 0 goes on watching its
        // counter until they decide how the piece ends (bounded; giving up
        // only loses the shortcut).
        if (got && lane == 0) {
          const long long t0 = clock64();
          while (snoop < 2 && !*reinterpret_cast<volatile int *>(&ctl->decided) &&
                 !*abort_flag && clock64() - t0 < kWaitTimeoutCycles) {
            // named before the end mark, or never: a whole final piece
            if (snoop == 0 && !*reinterpret_cast<volatile int *>(&ctl->fin_valid)) break;
            snoop_final(other_buf);
            if (snoop < 2) __nanosleep(64);
          }
        }
        // Copies this warp requested land before it signs off (bounded).
        if (lane == 0 && pf_issued) {
          volatile int never = 0;
          mbar_wait(smem_addr(&ctl->pf_bar), 0, &never, nullptr);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&ctl->ew_done));
        return;
      }
      // a cut piece arrives now, before the combine (relaxed: it publishes
      // its rows after writing them), so that its arrival is not late
      int early_word = 0;
      if (!SPLIT_MERGE && d.kind == kPieceCut && lane == 0)
        early_word = atom_add_relaxed_gpu(p.counters + d.cs1, kArrive);
      if constexpr (S::NPH > 1) {
        const float *rk = red + k * S::RED_ONE_FLOATS;
        // per query head: the normalised weight of each of its NPH warps
        for (int qh = lane; qh < S::HQ; qh += 32) {
          const int gh = qh / G, h = qh % G;
          float mk[S::NPH], M = -INFINITY;
#pragma unroll
          for (int w = 0; w < S::NPH; ++w) {
            mk[w] = rk[((gh + w * HKV) * G + h) * S::RED_FLOATS_PER_HEAD + S::RED_M];
            M = fmaxf(M, mk[w]);
          }
          float L = 0.f;
#pragma unroll
          for (int w = 0; w < S::NPH; ++w) {
            mk[w] = mk[w] == -INFINITY ? 0.f : exp2f(mk[w] - M);
            L += rk[((gh + w * HKV) * G + h) * S::RED_FLOATS_PER_HEAD + S::RED_L] * mk[w];
          }
          const float inv = L > 0.f ? 1.f / L : 0.f;
#pragma unroll
          for (int w = 0; w < S::NPH; ++w) eww[w * S::HQ + qh] = mk[w] * inv;
          if (d.kind == kPieceCut)
            p.part_lse[d.slot_row + qh] =
                L > 0.f ? (M + __log2f(L)) * 0.69314718055994531f : -INFINITY;
        }
        __syncwarp();
        for (int item = lane; item < S::HQ * (kHeadDim / 4); item += 32) {
          const int qh = item / (kHeadDim / 4);
          const int dd = (item % (kHeadDim / 4)) * 4;
          const int gh = qh / G, h = qh % G;
          float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
          for (int w = 0; w < S::NPH; ++w) {
            const float wk = eww[w * S::HQ + qh];
            const float4 v = *reinterpret_cast<const float4 *>(
                rk + ((gh + w * HKV) * G + h) * S::RED_FLOATS_PER_HEAD + dd);
            acc.x += wk * v.x;
            acc.y += wk * v.y;
            acc.z += wk * v.z;
            acc.w += wk * v.w;
          }
          if (d.kind == kPieceWhole)
            store_out4(p.out, p.out_f32, ((long long)d.b * S::HQ + qh) * kHeadDim + dd, acc);
          else
            *reinterpret_cast<float4 *>(p.part_o + (d.slot_row + qh) * kHeadDim + dd) = acc;
        }
        __syncwarp();
      }
      if (lane == 0) mbar_arrive(smem_addr(&ctl->red_empty[k]));  // buffer k is free again
      if (!SPLIT_MERGE && d.kind == kPieceCut) {
        int last = 0;
        if (lane == 0) {
          // release: the partial rows (this warp's, or the consumers' that
          // the red_full barrier ordered before) precede the arrival, which
          // publishes them too
          last = arrived_count(early_word) == d.pieces - 1;
          if (!last) atom_add_release_gpu(p.counters + d.cs1, kPublish);
        }
        if (lane == 0 && last) {
          // arrived last: its own rows stay unpublished (this CTA merges);
          // wait (acquire) until every other piece is published and leave
          // the merge to the consumer warps
          asm volatile("fence.proxy.async.global;" ::: "memory");
          wait_published(p.counters + d.cs1, d.pieces - 1, abort_flag, p.err);
          ctl->def_b = d.b;
          ctl->def_cs0 = d.cs0;
          ctl->def_cs1 = d.cs1;
          ctl->def_pending = 1;
        }
        __syncwarp();
      }
    }
  }

  // ---- 5b. consumers ----------------------------------------------------------
  const int cw = warp - kDecodeFirstConsumerWarp;  // consumer warp 0..CW-1
  const int ct = tid - 32 * kDecodeFirstConsumerWarp;  // consumer thread index
  // The first chunk's walk reads only context lengths, so it comes before
  // the wait for the previous kernel (taken inside the loop, after the first
  // walk): after the wait every global load misses the SM's caches, and the
  // walk's loads would otherwise be dependent round trips between the wait
  // and the first stage.  (The rows of empty sequences are the epilogue
  // warp's.)
  int wb = first_b;
  int wctx = __ldg(p.context_lens + wb);
  int wj = (int)(lo - first_prefix);
  bool cons_waited = false;
  const int g = cw % HKV;     // kv head of this warp
  const int ph = cw / HKV;    // stage phase of this warp
  const int gid = lane >> 2;  // fragment row group
  const int qd = lane & 3;    // fragment column pair
  // this warp's kv head inside the TMA boxes: box group, row offset
  const int gpair = g / S::HB, gsub = g % S::HB;
  // F8: the K scale of this kv head folds into the score scale, the V scale
  // into the rows at each piece end (codes widen exactly, so the products
  // equal those of the widened values)
  // (F8: the scales are read after the wait, below)
  float cl2 = p.qk_scale_log2;
  float vsc = 1.f;
  // F8: the 16 score rows of an MMA are the tokens tperm(r), so that a
  // thread's two token pairs of the PV operand are 4 consecutive bytes of
  // a dim-major V row: rows 2i, 2i + 1 -> tokens 4i, 4i + 1 and rows
  // 8 + 2i, 9 + 2i -> tokens 4i + 2, 4i + 3 (any order of the tokens gives
  // the same sums; the same order is used for K, the mask and V)
  const int tok0 = F8 ? (((gid >> 1) << 2) | (gid & 1)) : gid;           // row gid
  const int tok1 = F8 ? (((gid >> 1) << 2) | 2 | (gid & 1)) : gid + 8;   // row gid + 8

  uint32_t qf[8][2];  // Q^T fragments of the group, per 16-dim k-step
  float o[8][4];      // O^T rows 16 mt + {gid, gid + 8}, head columns 2 qd, 2 qd + 1
  // m0, m1: reference max of the scaled scores (base 2), heads 2qd, 2qd + 1.
  // It moves only when a block's max exceeds it by more than 8, so the
  // exponentials stay <= 256 and o, l are rescaled rarely.
  float m0 = -INFINITY, m1 = -INFINITY;
  float l0 = 0.f, l1 = 0.f;              // running sum over this lane's tokens
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) qf[ks][0] = qf[ks][1] = 0u;
#pragma unroll
  for (int mt = 0; mt < 8; ++mt)
#pragma unroll
    for (int i = 0; i < 4; ++i) o[mt][i] = 0.f;

  int npieces = 0;  // pieces ended so far (every consumer warp counts the same)
  bool def_done = false;  // an owed merge was handled with the final piece's
  bool no_final = false;  // the block walk stopped early (inconsistent input)
  // consumer thread 0: the current piece's split words are in ctl
  bool pc_done = false;
  auto piece_splits = [&](long long gb, int j, int n) {
    const long long P = gb - j;  // global index of block 0 of the sequence
    const long long cs0 = split_of_block(P, nsplit, N);
    const long long cs1 = split_of_block(P + n - 1, nsplit, N);
    long long pieces = cs1 - cs0 + 1;
    if (N < nsplit) {
      pieces = 1;
      for (long long cc = cs0 + 1; cc <= cs1; ++cc)
        pieces += split_begin(cc, nsplit, N) < split_begin(cc + 1, nsplit, N) ? 1 : 0;
    }
    ctl->pc_cs0 = cs0;
    ctl->pc_cs1 = cs1;
    ctl->pc_pieces = (int)pieces;
    pc_done = true;
    const long long last_blk = P + n - 1;
    if (last_blk >= hi - 1 && (P < lo || last_blk > hi - 1) && N >= nsplit &&
        pieces <= S::MERGE_MAX_PIECES) {
      // the CTA's final piece, cut (and mergeable from shared memory): the
      // epilogue warp watches its sequence's arrival counter meanwhile
      ctl->fin_cs0 = cs0;
      ctl->fin_cs1 = cs1;
      ctl->fin_pieces = (int)pieces;
      ctl->fin_npe = npieces;
      __threadfence_block();
      *reinterpret_cast<volatile int *>(&ctl->fin_valid) = 1;
    }
  };
  bool need_q = true;  // the q rows of the current piece are not loaded yet
  long long it0 = 0;  // stage index of the chunk's first block
  for (long long gb0 = lo; gb0 < hi;) {
    // the next (up to) 32 blocks: lane L describes block gb0 + L
    int lb = 0, lj = 0, lctx = 0;
    const int count =
        walk_chunk(p.context_lens, p.batch, wb, wctx, wj, hi - gb0, lane, lb, lj, lctx);
    if (!cons_waited) {
      // the first chunk is walked: now wait for the previous kernel, then
      // read the FP8 scales
      cons_waited = true;
      wait_prev_then_release();
      if constexpr (F8) {
        cl2 *= __ldg(p.k_scale + g);
        vsc = __ldg(p.v_scale + g);
      }
    }
    if (count == 0) {
      // same decision in every consumer warp and the producer; no final
      // piece follows: the epilogue warp gets its end mark at the consumers'
      // end
      no_final = true;
      break;
    }
    // A warp visits only the blocks that concern it: its own stages (index
    // = ph mod NPH) and every piece end (all warps combine there).
    const bool in_chunk = lane < count;
    const int lnb = ceil_div_blocks(lctx);
    const unsigned m_last =
        __ballot_sync(0xffffffffu, in_chunk && (gb0 + lane == hi - 1 || lj == lnb - 1));
    const unsigned m_mine =
        __ballot_sync(0xffffffffu, in_chunk && (int)((it0 + lane) % S::NPH) == ph);
    unsigned todo = m_last | m_mine;
    while (todo) {
      const int pos = __ffs(todo) - 1;
      todo &= todo - 1;
      const int b = __shfl_sync(0xffffffffu, lb, pos);
      const int j = __shfl_sync(0xffffffffu, lj, pos);
      const int ctx = __shfl_sync(0xffffffffu, lctx, pos);
      const int n = ceil_div_blocks(ctx);
      const long long gb = gb0 + pos, it = it0 + pos;
      const bool piece_last = (m_last >> pos) & 1u;
      if ((m_mine >> pos) & 1u) {
        const int sidx = (int)(it % S::NST);
        const uint32_t sbase = stage0 + sidx * S::STAGE_BYTES;
        // warp-uniform: the collective instructions below need every lane
        const bool have = __all_sync(
            0xffffffffu, mbar_wait(full0 + 8 * sidx, (int)((it / S::NST) & 1), abort_flag, p.err));
        if (need_q) {
          // this warp's first stage of the piece: it carries the q rows
          need_q = false;
          if (!SPLIT_MERGE && ct == 0 && !pc_done) piece_splits(gb, j, n);
          if (have) {
            const uint32_t qrow = sbase + 2 * S::KV_BYTES + (g * G + gid) * kHeadDim * 2;
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
              uint32_t x0 = 0, x1 = 0;
              if (gid < G) {
                if constexpr (F8) {
                  // f16 operands; the k-step's dims in the order the K
                  // fragments use: columns 2qd, 2qd + 1 = dims dk, dk + 1,
                  // columns 2qd + 8, 2qd + 9 = dims dk + 2, dk + 3
                  const int dk = 16 * f8_k_chunk<S::HB>(qd, ks >> 2) + 4 * (ks & 3);
                  const uint32_t w0 = lds32(qrow + dk * 2);
                  const uint32_t w1 = lds32(qrow + (dk + 2) * 2);
                  const float2 f0 = bf16x2_to_float2(w0), f1 = bf16x2_to_float2(w1);
                  x0 = float2_to_f16x2(f0.x, f0.y);
                  x1 = float2_to_f16x2(f1.x, f1.y);
                } else {
                  x0 = lds32(qrow + (16 * ks + 2 * qd) * 2);
                  x1 = lds32(qrow + (16 * ks + 8 + 2 * qd) * 2);
                }
              }
              qf[ks][0] = x0;
              qf[ks][1] = x1;
            }
            if constexpr (ROPE) {
              // rotate-half: dims d < 64 (k-steps 0..3) pair with d + 64
              // (k-steps 4..7) in the same fragment registers; the same
              // products and one bf16 rounding as pa_rope_store_kv
              const uint32_t crow = sbase + 2 * S::KV_BYTES + S::Q_BYTES;
              const uint32_t srow = crow + S::ROPE_BYTES / 2;
#pragma unroll
              for (int ks = 0; ks < 4; ++ks) {
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                  const int d = 16 * ks + 8 * h + 2 * qd;
                  const float2 c2 = make_float2(__uint_as_float(lds32(crow + d * 4)),
                                                __uint_as_float(lds32(crow + d * 4 + 4)));
                  const float2 s2 = make_float2(__uint_as_float(lds32(srow + d * 4)),
                                                __uint_as_float(lds32(srow + d * 4 + 4)));
                  const float2 x1 = bf16x2_to_float2(qf[ks][h]);
                  const float2 x2 = bf16x2_to_float2(qf[ks + 4][h]);
                  if (gid < G) {
                    qf[ks][h] = float2_to_bf16x2(fmaf(x1.x, c2.x, -(x2.x * s2.x)),
                                                 fmaf(x1.y, c2.y, -(x2.y * s2.y)));
                    qf[ks + 4][h] = float2_to_bf16x2(fmaf(x2.x, c2.x, x1.x * s2.x),
                                                     fmaf(x2.y, c2.y, x1.y * s2.y));
                  }
                }
              }
            }
          }
        }
        const int valid = min(kBlockSize, ctx - j * kBlockSize);  // keys of this block (>= 1)
        bool patched = false;  // generic-proxy writes into the stage (fence before release)
        if (have) {
          // boxes of this head group: K at kb (bf16: +BOX_BYTES for dims
          // 64..127), V at vb
          const uint32_t kb = sbase + gpair * (F8 ? 1 : 2) * S::BOX_BYTES;
          const uint32_t vb = sbase + S::KV_BYTES + gpair * (F8 ? 1 : 2) * S::BOX_BYTES;
          if constexpr (!F8) {
            if (p.new_k != nullptr && j == n - 1) {
              // Fused store: this is the sequence's last block, the one that
              // holds its new token (row valid - 1).  The pool row may not
              // hold it yet: its K/V rows of this warp's head go into the
              // staged tile (lane L: 16-byte chunk L & 15 of K, L < 16, or of
              // V) and to the pool slot, which must be that row's slot.
              const long long slot = __ldg(p.slot_mapping + b);
              if (slot >= 0) {
                const long long want =
                    (long long)__ldg(p.block_tables + (long long)b * p.bt_stride + j) *
                        kBlockSize + (valid - 1);
                // the slot must be the new position's, and inside the pool
                // (a table entry outside it would make both agree on a slot
                // past the pool)
                long long pos = 0;
                if constexpr (ROPE) pos = __ldg(p.positions + b);
                if (slot != want || slot >= p.num_blocks * kBlockSize) {
                  if (lane == 0) report(p.err, PA_DEVERR_SLOT_INDEX);
                } else if (ROPE && (pos < 0 || pos >= p.max_position)) {
                  // reported by the producer: the row is neither stored nor patched
                } else {
                  const int c = lane & 15;
                  const bool is_v = lane >= 16;
                  const uint16_t *src =
                      (is_v ? p.new_v + b * p.new_v_tok : p.new_k + b * p.new_k_tok) +
                      g * kHeadDim + c * 8;
                  uint4 val = *reinterpret_cast<const uint4 *>(src);
                  if constexpr (ROPE) {
                    // the K row rotated at its position: chunk c pairs with
                    // chunk c ^ 8 (dims +- 64), held by lane ^ 8
                    uint4 pv;
                    pv.x = __shfl_xor_sync(0xffffffffu, val.x, 8);
                    pv.y = __shfl_xor_sync(0xffffffffu, val.y, 8);
                    pv.z = __shfl_xor_sync(0xffffffffu, val.z, 8);
                    pv.w = __shfl_xor_sync(0xffffffffu, val.w, 8);
                    if (!is_v) {
                      const long long t0 = pos * (kHeadDim / 2) + (c & 7) * 8;
                      const float4 c0 = __ldg(reinterpret_cast<const float4 *>(p.cos_table + t0));
                      const float4 c1 =
                          __ldg(reinterpret_cast<const float4 *>(p.cos_table + t0 + 4));
                      const float4 s0 = __ldg(reinterpret_cast<const float4 *>(p.sin_table + t0));
                      const float4 s1 =
                          __ldg(reinterpret_cast<const float4 *>(p.sin_table + t0 + 4));
                      uint4 ra, rb;
                      if (c < 8) {
                        rope_rotate8(val, pv, c0, c1, s0, s1, ra, rb);
                        val = ra;
                      } else {
                        rope_rotate8(pv, val, c0, c1, s0, s1, ra, rb);
                        val = rb;
                      }
                    }
                  }
                  uint16_t *dstg = (is_v ? p.v_pool16 : p.k_pool) +
                                   (slot * HKV + g) * kHeadDim + c * 8;
                  *reinterpret_cast<uint4 *>(dstg) = val;
                  const uint32_t a = (is_v ? vb : kb) + (c >> 3) * S::BOX_BYTES +
                                     swz((valid - 1) * S::HB + gsub, c & 7);
                  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(val.x),
                               "r"(val.y), "r"(val.z), "r"(val.w)
                               : "memory");
                  patched = true;
                  __syncwarp();
                }
              }
            }
          } else {
            if (p.new_k != nullptr && j == n - 1) {
              // Fused FP8 store: quantise the new token's rows of this head
              // (code = nearest-even E4M3 of x / scale, saturated) into the
              // staged tiles and the pools.  K: lane L < 8 takes dims
              // 16L .. 16L + 15 (one 16-byte chunk of the swizzled row); V:
              // lane L takes dims 4L .. 4L + 3 (the token's byte in each of
              // four dim-major rows).
              const long long slot = __ldg(p.slot_mapping + b);
              if (slot >= 0) {
                const long long phys_j = __ldg(p.block_tables + (long long)b * p.bt_stride + j);
                const long long want = phys_j * kBlockSize + (valid - 1);
                // the slot must be the new position's, and inside the pool
                // (a table entry outside it would make both agree on a slot
                // past the pool)
                if (slot != want || slot >= p.num_blocks * kBlockSize) {
                  if (lane == 0) report(p.err, PA_DEVERR_SLOT_INDEX);
                } else {
                  const int trow = valid - 1;
                  if (lane < 8) {
                    const float ksc = __ldg(p.k_scale + g);
                    const uint4 *src = reinterpret_cast<const uint4 *>(
                        p.new_k + b * p.new_k_tok + g * kHeadDim + 16 * lane);
                    const uint4 x0 = src[0], x1 = src[1];
                    const uint32_t xw[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
                    uint32_t cw[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                      const float2 f0 = bf16x2_to_float2(xw[2 * i]);
                      const float2 f1 = bf16x2_to_float2(xw[2 * i + 1]);
                      cw[i] = float2_to_e4m3x2_sat(__fdiv_rn(f0.x, ksc), __fdiv_rn(f0.y, ksc)) |
                              (float2_to_e4m3x2_sat(__fdiv_rn(f1.x, ksc), __fdiv_rn(f1.y, ksc))
                               << 16);
                    }
                    *reinterpret_cast<uint4 *>(p.k_pool8 + (slot * HKV + g) * kHeadDim +
                                               16 * lane) = make_uint4(cw[0], cw[1], cw[2], cw[3]);
                    const uint32_t a = kb + swz(trow * S::HB + gsub, lane);
                    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(cw[0]),
                                 "r"(cw[1]), "r"(cw[2]), "r"(cw[3])
                                 : "memory");
                  }
                  {
                    const float vsc_raw = __ldg(p.v_scale + g);
                    const uint2 xv = *reinterpret_cast<const uint2 *>(
                        p.new_v + b * p.new_v_tok + g * kHeadDim + 4 * lane);
                    const float2 f0 = bf16x2_to_float2(xv.x), f1 = bf16x2_to_float2(xv.y);
                    const uint32_t c01 =
                        float2_to_e4m3x2_sat(__fdiv_rn(f0.x, vsc_raw), __fdiv_rn(f0.y, vsc_raw));
                    const uint32_t c23 =
                        float2_to_e4m3x2_sat(__fdiv_rn(f1.x, vsc_raw), __fdiv_rn(f1.y, vsc_raw));
                    const uint32_t codes = c01 | (c23 << 16);
                    uint8_t *vg = p.v_pool8 + ((phys_j * HKV + g) * kHeadDim + 4 * lane) *
                                                  kBlockSize + trow;
                    const uint32_t vsm =
                        vb + gsub * (kHeadDim * kBlockSize) + 4 * lane * kBlockSize + trow;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                      const uint32_t c = (codes >> (8 * i)) & 0xFFu;
                      vg[i * kBlockSize] = (uint8_t)c;
                      asm volatile("st.shared.u8 [%0], %1;" ::"r"(vsm + i * kBlockSize), "r"(c)
                                   : "memory");
                    }
                  }
                  patched = true;
                  __syncwarp();
                }
              }
            }
          }
          // S^T = K . Q^T, two accumulation chains over the eight 16-dim k-steps
          float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
          if constexpr (F8) {
            // 128-byte rows of E4M3 codes (token, head), 128-byte swizzle.
            // Thread qd reads 16-byte chunks kc0 and kc1 of rows tok0 and
            // tok1 (one vector load each); k-step ks = 4 h + i takes word i
            // of chunk kc_h: four consecutive dims per row.
            const int row0 = tok0 * S::HB + gsub, row1 = tok1 * S::HB + gsub;
            const int kc0 = f8_k_chunk<S::HB>(qd, 0), kc1 = f8_k_chunk<S::HB>(qd, 1);
            const uint4 r0a = lds128(kb + swz(row0, kc0)), r0b = lds128(kb + swz(row0, kc1));
            const uint4 r1a = lds128(kb + swz(row1, kc0)), r1b = lds128(kb + swz(row1, kc1));
            const uint32_t k0w[8] = {r0a.x, r0a.y, r0a.z, r0a.w, r0b.x, r0b.y, r0b.z, r0b.w};
            const uint32_t k1w[8] = {r1a.x, r1a.y, r1a.z, r1a.w, r1b.x, r1b.y, r1b.z, r1b.w};
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
              const uint32_t w0 = k0w[ks];
              const uint32_t w1 = k1w[ks];
              const uint32_t a0 = e4m3x2_to_f16x2(w0), a2 = e4m3x2_to_f16x2(w0 >> 16);
              const uint32_t a1 = e4m3x2_to_f16x2(w1), a3 = e4m3x2_to_f16x2(w1 >> 16);
              if (ks & 1)
                mma_f16(sb, a0, a1, a2, a3, qf[ks][0], qf[ks][1]);
              else
                mma_f16(sa, a0, a1, a2, a3, qf[ks][0], qf[ks][1]);
            }
          } else {
            const int mi = lane >> 3, r = lane & 7;
            const int t = r + ((mi & 1) << 3);
            const int row = t * S::HB + gsub;  // 128-byte row of token t, this head
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
              const int chunk = ((ks & 3) << 1) + (mi >> 1);
              uint32_t a0, a1, a2, a3;
              ldsm_x4(kb + (ks >> 2) * S::BOX_BYTES + swz(row, chunk), a0, a1, a2, a3);
              if (ks & 1)
                mma_bf16(sb, a0, a1, a2, a3, qf[ks][0], qf[ks][1]);
              else
                mma_bf16(sa, a0, a1, a2, a3, qf[ks][0], qf[ks][1]);
            }
          }
          // scaled scores (base 2): [0] (token tok0, head 2qd) [1] (tok0, 2qd+1)
          // [2] (tok1, 2qd) [3] (tok1, 2qd+1); keys past the end are -inf
          const bool v0 = tok0 < valid, v1 = tok1 < valid;
          const float s0 = v0 ? (sa[0] + sb[0]) * cl2 : -INFINITY;
          const float s1 = v0 ? (sa[1] + sb[1]) * cl2 : -INFINITY;
          const float s2 = v1 ? (sa[2] + sb[2]) * cl2 : -INFINITY;
          const float s3 = v1 ? (sa[3] + sb[3]) * cl2 : -INFINITY;
          float x0 = fmaxf(s0, s2), x1 = fmaxf(s1, s3);
#pragma unroll
          for (int off = 4; off < 32; off <<= 1) {
            x0 = fmaxf(x0, __shfl_xor_sync(0xffffffffu, x0, off));
            x1 = fmaxf(x1, __shfl_xor_sync(0xffffffffu, x1, off));
          }
          // token 0 of every block is a key, so x0, x1 are finite (and the
          // first block moves the reference: x - (-inf) = +inf)
          const bool g0 = x0 - m0 > 8.f, g1 = x1 - m1 > 8.f;
          if (__any_sync(0xffffffffu, g0 || g1)) {
            const float al0 = g0 ? exp2f(m0 - x0) : 1.f, al1 = g1 ? exp2f(m1 - x1) : 1.f;
            if (g0) m0 = x0;
            if (g1) m1 = x1;
            l0 *= al0;
            l1 *= al1;
#pragma unroll
            for (int mt = 0; mt < 8; ++mt) {
              o[mt][0] *= al0;
              o[mt][1] *= al1;
              o[mt][2] *= al0;
              o[mt][3] *= al1;
            }
          }
          const float p0 = exp2f(s0 - m0), p1 = exp2f(s1 - m1);
          const float p2 = exp2f(s2 - m0), p3 = exp2f(s3 - m1);
          l0 += p0 + p2;
          l1 += p1 + p3;
          // P^T fragments: bf16 hi + lo split, or with F8 pools one f16
          // term (11-bit significand, far finer than the E4M3 values it
          // weighs)
          uint32_t hA, hB, lA = 0u, lB = 0u;
          if constexpr (F8) {
            hA = float2_to_f16x2(p0, p1);
            hB = float2_to_f16x2(p2, p3);
          } else {
            hA = float2_to_bf16x2(p0, p1);
            hB = float2_to_bf16x2(p2, p3);
            const float2 fA = bf16x2_to_float2(hA), fB = bf16x2_to_float2(hB);
            lA = float2_to_bf16x2(p0 - fA.x, p1 - fA.y);
            lB = float2_to_bf16x2(p2 - fB.x, p3 - fB.y);
          }
          const uint32_t bh0 = movm_t(hA), bh1 = movm_t(hB);
          const uint32_t bl0 = movm_t(lA), bl1 = movm_t(lB);
          if (valid < kBlockSize) {
            // rows past the last key may hold anything (NaN): zero them so that
            // 0-weight rows contribute exactly 0 to the MMA
            if constexpr (F8) {
              // dim-major: bytes valid .. 15 of each of this head's 128 dim rows
              const uint32_t hb = vb + gsub * (kHeadDim * kBlockSize);
              for (int d = lane; d < kHeadDim; d += 32) {
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                  const int keep = min(max(valid - 4 * w, 0), 4);
                  if (keep < 4) {
                    const uint32_t a = hb + d * kBlockSize + 4 * w;
                    const uint32_t mask = keep == 0 ? 0u : (1u << (8 * keep)) - 1u;
                    asm volatile("st.shared.u32 [%0], %1;" ::"r"(a), "r"(lds32(a) & mask)
                                 : "memory");
                  }
                }
              }
            } else {
              for (int i = lane; i < (kBlockSize - valid) * 16; i += 32) {
                const int t = valid + (i >> 4), ch = i & 15;
                const uint32_t a = vb + (ch >> 3) * S::BOX_BYTES + swz(t * S::HB + gsub, ch & 7);
                asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(a), "r"(0u)
                             : "memory");
              }
            }
            __syncwarp();
          }
          // O^T += V^T . P^T
          if constexpr (F8) {
            // dim rows 16 mt + gid (a0, a2) and + 8 (a1, a3): bytes 4qd .. 4qd + 3
            // are the tokens of k-rows 2qd, 2qd + 1 (a0 / a1) and 2qd + 8,
            // 2qd + 9 (a2 / a3) in the score-row order above
            const uint32_t hb = vb + gsub * (kHeadDim * kBlockSize) + gid * kBlockSize + 4 * qd;
#pragma unroll
            for (int mt = 0; mt < 8; ++mt) {
              const uint32_t w0 = lds32(hb + 16 * mt * kBlockSize);
              const uint32_t w1 = lds32(hb + (16 * mt + 8) * kBlockSize);
              const uint32_t a0 = e4m3x2_to_f16x2(w0), a2 = e4m3x2_to_f16x2(w0 >> 16);
              const uint32_t a1 = e4m3x2_to_f16x2(w1), a3 = e4m3x2_to_f16x2(w1 >> 16);
              mma_f16(o[mt], a0, a1, a2, a3, bh0, bh1);
            }
          } else {
            const int mi = lane >> 3, r = lane & 7;
            const int t = r + ((mi >> 1) << 3);
            const int row = t * S::HB + gsub;
#pragma unroll
            for (int mt = 0; mt < 8; ++mt) {
              const int chunk = 2 * mt + (mi & 1);  // 8-dim chunk 0..15
              uint32_t a0, a1, a2, a3;
              ldsm_x4_t(vb + (chunk >> 3) * S::BOX_BYTES + swz(row, chunk & 7), a0, a1, a2, a3);
              mma_bf16(o[mt], a0, a1, a2, a3, bh0, bh1);
              mma_bf16(o[mt], a0, a1, a2, a3, bl0, bl1);
            }
          }
          // generic-proxy writes above must be ordered before the TMA that
          // reuses this stage
          if (valid < kBlockSize || patched)
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty0 + 8 * sidx);  // one of the slot's Hkv readers
      }
      if (!piece_last) continue;

      // ---- end of a piece: merge the warps of each kv head, write rows -------
      if constexpr (F8) {
        // the V scale of this warp's kv head, once per piece
#pragma unroll
        for (int mt = 0; mt < 8; ++mt)
#pragma unroll
          for (int i = 0; i < 4; ++i) o[mt][i] *= vsc;
      }
      // (warp 0 may have had no stage in the piece)
      if (!SPLIT_MERGE && ct == 0 && !pc_done) piece_splits(gb, j, n);
      const bool head_cut = gb - j < lo;  // the sequence starts before this CTA's blocks
      const bool tail_cut = j < n - 1;
      const bool whole = !head_cut && !tail_cut;
      // A cut piece is the CTA's first piece (cut at its head) or its final
      // one (cut at its tail); pieces in between are whole sequences.
      const bool final_piece = gb == hi - 1;
      // own rows of a final cut piece, kept in the ring (every stage consumed);
      // the rest of the ring receives the other pieces' rows for the merge
      float *own_o = reinterpret_cast<float *>(smem);
      float *own_lse = own_o + S::HQ * kHeadDim;
      const bool keep_own = !SPLIT_MERGE && !whole && final_piece;
      float L0 = l0, L1 = l1;
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        L0 += __shfl_xor_sync(0xffffffffu, L0, off);
        L1 += __shfl_xor_sync(0xffffffffu, L1, off);
      }
      const long long slot_row = ((head_cut ? 0 : 1) * nsplit + c) * S::HQ;
      const int ha = 2 * qd, hb = 2 * qd + 1;  // heads of this lane's fragment columns
      // red buffer of this piece; the epilogue warp must be done with its use
      // two pieces ago
      const int kbuf = npieces & 1;
      float *const rbuf = red + kbuf * S::RED_ONE_FLOATS;
      if (npieces >= 2)
        __all_sync(0xffffffffu, mbar_wait(smem_addr(&ctl->red_empty[kbuf]),
                                          ((npieces >> 1) - 1) & 1, abort_flag, p.err));
      if constexpr (S::NPH == 1) {
        // one warp per kv head: write straight from the fragments
        if (keep_own) named_barrier(1, S::CW * 32);  // all warps are past the ring
        const float ia = L0 > 0.f ? 1.f / L0 : 0.f, ib = L1 > 0.f ? 1.f / L1 : 0.f;
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            const int d = 16 * mt + gid + 8 * half;
            if (ha < G) {
              const int qh = g * G + ha;
              const float v = o[mt][2 * half] * ia;
              if (whole) {
                store_out1(p.out, p.out_f32, ((long long)b * S::HQ + qh) * kHeadDim + d, v);
              } else {
                p.part_o[(slot_row + qh) * kHeadDim + d] = v;
                if (keep_own) own_o[qh * kHeadDim + d] = v;
              }
            }
            if (hb < G) {
              const int qh = g * G + hb;
              const float v = o[mt][2 * half + 1] * ib;
              if (whole) {
                store_out1(p.out, p.out_f32, ((long long)b * S::HQ + qh) * kHeadDim + d, v);
              } else {
                p.part_o[(slot_row + qh) * kHeadDim + d] = v;
                if (keep_own) own_o[qh * kHeadDim + d] = v;
              }
            }
          }
        }
        if (!whole && gid == 0) {
          const float lse_a = L0 > 0.f ? (m0 + __log2f(L0)) * 0.69314718055994531f : -INFINITY;
          const float lse_b = L1 > 0.f ? (m1 + __log2f(L1)) * 0.69314718055994531f : -INFINITY;
          if (ha < G) {
            p.part_lse[slot_row + g * G + ha] = lse_a;
            if (keep_own) own_lse[g * G + ha] = lse_a;
          }
          if (hb < G) {
            p.part_lse[slot_row + g * G + hb] = lse_b;
            if (keep_own) own_lse[g * G + hb] = lse_b;
          }
        }
        if (final_piece && !whole) named_barrier(1, S::CW * 32);
      } else {
        // several warps share a kv head: combine through shared memory
        if (ha < G) {
          float *ra = rbuf + (cw * G + ha) * S::RED_FLOATS_PER_HEAD;
          if (gid == 0) {
            ra[S::RED_M] = m0;
            ra[S::RED_L] = L0;
          }
#pragma unroll
          for (int mt = 0; mt < 8; ++mt) {
            ra[16 * mt + gid] = o[mt][0];
            ra[16 * mt + gid + 8] = o[mt][2];
          }
        }
        if (hb < G) {
          float *rb = rbuf + (cw * G + hb) * S::RED_FLOATS_PER_HEAD;
          if (gid == 0) {
            rb[S::RED_M] = m1;
            rb[S::RED_L] = L1;
          }
#pragma unroll
          for (int mt = 0; mt < 8; ++mt) {
            rb[16 * mt + gid] = o[mt][1];
            rb[16 * mt + gid + 8] = o[mt][3];
          }
        }
      }
      if constexpr (S::NPH > 1) {
        // the final piece: the consumers combine it themselves (nothing else
        // is left for them to do); other pieces go to the epilogue warp
        if (final_piece) {
          named_barrier(1, S::CW * 32);
          // one thread per query head: the normalised weight of each of its NPH
          // warps (into the merge scratch) and the piece's lse
          float *cwt = mw;  // [NPH][HQ]
          if (ct < S::HQ) {
            const int qh = ct, gh = qh / G, h = qh % G;
            float mk[S::NPH], M = -INFINITY;
#pragma unroll
            for (int k = 0; k < S::NPH; ++k) {
              mk[k] = rbuf[((gh + k * HKV) * G + h) * S::RED_FLOATS_PER_HEAD + S::RED_M];
              M = fmaxf(M, mk[k]);
            }
            float L = 0.f;
#pragma unroll
            for (int k = 0; k < S::NPH; ++k) {
              mk[k] = mk[k] == -INFINITY ? 0.f : exp2f(mk[k] - M);
              L += rbuf[((gh + k * HKV) * G + h) * S::RED_FLOATS_PER_HEAD + S::RED_L] * mk[k];
            }
            const float inv = L > 0.f ? 1.f / L : 0.f;
#pragma unroll
            for (int k = 0; k < S::NPH; ++k) cwt[k * S::HQ + qh] = mk[k] * inv;
            if (!whole) {
              const float lse = L > 0.f ? (M + __log2f(L)) * 0.69314718055994531f : -INFINITY;
              p.part_lse[slot_row + qh] = lse;
              if (keep_own) own_lse[qh] = lse;
            }
          }
          named_barrier(1, S::CW * 32);
          for (int item = ct; item < S::HQ * (kHeadDim / 4); item += S::CW * 32) {
            const int qh = item / (kHeadDim / 4);
            const int d = (item % (kHeadDim / 4)) * 4;
            const int gh = qh / G, h = qh % G;
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int k = 0; k < S::NPH; ++k) {
              const float wk = cwt[k * S::HQ + qh];
              const float4 v = *reinterpret_cast<const float4 *>(
                  rbuf + ((gh + k * HKV) * G + h) * S::RED_FLOATS_PER_HEAD + d);
              acc.x += wk * v.x;
              acc.y += wk * v.y;
              acc.z += wk * v.z;
              acc.w += wk * v.w;
            }
            if (whole) {
              store_out4(p.out, p.out_f32, ((long long)b * S::HQ + qh) * kHeadDim + d, acc);
            } else {
              *reinterpret_cast<float4 *>(p.part_o + (slot_row + qh) * kHeadDim + d) = acc;
              if (keep_own) *reinterpret_cast<float4 *>(own_o + qh * kHeadDim + d) = acc;
            }
          }
          named_barrier(1, S::CW * 32);
        }
      }

      if (final_piece) {
        // no piece follows: the end mark goes to the epilogue warp now,
        // before the final piece is published and merged, so that the
        // epilogue warp is done before the consumers' end (buffer kbuf was
        // released to the consumers above; they are done with it)
        if (ct == 0) ctl->desc[kbuf].kind = kPieceEnd;
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&ctl->red_full[kbuf]));
      }
      if (!final_piece) {
        // hand the piece to the epilogue warp (its rows are in rbuf, or
        // already written with one warp per kv head) and stream on
        if (ct == 0) {
          PieceDesc &pd = ctl->desc[kbuf];
          pd.slot_row = slot_row;
          pd.cs0 = ctl->pc_cs0;
          pd.cs1 = ctl->pc_cs1;
          pd.b = b;
          pd.kind = whole ? kPieceWhole : kPieceCut;
          pd.pieces = ctl->pc_pieces;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&ctl->red_full[kbuf]));
        ++npieces;
      } else if (keep_own) {
        // The final piece, cut: publish it; the last piece of the sequence to
        // arrive merges.  Nothing follows the final piece, which the jump out
        // of the loops makes explicit: the accumulators are dead and the merge
        // may use their registers.  Every consumer thread is past a barrier
        // since consumer thread 0 wrote the piece's split words.
        const long long cs0 = ctl->pc_cs0, cs1 = ctl->pc_cs1;
        const int pieces = ctl->pc_pieces;
        if (ct == 0) {
          *reinterpret_cast<volatile int *>(&ctl->decided) = 1;
          if (mbar_test_wait(smem_addr(&ctl->seen_bar), 0)) {
            // every other piece had arrived (the epilogue warp acquired their
            // rows): this piece is the last, no arrival and no publication
            ctl->last = 1;
          } else {
            // arrive first (relaxed: nothing of this piece is published yet).
            // The last arrival merges and needs only every other piece
            // published (acquire); any other publishes its rows (release).
            const bool last =
                arrived_count(atom_add_relaxed_gpu(p.counters + cs1, kArrive)) == pieces - 1;
            if (last)
              wait_published(p.counters + cs1, pieces - 1, abort_flag, p.err);
            else
              atom_add_release_gpu(p.counters + cs1, kPublish);
            ctl->last = last && !*abort_flag;
          }
          // the epilogue warp requested the other partials only once every
          // other piece had arrived: when it has, they are this merge's
          ctl->use_pf = ctl->last && *reinterpret_cast<volatile int *>(&ctl->pf_ready);
          // The epilogue warp has published every earlier piece once it took
          // the end mark: then whether the CTA owes a merge (a piece it
          // published arrived last) is known, and an owed merge runs now,
          // beside the final piece's (on the two halves of the consumer
          // threads, with their own buffers, barriers and weights).  If the
          // epilogue warp is not there yet, the owed merge waits for the end.
          ctl->owed_now = mbar_test_wait(smem_addr(&ctl->pub_done), 0) &&
                          *reinterpret_cast<volatile int *>(&ctl->def_pending);
        }
        named_barrier(1, S::CW * 32);
        const bool fin_merge = ctl->last != 0;
        const bool def_merge = ctl->owed_now != 0;
        // the final piece's merge: threads [0, nt) of the consumers, named
        // barrier bar; the rows of the other pieces come into the ring after
        // the own rows, up to buf_end floats from the ring start
        auto final_merge = [&](auto nt_tag, int t, int bar, long long buf_end) {
          constexpr int NT = decltype(nt_tag)::value;
          float *mbuf = own_lse + ((S::HQ + 3) & ~3);
          const long long mbuf_bytes = (buf_end - (long long)(mbuf - own_o)) * 4;
          const bool use_pf = ctl->use_pf != 0;
          bool merged = false;
          if constexpr (S::PF_PIECES > 0) {
            if (use_pf)
              merged = merge_sequence_bulk<S::HQ, S::PF_PIECES, NT>(
                  p, b, cs0, cs1, nsplit, N, mw + S::PF_W, t, bar, c, own_o, own_lse,
                  red + ((npieces & 1) ^ 1) * S::RED_ONE_FLOATS,
                  (long long)S::RED_ONE_FLOATS * 4, smem_addr(&ctl->pf_bar), abort_flag, true);
          }
          // (beside an owed merge, the weights stay below DEF_W)
          constexpr int MAXP = NT == S::CW * 32 ? S::MERGE_MAX_PIECES : S::DEF_W / S::HQ - 1;
          if (!merged && !use_pf)
            merged = merge_sequence_bulk<S::HQ, MAXP, NT>(
                p, b, cs0, cs1, nsplit, N, mw, t, bar, c, own_o, own_lse, mbuf, mbuf_bytes,
                smem_addr(&ctl->merge_bar), abort_flag);
          if (!merged)
            for (int h = t >> 5; h < S::HQ; h += NT / 32)
              merge_row(p.part_o, p.part_lse, p.out, p.out_f32, (long long)b * S::HQ + h, S::HQ, h,
                        cs0, cs1, nsplit, N, lane);
          if (t == 0) p.counters[cs1] = 0;
        };
        // the owed merge: every piece from the workspace, rows into the ring
        // from buf_begin floats on
        auto owed_merge = [&](auto nt_tag, int t, int bar, long long buf_begin) {
          constexpr int NT = decltype(nt_tag)::value;
          const int db = ctl->def_b;
          const long long d0 = ctl->def_cs0, d1 = ctl->def_cs1;
          float *dbuf = own_o + buf_begin;
          const long long dbuf_bytes = ((long long)S::NST * S::STAGE_BYTES / 4 - buf_begin) * 4;
          if (!merge_sequence_bulk<S::HQ, S::DEF_MAX_PIECES, NT>(
                  p, db, d0, d1, nsplit, N, mw + S::DEF_W, t, bar, -1, nullptr, nullptr, dbuf,
                  dbuf_bytes, smem_addr(&ctl->merge_bar2), abort_flag))
            for (int h = t >> 5; h < S::HQ; h += NT / 32)
              merge_row(p.part_o, p.part_lse, p.out, p.out_f32, (long long)db * S::HQ + h, S::HQ,
                        h, d0, d1, nsplit, N, lane);
          if (t == 0) p.counters[d1] = 0;
        };
        constexpr int RING_FLOATS = S::NST * S::STAGE_BYTES / 4;
        // the ring split in two (1 KB aligned) when both merges run
        constexpr int HALF_FLOATS = RING_FLOATS / 2 / 256 * 256;
        if (fin_merge && def_merge) {
          if (ct < S::CW * 16)
            final_merge(std::integral_constant<int, S::CW * 16>{}, ct, 3, HALF_FLOATS);
          else
            owed_merge(std::integral_constant<int, S::CW * 16>{}, ct - S::CW * 16, 4, HALF_FLOATS);
        } else if (fin_merge) {
          final_merge(std::integral_constant<int, S::CW * 32>{}, ct, 1, RING_FLOATS);
        } else if (def_merge) {
          owed_merge(std::integral_constant<int, S::CW * 32>{}, ct, 1, 0);
        }
        def_done = def_merge;
        goto consumers_done;
      }
      // the next piece starts from nothing
#pragma unroll
      for (int mt = 0; mt < 8; ++mt)
#pragma unroll
        for (int i = 0; i < 4; ++i) o[mt][i] = 0.f;
      m0 = m1 = -INFINITY;
      l0 = l1 = 0.f;
      need_q = true;
      pc_done = false;
    }
    gb0 += count;
    it0 += count;
  }
consumers_done:
  {
    if (no_final) {
      // no final piece came (inconsistent input): tell the epilogue warp
      // that no piece follows, once it is done with the buffer it would look
      // at next
      const int kbuf = npieces & 1;
      if (npieces >= 2)
        __all_sync(0xffffffffu, mbar_wait(smem_addr(&ctl->red_empty[kbuf]),
                                          ((npieces >> 1) - 1) & 1, abort_flag, p.err));
      if (ct == 0) ctl->desc[kbuf].kind = kPieceEnd;
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&ctl->red_full[kbuf]));
    }
    if (ct == 0) *reinterpret_cast<volatile int *>(&ctl->decided) = 1;
    // the epilogue warp has finished (copies it requested have landed); a
    // merge it left, unless run beside the final one above
    __all_sync(0xffffffffu, mbar_wait(smem_addr(&ctl->ew_done), 0, abort_flag, p.err));
    if (!def_done && ctl->def_pending) {
      named_barrier(1, S::CW * 32);  // every consumer is done with the ring
      const int db = ctl->def_b;
      const long long d0 = ctl->def_cs0, d1 = ctl->def_cs1;
      if (!merge_sequence_bulk<S::HQ, S::MERGE_MAX_PIECES, S::CW * 32>(
              p, db, d0, d1, nsplit, N, mw, ct, 1, -1, nullptr, nullptr,
              reinterpret_cast<float *>(smem), (long long)S::NST * S::STAGE_BYTES,
              smem_addr(&ctl->merge_bar2), abort_flag))
        for (int h = cw; h < S::HQ; h += S::CW)
          merge_row(p.part_o, p.part_lse, p.out, p.out_f32, (long long)db * S::HQ + h, S::HQ, h,
                    d0, d1, nsplit, N, lane);
      if (ct == 0) p.counters[d1] = 0;
    }
  }
}

// Launches decode_kernel<G, HKV, F8, ROPE, SPLIT_MERGE> for one G (defined per
// HKV and variant in pa_decode_h*.cu, pa_decode_f8_h*.cu, pa_decode_rope_h*.cu
// and, with SPLIT_MERGE, pa_decode_sm_h{4,8}.cu and pa_decode_f8_sm_h{4,8}.cu).
template <int HKV, bool F8, bool ROPE = false, bool SPLIT_MERGE = false>
cudaError_t launch_decode(int G, const CUtensorMap &tk, const CUtensorMap &tv,
                          const DecodeParams &p, cudaStream_t s, int device, bool pdl);

}  // namespace pa
