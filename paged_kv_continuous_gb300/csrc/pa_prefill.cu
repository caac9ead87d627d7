// pa_prefill_varlen: causal varlen attention of cu_seqlens-packed query
// chunks over each sequence's paged keys (mini-vllm tutorial, "step14_7 --
// Batched Forward", sections "解决方案：变长 batch（varlen）" and "cu_seqlens 只在
// Attention 里才需要": tokens of all sequences are flattened and cu_seqlens
// marks the boundaries; attention stays inside a sequence and is causal;
// keys come from the sequence's pages through its block table).
//
// One CTA computes a 128-row tile of one (sequence, kv head): rows are the
// (query position, query head) pairs of PT = 128 / G consecutive positions
// times the G query heads of the kv head, so every K/V tile read from the
// pool serves the whole GQA group.  Per 64-key tile j:
//   S   = Q K_j^T      tcgen05.mma (M 128, N 64, K 128), fp32 in TMEM
//   P   = exp2(S * c - m)  per row, with the causal and length masks (fp32)
//   O  += P V_j        tcgen05.mma (M 128, N 128, K 64), O accumulated in
//                      TMEM.  A row's exponentials use a reference max that
//                      moves only when a tile's max exceeds it by more than 8
//                      (base 2), so O is rescaled in TMEM rarely; P stays
//                      <= 256.  P is split into bf16 hi + lo parts (two MMA
//                      passes) so the product keeps ~16 bits of the fp32
//                      weights.
// Two CTAs share an SM (under half its shared memory, registers and tensor
// memory each), so one CTA's softmax runs while the other's MMAs keep the
// tensor pipe busy.  Warps: 0 loads K tiles and 2 loads V tiles (TMA, two
// stages each; the block-table entries of eight tiles come in one round of
// lane loads); 1 issues the score MMAs and owns the TMEM allocation (two
// score buffers and O), 3 issues the PV MMAs (each a converged warp, one
// elected lane, so neither chain waits behind the other); 4..7 run the
// softmax, one warp per TMEM lane quarter and one row per thread: they write
// their Q rows into shared memory, read each tile's scores, write P over them
// (the A operand of the PV MMAs comes from tensor memory) and store the
// output.  Tile j's scores go to buffer j % 2 once the PV MMA of tile j - 2
// that read that buffer is done, so the score MMA of tile j + 1 runs under
// the softmax of tile j.  CTAs take their tiles longest first (the most KV
// tiles to attend), so the long ones do not start at the end of the grid.
//
// pa_prefill_store_varlen (the store of the chunks' K/V fused in): other CTAs
// of a sequence need chunk keys this CTA stores, so the chunk is never read
// back from the pool.  Pages wholly before the prefix come from the pool,
// pages wholly inside the chunk by TMA from the new rows, and the page that
// straddles the prefix is assembled by the loader warp from both; after its
// last tile each loader warp stores the CTA's own positions (K: warp 0, V:
// warp 2) through slot_mapping.
#include <cmath>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "pa_common.cuh"

namespace pa {
namespace {

constexpr int kPfSoftWarps = 4;   // one per TMEM lane quarter: a thread owns a row
constexpr int kPfThreads = 32 * (4 + kPfSoftWarps);  // K loader, QK, V loader, PV, softmax
constexpr int kPfFirstSoftWarp = 4;
constexpr int kPfRows = 128;      // M
constexpr int kPfKeys = 64;       // keys per KV tile (N of the score MMA)
constexpr int kPfPages = kPfKeys / kBlockSize;  // pages per KV tile
constexpr int kHalfBytes = kPfKeys * 128;  // 64 keys x 64 dims (bf16) with the 128-byte swizzle
constexpr int kTileBytes2 = 2 * kHalfBytes;  // one 64 x 128 bf16 K or V tile = 16 KB
constexpr int kQHalf = kPfRows * 128;        // 128 rows x 64 dims of Q
// Shared memory (offsets from a 1024-aligned base), under half an SM's so
// that two CTAs share one: while one runs its softmax the other's MMAs keep
// the tensor pipe busy.
constexpr int kKStages = 2, kVStages = 2;
constexpr int kOffQ = 0;                                  // Q tile, two 64-dim halves
constexpr int kOffK = kOffQ + 2 * kQHalf;                 // K tile j in stage j % 2
constexpr int kOffV = kOffK + kKStages * kTileBytes2;     // V tile j in stage j % 2
constexpr int kOffBar = kOffV + kVStages * kTileBytes2;
// 8-byte slots from kOffBar: K full / empty, V full / empty (one per stage),
// Q ready, two score, two P and two PV barriers, the TMEM address, the abort flag
constexpr int kBarKFull = 0, kBarKEmpty = kBarKFull + kKStages;
constexpr int kBarVFull = kBarKEmpty + kKStages, kBarVEmpty = kBarVFull + kVStages;
constexpr int kBarQ = kBarVEmpty + kVStages, kBarS = kBarQ + 1, kBarP = kBarS + 2;
constexpr int kBarO = kBarP + 2, kBarTmem = kBarO + 2, kBarAbort = kBarTmem + 1;
constexpr int kBarBytes = 256;
static_assert((kBarAbort + 1) * 8 <= kBarBytes, "barrier slots do not fit");
constexpr int kPfSmem = 1024 + kOffBar + kBarBytes;
static_assert(kPfSmem <= 227 * 1024, "shared memory over the per-CTA limit");
// TMEM columns (256 of the SM's 512, two CTAs per SM): two score buffers
// S_0, S_1 at 0..63 and 64..127 (fp32, tile j in buffer j % 2; the softmax
// writes P over the scores it has read: bf16 hi parts in the buffer's
// columns 0..31, lo parts in 32..63, two keys per column), O at 128..255.
constexpr int kTmemCols = 256;
constexpr int kTmemSCols = 64, kTmemO = 128;

struct PrefillParams {
  void *out;
  int out_f32;
  const uint16_t *q;
  const int32_t *cu_seqlens;
  int num_seqs;
  long long num_blocks;
  const int32_t *block_tables;
  long long bt_stride;
  const int32_t *context_lens;
  int hq, hkv;
  float qk_scale_log2;  // > 0: a scale <= 0 is folded into q as staged
  uint32_t q_and, q_xor;  // staged q pairs = (q & q_and) ^ q_xor
  int32_t *err;
  // Fused store (new_k == nullptr: none).  The chunk rows of token t are
  // new_k / new_v + t * new_*_tok + h * 128; they are stored at
  // slot_mapping[t], and the chunk's keys are read from them (not from the
  // pool, where other CTAs of the sequence may not have stored them yet).
  const uint16_t *new_k;
  const uint16_t *new_v;
  long long new_k_tok, new_v_tok;
  const int32_t *slot_mapping;
  const uint16_t *k_cache;  // pools, for the page that straddles the prefix
  const uint16_t *v_cache;
  uint16_t *k_store;  // the same pools, written by the fused store
  uint16_t *v_store;
};

// ---- tcgen05 helpers ----------------------------------------------------------

// Shared-memory matrix descriptor (K- or MN-major, 128-byte swizzle):
// start address, leading / stride byte offsets (>> 4), version 1, layout 2.
__device__ __forceinline__ uint64_t umma_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFF);
  d |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFF) << 32;
  d |= (uint64_t)1 << 46;  // descriptor version for tcgen05
  d |= (uint64_t)2 << 61;  // SWIZZLE_128B
  return d;
}

// Instruction descriptor, kind::f16: bf16 A and B, fp32 D, M = 128, N = n,
// A K-major, B K-major (b_mn = 0) or MN-major (b_mn = 1).
__host__ __device__ constexpr uint32_t umma_idesc(int b_mn, int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)b_mn << 16) |
         ((uint32_t)(n >> 3) << 17) | ((uint32_t)(kPfRows >> 4) << 24);
}

// The MMA, commit and TMA helpers below are executed by a whole converged
// warp whose role branch the compiler can see is warp-uniform: every lane
// computes the same operands (kept in uniform registers) and one lane, picked
// by elect.sync, issues.  Issued from a lone lane in a divergent branch, each
// MMA cost about three times its tensor-pipe time.
//
// D (+)= A B with A (M x 16, K-major, two bf16 per 32-bit column) read from
// tensor memory at column address a_tmem and B described by b.
__device__ __forceinline__ void umma_f16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D (+)= A B with both operands described in shared memory.
__device__ __forceinline__ void umma_f16_ss(uint32_t d_tmem, uint64_t a, uint64_t b,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(
          bar)
      : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// 32 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
      "%28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// 64 consecutive fp32 columns of this thread's TMEM lane (two loads, one wait).
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, float (&v)[2][32]) {
  uint32_t r[64];
#pragma unroll
  for (int h = 0; h < 2; ++h)
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
        "%28, %29, %30, %31}, [%32];"
        : "=r"(r[32 * h + 0]), "=r"(r[32 * h + 1]), "=r"(r[32 * h + 2]), "=r"(r[32 * h + 3]),
          "=r"(r[32 * h + 4]), "=r"(r[32 * h + 5]), "=r"(r[32 * h + 6]), "=r"(r[32 * h + 7]),
          "=r"(r[32 * h + 8]), "=r"(r[32 * h + 9]), "=r"(r[32 * h + 10]), "=r"(r[32 * h + 11]),
          "=r"(r[32 * h + 12]), "=r"(r[32 * h + 13]), "=r"(r[32 * h + 14]),
          "=r"(r[32 * h + 15]), "=r"(r[32 * h + 16]), "=r"(r[32 * h + 17]),
          "=r"(r[32 * h + 18]), "=r"(r[32 * h + 19]), "=r"(r[32 * h + 20]),
          "=r"(r[32 * h + 21]), "=r"(r[32 * h + 22]), "=r"(r[32 * h + 23]),
          "=r"(r[32 * h + 24]), "=r"(r[32 * h + 25]), "=r"(r[32 * h + 26]),
          "=r"(r[32 * h + 27]), "=r"(r[32 * h + 28]), "=r"(r[32 * h + 29]),
          "=r"(r[32 * h + 30]), "=r"(r[32 * h + 31])
        : "r"(taddr + 32 * h));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int h = 0; h < 2; ++h)
#pragma unroll
    for (int i = 0; i < 32; ++i) v[h][i] = __uint_as_float(r[32 * h + i]);
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
      "%28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
      "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
      "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
      "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
      "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
      "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
      : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// 16 consecutive 32-bit columns of this thread's TMEM lane; completes at the
// next tmem_wait_st().
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
      "r"(v[15])
      : "memory");
}

__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&v)[8]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
      : "memory");
}

__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *map, int x, int y,
                                            int z, uint32_t bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];\n\t}" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}

// Packed pairs of floats (lo half first) and the f32x2 arithmetic on them:
// each half is rounded as the scalar instruction would round it.
__device__ __forceinline__ uint64_t pack_f32x2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void unpack_f32x2(uint64_t v, float &lo, float &hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t fma_f32x2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ uint64_t add_f32x2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t sub_f32x2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}

// max of three floats (exact; a NaN operand is ignored, as by fmaxf)
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// 2^x by the special-function unit (ex2.approx, relative error ~2^-22).
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Byte offset of (row, 16-byte chunk) inside a [128 rows][128 B] swizzled half.
__device__ __forceinline__ uint32_t sw128(int row, int chunk) {
  return row * 128 + ((chunk ^ (row & 7)) << 4);
}

// ---- work order -------------------------------------------------------------
// The work items are (sequence s, query tile mt, kv head g) with a query
// tile of PT positions; an item costs one step per 64-key tile it attends,
// nkv = (prefix + last position of the tile) / 64 + 1, which grows with mt.
// CTAs start in block-index order, so the CTA of linear index r takes the
// item of rank r in the order "most steps first" (ties: by s, then mt, then
// g): long items start first and short ones fill the end of the grid.  Every
// CTA finds its item from a histogram of the step counts (one thread per
// sequence, counts clamped to kLptBins - 1, which only merges ties) and two
// block scans; the kernel uses it only while num_seqs <= kPfThreads, so
// that this prologue stays one round of loads.  Returns false when the CTA has no item.  Sequences
// with rows beyond the grid's tiles or with context_lens < q_len are
// reported (PA_DEVERR_SHAPE); the latter have no items.
constexpr int kLptBins = 1024;
static_assert((kLptBins + 32 + 5) * 4 <= kKStages * kTileBytes2,
              "work-order scratch does not fit the K stages");
__device__ __forceinline__ int lpt_bin(int prefix, int q_len, int mt, int PT) {
  const int last = mt * PT + min(PT, q_len - mt * PT) - 1;  // last position of the tile
  return min((prefix + last) / kPfKeys + 1, kLptBins - 1);
}
// exclusive block scan of one int per thread (kPfThreads threads)
__device__ __forceinline__ int block_excl_scan(int v, int *wsum, int &total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) wsum[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int t = lane < kPfThreads / 32 ? wsum[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, t, o);
      if (lane >= o) t += y;
    }
    if (lane < kPfThreads / 32) wsum[lane] = t;  // inclusive warp prefix
  }
  __syncthreads();
  total = wsum[kPfThreads / 32 - 1];
  const int before = warp > 0 ? wsum[warp - 1] : 0;
  __syncthreads();  // wsum is reused by the next scan
  return before + x - v;
}
template <int PT>
__device__ bool pick_work_item(const PrefillParams &p, int gx, int *sc, int &s_out, int &mt_out,
                               int &g_out) {
  int *hist = sc;                     // [kLptBins] items per step count
  int *wsum = sc + kLptBins;          // [kPfThreads / 32] block-scan scratch
  int *res = sc + kLptBins + 32;      // picked bin, items before it, s, mt, g
  const int tid = threadIdx.x;
  const int r = (int)(blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z));
  for (int i = tid; i < kLptBins; i += kPfThreads) hist[i] = 0;
  if (tid == 0) res[0] = -1;
  __syncthreads();
  const int ns = p.num_seqs, hkv = p.hkv;
  const int spt = (ns + kPfThreads - 1) / kPfThreads;
  const int s0 = min(ns, tid * spt), s1 = min(ns, s0 + spt);
  // pass 1: the histogram (runs of equal counts added at once)
  for (int s = s0; s < s1; ++s) {
    const int q_len = __ldg(p.cu_seqlens + s + 1) - __ldg(p.cu_seqlens + s);
    if (q_len <= 0) continue;
    const int prefix = __ldg(p.context_lens + s) - q_len;
    if (prefix < 0) {
      report(p.err, PA_DEVERR_SHAPE);
      continue;
    }
    if (q_len > gx * PT) report(p.err, PA_DEVERR_SHAPE);  // rows no CTA covers
    const int T = min((q_len + PT - 1) / PT, gx);
    int run_bin = lpt_bin(prefix, q_len, 0, PT), run = 0;
    for (int mt = 0; mt < T; ++mt) {
      const int b = lpt_bin(prefix, q_len, mt, PT);
      if (b != run_bin) {
        atomicAdd(hist + run_bin, run * hkv);
        run_bin = b;
        run = 0;
      }
      ++run;
    }
    if (T > 0) atomicAdd(hist + run_bin, run * hkv);
  }
  __syncthreads();
  // pass 2 (warp 0): the bin of rank r, counting bins from the top
  if (tid < 32) {
    constexpr int kPer = kLptBins / 32;
    int sum = 0;
#pragma unroll 4
    for (int k = 0; k < kPer; ++k) sum += hist[kLptBins - 1 - tid * kPer - k];
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (tid >= o) incl += y;
    }
    const int excl = incl - sum;
    if (r >= excl && r < incl) {
      int acc = excl;
      for (int k = 0; k < kPer; ++k) {
        const int b = kLptBins - 1 - tid * kPer - k;
        if (r < acc + hist[b]) {
          res[0] = b;
          res[1] = acc;
          break;
        }
        acc += hist[b];
      }
    }
  }
  __syncthreads();
  const int vb = res[0];
  if (vb < 0) return false;  // rank past the last item
  const int j = r - res[1];
  // pass 3: the j-th item of bin vb in (s, mt, g) order
  int cnt = 0;
  for (int s = s0; s < s1; ++s) {
    const int q_len = __ldg(p.cu_seqlens + s + 1) - __ldg(p.cu_seqlens + s);
    const int prefix = __ldg(p.context_lens + s) - q_len;
    if (q_len <= 0 || prefix < 0) continue;
    const int T = min((q_len + PT - 1) / PT, gx);
    for (int mt = 0; mt < T; ++mt) cnt += lpt_bin(prefix, q_len, mt, PT) == vb ? hkv : 0;
  }
  int total;
  const int before = block_excl_scan(cnt, wsum, total);
  if (j >= before && j < before + cnt) {
    int k = j - before;
    for (int s = s0; s < s1 && k >= 0; ++s) {
      const int q_len = __ldg(p.cu_seqlens + s + 1) - __ldg(p.cu_seqlens + s);
      const int prefix = __ldg(p.context_lens + s) - q_len;
      if (q_len <= 0 || prefix < 0) continue;
      const int T = min((q_len + PT - 1) / PT, gx);
      for (int mt = 0; mt < T; ++mt) {
        if (lpt_bin(prefix, q_len, mt, PT) != vb) continue;
        if (k < hkv) {
          res[2] = s;
          res[3] = mt;
          res[4] = k;
          k = -1;
          break;
        }
        k -= hkv;
      }
    }
  }
  __syncthreads();
  s_out = res[2];
  mt_out = res[3];
  g_out = res[4];
  // the scratch becomes a TMA destination: order these generic writes first
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  return true;
}

template <int G>
__global__ void __launch_bounds__(kPfThreads, 2)
    prefill_kernel(const __grid_constant__ CUtensorMap tmap_k,
                   const __grid_constant__ CUtensorMap tmap_v,
                   const __grid_constant__ CUtensorMap tmap_nk,
                   const __grid_constant__ CUtensorMap tmap_nv, const PrefillParams p) {
  constexpr int PT = kPfRows / G;  // query positions per tile
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t base = smem_addr(smem);
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kOffBar);
  // barrier slots ("0" slots: + 8 * stage, or + 8 * (tile & 1)), laid out
  // from the stage counts: no two barriers share a slot
  const uint32_t b_k_full0 = smem_addr(bars + kBarKFull);
  const uint32_t b_k_empty0 = smem_addr(bars + kBarKEmpty);
  const uint32_t b_v_full0 = smem_addr(bars + kBarVFull);
  const uint32_t b_v_empty0 = smem_addr(bars + kBarVEmpty);
  const uint32_t b_q_ready = smem_addr(bars + kBarQ);
  const uint32_t b_s_full0 = smem_addr(bars + kBarS);  // scores of tile j in buffer j & 1
  const uint32_t b_p_full0 = smem_addr(bars + kBarP);  // P of tile j written over them
  const uint32_t b_o_full0 = smem_addr(bars + kBarO);  // PV of tile j done (j & 1)
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + kBarTmem);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(bars + kBarAbort);

  const int tid = threadIdx.x, lane = tid & 31;
  // broadcast from lane 0: the compiler then knows every role branch below
  // is warp-uniform
  const int warp = __shfl_sync(0xffffffffu, tid >> 5, 0);
  // the work item of this CTA: longest first (pick_work_item; the scratch
  // is the K stage region, which no TMA has written yet) while one thread
  // per sequence suffices, else in grid order with the last tiles of a
  // chunk (the most keys, causal) first
  int s, mt, g;
  if (p.num_seqs <= kPfThreads) {
    if (!pick_work_item<PT>(p, (int)gridDim.x, reinterpret_cast<int *>(smem + kOffK), s, mt, g))
      return;
  } else {
    mt = (int)gridDim.x - 1 - (int)blockIdx.x;
    g = blockIdx.y;
    s = blockIdx.z;
    const int ql = __ldg(p.cu_seqlens + s + 1) - __ldg(p.cu_seqlens + s);
    if (mt * PT >= ql) return;  // this tile has no query
    if (__ldg(p.context_lens + s) < ql) {
      if (tid == 0) report(p.err, PA_DEVERR_SHAPE);
      return;
    }
    // a chunk longer than max_q_len has rows no CTA covers: reported
    if (mt == (int)gridDim.x - 1 && mt * PT + PT < ql && tid == 0)
      report(p.err, PA_DEVERR_SHAPE);
  }
  const int q0 = __ldg(p.cu_seqlens + s);
  const int q_len = __ldg(p.cu_seqlens + s + 1) - q0;
  const int pos0 = mt * PT;
  const int n = __ldg(p.context_lens + s);
  const int prefix = n - q_len;
  const int npos = min(PT, q_len - pos0);
  const int rows = npos * G;
  const int kmax = prefix + pos0 + npos - 1;  // last key any row of the tile sees
  const int nkv = kmax / kPfKeys + 1;
  const float c = p.qk_scale_log2;

  if (tid == 0) {
    for (int i = 0; i < kKStages; ++i) {
      mbar_init(b_k_full0 + 8 * i, 1);
      mbar_init(b_k_empty0 + 8 * i, 1);
    }
    for (int i = 0; i < kVStages; ++i) {
      mbar_init(b_v_full0 + 8 * i, 1);
      mbar_init(b_v_empty0 + 8 * i, 1);
    }
    constexpr int kSoft = 32 * kPfSoftWarps;
    mbar_init(b_q_ready, kSoft);
    for (int i = 0; i < 2; ++i) {
      mbar_init(b_s_full0 + 8 * i, 1);
      mbar_init(b_p_full0 + 8 * i, kSoft);
      mbar_init(b_o_full0 + 8 * i, 1);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tmem_o = tmem + kTmemO;

  if (warp == 0 || warp == 2) {
    // ---- TMA loaders: warp 0 brings the K tiles, warp 2 the V tiles, each
    //      into stage j % stages once the MMA that read the stage's previous
    //      tile is done;
    //      separate loaders halve the per-tile issue time (16 boxes each) ----
    const bool is_k = warp == 0;
    const CUtensorMap *map = is_k ? &tmap_k : &tmap_v;
    // fused store: pages of the chunk come from the new rows
    const bool fused = p.new_k != nullptr;
    const CUtensorMap *nmap = is_k ? &tmap_nk : &tmap_nv;
    const uint16_t *nrows = is_k ? p.new_k : p.new_v;
    const long long ntok = is_k ? p.new_k_tok : p.new_v_tok;
    const uint16_t *pool = is_k ? p.k_cache : p.v_cache;
    const uint32_t dst0 = base + (is_k ? kOffK : kOffV);
    const uint32_t b_full0 = is_k ? b_k_full0 : b_v_full0;
    const uint32_t b_empty0 = is_k ? b_k_empty0 : b_v_empty0;
    const int nst = is_k ? kKStages : kVStages;
    if (lane == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
      if (fused)
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(nmap))
                     : "memory");
    }
    const int32_t *row = p.block_tables + (long long)s * p.bt_stride;
    // block-table entries of eight tiles (32 pages) per round of loads, one
    // per lane: -1 = no key in the page (left as it is: masked), -2 = bad entry
    long long ph_lane = -1;
    int j = 0;
    for (; j < nkv; ++j) {
      const int st = j % nst, round = j / nst;
      const uint32_t dst = dst0 + st * kTileBytes2, b_full = b_full0 + 8 * st;
      if (j % (32 / kPfPages) == 0) {
        const int lb = j * kPfPages + lane;
        const bool has = lb * kBlockSize < n;
        const long long ph = has && lb < p.bt_stride ? __ldg(row + lb) : -2;
        ph_lane = !has ? -1 : (ph >= 0 && ph < p.num_blocks) ? ph : -2;
      }
      if (round > 0 && !__all_sync(0xffffffffu, mbar_wait(b_empty0 + 8 * st, (round - 1) & 1,
                                                           abort_flag, p.err)))
        break;
      // lane L < 4 handles page L of the tile; its kind: pool page (TMA
      // from the pool), chunk page (fused: TMA from the new rows), the page
      // that straddles the prefix (fused: assembled by the warp) or none
      const long long phys =
          __shfl_sync(0xffffffffu, ph_lane, (j % (32 / kPfPages)) * kPfPages + lane % kPfPages);
      const bool mine = lane < kPfPages;
      const int kp0 = j * kPfKeys + (lane % kPfPages) * kBlockSize;  // first key of the page
      const bool in_chunk = fused && kp0 >= prefix;
      const bool straddle = fused && kp0 < prefix && kp0 + kBlockSize > prefix;
      const bool by_tma = phys != -1 && !straddle && (in_chunk || phys >= 0);
      const unsigned okm = __ballot_sync(0xffffffffu, mine && by_tma);
      if (is_k && (__ballot_sync(0xffffffffu, mine && phys == -2 && !in_chunk) != 0u) &&
          lane == 0)
        report(p.err, PA_DEVERR_BLOCK_INDEX);
      const unsigned mixm = __ballot_sync(0xffffffffu, mine && straddle && phys >= 0);
      if (mixm) {
        // rows 0 .. prefix - kp - 1 from the pool page, the rest from the new
        // rows (rows past the sequence: zero), written in the layout the TMA
        // uses (128-byte swizzle); then made visible to the tensor core
        const int pg = __ffs(mixm) - 1;
        const long long ph = __shfl_sync(0xffffffffu, phys, pg);
        const int kp = j * kPfKeys + pg * kBlockSize;
        // 16 rows x 16 chunks: 8 per lane, all loads issued before the stores
        uint4 v[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int i = lane + 32 * k, r = i >> 4, c = i & 15;
          v[k] = make_uint4(0u, 0u, 0u, 0u);
          if (kp + r < n) {
            const uint16_t *src =
                kp + r < prefix
                    ? pool + ((ph * kBlockSize + r) * p.hkv + g) * kHeadDim + c * 8
                    : nrows + (long long)(q0 + kp + r - prefix) * ntok + g * kHeadDim + c * 8;
            v[k] = __ldg(reinterpret_cast<const uint4 *>(src));
          }
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int i = lane + 32 * k, r = i >> 4, c = i & 15;
          const uint32_t a = dst + (c >> 3) * kHalfBytes + pg * kBlockSize * 128 + sw128(r, c & 7);
          asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(v[k].x),
                       "r"(v[k].y), "r"(v[k].z), "r"(v[k].w)
                       : "memory");
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      }
      __syncwarp();
      if (lane == 0) mbar_arrive_expect_tx(b_full, __popc(okm) * 2u * kBlockSize * 64 * 2);
      __syncwarp();
      // one page at a time, its index broadcast to the whole warp
#pragma unroll
      for (int pg = 0; pg < kPfPages; ++pg) {
        if (!((okm >> pg) & 1u)) continue;
        const long long ph = __shfl_sync(0xffffffffu, phys, pg);
        const int kp = j * kPfKeys + pg * kBlockSize;
        const bool from_new = fused && kp >= prefix;
        // pool page: token slots of block ph; chunk page: the new rows from
        // token q0 + kp - prefix (rows past the last token are zero-filled)
        const int z = from_new ? q0 + kp - prefix : (int)(ph * kBlockSize);
#pragma unroll
        for (int h = 0; h < 2; ++h)
          tma_load_3d(dst + h * kHalfBytes + pg * kBlockSize * 128, from_new ? nmap : map, h * 64,
                      g, z, b_full);
      }
    }
    if (fused && !*abort_flag) {
      // the fused store: this CTA's positions pos0 .. pos0 + npos - 1, kv
      // head g (warp 0: K rows, warp 2: V rows), 16-byte chunks over the lanes
      uint16_t *dstp = is_k ? p.k_store : p.v_store;
      const long long num_slots = p.num_blocks * kBlockSize;
      // up to 21 positions x 16 chunks; four per lane per round, the loads of
      // a round issued before its stores
      for (int i0 = 0; i0 < npos * 16; i0 += 4 * 32) {
        long long slot[4];
        uint4 v[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int i = i0 + lane + 32 * k, r = i >> 4, c = i & 15;
          slot[k] = -1;
          if (i < npos * 16) {
            const long long t = q0 + pos0 + r;
            slot[k] = __ldg(p.slot_mapping + t);
            v[k] = __ldg(reinterpret_cast<const uint4 *>(nrows + t * ntok + g * kHeadDim + c * 8));
          }
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int c = (i0 + lane + 32 * k) & 15;
          if (slot[k] < 0) continue;  // padding, or past this CTA's rows
          if (slot[k] >= num_slots) {
            if (c == 0) report(p.err, PA_DEVERR_SLOT_INDEX);
            continue;
          }
          *reinterpret_cast<uint4 *>(dstp + (slot[k] * p.hkv + g) * kHeadDim + c * 8) = v[k];
        }
      }
    }
    if (lane == 0 && *abort_flag) {
      // copies in flight must land before the CTA's shared memory is released
      volatile int never = 0;
      for (int i = j > nst ? j - nst : 0; i < j; ++i)
        mbar_wait(b_full0 + 8 * (i % nst), (i / nst) & 1, &never, nullptr);
    }
    __syncwarp();
  } else if (warp == 1 || warp == 3) {
    // ---- MMA issuers, each a whole converged warp (see umma_f16_ta).  Warp
    //      1 issues S_j = Q K_j^T into buffer j & 1 (Q from shared memory)
    //      once the PV MMA of tile j - 2, which read that buffer, is done;
    //      warp 3 issues O += (P_hi + P_lo) V_j with P from buffer j & 1.
    //      Two issuers keep either chain from waiting behind the other ----
    constexpr uint32_t idesc_qk = umma_idesc(0, kPfKeys), idesc_pv = umma_idesc(1, kHeadDim);
    constexpr unsigned kAll = 0xffffffffu;
    uint32_t last_bar = 0;  // barrier of this warp's latest commit (drained on abort)
    int last_par = 0;
    if (warp == 1) {
      bool ok = __all_sync(kAll, mbar_wait(b_q_ready, 0, abort_flag, p.err));
      tc_fence_after();
      for (int j = 0; j < nkv && ok; ++j) {
        const int ks2 = j % kKStages;
        ok = __all_sync(kAll, mbar_wait(b_k_full0 + 8 * ks2, (j / kKStages) & 1, abort_flag,
                                        p.err));
        // buffer j & 1 held P of tile j - 2: the PV that read it is done
        if (ok && j >= 2)
          ok = __all_sync(kAll, mbar_wait(b_o_full0 + 8 * (j & 1), ((j - 2) >> 1) & 1,
                                          abort_flag, p.err));
        if (!ok) break;
        tc_fence_after();
        const uint32_t sb = tmem + (j & 1) * kTmemSCols;
        // 8 k-steps of 16 dims (4 per 64-dim half)
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          const uint32_t koff = (ks >> 2) * kHalfBytes + (ks & 3) * 32;
          const uint32_t qoff = (ks >> 2) * kQHalf + (ks & 3) * 32;
          umma_f16_ss(sb, umma_desc(base + kOffQ + qoff, 16, 1024),
                      umma_desc(base + kOffK + ks2 * kTileBytes2 + koff, 16, 1024), idesc_qk,
                      ks > 0);
        }
        umma_commit(b_s_full0 + 8 * (j & 1));
        umma_commit(b_k_empty0 + 8 * ks2);  // the K stage may be refilled
        last_bar = b_s_full0 + 8 * (j & 1);
        last_par = (j >> 1) & 1;
      }
    } else {
      for (int j = 0; j < nkv; ++j) {
        // 2 x 4 k-steps of 16 keys, P_j from buffer j & 1 (8 columns per
        // step); V is MN-major (dims contiguous): LBO = distance between the
        // two 64-dim halves, SBO = 8 keys
        if (!__all_sync(kAll, mbar_wait(b_p_full0 + 8 * (j & 1), (j >> 1) & 1, abort_flag, p.err)))
          break;
        if (!__all_sync(kAll, mbar_wait(b_v_full0 + 8 * (j % kVStages), (j / kVStages) & 1,
                                        abort_flag, p.err)))
          break;
        tc_fence_after();
        const uint32_t vb = base + kOffV + (j % kVStages) * kTileBytes2;
        const uint32_t pb = tmem + (j & 1) * kTmemSCols;
#pragma unroll
        for (int part = 0; part < 2; ++part) {
#pragma unroll
          for (int ks = 0; ks < kPfKeys / 16; ++ks)
            umma_f16_ta(tmem_o, pb + part * (kTmemSCols / 2) + ks * 8,
                        umma_desc(vb + ks * 16 * 128, kHalfBytes, 1024), idesc_pv,
                        (j > 0 || part > 0 || ks > 0) ? 1u : 0u);
        }
        umma_commit(b_o_full0 + 8 * (j & 1));
        umma_commit(b_v_empty0 + 8 * (j % kVStages));  // the V stage may be refilled
        last_bar = b_o_full0 + 8 * (j & 1);
        last_par = (j >> 1) & 1;
      }
    }
    if (__any_sync(kAll, *abort_flag != 0) && last_bar) {
      // let this warp's issued MMAs finish before TMEM is released (bounded)
      volatile int never = 0;
      mbar_wait(last_bar, last_par, &never, nullptr);
    }
    __syncwarp();
  } else {
    // ---- softmax / epilogue warps 4..7: warp w serves TMEM lane quarter
    //      w % 4 (rows 32 (w % 4) .. + 31); a thread owns its row's scores,
    //      P and output columns ----------------------------------------------
    const int lb = 32 * (warp & 3);  // TMEM lanes this warp may access
    const int r = lb + lane;         // row of the tile
    const int rpos = r / G;          // query position in the tile
    const int hs = r % G;            // query head in the group
    const bool rvalid = r < rows;
    const int limit = rvalid ? prefix + pos0 + rpos : -1;  // last key this row sees
    const uint32_t trow = (uint32_t)lb << 16;

    // Q row r = q[q0 + pos0 + rpos][g * G + hs][:] into the Q tile in shared
    // memory (K-major, two 64-dim halves, 128-byte swizzle, the layout the
    // TMA gives the K tiles), then made visible to the tensor core
    {
      const uint4 *src = reinterpret_cast<const uint4 *>(
          p.q + ((long long)(q0 + pos0 + rpos) * p.hq + g * G + hs) * kHeadDim);
      uint4 qv[16];
#pragma unroll
      for (int c16 = 0; c16 < 16; ++c16)
        qv[c16] = rvalid ? __ldg(src + c16) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
      for (int c16 = 0; c16 < 16; ++c16) {
        qv[c16].x = (qv[c16].x & p.q_and) ^ p.q_xor;
        qv[c16].y = (qv[c16].y & p.q_and) ^ p.q_xor;
        qv[c16].z = (qv[c16].z & p.q_and) ^ p.q_xor;
        qv[c16].w = (qv[c16].w & p.q_and) ^ p.q_xor;
      }
#pragma unroll
      for (int c16 = 0; c16 < 16; ++c16) {
        const uint32_t a = base + kOffQ + (c16 >> 3) * kQHalf + sw128(r, c16 & 7);
        asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(qv[c16].x),
                     "r"(qv[c16].y), "r"(qv[c16].z), "r"(qv[c16].w)
                     : "memory");
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      mbar_arrive(b_q_ready);
    }

    // m: reference max (base-2 units) of this row's exponentials.  It moves
    // only when a tile's max exceeds it by more than 8 (a factor 256), so P
    // stays <= 256 and O needs rescaling (after the previous PV) rarely.
    // l: the row sum.
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < nkv && ok; ++j) {
      // warp-uniform: tcgen05.ld / st below are warp-collective
      ok = __all_sync(0xffffffffu, mbar_wait(b_s_full0 + 8 * (j & 1), (j >> 1) & 1, abort_flag,
                                            p.err));
      if (!ok) break;
      tc_fence_after();
      const uint32_t sb = tmem + (j & 1) * kTmemSCols;
      const int key0 = j * kPfKeys;
      // every row of the tile sees every key of it: no masks
      const bool tile_full = key0 + kPfKeys - 1 <= prefix + pos0;
      float sv[2][32];
      tmem_ld64(sb + trow, sv);
      // masked keys (diagonal and last tiles only) become -inf before the
      // max, so the max and the exponentials below have a single, unmasked
      // body (selects, not branches)
      if (!tile_full) {
#pragma unroll
        for (int cc = 0; cc < 2; ++cc)
#pragma unroll
          for (int i = 0; i < 32; ++i)
            sv[cc][i] = key0 + cc * 32 + i <= limit ? sv[cc][i] : -INFINITY;
      }
      // eight independent max chains, two keys per three-input max
      float mx8[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) mx8[u] = -INFINITY;
#pragma unroll
      for (int cc = 0; cc < 2; ++cc)
#pragma unroll
        for (int i = 0; i < 32; i += 2)
          mx8[(i >> 1) & 7] = fmax3(mx8[(i >> 1) & 7], sv[cc][i], sv[cc][i + 1]);
      const float mx = fmax3(fmax3(mx8[0], mx8[1], mx8[2]), fmax3(mx8[3], mx8[4], mx8[5]),
                             fmaxf(mx8[6], mx8[7]));
      const float mxc = mx * c;
      const bool grow = mxc > m + 8.f;
      const float m_new = grow ? mxc : m;
      const float alpha = grow && m != -INFINITY ? exp2f(m - m_new) : 1.f;
      m = m_new;
      // P = exp2(S c - m) in place (its row sum is taken with the split of P
      // below).  A masked
      // key has S = -inf, so its exponent is -inf and 2^x = +0; a row with no
      // key yet (m = -inf: rows past the chunk) takes offset 0 instead of
      // +inf, which keeps it -inf rather than NaN.
      const float neg_m = m == -INFINITY ? 0.f : -m;
      // (the exponents of a key pair in one packed f32x2 multiply-add)
      const uint64_t c2 = pack_f32x2(c, c), nm2 = pack_f32x2(neg_m, neg_m);
#pragma unroll
      for (int cc = 0; cc < 2; ++cc)
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          float x0, x1;
          unpack_f32x2(fma_f32x2(pack_f32x2(sv[cc][i], sv[cc][i + 1]), c2, nm2), x0, x1);
          sv[cc][i] = ex2_approx(x0);
          sv[cc][i + 1] = ex2_approx(x1);
        }
      // rows whose reference max moved rescale their O row, once the PV of
      // tile j - 1 is done and before that of tile j (warp-wide: tcgen05.ld /
      // st are collective)
      if (__any_sync(0xffffffffu, alpha != 1.f)) {
        if (j >= 1) {
          ok = __all_sync(0xffffffffu, mbar_wait(b_o_full0 + 8 * ((j - 1) & 1),
                                                ((j - 1) >> 1) & 1, abort_flag, p.err));
          if (!ok) break;
          tc_fence_after();
        }
#pragma unroll 1
        for (int cc = 0; cc < kHeadDim / 32; ++cc) {
          float ov[32];
          tmem_ld32(tmem_o + trow + cc * 32, ov);
#pragma unroll
          for (int i = 0; i < 32; ++i) ov[i] *= alpha;
          tmem_st32(tmem_o + trow + cc * 32, ov);
        }
      }
      const float l_scaled = l * alpha;
      // P as bf16 hi + lo over the scores of this row's TMEM lane (A operands
      // of the PV MMAs; keys 2i and 2i + 1 share column i, the even key in the
      // low half; hi parts in the buffer's columns 0..31, lo parts in
      // 32..63).  hi is e with the low 16 mantissa bits cleared (exactly a
      // bf16, one byte permute per key pair); lo = e - hi is exact in fp32
      // (one packed subtraction per pair) and rounded to nearest even bf16
      // (one packed conversion per pair), so hi + lo is e within 2^-15
      // relative, without bias.
      // The row sum of the exponentials is taken here, on the key pairs the
      // subtraction packs anyway (eight chains, two per packed add); 8-column
      // stores keep the loop within the registers of two CTAs per SM.
      uint64_t ps4[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        uint32_t hi[8], lo[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float e0 = sv[cc >> 1][16 * (cc & 1) + 2 * i];
          const float e1 = sv[cc >> 1][16 * (cc & 1) + 2 * i + 1];
          const uint32_t u0 = __float_as_uint(e0), u1 = __float_as_uint(e1);
          hi[i] = __byte_perm(u0, u1, 0x7632);
          const uint64_t e2 = pack_f32x2(e0, e1);
          ps4[i & 3] = add_f32x2(ps4[i & 3], e2);
          float d0, d1;
          unpack_f32x2(sub_f32x2(e2, pack_f32x2(__uint_as_float(u0 & 0xFFFF0000u),
                                                __uint_as_float(u1 & 0xFFFF0000u))),
                       d0, d1);
          asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(lo[i]) : "f"(d1), "f"(d0));
        }
        tmem_st8(sb + trow + cc * 8, hi);
        tmem_st8(sb + trow + kTmemSCols / 2 + cc * 8, lo);
      }
      {
        float ps8[8];
#pragma unroll
        for (int u = 0; u < 4; ++u) unpack_f32x2(ps4[u], ps8[2 * u], ps8[2 * u + 1]);
        l = l_scaled + (((ps8[0] + ps8[1]) + (ps8[2] + ps8[3])) +
                        ((ps8[4] + ps8[5]) + (ps8[6] + ps8[7])));
      }
      tmem_wait_st();
      // keys past the end of the sequence: their V rows may hold anything;
      // zero them so that 0-weight rows add exactly 0 (last tile only, once
      // the V tile has landed)
      if (key0 + kPfKeys > n) {
        ok = __all_sync(0xffffffffu, mbar_wait(b_v_full0 + 8 * (j % kVStages),
                                              (j / kVStages) & 1, abort_flag, p.err));
        if (!ok) break;
        const uint32_t vb = base + kOffV + (j % kVStages) * kTileBytes2;
        for (int i = r; i < kPfKeys * 16; i += kPfRows) {
          const int key = i >> 4, ch = i & 15;
          if (key0 + key >= n) {
            const uint32_t a = vb + (ch >> 3) * kHalfBytes + sw128(key, ch & 7);
            asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(a), "r"(0u) : "memory");
          }
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      }
      tc_fence_before();
      mbar_arrive(b_p_full0 + 8 * (j & 1));
    }
    // epilogue: O / l -> out[q0 + pos0 + rpos][g * G + hs][:]
    if (ok && nkv > 0)
      ok = __all_sync(0xffffffffu, mbar_wait(b_o_full0 + 8 * ((nkv - 1) & 1),
                                            ((nkv - 1) >> 1) & 1, abort_flag, p.err));
    tc_fence_after();
    if (ok) {
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const long long orow = ((long long)(q0 + pos0 + rpos) * p.hq + g * G + hs) * kHeadDim;
#pragma unroll 1
      for (int cc = 0; cc < kHeadDim / 32; ++cc) {
        float ov[32];
        tmem_ld32(tmem_o + trow + cc * 32, ov);
        if (rvalid) {
          if (p.out_f32) {
            float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(p.out) + orow + cc * 32);
#pragma unroll
            for (int i = 0; i < 8; ++i)
              dst[i] = make_float4(ov[4 * i] * inv, ov[4 * i + 1] * inv, ov[4 * i + 2] * inv,
                                   ov[4 * i + 3] * inv);
          } else {
            uint4 *dst = reinterpret_cast<uint4 *>(static_cast<uint16_t *>(p.out) + orow + cc * 32);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              uint4 w;
              w.x = float2_to_bf16x2(ov[8 * i] * inv, ov[8 * i + 1] * inv);
              w.y = float2_to_bf16x2(ov[8 * i + 2] * inv, ov[8 * i + 3] * inv);
              w.z = float2_to_bf16x2(ov[8 * i + 4] * inv, ov[8 * i + 5] * inv);
              w.w = float2_to_bf16x2(ov[8 * i + 6] * inv, ov[8 * i + 7] * inv);
              dst[i] = w;
            }
          }
        }
      }
    }
    tc_fence_before();
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kTmemCols)
                 : "memory");
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// (dim 128, kv head, token slot) view of a pool; one box = 64 dims x 1 head x
// 16 slots (one page of one head), 128-byte swizzle.
bool pool_map(CUtensorMap *map, const void *pool, long long num_blocks, int hkv) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encoder();
  if (!enc) return false;
  cuuint64_t dims[3] = {(cuuint64_t)kHeadDim, (cuuint64_t)hkv,
                        (cuuint64_t)num_blocks * kBlockSize};
  cuuint64_t strides[2] = {(cuuint64_t)kHeadDim * 2, (cuuint64_t)hkv * kHeadDim * 2};
  cuuint32_t box[3] = {64, 1, (cuuint32_t)kBlockSize};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(pool), dims, strides,
             box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// (dim 128, kv head, token) view of the new rows (token stride in elements,
// a multiple of 8); the same box as pool_map: 64 dims x 1 head x 16 tokens.
bool rows_map(CUtensorMap *map, const void *rows, long long num_tokens, int hkv,
              long long tok_stride) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encoder();
  if (!enc) return false;
  cuuint64_t dims[3] = {(cuuint64_t)kHeadDim, (cuuint64_t)hkv, (cuuint64_t)num_tokens};
  cuuint64_t strides[2] = {(cuuint64_t)kHeadDim * 2, (cuuint64_t)tok_stride * 2};
  cuuint32_t box[3] = {64, 1, (cuuint32_t)kBlockSize};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(rows), dims, strides,
             box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int G>
cudaError_t launch_prefill(const CUtensorMap &tk, const CUtensorMap &tv, const CUtensorMap &tnk,
                           const CUtensorMap &tnv, const PrefillParams &pp,
                           int max_q_len, cudaStream_t s, int device) {
  static std::atomic<bool> configured[64] = {};
  const cudaError_t e = set_smem_once(configured, prefill_kernel<G>, device, kPfSmem);
  if (e != cudaSuccess) return e;
  // two CTAs per SM: all of the unified L1 / shared memory as shared memory
  // (a hint; setting it again is harmless)
  cudaFuncSetAttribute(prefill_kernel<G>, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
  constexpr int PT = kPfRows / G;
  dim3 grid((max_q_len + PT - 1) / PT, pp.hkv, pp.num_seqs);
  prefill_kernel<G><<<grid, kPfThreads, kPfSmem, s>>>(tk, tv, tnk, tnv, pp);
  return cudaGetLastError();
}

}  // namespace
}  // namespace pa

namespace pa {
namespace {
pa_status prefill_entry(void *out, int32_t out_dtype, const void *q, const int32_t *cu_seqlens,
                        int32_t num_seqs, int32_t total_tokens, int32_t max_q_len,
                        const void *k_cache, const void *v_cache, int64_t num_blocks,
                        const int32_t *block_tables, int32_t block_table_stride,
                        const int32_t *context_lens, int32_t num_q_heads, int32_t num_kv_heads,
                        int32_t head_dim, int32_t block_size, float scale, int32_t *error_flags,
                        void *stream, const void *new_k, const void *new_v,
                        int64_t new_k_tok_stride, int64_t new_v_tok_stride,
                        const int32_t *slot_mapping) {
  if (num_seqs < 0 || total_tokens < 0 || max_q_len < 0 || num_blocks < 0)
    return PA_ERR_INVALID_ARG;
  if (out_dtype != PA_DTYPE_BF16 && out_dtype != PA_DTYPE_F32) return PA_ERR_INVALID_ARG;
  if (head_dim != kHeadDim || block_size != kBlockSize) return PA_ERR_UNSUPPORTED;
  if (!(num_kv_heads == 1 || num_kv_heads == 2 || num_kv_heads == 4 || num_kv_heads == 8))
    return PA_ERR_UNSUPPORTED;
  if (num_q_heads < num_kv_heads || num_q_heads % num_kv_heads || num_q_heads / num_kv_heads > 8)
    return PA_ERR_UNSUPPORTED;
  if (!std::isfinite(scale)) return PA_ERR_INVALID_ARG;
  if (num_seqs == 0 || total_tokens == 0 || max_q_len == 0) return PA_OK;
  if (num_seqs > 65535) return PA_ERR_UNSUPPORTED;
  if (num_blocks < 1 || num_blocks > (long long)(0x7fffffff / kBlockSize))
    return PA_ERR_INVALID_ARG;
  if (!out || !q || !cu_seqlens || !k_cache || !v_cache || !block_tables || !context_lens)
    return PA_ERR_INVALID_ARG;
  if (block_table_stride < 1) return PA_ERR_INVALID_ARG;
  auto misaligned = [](const void *x) { return (reinterpret_cast<uintptr_t>(x) & 15) != 0; };
  if (misaligned(out) || misaligned(q) || misaligned(k_cache) || misaligned(v_cache))
    return PA_ERR_INVALID_ARG;
  const bool fused = new_k != nullptr;
  if (fused) {
    if (!new_v || !slot_mapping || misaligned(new_k) || misaligned(new_v)) return PA_ERR_INVALID_ARG;
    if (new_k_tok_stride < (int64_t)num_kv_heads * kHeadDim ||
        new_v_tok_stride < (int64_t)num_kv_heads * kHeadDim || new_k_tok_stride % 8 ||
        new_v_tok_stride % 8)
      return PA_ERR_INVALID_ARG;
  }
  int device = -1;
  if (cudaGetDevice(&device) != cudaSuccess) return PA_ERR_DEVICE;
  CUtensorMap tk, tv, tnk, tnv;
  memset(&tk, 0, sizeof tk);
  memset(&tv, 0, sizeof tv);
  if (!pool_map(&tk, k_cache, num_blocks, num_kv_heads) ||
      !pool_map(&tv, v_cache, num_blocks, num_kv_heads))
    return PA_ERR_DEVICE;
  tnk = tk;
  tnv = tv;
  if (fused && (!rows_map(&tnk, new_k, total_tokens, num_kv_heads, new_k_tok_stride) ||
                !rows_map(&tnv, new_v, total_tokens, num_kv_heads, new_v_tok_stride)))
    return PA_ERR_DEVICE;
  PrefillParams pp;
  pp.out = out;
  pp.out_f32 = out_dtype == PA_DTYPE_F32;
  pp.q = static_cast<const uint16_t *>(q);
  pp.cu_seqlens = cu_seqlens;
  pp.num_seqs = num_seqs;
  pp.num_blocks = num_blocks;
  pp.block_tables = block_tables;
  pp.bt_stride = block_table_stride;
  pp.context_lens = context_lens;
  pp.hq = num_q_heads;
  pp.hkv = num_kv_heads;
  // The softmax keeps its reference max in raw score units and masks keys
  // with -inf before scaling, which needs a positive score scale: a negative
  // scale is folded into q (its sign bits flipped, exact), a zero one makes
  // q zero (every score 0, scale 1).
  pp.qk_scale_log2 = (scale > 0.f ? scale : scale < 0.f ? -scale : 1.f) * 1.4426950408889634f;
  pp.q_and = scale == 0.f ? 0u : 0xFFFFFFFFu;
  pp.q_xor = scale < 0.f ? 0x80008000u : 0u;
  pp.err = error_flags;
  pp.new_k = static_cast<const uint16_t *>(new_k);
  pp.new_v = static_cast<const uint16_t *>(new_v);
  pp.new_k_tok = new_k_tok_stride;
  pp.new_v_tok = new_v_tok_stride;
  pp.slot_mapping = slot_mapping;
  pp.k_cache = static_cast<const uint16_t *>(k_cache);
  pp.v_cache = static_cast<const uint16_t *>(v_cache);
  pp.k_store = static_cast<uint16_t *>(const_cast<void *>(k_cache));
  pp.v_store = static_cast<uint16_t *>(const_cast<void *>(v_cache));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int G = num_q_heads / num_kv_heads;
  cudaError_t e;
  switch (G) {
    case 1: e = launch_prefill<1>(tk, tv, tnk, tnv, pp, max_q_len, st, device); break;
    case 2: e = launch_prefill<2>(tk, tv, tnk, tnv, pp, max_q_len, st, device); break;
    case 3: e = launch_prefill<3>(tk, tv, tnk, tnv, pp, max_q_len, st, device); break;
    case 4: e = launch_prefill<4>(tk, tv, tnk, tnv, pp, max_q_len, st, device); break;
    case 5: e = launch_prefill<5>(tk, tv, tnk, tnv, pp, max_q_len, st, device); break;
    case 6: e = launch_prefill<6>(tk, tv, tnk, tnv, pp, max_q_len, st, device); break;
    case 7: e = launch_prefill<7>(tk, tv, tnk, tnv, pp, max_q_len, st, device); break;
    default: e = launch_prefill<8>(tk, tv, tnk, tnv, pp, max_q_len, st, device); break;
  }
  return e == cudaSuccess ? PA_OK : PA_ERR_LAUNCH;
}
}  // namespace
}  // namespace pa

extern "C" pa_status pa_prefill_varlen(void *out, int32_t out_dtype, const void *q,
                                       const int32_t *cu_seqlens, int32_t num_seqs,
                                       int32_t total_tokens, int32_t max_q_len,
                                       const void *k_cache, const void *v_cache,
                                       int64_t num_blocks, const int32_t *block_tables,
                                       int32_t block_table_stride, const int32_t *context_lens,
                                       int32_t num_q_heads, int32_t num_kv_heads,
                                       int32_t head_dim, int32_t block_size, float scale,
                                       int32_t *error_flags, void *stream) {
  return pa::prefill_entry(out, out_dtype, q, cu_seqlens, num_seqs, total_tokens, max_q_len,
                           k_cache, v_cache, num_blocks, block_tables, block_table_stride,
                           context_lens, num_q_heads, num_kv_heads, head_dim, block_size, scale,
                           error_flags, stream, nullptr, nullptr, 0, 0, nullptr);
}

extern "C" pa_status pa_prefill_store_varlen(
    void *out, int32_t out_dtype, const void *q, const void *new_k, const void *new_v,
    int64_t new_k_tok_stride, int64_t new_v_tok_stride, const int32_t *slot_mapping,
    const int32_t *cu_seqlens, int32_t num_seqs, int32_t total_tokens, int32_t max_q_len,
    void *k_cache, void *v_cache, int64_t num_blocks, const int32_t *block_tables,
    int32_t block_table_stride, const int32_t *context_lens, int32_t num_q_heads,
    int32_t num_kv_heads, int32_t head_dim, int32_t block_size, float scale,
    int32_t *error_flags, void *stream) {
  if (total_tokens > 0 && num_seqs > 0 && max_q_len > 0 && (!new_k || !new_v || !slot_mapping))
    return PA_ERR_INVALID_ARG;
  return pa::prefill_entry(out, out_dtype, q, cu_seqlens, num_seqs, total_tokens, max_q_len,
                           k_cache, v_cache, num_blocks, block_tables, block_table_stride,
                           context_lens, num_q_heads, num_kv_heads, head_dim, block_size, scale,
                           error_flags, stream, new_k, new_v, new_k_tok_stride,
                           new_v_tok_stride, slot_mapping);
}
