/*
 * pa.h -- C ABI of the GB300 paged-KV attention library (libpa_gb300.so).
 *
 * Five operations over a block-paged KV cache, each a hand-written sm_103a
 * CUDA kernel enqueued on the caller's stream:
 *
 *   pa_store_kv        write each new token's K/V rows into the pool slot
 *                      named by slot_mapping;
 *   pa_rope_store_kv   the same store fused with the rotary position
 *                      embedding of q and k;
 *   pa_decode          paged GQA decode attention (one query per sequence),
 *                      split across CTAs with log-sum-exp partials;
 *   pa_decode_merge    combine those partials into the final rows;
 *   pa_prefill_varlen  causal varlen attention of cu_seqlens-packed query
 *                      chunks over each sequence's paged keys
 *                      (pa_prefill_store_varlen: with the chunks' store);
 * pa_store_decode fuses pa_store_kv and pa_decode for a decode step; and an
 * FP8 (E4M3) KV cache: pa_store_kv_fp8 quantises into it, pa_decode_fp8
 * decodes over it and pa_store_decode_fp8 does both for a decode step.
 *
 * Sources (web pages that describe the method):
 *   [EAS] koas-w, "errors and solutions" (Qwen2.5-1.5B inference from
 *         scratch): sections "KV Cache 管理" (global pool of 16-token
 *         blocks, logical->physical block_table), "自写 Triton Kernel"
 *         (store_kvcache_kernel; Decode_Paged_GQAAttention_Kernel;
 *         fused_rope_and_cache_store_kernel), "开发时间线" (days 4-5: RoPE
 *         as a real-valued table lookup), "算子融合与模型优化"
 *         (rotate_half), "CUDA Graph" (static slot_mapping / block_table /
 *         context_lens buffers) and "开发过程遇到的错误汇总" types 1, 2 and 5.
 *   [MVT] mini-vllm tutorial, "step14_7 -- Batched Forward": sections
 *         "解决方案：变长 batch（varlen）" and "cu_seqlens 只在 Attention 里才需要".
 *   [CEB] PocketLLM, "cpp_engine Batching Implementation (Phase 3.1)",
 *         section "当前 KV cache 结构" (one token row is [kv_heads, head_dim];
 *         k_scale / v_scale kept beside the caches for FP8/INT8).
 *
 * Conventions shared by every entry point
 *   - All array arguments are DEVICE pointers into caller-owned memory, with
 *     two exceptions: the `out` of the decode entry points and both buffers
 *     of pa_copy may also be pinned host memory (cudaHostAlloc / a pinned
 *     torch tensor), which the device reaches through the same address over
 *     the CPU-GPU link -- a decode's `out` there delivers the result to the
 *     host with no copy.  The
 *     library allocates nothing and keeps no data between calls (its only
 *     host-side state: per-device flags recording that a kernel's shared
 *     memory limit was raised, the driver entry points it looked up, and
 *     pa_decode_noalloc's cached array address -- all set once, under
 *     atomics or a lock, so the entry points may be called from several host
 *     threads at once; two calls in flight must not share a workspace or an
 *     output buffer).  Scalars are passed by value.  `stream` is a cudaStream_t (NULL = legacy default
 *     stream); all work is enqueued there and the call returns without
 *     synchronising.  PA_OK means "validated and launched", not "finished".
 *   - Element type of q, k, v and the pools is bf16.  Outputs are bf16
 *     (out_dtype = PA_DTYPE_BF16, round to nearest even) or fp32
 *     (PA_DTYPE_F32).  Arithmetic is fp32.
 *   - KV pool layout: k_cache and v_cache are contiguous
 *     [num_blocks][block_size][num_kv_heads][head_dim]; slot s is physical
 *     block s / block_size, row s % block_size ([EAS] "KV Cache 管理";
 *     token row as in [CEB]).
 *   - block_tables is int32 [batch][block_table_stride] (row-major, row
 *     stride in elements); entry j of row b is the physical block holding
 *     positions 16j .. 16j+15 of sequence b.  Only entries
 *     j < ceil(context_lens[b] / block_size) are read; the rest may hold
 *     anything.
 *   - context_lens[b] is the number of keys sequence b attends to, INCLUDING
 *     tokens stored in the same step ([EAS] error type 1).
 *   - GQA: query head h reads kv head h / (num_q_heads / num_kv_heads).
 *   - Supported shapes: head_dim = 128, block_size = 16, num_kv_heads in
 *     {1, 2, 4, 8}, num_q_heads / num_kv_heads in 1..8.  Other shapes return
 *     PA_ERR_UNSUPPORTED without launching.
 *   - Errors: host-side checks return a status and launch nothing.  Device-
 *     side checks (a block-table entry outside [0, num_blocks), a slot past
 *     the pool, a prefix shorter than zero, a pipeline wait that gave up)
 *     never fault: the kernel skips the access, ORs a PA_DEVERR_* bit into
 *     the caller's error word and leaves the affected output rows
 *     unspecified.
 */
#ifndef PA_GB300_H
#define PA_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define PA_ABI_VERSION 11

#if defined(__GNUC__)
#define PA_API __attribute__((visibility("default")))
#else
#define PA_API
#endif

typedef int32_t pa_status;
#define PA_OK 0
#define PA_ERR_INVALID_ARG 1   /* null pointer, negative size, bad stride, ... */
#define PA_ERR_UNSUPPORTED 2   /* shape outside the supported set */
#define PA_ERR_WORKSPACE 3     /* workspace missing or too small */
#define PA_ERR_LAUNCH 4        /* the CUDA runtime rejected the launch */
#define PA_ERR_DEVICE 5        /* a device query or copy failed */

/* Largest split count pa_decode accepts. */
#define PA_DECODE_MAX_SPLITS 4096

#define PA_DTYPE_BF16 0
#define PA_DTYPE_F32 1

/* Bits a kernel ORs into the caller's int32 error word. */
#define PA_DEVERR_BLOCK_INDEX 1   /* block table entry outside [0, num_blocks) */
#define PA_DEVERR_SLOT_INDEX 2    /* slot_mapping entry outside the pool */
#define PA_DEVERR_WAIT_TIMEOUT 4  /* a pipeline wait gave up after ~2 s */
#define PA_DEVERR_SHAPE 8         /* context_lens / cu_seqlens inconsistent */
#define PA_DEVERR_POSITION 16     /* a position outside the rotary tables */

/*
 * Launch flags (the `flags` argument of pa_store_kv, pa_store_kv_fp8,
 * pa_rope_store_kv, pa_decode, pa_store_decode, pa_rope_store_decode,
 * pa_decode_fp8, pa_store_decode_fp8 and pa_decode_noalloc).  Any other bit returns
 * PA_ERR_INVALID_ARG.
 *
 * PA_LAUNCH_PDL: programmatic dependent launch.  The call's kernel may begin
 * while the kernel launched just before it on the same stream is still
 * running, and lets the kernel launched after it begin early; a chain of
 * such calls overlaps each kernel's start-up (launch, set-up, first loads)
 * with the tail of the one before.  Before waiting for the previous kernel
 * to complete, pa_decode / pa_decode_noalloc read context_lens and
 * block_tables only (to partition the work and find the first pages); so
 * with this flag those two must not be written by the kernel launched
 * immediately before the call (host copies and earlier kernels are fine).
 * pa_store_kv and pa_rope_store_kv read nothing before that wait.
 * Every write and every other read happens after it, so the results are the
 * same with and without the flag.  The decode kernels let the kernel after
 * them begin only once they have passed their own wait: when that next
 * kernel starts, every kernel before them has completed.  A decode call that
 * also launches the merge kernel (the partition below) lets the next call
 * begin at once from that kernel, so its decode kernel may still run when
 * the next call's first kernel begins: the "kernel launched immediately
 * before" in the guarantees here and below is then that whole call.
 *
 * PA_LAUNCH_EARLY_KV (decode entry points only, together with
 * PA_LAUNCH_PDL): the kernel also requests the K/V pages of its first ring
 * stages (up to 6 blocks per CTA) before the previous kernel completes, so
 * that the copies overlap that kernel's tail.  q, the new rows, the
 * workspace and every write still wait for it.  The caller guarantees that
 * the kernel launched immediately before the call does not write k_cache /
 * v_cache; in a layer-by-layer decode step with pa_store_decode this holds
 * (the kernel before layer l's call writes layer l - 1's pools or
 * activations), while a pa_store_kv or pa_rope_store_kv into the same pools
 * just before the call rules the flag out.  Results are the same with and
 * without it.  Without PA_LAUNCH_PDL it returns PA_ERR_INVALID_ARG.
 */
#define PA_LAUNCH_PDL 1u
#define PA_LAUNCH_EARLY_KV 2u
#define PA_COPY_BEFORE_WAIT 4u

/* ABI version of the loaded library (PA_ABI_VERSION it was built with). */
PA_API int32_t pa_abi_version(void);

/* Static, human-readable name of a pa_status value. */
PA_API const char *pa_status_string(pa_status status);

/*
 * pa_copy -- a byte copy, as a kernel (host plumbing for a serving loop; the
 * pages have no counterpart).
 *
 * Copies num_bytes from src to dst, two buffers the device can address:
 * device memory, or pinned host memory (cudaHostAlloc / a pinned torch
 * tensor), which the device reaches through the same address.  A
 * cudaMemcpyAsync between two kernels of a stream ends their programmatic
 * overlap; this copy keeps it.  flags: 0, PA_LAUNCH_PDL (the copy waits for
 * the kernel launched just before it, then moves the bytes; the kernel after
 * it begins once it has passed that wait), or PA_LAUNCH_PDL |
 * PA_COPY_BEFORE_WAIT (it moves the bytes and lets the kernel after it begin
 * while the kernel before it may still run, then waits for that one).  With
 * PA_COPY_BEFORE_WAIT the caller guarantees that the kernel launched just
 * before the copy neither writes src nor reads or writes dst, and that the
 * kernel launched just after it reads dst only after its own wait (the
 * decode entry points read context_lens and block_tables before theirs: stage
 * those a launch earlier).  That next kernel may begin while the kernel
 * before the copy still runs, so what it reads before its wait
 * (context_lens, block_tables, and with PA_LAUNCH_EARLY_KV the pages) must
 * not be written by that kernel either.  16-byte aligned
 * addresses move in 16-byte chunks; otherwise at most 256 bytes may be
 * copied (PA_ERR_UNSUPPORTED beyond).  Returns PA_ERR_INVALID_ARG for a
 * null pointer, a negative size or a bad flag, before launching anything;
 * num_bytes = 0 launches nothing.  Allocates nothing.
 */
PA_API pa_status pa_copy(void *dst, const void *src, int64_t num_bytes, uint32_t flags,
                         void *stream);

/*
 * pa_get_device_error -- read back a device error word (host helper; the
 * pages have no counterpart: it stands in for a debug-build error query).
 *
 * error_word is the caller's int32 word that a call ORs PA_DEVERR_* bits
 * into: byte 0 of a decode workspace (pa_decode, pa_store_decode,
 * pa_rope_store_decode, pa_decode_fp8, pa_store_decode_fp8), or the
 * `error_flags` argument of the other entry points.  The helper enqueues a
 * copy of the word to the host on `stream` (and, when `clear` is nonzero, a
 * reset of the word to 0 after the copy), synchronises the stream, and
 * stores the word in *out_flags.  It is the one entry point that blocks the
 * calling thread; it allocates nothing.  Returns PA_ERR_INVALID_ARG for a
 * null pointer (nothing enqueued) and PA_ERR_DEVICE when the copy, the reset
 * or the synchronisation fails (*out_flags is then left untouched).
 */
PA_API pa_status pa_get_device_error(int32_t *error_word, int32_t *out_flags, int32_t clear,
                                     void *stream);

/*
 * pa_store_kv -- slot_mapping store ([EAS] "自写 Triton Kernel",
 * store_kvcache_kernel; strides as in [EAS] error type 2).
 *
 * For every token t < num_tokens with slot = slot_mapping[t] >= 0, copies
 * k[t][h][0..head_dim) and v[t][h][0..head_dim) for every kv head h into
 * k_cache / v_cache at physical block slot / block_size, row
 * slot % block_size.  Tokens with slot < 0 are padding and are skipped.
 * The copy is bit-exact.  Two tokens naming the same slot is a caller error
 * (one of them wins, unspecified which).
 *
 *   k, v           bf16 source rows; element (t, h, d) lives at
 *                  k + t * k_tok_stride + h * k_head_stride + d (strides in
 *                  elements, d contiguous), same for v.
 *   k_cache,
 *   v_cache        pools, [num_blocks][block_size][num_kv_heads][head_dim].
 *   slot_mapping   int32 [num_tokens].
 *   error_flags    optional int32 word (may be NULL); a slot >= num_blocks *
 *                  block_size sets PA_DEVERR_SLOT_INDEX and that token is
 *                  skipped.
 *   flags          0 or PA_LAUNCH_PDL.
 */
PA_API pa_status pa_store_kv(const void *k, const void *v, int64_t num_tokens,
                      int64_t k_tok_stride, int64_t k_head_stride,
                      int64_t v_tok_stride, int64_t v_head_stride,
                      void *k_cache, void *v_cache, int64_t num_blocks,
                      int32_t block_size, int32_t num_kv_heads, int32_t head_dim,
                      const int32_t *slot_mapping, int32_t *error_flags,
                      uint32_t flags, void *stream);

/*
 * pa_rope_store_kv -- rotary position embedding fused with the slot_mapping
 * store ([EAS] "自写 Triton Kernel", fused_rope_and_cache_store_kernel: q is
 * rotated and written back contiguous, k is rotated and stored with v
 * through slot_mapping; RoPE by table lookup, "开发时间线" days 4-5;
 * rotate_half, "算子融合与模型优化").
 *
 * With D = head_dim, for every token t < num_tokens at p = positions[t] and
 * every i < D/2, c = cos_table[p * D/2 + i], s = sin_table[p * D/2 + i], a
 * head row x is rotated in rotate-half pairs:
 *     x'[i]       = x[i] * c - x[i + D/2] * s
 *     x'[i + D/2] = x[i + D/2] * c + x[i] * s.
 * Every q head of token t is rotated into q_out.  Every kv head of k is
 * rotated and stored, with the v row unrotated, at slot_mapping[t] exactly
 * as pa_store_kv stores (slot < 0: padding, no pool row is written, q_out
 * still is).  Arithmetic is fp32 from the bf16 rows and fp32 tables (fused
 * multiply-add), rounded once to bf16 (nearest even); v moves bit-exactly.
 *
 *   q, k, v        bf16; element (t, h, d) of x lives at
 *                  x + t * x_tok_stride + h * head_dim + d (heads
 *                  contiguous, so the three may be column slices of one
 *                  fused QKV row).
 *   q_out          bf16, (t, h, d) at q_out + t * q_out_tok_stride +
 *                  h * head_dim + d.  May be q itself (rotation in place);
 *                  any other overlap with q, k or v is a caller error.
 *   positions      int32 [num_tokens], absolute positions.
 *   cos_table,
 *   sin_table      fp32 [max_position][head_dim / 2], 16-byte aligned; the
 *                  caller chooses the angles (e.g. p * base^(-2i / D)).
 *   k_cache,
 *   v_cache        pools, [num_blocks][block_size][num_kv_heads][head_dim].
 *   slot_mapping   int32 [num_tokens].
 *   error_flags    optional int32 word (may be NULL): a position outside
 *                  [0, max_position) sets PA_DEVERR_POSITION and the whole
 *                  token is skipped (no q_out row, no pool row); a slot >=
 *                  num_blocks * block_size sets PA_DEVERR_SLOT_INDEX and
 *                  the token's pool rows are skipped.
 *   flags          0 or PA_LAUNCH_PDL.
 * Supported: head_dim 128, block_size 16, 1 <= num_kv_heads <= 64,
 * 1 <= num_q_heads <= 512.
 */
PA_API pa_status pa_rope_store_kv(const void *q, int64_t q_tok_stride, void *q_out,
                                  int64_t q_out_tok_stride, const void *k, int64_t k_tok_stride,
                                  const void *v, int64_t v_tok_stride, int64_t num_tokens,
                                  int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                  const int32_t *positions, const float *cos_table,
                                  const float *sin_table, int64_t max_position, void *k_cache,
                                  void *v_cache, int64_t num_blocks, int32_t block_size,
                                  const int32_t *slot_mapping, int32_t *error_flags,
                                  uint32_t flags, void *stream);

/*
 * FP8 KV cache ([CEB] "当前 KV cache 结构": k_scale / v_scale beside the
 * caches, "FP8/INT8 量化时使用"; the pages fix nothing more, so:)
 *   - every element is an E4M3 code (1 sign bit, 4 exponent bits with bias
 *     7, 3 mantissa bits; largest finite 448; 0x7F / 0xFF are NaN);
 *   - k_scale and v_scale are fp32 [num_kv_heads] device arrays; the value
 *     of a K code of head h is code * k_scale[h] (V likewise);
 *   - K pool: uint8 [num_blocks][block_size][num_kv_heads][head_dim], the
 *     bf16 layout with one byte per element;
 *   - V pool: uint8 [num_blocks][num_kv_heads][head_dim][block_size]:
 *     dim-major inside a block (token row s % block_size of dim d of head h
 *     of block s / block_size is byte (((s / bs) * Hkv + h) * D + d) * bs +
 *     s % bs), so that the decode's tensor-core operands are whole words.
 *
 * pa_store_kv_fp8 -- pa_store_kv into FP8 pools: the code of element x of
 * kv head h is the E4M3 value nearest to x / scale[h] (IEEE fp32 division;
 * ties to the even code; magnitudes past 448 saturate to +-448).  Arguments
 * as pa_store_kv, plus k_scale / v_scale; k_cache must be 8-byte aligned.
 */
PA_API pa_status pa_store_kv_fp8(const void *k, const void *v, int64_t num_tokens,
                                 int64_t k_tok_stride, int64_t k_head_stride,
                                 int64_t v_tok_stride, int64_t v_head_stride, void *k_cache,
                                 void *v_cache, const float *k_scale, const float *v_scale,
                                 int64_t num_blocks, int32_t block_size, int32_t num_kv_heads,
                                 int32_t head_dim, const int32_t *slot_mapping,
                                 int32_t *error_flags, uint32_t flags, void *stream);

/*
 * Decode split partition.  The decode work is the list of all KV blocks of
 * all sequences, sequence after sequence: sequence b owns
 * n_b = ceil(context_lens[b] / block_size) blocks, the global block index of
 * its block j is P_b + j with P_b = n_0 + ... + n_{b-1}, and
 * N = n_0 + ... + n_{batch-1}.  With S = num_splits, split c in [0, S)
 * processes global blocks [floor(N W(c) / W(S)), floor(N W(c + 1) / W(S))),
 * where W(c) sums the weights of splits 0 .. c - 1: every split weighs 4,
 * except that when S >= 32 and N >= 4 S the last four weigh 3, 3, 3 and 2
 * (a grid's highest-indexed CTAs start last behind a previous kernel, on
 * the SMs it frees last; their lighter shares let them end with the rest).
 * Every split therefore moves the same number of KV bytes (+-1 block), the
 * last four less, however skewed the lengths are.
 *
 * A sequence whose blocks all fall in one split is finished by that split,
 * which writes its output rows directly.  A sequence spread over splits
 * c0 < c1 leaves a partial result in every split it touches: split c0 in
 * slot 1, row block c0, and every non-empty split c in (c0, c1] in slot 0,
 * row block c (so the slot-0 partials of one sequence are consecutive).  A
 * partial is the attention output over that split's keys only, normalised
 * over those keys, plus the natural-log sum-exp of its scaled scores.  The
 * split that completes a sequence's set of partials (counted in
 * counters[c1]) merges them into the output rows and sets the counter back
 * to zero, all inside the decode kernel.  Launches with num_kv_heads >= 4
 * and S >= 8 * batch (few sequences, each cut into many pieces of many query
 * heads) merge differently: the decode kernel only writes the partials, and
 * the call's second kernel (the merge kernel, a programmatic dependent launch
 * right behind it) merges every cut sequence once the decode kernel has
 * completed; the counters are not used.
 *
 * Workspace layout (bytes from the workspace pointer; R(x) rounds x up to
 * a multiple of 256; H = num_q_heads, D = head_dim, C = 256 + 4 *
 * PA_DECODE_MAX_SPLITS):
 *   [0, 4)              int32 error word (PA_DEVERR_* bits; the library
 *                       only ORs bits in);
 *   [256, C)            int32 counters[PA_DECODE_MAX_SPLITS], zero between
 *                       calls, at the same place for every S;
 *   [C, ...)            float partial_o[2][S][H][D]  (slot, split, head, dim);
 *   C + R(8SHD)         float partial_lse[2][S][H].
 * Zero the whole workspace once when allocating it; every completed call
 * leaves the counters at zero again, so the workspace can be reused with
 * any split count.  After a call that reported PA_DEVERR_WAIT_TIMEOUT,
 * zero it again.  One workspace serves one call in flight at a time.
 */
PA_API size_t pa_decode_workspace_size(int32_t num_splits, int32_t num_q_heads, int32_t head_dim);

/* num_splits used when pa_decode is given 0 for this head shape: one split
 * per CTA the decode kernel keeps resident on `device` (its SM count for the
 * shipped kernel, whatever the head counts).  Returns <= 0 on error. */
PA_API int32_t pa_decode_default_splits(int32_t device, int32_t num_q_heads,
                                        int32_t num_kv_heads);

/*
 * pa_decode -- paged GQA decode attention ([EAS] "自写 Triton Kernel",
 * Decode_Paged_GQAAttention_Kernel; flash-decoding split-K with a balanced
 * block partition).
 *
 * For each sequence b and query head h, with g = h / (num_q_heads /
 * num_kv_heads) and n = context_lens[b]:
 *   out[b][h] = sum_{j<n} softmax_j(scale * q[b][h] . K_b[j][g]) V_b[j][g]
 * where K_b[j] is row j % block_size of physical block
 * block_tables[b][j / block_size].  The kernel walks the block table and
 * streams pages through shared memory; nothing is gathered into contiguous
 * memory.  Sequences with context 0 get a zero row.  Sequences spread over
 * splits (see the partition above) are merged inside the same kernel, so
 * `out` is complete when the stream reaches the end of the call.
 *
 *   out            [batch][num_q_heads][head_dim], out_dtype.
 *   q              bf16 [batch][num_q_heads][head_dim], contiguous.
 *   k_cache,
 *   v_cache        bf16 pools (layout above), num_blocks blocks each.
 *   block_tables   int32 [batch][block_table_stride].
 *   context_lens   int32 [batch]; negative values are treated as 0.
 *   scale          softmax scale applied to q . k (e.g. 1/sqrt(head_dim));
 *                  any finite value, of either sign (non-finite:
 *                  PA_ERR_INVALID_ARG).
 *   num_splits     S of the partition, at most PA_DECODE_MAX_SPLITS;
 *                  0 = pa_decode_default_splits.
 *   workspace      device buffer of workspace_bytes >=
 *                  pa_decode_workspace_size(S, num_q_heads, head_dim).
 *   flags          0, PA_LAUNCH_PDL (then context_lens and block_tables
 *                  must not be written by the kernel launched just before
 *                  this call) or PA_LAUNCH_PDL | PA_LAUNCH_EARLY_KV (then
 *                  not k_cache / v_cache either).
 * Results do not depend on how sequences are laid out in the pool; with a
 * fixed num_splits they are deterministic run to run.
 */
PA_API pa_status pa_decode(void *out, int32_t out_dtype, const void *q, const void *k_cache,
                    const void *v_cache, int64_t num_blocks, const int32_t *block_tables,
                    int32_t block_table_stride, const int32_t *context_lens, int32_t batch,
                    int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                    int32_t block_size, float scale, int32_t num_splits, void *workspace,
                    size_t workspace_bytes, uint32_t flags, void *stream);

/*
 * pa_store_decode -- pa_store_kv and pa_decode of one decode step in one
 * kernel (bf16 pools).  Every sequence b has one new token, at position
 * context_lens[b] - 1, whose K/V rows are new_k / new_v + b *
 * new_*_tok_stride + h * head_dim (heads contiguous; 16-byte aligned rows,
 * token strides multiples of 8 elements); slot_mapping[b] is its pool slot
 * (< 0: the token is not stored and the pool row is used as it is).
 * The result equals pa_store_kv followed by pa_decode, but the new rows
 * reach the attention directly: the CTA that consumes a sequence's last
 * block patches them into its staged tile and writes them to the pool, so
 * no second launch and no store-to-load dependency stands between the two.
 * slot_mapping[b] must be the slot of that position under the block table
 * (table[b][(ctx - 1) / 16] * 16 + (ctx - 1) % 16); any other value sets
 * PA_DEVERR_SLOT_INDEX in the workspace error word and that row is neither
 * stored nor patched.  Other arguments, the workspace and the flags as for
 * pa_decode.
 */
PA_API pa_status pa_store_decode(void *out, int32_t out_dtype, const void *q, const void *new_k,
                                 const void *new_v, int64_t new_k_tok_stride,
                                 int64_t new_v_tok_stride, const int32_t *slot_mapping,
                                 void *k_cache, void *v_cache, int64_t num_blocks,
                                 const int32_t *block_tables, int32_t block_table_stride,
                                 const int32_t *context_lens, int32_t batch, int32_t num_q_heads,
                                 int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                 float scale, int32_t num_splits, void *workspace,
                                 size_t workspace_bytes, uint32_t flags, void *stream);

/*
 * pa_rope_store_decode -- pa_rope_store_kv, pa_store_kv and pa_decode of one
 * decode step in one kernel (bf16 pools): the rotary embedding of
 * pa_rope_store_kv (koas-w, "errors and solutions", fused_rope_and_cache_store_kernel)
 * applied inside pa_store_decode.  Sequence b's new token sits at position
 * positions[b]; its q rows (q + b * num_q_heads * head_dim, as for
 * pa_decode) and its new K row are rotated with row positions[b] of
 * cos_table / sin_table (float32 [max_position][head_dim / 2], 16-byte
 * aligned), rotate-half pairs (i, i + head_dim / 2), with the same arithmetic
 * and rounding as pa_rope_store_kv: the output equals, bit for bit,
 * pa_rope_store_kv (q rotated into q_out, K rotated and stored with V)
 * followed by pa_decode on q_out, with the same split count; the pools
 * after the call equal those pa_rope_store_kv leaves.  q itself is not
 * written.  new_k / new_v / slot_mapping as for pa_store_decode.  A position
 * outside [0, max_position) sets PA_DEVERR_POSITION in the workspace error
 * word; that sequence's q is rotated with row 0 and its new row is neither
 * stored nor patched.  Returns PA_ERR_INVALID_ARG for a missing pointer,
 * max_position < 1 or unaligned tables (before any device query); other
 * arguments, the workspace and the flags as for pa_decode.
 */
PA_API pa_status pa_rope_store_decode(
    void *out, int32_t out_dtype, const void *q, const void *new_k, const void *new_v,
    int64_t new_k_tok_stride, int64_t new_v_tok_stride, const int32_t *positions,
    const float *cos_table, const float *sin_table, int64_t max_position,
    const int32_t *slot_mapping, void *k_cache, void *v_cache, int64_t num_blocks,
    const int32_t *block_tables, int32_t block_table_stride, const int32_t *context_lens,
    int32_t batch, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
    int32_t block_size, float scale, int32_t num_splits, void *workspace,
    size_t workspace_bytes, uint32_t flags, void *stream);

/*
 * pa_store_decode_fp8 -- pa_store_decode over FP8 pools: each sequence's new
 * token is quantised (as pa_store_kv_fp8 does, bit for bit) into the pools
 * and into the staged tiles of its last block, and every sequence is decoded
 * as pa_decode_fp8 does, in one kernel.  Arguments as pa_store_decode plus
 * k_scale / v_scale (NULL: PA_ERR_INVALID_ARG).
 */
PA_API pa_status pa_store_decode_fp8(void *out, int32_t out_dtype, const void *q,
                                     const void *new_k, const void *new_v,
                                     int64_t new_k_tok_stride, int64_t new_v_tok_stride,
                                     const int32_t *slot_mapping, void *k_cache, void *v_cache,
                                     const float *k_scale, const float *v_scale,
                                     int64_t num_blocks, const int32_t *block_tables,
                                     int32_t block_table_stride, const int32_t *context_lens,
                                     int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                                     int32_t head_dim, int32_t block_size, float scale,
                                     int32_t num_splits, void *workspace, size_t workspace_bytes,
                                     uint32_t flags, void *stream);

/*
 * pa_decode_fp8 -- pa_decode over FP8 pools (layout and scales above).
 * Codes are widened exactly; the dot products and P . V run on the tensor
 * cores in f16 (q is rounded to f16, which is exact for bf16 values of
 * magnitude 2^-14 .. 65504; larger magnitudes saturate to 65504), with fp32
 * accumulation, and the result meets the same tolerance as pa_decode
 * against the attention over the widened values.  Same workspace, splits,
 * flags and outputs as pa_decode.  Returns PA_ERR_INVALID_ARG when k_scale
 * or v_scale is NULL.
 */
PA_API pa_status pa_decode_fp8(void *out, int32_t out_dtype, const void *q, const void *k_cache,
                               const void *v_cache, const float *k_scale, const float *v_scale,
                               int64_t num_blocks, const int32_t *block_tables,
                               int32_t block_table_stride, const int32_t *context_lens,
                               int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                               int32_t head_dim, int32_t block_size, float scale,
                               int32_t num_splits, void *workspace, size_t workspace_bytes,
                               uint32_t flags, void *stream);

/*
 * pa_decode_merge -- log-sum-exp merge of decode partials (flash-decoding).
 *
 * For every sequence spread over splits c0 < c1 (partition above, from
 * context_lens, block_size and num_splits) and every query head, with
 * partials (o_i, lse_i) read from the workspace slots listed above:
 *   M = max_i lse_i,  w_i = exp(lse_i - M),  out = sum_i w_i o_i / sum_i w_i.
 * Rows of sequences held by a single split are not touched.  This is the
 * merge kernel that pa_decode launches behind its decode kernel for launches
 * with few long sequences (partition above); it also combines partials that
 * are already in a workspace (e.g. written by another producer, or kept for
 * inspection) and lets the merge be tested and timed on its own.  Counters
 * are neither read nor written.
 */
PA_API pa_status pa_decode_merge(void *out, int32_t out_dtype, const void *workspace,
                          size_t workspace_bytes, const int32_t *context_lens,
                          int32_t batch, int32_t num_q_heads, int32_t head_dim,
                          int32_t block_size, int32_t num_splits, void *stream);

/*
 * pa_decode_noalloc -- pa_decode without a workspace argument, for callers
 * that cannot allocate device memory: an engine that gives nearly all free
 * memory to its KV block pool at start-up and must not allocate on the
 * decode path, a caller that only receives device pointers from a framework
 * owning the allocator, or a decode loop that cannot take the device-wide
 * synchronisation an allocation may cause.  The pages describe no such
 * entry point; it has no counterpart there.
 *
 * Same arguments and result as pa_decode, except: the split partials live
 * in a fixed 8 MiB array inside the library (a file-scope __device__ array,
 * held by every GPU that loads the library until the process exits);
 * device-side error bits go to `error_flags` (optional int32 word, may be
 * NULL).  num_splits = 0 takes pa_decode_default_splits, lowered where
 * needed to the largest S whose pa_decode_workspace_size(S, num_q_heads,
 * head_dim) fits in 8 MiB.  An explicit S that does not fit (S > 676 at 12
 * query heads, S > 253 at 32) returns PA_ERR_WORKSPACE, launching nothing.  The
 * call allocates nothing: no cudaMalloc, no cudaFree, no allocating library
 * routine.  The first call on a device, with that device current, looks up
 * the array's device address and caches it with the current CUDA context;
 * make that first call before any stream capture.  A call under another
 * context on that device (after cudaDeviceReset, or after the primary
 * context was released and created again) looks the address up again, so
 * the first call after such a change must also come before any capture.
 * All calls on a device share the array: calls that overlap on the GPU race
 * on it.  Each call clears the split arrival counters in the array (an
 * asynchronous memset on `stream`) before its kernel; nothing else in it
 * needs to start at zero.  That memset sits between the previous kernel on
 * the stream and the decode kernel, so PA_LAUNCH_PDL and PA_LAUNCH_EARLY_KV
 * are accepted but give no overlap through this entry point (the kernel
 * starts after the memset, as without the flags); results are the same.
 */
PA_API pa_status pa_decode_noalloc(void *out, int32_t out_dtype, const void *q,
                                   const void *k_cache, const void *v_cache,
                                   int64_t num_blocks, const int32_t *block_tables,
                                   int32_t block_table_stride, const int32_t *context_lens,
                                   int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                                   int32_t head_dim, int32_t block_size, float scale,
                                   int32_t num_splits, int32_t *error_flags, uint32_t flags,
                                   void *stream);

/*
 * pa_prefill_varlen -- causal varlen attention over a paged prefix ([MVT]
 * "解决方案：变长 batch（varlen）", "cu_seqlens 只在 Attention 里才需要"; the
 * per-sequence loop there is the one this kernel removes).
 *
 * Query rows of sequence s are rows cu_seqlens[s] .. cu_seqlens[s+1]-1 of q
 * (q_len_s of them).  The sequence has n_s = context_lens[s] keys in the
 * pool, its chunk's own keys included: store the chunk with pa_store_kv
 * first.  Query i of the chunk sits at absolute position P_s + i with
 * P_s = n_s - q_len_s (the paged prefix, [MVT] start_positions) and attends
 * keys 0 .. P_s + i inclusive of its own sequence only.
 *
 *   out            [total_tokens][num_q_heads][head_dim], out_dtype.
 *   q              bf16 [total_tokens][num_q_heads][head_dim], contiguous.
 *   cu_seqlens     int32 [num_seqs + 1], non-decreasing, cu_seqlens[0] = 0,
 *                  cu_seqlens[num_seqs] = total_tokens.
 *   max_q_len      upper bound of every q_len_s (sizes the launch grid).
 *   context_lens   int32 [num_seqs]; q_len_s > n_s sets PA_DEVERR_SHAPE and
 *                  that sequence's rows are left unspecified.
 *   scale          softmax scale applied to q . k; any finite value, of
 *                  either sign (non-finite: PA_ERR_INVALID_ARG).
 *   error_flags    optional int32 word (may be NULL).
 * Rows of different sequences never attend to each other, so a sequence's
 * rows equal what the same call gives for that sequence alone.  The order
 * in which the launch's tiles run (longest first) does not change any
 * result.
 */
PA_API pa_status pa_prefill_varlen(void *out, int32_t out_dtype, const void *q,
                            const int32_t *cu_seqlens, int32_t num_seqs,
                            int32_t total_tokens, int32_t max_q_len, const void *k_cache,
                            const void *v_cache, int64_t num_blocks,
                            const int32_t *block_tables, int32_t block_table_stride,
                            const int32_t *context_lens, int32_t num_q_heads,
                            int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                            float scale, int32_t *error_flags, void *stream);

/*
 * pa_prefill_store_varlen -- pa_store_kv of the chunks' tokens and
 * pa_prefill_varlen over them in one kernel ([EAS] "自写 Triton Kernel": the
 * store through slot_mapping, here fused with the attention that follows).
 * Token t of the packed chunks has K/V rows new_k / new_v + t *
 * new_*_tok_stride + h * head_dim (heads contiguous, 16-byte aligned, token
 * strides multiples of 8 elements) and pool slot slot_mapping[t] (< 0:
 * padding, not stored).  Each chunk's own keys are read from these rows, the
 * prefix keys from the pool; the rows are also stored, so the pools end as
 * pa_store_kv leaves them and the output equals pa_store_kv followed by
 * pa_prefill_varlen.  slot_mapping[t] must be the slot of token t's
 * position under the block table (the attention reads the chunk from
 * new_k / new_v); a slot past the pool sets PA_DEVERR_SLOT_INDEX and is
 * skipped.  Other arguments as pa_prefill_varlen.
 */
PA_API pa_status pa_prefill_store_varlen(void *out, int32_t out_dtype, const void *q,
                                         const void *new_k, const void *new_v,
                                         int64_t new_k_tok_stride, int64_t new_v_tok_stride,
                                         const int32_t *slot_mapping, const int32_t *cu_seqlens,
                                         int32_t num_seqs, int32_t total_tokens,
                                         int32_t max_q_len, void *k_cache, void *v_cache,
                                         int64_t num_blocks, const int32_t *block_tables,
                                         int32_t block_table_stride,
                                         const int32_t *context_lens, int32_t num_q_heads,
                                         int32_t num_kv_heads, int32_t head_dim,
                                         int32_t block_size, float scale, int32_t *error_flags,
                                         void *stream);

#ifdef __cplusplus
}
#endif

#endif /* PA_GB300_H */
