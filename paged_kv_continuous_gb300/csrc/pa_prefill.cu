// pa_prefill_varlen: causal varlen attention over a paged prefix.  The
// tcgen05 tensor-core kernel is not built yet; the entry point validates its
// arguments and reports PA_ERR_UNSUPPORTED.
#include "pa_common.cuh"

extern "C" pa_status pa_prefill_varlen(void *out, int32_t out_dtype, const void *q,
                                       const int32_t *cu_seqlens, int32_t num_seqs,
                                       int32_t total_tokens, int32_t max_q_len,
                                       const void *k_cache, const void *v_cache,
                                       int64_t num_blocks, const int32_t *block_tables,
                                       int32_t block_table_stride, const int32_t *context_lens,
                                       int32_t num_q_heads, int32_t num_kv_heads,
                                       int32_t head_dim, int32_t block_size, float scale,
                                       int32_t *error_flags, void *stream) {
  (void)out; (void)out_dtype; (void)q; (void)cu_seqlens; (void)num_seqs; (void)total_tokens;
  (void)max_q_len; (void)k_cache; (void)v_cache; (void)num_blocks; (void)block_tables;
  (void)block_table_stride; (void)context_lens; (void)num_q_heads; (void)num_kv_heads;
  (void)head_dim; (void)block_size; (void)scale; (void)error_flags; (void)stream;
  return PA_ERR_UNSUPPORTED;
}
