// Host-side pieces shared by pa_decode.cu and pa_decode_noalloc.cu (not part
// of the public ABI).
#pragma once

#include <stddef.h>
#include <stdint.h>

#include "../../include/pa.h"

namespace pa {

constexpr size_t kWorkspaceHeader = 256;  // int32 error word + reserved
// The arrival counters sit at a fixed place for every split count, so a
// workspace reused with another split count still finds them at zero.
constexpr size_t kCounterOffset = kWorkspaceHeader;
constexpr size_t kCounterBytes = size_t(PA_DECODE_MAX_SPLITS) * 4;

// Byte offsets inside a decode workspace for `splits` splits.
struct WorkspaceLayout {
  size_t counters;  // int32 [PA_DECODE_MAX_SPLITS], zero between calls
  size_t part_o;    // float [2][splits][hq][128]
  size_t part_lse;  // float [2][splits][hq]
  size_t total;
};
WorkspaceLayout workspace_layout(long long splits, int hq);

struct DecodeRequest {
  void *out;
  int32_t out_dtype;
  const void *q, *k_cache, *v_cache;
  int64_t num_blocks;
  const int32_t *block_tables;
  int32_t block_table_stride;
  const int32_t *context_lens;
  int32_t batch, num_q_heads, num_kv_heads, head_dim, block_size;
  float scale;
  int32_t num_splits;  // as given (0 = default)
  int32_t splits;      // resolved by check_decode_request
  uint32_t flags;      // PA_LAUNCH_* bits
  void *stream;
  // FP8 (E4M3) pools: K token-major, V dim-major per block, per-kv-head scales
  bool fp8 = false;
  const float *k_scale = nullptr;
  const float *v_scale = nullptr;
  // fused store of each sequence's new token (bf16 pools; null: none)
  const void *new_k = nullptr;
  const void *new_v = nullptr;
  int64_t new_k_tok = 0, new_v_tok = 0;
  const int32_t *slot_mapping = nullptr;
  // rotary embedding of q and the new K rows inside the fused store (null:
  // none): float32 tables [max_position][head_dim / 2]
  const int32_t *positions = nullptr;
  const float *cos_table = nullptr;
  const float *sin_table = nullptr;
  int64_t max_position = 0;
};

// Host checks shared by both decode entry points; resolves r.splits.
pa_status check_decode_request(DecodeRequest &r, int *device);

// Encodes the pool tensor maps and launches the decode kernel (which merges
// cut sequences itself).  `clear_counters` enqueues a memset of the arrival
// counters first.
pa_status run_decode(const DecodeRequest &r, void *workspace, int32_t *err, int device,
                     bool clear_counters);

}  // namespace pa
