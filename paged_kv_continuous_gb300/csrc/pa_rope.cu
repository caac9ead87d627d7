// pa_rope_store_kv: rotary position embedding fused with the slot_mapping
// KV-cache store (koas-w, "errors and solutions": section "自写 Triton
// Kernel", fused_rope_and_cache_store_kernel -- q rotated in registers and
// written back contiguous, k rotated and stored with v through slot_mapping;
// section "开发时间线", days 4-5 -- RoPE as a real-valued table lookup;
// section "算子融合与模型优化" -- rotate_half).
//
// Rotate-half pairs: dimension i of a head pairs with i + D/2, and with
// c = cos_table[p][i], s = sin_table[p][i] for the token's position p,
//   x'[i] = x[i] c - x[i + D/2] s,   x'[i + D/2] = x[i + D/2] c + x[i] s.
//
// One thread owns one "chunk pair" of one (token, head row): dims
// 8c .. 8c + 7 and their partners 64 + 8c .. 64 + 8c + 7 (c < 8), i.e. two
// 16-byte loads of the row, 32 bytes each of the cos and sin row, and two
// 16-byte stores.  Head rows are taken in the order q heads, k heads, v
// heads, so a warp covers four 256-byte rows with full 32-byte sectors, and
// a token's rows sit in consecutive threads (its table rows are read from
// L1 after the first warp).
#include "pa_common.cuh"

namespace pa {

namespace {

template <bool kVec>
__device__ __forceinline__ uint4 load8(const uint16_t *p) {
  if constexpr (kVec) {
    return __ldg(reinterpret_cast<const uint4 *>(p));
  } else {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) w[i] = (uint32_t)p[2 * i] | ((uint32_t)p[2 * i + 1] << 16);
    return make_uint4(w[0], w[1], w[2], w[3]);
  }
}

template <bool kVec>
__device__ __forceinline__ void store8(uint16_t *p, const uint4 &v) {
  if constexpr (kVec) {
    *reinterpret_cast<uint4 *>(p) = v;
  } else {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      p[2 * i] = (uint16_t)(w[i] & 0xFFFFu);
      p[2 * i + 1] = (uint16_t)(w[i] >> 16);
    }
  }
}

struct RopeParams {
  const uint16_t *q;
  long long q_tok;
  uint16_t *q_out;
  long long q_out_tok;
  const uint16_t *k;
  long long k_tok;
  const uint16_t *v;
  long long v_tok;
  long long num_tokens;
  int hq, hkv;
  const int32_t *positions;
  const float *cos_t;
  const float *sin_t;
  long long max_position;
  uint16_t *k_cache;
  uint16_t *v_cache;
  long long num_slots;
  const int32_t *slot_mapping;
  int32_t *err;
};

template <bool kVec>
__global__ void __launch_bounds__(256) rope_store_kernel(const RopeParams p) {
  constexpr int kHalf = kHeadDim / 2;     // 64 pairs per head
  constexpr int kPairChunks = kHalf / 8;  // 8 threads per head row
  // the rows, positions, slots and pools may come from or go to the
  // previous kernel
  griddep_wait();
  griddep_launch_dependents();
  const int rows = p.hq + 2 * p.hkv;  // head rows of a token: q, k, v
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= p.num_tokens * rows * kPairChunks) return;
  const int c = (int)(idx % kPairChunks);
  const long long tr = idx / kPairChunks;
  const int r = (int)(tr % rows);
  const long long t = tr / rows;
  const int d0 = c * 8;  // first-half dims d0 .. d0 + 7, partners + 64
  const long long pos = __ldg(p.positions + t);
  if (pos < 0 || pos >= p.max_position) {
    if (r == 0 && c == 0) report(p.err, PA_DEVERR_POSITION);
    return;
  }
  if (r < p.hq) {
    // q head r: rotate, write back contiguous
    const uint16_t *src = p.q + t * p.q_tok + (long long)r * kHeadDim;
    const uint4 a = load8<kVec>(src + d0), b = load8<kVec>(src + kHalf + d0);
    const float *cr = p.cos_t + pos * kHalf + d0, *sr = p.sin_t + pos * kHalf + d0;
    uint4 ra, rb;
    rope_rotate8(a, b, __ldg(reinterpret_cast<const float4 *>(cr)),
          __ldg(reinterpret_cast<const float4 *>(cr + 4)),
          __ldg(reinterpret_cast<const float4 *>(sr)),
          __ldg(reinterpret_cast<const float4 *>(sr + 4)), ra, rb);
    uint16_t *dst = p.q_out + t * p.q_out_tok + (long long)r * kHeadDim;
    store8<kVec>(dst + d0, ra);
    store8<kVec>(dst + kHalf + d0, rb);
    return;
  }
  const long long slot = __ldg(p.slot_mapping + t);
  if (slot < 0) return;  // padding token: no pool row
  if (slot >= p.num_slots) {
    if (r == p.hq && c == 0) report(p.err, PA_DEVERR_SLOT_INDEX);
    return;
  }
  if (r < p.hq + p.hkv) {
    // k head: rotate, store at the slot
    const int h = r - p.hq;
    const uint16_t *src = p.k + t * p.k_tok + (long long)h * kHeadDim;
    const uint4 a = load8<kVec>(src + d0), b = load8<kVec>(src + kHalf + d0);
    const float *cr = p.cos_t + pos * kHalf + d0, *sr = p.sin_t + pos * kHalf + d0;
    uint4 ra, rb;
    rope_rotate8(a, b, __ldg(reinterpret_cast<const float4 *>(cr)),
          __ldg(reinterpret_cast<const float4 *>(cr + 4)),
          __ldg(reinterpret_cast<const float4 *>(sr)),
          __ldg(reinterpret_cast<const float4 *>(sr + 4)), ra, rb);
    uint16_t *dst = p.k_cache + (slot * p.hkv + h) * kHeadDim;
    store8<kVec>(dst + d0, ra);
    store8<kVec>(dst + kHalf + d0, rb);
  } else {
    // v head: stored as it is
    const int h = r - p.hq - p.hkv;
    const uint16_t *src = p.v + t * p.v_tok + (long long)h * kHeadDim;
    uint16_t *dst = p.v_cache + (slot * p.hkv + h) * kHeadDim;
    store8<kVec>(dst + d0, load8<kVec>(src + d0));
    store8<kVec>(dst + kHalf + d0, load8<kVec>(src + kHalf + d0));
  }
}

}  // namespace

}  // namespace pa

extern "C" pa_status pa_rope_store_kv(const void *q, int64_t q_tok_stride, void *q_out,
                                      int64_t q_out_tok_stride, const void *k,
                                      int64_t k_tok_stride, const void *v, int64_t v_tok_stride,
                                      int64_t num_tokens, int32_t num_q_heads,
                                      int32_t num_kv_heads, int32_t head_dim,
                                      const int32_t *positions, const float *cos_table,
                                      const float *sin_table, int64_t max_position,
                                      void *k_cache, void *v_cache, int64_t num_blocks,
                                      int32_t block_size, const int32_t *slot_mapping,
                                      int32_t *error_flags, uint32_t flags, void *stream) {
  using namespace pa;
  if (num_tokens < 0 || num_blocks < 0 || max_position < 0) return PA_ERR_INVALID_ARG;
  if (head_dim != kHeadDim || block_size != kBlockSize) return PA_ERR_UNSUPPORTED;
  if (num_kv_heads < 1 || num_kv_heads > 64 || num_q_heads < 1 || num_q_heads > 512)
    return PA_ERR_UNSUPPORTED;
  if (flags & ~static_cast<uint32_t>(PA_LAUNCH_PDL)) return PA_ERR_INVALID_ARG;
  if (num_tokens == 0) return PA_OK;
  if (!q || !q_out || !k || !v || !positions || !cos_table || !sin_table || !k_cache ||
      !v_cache || !slot_mapping)
    return PA_ERR_INVALID_ARG;
  if (q_tok_stride < 0 || q_out_tok_stride < 0 || k_tok_stride < 0 || v_tok_stride < 0)
    return PA_ERR_INVALID_ARG;
  // the table rows are read as float4: 16-byte aligned tables (rows are
  // 256 bytes, so every row then is)
  if ((reinterpret_cast<uintptr_t>(cos_table) | reinterpret_cast<uintptr_t>(sin_table)) % 16)
    return PA_ERR_INVALID_ARG;
  // 16-byte row accesses when every row chunk is 16-byte aligned
  const bool aligned =
      ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(q_out) |
        reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(v) |
        reinterpret_cast<uintptr_t>(k_cache) | reinterpret_cast<uintptr_t>(v_cache)) % 16 ==
       0) &&
      (q_tok_stride % 8 == 0) && (q_out_tok_stride % 8 == 0) && (k_tok_stride % 8 == 0) &&
      (v_tok_stride % 8 == 0);
  const long long total =
      (long long)num_tokens * (num_q_heads + 2 * num_kv_heads) * (kHeadDim / 16);
  const int threads = 256;
  const long long blocks = (total + threads - 1) / threads;
  if (blocks > 0x7fffffffLL) return PA_ERR_UNSUPPORTED;
  RopeParams rp;
  rp.q = static_cast<const uint16_t *>(q);
  rp.q_tok = q_tok_stride;
  rp.q_out = static_cast<uint16_t *>(q_out);
  rp.q_out_tok = q_out_tok_stride;
  rp.k = static_cast<const uint16_t *>(k);
  rp.k_tok = k_tok_stride;
  rp.v = static_cast<const uint16_t *>(v);
  rp.v_tok = v_tok_stride;
  rp.num_tokens = num_tokens;
  rp.hq = num_q_heads;
  rp.hkv = num_kv_heads;
  rp.positions = positions;
  rp.cos_t = cos_table;
  rp.sin_t = sin_table;
  rp.max_position = max_position;
  rp.k_cache = static_cast<uint16_t *>(k_cache);
  rp.v_cache = static_cast<uint16_t *>(v_cache);
  rp.num_slots = (long long)num_blocks * kBlockSize;
  rp.slot_mapping = slot_mapping;
  rp.err = error_flags;
  const bool pdl = (flags & PA_LAUNCH_PDL) != 0;
  const cudaError_t e =
      launch_kernel(aligned ? rope_store_kernel<true> : rope_store_kernel<false>,
                    dim3((unsigned)blocks), dim3(threads), 0, static_cast<cudaStream_t>(stream),
                    pdl, rp);
  return e == cudaSuccess ? PA_OK : PA_ERR_LAUNCH;
}
