// Host side of pa_decode / pa_decode_merge: argument checks, the workspace
// layout, the split count, the TMA tensor maps of the two pools and the
// launches.  The decode kernel is in pa_decode_kernel.cuh (instantiated in
// pa_decode_h*.cu); the standalone merge kernel is below.
#include <climits>
#include <cstring>
#include <cmath>
#include <mutex>

#include <cudaTypedefs.h>

#include "pa_decode_internal.h"
#include "pa_decode_kernel.cuh"

namespace pa {

// ---- merge of cut sequences ---------------------------------------------------

struct MergeParams {
  void *out;
  int out_f32;
  const float *part_o;
  const float *part_lse;
  const int32_t *context_lens;
  int batch;
  int num_q_heads;
  int num_splits;
};

constexpr int kMergeWarps = 4;   // warps per (sequence, head) row, a quarter of its pieces each
constexpr int kMergeChunk = 16;  // pieces whose loads are in flight together in one warp

// One warp's share of a log-sum-exp merge: the partials of splits ca..cb of
// a sequence whose first split is c0 (slot 1 of c0, slot 0 of the others;
// partials are [slot][split][head][dim]), row h; lane l owns dims 4l..4l+3.
// When N >= S every split holds at least one block; otherwise empty splits
// are skipped.  Pieces go in split order, kMergeChunk at a time with all
// their loads (lane i < kMergeChunk: the lse of piece i; every lane: its
// four dims of each piece's row) in flight together.  Returns M (the
// largest lse), W = sum_i e_i and acc = sum_i e_i o_i with e_i =
// exp(lse_i - M); a chunk that raises M rescales the sums so far by
// exp(M_old - M_new).
struct MergePart {
  float M, W;
  float4 acc;
};
__device__ __forceinline__ MergePart merge_part(const float *part_o, const float *part_lse,
                                                int HQ, int h, long long c0, long long ca,
                                                long long cb, long long S, long long N,
                                                int lane) {
  const bool dense = N >= S;
  auto piece = [&](long long cc) -> bool {
    return cc <= cb && (dense || cc == c0 || split_begin(cc, S, N) < split_begin(cc + 1, S, N));
  };
  auto row_of = [&](long long cc) -> long long { return ((cc == c0 ? 1 : 0) * S + cc) * HQ + h; };
  MergePart r{-INFINITY, 0.f, make_float4(0.f, 0.f, 0.f, 0.f)};
  for (long long base = ca; base <= cb; base += kMergeChunk) {
    const long long mine = base + lane;
    const float ls =
        lane < kMergeChunk && piece(mine) ? __ldcg(part_lse + row_of(mine)) : -INFINITY;
    float4 v[kMergeChunk];
#pragma unroll
    for (int u = 0; u < kMergeChunk; ++u)
      v[u] = piece(base + u)
                 ? __ldcg(reinterpret_cast<const float4 *>(part_o + row_of(base + u) * kHeadDim) +
                          lane)
                 : make_float4(0.f, 0.f, 0.f, 0.f);
    float mc = ls;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mc = fmaxf(mc, __shfl_xor_sync(0xffffffffu, mc, off));
    const float Mn = fmaxf(r.M, mc);
    if (Mn == -INFINITY) continue;  // no piece with a key so far
    const float sc = __expf(r.M - Mn);  // 0 for the first chunk (M = -inf)
    r.W *= sc;
    r.acc.x *= sc;
    r.acc.y *= sc;
    r.acc.z *= sc;
    r.acc.w *= sc;
#pragma unroll
    for (int u = 0; u < kMergeChunk; ++u) {
      const float lu = __shfl_sync(0xffffffffu, ls, u);
      const float e = lu == -INFINITY ? 0.f : __expf(lu - Mn);
      r.W += e;
      r.acc.x = fmaf(e, v[u].x, r.acc.x);
      r.acc.y = fmaf(e, v[u].y, r.acc.y);
      r.acc.z = fmaf(e, v[u].z, r.acc.z);
      r.acc.w = fmaf(e, v[u].w, r.acc.w);
    }
    r.M = Mn;
  }
  return r;
}

// grid (batch, num_q_heads): CTA (b, h) merges row h of sequence b when the
// partition cut it (splits c0 < c1), its kMergeWarps warps taking a quarter
// of the splits each (one round of loads for up to 64 pieces); warp 0 then
// combines the four shares:
//   M = max_w M_w,  s_w = exp(M_w - M),  out = sum_w s_w acc_w / sum_w s_w W_w.
// The block counts and the partition come from context_lens alone, before
// the wait for the kernel before it (the decode kernel, under a
// programmatic dependent launch); the partials after it.  The next kernel in
// the stream may begin at once: its own wait covers this one.
__global__ void __launch_bounds__(32 * kMergeWarps) merge_kernel(const MergeParams p) {
  griddep_launch_dependents();
  __shared__ long long red[2][kMergeWarps];
  __shared__ float share_mw[kMergeWarps][2];
  __shared__ float4 share_acc[kMergeWarps][32];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int b = blockIdx.x, h = blockIdx.y;
  const long long S = p.num_splits;
  // N and the blocks before sequence b
  long long all = 0, before = 0;
  for (int x = tid; x < p.batch; x += 32 * kMergeWarps) {
    const int n = seq_blocks(p.context_lens, x);
    all += n;
    if (x < b) before += n;
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    all += __shfl_xor_sync(0xffffffffu, all, off);
    before += __shfl_xor_sync(0xffffffffu, before, off);
  }
  if (lane == 0) {
    red[0][warp] = all;
    red[1][warp] = before;
  }
  __syncthreads();
  long long N = 0, P = 0;
#pragma unroll
  for (int w = 0; w < kMergeWarps; ++w) {
    N += red[0][w];
    P += red[1][w];
  }
  const int n = seq_blocks(p.context_lens, b);
  if (n == 0) return;
  const long long c0 = split_of_block(P, S, N), c1 = split_of_block(P + n - 1, S, N);
  if (c0 == c1) return;  // held by one split: its rows are written already
  griddep_wait();
  const long long q = (c1 - c0 + kMergeWarps) / kMergeWarps;  // splits per warp
  const long long ca = c0 + warp * q, cb = min(c1, ca + q - 1);
  const MergePart r = merge_part(p.part_o, p.part_lse, p.num_q_heads, h, c0, ca, cb, S, N, lane);
  share_acc[warp][lane] = r.acc;
  if (lane == 0) {
    share_mw[warp][0] = r.M;
    share_mw[warp][1] = r.W;
  }
  __syncthreads();
  if (warp != 0) return;
  float M = -INFINITY;
#pragma unroll
  for (int w = 0; w < kMergeWarps; ++w) M = fmaxf(M, share_mw[w][0]);
  float W = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int w = 0; w < kMergeWarps; ++w) {
    const float mw = share_mw[w][0];
    const float sw = mw == -INFINITY ? 0.f : __expf(mw - M);
    const float4 a = share_acc[w][lane];
    W = fmaf(sw, share_mw[w][1], W);
    acc.x = fmaf(sw, a.x, acc.x);
    acc.y = fmaf(sw, a.y, acc.y);
    acc.z = fmaf(sw, a.z, acc.z);
    acc.w = fmaf(sw, a.w, acc.w);
  }
  const float inv = W > 0.f ? 1.f / W : 0.f;
  store_out4(p.out, p.out_f32, ((long long)b * p.num_q_heads + h) * kHeadDim + lane * 4,
             make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv));
}

namespace {

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
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

// 3-D view of a pool: (dim 128, kv head Hkv, token slot num_blocks * 16).
// One TMA box = 64 dims x min(Hkv, 2) heads x 16 slots (one page), with the
// 128-byte swizzle.
bool encode_pool_map(CUtensorMap *map, const void *pool, long long num_blocks, int hkv) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return false;
  cuuint64_t dims[3] = {(cuuint64_t)kHeadDim, (cuuint64_t)hkv,
                        (cuuint64_t)num_blocks * kBlockSize};
  cuuint64_t strides[2] = {(cuuint64_t)kHeadDim * 2, (cuuint64_t)hkv * kHeadDim * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)(hkv >= 2 ? 2 : 1), (cuuint32_t)kBlockSize};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(pool), dims, strides,
             box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// FP8 pools.  K: (128 dims, kv head, token slot) of bytes; one box = 128
// dims x min(Hkv, 2) heads x 16 slots, 128-byte swizzle.  V, dim-major inside
// a block, is read by plain bulk copies (one per block); its map -- (16
// tokens, 128 dims, block * Hkv + head) -- only validates the pool.
bool encode_pool_maps_fp8(CUtensorMap *mk, CUtensorMap *mv, const void *k_pool,
                          const void *v_pool, long long num_blocks, int hkv) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return false;
  const cuuint32_t hb = (cuuint32_t)(hkv >= 2 ? 2 : 1);
  cuuint32_t estr[3] = {1, 1, 1};
  cuuint64_t kd[3] = {(cuuint64_t)kHeadDim, (cuuint64_t)hkv,
                      (cuuint64_t)num_blocks * kBlockSize};
  cuuint64_t ks[2] = {(cuuint64_t)kHeadDim, (cuuint64_t)hkv * kHeadDim};
  cuuint32_t kbox[3] = {(cuuint32_t)kHeadDim, hb, (cuuint32_t)kBlockSize};
  cuuint64_t vd[3] = {(cuuint64_t)kBlockSize, (cuuint64_t)kHeadDim,
                      (cuuint64_t)num_blocks * hkv};
  cuuint64_t vs[2] = {(cuuint64_t)kBlockSize, (cuuint64_t)kHeadDim * kBlockSize};
  cuuint32_t vbox[3] = {(cuuint32_t)kBlockSize, (cuuint32_t)kHeadDim, hb};
  return enc(mk, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(k_pool), kd, ks, kbox,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
             CUDA_SUCCESS &&
         enc(mv, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(v_pool), vd, vs, vbox,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
             CUDA_SUCCESS;
}

cudaError_t launch_merge(const MergeParams &m, cudaStream_t s, bool pdl) {
  const dim3 grid((unsigned)m.batch, (unsigned)m.num_q_heads);
  return launch_kernel(merge_kernel, grid, dim3(32 * kMergeWarps), 0, s, pdl, m);
}

}  // namespace

WorkspaceLayout workspace_layout(long long splits, int hq) {
  WorkspaceLayout w;
  w.counters = kCounterOffset;
  w.part_o = kCounterOffset + kCounterBytes;
  w.part_lse = w.part_o + align256((size_t)splits * 2 * hq * kHeadDim * sizeof(float));
  w.total = w.part_lse + align256((size_t)splits * 2 * hq * sizeof(float));
  return w;
}

pa_status run_decode(const DecodeRequest &r, void *workspace, int32_t *err, int device,
                     bool clear_counters) {
  const WorkspaceLayout L = workspace_layout(r.splits, r.num_q_heads);
  char *ws = static_cast<char *>(workspace);
  CUtensorMap tk, tv;
  memset(&tk, 0, sizeof tk);
  memset(&tv, 0, sizeof tv);
  if (r.num_blocks > 0) {
    const bool ok =
        r.fp8 ? encode_pool_maps_fp8(&tk, &tv, r.k_cache, r.v_cache, r.num_blocks,
                                     r.num_kv_heads)
              : encode_pool_map(&tk, r.k_cache, r.num_blocks, r.num_kv_heads) &&
                    encode_pool_map(&tv, r.v_cache, r.num_blocks, r.num_kv_heads);
    if (!ok) return PA_ERR_DEVICE;
  }
  DecodeParams p;
  p.out = r.out;
  p.out_f32 = r.out_dtype == PA_DTYPE_F32;
  p.q = static_cast<const uint16_t *>(r.q);
  p.num_blocks = r.num_blocks;
  p.block_tables = r.block_tables;
  p.bt_stride = r.block_table_stride;
  p.context_lens = r.context_lens;
  p.batch = r.batch;
  p.qk_scale_log2 = r.scale * 1.4426950408889634f;
  p.num_splits = r.splits;
  p.part_o = reinterpret_cast<float *>(ws + L.part_o);
  p.part_lse = reinterpret_cast<float *>(ws + L.part_lse);
  p.counters = reinterpret_cast<int32_t *>(ws + L.counters);
  p.err = err;
  p.k_scale = r.k_scale;
  p.v_scale = r.v_scale;
  p.v_pool = r.fp8 ? static_cast<const uint8_t *>(r.v_cache) : nullptr;
  p.new_k = static_cast<const uint16_t *>(r.new_k);
  p.new_v = static_cast<const uint16_t *>(r.new_v);
  p.new_k_tok = r.new_k_tok;
  p.new_v_tok = r.new_v_tok;
  p.slot_mapping = r.slot_mapping;
  p.k_pool = r.fp8 ? nullptr : static_cast<uint16_t *>(const_cast<void *>(r.k_cache));
  p.v_pool16 = r.fp8 ? nullptr : static_cast<uint16_t *>(const_cast<void *>(r.v_cache));
  p.k_pool8 = r.fp8 ? static_cast<uint8_t *>(const_cast<void *>(r.k_cache)) : nullptr;
  p.v_pool8 = r.fp8 ? static_cast<uint8_t *>(const_cast<void *>(r.v_cache)) : nullptr;
  p.early_kv = (r.flags & PA_LAUNCH_EARLY_KV) != 0;
  p.positions = r.positions;
  p.cos_table = r.cos_table;
  p.sin_table = r.sin_table;
  p.max_position = r.max_position;
  cudaStream_t s = static_cast<cudaStream_t>(r.stream);
  if (clear_counters &&
      cudaMemsetAsync(p.counters, 0, (size_t)r.splits * sizeof(int32_t), s) != cudaSuccess)
    return PA_ERR_LAUNCH;
  const int G = r.num_q_heads / r.num_kv_heads;
  const bool pdl = (r.flags & PA_LAUNCH_PDL) != 0;
  // Few sequences over many splits (at least 8 per sequence) with 4 or 8 kv
  // heads: every cut sequence has many pieces of many query heads, and one
  // CTA merging them at the end of the decode kernel sets its end; merge
  // them in merge_kernel instead, spread over all splits and heads.
  const bool split_merge = !r.positions && r.num_kv_heads >= 4 &&
                           (long long)r.splits >= 8LL * r.batch;
  cudaError_t e;
  if (r.fp8) {
    switch (r.num_kv_heads) {
      case 1: e = launch_decode<1, true>(G, tk, tv, p, s, device, pdl); break;
      case 2: e = launch_decode<2, true>(G, tk, tv, p, s, device, pdl); break;
      case 4:
        e = split_merge ? launch_decode<4, true, false, true>(G, tk, tv, p, s, device, pdl)
                        : launch_decode<4, true>(G, tk, tv, p, s, device, pdl);
        break;
      default:
        e = split_merge ? launch_decode<8, true, false, true>(G, tk, tv, p, s, device, pdl)
                        : launch_decode<8, true>(G, tk, tv, p, s, device, pdl);
        break;
    }
  } else if (r.positions) {
    switch (r.num_kv_heads) {
      case 1: e = launch_decode<1, false, true>(G, tk, tv, p, s, device, pdl); break;
      case 2: e = launch_decode<2, false, true>(G, tk, tv, p, s, device, pdl); break;
      case 4: e = launch_decode<4, false, true>(G, tk, tv, p, s, device, pdl); break;
      default: e = launch_decode<8, false, true>(G, tk, tv, p, s, device, pdl); break;
    }
  } else {
    switch (r.num_kv_heads) {
      case 1: e = launch_decode<1, false>(G, tk, tv, p, s, device, pdl); break;
      case 2: e = launch_decode<2, false>(G, tk, tv, p, s, device, pdl); break;
      case 4:
        e = split_merge ? launch_decode<4, false, false, true>(G, tk, tv, p, s, device, pdl)
                        : launch_decode<4, false>(G, tk, tv, p, s, device, pdl);
        break;
      default:
        e = split_merge ? launch_decode<8, false, false, true>(G, tk, tv, p, s, device, pdl)
                        : launch_decode<8, false>(G, tk, tv, p, s, device, pdl);
        break;
    }
  }
  if (e != cudaSuccess) return PA_ERR_LAUNCH;
  if (split_merge) {
    // a programmatic dependent launch behind the decode kernel: it waits
    // for the partials, and lets the next kernel in the stream begin at once
    MergeParams m;
    m.out = r.out;
    m.out_f32 = p.out_f32;
    m.part_o = p.part_o;
    m.part_lse = p.part_lse;
    m.context_lens = r.context_lens;
    m.batch = r.batch;
    m.num_q_heads = r.num_q_heads;
    m.num_splits = r.splits;
    if (launch_merge(m, s, true) != cudaSuccess) return PA_ERR_LAUNCH;
  }
  return PA_OK;
}

pa_status check_decode_request(DecodeRequest &r, int *device_out) {
  if (r.batch < 0 || r.num_blocks < 0 || r.num_splits < 0) return PA_ERR_INVALID_ARG;
  if (r.flags & ~static_cast<uint32_t>(PA_LAUNCH_PDL | PA_LAUNCH_EARLY_KV))
    return PA_ERR_INVALID_ARG;
  if ((r.flags & PA_LAUNCH_EARLY_KV) && !(r.flags & PA_LAUNCH_PDL)) return PA_ERR_INVALID_ARG;
  if (r.num_splits > PA_DECODE_MAX_SPLITS) return PA_ERR_UNSUPPORTED;
  if (r.out_dtype != PA_DTYPE_BF16 && r.out_dtype != PA_DTYPE_F32) return PA_ERR_INVALID_ARG;
  if (r.head_dim != kHeadDim || r.block_size != kBlockSize) return PA_ERR_UNSUPPORTED;
  const int hkv = r.num_kv_heads, hq = r.num_q_heads;
  if (!(hkv == 1 || hkv == 2 || hkv == 4 || hkv == 8)) return PA_ERR_UNSUPPORTED;
  if (hq < hkv || hq % hkv != 0 || hq / hkv > 8) return PA_ERR_UNSUPPORTED;
  if (!std::isfinite(r.scale)) return PA_ERR_INVALID_ARG;
  if (r.num_blocks > (long long)(INT_MAX / kBlockSize)) return PA_ERR_UNSUPPORTED;
  if (r.batch == 0) return PA_OK;
  if (!r.out || !r.q || !r.k_cache || !r.v_cache || !r.block_tables || !r.context_lens)
    return PA_ERR_INVALID_ARG;
  if (r.block_table_stride < 1) return PA_ERR_INVALID_ARG;
  if (!aligned16(r.out) || !aligned16(r.q) || !aligned16(r.k_cache) || !aligned16(r.v_cache))
    return PA_ERR_INVALID_ARG;
  int device = -1;
  if (cudaGetDevice(&device) != cudaSuccess || device < 0) return PA_ERR_DEVICE;
  r.splits = r.num_splits > 0 ? r.num_splits : pa_decode_default_splits(device, hq, hkv);
  if (r.splits < 1) return PA_ERR_DEVICE;
  if (r.splits > PA_DECODE_MAX_SPLITS) r.splits = PA_DECODE_MAX_SPLITS;
  *device_out = device;
  return PA_OK;
}

}  // namespace pa

extern "C" size_t pa_decode_workspace_size(int32_t num_splits, int32_t num_q_heads,
                                           int32_t head_dim) {
  using namespace pa;
  if (num_splits < 1 || num_splits > PA_DECODE_MAX_SPLITS || num_q_heads < 1 ||
      head_dim != kHeadDim)
    return 0;
  return workspace_layout(num_splits, num_q_heads).total;
}

extern "C" int32_t pa_decode_default_splits(int32_t device, int32_t num_q_heads,
                                            int32_t num_kv_heads) {
  if (num_q_heads < 1 || num_kv_heads < 1) return -1;
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess)
    return -1;
  return sms;  // the decode kernel keeps one CTA per SM for every head shape
}

extern "C" pa_status pa_decode(void *out, int32_t out_dtype, const void *q, const void *k_cache,
                               const void *v_cache, int64_t num_blocks,
                               const int32_t *block_tables, int32_t block_table_stride,
                               const int32_t *context_lens, int32_t batch, int32_t num_q_heads,
                               int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                               float scale, int32_t num_splits, void *workspace,
                               size_t workspace_bytes, uint32_t flags, void *stream) {
  using namespace pa;
  DecodeRequest r{out, out_dtype, q, k_cache, v_cache, num_blocks, block_tables,
                  block_table_stride, context_lens, batch, num_q_heads, num_kv_heads, head_dim,
                  block_size, scale, num_splits, 0, flags, stream};
  int device = -1;
  const pa_status st = check_decode_request(r, &device);
  if (st != PA_OK || batch == 0) return st;
  if (!workspace || !aligned16(workspace) ||
      workspace_bytes < pa_decode_workspace_size(r.splits, num_q_heads, head_dim))
    return PA_ERR_WORKSPACE;
  return run_decode(r, workspace, static_cast<int32_t *>(workspace), device, false);
}

extern "C" pa_status pa_store_decode(void *out, int32_t out_dtype, const void *q,
                                     const void *new_k, const void *new_v,
                                     int64_t new_k_tok_stride, int64_t new_v_tok_stride,
                                     const int32_t *slot_mapping, void *k_cache, void *v_cache,
                                     int64_t num_blocks, const int32_t *block_tables,
                                     int32_t block_table_stride, const int32_t *context_lens,
                                     int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                                     int32_t head_dim, int32_t block_size, float scale,
                                     int32_t num_splits, void *workspace, size_t workspace_bytes,
                                     uint32_t flags, void *stream) {
  using namespace pa;
  DecodeRequest r{out, out_dtype, q, k_cache, v_cache, num_blocks, block_tables,
                  block_table_stride, context_lens, batch, num_q_heads, num_kv_heads, head_dim,
                  block_size, scale, num_splits, 0, flags, stream};
  r.new_k = new_k;
  r.new_v = new_v;
  r.new_k_tok = new_k_tok_stride;
  r.new_v_tok = new_v_tok_stride;
  r.slot_mapping = slot_mapping;
  if (batch > 0 && (!new_k || !new_v || !slot_mapping)) return PA_ERR_INVALID_ARG;
  int device = -1;
  const pa_status st = check_decode_request(r, &device);
  if (st != PA_OK || batch == 0) return st;
  // the new rows are moved in 16-byte chunks
  if (!aligned16(new_k) || !aligned16(new_v) || new_k_tok_stride < num_kv_heads * head_dim ||
      new_v_tok_stride < num_kv_heads * head_dim || new_k_tok_stride % 8 ||
      new_v_tok_stride % 8)
    return PA_ERR_INVALID_ARG;
  if (!workspace || !aligned16(workspace) ||
      workspace_bytes < pa_decode_workspace_size(r.splits, num_q_heads, head_dim))
    return PA_ERR_WORKSPACE;
  return run_decode(r, workspace, static_cast<int32_t *>(workspace), device, false);
}

extern "C" pa_status pa_rope_store_decode(
    void *out, int32_t out_dtype, const void *q, const void *new_k, const void *new_v,
    int64_t new_k_tok_stride, int64_t new_v_tok_stride, const int32_t *positions,
    const float *cos_table, const float *sin_table, int64_t max_position,
    const int32_t *slot_mapping, void *k_cache, void *v_cache, int64_t num_blocks,
    const int32_t *block_tables, int32_t block_table_stride, const int32_t *context_lens,
    int32_t batch, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
    int32_t block_size, float scale, int32_t num_splits, void *workspace,
    size_t workspace_bytes, uint32_t flags, void *stream) {
  using namespace pa;
  DecodeRequest r{out, out_dtype, q, k_cache, v_cache, num_blocks, block_tables,
                  block_table_stride, context_lens, batch, num_q_heads, num_kv_heads, head_dim,
                  block_size, scale, num_splits, 0, flags, stream};
  r.new_k = new_k;
  r.new_v = new_v;
  r.new_k_tok = new_k_tok_stride;
  r.new_v_tok = new_v_tok_stride;
  r.slot_mapping = slot_mapping;
  r.positions = positions;
  r.cos_table = cos_table;
  r.sin_table = sin_table;
  r.max_position = max_position;
  if (batch > 0 &&
      (!new_k || !new_v || !slot_mapping || !positions || !cos_table || !sin_table))
    return PA_ERR_INVALID_ARG;
  // table rows are brought by bulk copies: 16-byte aligned bases
  if (batch > 0 && (max_position < 1 || !aligned16(cos_table) || !aligned16(sin_table)))
    return PA_ERR_INVALID_ARG;
  int device = -1;
  const pa_status st = check_decode_request(r, &device);
  if (st != PA_OK || batch == 0) return st;
  if (!aligned16(new_k) || !aligned16(new_v) || new_k_tok_stride < num_kv_heads * head_dim ||
      new_v_tok_stride < num_kv_heads * head_dim || new_k_tok_stride % 8 ||
      new_v_tok_stride % 8)
    return PA_ERR_INVALID_ARG;
  if (!workspace || !aligned16(workspace) ||
      workspace_bytes < pa_decode_workspace_size(r.splits, num_q_heads, head_dim))
    return PA_ERR_WORKSPACE;
  return run_decode(r, workspace, static_cast<int32_t *>(workspace), device, false);
}

extern "C" pa_status pa_store_decode_fp8(
    void *out, int32_t out_dtype, const void *q, const void *new_k, const void *new_v,
    int64_t new_k_tok_stride, int64_t new_v_tok_stride, const int32_t *slot_mapping,
    void *k_cache, void *v_cache, const float *k_scale, const float *v_scale, int64_t num_blocks,
    const int32_t *block_tables, int32_t block_table_stride, const int32_t *context_lens,
    int32_t batch, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
    int32_t block_size, float scale, int32_t num_splits, void *workspace,
    size_t workspace_bytes, uint32_t flags, void *stream) {
  using namespace pa;
  DecodeRequest r{out, out_dtype, q, k_cache, v_cache, num_blocks, block_tables,
                  block_table_stride, context_lens, batch, num_q_heads, num_kv_heads, head_dim,
                  block_size, scale, num_splits, 0, flags, stream};
  r.fp8 = true;
  r.k_scale = k_scale;
  r.v_scale = v_scale;
  r.new_k = new_k;
  r.new_v = new_v;
  r.new_k_tok = new_k_tok_stride;
  r.new_v_tok = new_v_tok_stride;
  r.slot_mapping = slot_mapping;
  if (batch > 0 && (!k_scale || !v_scale || !new_k || !new_v || !slot_mapping))
    return PA_ERR_INVALID_ARG;
  int device = -1;
  const pa_status st = check_decode_request(r, &device);
  if (st != PA_OK || batch == 0) return st;
  if (!aligned16(new_k) || !aligned16(new_v) || new_k_tok_stride < num_kv_heads * head_dim ||
      new_v_tok_stride < num_kv_heads * head_dim || new_k_tok_stride % 8 ||
      new_v_tok_stride % 8)
    return PA_ERR_INVALID_ARG;
  if (!workspace || !aligned16(workspace) ||
      workspace_bytes < pa_decode_workspace_size(r.splits, num_q_heads, head_dim))
    return PA_ERR_WORKSPACE;
  return run_decode(r, workspace, static_cast<int32_t *>(workspace), device, false);
}

extern "C" pa_status pa_decode_fp8(void *out, int32_t out_dtype, const void *q,
                                   const void *k_cache, const void *v_cache, const float *k_scale,
                                   const float *v_scale, int64_t num_blocks,
                                   const int32_t *block_tables, int32_t block_table_stride,
                                   const int32_t *context_lens, int32_t batch,
                                   int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                   int32_t block_size, float scale, int32_t num_splits,
                                   void *workspace, size_t workspace_bytes, uint32_t flags,
                                   void *stream) {
  using namespace pa;
  DecodeRequest r{out, out_dtype, q, k_cache, v_cache, num_blocks, block_tables,
                  block_table_stride, context_lens, batch, num_q_heads, num_kv_heads, head_dim,
                  block_size, scale, num_splits, 0, flags, stream};
  r.fp8 = true;
  r.k_scale = k_scale;
  r.v_scale = v_scale;
  if (batch > 0 && (!k_scale || !v_scale)) return PA_ERR_INVALID_ARG;
  int device = -1;
  const pa_status st = check_decode_request(r, &device);
  if (st != PA_OK || batch == 0) return st;
  if (!workspace || !aligned16(workspace) ||
      workspace_bytes < pa_decode_workspace_size(r.splits, num_q_heads, head_dim))
    return PA_ERR_WORKSPACE;
  return run_decode(r, workspace, static_cast<int32_t *>(workspace), device, false);
}

extern "C" pa_status pa_decode_merge(void *out, int32_t out_dtype, const void *workspace,
                                     size_t workspace_bytes, const int32_t *context_lens,
                                     int32_t batch, int32_t num_q_heads, int32_t head_dim,
                                     int32_t block_size, int32_t num_splits, void *stream) {
  using namespace pa;
  if (batch < 0 || num_splits < 1 || num_q_heads < 1) return PA_ERR_INVALID_ARG;
  if (out_dtype != PA_DTYPE_BF16 && out_dtype != PA_DTYPE_F32) return PA_ERR_INVALID_ARG;
  if (head_dim != kHeadDim || block_size != kBlockSize) return PA_ERR_UNSUPPORTED;
  if (num_q_heads > 65535 || num_splits > PA_DECODE_MAX_SPLITS) return PA_ERR_UNSUPPORTED;
  if (batch == 0) return PA_OK;
  if (!out || !context_lens || !aligned16(out)) return PA_ERR_INVALID_ARG;
  if (!workspace || !aligned16(workspace) ||
      workspace_bytes < pa_decode_workspace_size(num_splits, num_q_heads, head_dim))
    return PA_ERR_WORKSPACE;
  const WorkspaceLayout L = workspace_layout(num_splits, num_q_heads);
  const char *ws = static_cast<const char *>(workspace);
  MergeParams m;
  m.out = out;
  m.out_f32 = out_dtype == PA_DTYPE_F32;
  m.part_o = reinterpret_cast<const float *>(ws + L.part_o);
  m.part_lse = reinterpret_cast<const float *>(ws + L.part_lse);
  m.context_lens = context_lens;
  m.batch = batch;
  m.num_q_heads = num_q_heads;
  m.num_splits = num_splits;
  return launch_merge(m, static_cast<cudaStream_t>(stream), false) == cudaSuccess
             ? PA_OK
             : PA_ERR_LAUNCH;
}
