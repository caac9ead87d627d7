// Host side of pa_decode / pa_decode_merge: argument checks, the workspace
// layout, the split count and the launches.  The kernels are in
// pa_decode_kernel.cuh (instantiated in pa_decode_h*.cu).
#include <cmath>

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

constexpr int kMergeSeqPerCta = 8;

// grid (ceil(batch / 8), num_q_heads); warp w merges row (b0 + w, head).
__global__ void __launch_bounds__(32 * kMergeSeqPerCta) merge_kernel(const MergeParams p) {
  __shared__ unsigned long long tot[2];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int b0 = blockIdx.x * kMergeSeqPerCta;
  const int h = blockIdx.y;
  if (tid < 2) tot[tid] = 0;
  __syncthreads();
  unsigned long long all = 0, before = 0;
  for (int b = tid; b < p.batch; b += blockDim.x) {
    const int n = seq_blocks(p.context_lens, b);
    all += n;
    if (b < b0) before += n;
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    all += __shfl_xor_sync(0xffffffffu, all, off);
    before += __shfl_xor_sync(0xffffffffu, before, off);
  }
  if (lane == 0) {
    if (all) atomicAdd(&tot[0], all);
    if (before) atomicAdd(&tot[1], before);
  }
  __syncthreads();
  const int b = b0 + warp;
  if (b >= p.batch) return;
  const long long N = (long long)tot[0];
  long long P = (long long)tot[1];
  for (int x = b0; x < b; ++x) P += seq_blocks(p.context_lens, x);
  const int n = seq_blocks(p.context_lens, b);
  if (n == 0) return;
  const long long S = p.num_splits;
  const long long c0 = split_of_block(P, S, N);
  const long long c1 = split_of_block(P + n - 1, S, N);
  if (c0 == c1) return;
  const int HQ = p.num_q_heads;
  auto piece_row = [&](long long cc) -> long long {
    return (cc * 2 + (cc == c0 ? 1 : 0)) * HQ + h;
  };
  auto nonempty = [&](long long cc) -> bool {
    return split_begin(cc, S, N) < split_begin(cc + 1, S, N);
  };
  float M = -INFINITY;
  for (long long cc = c0; cc <= c1; ++cc)
    if (cc == c0 || nonempty(cc)) M = fmaxf(M, __ldg(p.part_lse + piece_row(cc)));
  float W = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (long long cc = c0; cc <= c1; ++cc) {
    if (cc != c0 && !nonempty(cc)) continue;
    const long long r = piece_row(cc);
    const float lse = __ldg(p.part_lse + r);
    const float w = lse == -INFINITY ? 0.f : __expf(lse - M);
    const float4 o = __ldg(reinterpret_cast<const float4 *>(p.part_o + r * kHeadDim) + lane);
    W += w;
    acc.x += w * o.x;
    acc.y += w * o.y;
    acc.z += w * o.z;
    acc.w += w * o.w;
  }
  const float inv = W > 0.f ? 1.f / W : 0.f;
  const long long base = ((long long)b * HQ + h) * kHeadDim + lane * 4;
  if (p.out_f32) {
    *reinterpret_cast<float4 *>(static_cast<float *>(p.out) + base) =
        make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
  } else {
    uint2 w2;
    w2.x = float2_to_bf16x2(acc.x * inv, acc.y * inv);
    w2.y = float2_to_bf16x2(acc.z * inv, acc.w * inv);
    *reinterpret_cast<uint2 *>(static_cast<uint16_t *>(p.out) + base) = w2;
  }
}


namespace {

constexpr size_t kWsHeader = 256;

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

size_t part_o_bytes(long long splits, int hq) {
  return align256((size_t)splits * 2 * hq * kHeadDim * sizeof(float));
}
size_t part_lse_bytes(long long splits, int hq) {
  return align256((size_t)splits * 2 * hq * sizeof(float));
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

pa_status check_heads(int32_t hq, int32_t hkv, int32_t head_dim, int32_t block_size) {
  if (head_dim != kHeadDim || block_size != kBlockSize) return PA_ERR_UNSUPPORTED;
  if (!(hkv == 1 || hkv == 2 || hkv == 4 || hkv == 8)) return PA_ERR_UNSUPPORTED;
  if (hq < hkv || hq % hkv != 0 || hq / hkv > 8) return PA_ERR_UNSUPPORTED;
  return PA_OK;
}

int current_device() {
  int d = -1;
  return cudaGetDevice(&d) == cudaSuccess ? d : -1;
}

MergeParams merge_params(void *out, int32_t out_dtype, const void *workspace,
                         const int32_t *context_lens, int32_t batch, int32_t hq,
                         int32_t splits) {
  const char *ws = static_cast<const char *>(workspace);
  MergeParams m;
  m.out = out;
  m.out_f32 = out_dtype == PA_DTYPE_F32;
  m.part_o = reinterpret_cast<const float *>(ws + kWsHeader);
  m.part_lse = reinterpret_cast<const float *>(ws + kWsHeader + part_o_bytes(splits, hq));
  m.context_lens = context_lens;
  m.batch = batch;
  m.num_q_heads = hq;
  m.num_splits = splits;
  return m;
}

cudaError_t launch_merge(const MergeParams &m, cudaStream_t s) {
  dim3 grid((m.batch + kMergeSeqPerCta - 1) / kMergeSeqPerCta, m.num_q_heads);
  merge_kernel<<<grid, 32 * kMergeSeqPerCta, 0, s>>>(m);
  return cudaGetLastError();
}

}  // namespace
}  // namespace pa

extern "C" size_t pa_decode_workspace_size(int32_t num_splits, int32_t num_q_heads,
                                           int32_t head_dim) {
  using namespace pa;
  if (num_splits < 1 || num_q_heads < 1 || head_dim != kHeadDim) return 0;
  return kWsHeader + part_o_bytes(num_splits, num_q_heads) +
         part_lse_bytes(num_splits, num_q_heads);
}

extern "C" int32_t pa_decode_default_splits(int32_t device) {
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess)
    return -1;
  return sms;  // one 1-CTA-per-SM split per SM
}

extern "C" pa_status pa_decode(void *out, int32_t out_dtype, const void *q, const void *k_cache,
                               const void *v_cache, int64_t num_blocks,
                               const int32_t *block_tables, int32_t block_table_stride,
                               const int32_t *context_lens, int32_t batch, int32_t num_q_heads,
                               int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                               float scale, int32_t num_splits, void *workspace,
                               size_t workspace_bytes, void *stream) {
  using namespace pa;
  if (batch < 0 || num_blocks < 0 || num_splits < 0) return PA_ERR_INVALID_ARG;
  if (out_dtype != PA_DTYPE_BF16 && out_dtype != PA_DTYPE_F32) return PA_ERR_INVALID_ARG;
  const pa_status hs = check_heads(num_q_heads, num_kv_heads, head_dim, block_size);
  if (hs != PA_OK) return hs;
  if (!std::isfinite(scale)) return PA_ERR_INVALID_ARG;
  if (batch == 0) return PA_OK;
  if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens)
    return PA_ERR_INVALID_ARG;
  if (block_table_stride < 1) return PA_ERR_INVALID_ARG;
  if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache))
    return PA_ERR_INVALID_ARG;
  const int device = current_device();
  if (device < 0) return PA_ERR_DEVICE;
  const int32_t splits = num_splits > 0 ? num_splits : pa_decode_default_splits(device);
  if (splits < 1) return PA_ERR_DEVICE;
  if (!workspace || !aligned16(workspace) ||
      workspace_bytes < pa_decode_workspace_size(splits, num_q_heads, head_dim))
    return PA_ERR_WORKSPACE;

  char *ws = static_cast<char *>(workspace);
  DecodeParams p;
  p.out = out;
  p.out_f32 = out_dtype == PA_DTYPE_F32;
  p.q = static_cast<const uint16_t *>(q);
  p.k_cache = static_cast<const uint16_t *>(k_cache);
  p.v_cache = static_cast<const uint16_t *>(v_cache);
  p.num_blocks = num_blocks;
  p.block_tables = block_tables;
  p.bt_stride = block_table_stride;
  p.context_lens = context_lens;
  p.batch = batch;
  p.qk_scale_log2 = scale * 1.4426950408889634f;
  p.num_splits = splits;
  p.part_o = reinterpret_cast<float *>(ws + kWsHeader);
  p.part_lse = reinterpret_cast<float *>(ws + kWsHeader + part_o_bytes(splits, num_q_heads));
  p.err = reinterpret_cast<int32_t *>(ws);

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int G = num_q_heads / num_kv_heads;
  cudaError_t e;
  switch (num_kv_heads) {
    case 1: e = launch_decode<1>(G, p, s, device); break;
    case 2: e = launch_decode<2>(G, p, s, device); break;
    case 4: e = launch_decode<4>(G, p, s, device); break;
    default: e = launch_decode<8>(G, p, s, device); break;
  }
  if (e != cudaSuccess) return PA_ERR_LAUNCH;
  if (splits > 1) {
    e = launch_merge(merge_params(out, out_dtype, workspace, context_lens, batch, num_q_heads,
                                  splits),
                     s);
    if (e != cudaSuccess) return PA_ERR_LAUNCH;
  }
  return PA_OK;
}

extern "C" pa_status pa_decode_merge(void *out, int32_t out_dtype, const void *workspace,
                                     size_t workspace_bytes, const int32_t *context_lens,
                                     int32_t batch, int32_t num_q_heads, int32_t head_dim,
                                     int32_t block_size, int32_t num_splits, void *stream) {
  using namespace pa;
  if (batch < 0 || num_splits < 1 || num_q_heads < 1) return PA_ERR_INVALID_ARG;
  if (out_dtype != PA_DTYPE_BF16 && out_dtype != PA_DTYPE_F32) return PA_ERR_INVALID_ARG;
  if (head_dim != kHeadDim || block_size != kBlockSize) return PA_ERR_UNSUPPORTED;
  if (num_q_heads > 65535) return PA_ERR_UNSUPPORTED;
  if (batch == 0) return PA_OK;
  if (!out || !context_lens || !aligned16(out)) return PA_ERR_INVALID_ARG;
  if (!workspace || !aligned16(workspace) ||
      workspace_bytes < pa_decode_workspace_size(num_splits, num_q_heads, head_dim))
    return PA_ERR_WORKSPACE;
  const cudaError_t e = launch_merge(
      merge_params(out, out_dtype, workspace, context_lens, batch, num_q_heads, num_splits),
      static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PA_OK : PA_ERR_LAUNCH;
}
