// pa_store_kv: the slot_mapping KV-cache store (koas-w, "errors and
// solutions", section "自写 Triton Kernel", store_kvcache_kernel; source rows
// are addressed through strides as in error type 2 of the same page).
//
// One thread moves one 16-byte chunk (8 bf16) of one (token, kv head) row of
// K and of V.  A warp covers two 256-byte head rows, so both the strided
// source reads and the pool writes are full 32-byte sectors.  The pool
// address of (slot, head) is ((slot * Hkv) + head) * head_dim because the
// pool is [block][row][head][dim] and slot = block * block_size + row.
#include "pa_common.cuh"

namespace pa {

template <bool kVec>
__global__ void __launch_bounds__(256) store_kv_kernel(
    const uint16_t *__restrict__ k, const uint16_t *__restrict__ v, long long num_tokens,
    long long k_tok, long long k_head, long long v_tok, long long v_head,
    uint16_t *__restrict__ k_cache, uint16_t *__restrict__ v_cache, long long num_slots,
    int hkv, const int32_t *__restrict__ slot_mapping, int32_t *err) {
  constexpr int kChunks = kHeadDim / 8;  // 16-byte chunks per head row
  // the rows, slots and pools may come from or go to the previous kernel
  griddep_wait();
  griddep_launch_dependents();
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long total = num_tokens * hkv * kChunks;
  if (idx >= total) return;
  const int chunk = (int)(idx % kChunks);
  const long long th = idx / kChunks;
  const int h = (int)(th % hkv);
  const long long t = th / hkv;
  const long long slot = __ldg(slot_mapping + t);
  if (slot < 0) return;  // padding token
  if (slot >= num_slots) {
    if (chunk == 0 && h == 0) report(err, PA_DEVERR_SLOT_INDEX);
    return;
  }
  const long long dst = (slot * hkv + h) * kHeadDim + chunk * 8;
  const long long ks = t * k_tok + h * k_head + chunk * 8;
  const long long vs = t * v_tok + h * v_head + chunk * 8;
  if (kVec) {
    const uint4 kv = __ldg(reinterpret_cast<const uint4 *>(k + ks));
    const uint4 vv = __ldg(reinterpret_cast<const uint4 *>(v + vs));
    *reinterpret_cast<uint4 *>(k_cache + dst) = kv;
    *reinterpret_cast<uint4 *>(v_cache + dst) = vv;
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      k_cache[dst + i] = k[ks + i];
      v_cache[dst + i] = v[vs + i];
    }
  }
}

// Two floats to two E4M3 codes (lo in the low byte): nearest even, magnitudes
// past the largest finite value (448) saturated to it.
__device__ __forceinline__ uint32_t float2_to_e4m3x2(float lo, float hi) {
  unsigned short r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// FP8 store: one thread quantises one 8-element chunk of one (token, kv
// head) row of K and of V: code = nearest-even E4M3 of x / scale[h]
// (IEEE float32 division), saturated to +-448.  K codes go to the
// token-major row (8 bytes), V codes to the dim-major block
// [block][head][dim][16 tokens] (8 bytes, one per dim row).
__global__ void __launch_bounds__(256) store_kv_fp8_kernel(
    const uint16_t *__restrict__ k, const uint16_t *__restrict__ v, long long num_tokens,
    long long k_tok, long long k_head, long long v_tok, long long v_head,
    uint8_t *__restrict__ k_cache, uint8_t *__restrict__ v_cache, long long num_slots, int hkv,
    const float *__restrict__ k_scale, const float *__restrict__ v_scale,
    const int32_t *__restrict__ slot_mapping, int32_t *err) {
  constexpr int kChunks = kHeadDim / 8;
  griddep_wait();
  griddep_launch_dependents();
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= num_tokens * hkv * kChunks) return;
  const int chunk = (int)(idx % kChunks);
  const long long th = idx / kChunks;
  const int h = (int)(th % hkv);
  const long long t = th / hkv;
  const long long slot = __ldg(slot_mapping + t);
  if (slot < 0) return;  // padding token
  if (slot >= num_slots) {
    if (chunk == 0 && h == 0) report(err, PA_DEVERR_SLOT_INDEX);
    return;
  }
  const float ks = __ldg(k_scale + h), vs = __ldg(v_scale + h);
  const uint16_t *kr = k + t * k_tok + h * k_head + chunk * 8;
  const uint16_t *vr = v + t * v_tok + h * v_head + chunk * 8;
  uint32_t kc[2], vc[8];
#pragma unroll
  for (int i = 0; i < 8; i += 4) {
    const float k0 = __uint_as_float((uint32_t)kr[i] << 16);
    const float k1 = __uint_as_float((uint32_t)kr[i + 1] << 16);
    const float k2 = __uint_as_float((uint32_t)kr[i + 2] << 16);
    const float k3 = __uint_as_float((uint32_t)kr[i + 3] << 16);
    kc[i / 4] = float2_to_e4m3x2(__fdiv_rn(k0, ks), __fdiv_rn(k1, ks)) |
                (float2_to_e4m3x2(__fdiv_rn(k2, ks), __fdiv_rn(k3, ks)) << 16);
  }
#pragma unroll
  for (int i = 0; i < 8; i += 2)
    vc[i / 2] = float2_to_e4m3x2(__fdiv_rn(__uint_as_float((uint32_t)vr[i] << 16), vs),
                                 __fdiv_rn(__uint_as_float((uint32_t)vr[i + 1] << 16), vs));
  const long long block = slot / kBlockSize, row = slot % kBlockSize;
  *reinterpret_cast<uint2 *>(k_cache + (slot * hkv + h) * kHeadDim + chunk * 8) =
      make_uint2(kc[0], kc[1]);
  uint8_t *vd = v_cache + ((block * hkv + h) * kHeadDim + chunk * 8) * kBlockSize + row;
#pragma unroll
  for (int i = 0; i < 8; ++i)
    vd[i * kBlockSize] = (uint8_t)(vc[i / 2] >> (8 * (i & 1)));
}

}  // namespace pa

extern "C" pa_status pa_store_kv_fp8(const void *k, const void *v, int64_t num_tokens,
                                     int64_t k_tok_stride, int64_t k_head_stride,
                                     int64_t v_tok_stride, int64_t v_head_stride, void *k_cache,
                                     void *v_cache, const float *k_scale, const float *v_scale,
                                     int64_t num_blocks, int32_t block_size,
                                     int32_t num_kv_heads, int32_t head_dim,
                                     const int32_t *slot_mapping, int32_t *error_flags,
                                     uint32_t flags, void *stream) {
  using namespace pa;
  if (num_tokens < 0 || num_blocks < 0) return PA_ERR_INVALID_ARG;
  if (head_dim != kHeadDim || block_size != kBlockSize) return PA_ERR_UNSUPPORTED;
  if (num_kv_heads < 1 || num_kv_heads > 64) return PA_ERR_UNSUPPORTED;
  if (flags & ~static_cast<uint32_t>(PA_LAUNCH_PDL)) return PA_ERR_INVALID_ARG;
  if (num_tokens == 0) return PA_OK;
  if (!k || !v || !k_cache || !v_cache || !slot_mapping || !k_scale || !v_scale)
    return PA_ERR_INVALID_ARG;
  if (k_tok_stride < 0 || k_head_stride < 0 || v_tok_stride < 0 || v_head_stride < 0)
    return PA_ERR_INVALID_ARG;
  // the K code rows are written 8 bytes at a time
  if (reinterpret_cast<uintptr_t>(k_cache) % 8) return PA_ERR_INVALID_ARG;
  const long long total = (long long)num_tokens * num_kv_heads * (kHeadDim / 8);
  const int threads = 256;
  const long long blocks = (total + threads - 1) / threads;
  if (blocks > 0x7fffffffLL) return PA_ERR_UNSUPPORTED;
  const cudaError_t e = launch_kernel(
      store_kv_fp8_kernel, dim3((unsigned)blocks), dim3(threads), 0,
      static_cast<cudaStream_t>(stream), (flags & PA_LAUNCH_PDL) != 0,
      static_cast<const uint16_t *>(k), static_cast<const uint16_t *>(v), num_tokens,
      (long long)k_tok_stride, (long long)k_head_stride, (long long)v_tok_stride,
      (long long)v_head_stride, static_cast<uint8_t *>(k_cache), static_cast<uint8_t *>(v_cache),
      (long long)num_blocks * kBlockSize, (int)num_kv_heads, k_scale, v_scale, slot_mapping,
      error_flags);
  return e == cudaSuccess ? PA_OK : PA_ERR_LAUNCH;
}

extern "C" pa_status pa_store_kv(const void *k, const void *v, int64_t num_tokens,
                                 int64_t k_tok_stride, int64_t k_head_stride,
                                 int64_t v_tok_stride, int64_t v_head_stride, void *k_cache,
                                 void *v_cache, int64_t num_blocks, int32_t block_size,
                                 int32_t num_kv_heads, int32_t head_dim,
                                 const int32_t *slot_mapping, int32_t *error_flags,
                                 uint32_t flags, void *stream) {
  using namespace pa;
  if (num_tokens < 0 || num_blocks < 0) return PA_ERR_INVALID_ARG;
  if (head_dim != kHeadDim || block_size != kBlockSize) return PA_ERR_UNSUPPORTED;
  if (num_kv_heads < 1 || num_kv_heads > 64) return PA_ERR_UNSUPPORTED;
  if (flags & ~static_cast<uint32_t>(PA_LAUNCH_PDL)) return PA_ERR_INVALID_ARG;
  if (num_tokens == 0) return PA_OK;
  if (!k || !v || !k_cache || !v_cache || !slot_mapping) return PA_ERR_INVALID_ARG;
  if (k_tok_stride < 0 || k_head_stride < 0 || v_tok_stride < 0 || v_head_stride < 0)
    return PA_ERR_INVALID_ARG;
  // 16-byte vector path when every source row chunk is 16-byte aligned.
  const bool aligned =
      ((reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(v) |
        reinterpret_cast<uintptr_t>(k_cache) | reinterpret_cast<uintptr_t>(v_cache)) % 16 == 0) &&
      (k_tok_stride % 8 == 0) && (k_head_stride % 8 == 0) && (v_tok_stride % 8 == 0) &&
      (v_head_stride % 8 == 0);
  const long long total = (long long)num_tokens * num_kv_heads * (kHeadDim / 8);
  const int threads = 256;
  const long long blocks = (total + threads - 1) / threads;
  if (blocks > 0x7fffffffLL) return PA_ERR_UNSUPPORTED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const long long num_slots = (long long)num_blocks * kBlockSize;
  auto *kp = static_cast<const uint16_t *>(k);
  auto *vp = static_cast<const uint16_t *>(v);
  auto *kc = static_cast<uint16_t *>(k_cache);
  auto *vc = static_cast<uint16_t *>(v_cache);
  const bool pdl = (flags & PA_LAUNCH_PDL) != 0;
  const cudaError_t e = launch_kernel(
      aligned ? store_kv_kernel<true> : store_kv_kernel<false>, dim3((unsigned)blocks),
      dim3(threads), 0, s, pdl, kp, vp, num_tokens, (long long)k_tok_stride,
      (long long)k_head_stride, (long long)v_tok_stride, (long long)v_head_stride, kc, vc,
      num_slots, (int)num_kv_heads, slot_mapping, error_flags);
  return e == cudaSuccess ? PA_OK : PA_ERR_LAUNCH;
}
