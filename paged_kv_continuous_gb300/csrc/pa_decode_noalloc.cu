// pa_decode_noalloc: pa_decode for callers that cannot allocate device
// memory.  The split partials live in one file-scope __device__ array of
// fixed size instead of a caller-provided workspace.
//
// Who needs this: an engine that hands nearly all device memory to its KV
// block pool at start-up and must not allocate on the decode path; a caller
// that only receives device pointers from a framework that owns the
// allocator; a decode loop that cannot afford the device-wide
// synchronisation a cudaMalloc/cudaFree may cause.
//
// Set-up: the first call on each device, with that device current, resolves
// the array's device address with cudaGetSymbolAddress (a host-side use of
// the array's name is only a host stand-in, never a device address) and
// caches it; make that first call before any stream capture.  Nothing here
// calls cudaMalloc, cudaFree or any allocating routine.
//
// Sharing: every call on a device uses the same array and leaves its
// partials there.  Nothing in it has to start at zero -- each partial the
// merge reads is written earlier in the same call -- but calls that overlap
// on the GPU (two streams, or two threads) race on it and give wrong rows.
#include <cmath>
#include <mutex>

#include "pa_decode_kernel.cuh"

namespace pa {
namespace {

constexpr size_t kStaticScratchBytes = size_t(8) << 20;  // 8 MiB per device
constexpr size_t kWsHeader = 256;                          // same layout as pa_decode's
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_decode_scratch[kStaticScratchBytes];

std::mutex g_scratch_mutex;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of g_decode_scratch on `device` (the current device).
cudaError_t scratch_address(int device, void **ptr) {
  if (device < 0 || device >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (!g_scratch_ptr[device]) {
    void *p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[device] = p;
  }
  *ptr = g_scratch_ptr[device];
  return cudaSuccess;
}

}  // namespace
}  // namespace pa

extern "C" pa_status pa_decode_noalloc(void *out, int32_t out_dtype, const void *q,
                                       const void *k_cache, const void *v_cache,
                                       int64_t num_blocks, const int32_t *block_tables,
                                       int32_t block_table_stride, const int32_t *context_lens,
                                       int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                                       int32_t head_dim, int32_t block_size, float scale,
                                       int32_t num_splits, int32_t *error_flags, void *stream) {
  using namespace pa;
  if (batch < 0 || num_blocks < 0 || num_splits < 0) return PA_ERR_INVALID_ARG;
  if (out_dtype != PA_DTYPE_BF16 && out_dtype != PA_DTYPE_F32) return PA_ERR_INVALID_ARG;
  if (head_dim != kHeadDim || block_size != kBlockSize) return PA_ERR_UNSUPPORTED;
  if (!(num_kv_heads == 1 || num_kv_heads == 2 || num_kv_heads == 4 || num_kv_heads == 8))
    return PA_ERR_UNSUPPORTED;
  if (num_q_heads < num_kv_heads || num_q_heads % num_kv_heads || num_q_heads / num_kv_heads > 8)
    return PA_ERR_UNSUPPORTED;
  if (!std::isfinite(scale)) return PA_ERR_INVALID_ARG;
  if (batch == 0) return PA_OK;
  if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens)
    return PA_ERR_INVALID_ARG;
  if (block_table_stride < 1) return PA_ERR_INVALID_ARG;
  auto misaligned = [](const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) != 0; };
  if (misaligned(out) || misaligned(q) || misaligned(k_cache) || misaligned(v_cache))
    return PA_ERR_INVALID_ARG;
  int device = -1;
  if (cudaGetDevice(&device) != cudaSuccess) return PA_ERR_DEVICE;
  const int32_t splits = num_splits > 0 ? num_splits : pa_decode_default_splits(device);
  if (splits < 1) return PA_ERR_DEVICE;
  // the partials of `splits` splits must fit in the fixed array
  const size_t need = pa_decode_workspace_size(splits, num_q_heads, head_dim);
  if (need == 0 || need > kStaticScratchBytes) return PA_ERR_WORKSPACE;
  void *scratch = nullptr;
  if (scratch_address(device, &scratch) != cudaSuccess) return PA_ERR_DEVICE;

  char *ws = static_cast<char *>(scratch);
  const size_t part_o_bytes =
      ((size_t)splits * 2 * num_q_heads * kHeadDim * sizeof(float) + 255) / 256 * 256;
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
  p.part_lse = reinterpret_cast<float *>(ws + kWsHeader + part_o_bytes);
  p.err = error_flags;

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
  if (splits > 1)
    return pa_decode_merge(out, out_dtype, scratch, kStaticScratchBytes, context_lens, batch,
                           num_q_heads, head_dim, block_size, splits, stream);
  return PA_OK;
}
