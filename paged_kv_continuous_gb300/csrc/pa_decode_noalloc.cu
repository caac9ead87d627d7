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
// caches it with the CUDA context it belongs to; make that first call before
// any stream capture.  A later call under another context on that device
// (after cudaDeviceReset, or a primary context released and made again)
// looks the address up again, since the old one belonged to the old
// context; that call, too, must come before any capture.  Nothing here calls
// cudaMalloc, cudaFree or any allocating routine.
//
// Sharing: every call on a device uses the same array and leaves its
// partials there.  The split-K arrival counters in it must start at zero:
// each call clears them on its stream (a memset, not an allocation) before
// the kernel; the partials need no clearing (each one the merge reads is
// written earlier in the same call).  Calls that overlap on the GPU (two
// streams, or two threads) race on the array and give wrong rows.
#include <cmath>
#include <mutex>

#include <cudaTypedefs.h>

#include "pa_decode_internal.h"
#include "pa_decode_kernel.cuh"

namespace pa {
namespace {

constexpr size_t kStaticScratchBytes = size_t(8) << 20;  // 8 MiB per device
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_decode_scratch[kStaticScratchBytes];

std::mutex g_scratch_mutex;
void *g_scratch_ptr[kMaxDevices] = {};
CUcontext g_scratch_ctx[kMaxDevices] = {};

// The driver's cuCtxGetCurrent (the runtime has no call that names the
// current context), looked up once.
PFN_cuCtxGetCurrent_v4000 ctx_get_current() {
  static PFN_cuCtxGetCurrent_v4000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 4000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(f);
  });
  return fn;
}

// Device address of g_decode_scratch on `device` (the current device), for
// the current context: cached per device with the context it was looked up
// in, and looked up again when the current context is another one.
cudaError_t scratch_address(int device, void **ptr) {
  if (device < 0 || device >= kMaxDevices) return cudaErrorInvalidDevice;
  PFN_cuCtxGetCurrent_v4000 get_ctx = ctx_get_current();
  if (!get_ctx) return cudaErrorNotSupported;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  CUcontext cur = nullptr;
  if (get_ctx(&cur) != CUDA_SUCCESS) return cudaErrorUnknown;
  if (!g_scratch_ptr[device] || cur == nullptr || cur != g_scratch_ctx[device]) {
    void *p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e != cudaSuccess) return e;
    // the lookup made the runtime's context current if none was
    if (get_ctx(&cur) != CUDA_SUCCESS || cur == nullptr) return cudaErrorUnknown;
    g_scratch_ptr[device] = p;
    g_scratch_ctx[device] = cur;
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
                                       int32_t num_splits, int32_t *error_flags, uint32_t flags,
                                       void *stream) {
  using namespace pa;
  DecodeRequest r{out, out_dtype, q, k_cache, v_cache, num_blocks, block_tables,
                  block_table_stride, context_lens, batch, num_q_heads, num_kv_heads, head_dim,
                  block_size, scale, num_splits, 0, flags, stream};
  int device = -1;
  const pa_status st = check_decode_request(r, &device);
  if (st != PA_OK || batch == 0) return st;
  // the partials and counters of `splits` splits must fit in the fixed array;
  // a default split count is lowered to the largest that fits
  if (num_splits == 0)
    while (r.splits > 1 &&
           pa_decode_workspace_size(r.splits, num_q_heads, head_dim) > kStaticScratchBytes)
      --r.splits;
  const size_t need = pa_decode_workspace_size(r.splits, num_q_heads, head_dim);
  if (need == 0 || need > kStaticScratchBytes) return PA_ERR_WORKSPACE;
  void *scratch = nullptr;
  if (scratch_address(device, &scratch) != cudaSuccess) return PA_ERR_DEVICE;
  // the arrival counters must start at zero: clear them on the stream first
  return run_decode(r, scratch, error_flags, device, /*clear_counters=*/true);
}
