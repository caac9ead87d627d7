// pa_copy: a byte copy, as a kernel, between two buffers the device can
// address -- device memory, or pinned host memory, which on this machine the
// device reads and writes through the same address over the CPU-GPU link.
//
// A serving loop stages each step's inputs from host memory and reads its
// result back.  A cudaMemcpyAsync between two kernels of a stream ends their
// programmatic-launch overlap: the second kernel cannot start before the
// copy, which cannot start before the first kernel completes.  As a kernel
// launched with programmatic dependent launch, the copy keeps the chain: it
// begins during the previous kernel's tail.  With PA_COPY_BEFORE_WAIT it
// moves its bytes and lets the next kernel begin before that kernel
// completes (the caller guarantees that no kernel still running writes the
// source or touches the destination, and that the next kernel reads the
// destination only after its own wait).
//
// One thread moves 16-byte chunks in a grid-stride loop, four loads in
// flight; the bytes past the last whole chunk are copied one by one.
#include "pa_common.cuh"

namespace pa {
namespace {

constexpr int kCopyThreads = 256;

__global__ void __launch_bounds__(kCopyThreads)
    copy_kernel(uint8_t *__restrict__ dst, const uint8_t *__restrict__ src, long long n16,
                int tail, int before_wait) {
  if (!before_wait) griddep_wait();
  uint4 *d = reinterpret_cast<uint4 *>(dst);
  const uint4 *s = reinterpret_cast<const uint4 *>(src);
  const long long stride = (long long)gridDim.x * blockDim.x;
  long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  for (; i + 3 * stride < n16; i += 4 * stride) {
    uint4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) v[u] = s[i + u * stride];
#pragma unroll
    for (int u = 0; u < 4; ++u) d[i + u * stride] = v[u];
  }
  for (; i < n16; i += stride) d[i] = s[i];
  if (blockIdx.x == 0 && threadIdx.x < tail) dst[n16 * 16 + threadIdx.x] = src[n16 * 16 + threadIdx.x];
  // Before the wait, the copy also lets the next kernel begin at once: a
  // staging copy between two decode steps then keeps the next step's start
  // overlapping the previous step's tail.  That next kernel's own wait still
  // covers every kernel before it (this one completes only after its wait).
  if (before_wait) {
    griddep_launch_dependents();
    griddep_wait();
  } else {
    griddep_launch_dependents();
  }
}

}  // namespace
}  // namespace pa

extern "C" pa_status pa_copy(void *dst, const void *src, int64_t num_bytes, uint32_t flags,
                             void *stream) {
  using namespace pa;
  if (flags & ~static_cast<uint32_t>(PA_LAUNCH_PDL | PA_COPY_BEFORE_WAIT))
    return PA_ERR_INVALID_ARG;
  if ((flags & PA_COPY_BEFORE_WAIT) && !(flags & PA_LAUNCH_PDL)) return PA_ERR_INVALID_ARG;
  if (num_bytes < 0) return PA_ERR_INVALID_ARG;
  if (num_bytes == 0) return PA_OK;
  if (!dst || !src) return PA_ERR_INVALID_ARG;
  // 16-byte chunks need both addresses 16-byte aligned; otherwise every byte
  // goes through the tail path, which takes at most one block's threads
  const bool vec = ((reinterpret_cast<uintptr_t>(dst) | reinterpret_cast<uintptr_t>(src)) & 15) == 0;
  const long long n16 = vec ? num_bytes / 16 : 0;
  const long long tail = num_bytes - n16 * 16;
  if (tail > kCopyThreads) return PA_ERR_UNSUPPORTED;
  int device = -1, sms = 0;
  if (cudaGetDevice(&device) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess)
    return PA_ERR_DEVICE;
  long long blocks = (n16 + kCopyThreads - 1) / kCopyThreads;
  if (blocks > 2LL * sms) blocks = 2LL * sms;
  if (blocks < 1) blocks = 1;
  const cudaError_t e =
      launch_kernel(copy_kernel, dim3((unsigned)blocks), dim3(kCopyThreads), 0,
                    static_cast<cudaStream_t>(stream), (flags & PA_LAUNCH_PDL) != 0,
                    static_cast<uint8_t *>(dst), static_cast<const uint8_t *>(src), n16,
                    (int)tail, (flags & PA_COPY_BEFORE_WAIT) ? 1 : 0);
  return e == cudaSuccess ? PA_OK : PA_ERR_LAUNCH;
}
