// Instantiates decode_kernel<G, PA_HKV> for G = 1..8 and the launcher the
// host ABI dispatches to.  Included once per kv-head count by
// pa_decode_h{1,2,4,8}.cu so that the instantiations compile in parallel.
#include "pa_decode_kernel.cuh"

#ifndef PA_HKV
#error "define PA_HKV before including pa_decode_inst.cuh"
#endif

namespace pa {

namespace {
template <int G>
cudaError_t launch_g(const CUtensorMap &tk, const CUtensorMap &tv, const DecodeParams &p,
                     cudaStream_t s, int device) {
  using Sh = DecodeShape<G, PA_HKV>;
  static bool configured[64] = {};
  if (device < 0 || device >= 64 || !configured[device]) {
    const cudaError_t e = cudaFuncSetAttribute(
        decode_kernel<G, PA_HKV>, cudaFuncAttributeMaxDynamicSharedMemorySize, Sh::SMEM);
    if (e != cudaSuccess) return e;
    if (device >= 0 && device < 64) configured[device] = true;
  }
  decode_kernel<G, PA_HKV><<<p.num_splits, kDecodeThreads, Sh::SMEM, s>>>(tk, tv, p);
  return cudaGetLastError();
}
}  // namespace

template <>
cudaError_t launch_decode<PA_HKV>(int G, const CUtensorMap &tk, const CUtensorMap &tv,
                                  const DecodeParams &p, cudaStream_t s, int device) {
  switch (G) {
    case 1: return launch_g<1>(tk, tv, p, s, device);
    case 2: return launch_g<2>(tk, tv, p, s, device);
    case 3: return launch_g<3>(tk, tv, p, s, device);
    case 4: return launch_g<4>(tk, tv, p, s, device);
    case 5: return launch_g<5>(tk, tv, p, s, device);
    case 6: return launch_g<6>(tk, tv, p, s, device);
    case 7: return launch_g<7>(tk, tv, p, s, device);
    case 8: return launch_g<8>(tk, tv, p, s, device);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace pa
