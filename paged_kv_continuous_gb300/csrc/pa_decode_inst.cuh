// Instantiates decode_kernel<G, PA_HKV, PA_F8, PA_ROPE, PA_SPLIT> for G = 1..8
// and the launcher the host ABI dispatches to.  Included once per kv-head
// count and variant by pa_decode_h{1,2,4,8}.cu (bf16 pools),
// pa_decode_f8_h{1,2,4,8}.cu (FP8 pools), pa_decode_rope_h{1,2,4,8}.cu (bf16
// pools, rotary embedding in the fused store), and pa_decode_sm_h{4,8}.cu /
// pa_decode_f8_sm_h{4,8}.cu (merges left to merge_kernel) so that the
// instantiations compile in parallel.
#include "pa_decode_kernel.cuh"

#ifndef PA_HKV
#error "define PA_HKV before including pa_decode_inst.cuh"
#endif
#ifndef PA_F8
#define PA_F8 false
#endif
#ifndef PA_ROPE
#define PA_ROPE false
#endif
#ifndef PA_SPLIT
#define PA_SPLIT false
#endif

namespace pa {

namespace {
template <int G>
cudaError_t launch_g(const CUtensorMap &tk, const CUtensorMap &tv, const DecodeParams &p,
                     cudaStream_t s, int device, bool pdl) {
  using Sh = DecodeShape<G, PA_HKV, PA_F8, PA_ROPE>;
  static std::atomic<bool> configured[64] = {};
  const cudaError_t e = set_smem_once(
      configured, decode_kernel<G, PA_HKV, PA_F8, PA_ROPE, PA_SPLIT>, device, Sh::SMEM);
  if (e != cudaSuccess) return e;
  return launch_kernel(decode_kernel<G, PA_HKV, PA_F8, PA_ROPE, PA_SPLIT>, dim3(p.num_splits),
                       dim3(kDecodeThreads), Sh::SMEM, s, pdl, tk, tv, p);
}
}  // namespace

template <>
cudaError_t launch_decode<PA_HKV, PA_F8, PA_ROPE, PA_SPLIT>(int G, const CUtensorMap &tk, const CUtensorMap &tv,
                                  const DecodeParams &p, cudaStream_t s, int device,
                                  bool pdl) {
  switch (G) {
    case 1: return launch_g<1>(tk, tv, p, s, device, pdl);
    case 2: return launch_g<2>(tk, tv, p, s, device, pdl);
    case 3: return launch_g<3>(tk, tv, p, s, device, pdl);
    case 4: return launch_g<4>(tk, tv, p, s, device, pdl);
    case 5: return launch_g<5>(tk, tv, p, s, device, pdl);
    case 6: return launch_g<6>(tk, tv, p, s, device, pdl);
    case 7: return launch_g<7>(tk, tv, p, s, device, pdl);
    case 8: return launch_g<8>(tk, tv, p, s, device, pdl);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace pa
