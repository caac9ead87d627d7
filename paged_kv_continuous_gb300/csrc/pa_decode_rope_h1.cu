// decode_kernel instantiations for bf16 pools with rotary embedding in the
// fused store, 1 kv head(s) per sequence.
#define PA_HKV 1
#define PA_ROPE true
#include "pa_decode_inst.cuh"
