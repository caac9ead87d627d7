// decode_kernel instantiations for bf16 pools with rotary embedding in the
// fused store, 2 kv head(s) per sequence.
#define PA_HKV 2
#define PA_ROPE true
#include "pa_decode_inst.cuh"
