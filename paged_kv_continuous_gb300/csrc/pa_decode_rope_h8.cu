// decode_kernel instantiations for bf16 pools with rotary embedding in the
// fused store, 8 kv head(s) per sequence.
#define PA_HKV 8
#define PA_ROPE true
#include "pa_decode_inst.cuh"
