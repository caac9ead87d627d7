// decode_kernel instantiations for 8 kv head(s) per sequence.
#define PA_HKV 8
#include "pa_decode_inst.cuh"
