// decode_kernel instantiations for 1 kv head(s) per sequence.
#define PA_HKV 1
#include "pa_decode_inst.cuh"
