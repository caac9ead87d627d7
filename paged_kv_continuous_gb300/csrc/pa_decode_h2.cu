// decode_kernel instantiations for 2 kv head(s) per sequence.
#define PA_HKV 2
#include "pa_decode_inst.cuh"
