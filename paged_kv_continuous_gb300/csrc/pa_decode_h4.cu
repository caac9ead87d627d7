// decode_kernel instantiations for 4 kv head(s) per sequence.
#define PA_HKV 4
#include "pa_decode_inst.cuh"
