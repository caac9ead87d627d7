// decode_kernel instantiations for FP8 (E4M3) pools, 1 kv head(s) per sequence.
#define PA_HKV 1
#define PA_F8 true
#include "pa_decode_inst.cuh"
