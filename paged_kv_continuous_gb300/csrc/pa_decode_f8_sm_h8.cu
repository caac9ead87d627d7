// decode_kernel instantiations for 8 kv heads per sequence, FP8 pools,
// merges of cut sequences left to merge_kernel.
#define PA_HKV 8
#define PA_F8 true
#define PA_SPLIT true
#include "pa_decode_inst.cuh"
