// decode_kernel instantiations for 4 kv heads per sequence, bf16 pools,
// merges of cut sequences left to merge_kernel.
#define PA_HKV 4
#define PA_SPLIT true
#include "pa_decode_inst.cuh"
