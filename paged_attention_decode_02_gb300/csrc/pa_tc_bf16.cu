// tcgen05 decode kernel, bf16 KV.
#define PA_TC_PART_BF16
#include "pa_tc_launch.cuh"
