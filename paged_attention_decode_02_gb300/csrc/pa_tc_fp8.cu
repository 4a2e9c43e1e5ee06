// tcgen05 decode kernel, fp8 KV.
#define PA_TC_PART_FP8
#include "pa_tc_launch.cuh"
