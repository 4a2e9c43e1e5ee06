// tcgen05 decode kernel, mxfp4 KV.
#define PA_TC_PART_FP4
#include "pa_tc_launch.cuh"
