// inst_i64.cu -- every kernel launcher for int64_t elements (one translation unit per
// element type, so the library builds in parallel).
#include "compact.cuh"
#include "partition.cuh"
#include "segmented.cuh"
#include "rts.cuh"
#include "scan.cuh"

GBS_INSTANTIATE(int64_t)
