// inst_f64.cu -- every kernel launcher for double elements (one translation unit per
// element type, so the library builds in parallel).
#include "compact.cuh"
#include "partition.cuh"
#include "segmented.cuh"
#include "rts.cuh"
#include "scan.cuh"

GBS_INSTANTIATE(double)
