// inst_f32.cu -- every kernel launcher for float elements (one translation unit per
// element type, so the library builds in parallel).
#include "compact.cuh"
#include "partition.cuh"
#include "segmented.cuh"
#include "rts.cuh"
#include "scan.cuh"

GBS_INSTANTIATE(float)
