// inst_u32.cu -- every kernel launcher for uint32_t elements (one translation unit per
// element type, so the library builds in parallel).
#include "compact.cuh"
#include "partition.cuh"
#include "segmented.cuh"
#include "rts.cuh"
#include "scan.cuh"

GBS_INSTANTIATE(uint32_t)
