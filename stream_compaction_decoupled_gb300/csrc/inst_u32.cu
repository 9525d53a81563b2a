// inst_u32.cu -- every kernel launcher for uint32_t elements (one translation unit per
// element type, so the library builds in parallel).
#include "compact.cuh"
#include "partition.cuh"
#include "segmented.cuh"
#include "rts.cuh"
#include "scan.cuh"
#include "scan_affine.cuh"

GBS_INSTANTIATE(uint32_t)

// Composition of affine maps: the signed type of the same width shares these.
namespace gbs {
template size_t affine_temp_bytes<uint32_t>(long long);
template cudaError_t launch_affine<uint32_t>(const ScanJob&, const LaunchCtx&);
}
