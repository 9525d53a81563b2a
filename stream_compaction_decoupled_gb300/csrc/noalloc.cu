// noalloc.cu -- an inclusive scan for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc or cudaMallocAsync at all: code that runs
// under an allocator it does not own (a host framework that forbids allocation in
// its hot path, or one that hands out only the buffers it manages), or code that
// must not change the process's memory footprint after start-up.  For them this
// file keeps the scan's scratch (the tile-claim counter and the tile-status words)
// in one static device array, allocated with the library's module, so the call
// itself allocates nothing.
//
// The array is a fixed size, kNoAllocScratchBytes, held by every GPU that loads the
// library until the process exits.  All calls share it and it keeps the previous
// call's contents; the scan clears the parts that must start at zero (counter and
// status words) on every call, on the caller's stream.  Two calls that can overlap
// on the GPU (on different streams without ordering between them, or on different
// host threads) race on the array and give wrong results.
#include <mutex>

#include "gbscan.h"

namespace {

// 1 MiB: 256 header bytes plus the status words of 131,040 tiles of 4-byte values
// (n up to 536,739,840 elements) or of 52,416 tiles of 8-byte values (n up to
// 107,347,968 elements).
constexpr size_t kNoAllocScratchBytes = 1u << 20;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the static array on the current device.  In host code the
// array's name is only a host-side stand-in, so the address is looked up once per
// device (with that device current) and reused.
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return GB_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return GB_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_setup_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p) return GB_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return GB_OK;
}

}  // namespace

extern "C" int gb_scan_inclusive_noalloc(int dtype, int op, const void* in, void* out, int64_t n,
                                         void* stream) {
  // The same argument checks as gb_scan_inclusive, in the same order: a bad type or
  // operator is refused even when there is nothing to scan.
  if (n < 0 || gb_temp_storage_bytes(GB_KIND_SCAN, dtype, 1, 1, 0) == 0) return GB_ERR_INVALID;
  if (op != GB_ADD && op != GB_MAX && op != GB_MIN && op != GB_MUL) return GB_ERR_INVALID;
  if (n == 0) return GB_OK;
  const size_t need = gb_temp_storage_bytes(GB_KIND_SCAN, dtype, 1, n, 0);
  if (need == 0) return GB_ERR_INVALID;
  if (need > kNoAllocScratchBytes) return GB_ERR_RANGE;
  void* scratch = nullptr;
  const int rc = scratch_address(&scratch);
  if (rc != GB_OK) return rc;
  // The ordinary entry point with caller-supplied scratch: it never allocates.
  return gb_scan_inclusive(dtype, 1, op, in, out, n, scratch, kNoAllocScratchBytes, stream);
}
