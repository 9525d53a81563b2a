// launch.h -- host-side interface between the C ABI (api.cu) and the kernel
// launchers (one translation unit per element type, compiled in parallel).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <utility>

namespace gbs {

// Where kernels report a device-side error (a wait that ran out, a packing total
// over capacity, a negative count): the device's sticky word, read and cleared by
// gb_device_error, and the call's own word in its scratch header (nullable), read
// by gb_last_device_error.  The call's word is cleared with the rest of the header
// by the call's status clear, so it holds what this call found and nothing older.
struct ErrSink {
  unsigned* dev = nullptr;
  unsigned* call = nullptr;
};

// Byte offset of the call's error word in the scratch header (kHeaderBytes below);
// the tile-claim counter is at offset 0.
constexpr size_t kCallErrOffset = 128;

#ifdef __CUDACC__
__device__ __forceinline__ void raise_err(const ErrSink& e, unsigned bits) {
  atomicOr(e.dev, bits);
  if (e.call) atomicOr(e.call, bits);
}
#endif

// Settings the C ABI attaches to every launch.
struct LaunchCtx {
  cudaStream_t stream = nullptr;
  ErrSink err;                         // device-wide and per-call error words
  unsigned long long wait_ns = 0;      // limit of every in-kernel wait
  long long stalled_tile = -1;         // fault injection: tile that never publishes
  cudaEvent_t ev_before = nullptr;     // optional events around the main kernel
  cudaEvent_t ev_after = nullptr;
  int num_sms = 0;
};

// Scan along the middle axis of a row-major (B, R, C) array.
struct ScanJob {
  int op = 0;
  int inclusive = 1;
  const void* in = nullptr;
  void* out = nullptr;
  long long B = 0, R = 0, C = 0;
  const void* init_host = nullptr;  // exclusive: init_lanes values (host); lane c uses c % init_lanes
  int init_lanes = 1;
  void* temp = nullptr;             // >= scan_temp_bytes<T>(B, R, C), 256-byte aligned
  // One row, inclusive, segment kernels only: a device value combined on the left of
  // every output (the total of earlier pieces of a longer array), and where the row's
  // last output (its inclusive total, carry_in included) is copied.  Either may be null.
  const void* carry_in = nullptr;
  void* carry_out = nullptr;
};

struct CompactJob {
  const void* in = nullptr;
  long long n = 0;
  int pred = 0;
  const void* threshold_host = nullptr;
  int32_t* out_idx = nullptr;
  int32_t* out_count = nullptr;
  void* temp = nullptr;
};

struct PartitionJob {
  const void* in = nullptr;
  long long n = 0;
  int pred = 0;  // gb_pred, or 6 (bit clear, integers)
  const void* threshold_host = nullptr;
  void* out = nullptr;
  int32_t* out_idx = nullptr;
  int32_t* out_count = nullptr;
  void* temp = nullptr;
};

struct SegmentedJob {
  int op = 0;
  int inclusive = 1;
  const void* in = nullptr;
  const void* flags = nullptr;  // n bytes, nonzero = head
  void* out = nullptr;
  long long n = 0;
  const void* init_host = nullptr;  // exclusive: the value each segment starts from
  void* temp = nullptr;
};

struct PackJob {
  const int32_t* counts = nullptr;
  long long n = 0;
  int32_t* offsets = nullptr;
  int32_t* records = nullptr;
  long long capacity = 0;
  int32_t* out_total = nullptr;
  void* temp = nullptr;
};

struct RtsJob {
  int op = 0;
  int inclusive = 1;
  const void* in = nullptr;
  void* out = nullptr;
  long long n = 0;
  const void* init_host = nullptr;
  void* temp = nullptr;
  int scan_then_fan = 0;  // 0: reduce-then-scan, 1: scan-then-fan
};

// Each returns a cudaError_t (cudaSuccess on success).  Defined in scan_rows.cuh /
// scan_lanes.cuh / compact.cuh / rts.cuh, instantiated in inst_<type>.cu.
template <class T> size_t scan_temp_bytes(long long B, long long R, long long C);
template <class T> cudaError_t launch_scan(const ScanJob& job, const LaunchCtx& ctx);
template <class T> size_t compact_temp_bytes(long long n);
template <class T> cudaError_t launch_compact(const CompactJob& job, const LaunchCtx& ctx);
template <class T> size_t partition_temp_bytes();
template <class T> cudaError_t launch_partition(const PartitionJob& job, const LaunchCtx& ctx);
template <class T> size_t segmented_temp_bytes();
template <class T> cudaError_t launch_segmented(const SegmentedJob& job, const LaunchCtx& ctx);
template <class T> size_t rts_temp_bytes(long long n, int num_sms);
template <class T> cudaError_t launch_rts(const RtsJob& job, const LaunchCtx& ctx);
size_t pack_temp_bytes(long long n);
cudaError_t launch_pack(const PackJob& job, const LaunchCtx& ctx);
// Composition of affine maps (scan_affine.cuh): T is uint32_t or uint64_t, the job
// one row (B = 1) of R maps stored as C = 2 values each.  Instantiated in
// inst_u32.cu / inst_u64.cu.
template <class T> size_t affine_temp_bytes(long long n);
template <class T> cudaError_t launch_affine(const ScanJob& job, const LaunchCtx& ctx);

// Launches `kernel` with programmatic stream serialization, so that it may be
// scheduled while the previous grid in the stream still runs; the kernel must begin
// with pdl_entry() (common.cuh), which holds it until that grid has completed.
template <class... P, class... A>
cudaError_t launch_pdl(void (*kernel)(P...), unsigned grid, unsigned block, size_t smem, cudaStream_t stream,
                       A&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<A>(args)...);
}

// Zeroes [p0, p0 + b0) and, if p1 is set, [p1, p1 + b1) with one small kernel
// launched like the others (it waits for the previous grid, so a call never clears
// scratch that the call before it still reads).  Both bases 16-byte aligned; the
// sizes are rounded up to 16 bytes, which the 256-byte-rounded scratch regions hold.
// Defined in api.cu.
cudaError_t clear_status(void* p0, size_t b0, void* p1, size_t b1, const LaunchCtx& ctx);

// Records ctx.ev_before / ctx.ev_after around a call's launches (the status clear
// and the main kernel) when both are set.  Nothing is recorded between the two
// launches: an event there would stop the second from overlapping the first.
inline void profile_before(const LaunchCtx& ctx) {
  if (ctx.ev_before && ctx.ev_after) cudaEventRecord(ctx.ev_before, ctx.stream);
}
inline void profile_after(const LaunchCtx& ctx) {
  if (ctx.ev_before && ctx.ev_after) cudaEventRecord(ctx.ev_after, ctx.stream);
}

inline size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Temp-storage header: the tile-claim counter lives at offset 0.
constexpr size_t kHeaderBytes = 256;

}  // namespace gbs
