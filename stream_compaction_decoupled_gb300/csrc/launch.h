// launch.h -- host-side interface between the C ABI (api.cu) and the kernel
// launchers (one translation unit per element type, compiled in parallel).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace gbs {

// Settings the C ABI attaches to every launch.
struct LaunchCtx {
  cudaStream_t stream = nullptr;
  unsigned* err = nullptr;             // sticky device error word of this device
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
};

// Each returns a cudaError_t (cudaSuccess on success).  Defined in scan_rows.cuh /
// scan_lanes.cuh / compact.cuh / rts.cuh, instantiated in inst_<type>.cu.
template <class T> size_t scan_temp_bytes(long long B, long long R, long long C);
template <class T> cudaError_t launch_scan(const ScanJob& job, const LaunchCtx& ctx);
template <class T> size_t compact_temp_bytes(long long n);
template <class T> cudaError_t launch_compact(const CompactJob& job, const LaunchCtx& ctx);
template <class T> size_t rts_temp_bytes(long long n, int num_sms);
template <class T> cudaError_t launch_rts(const RtsJob& job, const LaunchCtx& ctx);
size_t pack_temp_bytes(long long n);
cudaError_t launch_pack(const PackJob& job, const LaunchCtx& ctx);

// Records ctx.ev_before / ctx.ev_after around the main launch when both are set.
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
