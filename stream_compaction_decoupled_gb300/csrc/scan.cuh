// scan.cuh -- dispatch of a scan along the middle axis of a row-major (B, R, C)
// array.  C == 1 (contiguous rows): one row, or a few long rows, that fit in L2 go
// to the segment kernel (fp64: its thread-contiguous variant, one row), one row many
// times larger than L2 to the L2-resident look-back kernel, everything else to the
// row kernel.  C > 1 (lanes / columns): one aligned chain of 4, 8 or 16 four-byte
// lanes that fits in L2 goes to the lane segment kernel, 8-byte lanes in a few long
// chains that fit in L2 to reduce-then-scan, everything else to the lane look-back
// kernel.
#pragma once

#include "scan_lanes.cuh"
#include "scan_lanes_rts.cuh"
#include "scan_lanes_seg.cuh"
#include "scan_strips.cuh"
#include "scan_rows.cuh"
#include "scan_seg.cuh"
#include "scan_stash.cuh"

namespace gbs {

template <class T> size_t scan_temp_bytes(long long B, long long R, long long C) {
  if (C == 1) {
    // Either kernel may run (the choice depends on the pointers' alignment).
    const size_t rows = kHeaderBytes + rows_status_bytes<T>(rows_tiles<T>(B, R));
    const size_t stash = B == 1 ? kHeaderBytes + stash_status_bytes<T>(R) : 0;
    const size_t seg = kHeaderBytes + seg_status_bytes<T>();
    const size_t m = rows > stash ? rows : stash;
    return m > seg ? m : seg;
  }
  const size_t sp = strips_temp_bytes<T>(C);  // the strip kernel may run (it depends on the pointers)
  if (lanes_rts_applies<T>(B, R, C)) {
    const size_t rt = lanes_rts_temp_bytes<T>(B, R, C);
    return rt > sp ? rt : sp;
  }
  size_t lt = lanes_temp_bytes<T>(B, R, C);
  if (sp > lt) lt = sp;
  if constexpr (sizeof(T) == 4) {
    if (B == 1 && (C == 4 || C == 8 || C == 16)) {  // the lane segment kernel may run
      const size_t st = lanes_seg_temp_bytes<T>();
      return lt > st ? lt : st;
    }
  }
  return lt;
}

template <class T> cudaError_t launch_scan(const ScanJob& job, const LaunchCtx& ctx) {
  if (job.carry_in || job.carry_out) {  // pieces of a longer row: the segment kernels, inclusive
    const bool ok = std::is_same<T, double>::value ? seg_chunk_applies<T>(job, ctx.num_sms) : seg_applies<T>(job);
    if (!ok || job.B != 1 || job.C != 1 || !job.inclusive) return cudaErrorInvalidValue;
  }
  if constexpr (std::is_same<T, double>::value) {
    if (seg_chunk_applies<T>(job, ctx.num_sms)) {
      switch (job.op) {
        case OP_ADD: return launch_seg_chunk<T, OP_ADD>(job, ctx);
        case OP_MAX: return launch_seg_chunk<T, OP_MAX>(job, ctx);
        case OP_MUL: return launch_seg_chunk<T, OP_MUL>(job, ctx);
        default: return launch_seg_chunk<T, OP_MIN>(job, ctx);
      }
    }
  }
  if constexpr (!std::is_same<T, double>::value) {  // fp64 takes the chunked variant above
    if (seg_applies<T>(job)) {
      switch (job.op) {
        case OP_ADD: return launch_seg_op<T, OP_ADD>(job, ctx);
        case OP_MAX: return launch_seg_op<T, OP_MAX>(job, ctx);
        case OP_MUL: return launch_seg_op<T, OP_MUL>(job, ctx);
        default: return launch_seg_op<T, OP_MIN>(job, ctx);
      }
    }
  }
  if (job.C == 1 && stash_applies<T>(job, ctx.num_sms)) {
    switch (job.op) {
      case OP_ADD: return launch_stash_op<T, OP_ADD>(job, ctx);
      case OP_MAX: return launch_stash_op<T, OP_MAX>(job, ctx);
      case OP_MUL: return launch_stash_op<T, OP_MUL>(job, ctx);
      default: return launch_stash_op<T, OP_MIN>(job, ctx);
    }
  }
  if (job.C == 1) {
    switch (job.op) {
      case OP_ADD: return launch_rows_op<T, OP_ADD>(job, ctx);
      case OP_MAX: return launch_rows_op<T, OP_MAX>(job, ctx);
      case OP_MUL: return launch_rows_op<T, OP_MUL>(job, ctx);
      default: return launch_rows_op<T, OP_MIN>(job, ctx);
    }
  }
  if (strips_applies<T>(job, ctx.num_sms)) {
    switch (job.op) {
      case OP_ADD: return launch_strips_op<T, OP_ADD>(job, ctx);
      case OP_MAX: return launch_strips_op<T, OP_MAX>(job, ctx);
      case OP_MUL: return launch_strips_op<T, OP_MUL>(job, ctx);
      default: return launch_strips_op<T, OP_MIN>(job, ctx);
    }
  }
  if constexpr (sizeof(T) == 4) {
    if (lanes_seg_applies<T>(job)) {
      switch (job.op) {
        case OP_ADD: return launch_lanes_seg_op<T, OP_ADD>(job, ctx);
        case OP_MAX: return launch_lanes_seg_op<T, OP_MAX>(job, ctx);
        case OP_MUL: return launch_lanes_seg_op<T, OP_MUL>(job, ctx);
        default: return launch_lanes_seg_op<T, OP_MIN>(job, ctx);
      }
    }
  }
  if constexpr (sizeof(T) == 8) {
    if (lanes_rts_applies<T>(job.B, job.R, job.C)) {
      switch (job.op) {
        case OP_ADD: return launch_lanes_rts_op<T, OP_ADD>(job, ctx);
        case OP_MAX: return launch_lanes_rts_op<T, OP_MAX>(job, ctx);
        case OP_MUL: return launch_lanes_rts_op<T, OP_MUL>(job, ctx);
        default: return launch_lanes_rts_op<T, OP_MIN>(job, ctx);
      }
    }
  }
  switch (job.op) {
    case OP_ADD: return launch_lanes_op<T, OP_ADD>(job, ctx);
    case OP_MAX: return launch_lanes_op<T, OP_MAX>(job, ctx);
    case OP_MUL: return launch_lanes_op<T, OP_MUL>(job, ctx);
    default: return launch_lanes_op<T, OP_MIN>(job, ctx);
  }
}

}  // namespace gbs

// Explicit instantiation of every launcher for one element type.
#define GBS_INSTANTIATE(T)                                                                   \
  namespace gbs {                                                                            \
  template size_t scan_temp_bytes<T>(long long, long long, long long);                      \
  template cudaError_t launch_scan<T>(const ScanJob&, const LaunchCtx&);                    \
  template size_t compact_temp_bytes<T>(long long);                                         \
  template cudaError_t launch_compact<T>(const CompactJob&, const LaunchCtx&);              \
  template size_t partition_temp_bytes<T>();                                                \
  template cudaError_t launch_partition<T>(const PartitionJob&, const LaunchCtx&);          \
  template size_t segmented_temp_bytes<T>();                                                \
  template cudaError_t launch_segmented<T>(const SegmentedJob&, const LaunchCtx&);          \
  template size_t rts_temp_bytes<T>(long long, int);                                        \
  template cudaError_t launch_rts<T>(const RtsJob&, const LaunchCtx&);                      \
  }
