/*
 * gbscan.h -- device-wide prefix sums and stream compaction for the NVIDIA GB300
 * (sm_103a), as a plain C ABI.
 *
 * The operations are those of three pages on the subject:
 *   [HB]  The CUDA Handbook, ch. 13 "Scan", section 13.3 "CUDA implementations"
 *         (13.3.1 warp and block scans; 13.3.3 reduce-then-scan, Listings 13-10..
 *         13-12, Figure 13-10; 13.3.4 single-pass decoupled look-back, Figure
 *         13-11, Listings 13-13..13-15; 13.3.5 items per thread, Listing 13-16).
 *   [PS]  B. Merry, "Prefix sums on GPUs", GPGPU2 2014: slides "Exclusive Prefix
 *         Sum", "Inclusive Prefix Sum", "Output Format", "Solution", "Other
 *         Applications", "Fixed Block Count", "Prefix-Summing a Block".
 *   [AK]  AcceleratedKernels.jl PR #208, "Fit the scans' tiles in local memory for
 *         large element types": tiles sized per element type; ScanPrefixes,
 *         SliceScan along `dims`, findall.
 *
 * Conventions shared by every call:
 *   - All data pointers (in, out, out_idx, counts, offsets, records, out_count,
 *     out_total, temp) are DEVICE pointers owned by the caller.  `init` and
 *     `threshold` are HOST pointers to one element, read during the call.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *     stream).  Every call is asynchronous on that stream; nothing synchronises
 *     unless stated.  A call enqueues a small status-clearing kernel and its main
 *     kernel(s), each launched with programmatic stream serialization (programmatic
 *     dependent launch): each may be scheduled while the grid before it in the
 *     stream still runs, and each waits (griddepcontrol.wait) for that grid to
 *     complete before touching memory, so stream order is kept.  The library's
 *     kernels let the next launch in the stream be scheduled early; a caller's
 *     kernel launched after a call with the same attribute must itself execute
 *     griddepcontrol.wait (cudaGridDependencySynchronize) before reading the
 *     call's outputs, as that attribute requires of any kernel.
 *   - An "element" is `lanes` consecutive values of `dtype` (lanes = 1 for plain
 *     arrays; 24 fp32 lanes for a 96-byte struct; 17 fp64 lanes for a dual number
 *     with 16 partials).  Operators act lane-wise.
 *   - `temp` may be NULL: the library then draws scratch from the stream-ordered
 *     allocator (cudaMallocAsync / cudaFreeAsync on `stream`), as [HB] 13.3.4's
 *     host function does (Listing 13-15).  Otherwise it must point to at least
 *     gb_temp_storage_bytes(...) bytes, 256-byte aligned, not used concurrently
 *     by another call.  The library resets the parts it needs on every call.
 *   - In-place scans (in == out) are allowed.  out_idx / out_records must not
 *     overlap the inputs.
 *   - n = 0 (or rows*cols = 0) is a no-op that returns GB_OK; compaction and
 *     packing still write a count of 0.
 *   - Return value: GB_OK or one of the GB_ERR_* codes below.  Argument errors
 *     are reported before anything is enqueued.  Errors found on the device
 *     (a look-back that waited too long, a packing capacity exceeded, a negative
 *     count) are recorded twice: in a word in the call's own scratch, read with
 *     gb_last_device_error(temp, stream), and in a word per device that every
 *     call shares, read (and cleared) with gb_device_error(stream).
 */
#ifndef GBSCAN_H
#define GBSCAN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Element types. */
enum gb_dtype { GB_I32 = 0, GB_U32 = 1, GB_I64 = 2, GB_U64 = 3, GB_F32 = 4, GB_F64 = 5 };

/* Associative operators ([PS] "Exclusive Prefix Sum": an operator (+) with an
 * identity I; "Other Applications": max for visibility; [AK]: the accumulate API's
 * cumsum and cumprod).  ADD and MUL wrap modulo 2^32 / 2^64 for integers (the low
 * bits of the exact sum or product, two's complement).  MAX / MIN on floats follow
 * fmax / fmin (a NaN operand is ignored).  MAX and MIN are treated as operators
 * WITHOUT a neutral element ([AK]): inclusive scans need none, exclusive scans need
 * `init`.  ADD's neutral element is 0, MUL's 1.  Float ADD and MUL round in the
 * element type; results are compared against exact (fp64) prefixes within the
 * rounding bounds of any bracketing: sums within 1e-5 of the prefix sum of |x|,
 * products within a relative (i + 1) u / (1 - (i + 1) u) at position i (u the
 * unit roundoff of the type). */
enum gb_op { GB_ADD = 0, GB_MAX = 1, GB_MIN = 2, GB_MUL = 3, GB_AFFINE = 4 };

/* GB_AFFINE: composition of affine maps, an operator that is associative but NOT
 * commutative ([HB] 13.3.4 notes that its packed single-pass descriptor assumes a
 * commutative operator; this library combines in index order throughout).  An
 * element is the map y -> a*y + b over an integer type, stored as lanes = 2 values
 * (a, b); the earlier map is applied first:
 *     (a1, b1) (+) (a2, b2) = (a1*a2, a2*b1 + b2),    neutral element (1, 0).
 * The b of inclusive output i is y_i of the recurrence y_i = a_i*y_{i-1} + b_i
 * from y_{-1} = 0.  Arithmetic wraps modulo 2^32 / 2^64 (signed and unsigned types
 * give the same bits).  Served by gb_scan_inclusive / gb_scan_exclusive with
 * lanes = 2 and an integer dtype (else GB_ERR_UNSUPPORTED), `in` and `out` aligned
 * to the element type; exclusive init is a host pointer to one map (a, b), NULL
 * meaning (1, 0).  gb_temp_storage_bytes(GB_KIND_SCAN, dtype, 2, n, 0) covers it.
 * The other entry points return GB_ERR_UNSUPPORTED for it. */

/* Compaction and partition predicates: element x is selected when  x <op> threshold,
 * compared in the element type (a NaN fails every comparison but NE).  GB_BIT_CLEAR
 * (partition, integer types): x is selected when bit `threshold` (0 .. bits - 1) of
 * x is 0 -- the one-bit split of a radix sort. */
enum gb_pred { GB_LT = 0, GB_LE = 1, GB_GT = 2, GB_GE = 3, GB_EQ = 4, GB_NE = 5, GB_BIT_CLEAR = 6 };

/* Kinds for gb_temp_storage_bytes. */
enum gb_kind {
  GB_KIND_SCAN = 0,          /* gb_scan_inclusive / gb_scan_exclusive: rows = n      */
  GB_KIND_BATCHED_AXIS1 = 1, /* gb_scan_batched axis 1: rows x cols                   */
  GB_KIND_BATCHED_AXIS0 = 2, /* gb_scan_batched axis 0: rows x cols                   */
  GB_KIND_COMPACT = 3,       /* gb_compact: rows = n                                  */
  GB_KIND_PACK = 4,          /* gb_pack_by_counts: rows = n                           */
  GB_KIND_REDUCE_THEN_SCAN = 5, /* gb_scan_reduce_then_scan: rows = n                 */
  GB_KIND_PARTITION = 6,       /* gb_partition: rows = n                              */
  GB_KIND_SEGMENTED = 7        /* gb_scan_segmented: rows = n                         */
};

/* Status codes. */
enum gb_status {
  GB_OK = 0,
  GB_ERR_INVALID = 1,     /* null pointer, negative size, lanes < 1, bad axis/enum   */
  GB_ERR_UNSUPPORTED = 2, /* dtype / op / lanes combination not provided              */
  GB_ERR_TEMP = 3,        /* temp_bytes smaller than gb_temp_storage_bytes           */
  GB_ERR_NO_IDENTITY = 4, /* exclusive MAX / MIN without init                         */
  GB_ERR_RANGE = 5,       /* too large for int32 indices, or packing over capacity   */
  GB_ERR_CUDA = 6,        /* a CUDA runtime call failed: see gb_last_cuda_error()     */
  GB_ERR_TIMEOUT = 7      /* (device) a look-back or copy wait hit its time limit     */
};

/*
 * Inclusive scan  s_i = a_0 (+) ... (+) a_i  of n elements ([PS] "Inclusive Prefix
 * Sum"), computed in one pass by decoupled look-back ([HB] 13.3.4-13.3.5).
 *   dtype, lanes, op  element type, lanes per element (1..4096), operator
 *   in, out           n*lanes values each, contiguous, row-major (element-major)
 *   temp, temp_bytes  scratch (see conventions); kind GB_KIND_SCAN
 * Errors: GB_ERR_INVALID, GB_ERR_UNSUPPORTED, GB_ERR_TEMP, GB_ERR_CUDA.
 */
int gb_scan_inclusive(int dtype, int lanes, int op, const void* in, void* out, int64_t n,
                      void* temp, size_t temp_bytes, void* stream);

/*
 * Exclusive scan  e_i = init (+) a_0 (+) ... (+) a_{i-1}  ([PS] "Exclusive Prefix
 * Sum"; the caller's init takes the place of the identity I and is folded in on
 * the left of every output).  `init` is a host pointer to one element (lanes
 * values) or NULL: NULL means 0 for GB_ADD and 1 for GB_MUL, and is refused for
 * MAX / MIN with GB_ERR_NO_IDENTITY.  The exclusive value is the prefix of the predecessors (a
 * shift), not inclusive minus x ([HB] 13.3.1 derives it by subtraction, which
 * holds for add only).
 */
int gb_scan_exclusive(int dtype, int lanes, int op, const void* in, void* out, int64_t n,
                      const void* init, void* temp, size_t temp_bytes, void* stream);

/*
 * Batched scans of a row-major (rows, cols) matrix of elements ([AK] SliceScan
 * along `dims`).
 *   axis = 1  scan along each row (contiguous; every row is independent)
 *   axis = 0  scan down each column (stride cols*lanes)
 *   inclusive 1 for inclusive, 0 for exclusive (init as in gb_scan_exclusive,
 *             applied to every row / column)
 * temp kind: GB_KIND_BATCHED_AXIS1 or GB_KIND_BATCHED_AXIS0.
 */
int gb_scan_batched(int dtype, int lanes, int op, int inclusive, const void* in, void* out,
                    int64_t rows, int64_t cols, int axis, const void* init,
                    void* temp, size_t temp_bytes, void* stream);

/*
 * Stream compaction ([PS] "Other Applications": compaction; "Solution": count,
 * scan, emit): writes to out_idx, in ascending order, the int32 index of every
 * element x_i (lanes = 1) with  x_i <pred> *threshold, the comparison made in
 * `dtype`, and the number selected to *out_count (device).  One pass: per-tile
 * counts, decoupled look-back over the counts, staged scatter.  Stable ([PS]
 * "Atomics": order must be preserved).  out_idx must hold up to n entries.
 * Errors: GB_ERR_RANGE if n > INT32_MAX.  temp kind: GB_KIND_COMPACT.
 */
int gb_compact(int dtype, const void* in, int64_t n, int pred, const void* threshold,
               int32_t* out_idx, int32_t* out_count, void* temp, size_t temp_bytes,
               void* stream);

/*
 * Stable partition ([PS] "Other Applications": partitioning, and the split that a
 * radix sort repeats; "Solution": count, scan, emit, here with two destinations):
 * the elements x_i (lanes = 1) with  x_i <pred> *threshold  go first, in input
 * order, then all the others, in input order.
 *   out        n elements of `dtype` (device): out[0 .. m) selected, out[m .. n) the rest
 *   out_idx    n int32 (device) or NULL: the input index of each element of out
 *   out_count  one int32 (device): m
 * pred is a gb_pred; GB_BIT_CLEAR (integer dtypes only) selects the elements whose
 * bit *threshold is 0.  `in` must hold naturally aligned elements and must not
 * overlap out or out_idx.  One launch with every CTA resident at once (cooperative):
 * count, gather all segments' counts, rescan and write both windows.
 * Errors: GB_ERR_RANGE if n > INT32_MAX; GB_ERR_UNSUPPORTED for GB_BIT_CLEAR on
 * floats; GB_ERR_INVALID for a bit index outside the type.  temp kind:
 * GB_KIND_PARTITION.
 */
int gb_partition(int dtype, const void* in, int64_t n, int pred, const void* threshold, void* out,
                 int32_t* out_idx, int32_t* out_count, void* temp, size_t temp_bytes, void* stream);

/*
 * Segmented scan by head flags (lanes = 1): flags[i] != 0 marks element i as the
 * first of a segment (element 0 always is one), and every segment is scanned on its
 * own: inclusive  out_i = x_h (+) ... (+) x_i,  exclusive  out_i = init (+) x_h (+)
 * ... (+) x_{i-1}  (out_h = init), h the last head at or before i.  The segmented
 * operator on (value, flag) pairs is associative but not commutative ([HB] 13.3.4's
 * caveat on the packed descriptor), and the kernel combines in index order
 * throughout.  flags: n bytes (device).  init as in gb_scan_exclusive (NULL: 0 for
 * ADD, 1 for MUL; required for MAX / MIN).  in == out is allowed.  temp kind:
 * GB_KIND_SEGMENTED.
 */
int gb_scan_segmented(int dtype, int op, int inclusive, const void* in, const uint8_t* flags, void* out,
                      int64_t n, const void* init, void* temp, size_t temp_bytes, void* stream);

/*
 * Variable-length packing ([PS] "Output Format" and "Solution"): object i emits
 * counts[i] records holding the value i; its run starts at the exclusive prefix
 * sum of the counts, and the runs are packed contiguously into out_records.
 *   offsets       NULL, or n int32 entries that receive the start of each run
 *   out_capacity  entries available in out_records; records past it are dropped
 *   out_total     device int32: the total record count (sum of counts)
 * Device errors (gb_last_device_error, gb_device_error): GB_ERR_RANGE when the total exceeds
 * out_capacity or INT32_MAX; GB_ERR_INVALID when a count is negative (it is then
 * treated as 0).  temp kind: GB_KIND_PACK.
 */
int gb_pack_by_counts(const int32_t* counts, int64_t n, int32_t* offsets,
                      int32_t* out_records, int64_t out_capacity, int32_t* out_total,
                      void* temp, size_t temp_bytes, void* stream);

/*
 * The reduce-then-scan comparison variant ([HB] 13.3.3, Listings 13-10..13-12;
 * [PS] "Fixed Block Count"): a fixed number C of blocks (a multiple of the SM
 * count) each reduce a contiguous subarray, one block scans the C partials, then
 * each block scans its subarray starting from its base.  Three launches, 3n
 * element transfers instead of 2n.  lanes = 1.  Same results and errors as the
 * single-pass scans; temp kind GB_KIND_REDUCE_THEN_SCAN.
 */
int gb_scan_reduce_then_scan(int dtype, int op, int inclusive, const void* in, void* out,
                             int64_t n, const void* init, void* temp, size_t temp_bytes,
                             void* stream);

/*
 * The scan-then-fan comparison variant ([HB] 13.3.2): the same C blocks each scan
 * their contiguous subarray into `out` and record its total, one block scans the C
 * totals, then every block after the first combines its base into its outputs (the
 * fan).  Three launches, 4n element transfers.  lanes = 1.  Same results and errors
 * as the single-pass scans; temp kind GB_KIND_REDUCE_THEN_SCAN (the same scratch).
 * `in` and `out` may be the same array.
 */
int gb_scan_then_fan(int dtype, int op, int inclusive, const void* in, void* out, int64_t n,
                     const void* init, void* temp, size_t temp_bytes, void* stream);

/*
 * Inclusive scan of a HOST array into a host array (lanes = 1): the library copies
 * the input to the device, scans it and copies the result back, chunk by chunk, so
 * that the copy of one chunk in and of another out overlap the scan of a third
 * (separate copy streams, a ring of three device buffers, events between them).
 * Each chunk is scanned by the segment kernel starting from the running total of
 * the chunks before it, which stays in device memory: the result is that of one
 * inclusive scan of the whole array ([HB] 13.3.3's reduce-then-scan of a long
 * array, piece by piece).  The pages have no counterpart: their host functions take
 * device arrays.
 *   dtype, op         as gb_scan_inclusive
 *   in_host, out_host HOST pointers to n elements each, owned by the caller; pinned
 *                     (cudaMallocHost / cudaHostRegister) for the copies to overlap,
 *                     pageable memory works but copies synchronously; out_host may
 *                     equal in_host; neither is touched after the work on `stream`
 *                     completes
 *   n                 element count (0: no-op)
 *   chunk_elems       elements per chunk, 0 for the default (48 MiB of elements);
 *                     capped at 48 MiB and rounded up to 16 bytes
 *   work, work_bytes  device scratch of at least gb_host_scan_work_bytes(dtype, n,
 *                     chunk_elems) bytes (256-byte aligned), or NULL: the library
 *                     then allocates it on `stream` (cudaMallocAsync) and frees it
 *                     there
 *   stream            the caller's stream: the scans run on it, and it waits for the
 *                     last chunk to be back in host memory, so synchronising it (or
 *                     an event recorded on it after the call) means out_host is ready
 * The copy streams and events are the library's, one set per device; calls on one
 * device from several host threads are enqueued one after the other.  Floating-
 * point results may differ from gb_scan_inclusive's in the last bits (the sum is
 * combined in another order).  Errors: as gb_scan_inclusive; a failed CUDA call
 * mid-way returns GB_ERR_CUDA with the chunks before it enqueued.
 */
int gb_scan_inclusive_host(int dtype, int op, const void* in_host, void* out_host, int64_t n,
                           int64_t chunk_elems, void* work, size_t work_bytes, void* stream);

/* Device scratch bytes for gb_scan_inclusive_host (0 for an invalid dtype or n <= 0). */
size_t gb_host_scan_work_bytes(int dtype, int64_t n, int64_t chunk_elems);

/*
 * Inclusive scan that allocates nothing, for callers that cannot call cudaMalloc or
 * cudaMallocAsync (code running under an allocator it does not own, or that must not
 * grow the process's device memory after start-up).  The pages have no counterpart:
 * their host functions draw scratch from the stream-ordered allocator.
 *   dtype, op       as gb_scan_inclusive; one lane per element (lanes = 1)
 *   in, out, n      device pointers and element count, as gb_scan_inclusive
 *   stream          cudaStream_t as void*
 * The scratch (tile counter and tile-status words) is one static device array of
 * 1 MiB (1048576 bytes) inside the library, held by every GPU that loads the library
 * until the process exits.  Sizes whose scratch does not fit
 * (gb_temp_storage_bytes(GB_KIND_SCAN, dtype, 1, n, 0) > 1048576: n above
 * 536,739,840 for 4-byte types, above 107,347,968 for 8-byte types) are rejected
 * with GB_ERR_RANGE before anything is enqueued.  The first call on a device looks up
 * the array's device address (cudaGetSymbolAddress) with that device current; make
 * that first call before any stream capture.  Every call shares the array and clears
 * what must start at zero on `stream`; calls that can overlap on the GPU (different
 * streams without ordering, or concurrent host threads) race on it.
 * Errors: as gb_scan_inclusive, plus GB_ERR_RANGE for the size limit.
 */
int gb_scan_inclusive_noalloc(int dtype, int op, const void* in, void* out, int64_t n, void* stream);

/*
 * Scratch bytes a call needs for the given kind and sizes (rows = n for the 1-D
 * kinds; cols ignored there).  Returns 0 for an invalid combination.
 */
size_t gb_temp_storage_bytes(int kind, int dtype, int lanes, int64_t rows, int64_t cols);

/*
 * Synchronise `stream`, then return and clear the sticky device-side error of the
 * current device: GB_OK, GB_ERR_TIMEOUT, GB_ERR_RANGE or GB_ERR_INVALID (the most
 * serious kind seen by any call on the device since the last read), or GB_ERR_CUDA
 * if the sync failed.  Calls on independent streams all report here.
 */
int gb_device_error(void* stream);

/*
 * The device-side status of the last call that ran kernels with this scratch
 * ([HB] 13.3.4, Listing 13-15: the scan's scratch is the call's own; the error
 * word sits in its header and the call clears it together with the tile-status
 * words, so nothing from an earlier call shows): synchronises `stream` (the stream
 * that call ran on), then returns GB_OK, GB_ERR_TIMEOUT, GB_ERR_RANGE or
 * GB_ERR_INVALID, or GB_ERR_CUDA if the sync failed.  Unlike gb_device_error it
 * sees only that call, so calls on other streams with their own scratch do not
 * mix in, and it clears nothing.
 *   temp    the `temp` the call was given (256-byte aligned), or the `work` of
 *           gb_scan_inclusive_host (whose word gathers every chunk of the call).
 *           A call given temp = NULL uses library scratch that is gone when it
 *           returns: read such calls with gb_device_error.  A call that ran no
 *           kernel (n = 0, an argument error) leaves the word as it was.
 * Errors: GB_ERR_INVALID for a NULL or unaligned temp.
 */
int gb_last_device_error(void* temp, void* stream);

/* Human-readable name of a status code (static storage). */
const char* gb_status_string(int status);

/* The cudaError_t value behind the last GB_ERR_CUDA returned on this thread. */
int gb_last_cuda_error(void);

/* Library version, as major*10000 + minor*100 + patch. */
int gb_version(void);

/*
 * Observability hook: when both are non-NULL cudaEvent_t handles, the next calls
 * on this host thread record `before` and `after` on their stream around their
 * launches (the status clear and the single-pass kernel, or the three
 * reduce-then-scan launches), so a caller can time a call's device work without
 * host overhead.  Nothing is recorded between the launches of a call: an event
 * there would stop them from overlapping.  Pass NULL, NULL to turn it off.
 */
void gb_set_profile_events(void* before, void* after);

/*
 * Time limit, in nanoseconds of the GPU's global timer, of every wait inside the
 * kernels (a look-back waiting on a predecessor, a tile waiting for its copy).  A
 * wait that runs out records GB_ERR_TIMEOUT (see gb_last_device_error), publishes what
 * it has so that later tiles do not wait as well, and the kernel returns normally.
 * 0 restores the default of one second.  Process-wide.
 */
void gb_set_wait_limit_ns(uint64_t ns);

/*
 * Fault injection for tests: the tile with this index (in claim order) of the
 * next single-pass launches never publishes its status, so its successors' waits
 * run out.  -1 (the default) turns it off.  Process-wide.
 */
void gb_set_stalled_tile(int64_t tile);

#ifdef __cplusplus
}
#endif

#endif /* GBSCAN_H */
