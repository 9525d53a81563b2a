// api.cu -- the C ABI declared in include/gbscan.h: argument checks, scratch
// (temp) handling, element-type dispatch and the sticky device error word.
// Every check that can fail does so before anything is enqueued.
#include <atomic>
#include <cstring>
#include <mutex>
#include <type_traits>
#include <vector>

#include "common.cuh"
#include "gbscan.h"
#include "launch.h"

// Sticky device-side error bits (look-back / copy timeouts, packing overflow,
// negative counts), one word per device, set with atomicOr by the kernels.
__device__ unsigned g_gbscan_device_error;

namespace gbs {

// The status clear (see clear_status in launch.h): 16-byte stores over both ranges.
__global__ void __launch_bounds__(256) clear_status_kernel(uint4* p0, size_t n0, uint4* p1, size_t n1) {
  pdl_entry();
  const size_t n = n0 + n1;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
    if (i < n0) p0[i] = make_uint4(0u, 0u, 0u, 0u);
    else p1[i - n0] = make_uint4(0u, 0u, 0u, 0u);
  }
}

cudaError_t clear_status(void* p0, size_t b0, void* p1, size_t b1, const LaunchCtx& ctx) {
  const size_t n0 = (b0 + 15) / 16, n1 = p1 ? (b1 + 15) / 16 : 0;
  size_t grid = (n0 + n1 + 1023) / 1024;  // about four stores a thread
  const size_t max_grid = 2 * (size_t)(ctx.num_sms > 0 ? ctx.num_sms : 1);
  if (grid > max_grid) grid = max_grid;
  if (grid < 1) grid = 1;
  return launch_pdl(clear_status_kernel, (unsigned)grid, 256, 0, ctx.stream, (uint4*)p0, n0, (uint4*)p1, n1);
}

}  // namespace gbs

namespace {

using gbs::LaunchCtx;

constexpr int kMaxDevices = 64;
constexpr int kMaxLanes = 4096;
constexpr unsigned long long kDefaultWaitNs = 1000000000ull;  // 1 s

std::mutex g_mu;
unsigned* g_err_ptr[kMaxDevices] = {};
int g_num_sms[kMaxDevices] = {};
std::atomic<unsigned long long> g_wait_ns{0};
std::atomic<long long> g_stalled_tile{-1};
thread_local int t_last_cuda = 0;
thread_local cudaEvent_t t_ev_before = nullptr;
thread_local cudaEvent_t t_ev_after = nullptr;

int cuda_fail(cudaError_t e) {
  t_last_cuda = (int)e;
  return GB_ERR_CUDA;
}

// The status code of a set of device error bits (the most serious first).
int status_of_bits(unsigned bits) {
  if (bits & gbs::ERRBIT_TIMEOUT) return GB_ERR_TIMEOUT;
  if (bits & gbs::ERRBIT_RANGE) return GB_ERR_RANGE;
  if (bits & gbs::ERRBIT_INVALID) return GB_ERR_INVALID;
  return GB_OK;
}

// Per-device set-up (once): the address of the error word and the SM count.
int make_ctx(void* stream, LaunchCtx& ctx) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dev < 0 || dev >= kMaxDevices) return GB_ERR_UNSUPPORTED;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_err_ptr[dev]) {
      void* p = nullptr;
      e = cudaGetSymbolAddress(&p, g_gbscan_device_error);
      if (e != cudaSuccess) return cuda_fail(e);
      int sms = 0;
      e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
      if (e != cudaSuccess) return cuda_fail(e);
      g_num_sms[dev] = sms;
      g_err_ptr[dev] = (unsigned*)p;
    }
    ctx.err.dev = g_err_ptr[dev];
    ctx.err.call = nullptr;
    ctx.num_sms = g_num_sms[dev];
  }
  ctx.stream = (cudaStream_t)stream;
  const unsigned long long w = g_wait_ns.load();
  ctx.wait_ns = w ? w : kDefaultWaitNs;
  ctx.stalled_tile = g_stalled_tile.load();
  ctx.ev_before = t_ev_before;
  ctx.ev_after = t_ev_after;
  return GB_OK;
}

// Caller-supplied scratch, or stream-ordered scratch freed when the call ends.
struct Temp {
  void* p = nullptr;
  bool owned = false;
  cudaStream_t s = nullptr;
  ~Temp() {
    if (owned && p) cudaFreeAsync(p, s);
  }
};

// The call's own error word lives in its scratch header (cleared by the call's
// status clear), so gb_last_device_error(temp, ...) reports what this call found.
void attach_call_err(LaunchCtx& ctx, void* temp) {
  ctx.err.call = (unsigned*)((char*)temp + gbs::kCallErrOffset);
}

int get_temp(void* temp, size_t temp_bytes, size_t need, cudaStream_t s, Temp& t) {
  t.s = s;
  if (temp) {
    if (temp_bytes < need) return GB_ERR_TEMP;
    if ((uintptr_t)temp % 256) return GB_ERR_INVALID;
    t.p = temp;
    return GB_OK;
  }
  cudaError_t e = cudaMallocAsync(&t.p, need, s);
  if (e != cudaSuccess) {
    t.p = nullptr;
    return cuda_fail(e);
  }
  t.owned = true;
  return GB_OK;
}

size_t dtype_size(int dtype) {
  switch (dtype) {
    case GB_I32: case GB_U32: case GB_F32: return 4;
    case GB_I64: case GB_U64: case GB_F64: return 8;
    default: return 0;
  }
}

bool valid_op(int op) { return op == GB_ADD || op == GB_MAX || op == GB_MIN || op == GB_MUL; }
bool is_int(int dtype) { return dtype == GB_I32 || dtype == GB_U32 || dtype == GB_I64 || dtype == GB_U64; }

// Scratch for a 1-D scan of affine maps (8- or 16-byte pairs of an integer type).
size_t affine_temp(int dtype, long long n) {
  return dtype_size(dtype) == 4 ? gbs::affine_temp_bytes<uint32_t>(n) : gbs::affine_temp_bytes<uint64_t>(n);
}

// The scan of affine maps: one row of n maps, each `lanes` = 2 integers (a, b); the
// signed types run as the unsigned ones of their width (the same bits).
int run_affine(int dtype, int inclusive, const void* in, void* out, long long n, const void* init, int lanes,
               void* temp, size_t temp_bytes, void* stream) {
  if (!dtype_size(dtype) || lanes < 1 || n < 0) return GB_ERR_INVALID;
  if (!is_int(dtype) || lanes != 2) return GB_ERR_UNSUPPORTED;
  if (n == 0) return GB_OK;
  if (!in || !out) return GB_ERR_INVALID;
  if ((uintptr_t)in % dtype_size(dtype) || (uintptr_t)out % dtype_size(dtype)) return GB_ERR_INVALID;
  LaunchCtx ctx;
  int rc = make_ctx(stream, ctx);
  if (rc) return rc;
  Temp t;
  rc = get_temp(temp, temp_bytes, affine_temp(dtype, n), ctx.stream, t);
  if (rc) return rc;
  attach_call_err(ctx, t.p);
  gbs::ScanJob job;
  job.op = GB_AFFINE;
  job.inclusive = inclusive ? 1 : 0;
  job.in = in;
  job.out = out;
  job.B = 1;
  job.R = n;
  job.C = 2;
  job.init_host = inclusive ? nullptr : init;
  job.init_lanes = 2;
  job.temp = t.p;
  const cudaError_t e = dtype_size(dtype) == 4 ? gbs::launch_affine<uint32_t>(job, ctx)
                                               : gbs::launch_affine<uint64_t>(job, ctx);
  return e == cudaSuccess ? GB_OK : cuda_fail(e);
}
bool has_identity(int op) { return op == GB_ADD || op == GB_MUL; }

// Calls f.template operator()<T>() with T the C++ type of `dtype`.
template <class F> auto with_type(int dtype, F&& f) {
  switch (dtype) {
    case GB_I32: return f((int32_t*)nullptr);
    case GB_U32: return f((uint32_t*)nullptr);
    case GB_I64: return f((int64_t*)nullptr);
    case GB_U64: return f((uint64_t*)nullptr);
    case GB_F32: return f((float*)nullptr);
    default: return f((double*)nullptr);
  }
}

// The neutral element of ADD (0) or MUL (1), `lanes` copies in the element type.
std::vector<unsigned char> identity_bytes(int dtype, int op, int lanes) {
  const size_t es = dtype_size(dtype);
  std::vector<unsigned char> v((size_t)lanes * es, 0);
  if (op == GB_MUL) {
    with_type(dtype, [&](auto* tp) {
      using T = std::remove_pointer_t<decltype(tp)>;
      const T one = T(1);
      for (int l = 0; l < lanes; ++l) std::memcpy(v.data() + (size_t)l * es, &one, es);
      return 0;
    });
  }
  return v;
}

// Tiles are claimed with a 32-bit counter and indexed with grid.x.
constexpr size_t kMaxTiles = 0x7fffffffull;

size_t scan_temp(int dtype, long long B, long long R, long long C) {
  return with_type(dtype, [&](auto* tp) -> size_t {
    using T = std::remove_pointer_t<decltype(tp)>;
    return gbs::scan_temp_bytes<T>(B, R, C);
  });
}

bool scan_fits(int dtype, long long B, long long R, long long C) {
  // Conservative bound on the tile count of either kernel (tiles hold >= 64 positions
  // of a lane strip, or >= 2048 positions of a row).
  const size_t es = dtype_size(dtype);
  const long long strips = C <= 1 ? 1 : (C + 31) / 32;
  const long long per = C <= 1 ? (es == 4 ? 4096 : 2048) : 8;
  const long double tiles = (long double)B * strips * ((R + per - 1) / per);
  return tiles < (long double)kMaxTiles;
}

// Shared body of every scan entry point: (B, R, C) layout, init lanes.
int run_scan(int dtype, int op, int inclusive, const void* in, void* out, long long B, long long R,
             long long C, const void* init, int lanes, void* temp, size_t temp_bytes, void* stream) {
  if (!dtype_size(dtype) || !valid_op(op)) return GB_ERR_INVALID;
  if (lanes < 1 || lanes > kMaxLanes || B < 0 || R < 0 || C < 0) return GB_ERR_INVALID;
  if (!inclusive && !init && !has_identity(op)) return GB_ERR_NO_IDENTITY;
  if (B == 0 || R == 0 || C == 0) return GB_OK;
  if (!in || !out) return GB_ERR_INVALID;
  if ((long double)B * R * C > 9.0e18L) return GB_ERR_RANGE;
  if (!scan_fits(dtype, B, R, C)) return GB_ERR_RANGE;
  LaunchCtx ctx;
  int rc = make_ctx(stream, ctx);
  if (rc) return rc;
  Temp t;
  rc = get_temp(temp, temp_bytes, scan_temp(dtype, B, R, C), ctx.stream, t);
  if (rc) return rc;
  attach_call_err(ctx, t.p);
  std::vector<unsigned char> neutral;
  if (!inclusive && !init) {  // add / multiply without init: start from 0 / 1
    neutral = identity_bytes(dtype, op, lanes);
    init = neutral.data();
  }
  gbs::ScanJob job;
  job.op = op;
  job.inclusive = inclusive ? 1 : 0;
  job.in = in;
  job.out = out;
  job.B = B;
  job.R = R;
  job.C = C;
  job.init_host = init;
  job.init_lanes = lanes;
  job.temp = t.p;
  const cudaError_t e = with_type(dtype, [&](auto* tp) {
    using T = std::remove_pointer_t<decltype(tp)>;
    return gbs::launch_scan<T>(job, ctx);
  });
  if (e != cudaSuccess) return cuda_fail(e);
  return GB_OK;
}

// ---- scans between host buffers: chunks whose copies overlap the scans --------------

// Device copies of a host array move in chunks through a ring of kRing device buffers:
// chunk i is copied in on one stream, scanned in place on the caller's stream (its
// first element combined with the running total of chunks 0..i-1, which the previous
// chunk's scan left in device memory), and copied out on another stream, so the copy
// of chunk i+1 in and of chunk i-1 out run while chunk i is scanned.  Events order
// each buffer's reuse.  The streams and events are made once per device.
constexpr int kRing = 3;
constexpr size_t kHostChunkBytes = 48ull << 20;  // a segment-kernel size (at most 96 MiB)

struct HostPipe {
  cudaStream_t h2d = nullptr, d2h = nullptr;
  cudaEvent_t start = nullptr;
  cudaEvent_t in_done[kRing] = {}, scan_done[kRing] = {}, out_done[kRing] = {};
  std::mutex mu;  // one call enqueues its chunks at a time on a device
};
HostPipe* g_pipe[kMaxDevices] = {};

int get_pipe(HostPipe*& out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_pipe[dev]) {
    HostPipe* p = new HostPipe();
    const unsigned fl = cudaEventDisableTiming;
    e = cudaStreamCreateWithFlags(&p->h2d, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&p->d2h, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p->start, fl);
    for (int k = 0; k < kRing && e == cudaSuccess; ++k) {
      e = cudaEventCreateWithFlags(&p->in_done[k], fl);
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p->scan_done[k], fl);
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p->out_done[k], fl);
    }
    if (e != cudaSuccess) return cuda_fail(e);  // the partly made pipe is leaked, not reused
    g_pipe[dev] = p;
  }
  out = g_pipe[dev];
  return GB_OK;
}

long long host_chunk_elems(int dtype, long long n, long long req) {
  const long long es = (long long)dtype_size(dtype);
  long long c = req > 0 ? req : (long long)(kHostChunkBytes / es);
  if (c * es > (long long)kHostChunkBytes) c = (long long)(kHostChunkBytes / es);
  c = (c + 15) / 16 * 16;  // whole 16-byte vectors (ring slots stay aligned)
  return c < n ? c : n;
}

// Work area: [header: the call's error word][scan scratch][two carries][ring].  The
// chunk scans clear only their own scratch, so the header's error word collects what
// every chunk of the call found.
struct HostLayout {
  size_t header = 0, scan_temp = 0, carry = 0, slot = 0, total = 0;
};
HostLayout host_layout(int dtype, long long chunk) {
  HostLayout L;
  L.header = gbs::kHeaderBytes;
  L.scan_temp = gbs::round_up(scan_temp(dtype, 1, chunk, 1), 256);
  L.carry = 256;  // two carries
  L.slot = gbs::round_up((size_t)chunk * dtype_size(dtype), 256);
  L.total = L.header + L.scan_temp + L.carry + kRing * L.slot;
  return L;
}

// The reduce-then-scan (stf = 0) and scan-then-fan (stf = 1) comparators.
int run_comparator(int stf, int dtype, int op, int inclusive, const void* in, void* out, int64_t n,
                   const void* init, void* temp, size_t temp_bytes, void* stream) {
  if (op == GB_AFFINE) return GB_ERR_UNSUPPORTED;
  if (!dtype_size(dtype) || !valid_op(op) || n < 0) return GB_ERR_INVALID;
  if (!inclusive && !init && !has_identity(op)) return GB_ERR_NO_IDENTITY;
  if (n == 0) return GB_OK;
  if (!in || !out) return GB_ERR_INVALID;
  LaunchCtx ctx;
  int rc = make_ctx(stream, ctx);
  if (rc) return rc;
  const size_t need = with_type(dtype, [&](auto* tp) {
    using T = std::remove_pointer_t<decltype(tp)>;
    return gbs::rts_temp_bytes<T>(n, ctx.num_sms);
  });
  Temp t;
  rc = get_temp(temp, temp_bytes, need, ctx.stream, t);
  if (rc) return rc;
  attach_call_err(ctx, t.p);
  const std::vector<unsigned char> neutral = identity_bytes(dtype, op, 1);
  gbs::RtsJob job;
  job.op = op;
  job.inclusive = inclusive ? 1 : 0;
  job.in = in;
  job.out = out;
  job.n = n;
  job.init_host = init ? init : neutral.data();
  job.temp = t.p;
  job.scan_then_fan = stf;
  const cudaError_t e = with_type(dtype, [&](auto* tp) {
    using T = std::remove_pointer_t<decltype(tp)>;
    return gbs::launch_rts<T>(job, ctx);
  });
  return e == cudaSuccess ? GB_OK : cuda_fail(e);
}

}  // namespace

extern "C" {

size_t gb_host_scan_work_bytes(int dtype, int64_t n, int64_t chunk_elems) {
  if (!dtype_size(dtype) || n <= 0) return 0;
  return host_layout(dtype, host_chunk_elems(dtype, n, chunk_elems)).total;
}

int gb_scan_inclusive_host(int dtype, int op, const void* in_host, void* out_host, int64_t n, int64_t chunk_elems,
                           void* work, size_t work_bytes, void* stream) {
  if (op == GB_AFFINE) return GB_ERR_UNSUPPORTED;
  if (!dtype_size(dtype) || !valid_op(op) || n < 0 || chunk_elems < 0) return GB_ERR_INVALID;
  if (n == 0) return GB_OK;
  if (!in_host || !out_host) return GB_ERR_INVALID;
  LaunchCtx ctx;
  int rc = make_ctx(stream, ctx);
  if (rc) return rc;
  ctx.ev_before = ctx.ev_after = nullptr;  // the profile hook times single-kernel calls only
  HostPipe* pipe = nullptr;
  rc = get_pipe(pipe);
  if (rc) return rc;
  const long long chunk = host_chunk_elems(dtype, n, chunk_elems);
  const HostLayout L = host_layout(dtype, chunk);
  Temp t;
  rc = get_temp(work, work_bytes, L.total, ctx.stream, t);
  if (rc) return rc;
  char* base = (char*)t.p;
  attach_call_err(ctx, base);
  void* scan_tmp = base + L.header;
  char* carry = base + L.header + L.scan_temp;
  char* ring = carry + L.carry;
  const size_t es = dtype_size(dtype);
  const long long nchunks = (n + chunk - 1) / chunk;

  std::lock_guard<std::mutex> lk(pipe->mu);
  cudaError_t e = cudaMemsetAsync(ctx.err.call, 0, sizeof(unsigned), ctx.stream);
  if (e == cudaSuccess) e = cudaEventRecord(pipe->start, ctx.stream);  // after the caller's earlier work
  if (e == cudaSuccess) e = cudaStreamWaitEvent(pipe->h2d, pipe->start, 0);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(pipe->d2h, pipe->start, 0);
  for (long long i = 0; i < nchunks && e == cudaSuccess; ++i) {
    const int k = (int)(i % kRing);
    const long long off = i * chunk, len = n - off < chunk ? n - off : chunk;
    const size_t bytes = (size_t)len * es;
    char* buf = ring + (size_t)k * L.slot;
    if (i >= kRing) e = cudaStreamWaitEvent(pipe->h2d, pipe->out_done[k], 0);  // slot copied out
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(buf, (const char*)in_host + (size_t)off * es, bytes, cudaMemcpyHostToDevice, pipe->h2d);
    if (e == cudaSuccess) e = cudaEventRecord(pipe->in_done[k], pipe->h2d);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(ctx.stream, pipe->in_done[k], 0);
    if (e == cudaSuccess) {
      gbs::ScanJob job;
      job.op = op;
      job.inclusive = 1;
      job.in = buf;
      job.out = buf;
      job.B = 1;
      job.R = len;
      job.C = 1;
      job.temp = scan_tmp;
      job.carry_in = i > 0 ? carry + ((i - 1) % 2) * 16 : nullptr;
      job.carry_out = i + 1 < nchunks ? carry + (i % 2) * 16 : nullptr;
      e = with_type(dtype, [&](auto* tp) {
        using T = std::remove_pointer_t<decltype(tp)>;
        return gbs::launch_scan<T>(job, ctx);
      });
    }
    if (e == cudaSuccess) e = cudaEventRecord(pipe->scan_done[k], ctx.stream);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(pipe->d2h, pipe->scan_done[k], 0);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync((char*)out_host + (size_t)off * es, buf, bytes, cudaMemcpyDeviceToHost, pipe->d2h);
    if (e == cudaSuccess) e = cudaEventRecord(pipe->out_done[k], pipe->d2h);
  }
  // The caller's stream resumes once the last chunk is back in host memory (copies
  // leave each stream in order, so every earlier copy has finished too).
  if (e == cudaSuccess) e = cudaStreamWaitEvent(ctx.stream, pipe->out_done[(nchunks - 1) % kRing], 0);
  return e == cudaSuccess ? GB_OK : cuda_fail(e);
}



int gb_scan_inclusive(int dtype, int lanes, int op, const void* in, void* out, int64_t n, void* temp,
                      size_t temp_bytes, void* stream) {
  if (n < 0) return GB_ERR_INVALID;
  if (op == GB_AFFINE) return run_affine(dtype, 1, in, out, n, nullptr, lanes, temp, temp_bytes, stream);
  return run_scan(dtype, op, 1, in, out, 1, n, lanes, nullptr, lanes, temp, temp_bytes, stream);
}

int gb_scan_exclusive(int dtype, int lanes, int op, const void* in, void* out, int64_t n, const void* init,
                      void* temp, size_t temp_bytes, void* stream) {
  if (n < 0) return GB_ERR_INVALID;
  if (op == GB_AFFINE) return run_affine(dtype, 0, in, out, n, init, lanes, temp, temp_bytes, stream);
  return run_scan(dtype, op, 0, in, out, 1, n, lanes, init, lanes, temp, temp_bytes, stream);
}

int gb_scan_batched(int dtype, int lanes, int op, int inclusive, const void* in, void* out, int64_t rows,
                    int64_t cols, int axis, const void* init, void* temp, size_t temp_bytes, void* stream) {
  if (op == GB_AFFINE) return GB_ERR_UNSUPPORTED;
  if (rows < 0 || cols < 0 || lanes < 1 || lanes > kMaxLanes) return GB_ERR_INVALID;
  if (axis == 1) return run_scan(dtype, op, inclusive, in, out, rows, cols, lanes, init, lanes, temp, temp_bytes, stream);
  if (axis == 0) {
    if (cols != 0 && (long double)cols * lanes > 9.0e18L) return GB_ERR_RANGE;
    return run_scan(dtype, op, inclusive, in, out, 1, rows, (long long)cols * lanes, init, lanes, temp, temp_bytes,
                    stream);
  }
  return GB_ERR_INVALID;
}

int gb_compact(int dtype, const void* in, int64_t n, int pred, const void* threshold, int32_t* out_idx,
               int32_t* out_count, void* temp, size_t temp_bytes, void* stream) {
  if (!dtype_size(dtype) || pred < GB_LT || pred > GB_NE || n < 0) return GB_ERR_INVALID;
  if (!out_count || !threshold) return GB_ERR_INVALID;
  if (n > 0x7fffffffll) return GB_ERR_RANGE;
  if (n > 0 && (!in || !out_idx)) return GB_ERR_INVALID;
  LaunchCtx ctx;
  int rc = make_ctx(stream, ctx);
  if (rc) return rc;
  if (n == 0) {
    cudaError_t e = cudaMemsetAsync(out_count, 0, sizeof(int32_t), ctx.stream);
    return e == cudaSuccess ? GB_OK : cuda_fail(e);
  }
  const size_t need = with_type(dtype, [&](auto* tp) {
    using T = std::remove_pointer_t<decltype(tp)>;
    return gbs::compact_temp_bytes<T>(n);
  });
  Temp t;
  rc = get_temp(temp, temp_bytes, need, ctx.stream, t);
  if (rc) return rc;
  attach_call_err(ctx, t.p);
  gbs::CompactJob job;
  job.in = in;
  job.n = n;
  job.pred = pred;
  job.threshold_host = threshold;
  job.out_idx = out_idx;
  job.out_count = out_count;
  job.temp = t.p;
  const cudaError_t e = with_type(dtype, [&](auto* tp) {
    using T = std::remove_pointer_t<decltype(tp)>;
    return gbs::launch_compact<T>(job, ctx);
  });
  return e == cudaSuccess ? GB_OK : cuda_fail(e);
}

int gb_partition(int dtype, const void* in, int64_t n, int pred, const void* threshold, void* out,
                 int32_t* out_idx, int32_t* out_count, void* temp, size_t temp_bytes, void* stream) {
  if (!dtype_size(dtype) || pred < GB_LT || pred > GB_BIT_CLEAR || n < 0) return GB_ERR_INVALID;
  if (!out_count || !threshold) return GB_ERR_INVALID;
  const bool is_float = dtype == GB_F32 || dtype == GB_F64;
  if (pred == GB_BIT_CLEAR) {
    if (is_float) return GB_ERR_UNSUPPORTED;
    unsigned long long b = 0;
    std::memcpy(&b, threshold, dtype_size(dtype));
    if (dtype == GB_I32 || dtype == GB_U32) b &= 0xffffffffull;
    if (b >= 8 * dtype_size(dtype)) return GB_ERR_INVALID;
  }
  if (n > 0x7fffffffll) return GB_ERR_RANGE;
  if (n > 0 && (!in || !out)) return GB_ERR_INVALID;
  if (n > 0 && (uintptr_t)in % dtype_size(dtype) != 0) return GB_ERR_INVALID;
  LaunchCtx ctx;
  int rc = make_ctx(stream, ctx);
  if (rc) return rc;
  if (n == 0) {
    cudaError_t e = cudaMemsetAsync(out_count, 0, sizeof(int32_t), ctx.stream);
    return e == cudaSuccess ? GB_OK : cuda_fail(e);
  }
  const size_t need = with_type(dtype, [&](auto* tp) {
    using T = std::remove_pointer_t<decltype(tp)>;
    return gbs::partition_temp_bytes<T>();
  });
  Temp t;
  rc = get_temp(temp, temp_bytes, need, ctx.stream, t);
  if (rc) return rc;
  attach_call_err(ctx, t.p);
  gbs::PartitionJob job;
  job.in = in;
  job.n = n;
  job.pred = pred;
  job.threshold_host = threshold;
  job.out = out;
  job.out_idx = out_idx;
  job.out_count = out_count;
  job.temp = t.p;
  const cudaError_t e = with_type(dtype, [&](auto* tp) {
    using T = std::remove_pointer_t<decltype(tp)>;
    return gbs::launch_partition<T>(job, ctx);
  });
  return e == cudaSuccess ? GB_OK : cuda_fail(e);
}

int gb_scan_segmented(int dtype, int op, int inclusive, const void* in, const uint8_t* flags, void* out,
                      int64_t n, const void* init, void* temp, size_t temp_bytes, void* stream) {
  if (op == GB_AFFINE) return GB_ERR_UNSUPPORTED;
  if (!dtype_size(dtype) || !valid_op(op) || n < 0) return GB_ERR_INVALID;
  if (!inclusive && !init && !has_identity(op)) return GB_ERR_NO_IDENTITY;
  if (n == 0) return GB_OK;
  if (!in || !out || !flags) return GB_ERR_INVALID;
  LaunchCtx ctx;
  int rc = make_ctx(stream, ctx);
  if (rc) return rc;
  const size_t need = with_type(dtype, [&](auto* tp) {
    using T = std::remove_pointer_t<decltype(tp)>;
    return gbs::segmented_temp_bytes<T>();
  });
  Temp t;
  rc = get_temp(temp, temp_bytes, need, ctx.stream, t);
  if (rc) return rc;
  attach_call_err(ctx, t.p);
  const std::vector<unsigned char> neutral = identity_bytes(dtype, op, 1);
  gbs::SegmentedJob job;
  job.op = op;
  job.inclusive = inclusive ? 1 : 0;
  job.in = in;
  job.flags = flags;
  job.out = out;
  job.n = n;
  job.init_host = init ? init : neutral.data();
  job.temp = t.p;
  const cudaError_t e = with_type(dtype, [&](auto* tp) {
    using T = std::remove_pointer_t<decltype(tp)>;
    return gbs::launch_segmented<T>(job, ctx);
  });
  return e == cudaSuccess ? GB_OK : cuda_fail(e);
}

int gb_pack_by_counts(const int32_t* counts, int64_t n, int32_t* offsets, int32_t* out_records,
                      int64_t out_capacity, int32_t* out_total, void* temp, size_t temp_bytes, void* stream) {
  if (n < 0 || out_capacity < 0 || !out_total) return GB_ERR_INVALID;
  if (n > 0x7fffffffll) return GB_ERR_RANGE;
  if (n > 0 && !counts) return GB_ERR_INVALID;
  if (out_capacity > 0 && !out_records) return GB_ERR_INVALID;
  LaunchCtx ctx;
  int rc = make_ctx(stream, ctx);
  if (rc) return rc;
  if (n == 0) {
    cudaError_t e = cudaMemsetAsync(out_total, 0, sizeof(int32_t), ctx.stream);
    return e == cudaSuccess ? GB_OK : cuda_fail(e);
  }
  Temp t;
  rc = get_temp(temp, temp_bytes, gbs::pack_temp_bytes(n), ctx.stream, t);
  if (rc) return rc;
  attach_call_err(ctx, t.p);
  gbs::PackJob job;
  job.counts = counts;
  job.n = n;
  job.offsets = offsets;
  job.records = out_records;
  job.capacity = out_capacity;
  job.out_total = out_total;
  job.temp = t.p;
  const cudaError_t e = gbs::launch_pack(job, ctx);
  return e == cudaSuccess ? GB_OK : cuda_fail(e);
}

int gb_scan_then_fan(int dtype, int op, int inclusive, const void* in, void* out, int64_t n,
                     const void* init, void* temp, size_t temp_bytes, void* stream) {
  return run_comparator(1, dtype, op, inclusive, in, out, n, init, temp, temp_bytes, stream);
}

int gb_scan_reduce_then_scan(int dtype, int op, int inclusive, const void* in, void* out, int64_t n,
                             const void* init, void* temp, size_t temp_bytes, void* stream) {
  return run_comparator(0, dtype, op, inclusive, in, out, n, init, temp, temp_bytes, stream);
}


size_t gb_temp_storage_bytes(int kind, int dtype, int lanes, int64_t rows, int64_t cols) {
  if (!dtype_size(dtype) || lanes < 1 || lanes > kMaxLanes || rows < 0 || cols < 0) return 0;
  switch (kind) {
    case GB_KIND_SCAN: {
      // Two lanes of an integer type may be affine maps (GB_AFFINE): cover that too.
      const size_t s = scan_temp(dtype, 1, rows, lanes);
      if (lanes == 2 && is_int(dtype)) {
        const size_t a = affine_temp(dtype, rows);
        return a > s ? a : s;
      }
      return s;
    }
    case GB_KIND_BATCHED_AXIS1:
      return scan_temp(dtype, rows, cols, lanes);
    case GB_KIND_BATCHED_AXIS0:
      return scan_temp(dtype, 1, rows, (long long)cols * lanes);
    case GB_KIND_COMPACT:
      return with_type(dtype, [&](auto* tp) {
        using T = std::remove_pointer_t<decltype(tp)>;
        return gbs::compact_temp_bytes<T>(rows);
      });
    case GB_KIND_PACK:
      return gbs::pack_temp_bytes(rows);
    case GB_KIND_PARTITION:
      return with_type(dtype, [&](auto* tp) {
        using T = std::remove_pointer_t<decltype(tp)>;
        return gbs::partition_temp_bytes<T>();
      });
    case GB_KIND_SEGMENTED:
      return with_type(dtype, [&](auto* tp) {
        using T = std::remove_pointer_t<decltype(tp)>;
        return gbs::segmented_temp_bytes<T>();
      });
    case GB_KIND_REDUCE_THEN_SCAN:
      return with_type(dtype, [&](auto* tp) {
        using T = std::remove_pointer_t<decltype(tp)>;
        return gbs::rts_temp_bytes<T>(rows, 0);
      });
    default:
      return 0;
  }
}

int gb_device_error(void* stream) {
  LaunchCtx ctx;
  int rc = make_ctx(stream, ctx);
  if (rc) return rc;
  cudaError_t e = cudaStreamSynchronize(ctx.stream);
  if (e != cudaSuccess) return cuda_fail(e);
  unsigned bits = 0;
  e = cudaMemcpy(&bits, ctx.err.dev, sizeof(bits), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e);
  if (bits) {
    e = cudaMemset(ctx.err.dev, 0, sizeof(unsigned));
    if (e != cudaSuccess) return cuda_fail(e);
  }
  return status_of_bits(bits);
}

int gb_last_device_error(void* temp, void* stream) {
  if (!temp || (uintptr_t)temp % 256) return GB_ERR_INVALID;
  LaunchCtx ctx;
  int rc = make_ctx(stream, ctx);
  if (rc) return rc;
  cudaError_t e = cudaStreamSynchronize(ctx.stream);
  if (e != cudaSuccess) return cuda_fail(e);
  unsigned bits = 0;
  e = cudaMemcpy(&bits, (const char*)temp + gbs::kCallErrOffset, sizeof(bits), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e);
  return status_of_bits(bits);
}

const char* gb_status_string(int status) {
  switch (status) {
    case GB_OK: return "GB_OK";
    case GB_ERR_INVALID: return "GB_ERR_INVALID: invalid argument";
    case GB_ERR_UNSUPPORTED: return "GB_ERR_UNSUPPORTED: unsupported type, operator or size";
    case GB_ERR_TEMP: return "GB_ERR_TEMP: temporary storage too small";
    case GB_ERR_NO_IDENTITY: return "GB_ERR_NO_IDENTITY: exclusive max/min needs an initial value";
    case GB_ERR_RANGE: return "GB_ERR_RANGE: size or output capacity out of range";
    case GB_ERR_CUDA: return "GB_ERR_CUDA: a CUDA runtime call failed";
    case GB_ERR_TIMEOUT: return "GB_ERR_TIMEOUT: a device-side wait ran out of time";
    default: return "unknown gbscan status";
  }
}

int gb_last_cuda_error(void) { return t_last_cuda; }

int gb_version(void) { return 1 * 10000 + 0 * 100 + 0; }

void gb_set_profile_events(void* before, void* after) {
  t_ev_before = (cudaEvent_t)before;
  t_ev_after = (cudaEvent_t)after;
}

void gb_set_wait_limit_ns(uint64_t ns) { g_wait_ns.store(ns); }

void gb_set_stalled_tile(int64_t tile) { g_stalled_tile.store(tile); }

}  // extern "C"
