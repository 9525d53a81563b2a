// scan_seg.cuh -- reduce-then-scan in one launch, for 1-D inputs that fit in L2.
//
// The CUDA Handbook, 13.3.3 (Figure 13-10) splits the input into subarrays, reduces
// each (pass 1), scans the partial sums, and rescans each subarray seeded with its
// base sum (pass 2): 3N global operations over three launches.  Here the three
// steps run in one kernel and the second read of every element is served from L2,
// so HBM sees one read and one write per element, as a single-pass scan does:
//
//   1. each CTA claims a segment (an atomic counter: a CTA only ever waits for
//      segments claimed before its own, so no co-residency is assumed) and its
//      warps reduce their contiguous parts of it, loading with an L2 evict-last
//      hint; the block combines the warp totals and publishes the segment
//      aggregate;
//   2. warp 0 reads the aggregates of ALL earlier segments at once (lane l owns
//      segments l, l+32, ...) and combines them in a fixed order: the segment's
//      base sum.  There is no chain of inclusive prefixes to walk, so every
//      segment has its base one memory round trip after the slowest earlier
//      segment has published, however many segments there are;
//   3. each warp rescans its part chunk by chunk from L2 (evict-first: last use),
//      seeded with base sum (+) earlier warps of the segment (+) earlier chunks,
//      and streams the result out.
//
// Decoupled look-back (The CUDA Handbook, 13.3.4) is the better scheme once the
// input is many times larger than L2 and tiles start at different times; with all
// tiles of a mid-size input starting together, the look-back's inclusive prefixes
// can only advance one window of tiles per memory round trip, which this kernel
// avoids.  The fixed combination order makes floating-point results reproducible
// from run to run.
//
// Stream compaction (B. Merry, "Prefix sums on GPUs", slide "Solution") runs the
// same three phases on selection counts.
#pragma once

#include "launch.h"
#include "tile.cuh"

namespace gbs {

// A warp's unit of work is a chunk of 32 lanes x ROUNDS x one 16-byte vector; in
// round j lane l holds vector j*32 + l of the chunk (the row kernel's run layout).
template <class T, int NT_, int ROUNDS_, int MINB_> struct SegCfg {
  static constexpr int NT = NT_, NW = NT_ / 32, ROUNDS = ROUNDS_, MINB = MINB_;
  static constexpr int VEC = Vec<T>::N;
  static constexpr int CH = 32 * ROUNDS * VEC;  // elements per chunk
  // Segments (CTAs) per launch at most; 8-byte values keep the gather's loads (two
  // words a segment) within the registers of a 1024-thread CTA.
  static constexpr int MAXSEG = sizeof(T) == 8 ? 256 : 512;
  static constexpr int M = MAXSEG / 32;         // earlier aggregates per lane in phase 2
};
// 8-byte elements take 2 rounds a chunk (the chunk and the one prefetched behind it
// then fit the 64 registers a thread of a 1024-thread CTA has).
template <class T> using SegGeom = SegCfg<T, 1024, sizeof(T) == 8 ? 2 : 4, 1>;

// Work split of `rows` independent rows of n elements (a 1-D scan is one row): each
// row's nc chunks are spread over `segs` segments (CTAs; segment p of a row takes
// chunks [p*nc/segs, (p+1)*nc/segs), at least one), then over the segment's NW warps
// (the first k mod NW warps take one chunk more, so warps without chunks come last).
// Spreading over CTAs first keeps every SM busy when there are fewer chunks than
// warps.  Segments never cross a row, so a row's scan only gathers its own segments'
// aggregates.
struct SegPlan {
  unsigned rows = 0;
  long long nc = 0;   // chunks per row
  unsigned segs = 0;  // segments per row
  unsigned ctas = 0;
  long long cpw = 0;  // most chunks any warp takes
};
template <class G> SegPlan seg_plan(long long rows, long long n, int num_sms) {
  SegPlan p;
  if (rows <= 0 || n <= 0) return p;
  p.rows = (unsigned)rows;
  p.nc = (n + G::CH - 1) / G::CH;
  long long segs = (long long)num_sms * G::MINB / rows;
  if (segs < 1) segs = 1;
  if (segs > p.nc) segs = p.nc;
  if (segs * rows > G::MAXSEG) {
    segs = G::MAXSEG / rows;
    if (segs < 1) return SegPlan{};  // too many rows for the status slots
  }
  p.segs = (unsigned)segs;
  p.ctas = (unsigned)(segs * rows);
  const long long cps = (p.nc + segs - 1) / segs;  // most chunks in a segment
  p.cpw = (cps + G::NW - 1) / G::NW;
  return p;
}

struct SegArgsBase {
  long long n;  // elements per row
  long long nc;
  unsigned segs;
  unsigned ctas;
  unsigned* counter;
  ErrSink err;
  unsigned long long wait_ns;
  long long stalled;  // fault injection: this segment never publishes
};

template <class T> struct SegArgs : SegArgsBase {
  const T* in;
  T* out;
  T init;
  int inclusive;
  const T* carry_in;  // nullable: combined on the left of everything (one row only)
  T* carry_out;       // nullable: the row's last inclusive value (inclusive scans, one row)
};

// Phase 2's result for one segment, by lane 0 of warp 0: the base, carry-in on the
// left of the gathered aggregates of the row's earlier segments.  (The row's total
// for carry_out is taken from its last scanned element in phase 3: the aggregates
// of a ragged last chunk hold the padding read past n.)
template <class T, int OP>
__device__ __forceinline__ void seg_finish_base(const SegArgs<T>& a, bool have_gather, T gathered, T& base,
                                                bool& has) {
  has = false;
  if (a.carry_in) {
    base = *a.carry_in;
    has = true;
  }
  if (have_gather) {
    base = has ? Op<T, OP>::f(base, gathered) : gathered;
    has = true;
  }
}

// Chunk loads and stores.  A full chunk moves as 16-byte vectors with an L2 policy;
// the one ragged chunk at the end of the input moves element by element (elements
// past n read as T{}: they only ever reach totals that nothing reads).
template <class T, int ROUNDS>
__device__ __forceinline__ void seg_load(Vec<T> (&x)[ROUNDS], const T* in, long long c0, long long n, int lane,
                                         unsigned long long pol) {
  constexpr int VEC = Vec<T>::N, CH = 32 * ROUNDS * VEC;
  if (c0 + CH <= n) {
    const uint4* p = reinterpret_cast<const uint4*>(in + c0) + lane;
#pragma unroll
    for (int j = 0; j < ROUNDS; ++j) {
      const uint4 u = ld_hint(p + j * 32, pol);
      memcpy(x[j].v, &u, 16);
    }
  } else {
#pragma unroll
    for (int j = 0; j < ROUNDS; ++j)
#pragma unroll
      for (int e = 0; e < VEC; ++e) {
        const long long i = c0 + (long long)(j * 32 + lane) * VEC + e;
        x[j].v[e] = i < n ? in[i] : T{};
      }
  }
}
template <class T, int ROUNDS>
__device__ __forceinline__ void seg_store(const Vec<T> (&x)[ROUNDS], T* out, long long c0, long long n, int lane,
                                          unsigned long long pol) {
  constexpr int VEC = Vec<T>::N, CH = 32 * ROUNDS * VEC;
  if (c0 + CH <= n) {
    uint4* p = reinterpret_cast<uint4*>(out + c0) + lane;
#pragma unroll
    for (int j = 0; j < ROUNDS; ++j) {
      uint4 u;
      memcpy(&u, x[j].v, 16);
      st_hint(p + j * 32, u, pol);
    }
  } else {
#pragma unroll
    for (int j = 0; j < ROUNDS; ++j)
#pragma unroll
      for (int e = 0; e < VEC; ++e) {
        const long long i = c0 + (long long)(j * 32 + lane) * VEC + e;
        if (i < n) out[i] = x[j].v[e];
      }
  }
}

// Butterfly combination over the warp (every lane gets the same result; the order
// is fixed, so floating-point sums are reproducible).
template <class T, int OP> __device__ __forceinline__ T warp_allreduce(T v) {
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const T o = __shfl_xor_sync(0xffffffffu, v, off);
    v = (threadIdx.x & off) ? Op<T, OP>::f(o, v) : Op<T, OP>::f(v, o);
  }
  return v;
}

// Phase 1 of a warp: the combination of the elements of its chunks [c0, c1), read
// as coalesced 16-byte vectors, U per lane in flight (the reduction's order is free:
// only the scan in phase 3 follows element order).  Loads carry the L2 evict-last
// hint so that phase 3 finds the lines in L2.  Every lane of a warp with whole
// chunks has elements; only the last warp (whose total nothing reads) may not.
template <class T, int OP, class G>
__device__ __forceinline__ T seg_reduce_part(const T* in, long long n, long long c0, long long c1, int lane) {
  constexpr int VEC = G::VEC, CH = G::CH, U = 8;
  const unsigned long long keep = l2_policy_evict_last();
  const long long e1 = c1 * CH < n ? c1 * CH : n;
  const long long v1 = e1 / VEC;  // whole vectors end
  const uint4* p = reinterpret_cast<const uint4*>(in);
  long long v = c0 * CH / VEC + lane;
  T acc{};
  if (v < v1) {
    const uint4 u = ld_hint(p + v, keep);
    Vec<T> x;
    memcpy(x.v, &u, 16);
    acc = x.v[0];
#pragma unroll
    for (int e = 1; e < VEC; ++e) acc = Op<T, OP>::f(acc, x.v[e]);
    v += 32;
  }
  for (; v + 32 * (U - 1) < v1; v += 32 * U) {  // U loads in flight
    uint4 u[U];
#pragma unroll
    for (int k = 0; k < U; ++k) u[k] = ld_hint(p + v + 32 * k, keep);
#pragma unroll
    for (int k = 0; k < U; ++k) {
      Vec<T> x;
      memcpy(x.v, &u[k], 16);
#pragma unroll
      for (int e = 0; e < VEC; ++e) acc = Op<T, OP>::f(acc, x.v[e]);
    }
  }
  if (v < v1) {  // the rest in one guarded round, its loads still all in flight
    uint4 u[U];
#pragma unroll
    for (int k = 0; k < U; ++k)
      if (v + 32 * k < v1) u[k] = ld_hint(p + v + 32 * k, keep);
#pragma unroll
    for (int k = 0; k < U; ++k)
      if (v + 32 * k < v1) {
        Vec<T> x;
        memcpy(x.v, &u[k], 16);
#pragma unroll
        for (int e = 0; e < VEC; ++e) acc = Op<T, OP>::f(acc, x.v[e]);
      }
  }
  if (lane == 0)
    for (long long i = v1 * VEC; i < e1; ++i) acc = Op<T, OP>::f(acc, in[i]);
  return acc;
}

// Phase 2, by one whole warp: the combination of the aggregates of segments
// first .. first+cnt-1 (1 <= cnt <= 32 M, the earlier segments of the row), waiting
// (bounded by wait_ns) for each to be published.  Lane l owns the consecutive
// segments first + l P .. first + l P + P - 1, P = ceil(cnt / 32): all are requested
// at once, and only those not yet published are read again.  Every partial result
// then combines consecutive segments in order (as the look-back's ordered combine
// does), which keeps float products from overflowing where the prefix itself does
// not.  Returns the base sum in every lane.
template <class T, int OP, int M, class S>
__device__ __forceinline__ T seg_gather(const S& st, unsigned first, unsigned cnt, unsigned long long wait_ns,
                                        bool& timed_out) {
  const int lane = threadIdx.x & 31;
  const unsigned seg = cnt;
  const unsigned per = (cnt + 31) / 32;      // segments per lane, <= M
  const unsigned mine = (unsigned)lane * per; // this lane's first segment (relative)
  T val[M];
  unsigned pending = 0;
#pragma unroll
  for (int k = 0; k < M; ++k)
    if ((unsigned)k < per && mine + k < seg) pending |= 1u << k;
  unsigned long long t0 = 0;
  timed_out = false;
  for (int spins = 0;; ++spins) {
#pragma unroll
    for (int k = 0; k < M; ++k) {
      if (pending & (1u << k)) {
        T v;
        const unsigned f = st.poll(first + mine + k, v);
        if (f != FLAG_X) {
          val[k] = st.fetch(first + mine + k, f, v);
          pending &= ~(1u << k);
        }
      }
    }
    if (__all_sync(0xffffffffu, pending == 0)) break;
    unsigned long long now = 0;
    if (lane == 0) now = globaltimer();
    now = __shfl_sync(0xffffffffu, now, 0);
    if (spins == 0) t0 = now;
    else if (now - t0 > wait_ns) {
      timed_out = true;
#pragma unroll
      for (int k = 0; k < M; ++k)
        if (pending & (1u << k)) val[k] = T{};
      break;
    }
    backoff(spins);
  }
  // Lane fold in segment order, then the lanes in lane order.  A lane with no
  // segment contributes the neutral element of add (and of the saturating add) or
  // of multiply, or (max / min being idempotent) lane 0's first value.
  T acc = val[0];
#pragma unroll
  for (int k = 1; k < M; ++k)
    if ((unsigned)k < per && mine + k < seg) acc = Op<T, OP>::f(acc, val[k]);
  const T v00 = __shfl_sync(0xffffffffu, val[0], 0);
  if (mine >= seg) acc = (OP == OP_ADD || OP == OP_SATADD) ? T{} : OP == OP_MUL ? T(1) : v00;
  const T inc = warp_inclusive<T, OP>(acc, lane);
  return __shfl_sync(0xffffffffu, inc, 31);
}

// The chunks [c0, c1) of the segment's row for warp `warp` of the CTA, `part` being
// the segment's index within its row; returns how many of the CTA's warps have
// chunks (they are the first ones).
__device__ __forceinline__ int seg_chunks(const SegArgsBase& a, unsigned part, int warp, int nw, long long& c0,
                                          long long& c1) {
  const long long cb = (long long)part * a.nc / a.segs, ce = (long long)(part + 1) * a.nc / a.segs;
  const long long k = ce - cb, q = k / nw, r = k % nw;
  c0 = cb + warp * q + (warp < r ? warp : r);
  c1 = c0 + q + (warp < r ? 1 : 0);
  return k < nw ? (int)k : nw;
}

template <class T, int OP, class G, class S>
__global__ void __launch_bounds__(G::NT, G::MINB) scan_seg_kernel(SegArgs<T> a, S st) {
  pdl_entry();
  constexpr int NW = G::NW, ROUNDS = G::ROUNDS, CH = G::CH;
  __shared__ unsigned s_seg;
  __shared__ T s_warp[NW];
  __shared__ T s_base;
  __shared__ int s_hbase;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) s_seg = atomicAdd(a.counter, 1u);
  __syncthreads();
  const unsigned seg = s_seg;
  const unsigned row = seg / a.segs, part = seg - row * a.segs;
  const T* in = a.in + (long long)row * a.n;
  T* out = a.out + (long long)row * a.n;
  long long c0, c1;
  const int nact = seg_chunks(a, part, warp, NW, c0, c1);

  // Phase 1: the warp's total (lanes accumulate their vectors, then one butterfly).
  const T acc = seg_reduce_part<T, OP, G>(in, a.n, c0, c1, lane);
  const T wtot = warp_allreduce<T, OP>(acc);
  if (lane == 0) s_warp[warp] = wtot;  // warps without chunks come last: their totals are never read
  __syncthreads();

  // Phase 2: publish the segment aggregate, gather the row's earlier ones.
  if (warp == 0) {
    block_scan_warp_totals<T, OP, NW>(s_warp, lane);
    __syncwarp();
    const T agg = s_warp[nact - 1];
    if (lane == 0 && (long long)seg != a.stalled) st.publish(seg, FLAG_A, agg);
    T gathered{};
    if (part > 0) {
      bool timed_out;
      gathered = seg_gather<T, OP, G::M>(st, seg - part, part, a.wait_ns, timed_out);
      if (lane == 0 && timed_out) raise_err(a.err, ERRBIT_TIMEOUT);
    }
    if (lane == 0) {
      T b{};
      bool h;
      seg_finish_base<T, OP>(a, part > 0, gathered, b, h);
      s_base = b;
      s_hbase = h;
    }
  }
  __syncthreads();

  // Phase 3: rescan the warp's chunks from L2, seeded.
  bool hb = s_hbase != 0;
  T base = s_base;
  if (warp > 0) {
    const T wp = s_warp[warp - 1];
    base = hb ? Op<T, OP>::f(base, wp) : wp;
    hb = true;
  }
  if (!a.inclusive) {
    base = hb ? Op<T, OP>::f(a.init, base) : a.init;
    hb = true;
  }
  const unsigned long long drop = l2_policy_evict_first();
  Vec<T> x[ROUNDS];
  if (c0 < c1) seg_load<T, ROUNDS>(x, in, c0 * CH, a.n, lane, drop);
  for (long long c = c0; c < c1; ++c) {
    Vec<T> y[ROUNDS];  // the next chunk, requested before this one is scanned
    if (c + 1 < c1) seg_load<T, ROUNDS>(y, in, (c + 1) * CH, a.n, lane, drop);
    T pre[ROUNDS];
    const T ctot = regs_reduce_pass<T, OP, ROUNDS>(x, lane, pre);
    regs_apply_pass<T, OP, ROUNDS>(x, lane, pre, base, hb, a.inclusive);
    seg_store<T, ROUNDS>(x, out, c * CH, a.n, lane, drop);
    if (a.carry_out && c == a.nc - 1) {  // the row's last element: its inclusive value
      constexpr int VEC = G::VEC;
      const int el = (int)(a.n - 1 - c * CH);
      T last = x[0].v[0];  // register selects: a runtime index would put x[] in local memory
#pragma unroll
      for (int j = 0; j < ROUNDS; ++j)
#pragma unroll
        for (int e = 0; e < VEC; ++e) last = ((j * 32 + lane) * VEC + e == el) ? x[j].v[e] : last;
      if (lane == (el / VEC) % 32) *a.carry_out = last;
    }
    base = hb ? Op<T, OP>::f(base, ctot) : ctot;
    hb = true;
#pragma unroll
    for (int j = 0; j < ROUNDS; ++j) x[j] = y[j];
  }
}

// Status area right after the header: descriptors for up to kSegSlots segments (the
// most any segment-scheme kernel launches), as the flag-carrying layouts of the
// segmented scans (StatusFor) or as the segment kernels' words (SegStatusFor).
constexpr int kSegSlots = 512;
template <class T> size_t seg_status_bytes() {
  if (sizeof(T) == 4) return round_up((size_t)kSegSlots * 8, 256);
  return round_up((size_t)kSegSlots * 4, 256) + 2 * round_up((size_t)kSegSlots * sizeof(T), 256);
}
template <class T> typename StatusFor<T>::type seg_status(void* temp) {
  typename StatusFor<T>::type st;
  char* base = (char*)temp + kHeaderBytes;
  if constexpr (sizeof(T) == 4) {
    st.w = (unsigned long long*)base;
  } else {
    st.flag = (unsigned*)base;
    base += round_up((size_t)kSegSlots * 4, 256);
    st.agg = (T*)base;
    base += round_up((size_t)kSegSlots * sizeof(T), 256);
    st.pfx = (T*)base;
  }
  return st;
}
// Bytes to clear before a launch: the header and the flags.
template <class T> size_t seg_reset_bytes() {
  return kHeaderBytes + (sizeof(T) == 4 ? (size_t)kSegSlots * 8 : (size_t)kSegSlots * 4);
}

// Status of the segment kernels' aggregates (they publish aggregates only).  4-byte
// values: the packed (flag, value) word.  8-byte values: the value's bits and their
// complement in two relaxed stores; a reader loads both, in flight together, and
// takes the value once one word is the complement of the other.  Both words are
// zero before the launch, so every pair a reader accepts holds the value written
// ((v, 0) passes only when v is all ones, (0, ~v) only when v is 0).  Unlike a flag
// released after the value, this needs no acquire: a gather keeps all its loads in
// flight at once.
template <class T> struct WordPairStatus {
  unsigned long long* w;  // [segment][2]
  __device__ __forceinline__ void publish(long long i, unsigned, T v) const {
    const unsigned long long x = to_u64(v);
    st_relaxed_u64(w + 2 * i, x);
    st_relaxed_u64(w + 2 * i + 1, ~x);
  }
  __device__ __forceinline__ unsigned poll(long long i, T& v) const {
    const unsigned long long x0 = ld_relaxed_u64(w + 2 * i), x1 = ld_relaxed_u64(w + 2 * i + 1);
    v = from_u64<T>(x0);
    return x1 == ~x0 ? FLAG_A : FLAG_X;
  }
  __device__ __forceinline__ T fetch(long long, unsigned, T polled) const { return polled; }
};
template <class T> struct SegStatusFor {
  using type = typename std::conditional<sizeof(T) == 4, PackedStatus<T>, WordPairStatus<T>>::type;
};
template <class T> typename SegStatusFor<T>::type seg_word_status(void* temp) {
  typename SegStatusFor<T>::type st;
  st.w = (unsigned long long*)((char*)temp + kHeaderBytes);
  return st;
}
// Bytes to clear before a launch of `ctas` segments (within seg_status_bytes).
static_assert(kSegSlots * 16 <= kSegSlots * 4 + 2 * kSegSlots * 8, "word pairs fit the 8-byte status area");
template <class T> size_t seg_word_reset_bytes(unsigned ctas) {
  return kHeaderBytes + (size_t)ctas * (sizeof(T) == 4 ? 8 : 16);
}

// Inputs up to this size go to this kernel.  Measured on GB300 (fp32 add, L2
// flushed): 12.3 / 24.6 / 32.8 us at 1e6 / 1e7 / 1.6e7 elements against 17.4 /
// 33.0 / 45.1 us for the row kernel and 30.7 / 38.9 us for the L2-resident
// look-back kernel at 1e7 / 1.6e7; at 3.2e7 (128 MB) the two meet.
constexpr long long kSegMaxBytes = 96ll << 20;

// Not for fp64: this kernel's run layout costs about five fp64 adds per element
// (warp scans of 2-element vectors), the row kernel's thread-contiguous chunks
// about 2.4, and fp64 adds, not bytes, bound fp64 scans on GB300.
// Batched rows (B > 1) come here when they are few and long: each row then gets
// several CTAs (short rows go to the row kernel, whose tiles never wait across a
// row); rows must start on 16-byte boundaries.
constexpr long long kSegMaxRows = 64;
constexpr long long kSegMinRowElems = 1 << 16;

template <class T> bool seg_applies(const ScanJob& job) {
  if (std::is_same<T, double>::value) return false;
  if (job.C != 1 || job.B < 1 || (uintptr_t)job.in % 16 != 0 || (uintptr_t)job.out % 16 != 0) return false;
  if (job.B * job.R * (long long)sizeof(T) > kSegMaxBytes) return false;
  if (job.B == 1) return true;
  return job.B <= kSegMaxRows && job.R >= kSegMinRowElems && (job.R * (long long)sizeof(T)) % 16 == 0;
}

template <class T, int OP, class G = SegGeom<T>>
cudaError_t launch_seg_op(const ScanJob& job, const LaunchCtx& ctx) {
  const SegPlan p = seg_plan<G>(job.B, job.R, ctx.num_sms);
  if (p.ctas == 0) return cudaErrorInvalidValue;  // callers check seg_applies
  SegArgs<T> a;
  a.n = job.R;
  a.nc = p.nc;
  a.segs = p.segs;
  a.ctas = p.ctas;
  a.counter = (unsigned*)job.temp;
  a.err = ctx.err;
  a.wait_ns = ctx.wait_ns;
  a.stalled = ctx.stalled_tile;
  a.in = (const T*)job.in;
  a.out = (T*)job.out;
  a.init = T{};
  if (!job.inclusive && job.init_host) memcpy(&a.init, job.init_host, sizeof(T));
  a.inclusive = job.inclusive;
  a.carry_in = (const T*)job.carry_in;
  a.carry_out = (T*)job.carry_out;
  auto st = seg_word_status<T>(job.temp);
  profile_before(ctx);
  cudaError_t e = clear_status(job.temp, seg_word_reset_bytes<T>(p.ctas), nullptr, 0, ctx);
  if (e == cudaSuccess) e = launch_pdl(scan_seg_kernel<T, OP, G, decltype(st)>, p.ctas, G::NT, 0, ctx.stream, a, st);
  profile_after(ctx);
  return e;
}

// ---- fp64: thread-contiguous chunks ----------------------------------------------
//
// GB300 adds fp64 at about 1/70 of its fp32 rate (501.6 G adds/s measured), so an
// fp64 scan is bound by adds, not bytes, and the layout above (a warp scan per pair
// of elements) costs about five adds per element.  Here lane l of a warp owns K
// consecutive elements of each chunk (a chunk is 32 x K elements), reduced serially:
//   phase 1: lane total (K - 1 adds), kept in shared memory, plus one add into the
//            warp's running total;
//   phase 3: a warp scan of the 32 kept lane totals (5 adds), the lane's base (2),
//            and the seeded serial scan of its K elements (K adds);
// about 2 + 8/K adds per element in all, against 2 for any work-efficient scan.  The
// lane's elements are loaded as 16-byte vectors K elements apart across the warp (the
// L1 cache serves the second half of every 32-byte sector).  Results go out through a
// per-warp staging buffer so that every store writes whole 128-byte lines (lane-
// strided 16-byte stores cost L2 eight partial writes per line and made the rescan
// phase take 1.8x its fp64-add time).
template <class T, int NT_, int KH_, int NH_, int MAXCPW_, int MINB_> struct SegChunkCfg {
  static constexpr int NT = NT_, NW = NT_ / 32, MINB = MINB_;
  static constexpr int VEC = Vec<T>::N;
  static constexpr int KH = KH_;                 // elements a lane holds in registers at once
  static constexpr int NH = NH_;                 // register loads per lane per chunk
  static constexpr int K = KH * NH;              // consecutive elements a lane owns per chunk
  static constexpr int CH = 32 * K;              // elements per chunk
  static constexpr int MAXCPW = MAXCPW_;         // chunks a warp can take (shared-memory slots)
  static constexpr int MAXSEG = 512;
  static constexpr int M = MAXSEG / 32;
  static constexpr size_t TOT_BYTES = (size_t)NW * MAXCPW * 32 * sizeof(T);  // kept lane totals
  static constexpr size_t STAGE_BYTES = (size_t)NW * 32 * KH * sizeof(T);     // output staging
  static constexpr size_t SMEM = TOT_BYTES + STAGE_BYTES;
  static_assert(KH % VEC == 0, "whole vectors per lane");
  static_assert(sizeof(T) != 8 || KH == 16, "the staging swizzle is laid out for 16 doubles a lane");
};
// 512 threads (126 registers a thread), 16 doubles a lane in registers at once, up to 12
// chunks a warp (112 KB of shared memory).  A lane owns 32 or 48 consecutive doubles of
// a chunk (two or three register loads): the warp scan and base of each chunk (7 adds a
// lane) are then spread over more elements, 2.22 or 2.15 adds per element against 2.44
// for 16.  Measured on GB300, fp64 add, L2 flushed, 1e7 elements: 65.4-65.9 us for 16
// doubles a lane, 61.8-62.0 us for 32, 59.7-59.8 us for 48, 63.9-65.3 us for 64.
template <class T> using SegChunkGeom = SegChunkCfg<T, 512, 16, 2, 12, 1>;
template <class T> using SegChunkGeomL = SegChunkCfg<T, 512, 16, 3, 12, 1>;

template <class T, int KH>
__device__ __forceinline__ void lane_load(T (&x)[KH], const T* in, long long e0, long long n, unsigned long long pol) {
  constexpr int VEC = Vec<T>::N;
  if (e0 + KH <= n) {
    const uint4* p = reinterpret_cast<const uint4*>(in + e0);
    if ((KH / VEC) % 2 == 0 && ((uintptr_t)p & 31) == 0) {  // 32-byte loads of whole sectors
#pragma unroll
      for (int j = 0; j < KH / VEC; j += 2) {
        uint4 lo, hi;
        ld_hint32(p + j, pol, lo, hi);
        memcpy(&x[j * VEC], &lo, 16);
        memcpy(&x[(j + 1) * VEC], &hi, 16);
      }
    } else {
#pragma unroll
      for (int j = 0; j < KH / VEC; ++j) {
        const uint4 u = ld_hint_l1(p + j, pol);
        memcpy(&x[j * VEC], &u, 16);
      }
    }
  } else {
#pragma unroll
    for (int k = 0; k < KH; ++k) x[k] = e0 + k < n ? in[e0 + k] : T{};
  }
}
// Writes the warp's 32 x 16 doubles (lane l's x[] belongs at out + e0 + l * K) as
// whole lines.  Lane l puts its element k at stage[l*16 + (k ^ (l & 15))]: for a fixed
// k the 16 lanes of a half-warp hit 16 different 8-byte bank pairs.  Store i then
// covers the pieces of lanes 4i..4i+3: lane L reads the aligned pair holding elements
// 2(L%8), 2(L%8)+1 of lane p = 4i + L/8 (swapped when the swizzle is odd) and writes
// it at its place, so eight lanes write one 128-byte piece.  A piece cut by the end of
// the input is written element by element.
template <class T, int K>
__device__ __forceinline__ void lane_store_staged(const T (&x)[16], T* stage, T* out, long long e_lane0,
                                                  long long n, int lane, unsigned long long pol) {
  static_assert(sizeof(T) == 8, "16 doubles a lane");
  __syncwarp();
  const int sw = lane & 15;
#pragma unroll
  for (int k = 0; k < 16; ++k) stage[lane * 16 + (k ^ sw)] = x[k];
  __syncwarp();
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int pl = 4 * i + (lane >> 3);  // the lane whose piece this is
    const int k = 2 * (lane & 7);
    const int ps = pl & 15;
    const double2 v2 = *reinterpret_cast<const double2*>(&stage[pl * 16 + ((k ^ ps) & ~1)]);
    T lo, hi;
    {
      const double a0 = (ps & 1) ? v2.y : v2.x, a1 = (ps & 1) ? v2.x : v2.y;
      memcpy(&lo, &a0, 8);
      memcpy(&hi, &a1, 8);
    }
    const long long e = e_lane0 + (long long)pl * K + k;
    if (e + 2 <= n) {
      uint4 u;
      memcpy(&u.x, &lo, 8);
      memcpy(&u.z, &hi, 8);
      st_hint(reinterpret_cast<uint4*>(out + e), u, pol);
    } else {
      if (e < n) out[e] = lo;
      if (e + 1 < n) out[e + 1] = hi;
    }
  }
}

template <class T, int OP, class G, class S>
__global__ void __launch_bounds__(G::NT, G::MINB) scan_seg_chunk_kernel(SegArgs<T> a, S st) {
  pdl_entry();
  constexpr int NW = G::NW, KH = G::KH, NH = G::NH, K = G::K, CH = G::CH, MAXCPW = G::MAXCPW;
  extern __shared__ __align__(16) unsigned char seg_chunk_smem[];
  __shared__ unsigned s_seg;
  __shared__ T s_warp[NW];
  __shared__ T s_base;
  __shared__ int s_hbase;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  T* s_tot = reinterpret_cast<T*>(seg_chunk_smem) + warp * MAXCPW * 32;  // [chunk][lane]
  T* s_stage = reinterpret_cast<T*>(seg_chunk_smem + G::TOT_BYTES) + warp * 32 * KH;
  if (tid == 0) s_seg = atomicAdd(a.counter, 1u);
  __syncthreads();
  const unsigned seg = s_seg;  // one row: the segment is its part
  long long c0, c1;
  const int nact = seg_chunks(a, seg, warp, NW, c0, c1);

  // Phase 1: lane totals of every chunk (kept), and the warp's total.
  const unsigned long long keep = l2_policy_evict_last();
  T acc{};
  for (long long c = c0; c < c1; ++c) {
    const long long e0 = c * CH + (long long)lane * K;
    T t{};
#pragma unroll
    for (int h = 0; h < NH; ++h) {
      T x[KH];
      lane_load<T, KH>(x, a.in, e0 + h * KH, a.n, keep);
#pragma unroll
      for (int k = 0; k < KH; ++k) t = (h == 0 && k == 0) ? x[0] : Op<T, OP>::f(t, x[k]);
    }
    s_tot[(c - c0) * 32 + lane] = t;
    acc = c == c0 ? t : Op<T, OP>::f(acc, t);
  }
  const T wtot = warp_allreduce<T, OP>(acc);
  if (lane == 0) s_warp[warp] = wtot;  // warps without chunks come last: their totals are never read
  __syncthreads();

  // Phase 2: as in scan_seg_kernel.
  if (warp == 0) {
    block_scan_warp_totals<T, OP, NW>(s_warp, lane);
    __syncwarp();
    const T agg = s_warp[nact - 1];
    if (lane == 0 && (long long)seg != a.stalled) st.publish(seg, FLAG_A, agg);
    T gathered{};
    if (seg > 0) {
      bool timed_out;
      gathered = seg_gather<T, OP, G::M>(st, 0, seg, a.wait_ns, timed_out);
      if (lane == 0 && timed_out) raise_err(a.err, ERRBIT_TIMEOUT);
    }
    if (lane == 0) {
      T b{};
      bool h;
      seg_finish_base<T, OP>(a, seg > 0, gathered, b, h);
      s_base = b;
      s_hbase = h;
    }
  }
  __syncthreads();

  // Phase 3: per chunk, a warp scan of the kept lane totals seeds each lane's serial
  // scan of its own elements.
  bool hb = s_hbase != 0;
  T base = s_base;
  if (warp > 0) {
    const T wp = s_warp[warp - 1];
    base = hb ? Op<T, OP>::f(base, wp) : wp;
    hb = true;
  }
  if (!a.inclusive) {
    base = hb ? Op<T, OP>::f(a.init, base) : a.init;
    hb = true;
  }
  const unsigned long long drop = l2_policy_evict_first();
  for (long long c = c0; c < c1; ++c) {
    const long long e0 = c * CH + (long long)lane * K;
    const T t = s_tot[(c - c0) * 32 + lane];
    const T inc = warp_inclusive<T, OP>(t, lane);
    const T exc = __shfl_up_sync(0xffffffffu, inc, 1);
    const T ctot = __shfl_sync(0xffffffffu, inc, 31);
    T r;
    bool h;
    if (lane > 0) {
      r = hb ? Op<T, OP>::f(base, exc) : exc;
      h = true;
    } else {
      r = base;
      h = hb;
    }
#pragma unroll
    for (int hh = 0; hh < NH; ++hh) {
      T x[KH];
      lane_load<T, KH>(x, a.in, e0 + hh * KH, a.n, drop);
      if (a.inclusive) {
#pragma unroll
        for (int k = 0; k < KH; ++k) {
          r = h ? Op<T, OP>::f(r, x[k]) : x[k];
          h = true;
          x[k] = r;
        }
      } else {  // exclusive: r always holds (the initial value at least)
#pragma unroll
        for (int k = 0; k < KH; ++k) {
          const T v = x[k];
          x[k] = r;
          r = Op<T, OP>::f(r, v);
        }
      }
      lane_store_staged<T, K>(x, s_stage, a.out, c * CH + hh * KH, a.n, lane, drop);
      if (a.carry_out && c == a.nc - 1) {  // the row's last element: its inclusive value
        const long long el = a.n - 1 - (e0 + hh * KH);
        T last = x[0];  // register selects, as in scan_seg_kernel
#pragma unroll
        for (int k = 0; k < KH; ++k) last = (el == k) ? x[k] : last;
        if (el >= 0 && el < KH) *a.carry_out = last;
      }
    }
    base = hb ? Op<T, OP>::f(base, ctot) : ctot;
    hb = true;
  }
}

// The warps' lane totals live in G::MAXCPW shared-memory slots per warp, so a plan
// whose warps take more chunks than that does not fit this geometry.
template <class G> bool seg_chunk_plan_fits(const SegPlan& p) {
  return p.ctas > 0 && p.cpw <= G::MAXCPW;
}

// Of the two lane lengths, the one whose busiest warp holds fewer elements (its chunk
// count times the chunk), the shorter on a tie: measured at 1e6 / 3e6 / 1e7 / 1.2e7
// doubles (19.1 / 29.3 / 61.9 / 70.3 us with 32 a lane, 19.1 / 27.2 / 59.7 / 72.3 us
// with 48), this picks the faster each time.
template <class T> bool seg_chunk_long(long long n, int num_sms) {
  using G2 = SegChunkGeom<T>;
  using G3 = SegChunkGeomL<T>;
  const SegPlan p2 = seg_plan<G2>(1, n, num_sms), p3 = seg_plan<G3>(1, n, num_sms);
  return p3.cpw * G3::CH < p2.cpw * G2::CH;
}

template <class T> bool seg_chunk_applies(const ScanJob& job, int num_sms) {
  if (!(job.B == 1 && job.C == 1 && (uintptr_t)job.in % 16 == 0 && (uintptr_t)job.out % 16 == 0 &&
        job.R * (long long)sizeof(T) <= kSegMaxBytes))
    return false;
  if (seg_chunk_long<T>(job.R, num_sms))
    return seg_chunk_plan_fits<SegChunkGeomL<T>>(seg_plan<SegChunkGeomL<T>>(1, job.R, num_sms));
  return seg_chunk_plan_fits<SegChunkGeom<T>>(seg_plan<SegChunkGeom<T>>(1, job.R, num_sms));
}

template <class T, int OP, class G>
cudaError_t launch_seg_chunk_op(const ScanJob& job, const LaunchCtx& ctx) {
  const SegPlan p = seg_plan<G>(1, job.R, ctx.num_sms);
  if (p.ctas == 0 || !seg_chunk_plan_fits<G>(p)) return cudaErrorInvalidValue;  // callers check seg_chunk_applies
  SegArgs<T> a;
  a.n = job.R;
  a.nc = p.nc;
  a.segs = p.segs;
  a.ctas = p.ctas;
  a.counter = (unsigned*)job.temp;
  a.err = ctx.err;
  a.wait_ns = ctx.wait_ns;
  a.stalled = ctx.stalled_tile;
  a.in = (const T*)job.in;
  a.out = (T*)job.out;
  a.init = T{};
  if (!job.inclusive && job.init_host) memcpy(&a.init, job.init_host, sizeof(T));
  a.inclusive = job.inclusive;
  a.carry_in = (const T*)job.carry_in;
  a.carry_out = (T*)job.carry_out;
  auto st = seg_word_status<T>(job.temp);
  auto kern = scan_seg_chunk_kernel<T, OP, G, decltype(st)>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)G::SMEM);
  if (e != cudaSuccess) return e;
  profile_before(ctx);
  e = clear_status(job.temp, seg_word_reset_bytes<T>(p.ctas), nullptr, 0, ctx);
  if (e == cudaSuccess) e = launch_pdl(kern, p.ctas, G::NT, G::SMEM, ctx.stream, a, st);
  profile_after(ctx);
  return e;
}

template <class T, int OP> cudaError_t launch_seg_chunk(const ScanJob& job, const LaunchCtx& ctx) {
  return seg_chunk_long<T>(job.R, ctx.num_sms) ? launch_seg_chunk_op<T, OP, SegChunkGeomL<T>>(job, ctx)
                                               : launch_seg_chunk_op<T, OP, SegChunkGeom<T>>(job, ctx);
}

}  // namespace gbs
