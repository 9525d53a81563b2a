// scan_lanes.cuh -- single-pass decoupled look-back scan along the middle axis of a
// row-major (B, R, C) array with C > 1 lanes: scans down the columns of a matrix,
// and scans of elements made of several values (a 96-byte struct is 24 fp32
// lanes, a dual number with 16 partials is 17 fp64 lanes), each lane on its own.
//
// A tile is RT consecutive positions (rows) x CT consecutive lanes (a strip of the
// columns; CT = C when C is small).  Its row count is chosen from the lane count so
// that its size stays fixed (32 KB for 4-byte, 64 KB for 8-byte lanes) whatever the
// element width, which is what lets 96- and 136-byte elements fit shared memory
// (AcceleratedKernels.jl PR #208 sizes its tiles from the element type for the same
// reason).  Threads map
// to (lane c, row group g); each thread combines RPG rows of one lane serially in
// shared memory, a warp scans the G group totals of a lane, and one thread per
// lane looks back along that lane.  Tiles of one (batch, strip) chain are scanned
// in order through the look-back; chains are independent.
#pragma once

#include "launch.h"
#include "tile.cuh"

namespace gbs {

template <class T> struct LanesArgs {
  const T* in;
  T* out;
  long long R, C;           // positions per chain, lanes per position
  int CT, G, RT;            // strip width, row groups, rows per tile (= G * RPG)
  unsigned strips;          // ceil(C / CT)
  unsigned tiles_per_chain; // ceil(R / RT)
  unsigned num_tiles;       // B * strips * tiles_per_chain
  unsigned* counter;
  ErrSink err;
  const T* init;            // device copy of the initial value (exclusive)
  int init_lanes;           // lane c starts from init[c % init_lanes]
  int inclusive;
  unsigned long long wait_ns;
  long long stalled_tile;
};

// Rows per thread: 32 (tiles of 32 KB for 4-byte and 64 KB for 8-byte lanes).  A
// sweep over 8..64 rows per thread on the column and lane-vector workloads (4096x4096
// and 1e6x8 axis 0, 96-byte structs, 17-lane duals, 1000x1e4 fp64 axis 0) put 32 at
// or near the best everywhere: fewer, larger tiles mean fewer look-backs along a
// chain, which is what limits these scans (dual16 1e6: 372 us at 8, 165 us at 32).
template <class T, int RPG_ = 32, int D_ = 4, int CTMAX_ = 0> struct LanesGeomT {
  static constexpr int NT = 256;
  static constexpr int NW = NT / 32;
  static constexpr int RPG = RPG_;                        // rows per thread
  // Look-back: predecessors per round trip of a lane's thread.  4 is best on every
  // lane workload measured (96-byte structs 1e6: 51.9 / 59.5 / 62.1 us at 4 / 8 / 16;
  // 17-lane duals 1e6: 162 / 176 / 232 us): wider windows cost registers and occupancy.
  static constexpr int D = D_;
  // Strip width: 128-byte strips for 4-byte lanes, 256-byte for 8-byte.  Wider strips
  // (fewer, larger per-row copies, longer chains) measured slower everywhere (4096 x
  // 4096 fp32 columns: 43.6 / 49.8 / 62.0 us at 64 / 128 / 256 lanes; 1000 x 1e4 fp64:
  // 72-74 / 74.3 / 76.4 us at 32 / 64 / 128), and 32 fp32 lanes beat 64 on 2080-byte
  // elements (32.9 against 35.0 us: twice the chains, half as long).
  static constexpr int CTMAX = CTMAX_ > 0 ? CTMAX_ : 32;
  static int ct(long long C) { return C <= CTMAX ? (int)C : CTMAX; }
  static int groups(int CT) {
    int g = NT / CT;
    return g > 32 ? 32 : g;
  }
};
template <class T> using LanesGeom = LanesGeomT<T>;

template <class T, int OP, class S, class Gm = LanesGeom<T>>
__global__ void __launch_bounds__(Gm::NT) scan_lanes_kernel(LanesArgs<T> a, S st) {
  pdl_entry();
  constexpr int NT = Gm::NT, NW = Gm::NW, RPG = Gm::RPG;
  __shared__ __align__(128) T s_tile[NT * RPG];
  __shared__ T s_gx[NT];     // group totals, then exclusive group prefixes, [g*CT + c]
  __shared__ T s_pfx[NT];    // per lane: aggregate, then the tile's exclusive prefix
  __shared__ __align__(8) unsigned long long s_bar;
  __shared__ unsigned s_t;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int CT = a.CT, G = a.G, RT = a.RT;

  // Thread 0 claims the tile, decides how to load it and arms the mbarrier with
  // the expected byte count before any copy is issued.
  __shared__ int s_bulk;
  if (tid == 0) {
    const unsigned t0 = atomicAdd(a.counter, 1u);
    s_t = t0;
    const unsigned ch = t0 / a.tiles_per_chain, t_in = t0 - ch * a.tiles_per_chain;
    const unsigned bb = ch / a.strips, sp = ch - bb * a.strips;
    const long long rr0 = (long long)t_in * RT;
    const int nrows = a.R - rr0 >= RT ? RT : (int)(a.R - rr0);
    const long long cc0 = (long long)sp * CT;
    const int ncols = a.C - cc0 >= CT ? CT : (int)(a.C - cc0);
    const long long gb0 = ((long long)bb * a.R + rr0) * a.C + cc0;
    const size_t rbytes = (size_t)ncols * sizeof(T);
    bool blk = aligned16(a.in + gb0) && aligned16(a.out + gb0);
    if (ncols == a.C) blk = blk && ((size_t)nrows * rbytes) % 16 == 0;
    else blk = blk && rbytes % 16 == 0 && ((size_t)a.C * sizeof(T)) % 16 == 0 && ((size_t)CT * sizeof(T)) % 16 == 0;
    s_bulk = blk;
    if (blk) {
      mbar_init(&s_bar, 1);
      fence_mbar_init();
      mbar_arrive_expect_tx(&s_bar, (unsigned)(nrows * rbytes));
    }
  }
  __syncthreads();
  const unsigned t = s_t;
  const unsigned chain = t / a.tiles_per_chain, tt = t - chain * a.tiles_per_chain;
  const unsigned b = chain / a.strips, strip = chain - b * a.strips;
  const long long r0 = (long long)tt * RT;
  const int rows = a.R - r0 >= RT ? RT : (int)(a.R - r0);
  const long long c0 = (long long)strip * CT;
  const int cols = a.C - c0 >= CT ? CT : (int)(a.C - c0);
  const long long gbase = ((long long)b * a.R + r0) * a.C + c0;
  const T* src = a.in + gbase;
  T* dst = a.out + gbase;

  // Load.  Whole rows (CT == C): one contiguous copy.  A strip: one copy per row.
  const bool whole = cols == a.C;
  const size_t row_bytes = (size_t)cols * sizeof(T);
  const bool bulk = s_bulk != 0;
  bool failed = false;
  if (bulk) {
    if (whole) {
      if (tid == 0) bulk_g2s(s_tile, src, (unsigned)(rows * row_bytes), &s_bar);
    } else {
      for (int r = tid; r < rows; r += NT) bulk_g2s(s_tile + r * CT, src + r * a.C, (unsigned)row_bytes, &s_bar);
    }
    failed = !mbar_wait(&s_bar, 0, a.wait_ns);
  } else {
    for (int k = tid; k < rows * cols; k += NT) {
      const int r = k / cols, c = k - r * cols;
      s_tile[r * CT + c] = src[(long long)r * a.C + c];
    }
  }
  if (__syncthreads_or(failed)) {
    if (tid == 0) {
      raise_err(a.err, ERRBIT_TIMEOUT);
      mbar_wait(&s_bar, 0, a.wait_ns);
    }
    if (tid < cols && (long long)t != a.stalled_tile) st.publish((long long)t * CT + tid, FLAG_P, T{});
    return;
  }

  // Pass 1: each (lane c, group g) combines its RPG rows.
  const int c = tid % CT, g = tid / CT;
  const int rb = g * RPG, re = rb + RPG < rows ? rb + RPG : rows;
  const bool active = g < G && c < cols && rb < rows;
  if (active) {
    T acc = s_tile[rb * CT + c];
    for (int r = rb + 1; r < re; ++r) acc = Op<T, OP>::f(acc, s_tile[r * CT + c]);
    s_gx[g * CT + c] = acc;
  }
  __syncthreads();

  // Exclusive scan of the group totals of each lane.  fp64: one thread per lane,
  // serially (G - 1 adds a lane, where a warp-wide scan costs 5 x 32: fp64 adds are
  // what bounds 8-byte float lanes on this GPU); else one warp per lane.
  const int ngroups = (rows + RPG - 1) / RPG;
  if constexpr (std::is_same<T, double>::value) {
    if (tid < cols) {
      T run = s_gx[tid];
      for (int g0 = 1; g0 < ngroups; g0 += 8) {
        T v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u)
          if (g0 + u < ngroups) v[u] = s_gx[(g0 + u) * CT + tid];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          if (g0 + u < ngroups) {
            s_gx[(g0 + u) * CT + tid] = run;
            run = Op<T, OP>::f(run, v[u]);
          }
        }
      }
      s_pfx[tid] = run;
    }
  } else {
    for (int cc = warp; cc < cols; cc += NW) {
      const T v = s_gx[(lane < ngroups ? lane : ngroups - 1) * CT + cc];
      const T inc = warp_inclusive<T, OP>(v, lane);
      const T exc = __shfl_up_sync(0xffffffffu, inc, 1);
      const T agg = __shfl_sync(0xffffffffu, inc, ngroups - 1);
      __syncwarp();
      if (lane < ngroups && lane > 0) s_gx[lane * CT + cc] = exc;
      if (lane == 0) s_pfx[cc] = agg;
    }
  }
  __syncthreads();

  // Publish and look back, one thread per lane.
  if (tid < cols) {
    const T agg = s_pfx[tid];
    const long long first = (long long)t - tt;  // tile index of the chain's tile 0
    const bool stalled = (long long)t == a.stalled_tile;
    const long long si = (long long)t * CT + tid;
    if (tt == 0) {
      if (!stalled) st.publish(si, FLAG_P, agg);
    } else {
      if (!stalled) st.publish(si, FLAG_A, agg);
      bool timed_out;
      const T pfx = lookback_lane<T, OP, Gm::D>(st, first, tt, tid, CT, a.wait_ns, timed_out);
      if (!stalled) st.publish(si, FLAG_P, Op<T, OP>::f(pfx, agg));
      s_pfx[tid] = pfx;
      if (timed_out) raise_err(a.err, ERRBIT_TIMEOUT);
    }
  }
  __syncthreads();

  // Pass 2: rewrite the rows in place.
  if (active) {
    bool h = tt > 0;
    T base = s_pfx[c];
    if (g > 0) {
      const T gx = s_gx[g * CT + c];
      base = h ? Op<T, OP>::f(base, gx) : gx;
      h = true;
    }
    if (!a.inclusive) {
      const T i0 = a.init[(c0 + c) % a.init_lanes];
      base = h ? Op<T, OP>::f(i0, base) : i0;
      h = true;
    }
    if (a.inclusive) {
      for (int r = rb; r < re; ++r) {
        const T x = s_tile[r * CT + c];
        base = h ? Op<T, OP>::f(base, x) : x;
        h = true;
        s_tile[r * CT + c] = base;
      }
    } else {
      for (int r = rb; r < re; ++r) {
        const T x = s_tile[r * CT + c];
        s_tile[r * CT + c] = base;
        base = Op<T, OP>::f(base, x);
      }
    }
  }

  if (bulk) {
    fence_proxy_async_smem();
    __syncthreads();
    if (whole) {
      if (tid == 0) {
        bulk_s2g(dst, s_tile, (unsigned)(rows * row_bytes));
        bulk_commit();
        bulk_wait_read_all();
      }
    } else {
      for (int r = tid; r < rows; r += NT) {
        bulk_s2g(dst + r * a.C, s_tile + r * CT, (unsigned)row_bytes);
        bulk_commit();
      }
      bulk_wait_read_all();
    }
  } else {
    __syncthreads();
    for (int k = tid; k < rows * cols; k += NT) {
      const int r = k / cols, cc = k - r * cols;
      dst[(long long)r * a.C + cc] = s_tile[r * CT + cc];
    }
  }
}

template <class T, class Gm = LanesGeom<T>> struct LanesPlan {
  int CT, G, RT;
  unsigned strips, tiles_per_chain, num_tiles;
};

template <class T, class Gm = LanesGeom<T>> LanesPlan<T, Gm> lanes_plan(long long B, long long R, long long C) {
  LanesPlan<T, Gm> p;
  p.CT = Gm::ct(C);
  p.G = Gm::groups(p.CT);
  p.RT = p.G * Gm::RPG;
  p.strips = (unsigned)((C + p.CT - 1) / p.CT);
  p.tiles_per_chain = (unsigned)((R + p.RT - 1) / p.RT);
  p.num_tiles = (unsigned)(B * p.strips * p.tiles_per_chain);
  return p;
}

// Layout after the header: [init: up to 4096 lanes][status]
template <class T> size_t lanes_init_bytes(long long C) {
  const long long n = C < 4096 ? C : 4096;
  return round_up((size_t)n * sizeof(T), 256);
}
template <class T, class Gm> size_t lanes_status_entries(const LanesPlan<T, Gm>& p) {
  return (size_t)p.num_tiles * p.CT;
}
template <class T, class Gm> size_t lanes_flag_bytes(const LanesPlan<T, Gm>& p) {
  return sizeof(T) == 4 ? round_up(lanes_status_entries(p) * 8, 256)
                        : round_up(lanes_status_entries(p) * 4, 256);
}
template <class T, class Gm = LanesGeom<T>> size_t lanes_temp_bytes(long long B, long long R, long long C) {
  const LanesPlan<T, Gm> p = lanes_plan<T, Gm>(B, R, C);
  size_t s = kHeaderBytes + lanes_init_bytes<T>(C) + lanes_flag_bytes(p);
  if (sizeof(T) == 8) s += 2 * round_up(lanes_status_entries(p) * sizeof(T), 256);
  return s;
}

template <class T, int OP, class Gm = LanesGeom<T>>
cudaError_t launch_lanes_op(const ScanJob& job, const LaunchCtx& ctx) {
  const LanesPlan<T, Gm> p = lanes_plan<T, Gm>(job.B, job.R, job.C);
  LanesArgs<T> a;
  a.in = (const T*)job.in;
  a.out = (T*)job.out;
  a.R = job.R;
  a.C = job.C;
  a.CT = p.CT;
  a.G = p.G;
  a.RT = p.RT;
  a.strips = p.strips;
  a.tiles_per_chain = p.tiles_per_chain;
  a.num_tiles = p.num_tiles;
  a.counter = (unsigned*)job.temp;
  a.err = ctx.err;
  char* init_area = (char*)job.temp + kHeaderBytes;
  a.init = (const T*)init_area;
  a.init_lanes = job.init_lanes;
  a.inclusive = job.inclusive;
  a.wait_ns = ctx.wait_ns;
  a.stalled_tile = ctx.stalled_tile;

  char* status = init_area + lanes_init_bytes<T>(job.C);
  typename StatusFor<T>::type st;
  if constexpr (sizeof(T) == 4) {
    st.w = (unsigned long long*)status;
  } else {
    st.flag = (unsigned*)status;
    st.agg = (T*)(status + lanes_flag_bytes(p));
    st.pfx = (T*)(status + lanes_flag_bytes(p) + round_up(lanes_status_entries(p) * sizeof(T), 256));
  }
  profile_before(ctx);
  cudaError_t e = cudaSuccess;
  if (!job.inclusive)
    e = cudaMemcpyAsync(init_area, job.init_host, (size_t)job.init_lanes * sizeof(T), cudaMemcpyHostToDevice,
                        ctx.stream);
  if (e == cudaSuccess) e = clear_status(job.temp, kHeaderBytes, status, lanes_flag_bytes(p), ctx);
  if (e == cudaSuccess) e = launch_pdl(scan_lanes_kernel<T, OP, decltype(st), Gm>, p.num_tiles, Gm::NT, 0, ctx.stream, a, st);
  profile_after(ctx);
  return e;
}

}  // namespace gbs
