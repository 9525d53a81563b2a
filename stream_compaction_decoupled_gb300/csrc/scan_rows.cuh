// scan_rows.cuh -- single-pass decoupled look-back scan of contiguous rows: a 1-D
// scan is one row; a batched scan along axis 1 of a row-major matrix is one row
// per matrix row.  Tiles never cross a row, and a row's tile 0 publishes its
// inclusive prefix at once, so the look-back stops at the start of the row.
//
// Per tile (one CTA, claimed in order from an atomic counter; The CUDA Handbook,
// 13.3.4-13.3.5, Listings 13-14 and 13-16):
//   1. claim the tile index; one thread issues a bulk (TMA) copy of the whole
//      tile into shared memory, completing on an mbarrier (a ragged or unaligned
//      tile is loaded with plain coalesced loads instead);
//   2. pass 1: per-(round, lane) serial combine of a 16-byte vector, warp scans
//      of the lane totals, per-warp totals;
//   3. block scan of the warp totals (warp 0) -> tile aggregate;
//   4. warp 0 publishes A (or P for a row's first tile) and looks back;
//      publishes P;
//   5. pass 2 rewrites the tile in shared memory with the final values;
//   6. one thread bulk-copies the tile back to global memory.
#pragma once

#include "launch.h"
#include "tile.cuh"

namespace gbs {

template <class T> struct RowsArgs {
  const T* in;
  T* out;
  long long R;              // elements per row
  unsigned tiles_per_row;   // ceil(R / TILE)
  unsigned num_tiles;       // rows * tiles_per_row
  unsigned* counter;        // tile-claim counter, 0 on entry
  ErrSink err;            // device-wide and per-call error words
  T init;                   // exclusive scans: folded in on the left of every row
  int inclusive;
  int bulk_ok;              // in, out and every row start are 16-byte aligned
  unsigned long long wait_ns;
  long long stalled_tile;
};

// Tile geometry: NT threads, ROUNDS 16-byte vectors per thread, K predecessors
// per lane in the look-back window, MINB resident CTAs per SM asked of the compiler.
template <class T, int NT_, int ROUNDS_, int K_, int MINB_> struct RowsCfg {
  static constexpr int NT = NT_;
  static constexpr int NW = NT / 32;
  static constexpr int ROUNDS = ROUNDS_;
  static constexpr int VEC = 16 / (int)sizeof(T);
  static constexpr int TILE = NW * ROUNDS * 32 * VEC;
  static constexpr int K = K_;
  static constexpr int MINB = MINB_;
};

// The configuration the library uses: 16 KB tiles of 128 threads, so that a dozen
// CTAs (tiles) are resident per SM, and a look-back window of 32 tiles (one per
// lane).  (A sweep on the fp32 1e8 scan: windows of 4 or 8 tiles per lane were
// slower, 6 CTAs of 256 threads were slower, 32 KB tiles were no faster.  A window
// of 2 tiles per lane made warp 0 spill its per-round prefixes at the 40 registers
// that 12 CTAs leave a thread.)  8-byte integers get 10 CTAs (48 registers), whose
// pairs of registers per value would spill at 40.
// fp64 runs the chunked variant (see scan_rows_chunk_kernel), which keeps a thread's
// 16 doubles in registers; 8 CTAs per SM (64 registers a thread) let one tile's
// FP64 adds overlap other tiles' loads and look-backs best (113 us against 130 us
// at 4 CTAs for 1e7 doubles).
template <class T>
using RowsGeom = RowsCfg<T, 128, 8, 1, std::is_same<T, double>::value ? 8 : (sizeof(T) == 8 ? 10 : 12)>;

template <class T, int OP, class G, class S>
__global__ void __launch_bounds__(G::NT, G::MINB) scan_rows_kernel(RowsArgs<T> a, S st) {
  pdl_entry();
  constexpr int NT = G::NT, NW = G::NW, ROUNDS = G::ROUNDS, TILE = G::TILE;
  __shared__ __align__(128) T s_tile[TILE];
  __shared__ __align__(8) unsigned long long s_bar;
  __shared__ unsigned s_t;
  __shared__ T s_warp[NW];
  __shared__ T s_prefix;
  __shared__ int s_has_prefix;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  if (tid == 0) {
    const unsigned t = atomicAdd(a.counter, 1u);
    s_t = t;
    const unsigned row = t / a.tiles_per_row, tt = t - row * a.tiles_per_row;
    const long long off = (long long)tt * TILE;
    if (a.bulk_ok && a.R - off >= TILE) {
      mbar_init(&s_bar, 1);
      fence_mbar_init();
      mbar_arrive_expect_tx(&s_bar, TILE * sizeof(T));
      bulk_g2s(s_tile, a.in + (long long)row * a.R + off, TILE * sizeof(T), &s_bar);
    }
  }
  __syncthreads();
  const unsigned t = s_t;
  const unsigned row = t / a.tiles_per_row, tt = t - row * a.tiles_per_row;
  const long long off = (long long)tt * TILE;
  const long long start = (long long)row * a.R + off;
  const int len = a.R - off >= TILE ? TILE : (int)(a.R - off);
  const bool bulk = a.bulk_ok && len == TILE;

  bool failed = false;
  if (bulk) {
    failed = !mbar_wait(&s_bar, 0, a.wait_ns);
  } else {
    const T* src = a.in + start;
    for (int k = tid; k < TILE; k += NT) s_tile[k] = k < len ? src[k] : T{};
  }
  if (__syncthreads_or(failed)) {
    // The copy never landed: record it, let successors go on, write nothing.
    if (tid == 0) {
      raise_err(a.err, ERRBIT_TIMEOUT);
      mbar_wait(&s_bar, 0, a.wait_ns);  // give the copy in flight one more bounded wait
      if ((long long)t != a.stalled_tile) {
        S(st).publish((long long)row * a.tiles_per_row + tt, FLAG_P, T{});
      }
    }
    return;
  }

  // Pass 1.
  uint4* run = reinterpret_cast<uint4*>(s_tile) + warp * ROUNDS * 32;
  T pre[ROUNDS];
  const T wtot = tile_reduce_pass<T, OP, ROUNDS>(run, lane, pre);
  if (lane == 0) s_warp[warp] = wtot;
  __syncthreads();

  // Block scan of warp totals, then the look-back, both by warp 0.
  if (warp == 0) {
    const T agg = block_scan_warp_totals<T, OP, NW>(s_warp, lane);
    const long long first = (long long)row * a.tiles_per_row;
    const bool stalled = (long long)t == a.stalled_tile;
    if (tt == 0) {
      if (lane == 0) {
        if (!stalled) st.publish(first, FLAG_P, agg);
        s_has_prefix = 0;
      }
    } else {
      if (lane == 0 && !stalled) st.publish(first + tt, FLAG_A, agg);
      bool timed_out;
      const T pfx = lookback_warp<T, OP, G::K>(st, first, tt, a.wait_ns, timed_out);
      if (lane == 0) {
        if (!stalled) st.publish(first + tt, FLAG_P, Op<T, OP>::f(pfx, agg));
        s_prefix = pfx;
        s_has_prefix = 1;
        if (timed_out) raise_err(a.err, ERRBIT_TIMEOUT);
      }
    }
  }
  __syncthreads();

  // Pass 2: base = tile prefix (+) warps before this one (+ init on the left).
  bool has_base = s_has_prefix != 0;
  T base = s_prefix;
  if (warp > 0) {
    const T wp = s_warp[warp - 1];
    base = has_base ? Op<T, OP>::f(base, wp) : wp;
    has_base = true;
  }
  if (!a.inclusive) {
    base = has_base ? Op<T, OP>::f(a.init, base) : a.init;
    has_base = true;
  }
  tile_apply_pass<T, OP, ROUNDS>(run, lane, pre, base, has_base, a.inclusive != 0);

  if (bulk) {
    fence_proxy_async_smem();
    __syncthreads();
    if (tid == 0) {
      bulk_s2g(a.out + start, s_tile, TILE * sizeof(T));
      bulk_commit();
      bulk_wait_read_all();
    }
  } else {
    __syncthreads();
    T* dst = a.out + start;
    for (int k = tid; k < len; k += NT) dst[k] = s_tile[k];
  }
}

// The same tile scan with thread-contiguous chunks (see chunk_load): thread l of
// warp w owns the CV vectors [(w*32 + l)*CV, +CV) of the tile.  Used where each
// operator application is expensive (fp64 on GB300 adds at ~1/68 of the fp32 rate):
// about 2.4 operator applications per element instead of ~5.5.
template <class T, int OP, class G, class S>
__global__ void __launch_bounds__(G::NT, G::MINB) scan_rows_chunk_kernel(RowsArgs<T> a, S st) {
  pdl_entry();
  constexpr int NT = G::NT, NW = G::NW, CV = G::ROUNDS, VEC = G::VEC, TILE = G::TILE;
  static_assert((CV & (CV - 1)) == 0, "chunk length must be a power of two");
  __shared__ __align__(128) T s_tile[TILE];
  __shared__ __align__(8) unsigned long long s_bar;
  __shared__ unsigned s_t;
  __shared__ T s_warp[NW];
  __shared__ T s_prefix;
  __shared__ int s_has_prefix;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    const unsigned t = atomicAdd(a.counter, 1u);
    s_t = t;
    const unsigned row = t / a.tiles_per_row, tt = t - row * a.tiles_per_row;
    const long long off = (long long)tt * TILE;
    if (a.bulk_ok && a.R - off >= TILE) {
      mbar_init(&s_bar, 1);
      fence_mbar_init();
      mbar_arrive_expect_tx(&s_bar, TILE * sizeof(T));
      bulk_g2s(s_tile, a.in + (long long)row * a.R + off, TILE * sizeof(T), &s_bar);
    }
  }
  __syncthreads();
  const unsigned t = s_t;
  const unsigned row = t / a.tiles_per_row, tt = t - row * a.tiles_per_row;
  const long long off = (long long)tt * TILE;
  const long long start = (long long)row * a.R + off;
  const int len = a.R - off >= TILE ? TILE : (int)(a.R - off);
  const bool bulk = a.bulk_ok && len == TILE;
  bool failed = false;
  if (bulk) {
    failed = !mbar_wait(&s_bar, 0, a.wait_ns);
  } else {
    const T* src = a.in + start;
    for (int k = tid; k < TILE; k += NT) s_tile[k] = k < len ? src[k] : T{};
  }
  if (__syncthreads_or(failed)) {
    if (tid == 0) {
      raise_err(a.err, ERRBIT_TIMEOUT);
      mbar_wait(&s_bar, 0, a.wait_ns);
      if ((long long)t != a.stalled_tile) st.publish((long long)row * a.tiles_per_row + tt, FLAG_P, T{});
    }
    return;
  }

  // Pass 1: the thread's chunk total, then one warp scan of the totals.  The chunk
  // is read again from shared memory in pass 2, so it does not occupy registers
  // across the look-back.
  uint4* chunk = reinterpret_cast<uint4*>(s_tile) + (warp * 32 + lane) * CV;
  T tot;
  {
    Vec<T> v[CV];
    chunk_load<T, CV>(chunk, lane, v);
    tot = v[0].v[0];  // any order: the total does not depend on it (up to rounding)
#pragma unroll
    for (int e = 1; e < VEC; ++e) tot = Op<T, OP>::f(tot, v[0].v[e]);
#pragma unroll
    for (int j = 1; j < CV; ++j)
#pragma unroll
      for (int e = 0; e < VEC; ++e) tot = Op<T, OP>::f(tot, v[j].v[e]);
  }
  const T wi = warp_inclusive<T, OP>(tot, lane);
  const T we = __shfl_up_sync(0xffffffffu, wi, 1);  // lane 0: none
  if (lane == 31) s_warp[warp] = wi;
  __syncthreads();

  if (warp == 0) {
    const T agg = block_scan_warp_totals<T, OP, NW>(s_warp, lane);
    const long long first = (long long)row * a.tiles_per_row;
    const bool stalled = (long long)t == a.stalled_tile;
    if (tt == 0) {
      if (lane == 0) {
        if (!stalled) st.publish(first, FLAG_P, agg);
        s_has_prefix = 0;
      }
    } else {
      if (lane == 0 && !stalled) st.publish(first + tt, FLAG_A, agg);
      bool timed_out;
      const T pfx = lookback_warp<T, OP, G::K>(st, first, tt, a.wait_ns, timed_out);
      if (lane == 0) {
        if (!stalled) st.publish(first + tt, FLAG_P, Op<T, OP>::f(pfx, agg));
        s_prefix = pfx;
        s_has_prefix = 1;
        if (timed_out) raise_err(a.err, ERRBIT_TIMEOUT);
      }
    }
  }
  __syncthreads();

  // Pass 2: base = tile prefix (+) earlier warps (+) earlier lanes (+ init on the left).
  bool hb = s_has_prefix != 0;
  T base = s_prefix;
  if (warp > 0) {
    const T wp = s_warp[warp - 1];
    base = hb ? Op<T, OP>::f(base, wp) : wp;
    hb = true;
  }
  if (lane > 0) {
    base = hb ? Op<T, OP>::f(base, we) : we;
    hb = true;
  }
  if (!a.inclusive) {
    base = hb ? Op<T, OP>::f(a.init, base) : a.init;
    hb = true;
  }
  Vec<T> v[CV];
  chunk_load<T, CV>(chunk, lane, v);
  chunk_rotate<T, CV, -1>(v, lane);  // v[k] is now chunk vector k
  if (a.inclusive) {
#pragma unroll
    for (int k = 0; k < CV; ++k)
#pragma unroll
      for (int e = 0; e < VEC; ++e) {
        base = hb ? Op<T, OP>::f(base, v[k].v[e]) : v[k].v[e];
        hb = true;
        v[k].v[e] = base;
      }
  } else {
#pragma unroll
    for (int k = 0; k < CV; ++k)
#pragma unroll
      for (int e = 0; e < VEC; ++e) {
        const T x = v[k].v[e];
        v[k].v[e] = base;
        base = Op<T, OP>::f(base, x);
      }
  }
  chunk_rotate<T, CV, +1>(v, lane);
  chunk_store<T, CV>(chunk, lane, v);

  if (bulk) {
    fence_proxy_async_smem();
    __syncthreads();
    if (tid == 0) {
      bulk_s2g(a.out + start, s_tile, TILE * sizeof(T));
      bulk_commit();
      bulk_wait_read_all();
    }
  } else {
    __syncthreads();
    T* dst = a.out + start;
    for (int k = tid; k < len; k += NT) dst[k] = s_tile[k];
  }
}

// Status area of the row kernel, right after the header.
template <class T> size_t rows_status_bytes(unsigned num_tiles) {
  if (sizeof(T) == 4) return round_up((size_t)num_tiles * 8, 256);
  return round_up((size_t)num_tiles * 4, 256) + 2 * round_up((size_t)num_tiles * sizeof(T), 256);
}
// Bytes the per-call reset has to clear (counter + flags).
template <class T> size_t rows_reset_bytes(unsigned num_tiles) {
  if (sizeof(T) == 4) return kHeaderBytes + round_up((size_t)num_tiles * 8, 256);
  return kHeaderBytes + round_up((size_t)num_tiles * 4, 256);
}

template <class T, class G = RowsGeom<T>> unsigned rows_tiles(long long B, long long R) {
  const long long tpr = (R + G::TILE - 1) / G::TILE;
  return (unsigned)(B * tpr);
}

template <class T> typename StatusFor<T>::type rows_status(void* temp, unsigned num_tiles) {
  char* base = (char*)temp + kHeaderBytes;
  typename StatusFor<T>::type st;
  if constexpr (sizeof(T) == 4) {
    st.w = (unsigned long long*)base;
  } else {
    st.flag = (unsigned*)base;
    base += round_up((size_t)num_tiles * 4, 256);
    st.agg = (T*)base;
    base += round_up((size_t)num_tiles * sizeof(T), 256);
    st.pfx = (T*)base;
  }
  return st;
}

template <class T, int OP, class G = RowsGeom<T>>
cudaError_t launch_rows_op(const ScanJob& job, const LaunchCtx& ctx) {
  RowsArgs<T> a;
  a.in = (const T*)job.in;
  a.out = (T*)job.out;
  a.R = job.R;
  a.tiles_per_row = (unsigned)((job.R + G::TILE - 1) / G::TILE);
  a.num_tiles = rows_tiles<T, G>(job.B, job.R);
  a.counter = (unsigned*)job.temp;
  a.err = ctx.err;
  a.init = T{};
  if (!job.inclusive && job.init_host) memcpy(&a.init, job.init_host, sizeof(T));
  a.inclusive = job.inclusive;
  a.bulk_ok = ((uintptr_t)job.in % 16 == 0) && ((uintptr_t)job.out % 16 == 0) &&
              (job.B == 1 || (job.R * (long long)sizeof(T)) % 16 == 0);
  a.wait_ns = ctx.wait_ns;
  a.stalled_tile = ctx.stalled_tile;
  auto st = rows_status<T>(job.temp, a.num_tiles);
  profile_before(ctx);
  cudaError_t e = clear_status(job.temp, rows_reset_bytes<T>(a.num_tiles), nullptr, 0, ctx);
  if (e == cudaSuccess) {
    if constexpr (std::is_same<T, double>::value) {
      // fp64: thread-contiguous chunks (fewer operator applications).
      e = launch_pdl(scan_rows_chunk_kernel<T, OP, G, decltype(st)>, a.num_tiles, G::NT, 0, ctx.stream, a, st);
    } else {
      e = launch_pdl(scan_rows_kernel<T, OP, G, decltype(st)>, a.num_tiles, G::NT, 0, ctx.stream, a, st);
    }
  }
  profile_after(ctx);
  return e;
}

}  // namespace gbs
