// tile.cuh -- the pieces of a single-pass tile scan shared by every kernel:
// tile-status descriptors, the decoupled look-back, and the two passes over a tile
// held in shared memory.
//
// A tile of TILE = NW warps x ROUNDS x 32 lanes x VEC elements lives in shared
// memory in its natural order.  Warp w owns the contiguous run
// [w*ROUNDS*32*VEC, (w+1)*ROUNDS*32*VEC); in round j lane l owns the 16-byte vector
// at j*32 + l of that run.  Reading the tile this way is a conflict-free 128-bit
// shared-memory access, and every element is read by exactly one thread.
//
// Pass 1 (reduce) gives each (round, lane) the combination of all warp elements
// before it and each warp its total; the block scan of the warp totals gives each
// warp its offset and the tile its aggregate; the look-back gives the tile its
// exclusive prefix; pass 2 (apply) rewrites the tile in place with the scanned
// values.  Each element is read twice and written once in shared memory; in global
// memory it is read once and written once (The CUDA Handbook, 13.3.4: 2N traffic).
#pragma once

#include "common.cuh"

namespace gbs {

// ---- tile-status descriptors -------------------------------------------------------

// 4-byte values: one 64-bit word per tile holding (flag << 32) | value bits,
// written and read whole, so a reader that sees the flag sees the matching value
// and no fence is needed between them (The CUDA Handbook, 13.3.4: the packed
// descriptor).  The value is bit-cast, not value-cast, so floats survive.
template <class T> struct PackedStatus {
  unsigned long long* w;
  __device__ __forceinline__ void publish(long long i, unsigned flag, T v) const {
    st_relaxed_u64(w + i, ((unsigned long long)flag << 32) | to_u32(v));
  }
  __device__ __forceinline__ unsigned poll(long long i, T& v) const {
    unsigned long long x = ld_relaxed_u64(w + i);
    v = from_u32<T>((unsigned)x);
    return (unsigned)(x >> 32);
  }
  __device__ __forceinline__ T fetch(long long, unsigned, T polled) const { return polled; }
};

// 8-byte (or wider) values: the two-word descriptor with an explicit fence that
// the same section names for 64-bit types.  The value goes to a slot of its own
// (aggregate and inclusive prefix have separate slots, so a reader that saw A can
// never pick up the later P value), then the flag is stored with release
// semantics; a reader loads the flag with acquire semantics before the value.
template <class T> struct SplitStatus {
  unsigned* flag;
  T* agg;
  T* pfx;
  __device__ __forceinline__ void publish(long long i, unsigned f, T v) const {
    st_relaxed(f == FLAG_A ? agg + i : pfx + i, v);
    st_release_u32(flag + i, f);
  }
  __device__ __forceinline__ unsigned poll(long long i, T&) const { return ld_acquire_u32(flag + i); }
  __device__ __forceinline__ T fetch(long long i, unsigned f, T) const {
    return ld_relaxed(f == FLAG_A ? agg + i : pfx + i);
  }
};

template <class T> struct StatusFor {
  using type = typename std::conditional<sizeof(T) == 4, PackedStatus<T>, SplitStatus<T>>::type;
};

// ---- decoupled look-back -------------------------------------------------------------

// Warp-cooperative look-back (The CUDA Handbook, 13.3.4, Figure 13-11), widened:
// lane l inspects the K predecessors frontier-K*l-i (i = 0..K-1, nearest first), so
// one round trip covers a window of 32*K tiles instead of 32.  A ballot finds the
// lane holding the nearest P; the values from the frontier back to that P are
// combined in tile order (earlier tiles on the left); with no P in the window all
// 32*K aggregates are combined and the warp steps back a whole window.  A tile only
// needs the part of its window up to the nearest P to be non-X.
//
// The window is read once; while it is not ready, only the entries that are still
// X and nearer than the nearest P are read again (an A or P already seen stays
// valid: an aggregate never changes, and any P is a correct inclusive prefix).  So
// a waiting warp costs the memory system a few words per poll, not its window:
// with hundreds of tiles resident per GPU, re-reading whole windows floods L2.
//
// `first` is the status index of tile 0 of this row (whose status is always P),
// `tt` >= 1 the tile's index within the row.  Called by all 32 lanes of one warp;
// returns the tile's exclusive prefix in every lane.  Every wait is bounded by
// wait_ns of global time; on expiry *timed_out is set and whatever was read is
// returned.
template <class T, int OP, int K, class S>
__device__ __forceinline__ T lookback_warp(const S& st, long long first, long long tt,
                                           unsigned long long wait_ns, bool& timed_out) {
  const int lane = threadIdx.x & 31;
  long long frontier = tt - 1;
  T acc{};
  bool have = false;
  timed_out = false;
  for (;;) {
    unsigned f[K];
    T v[K];
#pragma unroll
    for (int i = 0; i < K; ++i) {
      const long long p = frontier - (long long)K * lane - i;
      v[i] = T{};
      f[i] = (p >= 0) ? st.poll(first + p, v[i]) : FLAG_P;  // before the row: stops the walk
    }
    int fp = K;        // this lane's nearest P (K: none)
    int nearest = 32;  // lane holding the window's nearest P (32: none)
    int spins = 0;
    unsigned long long t0 = 0;
    for (;;) {
      fp = K;
#pragma unroll
      for (int i = K - 1; i >= 0; --i)
        if (f[i] == FLAG_P) fp = i;
      bool x_before_p = false, any_x = false;
#pragma unroll
      for (int i = 0; i < K; ++i)
        if (f[i] == FLAG_X) {
          any_x = true;
          if (i < fp) x_before_p = true;
        }
      const unsigned pm = __ballot_sync(0xffffffffu, fp < K);
      nearest = pm ? __ffs(pm) - 1 : 32;
      const bool bad = (lane < nearest && any_x) || (lane == nearest && x_before_p);
      if (!__any_sync(0xffffffffu, bad)) break;
      // The time-out decision is taken by the whole warp at once, so no lane leaves
      // the loop while others still poll (the ballots above need every lane).
      if (spins == 0) t0 = __shfl_sync(0xffffffffu, globaltimer(), 0);
      const bool late = spins > 0 && __shfl_sync(0xffffffffu, globaltimer(), 0) - t0 > wait_ns;
      if (late) {
        timed_out = true;
        break;
      }
      backoff(spins++);
      // Re-read only the blocking entries.
#pragma unroll
      for (int i = 0; i < K; ++i) {
        const bool needed = lane < nearest || (lane == nearest && i < fp);
        if (needed && f[i] == FLAG_X) {
          const long long p = frontier - (long long)K * lane - i;
          f[i] = (p >= 0) ? st.poll(first + p, v[i]) : FLAG_P;
        }
      }
    }
    // This lane's contribution: its tiles from its nearest P (or its farthest tile)
    // down to the nearest one, in tile order.
    const int m = lane == nearest ? fp : K - 1;
    T w{};
    if (lane <= nearest) {
#pragma unroll
      for (int i = K - 1; i >= 0; --i) {
        if (i <= m) {
          const long long p = frontier - (long long)K * lane - i;
          const T val = p >= 0 ? st.fetch(first + p, f[i], v[i]) : v[i];
          w = (i == m) ? val : Op<T, OP>::f(w, val);
        }
      }
    }
    // Ordered combination of lanes 0..min(nearest, 31) (lane k holds later tiles than k+1).
    const int last = nearest < 32 ? nearest : 31;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      T o = __shfl_down_sync(0xffffffffu, w, off);
      if (lane + off <= last) w = Op<T, OP>::f(o, w);
    }
    w = __shfl_sync(0xffffffffu, w, 0);
    acc = have ? Op<T, OP>::f(w, acc) : w;
    have = true;
    timed_out = __any_sync(0xffffffffu, timed_out);
    if (nearest < 32 || timed_out) break;
    frontier -= 32LL * K;
  }
  return acc;
}

// Per-lane look-back for lane-vector tiles: one thread walks back along one lane
// (column), reading D predecessors at a time; same protocol as lookback_warp.
// Status of (tile i, lane c) is at index i*CT + c.  `first` is the tile index of
// the chain's tile 0.
template <class T, int OP, int D, class S>
__device__ __forceinline__ T lookback_lane(const S& st, long long first, long long tt, int c, int CT,
                                           unsigned long long wait_ns, bool& timed_out) {
  long long f = tt - 1;
  T acc{};
  bool have = false;
  timed_out = false;
  for (;;) {
    unsigned fl[D];
    T v[D];
    int spins = 0;
    unsigned long long t0 = 0;
    for (;;) {
#pragma unroll
      for (int k = 0; k < D; ++k) {
        const long long p = f - k;
        v[k] = T{};
        fl[k] = p >= 0 ? st.poll((first + p) * CT + c, v[k]) : FLAG_P;
      }
      bool ready = true, seen_p = false;
#pragma unroll
      for (int k = 0; k < D; ++k) {
        if (!seen_p && fl[k] == FLAG_X) ready = false;
        if (fl[k] == FLAG_P) seen_p = true;
      }
      if (ready) break;
      if (spins == 0) {
        t0 = globaltimer();
      } else if (globaltimer() - t0 > wait_ns) {
        timed_out = true;
        break;
      }
      backoff(spins++);
    }
    int m = D - 1;
    bool found = false;
#pragma unroll
    for (int k = D - 1; k >= 0; --k)
      if (fl[k] == FLAG_P) {
        m = k;
        found = true;
      }
    T w{};
    bool hw = false;
#pragma unroll
    for (int k = D - 1; k >= 0; --k) {
      const long long p = f - k;
      if (k <= m && p >= 0) {
        T val = st.fetch((first + p) * CT + c, fl[k], v[k]);
        w = hw ? Op<T, OP>::f(w, val) : val;
        hw = true;
      }
    }
    if (hw) {
      acc = have ? Op<T, OP>::f(w, acc) : w;
      have = true;
    }
    if (found || timed_out) break;
    f -= D;
  }
  return acc;
}

// ---- the two passes over a tile in shared memory ------------------------------------

// Pass 1 over warp `warp`'s run: for each round j, pre[j] receives the combination
// of all of the warp's elements before lane `lane`'s vector (undefined for round 0,
// lane 0, which has none).  Returns the warp total (in every lane).
template <class T, int OP, int ROUNDS>
__device__ __forceinline__ T tile_reduce_pass(const uint4* run, int lane, T (&pre)[ROUNDS]) {
  constexpr int VEC = Vec<T>::N;
  T carry{};
#pragma unroll
  for (int j = 0; j < ROUNDS; ++j) {
    Vec<T> x = ld_vec<T>(run + j * 32 + lane);
    T t = x.v[0];
#pragma unroll
    for (int e = 1; e < VEC; ++e) t = Op<T, OP>::f(t, x.v[e]);
    const T wi = warp_inclusive<T, OP>(t, lane);
    const T we = __shfl_up_sync(0xffffffffu, wi, 1);
    const T rt = __shfl_sync(0xffffffffu, wi, 31);
    if (j == 0) {
      pre[0] = we;
      carry = rt;
    } else {
      pre[j] = lane == 0 ? carry : Op<T, OP>::f(carry, we);
      carry = Op<T, OP>::f(carry, rt);
    }
  }
  return carry;
}

// Pass 2: rewrite the warp's run in place with scanned values.  `base` (valid when
// has_base) is everything before the warp's run, already combined with the tile
// prefix and, for an exclusive scan, the initial value.
template <class T, int OP, int ROUNDS>
__device__ __forceinline__ void tile_apply_pass(uint4* run, int lane, const T (&pre)[ROUNDS], T base,
                                                bool has_base, bool inclusive) {
  constexpr int VEC = Vec<T>::N;
#pragma unroll
  for (int j = 0; j < ROUNDS; ++j) {
    Vec<T> x = ld_vec<T>(run + j * 32 + lane);
    T r;
    bool h;
    if (j > 0 || lane > 0) {
      r = has_base ? Op<T, OP>::f(base, pre[j]) : pre[j];
      h = true;
    } else {
      r = base;
      h = has_base;
    }
    Vec<T> y;
    if (inclusive) {
#pragma unroll
      for (int e = 0; e < VEC; ++e) {
        r = h ? Op<T, OP>::f(r, x.v[e]) : x.v[e];
        h = true;
        y.v[e] = r;
      }
    } else {  // exclusive: base always holds (the initial value at least)
#pragma unroll
      for (int e = 0; e < VEC; ++e) {
        y.v[e] = r;
        r = Op<T, OP>::f(r, x.v[e]);
      }
    }
    st_vec<T>(run + j * 32 + lane, y);
  }
}

// The same two passes on a tile held in registers: x[j] is the thread's 16-byte
// vector of round j (vector index (warp*ROUNDS + j)*32 + lane of the tile).
template <class T, int OP, int ROUNDS>
__device__ __forceinline__ T regs_reduce_pass(const Vec<T> (&x)[ROUNDS], int lane, T (&pre)[ROUNDS]) {
  constexpr int VEC = Vec<T>::N;
  T carry{};
#pragma unroll
  for (int j = 0; j < ROUNDS; ++j) {
    T t = x[j].v[0];
#pragma unroll
    for (int e = 1; e < VEC; ++e) t = Op<T, OP>::f(t, x[j].v[e]);
    const T wi = warp_inclusive<T, OP>(t, lane);
    const T we = __shfl_up_sync(0xffffffffu, wi, 1);
    const T rt = __shfl_sync(0xffffffffu, wi, 31);
    if (j == 0) {
      pre[0] = we;
      carry = rt;
    } else {
      pre[j] = lane == 0 ? carry : Op<T, OP>::f(carry, we);
      carry = Op<T, OP>::f(carry, rt);
    }
  }
  return carry;
}

template <class T, int OP, int ROUNDS>
__device__ __forceinline__ void regs_apply_pass(Vec<T> (&x)[ROUNDS], int lane, const T (&pre)[ROUNDS], T base,
                                                bool has_base, bool inclusive) {
  constexpr int VEC = Vec<T>::N;
#pragma unroll
  for (int j = 0; j < ROUNDS; ++j) {
    T r;
    bool h;
    if (j > 0 || lane > 0) {
      r = has_base ? Op<T, OP>::f(base, pre[j]) : pre[j];
      h = true;
    } else {
      r = base;
      h = has_base;
    }
    if (inclusive) {
#pragma unroll
      for (int e = 0; e < VEC; ++e) {
        r = h ? Op<T, OP>::f(r, x[j].v[e]) : x[j].v[e];
        h = true;
        x[j].v[e] = r;
      }
    } else {
#pragma unroll
      for (int e = 0; e < VEC; ++e) {
        const T xv = x[j].v[e];
        x[j].v[e] = r;
        r = Op<T, OP>::f(r, xv);
      }
    }
  }
}

// ---- thread-contiguous chunks (for operators that are costly per element) ------------

// Each thread owns CV consecutive 16-byte vectors of the tile (its "chunk").  A warp
// reading vector k of every lane's chunk would hit one bank group 8 times over, so
// lane l reads its vectors in the rotated order (j + l) mod CV: conflict-free.  The
// rotation is undone in registers with log2(CV) select stages before the ordered
// scan, and redone before the write-back.  Costs a few integer selects per element
// and saves the warp scans: one warp scan per CV*VEC elements instead of per VEC.
template <class T, int CV>
__device__ __forceinline__ void chunk_load(const uint4* chunk, int lane, Vec<T> (&v)[CV]) {
#pragma unroll
  for (int j = 0; j < CV; ++j) v[j] = ld_vec<T>(chunk + ((j + lane) & (CV - 1)));
}
template <class T, int CV>
__device__ __forceinline__ void chunk_store(uint4* chunk, int lane, const Vec<T> (&v)[CV]) {
#pragma unroll
  for (int j = 0; j < CV; ++j) st_vec<T>(chunk + ((j + lane) & (CV - 1)), v[j]);
}
// w[k] = v[(k - rot) mod CV] (dir = -1) or v[(k + rot) mod CV] (dir = +1).
template <class T, int CV, int DIR>
__device__ __forceinline__ void chunk_rotate(Vec<T> (&v)[CV], int rot) {
#pragma unroll
  for (int s = 1; s < CV; s <<= 1) {
    const bool b = (rot & s) != 0;
    Vec<T> t[CV];
#pragma unroll
    for (int k = 0; k < CV; ++k) {
      const Vec<T>& src = v[(k + DIR * s + CV) & (CV - 1)];
#pragma unroll
      for (int e = 0; e < Vec<T>::N; ++e) t[k].v[e] = b ? src.v[e] : v[k].v[e];
    }
#pragma unroll
    for (int k = 0; k < CV; ++k) v[k] = t[k];
  }
}

// Block scan of the NW warp totals by warp 0 (The CUDA Handbook, 13.3.1, Listing
// 13-5, with one shared slot per warp as in AcceleratedKernels.jl PR #208): on
// return s_warp[w] holds the inclusive total of warps 0..w; returns the tile
// aggregate in every lane of warp 0.
template <class T, int OP, int NW>
__device__ __forceinline__ T block_scan_warp_totals(T* s_warp, int lane) {
  T w = s_warp[lane < NW ? lane : NW - 1];
  w = warp_inclusive<T, OP>(w, lane);
  if (lane < NW) s_warp[lane] = w;
  return __shfl_sync(0xffffffffu, w, NW - 1);
}

}  // namespace gbs
