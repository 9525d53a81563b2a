// scan_lanes_rts.cuh -- reduce-then-scan for elements of C 8-byte lanes (The CUDA
// Handbook, 13.3.3, Figure 13-10; B. Merry, "Prefix sums on GPUs", slide "Fixed Block
// Count"), for arrays that fit in L2 and few long chains: three launches, no CTA ever
// waits for another.
//
// Tiles are the lane kernel's (RT rows x CT lanes; thread (lane c, group g) owns RPG
// consecutive rows of lane c), 32 KB here.  A range is TPR consecutive tiles of one
// chain (batch x lane strip); there are about as many ranges as CTAs that fit on the
// GPU at once.
//   1. reduce: one CTA per range streams its tiles through shared memory (bulk
//      copies with an L2 evict-last hint, two tiles in flight) and writes the
//      range's CT lane aggregates;
//   2. spine: one CTA per chain turns its ranges' aggregates into exclusive range
//      prefixes per lane, in place;
//   3. scan: one CTA per range streams its tiles again (now from L2, evict-first),
//      scans each tile from the range prefix carried lane by lane, and writes it.
// Why only 8-byte lanes: the single-pass lane kernel publishes an 8-byte lane's
// status as a flag and a value in separate words, so each step of its per-lane
// look-back costs two dependent round trips (about 75 ns a tile, measured), and a
// chain of thousands of tiles bounds it; 4-byte lanes pack flag and value in one
// word (about 16 ns a tile), and there the single pass is faster than three launches
// (96-byte structs 1e6: 51 against 64 us).  fp64 adds bound the fp64 case (about 500
// G/s on this GPU): the reduce keeps each tile's group partials so that the scan adds
// every element once, two fp64 adds per element in all.
#pragma once

#include "launch.h"
#include "scan_lanes.cuh"
#include "tile.cuh"

namespace gbs {

template <class T> struct LanesRtsArgs {
  const T* in;
  T* out;
  long long R, C;            // positions per chain, lanes per position
  int CT, G, RT;             // strip width, row groups, rows per tile (= G * RPG)
  unsigned strips;           // ceil(C / CT)
  unsigned tiles_per_chain;  // ceil(R / RT)
  unsigned tpr;              // tiles per range
  unsigned K;                // ranges per chain: ceil(tiles_per_chain / tpr)
  T* agg;                    // [chains][K][CT]: range aggregates, then exclusive prefixes
  const T* init;             // device copy of the initial values (exclusive)
  int init_lanes;            // lane c starts from init[c % init_lanes]
  int inclusive;
  ErrSink err;
  unsigned long long wait_ns;
  T* gp;                     // [tiles][G][CT]: group partials (fp64), else null
};

template <class T> __host__ __device__ constexpr bool lanes_rts_keeps_groups() {
  return std::is_same<T, double>::value;
}

// 32 KB tiles (16 rows per thread of 8-byte lanes), two per CTA.
template <class T> using LanesRtsGeom = LanesGeomT<T, 16>;

// Spine: ranges per thread, held in registers.  A chain has at most (1024 / CT) * U
// ranges (the plan raises TPR until it does).
template <class T> __host__ __device__ constexpr int lanes_spine_u() { return sizeof(T) == 8 ? 8 : 16; }

__device__ __forceinline__ void bulk_s2g_hint(void* gdst, const void* smem_src, unsigned bytes,
                                              unsigned long long pol) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group.L2::cache_hint [%0], [%1], %2, %3;" ::"l"(gdst),
               "r"(smem_u32(smem_src)), "r"(bytes), "l"(pol)
               : "memory");
}

// Tile tt of chain `chain`: where its rows sit and how many there are.
struct LanesTileAt {
  long long gbase;  // element offset of the tile's first row, first lane of the strip
  long long c0;     // the strip's first lane
  int rows, cols;
};
template <class T>
__device__ __forceinline__ LanesTileAt lanes_tile_at(const LanesRtsArgs<T>& a, unsigned chain, unsigned tt) {
  LanesTileAt w;
  const unsigned b = chain / a.strips, strip = chain - b * a.strips;
  const long long r0 = (long long)tt * a.RT;
  w.rows = a.R - r0 >= a.RT ? a.RT : (int)(a.R - r0);
  w.c0 = (long long)strip * a.CT;
  w.cols = a.C - w.c0 >= a.CT ? a.CT : (int)(a.C - w.c0);
  w.gbase = ((long long)b * a.R + r0) * a.C + w.c0;
  return w;
}

// Can tile w move by bulk copies?  Whole rows (CT == C): one contiguous copy; a strip:
// one copy per row.  `out` is null when only the load matters.
template <class T>
__device__ __forceinline__ bool lanes_tile_bulk(const LanesRtsArgs<T>& a, const LanesTileAt& w, const T* out) {
  const size_t rbytes = (size_t)w.cols * sizeof(T);
  bool blk = aligned16(a.in + w.gbase) && (out == nullptr || aligned16(out + w.gbase));
  if (w.cols == a.C) blk = blk && ((size_t)w.rows * rbytes) % 16 == 0;
  else blk = blk && rbytes % 16 == 0 && ((size_t)a.C * sizeof(T)) % 16 == 0 && ((size_t)a.CT * sizeof(T)) % 16 == 0;
  return blk;
}

// ---- two-stage tile pipeline: tile i of a range sits in buffer i & 1; the copy of
// tile i + 2 starts as soon as tile i has been consumed.

// Thread 0 arms buffer q's barrier for tile tt, if that tile moves by bulk copy.
template <class T>
__device__ __forceinline__ void lanes_stage_arm(const LanesRtsArgs<T>& a, unsigned chain, unsigned tt, unsigned t1,
                                                const T* out, unsigned long long* bar) {
  if (threadIdx.x == 0 && tt < t1) {
    const LanesTileAt w = lanes_tile_at(a, chain, tt);
    if (lanes_tile_bulk(a, w, out)) mbar_arrive_expect_tx(bar, (unsigned)(w.rows * w.cols * sizeof(T)));
  }
}
// Issue tile tt's bulk copies into buf (after the block barrier that follows the arm).
template <class T, int NT>
__device__ __forceinline__ void lanes_stage_issue(const LanesRtsArgs<T>& a, unsigned chain, unsigned tt, unsigned t1,
                                                  const T* out, T* buf, unsigned long long* bar,
                                                  unsigned long long pol) {
  if (tt >= t1) return;
  const LanesTileAt w = lanes_tile_at(a, chain, tt);
  if (!lanes_tile_bulk(a, w, out)) return;
  const T* src = a.in + w.gbase;
  const unsigned rbytes = (unsigned)(w.cols * sizeof(T));
  if (w.cols == a.C) {
    if (threadIdx.x == 0) bulk_g2s_hint(buf, src, (unsigned)w.rows * rbytes, bar, pol);
  } else {
    for (int r = threadIdx.x; r < w.rows; r += NT) bulk_g2s_hint(buf + r * a.CT, src + r * a.C, rbytes, bar, pol);
  }
}
// Wait for tile w in buffer q (or load it with plain loads if it does not move by
// bulk copy).  false on every thread if the copy did not land in time.
template <class T, int NT>
__device__ __forceinline__ bool lanes_stage_wait(const LanesRtsArgs<T>& a, const LanesTileAt& w, bool bulk, T* buf,
                                                 unsigned long long* bar, unsigned& phases, int q) {
  bool failed = false;
  if (bulk) {
    failed = !mbar_wait(bar, (phases >> q) & 1u, a.wait_ns);
    phases ^= 1u << q;
  } else {
    const T* src = a.in + w.gbase;
    for (int k = threadIdx.x; k < w.rows * w.cols; k += NT) {
      const int r = k / w.cols, c = k - r * w.cols;
      buf[r * a.CT + c] = src[(long long)r * a.C + c];
    }
  }
  return !__syncthreads_or(failed);
}
// After a copy timed out: record it, and give the copies still in flight into both
// buffers (tiles tt and tt + 1) a bounded time to land before the CTA exits.
template <class T>
__device__ __forceinline__ void lanes_stage_abort(const LanesRtsArgs<T>& a, unsigned chain, unsigned tt, unsigned t1,
                                                  const T* out, unsigned long long* bars, unsigned phases, int q) {
  if (threadIdx.x != 0) return;
  raise_err(a.err, ERRBIT_TIMEOUT);
  mbar_wait(&bars[q], ((phases >> q) & 1u) ^ 1u, a.wait_ns);  // the phase that did not complete
  if (tt + 1 < t1 && lanes_tile_bulk(a, lanes_tile_at(a, chain, tt + 1), out))
    mbar_wait(&bars[q ^ 1], (phases >> (q ^ 1)) & 1u, a.wait_ns);
}

template <class T, int OP, class Gm>
__global__ void __launch_bounds__(Gm::NT, 3) lanes_rts_reduce_kernel(LanesRtsArgs<T> a) {
  pdl_entry();
  constexpr int NT = Gm::NT, RPG = Gm::RPG;
  __shared__ __align__(128) T s_tile[2][NT * RPG];
  __shared__ T s_gx[NT];
  __shared__ __align__(8) unsigned long long s_bar[2];
  const int tid = threadIdx.x, CT = a.CT, c = tid % CT, g = tid / CT;
  const unsigned chain = blockIdx.x / a.K, k = blockIdx.x - chain * a.K;
  const unsigned t0 = k * a.tpr, t1 = t0 + a.tpr < a.tiles_per_chain ? t0 + a.tpr : a.tiles_per_chain;
  const unsigned long long keep = l2_policy_evict_last();
  const T* none = nullptr;
  if (tid == 0) {
    mbar_init(&s_bar[0], 1);
    mbar_init(&s_bar[1], 1);
    fence_mbar_init();
  }
  lanes_stage_arm(a, chain, t0, t1, none, &s_bar[0]);
  lanes_stage_arm(a, chain, t0 + 1, t1, none, &s_bar[1]);
  __syncthreads();
  lanes_stage_issue<T, NT>(a, chain, t0, t1, none, s_tile[0], &s_bar[0], keep);
  lanes_stage_issue<T, NT>(a, chain, t0 + 1, t1, none, s_tile[1], &s_bar[1], keep);
  T acc{};
  bool has = false;
  unsigned phases = 0;
  for (unsigned tt = t0; tt < t1; ++tt) {
    const int q = (tt - t0) & 1;
    const LanesTileAt w = lanes_tile_at(a, chain, tt);
    if (!lanes_stage_wait<T, NT>(a, w, lanes_tile_bulk(a, w, none), s_tile[q], &s_bar[q], phases, q)) {
      lanes_stage_abort(a, chain, tt, t1, none, s_bar, phases, q);
      return;
    }
    const T* tile = s_tile[q];
    const int rb = g * RPG, re = rb + RPG < w.rows ? rb + RPG : w.rows;
    if (g < a.G && c < w.cols && rb < w.rows) {
      T p = tile[rb * CT + c];
      for (int r = rb + 1; r < re; ++r) p = Op<T, OP>::f(p, tile[r * CT + c]);
      if constexpr (lanes_rts_keeps_groups<T>())
        a.gp[(((size_t)chain * a.tiles_per_chain + tt) * a.G + g) * CT + c] = p;
      acc = has ? Op<T, OP>::f(acc, p) : p;
      has = true;
    }
    lanes_stage_arm(a, chain, tt + 2, t1, none, &s_bar[q]);
    __syncthreads();  // buffer q is free
    lanes_stage_issue<T, NT>(a, chain, tt + 2, t1, none, s_tile[q], &s_bar[q], keep);
  }
  if (has) s_gx[g * CT + c] = acc;
  __syncthreads();
  const LanesTileAt w0 = lanes_tile_at(a, chain, t0);
  if (tid < w0.cols) {  // the groups in order (a group that holds rows holds them in the first tile)
    const int ngroups = (w0.rows + RPG - 1) / RPG;
    T v = s_gx[tid];
    for (int gg = 1; gg < ngroups; ++gg) v = Op<T, OP>::f(v, s_gx[gg * CT + tid]);
    a.agg[((size_t)chain * a.K + k) * CT + tid] = v;
  }
}

// One CTA per lane of each chain: the exclusive range prefixes of that lane, in place.
// Thread j holds the j-th of J = min(K, 1024) contiguous parts of the K ranges (at most
// U of them) in registers and folds them; the part totals are scanned by warp shuffles
// and one warp over the warp totals; each thread writes its running prefixes back.
// Range 0's entry is left as it is (it has no prefix).  Spreading the lanes over CTAs
// keeps the fp64 adds of a long chain off a single SM (one SM adds about 1.7 doubles a
// clock: 417 ranges x 17 lanes took 10-12 us on one CTA).
template <class T, int OP>
__global__ void __launch_bounds__(1024) lanes_rts_spine_kernel(LanesRtsArgs<T> a) {
  pdl_entry();
  constexpr int U = lanes_spine_u<T>();
  __shared__ T s_w[32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, CT = a.CT;
  const unsigned K = a.K, chain = blockIdx.x / CT;
  const int c = (int)(blockIdx.x - chain * CT);
  const unsigned strip = chain % a.strips;
  if ((long long)strip * CT + c >= a.C) return;  // a lane past C (the CTA leaves as one)
  const unsigned J = K < 1024u ? K : 1024u;
  const bool part = (unsigned)tid < J;  // the parts are threads 0 .. J-1: later threads never reach them
  const unsigned pb = part ? (unsigned)((unsigned long long)tid * K / J) : 0u;
  const unsigned pe = part ? (unsigned)((unsigned long long)(tid + 1) * K / J) : 0u;  // 0 < pe - pb <= U
  T* mine = a.agg + ((size_t)chain * K + pb) * CT + c;
  const int cnt = (int)(pe - pb);
  T v[U] = {};
#pragma unroll
  for (int q = 0; q < U; ++q)
    if (q < cnt) v[q] = mine[(size_t)q * CT];
  T acc = v[0];  // unused past J: scans only pull from lower threads
#pragma unroll
  for (int q = 1; q < U; ++q)
    if (q < cnt) acc = Op<T, OP>::f(acc, v[q]);
  const T inc = warp_inclusive<T, OP>(acc, lane);
  if (lane == 31) s_w[warp] = inc;
  __syncthreads();
  if (warp == 0) s_w[lane] = warp_inclusive<T, OP>(s_w[lane], lane);
  __syncthreads();
  const T below = __shfl_up_sync(0xffffffffu, inc, 1);  // the parts before this one in the warp
  if (part && tid > 0) {
    T run;
    if (warp == 0) run = below;
    else run = lane == 0 ? s_w[warp - 1] : Op<T, OP>::f(s_w[warp - 1], below);
#pragma unroll
    for (int q = 0; q < U; ++q) {
      if (q < cnt) {
        mine[(size_t)q * CT] = run;  // the prefix of range pb + q
        run = Op<T, OP>::f(run, v[q]);
      }
    }
  } else if (part) {  // thread 0: range 0 keeps its aggregate, the rest of its part gets prefixes
    T run = v[0];
#pragma unroll
    for (int q = 1; q < U; ++q) {
      if (q < cnt) {
        mine[(size_t)q * CT] = run;
        run = Op<T, OP>::f(run, v[q]);
      }
    }
  }
}

template <class T, int OP, class Gm>
__global__ void __launch_bounds__(Gm::NT, 3) lanes_rts_scan_kernel(LanesRtsArgs<T> a) {
  pdl_entry();
  constexpr int NT = Gm::NT, NW = Gm::NW, RPG = Gm::RPG;
  __shared__ __align__(128) T s_tile[2][NT * RPG];
  __shared__ T s_gx[NT];    // group totals, then exclusive group prefixes, [g*CT + c]
  __shared__ T s_pfx[NT];   // per lane: the prefix carried into the current tile
  __shared__ T s_agg[NT];   // per lane: the current tile's aggregate
  __shared__ __align__(8) unsigned long long s_bar[2];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int CT = a.CT, c = tid % CT, g = tid / CT;
  const unsigned chain = blockIdx.x / a.K, k = blockIdx.x - chain * a.K;
  const unsigned t0 = k * a.tpr, t1 = t0 + a.tpr < a.tiles_per_chain ? t0 + a.tpr : a.tiles_per_chain;
  const unsigned long long drop = l2_policy_evict_first();
  const T* out = a.out;
  // The carried prefix: the initial value, then the range's exclusive prefix.
  bool has = k > 0 || !a.inclusive;
  {
    const LanesTileAt w = lanes_tile_at(a, chain, t0);
    if (tid < w.cols) {
      T p = k > 0 ? a.agg[((size_t)chain * a.K + k) * CT + tid] : T{};
      if (!a.inclusive) {
        const T i0 = a.init[(w.c0 + tid) % a.init_lanes];
        p = k > 0 ? Op<T, OP>::f(i0, p) : i0;
      }
      s_pfx[tid] = p;
    }
  }
  if (tid == 0) {
    mbar_init(&s_bar[0], 1);
    mbar_init(&s_bar[1], 1);
    fence_mbar_init();
  }
  lanes_stage_arm(a, chain, t0, t1, out, &s_bar[0]);
  lanes_stage_arm(a, chain, t0 + 1, t1, out, &s_bar[1]);
  __syncthreads();
  lanes_stage_issue<T, NT>(a, chain, t0, t1, out, s_tile[0], &s_bar[0], drop);
  lanes_stage_issue<T, NT>(a, chain, t0 + 1, t1, out, s_tile[1], &s_bar[1], drop);
  unsigned phases = 0;
  for (unsigned tt = t0; tt < t1; ++tt) {
    const int q = (tt - t0) & 1;
    T* tile = s_tile[q];
    const LanesTileAt w = lanes_tile_at(a, chain, tt);
    const bool bulk = lanes_tile_bulk(a, w, out);
    const int rb = g * RPG, re = rb + RPG < w.rows ? rb + RPG : w.rows;
    const bool active = g < a.G && c < w.cols && rb < w.rows;
    T gpart{};
    if constexpr (lanes_rts_keeps_groups<T>())  // fetched while the tile is in flight
      if (active) gpart = a.gp[(((size_t)chain * a.tiles_per_chain + tt) * a.G + g) * CT + c];
    if (!lanes_stage_wait<T, NT>(a, w, bulk, tile, &s_bar[q], phases, q)) {
      lanes_stage_abort(a, chain, tt, t1, out, s_bar, phases, q);
      return;
    }

    // Pass 1: each (lane c, group g) combines its RPG rows (fp64: kept by the reduce).
    if (active) {
      if constexpr (lanes_rts_keeps_groups<T>()) {
        s_gx[g * CT + c] = gpart;
      } else {
        T p = tile[rb * CT + c];
        for (int r = rb + 1; r < re; ++r) p = Op<T, OP>::f(p, tile[r * CT + c]);
        s_gx[g * CT + c] = p;
      }
    }
    __syncthreads();
    // Exclusive scan of each lane's group totals.  fp64: one thread per lane, serially
    // (G - 1 adds a lane; a warp-wide scan costs 5 x 32); else one warp per lane.
    const int ngroups = (w.rows + RPG - 1) / RPG;
    if constexpr (lanes_rts_keeps_groups<T>()) {
      if (tid < w.cols) {
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
        s_agg[tid] = run;
      }
    } else {
      for (int cc = warp; cc < w.cols; cc += NW) {
        const T v = s_gx[(lane < ngroups ? lane : ngroups - 1) * CT + cc];
        const T inc = warp_inclusive<T, OP>(v, lane);
        const T exc = __shfl_up_sync(0xffffffffu, inc, 1);
        const T tot = __shfl_sync(0xffffffffu, inc, ngroups - 1);
        __syncwarp();
        if (lane < ngroups && lane > 0) s_gx[lane * CT + cc] = exc;
        if (lane == 0) s_agg[cc] = tot;
      }
    }
    __syncthreads();
    // Pass 2: rewrite the rows in place from the carried prefix.
    if (active) {
      bool h = has;
      T base = s_pfx[c];
      if (g > 0) {
        const T gx = s_gx[g * CT + c];
        base = h ? Op<T, OP>::f(base, gx) : gx;
        h = true;
      }
      if (a.inclusive) {
        for (int r = rb; r < re; ++r) {
          const T x = tile[r * CT + c];
          base = h ? Op<T, OP>::f(base, x) : x;
          h = true;
          tile[r * CT + c] = base;
        }
      } else {
        for (int r = rb; r < re; ++r) {
          const T x = tile[r * CT + c];
          tile[r * CT + c] = base;
          base = Op<T, OP>::f(base, x);
        }
      }
    }
    if (bulk) fence_proxy_async_smem();
    __syncthreads();  // every thread has read s_pfx; the rows are final
    if (tid < w.cols) s_pfx[tid] = has ? Op<T, OP>::f(s_pfx[tid], s_agg[tid]) : s_agg[tid];
    has = true;

    T* dst = a.out + w.gbase;
    if (bulk) {
      const unsigned rbytes = (unsigned)(w.cols * sizeof(T));
      if (w.cols == a.C) {
        if (tid == 0) {
          bulk_s2g_hint(dst, tile, (unsigned)w.rows * rbytes, drop);
          bulk_commit();
        }
      } else {
        for (int r = tid; r < w.rows; r += NT) {
          bulk_s2g_hint(dst + r * a.C, tile + r * CT, rbytes, drop);
          bulk_commit();
        }
      }
      bulk_wait_read_all();
    } else {
      for (int qq = tid; qq < w.rows * w.cols; qq += NT) {
        const int r = qq / w.cols, cc = qq - r * w.cols;
        dst[(long long)r * a.C + cc] = tile[r * CT + cc];
      }
    }
    lanes_stage_arm(a, chain, tt + 2, t1, out, &s_bar[q]);
    __syncthreads();  // buffer q is free; s_pfx holds the new prefix
    lanes_stage_issue<T, NT>(a, chain, tt + 2, t1, out, s_tile[q], &s_bar[q], drop);
  }
}

// The path runs for 8-byte lanes whose array fits in L2 (the rows stay there from
// the reduce to the scan), in at most 4 chains of at least 128 of the lane kernel's
// tiles.  17-lane fp64 duals, 1e6 in one chain (2084 tiles): 118 us against 154 us for
// the lane kernel; 3 chains of 1e5 (209 tiles each): 49 against 60 us; 1000 x 1e4 fp64
// columns, 313 chains of 4 tiles: 105 against 72 us, where the look-back has nothing
// to wait for.
constexpr long long kLanesRtsMaxBytes = 160ll << 20;

template <class T> bool lanes_rts_applies(long long B, long long R, long long C) {
  if (sizeof(T) != 8 || C <= 1 || B * R * C * (long long)sizeof(T) > kLanesRtsMaxBytes) return false;
  const LanesPlan<T> lb = lanes_plan<T>(B, R, C);
  return lb.num_tiles / lb.tiles_per_chain <= 4 && lb.tiles_per_chain >= 128;
}

template <class T, class Gm = LanesRtsGeom<T>> struct LanesRtsPlan {
  LanesPlan<T, Gm> t;
  unsigned tpr, K, chains;
};

// Ranges per chain never exceed this (the spine holds them in registers).
template <class T, class Gm> long long lanes_rts_max_ranges(const LanesPlan<T, Gm>& t) {
  const long long cap = (long long)(1024 / t.CT) * lanes_spine_u<T>();
  return (long long)t.tiles_per_chain < cap ? (long long)t.tiles_per_chain : cap;
}

// CTAs of the reduce and scan kernels that fit on one SM at once (queried once).
template <class T, int OP, class Gm> int lanes_rts_ctas_per_sm() {
  static int cached = 0;
  if (cached == 0) {
    int r = 0, s = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&r, lanes_rts_reduce_kernel<T, OP, Gm>, Gm::NT, 0) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&s, lanes_rts_scan_kernel<T, OP, Gm>, Gm::NT, 0) != cudaSuccess)
      return 1;
    cached = r < s ? r : s;
    if (cached < 1) cached = 1;
  }
  return cached;
}

template <class T, class Gm = LanesRtsGeom<T>>
LanesRtsPlan<T, Gm> lanes_rts_plan(long long B, long long R, long long C, int num_sms, int ctas_per_sm) {
  LanesRtsPlan<T, Gm> p;
  p.t = lanes_plan<T, Gm>(B, R, C);
  p.chains = p.t.num_tiles / p.t.tiles_per_chain;
  // About one range per CTA slot, so that every range runs in the first wave.
  const long long slots = (long long)(num_sms > 0 ? num_sms : 1) * (ctas_per_sm > 0 ? ctas_per_sm : 1);
  long long tpr = ((long long)p.t.num_tiles + slots - 1) / slots;
  const long long maxk = lanes_rts_max_ranges(p.t);
  const long long tmin = ((long long)p.t.tiles_per_chain + maxk - 1) / maxk;
  if (tpr < tmin) tpr = tmin;
  p.tpr = (unsigned)tpr;
  p.K = (unsigned)(((long long)p.t.tiles_per_chain + tpr - 1) / tpr);
  return p;
}

// Layout after the header: [init: up to 4096 lanes][range aggregates][group partials
// (fp64)].  The aggregates are sized for the most ranges any SM count gives.
template <class T, class Gm> size_t lanes_rts_agg_bytes(const LanesPlan<T, Gm>& t) {
  const size_t chains = t.num_tiles / t.tiles_per_chain;
  return round_up(chains * (size_t)lanes_rts_max_ranges(t) * t.CT * sizeof(T), 256);
}
template <class T, class Gm> size_t lanes_rts_gp_bytes(const LanesPlan<T, Gm>& t) {
  return lanes_rts_keeps_groups<T>() ? round_up((size_t)t.num_tiles * t.G * t.CT * sizeof(T), 256) : 0;
}
template <class T, class Gm = LanesRtsGeom<T>> size_t lanes_rts_temp_bytes(long long B, long long R, long long C) {
  const LanesPlan<T, Gm> t = lanes_plan<T, Gm>(B, R, C);
  return kHeaderBytes + lanes_init_bytes<T>(C) + lanes_rts_agg_bytes(t) + lanes_rts_gp_bytes(t);
}

template <class T, int OP, class Gm = LanesRtsGeom<T>>
cudaError_t launch_lanes_rts_op(const ScanJob& job, const LaunchCtx& ctx) {
  const LanesRtsPlan<T, Gm> p =
      lanes_rts_plan<T, Gm>(job.B, job.R, job.C, ctx.num_sms, lanes_rts_ctas_per_sm<T, OP, Gm>());
  LanesRtsArgs<T> a;
  a.in = (const T*)job.in;
  a.out = (T*)job.out;
  a.R = job.R;
  a.C = job.C;
  a.CT = p.t.CT;
  a.G = p.t.G;
  a.RT = p.t.RT;
  a.strips = p.t.strips;
  a.tiles_per_chain = p.t.tiles_per_chain;
  a.tpr = p.tpr;
  a.K = p.K;
  char* init_area = (char*)job.temp + kHeaderBytes;
  a.init = (const T*)init_area;
  a.agg = (T*)(init_area + lanes_init_bytes<T>(job.C));
  a.gp = lanes_rts_keeps_groups<T>() ? (T*)((char*)a.agg + lanes_rts_agg_bytes(p.t)) : nullptr;
  a.init_lanes = job.init_lanes;
  a.inclusive = job.inclusive;
  a.err = ctx.err;
  a.wait_ns = ctx.wait_ns;
  const unsigned ranges = p.chains * p.K;
  profile_before(ctx);
  cudaError_t e = clear_status(job.temp, kHeaderBytes, nullptr, 0, ctx);  // the call's error word
  if (e == cudaSuccess && !job.inclusive)
    e = cudaMemcpyAsync(init_area, job.init_host, (size_t)job.init_lanes * sizeof(T), cudaMemcpyHostToDevice,
                        ctx.stream);
  if (e == cudaSuccess) e = launch_pdl(lanes_rts_reduce_kernel<T, OP, Gm>, ranges, Gm::NT, 0, ctx.stream, a);
  if (e == cudaSuccess) e = launch_pdl(lanes_rts_spine_kernel<T, OP>, p.chains * p.t.CT, 1024, 0, ctx.stream, a);
  if (e == cudaSuccess) e = launch_pdl(lanes_rts_scan_kernel<T, OP, Gm>, ranges, Gm::NT, 0, ctx.stream, a);
  profile_after(ctx);
  return e;
}

}  // namespace gbs
