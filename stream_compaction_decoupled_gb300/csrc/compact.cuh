// compact.cuh -- single-pass stable stream compaction: count, scan, scatter in one
// kernel (B. Merry, "Prefix sums on GPUs", slides "Solution" and "Other
// Applications"; the counts are scanned with the decoupled look-back of The CUDA
// Handbook, 13.3.4).
//
// Per tile (same geometry and claiming as the row scan):
//   1. bulk-copy the tile of inputs into shared memory;
//   2. each (round, lane) evaluates the predicate on its 16-byte vector; one ballot
//      per vector slot gives every element its rank inside the warp's round, and
//      the popcounts give the round totals (no shuffles needed for 0/1 flags);
//   3. block scan of the per-warp counts, look-back over packed (flag, count)
//      words -> the tile's output offset;
//   4. selected indices are staged in shared memory at their rank and written out
//      contiguously, so the global stores are coalesced;
//   5. the last tile writes the total count.
#pragma once

#include "launch.h"
#include "scan_rows.cuh"
#include "scan_seg.cuh"

namespace gbs {

template <class T> struct CompactArgs {
  const T* in;
  long long n;
  unsigned num_tiles;
  T thr;
  unsigned predmask;  // bit0: select x < t, bit1: x == t, bit2: x > t, bit3: unordered
  int* out_idx;
  int* out_count;
  unsigned* counter;
  ErrSink err;
  int bulk_ok;
  unsigned long long wait_ns;
  long long stalled_tile;
};

template <class T> __device__ __forceinline__ bool selects(T x, T t, unsigned mask) {
  const unsigned cls = x < t ? 1u : (x == t ? 2u : (x > t ? 4u : 8u));
  return (mask & cls) != 0;
}

// The same predicates fixed at compile time (LT LE GT GE EQ NE, the order of the C
// ABI's GB_LT..GB_NE): one comparison each.  A NaN x selects only under NE, as the
// class mask above gives (unordered is in NE's mask only).
template <int PRED, class T> __device__ __forceinline__ bool select_pred(T x, T t) {
  if constexpr (PRED == 0) return x < t;
  else if constexpr (PRED == 1) return x <= t;
  else if constexpr (PRED == 2) return x > t;
  else if constexpr (PRED == 3) return x >= t;
  else if constexpr (PRED == 4) return x == t;
  else if constexpr (PRED == 5) return !(x == t);
  else {  // 6, integers only: bit t of x is clear (the one-bit split)
    using U = typename std::make_unsigned<T>::type;
    return (((U)x >> (unsigned)t) & 1u) == 0;
  }
}

// Phase 1 of the selection segment kernels (compaction, partition): how many
// elements of the warp's chunks [c0, c1) satisfy PRED.  Coalesced 16-byte vectors,
// U per lane in flight, loaded with the L2 evict-last hint so that phase 3 finds
// them; the ragged end element by element.  Elements before d (a partition's
// unaligned head, read from the aligned base below the input) do not count; they
// can only sit in the base's first vector.  Returns this lane's share.
template <class T, int PRED, class G>
__device__ __forceinline__ unsigned count_selected(const T* in, long long n, long long c0, long long c1, T thr,
                                                   long long d, int lane) {
  constexpr int VEC = G::VEC, CH = G::CH, U = 8;
  const unsigned long long keep = l2_policy_evict_last();
  const long long e1 = c1 * CH < n ? c1 * CH : n;
  const long long v1 = e1 / VEC;
  const uint4* p = reinterpret_cast<const uint4*>(in);
  long long v = c0 * CH / VEC + lane;
  unsigned cnt = 0;
  if (d > 0 && v < 32 && v < v1) {  // the base's first vector may hold masked elements
    Vec<T> x;
    const uint4 u = ld_hint(p + v, keep);
    memcpy(x.v, &u, 16);
#pragma unroll
    for (int e = 0; e < VEC; ++e) cnt += (v * VEC + e >= d && select_pred<PRED>(x.v[e], thr)) ? 1u : 0u;
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
      for (int e = 0; e < VEC; ++e) cnt += select_pred<PRED>(x.v[e], thr) ? 1u : 0u;
    }
  }
  if (v < v1) {  // the rest in one guarded round
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
        for (int e = 0; e < VEC; ++e) cnt += select_pred<PRED>(x.v[e], thr) ? 1u : 0u;
      }
  }
  if (lane == 0)
    for (long long i = v1 * VEC; i < e1; ++i) cnt += (i >= d && select_pred<PRED>(in[i], thr)) ? 1u : 0u;
  return cnt;
}

// Nine tiles per SM (56 registers a thread): the selection bits, the tile's place and
// the look-back's state then stay in registers.
constexpr int kCompactTileMinBlocks = 9;

template <class T>
__global__ void __launch_bounds__(RowsGeom<T>::NT, kCompactTileMinBlocks) compact_kernel(CompactArgs<T> a, PackedStatus<unsigned> st) {
  pdl_entry();
  using G = RowsGeom<T>;
  constexpr int NT = G::NT, NW = G::NW, ROUNDS = G::ROUNDS, VEC = G::VEC, TILE = G::TILE;
  static_assert(ROUNDS * VEC <= 32, "selection bits must fit one word");
  __shared__ __align__(128) T s_tile[TILE];
  __shared__ __align__(8) unsigned long long s_bar;
  __shared__ unsigned s_t;
  __shared__ unsigned s_warp[NW];
  __shared__ unsigned s_prefix;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    const unsigned t = atomicAdd(a.counter, 1u);
    s_t = t;
    const long long off = (long long)t * TILE;
    if (a.bulk_ok && a.n - off >= TILE) {
      mbar_init(&s_bar, 1);
      fence_mbar_init();
      mbar_arrive_expect_tx(&s_bar, TILE * sizeof(T));
      bulk_g2s(s_tile, a.in + off, TILE * sizeof(T), &s_bar);
    }
  }
  __syncthreads();
  const unsigned t = s_t;
  const long long off = (long long)t * TILE;
  const int len = a.n - off >= TILE ? TILE : (int)(a.n - off);
  const bool bulk = a.bulk_ok && len == TILE;
  bool failed = false;
  if (bulk) {
    failed = !mbar_wait(&s_bar, 0, a.wait_ns);
  } else {
    for (int k = tid; k < TILE; k += NT) s_tile[k] = k < len ? a.in[off + k] : T{};
  }
  if (__syncthreads_or(failed)) {
    if (tid == 0) {
      raise_err(a.err, ERRBIT_TIMEOUT);
      mbar_wait(&s_bar, 0, a.wait_ns);
      if ((long long)t != a.stalled_tile) st.publish(t, FLAG_P, 0u);
    }
    return;
  }

  // Selection bits (a lane's 32 elements in one word) and the warp's count.  The
  // ranks are taken from the bits after the look-back, so nothing but the one word
  // stays live across it.
  const uint4* run = reinterpret_cast<const uint4*>(s_tile) + warp * ROUNDS * 32;
  const int run0 = warp * ROUNDS * 32 * VEC;  // tile position of the warp's first element
  unsigned bits = 0;
#pragma unroll
  for (int j = 0; j < ROUNDS; ++j) {
    const Vec<T> x = ld_vec<T>(run + j * 32 + lane);
#pragma unroll
    for (int e = 0; e < VEC; ++e) {
      const int pos = run0 + (j * 32 + lane) * VEC + e;
      bits |= (unsigned)(pos < len && selects(x.v[e], a.thr, a.predmask)) << (j * VEC + e);
    }
  }
  const unsigned wcount = __reduce_add_sync(0xffffffffu, (unsigned)__popc(bits));
  if (lane == 0) s_warp[warp] = wcount;
  __syncthreads();

  if (warp == 0) {
    const unsigned agg = block_scan_warp_totals<unsigned, OP_ADD, NW>(s_warp, lane);
    const bool stalled = (long long)t == a.stalled_tile;
    unsigned pfx = 0;
    if (t == 0) {
      if (lane == 0 && !stalled) st.publish(0, FLAG_P, agg);
    } else {
      if (lane == 0 && !stalled) st.publish(t, FLAG_A, agg);
      bool timed_out;
      pfx = lookback_warp<unsigned, OP_ADD, G::K>(st, 0, t, a.wait_ns, timed_out);
      if (lane == 0) {
        if (!stalled) st.publish(t, FLAG_P, pfx + agg);
        if (timed_out) raise_err(a.err, ERRBIT_TIMEOUT);
      }
    }
    if (lane == 0) {
      s_prefix = pfx;
      if (t == a.num_tiles - 1) *a.out_count = (int)(pfx + agg);
    }
  }
  __syncthreads();

  // Stage the selected indices at their rank in the tile (the input is no longer
  // needed: its selection bits are in registers), then store them contiguously.
  int* s_idx = reinterpret_cast<int*>(s_tile);
  const unsigned base_index = (unsigned)off + (unsigned)run0;
  const unsigned lt = lanemask_lt();
  unsigned carry = warp > 0 ? s_warp[warp - 1] : 0u;  // the warp's first slot in the tile
#pragma unroll
  for (int j = 0; j < ROUNDS; ++j) {
    // One ballot per vector slot: lane l's selected elements in round j follow those
    // of lanes 0 .. l-1 (all slots), in element order.
    unsigned before = 0, total = 0;
#pragma unroll
    for (int e = 0; e < VEC; ++e) {
      const unsigned bal = __ballot_sync(0xffffffffu, (bits >> (j * VEC + e)) & 1u);
      before += __popc(bal & lt);
      total += __popc(bal);
    }
    unsigned r = carry + before;
#pragma unroll
    for (int e = 0; e < VEC; ++e)
      if ((bits >> (j * VEC + e)) & 1u) s_idx[r++] = (int)(base_index + (unsigned)((j * 32 + lane) * VEC + e));
    carry += total;
  }
  __syncthreads();
  const unsigned cnt = s_warp[NW - 1];
  int* dst = a.out_idx + s_prefix;
  for (unsigned k = tid; k < cnt; k += NT) dst[k] = s_idx[k];
}

// The same selection for inputs that fit in L2, with the three phases of the
// segment scan (scan_seg.cuh): count per warp part, publish segment counts and
// gather the earlier ones, rescan from L2 and write the indices.  Within a round,
// a lane's selected elements get consecutive output slots after those of the
// lanes before it (one ballot per vector slot); the round's indices are staged in
// shared memory and stored as one contiguous window.
//
// The rescan does not wait for the gather.  Once the segment's count is published,
// warp 0 gathers the earlier counts while the other warps already re-read their
// chunks, rank the selected elements and stage their indices in a per-warp buffer
// of CAP entries (ranks within the warp's part need no base).  When warp 0 posts
// the base, each warp writes out what it has staged and continues round by round;
// a warp whose buffer fills first waits for the base.  So the latency of the
// gather (the slowest segment's count crossing a loaded memory system) overlaps
// the rescan instead of idling every warp of the CTA.
template <class T> struct CompactSegArgs : SegArgsBase {
  const T* in;
  T thr;
  int* out_idx;
  int* out_count;
};

constexpr int kCompactStageCap = 1536;  // indices a warp can stage before the base is known

template <class T, int PRED, class G>
__global__ void __launch_bounds__(G::NT, G::MINB) compact_seg_kernel(CompactSegArgs<T> a, PackedStatus<unsigned> st) {
  pdl_entry();
  constexpr int NW = G::NW, ROUNDS = G::ROUNDS, VEC = G::VEC, CH = G::CH, CAP = kCompactStageCap;
  extern __shared__ __align__(16) int compact_stage_smem[];  // NW x CAP staged indices
  __shared__ unsigned s_seg;
  __shared__ unsigned s_warp[NW];
  __shared__ unsigned s_base;
  __shared__ unsigned s_ready;  // the base and the warp offsets are posted
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int* stage = compact_stage_smem + warp * CAP;
  if (tid == 0) {
    s_seg = atomicAdd(a.counter, 1u);
    s_ready = 0u;
  }
  __syncthreads();
  const unsigned seg = s_seg;
  long long c0, c1;
  const int nact = seg_chunks(a, seg, warp, NW, c0, c1);

  // Phase 1: selected elements in the warp's part.
  unsigned cnt = count_selected<T, PRED, G>(a.in, a.n, c0, c1, a.thr, 0, lane);
  cnt = __reduce_add_sync(0xffffffffu, cnt);
  if (lane == 0) s_warp[warp] = cnt;
  __syncthreads();

  // Phase 2 (warp 0): publish the segment's count, gather the earlier counts, post
  // the base.  The other warps go on to phase 3 meanwhile.
  if (warp == 0) {
    block_scan_warp_totals<unsigned, OP_ADD, NW>(s_warp, lane);
    __syncwarp();
    const unsigned agg = s_warp[nact - 1];
    if (lane == 0 && (long long)seg != a.stalled) st.publish(seg, FLAG_A, agg);
    unsigned base = 0;
    if (seg > 0) {
      bool timed_out;
      base = seg_gather<unsigned, OP_ADD, G::M>(st, 0, seg, a.wait_ns, timed_out);
      if (lane == 0 && timed_out) raise_err(a.err, ERRBIT_TIMEOUT);
    }
    if (lane == 0) {
      s_base = base;
      if (seg == a.ctas - 1) *a.out_count = (int)(base + agg);
      st_release_cta_shared(&s_ready, 1u);
    }
    __syncwarp();
  }

  // Phase 3: rescan from L2 and write the selected indices (positions fit 32 bits:
  // compaction inputs hold fewer than 2^31 elements).  Until the base is posted the
  // indices go to the warp's buffer at staged + rank.
  bool ready = false;
  unsigned off = 0, staged = 0;
  // Takes the posted base: writes out the staged indices and returns the next slot.
  auto take_base = [&]() {
    off = s_base + (warp > 0 ? s_warp[warp - 1] : 0u);
    for (unsigned k = lane; k < staged; k += 32) a.out_idx[off + k] = stage[k];
    off += staged;
    ready = true;
    __syncwarp();  // the buffer is free again
  };
  const unsigned long long drop = l2_policy_evict_first();
  const unsigned lt = lanemask_lt();
  const unsigned n32 = (unsigned)a.n;
  Vec<T> x[ROUNDS];
  if (c0 < c1) seg_load<T, ROUNDS>(x, a.in, c0 * CH, a.n, lane, drop);
  for (long long c = c0; c < c1; ++c) {
    Vec<T> y[ROUNDS];  // the next chunk, requested before this one is processed
    if (c + 1 < c1) seg_load<T, ROUNDS>(y, a.in, (c + 1) * CH, a.n, lane, drop);
    const unsigned cbase = (unsigned)(c * CH);
    const bool full = cbase + CH <= n32;  // no element past n: no bound checks
#pragma unroll
    for (int j = 0; j < ROUNDS; ++j) {
      const unsigned p0 = cbase + (unsigned)((j * 32 + lane) * VEC);
      unsigned sel = 0, before = 0, total = 0;
#pragma unroll
      for (int e = 0; e < VEC; ++e) {
        const bool s = (full || p0 + e < n32) && select_pred<PRED>(x[j].v[e], a.thr);
        const unsigned bal = __ballot_sync(0xffffffffu, s);
        before += __popc(bal & lt);
        total += __popc(bal);
        sel |= (unsigned)s << e;
      }
      if (total == 0) continue;  // warp-uniform
      if (!ready) {
        // One lane reads the flag for the warp, so every lane takes the same branch.
        unsigned posted = 0;
        if (lane == 0) posted = ld_acquire_cta_shared(&s_ready);
        if (__shfl_sync(0xffffffffu, posted, 0)) take_base();
      }
      if (!ready && staged + total > (unsigned)CAP) {
        // The buffer is full: wait for the base (warp 0 always posts it, after at
        // most its bounded gather; the wait is bounded too, and a warp that still
        // sees no base drops its indices rather than write at an unknown offset).
        const unsigned long long t0 = globaltimer();
        unsigned posted = 0;
        for (int spins = 0;; ++spins) {
          if (lane == 0) posted = ld_acquire_cta_shared(&s_ready);
          posted = __shfl_sync(0xffffffffu, posted, 0);
          if (posted || globaltimer() - t0 > 2 * a.wait_ns) break;
          backoff(spins);
        }
        if (!posted) {
          if (lane == 0) raise_err(a.err, ERRBIT_TIMEOUT);
          return;
        }
        take_base();
      }
      // Stage the round's indices at their ranks, then (once the base is known)
      // store the round's contiguous output window with consecutive lanes on
      // consecutive slots (whole lines, not 4-byte pieces spread over 32 x VEC slots).
      int* dst = ready ? stage : stage + staged;
      unsigned r = before;
#pragma unroll
      for (int e = 0; e < VEC; ++e)
        if ((sel >> e) & 1u) dst[r++] = (int)(p0 + e);
      __syncwarp();
      if (ready) {
        for (unsigned k = lane; k < total; k += 32) a.out_idx[off + k] = stage[k];
        off += total;
        __syncwarp();  // the round's reads of the buffer are done before the next writes
      } else {
        staged += total;
      }
    }
#pragma unroll
    for (int j = 0; j < ROUNDS; ++j) x[j] = y[j];
  }
  if (!ready && staged > 0) {  // the part ended before the base was posted
    const unsigned long long t0 = globaltimer();
    unsigned posted = 0;
    for (int spins = 0;; ++spins) {
      if (lane == 0) posted = ld_acquire_cta_shared(&s_ready);
      posted = __shfl_sync(0xffffffffu, posted, 0);
      if (posted || globaltimer() - t0 > 2 * a.wait_ns) break;
      backoff(spins);
    }
    if (!posted) {
      if (lane == 0) raise_err(a.err, ERRBIT_TIMEOUT);
      return;
    }
    take_base();
  }
}

template <class T> bool compact_seg_applies(const CompactJob& job) {
  return (uintptr_t)job.in % 16 == 0 && job.n * (long long)sizeof(T) <= kSegMaxBytes;
}

template <class T> size_t compact_temp_bytes(long long n) {
  const size_t rows = kHeaderBytes + round_up((size_t)rows_tiles<T>(1, n) * 8, 256);
  const size_t seg = kHeaderBytes + seg_status_bytes<unsigned>();
  return rows > seg ? rows : seg;
}

template <class T, int PRED, class G = SegGeom<T>>
cudaError_t launch_compact_seg_p(const CompactJob& job, const LaunchCtx& ctx) {
  const SegPlan p = seg_plan<G>(1, job.n, ctx.num_sms);
  if (p.ctas == 0) return cudaSuccess;
  CompactSegArgs<T> a;
  a.n = job.n;
  a.nc = p.nc;
  a.segs = p.segs;
  a.ctas = p.ctas;
  a.counter = (unsigned*)job.temp;
  a.err = ctx.err;
  a.wait_ns = ctx.wait_ns;
  a.stalled = ctx.stalled_tile;
  a.in = (const T*)job.in;
  memcpy(&a.thr, job.threshold_host, sizeof(T));
  a.out_idx = job.out_idx;
  a.out_count = job.out_count;
  PackedStatus<unsigned> st = seg_status<unsigned>(job.temp);
  auto kern = compact_seg_kernel<T, PRED, G>;
  const size_t smem = (size_t)G::NW * kCompactStageCap * sizeof(int);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  profile_before(ctx);
  e = clear_status(job.temp, seg_reset_bytes<unsigned>(), nullptr, 0, ctx);
  if (e == cudaSuccess) e = launch_pdl(kern, p.ctas, G::NT, smem, ctx.stream, a, st);
  profile_after(ctx);
  return e;
}

template <class T> cudaError_t launch_compact_seg(const CompactJob& job, const LaunchCtx& ctx) {
  switch (job.pred) {
    case 0: return launch_compact_seg_p<T, 0>(job, ctx);
    case 1: return launch_compact_seg_p<T, 1>(job, ctx);
    case 2: return launch_compact_seg_p<T, 2>(job, ctx);
    case 3: return launch_compact_seg_p<T, 3>(job, ctx);
    case 4: return launch_compact_seg_p<T, 4>(job, ctx);
    default: return launch_compact_seg_p<T, 5>(job, ctx);
  }
}

template <class T> cudaError_t launch_compact(const CompactJob& job, const LaunchCtx& ctx) {
  using G = RowsGeom<T>;
  static const unsigned masks[6] = {1u, 3u, 4u, 6u, 2u, 13u};  // LT LE GT GE EQ NE
  if (compact_seg_applies<T>(job)) return launch_compact_seg<T>(job, ctx);
  CompactArgs<T> a;
  a.in = (const T*)job.in;
  a.n = job.n;
  a.num_tiles = rows_tiles<T>(1, job.n);
  memcpy(&a.thr, job.threshold_host, sizeof(T));
  a.predmask = masks[job.pred];
  a.out_idx = job.out_idx;
  a.out_count = job.out_count;
  a.counter = (unsigned*)job.temp;
  a.err = ctx.err;
  a.bulk_ok = ((uintptr_t)job.in % 16) == 0;
  a.wait_ns = ctx.wait_ns;
  a.stalled_tile = ctx.stalled_tile;
  PackedStatus<unsigned> st;
  st.w = (unsigned long long*)((char*)job.temp + kHeaderBytes);
  profile_before(ctx);
  cudaError_t e = clear_status(job.temp, kHeaderBytes + (size_t)a.num_tiles * 8, nullptr, 0, ctx);
  if (e == cudaSuccess) e = launch_pdl(compact_kernel<T>, a.num_tiles, G::NT, 0, ctx.stream, a, st);
  profile_after(ctx);
  return e;
}

}  // namespace gbs
