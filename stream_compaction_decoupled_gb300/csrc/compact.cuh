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
  unsigned* err;
  int bulk_ok;
  unsigned long long wait_ns;
  long long stalled_tile;
};

template <class T> __device__ __forceinline__ bool selects(T x, T t, unsigned mask) {
  const unsigned cls = x < t ? 1u : (x == t ? 2u : (x > t ? 4u : 8u));
  return (mask & cls) != 0;
}

template <class T>
__global__ void __launch_bounds__(RowsGeom<T>::NT, RowsGeom<T>::MINB) compact_kernel(CompactArgs<T> a, PackedStatus<unsigned> st) {
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
      atomicOr(a.err, ERRBIT_TIMEOUT);
      mbar_wait(&s_bar, 0, a.wait_ns);
      if ((long long)t != a.stalled_tile) st.publish(t, FLAG_P, 0u);
    }
    return;
  }

  // Flags, ranks within the warp, warp totals.
  const uint4* run = reinterpret_cast<const uint4*>(s_tile) + warp * ROUNDS * 32;
  const int run0 = warp * ROUNDS * 32 * VEC;  // tile position of the warp's first element
  const unsigned lt = lanemask_lt();
  unsigned bits = 0, carry = 0;
  unsigned rank0[ROUNDS];
#pragma unroll
  for (int j = 0; j < ROUNDS; ++j) {
    const Vec<T> x = ld_vec<T>(run + j * 32 + lane);
    unsigned before = 0, total = 0;
#pragma unroll
    for (int e = 0; e < VEC; ++e) {
      const int pos = run0 + (j * 32 + lane) * VEC + e;
      const bool s = pos < len && selects(x.v[e], a.thr, a.predmask);
      const unsigned bal = __ballot_sync(0xffffffffu, s);
      before += __popc(bal & lt);
      total += __popc(bal);
      bits |= (unsigned)s << (j * VEC + e);
    }
    rank0[j] = carry + before;
    carry += total;
  }
  if (lane == 0) s_warp[warp] = carry;
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
        if (timed_out) atomicOr(a.err, ERRBIT_TIMEOUT);
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
  const unsigned woff = warp > 0 ? s_warp[warp - 1] : 0u;
  const unsigned base_index = (unsigned)off + (unsigned)run0;
#pragma unroll
  for (int j = 0; j < ROUNDS; ++j) {
    unsigned r = woff + rank0[j];
#pragma unroll
    for (int e = 0; e < VEC; ++e)
      if ((bits >> (j * VEC + e)) & 1u) s_idx[r++] = (int)(base_index + (unsigned)((j * 32 + lane) * VEC + e));
  }
  __syncthreads();
  const unsigned cnt = s_warp[NW - 1];
  int* dst = a.out_idx + s_prefix;
  for (unsigned k = tid; k < cnt; k += NT) dst[k] = s_idx[k];
}

template <class T> size_t compact_temp_bytes(long long n) {
  return kHeaderBytes + round_up((size_t)rows_tiles<T>(1, n) * 8, 256);
}

template <class T> cudaError_t launch_compact(const CompactJob& job, const LaunchCtx& ctx) {
  using G = RowsGeom<T>;
  CompactArgs<T> a;
  a.in = (const T*)job.in;
  a.n = job.n;
  a.num_tiles = rows_tiles<T>(1, job.n);
  memcpy(&a.thr, job.threshold_host, sizeof(T));
  static const unsigned masks[6] = {1u, 3u, 4u, 6u, 2u, 13u};  // LT LE GT GE EQ NE
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
  cudaError_t e = cudaMemsetAsync(job.temp, 0, compact_temp_bytes<T>(job.n), ctx.stream);
  if (e != cudaSuccess) return e;
  profile_before(ctx);
  compact_kernel<T><<<a.num_tiles, G::NT, 0, ctx.stream>>>(a, st);
  profile_after(ctx);
  return cudaGetLastError();
}

}  // namespace gbs
