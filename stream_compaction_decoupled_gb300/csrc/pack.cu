// pack.cu -- variable-length output packing by counts in one pass (B. Merry,
// "Prefix sums on GPUs", slides "Output Format" and "Solution": every object
// counts its records, the counts are exclusive-scanned into start positions, and
// every object emits its records at its position).
//
// Per tile of 4096 counts (row-scan geometry, claimed in order): bulk-copy the
// counts into shared memory; exclusive-scan them there (pass 1, block scan,
// decoupled look-back over packed (flag, running total) words, pass 2); write the
// global start offsets if asked; then emit the tile's records contiguously: each
// thread takes runs of consecutive output slots of the tile, finds the object owning
// the first by a binary search over the tile's local offsets and walks forward, so
// the work per record is constant whatever the count distribution.  Offsets add
// with saturation at 2^31 so a total that does not fit int32 is caught, not
// wrapped.
#include "scan_rows.cuh"

namespace gbs {

struct PackArgs {
  const int* counts;
  long long n;
  unsigned num_tiles;
  int* offsets;          // nullable
  int* records;
  long long capacity;
  int* out_total;
  unsigned* counter;
  unsigned* err;
  int bulk_ok;           // counts 16-byte aligned
  int offsets_vec_ok;    // offsets 16-byte aligned
  unsigned long long wait_ns;
  long long stalled_tile;
};

template <class G>
__global__ void __launch_bounds__(G::NT, G::MINB) pack_kernel(PackArgs a, PackedStatus<unsigned> st) {
  pdl_entry();
  constexpr int NT = G::NT, NW = G::NW, ROUNDS = G::ROUNDS, VEC = G::VEC, TILE = G::TILE;
  __shared__ __align__(128) unsigned s_tile[TILE];
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
      mbar_arrive_expect_tx(&s_bar, TILE * sizeof(unsigned));
      bulk_g2s(s_tile, a.counts + off, TILE * sizeof(unsigned), &s_bar);
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
    for (int k = tid; k < TILE; k += NT) s_tile[k] = k < len ? (unsigned)a.counts[off + k] : 0u;
  }
  if (__syncthreads_or(failed)) {
    if (tid == 0) {
      atomicOr(a.err, ERRBIT_TIMEOUT);
      mbar_wait(&s_bar, 0, a.wait_ns);
      if ((long long)t != a.stalled_tile) st.publish(t, FLAG_P, 0u);
    }
    return;
  }

  // A negative count is an error; it counts as zero.
  uint4* run = reinterpret_cast<uint4*>(s_tile) + warp * ROUNDS * 32;
  bool negative = false;
#pragma unroll
  for (int j = 0; j < ROUNDS; ++j) {
    Vec<unsigned> x = ld_vec<unsigned>(run + j * 32 + lane);
    bool fix = false;
#pragma unroll
    for (int e = 0; e < VEC; ++e)
      if ((int)x.v[e] < 0) {
        x.v[e] = 0;
        fix = true;
      }
    if (fix) {
      st_vec<unsigned>(run + j * 32 + lane, x);
      negative = true;
    }
  }
  if (negative) atomicOr(a.err, ERRBIT_INVALID);
  __syncwarp();

  unsigned pre[ROUNDS];
  const unsigned wtot = tile_reduce_pass<unsigned, OP_SATADD, ROUNDS>(run, lane, pre);
  if (lane == 0) s_warp[warp] = wtot;
  __syncthreads();

  if (warp == 0) {
    const unsigned agg = block_scan_warp_totals<unsigned, OP_SATADD, NW>(s_warp, lane);
    const bool stalled = (long long)t == a.stalled_tile;
    unsigned pfx = 0;
    if (t == 0) {
      if (lane == 0 && !stalled) st.publish(0, FLAG_P, agg);
    } else {
      if (lane == 0 && !stalled) st.publish(t, FLAG_A, agg);
      bool timed_out;
      pfx = lookback_warp<unsigned, OP_SATADD, G::K>(st, 0, t, a.wait_ns, timed_out);
      if (lane == 0) {
        if (!stalled) st.publish(t, FLAG_P, Op<unsigned, OP_SATADD>::f(pfx, agg));
        if (timed_out) atomicOr(a.err, ERRBIT_TIMEOUT);
      }
    }
    if (lane == 0) {
      s_prefix = pfx;
      if (t == a.num_tiles - 1) {
        const unsigned total = Op<unsigned, OP_SATADD>::f(pfx, agg);
        *a.out_total = total >= 0x80000000u ? 0x7fffffff : (int)total;
        if (total >= 0x80000000u || (long long)total > a.capacity) atomicOr(a.err, ERRBIT_RANGE);
      }
    }
  }
  __syncthreads();

  // Local exclusive offsets, in place.
  const unsigned base = warp > 0 ? s_warp[warp - 1] : 0u;
  tile_apply_pass<unsigned, OP_SATADD, ROUNDS>(run, lane, pre, base, true, false);
  const unsigned pfx = s_prefix;
  if (a.offsets) {
    const int run0 = warp * ROUNDS * 32 * VEC;
#pragma unroll
    for (int j = 0; j < ROUNDS; ++j) {
      Vec<unsigned> x = ld_vec<unsigned>(run + j * 32 + lane);
#pragma unroll
      for (int e = 0; e < VEC; ++e) {
        const unsigned g = Op<unsigned, OP_SATADD>::f(pfx, x.v[e]);
        x.v[e] = g >= 0x80000000u ? 0x7fffffffu : g;
      }
      const int pos = run0 + (j * 32 + lane) * VEC;
      if (a.offsets_vec_ok && len == TILE) {
        st_vec<unsigned>(reinterpret_cast<uint4*>(a.offsets + off + pos), x);
      } else {
#pragma unroll
        for (int e = 0; e < VEC; ++e)
          if (pos + e < len) a.offsets[off + pos + e] = (int)x.v[e];
      }
    }
  }
  const unsigned agg = s_warp[NW - 1];
  __syncthreads();

  // Emit the tile's records: output slot j of the tile belongs to the last object
  // whose local offset is <= j.  Each thread takes V consecutive slots per round: one
  // binary search for its first slot, then a forward walk (objects with no records
  // share their successor's offset and are stepped over).
  constexpr int V = 32;
  for (unsigned base = 0; base < agg; base += NT * V) {
    const unsigned j0 = base + (unsigned)tid * V;
    if (j0 >= agg) continue;
    int lo = 0, hi = len;
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (s_tile[mid] <= j0) lo = mid + 1;
      else hi = mid;
    }
    int obj = lo - 1;
    const unsigned jend = j0 + V < agg ? j0 + V : agg;
    for (unsigned j = j0; j < jend; ++j) {
      while (obj + 1 < len && s_tile[obj + 1] <= j) ++obj;
      const long long pos = (long long)pfx + j;
      if (pos >= a.capacity) break;
      a.records[pos] = (int)(off + obj);
    }
  }
}

// Packing geometry: the record emission, not the scan, dominates, so tiles are
// a quarter of the scans' (1024 counts: four times as many CTAs share the emission).
using PackGeom = RowsCfg<unsigned, 128, 2, 2, 12>;

size_t pack_temp_bytes(long long n) {
  return kHeaderBytes + round_up((size_t)rows_tiles<unsigned, PackGeom>(1, n) * 8, 256);
}

template <class G> cudaError_t launch_pack_geom(const PackJob& job, const LaunchCtx& ctx) {
  PackArgs a;
  a.counts = job.counts;
  a.n = job.n;
  a.num_tiles = rows_tiles<unsigned, G>(1, job.n);
  a.offsets = job.offsets;
  a.records = job.records;
  a.capacity = job.capacity;
  a.out_total = job.out_total;
  a.counter = (unsigned*)job.temp;
  a.err = ctx.err;
  a.bulk_ok = ((uintptr_t)job.counts % 16) == 0;
  a.offsets_vec_ok = ((uintptr_t)job.offsets % 16) == 0;
  a.wait_ns = ctx.wait_ns;
  a.stalled_tile = ctx.stalled_tile;
  PackedStatus<unsigned> st;
  st.w = (unsigned long long*)((char*)job.temp + kHeaderBytes);
  profile_before(ctx);
  cudaError_t e = clear_status(job.temp, kHeaderBytes + (size_t)rows_tiles<unsigned, G>(1, job.n) * 8, nullptr, 0, ctx);
  if (e == cudaSuccess) e = launch_pdl(pack_kernel<G>, a.num_tiles, G::NT, 0, ctx.stream, a, st);
  profile_after(ctx);
  return e;
}

cudaError_t launch_pack(const PackJob& job, const LaunchCtx& ctx) { return launch_pack_geom<PackGeom>(job, ctx); }

}  // namespace gbs
