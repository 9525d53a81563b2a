// pack.cu -- variable-length output packing by counts in one launch (B. Merry,
// "Prefix sums on GPUs", slides "Output Format" and "Solution": every object
// counts its records, the counts are exclusive-scanned into start positions, and
// every object emits its records at its position).
//
// Two kernels.  Counts that fit in L2 (16-byte aligned, up to 96 MiB) take the
// segment kernel below (pack_seg_kernel).  Otherwise, per tile of 1024 counts (row-
// scan geometry, claimed in order): bulk-copy the counts into shared memory;
// exclusive-scan them there (pass 1, block scan, decoupled look-back over packed
// (flag, running total) words, pass 2); write the global start offsets if asked; then
// emit the tile's records contiguously: each thread takes runs of consecutive output
// slots of the tile, finds the object owning the first by a binary search over the
// tile's local offsets and walks forward, so the work per record is constant
// whatever the count distribution.  In both, offsets add with saturation at 2^31 so
// a total that does not fit int32 is caught, not wrapped.
#include "scan_rows.cuh"
#include "scan_seg.cuh"

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
  ErrSink err;
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
      raise_err(a.err, ERRBIT_TIMEOUT);
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
  if (negative) raise_err(a.err, ERRBIT_INVALID);
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
        if (timed_out) raise_err(a.err, ERRBIT_TIMEOUT);
      }
    }
    if (lane == 0) {
      s_prefix = pfx;
      if (t == a.num_tiles - 1) {
        const unsigned total = Op<unsigned, OP_SATADD>::f(pfx, agg);
        *a.out_total = total >= 0x80000000u ? 0x7fffffff : (int)total;
        if (total >= 0x80000000u || (long long)total > a.capacity) raise_err(a.err, ERRBIT_RANGE);
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

// ---- packing for inputs that fit in L2: the segment scheme (scan_seg.cuh) ----------
//
// Phase 1 sums each warp's counts (negative counts read as 0; 64-bit sums capped at
// 2^31, which is the saturating add of the counts), phase 2 publishes the segment
// sum and gathers the earlier ones, phase 3 walks the warp's chunks again from L2:
// the exclusive offsets of a chunk (saturating, seeded with the running base) are
// written out, and the chunk's records are emitted in blocks of 32 x PV output slots
// by a scatter of the run starts and a forward max over the block (no search; see
// the emission below), and the warp stores each block contiguously.
constexpr int PV = 8;
// Chunks of 128 counts (one 16-byte vector a lane): about 512 records each for the
// Poisson(4) workload, so that a million counts give every warp of every SM chunks
// to emit (emission is instruction-bound, not memory-bound).
using PackSegGeom = SegCfg<unsigned, 1024, 1, 1>;
constexpr size_t kPackSegSmem = (size_t)PackSegGeom::NW * 32 * PV * sizeof(unsigned);

struct PackSegArgs : SegArgsBase {
  const int* counts;
  int* offsets;  // nullable
  int* records;
  long long capacity;
  int* out_total;
};

__global__ void __launch_bounds__(PackSegGeom::NT, PackSegGeom::MINB) pack_seg_kernel(PackSegArgs a,
                                                                                    PackedStatus<unsigned> st) {
  pdl_entry();
  using G = PackSegGeom;
  constexpr int NW = G::NW, ROUNDS = G::ROUNDS, VEC = G::VEC, CH = G::CH;
  constexpr unsigned CAP = 0x80000000u;  // offsets saturate here
  extern __shared__ __align__(16) unsigned pack_seg_smem[];
  __shared__ unsigned s_seg;
  __shared__ unsigned s_warp[NW];
  __shared__ unsigned s_base;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  unsigned* s_stage = pack_seg_smem + warp * 32 * PV;  // one block of record slots
  if (tid == 0) s_seg = atomicAdd(a.counter, 1u);
  __syncthreads();
  const unsigned seg = s_seg;
  long long c0, c1;
  const int nact = seg_chunks(a, seg, warp, NW, c0, c1);

  // Phase 1: the warp's count sum.
  {
    constexpr int U = 8;
    const unsigned long long keep = l2_policy_evict_last();
    const long long e1 = c1 * CH < a.n ? c1 * CH : a.n;
    const long long v1 = e1 / VEC;
    const uint4* p = reinterpret_cast<const uint4*>(a.counts);
    unsigned long long sum = 0;
    long long v = c0 * CH / VEC + lane;
    for (; v + 32 * (U - 1) < v1; v += 32 * U) {  // U loads in flight
      uint4 u[U];
#pragma unroll
      for (int k = 0; k < U; ++k) u[k] = ld_hint(p + v + 32 * k, keep);
#pragma unroll
      for (int k = 0; k < U; ++k)
        sum += (unsigned long long)(unsigned)max((int)u[k].x, 0) + (unsigned)max((int)u[k].y, 0) +
               (unsigned)max((int)u[k].z, 0) + (unsigned)max((int)u[k].w, 0);
    }
    if (v < v1) {  // the rest in one guarded round
      uint4 u[U];
#pragma unroll
      for (int k = 0; k < U; ++k)
        if (v + 32 * k < v1) u[k] = ld_hint(p + v + 32 * k, keep);
#pragma unroll
      for (int k = 0; k < U; ++k)
        if (v + 32 * k < v1)
          sum += (unsigned long long)(unsigned)max((int)u[k].x, 0) + (unsigned)max((int)u[k].y, 0) +
                 (unsigned)max((int)u[k].z, 0) + (unsigned)max((int)u[k].w, 0);
    }
    if (lane == 0)
      for (long long i = v1 * VEC; i < e1; ++i) sum += (unsigned)max(a.counts[i], 0);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
    if (lane == 0) s_warp[warp] = sum >= CAP ? CAP : (unsigned)sum;
  }
  __syncthreads();

  // Phase 2: publish the segment's sum, gather the earlier sums; the last segment
  // writes the total.
  if (warp == 0) {
    block_scan_warp_totals<unsigned, OP_SATADD, NW>(s_warp, lane);
    __syncwarp();
    const unsigned agg = s_warp[nact - 1];
    if (lane == 0 && (long long)seg != a.stalled) st.publish(seg, FLAG_A, agg);
    unsigned base = 0;
    if (seg > 0) {
      bool timed_out;
      base = seg_gather<unsigned, OP_SATADD, G::M>(st, 0, seg, a.wait_ns, timed_out);
      if (lane == 0 && timed_out) raise_err(a.err, ERRBIT_TIMEOUT);
    }
    if (lane == 0) {
      s_base = base;
      if (seg == a.ctas - 1) {
        const unsigned total = Op<unsigned, OP_SATADD>::f(base, agg);
        *a.out_total = total >= CAP ? 0x7fffffff : (int)total;
        if (total >= CAP || (long long)total > a.capacity) raise_err(a.err, ERRBIT_RANGE);
      }
    }
  }
  __syncthreads();

  // Phase 3: offsets and records, chunk by chunk.
  unsigned run = s_base;
  if (warp > 0) run = Op<unsigned, OP_SATADD>::f(run, s_warp[warp - 1]);
  const unsigned long long drop = l2_policy_evict_first();
  bool negative = false;
  for (long long c = c0; c < c1; ++c) {
    Vec<unsigned> x[ROUNDS];
    seg_load<unsigned, ROUNDS>(x, reinterpret_cast<const unsigned*>(a.counts), c * CH, a.n, lane, drop);
#pragma unroll
    for (int j = 0; j < ROUNDS; ++j)
#pragma unroll
      for (int e = 0; e < VEC; ++e)
        if ((int)x[j].v[e] < 0) {
          x[j].v[e] = 0;
          negative = true;
        }
    static_assert(ROUNDS == 1, "a lane holds one vector of counts per chunk");
    const Vec<unsigned> cnt = x[0];  // the (clamped) counts, kept for the emission
    unsigned pre[ROUNDS];
    const unsigned ctot = regs_reduce_pass<unsigned, OP_SATADD, ROUNDS>(x, lane, pre);
    regs_apply_pass<unsigned, OP_SATADD, ROUNDS>(x, lane, pre, run, true, false);  // x: exclusive offsets
    __syncwarp();
#pragma unroll
    for (int j = 0; j < ROUNDS; ++j) {
      if (a.offsets) {
        const long long e0 = c * CH + (long long)(j * 32 + lane) * VEC;
        Vec<unsigned> o;
#pragma unroll
        for (int e = 0; e < VEC; ++e) o.v[e] = x[j].v[e] >= CAP ? 0x7fffffffu : x[j].v[e];
        if (e0 + VEC <= a.n && ((uintptr_t)(a.offsets + e0) & 15) == 0) {
          uint4 u;
          memcpy(&u, o.v, 16);
          st_hint(reinterpret_cast<uint4*>(a.offsets + e0), u, drop);
        } else {
#pragma unroll
          for (int e = 0; e < VEC; ++e)
            if (e0 + e < a.n) a.offsets[e0 + e] = (int)o.v[e];
        }
      }
    }
    __syncwarp();
    // Records of this chunk: slots [run, run + ctot), capped by the capacity (slots
    // and offsets stay below 2^31, so 32-bit arithmetic suffices).
    const unsigned cend_u = Op<unsigned, OP_SATADD>::f(run, ctot);
    const unsigned cb = run, ce = (long long)cend_u < a.capacity ? cend_u : (unsigned)a.capacity;
    const unsigned obj0 = (unsigned)(c * CH);
    // Records in blocks of 32 x PV slots, with no search: the block's slots are
    // cleared in shared memory, every object whose run starts in the block writes its
    // (chunk-local index + 1) at its first slot (distinct objects with records have
    // distinct offsets), and a forward max over the block fills each slot with its
    // owner (owners increase with the offset): lane l takes slots PV l .. PV l + PV - 1
    // serially, one warp max-scan joins the lanes, and `owner` carries the last slot's
    // owner into the next block.  The warp then stores the block contiguously.
    static_assert(PV == 8, "two 16-byte vectors of slots a lane");
    uint4* blk4 = reinterpret_cast<uint4*>(s_stage);
    unsigned owner = 0;
    for (unsigned b0 = cb; b0 < ce; b0 += 32 * PV) {
      blk4[2 * lane] = make_uint4(0u, 0u, 0u, 0u);
      blk4[2 * lane + 1] = make_uint4(0u, 0u, 0u, 0u);
      __syncwarp();
#pragma unroll
      for (int e = 0; e < VEC; ++e) {
        const unsigned o = x[0].v[e];
        if (cnt.v[e] != 0 && o >= b0 && o - b0 < 32u * PV) s_stage[o - b0] = (unsigned)(lane * VEC + e) + 1u;
      }
      __syncwarp();
      const uint4 lo = blk4[2 * lane], hi = blk4[2 * lane + 1];
      unsigned v[PV] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
#pragma unroll
      for (int i = 1; i < PV; ++i) v[i] = max(v[i], v[i - 1]);
      const unsigned inc = warp_inclusive<unsigned, OP_MAX>(v[PV - 1], lane);
      unsigned before = __shfl_up_sync(0xffffffffu, inc, 1);
      before = max(lane > 0 ? before : 0u, owner);
#pragma unroll
      for (int i = 0; i < PV; ++i) v[i] = max(v[i], before);
      owner = max(__shfl_sync(0xffffffffu, inc, 31), owner);
      __syncwarp();
      blk4[2 * lane] = make_uint4(v[0], v[1], v[2], v[3]);
      blk4[2 * lane + 1] = make_uint4(v[4], v[5], v[6], v[7]);
      __syncwarp();
      const unsigned nblk = ce - b0 < 32u * PV ? ce - b0 : 32u * PV;
      int* dst = a.records + b0;
#pragma unroll
      for (int i = 0; i < PV; ++i) {
        const unsigned k = (unsigned)(lane + 32 * i);
        if (k < nblk) dst[k] = (int)(obj0 + s_stage[k] - 1u);
      }
      __syncwarp();
    }
    run = cend_u;
  }
  if (negative) raise_err(a.err, ERRBIT_INVALID);
}

size_t pack_temp_bytes(long long n) {
  const size_t rows = kHeaderBytes + round_up((size_t)rows_tiles<unsigned, PackGeom>(1, n) * 8, 256);
  const size_t seg = kHeaderBytes + seg_status_bytes<unsigned>();
  return rows > seg ? rows : seg;
}

// Inputs up to this many counts take the segment kernel (16-byte aligned counts).
constexpr long long kPackSegMaxCounts = (96ll << 20) / 4;

cudaError_t launch_pack_seg(const PackJob& job, const LaunchCtx& ctx) {
  using G = PackSegGeom;
  const SegPlan p = seg_plan<G>(1, job.n, ctx.num_sms);
  if (p.ctas == 0) return cudaErrorInvalidValue;
  PackSegArgs a;
  a.n = job.n;
  a.nc = p.nc;
  a.segs = p.segs;
  a.ctas = p.ctas;
  a.counter = (unsigned*)job.temp;
  a.err = ctx.err;
  a.wait_ns = ctx.wait_ns;
  a.stalled = ctx.stalled_tile;
  a.counts = job.counts;
  a.offsets = job.offsets;
  a.records = job.records;
  a.capacity = job.capacity;
  a.out_total = job.out_total;
  PackedStatus<unsigned> st = seg_status<unsigned>(job.temp);
  cudaError_t e = cudaFuncSetAttribute(pack_seg_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kPackSegSmem);
  if (e != cudaSuccess) return e;
  profile_before(ctx);
  e = clear_status(job.temp, seg_reset_bytes<unsigned>(), nullptr, 0, ctx);
  if (e == cudaSuccess) e = launch_pdl(pack_seg_kernel, p.ctas, G::NT, kPackSegSmem, ctx.stream, a, st);
  profile_after(ctx);
  return e;
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

cudaError_t launch_pack(const PackJob& job, const LaunchCtx& ctx) {
  if ((uintptr_t)job.counts % 16 == 0 && job.n <= kPackSegMaxCounts) return launch_pack_seg(job, ctx);
  return launch_pack_geom<PackGeom>(job, ctx);
}

}  // namespace gbs
