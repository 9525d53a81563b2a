// partition.cuh -- stable partition by a predicate (B. Merry, "Prefix sums on GPUs",
// slides "Other Applications": partitioning and the one-bit split of radix sort;
// "Solution": count, scan, emit), as one launch of the segment scheme (scan_seg.cuh):
//   1. each warp counts the selected elements of its part (16-byte loads, evict-last);
//   2. warp 0 publishes the segment's count and gathers every segment's count: the
//      earlier ones give the segment's selected base, all of them the total m;
//   3. each warp rescans its part from L2 and writes a round's selected elements to
//      out[base + rank] and its rejected ones to out[m + (elements before - selected
//      before) + rank], both in input order (staged back to back in shared memory and
//      stored in one pass).
// Phase 2 waits for later segments too, so every segment must be resident at once:
// the kernel is launched cooperatively (one CTA per SM at most).  Inputs larger than
// L2 run the same way; their phase 3 then reads HBM again.
//
// An input view that does not start on a 16-byte boundary is read from the boundary
// below it (the same 16-byte block, inside the allocation, which starts aligned) with
// its d leading elements masked out, so all loads stay vector loads.
#pragma once

#include "compact.cuh"

namespace gbs {

template <class T> struct PartitionArgs : SegArgsBase {  // n counts the d masked elements too
  const T* in;   // 16-byte aligned base: in[d] is the input's element 0
  unsigned d;    // leading elements of the base that are not part of the input
  T thr;
  T* out;
  int* out_idx;  // nullable
  int* out_count;
};

template <class T, int PRED, class G>
__global__ void __launch_bounds__(G::NT, G::MINB) partition_seg_kernel(PartitionArgs<T> a, PackedStatus<unsigned> st) {
  pdl_entry();
  constexpr int NW = G::NW, ROUNDS = G::ROUNDS, VEC = G::VEC, CH = G::CH, SLOTS = 32 * VEC;
  __shared__ unsigned s_seg;
  __shared__ unsigned s_warp[NW];
  __shared__ unsigned s_base, s_total;
  __shared__ T s_val_all[NW * SLOTS];  // a round's selected values, then its rejected ones
  __shared__ int s_idx_all[NW * SLOTS];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  T* s_val = s_val_all + warp * SLOTS;
  int* s_idx = s_idx_all + warp * SLOTS;
  if (tid == 0) s_seg = atomicAdd(a.counter, 1u);
  __syncthreads();
  const unsigned seg = s_seg;
  long long c0, c1;
  const int nact = seg_chunks(a, seg, warp, NW, c0, c1);
  const long long d = a.d;

  // Phase 1: selected elements of the warp's part.
  unsigned cnt = count_selected<T, PRED, G>(a.in, a.n, c0, c1, a.thr, d, lane);
  cnt = __reduce_add_sync(0xffffffffu, cnt);
  if (lane == 0) s_warp[warp] = cnt;
  __syncthreads();

  // Phase 2: publish the count; gather the earlier segments' counts and all of them.
  if (warp == 0) {
    block_scan_warp_totals<unsigned, OP_ADD, NW>(s_warp, lane);
    __syncwarp();
    const unsigned agg = s_warp[nact - 1];
    if (lane == 0 && (long long)seg != a.stalled) st.publish(seg, FLAG_A, agg);
    bool t1 = false, t2 = false;
    const unsigned base = seg > 0 ? seg_gather<unsigned, OP_ADD, G::M>(st, 0, seg, a.wait_ns, t1) : 0u;
    const unsigned total = seg_gather<unsigned, OP_ADD, G::M>(st, 0, a.ctas, a.wait_ns, t2);
    if (lane == 0) {
      if (t1 || t2) raise_err(a.err, ERRBIT_TIMEOUT);
      s_base = base;
      s_total = total;
      if (seg == a.ctas - 1) *a.out_count = (int)total;
    }
  }
  __syncthreads();

  // Phase 3: rescan from L2; the selected and the rejected elements of a round go out
  // as two contiguous windows.  Positions fit 32 bits (n < 2^31).
  const unsigned total = s_total;
  unsigned sel = s_base + (warp > 0 ? s_warp[warp - 1] : 0u);  // selected before the part
  const long long first = c0 * CH;
  unsigned rej = (unsigned)(first > d ? first - d : 0) - sel;      // rejected before the part
  const unsigned long long drop = l2_policy_evict_first();
  const unsigned lt = lanemask_lt();
  const unsigned nb = (unsigned)a.n, d32 = a.d;
  Vec<T> x[ROUNDS];
  if (c0 < c1) seg_load<T, ROUNDS>(x, a.in, c0 * CH, a.n, lane, drop);
  for (long long c = c0; c < c1; ++c) {
    Vec<T> y[ROUNDS];
    if (c + 1 < c1) seg_load<T, ROUNDS>(y, a.in, (c + 1) * CH, a.n, lane, drop);
    const unsigned cbase = (unsigned)(c * CH);
    const bool full = cbase >= d32 && cbase + CH <= nb;  // every element of the chunk is input
#pragma unroll
    for (int j = 0; j < ROUNDS; ++j) {
      const unsigned p0 = cbase + (unsigned)((j * 32 + lane) * VEC);
      // Ranks: selected elements of the lanes before this one (sb), the round's
      // selected (st_) and rejected (rt) totals; in a full chunk every element is
      // valid, so the rejected ones follow from the selected ones.
      unsigned sbits = 0, rbits = 0, sb = 0, st_ = 0, rb, rt;
      if (full) {
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
          const bool s = select_pred<PRED>(x[j].v[e], a.thr);
          const unsigned bs = __ballot_sync(0xffffffffu, s);
          sb += __popc(bs & lt);
          st_ += __popc(bs);
          sbits |= (unsigned)s << e;
        }
        rbits = ~sbits & ((1u << VEC) - 1u);
        rb = (unsigned)lane * VEC - sb;
        rt = SLOTS - st_;
      } else {
        rb = rt = 0;
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
          const bool valid = p0 + e >= d32 && p0 + e < nb;
          const bool s = valid && select_pred<PRED>(x[j].v[e], a.thr);
          const bool r = valid && !s;
          const unsigned bs = __ballot_sync(0xffffffffu, s), br = __ballot_sync(0xffffffffu, r);
          sb += __popc(bs & lt);
          st_ += __popc(bs);
          rb += __popc(br & lt);
          rt += __popc(br);
          sbits |= (unsigned)s << e;
          rbits |= (unsigned)r << e;
        }
      }
      if (st_ + rt != 0) {  // warp-uniform
        // Stage the selected elements at [0, st_) and the rejected at [st_, st_ + rt),
        // each in input order, then write both windows in one pass.
        __syncwarp();
        unsigned rs = sb, rr = st_ + rb;
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
          const bool sel_e = (sbits >> e) & 1u, rej_e = (rbits >> e) & 1u;
          if (sel_e || rej_e) {
            const unsigned slot = sel_e ? rs++ : rr++;
            s_val[slot] = x[j].v[e];
            s_idx[slot] = (int)(p0 + e - d32);
          }
        }
        __syncwarp();
        const unsigned all = st_ + rt, rdst = total + rej - st_;
        for (unsigned k = lane; k < all; k += 32) {
          const unsigned dst = k < st_ ? sel + k : rdst + k;
          a.out[dst] = s_val[k];
          if (a.out_idx) a.out_idx[dst] = s_idx[k];
        }
        sel += st_;
        rej += rt;
      }
    }
#pragma unroll
    for (int j = 0; j < ROUNDS; ++j) x[j] = y[j];
  }
}

template <class T> size_t partition_temp_bytes() { return kHeaderBytes + seg_status_bytes<unsigned>(); }

// Launches with every CTA resident at once (phase 2 waits for all segments).
template <class... P, class... A>
cudaError_t launch_cooperative(void (*kernel)(P...), unsigned grid, unsigned block, cudaStream_t stream,
                               A&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<A>(args)...);
}

template <class T, int PRED> cudaError_t launch_partition_p(const PartitionJob& job, const LaunchCtx& ctx) {
  using G = SegGeom<T>;
  const unsigned d = (unsigned)(((uintptr_t)job.in % 16) / sizeof(T));
  const SegPlan p = seg_plan<G>(1, job.n + d, ctx.num_sms);
  if (p.ctas == 0) return cudaSuccess;
  PartitionArgs<T> a;
  a.n = job.n + d;
  a.nc = p.nc;
  a.segs = p.segs;
  a.ctas = p.ctas;
  a.counter = (unsigned*)job.temp;
  a.err = ctx.err;
  a.wait_ns = ctx.wait_ns;
  a.stalled = ctx.stalled_tile;
  a.in = (const T*)job.in - d;
  a.d = d;
  memcpy(&a.thr, job.threshold_host, sizeof(T));
  a.out = (T*)job.out;
  a.out_idx = job.out_idx;
  a.out_count = job.out_count;
  PackedStatus<unsigned> st = seg_status<unsigned>(job.temp);
  profile_before(ctx);
  cudaError_t e = clear_status(job.temp, seg_reset_bytes<unsigned>(), nullptr, 0, ctx);
  if (e == cudaSuccess) e = launch_cooperative(partition_seg_kernel<T, PRED, G>, p.ctas, G::NT, ctx.stream, a, st);
  profile_after(ctx);
  return e;
}

template <class T> cudaError_t launch_partition(const PartitionJob& job, const LaunchCtx& ctx) {
  if ((uintptr_t)job.in % sizeof(T) != 0) return cudaErrorMisalignedAddress;
  switch (job.pred) {
    case 0: return launch_partition_p<T, 0>(job, ctx);
    case 1: return launch_partition_p<T, 1>(job, ctx);
    case 2: return launch_partition_p<T, 2>(job, ctx);
    case 3: return launch_partition_p<T, 3>(job, ctx);
    case 4: return launch_partition_p<T, 4>(job, ctx);
    case 5: return launch_partition_p<T, 5>(job, ctx);
    default:
      if constexpr (std::is_integral<T>::value) return launch_partition_p<T, 6>(job, ctx);
      else return cudaErrorInvalidValue;
  }
}

}  // namespace gbs
