// rts.cuh -- the reduce-then-scan comparison variant (The CUDA Handbook, 13.3.3,
// Figure 13-10 and Listings 13-10..13-12; B. Merry, "Prefix sums on GPUs", slides
// "Fixed Block Count" and "Prefix-Summing a Block"): a fixed number C of blocks,
// a multiple of the SM count and at most 1024, each own one contiguous subarray
// (a whole number of tiles).
//   launch 1  each block reduces its subarray to one partial       (reads n)
//   launch 2  one block scans the C partials into exclusive bases
//   launch 3  each block scans its subarray tile by tile, carrying the running
//             total from its base, double-buffering the tile loads  (reads n, writes n)
// No tile status, no look-back and no waiting between blocks; 3n element transfers
// against the single-pass kernel's 2n.  The reduction in launch 1 visits the
// elements in a strided order, which is fine for the operators provided (all
// commutative); launch 3 keeps scan order.
//
// The scan-then-fan variant (The CUDA Handbook, 13.3.2) uses the same blocks:
//   launch 1  each block scans its subarray (tile by tile, carrying its own running
//             total) and writes its total to the partials     (reads n, writes n)
//   launch 2  one block scans the C partials into exclusive bases
//   launch 3  each block but the first combines its base into its outputs (fan)
//                                                            (reads n, writes n)
// 4n element transfers.  An exclusive scan seeds every block's local scan with the
// initial value (0 for add, 1 for multiply when none is given; max and min take it
// more than once harmlessly, being idempotent), so the fan is one combine per
// element for both kinds.
#pragma once

#include "launch.h"
#include "tile.cuh"
#include "scan_rows.cuh"

namespace gbs {

template <class T> struct RtsArgs {
  const T* in;
  T* out;
  long long n;
  long long per_block;  // elements per block, a multiple of the tile
  int nblocks;
  T* partials;          // nblocks reductions, then (from index 1) exclusive bases
  T init;
  int inclusive;
  int vec_ok;           // in and out 16-byte aligned
  ErrSink err;
  unsigned long long wait_ns;
};

constexpr int kRtsMaxBlocks = 1024;

template <class T, int OP>
__global__ void __launch_bounds__(256) rts_reduce_kernel(RtsArgs<T> a) {
  pdl_entry();
  constexpr int NT = 256, VEC = Vec<T>::N, U = 4;
  __shared__ T s_v[NT / 32];
  __shared__ int s_h[NT / 32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const long long begin = (long long)blockIdx.x * a.per_block;
  const long long end = begin + a.per_block < a.n ? begin + a.per_block : a.n;
  T acc{};
  bool has = false;
  long long i = begin + (long long)tid * VEC;
  if (a.vec_ok) {
    // U independent 16-byte loads in flight per thread.
    for (; i + (long long)(U - 1) * NT * VEC + VEC <= end; i += (long long)U * NT * VEC) {
      Vec<T> x[U];
#pragma unroll
      for (int u = 0; u < U; ++u) x[u] = ld_vec<T>(reinterpret_cast<const uint4*>(a.in + i + (long long)u * NT * VEC));
#pragma unroll
      for (int u = 0; u < U; ++u)
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
          acc = has ? Op<T, OP>::f(acc, x[u].v[e]) : x[u].v[e];
          has = true;
        }
    }
    for (; i + VEC <= end; i += (long long)NT * VEC) {
      const Vec<T> x = ld_vec<T>(reinterpret_cast<const uint4*>(a.in + i));
#pragma unroll
      for (int e = 0; e < VEC; ++e) {
        acc = has ? Op<T, OP>::f(acc, x.v[e]) : x.v[e];
        has = true;
      }
    }
    for (; i < end; i += (long long)NT * VEC)  // ragged tail of the array
      for (long long k = i; k < end && k < i + VEC; ++k) {
        acc = has ? Op<T, OP>::f(acc, a.in[k]) : a.in[k];
        has = true;
      }
  } else {
    for (long long k = begin + tid; k < end; k += NT) {
      acc = has ? Op<T, OP>::f(acc, a.in[k]) : a.in[k];
      has = true;
    }
  }
  // Block reduction with presence flags (no identity element needed).
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const T o = __shfl_down_sync(0xffffffffu, acc, off);
    const int oh = __shfl_down_sync(0xffffffffu, (int)has, off);
    if (lane + off < 32 && oh) {
      acc = has ? Op<T, OP>::f(acc, o) : o;
      has = true;
    }
  }
  if (lane == 0) {
    s_v[warp] = acc;
    s_h[warp] = has;
  }
  __syncthreads();
  if (tid == 0) {
    T r{};
    bool h = false;
    for (int w = 0; w < NT / 32; ++w)
      if (s_h[w]) {
        r = h ? Op<T, OP>::f(r, s_v[w]) : s_v[w];
        h = true;
      }
    a.partials[blockIdx.x] = r;
  }
}

template <class T, int OP>
__global__ void __launch_bounds__(kRtsMaxBlocks) rts_spine_kernel(T* partials, int nb) {
  pdl_entry();
  __shared__ T s_w[32];
  __shared__ T s_incl[kRtsMaxBlocks];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const T v = partials[tid < nb ? tid : nb - 1];
  const T wi = warp_inclusive<T, OP>(v, lane);
  if (lane == 31) s_w[warp] = wi;
  __syncthreads();
  if (warp == 0) {
    const T w = warp_inclusive<T, OP>(s_w[lane], lane);
    s_w[lane] = w;
  }
  __syncthreads();
  s_incl[tid] = warp > 0 ? Op<T, OP>::f(s_w[warp - 1], wi) : wi;
  __syncthreads();
  if (tid > 0 && tid < nb) partials[tid] = s_incl[tid - 1];  // exclusive base of block tid
}

template <class T, int OP, bool STF>
__global__ void __launch_bounds__(RowsGeom<T>::NT) rts_scan_kernel(RtsArgs<T> a) {
  pdl_entry();
  using G = RowsGeom<T>;
  constexpr int NT = G::NT, NW = G::NW, ROUNDS = G::ROUNDS, TILE = G::TILE;
  __shared__ __align__(128) T s_tile[2][TILE];
  __shared__ __align__(8) unsigned long long s_bar[2];
  __shared__ T s_warp[NW];
  __shared__ int s_fail;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const long long begin = (long long)blockIdx.x * a.per_block;
  const long long end = begin + a.per_block < a.n ? begin + a.per_block : a.n;
  const long long ntiles = (end - begin + TILE - 1) / TILE;

  // Carry-in: the block's base (block 0 has none; scan-then-fan: none yet), behind
  // the initial value.  Scan-then-fan also keeps the block's own total.
  bool has = !STF && blockIdx.x > 0;
  T carry = has ? a.partials[blockIdx.x] : T{};
  if (!a.inclusive) {
    carry = has ? Op<T, OP>::f(a.init, carry) : a.init;
    has = true;
  }
  T total{};
  bool htotal = false;

  auto tile_len = [&](long long k) -> int {
    const long long s = begin + k * TILE;
    return end - s >= TILE ? TILE : (int)(end - s);
  };
  auto issue = [&](long long k) {  // thread 0 only
    if (a.vec_ok && tile_len(k) == TILE) {
      const int q = (int)(k & 1);
      mbar_arrive_expect_tx(&s_bar[q], TILE * sizeof(T));
      bulk_g2s(s_tile[q], a.in + begin + k * TILE, TILE * sizeof(T), &s_bar[q]);
    }
  };
  if (tid == 0) {
    mbar_init(&s_bar[0], 1);
    mbar_init(&s_bar[1], 1);
    fence_mbar_init();
    s_fail = 0;
    issue(0);
  }
  __syncthreads();

  for (long long k = 0; k < ntiles; ++k) {
    const int q = (int)(k & 1);
    const int len = tile_len(k);
    const bool bulk = a.vec_ok && len == TILE;
    const long long start = begin + k * TILE;
    if (tid == 0 && k + 1 < ntiles) {
      bulk_wait_read_all();  // the other buffer's store (tile k-1) has been read out
      issue(k + 1);
    }
    bool failed = false;
    if (bulk) {
      failed = !mbar_wait(&s_bar[q], (unsigned)((k >> 1) & 1), a.wait_ns);
    } else {
      for (int i = tid; i < TILE; i += NT) s_tile[q][i] = i < len ? a.in[start + i] : T{};
    }
    if (__syncthreads_or(failed)) {
      if (tid == 0) {
        raise_err(a.err, ERRBIT_TIMEOUT);
        mbar_wait(&s_bar[q], (unsigned)((k >> 1) & 1), a.wait_ns);
        if (k + 1 < ntiles) mbar_wait(&s_bar[q ^ 1], (unsigned)(((k + 1) >> 1) & 1), a.wait_ns);
      }
      return;
    }
    uint4* run = reinterpret_cast<uint4*>(s_tile[q]) + warp * ROUNDS * 32;
    T pre[ROUNDS];
    const T wtot = tile_reduce_pass<T, OP, ROUNDS>(run, lane, pre);
    if (lane == 0) s_warp[warp] = wtot;
    __syncthreads();
    if (warp == 0) block_scan_warp_totals<T, OP, NW>(s_warp, lane);
    __syncthreads();
    bool hb = has;
    T b = carry;
    if (warp > 0) {
      const T wp = s_warp[warp - 1];
      b = hb ? Op<T, OP>::f(b, wp) : wp;
      hb = true;
    }
    tile_apply_pass<T, OP, ROUNDS>(run, lane, pre, b, hb, a.inclusive != 0);
    const T agg = s_warp[NW - 1];
    carry = has ? Op<T, OP>::f(carry, agg) : agg;
    has = true;
    if (STF) {
      total = htotal ? Op<T, OP>::f(total, agg) : agg;
      htotal = true;
    }
    if (bulk) {
      fence_proxy_async_smem();
      __syncthreads();
      if (tid == 0) {
        bulk_s2g(a.out + start, s_tile[q], TILE * sizeof(T));
        bulk_commit();
      }
    } else {
      __syncthreads();
      for (int i = tid; i < len; i += NT) a.out[start + i] = s_tile[q][i];
    }
    __syncthreads();  // s_warp and the buffer are reused by the next tile
  }
  if (tid == 0) {
    bulk_wait_read_all();
    if (STF) a.partials[blockIdx.x] = total;
  }
}

// Scan-then-fan, launch 3: block b > 0 combines its exclusive base into each of its
// outputs, on the left (16-byte vectors when aligned, U in flight per thread).
template <class T, int OP>
__global__ void __launch_bounds__(256) stf_fan_kernel(RtsArgs<T> a) {
  pdl_entry();
  if (blockIdx.x == 0) return;
  constexpr int NT = 256, VEC = Vec<T>::N, U = 4;
  const long long begin = (long long)blockIdx.x * a.per_block;
  const long long end = begin + a.per_block < a.n ? begin + a.per_block : a.n;
  const T base = a.partials[blockIdx.x];
  long long i = begin + (long long)threadIdx.x * VEC;
  if (a.vec_ok) {
    for (; i + (long long)(U - 1) * NT * VEC + VEC <= end; i += (long long)U * NT * VEC) {
      Vec<T> x[U];
#pragma unroll
      for (int u = 0; u < U; ++u) x[u] = ld_vec<T>(reinterpret_cast<const uint4*>(a.out + i + (long long)u * NT * VEC));
#pragma unroll
      for (int u = 0; u < U; ++u) {
#pragma unroll
        for (int e = 0; e < VEC; ++e) x[u].v[e] = Op<T, OP>::f(base, x[u].v[e]);
        uint4 w;
        memcpy(&w, x[u].v, 16);
        *reinterpret_cast<uint4*>(a.out + i + (long long)u * NT * VEC) = w;
      }
    }
    for (; i < end; i += (long long)NT * VEC)
      for (long long k = i; k < end && k < i + VEC; ++k) a.out[k] = Op<T, OP>::f(base, a.out[k]);
  } else {
    for (long long k = begin + threadIdx.x; k < end; k += NT) a.out[k] = Op<T, OP>::f(base, a.out[k]);
  }
}

template <class T> size_t rts_temp_bytes(long long, int) {
  return kHeaderBytes + round_up((size_t)kRtsMaxBlocks * sizeof(T), 256);
}

template <class T, int OP> cudaError_t launch_rts_op(const RtsJob& job, const LaunchCtx& ctx) {
  constexpr int TILE = RowsGeom<T>::TILE;
  RtsArgs<T> a;
  a.in = (const T*)job.in;
  a.out = (T*)job.out;
  a.n = job.n;
  const long long tiles = (job.n + TILE - 1) / TILE;
  long long c = (long long)ctx.num_sms * 6;  // about the resident CTAs of the scan pass
  if (c > kRtsMaxBlocks) c = kRtsMaxBlocks;
  if (c > tiles) c = tiles;
  if (c < 1) c = 1;
  const long long tiles_per_block = (tiles + c - 1) / c;
  a.per_block = tiles_per_block * TILE;
  a.nblocks = (int)((job.n + a.per_block - 1) / a.per_block);
  a.partials = (T*)((char*)job.temp + kHeaderBytes);
  a.init = T{};
  if (!job.inclusive && job.init_host) memcpy(&a.init, job.init_host, sizeof(T));
  a.inclusive = job.inclusive;
  a.vec_ok = ((uintptr_t)job.in % 16 == 0) && ((uintptr_t)job.out % 16 == 0);
  a.err = ctx.err;
  a.wait_ns = ctx.wait_ns;
  // The three launches follow one another with programmatic dependent launch; the
  // profile events (when set) bracket all three.
  profile_before(ctx);
  cudaError_t e = clear_status(job.temp, kHeaderBytes, nullptr, 0, ctx);  // the call's error word
  if (e == cudaSuccess) e = launch_pdl(rts_reduce_kernel<T, OP>, a.nblocks, 256, 0, ctx.stream, a);
  if (e == cudaSuccess)
    e = launch_pdl(rts_spine_kernel<T, OP>, 1, kRtsMaxBlocks, 0, ctx.stream, a.partials, a.nblocks);
  if (e == cudaSuccess) e = launch_pdl(rts_scan_kernel<T, OP, false>, a.nblocks, RowsGeom<T>::NT, 0, ctx.stream, a);
  profile_after(ctx);
  return e;
}

template <class T, int OP> cudaError_t launch_stf_op(const RtsJob& job, const LaunchCtx& ctx) {
  constexpr int TILE = RowsGeom<T>::TILE;
  RtsArgs<T> a;
  a.in = (const T*)job.in;
  a.out = (T*)job.out;
  a.n = job.n;
  const long long tiles = (job.n + TILE - 1) / TILE;
  long long c = (long long)ctx.num_sms * 6;
  if (c > kRtsMaxBlocks) c = kRtsMaxBlocks;
  if (c > tiles) c = tiles;
  if (c < 1) c = 1;
  const long long tiles_per_block = (tiles + c - 1) / c;
  a.per_block = tiles_per_block * TILE;
  a.nblocks = (int)((job.n + a.per_block - 1) / a.per_block);
  a.partials = (T*)((char*)job.temp + kHeaderBytes);
  a.init = T{};
  if (!job.inclusive && job.init_host) memcpy(&a.init, job.init_host, sizeof(T));
  a.inclusive = job.inclusive;
  a.vec_ok = ((uintptr_t)job.in % 16 == 0) && ((uintptr_t)job.out % 16 == 0);
  a.err = ctx.err;
  a.wait_ns = ctx.wait_ns;
  profile_before(ctx);
  cudaError_t e = clear_status(job.temp, kHeaderBytes, nullptr, 0, ctx);  // the call's error word
  if (e == cudaSuccess) e = launch_pdl(rts_scan_kernel<T, OP, true>, a.nblocks, RowsGeom<T>::NT, 0, ctx.stream, a);
  if (e == cudaSuccess)
    e = launch_pdl(rts_spine_kernel<T, OP>, 1, kRtsMaxBlocks, 0, ctx.stream, a.partials, a.nblocks);
  if (e == cudaSuccess) e = launch_pdl(stf_fan_kernel<T, OP>, a.nblocks, 256, 0, ctx.stream, a);
  profile_after(ctx);
  return e;
}

template <class T> cudaError_t launch_rts(const RtsJob& job, const LaunchCtx& ctx) {
  if (job.scan_then_fan) {
    switch (job.op) {
      case OP_ADD: return launch_stf_op<T, OP_ADD>(job, ctx);
      case OP_MAX: return launch_stf_op<T, OP_MAX>(job, ctx);
      case OP_MUL: return launch_stf_op<T, OP_MUL>(job, ctx);
      default: return launch_stf_op<T, OP_MIN>(job, ctx);
    }
  }
  switch (job.op) {
    case OP_ADD: return launch_rts_op<T, OP_ADD>(job, ctx);
    case OP_MAX: return launch_rts_op<T, OP_MAX>(job, ctx);
    case OP_MUL: return launch_rts_op<T, OP_MUL>(job, ctx);
    default: return launch_rts_op<T, OP_MIN>(job, ctx);
  }
}

}  // namespace gbs
