// segmented.cuh -- scans that restart at head flags: out_i combines x_h .. x_i, h the
// last head at or before i (element 0 is always a head).  The segmented operator on
// (value, flag) pairs,
//     (v1, f1) (+) (v2, f2) = (f2 ? v2 : v1 (+) v2,  f1 | f2),
// is associative but not commutative (The CUDA Handbook, 13.3.4: the single-pass
// descriptor as printed assumes a commutative operator; combining in tile order
// lifts that), so every combine in this kernel keeps index order:
//   - a lane owns K consecutive elements of a chunk (32 K elements) and folds them
//     serially; lanes, warps, chunks and segments are then combined in index order
//     (shuffle-up warp scans, a warp scan of the warp totals, and the segment gather
//     of scan_seg.cuh, whose lanes take consecutive blocks of segments);
//   - a segment's status word carries its aggregate value and, in the flag, whether
//     it holds a head (the FLAG_HEAD bit).
// One launch of the segment scheme: reduce (evict-last), publish, gather the earlier
// segments, rescan from L2 (evict-first) and write.
#pragma once

#include "scan_seg.cuh"

namespace gbs {

enum : unsigned { FLAG_HEAD = 4u };

// 8-byte values: one CTA per SM, so a lane's 8 values and flags stay in registers.
template <class T> struct SegmentedCfg {
  static constexpr int NT = 512, NW = NT / 32, MINB = sizeof(T) == 8 ? 1 : 2;
  static constexpr int K = 64 / (int)sizeof(T);  // elements per lane per chunk: 64 bytes
  static constexpr int CH = 32 * K;
  static constexpr int MAXSEG = 512, M = MAXSEG / 32;
};

template <class T> struct SegmentedArgs : SegArgsBase {
  const T* in;
  const unsigned char* flags;
  T* out;
  T init;
  int inclusive;
  int vec;  // in, out and flags 16-byte aligned: chunks move as vectors
};

// (av, af) <- (av, af) (+) (bv, bf)
template <class T, int OP>
__device__ __forceinline__ void pair_combine(T& av, bool& af, T bv, bool bf) {
  av = bf ? bv : Op<T, OP>::f(av, bv);
  af = af || bf;
}

// Inclusive warp scan of (value, flag) pairs in lane order.
template <class T, int OP> __device__ __forceinline__ void warp_inclusive_pair(T& v, bool& f, int lane) {
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const T nv = __shfl_up_sync(0xffffffffu, v, off);
    const bool nf = __shfl_up_sync(0xffffffffu, (int)f, off) != 0;
    if (lane >= off) {
      T a = nv;
      bool af = nf;
      pair_combine<T, OP>(a, af, v, f);
      v = a;
      f = af;
    }
  }
}

// A lane's K elements and head flags of chunk c (element 0 of the array is a head).
// Past n: value T{}, flag set (a head), so padding never reaches real elements.
template <class T, class G>
__device__ __forceinline__ void seg_pair_load(const SegmentedArgs<T>& a, long long c, int lane, T (&x)[G::K],
                                              unsigned& fl, unsigned long long pol) {
  constexpr int K = G::K, CH = G::CH;
  const long long e0 = c * CH + (long long)lane * K;
  if (a.vec && c * CH + CH <= a.n) {
    const uint4* p = reinterpret_cast<const uint4*>(a.in + e0);
    constexpr int Q = K * (int)sizeof(T) / 16;  // 16-byte pieces of the lane's values
    if (Q % 2 == 0 && ((uintptr_t)p & 31) == 0) {  // loads of whole sectors
#pragma unroll
      for (int q = 0; q < Q; q += 2) {
        uint4 lo, hi;
        ld_hint32(p + q, pol, lo, hi);
        memcpy(&x[q * 16 / sizeof(T)], &lo, 16);
        memcpy(&x[(q + 1) * 16 / sizeof(T)], &hi, 16);
      }
    } else {
#pragma unroll
      for (int q = 0; q < Q; ++q) {
        const uint4 u = ld_hint_l1(p + q, pol);
        memcpy(&x[q * 16 / sizeof(T)], &u, 16);
      }
    }
    unsigned w[4];  // the lane's K flag bytes (16, or 8 for 8-byte elements)
    if constexpr (K == 16) {
      const uint4 u = ld_hint(reinterpret_cast<const uint4*>(a.flags + e0), pol);
      w[0] = u.x, w[1] = u.y, w[2] = u.z, w[3] = u.w;
    } else {
      const uint2 u = *reinterpret_cast<const uint2*>(a.flags + e0);
      w[0] = u.x, w[1] = u.y, w[2] = w[3] = 0;
    }
    unsigned m = 0;
#pragma unroll
    for (int k = 0; k < K; ++k) m |= (((w[k >> 2] >> ((k & 3) * 8)) & 0xffu) != 0 ? 1u : 0u) << k;
    fl = m;
  } else {
    unsigned m = 0;
#pragma unroll
    for (int k = 0; k < K; ++k) {
      const long long i = e0 + k;
      x[k] = i < a.n ? a.in[i] : T{};
      m |= (i >= a.n || a.flags[i] != 0 ? 1u : 0u) << k;
    }
    fl = m;
  }
  if (e0 == 0) fl |= 1u;
}

// A full chunk leaves through the warp's staging buffer (32 lanes x 4 granules of 16
// bytes): lane l puts its granule q at l*4 + (q ^ ((l >> 1) & 3)), which spreads every
// 8 lanes over the 8 granule slots of 128 bytes (no bank conflict), then the warp
// stores the chunk's 2 KB as consecutive 16-byte pieces, whole lines per instruction.
// A lane's 64-byte stride alone would leave each store instruction half lines.
template <class T, class G>
__device__ __forceinline__ void seg_pair_store(const SegmentedArgs<T>& a, long long c, int lane, const T (&y)[G::K],
                                               uint4* stage, unsigned long long pol) {
  constexpr int K = G::K, CH = G::CH, GR = K * (int)sizeof(T) / 16;  // granules per lane: 4
  const long long e0 = c * CH + (long long)lane * K;
  if (a.vec && c * CH + CH <= a.n) {
    __syncwarp();  // the previous chunk's stores have read the buffer
#pragma unroll
    for (int q = 0; q < GR; ++q) {
      uint4 u;
      memcpy(&u, &y[q * 16 / sizeof(T)], 16);
      stage[lane * GR + (q ^ ((lane >> 1) & 3))] = u;
    }
    __syncwarp();
    uint4* base = reinterpret_cast<uint4*>(a.out + c * CH);
#pragma unroll
    for (int it = 0; it < GR; ++it) {
      const int g = it * 32 + lane, l = g / GR, q = (g % GR) ^ ((l >> 1) & 3);
      st_hint(base + l * GR + q, stage[g], pol);
    }
  } else {
#pragma unroll
    for (int k = 0; k < K; ++k)
      if (e0 + k < a.n) a.out[e0 + k] = y[k];
  }
}

// Phase 2 for pairs: the ordered combination of segments 0 .. cnt-1 (lane l takes a
// block of consecutive segments), the head bit riding in the flag.
template <class T, int OP, int M, class S>
__device__ __forceinline__ void seg_gather_pair(const S& st, unsigned cnt, unsigned long long wait_ns, T& rv, bool& rf,
                                                bool& timed_out) {
  const int lane = threadIdx.x & 31;
  const unsigned per = (cnt + 31) / 32, mine = (unsigned)lane * per;
  T val[M];
  unsigned fl[M];
  unsigned pending = 0;
#pragma unroll
  for (int k = 0; k < M; ++k)
    if ((unsigned)k < per && mine + k < cnt) pending |= 1u << k;
  unsigned long long t0 = 0;
  timed_out = false;
  for (int spins = 0;; ++spins) {
#pragma unroll
    for (int k = 0; k < M; ++k) {
      if (pending & (1u << k)) {
        T v;
        const unsigned f = st.poll(mine + k, v);
        if (f != FLAG_X) {
          val[k] = st.fetch(mine + k, f, v);
          fl[k] = f;
          pending &= ~(1u << k);
        }
      }
    }
    if (__all_sync(0xffffffffu, pending == 0)) break;
    unsigned long long now = 0;
    if (lane == 0) now = globaltimer();
    now = __shfl_sync(0xffffffffu, now, 0);
    if (spins == 0) t0 = now;
    else if (now - t0 > wait_ns) {
      timed_out = true;
#pragma unroll
      for (int k = 0; k < M; ++k)
        if (pending & (1u << k)) {
          val[k] = T{};
          fl[k] = FLAG_A | FLAG_HEAD;
        }
      break;
    }
    backoff(spins);
  }
  // Lanes hold consecutive blocks from lane 0 on; lanes past the last one hold none
  // and take no part.
  const bool real = mine < cnt;
  T v = real ? val[0] : T{};
  bool f = real && (fl[0] & FLAG_HEAD) != 0;
#pragma unroll
  for (int k = 1; k < M; ++k)
    if ((unsigned)k < per && mine + k < cnt) pair_combine<T, OP>(v, f, val[k], (fl[k] & FLAG_HEAD) != 0);
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const T nv = __shfl_up_sync(0xffffffffu, v, off);
    const bool nf = __shfl_up_sync(0xffffffffu, (int)f, off) != 0;
    if (lane >= off && real) {  // lanes below a real lane are real
      T t = nv;
      bool tf = nf;
      pair_combine<T, OP>(t, tf, v, f);
      v = t;
      f = tf;
    }
  }
  const int last = (int)((cnt + per - 1) / per) - 1;  // the last lane holding segments
  rv = __shfl_sync(0xffffffffu, v, last);
  rf = __shfl_sync(0xffffffffu, (int)f, last) != 0;
}

template <class T, int OP, class G, class S>
__global__ void __launch_bounds__(G::NT, G::MINB) scan_segmented_kernel(SegmentedArgs<T> a, S st) {
  pdl_entry();
  constexpr int NW = G::NW, K = G::K;
  __shared__ unsigned s_seg;
  __shared__ T s_wv[NW];
  __shared__ int s_wf[NW];
  __shared__ T s_bv;
  __shared__ int s_bf, s_bhas;
  __shared__ uint4 s_stage_all[NW * 32 * (K * sizeof(T) / 16)];  // a chunk's outputs per warp
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint4* s_stage = s_stage_all + warp * 32 * (K * sizeof(T) / 16);
  if (tid == 0) s_seg = atomicAdd(a.counter, 1u);
  __syncthreads();
  const unsigned seg = s_seg;
  long long c0, c1;
  const int nact = seg_chunks(a, seg, warp, NW, c0, c1);

  // Phase 1: the warp's aggregate pair over its chunks, in order.
  {
    const unsigned long long keep = l2_policy_evict_last();
    T wv{};
    bool wf = false, whas = false;
    for (long long c = c0; c < c1; ++c) {
      T x[K];
      unsigned fl;
      seg_pair_load<T, G>(a, c, lane, x, fl, keep);
      T lv = x[0];
      bool lf = fl & 1u;
#pragma unroll
      for (int k = 1; k < K; ++k) pair_combine<T, OP>(lv, lf, x[k], (fl >> k) & 1u);
      warp_inclusive_pair<T, OP>(lv, lf, lane);
      const T cv = __shfl_sync(0xffffffffu, lv, 31);
      const bool cf = __shfl_sync(0xffffffffu, (int)lf, 31) != 0;
      if (whas) pair_combine<T, OP>(wv, wf, cv, cf);
      else {
        wv = cv;
        wf = cf;
        whas = true;
      }
    }
    if (lane == 0) {
      s_wv[warp] = wv;
      s_wf[warp] = wf;
    }
  }
  __syncthreads();

  // Phase 2: warp 0 scans the warp pairs, publishes the segment's pair and gathers
  // the earlier segments' pairs.
  if (warp == 0) {
    T v = s_wv[lane < nact ? lane : nact - 1];
    bool f = s_wf[lane < nact ? lane : nact - 1] != 0;
    warp_inclusive_pair<T, OP>(v, f, lane);
    if (lane < nact) {
      s_wv[lane] = v;
      s_wf[lane] = f;
    }
    const T av = __shfl_sync(0xffffffffu, v, nact - 1);
    const bool af = __shfl_sync(0xffffffffu, (int)f, nact - 1) != 0;
    if (lane == 0 && (long long)seg != a.stalled) st.publish(seg, FLAG_A | (af ? FLAG_HEAD : 0u), av);
    T bv{};
    bool bf = false, timed_out = false;
    if (seg > 0) seg_gather_pair<T, OP, G::M>(st, seg, a.wait_ns, bv, bf, timed_out);
    if (lane == 0) {
      if (timed_out) raise_err(a.err, ERRBIT_TIMEOUT);
      s_bv = bv;
      s_bf = bf;
      s_bhas = seg > 0;
    }
  }
  __syncthreads();

  // Phase 3: rescan from L2.  The carry into the warp's part: the segment base, then
  // the earlier warps of the segment.
  T cv = s_bv;
  bool chas = s_bhas != 0;
  if (warp > 0) {
    const T pv = s_wv[warp - 1];
    const bool pf = s_wf[warp - 1] != 0;
    if (chas) {
      bool dummy = false;
      pair_combine<T, OP>(cv, dummy, pv, pf);
    } else {
      cv = pv;
      chas = true;
    }
  }
  const unsigned long long drop = l2_policy_evict_first();
  for (long long c = c0; c < c1; ++c) {
    T x[K];
    unsigned fl;
    seg_pair_load<T, G>(a, c, lane, x, fl, drop);
    // The lane's pair, the exclusive scan of the lanes before it, then the chunk's
    // carry on their left.
    T lv = x[0];
    bool lf = fl & 1u;
#pragma unroll
    for (int k = 1; k < K; ++k) pair_combine<T, OP>(lv, lf, x[k], (fl >> k) & 1u);
    T iv = lv;
    bool ifl = lf;
    warp_inclusive_pair<T, OP>(iv, ifl, lane);
    T ev = __shfl_up_sync(0xffffffffu, iv, 1);
    bool ef = __shfl_up_sync(0xffffffffu, (int)ifl, 1) != 0;
    bool ehas = lane > 0;
    if (chas) {
      if (ehas) {
        T t = cv;
        bool tf = false;
        pair_combine<T, OP>(t, tf, ev, ef);
        ev = t;
      } else {
        ev = cv;
      }
      ehas = true;
    }
    // The chunk's carry for the next one: carry (+) the chunk's pair.
    const T tv = __shfl_sync(0xffffffffu, iv, 31);
    const bool tf = __shfl_sync(0xffffffffu, (int)ifl, 31) != 0;
    if (chas) {
      bool dummy = false;
      pair_combine<T, OP>(cv, dummy, tv, tf);
    } else {
      cv = tv;
      chas = true;
    }
    // Serial scan of the lane's elements: `run` is the segment-local inclusive value
    // of the previous element (ehas: it exists, i.e. this is not element 0).
    T run = ev;
    bool rhas = ehas;
    T y[K];
#pragma unroll
    for (int k = 0; k < K; ++k) {
      const bool head = (fl >> k) & 1u;
      if (a.inclusive) {
        run = (head || !rhas) ? x[k] : Op<T, OP>::f(run, x[k]);
        y[k] = run;
      } else {
        y[k] = (head || !rhas) ? a.init : Op<T, OP>::f(a.init, run);
        run = (head || !rhas) ? x[k] : Op<T, OP>::f(run, x[k]);
      }
      rhas = true;
    }
    seg_pair_store<T, G>(a, c, lane, y, s_stage, drop);
  }
}

template <class T> size_t segmented_temp_bytes() { return kHeaderBytes + seg_status_bytes<T>(); }

template <class T, int OP> cudaError_t launch_segmented_op(const SegmentedJob& job, const LaunchCtx& ctx) {
  using G = SegmentedCfg<T>;
  const SegPlan p = seg_plan<G>(1, job.n, ctx.num_sms);
  if (p.ctas == 0) return cudaSuccess;
  SegmentedArgs<T> a;
  a.n = job.n;
  a.nc = p.nc;
  a.segs = p.segs;
  a.ctas = p.ctas;
  a.counter = (unsigned*)job.temp;
  a.err = ctx.err;
  a.wait_ns = ctx.wait_ns;
  a.stalled = ctx.stalled_tile;
  a.in = (const T*)job.in;
  a.flags = (const unsigned char*)job.flags;
  a.out = (T*)job.out;
  a.init = T{};
  if (job.init_host) memcpy(&a.init, job.init_host, sizeof(T));
  a.inclusive = job.inclusive;
  a.vec = ((uintptr_t)job.in % 16 == 0) && ((uintptr_t)job.out % 16 == 0) && ((uintptr_t)job.flags % 16 == 0);
  auto st = seg_status<T>(job.temp);
  profile_before(ctx);
  cudaError_t e = clear_status(job.temp, seg_reset_bytes<T>(), nullptr, 0, ctx);
  if (e == cudaSuccess)
    e = launch_pdl(scan_segmented_kernel<T, OP, G, decltype(st)>, p.ctas, G::NT, 0, ctx.stream, a, st);
  profile_after(ctx);
  return e;
}

template <class T> cudaError_t launch_segmented(const SegmentedJob& job, const LaunchCtx& ctx) {
  switch (job.op) {
    case OP_ADD: return launch_segmented_op<T, OP_ADD>(job, ctx);
    case OP_MAX: return launch_segmented_op<T, OP_MAX>(job, ctx);
    case OP_MUL: return launch_segmented_op<T, OP_MUL>(job, ctx);
    default: return launch_segmented_op<T, OP_MIN>(job, ctx);
  }
}

}  // namespace gbs
