// scan_affine.cuh -- scans under an operator that is associative but not
// commutative: composition of affine maps.
//
// Element i is the map f_i(y) = a_i * y + b_i over one unsigned integer type
// (signed types give the same bits), stored as the pair (a_i, b_i).  The operator
// applies the earlier map first:
//     (a1, b1) (+) (a2, b2) = (a1 a2,  a2 b1 + b2),       identity (1, 0),
// so the b of an inclusive prefix is the value y_i of the first-order linear
// recurrence y_i = a_i y_{i-1} + b_i started from 0.  The CUDA Handbook, 13.3.4,
// notes that its packed single-pass descriptor assumes a commutative operator;
// here every combination keeps index order (earlier terms on the left):
//   - a lane owns K consecutive elements (64 bytes) of a chunk or tile and folds
//     them serially; lanes combine by shuffle-up scans in lane order, warps by a
//     scan of the warp totals in warp order, segments by the ordered gather;
//   - the look-back combines the predecessors' values from the nearest inclusive
//     prefix forward.
// Two kernels, as for the other scans:
//   scan_affine_seg_kernel   one aligned row that fits in L2 (96 MiB): reduce,
//                            publish, gather every earlier segment, rescan from L2;
//   scan_affine_tile_kernel  any other row: one CTA per tile claimed in order, the
//                            tile's aggregate published, decoupled look-back over
//                            flag + value status words (a value of 8 or 16 bytes
//                            never fits one word with its flag, so the flag is
//                            stored with release semantics after the value).
#pragma once

#include "scan_seg.cuh"

namespace gbs {

template <class T> struct Aff {
  T a, b;
};

template <class T> __device__ __forceinline__ Aff<T> aff_identity() {
  Aff<T> r;
  r.a = T(1);
  r.b = T(0);
  return r;
}
// l (+) r: apply l, then r.  Unsigned arithmetic wraps modulo 2^w.
template <class T> __device__ __forceinline__ Aff<T> aff_then(const Aff<T>& l, const Aff<T>& r) {
  Aff<T> o;
  o.a = l.a * r.a;
  o.b = r.a * l.b + r.b;
  return o;
}
template <class T> __device__ __forceinline__ Aff<T> aff_shfl_up(const Aff<T>& v, int d) {
  Aff<T> o;
  o.a = __shfl_up_sync(0xffffffffu, v.a, d);
  o.b = __shfl_up_sync(0xffffffffu, v.b, d);
  return o;
}
template <class T> __device__ __forceinline__ Aff<T> aff_shfl_down(const Aff<T>& v, int d) {
  Aff<T> o;
  o.a = __shfl_down_sync(0xffffffffu, v.a, d);
  o.b = __shfl_down_sync(0xffffffffu, v.b, d);
  return o;
}
template <class T> __device__ __forceinline__ Aff<T> aff_shfl_idx(const Aff<T>& v, int src) {
  Aff<T> o;
  o.a = __shfl_sync(0xffffffffu, v.a, src);
  o.b = __shfl_sync(0xffffffffu, v.b, src);
  return o;
}

// Inclusive scan over the warp in lane order.  The map a lane receives from below
// its own range is replaced by the identity, so every step is one unconditional
// composition and no lane needs a guard.
template <class T> __device__ __forceinline__ Aff<T> aff_warp_inclusive(Aff<T> v, int lane) {
  const Aff<T> id = aff_identity<T>();
#pragma unroll
  for (int d = 1; d < 32; d *= 2) {
    const Aff<T> below = aff_shfl_up(v, d);
    v = aff_then(lane >= d ? below : id, v);
  }
  return v;
}
// The exclusive value of each lane (the identity in lane 0) from the inclusive one.
template <class T> __device__ __forceinline__ Aff<T> aff_lane_exclusive(const Aff<T>& inc, int lane) {
  const Aff<T> e = aff_shfl_up(inc, 1);
  return lane > 0 ? e : aff_identity<T>();
}

// A lane's K consecutive maps (64 bytes) starting at element e0; maps past n read as
// the identity (they only reach outputs that are not stored).  `vec`: the 64 bytes
// are whole and 16-byte aligned.
template <class T, int K>
__device__ __forceinline__ void aff_load(Aff<T> (&x)[K], const T* in, long long e0, long long n, bool vec,
                                         unsigned long long pol) {
  static_assert(K * sizeof(Aff<T>) == 64, "a lane owns 64 bytes");
  if (vec && e0 + K <= n) {
    const uint4* p = reinterpret_cast<const uint4*>(in + 2 * e0);
    if (((uintptr_t)p & 31) == 0) {  // two loads of whole sectors
#pragma unroll
      for (int q = 0; q < 4; q += 2) {
        uint4 lo, hi;
        ld_hint32(p + q, pol, lo, hi);
        memcpy(reinterpret_cast<char*>(x) + 16 * q, &lo, 16);
        memcpy(reinterpret_cast<char*>(x) + 16 * q + 16, &hi, 16);
      }
    } else {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint4 u = ld_hint_l1(p + q, pol);
        memcpy(reinterpret_cast<char*>(x) + 16 * q, &u, 16);
      }
    }
  } else {
#pragma unroll
    for (int k = 0; k < K; ++k) {
      if (e0 + k < n) {
        x[k].a = in[2 * (e0 + k)];
        x[k].b = in[2 * (e0 + k) + 1];
      } else {
        x[k] = aff_identity<T>();
      }
    }
  }
}

// Writes a warp's 32 lanes x 64 bytes of whole, aligned output through the warp's
// 2 KB staging buffer: lane l puts its granule q at l*4 + (q ^ ((l >> 1) & 3)), which
// spreads every 8 lanes over the 8 granule slots of a 128-byte line (no bank
// conflict); the warp then stores the 2 KB as consecutive 16-byte pieces, whole lines
// per instruction.  A lane's own 64-byte stride would leave each store half lines.
template <class T, int K>
__device__ __forceinline__ void aff_store_staged(T* out_warp, const Aff<T> (&y)[K], uint4* stage, int lane,
                                                 unsigned long long pol) {
  __syncwarp();  // the previous stores have read the buffer
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint4 u;
    memcpy(&u, reinterpret_cast<const char*>(y) + 16 * q, 16);
    stage[lane * 4 + (q ^ ((lane >> 1) & 3))] = u;
  }
  __syncwarp();
  uint4* base = reinterpret_cast<uint4*>(out_warp);
#pragma unroll
  for (int it = 0; it < 4; ++it) {
    const int g = it * 32 + lane, l = g / 4, q = (g % 4) ^ ((l >> 1) & 3);
    st_hint(base + l * 4 + q, stage[g], pol);
  }
}
template <class T, int K>
__device__ __forceinline__ void aff_store_plain(T* out, const Aff<T> (&y)[K], long long e0, long long n) {
#pragma unroll
  for (int k = 0; k < K; ++k)
    if (e0 + k < n) {
      out[2 * (e0 + k)] = y[k].a;
      out[2 * (e0 + k) + 1] = y[k].b;
    }
}

// Serial scan of a lane's maps from `pre` (everything before the lane's first map,
// the initial map included).  Inclusive: y_k = pre (+) x_0 (+) ... (+) x_k;
// exclusive: y_k = pre (+) x_0 (+) ... (+) x_{k-1}.
template <class T, int K>
__device__ __forceinline__ void aff_lane_scan(Aff<T> (&x)[K], Aff<T> pre, bool inclusive) {
#pragma unroll
  for (int k = 0; k < K; ++k) {
    const Aff<T> nxt = aff_then(pre, x[k]);
    x[k] = inclusive ? nxt : pre;
    pre = nxt;
  }
}

template <class T, int K> __device__ __forceinline__ Aff<T> aff_fold(const Aff<T> (&x)[K]) {
  Aff<T> t = x[0];
#pragma unroll
  for (int k = 1; k < K; ++k) t = aff_then(t, x[k]);
  return t;
}

// Status words of a map: a flag per unit, and the map in its own slot (aggregate and
// inclusive prefix separate, so a reader that saw A never picks up a later P).  The
// value is stored first, then the flag with release semantics; a reader loads the
// flag with acquire semantics, then the value.
template <class T> struct AffStatus {
  unsigned* flag;
  Aff<T>* agg;
  Aff<T>* pfx;
  __device__ __forceinline__ void publish(long long i, unsigned f, const Aff<T>& v) const {
    Aff<T>* s = (f == FLAG_A ? agg : pfx) + i;
    st_relaxed(&s->a, v.a);
    st_relaxed(&s->b, v.b);
    st_release_u32(flag + i, f);
  }
  __device__ __forceinline__ unsigned poll(long long i) const { return ld_acquire_u32(flag + i); }
  __device__ __forceinline__ Aff<T> fetch(long long i, unsigned f) const {
    const Aff<T>* s = (f == FLAG_A ? agg : pfx) + i;
    Aff<T> v;
    v.a = ld_relaxed(&s->a);
    v.b = ld_relaxed(&s->b);
    return v;
  }
};

// The segment kernel's status (aggregates only): every 8-byte piece of a segment's
// map and its complement, in relaxed stores; a reader takes the map once each piece
// has its complement beside it (the words start at zero each launch, so an accepted
// pair always holds the piece written).  No flag is released after the values, so a
// gather needs no acquire and keeps all its loads in flight together.
template <class T> struct AffSegStatus {
  static constexpr int P = sizeof(Aff<T>) / 8;  // 8-byte pieces of a map
  unsigned long long* w;                        // [segment][P][2]
  __device__ __forceinline__ void publish(long long i, const Aff<T>& v) const {
    unsigned long long x[P];
    memcpy(x, &v, sizeof(x));
#pragma unroll
    for (int j = 0; j < P; ++j) {
      st_relaxed_u64(w + (i * P + j) * 2, x[j]);
      st_relaxed_u64(w + (i * P + j) * 2 + 1, ~x[j]);
    }
  }
  __device__ __forceinline__ bool poll(long long i, Aff<T>& v) const {
    unsigned long long x[P];
    bool ok = true;
#pragma unroll
    for (int j = 0; j < P; ++j) {
      x[j] = ld_relaxed_u64(w + (i * P + j) * 2);
      ok = ok && ld_relaxed_u64(w + (i * P + j) * 2 + 1) == ~x[j];
    }
    memcpy(&v, x, sizeof(x));
    return ok;
  }
};
static_assert(sizeof(Aff<unsigned>) == 8 && sizeof(Aff<unsigned long long>) == 16, "maps are whole 8-byte pieces");

template <class T> size_t aff_status_bytes(size_t units) {
  return round_up(units * 4, 256) + 2 * round_up(units * sizeof(Aff<T>), 256);
}
template <class T> AffStatus<T> aff_status(void* temp, size_t units) {
  AffStatus<T> st;
  char* p = (char*)temp + kHeaderBytes;
  st.flag = (unsigned*)p;
  p += round_up(units * 4, 256);
  st.agg = (Aff<T>*)p;
  p += round_up(units * sizeof(Aff<T>), 256);
  st.pfx = (Aff<T>*)p;
  return st;
}

template <class T> struct AffArgs : SegArgsBase {
  const T* in;
  T* out;
  Aff<T> start;  // identity (inclusive) or the caller's initial map (exclusive)
  int inclusive;
  int vec;       // in and out 16-byte aligned
};

// ---- one aligned row that fits in L2: the segment scheme -------------------------------

// 64-bit maps take twice the registers (and emulated 64-bit multiplies): one CTA of
// 512 threads per SM keeps them out of local memory.
template <class T> struct AffSegCfg {
  static constexpr int NT = 512, NW = NT / 32, MINB = sizeof(T) == 8 ? 1 : 2;
  static constexpr int K = 64 / (int)sizeof(Aff<T>);  // maps per lane per chunk
  static constexpr int CH = 32 * K;                    // maps per chunk (2 KB)
  static constexpr int MAXSEG = 512, M = MAXSEG / 32;
};

// Phase 2: the ordered composition of segments 0 .. cnt-1 (cnt >= 1), each waited
// for (bounded by wait_ns).  Lane l takes the consecutive block [l P, l P + P), P =
// ceil(cnt / 32); blocks then combine in lane order.  Returns it in every lane.
template <class T, int M>
__device__ __forceinline__ Aff<T> aff_gather(const AffSegStatus<T>& st, unsigned cnt, unsigned long long wait_ns,
                                             bool& timed_out) {
  const int lane = threadIdx.x & 31;
  const unsigned per = (cnt + 31) / 32, mine = (unsigned)lane * per;
  Aff<T> val[M];
  unsigned pending = 0;
#pragma unroll
  for (int k = 0; k < M; ++k) {
    val[k] = aff_identity<T>();
    if ((unsigned)k < per && mine + k < cnt) pending |= 1u << k;
  }
  unsigned long long t0 = 0;
  timed_out = false;
  for (int spins = 0;; ++spins) {
#pragma unroll
    for (int k = 0; k < M; ++k)
      if (pending & (1u << k)) {
        Aff<T> v;
        if (st.poll(mine + k, v)) {
          val[k] = v;
          pending &= ~(1u << k);
        }
      }
    if (__all_sync(0xffffffffu, pending == 0)) break;
    unsigned long long now = 0;
    if (lane == 0) now = globaltimer();
    now = __shfl_sync(0xffffffffu, now, 0);
    if (spins == 0) t0 = now;
    else if (now - t0 > wait_ns) {
      timed_out = true;
      break;  // what was not read stays the identity
    }
    backoff(spins);
  }
  Aff<T> v = val[0];
#pragma unroll
  for (int k = 1; k < M; ++k) v = aff_then(v, val[k]);  // entries past the block are the identity
  v = aff_warp_inclusive(v, lane);
  return aff_shfl_idx(v, 31);
}

template <class T, class G>
__global__ void __launch_bounds__(G::NT, G::MINB) scan_affine_seg_kernel(AffArgs<T> a, AffSegStatus<T> st) {
  pdl_entry();
  constexpr int NW = G::NW, K = G::K, CH = G::CH;
  __shared__ unsigned s_seg;
  __shared__ Aff<T> s_w[NW];
  __shared__ Aff<T> s_base;
  __shared__ uint4 s_stage_all[NW * 32 * 4];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint4* stage = s_stage_all + warp * 32 * 4;
  if (tid == 0) s_seg = atomicAdd(a.counter, 1u);
  __syncthreads();
  const unsigned seg = s_seg;
  long long c0, c1;
  const int nact = seg_chunks(a, seg, warp, NW, c0, c1);

  // Phase 1: the warp's composition of its chunks, in order (evict-last loads, so
  // the rescan finds the lines in L2).  The next chunk is requested before the
  // current one is folded: with one 2 KB chunk per warp in flight, the SM would wait
  // on HBM latency instead of moving the input at the bandwidth it shares.
  {
    const unsigned long long keep = l2_policy_evict_last();
    Aff<T> w = aff_identity<T>();
    Aff<T> x[K];
    if (c0 < c1) aff_load<T, K>(x, a.in, c0 * CH + (long long)lane * K, a.n, true, keep);
    for (long long c = c0; c < c1; ++c) {
      Aff<T> nx[K];
      if (c + 1 < c1) aff_load<T, K>(nx, a.in, (c + 1) * CH + (long long)lane * K, a.n, true, keep);
      const Aff<T> inc = aff_warp_inclusive(aff_fold<T, K>(x), lane);
      w = aff_then(w, aff_shfl_idx(inc, 31));
#pragma unroll
      for (int k = 0; k < K; ++k) x[k] = nx[k];
    }
    if (lane == 0) s_w[warp] = w;
  }
  __syncthreads();

  // Phase 2: warp 0 scans the warp totals in order, publishes the segment's map and
  // composes every earlier segment's.
  if (warp == 0) {
    Aff<T> v = lane < nact ? s_w[lane] : aff_identity<T>();
    v = aff_warp_inclusive(v, lane);
    if (lane < nact) s_w[lane] = v;
    const Aff<T> agg = aff_shfl_idx(v, 31);
    if (lane == 0 && (long long)seg != a.stalled) st.publish(seg, agg);
    Aff<T> before = aff_identity<T>();
    bool timed_out = false;
    if (seg > 0) before = aff_gather<T, G::M>(st, seg, a.wait_ns, timed_out);
    if (lane == 0) {
      if (timed_out) raise_err(a.err, ERRBIT_TIMEOUT);
      s_base = aff_then(a.start, before);
    }
  }
  __syncthreads();

  // Phase 3: rescan from L2 (evict-first) and write.
  Aff<T> carry = s_base;
  if (warp > 0) carry = aff_then(carry, s_w[warp - 1]);
  const unsigned long long drop = l2_policy_evict_first();
  Aff<T> nx[K];  // the next chunk, requested before this one is scanned
  if (c0 < c1) aff_load<T, K>(nx, a.in, c0 * CH + (long long)lane * K, a.n, true, drop);
  for (long long c = c0; c < c1; ++c) {
    Aff<T> x[K];
#pragma unroll
    for (int k = 0; k < K; ++k) x[k] = nx[k];
    const long long e0 = c * CH + (long long)lane * K;
    if (c + 1 < c1) aff_load<T, K>(nx, a.in, e0 + CH, a.n, true, drop);
    const Aff<T> inc = aff_warp_inclusive(aff_fold<T, K>(x), lane);
    const Aff<T> pre = aff_then(carry, aff_lane_exclusive(inc, lane));
    carry = aff_then(carry, aff_shfl_idx(inc, 31));
    aff_lane_scan<T, K>(x, pre, a.inclusive != 0);
    if (c * CH + CH <= a.n) aff_store_staged<T, K>(a.out + 2 * c * CH, x, stage, lane, drop);
    else aff_store_plain<T, K>(a.out, x, e0, a.n);
  }
}

// ---- any other row: one CTA per tile, decoupled look-back ---------------------------

template <class T> struct AffTileCfg {
  static constexpr int NT = 256, NW = NT / 32, MINB = 4;
  static constexpr int K = 64 / (int)sizeof(Aff<T>);
  static constexpr int TILE = NW * 32 * K;  // maps per tile (16 KB)
};

// Warp-cooperative look-back in tile order: lane l reads the status of tile
// tt-1-l (lane 0 the nearest).  While any tile from the frontier back to the nearest
// P is still X, those entries (only) are read again, bounded by wait_ns.  Then lanes
// 0 .. nearest compose their maps with earlier tiles on the left; with no P in the
// window, all 32 aggregates are composed and the walk steps back 32 tiles.  Returns
// the tile's exclusive prefix in every lane.
template <class T>
__device__ __forceinline__ Aff<T> aff_lookback(const AffStatus<T>& st, long long tt, unsigned long long wait_ns,
                                               bool& timed_out) {
  const int lane = threadIdx.x & 31;
  long long frontier = tt - 1;
  Aff<T> acc = aff_identity<T>();
  timed_out = false;
  for (;;) {
    const long long p = frontier - lane;
    unsigned f = p >= 0 ? st.poll(p) : FLAG_P;  // before tile 0: stops the walk
    int spins = 0;
    unsigned long long t0 = 0;
    int nearest;
    for (;;) {
      const unsigned pm = __ballot_sync(0xffffffffu, f == FLAG_P);
      nearest = pm ? __ffs(pm) - 1 : 32;
      const bool blocking = lane <= nearest && f == FLAG_X;
      if (!__any_sync(0xffffffffu, blocking)) break;
      if (spins == 0) t0 = __shfl_sync(0xffffffffu, globaltimer(), 0);
      else if (__shfl_sync(0xffffffffu, globaltimer(), 0) - t0 > wait_ns) {
        timed_out = true;
        break;
      }
      backoff(spins++);
      if (blocking) f = st.poll(p);
    }
    Aff<T> v = aff_identity<T>();
    if (lane <= nearest && p >= 0 && f != FLAG_X) v = st.fetch(p, f);
    // Ordered composition of lanes 0 .. last: lane k holds a later tile than k + 1,
    // so the value from the higher lane goes on the left.
    const int last = nearest < 32 ? nearest : 31;
#pragma unroll
    for (int d = 1; d < 32; d *= 2) {
      const Aff<T> hi = aff_shfl_down(v, d);
      if (lane + d <= last) v = aff_then(hi, v);
    }
    acc = aff_then(aff_shfl_idx(v, 0), acc);
    timed_out = __any_sync(0xffffffffu, timed_out);
    if (nearest < 32 || timed_out) break;
    frontier -= 32;
  }
  return acc;
}

template <class T, class G>
__global__ void __launch_bounds__(G::NT, G::MINB) scan_affine_tile_kernel(AffArgs<T> a, AffStatus<T> st) {
  pdl_entry();
  constexpr int NW = G::NW, K = G::K, TILE = G::TILE;
  __shared__ unsigned s_tile;
  __shared__ Aff<T> s_w[NW];
  __shared__ Aff<T> s_prefix;
  __shared__ uint4 s_stage_all[NW * 32 * 4];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint4* stage = s_stage_all + warp * 32 * 4;
  if (tid == 0) s_tile = atomicAdd(a.counter, 1u);
  __syncthreads();
  const long long t = s_tile;
  const long long e0 = t * TILE + (long long)(warp * 32 + lane) * K;
  const unsigned long long drop = l2_policy_evict_first();
  Aff<T> x[K];
  aff_load<T, K>(x, a.in, e0, a.n, a.vec != 0, drop);
  const Aff<T> inc = aff_warp_inclusive(aff_fold<T, K>(x), lane);
  if (lane == 31) s_w[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    Aff<T> v = lane < NW ? s_w[lane] : aff_identity<T>();
    v = aff_warp_inclusive(v, lane);
    if (lane < NW) s_w[lane] = v;
    const Aff<T> agg = aff_shfl_idx(v, NW - 1);
    Aff<T> pfx = aff_identity<T>();
    if (t == 0) {
      if (lane == 0 && t != a.stalled) st.publish(0, FLAG_P, agg);
    } else {
      if (lane == 0 && t != a.stalled) st.publish(t, FLAG_A, agg);
      bool timed_out;
      pfx = aff_lookback<T>(st, t, a.wait_ns, timed_out);
      if (lane == 0) {
        if (t != a.stalled) st.publish(t, FLAG_P, aff_then(pfx, agg));
        if (timed_out) raise_err(a.err, ERRBIT_TIMEOUT);
      }
    }
    if (lane == 0) s_prefix = aff_then(a.start, pfx);
  }
  __syncthreads();
  Aff<T> pre = s_prefix;
  if (warp > 0) pre = aff_then(pre, s_w[warp - 1]);
  pre = aff_then(pre, aff_lane_exclusive(inc, lane));
  aff_lane_scan<T, K>(x, pre, a.inclusive != 0);
  const long long w0 = t * TILE + (long long)warp * 32 * K;  // the warp's first map
  if (a.vec && w0 + 32 * K <= a.n) aff_store_staged<T, K>(a.out + 2 * w0, x, stage, lane, drop);
  else aff_store_plain<T, K>(a.out, x, e0, a.n);
}

// ---- dispatch --------------------------------------------------------------------

template <class T> bool aff_seg_applies(const ScanJob& job) {
  return job.B == 1 && (uintptr_t)job.in % 16 == 0 && (uintptr_t)job.out % 16 == 0 &&
         job.R * (long long)sizeof(Aff<T>) <= kSegMaxBytes;
}

template <class T> size_t affine_temp_bytes(long long n) {
  const size_t tiles = (size_t)((n + AffTileCfg<T>::TILE - 1) / AffTileCfg<T>::TILE);
  const size_t a = kHeaderBytes + aff_status_bytes<T>(tiles);
  const size_t b = kHeaderBytes + aff_status_bytes<T>(AffSegCfg<T>::MAXSEG);
  return a > b ? a : b;
}

// One row of job.R maps (job.in / job.out hold 2 R values of T); job.init_host is
// the initial map (exclusive scans; NULL: the identity).
template <class T> cudaError_t launch_affine(const ScanJob& job, const LaunchCtx& ctx) {
  static_assert(std::is_unsigned<T>::value, "affine maps wrap: unsigned arithmetic");
  if (job.B != 1 || job.C != 2) return cudaErrorInvalidValue;
  AffArgs<T> a;
  a.n = job.R;
  a.counter = (unsigned*)job.temp;
  a.err = ctx.err;
  a.wait_ns = ctx.wait_ns;
  a.stalled = ctx.stalled_tile;
  a.in = (const T*)job.in;
  a.out = (T*)job.out;
  a.start.a = T(1);
  a.start.b = T(0);
  if (!job.inclusive && job.init_host) memcpy(&a.start, job.init_host, sizeof(Aff<T>));
  a.inclusive = job.inclusive;
  a.vec = (uintptr_t)job.in % 16 == 0 && (uintptr_t)job.out % 16 == 0;
  cudaError_t e;
  if (aff_seg_applies<T>(job)) {
    using G = AffSegCfg<T>;
    const SegPlan p = seg_plan<G>(1, job.R, ctx.num_sms);
    if (p.ctas == 0) return cudaErrorInvalidValue;
    a.nc = p.nc;
    a.segs = p.segs;
    a.ctas = p.ctas;
    AffSegStatus<T> st;
    st.w = (unsigned long long*)((char*)job.temp + kHeaderBytes);  // within aff_status_bytes(MAXSEG)
    profile_before(ctx);
    e = clear_status(job.temp, kHeaderBytes + (size_t)p.ctas * 2 * sizeof(Aff<T>), nullptr, 0, ctx);
    if (e == cudaSuccess) e = launch_pdl(scan_affine_seg_kernel<T, G>, p.ctas, G::NT, 0, ctx.stream, a, st);
    profile_after(ctx);
    return e;
  }
  using G = AffTileCfg<T>;
  const long long tiles = (job.R + G::TILE - 1) / G::TILE;
  if (tiles > 0x7fffffffll) return cudaErrorInvalidValue;
  a.nc = tiles;
  a.segs = 0;
  a.ctas = (unsigned)tiles;
  const AffStatus<T> st = aff_status<T>(job.temp, (size_t)tiles);
  profile_before(ctx);
  e = clear_status(job.temp, kHeaderBytes + (size_t)tiles * 4, nullptr, 0, ctx);
  if (e == cudaSuccess)
    e = launch_pdl(scan_affine_tile_kernel<T, G>, (unsigned)tiles, G::NT, 0, ctx.stream, a, st);
  profile_after(ctx);
  return e;
}

}  // namespace gbs
