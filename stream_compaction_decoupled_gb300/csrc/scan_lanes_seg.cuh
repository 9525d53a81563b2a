// scan_lanes_seg.cuh -- lane-vector scans of one long chain of small elements (C = 4,
// 8 or 16 lanes of a 4-byte type) that fits in L2: the segment scheme of scan_seg.cuh
// (reduce, publish, gather every earlier segment, rescan from L2) with warp scans
// that step over whole elements.
//
// A single chain of such elements (a 32-byte struct of 8 fp32 lanes, or the columns
// of an (R, 8) matrix scanned down axis 0) is thousands of tiles long, and the lane
// kernel's per-lane look-back walks it tile by tile.  Here every segment (CTA) gets
// the combination of all earlier segments in one gather, as the 1-D segment kernel
// does.  A segment publishes each lane's aggregate in a word of its own that carries
// its flag, right after phase 1, and the gather is spread over all but one warp of
// the CTA, so that every earlier word is requested at once and the base is known
// one memory round trip after the last of them is visible.
//
// An element is V = C / 4 vectors of 16 bytes.  A warp reads a chunk as ROUNDS
// coalesced rounds of 32 vectors (512 bytes, E = 32 / V whole elements); lane l
// always holds vector slot s = l mod V of an element (its lanes 4s .. 4s+3), and the
// lanes with the same slot, V apart, hold consecutive elements.  A round is scanned
// with one warp scan in steps of V lanes (every slot at once), seeded with the carry
// of the rounds before it.  (A layout in which each lane owned consecutive elements
// needed fewer shuffles, but each of its accesses touched 16 lines instead of 4 and
// ran slower.)
#pragma once

#include "scan_seg.cuh"

namespace gbs {

template <class T, int V_> struct LanesSegCfg {
  static constexpr int V = V_, C = 4 * V_, E = 32 / V_;
  static constexpr int NT = 768, NW = NT / 32, MINB = 1;
  static constexpr int ROUNDS = 4;         // coalesced rounds of 32 vectors per chunk
  static constexpr int CHE = ROUNDS * E;   // elements per chunk
  static constexpr int CH = CHE * V;       // 16-byte vectors per chunk (128: 2 KB)
  static constexpr int MAXSEG = 512, M = MAXSEG / 32;
  static_assert(sizeof(T) == 4, "4-byte lanes");
};

template <class T, int C> struct LanesSegArgs : SegArgsBase {  // n: elements (positions)
  const T* in;
  T* out;
  T init[C];      // exclusive scans: the initial value of every lane
  int inclusive;
};

// Status of a segment: C words, one per lane, each (flag << 32 | the lane
// aggregate's bits).  A lane's value and its flag travel in one 64-bit store, so a
// reader that sees the flag has the value, with no fence between them.
template <class T, int C> struct LanesSegStatus {
  unsigned long long* w;  // [segment][lane]
};

// A lane's 4 values: one 16-byte vector, the lanes 4s .. 4s+3 of one element.
template <class T> struct Quad {
  T v[4];
};
template <class T, int OP> __device__ __forceinline__ void quad_then(Quad<T>& a, const Quad<T>& b) {
#pragma unroll
  for (int k = 0; k < 4; ++k) a.v[k] = Op<T, OP>::f(a.v[k], b.v[k]);
}
template <class T> __device__ __forceinline__ Quad<T> quad_shfl_up(const Quad<T>& q, int d) {
  Quad<T> r;
#pragma unroll
  for (int k = 0; k < 4; ++k) r.v[k] = __shfl_up_sync(0xffffffffu, q.v[k], d);
  return r;
}
template <class T> __device__ __forceinline__ Quad<T> quad_shfl_xor(const Quad<T>& q, int d) {
  Quad<T> r;
#pragma unroll
  for (int k = 0; k < 4; ++k) r.v[k] = __shfl_xor_sync(0xffffffffu, q.v[k], d);
  return r;
}
template <class T> __device__ __forceinline__ Quad<T> quad_shfl(const Quad<T>& q, int src) {
  Quad<T> r;
#pragma unroll
  for (int k = 0; k < 4; ++k) r.v[k] = __shfl_sync(0xffffffffu, q.v[k], src);
  return r;
}
template <class T> __device__ __forceinline__ Quad<T> quad_load(const uint4* p, unsigned long long pol) {
  const uint4 u = ld_hint(p, pol);
  Quad<T> q;
  memcpy(q.v, &u, 16);
  return q;
}
template <class T> __device__ __forceinline__ void quad_store(uint4* p, const Quad<T>& q, unsigned long long pol) {
  uint4 u;
  memcpy(&u, q.v, 16);
  st_hint(p, u, pol);
}

// Phase 1 of a warp: every lane combines the vectors v = first + lane + 32 k of its
// chunks (always slot lane mod V); then the members of each slot group combine
// theirs (the order is free: the operators of this kernel commute).  Lanes that got
// no vector take no part (`has`).  Returns the warp's total of the lane's slot.
template <class T, int OP, class G>
__device__ __forceinline__ Quad<T> lanes_seg_reduce(const uint4* p, long long v0, long long v1, int lane,
                                                    bool& has) {
  constexpr int U = 8, V = G::V;
  const unsigned long long keep = l2_policy_evict_last();
  Quad<T> acc{};
  has = false;
  long long v = v0 + lane;
  for (; v + 32 * (U - 1) < v1; v += 32 * U) {  // U loads in flight
    Quad<T> q[U];
#pragma unroll
    for (int k = 0; k < U; ++k) q[k] = quad_load<T>(p + v + 32 * k, keep);
#pragma unroll
    for (int k = 0; k < U; ++k) {
      if (has) quad_then<T, OP>(acc, q[k]);
      else acc = q[k];
      has = true;
    }
  }
  for (; v < v1; v += 32) {
    const Quad<T> q = quad_load<T>(p + v, keep);
    if (has) quad_then<T, OP>(acc, q);
    else acc = q;
    has = true;
  }
#pragma unroll
  for (int d = V; d < 32; d *= 2) {  // across the members of the slot group
    const Quad<T> o = quad_shfl_xor(acc, d);
    const bool oh = __shfl_xor_sync(0xffffffffu, (int)has, d) != 0;
    if (oh) {
      if (has) {  // a fixed order (the lower lane on the left): reproducible float sums
        Quad<T> lo = (lane & d) ? o : acc;
        quad_then<T, OP>(lo, (lane & d) ? acc : o);
        acc = lo;
      } else {
        acc = o;
      }
      has = true;
    }
  }
  return acc;
}

template <class T, int OP, class G>
__global__ void __launch_bounds__(G::NT, G::MINB)
    scan_lanes_seg_kernel(LanesSegArgs<T, G::C> a, LanesSegStatus<T, G::C> st) {
  pdl_entry();
  constexpr int NW = G::NW, V = G::V, C = G::C, ROUNDS = G::ROUNDS, CH = G::CH;
  __shared__ unsigned s_seg;
  __shared__ T s_w[NW][C];  // warp totals, then their inclusive scan over the warps
  __shared__ T s_base[C];
  __shared__ T s_init[C];
  __shared__ int s_hbase;
  constexpr int GG = (NW - 1) * 32 / C;  // phase 2's gathering blocks (warps 1..)
  __shared__ T s_part[GG][C];            // their folds
  __shared__ int s_phas[GG];
  __shared__ int s_tmo;                  // a gatherer's wait ran out
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int slot = lane % V;
  if (tid == 0) {
    s_seg = atomicAdd(a.counter, 1u);
    s_tmo = 0;
#pragma unroll
    for (int c = 0; c < C; ++c) s_init[c] = a.init[c];  // constant indices: no local copy of the parameter
  }
  __syncthreads();
  const unsigned seg = s_seg;
  long long c0, c1;
  const int nact = seg_chunks(a, seg, warp, NW, c0, c1);
  const uint4* vin = reinterpret_cast<const uint4*>(a.in);
  uint4* vout = reinterpret_cast<uint4*>(a.out);
  const long long nv = a.n * V;  // vectors in the row

  // Phase 1: the warp's total of every lane (warps without chunks come last; their
  // totals are never read).  Float products combine in order, round by round, so
  // that only adjacent ranges are ever multiplied: a product of factors that are
  // not adjacent can overflow where every prefix stays in range.  The other
  // operators fold each lane's vectors in any order first.
  if constexpr (OP == OP_MUL && std::is_floating_point<T>::value) {
    const unsigned long long keep = l2_policy_evict_last();
    Quad<T> w{};
    bool hw = false;
    for (long long c = c0; c < c1; ++c) {
      Quad<T> q[ROUNDS];
#pragma unroll
      for (int j = 0; j < ROUNDS; ++j) {
        const long long v = c * CH + j * 32 + lane;
        q[j] = v < nv ? quad_load<T>(vin + v, keep) : Quad<T>{};
      }
#pragma unroll
      for (int j = 0; j < ROUNDS; ++j) {
        const long long vlast = c * CH + j * 32;   // the round's first vector
        if (vlast >= nv) break;                    // warp-uniform
        Quad<T> t = q[j];
#pragma unroll
        for (int d = V; d < 32; d *= 2) {
          Quad<T> o = quad_shfl_up(t, d);
          if (lane >= d) {
            quad_then<T, OP>(o, t);
            t = o;
          }
        }
        // The round's product per slot: the last lane of the slot group still inside n.
        const long long nin = nv - vlast < 32 ? nv - vlast : 32;
        const Quad<T> r = quad_shfl(t, (int)(nin - V) + slot);
        if (hw) quad_then<T, OP>(w, r);
        else w = r;
        hw = true;
      }
    }
    if (lane < V && c0 < c1) {
#pragma unroll
      for (int k = 0; k < 4; ++k) s_w[warp][4 * slot + k] = w.v[k];
    }
  } else {
    bool has;
    const long long v0 = c0 * CH, v1 = c1 * CH < nv ? c1 * CH : nv;
    const Quad<T> t = lanes_seg_reduce<T, OP, G>(vin, v0, v1, lane, has);
    if (lane < V && c0 < c1) {
#pragma unroll
      for (int k = 0; k < 4; ++k) s_w[warp][4 * slot + k] = t.v[k];
    }
  }
  __syncthreads();

  // Phase 2.  Warp 0 combines the warp totals into the segment's C aggregates and
  // publishes them at once, then scans the warp totals per lane for phase 3.
  // Meanwhile the other warps wait for the earlier segments' words and fold them:
  // thread t of warps 1.. takes lane value t mod C of the consecutive block of
  // segments (t / C) q .. (t / C) q + q - 1, q = ceil(seg / GG), all its words
  // requested at once and only the missing ones polled again.  Then warp 0 joins the
  // blocks, lower ones on the left.  Every combination joins adjacent ranges in order
  // (a product of ranges that are not adjacent can overflow where every prefix
  // stays in range).
  constexpr int K = 32 / C;                        // lanes of warp 0 per lane value
  constexpr int QMAX = (G::MAXSEG + GG - 1) / GG;  // segments a block takes at most
  static_assert(QMAX <= 32, "pending bits of one word");
  if (warp == 0) {
    const int c = lane % C, k = lane / C;
    T acc{};
    bool h = false;
    for (int w = k * nact / K; w < (k + 1) * nact / K; ++w) {
      const T x = s_w[w][c];
      acc = h ? Op<T, OP>::f(acc, x) : x;
      h = true;
    }
#pragma unroll
    for (int d = C; d < 32; d *= 2) {  // across k, the lower warps on the left
      const T o = __shfl_xor_sync(0xffffffffu, acc, d);
      const bool oh = __shfl_xor_sync(0xffffffffu, (int)h, d) != 0;
      if (oh) acc = h ? ((lane & d) ? Op<T, OP>::f(o, acc) : Op<T, OP>::f(acc, o)) : o;
      h = h || oh;
    }
    if (k == 0 && (long long)seg != a.stalled)
      st_relaxed_u64(st.w + (size_t)seg * C + c, ((unsigned long long)FLAG_A << 32) | to_u32(acc));
    __syncwarp();  // every lane's reads of s_w before the scan rewrites it
    if (lane < C) {
      T run = s_w[0][lane];
      for (int w = 1; w < nact; ++w) {
        run = Op<T, OP>::f(run, s_w[w][lane]);
        s_w[w][lane] = run;
      }
    }
  } else {
    const int t = tid - 32, c = t % C, g = t / C;
    const unsigned q = (seg + GG - 1) / GG, s0 = (unsigned)g * q, s1 = s0 + q < seg ? s0 + q : seg;
    if (s0 < s1) {
      unsigned long long wv[QMAX];
      unsigned pending = 0;
#pragma unroll
      for (int j = 0; j < QMAX; ++j)
        if (s0 + j < s1) pending |= 1u << j;
      unsigned long long t0 = 0;
      for (int spins = 0;; ++spins) {
#pragma unroll
        for (int j = 0; j < QMAX; ++j)
          if (pending & (1u << j)) {
            wv[j] = ld_relaxed_u64(st.w + (size_t)(s0 + j) * C + c);
            if ((unsigned)(wv[j] >> 32) != FLAG_X) pending &= ~(1u << j);
          }
        if (pending == 0) break;
        const unsigned long long now = globaltimer();
        if (spins == 0) t0 = now;
        else if (now - t0 > a.wait_ns) {  // the words still missing are left out
          s_tmo = 1;
          break;
        }
        backoff(spins);
      }
      T acc{};
      bool h = false;
#pragma unroll
      for (int j = 0; j < QMAX; ++j)
        if (s0 + j < s1 && !(pending & (1u << j))) {
          const T x = from_u32<T>((unsigned)wv[j]);
          acc = h ? Op<T, OP>::f(acc, x) : x;
          h = true;
        }
      s_part[g][c] = acc;
      if (c == 0) s_phas[g] = h;
    } else if (c == 0) {
      s_phas[g] = 0;
    }
  }
  __syncthreads();
  if (warp == 0) {
    const int c = lane % C, k = lane / C;
    T acc{};
    bool have = false;
    for (int g = k * GG / K; g < (k + 1) * GG / K; ++g)
      if (s_phas[g]) {
        const T x = s_part[g][c];
        acc = have ? Op<T, OP>::f(acc, x) : x;
        have = true;
      }
#pragma unroll
    for (int d = C; d < 32; d *= 2) {  // across the blocks of k, the lower ones on the left
      const T o = __shfl_xor_sync(0xffffffffu, acc, d);
      const bool oh = __shfl_xor_sync(0xffffffffu, (int)have, d) != 0;
      if (oh) acc = have ? ((lane & d) ? Op<T, OP>::f(o, acc) : Op<T, OP>::f(acc, o)) : o;
      have = have || oh;
    }
    if (lane < C) s_base[lane] = acc;
    if (lane == 0) {
      if (s_tmo) raise_err(a.err, ERRBIT_TIMEOUT);
      s_hbase = have;
    }
  }
  __syncthreads();

  // Phase 3: the carry into the warp's part (init, the earlier segments, the earlier
  // warps of this one), then chunk by chunk from L2.
  Quad<T> carry;
  bool hc = s_hbase != 0;
#pragma unroll
  for (int k = 0; k < 4; ++k) carry.v[k] = s_base[4 * slot + k];
  if (warp > 0) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const T w = s_w[warp - 1][4 * slot + k];
      carry.v[k] = hc ? Op<T, OP>::f(carry.v[k], w) : w;
    }
    hc = true;
  }
  if (!a.inclusive) {
#pragma unroll
    for (int k = 0; k < 4; ++k) carry.v[k] = hc ? Op<T, OP>::f(s_init[4 * slot + k], carry.v[k]) : s_init[4 * slot + k];
    hc = true;
  }
  const unsigned long long drop = l2_policy_evict_first();
  auto load_chunk = [&](Quad<T> (&x)[ROUNDS], long long c) {
#pragma unroll
    for (int j = 0; j < ROUNDS; ++j) {
      const long long v = c * CH + j * 32 + lane;
      x[j] = v < nv ? quad_load<T>(vin + v, drop) : Quad<T>{};  // past n: never stored
    }
  };
  Quad<T> x[ROUNDS];
  if (c0 < c1) load_chunk(x, c0);
  for (long long c = c0; c < c1; ++c) {
    Quad<T> nxt[ROUNDS];  // the next chunk, requested before this one is scanned
    if (c + 1 < c1) load_chunk(nxt, c + 1);
#pragma unroll
    for (int j = 0; j < ROUNDS; ++j) {
      // Round j holds the E whole elements c*CHE + j*E .. + E - 1, element (j*32 +
      // lane) / V in lane `lane`: an inclusive scan over the slot group (steps of V).
      Quad<T> t = x[j];
#pragma unroll
      for (int d = V; d < 32; d *= 2) {
        Quad<T> o = quad_shfl_up(t, d);
        if (lane >= d) {
          quad_then<T, OP>(o, t);
          t = o;
        }
      }
      const Quad<T> round_total = quad_shfl(t, 32 - V + slot);
      Quad<T> y;
      if (a.inclusive) {
        y = t;
        if (hc) {
          y = carry;
          quad_then<T, OP>(y, t);
        }
      } else {  // exclusive: hc always holds (the initial value at least)
        const Quad<T> e = quad_shfl_up(t, V);
        y = carry;
        if (lane >= V) quad_then<T, OP>(y, e);
      }
      const long long v = c * CH + j * 32 + lane;
      if (v < nv) quad_store<T>(vout + v, y, drop);
      if (hc) quad_then<T, OP>(carry, round_total);
      else carry = round_total;
      hc = true;
    }
#pragma unroll
    for (int j = 0; j < ROUNDS; ++j) x[j] = nxt[j];
  }
}

template <class T, int V> size_t lanes_seg_status_bytes() {
  using G = LanesSegCfg<T, V>;
  return round_up((size_t)G::MAXSEG * G::C * 8, 256);
}
// Scratch for any lane count this kernel serves (the largest, 16 lanes).
template <class T> size_t lanes_seg_temp_bytes() { return kHeaderBytes + lanes_seg_status_bytes<T, 4>(); }

// One aligned chain (B = 1) of C = 4, 8 or 16 four-byte lanes that fits in L2.
template <class T> bool lanes_seg_applies(const ScanJob& job) {
  if (sizeof(T) != 4 || job.B != 1 || !(job.C == 4 || job.C == 8 || job.C == 16)) return false;
  if ((uintptr_t)job.in % 16 != 0 || (uintptr_t)job.out % 16 != 0) return false;
  return job.R * job.C * (long long)sizeof(T) <= kSegMaxBytes;
}

template <class T, int OP, int V> cudaError_t launch_lanes_seg_v(const ScanJob& job, const LaunchCtx& ctx) {
  using G = LanesSegCfg<T, V>;
  const long long nvec = job.R * V;
  const SegPlan p = seg_plan<G>(1, nvec, ctx.num_sms);  // plans in vectors (G::CH per chunk)
  if (p.ctas == 0) return cudaErrorInvalidValue;
  LanesSegArgs<T, G::C> a;
  a.n = job.R;
  a.nc = p.nc;
  a.segs = p.segs;
  a.ctas = p.ctas;
  a.counter = (unsigned*)job.temp;
  a.err = ctx.err;
  a.wait_ns = ctx.wait_ns;
  a.stalled = ctx.stalled_tile;
  a.in = (const T*)job.in;
  a.out = (T*)job.out;
  for (int c = 0; c < G::C; ++c) {
    a.init[c] = T{};
    if (!job.inclusive && job.init_host)
      memcpy(&a.init[c], (const char*)job.init_host + (size_t)(c % job.init_lanes) * sizeof(T), sizeof(T));
  }
  a.inclusive = job.inclusive;
  LanesSegStatus<T, G::C> st;
  st.w = (unsigned long long*)((char*)job.temp + kHeaderBytes);
  profile_before(ctx);
  cudaError_t e = clear_status(job.temp, kHeaderBytes + (size_t)p.ctas * G::C * 8, nullptr, 0, ctx);
  if (e == cudaSuccess) e = launch_pdl(scan_lanes_seg_kernel<T, OP, G>, p.ctas, G::NT, 0, ctx.stream, a, st);
  profile_after(ctx);
  return e;
}

template <class T, int OP> cudaError_t launch_lanes_seg_op(const ScanJob& job, const LaunchCtx& ctx) {
  if constexpr (sizeof(T) == 4) {
    switch (job.C) {
      case 4: return launch_lanes_seg_v<T, OP, 1>(job, ctx);
      case 8: return launch_lanes_seg_v<T, OP, 2>(job, ctx);
      default: return launch_lanes_seg_v<T, OP, 4>(job, ctx);
    }
  } else {
    return cudaErrorInvalidValue;
  }
}

}  // namespace gbs
