// scan_strips.cuh -- scans down the columns of a wide row-major (B, R, C) array, one
// strip of columns per CTA at a time, with no status words and no look-back.
//
// The lane kernel (scan_lanes.cuh) cuts every chain of positions into tiles and
// chains the tiles through the decoupled look-back; along a chain of tens of tiles
// that chain of publishes is what bounds it.  When the array has at least as many
// strips of 64 bytes as the GPU has SMs, every CTA can own whole strips instead: it
// walks its strip's rows tile by tile and carries the running prefix of each lane in
// registers, so no CTA ever waits for another (The CUDA Handbook, 13.3: a scan whose
// pieces are independent needs no inter-block communication at all).
//
// A strip is 64 bytes of a row (16 four-byte or 8 eight-byte lanes) = Q = 4 vectors
// of 16 bytes.  Thread t of a CTA takes vector q = t mod Q of the strip and L
// consecutive rows of each tile, starting at row (t / Q) L.  It requests its rows of
// the next P tiles into shared memory with asynchronous 16-byte copies and reads back
// only its own rows, so no barrier guards the buffers; it folds its rows serially,
// the CTA scans the NT / Q row groups of each vector (a shuffle scan over the 8
// groups of a warp, then one warp over the warp totals), and each thread rescans its
// rows seeded with everything before them and stores them.  Rows past R are read as
// zero: they only reach outputs past R, which are not stored (a scan propagates
// forward).  Measured on GB300 (fp32 4096 x 4096 down the columns, 256 strips): 30.1-
// 30.8 us against 40.6 us for the lane kernel; strips of 32 bytes (512 of them, better
// spread over the SMs) took 49.3 us, each row piece then being a lone DRAM sector.
#pragma once

#include "launch.h"
#include "tile.cuh"

namespace gbs {

template <class T> struct StripsCfg {
  static constexpr int NT = 512, NW = NT / 32, MINB = 2;
  static constexpr int VEC = Vec<T>::N;      // lanes of a 16-byte vector
  static constexpr int Q = 4;                // vectors of a strip row (64 bytes)
  static constexpr int W = Q * VEC;          // lanes of a strip
  static constexpr int GW = 32 / Q;          // row groups of a warp
  static constexpr int L = 4;                // rows of a thread per tile
  static constexpr int RT = (NT / Q) * L;    // rows of a tile
  static constexpr int P = 2;                // tiles requested ahead of the one scanned
  static constexpr int NBUF = P + 1;         // tile buffers in shared memory
  static constexpr size_t SMEM = (size_t)NBUF * L * NT * 16;  // 96 KB
};

template <class T> struct StripsArgs {
  const T* in;
  T* out;
  long long B, R, C;      // chains of R positions of C lanes; C * sizeof(T) % 16 == 0
  long long strips;       // ceil(C / W)
  long long tiles;        // ceil(R / RT): tiles of a chain
  const T* init;          // exclusive: device copy of the initial values
  int init_lanes;         // lane c starts from init[c % init_lanes]
  int inclusive;
  unsigned* call_err;     // the call's error word: cleared here (nothing in this kernel waits)
};

template <class T, int OP>
__device__ __forceinline__ Vec<T> vec_then(const Vec<T>& a, const Vec<T>& b) {
  Vec<T> r;
#pragma unroll
  for (int k = 0; k < Vec<T>::N; ++k) r.v[k] = Op<T, OP>::f(a.v[k], b.v[k]);
  return r;
}
template <class T> __device__ __forceinline__ Vec<T> vec_shfl_up(const Vec<T>& a, int d) {
  Vec<T> r;
#pragma unroll
  for (int k = 0; k < Vec<T>::N; ++k) r.v[k] = __shfl_up_sync(0xffffffffu, a.v[k], d);
  return r;
}

// 16-byte asynchronous copies into shared memory (L2 only); src_bytes 0 writes zeros
// and reads nothing.
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem, unsigned src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(smem)), "l"(gmem), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N> __device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

template <class T, int OP, class G>
__global__ void __launch_bounds__(G::NT, G::MINB) scan_strips_kernel(StripsArgs<T> a) {
  pdl_entry();
  constexpr int NT = G::NT, NW = G::NW, VEC = G::VEC, Q = G::Q, W = G::W, GW = G::GW, L = G::L, RT = G::RT;
  constexpr int P = G::P, NBUF = G::NBUF;
  extern __shared__ __align__(16) uint4 strips_smem[];  // [NBUF][L][NT]: each thread's own rows
  __shared__ Vec<T> s_wt[NW][Q];  // warp totals, then the inclusive scan over the warps
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int q = tid % Q, g = tid / Q, gl = lane / Q;  // vector, row group, row group in the warp
  if (blockIdx.x == 0 && tid == 0 && a.call_err) *a.call_err = 0u;
  const long long chains = a.B * a.strips;
  // This CTA's work: chains blockIdx.x, blockIdx.x + gridDim.x, ..., each a.tiles tiles,
  // taken as one sequence of items so that copies run ahead across chain boundaries.
  // Two cursors walk it (requests P items ahead of the scan); divisions happen once a
  // chain, not once a tile.
  const long long my_chains = (chains - blockIdx.x + gridDim.x - 1) / gridDim.x;
  const long long items = my_chains * a.tiles;
  struct Cursor {
    long long ch, tl;  // chain, tile in the chain
    long long c0;      // this thread's first lane
    long long off;     // element offset of the chain's row 0 at lane c0
  };
  auto start_chain = [&](Cursor& k) {
    const long long b = a.strips == 1 ? k.ch : k.ch / a.strips, sp = k.ch - b * a.strips;
    k.c0 = sp * W + (long long)q * VEC;
    k.off = b * a.R * a.C + k.c0;
  };
  auto advance = [&](Cursor& k) {
    if (++k.tl == a.tiles) {
      k.tl = 0;
      k.ch += gridDim.x;
      if (k.ch < chains) start_chain(k);
    }
  };
  Cursor rq{(long long)blockIdx.x, 0, 0, 0}, sc{(long long)blockIdx.x, 0, 0, 0};
  start_chain(rq);
  start_chain(sc);
  int rq_buf = 0, sc_buf = 0;

  // Request the rows of item rq of this thread into buffer rq_buf (zeros past R or C).
  long long requested = 0;
  auto request = [&]() {
    if (requested < items) {
      const long long r = rq.tl * RT + (long long)g * L;
      const T* p = a.in + rq.off + r * a.C;
      uint4* buf = strips_smem + (size_t)rq_buf * L * NT + tid;
      const bool cv = rq.c0 < a.C;
#pragma unroll
      for (int i = 0; i < L; ++i) {
        const bool ok = cv && r + i < a.R;
        cp_async16(buf + i * NT, ok ? (const void*)p : (const void*)a.in, ok ? 16u : 0u);
        p += a.C;
      }
      advance(rq);
      rq_buf = rq_buf + 1 == NBUF ? 0 : rq_buf + 1;
      ++requested;
    }
    cp_async_commit();  // an empty group past the end keeps the group count in step
  };
#pragma unroll
  for (int k = 0; k < P; ++k) request();

  const unsigned long long drop = l2_policy_evict_first();
  Vec<T> carry;  // everything before the current tile in this thread's lanes
  bool hc = false;
  for (long long j = 0; j < items; ++j) {
    request();
    cp_async_wait<P>();  // item j has landed (this thread's own rows only: no barrier)
    const bool qvalid = sc.c0 < a.C;  // C is a multiple of VEC
    const long long r0 = sc.tl * RT;
    if (sc.tl == 0) {  // a new chain
      hc = false;
      if (!a.inclusive) {
#pragma unroll
        for (int e = 0; e < VEC; ++e) carry.v[e] = qvalid ? a.init[(sc.c0 + e) % a.init_lanes] : T{};
        hc = true;
      }
    }
    const uint4* buf = strips_smem + (size_t)sc_buf * L * NT + tid;
    Vec<T> x[L];
#pragma unroll
    for (int i = 0; i < L; ++i) {
      const uint4 u = buf[i * NT];
      memcpy(x[i].v, &u, 16);
    }

    // The thread's rows, then the row groups of the warp (steps of Q lanes).
    Vec<T> t = x[0];
#pragma unroll
    for (int i = 1; i < L; ++i) t = vec_then<T, OP>(t, x[i]);
    Vec<T> inc = t;
#pragma unroll
    for (int d = Q; d < 32; d *= 2) {
      const Vec<T> o = vec_shfl_up(inc, d);
      if (lane >= d) inc = vec_then<T, OP>(o, inc);
    }
    const Vec<T> before_in_warp = vec_shfl_up(inc, Q);  // groups before this one in the warp
    if (gl == GW - 1) s_wt[warp][q] = inc;
    __syncthreads();
    if (warp == 0 && lane < Q) {  // inclusive scan of the warp totals, per vector
      Vec<T> run = s_wt[0][lane];
      for (int w = 1; w < NW; ++w) {
        run = vec_then<T, OP>(run, s_wt[w][lane]);
        s_wt[w][lane] = run;
      }
    }
    __syncthreads();

    // Everything before the thread's first row: the carry, the earlier warps, the
    // earlier groups of the warp.
    Vec<T> base = carry;
    bool hb = hc;
    if (warp > 0) {
      const Vec<T> pw = s_wt[warp - 1][q];
      base = hb ? vec_then<T, OP>(base, pw) : pw;
      hb = true;
    }
    if (gl > 0) {
      base = hb ? vec_then<T, OP>(base, before_in_warp) : before_in_warp;
      hb = true;
    }
    const Vec<T> tile_total = s_wt[NW - 1][q];
    T* dst = a.out + sc.off + (r0 + (long long)g * L) * a.C;
#pragma unroll
    for (int i = 0; i < L; ++i) {
      const long long r = r0 + (long long)g * L + i;
      Vec<T> y;
      if (a.inclusive) {
        y = hb ? vec_then<T, OP>(base, x[i]) : x[i];
        base = y;
        hb = true;
      } else {
        y = base;  // hb holds: the initial values at least
        base = vec_then<T, OP>(base, x[i]);
      }
      if (qvalid && r < a.R) {
        uint4 u;
        memcpy(&u, y.v, 16);
        st_hint(reinterpret_cast<uint4*>(dst), u, drop);
      }
      dst += a.C;
    }
    carry = hc ? vec_then<T, OP>(carry, tile_total) : tile_total;
    hc = true;
    advance(sc);
    sc_buf = sc_buf + 1 == NBUF ? 0 : sc_buf + 1;
    __syncthreads();  // s_wt is rewritten by the next tile
  }
  cp_async_wait<0>();
}

// Strips need 16-byte vectors in every row and enough of them to give every SM one.
// Not for fp64: a strip costs about 3 adds per element against the lane kernel's 2,
// and fp64 adds bound those scans on this GPU (1000 x 1e4 down the columns: 91.5 us
// here against 67.9 us).
template <class T> bool strips_applies(const ScanJob& job, int num_sms) {
  using G = StripsCfg<T>;
  if (std::is_same<T, double>::value) return false;
  if (job.C < 2 || (job.C * (long long)sizeof(T)) % 16 != 0) return false;
  if ((uintptr_t)job.in % 16 != 0 || (uintptr_t)job.out % 16 != 0) return false;
  const long long strips = (job.C + G::W - 1) / G::W;
  return job.B * strips >= num_sms;
}

template <class T> size_t strips_temp_bytes(long long C) {
  const long long n = C < 4096 ? C : 4096;
  return kHeaderBytes + round_up((size_t)n * sizeof(T), 256);
}

template <class T, int OP> cudaError_t launch_strips_op(const ScanJob& job, const LaunchCtx& ctx) {
  using G = StripsCfg<T>;
  StripsArgs<T> a;
  a.in = (const T*)job.in;
  a.out = (T*)job.out;
  a.B = job.B;
  a.R = job.R;
  a.C = job.C;
  a.strips = (job.C + G::W - 1) / G::W;
  a.tiles = (job.R + G::RT - 1) / G::RT;
  T* init_area = (T*)((char*)job.temp + kHeaderBytes);
  a.init = init_area;
  a.init_lanes = job.init_lanes;
  a.inclusive = job.inclusive;
  a.call_err = ctx.err.call;
  const long long chains = job.B * a.strips;
  const long long slots = (long long)ctx.num_sms * G::MINB;
  const unsigned grid = (unsigned)(chains < slots ? chains : slots);
  auto kern = scan_strips_kernel<T, OP, G>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)G::SMEM);
  if (e != cudaSuccess) return e;
  profile_before(ctx);
  if (!job.inclusive)
    e = cudaMemcpyAsync(init_area, job.init_host, (size_t)job.init_lanes * sizeof(T), cudaMemcpyHostToDevice,
                        ctx.stream);
  if (e == cudaSuccess) e = launch_pdl(kern, grid, G::NT, G::SMEM, ctx.stream, a);
  profile_after(ctx);
  return e;
}

}  // namespace gbs
