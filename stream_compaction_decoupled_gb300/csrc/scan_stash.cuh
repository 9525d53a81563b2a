// scan_stash.cuh -- single-pass decoupled look-back scan of one long contiguous row
// that keeps the tiles waiting for their prefix in L2 instead of shared memory.
//
// In a one-CTA-per-tile scan each CTA holds its tile in shared memory until its
// prefix is known, and the prefix of tile t cannot be known before the slowest load
// of any earlier tile has landed.  On a GB300 the load latency under full bandwidth
// has a tail several times its median, so every tile waits for that tail, and the
// ~200 KB of shared memory per SM cannot hold bandwidth x (latency + tail) of data:
// the scan then runs well below the copy bandwidth even though, without the wait,
// the same tiles move at copy speed.  The 129 MB L2 can hold that much.
//
// So each persistent CTA (one per SM) runs four decoupled roles over "runs" of
// RUN consecutive tiles, claimed in order from an atomic counter (The CUDA
// Handbook, 13.3.4: claimed order gives forward progress):
//   I  (one lane of warp 0)  claims runs (one claim ahead, while the CTA's queue of
//                 QD runs has room) and streams their tiles from HBM into NL
//                 shared-memory buffers by bulk copies (L2 evict-last hint);
//   R  (NR warps) reduce each tile as it lands and free its buffer at once; the
//                 reducer of a run's last tile publishes the run's aggregate (A, or
//                 P for run 0);
//   B  (one warp) takes the CTA's runs in order and computes each run's exclusive
//                 prefix with the warp-cooperative decoupled look-back over run
//                 status words (a window of 32 x K runs per round trip), then
//                 publishes P;
//   S  (NG groups of NSW warps) each own whole runs of the queue: a group re-loads a
//                 run's tiles from L2 (bulk copies, evict-first, a ring of NS
//                 buffers) as soon as its aggregate is out, so the copies overlap
//                 the look-back, then scans them in registers from the run's prefix
//                 (the row kernel's two passes) and stores them as 16-byte vectors
//                 (evict-first).
// HBM traffic stays one read and one write per element; the second read is served
// by L2.  I and R never wait on other CTAs, so every claimed run publishes its
// aggregate within one load latency, and B's look-backs always end.  I claims a
// run only when its queue has room, so the data resident in L2 is bounded by
// (CTAs x QD x RUN x tile) bytes.
#pragma once

#include "launch.h"
#include "scan_rows.cuh"
#include "tile.cuh"

namespace gbs {

// Defaults from sweeps on the fp32 1e8 and 2e8 inclusive scans (per-step time of 20
// chained calls, best of 5; the same box for every line):
//   4 load buffers, window 64 runs, runs of 4, 8 queued      140.3 us   265.5 us
//   5 load buffers, the rest as above                         140.5 us   267.2 us
//   window of 32 runs, the rest as above                      140.4 us   265.9 us
//   5 load buffers, window 32, runs of 4, 8 queued            137.0 us   261.5 us
//   5 load buffers, window 32, runs of 3, 10 queued           134.7 us   255.9 us
//   ... runs of 3, 9 queued (three repeats, interleaved)      132.6-133.0  252.0-252.3  <- defaults
//   ... runs of 3, 8 / 10 / 12 queued                         133.9 / 134.1 / 137.8   255.0 / 255.4 / 266.6
//   ... runs of 2, 14 / 16 queued                             147.1 / 151.6
//   3 / 4 load buffers (runs of 4 / 3)                       155.3 / 136.9 us
//   7 or 8 load buffers with 2 per group; 2 groups of 4       151.3 / 153.8; 143.7 us
//   1 or 3 reducers; two look-back warps on alternate runs    166.2 / 178.4; 179.7 us
//   12 KB or 8 KB tiles with more buffers (another box: 16 KB 136.9 us there)
//                                                             137.5-141.9; 165.1 us
// More loads in flight from HBM pay as long as each scanning group keeps 3 re-load
// buffers; shorter runs halve the wait for a run's prefix but need more runs queued,
// which presses L2 beyond about 30 queued tiles per SM.  More warps cost registers
// (all roles share one register budget, and the scanning warps then spill).
template <class T, int NR_ = 2, int NG_ = 3, int NL_ = 5, int NS_ = 3, int K_ = 1, int RUN_ = 3, int QD_ = 9,
          int NB_ = 1, int ROUNDS_ = 8>
struct StashCfgT {
  static constexpr int VEC = 16 / (int)sizeof(T);
  static constexpr int NR = NR_;                      // reducer warps
  static constexpr int NB = NB_;                      // look-back warps (alternate runs)
  static constexpr int NSW = 4;                       // warps per scanning group
  static constexpr int NG = NG_;                      // scanning groups (each owns whole runs)
  static constexpr int WB = 1 + NR;                   // first look-back warp
  static constexpr int WS = WB + NB;                  // first scanning warp
  static constexpr int NT = 32 * (WS + NG * NSW);
  static constexpr int ROUNDS = ROUNDS_;              // S: 16-byte vectors per thread per tile
  static constexpr int TILE = NSW * ROUNDS * 32 * VEC;  // 16 KB at 8 rounds
  static constexpr int RUN = RUN_;                    // tiles per run (one look-back per run)
  static constexpr int NL = NL_;                      // I/R buffers: bulk loads from HBM in flight
  static constexpr int NS = NS_;                      // buffers per scanning group (re-loads from L2)
  static constexpr int QD = QD_;                      // runs per CTA between I and S
  static constexpr int K = K_;                        // look-back window: 32 x K runs
  static constexpr size_t SMEM = (size_t)(NL + NG * NS) * TILE * sizeof(T);
};
template <class T> using StashCfg = StashCfgT<T>;

template <class T> struct StashArgs {
  const T* in;
  T* out;
  long long n;
  unsigned num_tiles;  // ceil(n / TILE)
  unsigned num_runs;   // ceil(num_tiles / RUN)
  unsigned* counter;   // run-claim counter, 0 on entry
  ErrSink err;
  T init;
  int inclusive;
  unsigned long long wait_ns;
  long long stalled_run;
};

// Barrier among the warps of one scanning group (named barrier 1 + group).
template <int N> __device__ __forceinline__ void s_group_sync(int g) {
  asm volatile("bar.sync %0, %1;" ::"r"(1 + g), "n"(N) : "memory");
}

// Barrier among the warps of one scanning group returning the AND of a predicate.
template <int N> __device__ __forceinline__ bool s_group_and(int g, bool v) {
  unsigned r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((unsigned)v), "r"(1 + g), "n"(N)
      : "memory");
  return r != 0;
}

// What a scanning group does next, decided by its first thread.
enum : int { S_SCAN = 0, S_EXIT = 1, S_EXIT_ERR = 2 };

// Shared state of one CTA.
template <class T, class C> struct StashShared {
  unsigned long long bar[C::NL];
  unsigned long long bar_s[C::NG][C::NS];
  // The tile stream: what buffer k % NL holds (written by I before it bumps `issued`).
  unsigned b_tile[C::NL];
  int b_entry[C::NL], b_pos[C::NL];
  volatile unsigned b_reduced[C::NL];  // stream index + 1 of the last tile reduced from the buffer
  // Run queue (entries reused in claim order).
  unsigned q_run[C::QD];
  int q_ntiles[C::QD];
  T q_tagg[C::QD][C::RUN];   // tile aggregates (R)
  int q_count[C::QD];        // tiles reduced so far (R, atomically)
  T q_agg[C::QD];            // run aggregate (R)
  volatile int q_aready[C::QD];  // run aggregate published (R); cleared by I on reuse
  T q_pfx[C::QD];            // exclusive prefix (B), valid when q_has[] != 0
  int q_has[C::QD];
  volatile int q_pready[C::QD];  // prefix known (B); cleared by I on reuse
  volatile int q_fin[C::QD]; // run written by S; cleared by I on reuse
  T s_warp[C::NG][C::NSW];
  // Control block of each scanning group, written by its first thread before each tile.
  int c_cmd[C::NG], c_has[C::NG], c_len[C::NG], c_slot[C::NG], c_parity[C::NG], c_run_start[C::NG],
      c_run_end[C::NG];
  unsigned c_tile[C::NG], c_entry[C::NG];
  T c_carry[C::NG];
  volatile unsigned issued;   // tiles issued by I
  volatile unsigned claimed;  // runs claimed by I (final once i_finished)
  volatile int i_finished;
  volatile int abort;
};

// Bounded wait (one thread) on a condition over shared state.  False on time-out.
template <class F> __device__ __forceinline__ bool stash_wait(F ready, unsigned long long limit, volatile int* abort) {
  if (ready()) return true;
  const unsigned long long t0 = globaltimer();
  for (int spins = 0;; ++spins) {
    __nanosleep(spins < 4 ? 32 : 128);
    if (ready()) return true;
    if (*abort || globaltimer() - t0 > limit) return false;
  }
}

template <class T, int OP, class S, class C>
__global__ void __launch_bounds__(C::NT, 1) scan_stash_kernel(StashArgs<T> a, S st) {
  pdl_entry();
  constexpr int VEC = C::VEC, TILE = C::TILE, RUN = C::RUN, NL = C::NL, QD = C::QD, NR = C::NR;
  constexpr int NSW = C::NSW, NG = C::NG, ROUNDS = C::ROUNDS, NST = 32 * NSW;
  constexpr unsigned FULL = 0xffffffffu;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  T* buf = reinterpret_cast<T*>(smem_raw);
  __shared__ StashShared<T, C> sh;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    for (int i = 0; i < NL; ++i) {
      mbar_init(&sh.bar[i], 1);
      sh.b_reduced[i] = 0;
    }
    for (int g = 0; g < NG; ++g)
      for (int i = 0; i < C::NS; ++i) mbar_init(&sh.bar_s[g][i], 1);
    fence_mbar_init();
    for (int i = 0; i < QD; ++i) {
      sh.q_fin[i] = 0;
      sh.q_aready[i] = 0;
      sh.q_pready[i] = 0;
      sh.q_count[i] = 0;
    }
    sh.issued = 0;
    sh.claimed = 0;
    sh.i_finished = 0;
    sh.abort = 0;
  }
  __syncthreads();

  auto tiles_in_run = [&](unsigned r) -> int {
    const unsigned t0 = r * RUN;
    return (int)(a.num_tiles - t0 < (unsigned)RUN ? a.num_tiles - t0 : (unsigned)RUN);
  };
  auto tile_len = [&](unsigned t) -> int {
    const long long off = (long long)t * TILE;
    return a.n - off >= TILE ? TILE : (int)(a.n - off);
  };
  auto fail = [&]() {
    raise_err(a.err, ERRBIT_TIMEOUT);
    sh.abort = 1;
  };

  if (warp == 0) {
    // ------------------------------------------------------ I: one lane --------
    if (lane == 0) {
      const unsigned long long pol = l2_policy_evict_last();
      unsigned claimed = 0, released = 0, issued = 0;
      unsigned next_run = atomicAdd(a.counter, 1u);  // claimed one run ahead
      bool exhausted = false;
      while (!exhausted) {
        // Release queue entries that S has written, in claim order.
        while (released < claimed && sh.q_fin[released % QD]) {
          const unsigned e = released % QD;
          sh.q_fin[e] = 0;
          sh.q_aready[e] = 0;
          sh.q_pready[e] = 0;
          sh.q_count[e] = 0;
          ++released;
        }
        if (claimed - released >= (unsigned)QD) {  // queue full: wait for S
          if (!stash_wait([&] { return sh.q_fin[released % QD] != 0; }, a.wait_ns, &sh.abort)) {
            fail();
            break;
          }
          continue;
        }
        const unsigned r = next_run;
        if (r >= a.num_runs) {
          exhausted = true;
          break;
        }
        const unsigned e = claimed % QD;
        const int nt = tiles_in_run(r);
        sh.q_run[e] = r;
        sh.q_ntiles[e] = nt;
        ++claimed;
        next_run = atomicAdd(a.counter, 1u);  // its result is needed only at the next claim
        for (int k = 0; k < nt; ++k) {
          const int slot = issued % NL;
          // The buffer's previous tile (stream index issued - NL) must be reduced.
          if (issued >= (unsigned)NL &&
              !stash_wait([&] { return sh.b_reduced[slot] >= issued - NL + 1; }, a.wait_ns, &sh.abort)) {
            fail();
            exhausted = true;
            break;
          }
          const unsigned t = r * RUN + k;
          sh.b_tile[slot] = t;
          sh.b_entry[slot] = e;
          sh.b_pos[slot] = k;
          if (tile_len(t) == TILE) {
            mbar_arrive_expect_tx(&sh.bar[slot], TILE * sizeof(T));
            bulk_g2s_hint(buf + (size_t)slot * TILE, a.in + (long long)t * TILE, TILE * sizeof(T), &sh.bar[slot], pol);
          }
          ++issued;
          __threadfence_block();
          sh.issued = issued;
        }
        __threadfence_block();
        sh.claimed = claimed;
      }
      // Runs may still be in flight: they are finished by R, B and S.
      __threadfence_block();
      sh.i_finished = 1;
    }
  } else if (warp <= NR) {
    // ------------------------------------------------------ R: reducers --------
    const int w = warp - 1;
    for (unsigned k = w;; k += NR) {  // stream indices of this reducer
      int go = 0;
      if (lane == 0) {
        const bool got = stash_wait([&] { return sh.issued > k || sh.i_finished; }, a.wait_ns, &sh.abort);
        __threadfence_block();
        go = !got ? 2 : (sh.issued > k ? 1 : 0);
        if (go == 2) fail();
      }
      go = __shfl_sync(FULL, go, 0);
      __syncwarp();
      if (go != 1) break;
      const int slot = k % NL;
      const unsigned t = sh.b_tile[slot];
      const int e = sh.b_entry[slot], pos = sh.b_pos[slot];
      const int len = tile_len(t);
      T acc{};
      if (len == TILE) {
        const bool landed = __all_sync(FULL, mbar_wait(&sh.bar[slot], (k / NL) & 1u, a.wait_ns));
        if (!landed) {
          if (lane == 0) fail();
          break;
        }
        // 2*VEC independent accumulators per lane: no long dependent chain.
        const uint4* v = reinterpret_cast<const uint4*>(buf + (size_t)slot * TILE);
        constexpr int J = TILE / VEC / 32;
        Vec<T> a0 = ld_vec<T>(v + lane), a1 = ld_vec<T>(v + 32 + lane);
#pragma unroll 4
        for (int j = 2; j < J; j += 2) {
          const Vec<T> x0 = ld_vec<T>(v + j * 32 + lane), x1 = ld_vec<T>(v + (j + 1) * 32 + lane);
#pragma unroll
          for (int e2 = 0; e2 < VEC; ++e2) {
            a0.v[e2] = Op<T, OP>::f(a0.v[e2], x0.v[e2]);
            a1.v[e2] = Op<T, OP>::f(a1.v[e2], x1.v[e2]);
          }
        }
        acc = Op<T, OP>::f(a0.v[0], a1.v[0]);
#pragma unroll
        for (int e2 = 1; e2 < VEC; ++e2) acc = Op<T, OP>::f(acc, Op<T, OP>::f(a0.v[e2], a1.v[e2]));
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) acc = Op<T, OP>::f(acc, __shfl_xor_sync(FULL, acc, off));
      } else {  // the ragged last tile: plain loads straight from global memory
        const T* src = a.in + (long long)t * TILE;
        bool has = false;
        for (int i = lane; i < len; i += 32) {
          acc = has ? Op<T, OP>::f(acc, src[i]) : src[i];
          has = true;
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
          const T o = __shfl_down_sync(FULL, acc, off);
          const int oh = __shfl_down_sync(FULL, (int)has, off);
          if (lane + off < 32 && oh) {
            acc = has ? Op<T, OP>::f(acc, o) : o;
            has = true;
          }
        }
        acc = __shfl_sync(FULL, acc, 0);
      }
      __syncwarp();
      if (lane == 0) {
        sh.q_tagg[e][pos] = acc;
        __threadfence_block();
        sh.b_reduced[slot] = k + 1;  // the buffer may take a new tile
        // The reducer of a run's last tile publishes the run's aggregate.
        if (atomicAdd(&sh.q_count[e], 1) + 1 == sh.q_ntiles[e]) {
          __threadfence_block();
          T ra = sh.q_tagg[e][0];
          for (int i = 1; i < sh.q_ntiles[e]; ++i) ra = Op<T, OP>::f(ra, sh.q_tagg[e][i]);
          const unsigned r = sh.q_run[e];
          if ((long long)r != a.stalled_run) st.publish(r, r == 0 ? FLAG_P : FLAG_A, ra);
          sh.q_agg[e] = ra;
          __threadfence_block();
          sh.q_aready[e] = 1;
        }
      }
    }
  } else if (warp < C::WS) {
    // ------------------------------------------------------ B: look-back -------
    // Look-back warp b takes the CTA's runs b, b+NB, ... in claim order.
    for (unsigned next = warp - C::WB;; next += C::NB) {
      const unsigned e = next % QD;
      int status = 0;  // 1: a run to process, 2: all done, 3: gave up
      if (lane == 0) {
        // Entry e holds run `next` only once I has claimed it (the slot may still
        // carry the flag of the run QD entries earlier until I reuses it).
        const bool got = stash_wait(
            [&] { return (next < sh.claimed && sh.q_aready[e]) || (sh.i_finished && sh.claimed <= next); },
            a.wait_ns, &sh.abort);
        __threadfence_block();
        status = !got ? 3 : ((next < sh.claimed && sh.q_aready[e]) ? 1 : 2);
        if (status == 3) fail();
      }
      status = __shfl_sync(FULL, status, 0);
      __syncwarp();
      if (status != 1) break;
      const unsigned r = sh.q_run[e];
      const T agg = sh.q_agg[e];
      T pfx{};
      if (r > 0) {
        bool timed_out;
        pfx = lookback_warp<T, OP, C::K>(st, 0, r, a.wait_ns, timed_out);
        if (lane == 0) {
          if ((long long)r != a.stalled_run) st.publish(r, FLAG_P, Op<T, OP>::f(pfx, agg));
          if (timed_out) raise_err(a.err, ERRBIT_TIMEOUT);
        }
      }
      if (lane == 0) {
        sh.q_pfx[e] = pfx;
        sh.q_has[e] = r > 0;
        __threadfence_block();
        sh.q_pready[e] = 1;
      }
      __syncwarp();
    }
  } else {
    // ------------------------------------------------------ S groups -----------
    // Group g scans the queue entries g, g+NG, g+2NG, ... (whole runs).  Its first
    // thread owns the group's control state (which tiles are being re-loaded, what
    // comes next) and hands each decision to the group through the control block,
    // so all threads of the group always take the same path through its barrier.
    constexpr int NS = C::NS;
    const int g = (warp - C::WS) / NSW, sw = (warp - C::WS) % NSW;
    const int stid = tid - 32 * C::WS - g * NST;
    T* buf_s = buf + (size_t)(NL + g * NS) * TILE;
    const unsigned long long pol = l2_policy_evict_first();
    unsigned issued = 0, scanned = 0, phase = 0;  // (first thread only)
    unsigned ient = g, sent = g;                  // entry sequence numbers being loaded / scanned
    int itile = 0, stile = 0;
    T carry{};
    bool has_carry = false;
    const int p0 = (sw * ROUNDS * 32 + lane) * VEC;  // the thread's first element within a tile
    for (;;) {
      if (stid == 0) {
        int cmd = S_SCAN;
        for (;;) {
          // Re-load (from L2) tiles of this group's runs whose aggregate is out (their
          // tiles are in L2 from then on); the prefix is needed only to scan them.
          while (issued - scanned < (unsigned)NS && ient < sh.claimed && sh.q_aready[ient % QD]) {
            __threadfence_block();
            const unsigned e = ient % QD;
            const unsigned r = sh.q_run[e];
            const unsigned t = r * RUN + itile;
            const int slot = issued % NS;
            if (tile_len(t) == TILE) {
              mbar_arrive_expect_tx(&sh.bar_s[g][slot], TILE * sizeof(T));
              bulk_g2s_hint(buf_s + (size_t)slot * TILE, a.in + (long long)t * TILE, TILE * sizeof(T),
                            &sh.bar_s[g][slot], pol);
            }
            ++issued;
            if (++itile == tiles_in_run(r)) {
              ient += NG;
              itile = 0;
            }
          }
          if (scanned < issued) {
            // The next tile to scan is loading; its run's prefix must be known.
            if (!stash_wait([&] { return sh.q_pready[sent % QD] != 0; }, a.wait_ns, &sh.abort)) {
              cmd = S_EXIT_ERR;
              fail();
            }
            __threadfence_block();
            break;
          }
          auto aready = [&] { return ient < sh.claimed && sh.q_aready[ient % QD] != 0; };
          const bool got = stash_wait([&] { return aready() || (sh.i_finished && ient >= sh.claimed); },
                                      a.wait_ns, &sh.abort);
          __threadfence_block();
          if (!got) {
            cmd = S_EXIT_ERR;
            fail();
            break;
          }
          if (aready()) continue;
          cmd = S_EXIT;
          break;
        }
        if (cmd == S_SCAN) {
          const unsigned e = sent % QD;
          const unsigned r = sh.q_run[e];
          const unsigned t = r * RUN + stile;
          const int slot = scanned % NS;
          sh.c_tile[g] = t;
          sh.c_entry[g] = e;
          sh.c_len[g] = tile_len(t);
          sh.c_slot[g] = slot;
          sh.c_parity[g] = (phase >> slot) & 1u;
          sh.c_run_start[g] = stile == 0;
          sh.c_run_end[g] = stile + 1 == tiles_in_run(r);
          if (stile == 0) {
            bool h = sh.q_has[e] != 0;
            T c = sh.q_pfx[e];
            if (!a.inclusive) {
              c = h ? Op<T, OP>::f(a.init, c) : a.init;
              h = true;
            }
            sh.c_carry[g] = c;
            sh.c_has[g] = h;
          }
          if (sh.c_len[g] == TILE) phase ^= 1u << slot;
          ++scanned;
          if (++stile == tiles_in_run(r)) {
            sent += NG;
            stile = 0;
          }
        }
        sh.c_cmd[g] = cmd;
      }
      s_group_sync<NST>(g);
      if (sh.c_cmd[g] != S_SCAN) break;
      const unsigned t = sh.c_tile[g], e = sh.c_entry[g];
      const int len = sh.c_len[g], slot = sh.c_slot[g];
      const bool run_end = sh.c_run_end[g] != 0;
      if (sh.c_run_start[g]) {
        carry = sh.c_carry[g];
        has_carry = sh.c_has[g] != 0;
      }
      Vec<T> x[ROUNDS];
      bool landed = true;
      if (len == TILE) {
        landed = mbar_wait(&sh.bar_s[g][slot], (unsigned)sh.c_parity[g], a.wait_ns);
        const uint4* v = reinterpret_cast<const uint4*>(buf_s + (size_t)slot * TILE) + sw * ROUNDS * 32 + lane;
#pragma unroll
        for (int j = 0; j < ROUNDS; ++j) x[j] = ld_vec<T>(v + j * 32);
      } else {  // the ragged last tile: element loads, zero past the end
#pragma unroll
        for (int j = 0; j < ROUNDS; ++j)
#pragma unroll
          for (int e2 = 0; e2 < VEC; ++e2) {
            const int p = p0 + j * 32 * VEC + e2;
            x[j].v[e2] = p < len ? a.in[(long long)t * TILE + p] : T{};
          }
      }
      T pre[ROUNDS];
      const T wtot = regs_reduce_pass<T, OP, ROUNDS>(x, lane, pre);
      if (lane == 0) sh.s_warp[g][sw] = wtot;
      // After this barrier every thread holds its part of the tile: the buffer is free.
      if (!s_group_and<NST>(g, landed)) {
        if (stid == 0) fail();
        break;
      }
      if (sw == 0) block_scan_warp_totals<T, OP, NSW>(sh.s_warp[g], lane);
      s_group_sync<NST>(g);
      T base = carry;
      bool hb = has_carry;
      if (sw > 0) {
        const T wp = sh.s_warp[g][sw - 1];
        base = hb ? Op<T, OP>::f(base, wp) : wp;
        hb = true;
      }
      const T tagg = sh.s_warp[g][NSW - 1];
      regs_apply_pass<T, OP, ROUNDS>(x, lane, pre, base, hb, a.inclusive != 0);
      carry = has_carry ? Op<T, OP>::f(carry, tagg) : tagg;
      has_carry = true;
      if (len == TILE) {
        uint4* dst = reinterpret_cast<uint4*>(a.out) + (long long)t * (TILE / VEC) + sw * ROUNDS * 32 + lane;
#pragma unroll
        for (int j = 0; j < ROUNDS; ++j) {
          uint4 u;
          memcpy(&u, x[j].v, 16);
          st_hint(dst + j * 32, u, pol);
        }
      } else {
#pragma unroll
        for (int j = 0; j < ROUNDS; ++j)
#pragma unroll
          for (int e2 = 0; e2 < VEC; ++e2) {
            const int p = p0 + j * 32 * VEC + e2;
            if (p < len) a.out[(long long)t * TILE + p] = x[j].v[e2];
          }
      }
      if (stid == 0 && run_end) {
        __threadfence_block();
        sh.q_fin[e] = 1;  // the run is written: I may reuse its queue entry
      }
    }
    if (stid == 0) {  // no bulk load may still be landing when the CTA exits
      for (unsigned i = scanned; i < issued; ++i)
        if (mbar_wait(&sh.bar_s[g][i % NS], (phase >> (i % NS)) & 1u, a.wait_ns)) phase ^= 1u << (i % NS);
    }
  }
}

template <class T> unsigned stash_runs(long long n) {
  const long long tiles = (n + StashCfg<T>::TILE - 1) / StashCfg<T>::TILE;
  return (unsigned)((tiles + StashCfg<T>::RUN - 1) / StashCfg<T>::RUN);
}
template <class T> size_t stash_status_bytes(long long n) {
  const size_t runs = stash_runs<T>(n);
  if (sizeof(T) == 4) return round_up(runs * 8, 256);
  return round_up(runs * 4, 256) + 2 * round_up(runs * sizeof(T), 256);
}
template <class T> size_t stash_reset_bytes(long long n) {
  const size_t runs = stash_runs<T>(n);
  return kHeaderBytes + (sizeof(T) == 4 ? round_up(runs * 8, 256) : round_up(runs * 4, 256));
}

// When the L2-resident scan applies: one row, 16-byte aligned data, and enough
// tiles that the persistent grid has work for every SM.
template <class T> bool stash_applies(const ScanJob& job, int num_sms) {
  // Not for fp64: there the arithmetic, not HBM, is the limit (GB300 adds fp64 at a
  // small fraction of its fp32 rate), and the extra reduction would cost one more
  // add per element.
  if (std::is_same<T, double>::value) return false;
  return job.B == 1 && job.C == 1 && (uintptr_t)job.in % 16 == 0 && (uintptr_t)job.out % 16 == 0 &&
         job.R >= (long long)num_sms * StashCfg<T>::TILE * StashCfg<T>::RUN * 4;
}

template <class T, int OP, class C = StashCfg<T>>
cudaError_t launch_stash_op(const ScanJob& job, const LaunchCtx& ctx) {
  StashArgs<T> a;
  a.in = (const T*)job.in;
  a.out = (T*)job.out;
  a.n = job.R;
  a.num_tiles = (unsigned)((job.R + C::TILE - 1) / C::TILE);
  a.num_runs = (a.num_tiles + C::RUN - 1) / C::RUN;
  a.counter = (unsigned*)job.temp;
  a.err = ctx.err;
  a.init = T{};
  if (!job.inclusive && job.init_host) memcpy(&a.init, job.init_host, sizeof(T));
  a.inclusive = job.inclusive;
  a.wait_ns = ctx.wait_ns;
  a.stalled_run = ctx.stalled_tile;
  typename StatusFor<T>::type st;
  char* base = (char*)job.temp + kHeaderBytes;
  if constexpr (sizeof(T) == 4) {
    st.w = (unsigned long long*)base;
  } else {
    const size_t runs = a.num_runs;
    st.flag = (unsigned*)base;
    st.agg = (T*)(base + round_up(runs * 4, 256));
    st.pfx = (T*)(base + round_up(runs * 4, 256) + round_up(runs * sizeof(T), 256));
  }
  auto kern = scan_stash_kernel<T, OP, decltype(st), C>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::SMEM);
  if (e != cudaSuccess) return e;
  int grid = ctx.num_sms;
  if ((unsigned)grid > a.num_runs) grid = (int)a.num_runs;
  profile_before(ctx);
  e = clear_status(job.temp, kHeaderBytes + (size_t)a.num_runs * (sizeof(T) == 4 ? 8 : 4), nullptr, 0, ctx);
  if (e == cudaSuccess) e = launch_pdl(kern, grid, C::NT, C::SMEM, ctx.stream, a, st);
  profile_after(ctx);
  return e;
}

}  // namespace gbs
