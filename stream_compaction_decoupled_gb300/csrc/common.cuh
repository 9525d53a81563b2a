// common.cuh -- device helpers shared by the scan, compaction and packing kernels:
// the operators, bit casts, inline-PTX memory accesses with explicit semantics
// (relaxed / acquire / release at GPU scope), the mbarrier and bulk-copy (TMA)
// primitives, and the register-only warp scan.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <type_traits>

namespace gbs {

// Tile-status flags of the decoupled look-back (The CUDA Handbook, 13.3.4,
// Listing 13-13): X = nothing published, A = aggregate available, P = inclusive
// prefix available.  X must be 0: a zeroed status array reads as all-X.
enum : unsigned { FLAG_X = 0, FLAG_A = 1, FLAG_P = 2 };

// Bits of the sticky device error word.
enum : unsigned { ERRBIT_TIMEOUT = 1u, ERRBIT_RANGE = 2u, ERRBIT_INVALID = 4u };

// Operators (the public gb_op values, plus OP_SATADD, internal to packing: unsigned
// add saturating at 2^31, which keeps record offsets from wrapping while staying
// associative).
enum { OP_ADD = 0, OP_MAX = 1, OP_MIN = 2, OP_MUL = 3, OP_SATADD = 16 };

// Op<T, OP>::f(a, b) = a (+) b, with `a` the earlier operand in scan order.
template <class T, int OP> struct Op;

template <class T> struct Op<T, OP_ADD> {
  static __device__ __forceinline__ T f(T a, T b) {
    if constexpr (std::is_integral<T>::value) {
      using U = typename std::make_unsigned<T>::type;
      return (T)((U)a + (U)b);  // two's-complement wraparound
    } else {
      return a + b;
    }
  }
};
template <class T> struct Op<T, OP_MUL> {
  static __device__ __forceinline__ T f(T a, T b) {
    if constexpr (std::is_integral<T>::value) {
      using U = typename std::make_unsigned<T>::type;
      return (T)((U)a * (U)b);  // the low bits of the product (two's complement)
    } else {
      return a * b;
    }
  }
};
template <class T> struct Op<T, OP_MAX> {
  static __device__ __forceinline__ T f(T a, T b) {
    if constexpr (std::is_same<T, float>::value) return fmaxf(a, b);
    else if constexpr (std::is_same<T, double>::value) return fmax(a, b);
    else return a > b ? a : b;
  }
};
template <class T> struct Op<T, OP_MIN> {
  static __device__ __forceinline__ T f(T a, T b) {
    if constexpr (std::is_same<T, float>::value) return fminf(a, b);
    else if constexpr (std::is_same<T, double>::value) return fmin(a, b);
    else return a < b ? a : b;
  }
};
template <> struct Op<unsigned, OP_SATADD> {
  static __device__ __forceinline__ unsigned f(unsigned a, unsigned b) {
    unsigned long long s = (unsigned long long)a + b;
    return s > 0x80000000ull ? 0x80000000u : (unsigned)s;
  }
};

// ---- bit casts ------------------------------------------------------------------

template <class T> __device__ __forceinline__ unsigned to_u32(T v) {
  static_assert(sizeof(T) == 4, "4-byte type");
  unsigned u;
  memcpy(&u, &v, 4);
  return u;
}
template <class T> __device__ __forceinline__ T from_u32(unsigned u) {
  T v;
  memcpy(&v, &u, 4);
  return v;
}
template <class T> __device__ __forceinline__ unsigned long long to_u64(T v) {
  static_assert(sizeof(T) == 8, "8-byte type");
  unsigned long long u;
  memcpy(&u, &v, 8);
  return u;
}
template <class T> __device__ __forceinline__ T from_u64(unsigned long long u) {
  T v;
  memcpy(&v, &u, 8);
  return v;
}

// 16-byte vectors of T, moved as uint4.
template <class T> struct Vec {
  static constexpr int N = 16 / sizeof(T);
  T v[N];
};
template <class T> __device__ __forceinline__ Vec<T> ld_vec(const uint4* p) {
  uint4 r = *p;
  Vec<T> out;
  memcpy(out.v, &r, 16);
  return out;
}
template <class T> __device__ __forceinline__ void st_vec(uint4* p, const Vec<T>& x) {
  uint4 r;
  memcpy(&r, x.v, 16);
  *p = r;
}

// ---- memory accesses with explicit semantics (GPU scope) -------------------------

__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_relaxed_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ unsigned ld_relaxed_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_relaxed_u32(unsigned* p, unsigned v) {
  asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_u32(unsigned* p, unsigned v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Relaxed GPU-scope load/store of a 4- or 8-byte value (through L2, never a
// stale L1 line).
template <class T> __device__ __forceinline__ T ld_relaxed(const T* p) {
  if constexpr (sizeof(T) == 8) return from_u64<T>(ld_relaxed_u64((const unsigned long long*)p));
  else return from_u32<T>(ld_relaxed_u32((const unsigned*)p));
}
template <class T> __device__ __forceinline__ void st_relaxed(T* p, T v) {
  if constexpr (sizeof(T) == 8) st_relaxed_u64((unsigned long long*)p, to_u64(v));
  else st_relaxed_u32((unsigned*)p, to_u32(v));
}

// Acquire / release on a shared-memory flag within the CTA (one warp posts values in
// shared memory, the others read them once they see the flag).
__device__ __forceinline__ unsigned ld_acquire_cta_shared(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.cta.shared.u32 %0, [%1];" : "=r"(v) : "r"((unsigned)__cvta_generic_to_shared(p)) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_cta_shared(unsigned* p, unsigned v) {
  asm volatile("st.release.cta.shared.u32 [%0], %1;" ::"r"((unsigned)__cvta_generic_to_shared(p)), "r"(v) : "memory");
}

__device__ __forceinline__ unsigned long long globaltimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---- mbarrier and bulk (TMA) copies ------------------------------------------

__device__ __forceinline__ unsigned smem_u32(const void* p) {
  return (unsigned)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(unsigned long long* bar, unsigned count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
// Make an mbarrier initialisation visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(unsigned long long* bar, unsigned bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(unsigned long long* bar, unsigned parity) {
  unsigned ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Wait for phase `parity` of an mbarrier, for at most limit_ns of global time.
__device__ __forceinline__ bool mbar_wait(unsigned long long* bar, unsigned parity,
                                          unsigned long long limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer() - t0 > limit_ns) return false;
  }
  return true;
}
// Global -> shared bulk copy completing on an mbarrier.  16-byte aligned addresses,
// size a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* smem_dst, const void* gsrc, unsigned bytes,
                                         unsigned long long* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(smem_dst)),
      "l"(gsrc), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}
// Shared -> global bulk copy tracked by the issuing thread's bulk groups.
__device__ __forceinline__ void bulk_s2g(void* gdst, const void* smem_src, unsigned bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gdst),
               "r"(smem_u32(smem_src)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Wait until the source shared memory of every committed bulk store has been read.
__device__ __forceinline__ void bulk_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// Order this thread's generic-proxy shared-memory writes before later async-proxy
// (bulk copy) reads of them.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---- L2 cache-eviction hints ---------------------------------------------------

// Policies for the .L2::cache_hint qualifier: evict_last keeps lines that will be
// read again (an input re-read from L2), evict_first marks lines at their last use
// (a streamed output, an input read for the last time).
__device__ __forceinline__ unsigned long long l2_policy_evict_last() {
  unsigned long long p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ unsigned long long l2_policy_evict_first() {
  unsigned long long p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ void bulk_g2s_hint(void* smem_dst, const void* gsrc, unsigned bytes,
                                              unsigned long long* bar, unsigned long long pol) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_u32(smem_dst)),
      "l"(gsrc), "r"(bytes), "r"(smem_u32(bar)), "l"(pol)
      : "memory");
}
__device__ __forceinline__ uint4 ld_hint(const uint4* p, unsigned long long pol) {
  uint4 r;
  asm volatile("ld.global.L1::no_allocate.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p), "l"(pol));
  return r;
}
// The same load allocating in L1: for layouts in which each lane owns 64 consecutive
// bytes, so that one instruction reads 16 bytes of each of 32 sectors 64 bytes apart
// and the next three read the rest of the same sectors.  Without L1 allocation each
// sector would travel from L2 twice.
__device__ __forceinline__ uint4 ld_hint_l1(const uint4* p, unsigned long long pol) {
  uint4 r;
  asm volatile("ld.global.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p), "l"(pol));
  return r;
}
// One 32-byte load (sm_100 and later; p 32-byte aligned) with an L2 policy: a lane
// that owns 64 consecutive bytes reads them in two instructions of whole sectors.
__device__ __forceinline__ void ld_hint32(const void* p, unsigned long long pol, uint4& lo, uint4& hi) {
  asm volatile("ld.global.L1::no_allocate.L2::cache_hint.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8], %9;"
               : "=r"(lo.x), "=r"(lo.y), "=r"(lo.z), "=r"(lo.w), "=r"(hi.x), "=r"(hi.y), "=r"(hi.z), "=r"(hi.w)
               : "l"(p), "l"(pol));
}
__device__ __forceinline__ void st_hint(uint4* p, uint4 v, unsigned long long pol) {
  asm volatile("st.global.L2::cache_hint.v4.u32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(p), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w), "l"(pol)
               : "memory");
}
__device__ __forceinline__ bool aligned16(const void* p) {
  return ((uintptr_t)p & 15u) == 0;
}

// ---- programmatic dependent launch ---------------------------------------------

// Every kernel of the library is launched with programmatic stream serialization
// (launch_pdl) and begins with pdl_entry(): griddepcontrol.wait returns once the
// previous grid in the stream has completed and its writes are visible, so inputs
// written by a preceding kernel, and scratch still in use by a preceding call, are
// safe to touch after it; griddepcontrol.launch_dependents then lets the next launch
// in the stream be scheduled while this grid runs (it, too, waits before it reads).
// The launches of a call thus overlap the kernels before them instead of following
// them.  Neither instruction spins in software: the wait is a hardware dependency.
__device__ __forceinline__ void pdl_entry() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---- warp scan -------------------------------------------------------------------

// Inclusive scan over the 32 lanes of a warp, in registers (The CUDA Handbook,
// 13.3.1).  In the step of distance d each lane takes the running value of the lane d
// below it and combines it on its left; after the step a lane covers the 2d lanes
// ending at it.  Lanes below d have nothing below them and keep their value, which is
// what lets operators without a neutral element (MAX, MIN) use it unchanged.
template <class T, int OP> __device__ __forceinline__ T warp_inclusive(T v, int lane) {
#pragma unroll
  for (int d = 1; d < 32; d *= 2) {
    const T below = __shfl_up_sync(0xffffffffu, v, d);
    v = lane >= d ? Op<T, OP>::f(below, v) : v;
  }
  return v;
}

__device__ __forceinline__ unsigned lanemask_lt() {
  unsigned m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// Pause between polls of a tile status: short, because a predecessor that is still
// X usually publishes within a memory round trip or two.
__device__ __forceinline__ void backoff(int spins) {
  __nanosleep(spins < 3 ? (32u << spins) : 256u);
}

}  // namespace gbs
