// kernels.cuh -- sm_103a kernels of the per-shard mixed-precision ZeRO step.
//
// Pass 1 (steps a1..a4) has two forms:
//   pass1_bulk_kernel (one gradient buffer, the usual case): chunks of 4 or 8
//     tiles are staged into shared memory by bulk copies (TMA, cp.async.bulk
//     on an mbarrier, two stages per CTA);
//   pass1_multi_kernel (R*K > 1 buffers): summed per element in binary32
//     (rank-major order, starting from +0), optionally stored (the stash).
//   Each accumulates the overflow flag and the exact sum of squares (in
//   binary32 pairs, binary64 only for values outside binary32's exact-square
//   range).  Every CTA publishes one binary64 partial, summed in binary32
//   pairs and rounded once; the CTA that finishes last (atomic ticket, no
//   waiting) folds the partials in a fixed order in binary64 (one warp for
//   grids of up to 128 CTAs), takes the per-step decisions (skip, clip
//   coefficient, Adam scalars) and advances the rank's loss-scaler state.
//   One extra CTA prepares the next step's update scalars while the others
//   stream.  Pass 1 is a programmatic dependent launch of whatever precedes
//   it on the stream and waits for it at its very start.
// pass2_kernel (steps a5..a7): a programmatic dependent launch of pass 1; it
//   loads the decision together with its first tile, and on a skip every CTA
//   stores nothing; otherwise it applies unscale x clip, AdamW on the fp32
//   master copy (or the widened 16-bit master) and m, v, and writes the
//   16-bit parameter copy.
//
// Both passes are HBM-bandwidth bound streaming kernels.  Tiles are 2048
// elements (256 threads x 8); a thread moves each of its streams with one
// 16-byte access per tile when every pointer of the run is 16-byte aligned
// (vector path) and element by element otherwise.  Pass 2 visits its tiles in
// the reverse of pass 1's order so that the gradients pass 1 touched last are
// still in L2 when pass 2 starts.
//
// Rounding: every binary32 operation of the update is an explicit IEEE
// round-to-nearest intrinsic (__fmul_rn, __fadd_rn, __fsqrt_rn, __fdiv_rn), so
// no multiply-add is ever contracted and results do not depend on the
// compiler's fusion choices; 16-bit stores use __float2half_rn /
// __float2bfloat16_rn.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "decide_core.h"
#include "zero_opt_internal.h"

// Resident CTAs per SM each kernel is compiled for (register budget 65536 /
// (256 * n) per thread).
#ifndef ZO_PASS1_MIN_CTAS
#define ZO_PASS1_MIN_CTAS 4
#endif
#ifndef ZO_PASS2_MIN_CTAS
#define ZO_PASS2_MIN_CTAS 2
#endif
// With 16-bit masters a thread has fewer bytes in flight per tile (96 instead
// of 112 with one gradient buffer), so pass 2 takes a third CTA per SM to keep
// enough reads in flight (not with re-read buffers, whose eight loads in
// flight need the registers of two).
#ifndef ZO_PASS2_M16_MIN_CTAS
#define ZO_PASS2_M16_MIN_CTAS 3
#endif
// The multi-buffer pass 1 holds eight 16-byte loads in flight per thread and
// needs the larger register budget of three CTAs per SM.
#ifndef ZO_MULTI_MIN_CTAS
#define ZO_MULTI_MIN_CTAS 3
#endif

namespace zo {

// ------------------------------------------------------------- 16-bit formats
template <typename T>
struct Fmt;

template <>
struct Fmt<__half> {
  static __device__ __forceinline__ float dec(unsigned short b) {
    return __half2float(__ushort_as_half(b));
  }
  static __device__ __forceinline__ unsigned short enc(float f) {
    return __half_as_ushort(__float2half_rn(f));
  }
  static __device__ __forceinline__ void dec8(const uint4& u, float (&f)[kVec]) {
    const __half2* h = reinterpret_cast<const __half2*>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 t = __half22float2(h[i]);
      f[2 * i] = t.x;
      f[2 * i + 1] = t.y;
    }
  }
  // the two fp16 values of a 32-bit word, low half first
  static __device__ __forceinline__ float2 dec2(uint32_t w) {
    return __half22float2(*reinterpret_cast<const __half2*>(&w));
  }
  static constexpr uint32_t kInf = 0x7C00u;      // |bits| >= kInf: inf or NaN
  // Every finite fp16 value lies in [2^-24, 2^16): inside the exact range of
  // the sum of squares, so only inf/NaN leave the fast path.
  static __device__ __forceinline__ bool fast16(uint32_t t16) { return t16 < kInf; }
  static __device__ __forceinline__ uint4 enc8(const float (&f)[kVec]) {
    uint4 u;
    __half2* h = reinterpret_cast<__half2*>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = __floats2half2_rn(f[2 * i], f[2 * i + 1]);
    return u;
  }
};

template <>
struct Fmt<__nv_bfloat16> {
  static __device__ __forceinline__ float dec(unsigned short b) {
    return __bfloat162float(__ushort_as_bfloat16(b));
  }
  static __device__ __forceinline__ unsigned short enc(float f) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(f));
  }
  static __device__ __forceinline__ void dec8(const uint4& u, float (&f)[kVec]) {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 t = __bfloat1622float2(h[i]);
      f[2 * i] = t.x;
      f[2 * i + 1] = t.y;
    }
  }
  // bf16 is the upper half of binary32: the widening is a shift or a mask
  static __device__ __forceinline__ float2 dec2(uint32_t w) {
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
  }
  static constexpr uint32_t kInf = 0x7F80u;
  // fast range [2^-40, 2^50) (or all zero), as for binary32 sums
  static __device__ __forceinline__ bool fast16(uint32_t t16) {
    return t16 < 0x5880u && (t16 >= 0x2B80u || t16 == 0u);
  }
  static __device__ __forceinline__ uint4 enc8(const float (&f)[kVec]) {
    uint4 u;
    __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
    return u;
  }
};

// ------------------------------------------------------------- run lookup
// Tiles of all runs form one index space; a CTA-uniform cursor finds the run
// of a tile by binary search over the runs' first tiles and keeps it while
// consecutive tiles stay inside it.
struct RunCursor {
  int64_t begin = 0, end = 0;
  Seg s;
  __device__ __forceinline__ void seek(const Seg* __restrict__ segs, int nseg,
                                       int64_t tile) {
    if (tile >= begin && tile < end) return;
    int lo = 0, hi = nseg - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (segs[mid].tile0 <= tile) lo = mid;
      else hi = mid - 1;
    }
    s = segs[lo];
    begin = s.tile0;
    end = s.tile0 + s.ntiles;
  }
};

// The fields of a run that pass 1 needs (it never touches master/m/v/p16),
// so that the cursor costs few registers.
struct RunCursorLite {
  int64_t begin = 0, end = 0;
  struct {
    int64_t tile0, n, stash_off;
    int32_t gbase, vec;
  } s;
  __device__ __forceinline__ void seek(const Seg* __restrict__ segs, int nseg,
                                       int64_t tile) {
    if (tile >= begin && tile < end) return;
    int lo = 0, hi = nseg - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (segs[mid].tile0 <= tile) lo = mid;
      else hi = mid - 1;
    }
    const Seg& g = segs[lo];
    s.tile0 = g.tile0;
    s.n = g.n;
    s.stash_off = g.stash_off;
    s.gbase = g.gbase;
    s.vec = g.vec;
    begin = g.tile0;
    end = g.tile0 + g.ntiles;
  }
};

template <typename S>
__device__ __forceinline__ const unsigned short* grad_ptr(const void* const* gptrs,
                                                          const S& s, int b) {
  const unsigned long long raw =
      __ldg(reinterpret_cast<const unsigned long long*>(gptrs) + s.gbase + b);
  return reinterpret_cast<const unsigned short*>(raw);
}

// Programmatic dependent launch: pass 1 lets pass 2 be scheduled before it
// ends (each CTA signals at its start); pass 2 waits for pass 1 to complete,
// with all its memory visible, before it reads anything pass 1 writes.
#ifndef ZO_PDL
#define ZO_PDL 1
#endif
__device__ __forceinline__ void pdl_launch_dependents() {
#if ZO_PDL
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
#endif
}
__device__ __forceinline__ void pdl_wait() {
#if ZO_PDL
  asm volatile("griddepcontrol.wait;" ::: "memory");
#endif
}
// Pass 1 as a dependent launch of whatever kernel precedes it on the stream
// (the previous step's pass 2, or the caller's last kernel): its CTAs may be
// scheduled before that kernel ends, and wait at their very start, before
// any memory access, for it to complete with all its memory visible.
#ifndef ZO_PDL_PASS1
#define ZO_PDL_PASS1 1
#endif
__device__ __forceinline__ void pass1_prologue() {
  pdl_launch_dependents();
#if ZO_PDL_PASS1
  pdl_wait();
#endif
}
// Return the 128-byte L2 line at `p` (128-byte aligned) to evict_normal.
__device__ __forceinline__ void l2_normal(const void* p) {
  asm volatile("applypriority.global.L2::evict_normal [%0], 128;" ::"l"(p) : "memory");
}
// Warm L2 with `bytes` at `p` (16-byte aligned, a multiple of 16 bytes).
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// ------------------------------------------------------------- sum of squares
// The global norm needs the sum of squares of the reduced gradients to well
// below binary32 precision (the clip coefficient is rounded to binary32 from
// it), but GB300's binary64 rate is far too low for a binary64 operation per
// element.  Each square is therefore formed exactly as p + e (p = s*s rounded,
// e = fma(s, s, -p)) and added into a per-thread double-binary32 accumulator
// (hi, lo) with Knuth's TwoSum; even and odd elements go to two independent
// accumulators (the two lanes of one f32x2 register pair)
// so consecutive additions do not wait on each other.  The thread's total
// hi + lo is taken in binary64; the accumulated error is a few units of 2^-48
// of the thread's sum.  Every operation is an explicit IEEE round-to-nearest
// operation (a scalar _rn intrinsic, or an f32x2 instruction with .rn in
// inline PTX), so nothing is contracted.  Tiles whose largest
// |s| is 2^50 or more (squares near the binary32 overflow range, or inf/NaN),
// or whose values are all nonzero and below 2^-40 (squares near underflow),
// are summed in binary64 instead.  amax (the largest |s| bit pattern seen)
// gives the overflow flag: inf and NaN patterns are >= 0x7f800000.

// Two binary32 lanes in one 64-bit register, for the f32x2 instructions.  The
// explicit .rn rounding keeps each lane an IEEE binary32 operation that the
// compiler never contracts, so a lane rounds exactly as the scalar _rn
// intrinsic does.
typedef unsigned long long f32x2;
__device__ __forceinline__ f32x2 f2_pack(float a, float b) {
  return (f32x2)__float_as_uint(a) | ((f32x2)__float_as_uint(b) << 32);
}
__device__ __forceinline__ float f2_lo(f32x2 v) { return __uint_as_float((uint32_t)v); }
__device__ __forceinline__ float f2_hi(f32x2 v) { return __uint_as_float((uint32_t)(v >> 32)); }
__device__ __forceinline__ f32x2 f2_add(f32x2 a, f32x2 b) {
  f32x2 d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ f32x2 f2_sub(f32x2 a, f32x2 b) {
  f32x2 d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ f32x2 f2_mul(f32x2 a, f32x2 b) {
  f32x2 d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ f32x2 f2_fma(f32x2 a, f32x2 b, f32x2 c) {
  f32x2 d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}

// (hi, lo) + (hi, lo) in binary32 operations: TwoSum of the high parts, the
// low parts added to its error, renormalised by Fast2Sum (Dekker).  Used on
// non-negative sums of squares, where the renormalisation's condition
// |s| >= |e| holds; the result carries about 44 significant bits.
__device__ __forceinline__ float2 add22(float2 a, float2 b) {
  const float s = __fadd_rn(a.x, b.x);
  const float bp = __fsub_rn(s, a.x);
  float e = __fadd_rn(__fsub_rn(a.x, __fsub_rn(s, bp)), __fsub_rn(b.x, bp));
  e = __fadd_rn(e, __fadd_rn(a.y, b.y));
  const float hi = __fadd_rn(s, e);
  return make_float2(hi, __fsub_rn(e, __fsub_rn(hi, s)));
}

struct SqAcc {
  f32x2 H = 0ull, L = 0ull;    // lane 0 and lane 1 in one register each
  f32x2 H2 = 0ull, L2 = 0ull;  // a second pair (add_raw16_2): two dependency chains
  double slow = 0.0;
  uint32_t amax = 0u;

  // a to lane 0, b to lane 1.
  __device__ __forceinline__ void pair(float a, float b) {
    const f32x2 X = f2_pack(a, b);
    const f32x2 P = f2_mul(X, X);
    const f32x2 E = f2_fma(X, X, P ^ 0x8000000080000000ull);
    const f32x2 T = f2_add(H, P);
    const f32x2 BP = f2_sub(T, H);
    const f32x2 AP = f2_sub(T, BP);
    L = f2_add(L, f2_add(f2_add(f2_sub(H, AP), f2_sub(P, BP)), E));
    H = T;
  }
  static __device__ __forceinline__ void pair_exact_into(f32x2& H, f32x2& L, float a, float b) {
    const f32x2 X = f2_pack(a, b);
    const f32x2 P = f2_mul(X, X);
    const f32x2 T = f2_add(H, P);
    const f32x2 BP = f2_sub(T, H);
    const f32x2 AP = f2_sub(T, BP);
    L = f2_add(L, f2_add(f2_sub(H, AP), f2_sub(P, BP)));
    H = T;
  }
  // The same accumulation when every lane of H is at least the square being
  // added: Dekker's Fast2Sum, whose error term (H + P) - T is exact under
  // that condition and therefore bit-identical to TwoSum's, in four packed
  // operations instead of seven.
  static __device__ __forceinline__ void pair_fast_into(f32x2& H, f32x2& L, float a, float b) {
    const f32x2 X = f2_pack(a, b);
    const f32x2 P = f2_mul(X, X);
    const f32x2 T = f2_add(H, P);
    L = f2_add(L, f2_sub(P, f2_sub(T, H)));
    H = T;
  }
  __device__ __forceinline__ void pair_exact(float a, float b) {
    pair_exact_into(H, L, a, b);
  }

  // EXACT_SQ: every s is a converted 16-bit value, whose square (fp16: 22
  // significant bits, bf16: 16) is exact in binary32 inside the fast range.
  template <bool EXACT_SQ = false>
  __device__ __forceinline__ void add(const float (&s)[kVec]) {
    uint32_t tmax = 0u;
#pragma unroll
    for (int i = 0; i < kVec; ++i) tmax = max(tmax, __float_as_uint(s[i]) & 0x7fffffffu);
    amax = max(amax, tmax);
    const bool fast = tmax < 0x58800000u && (tmax >= 0x2B800000u || tmax == 0u);
    if (fast) {
#pragma unroll
      for (int i = 0; i < kVec; i += 2) {
        if (EXACT_SQ) pair_exact(s[i], s[i + 1]);
        else pair(s[i], s[i + 1]);
      }
    } else {
      double d = 0.0;
#pragma unroll
      for (int i = 0; i < kVec; ++i) d = __dadd_rn(d, __dmul_rn((double)s[i], (double)s[i]));
      slow = __dadd_rn(slow, d);
    }
  }
  // Eight raw 16-bit gradients of a single buffer (the sum is the value
  // itself).  The range and overflow checks run on the 16-bit patterns, two
  // at a time (__vmaxu2); the squares are exact in binary32.
  uint32_t amax16 = 0u;
  template <typename GT>
  __device__ __forceinline__ void add_raw16(const uint4& r) {
    const uint32_t m01 = __vmaxu2(r.x & 0x7fff7fffu, r.y & 0x7fff7fffu);
    const uint32_t m23 = __vmaxu2(r.z & 0x7fff7fffu, r.w & 0x7fff7fffu);
    const uint32_t mm = __vmaxu2(m01, m23);
    const uint32_t t16 = max(mm & 0xffffu, mm >> 16);
    amax16 = max(amax16, t16);
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
    if (Fmt<GT>::fast16(t16)) {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float2 x = Fmt<GT>::dec2(w[k]);
        pair_exact(x.x, x.y);
      }
    } else {
      double d = 0.0;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float2 x = Fmt<GT>::dec2(w[k]);
        d = __dadd_rn(d, __dmul_rn((double)x.x, (double)x.x));
        d = __dadd_rn(d, __dmul_rn((double)x.y, (double)x.y));
      }
      slow = __dadd_rn(slow, d);
    }
  }
  // As add_raw16 for two blocks of eight, into the two accumulator pairs.
  template <typename GT>
  __device__ __forceinline__ void add_raw16_2(const uint4& r, const uint4& q) {
    const uint32_t m0 = __vmaxu2(__vmaxu2(r.x & 0x7fff7fffu, r.y & 0x7fff7fffu),
                                 __vmaxu2(r.z & 0x7fff7fffu, r.w & 0x7fff7fffu));
    const uint32_t m1 = __vmaxu2(__vmaxu2(q.x & 0x7fff7fffu, q.y & 0x7fff7fffu),
                                 __vmaxu2(q.z & 0x7fff7fffu, q.w & 0x7fff7fffu));
    const uint32_t mm = __vmaxu2(m0, m1);
    const uint32_t t16 = max(mm & 0xffffu, mm >> 16);
    amax16 = max(amax16, t16);
    if (Fmt<GT>::fast16(t16)) {
      const uint32_t w[4] = {r.x, r.y, r.z, r.w};
      const uint32_t u[4] = {q.x, q.y, q.z, q.w};
      // The sums only grow (the squares are >= 0), so if the smallest of the
      // four running sums is at least the largest square of the sixteen, each
      // addition meets Fast2Sum's condition |H| >= |P|.
      const float mx = Fmt<GT>::dec((unsigned short)t16);
      const float hmin = fminf(fminf(f2_lo(H), f2_hi(H)), fminf(f2_lo(H2), f2_hi(H2)));
      if (hmin >= __fmul_rn(mx, mx)) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float2 x = Fmt<GT>::dec2(w[k]);
          const float2 y = Fmt<GT>::dec2(u[k]);
          pair_fast_into(H, L, x.x, x.y);
          pair_fast_into(H2, L2, y.x, y.y);
        }
      } else {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float2 x = Fmt<GT>::dec2(w[k]);
          const float2 y = Fmt<GT>::dec2(u[k]);
          pair_exact_into(H, L, x.x, x.y);
          pair_exact_into(H2, L2, y.x, y.y);
        }
      }
    } else {
      add_raw16<GT>(r);
      add_raw16<GT>(q);
    }
  }
  template <typename GT>
  __device__ __forceinline__ bool overflowed() const {
    return amax >= 0x7f800000u || amax16 >= Fmt<GT>::kInf;
  }

  __device__ __forceinline__ double total() const {
    const float hi0 = f2_lo(H), lo0 = f2_lo(L), hi1 = f2_hi(H), lo1 = f2_hi(L);
    double a = __dadd_rn((double)hi0, (double)lo0);
    double b = __dadd_rn((double)hi1, (double)lo1);
    a = __dadd_rn(a, __dadd_rn((double)f2_lo(H2), (double)f2_lo(L2)));
    b = __dadd_rn(b, __dadd_rn((double)f2_hi(H2), (double)f2_hi(L2)));
    return __dadd_rn(__dadd_rn(a, b), slow);
  }
  // The same sum without the binary64 part, in binary32 pairs (add22), for a
  // CTA none of whose threads took the binary64 path (slow == 0).
  __device__ __forceinline__ float2 total_ff() const {
    const float2 a = add22(make_float2(f2_lo(H), f2_lo(L)), make_float2(f2_hi(H), f2_hi(L)));
    const float2 b = add22(make_float2(f2_lo(H2), f2_lo(L2)), make_float2(f2_hi(H2), f2_hi(L2)));
    return add22(a, b);
  }
};

// Fixed-shape CTA sum of binary32 pairs (add22), rounded once to binary64 in
// thread 0 (where it is valid): the hi + lo of one pair is exact there.  The
// same tree as block_sum at binary32 speed; GB300's binary64 rate is a small
// fraction of its binary32 rate, and this sum sits on every step's serial
// path.
__device__ __forceinline__ double block_sum_ff(float2 v, float2* red) {
  __syncthreads();
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float2 o = make_float2(__shfl_down_sync(0xffffffffu, v.x, off),
                                 __shfl_down_sync(0xffffffffu, v.y, off));
    v = add22(v, o);
  }
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  double t = 0.0;
  if (threadIdx.x == 0) {
    float2 w = red[0];
#pragma unroll
    for (int k = 1; k < kThreads / 32; ++k) w = add22(w, red[k]);
    t = __dadd_rn((double)w.x, (double)w.y);
  }
  return t;
}

// Fixed-shape CTA sum in binary64: the result (valid in thread 0) depends only
// on the inputs, never on timing.
__device__ __forceinline__ double block_sum(double x, double* red) {
  __syncthreads();
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) x = __dadd_rn(x, __shfl_down_sync(0xffffffffu, x, off));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = x;
  __syncthreads();
  double t = 0.0;
  if (threadIdx.x == 0) {
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) t = __dadd_rn(t, red[w]);
  }
  return t;
}

// ------------------------------------------------------------- decisions (a4)
// The decision itself is decide_core (decide_core.h); here are the device
// parts around it: the scalar CTA's early computation of the next step's
// update scalars, and the last CTA's call with the folded statistics.

// Run by thread 0 of pass 1's scalar CTA while the other CTAs stream: the
// scalars of the step that follows the current one (t + 1; the step counter
// only changes in the decision at the end of this launch), so that the
// decision, which waits for every CTA, does no binary64 pow.  The host
// supplies them for the step numbers it expects (cand): when t + 1 is one of
// them they are taken as they are, with no table load and no binary64
// division; otherwise they are computed here from the bias-correction table
// (or pow past its end).  The host computes them with the same operations
// from the same table entries, so either way the values are identical.
// 1 / (scale * divisor): for a power-of-two scale 2^e it is (1 / divisor)
// * 2^-e, and scaling by a power of two is exact, so the host's rounded
// 1 / divisor scaled by 2^-e is the correctly rounded quotient itself.
static __device__ __noinline__ void precompute_scalars(const Pass1Args& a) {
  PreScalars p;
  const RankState st = a.ranks[a.rank];
  p.t = st.t + 1;
  const int64_t j = a.cand_t0 - p.t;
  if (j >= 0 && j < a.ncand) {
    p.step_size = a.cand[j][0];
    p.isb2 = a.cand[j][1];
    p.decay = a.cand[j][2];
  } else if (a.bc_table && p.t <= kBcSteps) {
    const double* bc = a.bc_table + 2 * (p.t - 1);
    step_scalars_bc(a.hp, p.t, bc[0], bc[1], &p.step_size, &p.isb2, &p.decay);
  } else {
    step_scalars(a.hp, p.t, &p.step_size, &p.isb2, &p.decay);
  }
  p.pad_ = 0;
  const uint32_t sb = __float_as_uint(st.scale);
  const uint32_t ex = (sb >> 23) & 0xffu;
  if ((sb & 0x807fffffu) == 0u && ex != 0u && ex != 0xffu)
    p.inv = scalbn(a.inv_d, 127 - (int)ex);   // scale = 2^(ex - 127)
  else
    p.inv = 1.0 / ((double)st.scale * a.hp.divisor);
  a.ws->pre = p;
}

// Bias-correction table of a handle: entry t - 1 holds 1 - beta1^t and
// 1 - beta2^t, exactly as the decision computes them.
struct BcTableArgs {
  double* table;
  double beta1, beta2;
};
static __global__ void __launch_bounds__(kThreads) bc_table_kernel(const BcTableArgs a) {
  const int64_t i = blockIdx.x * (int64_t)kThreads + threadIdx.x;
  if (i >= kBcSteps) return;
  a.table[2 * i] = bias_correction(a.beta1, i + 1);
  a.table[2 * i + 1] = bias_correction(a.beta2, i + 1);
}

// True for the CTA that streams nothing (the last one, when scalar_cta is set).
__device__ __forceinline__ bool is_scalar_cta(const Pass1Args& a) {
  return a.scalar_cta && blockIdx.x == gridDim.x - 1;
}

// Run by one thread of the last CTA of pass 1.  A statistics-only pass just
// publishes its statistics (after a fault: an overflow, so that every rank
// that folds them skips).  A fault skips the step and leaves the scaler state
// alone.  Otherwise the rank's scaler replica advances through decide_core.
// The decision's inputs from memory: the fault flag, the rank's scaler state
// and the scalar CTA's precomputed scalars.  The last CTA's thread 0 loads
// them (from L2: they were written by other CTAs of this launch or by the
// previous one) before it folds the partials, so that their latency overlaps
// the fold instead of following it.
struct DecideInputs {
  RankState st;
  PreScalars pre;
  int32_t fault;
};
template <typename T>
__device__ __forceinline__ T ldcg_struct(const T* p) {
  static_assert(sizeof(T) % 8 == 0 && alignof(T) >= 8, "8-byte words");
  T v;
  const long long* src = reinterpret_cast<const long long*>(p);
  long long* dst = reinterpret_cast<long long*>(&v);
#pragma unroll
  for (int i = 0; i < (int)(sizeof(T) / 8); ++i) dst[i] = __ldcg(src + i);
  return v;
}
__device__ __forceinline__ DecideInputs load_decide_inputs(const Pass1Args& a) {
  DecideInputs in;
  in.fault = __ldcg(&a.ws->fault);
  in.st = ldcg_struct(a.ranks + a.rank);
  in.pre = ldcg_struct(&a.ws->pre);
  return in;
}

static __device__ __forceinline__ void decide(const Pass1Args& a, double own_sumsq, int own_flag,
                                           const DecideInputs in) {
  Workspace* ws = a.ws;
  ws->ticket = 0u;
  const int fault = in.fault;
  ws->fault = 0;
  if (a.mode == kStatsOnly) {
    ws->own_sumsq = fault ? quiet_nan() : own_sumsq;
    ws->own_nonfinite = fault ? 1 : own_flag;
    if (a.stats_out) {
      a.stats_out->sumsq = ws->own_sumsq;
      a.stats_out->nonfinite = ws->own_nonfinite;
      a.stats_out->reserved = 0;
    }
    return;
  }
  if (fault) {
    ws->dec = fault_decision(in.st);
    return;
  }
  double sumsq = a.mode == kStepGlobal ? a.g_sumsq : own_sumsq;
  int nonfinite = a.mode == kStepGlobal ? a.g_nonfinite : own_flag;
  if (a.mode == kStepGlobalDev) {
    // the scalar all-reduce, folded here in rank order exactly as
    // zero_opt_fold_stats folds it on the host
    sumsq = 0.0;
    nonfinite = 0;
    for (int r = 0; r < a.g_n; ++r) {
      sumsq = __dadd_rn(sumsq, a.g_dev[r].sumsq);
      if (a.g_dev[r].nonfinite) nonfinite = 1;
    }
  }
  RankState st = in.st;
  // every stepping launch has a scalar CTA, which stored the scalars of step
  // t + 1 before this CTA could take the last ticket
  const PreScalars& pre = in.pre;
  const double inv = pre.inv;
  const Decision d = decide_core(a.hp, st, sumsq, nonfinite,
                                 [&pre](int64_t, float* ss, float* isb2, float* decay) {
                                   *ss = pre.step_size;
                                   *isb2 = pre.isb2;
                                   *decay = pre.decay;
                                 },
                                 &inv);
  a.ranks[a.rank] = st;
  ws->dec = d;
}

// ------------------------------------------------------------- pass 1
// The ticket of the last-CTA fold.  Every write another CTA needs (its
// partial and flag, the scalar CTA's precomputed scalars, a fault flag) is
// made by the CTA's thread 0 before it takes the ticket, and the atomic
// increment has release and acquire semantics at GPU scope: the CTA that
// draws the last ticket synchronizes with every earlier increment (they form
// one release sequence), and its barrier then orders its other threads'
// loads after all of those writes.
__device__ __forceinline__ unsigned int ticket_add_acq_rel(unsigned int* p) {
  unsigned int old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(old) : "l"(p) : "memory");
  return old;
}

// Grids of up to this many CTAs have their partials folded by one warp (four
// per lane).
constexpr int kFoldWarpMax = 128;

// The epilogue shared by both pass-1 kernels: one binary64 partial and one
// overflow flag per CTA; the CTA that finishes last folds them in a fixed
// order and takes the decisions.
__device__ __forceinline__ void pass1_finish(const Pass1Args& a, const SqAcc& acc, int flag,
                                             double* red, int* s_last) {
  const int tid = threadIdx.x;
  // the CTA's partial: in binary32 pairs unless a thread holds binary64 sums
  // (values outside the range whose squares binary32 holds exactly)
  // (an integer test: slow is a sum of non-negative terms, never -0, and a
  // binary64 comparison would hold GB300's slow binary64 pipe on every warp)
  const int slow = __syncthreads_or(__double_as_longlong(acc.slow) != 0ll);
  const double blk = slow ? block_sum(acc.total(), red)
                          : block_sum_ff(acc.total_ff(), reinterpret_cast<float2*>(red));
  const int any = __syncthreads_or(flag);
  if (tid == 0) {
    a.ws->part_sumsq[blockIdx.x] = blk;
    a.ws->part_flag[blockIdx.x] = any;
    const unsigned int prev = ticket_add_acq_rel(&a.ws->ticket);
    *s_last = (prev == gridDim.x - 1) ? 1 : 0;
  }
  __syncthreads();
  if (!*s_last) return;
  DecideInputs in;
  if (tid == 0) in = load_decide_inputs(a);
  if (gridDim.x <= kFoldWarpMax) {
    // At most 128 partials (small shards): warp 0 folds them alone, with no
    // CTA barrier on the path to the decision.  Lane l adds the partials l,
    // l + 32, l + 64 and l + 96 in that order (all four loads issued first;
    // past the grid: +0), then the lanes are added pairwise, halving.  Saves
    // about 0.5 us per step on shards up to ~1M parameters.
    if (tid >= 32) return;
    double v[kFoldWarpMax / 32];
    int fl[kFoldWarpMax / 32];
#pragma unroll
    for (int q = 0; q < kFoldWarpMax / 32; ++q) {
      const int c = q * 32 + tid;
      v[q] = c < (int)gridDim.x ? __ldcg(&a.ws->part_sumsq[c]) : 0.0;
      fl[q] = c < (int)gridDim.x ? __ldcg(&a.ws->part_flag[c]) : 0;
    }
    double part = 0.0;
    int f = 0;
#pragma unroll
    for (int q = 0; q < kFoldWarpMax / 32; ++q) {
      part = __dadd_rn(part, v[q]);
      f |= fl[q];
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
      part = __dadd_rn(part, __shfl_down_sync(0xffffffffu, part, off));
    f = __any_sync(0xffffffffu, f);
    if (tid == 0) decide(a, part, f, in);
    return;
  }
  // each thread folds the partials c = tid, tid + 256, ... in that order; the
  // loads of four are issued before any is added (past the grid: +0, which
  // leaves the sum unchanged)
  double part = 0.0;
  int f = 0;
  for (int c0 = 0; c0 < (int)gridDim.x; c0 += 4 * kThreads) {
    double v[4];
    int fl[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int c = c0 + k * kThreads + tid;
      v[k] = c < (int)gridDim.x ? __ldcg(&a.ws->part_sumsq[c]) : 0.0;
      fl[k] = c < (int)gridDim.x ? __ldcg(&a.ws->part_flag[c]) : 0;
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      part = __dadd_rn(part, v[k]);
      f |= fl[k];
    }
  }
  const double tot = block_sum(part, red);
  const int anyf = __syncthreads_or(f);
  if (tid == 0) decide(a, tot, anyf, in);
}

// One tile element by element: a ragged tail of a vector run (e >= e0 within
// the thread's 8 elements) or any tile of a run with a misaligned pointer
// (elements base + i*256 + tid, coalesced).  Returns the thread's 8 sums (0
// past the end) by value, so that callers keep their accumulators in
// registers; kept out of line because it is rare.
struct Sums8 {
  float v[kVec];
};

template <typename GT, bool STASH>
__device__ __noinline__ Sums8 pass1_elementwise_sums(const Pass1Args& a, int64_t n,
                                                     int64_t stash_off, int32_t gbase,
                                                     int32_t vec, int64_t base) {
  const int tid = threadIdx.x;
  const int64_t e0 = base + tid * kVec;
  Sums8 x;
#pragma unroll
  for (int i = 0; i < kVec; ++i) {
    const int64_t e = vec ? e0 + i : base + (int64_t)i * kThreads + tid;
    float sum = 0.0f;
    if (e < n) {
      for (int b = 0; b < a.nbuf; ++b) {
        const unsigned long long raw =
            __ldg(reinterpret_cast<const unsigned long long*>(a.gptrs) + gbase + b);
        sum = __fadd_rn(sum, Fmt<GT>::dec(__ldcg(reinterpret_cast<const unsigned short*>(raw) + e)));
      }
      if (STASH) a.stash[stash_off + e] = sum;
    }
    x.v[i] = sum;
  }
  return x;
}

// ------------------------------------------------------------- bulk copies
// Thin wrappers of the PTX for Blackwell's asynchronous bulk copies (TMA) and
// shared-memory transaction barriers.
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(unsigned long long* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}
__device__ __forceinline__ void mbar_init_fence() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
// Arrive (the one expected arrival) and expect `bytes` of asynchronous copies.
__device__ __forceinline__ void mbar_arrive_expect_tx(unsigned long long* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(unsigned long long* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}
// Global -> shared copy of `bytes` (multiple of 16, both addresses 16-byte
// aligned) that completes its bytes on `bar`.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          unsigned long long* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}
// The same copy with an L2 evict_last policy on the lines it reads.
__device__ __forceinline__ void bulk_load_keep(void* dst, const void* src, uint32_t bytes,
                                               unsigned long long* bar) {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(pol)
      : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(unsigned long long* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Wait for the phase of `bar` with the given parity, giving up after about a
// second (returns false then).  No wait in this library is unbounded.
__device__ __forceinline__ bool mbar_wait_bounded(unsigned long long* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_ns() - t0 > 1000000000ull) return false;
  }
  return true;
}

#ifndef ZO_BULK_STAGES
#define ZO_BULK_STAGES 2
#endif

// Bytes of dynamic shared memory pass1_bulk_kernel<GT, CT> needs.
constexpr int bulk_smem_bytes(int chunk_tiles) {
  return ZO_BULK_STAGES * chunk_tiles * kThreads * 16;
}
// Resident CTAs per SM each chunk size is compiled for.
constexpr int bulk_min_ctas(int chunk_tiles) { return chunk_tiles >= 8 ? 3 : ZO_PASS1_MIN_CTAS; }

// Single gradient buffer, staged through shared memory by bulk copies.  The
// work unit is a chunk of CT consecutive tiles (each thread reduces 8*CT
// elements per chunk, in two independent TwoSum chains that take the tiles
// in turn); thread 0 keeps ZO_BULK_STAGES chunks in flight per CTA
// with one cp.async.bulk of CT * 4 KiB each, so the reducing threads read
// shared memory instead of waiting on global loads.  Chunks of 4 tiles at 4
// CTAs per SM balance short shards best; chunks of 8 tiles at 3 CTAs per SM
// move more per copy on long ones.  A chunk that is not CT full tiles of one
// 16-byte aligned run is not copied: its barrier phase is completed by a
// plain arrival and its tiles are reduced from global memory.  If a wait
// expires the CTA stops issuing, waits (bounded) for the copies in flight and
// records a fault, which makes the step a no-op.
template <typename GT, int CT>
__global__ void __launch_bounds__(kThreads, bulk_min_ctas(CT))
    pass1_bulk_kernel(const Pass1Args a) {
  pass1_prologue();
  constexpr int S = ZO_BULK_STAGES;
  constexpr int kChunkTiles = CT;
  extern __shared__ __align__(128) uint4 stage_buf[];  // [S][CT][kThreads]
  __shared__ __align__(8) unsigned long long bar[S];
  __shared__ int s_whole[S];  // 1: the stage holds its chunk (copied whole)
  __shared__ double red[kThreads / 32];
  __shared__ int s_last, s_err;
  const int tid = threadIdx.x;
  const int64_t G = gridDim.x - a.scalar_cta;
  const int64_t nchunks = (a.ntiles + kChunkTiles - 1) / kChunkTiles;
  const int64_t mine = (int64_t)blockIdx.x < G && nchunks > (int64_t)blockIdx.x
                           ? (nchunks - 1 - blockIdx.x) / G + 1
                           : 0;
  // Thread 0 looks each chunk up (a fresh cursor, so no run state stays live
  // across the loop) and tells the others through s_whole whether the chunk
  // was copied: it is when its tiles are full tiles of one vector run.
  auto issue = [&](int64_t i) {
    const int64_t t0 = (blockIdx.x + i * G) * kChunkTiles;
    unsigned long long* b = &bar[i % S];
    if (a.inject_wait_fault && blockIdx.x == 0 && i == 0) return;  // test hook
    RunCursorLite c;
    c.seek(a.segs, a.nseg, t0);
    const bool whole = c.s.vec && t0 + kChunkTiles <= c.end &&
                       (t0 + kChunkTiles - c.s.tile0) * kTile <= c.s.n;
    s_whole[i % S] = whole ? 1 : 0;
    if (whole) {
      mbar_arrive_expect_tx(b, kChunkTiles * kTile * 2);
      if (t0 >= a.keep_tile0)
        bulk_load_keep(&stage_buf[(i % S) * kChunkTiles * kThreads],
                       grad_ptr(a.gptrs, c.s, 0) + (t0 - c.s.tile0) * kTile,
                       kChunkTiles * kTile * 2, b);
      else
        bulk_load(&stage_buf[(i % S) * kChunkTiles * kThreads],
                  grad_ptr(a.gptrs, c.s, 0) + (t0 - c.s.tile0) * kTile,
                  kChunkTiles * kTile * 2, b);
    } else {
      mbar_arrive(b);
    }
  };
  if (tid == 0) {
    for (int k = 0; k < S; ++k) mbar_init(&bar[k], 1);
    mbar_init_fence();
    s_err = 0;
    if (is_scalar_cta(a)) precompute_scalars(a);
  }
  __syncthreads();
  if (tid == 0)
    for (int64_t i = 0; i < mine && i < S; ++i) issue(i);
  SqAcc acc;
  int64_t issued = mine < S ? mine : S;
  for (int64_t i = 0; i < mine; ++i) {
    if (!mbar_wait_bounded(&bar[i % S], (uint32_t)((i / S) & 1))) s_err = 1;
    const int64_t t0 = (blockIdx.x + i * G) * kChunkTiles;
    if (!s_err) {
      if (*reinterpret_cast<volatile int*>(&s_whole[i % S])) {
        const uint4* sb = &stage_buf[(i % S) * kChunkTiles * kThreads + tid];
        // tiles in pairs, into two accumulator chains (CT is even)
#pragma unroll
        for (int k = 0; k < kChunkTiles; k += 2)
          acc.add_raw16_2<GT>(sb[k * kThreads], sb[(k + 1) * kThreads]);
      } else {
        RunCursorLite cur;
        for (int k = 0; k < kChunkTiles; ++k) {
          const int64_t tile = t0 + k;
          if (tile >= a.ntiles) break;
          cur.seek(a.segs, a.nseg, tile);
          const int64_t base = (tile - cur.s.tile0) * kTile;
          // per thread, as in pass 2: a thread whose eight elements are all
          // in the run loads them with one 16-byte access (the accumulation
          // of their raw 16-bit values is bit-identical to the element-wise
          // one), a thread past the end adds nothing (its sums would be +0),
          // and only a thread that straddles the end goes element by element
          const int64_t e0 = base + tid * kVec;
          if (cur.s.vec && e0 + kVec <= cur.s.n) {
            acc.add_raw16<GT>(__ldcg(reinterpret_cast<const uint4*>(
                grad_ptr(a.gptrs, cur.s, 0) + e0)));
          } else if (cur.s.vec && e0 >= cur.s.n) {
            // nothing in range
          } else {
            const Sums8 x = pass1_elementwise_sums<GT, false>(a, cur.s.n, cur.s.stash_off,
                                                              cur.s.gbase, cur.s.vec, base);
            acc.add<false>(x.v);
          }
        }
      }
    }
    __syncthreads();  // every thread is done with stage i % S
    if (s_err) {
      // wait for the copies still in flight before the shared memory goes away
      if (tid == 0) {
        for (int64_t j = i; j < issued; ++j)
          (void)mbar_wait_bounded(&bar[j % S], (uint32_t)((j / S) & 1));
        atomicExch(&a.ws->fault, 1);
      }
      break;
    }
    if (tid == 0 && issued < mine) {
      issue(issued);
      ++issued;
    }
  }
  pass1_finish(a, acc, acc.overflowed<GT>() ? 1 : 0, red, &s_last);
}

// Any number of gradient buffers, loaded in batches of eight per tile, summed
// in buffer order; optionally stores the sums (the stash).
template <typename GT, bool STASH>
__global__ void __launch_bounds__(kThreads, ZO_MULTI_MIN_CTAS)
    pass1_multi_kernel(const Pass1Args a) {
  pass1_prologue();
  __shared__ double red[kThreads / 32];
  __shared__ int s_last;
  const int tid = threadIdx.x;
  const int64_t G = gridDim.x - a.scalar_cta;
  if (is_scalar_cta(a) && tid == 0) precompute_scalars(a);
  SqAcc acc;
  RunCursorLite cur;
  for (int64_t tile = blockIdx.x; tile < a.ntiles && blockIdx.x < G; tile += G) {
    cur.seek(a.segs, a.nseg, tile);
    const auto& s = cur.s;
    const int64_t base = (tile - s.tile0) * kTile;
    const int64_t e0 = base + tid * kVec;
    if (!(s.vec && e0 + kVec <= s.n)) {
      const Sums8 x = pass1_elementwise_sums<GT, STASH>(a, s.n, s.stash_off, s.gbase, s.vec, base);
      acc.add<false>(x.v);
      continue;
    }
    float x[kVec];
#pragma unroll
    for (int i = 0; i < kVec; ++i) x[i] = 0.0f;
    for (int b0 = 0; b0 < a.nbuf; b0 += 8) {
      uint4 r[8];
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (b0 + j < a.nbuf)
          r[j] = __ldcg(reinterpret_cast<const uint4*>(grad_ptr(a.gptrs, s, b0 + j) + e0));
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (b0 + j < a.nbuf) {
          float y[kVec];
          Fmt<GT>::dec8(r[j], y);
#pragma unroll
          for (int i = 0; i < kVec; ++i) x[i] = __fadd_rn(x[i], y[i]);
        }
      }
    }
    if (STASH) {
      float* dst = a.stash + s.stash_off + e0;
      reinterpret_cast<float4*>(dst)[0] = make_float4(x[0], x[1], x[2], x[3]);
      reinterpret_cast<float4*>(dst)[1] = make_float4(x[4], x[5], x[6], x[7]);
    }
    acc.add<false>(x);
  }
  pass1_finish(a, acc, acc.overflowed<GT>() ? 1 : 0, red, &s_last);
}

// ------------------------------------------------------------- pass 2
struct Scalars {
  float coef, b1, omb1, b2, omb2, isb2, eps, decay, step_size;
};

// a5..a6 for one element: the exact binary32 operation sequence of the step.
__device__ __forceinline__ void adam_elem(float sj, float& p, float& m, float& v,
                                          const Scalars& c) {
  const float g = __fmul_rn(sj, c.coef);
  m = __fadd_rn(__fmul_rn(c.b1, m), __fmul_rn(c.omb1, g));
  v = __fadd_rn(__fmul_rn(c.b2, v), __fmul_rn(c.omb2, __fmul_rn(g, g)));
  const float den = __fadd_rn(__fmul_rn(__fsqrt_rn(v), c.isb2), c.eps);
  p = __fmul_rn(p, c.decay);
  p = __fsub_rn(p, __fmul_rn(c.step_size, __fdiv_rn(m, den)));
}

// Eight floats at a 32-byte aligned address, as one 256-bit access with the
// streaming cache hint.
__device__ __forceinline__ void ld8cs(const float* p, float* d) {
  asm volatile("ld.global.cs.v8.f32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3]), "=f"(d[4]), "=f"(d[5]),
                 "=f"(d[6]), "=f"(d[7])
               : "l"(p));
}
__device__ __forceinline__ void st8cs(float* p, const float* d) {
  asm volatile("st.global.cs.v8.f32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "f"(d[0]),
               "f"(d[1]), "f"(d[2]), "f"(d[3]), "f"(d[4]), "f"(d[5]), "f"(d[6]), "f"(d[7])
               : "memory");
}

__device__ __forceinline__ void f4_to(const float4& a, float* d) {
  d[0] = a.x; d[1] = a.y; d[2] = a.z; d[3] = a.w;
}

// SRC == 1: one gradient buffer; SRC == 0: a.nbuf buffers; SRC == -1: stash.
// M16: low-precision master weights -- there is no fp32 master array; the
// 16-bit parameter is widened, updated and stored back rounded.
template <typename GT, typename PT, int SRC, bool M16>
__global__ void __launch_bounds__(kThreads, (M16 && SRC != 0) ? ZO_PASS2_M16_MIN_CTAS
                                                               : ZO_PASS2_MIN_CTAS)
    pass2_kernel(const Pass2Args a) {
#if ZO_PDL_PASS1
  pdl_launch_dependents();  // the next step's pass 1 may be scheduled
#endif
  const int64_t G0 = gridDim.x;
  if (threadIdx.x == 0 && (int64_t)blockIdx.x < a.ntiles) {
    // Before the wait this overlaps the end of pass 1, so only data pass 1
    // never writes is touched: warm L2 with the state (and a single gradient
    // buffer) of this CTA's first tile, when it is a full 16-byte aligned one.
    const int64_t first = blockIdx.x + (a.ntiles - 1 - blockIdx.x) / G0 * G0;
    RunCursor c;
    c.seek(a.segs, a.nseg, first);
    const int64_t base = (first - c.s.tile0) * kTile;
    if (c.s.vec && base + kTile <= c.s.n) {
      if (!M16) prefetch_l2(c.s.master + base, kTile * 4);
      prefetch_l2(c.s.m + base, kTile * 4);
      prefetch_l2(c.s.v + base, kTile * 4);
      if (M16) prefetch_l2(static_cast<const unsigned short*>(c.s.p16) + base, kTile * 2);
      if (SRC == 1) prefetch_l2(grad_ptr(a.gptrs, c.s, 0) + base, kTile * 2);
    }
  }
  pdl_wait();
  // The decision, the first tile's run and the first tile's data are loaded
  // together: nothing of a tile depends on the decision, so the skip test
  // waits until those loads are in flight (on a skipped step their values are
  // dropped and nothing is stored).  Three dependent L2 round trips become
  // one on the path from pass 1's decision to pass 2's first update.
  const Decision* dp = a.dec;
  const int skip = dp->skip;
  Scalars c;
  c.coef = dp->coef;
  c.b1 = dp->b1;
  c.omb1 = dp->omb1;
  c.b2 = dp->b2;
  c.omb2 = dp->omb2;
  c.isb2 = dp->isb2;
  c.eps = dp->eps;
  c.decay = dp->decay;
  c.step_size = dp->step_size;
  const int tid = threadIdx.x;
  const int64_t G = gridDim.x;
  const int64_t cnt = (int64_t)blockIdx.x < a.ntiles ? (a.ntiles - 1 - blockIdx.x) / G + 1 : 0;
  RunCursor cur;
  for (int64_t k = cnt - 1; k >= 0; --k) {
    const int64_t tile = blockIdx.x + k * G;
    cur.seek(a.segs, a.nseg, tile);
    const Seg& s = cur.s;
    const int64_t base = (tile - s.tile0) * kTile;
    const int64_t e0 = base + tid * kVec;
    if (s.vec && e0 + kVec <= s.n) {
      float x[kVec], p[kVec], m[kVec], v[kVec];
      const unsigned short* gp = nullptr;
      uint4 graw = make_uint4(0u, 0u, 0u, 0u);
      if (SRC == -1) {
        // one 256-bit load per lane when the run's stash is 32-byte aligned
        // (two 128-bit loads at a 32-byte lane stride touch every sector
        // twice); fused reduction, 250M parameters: 1.146 -> 1.116 ms
        if (((uintptr_t)(a.stash + s.stash_off) & 31) == 0) {
          ld8cs(a.stash + s.stash_off + e0, x);
        } else {
          const float4* st = reinterpret_cast<const float4*>(a.stash + s.stash_off + e0);
          f4_to(__ldcs(st), x);
          f4_to(__ldcs(st + 1), x + 4);
        }
      } else if (SRC == 1) {
        gp = grad_ptr(a.gptrs, s, 0) + e0;
        graw = __ldcs(reinterpret_cast<const uint4*>(gp));   // decoded below
      } else {
#pragma unroll
        for (int i = 0; i < kVec; ++i) x[i] = 0.0f;
        for (int b0 = 0; b0 < a.nbuf; b0 += 8) {
          uint4 r[8];
#pragma unroll
          for (int j = 0; j < 8; ++j)
            if (b0 + j < a.nbuf)
              r[j] = __ldcs(reinterpret_cast<const uint4*>(grad_ptr(a.gptrs, s, b0 + j) + e0));
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            if (b0 + j < a.nbuf) {
              float y[kVec];
              Fmt<GT>::dec8(r[j], y);
#pragma unroll
              for (int i = 0; i < kVec; ++i) x[i] = __fadd_rn(x[i], y[i]);
            }
          }
        }
      }
      unsigned short* p16 = static_cast<unsigned short*>(s.p16) + e0;
      // 256-bit accesses to the fp32 state when its arrays are 32-byte aligned
      // at this tile (a property of the run, the same for every thread)
      const bool w8 = ((((uintptr_t)(s.m + e0)) | ((uintptr_t)(s.v + e0)) |
                        (M16 ? (uintptr_t)0 : (uintptr_t)(s.master + e0))) &
                       31) == 0;
      if (M16) {
        Fmt<PT>::dec8(__ldcs(reinterpret_cast<const uint4*>(p16)), p);
      } else if (w8) {
        ld8cs(s.master + e0, p);
      } else {
        const float4* pm = reinterpret_cast<const float4*>(s.master + e0);
        f4_to(__ldcs(pm), p);
        f4_to(__ldcs(pm + 1), p + 4);
      }
      if (w8) {
        ld8cs(s.m + e0, m);
        ld8cs(s.v + e0, v);
      } else {
        const float4* mm = reinterpret_cast<const float4*>(s.m + e0);
        const float4* vm = reinterpret_cast<const float4*>(s.v + e0);
        f4_to(__ldcs(mm), m);
        f4_to(__ldcs(mm + 1), m + 4);
        f4_to(__ldcs(vm), v);
        f4_to(__ldcs(vm + 1), v + 4);
      }
      // every load of the tile is issued above this point; the decision is
      // used below it
      asm volatile("" ::: "memory");
      if (skip) break;
      if (SRC == 1) {
        Fmt<GT>::dec8(graw, x);
        if (tile >= a.keep_tile0 && (tid & 7) == 0) l2_normal(gp);
#pragma unroll
        for (int i = 0; i < kVec; ++i) x[i] = __fadd_rn(0.0f, x[i]);
      }
#pragma unroll
      for (int i = 0; i < kVec; ++i) adam_elem(x[i], p[i], m[i], v[i], c);
      if (w8) {
        if (!M16) st8cs(s.master + e0, p);
        st8cs(s.m + e0, m);
        st8cs(s.v + e0, v);
      } else {
        if (!M16) {
          float4* po = reinterpret_cast<float4*>(s.master + e0);
          __stcs(po, make_float4(p[0], p[1], p[2], p[3]));
          __stcs(po + 1, make_float4(p[4], p[5], p[6], p[7]));
        }
        float4* mo = reinterpret_cast<float4*>(s.m + e0);
        float4* vo = reinterpret_cast<float4*>(s.v + e0);
        __stcs(mo, make_float4(m[0], m[1], m[2], m[3]));
        __stcs(mo + 1, make_float4(m[4], m[5], m[6], m[7]));
        __stcs(vo, make_float4(v[0], v[1], v[2], v[3]));
        __stcs(vo + 1, make_float4(v[4], v[5], v[6], v[7]));
      }
      __stcs(reinterpret_cast<uint4*>(p16), Fmt<PT>::enc8(p));
    } else {
      if (skip) break;
#pragma unroll
      for (int i = 0; i < kVec; ++i) {
        const int64_t e = s.vec ? e0 + i : base + (int64_t)i * kThreads + tid;
        if (e >= s.n) continue;
        float x;
        if (SRC == -1) {
          x = __ldcs(a.stash + s.stash_off + e);
        } else {
          x = 0.0f;
          for (int b = 0; b < a.nbuf; ++b)
            x = __fadd_rn(x, Fmt<GT>::dec(__ldcs(grad_ptr(a.gptrs, s, b) + e)));
        }
        unsigned short* p16 = static_cast<unsigned short*>(s.p16) + e;
        float p = M16 ? Fmt<PT>::dec(*p16) : __ldcs(s.master + e);
        float m = __ldcs(s.m + e), v = __ldcs(s.v + e);
        adam_elem(x, p, m, v, c);
        if (!M16) __stcs(s.master + e, p);
        __stcs(s.m + e, m);
        __stcs(s.v + e, v);
        *p16 = Fmt<PT>::enc(p);
      }
    }
  }
  if (skip) {
    // nothing was updated; the gradient lines pass 1 kept in L2 go back to
    // evict_normal all the same (one lane per 128-byte line)
    if (SRC == 1 && a.keep_tile0 < a.ntiles && (tid & 7) == 0) {
      RunCursor kc;
      for (int64_t tile = a.keep_tile0 + blockIdx.x; tile < a.ntiles; tile += G) {
        kc.seek(a.segs, a.nseg, tile);
        const int64_t e0 = (tile - kc.s.tile0) * kTile + tid * kVec;
        if (kc.s.vec && e0 + kVec <= kc.s.n) l2_normal(grad_ptr(a.gptrs, kc.s, 0) + e0);
      }
    }
  }
}

// ------------------------------------------------------------- 16-bit copy
// Rewrite a 16-bit parameter slice as the rounding of fp32 master weights
// (when a shard is restored from a checkpoint).
struct CastArgs {
  const float* master;
  unsigned short* p16;
  int64_t n;
};

template <typename PT>
__global__ void __launch_bounds__(kThreads) cast_kernel(const CastArgs a) {
  for (int64_t i = blockIdx.x * (int64_t)kThreads + threadIdx.x; i < a.n;
       i += (int64_t)gridDim.x * kThreads)
    a.p16[i] = Fmt<PT>::enc(a.master[i]);
}

}  // namespace zo
