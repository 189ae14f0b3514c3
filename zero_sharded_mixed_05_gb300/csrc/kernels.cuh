// kernels.cuh -- sm_103a kernels of the per-shard mixed-precision ZeRO step.
//
// pass1_single_kernel / pass1_multi_kernel (steps a1..a4): each CTA walks its
//   tiles of the shard, sums the R*K 16-bit gradient buffers per element in
//   binary32 (rank-major order, starting from +0; one buffer or many),
//   optionally stores the sums (the stash), and accumulates
//   the overflow flag and the sum of squares.  CTAs publish one partial each;
//   the CTA that finishes last (atomic ticket, no waiting) folds the partials
//   in CTA order in binary64, takes the per-step decisions (skip, clip
//   coefficient, Adam scalars) and advances the rank's loss-scaler state.
// pass2_kernel (steps a5..a7): reads the decision; on a skip every CTA returns
//   at once; otherwise it applies unscale x clip, AdamW on the fp32 master
//   copy and m, v, and writes the 16-bit parameter copy.
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

#include "zero_opt_internal.h"

// Resident CTAs per SM each kernel is compiled for (register budget 65536 /
// (256 * n) per thread).
#ifndef ZO_PASS1_MIN_CTAS
#define ZO_PASS1_MIN_CTAS 4
#endif
#ifndef ZO_PASS2_MIN_CTAS
#define ZO_PASS2_MIN_CTAS 2
#endif
// Tiles whose 16-byte gradient loads pass 1 issues before reducing any of
// them, when there is a single gradient buffer.
#ifndef ZO_PASS1_UNROLL
#define ZO_PASS1_UNROLL 4
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

// ------------------------------------------------------------- sum of squares
// The global norm needs the sum of squares of the reduced gradients to well
// below binary32 precision (the clip coefficient is rounded to binary32 from
// it), but GB300's binary64 rate is far too low for a binary64 operation per
// element.  Each square is therefore formed exactly as p + e (p = s*s rounded,
// e = fma(s, s, -p)) and added into a per-thread double-binary32 accumulator
// (hi, lo) with Knuth's TwoSum; even and odd elements go to two independent
// accumulators so consecutive additions do not wait on each other.  The
// thread's total hi + lo is taken in binary64; the accumulated error is a few
// units of 2^-48 of the thread's sum.  Every operation is an explicit IEEE
// round-to-nearest intrinsic, so nothing is contracted.  Tiles whose largest
// |s| is 2^50 or more (squares near the binary32 overflow range, or inf/NaN),
// or whose values are all nonzero and below 2^-40 (squares near underflow),
// are summed in binary64 instead.  amax (the largest |s| bit pattern seen)
// gives the overflow flag: inf and NaN patterns are >= 0x7f800000.
struct SqAcc {
  float hi0 = 0.0f, lo0 = 0.0f, hi1 = 0.0f, lo1 = 0.0f;
  double slow = 0.0;
  uint32_t amax = 0u;

  static __device__ __forceinline__ void two_sum_add(float& hi, float& lo, float x) {
    const float p = __fmul_rn(x, x);
    const float e = __fmaf_rn(x, x, -p);
    const float t = __fadd_rn(hi, p);
    const float bp = __fsub_rn(t, hi);
    const float ap = __fsub_rn(t, bp);
    const float err = __fadd_rn(__fsub_rn(hi, ap), __fsub_rn(p, bp));
    lo = __fadd_rn(lo, __fadd_rn(err, e));
    hi = t;
  }

  // Square known to be exact in binary32 (a 16-bit value in the fast range):
  // TwoSum only.
  static __device__ __forceinline__ void two_sum_add_exact(float& hi, float& lo, float x) {
    const float p = __fmul_rn(x, x);
    const float t = __fadd_rn(hi, p);
    const float bp = __fsub_rn(t, hi);
    const float ap = __fsub_rn(t, bp);
    lo = __fadd_rn(lo, __fadd_rn(__fsub_rn(hi, ap), __fsub_rn(p, bp)));
    hi = t;
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
        if (EXACT_SQ) {
          two_sum_add_exact(hi0, lo0, s[i]);
          two_sum_add_exact(hi1, lo1, s[i + 1]);
        } else {
          two_sum_add(hi0, lo0, s[i]);
          two_sum_add(hi1, lo1, s[i + 1]);
        }
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
        two_sum_add_exact(hi0, lo0, x.x);
        two_sum_add_exact(hi1, lo1, x.y);
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
  template <typename GT>
  __device__ __forceinline__ bool overflowed() const {
    return amax >= 0x7f800000u || amax16 >= Fmt<GT>::kInf;
  }

  __device__ __forceinline__ double total() const {
    const double a = __dadd_rn((double)hi0, (double)lo0);
    const double b = __dadd_rn((double)hi1, (double)lo1);
    return __dadd_rn(__dadd_rn(a, b), slow);
  }
};

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
// Run by one thread of the last CTA.  Scalars are computed in binary64 and
// rounded once to binary32.  Overflow: skip, clean count restarts, and on the
// hysteresis-th overflow since the scale last changed scale /= factor (not
// below min_scale).  The update's lr is lr, or WarmupLR's linear value.  Otherwise: norm of the unscaled gradient,
// clip coefficient min(1, max_norm / (norm + 1e-6)), Adam step t += 1 with its
// bias corrections, and the scale grows by the factor after `window`
// consecutive applied steps.
static __device__ void decide(const Pass1Args& a, double own_sumsq, int own_flag) {
  Workspace* ws = a.ws;
  ws->ticket = 0u;
  const int fault = ws->fault;
  ws->fault = 0;
  if (a.mode == kStatsOnly) {
    // after a fault the statistics are incomplete: report an overflow so that
    // every rank that folds them skips the step
    ws->own_sumsq = fault ? __longlong_as_double(0x7ff8000000000000ll) : own_sumsq;
    ws->own_nonfinite = fault ? 1 : own_flag;
    return;
  }
  if (fault) {
    // a bounded wait expired: skip without touching the scaler state
    Decision d;
    d.sumsq = d.norm = __longlong_as_double(0x7ff8000000000000ll);
    d.coef = d.scale_used = 0.0f;
    d.skip = 1;
    d.nonfinite = 0;
    d.t = a.ranks[a.rank].t;
    d.fault = 1;
    d.pad_ = 0;
    d.step_size = d.isb2 = d.decay = d.b1 = d.omb1 = d.b2 = d.omb2 = d.eps = 0.0f;
    d.scale_used = a.ranks[a.rank].scale;
    ws->dec = d;
    return;
  }
  const double sumsq = a.mode == kStepGlobal ? a.g_sumsq : own_sumsq;
  const int nonfinite = a.mode == kStepGlobal ? a.g_nonfinite : own_flag;
  RankState st = a.ranks[a.rank];
  Decision d;
  d.fault = 0;
  d.pad_ = 0;
  d.sumsq = sumsq;
  d.nonfinite = nonfinite;
  d.scale_used = st.scale;
  d.coef = 0.0f;
  d.step_size = d.isb2 = d.decay = d.b1 = d.omb1 = d.b2 = d.omb2 = d.eps = 0.0f;
  const float scale = st.scale;
  const double inv = 1.0 / ((double)scale * a.hp.divisor);
  if (nonfinite) {
    d.skip = 1;
    d.norm = __longlong_as_double(0x7ff8000000000000ll);
    if (a.hp.dynamic) {
      st.overflows += 1;
      if (st.overflows >= a.hp.hysteresis) {
        double lowered = (double)scale / a.hp.factor;
        if (lowered < a.hp.min_scale) lowered = a.hp.min_scale;
        st.scale = (float)lowered;
        st.overflows = 0;
      }
    }
    st.clean = 0;
    st.skipped_total += 1;
    st.last_skipped = 1;
  } else {
    const double norm = sqrt(sumsq) * inv;
    double clip = 1.0;
    if (a.hp.max_norm > 0.0) {
      clip = a.hp.max_norm / (norm + 1e-6);
      if (clip > 1.0) clip = 1.0;
    }
    d.skip = 0;
    d.norm = norm;
    d.coef = (float)(inv * clip);
    st.t += 1;
    double bc1 = 1.0, bc2 = 1.0;
    if (a.hp.bias_correction) {
      bc1 = 1.0 - pow(a.hp.beta1, (double)st.t);
      bc2 = 1.0 - pow(a.hp.beta2, (double)st.t);
    }
    double lr = a.hp.lr;
    if (a.hp.warmup_num_steps > 0) {
      const double T = (double)a.hp.warmup_num_steps;
      const double t = (double)st.t;
      const double frac = t < T ? t / T : 1.0;
      lr = a.hp.warmup_min_lr + (a.hp.warmup_max_lr - a.hp.warmup_min_lr) * frac;
    }
    d.step_size = (float)(lr / bc1);
    d.isb2 = (float)(1.0 / sqrt(bc2));
    d.decay = (float)(1.0 - lr * a.hp.wd);
    d.b1 = (float)a.hp.beta1;
    d.omb1 = (float)(1.0 - a.hp.beta1);
    d.b2 = (float)a.hp.beta2;
    d.omb2 = (float)(1.0 - a.hp.beta2);
    d.eps = (float)a.hp.eps;
    st.last_skipped = 0;
    st.clean += 1;
    if (a.hp.dynamic && st.clean == a.hp.window) {
      st.scale = (float)((double)scale * a.hp.factor);
      st.clean = 0;
      st.overflows = 0;
    }
  }
  d.t = st.t;
  a.ranks[a.rank] = st;
  ws->dec = d;
}

// ------------------------------------------------------------- pass 1
// The epilogue shared by both pass-1 kernels: one binary64 partial and one
// overflow flag per CTA; the CTA that finishes last folds them in CTA order
// and takes the decisions.
__device__ __forceinline__ void pass1_finish(const Pass1Args& a, double mine, int flag,
                                             double* red, int* s_last) {
  const int tid = threadIdx.x;
  const double blk = block_sum(mine, red);
  const int any = __syncthreads_or(flag);
  if (tid == 0) {
    a.ws->part_sumsq[blockIdx.x] = blk;
    a.ws->part_flag[blockIdx.x] = any;
    __threadfence();
    const unsigned int prev = atomicAdd(&a.ws->ticket, 1u);
    *s_last = (prev == gridDim.x - 1) ? 1 : 0;
  }
  __syncthreads();
  if (!*s_last) return;
  __threadfence();
  double part = 0.0;
  int f = 0;
  for (int c = tid; c < (int)gridDim.x; c += kThreads) {
    part = __dadd_rn(part, __ldcg(&a.ws->part_sumsq[c]));
    f |= __ldcg(&a.ws->part_flag[c]);
  }
  const double tot = block_sum(part, red);
  const int anyf = __syncthreads_or(f);
  if (tid == 0) decide(a, tot, anyf);
}

// One tile element by element: a ragged tail of a vector run (e >= e0 within
// the thread's 8 elements) or any tile of a run with a misaligned pointer
// (elements base + i*256 + tid, coalesced).  Kept out of line: it is rare, and
// inlining it would cost the main loops registers.
template <typename GT, bool STASH>
__device__ __noinline__ void pass1_elementwise_tile(const Pass1Args& a, int64_t n,
                                                    int64_t stash_off, int32_t gbase,
                                                    int32_t vec, int64_t base, SqAcc& acc) {
  const int tid = threadIdx.x;
  const int64_t e0 = base + tid * kVec;
  float x[kVec];
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
    x[i] = sum;
  }
  acc.add<false>(x);
}

// Single gradient buffer (R*K = 1, never stashed).  ZO_PASS1_UNROLL tiles'
// 16-byte loads are issued before any is reduced; reduction works on the raw
// 16-bit words (SqAcc::add_raw16).
template <typename GT>
__global__ void __launch_bounds__(kThreads, ZO_PASS1_MIN_CTAS)
    pass1_single_kernel(const Pass1Args a) {
  __shared__ double red[kThreads / 32];
  __shared__ int s_last;
  constexpr int U = ZO_PASS1_UNROLL;
  const int tid = threadIdx.x;
  const int64_t G = gridDim.x;
  SqAcc acc;
  RunCursorLite cur;
  for (int64_t t0 = blockIdx.x; t0 < a.ntiles; t0 += U * G) {
    uint4 raw[U];
    bool fast[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t tile = t0 + u * G;
      fast[u] = false;
      if (tile < a.ntiles) {
        cur.seek(a.segs, a.nseg, tile);
        const int64_t e0 = (tile - cur.s.tile0) * kTile + tid * kVec;
        if (cur.s.vec && e0 + kVec <= cur.s.n) {
          raw[u] = __ldcg(reinterpret_cast<const uint4*>(grad_ptr(a.gptrs, cur.s, 0) + e0));
          fast[u] = true;
        }
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t tile = t0 + u * G;
      if (tile >= a.ntiles) continue;
      if (fast[u]) {
        // the sum is 0 + g, which differs from g only in the sign of a zero
        // (irrelevant to the statistics)
        acc.add_raw16<GT>(raw[u]);
      } else {
        cur.seek(a.segs, a.nseg, tile);
        pass1_elementwise_tile<GT, false>(a, cur.s.n, cur.s.stash_off, cur.s.gbase, cur.s.vec,
                                          (tile - cur.s.tile0) * kTile, acc);
      }
    }
  }
  pass1_finish(a, acc.total(), acc.overflowed<GT>() ? 1 : 0, red, &s_last);
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
#define ZO_BULK_STAGES 8
#endif

// Single gradient buffer, staged through shared memory by bulk copies: thread
// 0 keeps ZO_BULK_STAGES tiles (4 KiB each for 16-bit gradients) in flight per
// CTA, so the reducing threads never wait on global memory.  A tile that is
// not a full 16-byte aligned tile (a run's ragged tail, a misaligned run) is
// not copied: its barrier phase is completed by a plain arrival and the tile
// is reduced element by element from global memory.  If a wait expires the
// CTA stops issuing copies, waits (again bounded) for those in flight, and
// records a fault, which makes the step a no-op.
template <typename GT>
__global__ void __launch_bounds__(kThreads, ZO_PASS1_MIN_CTAS)
    pass1_bulk_kernel(const Pass1Args a) {
  constexpr int S = ZO_BULK_STAGES;
  __shared__ __align__(128) uint4 buf[S][kThreads];
  __shared__ __align__(8) unsigned long long bar[S];
  __shared__ double red[kThreads / 32];
  __shared__ int s_last, s_err;
  const int tid = threadIdx.x;
  const int64_t G = gridDim.x;
  const int64_t mine = (a.ntiles > (int64_t)blockIdx.x)
                           ? (a.ntiles - 1 - (int64_t)blockIdx.x) / G + 1
                           : 0;
  RunCursorLite pcur;  // thread 0's cursor for issuing copies
  auto issue = [&](int64_t i) {
    const int64_t tile = blockIdx.x + i * G;
    unsigned long long* b = &bar[i % S];
    if (a.inject_wait_fault && blockIdx.x == 0 && i == 1) return;  // test hook
    pcur.seek(a.segs, a.nseg, tile);
    const int64_t base = (tile - pcur.s.tile0) * kTile;
    if (pcur.s.vec && base + kTile <= pcur.s.n) {
      mbar_arrive_expect_tx(b, kTile * 2);
      bulk_load(&buf[i % S][0], grad_ptr(a.gptrs, pcur.s, 0) + base, kTile * 2, b);
    } else {
      mbar_arrive(b);
    }
  };
  if (tid == 0) {
    for (int k = 0; k < S; ++k) mbar_init(&bar[k], 1);
    mbar_init_fence();
    s_err = 0;
  }
  __syncthreads();
  if (tid == 0)
    for (int64_t i = 0; i < mine && i < S; ++i) issue(i);
  SqAcc acc;
  RunCursorLite cur;
  int64_t issued = mine < S ? mine : S;
  for (int64_t i = 0; i < mine; ++i) {
    const uint32_t parity = (uint32_t)((i / S) & 1);
    if (!mbar_wait_bounded(&bar[i % S], parity)) s_err = 1;
    const int64_t tile = blockIdx.x + i * G;
    cur.seek(a.segs, a.nseg, tile);
    const int64_t base = (tile - cur.s.tile0) * kTile;
    if (!s_err) {
      if (cur.s.vec && base + kTile <= cur.s.n)
        acc.add_raw16<GT>(buf[i % S][tid]);
      else
        pass1_elementwise_tile<GT, false>(a, cur.s.n, cur.s.stash_off, cur.s.gbase, cur.s.vec,
                                          base, acc);
    }
    __syncthreads();  // every thread is done with stage i % S
    if (s_err) {
      // drain the copies still in flight before the CTA's shared memory goes
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
  pass1_finish(a, acc.total(), acc.overflowed<GT>() ? 1 : 0, red, &s_last);
}

// Any number of gradient buffers, loaded in batches of eight per tile, summed
// in buffer order; optionally stores the sums (the stash).
template <typename GT, bool STASH>
__global__ void __launch_bounds__(kThreads, ZO_PASS1_MIN_CTAS)
    pass1_multi_kernel(const Pass1Args a) {
  __shared__ double red[kThreads / 32];
  __shared__ int s_last;
  const int tid = threadIdx.x;
  SqAcc acc;
  RunCursorLite cur;
  for (int64_t tile = blockIdx.x; tile < a.ntiles; tile += gridDim.x) {
    cur.seek(a.segs, a.nseg, tile);
    const auto& s = cur.s;
    const int64_t base = (tile - s.tile0) * kTile;
    const int64_t e0 = base + tid * kVec;
    if (!(s.vec && e0 + kVec <= s.n)) {
      pass1_elementwise_tile<GT, STASH>(a, s.n, s.stash_off, s.gbase, s.vec, base, acc);
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
  pass1_finish(a, acc.total(), acc.overflowed<GT>() ? 1 : 0, red, &s_last);
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

__device__ __forceinline__ void f4_to(const float4& a, float* d) {
  d[0] = a.x; d[1] = a.y; d[2] = a.z; d[3] = a.w;
}

// SRC == 1: one gradient buffer; SRC == 0: a.nbuf buffers; SRC == -1: stash.
template <typename GT, typename PT, int SRC>
__global__ void __launch_bounds__(kThreads, ZO_PASS2_MIN_CTAS) pass2_kernel(const Pass2Args a) {
  const Decision* dp = a.dec;
  if (dp->skip) return;
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
  if ((int64_t)blockIdx.x >= a.ntiles) return;
  const int64_t cnt = (a.ntiles - 1 - blockIdx.x) / G + 1;
  RunCursor cur;
  for (int64_t k = cnt - 1; k >= 0; --k) {
    const int64_t tile = blockIdx.x + k * G;
    cur.seek(a.segs, a.nseg, tile);
    const Seg& s = cur.s;
    const int64_t base = (tile - s.tile0) * kTile;
    const int64_t e0 = base + tid * kVec;
    if (s.vec && e0 + kVec <= s.n) {
      float x[kVec], p[kVec], m[kVec], v[kVec];
      if (SRC == -1) {
        const float4* st = reinterpret_cast<const float4*>(a.stash + s.stash_off + e0);
        f4_to(__ldcs(st), x);
        f4_to(__ldcs(st + 1), x + 4);
      } else if (SRC == 1) {
        Fmt<GT>::dec8(__ldcs(reinterpret_cast<const uint4*>(grad_ptr(a.gptrs, s, 0) + e0)), x);
#pragma unroll
        for (int i = 0; i < kVec; ++i) x[i] = __fadd_rn(0.0f, x[i]);
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
      const float4* pm = reinterpret_cast<const float4*>(s.master + e0);
      const float4* mm = reinterpret_cast<const float4*>(s.m + e0);
      const float4* vm = reinterpret_cast<const float4*>(s.v + e0);
      f4_to(__ldcs(pm), p);
      f4_to(__ldcs(pm + 1), p + 4);
      f4_to(__ldcs(mm), m);
      f4_to(__ldcs(mm + 1), m + 4);
      f4_to(__ldcs(vm), v);
      f4_to(__ldcs(vm + 1), v + 4);
#pragma unroll
      for (int i = 0; i < kVec; ++i) adam_elem(x[i], p[i], m[i], v[i], c);
      float4* po = reinterpret_cast<float4*>(s.master + e0);
      float4* mo = reinterpret_cast<float4*>(s.m + e0);
      float4* vo = reinterpret_cast<float4*>(s.v + e0);
      __stcs(po, make_float4(p[0], p[1], p[2], p[3]));
      __stcs(po + 1, make_float4(p[4], p[5], p[6], p[7]));
      __stcs(mo, make_float4(m[0], m[1], m[2], m[3]));
      __stcs(mo + 1, make_float4(m[4], m[5], m[6], m[7]));
      __stcs(vo, make_float4(v[0], v[1], v[2], v[3]));
      __stcs(vo + 1, make_float4(v[4], v[5], v[6], v[7]));
      __stcs(reinterpret_cast<uint4*>(static_cast<unsigned short*>(s.p16) + e0),
             Fmt<PT>::enc8(p));
    } else {
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
        float p = __ldcs(s.master + e), m = __ldcs(s.m + e), v = __ldcs(s.v + e);
        adam_elem(x, p, m, v, c);
        __stcs(s.master + e, p);
        __stcs(s.m + e, m);
        __stcs(s.v + e, v);
        static_cast<unsigned short*>(s.p16)[e] = Fmt<PT>::enc(p);
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
