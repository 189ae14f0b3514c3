/*
 * zero_oracle.cpp -- TEST INFRASTRUCTURE ONLY: the parity oracle.
 *
 * A plain, slow, single-threaded restatement of the per-shard mixed-precision
 * ZeRO optimizer step, written from the pages listed in zero_oracle.h.  No
 * blocking, threading, vectorisation or reordering: every loop runs over the
 * elements in index order exactly as the definition reads.  Build with
 * -O2 -ffp-contract=off (no fused multiply-add, no -ffast-math) so that every
 * binary32 operation below is one IEEE-rounded operation.
 */
#include "zero_oracle.h"

#include <cmath>
#include <cstring>

/* ------------------------------------------------------------------------
 * a0: flat partition into N equal shards.
 * "ZeRO三阶段" ([AIQZ]) cuts the model state into N parts by GPU count; a
 * rank updates only its own slice ([CSDN] §2.4).  The flat buffer is padded
 * up to a multiple of N so that all N shards have the same length S.
 * ------------------------------------------------------------------------ */
extern "C" int orc_shard_bounds(int64_t numel, int32_t world, int32_t rank,
                                int64_t out[4]) {
  if (numel < 0 || world < 1 || rank < 0 || rank >= world) return 1;
  int64_t shard = (numel + world - 1) / world;      /* S = ceil(numel / N) */
  int64_t padded = shard * world;                   /* P = S * N */
  int64_t begin = (int64_t)rank * shard;
  int64_t end = begin + shard;
  int64_t real_end = end < numel ? end : numel;     /* padding is not real */
  if (real_end < begin) real_end = begin;           /* all-padding shard */
  out[0] = begin;
  out[1] = real_end;
  out[2] = shard;
  out[3] = padded;
  return 0;
}

/* Per-GPU model-state bytes.  Mixed-precision Adam keeps 2 bytes of 16-bit
 * parameters, 2 bytes of 16-bit gradients and 12 bytes of fp32 master, m and v
 * per parameter ([CSDN] §2.1; [JWZ] §1.2, M_DDP = 2Ψ + 2Ψ + 12Ψ = 16Ψ).  Stage 1
 * shards the 12Ψ, stage 2 also the gradients, stage 3 everything ([JWZ] §1.2,
 * M_ZeRO-1 = 4Ψ + 12Ψ/N, M_ZeRO-2 = 2Ψ + 14Ψ/N, M_ZeRO-3 = 16Ψ/N).  Here Ψ/N is
 * the padded shard length S, so the forms are exact integers; when N divides Ψ
 * they equal the pages' equations. */
extern "C" int64_t orc_memory_bytes(int64_t numel, int32_t world, int32_t stage) {
  int64_t b[4];
  if (orc_shard_bounds(numel, world, 0, b) != 0) return -1;
  int64_t psi = numel, s = b[2];
  switch (stage) {
    case 0: return 2 * psi + 2 * psi + 12 * psi;
    case 1: return 2 * psi + 2 * psi + 12 * s;
    case 2: return 2 * psi + 2 * s + 12 * s;
    case 3: return 2 * s + 2 * s + 12 * s;
    default: return -1;
  }
}

/* ------------------------------------------------------------------------
 * 16-bit formats.  fp16 is IEEE binary16 (1 sign, 5 exponent, 10 mantissa
 * bits); bf16 keeps binary32's 8 exponent bits and 7 mantissa bits.  A
 * conversion from binary32 rounds to the nearest representable value, ties to
 * the even significand, and overflows to infinity.
 * ------------------------------------------------------------------------ */
static void format_of(int32_t dtype, int* mbits, int* ebits) {
  if (dtype == ORC_BF16) { *mbits = 7; *ebits = 8; }
  else { *mbits = 10; *ebits = 5; }
}

extern "C" uint16_t orc_f32_to_16(float f, int32_t dtype) {
  int mbits, ebits;
  format_of(dtype, &mbits, &ebits);
  const int bias = (1 << (ebits - 1)) - 1;
  const int emax_field = (1 << ebits) - 1;
  uint32_t x;
  std::memcpy(&x, &f, 4);
  const uint16_t sign = (uint16_t)((x >> 31) << 15);
  const uint32_t e32 = (x >> 23) & 0xffu;
  const uint32_t m32 = x & 0x7fffffu;
  if (e32 == 0xffu) {                       /* inf stays inf, NaN -> quiet NaN */
    uint16_t inf = (uint16_t)(emax_field << mbits);
    if (m32 == 0) return (uint16_t)(sign | inf);
    return (uint16_t)(sign | inf | (1u << (mbits - 1)));
  }
  if (e32 == 0 && m32 == 0) return sign;    /* signed zero */

  /* |f| = sig * 2^e2 with an integer significand. */
  uint64_t sig;
  int e2;
  if (e32 == 0) { sig = m32; e2 = -149; }
  else { sig = m32 | 0x800000u; e2 = (int)e32 - 150; }
  int blen = 0;
  for (uint64_t t = sig; t != 0; t >>= 1) ++blen;
  const int k = e2 + blen - 1;              /* |f| lies in [2^k, 2^(k+1)) */
  const int kmin = 1 - bias;                /* smallest normal binade */
  const int qexp = (k < kmin ? kmin : k) - mbits;  /* spacing of the target grid */

  /* n = |f| / 2^qexp rounded to the nearest integer, ties to even. */
  const int shift = qexp - e2;
  uint64_t n;
  if (shift <= 0) {
    n = sig << (-shift);
  } else if (shift > 40) {
    n = 0;
  } else {
    n = sig >> shift;
    const uint64_t rem = sig & ((1ull << shift) - 1);
    const uint64_t half = 1ull << (shift - 1);
    if (rem > half || (rem == half && (n & 1u))) n += 1;
  }
  if (n == 0) return sign;
  if (k < kmin) {
    /* Subnormal grid; n == 2^mbits is exactly the smallest normal, whose
     * encoding is the same integer. */
    return (uint16_t)(sign | (uint16_t)n);
  }
  int ef = k + bias;
  if (n == (1ull << (mbits + 1))) { n >>= 1; ef += 1; }   /* rounded up a binade */
  if (ef >= emax_field) return (uint16_t)(sign | (emax_field << mbits));
  return (uint16_t)(sign | (ef << mbits) | (uint16_t)(n - (1ull << mbits)));
}

extern "C" float orc_16_to_f32(uint16_t h, int32_t dtype) {
  int mbits, ebits;
  format_of(dtype, &mbits, &ebits);
  const int bias = (1 << (ebits - 1)) - 1;
  const int emax_field = (1 << ebits) - 1;
  const int s = h >> 15;
  const int ef = (h >> mbits) & emax_field;
  const int man = h & ((1 << mbits) - 1);
  double v;
  if (ef == emax_field) v = man ? NAN : INFINITY;
  else if (ef == 0) v = std::ldexp((double)man, 1 - bias - mbits);
  else v = std::ldexp((double)((1 << mbits) + man), ef - bias - mbits);
  return (float)(s ? -v : v);              /* exact: every value fits binary32 */
}

extern "C" void orc_cast_f32_to_16(const float* src, uint16_t* dst, int64_t n,
                                   int32_t dtype) {
  for (int64_t i = 0; i < n; ++i) dst[i] = orc_f32_to_16(src[i], dtype);
}

extern "C" void orc_cast_16_to_f32(const uint16_t* src, float* dst, int64_t n,
                                   int32_t dtype) {
  for (int64_t i = 0; i < n; ++i) dst[i] = orc_16_to_f32(src[i], dtype);
}

/* ------------------------------------------------------------------------
 * a1: local reduction of the simulated ranks' and micro-steps' gradients.
 * Gradient accumulation sums K micro-batch gradients before one step
 * ([CSDN] §2.3); the reduce half of reduce-scatter sums the ranks' copies of
 * this shard ([ALGO] "ZeRO 三阶段"; [JWZ] §1.2 stage table).  Buffers are
 * given rank-major (b = r*K + k) and summed in that order in binary32.
 * ------------------------------------------------------------------------ */
extern "C" void orc_reduce(const uint16_t* const* bufs, int32_t nbuf, int64_t n,
                           int32_t dtype, float* s) {
  for (int64_t j = 0; j < n; ++j) {
    float acc = 0.0f;
    for (int32_t b = 0; b < nbuf; ++b) acc = acc + orc_16_to_f32(bufs[b][j], dtype);
    s[j] = acc;
  }
}

/* a2, a3: overflow flag and the sum of squares for the L2 norm.  The loss
 * scaler watches for gradients that overflowed to infinity ([CSDN] §2.2);
 * NaN counts as overflow too.  The norm is a plain sum with no order, so the
 * oracle computes the sum of squares to within one binary64 rounding of the
 * exact value: each square is exact in binary64 (a binary32 product needs 48
 * significand bits) and the running sum carries Neumaier's compensation term
 * (A. Neumaier, "Rundungsfehleranalyse einiger Verfahren zur Summation
 * endlicher Summen", ZAMM 54, 1974). */
extern "C" orc_stats orc_stats_of(const float* s, int64_t n) {
  orc_stats st;
  st.nonfinite = 0;
  st.pad_ = 0;
  double sum = 0.0, comp = 0.0;
  for (int64_t j = 0; j < n; ++j) {
    if (!std::isfinite(s[j])) st.nonfinite = 1;
    const double x = (double)s[j] * (double)s[j];
    const double t = sum + x;
    if (std::fabs(sum) >= std::fabs(x)) comp += (sum - t) + x;
    else comp += (x - t) + sum;
    sum = t;
  }
  st.sumsq = sum + comp;
  return st;
}

/* The scalar all-reduce across data-parallel ranks, folded in rank order. */
extern "C" orc_stats orc_fold_stats(const orc_stats* per_rank, int32_t n) {
  orc_stats st;
  st.sumsq = 0.0;
  st.nonfinite = 0;
  st.pad_ = 0;
  for (int32_t r = 0; r < n; ++r) {
    st.sumsq += per_rank[r].sumsq;
    if (per_rank[r].nonfinite) st.nonfinite = 1;
  }
  return st;
}

/* ------------------------------------------------------------------------
 * a4: per-step decisions and the dynamic loss scale.
 * [CSDN] §2.2: the loss (hence every gradient) is multiplied by the scale,
 * gradients are divided by the same factor before the update, the scale is
 * lowered when an overflow is detected and raised again once training has
 * been stable; §3.2 gives initial_scale_power 16, loss_scale_window 1000 and
 * min_loss_scale 1.  Reading: an overflowing step is skipped (no state moves,
 * the Adam counter does not advance) and the clean-step counter restarts; the
 * scale is divided by the factor (down to the floor) on the `hysteresis`-th
 * overflow since the scale last changed (§3.2 lists "hysteresis" without a
 * definition; 1 lowers it on every overflow); after `scale_window`
 * consecutive applied steps the scale is multiplied by the factor.
 * The learning rate follows WarmupLR (§3.2: warmup_min_lr, warmup_max_lr,
 * warmup_num_steps; §2.4: the scheduler steps with every parameter update),
 * read as a linear rise: update t uses min + (max - min) * min(t, T) / T.
 * Clipping divides the unscaled gradient by max(1, norm / max_norm) in the
 * form coef = min(1, max_norm / (norm + 1e-6)).
 * ------------------------------------------------------------------------ */
extern "C" void orc_decide(const orc_hparams* hp, orc_scaler* st, orc_stats global,
                           double divisor, orc_decision* d) {
  std::memset(d, 0, sizeof(*d));
  const float scale = st->scale;
  const double inv = 1.0 / ((double)scale * divisor);
  d->scale_used = scale;
  d->inv = inv;
  if (global.nonfinite) {
    d->skip = 1;
    d->norm = NAN;
    if (hp->dynamic_scale) {
      st->overflows += 1;
      if (st->overflows >= hp->hysteresis) {
        double lowered = (double)scale / hp->scale_factor;
        if (lowered < hp->min_scale) lowered = hp->min_scale;
        st->scale = (float)lowered;
        st->overflows = 0;
      }
    }
    st->clean = 0;
    st->skipped_total += 1;
    st->last_skipped = 1;
    return;
  }
  const double norm = std::sqrt(global.sumsq) * inv;
  double clip = 1.0;
  if (hp->max_grad_norm > 0.0) {
    clip = hp->max_grad_norm / (norm + 1e-6);
    if (clip > 1.0) clip = 1.0;
  }
  d->skip = 0;
  d->norm = norm;
  d->coef = (float)(inv * clip);

  st->t += 1;                                   /* first update uses t = 1 */
  const double t = (double)st->t;
  double bc1 = 1.0, bc2 = 1.0;
  if (hp->bias_correction) {
    bc1 = 1.0 - std::pow(hp->beta1, t);
    bc2 = 1.0 - std::pow(hp->beta2, t);
  }
  double lr = hp->lr;
  if (hp->warmup_num_steps > 0) {
    const double frac = t < (double)hp->warmup_num_steps ? t / (double)hp->warmup_num_steps : 1.0;
    lr = hp->warmup_min_lr + (hp->warmup_max_lr - hp->warmup_min_lr) * frac;
  }
  d->lr = lr;
  d->step_size = (float)(lr / bc1);
  d->isb2 = (float)(1.0 / std::sqrt(bc2));
  d->decay = (float)(1.0 - lr * hp->weight_decay);
  d->b1 = (float)hp->beta1;
  d->omb1 = (float)(1.0 - hp->beta1);
  d->b2 = (float)hp->beta2;
  d->omb2 = (float)(1.0 - hp->beta2);
  d->eps = (float)hp->eps;

  st->last_skipped = 0;
  st->clean += 1;
  if (hp->dynamic_scale && st->clean == hp->scale_window) {
    st->scale = (float)((double)scale * hp->scale_factor);
    st->clean = 0;
    st->overflows = 0;
  }
}

/* ------------------------------------------------------------------------
 * a5..a7: unscale and clip, AdamW on the fp32 master copy, 16-bit copy.
 * The moment updates and the eps outside the square root follow the Adam of
 * the "Python 演示" in [AIQZ]; bias correction divides m by 1 - beta1^t and v by
 * 1 - beta2^t (standard Adam; off reproduces the demo).  AdamW ([CSDN] §2.4,
 * §3.2 "type": "AdamW", weight_decay 0.01) decays the master weight by
 * (1 - lr*wd) before the Adam term.  The update runs on the fp32 master copy
 * and the 16-bit copy is its rounding ([AIQZ] "混合精度"; [CSDN] §2.2).
 * ------------------------------------------------------------------------ */
extern "C" void orc_update(const orc_decision* d, const float* s, float* master,
                           float* m, float* v, uint16_t* p16, int64_t n,
                           int32_t pdtype) {
  if (d->skip) return;
  for (int64_t j = 0; j < n; ++j) {
    const float g = s[j] * d->coef;
    // low-precision master weights: with no fp32 master array the 16-bit
    // parameter is the master, widened here and rounded back below
    float mj = m[j], vj = v[j];
    float pj = master ? master[j] : orc_16_to_f32(p16[j], pdtype);
    mj = d->b1 * mj + d->omb1 * g;
    vj = d->b2 * vj + d->omb2 * (g * g);
    const float den = std::sqrt(vj) * d->isb2 + d->eps;
    pj = pj * d->decay;
    pj = pj - d->step_size * (mj / den);
    m[j] = mj;
    v[j] = vj;
    if (master) master[j] = pj;
    if (p16) p16[j] = orc_f32_to_16(pj, pdtype);
  }
}

extern "C" int orc_step(const orc_hparams* hp, orc_scaler* st,
                        const uint16_t* const* grads, int32_t nbuf, int32_t gdtype,
                        int64_t n, double divisor,
                        float* master, float* m, float* v, uint16_t* p16,
                        int32_t pdtype, const orc_stats* global, orc_stats* own,
                        orc_decision* dec) {
  if (n < 0 || nbuf < 1 || divisor <= 0.0) return 1;
  float* s = new float[n > 0 ? n : 1];
  orc_reduce(grads, nbuf, n, gdtype, s);
  const orc_stats mine = orc_stats_of(s, n);
  if (own) *own = mine;
  orc_decision d;
  orc_decide(hp, st, global ? *global : mine, divisor, &d);
  orc_update(&d, s, master, m, v, p16, n, pdtype);
  if (dec) *dec = d;
  delete[] s;
  return 0;
}

/* zero_to_fp32 ("DeepSpeed framework interview answer", "训练与恢复边界"):
 * merge the ZeRO shards into one full fp32 state, padding dropped. */
extern "C" void orc_consolidate(const float* const* shard_master, int32_t world,
                                int64_t numel, float* out) {
  for (int32_t r = 0; r < world; ++r) {
    int64_t b[4];
    orc_shard_bounds(numel, world, r, b);
    for (int64_t j = b[0]; j < b[1]; ++j) out[j] = shard_master[r][j - b[0]];
  }
}
