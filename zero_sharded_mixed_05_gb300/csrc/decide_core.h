// decide_core.h -- the per-step decision (a4): skip on overflow, the clip
// coefficient, the Adam/AdamW update scalars and the dynamic loss-scale state
// machine.  Shared by the device pass 1 (one thread of its last CTA) and the
// host (offloaded) step, so both take the same decisions from the same
// statistics.  Plain C++ apart from the host/device qualifiers.
//
// Sources: "DeepSpeed tutorial" (devpress.csdn.net) §2.2 (loss scaling: a
// step whose gradients overflow is skipped and lowers the scale, which rises
// again once training is stable) and §3.2 (the ds_config.json fp16 block:
// loss_scale 0 for dynamic scaling, initial_scale_power, loss_scale_window,
// hysteresis, min_loss_scale; the AdamW optimizer block and the WarmupLR
// scheduler block); "DeepSpeed ZeRO引擎深入" (aiqz.cc), "Python 演示" (the Adam
// update: first and second moments, eps added outside the square root).  So:
// an inf or NaN in the reduced gradients skips the step and lowers the loss
// scale (not below min_loss_scale); the scale grows by the factor after
// loss_scale_window consecutive applied steps; Adam keeps m and v with bias
// correction, eps outside the root, and AdamW's weight decay is decoupled.  Readings where the pages are
// silent: the global L2 norm of the unscaled gradient with coefficient
// min(1, max_norm / (norm + 1e-6)); hysteresis lowers the scale on the
// hysteresis-th overflow since it last changed; WarmupLR ramps the lr linearly
// from warmup_min_lr to warmup_max_lr over warmup_num_steps applied steps.
#pragma once

#include <math.h>
#include <stdint.h>

#include "zero_opt_internal.h"

#ifdef __CUDACC__
#define ZO_HD __host__ __device__
#else
#define ZO_HD
#endif

namespace zo {

ZO_HD inline double quiet_nan() {
  union {
    int64_t i;
    double d;
  } u;
  u.i = 0x7ff8000000000000ll;
  return u.d;
}

// Update scalars of Adam step t, computed in binary64 and rounded once to
// binary32: step_size = lr / bc1, isb2 = 1 / sqrt(bc2) with the bias
// corrections bc1 = 1 - beta1^t, bc2 = 1 - beta2^t (both 1 without bias
// correction), and the decoupled decay 1 - lr * wd, where lr is WarmupLR's
// value when warmup_num_steps > 0.
ZO_HD inline void step_scalars_bc(const Hyper& hp, int64_t t, double bc1, double bc2,
                                  float* step_size, float* isb2, float* decay) {
  if (!hp.bias_correction) bc1 = bc2 = 1.0;
  double lr = hp.lr;
  if (hp.warmup_num_steps > 0) {
    const double T = (double)hp.warmup_num_steps;
    const double frac = (double)t < T ? (double)t / T : 1.0;
    lr = hp.warmup_min_lr + (hp.warmup_max_lr - hp.warmup_min_lr) * frac;
  }
  *step_size = (float)(lr / bc1);
  *isb2 = (float)(1.0 / sqrt(bc2));
  *decay = (float)(1.0 - lr * hp.wd);
}

// The bias corrections of Adam step t: 1 - beta1^t and 1 - beta2^t.
ZO_HD inline double bias_correction(double beta, int64_t t) { return 1.0 - pow(beta, (double)t); }

ZO_HD inline void step_scalars(const Hyper& hp, int64_t t, float* step_size, float* isb2,
                               float* decay) {
  step_scalars_bc(hp, t, bias_correction(hp.beta1, t), bias_correction(hp.beta2, t), step_size,
                  isb2, decay);
}

// The decision of one step of a rank whose scaler state is `st` (updated in
// place), from the global statistics.  `scalars(t, &step_size, &isb2,
// &decay)` supplies the update scalars of Adam step t: step_scalars itself,
// or values computed ahead of time.
template <typename Scalars>
ZO_HD inline Decision decide_core(const Hyper& hp, RankState& st, double sumsq, int nonfinite,
                                  Scalars scalars, const double* inv_pre = nullptr) {
  Decision d;
  d.fault = 0;
  d.pad_ = 0;
  d.sumsq = sumsq;
  d.nonfinite = nonfinite;
  d.scale_used = st.scale;
  d.coef = 0.0f;
  d.step_size = d.isb2 = d.decay = d.b1 = d.omb1 = d.b2 = d.omb2 = d.eps = 0.0f;
  const float scale = st.scale;
  // inv_pre: the same quotient, computed ahead for this scale
  const double inv = inv_pre ? *inv_pre : 1.0 / ((double)scale * hp.divisor);
  if (nonfinite) {
    d.skip = 1;
    d.norm = quiet_nan();
    if (hp.dynamic) {
      st.overflows += 1;
      if (st.overflows >= hp.hysteresis) {
        double lowered = (double)scale / hp.factor;
        if (lowered < hp.min_scale) lowered = hp.min_scale;
        st.scale = (float)lowered;
        st.overflows = 0;
      }
    }
    st.clean = 0;
    st.skipped_total += 1;
    st.last_skipped = 1;
  } else {
    const double norm = sqrt(sumsq) * inv;
    // clip = min(1, max_norm / b) with b = norm + 1e-6.  For binary64
    // max_norm >= b the rounded quotient is at least 1; for max_norm < b the
    // exact quotient is at most 1 - 2^-53 (max_norm is at most b less one
    // unit in b's last place), so it rounds below 1.  The division is
    // therefore needed only in the second case, and gives the same clip.
    double clip = 1.0;
    if (hp.clip_on) {
      const double b = norm + 1e-6;
      if (hp.max_norm < b) clip = hp.max_norm / b;
    }
    d.skip = 0;
    d.norm = norm;
    d.coef = (float)(inv * clip);
    st.t += 1;
    scalars(st.t, &d.step_size, &d.isb2, &d.decay);
    d.b1 = hp.b1f;
    d.omb1 = hp.omb1f;
    d.b2 = hp.b2f;
    d.omb2 = hp.omb2f;
    d.eps = hp.epsf;
    st.last_skipped = 0;
    st.clean += 1;
    if (hp.dynamic && st.clean == hp.window) {
      st.scale = (float)((double)scale * hp.factor);
      st.clean = 0;
      st.overflows = 0;
    }
  }
  d.t = st.t;
  return d;
}

// The decision of a step whose statistics could not be completed (a bounded
// wait expired): skipped, nothing of the scaler state changes.
ZO_HD inline Decision fault_decision(const RankState& st) {
  Decision d;
  d.sumsq = d.norm = quiet_nan();
  d.coef = 0.0f;
  d.skip = 1;
  d.nonfinite = 0;
  d.t = st.t;
  d.fault = 1;
  d.pad_ = 0;
  d.step_size = d.isb2 = d.decay = d.b1 = d.omb1 = d.b2 = d.omb2 = d.eps = 0.0f;
  d.scale_used = st.scale;
  return d;
}

}  // namespace zo
