// zero_opt_internal.h -- device-visible data structures shared by the host
// side (zero_opt.cu) and the kernels (kernels.cuh).  Not part of the ABI.
#pragma once

#include <stdint.h>

#include "zero_opt.h"

namespace zo {

constexpr int kThreads = 256;            // threads per CTA
constexpr int kVec = 8;                  // elements per thread per tile
constexpr int kTile = kThreads * kVec;   // 2048 elements per tile
constexpr int kMaxCtas = 4096;           // partial-sum slots in the workspace
constexpr int kMaxBufs = 1024;           // R*K limit

// One contiguous run of elements with its own buffers: the whole shard of a
// flat buffer, or one tensor of a per-tensor list.  All pointers already point
// at the run's first element.
struct Seg {
  float* master;
  float* m;
  float* v;
  void* p16;
  int64_t n;          // elements in the run (> 0)
  int64_t tile0;      // first tile index of the run
  int64_t ntiles;     // ceil(n / kTile)
  int64_t stash_off;  // element offset of the run in the stash
  int32_t gbase;      // first entry of the run's gradient pointers
  int32_t vec;        // 1: every pointer 16-byte aligned (vector path)
};

// Loss-scaler replica of one rank; same layout as zero_opt_scaler_state.
struct RankState {
  float scale;
  int32_t last_skipped;
  int64_t clean;
  int64_t t;
  int64_t skipped_total;
  int32_t overflows;     // overflows since the scale last changed
  int32_t reserved;
};
static_assert(sizeof(RankState) == sizeof(zero_opt_scaler_state), "layout");

// Decision of one step.  The first fields have the layout of
// zero_opt_step_info; the binary32 scalars of the update follow.
struct Decision {
  double sumsq;
  double norm;
  float coef;
  float scale_used;
  int32_t skip;
  int32_t nonfinite;
  int64_t t;
  int32_t fault;
  int32_t pad_;
  float step_size, isb2, decay, b1, omb1, b2, omb2, eps;
};
static_assert(sizeof(zero_opt_step_info) <= sizeof(Decision), "layout");

// The step-dependent update scalars for Adam step t, computed ahead of the
// decision by pass 1's scalar CTA.
struct PreScalars {
  int64_t t;             // the step they belong to; 0: none
  float step_size, isb2, decay;
  int32_t pad_;
  double inv;            // 1 / (scale * divisor) for the scale of this launch
};

// Steps whose bias corrections are tabulated per handle (computed on the
// device at creation with the same pow as the decision's fallback).
constexpr int64_t kBcSteps = 1 << 16;

// Update scalars the host supplies with each stepping launch: those of Adam
// steps cand_t0, cand_t0 - 1, ..., cand_t0 - (kScalarCands - 1) (the step the
// host expects, and the ones after up to seven skipped steps it has not seen).
constexpr int kScalarCands = 8;

struct Workspace {
  unsigned int ticket;   // CTAs of pass 1 that finished; reset by the last
  int32_t fault;         // set by a CTA whose bounded wait expired; reset by decide
  Decision dec;          // written by the last CTA of pass 1, read by pass 2
  PreScalars pre;        // written by the scalar CTA, read by decide
  double own_sumsq;      // statistics-only result
  int32_t own_nonfinite;
  int32_t pad1;
  double part_sumsq[kMaxCtas];
  int32_t part_flag[kMaxCtas];
};

struct Hyper {
  double lr, beta1, beta2, eps, wd, max_norm, divisor, min_scale, factor;
  int64_t window;
  int32_t bias_correction, dynamic;
  int64_t hysteresis;
  double warmup_min_lr, warmup_max_lr;
  int64_t warmup_num_steps;
  // The decision's step-independent binary32 constants, rounded once on the
  // host from the binary64 values above (the device's binary64 rate is low):
  // beta1, 1 - beta1, beta2, 1 - beta2, eps; clip_on = max_norm > 0.
  float b1f, omb1f, b2f, omb2f, epsf;
  int32_t clip_on;
};

// kStepGlobalDev: the global statistics are folded on the device from the
// per-rank statistics at g_dev (g_n of them, rank order).
enum Mode : int32_t { kStepLocal = 0, kStepGlobal = 1, kStatsOnly = 2, kStepGlobalDev = 3 };

struct Pass1Args {
  const Seg* segs;
  const void* const* gptrs;
  int32_t nseg;
  int32_t nbuf;
  int64_t ntiles;        // 0: decide only
  float* stash;          // non-NULL: store the reduced sums
  int32_t mode;
  int32_t rank;
  double g_sumsq;        // kStepGlobal: the folded statistics
  int32_t g_nonfinite;
  int32_t pad;
  Hyper hp;
  Workspace* ws;
  RankState* ranks;
  int32_t inject_wait_fault;   // test hook: leave one bulk-copy barrier un-armed
  int32_t scalar_cta;          // 1: the last CTA streams nothing and precomputes
                               // the next step's update scalars
  const double* bc_table;      // [kBcSteps][2]: 1 - beta1^t, 1 - beta2^t for t = 1..kBcSteps
  const zero_opt_stats* g_dev; // kStepGlobalDev: per-rank statistics (device)
  zero_opt_stats* stats_out;   // kStatsOnly: also written here (device), or NULL
  int32_t g_n;
  int32_t pad3;
  int64_t keep_tile0;          // single-buffer chunks from this tile on are read
                               // with an L2 evict_last policy (ntiles: none)
  double inv_d;                // 1 / divisor, rounded once (binary64)
  int64_t cand_t0;             // the scalar candidates' first step (see above)
  int32_t ncand;               // candidates supplied (0: none)
  int32_t pad5;
  float cand[kScalarCands][3]; // step_size, isb2, decay of step cand_t0 - j
};

struct Pass2Args {
  const Seg* segs;
  const void* const* gptrs;
  int32_t nseg;
  int32_t nbuf;
  int64_t ntiles;
  const float* stash;    // non-NULL: read the reduced sums from here
  const Decision* dec;
  int64_t keep_tile0;    // gradients of tiles from here on were kept in L2 by
                         // pass 1; pass 2 returns their lines to evict_normal
};

}  // namespace zo
