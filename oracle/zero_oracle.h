/*
 * zero_oracle.h -- TEST INFRASTRUCTURE ONLY.
 *
 * Plain, single-threaded CPU definition of the per-shard mixed-precision
 * ZeRO optimizer step.  It is the parity oracle for the CUDA library and
 * nothing else: only the tests, the smoke check and the benchmark's CPU
 * baseline may load it.  It shares no code, header, table or constant with
 * the CUDA path (zero_sharded_mixed_05_gb300/csrc), and neither side includes
 * the other.
 *
 * Sources (page title, section):
 *   [CSDN]  "DeepSpeed tutorial" (devpress.csdn.net): §2.1 ZeRO memory
 *           accounting, §2.2 Loss Scaling, §2.3 gradient accumulation,
 *           §2.4 optimizer on the local slice, §3.2 ds_config.json.
 *   [AIQZ]  "DeepSpeed ZeRO引擎深入" (aiqz.cc): "显存四巨头", "ZeRO三阶段",
 *           "混合精度", "Python 演示" (the NumPy ZeROStage1 demo).
 *   [JWZ]   "LLM-train tutorials, ch01 项目背景与定位" (jwzheng96.github.io):
 *           §1.2, the M_DDP and M_ZeRO-1/2/3 equations and the stage table;
 *           §1.7, the list of later additions (low-precision master weights).
 *   [ALGO]  "DeepSpeed framework interview answer" (algomooc.com):
 *           "ZeRO 三阶段".
 *   [AIDH]  "DeepSpeed" (aidhplus.com): ZeRO-1/2/3 paragraphs, dynamic
 *           loss scaling bullet.
 *
 * Precision: the pages fix the storage types (16-bit parameters and
 * gradients, fp32 master weights, fp32 Adam m and v: [CSDN] §2.1, [AIQZ]
 * "显存四巨头") and that the update runs on the fp32 master copy ([AIQZ]
 * "混合精度").  The oracle therefore performs the per-element update as a
 * sequence of individually rounded IEEE binary32 operations (built with
 * -ffp-contract=off, never -ffast-math), computes per-step scalars in binary64
 * and rounds each once to binary32, and accumulates the squared-gradient sum
 * in binary64.
 *
 * Parity unpinned (readings of what the pages name without defining; each is
 * pinned to its reading, not to the pages): the hysteresis rule of
 * orc_decide (the scale falls on the hysteresis-th overflow since it last
 * changed), the linear shape of WarmupLR in orc_decide (its endpoints and
 * update counting are the pages'; the shape follows the linear warm-up of the
 * script the tutorial migrates from, get_linear_schedule_with_warmup in
 * [CSDN] §3.3, since the WarmupLR block itself gives no curve), and
 * low-precision master weights in
 * orc_update (master == NULL: the 16-bit copy is the master, [JWZ] §1.7).
 */
#ifndef ZERO_ORACLE_H
#define ZERO_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { ORC_FP16 = 0, ORC_BF16 = 1 };

/* Optimizer and loss-scaler hyper-parameters, as real numbers (the values a
 * ds_config.json holds, [CSDN] §3.2). */
typedef struct orc_hparams {
  double lr, beta1, beta2, eps, weight_decay;
  double max_grad_norm;        /* <= 0: no clipping */
  int32_t bias_correction;     /* 1: standard Adam; 0: the [AIQZ] demo form */
  int32_t dynamic_scale;       /* 1: dynamic loss scale; 0: fixed scale */
  double min_scale;            /* floor of the dynamic scale ("min_loss_scale") */
  double scale_factor;         /* 2: halve on overflow, double after window */
  int64_t scale_window;        /* "loss_scale_window" */
  int64_t hysteresis;          /* overflows that lower the scale once (>= 1) */
  double warmup_min_lr;        /* WarmupLR: lr of the first update ...          */
  double warmup_max_lr;        /* ... rising linearly to this one               */
  int64_t warmup_num_steps;    /* ... over this many updates (0: constant lr)   */
} orc_hparams;

/* Loss-scaler state of one rank plus the Adam step counter. */
typedef struct orc_scaler {
  float scale;
  int32_t last_skipped;
  int64_t clean;               /* consecutive clean steps since last change */
  int64_t t;                   /* Adam step counter (updates applied) */
  int64_t skipped_total;
  int32_t overflows;           /* overflows since the scale last changed */
  int32_t pad_;
} orc_scaler;

/* Gradient statistics of one shard (or the fold over all shards). */
typedef struct orc_stats {
  double sumsq;                /* sum of squares of the fp32 reduced grads */
  int32_t nonfinite;           /* 1 if any reduced grad is inf or NaN */
  int32_t pad_;
} orc_stats;

/* Per-step decision and the binary32 scalars of the update. */
typedef struct orc_decision {
  int32_t skip;
  float coef;                  /* unscale x clip factor applied to the sum */
  double norm;                 /* L2 norm of the unscaled reduced gradient */
  double inv;                  /* 1 / (scale * divisor) */
  float scale_used;            /* loss scale the gradients were produced with */
  float step_size, isb2, decay, b1, omb1, b2, omb2, eps;
  double lr;                   /* learning rate of this update */
} orc_decision;

/* a0: shard bounds.  out = {begin, real_end, shard_len, padded_numel}. */
int orc_shard_bounds(int64_t numel, int32_t world, int32_t rank, int64_t out[4]);

/* Per-GPU model-state bytes of ZeRO stage 0..3 on the padded shard. */
int64_t orc_memory_bytes(int64_t numel, int32_t world, int32_t stage);

/* IEEE round-to-nearest-even conversions, written from the formats. */
uint16_t orc_f32_to_16(float f, int32_t dtype);
float orc_16_to_f32(uint16_t h, int32_t dtype);
void orc_cast_f32_to_16(const float* src, uint16_t* dst, int64_t n, int32_t dtype);
void orc_cast_16_to_f32(const uint16_t* src, float* dst, int64_t n, int32_t dtype);

/* a1: s_j = sum over buffers b (in order) of float(g[b][j]), fp32. */
void orc_reduce(const uint16_t* const* bufs, int32_t nbuf, int64_t n,
                int32_t dtype, float* s);

/* a2, a3: statistics of a run of reduced gradients. */
orc_stats orc_stats_of(const float* s, int64_t n);

/* Fold per-rank statistics in rank order (the scalar all-reduce). */
orc_stats orc_fold_stats(const orc_stats* per_rank, int32_t n);

/* a4: decide skip / clip / scalars from the global statistics and advance
 * the loss-scaler state. */
void orc_decide(const orc_hparams* hp, orc_scaler* st, orc_stats global,
                double divisor, orc_decision* out);

/* a5..a7: unscale, clip, AdamW, 16-bit write-back over n elements.  With
 * master == NULL the 16-bit copy p16 is the master weight (low-precision
 * master weights): each element is widened to binary32, updated, and stored
 * back rounded to nearest even. */
void orc_update(const orc_decision* d, const float* s, float* master,
                float* m, float* v, uint16_t* p16, int64_t n, int32_t pdtype);

/* One whole step over one shard: reduce, statistics, decide (with `global`
 * when non-NULL, else the shard's own statistics), update. */
int orc_step(const orc_hparams* hp, orc_scaler* st,
             const uint16_t* const* grads, int32_t nbuf, int32_t gdtype,
             int64_t n, double divisor,
             float* master, float* m, float* v, uint16_t* p16, int32_t pdtype,
             const orc_stats* global, orc_stats* own, orc_decision* dec);

/* zero_to_fp32: the full fp32 weights are the real parts of the N shards'
 * master weights laid end to end in rank order, padding dropped. */
void orc_consolidate(const float* const* shard_master, int32_t world, int64_t numel,
                     float* out);

#ifdef __cplusplus
}
#endif
#endif
