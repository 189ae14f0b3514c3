/*
 * zero_opt.h -- C ABI of the GB300 per-shard mixed-precision ZeRO optimizer
 * step.
 *
 * One call of zero_opt_step performs, for the shard a data-parallel rank owns,
 * the whole optimizer step of a ZeRO training engine:
 *   (i)   the local reduction of the simulated ranks' and accumulation
 *         micro-steps' 16-bit gradients (the reduce half of reduce-scatter),
 *   (ii)  unscaling by the dynamic loss scale,
 *   (iii) overflow (inf/NaN) detection and the global L2 norm for clipping,
 *   (iv)  the fp32 Adam/AdamW update of the master weights, m and v, and
 *   (v)   the write-back of the 16-bit parameter copy,
 * and advances the loss scale: halve and skip on overflow, double after
 * scale_window clean steps.
 *
 * Sources (page title, section):
 *   "DeepSpeed tutorial" (devpress.csdn.net): §2.1 the 16Ψ model-state bytes
 *     and ZeRO-1/2/3; §2.2 loss scaling (scale the loss, unscale before the
 *     update, lower on overflow, raise when stable); §2.3 gradient
 *     accumulation; §2.4 each GPU's optimizer updates only its own slice;
 *     §3.2 ds_config.json (AdamW lr/betas/eps/weight_decay, fp16
 *     loss_scale_window / initial_scale_power / hysteresis / min_loss_scale).
 *   "DeepSpeed ZeRO引擎深入" (aiqz.cc): "显存四巨头" (2 + 2 + 12 bytes per
 *     parameter), "ZeRO三阶段" (cut the state into N parts), "混合精度"
 *     (update on the fp32 master copy), "Python 演示" (Adam moments, eps in
 *     the denominator).
 *   "LLM-train tutorials ch01" (jwzheng96.github.io): §1.2 M_DDP and
 *     M_ZeRO-1/2/3 equations; stage table (reduce-scatter / all-gather).
 *   "DeepSpeed framework interview answer" (algomooc.com): "ZeRO 三阶段"
 *     (reduce-scatter gradients, update local shard, all-gather parameters).
 *
 * Conventions for every call:
 *   - Every function returns a zero_status; arguments are checked before any
 *     CUDA work is issued, and a rejected call changes nothing.
 *   - "device" pointers are CUDA global-memory addresses on the device that
 *     was current when the handle was created; that device must be current
 *     for every call on the handle.  "host" pointers are ordinary CPU memory.
 *   - The library never allocates, frees or retains caller buffers.  Device
 *     buffers must stay valid until the stream has passed the work that uses
 *     them.  The handle owns a small device workspace (about 1.1 MB: the
 *     pass-1 partials and decision, the scaler replicas and a table of the
 *     Adam bias corrections of the first 65536 steps) and its run-table
 *     arena (1 MiB of device memory and 1 MiB of page-locked host memory by
 *     default, zero_opt_config.table_kib), all allocated by zero_opt_create
 *     and freed by zero_opt_destroy; no other call allocates or frees device
 *     or page-locked memory (zero_opt_get_counters counts any that would).
 *   - `stream` is a cudaStream_t (NULL is the legacy default stream).  Work is
 *     enqueued asynchronously unless the function says it synchronizes.
 *   - Calls on one handle must be ordered (one stream, or externally
 *     synchronized): they share the handle's workspace.
 *   - Pointers that are not 16-byte aligned are accepted; they select a
 *     slower element-wise path instead of 16-byte vector accesses.
 */
#ifndef ZERO_OPT_H
#define ZERO_OPT_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum zero_status {
  ZERO_OK = 0,
  ZERO_EINVAL = 1,   /* invalid argument (null pointer, bad value, bad dtype) */
  ZERO_ERANGE = 2,   /* index or size out of range (rank >= world, ...) */
  ZERO_ENOMEM = 3,   /* host or device allocation failed in zero_opt_create */
  ZERO_ECUDA = 4,    /* a CUDA call failed, or no CUDA device is present */
  ZERO_ENOTSUP = 5   /* option not supported                */
} zero_status;

typedef enum zero_dtype {
  ZERO_FP16 = 0,     /* IEEE binary16 */
  ZERO_BF16 = 1      /* bfloat16 */
} zero_dtype;

typedef struct zero_opt_handle* zero_opt_t;

/*
 * Optimizer and loss-scale configuration: the fields of a ds_config.json
 * ("DeepSpeed tutorial" §3.2) that the step needs.  Real numbers are given as
 * doubles; the per-step scalars derived from them are computed in double and
 * rounded once to float.
 */
typedef struct zero_opt_config {
  int64_t numel;            /* Ψ: real parameters of the flat buffer (>= 0) */
  int32_t world;            /* N: data-parallel degree (>= 1)               */
  int32_t grad_dtype;       /* zero_dtype of the gradient buffers           */
  int32_t param_dtype;      /* zero_dtype of the 16-bit parameter copy      */
  int32_t bias_correction;  /* 1: Adam bias correction; 0: none             */
  double lr;                /* learning rate (>= 0)                         */
  double beta1, beta2;      /* in [0, 1)                                    */
  double eps;               /* > 0, added outside the square root           */
  double weight_decay;      /* >= 0, decoupled (AdamW): p *= 1 - lr*wd      */
  double max_grad_norm;     /* > 0 clips the global L2 norm; <= 0 disables  */
  int32_t dynamic_scale;    /* 1: dynamic loss scale; 0: fixed init_scale   */
  int32_t hysteresis;       /* >= 1: the scale is lowered on the hysteresis-th
                               overflow since it last changed (1: every one) */
  double init_scale;        /* > 0, e.g. 2^initial_scale_power              */
  double min_scale;         /* > 0, "min_loss_scale"                        */
  double scale_factor;      /* >= 1, 2 halves / doubles                     */
  int64_t scale_window;     /* >= 1, "loss_scale_window"                    */
  double warmup_min_lr;     /* WarmupLR: update t uses warmup_min_lr +      */
  double warmup_max_lr;     /*   (max - min) * min(t, T) / T, T =           */
  int64_t warmup_num_steps; /*   warmup_num_steps; 0 keeps lr constant      */
  int32_t master16;         /* 1: low-precision master weights -- no fp32
                               master array (buffers' master is ignored, may
                               be NULL); the 16-bit parameter is the master,
                               widened to fp32 for the update and stored back
                               rounded to nearest even ("LLM-train tutorials
                               ch01" §1.7).  0: fp32 master (default)        */
  int32_t table_kib;        /* KiB of the handle's run-table arena (device
                               memory plus a page-locked host mirror of the
                               same size), allocated by zero_opt_create;
                               0 selects 1024.  A step's table takes 72 bytes
                               per run (the shard, or one tensor of a list)
                               plus 8 per run and gradient buffer, rounded up
                               to 256; 1024 KiB holds the table of a list of
                               13,000 tensors with one gradient buffer
                               each.  0..2^20                               */
} zero_opt_config;

/*
 * Buffers of one flat shard step.  Layout: the flat parameter buffer holds Ψ
 * real elements padded with zeros to P = N * S elements, S = ceil(Ψ / N); rank
 * r owns [r*S, r*S + S), of which [r*S, real_end) are real ("ZeRO三阶段";
 * "DeepSpeed tutorial" §2.4).  Only real elements are read or written.
 */
typedef struct zero_opt_buffers {
  float* master;            /* device, fp32 master weights of the shard (S)  */
  float* m;                 /* device, fp32 first moment of the shard (S)    */
  float* v;                 /* device, fp32 second moment of the shard (S)   */
  void* param16;            /* device, 16-bit parameters (param_dtype); the
                               full padded buffer (P) unless
                               param16_shard_local, then the shard (S)       */
  const void* const* grads; /* host array of n_ranks*n_micro device pointers,
                               rank-major (index r*n_micro + k); each is the
                               full padded gradient buffer (P) of simulated
                               rank r and micro-step k, unless
                               grads_shard_local, then the shard (S)         */
  int32_t n_ranks;          /* R >= 1: simulated data-parallel ranks         */
  int32_t n_micro;          /* K >= 1: gradient-accumulation micro-steps     */
  int32_t grads_shard_local;
  int32_t param16_shard_local;
  double divisor;           /* D: the reduced sum is divided by D*scale;
                               <= 0 selects R*K (the average)                */
  float* stash;             /* optional device fp32 scratch of S elements: when
                               R*K > 4 the reduced sum is kept here between the
                               two passes instead of re-reading R*K buffers;
                               NULL always re-reads                          */
} zero_opt_buffers;

/* One tensor of a per-tensor (non-flat) list, all its buffers separate. */
typedef struct zero_opt_tensor {
  int64_t numel;            /* elements of this tensor (>= 0)                */
  float* master;            /* device fp32, numel                            */
  float* m;                 /* device fp32, numel                            */
  float* v;                 /* device fp32, numel                            */
  void* param16;            /* device 16-bit, numel                          */
  const void* const* grads; /* host array of n_ranks*n_micro device pointers
                               to this tensor's gradients, rank-major        */
} zero_opt_tensor;

typedef struct zero_opt_tensor_list {
  const zero_opt_tensor* tensors;  /* host array of n_tensors entries        */
  int32_t n_tensors;               /* >= 0                                   */
  int32_t n_ranks, n_micro;        /* R, K as in zero_opt_buffers            */
  double divisor;                  /* as in zero_opt_buffers                 */
  float* stash;                    /* optional device fp32 scratch of the
                                      summed numel of all tensors, or NULL   */
} zero_opt_tensor_list;

/* Gradient statistics of one shard, or their fold over all ranks. */
typedef struct zero_opt_stats {
  double sumsq;             /* sum of squares of the fp32 reduced (still
                               scaled) gradient sums                         */
  int32_t nonfinite;        /* 1 if any reduced gradient is inf or NaN       */
  int32_t reserved;
} zero_opt_stats;

/* What the last step of a rank decided (zero_opt_last_step). */
typedef struct zero_opt_step_info {
  double sumsq;             /* global sum of squares used                    */
  double norm;              /* L2 norm of the unscaled gradient (NaN on skip) */
  float coef;               /* factor applied to each reduced sum            */
  float scale_used;         /* loss scale the gradients carried              */
  int32_t skipped;          /* 1 if the step was skipped (overflow or fault) */
  int32_t nonfinite;
  int64_t t;                /* Adam step counter after the step              */
  int32_t fault;            /* 1 if a kernel gave up waiting for its own data
                               copies (bounded wait expired): the step was
                               skipped and nothing, the loss scale included,
                               was changed                                   */
  int32_t reserved;
} zero_opt_step_info;

/* Loss-scaler state of one rank. */
typedef struct zero_opt_scaler_state {
  float scale;              /* current loss scale                            */
  int32_t last_skipped;     /* 1 if the last step was skipped                */
  int64_t clean_steps;      /* consecutive applied steps since last change   */
  int64_t t;                /* Adam step counter (applied updates)           */
  int64_t skipped_total;    /* skipped steps so far                          */
  int32_t overflows;        /* overflows since the scale last changed        */
  int32_t reserved;
} zero_opt_scaler_state;

/* Fill *cfg with the ds_config.json values of "DeepSpeed tutorial" §3.2:
 * AdamW lr 2e-5, betas (0.9, 0.999), eps 1e-8, weight_decay 0.01; dynamic
 * fp16 loss scale 2^16 (initial_scale_power 16), window 1000, min 1, factor
 * 2; bias correction on, no clipping; numel 0, world 1, fp16; hysteresis 2;
 * WarmupLR off (warmup_num_steps 0; set warmup_min_lr 0, warmup_max_lr 2e-5,
 * warmup_num_steps 1000 for the page's schedule).  Errors: EINVAL if cfg is
 * NULL. */
zero_status zero_opt_config_default(zero_opt_config* cfg);

/* Create an optimizer handle for one data-parallel group of `world` ranks.
 * Each rank r has its own loss-scaler replica (scale = init_scale, counters
 * 0).  Allocates the handle's device workspace on the current device when a
 * CUDA device is present; without one the handle serves only the host-side
 * calls and every launching call returns ZERO_ECUDA.
 * Errors: EINVAL (NULL pointers, numel < 0, world < 1, a dtype not in
 * zero_dtype, lr < 0, beta outside [0,1), eps <= 0, weight_decay < 0,
 * init_scale/min_scale <= 0, scale_factor < 1, scale_window < 1,
 * hysteresis < 1, warmup_num_steps < 0, a warm-up lr < 0); ENOMEM; ECUDA.
 * *out is NULL on failure. */
zero_status zero_opt_create(const zero_opt_config* cfg, zero_opt_t* out);

/* Destroy a handle (synchronizes the device first). NULL is accepted. */
zero_status zero_opt_destroy(zero_opt_t h);

/* Shard bounds of `rank` ("ZeRO三阶段": N equal parts; padding to P = N*S).
 * Host only.  Outputs (host, each may be NULL): begin = rank*S, real_end =
 * min(begin + S, Ψ) (>= begin), shard_len = S, padded_numel = P.
 * Errors: EINVAL (h NULL), ERANGE (rank outside [0, world)). */
zero_status zero_opt_shard_bounds(zero_opt_t h, int32_t rank, int64_t* begin,
                                  int64_t* real_end, int64_t* shard_len,
                                  int64_t* padded_numel);

/* Per-GPU model-state bytes of ZeRO stage 0..3 for Ψ = numel over N = world
 * ranks, on the padded shard S = ceil(Ψ/N): stage 0 (DDP) 16Ψ, stage 1
 * 4Ψ + 12S, stage 2 2Ψ + 14S, stage 3 16S ("LLM-train tutorials ch01" §1.2;
 * "DeepSpeed tutorial" §2.1).  Equal to the pages' forms when N divides Ψ.
 * Host only. Errors: EINVAL (bytes NULL, numel < 0, world < 1), ERANGE
 * (stage outside 0..3). */
zero_status zero_opt_memory_bytes(int64_t numel, int32_t world, int32_t stage,
                                  int64_t* bytes);

/* Statistics of `rank`'s shard only (steps a1..a3): the fp32 reduction of
 * the R*K gradient buffers, its overflow flag and its sum of squares.  This is
 * the local half of the scalar all-reduce; fold all ranks' results in rank
 * order (sum sumsq, OR nonfinite) and pass the fold to zero_opt_step.  Also
 * fills bufs->stash when it is used.  Synchronizes `stream`; *out is host.
 * Errors: as zero_opt_step. */
zero_status zero_opt_grad_stats(zero_opt_t h, int32_t rank,
                                const zero_opt_buffers* bufs, void* stream,
                                zero_opt_stats* out);

/* The scalar all-reduce of the statistics, done on the host: *out = the fold
 * of per_rank[0..n) in rank order (binary64 sum of sumsq starting from 0,
 * OR of nonfinite).  Every rank that folds the same array gets bit-identical
 * totals, as after an all-reduce ("DeepSpeed framework interview answer",
 * "ZeRO 三阶段": gradients are reduce-scattered before the local update).
 * Host only.  Errors: EINVAL (out NULL, n < 0, per_rank NULL with n > 0). */
zero_status zero_opt_fold_stats(const zero_opt_stats* per_rank, int32_t n,
                                zero_opt_stats* out);

/* The same two calls with the statistics kept on the device, so that a
 * multi-process step needs no host round trip (the statistics go from rank to
 * rank through a device collective, e.g. an all-gather of 16-byte records):
 *
 * zero_opt_grad_stats_async: as zero_opt_grad_stats, but the result is
 * written into the DEVICE zero_opt_stats `out_dev` on `stream`; nothing
 * synchronizes.
 * zero_opt_step_folded: as zero_opt_step with the global statistics, where the
 * fold of the n per-rank statistics at the DEVICE array `per_rank_dev` (rank
 * order) is taken on the device, bit-identical to zero_opt_fold_stats.  The
 * array is read when the step runs on `stream`.
 * Errors: as zero_opt_grad_stats / zero_opt_step, plus EINVAL (out_dev or
 * per_rank_dev NULL) and ERANGE (n outside [1, 2^20]). */
zero_status zero_opt_grad_stats_async(zero_opt_t h, int32_t rank, const zero_opt_buffers* bufs,
                                      void* stream, zero_opt_stats* out_dev);
zero_status zero_opt_step_folded(zero_opt_t h, int32_t rank, const zero_opt_buffers* bufs,
                                 void* stream, const zero_opt_stats* per_rank_dev, int32_t n);

/* One optimizer step of `rank`'s shard (steps a1..a7), asynchronous on
 * `stream`.  `global` (host, may be NULL) is the fold of all ranks'
 * zero_opt_grad_stats for these same gradients; NULL means this shard is the
 * whole world and its own statistics decide.  On overflow the step is skipped
 * (master, m, v, param16 and t untouched) and, on the hysteresis-th
 * overflow since the scale last changed, the scale is divided by
 * scale_factor, not below min_scale; otherwise AdamW is applied with the
 * update's learning rate (lr, or the WarmupLR value) and after scale_window
 * consecutive applied steps the scale is multiplied by scale_factor
 * ("DeepSpeed tutorial" §2.2, §2.4, §3.2).
 * Run tables: each call describes its buffers to the kernels in a small
 * table (72 bytes per run plus 8 per run and gradient buffer) kept in the
 * handle's arena.  A call whose buffers the handle has seen finds its table
 * there; for new buffers the table is copied in, ordered on `stream`, from
 * the arena's page-locked mirror.  Neither allocates, frees or synchronizes
 * the device, so fresh gradient buffers every step cost only that copy.  The
 * arena keeps up to 64 tables; the least recently used, or the ones a new
 * table's place overlaps, are dropped, and the host waits only if the copy
 * that filled the dropped bytes has not yet run (a host more than a whole
 * arena of new tables ahead of the device; zero_opt_get_counters counts
 * these waits).  Dropping is safe because calls on one handle are ordered:
 * the kernels that read a dropped table precede the copy that overwrites it.
 * Stream capture (CUDA graphs): a call with buffers the handle has already
 * stepped issues only its two kernel launches, with the decision on the
 * device, so it can be captured and the graph replayed every step; its table
 * is then kept for the life of the handle (the graph holds its address).  A
 * call with buffers never stepped before is refused under capture (ECUDA);
 * make one call with them first.
 * Both kernels are programmatic dependent launches: the first may be
 * scheduled while the kernel before it on `stream` still runs, and waits for
 * that kernel to complete, with all its writes visible, before it touches
 * memory.  So a caller sees plain stream order.
 * Errors: EINVAL (h/bufs/grads NULL, a NULL state or gradient pointer for a
 * non-empty shard, R or K < 1, R*K > 1024), ERANGE (rank outside [0, world);
 * a run table larger than the arena, or no room left beside the tables
 * that captures keep), ECUDA (no device, wrong current device, a launch
 * failure, or new buffers under stream capture). */
zero_status zero_opt_step(zero_opt_t h, int32_t rank, const zero_opt_buffers* bufs,
                          void* stream, const zero_opt_stats* global);

/* Statistics of a per-tensor list (multi-tensor apply): as
 * zero_opt_grad_stats, over the concatenation of the tensors in list order.
 * `rank` selects the loss-scaler replica. Synchronizes `stream`. */
zero_status zero_opt_grad_stats_tensors(zero_opt_t h, int32_t rank,
                                        const zero_opt_tensor_list* list,
                                        void* stream, zero_opt_stats* out);

/* One optimizer step over a per-tensor list: the same math as zero_opt_step,
 * with the L2 norm and the overflow flag taken over all tensors of the list
 * (plus the other ranks' through `global`).  Each tensor keeps its own
 * master/m/v/param16/gradient buffers.  Asynchronous on `stream`.
 * Errors: as zero_opt_step; EINVAL for n_tensors < 0 or a NULL tensors array
 * with n_tensors > 0. */
zero_status zero_opt_step_tensors(zero_opt_t h, int32_t rank,
                                  const zero_opt_tensor_list* list, void* stream,
                                  const zero_opt_stats* global);

/* Read `rank`'s loss-scaler state into *out (host).  Synchronizes `stream`.
 * Errors: EINVAL (NULL), ERANGE (rank), ECUDA. */
zero_status zero_opt_loss_scale(zero_opt_t h, int32_t rank, void* stream,
                                zero_opt_scaler_state* out);

/* Overwrite `rank`'s loss-scaler state (resume from a checkpoint), ordered on
 * `stream`.  Errors: EINVAL (NULL, scale <= 0, negative counters), ERANGE,
 * ECUDA. */
zero_status zero_opt_set_loss_scale(zero_opt_t h, int32_t rank, void* stream,
                                    const zero_opt_scaler_state* in);

/* Set the learning rate for subsequent steps (a scheduler such as WarmupLR,
 * "DeepSpeed tutorial" §3.2, changes it per step). Host only.
 * Errors: EINVAL (h NULL, lr < 0). */
zero_status zero_opt_set_lr(zero_opt_t h, double lr);

/* What the last step (on any rank) of this handle decided.  Synchronizes
 * `stream`. Errors: EINVAL, ECUDA. */
zero_status zero_opt_last_step(zero_opt_t h, void* stream, zero_opt_step_info* out);

/* Timing hook: subsequent steps (and statistics calls) of this handle record
 * the caller's CUDA events (cudaEvent_t, created by the caller; each may be
 * NULL) on the step's stream: ev_start before pass 1, ev_mid between pass 1
 * and pass 2, ev_end after pass 2 (after pass 1 when there is no pass 2).
 * Passing three NULLs turns the hook off.  The events measure each pass on
 * the stream it runs on.  Host only; records nothing by itself.
 * Errors: EINVAL (h NULL). */
zero_status zero_opt_set_events(zero_opt_t h, void* ev_start, void* ev_mid, void* ev_end);

/* Failure-detection test hook.  The next statistics pass of this handle that
 * stages a single gradient buffer through shared memory leaves one of its
 * copy barriers un-armed, so that the wait for it expires after its bound
 * (about a second).  The kernel then stops, waits (bounded) for its copies in
 * flight, and records a fault: that step is skipped without changing any
 * state, and zero_opt_last_step reports fault = 1.  Nothing hangs and the
 * context stays usable.  Host only; the hook arms one launch.
 * Errors: EINVAL (h NULL). */
zero_status zero_opt_inject_wait_fault(zero_opt_t h);

/* Kernels launched by this handle since creation (for launch accounting). */
zero_status zero_opt_launch_count(zero_opt_t h, int64_t* launches);

/* Accounting of a handle's launches and run tables. */
typedef struct zero_opt_counters {
  int64_t launches;         /* kernels launched since creation               */
  int64_t table_uploads;    /* run tables copied into the arena              */
  int64_t table_waits;      /* times the host waited for an earlier table
                               copy before reusing its arena bytes           */
  int64_t device_allocs;    /* device or page-locked allocations made after
                               zero_opt_create returned (none by design)     */
  int64_t device_frees;     /* frees made before zero_opt_destroy (none by
                               design)                                       */
  int64_t tables_cached;    /* run tables in the arena now (<= 64)           */
  int64_t tables_pinned;    /* of those, kept for captured CUDA graphs       */
  int64_t table_bytes;      /* size of the arena                             */
} zero_opt_counters;

/* Read the handle's counters into *out (host).  Host only.
 * Errors: EINVAL (NULL). */
zero_status zero_opt_get_counters(zero_opt_t h, zero_opt_counters* out);

/* ---------------------------------------------------------------------------
 * Sharded checkpoints.  A DeepSpeed engine saves one checkpoint per rank and
 * resumes from it under the same world size and stage; zero_to_fp32.py merges
 * the ZeRO shards into one full fp32 state dict ("DeepSpeed framework
 * interview answer" (algomooc.com), "训练与恢复边界").
 *
 * File format (little-endian): 8-byte magic "ZOPTSHD1", uint32 version (1),
 * uint32 reserved (0), the fields of zero_opt_ckpt_info in declaration order
 * (int64 numel, int32 world, int32 rank, int64 begin, int64 real_len, then
 * float scale, int32 last_skipped, int64 clean_steps, int64 t, int64
 * skipped_total, int32 overflows, int32 reserved), uint64 checksum of the
 * payload, then the payload: real_len
 * fp32 master weights, real_len fp32 m, real_len fp32 v.  Padding is not
 * stored.  The checksum is 64-bit FNV-1a over the payload taken as 8-byte
 * little-endian words (a trailing partial word zero-extended).
 * ------------------------------------------------------------------------- */
typedef struct zero_opt_ckpt_info {
  int64_t numel;            /* Ψ of the flat buffer                           */
  int32_t world;            /* N                                              */
  int32_t rank;             /* rank whose shard this is                       */
  int64_t begin;            /* first flat index of the shard (rank * S)       */
  int64_t real_len;         /* real elements stored (no padding)              */
  zero_opt_scaler_state scaler;
} zero_opt_ckpt_info;

/* Write one shard file from HOST arrays of info->real_len floats each.
 * Errors: EINVAL (NULL arguments; info not describing rank's shard of numel
 * over world; an I/O failure, with the system error in zero_opt_last_error()). */
zero_status zero_opt_ckpt_write(const char* path, const zero_opt_ckpt_info* info,
                                const float* master, const float* m, const float* v);

/* Read a shard file's header into *info and, for each non-NULL HOST array of
 * info->real_len floats, its payload; the checksum is verified whenever the
 * payload is read.  Errors: EINVAL (NULL path/info, unreadable file, bad magic
 * or version, size not matching the header, checksum mismatch). */
zero_status zero_opt_ckpt_read(const char* path, zero_opt_ckpt_info* info,
                               float* master, float* m, float* v);

/* Save `rank`'s shard: its DEVICE master, m and v (shard-local; the first
 * real_len elements are stored) and its loss-scaler replica.  Synchronizes
 * `stream`.  Errors: as zero_opt_ckpt_write, plus ERANGE (rank), ECUDA,
 * ENOTSUP (a master16 handle: its masters are in param16, see
 * zero_opt_save_shard16). */
zero_status zero_opt_save_shard(zero_opt_t h, int32_t rank, const float* master,
                                const float* m, const float* v, void* stream,
                                const char* path);

/* Save `rank`'s shard of a master16 handle: its DEVICE 16-bit parameters
 * (the master weights; the full padded buffer unless param16_shard_local),
 * m, v and its loss-scaler replica, in the same file format.  The masters
 * are stored widened to binary32, which is exact.  zero_opt_load_shard
 * therefore restores them bit for bit (NaN payloads included), and
 * zero_opt_consolidate_fp32 reads the files like any other.  Synchronizes
 * `stream`.  Errors: as zero_opt_save_shard, plus EINVAL (a handle without
 * master16). */
zero_status zero_opt_save_shard16(zero_opt_t h, int32_t rank, const void* param16,
                                  int32_t param16_shard_local, const float* m, const float* v,
                                  void* stream, const char* path);

/* Resume `rank`'s shard from a file written for the same numel, world and
 * rank: fills the DEVICE master, m and v (shard-local), restores the rank's
 * loss-scaler replica and, when param16 is non-NULL, rewrites the rank's
 * slice of the 16-bit parameter copy as the rounding of the restored master
 * weights (param16 is the full padded buffer unless param16_shard_local).
 * For a master16 handle `master` is not used and param16 is required: the
 * file's masters are written into param16.  That is exact for a file from
 * zero_opt_save_shard16; for a file of fp32 masters it rounds them to
 * nearest even.
 * Synchronizes `stream`.  Errors: EINVAL (file for another numel/world/rank,
 * unreadable or corrupt file, a NULL buffer), ERANGE, ECUDA. */
zero_status zero_opt_load_shard(zero_opt_t h, int32_t rank, float* master, float* m,
                                float* v, void* param16, int32_t param16_shard_local,
                                void* stream, const char* path);

/* zero_to_fp32: merge the shard files of one checkpoint (n_paths == world, in
 * any order) into the full fp32 master weights out[0..numel) (HOST), padding
 * dropped.  Every rank must appear exactly once and all files must agree on
 * numel and world.  Host only.  Errors: EINVAL (NULL, unreadable or corrupt
 * file, missing or duplicate rank, numel or world mismatch). */
zero_status zero_opt_consolidate_fp32(const char* const* paths, int32_t n_paths,
                                      int64_t numel, float* out);

/* Gradient statistics for callers that cannot allocate device memory.  (No
 * counterpart on the pages: this is a service of this library.)
 *
 * The same result as zero_opt_grad_stats for one shard -- the overflow flag
 * and the sum of squares of the binary32 sums of n_bufs 16-bit gradient
 * buffers of n elements each -- but with no handle and no allocation.  Some
 * callers may not call cudaMalloc: a runtime whose own allocator owns every
 * device byte, a process already at its memory limit, or a code path that
 * cannot afford the device-wide synchronization cudaMalloc may cause; a
 * handle (zero_opt_create) allocates a workspace, so those callers use this.
 *
 * grads: host array of n_bufs device pointers (fp16 or bf16 per grad_dtype),
 * summed in index order; n_bufs must be 1..64 (ERANGE beyond 64).  out: a
 * DEVICE pointer to one zero_opt_stats, written asynchronously on `stream`.
 * Its scratch is a fixed 12,544-byte array in the library's device image
 * (per-CTA partial sums for at most 1024 CTAs and a completion counter),
 * held by every GPU that loads the library until the process exits.  The
 * first call on a device looks up that array's device address (with that
 * device current) and keeps it for the life of the process; make that first
 * call before any stream capture, and do not use this entry point on a
 * device after cudaDeviceReset (or any other reset of its primary context)
 * in the same process: the kept address may then no longer name the array.
 * Every call shares the array, so calls that may overlap on the GPU
 * (different streams, or different host threads) race and must be
 * serialized by the caller.  This C function sees only pointers and cannot
 * check that each gradient buffer holds n elements of grad_dtype on the
 * current device, or that out points at 16 writable device bytes; the
 * caller must (the Python binding checks its tensors).  Errors: EINVAL (NULL grads/out, a NULL gradient pointer with
 * n > 0, n < 0, n_bufs < 1, bad dtype), ERANGE (n_bufs > 64), ECUDA. */
zero_status zero_opt_grad_stats_noalloc(const void* const* grads, int32_t n_bufs,
                                        int32_t grad_dtype, int64_t n, void* stream,
                                        zero_opt_stats* out);

/* ---------------------------------------------------------------------------
 * Offloaded step: the same per-shard step on HOST-resident state, computed by
 * a pool of CPU threads ("DeepSpeed tutorial" §4.3 CPU offload and
 * "DeepSpeed ZeRO引擎深入" 卸载策略: the optimizer states, and the
 * gradients, live in CPU memory and the update runs there, trading transfer
 * time for device memory).  No CUDA call is made; these functions work on a
 * machine without a GPU.  The results are those of zero_opt_step on the same
 * inputs: the same binary32 operation sequence per element, the same 16-bit
 * rounding, the same decisions (one shared implementation) and the same loss
 * scale sequence; only the sum of squares may differ from the device's, by
 * about 1e-13 relative or less (both are compensated sums, added in different
 * orders), and through the clip coefficient that can move the clipped
 * steps' results by a unit in their last place.
 *
 * zero_host_create: `n_threads` worker threads (<= 0: the number of hardware
 * threads; at most 1024), started here and kept until zero_host_destroy.
 * The handle keeps one loss-scaler replica per rank, initialised as
 * zero_opt_create does.  Errors: EINVAL (NULL cfg/out, invalid config),
 * ENOMEM.
 *
 * Buffers are zero_opt_buffers whose pointers are all HOST pointers (the
 * grads array and every gradient buffer, master, m, v, param16) with the same
 * meaning, lengths and indexing as for zero_opt_step; `stash` is ignored (the
 * sums are recomputed).  Calls on one handle must not overlap; the caller's
 * buffers must not be touched by other threads during a call.
 *
 * zero_host_grad_stats: statistics of the rank's shard (for a fold over ranks
 * with zero_opt_fold_stats).  zero_host_step: the step of `rank`; `global` as
 * in zero_opt_step (NULL: this shard's own statistics).  Both return when the
 * work is done.  zero_host_loss_scale / zero_host_set_loss_scale read and
 * replace a rank's scaler replica; zero_host_last_step reports the last step
 * of any rank.  Errors: EINVAL (NULL handle/buffers/pointer, R*K < 1),
 * ERANGE (rank outside [0, world), R*K > 1024). */
typedef struct zero_host_handle* zero_host_t;

zero_status zero_host_create(const zero_opt_config* cfg, int32_t n_threads, zero_host_t* out);
zero_status zero_host_destroy(zero_host_t h);
zero_status zero_host_threads(zero_host_t h, int32_t* n_threads);
zero_status zero_host_grad_stats(zero_host_t h, int32_t rank, const zero_opt_buffers* bufs,
                                 zero_opt_stats* out);
zero_status zero_host_step(zero_host_t h, int32_t rank, const zero_opt_buffers* bufs,
                           const zero_opt_stats* global);
/* The per-tensor list forms, as zero_opt_grad_stats_tensors and
 * zero_opt_step_tensors with host pointers: the statistics are those of the
 * concatenation in list order, and every tensor is updated with the one
 * decision.  The threads split the list by blocks of 1024 elements across
 * tensors.  Errors: as the device forms, with no ECUDA. */
zero_status zero_host_grad_stats_tensors(zero_host_t h, int32_t rank,
                                         const zero_opt_tensor_list* list, zero_opt_stats* out);
zero_status zero_host_step_tensors(zero_host_t h, int32_t rank, const zero_opt_tensor_list* list,
                                   const zero_opt_stats* global);
zero_status zero_host_loss_scale(zero_host_t h, int32_t rank, zero_opt_scaler_state* out);
zero_status zero_host_set_loss_scale(zero_host_t h, int32_t rank,
                                     const zero_opt_scaler_state* state);
zero_status zero_host_last_step(zero_host_t h, zero_opt_step_info* out);

/* Static string describing a status code; never NULL. */
const char* zero_opt_status_string(zero_status s);

/* Message of the last error on this thread (empty if none); never NULL. */
const char* zero_opt_last_error(void);

#ifdef __cplusplus
}
#endif
#endif
