// host_step.cpp -- the offloaded optimizer step: the per-shard step of
// zero_opt_step (reduce, overflow flag, sum of squares, decision, AdamW,
// 16-bit write-back) on host-resident buffers, computed by a pool of CPU
// threads.  Sources: "DeepSpeed tutorial" §4.3 (ZeRO-Offload keeps the
// optimizer states and gradients in CPU memory) and "DeepSpeed ZeRO引擎深入"
// 卸载策略 (the update moves to the CPU to relieve device memory).
//
// Work split: the shard's real elements are cut into one contiguous range per
// thread (multiples of kBlock elements).  Each thread reduces its range block
// by block in buffer order, and either accumulates the squares (statistics)
// or applies the update.  Partial sums of squares are folded in thread
// order, so a result depends only on the inputs and the thread count.
//
// Every binary32 operation of the update is a separate IEEE operation in
// round-to-nearest: this file is compiled without floating-point contraction
// (-ffp-contract=off) and without any fast-math option, so vectorised code
// computes exactly what the scalar source says.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <condition_variable>
#include <cstdint>
#include <cstring>
#include <functional>
#include <mutex>
#include <new>
#include <thread>
#include <vector>

#include "decide_core.h"
#include "host_cast.h"
#include "host_util.h"
#include "zero_opt.h"
#include "zero_opt_internal.h"

namespace {

using zo::fail;
using namespace zo::hc;

constexpr int64_t kBlock = 1024;  // elements reduced at a time per thread
constexpr int kMaxThreads = 1024;

// ------------------------------------------------------------------ threads
// A fixed set of workers; run(f) calls f(i) for i in [0, n) -- i = 0 on the
// calling thread -- and returns when every call has returned.
class Pool {
 public:
  explicit Pool(int n) : n_(n) {
    for (int i = 1; i < n; ++i) workers_.emplace_back([this, i] { loop(i); });
  }
  ~Pool() {
    {
      std::lock_guard<std::mutex> l(mu_);
      stop_ = true;
    }
    cv_.notify_all();
    for (auto& t : workers_) t.join();
  }
  int size() const { return n_; }
  void run(const std::function<void(int)>& f) {
    {
      std::lock_guard<std::mutex> l(mu_);
      job_ = &f;
      pending_ = n_ - 1;
      ++gen_;
    }
    cv_.notify_all();
    f(0);
    std::unique_lock<std::mutex> l(mu_);
    done_.wait(l, [this] { return pending_ == 0; });
    job_ = nullptr;
  }

 private:
  void loop(int i) {
    uint64_t seen = 0;
    for (;;) {
      const std::function<void(int)>* job;
      {
        std::unique_lock<std::mutex> l(mu_);
        cv_.wait(l, [&] { return stop_ || gen_ != seen; });
        if (stop_) return;
        seen = gen_;
        job = job_;
      }
      (*job)(i);
      std::lock_guard<std::mutex> l(mu_);
      if (--pending_ == 0) done_.notify_one();
    }
  }
  int n_;
  std::vector<std::thread> workers_;
  std::mutex mu_;
  std::condition_variable cv_, done_;
  const std::function<void(int)>* job_ = nullptr;
  uint64_t gen_ = 0;
  int pending_ = 0;
  bool stop_ = false;
};

// ------------------------------------------------------------------ 16-bit formats
// (host_cast.h: half_table, bf16_to_f32, f32_to_bf16, f32_to_f16)


// ------------------------------------------------------------------ sums of squares
// Compensated binary64 accumulation in four independent lanes.  The square of
// a binary32 value is exact in binary64; each lane adds groups of eight
// squares (a pairwise sum, a few units of 2^-53 of the group) into its
// (hi, lo) pair with Knuth's TwoSum, so the total stays within a few units of
// 2^-53 of the exact sum of squares, like the device's.  Lane l takes every
// fourth element, so the four lanes are the lanes of a vector.
struct SqSum {
  double hi[4] = {0, 0, 0, 0}, lo[4] = {0, 0, 0, 0};
  static inline void two_sum(double& hi, double& lo, double x) {
    const double t = hi + x;
    const double bp = t - hi;
    lo += (hi - (t - bp)) + (x - bp);
    hi = t;
  }
  static inline double sq(float x) { return (double)x * (double)x; }
  void add_block(const float* s, int64_t n) {
    int64_t j = 0;
    for (; j + 32 <= n; j += 32)
      for (int l = 0; l < 4; ++l) {  // lane l: elements j + l + 4k, k = 0..7
        const float* q = s + j + l;
        two_sum(hi[l], lo[l], ((sq(q[0]) + sq(q[4])) + (sq(q[8]) + sq(q[12]))) +
                                  ((sq(q[16]) + sq(q[20])) + (sq(q[24]) + sq(q[28]))));
      }
    for (; j < n; ++j) two_sum(hi[0], lo[0], sq(s[j]));
  }
  // fold into (h, l) in lane order
  void into(double& h, double& l) const {
    for (int k = 0; k < 4; ++k) {
      two_sum(h, l, hi[k]);
      two_sum(h, l, lo[k]);
    }
  }
};

// ------------------------------------------------------------------ the step
// One run of elements with its own buffers: a flat shard, or one tensor of a
// per-tensor list.
struct Job {
  const zero_opt_config* cfg;
  const uint16_t* const* g;  // per buffer: first element of the run
  int nbuf;
  int64_t n;                 // elements of the run
  float* master;
  float* m;
  float* v;
  uint16_t* p16;             // first element of the run
};

// The runs of a step and their blocks numbered across runs (run k's blocks
// are first[k] .. first[k + 1] - 1), so that threads split the whole step by
// block, whatever the run sizes.
struct Work {
  std::vector<Job> jobs;
  std::vector<int64_t> first;  // jobs.size() + 1 entries
  std::vector<const uint16_t*> gptrs;  // storage of every job's gradient pointers
  void number_blocks() {
    first.assign(1, 0);
    for (const Job& j : jobs) first.push_back(first.back() + (j.n + kBlock - 1) / kBlock);
  }
  int64_t blocks() const { return first.back(); }
};

// Reduced binary32 sums of elements [j0, j0 + len) in buffer order.
inline void reduce_block(const Job& jb, int64_t j0, int64_t len, float* s) {
  const bool half = jb.cfg->grad_dtype == ZERO_FP16;
  const float* tab = half ? half_table().v : nullptr;
  for (int64_t k = 0; k < len; ++k) s[k] = 0.0f;
  for (int b = 0; b < jb.nbuf; ++b) {
    const uint16_t* g = jb.g[b] + j0;
    if (half) {
      for (int64_t k = 0; k < len; ++k) s[k] = s[k] + tab[g[k]];
    } else {
      for (int64_t k = 0; k < len; ++k) s[k] = s[k] + bf16_to_f32(g[k]);
    }
  }
}

// Thread i of nt: calls f(job, lo, hi) for the element ranges of its
// contiguous share of the step's blocks, in block order.
template <typename F>
void for_share(const Work& w, int nt, int i, F&& f) {
  const int64_t per = (w.blocks() + nt - 1) / nt;
  const int64_t b0 = std::min(w.blocks(), (int64_t)i * per);
  const int64_t b1 = std::min(w.blocks(), (int64_t)(i + 1) * per);
  if (b0 >= b1) return;
  size_t k = (size_t)(std::upper_bound(w.first.begin(), w.first.end(), b0) - w.first.begin()) - 1;
  for (int64_t b = b0; b < b1; ++k) {
    const int64_t end = std::min(b1, w.first[k + 1]);
    if (end > b) {
      const Job& jb = w.jobs[k];
      const int64_t lo = (b - w.first[k]) * kBlock;
      f(jb, lo, std::min(jb.n, (end - w.first[k]) * kBlock));
      b = end;
    }
  }
}

struct Partial {
  double hi = 0.0, lo = 0.0;
  int nonfinite = 0;
  char pad[64 - 2 * sizeof(double) - sizeof(int)];
};

void stats_range(const Job& jb, int64_t lo, int64_t hi, SqSum* acc, int* bad) {
  alignas(64) float s[kBlock];
  for (int64_t j0 = lo; j0 < hi; j0 += kBlock) {
    const int64_t len = std::min(kBlock, hi - j0);
    reduce_block(jb, j0, len, s);
    int b = 0;
    for (int64_t k = 0; k < len; ++k) b |= !(std::fabs(s[k]) <= 3.40282347e38f);
    *bad |= b;
    acc->add_block(s, len);
  }
}

void update_range(const Job& jb, const zo::Decision& d, int64_t lo, int64_t hi) {
  alignas(64) float s[kBlock];
  alignas(64) float pw[kBlock];  // widened 16-bit masters (master16)
  const bool half16 = jb.cfg->param_dtype == ZERO_FP16;
  const bool m16 = jb.cfg->master16 != 0;
  const float* tab = half_table().v;
  const float coef = d.coef, b1 = d.b1, omb1 = d.omb1, b2 = d.b2, omb2 = d.omb2;
  const float isb2 = d.isb2, eps = d.eps, decay = d.decay, step_size = d.step_size;
  for (int64_t j0 = lo; j0 < hi; j0 += kBlock) {
    const int64_t len = std::min(kBlock, hi - j0);
    reduce_block(jb, j0, len, s);
    uint16_t* __restrict__ Q = jb.p16 + j0;
    // low-precision master weights: the 16-bit parameter, widened, is the
    // master; pw holds it for the block and is not stored back
    float* __restrict__ P = m16 ? pw : jb.master + j0;
    if (m16) {
      if (half16) {
        for (int64_t k = 0; k < len; ++k) pw[k] = tab[Q[k]];
      } else {
        for (int64_t k = 0; k < len; ++k) pw[k] = bf16_to_f32(Q[k]);
      }
    }
    float* __restrict__ M = jb.m + j0;
    float* __restrict__ V = jb.v + j0;
    for (int64_t k = 0; k < len; ++k) {
      const float g = s[k] * coef;
      const float mk = b1 * M[k] + omb1 * g;
      const float vk = b2 * V[k] + omb2 * (g * g);
      const float den = std::sqrt(vk) * isb2 + eps;
      float p = P[k] * decay;
      p = p - step_size * (mk / den);
      M[k] = mk;
      V[k] = vk;
      P[k] = p;
    }
    if (half16) {
      for (int64_t k = 0; k < len; ++k) Q[k] = f32_to_f16(P[k]);
    } else {
      for (int64_t k = 0; k < len; ++k) Q[k] = f32_to_bf16(P[k]);
    }
  }
}

}  // namespace

struct zero_host_handle {
  zero_opt_config cfg;
  std::vector<zo::RankState> ranks;
  zo::Decision last;
  Pool* pool = nullptr;
};

namespace {

zero_status check_rank(zero_host_t h, int32_t rank) {
  if (!h) return fail(ZERO_EINVAL, "handle is NULL");
  if (rank < 0 || rank >= h->cfg.world)
    return fail(ZERO_ERANGE, "rank %d outside [0, %d)", rank, h->cfg.world);
  return ZERO_OK;
}

// Validate `b` and describe the rank's shard as a one-run Work.
zero_status flat_work(zero_host_t h, int32_t rank, const zero_opt_buffers* b, bool need_state,
                      Work* w) {
  zero_status st = check_rank(h, rank);
  if (st != ZERO_OK) return st;
  if (!b) return fail(ZERO_EINVAL, "buffers is NULL");
  if (b->n_ranks < 1 || b->n_micro < 1) return fail(ZERO_EINVAL, "n_ranks and n_micro must be >= 1");
  const int64_t nbuf = (int64_t)b->n_ranks * b->n_micro;
  if (nbuf > zo::kMaxBufs)
    return fail(ZERO_ERANGE, "n_ranks*n_micro = %lld exceeds %d", (long long)nbuf, zo::kMaxBufs);
  if (!b->grads) return fail(ZERO_EINVAL, "grads array is NULL");
  int64_t begin, real, S;
  zo::shard_range(h->cfg.numel, h->cfg.world, rank, &begin, &real, &S);
  if (real > 0) {
    for (int64_t k = 0; k < nbuf; ++k)
      if (!b->grads[k]) return fail(ZERO_EINVAL, "gradient pointer %lld is NULL", (long long)k);
    if (need_state && ((!h->cfg.master16 && !b->master) || !b->m || !b->v || !b->param16))
      return fail(ZERO_EINVAL, "master (unless master16), m, v and param16 must not be NULL");
  }
  w->gptrs.resize((size_t)nbuf);
  const int64_t goff = b->grads_shard_local ? 0 : begin;
  for (int64_t k = 0; k < nbuf; ++k)
    w->gptrs[(size_t)k] = b->grads[k] ? static_cast<const uint16_t*>(b->grads[k]) + goff : nullptr;
  Job jb;
  jb.cfg = &h->cfg;
  jb.g = w->gptrs.data();
  jb.nbuf = (int)nbuf;
  jb.n = real;
  jb.master = h->cfg.master16 ? nullptr : b->master;
  jb.m = b->m;
  jb.v = b->v;
  jb.p16 = b->param16 ? static_cast<uint16_t*>(b->param16) + (b->param16_shard_local ? 0 : begin)
                      : nullptr;
  w->jobs.assign(1, jb);
  w->number_blocks();
  return ZERO_OK;
}

// Validate a per-tensor list and describe it as a Work of one run per tensor.
zero_status list_work(zero_host_t h, int32_t rank, const zero_opt_tensor_list* l,
                      bool need_state, Work* w) {
  zero_status st = check_rank(h, rank);
  if (st != ZERO_OK) return st;
  if (!l) return fail(ZERO_EINVAL, "tensor list is NULL");
  if (l->n_tensors < 0) return fail(ZERO_EINVAL, "n_tensors must be >= 0");
  if (l->n_tensors > 0 && !l->tensors) return fail(ZERO_EINVAL, "tensors is NULL");
  if (l->n_ranks < 1 || l->n_micro < 1) return fail(ZERO_EINVAL, "n_ranks and n_micro must be >= 1");
  const int64_t nbuf = (int64_t)l->n_ranks * l->n_micro;
  if (nbuf > zo::kMaxBufs)
    return fail(ZERO_ERANGE, "n_ranks*n_micro = %lld exceeds %d", (long long)nbuf, zo::kMaxBufs);
  w->gptrs.assign((size_t)(nbuf * l->n_tensors), nullptr);
  w->jobs.clear();
  for (int i = 0; i < l->n_tensors; ++i) {
    const zero_opt_tensor& t = l->tensors[i];
    if (t.numel < 0) return fail(ZERO_EINVAL, "tensor %d has numel < 0", i);
    if (t.numel == 0) continue;
    if (!t.grads) return fail(ZERO_EINVAL, "tensor %d: grads array is NULL", i);
    for (int64_t k = 0; k < nbuf; ++k) {
      if (!t.grads[k]) return fail(ZERO_EINVAL, "tensor %d: gradient pointer %lld is NULL", i,
                                   (long long)k);
      w->gptrs[(size_t)(i * nbuf + k)] = static_cast<const uint16_t*>(t.grads[k]);
    }
    if (need_state && ((!h->cfg.master16 && !t.master) || !t.m || !t.v || !t.param16))
      return fail(ZERO_EINVAL, "tensor %d: master (unless master16), m, v and param16 must "
                  "not be NULL", i);
    Job jb;
    jb.cfg = &h->cfg;
    jb.g = w->gptrs.data() + (size_t)(i * nbuf);
    jb.nbuf = (int)nbuf;
    jb.n = t.numel;
    jb.master = h->cfg.master16 ? nullptr : t.master;
    jb.m = t.m;
    jb.v = t.v;
    jb.p16 = static_cast<uint16_t*>(t.param16);
    w->jobs.push_back(jb);
  }
  w->number_blocks();
  return ZERO_OK;
}

zero_opt_stats work_stats(zero_host_t h, const Work& w) {
  const int nt = h->pool->size();
  std::vector<Partial> part((size_t)nt);
  h->pool->run([&](int i) {
    SqSum acc;
    int bad = 0;
    for_share(w, nt, i, [&](const Job& jb, int64_t lo, int64_t hi) {
      stats_range(jb, lo, hi, &acc, &bad);
    });
    acc.into(part[(size_t)i].hi, part[(size_t)i].lo);
    part[(size_t)i].nonfinite = bad;
  });
  double H = 0.0, L = 0.0;
  int bad = 0;
  for (const Partial& p : part) {
    SqSum::two_sum(H, L, p.hi);
    SqSum::two_sum(H, L, p.lo);
    bad |= p.nonfinite;
  }
  zero_opt_stats out;
  out.sumsq = H + L;
  out.nonfinite = bad;
  out.reserved = 0;
  return out;
}

// Statistics (or the given global ones), the decision, and the update of
// every run of `w`.
zero_status step_work(zero_host_t h, int32_t rank, const Work& w, double divisor,
                      double rk, const zero_opt_stats* global) {
  const zero_opt_stats s = global ? *global : work_stats(h, w);
  const zo::Hyper hp = zo::hyper_of(h->cfg, divisor > 0.0 ? divisor : rk);
  zo::RankState& rs = h->ranks[(size_t)rank];
  const zo::Decision d =
      zo::decide_core(hp, rs, s.sumsq, s.nonfinite ? 1 : 0,
                      [&hp](int64_t t, float* ss, float* isb2, float* decay) {
                        zo::step_scalars(hp, t, ss, isb2, decay);
                      });
  h->last = d;
  if (!d.skip && w.blocks() > 0) {
    const int nt = h->pool->size();
    h->pool->run([&](int i) {
      for_share(w, nt, i, [&](const Job& jb, int64_t lo, int64_t hi) {
        update_range(jb, d, lo, hi);
      });
    });
  }
  return ZERO_OK;
}

}  // namespace

extern "C" {

zero_status zero_host_create(const zero_opt_config* cfg, int32_t n_threads, zero_host_t* out) {
  if (!cfg || !out) return fail(ZERO_EINVAL, "cfg and out must not be NULL");
  zero_status st = zo::check_config(cfg);
  if (st != ZERO_OK) return st;
  int n = n_threads;
  if (n <= 0) n = (int)std::max(1u, std::thread::hardware_concurrency());
  n = std::min(n, kMaxThreads);
  zero_host_t h = new (std::nothrow) zero_host_handle();
  if (!h) return fail(ZERO_ENOMEM, "host handle");
  try {
    h->cfg = *cfg;
    h->ranks.resize((size_t)cfg->world);
    for (auto& r : h->ranks) {
      r.scale = (float)cfg->init_scale;
      r.last_skipped = 0;
      r.clean = 0;
      r.t = 0;
      r.skipped_total = 0;
      r.overflows = 0;
      r.reserved = 0;
    }
    std::memset(&h->last, 0, sizeof(h->last));
    half_table();
    h->pool = new Pool(n);
  } catch (...) {
    delete h;
    return fail(ZERO_ENOMEM, "host handle: allocation or thread start failed");
  }
  *out = h;
  return ZERO_OK;
}

zero_status zero_host_destroy(zero_host_t h) {
  if (!h) return fail(ZERO_EINVAL, "handle is NULL");
  delete h->pool;
  delete h;
  return ZERO_OK;
}

zero_status zero_host_threads(zero_host_t h, int32_t* n_threads) {
  if (!h || !n_threads) return fail(ZERO_EINVAL, "NULL argument");
  *n_threads = h->pool->size();
  return ZERO_OK;
}

zero_status zero_host_grad_stats(zero_host_t h, int32_t rank, const zero_opt_buffers* bufs,
                                 zero_opt_stats* out) {
  if (!out) return fail(ZERO_EINVAL, "out is NULL");
  Work w;
  zero_status st = flat_work(h, rank, bufs, false, &w);
  if (st != ZERO_OK) return st;
  *out = work_stats(h, w);
  return ZERO_OK;
}

zero_status zero_host_grad_stats_tensors(zero_host_t h, int32_t rank,
                                         const zero_opt_tensor_list* list, zero_opt_stats* out) {
  if (!out) return fail(ZERO_EINVAL, "out is NULL");
  Work w;
  zero_status st = list_work(h, rank, list, false, &w);
  if (st != ZERO_OK) return st;
  *out = work_stats(h, w);
  return ZERO_OK;
}

zero_status zero_host_step(zero_host_t h, int32_t rank, const zero_opt_buffers* bufs,
                           const zero_opt_stats* global) {
  Work w;
  zero_status st = flat_work(h, rank, bufs, true, &w);
  if (st != ZERO_OK) return st;
  return step_work(h, rank, w, bufs->divisor, (double)bufs->n_ranks * bufs->n_micro, global);
}

zero_status zero_host_step_tensors(zero_host_t h, int32_t rank, const zero_opt_tensor_list* list,
                                   const zero_opt_stats* global) {
  Work w;
  zero_status st = list_work(h, rank, list, true, &w);
  if (st != ZERO_OK) return st;
  return step_work(h, rank, w, list->divisor, (double)list->n_ranks * list->n_micro, global);
}
zero_status zero_host_loss_scale(zero_host_t h, int32_t rank, zero_opt_scaler_state* out) {
  zero_status st = check_rank(h, rank);
  if (st != ZERO_OK) return st;
  if (!out) return fail(ZERO_EINVAL, "out is NULL");
  std::memcpy(out, &h->ranks[(size_t)rank], sizeof(*out));
  return ZERO_OK;
}

zero_status zero_host_set_loss_scale(zero_host_t h, int32_t rank,
                                     const zero_opt_scaler_state* state) {
  zero_status st = check_rank(h, rank);
  if (st != ZERO_OK) return st;
  if (!state) return fail(ZERO_EINVAL, "state is NULL");
  if (!(state->scale > 0.0f) || state->clean_steps < 0 || state->t < 0 ||
      state->skipped_total < 0 || state->overflows < 0)
    return fail(ZERO_EINVAL, "scale must be > 0 and the counters >= 0");
  std::memcpy(&h->ranks[(size_t)rank], state, sizeof(*state));
  return ZERO_OK;
}

zero_status zero_host_last_step(zero_host_t h, zero_opt_step_info* out) {
  if (!h || !out) return fail(ZERO_EINVAL, "NULL argument");
  std::memcpy(out, &h->last, sizeof(*out));
  return ZERO_OK;
}

}  // extern "C"
