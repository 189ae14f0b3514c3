// zero_opt.cu -- host side of the C ABI declared in include/zero_opt.h.
//
// The host code validates arguments, turns the caller's buffers into a "plan"
// (a table of runs: the shard of a flat buffer or the tensors of a per-tensor
// list, each with its gradient pointers), and launches the two passes of
// kernels.cuh on the caller's stream.  Plan tables live in a device arena that
// zero_opt_create allocates with the rest of the handle: a table is copied in
// once (stream-ordered, from a pinned mirror of the arena) and found again by
// content, so a training loop that passes the same buffers every step uploads
// its table once, and one that passes new buffers every step uploads a few
// hundred bytes per step -- in neither case does a step allocate, free or
// synchronize.  The loss-scaler state of every rank lives in the handle's
// device workspace and is only advanced by the kernels, so a step never waits
// for the host.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "host_util.h"
#include "host_cast.h"
#include "kernels.cuh"

// Bytes of gradients at the top of a single buffer that pass 1 reads with an
// L2 evict_last policy for pass 2 (0: none).
#ifndef ZO_L2_KEEP_BYTES
#define ZO_L2_KEEP_BYTES (64ll << 20)
#endif


// Pass 2 of a shard of at least ZO_L1_MIN_TILES tiles prefers the largest L1
// (shared-memory carveout 0); smaller shards get ZO_SMALL_CARVEOUT percent.
#ifndef ZO_L1_MIN_TILES
#define ZO_L1_MIN_TILES 1024
#endif
#ifndef ZO_SMALL_CARVEOUT
#define ZO_SMALL_CARVEOUT 58
#endif
#include "zero_opt.h"


namespace {
thread_local std::string g_err;
}  // namespace

namespace zo {

zero_status fail(zero_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_err = buf;
  return s;
}

void shard_range(int64_t numel, int32_t world, int32_t rank, int64_t* begin,
                 int64_t* real_len, int64_t* shard_len) {
  const int64_t S = (numel + world - 1) / world;
  const int64_t b = (int64_t)rank * S;
  int64_t e = std::min(b + S, numel);
  if (e < b) e = b;
  *begin = b;
  *real_len = e - b;
  *shard_len = S;
}

// Validation of a configuration shared by the device and host handles.
zero_status check_config(const zero_opt_config* c) {
  if (c->numel < 0) return fail(ZERO_EINVAL, "numel must be >= 0");
  if (c->world < 1) return fail(ZERO_EINVAL, "world must be >= 1");
  if ((c->grad_dtype != ZERO_FP16 && c->grad_dtype != ZERO_BF16) ||
      (c->param_dtype != ZERO_FP16 && c->param_dtype != ZERO_BF16))
    return fail(ZERO_EINVAL, "dtype must be ZERO_FP16 or ZERO_BF16");
  if (!(c->lr >= 0.0)) return fail(ZERO_EINVAL, "lr must be >= 0");
  if (!(c->beta1 >= 0.0 && c->beta1 < 1.0) || !(c->beta2 >= 0.0 && c->beta2 < 1.0))
    return fail(ZERO_EINVAL, "betas must lie in [0, 1)");
  if (!(c->eps > 0.0)) return fail(ZERO_EINVAL, "eps must be > 0");
  if (!(c->weight_decay >= 0.0)) return fail(ZERO_EINVAL, "weight_decay must be >= 0");
  if (std::isnan(c->max_grad_norm)) return fail(ZERO_EINVAL, "max_grad_norm is NaN");
  if (!(c->init_scale > 0.0) || !(c->min_scale > 0.0))
    return fail(ZERO_EINVAL, "init_scale and min_scale must be > 0");
  if (!(c->scale_factor >= 1.0)) return fail(ZERO_EINVAL, "scale_factor must be >= 1");
  if (c->scale_window < 1) return fail(ZERO_EINVAL, "scale_window must be >= 1");
  if (c->bias_correction != 0 && c->bias_correction != 1)
    return fail(ZERO_EINVAL, "bias_correction must be 0 or 1");
  if (c->dynamic_scale != 0 && c->dynamic_scale != 1)
    return fail(ZERO_EINVAL, "dynamic_scale must be 0 or 1");
  if (c->hysteresis < 1) return fail(ZERO_EINVAL, "hysteresis must be >= 1");
  if (c->warmup_num_steps < 0 || !(c->warmup_min_lr >= 0.0) || !(c->warmup_max_lr >= 0.0))
    return fail(ZERO_EINVAL, "warm-up steps and learning rates must be >= 0");
  if (c->master16 != 0 && c->master16 != 1) return fail(ZERO_EINVAL, "master16 must be 0 or 1");
  if (c->table_kib < 0 || c->table_kib > (1 << 20))
    return fail(ZERO_EINVAL, "table_kib must lie in [0, 2^20]");
  return ZERO_OK;
}

// Kernel-side hyperparameters of a configuration, in binary64.
Hyper hyper_of(const zero_opt_config& c, double divisor) {
  Hyper hp;
  hp.lr = c.lr;
  hp.beta1 = c.beta1;
  hp.beta2 = c.beta2;
  hp.eps = c.eps;
  hp.wd = c.weight_decay;
  hp.max_norm = c.max_grad_norm;
  hp.divisor = divisor;
  hp.min_scale = c.min_scale;
  hp.factor = c.scale_factor;
  hp.window = c.scale_window;
  hp.bias_correction = c.bias_correction;
  hp.dynamic = c.dynamic_scale;
  hp.hysteresis = c.hysteresis;
  hp.warmup_min_lr = c.warmup_min_lr;
  hp.warmup_max_lr = c.warmup_max_lr;
  hp.warmup_num_steps = c.warmup_num_steps;
  hp.b1f = (float)hp.beta1;
  hp.omb1f = (float)(1.0 - hp.beta1);
  hp.b2f = (float)hp.beta2;
  hp.omb2f = (float)(1.0 - hp.beta2);
  hp.epsf = (float)hp.eps;
  hp.clip_on = hp.max_norm > 0.0 ? 1 : 0;
  return hp;
}

}  // namespace zo

namespace {

using zo::fail;

zero_status cuda_fail(cudaError_t e, const char* what) {
  return fail(ZERO_ECUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// One run of elements as the caller described it.
struct HostRun {
  float* master;
  float* m;
  float* v;
  void* p16;
  int64_t n;
  int64_t stash_off;
  std::vector<const void*> g;
};

// A run table in the handle's arena: [Seg x nseg][const void* x nseg*nbuf].
struct Plan {
  std::vector<unsigned char> blob;  // the table as uploaded (the cache key)
  uint64_t hash = 0;                // FNV-1a of blob, checked before the bytes
  int64_t off = -1;                 // byte offset in the arena (-1: empty table)
  int64_t size = 0;                 // bytes reserved in the arena
  int nseg = 0;
  int nbuf = 0;
  int64_t ntiles = 0;
  uint64_t stamp = 0;               // last use (least recently used is evicted first)
  int ev = -1;                      // the handle's event recorded after the upload
  bool pinned = false;              // used under stream capture: never evicted
};

// Run tables kept at once (one upload event each).
constexpr int kMaxPlans = 64;
// Arena bytes when the configuration leaves table_kib at 0.
constexpr int64_t kDefaultTableBytes = 1 << 20;
// Placement granularity of tables in the arena.
constexpr int64_t kTableAlign = 256;

uint64_t fnv1a(const std::vector<unsigned char>& b) {
  uint64_t x = 1469598103934665603ull;
  for (unsigned char c : b) {
    x ^= c;
    x *= 1099511628211ull;
  }
  return x;
}

}  // namespace

struct zero_opt_handle {
  zero_opt_config cfg;
  bool has_device = false;
  bool created = false;  // zero_opt_create has returned: allocations are counted
  int device = -1;
  int sms = 0;
  zo::Workspace* ws = nullptr;
  zo::RankState* ranks = nullptr;
  double* bc_table = nullptr;  // device bias corrections of steps 1..kBcSteps
  std::vector<double> bc_host;   // the same table, read back once at creation
  // Adam step counter of each rank as the host expects it: advanced by every
  // stepping launch as if it applies, and set exactly whenever a call reads or
  // writes the rank's scaler state.  A skipped step the host has not seen
  // leaves it ahead of the device; the scalar candidates cover seven of those.
  std::vector<int64_t> t_mirror;
  void* pinned = nullptr;  // page-locked staging for small reads
  int64_t launches = 0;
  uint64_t clock = 0;
  cudaEvent_t ev[3] = {nullptr, nullptr, nullptr};  // timing hook
  int32_t inject_wait_fault = 0;                      // test hook, one launch
  // run-table arena: device copy, page-locked host mirror, placement head
  unsigned char* table_dev = nullptr;
  unsigned char* table_host = nullptr;
  int64_t table_bytes = 0;
  int64_t table_head = 0;
  cudaEvent_t table_ev[kMaxPlans] = {};
  std::vector<int> free_ev;      // indices of table_ev not held by a plan
  std::vector<Plan*> plans;
  Plan empty_plan;               // the table of a shard with no elements
  int64_t table_uploads = 0;
  int64_t table_waits = 0;
  int64_t device_allocs = 0;     // allocations after creation (none by design)
  int64_t device_frees = 0;      // frees before destruction (none by design)
  std::vector<std::pair<const void*, int>> occ;  // kernel -> CTAs per SM
  std::mutex mu;
};

namespace {

constexpr size_t kPinnedBytes = 256;

void shard_of(const zero_opt_config& c, int rank, int64_t* begin, int64_t* real_end,
              int64_t* shard, int64_t* padded) {
  const int64_t S = (c.numel + c.world - 1) / c.world;
  const int64_t b = (int64_t)rank * S;
  int64_t e = std::min(b + S, c.numel);
  if (e < b) e = b;
  *begin = b;
  *real_end = e;
  *shard = S;
  *padded = S * c.world;
}

zero_status check_handle_rank(zero_opt_t h, int32_t rank) {
  if (!h) return fail(ZERO_EINVAL, "handle is NULL");
  if (rank < 0 || rank >= h->cfg.world)
    return fail(ZERO_ERANGE, "rank %d outside [0, %d)", rank, h->cfg.world);
  return ZERO_OK;
}

zero_status check_device(zero_opt_t h) {
  if (!h->has_device) return fail(ZERO_ECUDA, "no CUDA device for this handle");
  int cur = -1;
  cudaError_t e = cudaGetDevice(&cur);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (cur != h->device)
    return fail(ZERO_ECUDA, "current device %d is not the handle's device %d", cur, h->device);
  return ZERO_OK;
}

// Dynamic shared memory a kernel is launched with (the bulk-copy pass 1 stages
// its chunks there; everything else uses none).
size_t dyn_smem(const void* fn) {
  if (fn == reinterpret_cast<const void*>(zo::pass1_bulk_kernel<__half, 4>) ||
      fn == reinterpret_cast<const void*>(zo::pass1_bulk_kernel<__nv_bfloat16, 4>))
    return zo::bulk_smem_bytes(4);
  if (fn == reinterpret_cast<const void*>(zo::pass1_bulk_kernel<__half, 8>) ||
      fn == reinterpret_cast<const void*>(zo::pass1_bulk_kernel<__nv_bfloat16, 8>))
    return zo::bulk_smem_bytes(8);
  return 0;
}

int occupancy(zero_opt_t h, const void* fn) {
  for (auto& kv : h->occ)
    if (kv.first == fn) return kv.second;
  // the opt-in limit counts static + dynamic shared memory against 48 KiB, so
  // it is raised for every kernel that takes dynamic shared memory
  const size_t smem = dyn_smem(fn);
  if (smem > 0)
    cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, zo::kThreads, smem) != cudaSuccess ||
      n < 1)
    n = 1;
  h->occ.emplace_back(fn, n);
  return n;
}

bool run_is_vec(const HostRun& r, const float* stash) {
  if (!aligned16(r.master) || !aligned16(r.m) || !aligned16(r.v) || !aligned16(r.p16))
    return false;
  for (const void* g : r.g)
    if (!aligned16(g)) return false;
  if (stash && !aligned16(stash + r.stash_off)) return false;
  return true;
}

// Device allocations of a handle go through these two, so that any made after
// zero_opt_create (none, by design) show in zero_opt_get_counters.
cudaError_t handle_malloc(zero_opt_t h, void** p, size_t bytes) {
  if (h->created) h->device_allocs += 1;
  return cudaMalloc(p, bytes);
}
cudaError_t handle_malloc_host(zero_opt_t h, void** p, size_t bytes) {
  if (h->created) h->device_allocs += 1;
  return cudaMallocHost(p, bytes);
}
void handle_free(zero_opt_t h, void* p) {
  if (h->created) h->device_frees += 1;
  if (p) cudaFree(p);
}
void handle_free_host(zero_opt_t h, void* p) {
  if (h->created) h->device_frees += 1;
  if (p) cudaFreeHost(p);
}

// Make plan `p`'s arena bytes reusable: its upload must have left the pinned
// mirror (the host is about to overwrite it).  Kernels that read its device
// copy were enqueued before the caller's current call, which is ordered after
// them (calls on one handle are ordered), and so is the next upload.
zero_status retire_plan(zero_opt_t h, Plan* p) {
  if (p->ev >= 0) {
    cudaError_t e = cudaEventQuery(h->table_ev[p->ev]);
    if (e == cudaErrorNotReady) {
      h->table_waits += 1;
      e = cudaEventSynchronize(h->table_ev[p->ev]);
    }
    if (e != cudaSuccess) return cuda_fail(e, "run-table upload");
    h->free_ev.push_back(p->ev);
  }
  delete p;
  return ZERO_OK;
}

zero_status evict(zero_opt_t h, std::vector<Plan*>::iterator it) {
  Plan* p = *it;
  h->plans.erase(it);
  return retire_plan(h, p);
}

// Arena offset for a table of `size` bytes: from the placement head on (or
// from 0 when it does not fit before the end), skipping tables pinned by a
// stream capture; the tables it overlaps are evicted.
zero_status place(zero_opt_t h, int64_t size, int64_t* out) {
  int64_t start = h->table_head;
  bool wrapped = false;
  for (;;) {
    if (start + size > h->table_bytes) {
      if (wrapped)
        return fail(ZERO_ERANGE,
                    "run-table arena of %lld bytes is full: tables used under stream capture "
                    "hold it (raise zero_opt_config.table_kib)",
                    (long long)h->table_bytes);
      start = 0;
      wrapped = true;
    }
    int64_t skip_to = -1;
    for (const Plan* p : h->plans)
      if (p->pinned && p->off < start + size && start < p->off + p->size)
        skip_to = std::max(skip_to, p->off + p->size);
    if (skip_to < 0) break;
    start = skip_to;
  }
  for (auto it = h->plans.begin(); it != h->plans.end();) {
    Plan* p = *it;
    if (p->off < start + size && start < p->off + p->size) {
      zero_status st = evict(h, it);
      if (st != ZERO_OK) return st;
      it = h->plans.begin();   // erase invalidated the iterator; rescan
    } else {
      ++it;
    }
  }
  h->table_head = start + size;
  *out = start;
  return ZERO_OK;
}

// Serialize the runs into the device table layout; find the identical table
// in the arena or copy it in (ordered on `stream`).  Under stream capture a
// table that is found is pinned (the graph keeps its address); a new table is
// refused there, since placing it may need a host wait.
zero_status get_plan(zero_opt_t h, const std::vector<HostRun>& runs, int nbuf,
                     const float* stash, cudaStream_t stream, Plan** out) {
  const int nseg = (int)runs.size();
  if (nseg == 0) {
    *out = &h->empty_plan;
    return ZERO_OK;
  }
  std::vector<zo::Seg> segs(nseg);
  std::vector<const void*> gp;
  gp.reserve((size_t)nseg * nbuf);
  int64_t tile0 = 0;
  for (int i = 0; i < nseg; ++i) {
    const HostRun& r = runs[i];
    zo::Seg& s = segs[i];
    std::memset(&s, 0, sizeof(s));
    s.master = r.master;
    s.m = r.m;
    s.v = r.v;
    s.p16 = r.p16;
    s.n = r.n;
    s.tile0 = tile0;
    s.ntiles = (r.n + zo::kTile - 1) / zo::kTile;
    s.stash_off = r.stash_off;
    s.gbase = (int32_t)gp.size();
    s.vec = run_is_vec(r, stash) ? 1 : 0;
    tile0 += s.ntiles;
    for (const void* g : r.g) gp.push_back(g);
  }
  std::vector<unsigned char> blob(sizeof(zo::Seg) * nseg + sizeof(void*) * gp.size());
  std::memcpy(blob.data(), segs.data(), sizeof(zo::Seg) * nseg);
  std::memcpy(blob.data() + sizeof(zo::Seg) * nseg, gp.data(), sizeof(void*) * gp.size());
  const uint64_t hash = fnv1a(blob);
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing(stream, &cap);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamIsCapturing");
  const bool capturing = cap != cudaStreamCaptureStatusNone;

  std::lock_guard<std::mutex> lock(h->mu);
  h->clock += 1;
  for (Plan* p : h->plans) {
    if (p->hash == hash && p->nbuf == nbuf && p->nseg == nseg && p->blob == blob) {
      p->stamp = h->clock;
      if (capturing) p->pinned = true;
      *out = p;
      return ZERO_OK;
    }
  }
  if (capturing)
    return fail(ZERO_ECUDA,
                "these buffers were never stepped before the stream capture began: make one "
                "call with them outside the capture first (it copies their run table in)");
  const int64_t size = ((int64_t)blob.size() + kTableAlign - 1) / kTableAlign * kTableAlign;
  if (size > h->table_bytes)
    return fail(ZERO_ERANGE,
                "run table of %lld bytes (%d runs x %d gradient buffers) exceeds the handle's "
                "arena of %lld bytes (raise zero_opt_config.table_kib)",
                (long long)blob.size(), nseg, nbuf, (long long)h->table_bytes);
  if ((int)h->plans.size() >= kMaxPlans) {
    auto lru = h->plans.end();
    for (auto it = h->plans.begin(); it != h->plans.end(); ++it)
      if (!(*it)->pinned && (lru == h->plans.end() || (*it)->stamp < (*lru)->stamp)) lru = it;
    if (lru == h->plans.end())
      return fail(ZERO_ERANGE, "all %d run tables are pinned by stream captures", kMaxPlans);
    zero_status st = evict(h, lru);
    if (st != ZERO_OK) return st;
  }
  int64_t off = 0;
  zero_status st = place(h, size, &off);
  if (st != ZERO_OK) return st;
  Plan* p = new Plan;
  p->blob = std::move(blob);
  p->hash = hash;
  p->off = off;
  p->size = size;
  p->nseg = nseg;
  p->nbuf = nbuf;
  p->ntiles = tile0;
  p->stamp = h->clock;
  p->ev = h->free_ev.back();
  h->free_ev.pop_back();
  // The pinned mirror is not touched again until this copy has run (its event
  // is waited on before the bytes are reused).
  std::memcpy(h->table_host + off, p->blob.data(), p->blob.size());
  e = cudaMemcpyAsync(h->table_dev + off, h->table_host + off, p->blob.size(),
                      cudaMemcpyHostToDevice, stream);
  if (e == cudaSuccess) e = cudaEventRecord(h->table_ev[p->ev], stream);
  if (e != cudaSuccess) {
    h->free_ev.push_back(p->ev);
    delete p;
    return cuda_fail(e, "run-table upload");
  }
  h->table_uploads += 1;
  h->plans.push_back(p);
  *out = p;
  return ZERO_OK;
}

using Pass1Fn = void (*)(zo::Pass1Args);
using Pass2Fn = void (*)(zo::Pass2Args);

// Tiles from which a single-buffer shard takes 8-tile bulk chunks (about 410M
// elements: at least ~60 chunks per CTA, so the coarser unit costs little
// balance).
constexpr int64_t kBigChunkTiles = 200000;

Pass1Fn pick_pass1(int gdt, bool stash, bool one, int64_t ntiles) {
  // a single buffer is never stashed (the stash needs more than four)
  if (one) {
    const bool big = ntiles >= kBigChunkTiles;
    if (gdt == ZERO_FP16)
      return big ? zo::pass1_bulk_kernel<__half, 8> : zo::pass1_bulk_kernel<__half, 4>;
    return big ? zo::pass1_bulk_kernel<__nv_bfloat16, 8> : zo::pass1_bulk_kernel<__nv_bfloat16, 4>;
  }
  if (gdt == ZERO_FP16)
    return stash ? zo::pass1_multi_kernel<__half, true> : zo::pass1_multi_kernel<__half, false>;
  return stash ? zo::pass1_multi_kernel<__nv_bfloat16, true>
               : zo::pass1_multi_kernel<__nv_bfloat16, false>;
}

template <typename GT, typename PT, bool M16>
Pass2Fn pick_pass2_src(int src) {
  if (src == -1) return zo::pass2_kernel<GT, PT, -1, M16>;
  if (src == 1) return zo::pass2_kernel<GT, PT, 1, M16>;
  return zo::pass2_kernel<GT, PT, 0, M16>;
}

template <typename GT, typename PT>
Pass2Fn pick_pass2_t(int src, bool m16) {
  return m16 ? pick_pass2_src<GT, PT, true>(src) : pick_pass2_src<GT, PT, false>(src);
}

Pass2Fn pick_pass2(int gdt, int pdt, int src, bool m16) {
  if (gdt == ZERO_FP16)
    return pdt == ZERO_FP16 ? pick_pass2_t<__half, __half>(src, m16)
                            : pick_pass2_t<__half, __nv_bfloat16>(src, m16);
  return pdt == ZERO_FP16 ? pick_pass2_t<__nv_bfloat16, __half>(src, m16)
                          : pick_pass2_t<__nv_bfloat16, __nv_bfloat16>(src, m16);
}


// Pass 2's shared-memory carveout preference for a shard of `ntiles` tiles.
// On large shards the largest L1 measured 10.42 -> 10.34 ms per step on the
// 2.27B-parameter list and 4.559 -> 4.535 ms on the 1B-parameter shard.  On a
// 1M-parameter shard (489 tiles) it cost 14.1 -> 18.6 us, since the pass-2
// CTAs then cannot wait on the SMs pass 1 still holds; left to the CUDA driver's
// choice the same step took 14.1, 15.5, 16.2 or 18.2 us from one process to
// the next, while 58% (room for the four resident pass-1 CTAs of a small
// shard) gave 14.33 us in every process.  The attribute belongs to the kernel
// function (process-wide), so it is set on first use and again only when the
// wanted value changes (per device: the attribute is set in the current
// device's context); a stale value costs time, never correctness.
void prefer_l1(int device, const void* fn, int64_t ntiles) {
  struct Entry {
    int device;
    const void* fn;
    int value;
  };
  static std::mutex mu;
  static std::vector<Entry> set;
  const int want = ntiles >= ZO_L1_MIN_TILES ? 0 : ZO_SMALL_CARVEOUT;
  std::lock_guard<std::mutex> lock(mu);
  for (Entry& e : set) {
    if (e.device == device && e.fn == fn) {
      if (e.value != want &&
          cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout, want) ==
              cudaSuccess)
        e.value = want;
      return;
    }
  }
  if (cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout, want) != cudaSuccess)
    return;
  set.push_back({device, fn, want});
}

// `dependent`: launched as a programmatic dependent of the previous kernel on
// the stream (pass 2 after pass 1): it may start while that kernel ends and
// waits for its completion itself (griddepcontrol.wait) before using results.
zero_status launch_kernel(zero_opt_t h, const void* fn, int grid, void* args,
                          cudaStream_t stream, bool dependent = false) {
  void* params[] = {args};
  cudaLaunchConfig_t lc;
  std::memset(&lc, 0, sizeof(lc));
  lc.gridDim = dim3(grid);
  lc.blockDim = dim3(zo::kThreads);
  lc.dynamicSmemBytes = dyn_smem(fn);
  lc.stream = stream;
  cudaLaunchAttribute attr[1];
  if (dependent && ZO_PDL) {
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    lc.attrs = attr;
    lc.numAttrs = 1;
  }
  cudaError_t e = cudaLaunchKernelExC(&lc, fn, params);
  if (e != cudaSuccess) return cuda_fail(e, "cudaLaunchKernelExC");
  h->launches += 1;
  return ZERO_OK;
}

// Pass 1 (always: it takes the decision), then pass 2 unless only the
// statistics are wanted.
// `global`: host statistics (kStepGlobal) or, for kStepGlobalDev, `g_n`
// per-rank device statistics; `stats_out`: device copy of a statistics-only
// result, or NULL.
zero_status run(zero_opt_t h, int32_t rank, const std::vector<HostRun>& runs, int nbuf,
                double divisor, float* stash, void* stream_v, zo::Mode mode,
                const zero_opt_stats* global, int32_t g_n = 0,
                zero_opt_stats* stats_out = nullptr) {
  cudaStream_t stream = static_cast<cudaStream_t>(stream_v);
  float* use_stash = (stash != nullptr && nbuf > 4) ? stash : nullptr;
  Plan* plan = nullptr;
  zero_status st = get_plan(h, runs, nbuf, use_stash, stream, &plan);
  if (st != ZERO_OK) return st;

  const unsigned char* table = plan->off >= 0 ? h->table_dev + plan->off : nullptr;
  const zo::Seg* segs = reinterpret_cast<const zo::Seg*>(table);
  const void* const* gptrs =
      table ? reinterpret_cast<const void* const*>(table + sizeof(zo::Seg) * plan->nseg)
            : nullptr;

  zo::Pass1Args a1;
  std::memset(&a1, 0, sizeof(a1));
  a1.segs = segs;
  a1.gptrs = gptrs;
  a1.nseg = plan->nseg;
  a1.nbuf = nbuf;
  // With the global statistics given and nothing to stash, pass 1 only
  // decides: one CTA, no tiles.
  const bool reduce =
      !((mode == zo::kStepGlobal || mode == zo::kStepGlobalDev) && use_stash == nullptr);
  a1.ntiles = reduce ? plan->ntiles : 0;
  a1.stash = use_stash;
  a1.mode = mode;
  a1.rank = rank;
  if (global && mode == zo::kStepGlobal) {
    a1.g_sumsq = global->sumsq;
    a1.g_nonfinite = global->nonfinite ? 1 : 0;
  }
  if (mode == zo::kStepGlobalDev) {
    a1.g_dev = global;
    a1.g_n = g_n;
  }
  a1.stats_out = stats_out;
  a1.hp = zo::hyper_of(h->cfg, divisor);
  a1.ws = h->ws;
  a1.ranks = h->ranks;
  a1.bc_table = h->bc_table;
  a1.inject_wait_fault = h->inject_wait_fault;
  h->inject_wait_fault = 0;
  // The gradients pass 2 reads first (the top of a single buffer, where its
  // reverse walk starts) are read by pass 1 with an L2 evict_last policy, up
  // to ZO_L2_KEEP_BYTES; pass 2 returns their lines to evict_normal.  Only for
  // steps over one 128-byte aligned run of one buffer.
  a1.keep_tile0 = plan->ntiles;
  if (ZO_L2_KEEP_BYTES > 0 && mode != zo::kStatsOnly && a1.ntiles > 0 && nbuf == 1 &&
      use_stash == nullptr && runs.size() == 1 &&
      (reinterpret_cast<uintptr_t>(runs[0].g[0]) & 127) == 0) {
    const int64_t keep = (int64_t)ZO_L2_KEEP_BYTES / (zo::kTile * 2);
    a1.keep_tile0 = std::max<int64_t>(0, plan->ntiles - keep);
  }

  // The update scalars of the step numbers this rank's step can have: the one
  // the host expects (its mirror + 1) and the seven below it (steps skipped
  // since the host last read the rank's state).  Computed here in binary64
  // exactly as the device would, from the device's own bias-correction table,
  // so that pass 1's scalar CTA only picks the one that applies.
  a1.inv_d = 1.0 / divisor;
  if (mode != zo::kStatsOnly) {
    const int64_t t_pred = h->t_mirror[rank] + 1;
    if (t_pred >= 1 && t_pred <= zo::kBcSteps) {
      a1.cand_t0 = t_pred;
      a1.ncand = (int32_t)std::min<int64_t>(zo::kScalarCands, t_pred);
      for (int j = 0; j < a1.ncand; ++j) {
        const int64_t t = t_pred - j;
        zo::step_scalars_bc(a1.hp, t, h->bc_host[2 * (t - 1)], h->bc_host[2 * (t - 1) + 1],
                            &a1.cand[j][0], &a1.cand[j][1], &a1.cand[j][2]);
      }
    }
    h->t_mirror[rank] = t_pred;
  }

  const void* f1 = reinterpret_cast<const void*>(
      pick_pass1(h->cfg.grad_dtype, use_stash != nullptr, nbuf == 1, plan->ntiles));
  // Every step launch gets one extra CTA that computes the next step's update
  // scalars (binary64 pow) while the others stream, so the decision at the
  // end of the launch does none; it takes one of the resident slots so that
  // every CTA runs at once.
  a1.scalar_cta = mode != zo::kStatsOnly ? 1 : 0;
  // work units: tiles, or the bulk kernel's chunks of 4 or 8 tiles
  int64_t units = a1.ntiles;
  if (nbuf == 1 && use_stash == nullptr) {
    const int64_t ct = plan->ntiles >= kBigChunkTiles ? 8 : 4;
    units = (a1.ntiles + ct - 1) / ct;
  }
  int64_t g1 = (int64_t)occupancy(h, f1) * h->sms - a1.scalar_cta;
  g1 = std::min<int64_t>(g1, std::max<int64_t>(units, 1));
  g1 = std::max<int64_t>(std::min<int64_t>(g1, zo::kMaxCtas - 1), 1) + a1.scalar_cta;
  if (h->ev[0]) cudaEventRecord(h->ev[0], stream);
  st = launch_kernel(h, f1, (int)g1, &a1, stream, ZO_PDL_PASS1 && h->ev[0] == nullptr);
  if (h->ev[1]) cudaEventRecord(h->ev[1], stream);
  if (st != ZERO_OK || mode == zo::kStatsOnly || plan->ntiles == 0) {
    if (h->ev[2]) cudaEventRecord(h->ev[2], stream);
    return st;
  }

  zo::Pass2Args a2;
  std::memset(&a2, 0, sizeof(a2));
  a2.segs = segs;
  a2.gptrs = gptrs;
  a2.nseg = plan->nseg;
  a2.nbuf = nbuf;
  a2.ntiles = plan->ntiles;
  a2.stash = use_stash;
  a2.dec = &h->ws->dec;
  a2.keep_tile0 = a1.keep_tile0;
  const int src = use_stash ? -1 : (nbuf == 1 ? 1 : 0);
  const void* f2 = reinterpret_cast<const void*>(
      pick_pass2(h->cfg.grad_dtype, h->cfg.param_dtype, src, h->cfg.master16 != 0));
  int64_t g2 = (int64_t)occupancy(h, f2) * h->sms;
  g2 = std::min<int64_t>(g2, plan->ntiles);
  prefer_l1(h->device, f2, plan->ntiles);
  // with the timing hook an event sits between the passes, and pass 2 is
  // an ordinary launch
  st = launch_kernel(h, f2, (int)g2, &a2, stream, h->ev[1] == nullptr);
  if (h->ev[2]) cudaEventRecord(h->ev[2], stream);
  return st;
}

// ---- turning the caller's descriptions into runs

zero_status check_grads(const void* const* grads, int nbuf, bool need_nonnull) {
  if (!grads) return fail(ZERO_EINVAL, "grads array is NULL");
  if (need_nonnull)
    for (int b = 0; b < nbuf; ++b)
      if (!grads[b]) return fail(ZERO_EINVAL, "gradient pointer %d is NULL", b);
  return ZERO_OK;
}

zero_status check_rk(int32_t R, int32_t K) {
  if (R < 1 || K < 1) return fail(ZERO_EINVAL, "n_ranks and n_micro must be >= 1");
  if ((int64_t)R * K > zo::kMaxBufs)
    return fail(ZERO_EINVAL, "n_ranks * n_micro must be <= %d", zo::kMaxBufs);
  return ZERO_OK;
}

zero_status flat_runs(zero_opt_t h, int32_t rank, const zero_opt_buffers* b,
                      std::vector<HostRun>* runs, int* nbuf, double* divisor) {
  if (!b) return fail(ZERO_EINVAL, "buffers are NULL");
  zero_status st = check_rk(b->n_ranks, b->n_micro);
  if (st != ZERO_OK) return st;
  const int nb = b->n_ranks * b->n_micro;
  int64_t begin, end, S, P;
  shard_of(h->cfg, rank, &begin, &end, &S, &P);
  const int64_t n = end - begin;
  st = check_grads(b->grads, nb, n > 0);
  if (st != ZERO_OK) return st;
  const bool m16 = h->cfg.master16 != 0;
  if (n > 0 && ((!m16 && !b->master) || !b->m || !b->v || !b->param16))
    return fail(ZERO_EINVAL, "master (unless master16), m, v and param16 must be non-NULL");
  *nbuf = nb;
  *divisor = b->divisor > 0.0 ? b->divisor : (double)nb;
  runs->clear();
  if (n == 0) return ZERO_OK;
  HostRun r;
  r.master = m16 ? nullptr : b->master;
  r.m = b->m;
  r.v = b->v;
  r.p16 = static_cast<unsigned char*>(b->param16) + (b->param16_shard_local ? 0 : begin * 2);
  r.n = n;
  r.stash_off = 0;
  const int64_t goff = b->grads_shard_local ? 0 : begin * 2;
  for (int i = 0; i < nb; ++i)
    r.g.push_back(static_cast<const unsigned char*>(b->grads[i]) + goff);
  runs->push_back(std::move(r));
  return ZERO_OK;
}

zero_status list_runs(const zero_opt_tensor_list* l, bool m16, std::vector<HostRun>* runs,
                      int* nbuf, double* divisor) {
  if (!l) return fail(ZERO_EINVAL, "tensor list is NULL");
  if (l->n_tensors < 0) return fail(ZERO_EINVAL, "n_tensors must be >= 0");
  if (l->n_tensors > 0 && !l->tensors) return fail(ZERO_EINVAL, "tensors array is NULL");
  zero_status st = check_rk(l->n_ranks, l->n_micro);
  if (st != ZERO_OK) return st;
  const int nb = l->n_ranks * l->n_micro;
  runs->clear();
  int64_t off = 0;
  for (int i = 0; i < l->n_tensors; ++i) {
    const zero_opt_tensor& t = l->tensors[i];
    if (t.numel < 0) return fail(ZERO_EINVAL, "tensor %d has numel < 0", i);
    if (t.numel > 0) {
      if ((!m16 && !t.master) || !t.m || !t.v || !t.param16)
        return fail(ZERO_EINVAL,
                    "tensor %d: master (unless master16), m, v and param16 must be non-NULL", i);
      st = check_grads(t.grads, nb, true);
      if (st != ZERO_OK) return st;
      HostRun r;
      r.master = m16 ? nullptr : t.master;
      r.m = t.m;
      r.v = t.v;
      r.p16 = t.param16;
      r.n = t.numel;
      r.stash_off = off;
      for (int b = 0; b < nb; ++b) r.g.push_back(t.grads[b]);
      runs->push_back(std::move(r));
    }
    off += t.numel;
  }
  *nbuf = nb;
  *divisor = l->divisor > 0.0 ? l->divisor : (double)nb;
  return ZERO_OK;
}

zero_status read_small(zero_opt_t h, const void* dev_src, size_t bytes, void* stream_v,
                       void* out) {
  cudaStream_t stream = static_cast<cudaStream_t>(stream_v);
  cudaError_t e = cudaMemcpyAsync(h->pinned, dev_src, bytes, cudaMemcpyDeviceToHost, stream);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyAsync");
  e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  std::memcpy(out, h->pinned, bytes);
  return ZERO_OK;
}

}  // namespace

// ====================================================================== ABI

extern "C" {

zero_status zero_opt_config_default(zero_opt_config* c) {
  if (!c) return fail(ZERO_EINVAL, "cfg is NULL");
  std::memset(c, 0, sizeof(*c));
  c->numel = 0;
  c->world = 1;
  c->grad_dtype = ZERO_FP16;
  c->param_dtype = ZERO_FP16;
  c->bias_correction = 1;
  c->lr = 2e-5;
  c->beta1 = 0.9;
  c->beta2 = 0.999;
  c->eps = 1e-8;
  c->weight_decay = 0.01;
  c->max_grad_norm = 0.0;
  c->dynamic_scale = 1;
  c->hysteresis = 2;
  c->init_scale = 65536.0;
  c->min_scale = 1.0;
  c->scale_factor = 2.0;
  c->scale_window = 1000;
  return ZERO_OK;
}

zero_status zero_opt_create(const zero_opt_config* cfg, zero_opt_t* out) {
  if (!out) return fail(ZERO_EINVAL, "out is NULL");
  *out = nullptr;
  if (!cfg) return fail(ZERO_EINVAL, "cfg is NULL");
  zero_status st = zo::check_config(cfg);
  if (st != ZERO_OK) return st;
  zero_opt_handle* h = new (std::nothrow) zero_opt_handle;
  if (!h) return fail(ZERO_ENOMEM, "handle allocation failed");
  h->cfg = *cfg;
  int count = 0;
  if (cudaGetDeviceCount(&count) != cudaSuccess || count < 1) {
    cudaGetLastError();  // clear the sticky "no device" error
    *out = h;            // host-only handle
    return ZERO_OK;
  }
  cudaError_t e = cudaGetDevice(&h->device);
  if (e == cudaSuccess)
    e = cudaDeviceGetAttribute(&h->sms, cudaDevAttrMultiProcessorCount, h->device);
  const size_t ws_bytes = sizeof(zo::Workspace) + sizeof(zo::RankState) * (size_t)cfg->world;
  void* ws = nullptr;
  if (e == cudaSuccess) e = handle_malloc(h, &ws, ws_bytes);
  if (e != cudaSuccess) {
    delete h;
    return e == cudaErrorMemoryAllocation ? fail(ZERO_ENOMEM, "workspace allocation failed")
                                          : cuda_fail(e, "zero_opt_create");
  }
  h->ws = static_cast<zo::Workspace*>(ws);
  h->ranks = reinterpret_cast<zo::RankState*>(static_cast<unsigned char*>(ws) +
                                              sizeof(zo::Workspace));
  std::vector<unsigned char> init(ws_bytes, 0);
  zo::RankState* r0 =
      reinterpret_cast<zo::RankState*>(init.data() + sizeof(zo::Workspace));
  for (int r = 0; r < cfg->world; ++r) {
    r0[r].scale = (float)cfg->init_scale;
    r0[r].last_skipped = 0;
    r0[r].clean = 0;
    r0[r].t = 0;
    r0[r].skipped_total = 0;
    r0[r].overflows = 0;
    r0[r].reserved = 0;
  }
  e = cudaMemcpy(ws, init.data(), ws_bytes, cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = handle_malloc_host(h, &h->pinned, kPinnedBytes);
  if (e == cudaSuccess)
    e = handle_malloc(h, reinterpret_cast<void**>(&h->bc_table),
                      sizeof(double) * 2 * zo::kBcSteps);
  // the run-table arena and its page-locked mirror: every table a step needs
  // is placed here, so no step allocates
  h->table_bytes = cfg->table_kib > 0 ? (int64_t)cfg->table_kib * 1024 : kDefaultTableBytes;
  if (e == cudaSuccess)
    e = handle_malloc(h, reinterpret_cast<void**>(&h->table_dev), (size_t)h->table_bytes);
  if (e == cudaSuccess)
    e = handle_malloc_host(h, reinterpret_cast<void**>(&h->table_host), (size_t)h->table_bytes);
  for (int i = 0; i < kMaxPlans && e == cudaSuccess; ++i) {
    e = cudaEventCreateWithFlags(&h->table_ev[i], cudaEventDisableTiming);
    if (e == cudaSuccess) h->free_ev.push_back(kMaxPlans - 1 - i);
  }
  if (e == cudaSuccess) {
    zo::BcTableArgs ta;
    ta.table = h->bc_table;
    ta.beta1 = cfg->beta1;
    ta.beta2 = cfg->beta2;
    void* params[] = {&ta};
    e = cudaLaunchKernel(reinterpret_cast<const void*>(zo::bc_table_kernel),
                         dim3((unsigned)((zo::kBcSteps + zo::kThreads - 1) / zo::kThreads)),
                         dim3(zo::kThreads), params, 0, nullptr);
    // ready before any stream, blocking or not, can use the handle
    if (e == cudaSuccess) e = cudaStreamSynchronize(nullptr);
  }
  if (e == cudaSuccess) {
    // the host computes the update scalars it supplies from these very values
    h->bc_host.resize(2 * (size_t)zo::kBcSteps);
    e = cudaMemcpy(h->bc_host.data(), h->bc_table, sizeof(double) * 2 * zo::kBcSteps,
                   cudaMemcpyDeviceToHost);
  }
  h->t_mirror.assign((size_t)cfg->world, 0);
  if (e != cudaSuccess) {
    for (cudaEvent_t ev : h->table_ev)
      if (ev) cudaEventDestroy(ev);
    handle_free(h, h->table_dev);
    handle_free_host(h, h->table_host);
    handle_free(h, h->bc_table);
    handle_free_host(h, h->pinned);
    handle_free(h, ws);
    delete h;
    return e == cudaErrorMemoryAllocation ? fail(ZERO_ENOMEM, "zero_opt_create: out of memory")
                                          : cuda_fail(e, "zero_opt_create");
  }
  h->has_device = true;
  h->created = true;
  *out = h;
  return ZERO_OK;
}

zero_status zero_opt_destroy(zero_opt_t h) {
  if (!h) return ZERO_OK;
  if (h->has_device) {
    int prev = -1;
    cudaGetDevice(&prev);
    cudaSetDevice(h->device);
    cudaDeviceSynchronize();
    h->created = false;  // the frees of destruction are not counted
    for (Plan* p : h->plans) delete p;
    for (cudaEvent_t ev : h->table_ev)
      if (ev) cudaEventDestroy(ev);
    handle_free(h, h->table_dev);
    handle_free_host(h, h->table_host);
    handle_free(h, h->ws);
    handle_free(h, h->bc_table);
    handle_free_host(h, h->pinned);
    if (prev >= 0) cudaSetDevice(prev);
  }
  delete h;
  return ZERO_OK;
}

zero_status zero_opt_shard_bounds(zero_opt_t h, int32_t rank, int64_t* begin,
                                  int64_t* real_end, int64_t* shard_len,
                                  int64_t* padded_numel) {
  zero_status st = check_handle_rank(h, rank);
  if (st != ZERO_OK) return st;
  int64_t b, e, s, p;
  shard_of(h->cfg, rank, &b, &e, &s, &p);
  if (begin) *begin = b;
  if (real_end) *real_end = e;
  if (shard_len) *shard_len = s;
  if (padded_numel) *padded_numel = p;
  return ZERO_OK;
}

zero_status zero_opt_memory_bytes(int64_t numel, int32_t world, int32_t stage,
                                  int64_t* bytes) {
  if (!bytes) return fail(ZERO_EINVAL, "bytes is NULL");
  if (numel < 0 || world < 1) return fail(ZERO_EINVAL, "numel must be >= 0 and world >= 1");
  if (stage < 0 || stage > 3) return fail(ZERO_ERANGE, "stage must be 0..3");
  const int64_t S = (numel + world - 1) / world;
  // 2 bytes of 16-bit parameters, 2 of 16-bit gradients, 12 of fp32 state.
  const int64_t params = stage >= 3 ? 2 * S : 2 * numel;
  const int64_t grads = stage >= 2 ? 2 * S : 2 * numel;
  const int64_t state = stage >= 1 ? 12 * S : 12 * numel;
  *bytes = params + grads + state;
  return ZERO_OK;
}

zero_status zero_opt_grad_stats(zero_opt_t h, int32_t rank, const zero_opt_buffers* bufs,
                                void* stream, zero_opt_stats* out) {
  zero_status st = check_handle_rank(h, rank);
  if (st != ZERO_OK) return st;
  if (!out) return fail(ZERO_EINVAL, "out is NULL");
  std::vector<HostRun> runs;
  int nbuf = 0;
  double divisor = 1.0;
  st = flat_runs(h, rank, bufs, &runs, &nbuf, &divisor);
  if (st != ZERO_OK) return st;
  st = check_device(h);
  if (st != ZERO_OK) return st;
  st = run(h, rank, runs, nbuf, divisor, bufs->stash, stream, zo::kStatsOnly, nullptr);
  if (st != ZERO_OK) return st;
  struct {
    double sumsq;
    int32_t nonfinite;
    int32_t pad;
  } got;
  st = read_small(h, &h->ws->own_sumsq, sizeof(got), stream, &got);
  if (st != ZERO_OK) return st;
  out->sumsq = got.sumsq;
  out->nonfinite = got.nonfinite;
  out->reserved = 0;
  return ZERO_OK;
}

zero_status zero_opt_grad_stats_async(zero_opt_t h, int32_t rank, const zero_opt_buffers* bufs,
                                      void* stream, zero_opt_stats* out_dev) {
  zero_status st = check_handle_rank(h, rank);
  if (st != ZERO_OK) return st;
  if (!out_dev) return fail(ZERO_EINVAL, "out_dev is NULL");
  std::vector<HostRun> runs;
  int nbuf = 0;
  double divisor = 1.0;
  st = flat_runs(h, rank, bufs, &runs, &nbuf, &divisor);
  if (st != ZERO_OK) return st;
  st = check_device(h);
  if (st != ZERO_OK) return st;
  return run(h, rank, runs, nbuf, divisor, bufs->stash, stream, zo::kStatsOnly, nullptr, 0,
             out_dev);
}

zero_status zero_opt_step_folded(zero_opt_t h, int32_t rank, const zero_opt_buffers* bufs,
                                 void* stream, const zero_opt_stats* per_rank_dev, int32_t n) {
  zero_status st = check_handle_rank(h, rank);
  if (st != ZERO_OK) return st;
  if (!per_rank_dev) return fail(ZERO_EINVAL, "per_rank_dev is NULL");
  if (n < 1 || n > (1 << 20)) return fail(ZERO_ERANGE, "n = %d outside [1, 2^20]", n);
  std::vector<HostRun> runs;
  int nbuf = 0;
  double divisor = 1.0;
  st = flat_runs(h, rank, bufs, &runs, &nbuf, &divisor);
  if (st != ZERO_OK) return st;
  st = check_device(h);
  if (st != ZERO_OK) return st;
  return run(h, rank, runs, nbuf, divisor, bufs->stash, stream, zo::kStepGlobalDev, per_rank_dev,
             n);
}

zero_status zero_opt_fold_stats(const zero_opt_stats* per_rank, int32_t n,
                                zero_opt_stats* out) {
  if (!out) return fail(ZERO_EINVAL, "out is NULL");
  if (n < 0 || (n > 0 && !per_rank)) return fail(ZERO_EINVAL, "bad per-rank array");
  double sumsq = 0.0;
  int32_t nonfinite = 0;
  for (int32_t r = 0; r < n; ++r) {
    sumsq += per_rank[r].sumsq;
    if (per_rank[r].nonfinite) nonfinite = 1;
  }
  out->sumsq = sumsq;
  out->nonfinite = nonfinite;
  out->reserved = 0;
  return ZERO_OK;
}

zero_status zero_opt_step(zero_opt_t h, int32_t rank, const zero_opt_buffers* bufs,
                          void* stream, const zero_opt_stats* global) {
  zero_status st = check_handle_rank(h, rank);
  if (st != ZERO_OK) return st;
  std::vector<HostRun> runs;
  int nbuf = 0;
  double divisor = 1.0;
  st = flat_runs(h, rank, bufs, &runs, &nbuf, &divisor);
  if (st != ZERO_OK) return st;
  st = check_device(h);
  if (st != ZERO_OK) return st;
  return run(h, rank, runs, nbuf, divisor, bufs->stash, stream,
             global ? zo::kStepGlobal : zo::kStepLocal, global);
}

zero_status zero_opt_grad_stats_tensors(zero_opt_t h, int32_t rank,
                                        const zero_opt_tensor_list* list, void* stream,
                                        zero_opt_stats* out) {
  zero_status st = check_handle_rank(h, rank);
  if (st != ZERO_OK) return st;
  if (!out) return fail(ZERO_EINVAL, "out is NULL");
  std::vector<HostRun> runs;
  int nbuf = 0;
  double divisor = 1.0;
  st = list_runs(list, h->cfg.master16 != 0, &runs, &nbuf, &divisor);
  if (st != ZERO_OK) return st;
  st = check_device(h);
  if (st != ZERO_OK) return st;
  st = run(h, rank, runs, nbuf, divisor, list->stash, stream, zo::kStatsOnly, nullptr);
  if (st != ZERO_OK) return st;
  struct {
    double sumsq;
    int32_t nonfinite;
    int32_t pad;
  } got;
  st = read_small(h, &h->ws->own_sumsq, sizeof(got), stream, &got);
  if (st != ZERO_OK) return st;
  out->sumsq = got.sumsq;
  out->nonfinite = got.nonfinite;
  out->reserved = 0;
  return ZERO_OK;
}

zero_status zero_opt_step_tensors(zero_opt_t h, int32_t rank, const zero_opt_tensor_list* list,
                                  void* stream, const zero_opt_stats* global) {
  zero_status st = check_handle_rank(h, rank);
  if (st != ZERO_OK) return st;
  std::vector<HostRun> runs;
  int nbuf = 0;
  double divisor = 1.0;
  st = list_runs(list, h->cfg.master16 != 0, &runs, &nbuf, &divisor);
  if (st != ZERO_OK) return st;
  st = check_device(h);
  if (st != ZERO_OK) return st;
  return run(h, rank, runs, nbuf, divisor, list->stash, stream,
             global ? zo::kStepGlobal : zo::kStepLocal, global);
}

zero_status zero_opt_loss_scale(zero_opt_t h, int32_t rank, void* stream,
                                zero_opt_scaler_state* out) {
  zero_status st = check_handle_rank(h, rank);
  if (st != ZERO_OK) return st;
  if (!out) return fail(ZERO_EINVAL, "out is NULL");
  st = check_device(h);
  if (st != ZERO_OK) return st;
  st = read_small(h, &h->ranks[rank], sizeof(zo::RankState), stream, out);
  if (st == ZERO_OK) h->t_mirror[rank] = out->t;
  return st;
}

zero_status zero_opt_set_loss_scale(zero_opt_t h, int32_t rank, void* stream,
                                    const zero_opt_scaler_state* in) {
  zero_status st = check_handle_rank(h, rank);
  if (st != ZERO_OK) return st;
  if (!in) return fail(ZERO_EINVAL, "in is NULL");
  if (!(in->scale > 0.0f) || in->clean_steps < 0 || in->t < 0 || in->skipped_total < 0 ||
      in->overflows < 0)
    return fail(ZERO_EINVAL, "scale must be > 0 and counters >= 0");
  st = check_device(h);
  if (st != ZERO_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // Pageable source: staged before the call returns, ordered on the stream.
  cudaError_t e = cudaMemcpyAsync(&h->ranks[rank], in, sizeof(zo::RankState),
                                  cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyAsync");
  h->t_mirror[rank] = in->t;
  return ZERO_OK;
}

zero_status zero_opt_set_lr(zero_opt_t h, double lr) {
  if (!h) return fail(ZERO_EINVAL, "handle is NULL");
  if (!(lr >= 0.0)) return fail(ZERO_EINVAL, "lr must be >= 0");
  h->cfg.lr = lr;
  return ZERO_OK;
}

zero_status zero_opt_last_step(zero_opt_t h, void* stream, zero_opt_step_info* out) {
  if (!h) return fail(ZERO_EINVAL, "handle is NULL");
  if (!out) return fail(ZERO_EINVAL, "out is NULL");
  zero_status st = check_device(h);
  if (st != ZERO_OK) return st;
  return read_small(h, &h->ws->dec, sizeof(zero_opt_step_info), stream, out);
}

zero_status zero_opt_save_shard(zero_opt_t h, int32_t rank, const float* master,
                                const float* m, const float* v, void* stream,
                                const char* path) {
  zero_status st = check_handle_rank(h, rank);
  if (st != ZERO_OK) return st;
  if (h->cfg.master16)
    return fail(ZERO_ENOTSUP,
                "a master16 handle keeps its masters in param16: use zero_opt_save_shard16");
  if (!path) return fail(ZERO_EINVAL, "path is NULL");
  zero_opt_ckpt_info info;
  std::memset(&info, 0, sizeof(info));
  int64_t shard = 0;
  zo::shard_range(h->cfg.numel, h->cfg.world, rank, &info.begin, &info.real_len, &shard);
  info.numel = h->cfg.numel;
  info.world = h->cfg.world;
  info.rank = rank;
  if (info.real_len > 0 && (!master || !m || !v))
    return fail(ZERO_EINVAL, "master, m and v must be non-NULL");
  st = check_device(h);
  if (st != ZERO_OK) return st;
  st = zero_opt_loss_scale(h, rank, stream, &info.scaler);
  if (st != ZERO_OK) return st;
  const size_t n = (size_t)info.real_len;
  std::vector<float> hm(n), hmm(n), hv(n);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSuccess;
  if (n > 0) {
    e = cudaMemcpyAsync(hm.data(), master, n * 4, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaMemcpyAsync(hmm.data(), m, n * 4, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaMemcpyAsync(hv.data(), v, n * 4, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  }
  if (e != cudaSuccess) return cuda_fail(e, "zero_opt_save_shard");
  return zero_opt_ckpt_write(path, &info, hm.data(), hmm.data(), hv.data());
}

zero_status zero_opt_save_shard16(zero_opt_t h, int32_t rank, const void* param16,
                                  int32_t param16_shard_local, const float* m, const float* v,
                                  void* stream, const char* path) {
  zero_status st = check_handle_rank(h, rank);
  if (st != ZERO_OK) return st;
  if (!h->cfg.master16)
    return fail(ZERO_EINVAL, "not a master16 handle: use zero_opt_save_shard");
  if (!path) return fail(ZERO_EINVAL, "path is NULL");
  zero_opt_ckpt_info info;
  std::memset(&info, 0, sizeof(info));
  int64_t shard = 0;
  zo::shard_range(h->cfg.numel, h->cfg.world, rank, &info.begin, &info.real_len, &shard);
  info.numel = h->cfg.numel;
  info.world = h->cfg.world;
  info.rank = rank;
  if (info.real_len > 0 && (!param16 || !m || !v))
    return fail(ZERO_EINVAL, "param16, m and v must be non-NULL");
  st = check_device(h);
  if (st != ZERO_OK) return st;
  st = zero_opt_loss_scale(h, rank, stream, &info.scaler);
  if (st != ZERO_OK) return st;
  const size_t n = (size_t)info.real_len;
  std::vector<uint16_t> hq(n);
  std::vector<float> hm(n), hmm(n), hv(n);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSuccess;
  if (n > 0) {
    const uint16_t* q =
        static_cast<const uint16_t*>(param16) + (param16_shard_local ? 0 : info.begin);
    e = cudaMemcpyAsync(hq.data(), q, n * 2, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaMemcpyAsync(hmm.data(), m, n * 4, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaMemcpyAsync(hv.data(), v, n * 4, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  }
  if (e != cudaSuccess) return cuda_fail(e, "zero_opt_save_shard16");
  const bool fp16 = h->cfg.param_dtype == ZERO_FP16;
  for (size_t i = 0; i < n; ++i) hm[i] = zo::hc::widen16(hq[i], fp16);
  return zero_opt_ckpt_write(path, &info, hm.data(), hmm.data(), hv.data());
}

zero_status zero_opt_load_shard(zero_opt_t h, int32_t rank, float* master, float* m,
                                float* v, void* param16, int32_t param16_shard_local,
                                void* stream, const char* path) {
  zero_status st = check_handle_rank(h, rank);
  if (st != ZERO_OK) return st;
  const bool m16 = h->cfg.master16 != 0;
  if (!path) return fail(ZERO_EINVAL, "path is NULL");
  zero_opt_ckpt_info info;
  st = zero_opt_ckpt_read(path, &info, nullptr, nullptr, nullptr);
  if (st != ZERO_OK) return st;
  if (info.numel != h->cfg.numel || info.world != h->cfg.world || info.rank != rank)
    return fail(ZERO_EINVAL, "%s was written for numel %lld, world %d, rank %d", path,
                (long long)info.numel, info.world, info.rank);
  if (info.real_len > 0 && (m16 ? (!param16 || !m || !v) : (!master || !m || !v)))
    return fail(ZERO_EINVAL, m16 ? "param16 (the masters of a master16 handle), m and v must be "
                                   "non-NULL"
                                 : "master, m and v must be non-NULL");
  st = check_device(h);
  if (st != ZERO_OK) return st;
  const size_t n = (size_t)info.real_len;
  std::vector<float> hm(n), hmm(n), hv(n);
  st = zero_opt_ckpt_read(path, &info, hm.data(), hmm.data(), hv.data());
  if (st != ZERO_OK) return st;
  // 16-bit masters: the file's binary32 masters narrowed (exactly, when they
  // were written by zero_opt_save_shard16; else rounded to nearest even)
  std::vector<uint16_t> hq(m16 ? n : 0);
  const bool fp16 = h->cfg.param_dtype == ZERO_FP16;
  for (size_t i = 0; i < hq.size(); ++i) hq[i] = zo::hc::narrow16(hm[i], fp16);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSuccess;
  if (n > 0) {
    if (m16) {
      uint16_t* q = static_cast<uint16_t*>(param16) + (param16_shard_local ? 0 : info.begin);
      e = cudaMemcpyAsync(q, hq.data(), n * 2, cudaMemcpyHostToDevice, s);
    } else {
      e = cudaMemcpyAsync(master, hm.data(), n * 4, cudaMemcpyHostToDevice, s);
    }
    if (e == cudaSuccess) e = cudaMemcpyAsync(m, hmm.data(), n * 4, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = cudaMemcpyAsync(v, hv.data(), n * 4, cudaMemcpyHostToDevice, s);
  }
  if (e != cudaSuccess) return cuda_fail(e, "zero_opt_load_shard");
  st = zero_opt_set_loss_scale(h, rank, stream, &info.scaler);
  if (st != ZERO_OK) return st;
  if (!m16 && param16 && n > 0) {
    zo::CastArgs ca;
    ca.master = master;
    ca.p16 = static_cast<unsigned short*>(param16) + (param16_shard_local ? 0 : info.begin);
    ca.n = (int64_t)n;
    const void* fn = h->cfg.param_dtype == ZERO_FP16
                         ? reinterpret_cast<const void*>(zo::cast_kernel<__half>)
                         : reinterpret_cast<const void*>(zo::cast_kernel<__nv_bfloat16>);
    const int64_t grid = std::max<int64_t>(
        1, std::min<int64_t>((int64_t)h->sms * 8, ((int64_t)n + zo::kThreads - 1) / zo::kThreads));
    st = launch_kernel(h, fn, (int)grid, &ca, s);
    if (st != ZERO_OK) return st;
  }
  e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "zero_opt_load_shard");
  return ZERO_OK;
}

zero_status zero_opt_set_events(zero_opt_t h, void* ev_start, void* ev_mid, void* ev_end) {
  if (!h) return fail(ZERO_EINVAL, "handle is NULL");
  h->ev[0] = static_cast<cudaEvent_t>(ev_start);
  h->ev[1] = static_cast<cudaEvent_t>(ev_mid);
  h->ev[2] = static_cast<cudaEvent_t>(ev_end);
  return ZERO_OK;
}

zero_status zero_opt_inject_wait_fault(zero_opt_t h) {
  if (!h) return fail(ZERO_EINVAL, "handle is NULL");
  h->inject_wait_fault = 1;
  return ZERO_OK;
}

zero_status zero_opt_launch_count(zero_opt_t h, int64_t* launches) {
  if (!h || !launches) return fail(ZERO_EINVAL, "NULL argument");
  *launches = h->launches;
  return ZERO_OK;
}

zero_status zero_opt_get_counters(zero_opt_t h, zero_opt_counters* out) {
  if (!h || !out) return fail(ZERO_EINVAL, "NULL argument");
  std::lock_guard<std::mutex> lock(h->mu);
  out->launches = h->launches;
  out->table_uploads = h->table_uploads;
  out->table_waits = h->table_waits;
  out->device_allocs = h->device_allocs;
  out->device_frees = h->device_frees;
  out->tables_cached = (int64_t)h->plans.size();
  int64_t pinned = 0;
  for (const Plan* p : h->plans) pinned += p->pinned ? 1 : 0;
  out->tables_pinned = pinned;
  out->table_bytes = h->table_bytes;
  return ZERO_OK;
}

const char* zero_opt_status_string(zero_status s) {
  switch (s) {
    case ZERO_OK: return "ZERO_OK";
    case ZERO_EINVAL: return "ZERO_EINVAL: invalid argument";
    case ZERO_ERANGE: return "ZERO_ERANGE: index or size out of range";
    case ZERO_ENOMEM: return "ZERO_ENOMEM: allocation failed";
    case ZERO_ECUDA: return "ZERO_ECUDA: CUDA error or no device";
    case ZERO_ENOTSUP: return "ZERO_ENOTSUP: unsupported option";
  }
  return "unknown zero_status";
}

const char* zero_opt_last_error(void) { return g_err.c_str(); }

}  // extern "C"
