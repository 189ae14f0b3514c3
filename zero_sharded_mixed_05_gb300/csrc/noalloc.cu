// noalloc.cu -- gradient statistics without any device allocation.
//
// zero_opt_grad_stats_noalloc computes what zero_opt_grad_stats computes for
// one shard -- the overflow flag and the sum of squares of the binary32 sums
// of n_bufs 16-bit gradient buffers -- for callers that cannot allocate device
// memory: the handle behind zero_opt_grad_stats owns a cudaMalloc'ed workspace
// and device-side buffer tables, and some callers may not call cudaMalloc at
// all (a runtime whose external allocator owns every device byte, a process
// already at its memory limit, or a code path that cannot afford the device
// synchronization cudaMalloc may cause).  Its only scratch -- the per-CTA
// partial sums and the completion ticket -- lives in the file-scope array
// g_stats_scratch below, which every GPU that loads the library holds until
// the process exits.  Gradient pointers travel by value in the kernel
// arguments, and the result is written to a caller-owned device struct.
#include <cuda_runtime.h>

#include <mutex>

#include "host_util.h"
#include "kernels.cuh"
#include "zero_opt.h"

namespace {

constexpr int kNoAllocMaxBufs = 64;     // gradient buffers per call
constexpr int kNoAllocMaxCtas = 1024;   // partial-sum slots, one per CTA
constexpr int kMaxDevices = 64;

struct StatsScratch {
  unsigned int ticket;                  // CTAs that finished; must start at 0
  int32_t pad[63];
  double part_sumsq[kNoAllocMaxCtas];
  int32_t part_flag[kNoAllocMaxCtas];
};

// 256 + 8 KiB + 4 KiB = 12,544 bytes per device.
static __device__ __align__(256) unsigned char g_stats_scratch[sizeof(StatsScratch)];

struct NoAllocArgs {
  const void* g[kNoAllocMaxBufs];
  int32_t nbuf;
  int32_t vec;                          // all pointers 16-byte aligned
  int64_t n;
  int64_t ntiles;
  StatsScratch* scratch;                // device address of g_stats_scratch
  zero_opt_stats* out;                  // caller's device result
};

// The sum over buffers, the exact-square accumulator and the fixed-order fold
// are those of pass 1, so the result agrees with zero_opt_grad_stats to within
// the accuracy of the sum of squares (the two may split the work differently).
template <typename GT>
__global__ void __launch_bounds__(zo::kThreads) stats_noalloc_kernel(const NoAllocArgs a) {
  __shared__ double red[zo::kThreads / 32];
  __shared__ int s_last;
  const int tid = threadIdx.x;
  zo::SqAcc acc;
  for (int64_t tile = blockIdx.x; tile < a.ntiles; tile += gridDim.x) {
    const int64_t base = tile * zo::kTile;
    const int64_t e0 = base + tid * zo::kVec;
    float x[zo::kVec];
    if (a.vec && e0 + zo::kVec <= a.n) {
#pragma unroll
      for (int i = 0; i < zo::kVec; ++i) x[i] = 0.0f;
      for (int b = 0; b < a.nbuf; ++b) {
        float y[zo::kVec];
        zo::Fmt<GT>::dec8(__ldcg(reinterpret_cast<const uint4*>(
                               static_cast<const unsigned short*>(a.g[b]) + e0)),
                           y);
#pragma unroll
        for (int i = 0; i < zo::kVec; ++i) x[i] = __fadd_rn(x[i], y[i]);
      }
    } else {
#pragma unroll
      for (int i = 0; i < zo::kVec; ++i) {
        const int64_t e = a.vec ? e0 + i : base + (int64_t)i * zo::kThreads + tid;
        float sum = 0.0f;
        if (e < a.n)
          for (int b = 0; b < a.nbuf; ++b)
            sum = __fadd_rn(sum, zo::Fmt<GT>::dec(
                                     __ldcg(static_cast<const unsigned short*>(a.g[b]) + e)));
        x[i] = sum;
      }
    }
    acc.add<false>(x);
  }
  const double blk = zo::block_sum(acc.total(), red);
  const int any = __syncthreads_or(acc.amax >= 0x7f800000u ? 1 : 0);
  if (tid == 0) {
    a.scratch->part_sumsq[blockIdx.x] = blk;
    a.scratch->part_flag[blockIdx.x] = any;
    __threadfence();
    const unsigned int prev = atomicAdd(&a.scratch->ticket, 1u);
    s_last = (prev == gridDim.x - 1) ? 1 : 0;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  double part = 0.0;
  int f = 0;
  for (int c = tid; c < (int)gridDim.x; c += zo::kThreads) {
    part = __dadd_rn(part, __ldcg(&a.scratch->part_sumsq[c]));
    f |= __ldcg(&a.scratch->part_flag[c]);
  }
  const double tot = zo::block_sum(part, red);
  const int anyf = __syncthreads_or(f);
  if (tid == 0) {
    a.out->sumsq = tot;
    a.out->nonfinite = anyf;
    a.out->reserved = 0;
    a.scratch->ticket = 0u;
  }
}

// Device address of g_stats_scratch, looked up once per device with that
// device current (in host code the array's name is not a device address).
std::mutex g_setup_mu;
void* g_scratch_addr[kMaxDevices] = {nullptr};

zero_status scratch_for(int dev, StatsScratch** out) {
  if (dev < 0 || dev >= kMaxDevices) return zo::fail(ZERO_ECUDA, "device %d unsupported", dev);
  std::lock_guard<std::mutex> lock(g_setup_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_stats_scratch);
    if (e != cudaSuccess)
      return zo::fail(ZERO_ECUDA, "cudaGetSymbolAddress: %s", cudaGetErrorString(e));
    g_scratch_addr[dev] = p;
  }
  *out = static_cast<StatsScratch*>(g_scratch_addr[dev]);
  return ZERO_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" zero_status zero_opt_grad_stats_noalloc(const void* const* grads, int32_t n_bufs,
                                                   int32_t grad_dtype, int64_t n,
                                                   void* stream, zero_opt_stats* out) {
  if (!grads || !out) return zo::fail(ZERO_EINVAL, "grads and out must be non-NULL");
  if (n_bufs < 1) return zo::fail(ZERO_EINVAL, "n_bufs must be >= 1");
  if (n_bufs > kNoAllocMaxBufs)
    return zo::fail(ZERO_ERANGE, "n_bufs %d exceeds the maximum of %d gradient buffers",
                    n_bufs, kNoAllocMaxBufs);
  if (n < 0) return zo::fail(ZERO_EINVAL, "n must be >= 0");
  if (grad_dtype != ZERO_FP16 && grad_dtype != ZERO_BF16)
    return zo::fail(ZERO_EINVAL, "grad_dtype must be ZERO_FP16 or ZERO_BF16");
  NoAllocArgs a;
  a.nbuf = n_bufs;
  a.n = n;
  a.vec = 1;
  for (int b = 0; b < kNoAllocMaxBufs; ++b) a.g[b] = nullptr;
  for (int b = 0; b < n_bufs; ++b) {
    if (!grads[b] && n > 0) return zo::fail(ZERO_EINVAL, "gradient pointer %d is NULL", b);
    a.g[b] = grads[b];
    if (!aligned16(grads[b])) a.vec = 0;
  }
  a.ntiles = (n + zo::kTile - 1) / zo::kTile;
  a.out = out;
  int dev = -1, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return zo::fail(ZERO_ECUDA, "no usable CUDA device: %s", cudaGetErrorString(e));
  }
  zero_status st = scratch_for(dev, &a.scratch);
  if (st != ZERO_OK) return st;
  const void* fn = grad_dtype == ZERO_FP16
                       ? reinterpret_cast<const void*>(stats_noalloc_kernel<__half>)
                       : reinterpret_cast<const void*>(stats_noalloc_kernel<__nv_bfloat16>);
  int occ = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, fn, zo::kThreads, 0) != cudaSuccess ||
      occ < 1)
    occ = 1;
  int64_t grid = (int64_t)occ * sms;
  if (grid > a.ntiles) grid = a.ntiles;
  if (grid > kNoAllocMaxCtas) grid = kNoAllocMaxCtas;
  if (grid < 1) grid = 1;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // The ticket must start at zero; a memset is not an allocation.
  e = cudaMemsetAsync(&a.scratch->ticket, 0, sizeof(unsigned int), s);
  if (e != cudaSuccess) return zo::fail(ZERO_ECUDA, "cudaMemsetAsync: %s", cudaGetErrorString(e));
  void* params[] = {&a};
  e = cudaLaunchKernel(fn, dim3((unsigned)grid), dim3(zo::kThreads), params, 0, s);
  if (e != cudaSuccess) return zo::fail(ZERO_ECUDA, "cudaLaunchKernel: %s", cudaGetErrorString(e));
  return ZERO_OK;
}
