// synth_gen.cu -- GPU side of the seeded synthetic-input generator.
//
// Produces exactly the values of synth.normal_np (see synth/__init__.py for
// the definition): SplitMix64 output function over a counter, Irwin-Hall sum
// of twelve 24-bit uniforms, scaled in binary64, rounded to binary32 and then
// to fp16 / bf16.  This file holds no optimizer arithmetic; it only makes
// inputs.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace {

constexpr uint64_t kGamma = 0x9E3779B97F4A7C15ull;

__device__ __forceinline__ uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

__global__ void normal_kernel(uint64_t key, int64_t offset, int64_t n,
                              double sigma, int kind, void* out) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const uint64_t j = (uint64_t)(offset + i);
    int64_t acc = 0;
#pragma unroll
    for (int u = 0; u < 12; ++u) {
      const uint64_t ctr = j * 12ull + (uint64_t)(u + 1);
      acc += (int64_t)(mix64(key + ctr * kGamma) >> 40);
    }
    const int64_t z = acc - 6ll * (1ll << 24);
    const double x = __dmul_rn((double)z * 0x1p-24, sigma);
    const float f = __double2float_rn(x);
    if (kind == 0) {
      static_cast<float*>(out)[i] = f;
    } else if (kind == 1) {
      static_cast<__half*>(out)[i] = __float2half_rn(f);
    } else {
      static_cast<__nv_bfloat16*>(out)[i] = __float2bfloat16_rn(f);
    }
  }
}

}  // namespace

extern "C" int synth_normal(uint64_t key, int64_t offset, int64_t n, double sigma,
                            int32_t kind, void* out, void* stream) {
  if (n <= 0) return 0;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  int64_t blocks = (n + 255) / 256;
  const int64_t cap = (int64_t)(sms > 0 ? sms : 1) * 16;
  if (blocks > cap) blocks = cap;
  normal_kernel<<<(unsigned)blocks, 256, 0, (cudaStream_t)stream>>>(key, offset, n,
                                                                     sigma, kind, out);
  return (int)cudaGetLastError();
}
