// Device implementation of the counter-based normal generator defined in synth/__init__.py:
// splitmix64 output function over key + (i + 1) * golden, Box-Muller on the two 32-bit halves
// in fp64, then fp64 -> fp32 -> 16-bit storage type, round-to-nearest-even at each step.
// Synthetic-input plumbing only: it holds none of the decode step's arithmetic.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace {

__device__ __forceinline__ uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

__global__ void fill_normal_kernel(uint16_t* dst, uint64_t count, uint64_t key, uint64_t offset,
                                   double mean, double std_, int is_bf16) {
  const uint64_t stride = static_cast<uint64_t>(gridDim.x) * blockDim.x;
  for (uint64_t i = static_cast<uint64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < count;
       i += stride) {
    const uint64_t w = mix64(key + (offset + i + 1) * 0x9E3779B97F4A7C15ull);
    const double u1 = (static_cast<double>(w >> 32) + 1.0) * (1.0 / 4294967296.0);
    const double u2 = static_cast<double>(w & 0xFFFFFFFFull) * (1.0 / 4294967296.0);
    const double z = sqrt(-2.0 * log(u1)) * cos(6.283185307179586 * u2);
    const float v = static_cast<float>(mean + std_ * z);
    uint16_t bits;
    if (is_bf16) {
      const __nv_bfloat16 b = __float2bfloat16_rn(v);
      bits = *reinterpret_cast<const uint16_t*>(&b);
    } else {
      const __half h = __float2half_rn(v);
      bits = *reinterpret_cast<const uint16_t*>(&h);
    }
    dst[i] = bits;
  }
}

}  // namespace

extern "C" int synth_fill_normal(void* dst, unsigned long long count, unsigned long long key,
                                 unsigned long long offset, double mean, double std_, int is_bf16,
                                 void* stream) {
  if (count == 0) return 0;
  int dev = 0, sms = 1;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  unsigned long long blocks = (count + 255) / 256;
  const unsigned long long cap = static_cast<unsigned long long>(sms) * 16;
  if (blocks > cap) blocks = cap;
  fill_normal_kernel<<<static_cast<unsigned>(blocks), 256, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<uint16_t*>(dst), count, key, offset, mean, std_, is_bf16);
  return static_cast<int>(cudaGetLastError());
}
