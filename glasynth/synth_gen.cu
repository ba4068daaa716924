// Device implementation of the seeded input generator of glasynth/__init__.py (same definition,
// same bits): SplitMix64 output i of the stream keyed by `key` is mix64(key + (i+1)*GAMMA); the
// value is (float(sum of its four 16-bit fields) - 131070) * c, rounded once in fp32, then to
// bf16 nearest-even for bf16 tensors.  Holds no part of the GLA arithmetic.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace {

__device__ __forceinline__ uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

__device__ __forceinline__ float ih4(uint64_t x, float c) {
  const uint32_t s = (uint32_t)(x & 0xFFFF) + (uint32_t)((x >> 16) & 0xFFFF) +
                     (uint32_t)((x >> 32) & 0xFFFF) + (uint32_t)((x >> 48) & 0xFFFF);
  return __fmul_rn(__fsub_rn((float)s, 131070.0f), c);
}

template <class T> __device__ __forceinline__ T cast(float x);
template <> __device__ __forceinline__ float cast<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 cast<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

template <class T>
__global__ void fill_normal_kernel(T* out, long long count, unsigned long long start,
                                   unsigned long long key, float c) {
  const unsigned long long gamma = 0x9E3779B97F4A7C15ull;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < count;
       i += (long long)gridDim.x * blockDim.x) {
    const uint64_t x = mix64(key + (start + (unsigned long long)i + 1ull) * gamma);
    out[i] = cast<T>(ih4(x, c));
  }
}

}  // namespace

extern "C" int glasynth_fill_normal(void* out, int is_bf16, long long count, unsigned long long start,
                                    unsigned long long key, float c, void* stream) {
  if (count <= 0) return 0;
  int dev = 0, sms = 1;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  long long blocks = (count + 255) / 256;
  const long long cap = (long long)sms * 16;
  if (blocks > cap) blocks = cap;
  cudaStream_t s = (cudaStream_t)stream;
  if (is_bf16)
    fill_normal_kernel<__nv_bfloat16><<<(unsigned)blocks, 256, 0, s>>>((__nv_bfloat16*)out, count, start, key, c);
  else
    fill_normal_kernel<float><<<(unsigned)blocks, 256, 0, s>>>((float*)out, count, start, key, c);
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}
