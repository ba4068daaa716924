// Device implementation of the seeded input generator of glasynth/__init__.py (same definition,
// same bits): SplitMix64 output i of the stream keyed by `key` is mix64(key + (i+1)*GAMMA); the
// value is the Box-Muller variate sqrt(-2 ln u1) cos(2 pi u2) of its two 32-bit halves, with the
// logarithm and cosine evaluated from their series in fp64 (the same operations, constants and
// order as the numpy side, each an IEEE-rounded +, -, x, / or sqrt, never fused), then
// multiplied by sigma and rounded once to fp32 (and to bf16 nearest-even for bf16 tensors).
// Holds no part of the GLA arithmetic.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace {

__device__ __forceinline__ uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

// Constants as in glasynth: ln 2, pi/2, sqrt 2 rounded to double; series coefficients 1/(2j+1)
// (atanh), (-1)^j/(2j)! (cos), (-1)^j/(2j+1)! (sin), j = 0..10, correctly rounded (each factorial
// is an exact double, and the compiler folds the division with IEEE rounding).
constexpr double LN2 = 0.6931471805599453;
constexpr double PIO2 = 1.5707963267948966;
constexpr double SQRT2 = 1.4142135623730951;
__constant__ double LOG_C[11] = {1.0 / 1, 1.0 / 3, 1.0 / 5, 1.0 / 7, 1.0 / 9, 1.0 / 11,
                                 1.0 / 13, 1.0 / 15, 1.0 / 17, 1.0 / 19, 1.0 / 21};
__constant__ double COS_C[11] = {1.0,
                                 -1.0 / 2.0,
                                 1.0 / 24.0,
                                 -1.0 / 720.0,
                                 1.0 / 40320.0,
                                 -1.0 / 3628800.0,
                                 1.0 / 479001600.0,
                                 -1.0 / 87178291200.0,
                                 1.0 / 20922789888000.0,
                                 -1.0 / 6402373705728000.0,
                                 1.0 / 2432902008176640000.0};
__constant__ double SIN_C[11] = {1.0,
                                 -1.0 / 6.0,
                                 1.0 / 120.0,
                                 -1.0 / 5040.0,
                                 1.0 / 362880.0,
                                 -1.0 / 39916800.0,
                                 1.0 / 6227020800.0,
                                 -1.0 / 1307674368000.0,
                                 1.0 / 355687428096000.0,
                                 -1.0 / 121645100408832000.0,
                                 1.0 / 51090942171709440000.0};

__device__ __forceinline__ double horner(const double* c, double s) {
  double p = c[10];
#pragma unroll
  for (int j = 9; j >= 0; --j) p = __dadd_rn(__dmul_rn(p, s), c[j]);
  return p;
}

// ln((a + 1/2) / 2^32): a + 1/2 = 2^e m with m in [1/sqrt 2, sqrt 2], ln m by the atanh series.
__device__ __forceinline__ double ln_u1(uint32_t a) {
  const uint64_t n = 2ull * a + 1ull;           // a + 1/2 = n / 2
  int e = 64 - __clzll((long long)n) - 2;       // n / 2 in [2^e, 2^(e+1))
  const double y = __dadd_rn((double)a, 0.5);   // exact
  double m = __dmul_rn(y, __longlong_as_double((long long)(1023 - e) << 52));  // y 2^-e, exact
  if (m > SQRT2) {
    m = __dmul_rn(m, 0.5);
    e += 1;
  }
  const double t = __ddiv_rn(__dsub_rn(m, 1.0), __dadd_rn(m, 1.0));
  const double lnm = __dmul_rn(__dmul_rn(2.0, t), horner(LOG_C, __dmul_rn(t, t)));
  return __dadd_rn(__dmul_rn((double)(e - 32), LN2), lnm);
}

// cos(2 pi b / 2^32): 4 u2 = n + f, |f| <= 1/2, phi = f pi/2, the quadrant n mod 4.
__device__ __forceinline__ double cos_2pi(uint32_t b) {
  const double w = __dmul_rn((double)b, 0x1p-30);  // b 2^-30, exact
  const double n = floor(__dadd_rn(w, 0.5));
  const double phi = __dmul_rn(__dsub_rn(w, n), PIO2);
  const double s = __dmul_rn(phi, phi);
  const int q = (int)n & 3;
  if (q == 0 || q == 2) {
    const double c = horner(COS_C, s);
    return q == 0 ? c : -c;
  }
  const double sn = __dmul_rn(phi, horner(SIN_C, s));
  return q == 1 ? -sn : sn;
}

__device__ __forceinline__ float box_muller(uint64_t x, double sigma) {
  const double r = __dsqrt_rn(__dmul_rn(-2.0, ln_u1((uint32_t)(x >> 32))));
  const double z = __dmul_rn(r, cos_2pi((uint32_t)(x & 0xFFFFFFFFull)));
  return __double2float_rn(__dmul_rn(z, sigma));
}

template <class T> __device__ __forceinline__ T cast(float x);
template <> __device__ __forceinline__ float cast<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 cast<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

template <class T>
__global__ void fill_normal_kernel(T* out, long long count, unsigned long long start,
                                   unsigned long long key, double sigma) {
  const unsigned long long gamma = 0x9E3779B97F4A7C15ull;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < count;
       i += (long long)gridDim.x * blockDim.x) {
    const uint64_t x = mix64(key + (start + (unsigned long long)i + 1ull) * gamma);
    out[i] = cast<T>(box_muller(x, sigma));
  }
}

}  // namespace

extern "C" int glasynth_fill_normal(void* out, int is_bf16, long long count, unsigned long long start,
                                    unsigned long long key, double sigma, void* stream) {
  if (count <= 0) return 0;
  int dev = 0, sms = 1;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  long long blocks = (count + 255) / 256;
  const long long cap = (long long)sms * 16;
  if (blocks > cap) blocks = cap;
  cudaStream_t s = (cudaStream_t)stream;
  if (is_bf16)
    fill_normal_kernel<__nv_bfloat16><<<(unsigned)blocks, 256, 0, s>>>((__nv_bfloat16*)out, count, start, key, sigma);
  else
    fill_normal_kernel<float><<<(unsigned)blocks, 256, 0, s>>>((float*)out, count, start, key, sigma);
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}
