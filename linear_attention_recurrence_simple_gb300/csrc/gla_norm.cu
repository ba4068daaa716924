// Per-tier Head RMSNorm and SiLU output gate of the mixer's output.
//
// "Beyond the KV cache" (Laplace 3B on Trainium2), section "i14 and the Laplace 3B architecture":
// the per-head outputs pass through a Head RMSNorm within each decay tier (the heads of a tier
// share one norm: "Head RMSNorm (per tier)" in the architecture table), are concatenated and
// gated by SiLU(g_t), g_t being the gate stream of the QKVG projection.  For row t, head h:
//     y = o / sqrt(mean_c o_c^2 + eps) * w_{tier(h)} * SiLU(g),   SiLU(x) = x sigmoid(x).
// The RMS needs all 192 channels of a head's row, which the chunk scans split over three CTAs,
// so this is its own pass: a stream over o and g (read once) and y (written once).  A warp takes
// four consecutive (row, head) pairs, 4 x 192 contiguous values cut into 96 pieces of 8; lane l
// holds pieces l, l + 32 and l + 64 (every lane busy, each load instruction one contiguous 512-byte
// run in bf16), issues all its loads before any arithmetic, and the four pairs' sums of squares
// are reduced across the warp.  The tier gains and the head-to-tier map are read through the
// read-only cache (a few KB, shared by every CTA).
#include "gla_common.cuh"

namespace gla {
namespace {

constexpr int NG_WARPS = 8;                          // warps per CTA
constexpr int NG_PAIRS = 4;                          // (row, head) pairs per warp
constexpr int NG_PIECES = NG_PAIRS * DV / 8 / 32;    // pieces of 8 values per lane (3)
static_assert(NG_PIECES * 32 * 8 == NG_PAIRS * DV, "a warp's pairs split evenly over its lanes");

// 8 consecutive values as loaded (bf16: one 16-byte word; fp32: two), unpacked at use, so that
// the loads in flight hold as few registers as possible.
template <class T> struct Raw8;
template <> struct Raw8<__nv_bfloat16> { uint4 u[1]; };
template <> struct Raw8<float> { uint4 u[2]; };
template <class T>
__device__ __forceinline__ Raw8<T> load_raw8(const T* p) {
  Raw8<T> r;
#pragma unroll
  for (int i = 0; i < (int)(sizeof(r.u) / 16); ++i) r.u[i] = reinterpret_cast<const uint4*>(p)[i];
  return r;
}
// Pairs of fp32 values go through the packed two-lane fp32 instructions (each lane rounded as
// its scalar counterpart).
__device__ __forceinline__ uint64_t f2_bits(float2 a) { return ((uint64_t)__float_as_uint(a.y) << 32) | __float_as_uint(a.x); }
__device__ __forceinline__ float2 bits_f2(uint64_t b) { return make_float2(__uint_as_float((uint32_t)b), __uint_as_float((uint32_t)(b >> 32))); }
__device__ __forceinline__ float2 pmul(float2 a, float2 b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(f2_bits(a)), "l"(f2_bits(b)));
  return bits_f2(r);
}
__device__ __forceinline__ float2 pfma(float2 a, float2 b, float2 c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(f2_bits(a)), "l"(f2_bits(b)), "l"(f2_bits(c)));
  return bits_f2(r);
}

__device__ __forceinline__ void unpack8(const Raw8<__nv_bfloat16>& r, float2 (&x)[4]) {
  const uint32_t w[4] = {r.u[0].x, r.u[0].y, r.u[0].z, r.u[0].w};
#pragma unroll
  for (int e = 0; e < 4; ++e) x[e] = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[e]));
}
__device__ __forceinline__ void unpack8(const Raw8<float>& r, float2 (&x)[4]) {
  const uint32_t w[8] = {r.u[0].x, r.u[0].y, r.u[0].z, r.u[0].w, r.u[1].x, r.u[1].y, r.u[1].z, r.u[1].w};
#pragma unroll
  for (int e = 0; e < 4; ++e) x[e] = make_float2(__uint_as_float(w[2 * e]), __uint_as_float(w[2 * e + 1]));
}
__device__ __forceinline__ void store8(__nv_bfloat16* p, const float2 (&x)[4]) {
  uint32_t w[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const __nv_bfloat162 b = __floats2bfloat162_rn(x[e].x, x[e].y);
    w[e] = *reinterpret_cast<const uint32_t*>(&b);
  }
  *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
}
__device__ __forceinline__ void store8(float* p, const float2 (&x)[4]) {
  reinterpret_cast<float4*>(p)[0] = make_float4(x[0].x, x[0].y, x[1].x, x[1].y);
  reinterpret_cast<float4*>(p)[1] = make_float4(x[2].x, x[2].y, x[3].x, x[3].y);
}

// SiLU(g) = g sigmoid(g) = g (1 + tanh(g / 2)) / 2.  bf16 data: the hardware tanh approximation
// (relative error about 2^-11, far inside a bf16 rounding); fp32 data: CUDA's accurate tanhf.
__device__ __forceinline__ float tanh_fast(float x) {
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
template <class T> __device__ __forceinline__ float2 tanh2(float2 x);
template <> __device__ __forceinline__ float2 tanh2<__nv_bfloat16>(float2 x) {
  return make_float2(tanh_fast(x.x), tanh_fast(x.y));
}
template <> __device__ __forceinline__ float2 tanh2<float>(float2 x) { return make_float2(tanhf(x.x), tanhf(x.y)); }
template <class T>
__device__ __forceinline__ float2 silu2(float2 g) {
  const float2 h = make_float2(0.5f, 0.5f);
  return pmul(g, pfma(h, tanh2<T>(pmul(h, g)), h));
}

template <class T>
__global__ void __launch_bounds__(NG_WARPS * 32)
head_norm_gate_kernel(const T* __restrict__ o, const T* __restrict__ g, const float* __restrict__ w,
                      const int32_t* __restrict__ tier, int n_tiers, float eps, T* __restrict__ y,
                      long long pairs, int H, unsigned* err) {
  const int lane = threadIdx.x & 31;
  const long long base = ((long long)blockIdx.x * NG_WARPS + (threadIdx.x >> 5)) * NG_PAIRS;  // row * H + head
  const long long n_el = pairs * DV;
  // Piece j of this lane: values [8p, 8p + 8) of the warp's block, p = lane + 32 j, in pair p / 24
  // (which is j or j + 1), channels 8 (p mod 24) onwards.  Loads past the last pair are clamped
  // into range and their results never stored.
  Raw8<T> ro[NG_PIECES], rg[NG_PIECES];
#pragma unroll
  for (int j = 0; j < NG_PIECES; ++j) {
    const long long e = min(base * DV + 8 * (lane + 32 * j), n_el - 8);
    ro[j] = load_raw8(o + e);
    rg[j] = load_raw8(g + e);
  }
  float2 x[NG_PIECES][4];
  float acc[NG_PAIRS];
#pragma unroll
  for (int r = 0; r < NG_PAIRS; ++r) acc[r] = 0.f;
#pragma unroll
  for (int j = 0; j < NG_PIECES; ++j) {
    unpack8(ro[j], x[j]);
    float2 s2 = pmul(x[j][0], x[j][0]);
#pragma unroll
    for (int e = 1; e < 4; ++e) s2 = pfma(x[j][e], x[j][e], s2);
    const float ss = s2.x + s2.y;
    const bool lower = lane + 32 * j < 24 * (j + 1);
    acc[j] += lower ? ss : 0.f;
    acc[j + 1] += lower ? 0.f : ss;
  }
  // The four sums over the warp by recursive halving: after the exchanges at distances 16 and 8
  // each lane carries one pair's partial sum, pair (lane >> 3) & 3, which the last three levels
  // complete; each piece then reads its pair's total from lane 8 q.
  const bool b4 = lane & 16, b3 = lane & 8;
  const float k0 = b4 ? acc[2] : acc[0], k1 = b4 ? acc[3] : acc[1];
  const float r0 = __shfl_xor_sync(0xffffffffu, b4 ? acc[0] : acc[2], 16);
  const float r1 = __shfl_xor_sync(0xffffffffu, b4 ? acc[1] : acc[3], 16);
  const float m0 = k0 + r0, m1 = k1 + r1;
  float tot = (b3 ? m1 : m0) + __shfl_xor_sync(0xffffffffu, b3 ? m0 : m1, 8);
#pragma unroll
  for (int off = 4; off > 0; off >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, off);
  const int h0 = (int)(base % H);
#pragma unroll
  for (int j = 0; j < NG_PIECES; ++j) {
    const int p = lane + 32 * j;
    const bool lower = p < 24 * (j + 1);
    const int q = lower ? j : j + 1, c = 8 * (p - 24 * q);
    const float ssq = __shfl_sync(0xffffffffu, tot, 8 * q);
    int hq = h0 + q;  // (h0 + q) mod H, q < 4
#pragma unroll
    for (int t = 1; t < NG_PAIRS; ++t) hq = hq >= H ? hq - H : hq;
    const int tr = base + q < pairs ? __ldg(tier + hq) : 0;
    if (base + q < pairs && (tr < 0 || tr >= n_tiers)) {  // a tier outside the gains: the row is left untouched
      if (c == 0) raise_error(err, ERR_SHAPE);
    } else if (base + q < pairs) {
      const float inv = rsqrtf(ssq * (1.f / DV) + eps);
      const float2 inv2 = make_float2(inv, inv);
      const float4 w0 = __ldg(reinterpret_cast<const float4*>(w + tr * DV + c));
      const float4 w1 = __ldg(reinterpret_cast<const float4*>(w + tr * DV + c) + 1);
      const float2 wv[4] = {make_float2(w0.x, w0.y), make_float2(w0.z, w0.w), make_float2(w1.x, w1.y),
                            make_float2(w1.z, w1.w)};
      float2 gg[4], r[4];
      unpack8(rg[j], gg);
#pragma unroll
      for (int e = 0; e < 4; ++e) r[e] = pmul(pmul(x[j][e], inv2), pmul(wv[e], silu2<T>(gg[e])));
      store8(y + base * DV + p * 8, r);
    }
  }
}

}  // namespace

cudaError_t launch_head_norm_gate(int dtype_f32, const void* o, const void* g, const float* w,
                                  const int32_t* tier, int n_tiers, float eps, void* y, long long rows,
                                  int H, unsigned* err, cudaStream_t stream) {
  const long long pairs = rows * H;
  if (pairs == 0) return cudaSuccess;
  const long long blocks = (pairs + NG_WARPS * NG_PAIRS - 1) / (NG_WARPS * NG_PAIRS);
  if (dtype_f32) {
    head_norm_gate_kernel<float><<<(unsigned)blocks, NG_WARPS * 32, 0, stream>>>(
        (const float*)o, (const float*)g, w, tier, n_tiers, eps, (float*)y, pairs, H, err);
  } else {
    head_norm_gate_kernel<__nv_bfloat16><<<(unsigned)blocks, NG_WARPS * 32, 0, stream>>>(
        (const __nv_bfloat16*)o, (const __nv_bfloat16*)g, w, tier, n_tiers, eps, (__nv_bfloat16*)y,
        pairs, H, err);
  }
  return cudaGetLastError();
}

}  // namespace gla
