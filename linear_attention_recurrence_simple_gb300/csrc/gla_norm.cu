// Per-tier Head RMSNorm and SiLU output gate of the mixer's output.
//
// "Beyond the KV cache" (Laplace 3B on Trainium2), section "i14 and the Laplace 3B architecture":
// the per-head outputs pass through a Head RMSNorm within each decay tier (the heads of a tier
// share one norm: "Head RMSNorm (per tier)" in the architecture table), are concatenated and
// gated by SiLU(g_t), g_t being the gate stream of the QKVG projection.  For row t, head h:
//     y = o / sqrt(mean_c o_c^2 + eps) * w_{tier(h)} * SiLU(g),   SiLU(x) = x sigmoid(x).
// The RMS needs all 192 channels of a head's row, which the chunk scans split over three CTAs,
// so this is its own pass: a stream over o and g (read once) and y (written once).  Each CTA
// first copies the tier gains and the head-to-tier map into shared memory; a warp then takes
// four consecutive (row, head) pairs and issues all their loads first (enough bytes in flight
// to cover the memory latency); per pair, 24 lanes hold 8 consecutive channels each (16-byte
// bf16 / two 16-byte fp32 loads) and the sum of squares is reduced across the warp.
#include "gla_common.cuh"

namespace gla {
namespace {

constexpr int NG_WARPS = 8;  // warps per CTA
constexpr int NG_PAIRS = 4;  // (row, head) pairs per warp
// The shared-memory copies hold at most 32 tiers of gains and 4,096 heads' tiers (40 KB, within
// the default dynamic shared-memory limit); the caller refuses larger calls.

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
__device__ __forceinline__ void unpack8(const Raw8<__nv_bfloat16>& r, float (&x)[8]) {
  const uint32_t w[4] = {r.u[0].x, r.u[0].y, r.u[0].z, r.u[0].w};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[e]));
    x[2 * e] = f.x;
    x[2 * e + 1] = f.y;
  }
}
__device__ __forceinline__ void unpack8(const Raw8<float>& r, float (&x)[8]) {
  const uint32_t w[8] = {r.u[0].x, r.u[0].y, r.u[0].z, r.u[0].w, r.u[1].x, r.u[1].y, r.u[1].z, r.u[1].w};
#pragma unroll
  for (int e = 0; e < 8; ++e) x[e] = __uint_as_float(w[e]);
}
__device__ __forceinline__ void store8(__nv_bfloat16* p, const float (&x)[8]) {
  uint32_t w[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const __nv_bfloat162 b = __floats2bfloat162_rn(x[2 * e], x[2 * e + 1]);
    w[e] = *reinterpret_cast<const uint32_t*>(&b);
  }
  *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
}
__device__ __forceinline__ void store8(float* p, const float (&x)[8]) {
  reinterpret_cast<float4*>(p)[0] = make_float4(x[0], x[1], x[2], x[3]);
  reinterpret_cast<float4*>(p)[1] = make_float4(x[4], x[5], x[6], x[7]);
}

// SiLU(g) = g sigmoid(g) = g (1 + tanh(g / 2)) / 2.  bf16 data: the hardware tanh approximation
// (relative error about 2^-11, far inside a bf16 rounding); fp32 data: CUDA's accurate tanhf.
__device__ __forceinline__ float tanh_fast(float x) {
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
template <class T> __device__ __forceinline__ float silu(float g);
template <> __device__ __forceinline__ float silu<__nv_bfloat16>(float g) {
  return g * fmaf(0.5f, tanh_fast(0.5f * g), 0.5f);
}
template <> __device__ __forceinline__ float silu<float>(float g) {
  return g * fmaf(0.5f, tanhf(0.5f * g), 0.5f);
}

template <class T>
__global__ void __launch_bounds__(NG_WARPS * 32)
head_norm_gate_kernel(const T* __restrict__ o, const T* __restrict__ g, const float* __restrict__ w,
                      const int32_t* __restrict__ tier, int n_tiers, float eps, T* __restrict__ y,
                      long long pairs, int H, unsigned* err) {
  extern __shared__ float ng_smem[];
  float* const ws = ng_smem;                                            // [n_tiers][192]
  int* const ts = reinterpret_cast<int*>(ng_smem + n_tiers * DV);     // [H]
  for (int e = threadIdx.x; e < n_tiers * DV; e += NG_WARPS * 32) ws[e] = w[e];
  for (int e = threadIdx.x; e < H; e += NG_WARPS * 32) ts[e] = tier[e];
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const long long rh0 = ((long long)blockIdx.x * NG_WARPS + (threadIdx.x >> 5)) * NG_PAIRS;  // row * H + head
  Raw8<T> ro[NG_PAIRS], rg[NG_PAIRS];
  // Unconditional loads (indices clamped into range; lanes 24..31 repeat lane 23's piece), so
  // that all of them issue before the first use.
  const int lp = lane < DV / 8 ? lane : DV / 8 - 1;
#pragma unroll
  for (int k = 0; k < NG_PAIRS; ++k) {
    const long long rk = rh0 + k < pairs ? rh0 + k : pairs - 1;
    ro[k] = load_raw8(o + rk * DV + 8 * lp);
    rg[k] = load_raw8(g + rk * DV + 8 * lp);
  }
#pragma unroll
  for (int k = 0; k < NG_PAIRS; ++k) {
    const long long rh = rh0 + k;
    if (rh >= pairs) break;
    const int h = (int)(rh % H);
    const int tr = ts[h];
    if (tr < 0 || tr >= n_tiers) {  // a tier outside the gains: the row is left untouched
      if (lane == 0) raise_error(err, ERR_SHAPE);
      continue;
    }
    float x[8], gg[8];
    unpack8(ro[k], x);
    float ss = 0.f;
    if (lane < DV / 8) {
#pragma unroll
      for (int e = 0; e < 8; ++e) ss = fmaf(x[e], x[e], ss);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    if (lane < DV / 8) {
      const float inv = rsqrtf(ss * (1.f / DV) + eps);
      const float4 w0 = reinterpret_cast<const float4*>(ws + tr * DV + 8 * lane)[0];
      const float4 w1 = reinterpret_cast<const float4*>(ws + tr * DV + 8 * lane)[1];
      const float wv[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
      unpack8(rg[k], gg);
      float r[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) r[e] = (x[e] * inv) * (wv[e] * silu<T>(gg[e]));
      store8(y + rh * DV + 8 * lane, r);
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
  const size_t smem = (size_t)n_tiers * DV * sizeof(float) + (size_t)H * sizeof(int);
  if (dtype_f32) {
    head_norm_gate_kernel<float><<<(unsigned)blocks, NG_WARPS * 32, smem, stream>>>(
        (const float*)o, (const float*)g, w, tier, n_tiers, eps, (float*)y, pairs, H, err);
  } else {
    head_norm_gate_kernel<__nv_bfloat16><<<(unsigned)blocks, NG_WARPS * 32, smem, stream>>>(
        (const __nv_bfloat16*)o, (const __nv_bfloat16*)g, w, tier, n_tiers, eps, (__nv_bfloat16*)y,
        pairs, H, err);
  }
  return cudaGetLastError();
}

}  // namespace gla
