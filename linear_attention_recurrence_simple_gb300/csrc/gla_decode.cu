// One-token decode step over a pool of fp32 GLA states, in place.
//
// "Beyond the KV cache" (Laplace 3B on Trainium2), section "i14 and the Laplace 3B
// architecture", GLA mixer: S <- lambda_h S + k v^T (rank-1 write of the current key/value,
// fixed per-head decay), then the readout o = S^T (scale q) queries the updated state.  Section
// "Optimizing inference on Trainium2": the serving wrapper keeps one fixed page of recurrent state
// per sequence in a pool, which `slot` indexes here.  With `aug` (aug_balance, [H, 96]) the
// output also gains the self-augmentation copy of the value, sigmoid(q . (a_h * k)) v (the
// paragraph after the readout in the same section; the query enters the gate unscaled).
// The state may also be stored in bf16 (not on the pages: a storage variant that halves the
// stream): it is read and widened to fp32, updated and read out in fp32, and rounded to bf16 (to
// nearest, ties to even) when it is written back.
//
// With the fused norm (NormGate given), the output row is not stored as o: it goes through the
// per-tier Head RMSNorm and the SiLU(g) gate of the same section ("the per-head outputs pass
// through a Head RMSNorm within each decay tier, then the SiLU(g) gate"), and y is stored:
//     y = o / sqrt(mean_c o_c^2 + eps) * w_{tier(h)} * SiLU(g),
// from the fp32 readout (before any rounding of o).  The CTA holds the head's whole 192-wide
// row, so the mean square is a reduction over its first 48 threads.
//
// The step is a pure stream over the 72 KB state of each (sequence, head): read once, update,
// write once.  One CTA owns one state; thread (r, c), c < 48, holds columns 4c..4c+3 (one
// vector) of the rows r, r + G, r + 2G, ... for G row groups, so consecutive lanes touch
// consecutive pieces of a row: fp32 states with 576 threads (G = 12, 8 rows of 16-byte vectors
// each, 2 CTAs per SM), bf16 states with 288 threads (G = 6, 16 rows of 8-byte vectors kept packed
// until use, 4 CTAs per SM: twice the bytes in flight per SM of 576-thread CTAs).  All of a
// thread's loads are issued before any arithmetic.  The readout's sum over d_k runs in
// registers, then over the G row groups through shared memory.  Loads and stores carry the
// streaming cache hint, since each state is touched once per step.
#include "gla_common.cuh"

namespace gla {
namespace {

constexpr int DEC_COLS = DV / 4;              // 48 four-column vectors per state row
// CTA shape per state storage type: threads (48 column groups x RGROUPS row groups), rows per
// thread, CTAs per SM.
template <class ST> struct DecCfg;
template <> struct DecCfg<float> { static constexpr int THREADS = 576, MIN_BLOCKS = 2; };
template <> struct DecCfg<__nv_bfloat16> { static constexpr int THREADS = 288, MIN_BLOCKS = 4; };

struct Bf16x4 { __nv_bfloat162 a, b; };

__device__ __forceinline__ float4 load4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ float4 load4(const __nv_bfloat16* p) {
  const uint2 u = *reinterpret_cast<const uint2*>(p);
  const float2 lo = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
  const float2 hi = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
  return make_float4(lo.x, lo.y, hi.x, hi.y);
}
__device__ __forceinline__ void store4(float* p, float4 x) { *reinterpret_cast<float4*>(p) = x; }
// State vectors (4 consecutive columns) with the streaming cache hint: fp32 storage as float4,
// bf16 storage as uint2 (four bf16).
template <class ST> struct StateVec;
template <> struct StateVec<float> { using type = float4; };
template <> struct StateVec<__nv_bfloat16> { using type = uint2; };
// A state vector as loaded, widened to fp32 at use (bf16 vectors stay packed in between, so the
// loads in flight hold half the registers).
__device__ __forceinline__ float4 widen_state(float4 x) { return x; }
__device__ __forceinline__ float4 widen_state(uint2 u) {
  const float2 lo = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
  const float2 hi = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
  return make_float4(lo.x, lo.y, hi.x, hi.y);
}
__device__ __forceinline__ void store_state(float4* p, float4 x) { __stcs(p, x); }
__device__ __forceinline__ void store_state(uint2* p, float4 x) {
  const __nv_bfloat162 a = __floats2bfloat162_rn(x.x, x.y), b = __floats2bfloat162_rn(x.z, x.w);
  __stcs(p, make_uint2(*reinterpret_cast<const uint32_t*>(&a), *reinterpret_cast<const uint32_t*>(&b)));
}
__device__ __forceinline__ void store4(__nv_bfloat16* p, float4 x) {
  Bf16x4 r;
  r.a = __floats2bfloat162_rn(x.x, x.y);
  r.b = __floats2bfloat162_rn(x.z, x.w);
  *reinterpret_cast<Bf16x4*>(p) = r;
}

// The fused Head RMSNorm + SiLU gate's inputs: g [N, H, 192] (the gate stream, dtype of o),
// weight [n_tiers, 192] fp32 (each tier's gain), tier [H] int32, eps.
template <class T>
struct NormGate {
  const T* g;
  const float* w;
  const int32_t* tier;
  int n_tiers;
  float eps;
};

// SiLU(x) = x sigmoid(x) = x (1 + tanh(x / 2)) / 2: the hardware tanh approximation for bf16
// data (relative error about 2^-11, inside a bf16 rounding), CUDA's tanhf for fp32 data.
__device__ __forceinline__ float dec_tanh_fast(float x) {
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float dec_silu(float g, __nv_bfloat16) { return g * fmaf(0.5f, dec_tanh_fast(0.5f * g), 0.5f); }
__device__ __forceinline__ float dec_silu(float g, float) { return g * fmaf(0.5f, tanhf(0.5f * g), 0.5f); }

template <class T, class ST, bool NG>
__global__ void __launch_bounds__(DecCfg<ST>::THREADS, DecCfg<ST>::MIN_BLOCKS)
decode_step_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                   const float* __restrict__ log_lambda, float scale, ST* __restrict__ state,
                   const int32_t* __restrict__ slot, int pool_rows, T* __restrict__ o, int H,
                   const float* __restrict__ aug, unsigned* err, const NormGate<T> ng) {
  __shared__ float s_q[DK];
  __shared__ float s_k[DK];
  __shared__ float s_gate;
  __shared__ float s_ss[2];
  constexpr int RG = DecCfg<ST>::THREADS / DEC_COLS, ROWS = DK / RG;
  __shared__ float4 s_part[RG][DEC_COLS];

  const long long nh = blockIdx.x;  // n * H + h
  const int n = (int)(nh / H);
  const int h = (int)(nh % H);
  const int tid = threadIdx.x;
  const int c = tid % DEC_COLS;
  const int r = tid / DEC_COLS;

  const int row = slot ? slot[n] : n;
  if (row < 0 || row >= pool_rows) {
    if (tid == 0) raise_error(err, ERR_SHAPE);
    return;
  }
  using SV = typename StateVec<ST>::type;
  SV* S = reinterpret_cast<SV*>(state + ((long long)row * H + h) * (DK * DV));

  SV s[ROWS];
#pragma unroll
  for (int i = 0; i < ROWS; ++i) s[i] = __ldcs(S + (r + RG * i) * DEC_COLS + c);

  if (tid < DK) {
    s_q[tid] = scale * to_f(q[nh * DK + tid]);
    s_k[tid] = to_f(k[nh * DK + tid]);
  }
  const float4 vv = load4(v + nh * DV + 4 * c);
  float4 gv = make_float4(0.f, 0.f, 0.f, 0.f);  // the gate stream's 4 channels (fused norm)
  if (NG && tid < DEC_COLS) gv = load4(ng.g + nh * DV + 4 * tid);
  const float lam = expf(log_lambda[h]);
  __syncthreads();

  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int i = 0; i < ROWS; ++i) {
    const int a = r + RG * i;
    const float ka = s_k[a], qa = s_q[a];
    float4 x = widen_state(s[i]);
    x.x = fmaf(lam, x.x, ka * vv.x);
    x.y = fmaf(lam, x.y, ka * vv.y);
    x.z = fmaf(lam, x.z, ka * vv.z);
    x.w = fmaf(lam, x.w, ka * vv.w);
    store_state(S + a * DEC_COLS + c, x);
    acc.x = fmaf(qa, x.x, acc.x);
    acc.y = fmaf(qa, x.y, acc.y);
    acc.z = fmaf(qa, x.z, acc.z);
    acc.w = fmaf(qa, x.w, acc.w);
  }
  s_part[r][c] = acc;
  if (aug && tid < 32) {  // gate = sigmoid(q . (a_h * k)), q unscaled
    float g = 0.f;
#pragma unroll
    for (int d = tid; d < DK; d += 32) g = fmaf(to_f(q[nh * DK + d]) * aug[h * DK + d], s_k[d], g);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) g += __shfl_xor_sync(0xffffffffu, g, off);
    if (tid == 0) s_gate = 1.f / (1.f + expf(-g));
  }
  __syncthreads();
  if (tid < (NG ? 64 : DEC_COLS)) {  // (fused norm: warps 0 and 1 whole, for the reduction)
    float4 t = make_float4(0.f, 0.f, 0.f, 0.f);
    if (tid < DEC_COLS) {
      t = s_part[0][tid];
#pragma unroll
      for (int g = 1; g < RG; ++g) {
        const float4 p = s_part[g][tid];
        t.x += p.x;
        t.y += p.y;
        t.z += p.z;
        t.w += p.w;
      }
      if (aug) {
        const float gate = s_gate;
        t.x = fmaf(gate, vv.x, t.x);
        t.y = fmaf(gate, vv.y, t.y);
        t.z = fmaf(gate, vv.z, t.z);
        t.w = fmaf(gate, vv.w, t.w);
      }
    }
    if constexpr (NG) {
      // mean square of the row's 192 channels: within warps 0 and 1, then across the two
      float ss = t.x * t.x + t.y * t.y + t.z * t.z + t.w * t.w;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
      if ((tid & 31) == 0) s_ss[tid >> 5] = ss;
      asm volatile("bar.sync 1, 64;" ::: "memory");
      const int tr = ng.tier[h];
      if (tr < 0 || tr >= ng.n_tiers) {  // a tier outside the gains: y is left untouched
        if (tid == 0) raise_error(err, ERR_SHAPE);
        return;
      }
      if (tid < DEC_COLS) {
        const float inv = rsqrtf((s_ss[0] + s_ss[1]) * (1.f / DV) + ng.eps);
        const float4 w = *reinterpret_cast<const float4*>(ng.w + tr * DV + 4 * tid);
        const T tag{};
        t.x = (t.x * inv) * (w.x * dec_silu(gv.x, tag));
        t.y = (t.y * inv) * (w.y * dec_silu(gv.y, tag));
        t.z = (t.z * inv) * (w.z * dec_silu(gv.z, tag));
        t.w = (t.w * inv) * (w.w * dec_silu(gv.w, tag));
        store4(o + nh * DV + 4 * tid, t);
      }
    } else {
      store4(o + nh * DV + 4 * tid, t);
    }
  }
}

template <class T, class ST>
void launch_decode_t(long long blocks, const void* q, const void* k, const void* v, const float* log_lambda,
                     float scale, void* state, const int32_t* slot, int pool_rows, void* o, int H,
                     const float* aug, unsigned* err, const DecodeNormGate* ngp, cudaStream_t stream) {
  if (ngp) {
    const NormGate<T> ng = {(const T*)ngp->g, ngp->w, ngp->tier, ngp->n_tiers, ngp->eps};
    decode_step_kernel<T, ST, true><<<(unsigned)blocks, DecCfg<ST>::THREADS, 0, stream>>>(
        (const T*)q, (const T*)k, (const T*)v, log_lambda, scale, (ST*)state, slot, pool_rows, (T*)o, H, aug,
        err, ng);
  } else {
    decode_step_kernel<T, ST, false><<<(unsigned)blocks, DecCfg<ST>::THREADS, 0, stream>>>(
        (const T*)q, (const T*)k, (const T*)v, log_lambda, scale, (ST*)state, slot, pool_rows, (T*)o, H, aug,
        err, NormGate<T>{});
  }
}

}  // namespace

// ngp: the fused Head RMSNorm + SiLU gate (o then receives y), or null for the plain readout.
cudaError_t launch_decode_step(int dtype_f32, int state_bf16, const void* q, const void* k, const void* v,
                               const float* log_lambda, float scale, void* state,
                               const int32_t* slot, int pool_rows, void* o, int N, int H,
                               const float* aug, unsigned* err, cudaStream_t stream,
                               const DecodeNormGate* ngp) {
  const long long blocks = (long long)N * H;
  if (blocks == 0) return cudaSuccess;
  using BF = __nv_bfloat16;
  if (dtype_f32 && !state_bf16)
    launch_decode_t<float, float>(blocks, q, k, v, log_lambda, scale, state, slot, pool_rows, o, H, aug, err, ngp, stream);
  else if (dtype_f32)
    launch_decode_t<float, BF>(blocks, q, k, v, log_lambda, scale, state, slot, pool_rows, o, H, aug, err, ngp, stream);
  else if (!state_bf16)
    launch_decode_t<BF, float>(blocks, q, k, v, log_lambda, scale, state, slot, pool_rows, o, H, aug, err, ngp, stream);
  else
    launch_decode_t<BF, BF>(blocks, q, k, v, log_lambda, scale, state, slot, pool_rows, o, H, aug, err, ngp, stream);
  return cudaGetLastError();
}

}  // namespace gla
