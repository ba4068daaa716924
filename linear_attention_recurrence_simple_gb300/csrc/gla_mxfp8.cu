// Decode state stored as MXFP8 (not on the pages: a storage variant that quarters the state
// stream of the decode step; the pages keep fp32 states, 29.5 MB per sequence).
//
// Format: OCP "Microscaling Formats (MX)" v1.0, MXFP8 with E4M3 elements.  Each state row of 192
// values is six blocks of 32; a block holds 32 E4M3 codes (OCP 8-bit floating point: bias 7,
// largest finite 448, subnormals m 2^-9) and one E8M0 scale byte b, value 2^(b - 127).  A state
// [96 x 192] is 18,432 code bytes plus 576 scale bytes (19,008 bytes against 73,728 in fp32).
// Quantisation of a block of fp32 values: the shared exponent is floor(log2(max |x|)) - 8, raised
// by one when the block maximum would then exceed 448 (so nothing saturates; the MX rule alone
// would clip maxima in [448, 512) 2^se to 448), clamped to [-127, 127] (-127 for an all-zero
// block); each element is x 2^-se (exact: a power of two) rounded to E4M3, to nearest, ties to
// even (cvt.rn.satfinite).  Every decision is a function of the fp32 values alone.
//
// Decode step ("Beyond the KV cache", section "i14 and the Laplace 3B architecture", GLA mixer;
// section "Optimizing inference on Trainium2", one state page per sequence): the state is widened
// exactly to fp32, S <- lambda S + k v^T and o = S^T (scale q) run in fp32 as in the fp32-state
// step (the readout from the update before it is stored), and the update is quantised back.
// One CTA of 192 threads per state: thread (g, p), g < 16, p < 12, holds the 16-byte piece p
// (columns 16p .. 16p + 15) of rows g, g + 16, ..., g + 80; the two pieces of a 32-column block
// sit in lanes t and t ^ 1 of one warp, which exchange their maxima with one shuffle.  All six
// code loads are issued before any arithmetic; the readout's sum over d_k runs in registers,
// then over the 16 row groups through shared memory.
#include <cuda_fp16.h>

#include <algorithm>

#include "gla_common.cuh"

namespace gla {
namespace {

constexpr int MX_THREADS = 192;
constexpr int MX_PIECES = DV / 16;                 // 12 16-byte pieces per row
constexpr int MX_GROUPS = MX_THREADS / MX_PIECES;  // 16 row groups
constexpr int MX_ROWS = DK / MX_GROUPS;            // 6 rows per thread
constexpr int MX_BLOCKS = DV / 32;                 // 6 scales per row
constexpr int MX_SCALE_BYTES = DK * MX_BLOCKS;     // 576 per state

// Two E4M3 codes (low byte first in memory) to fp32, exactly.
__device__ __forceinline__ float2 e4m3x2_to_f2(uint32_t two) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"((unsigned short)two));
  return __half22float2(*reinterpret_cast<const __half2*>(&h2));
}
// Two fp32 values to E4M3 (to nearest, ties to even, saturating), `lo` in the low byte.
__device__ __forceinline__ uint32_t f2_to_e4m3x2(float lo, float hi) {
  unsigned short r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}
// E8M0 scale byte to its fp32 value 2^(b - 127) (b = 0: the subnormal 2^-127; 255: NaN).
__device__ __forceinline__ float e8m0_to_f(uint32_t b) {
  return b == 0 ? __uint_as_float(0x00400000u) : (b == 255 ? __uint_as_float(0x7FC00000u) : __uint_as_float(b << 23));
}
// Shared exponent of a block whose largest magnitude is m (fp32, finite): floor(log2 m) - 8,
// plus one when m's significand exceeds 1.75 (then m 2^-(floor - 8) > 448), clamped to
// [-127, 127]; -127 for zero or subnormal m.
__device__ __forceinline__ int mx_shared_exp(float m) {
  const uint32_t bits = __float_as_uint(m);
  const int E = (int)((bits >> 23) & 0xFFu);
  if (E == 0) return -127;
  const int se = E - 135 + ((bits & 0x7FFFFFu) > 0x600000u ? 1 : 0);
  return max(se, -127);
}
// Pairs of fp32 values through the packed two-lane instructions (each lane rounded as its scalar
// counterpart, so the results are those of the scalar code).
__device__ __forceinline__ uint64_t f2b(float a, float b) { return ((uint64_t)__float_as_uint(b) << 32) | __float_as_uint(a); }
__device__ __forceinline__ void b2f(uint64_t r, float& a, float& b) {
  a = __uint_as_float((uint32_t)r);
  b = __uint_as_float((uint32_t)(r >> 32));
}
__device__ __forceinline__ uint64_t pmul(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t pfma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
// 2^-se as fp32 (se in [-127, 120]).
__device__ __forceinline__ float pow2_neg(int se) { return __uint_as_float((uint32_t)(127 - se) << 23); }

// 16 fp32 values -> 16 codes (one uint4), given the block's shared exponent.
__device__ __forceinline__ uint4 quantise16(const float (&x)[16], int se) {
  const float inv = pow2_neg(se);
  const uint64_t inv2 = f2b(inv, inv);
  uint32_t w[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    float y0, y1, y2, y3;
    b2f(pmul(f2b(x[4 * j], x[4 * j + 1]), inv2), y0, y1);
    b2f(pmul(f2b(x[4 * j + 2], x[4 * j + 3]), inv2), y2, y3);
    w[j] = f2_to_e4m3x2(y0, y1) | (f2_to_e4m3x2(y2, y3) << 16);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}
__device__ __forceinline__ void dequantise16(uint4 c, float scale, float (&x)[16]) {
  const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float2 a = e4m3x2_to_f2(w[j] & 0xFFFFu), b = e4m3x2_to_f2(w[j] >> 16);
    x[4 * j] = a.x * scale;
    x[4 * j + 1] = a.y * scale;
    x[4 * j + 2] = b.x * scale;
    x[4 * j + 3] = b.y * scale;
  }
}
__device__ __forceinline__ void fence_async_smem_mx() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// Largest magnitude of the block whose two 16-value halves sit in lanes t and t ^ 1.
__device__ __forceinline__ float block_max(const float (&x)[16]) {
  float m = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) m = fmaxf(m, fabsf(x[i]));
  return fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
}

// fp32 rows of 192 -> MXFP8 codes and scales; one thread per 16-value piece (12 per row).
__global__ void mxfp8_quantise_kernel(const float4* __restrict__ x, uint4* __restrict__ codes,
                                      uint8_t* __restrict__ scales, long long pieces) {
  const long long stride = (long long)gridDim.x * blockDim.x;  // a multiple of 32 (even)
  for (long long t = blockIdx.x * (long long)blockDim.x + threadIdx.x; t - (threadIdx.x & 31) < pieces; t += stride) {
    const bool live = t < pieces;  // whole warps stay in the loop for the shuffle
    const long long tt = live ? t : pieces - 1;
    float v[16];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float4 f = x[tt * 4 + j];
      v[4 * j] = f.x;
      v[4 * j + 1] = f.y;
      v[4 * j + 2] = f.z;
      v[4 * j + 3] = f.w;
    }
    const int se = mx_shared_exp(block_max(v));
    if (live) {
      codes[t] = quantise16(v, se);
      if ((t & 1) == 0) scales[t >> 1] = (uint8_t)(se + 127);
    }
  }
}

__global__ void mxfp8_dequantise_kernel(const uint4* __restrict__ codes, const uint8_t* __restrict__ scales,
                                        float4* __restrict__ x, long long pieces) {
  for (long long t = blockIdx.x * (long long)blockDim.x + threadIdx.x; t < pieces;
       t += (long long)gridDim.x * blockDim.x) {
    float v[16];
    dequantise16(codes[t], e8m0_to_f(scales[t >> 1]), v);
#pragma unroll
    for (int j = 0; j < 4; ++j) x[t * 4 + j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
  }
}

template <class T>
__device__ __forceinline__ void load16(const T* p, float (&v)[16]);
template <>
__device__ __forceinline__ void load16<float>(const float* p, float (&v)[16]) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float4 f = reinterpret_cast<const float4*>(p)[j];
    v[4 * j] = f.x;
    v[4 * j + 1] = f.y;
    v[4 * j + 2] = f.z;
    v[4 * j + 3] = f.w;
  }
}
template <>
__device__ __forceinline__ void load16<__nv_bfloat16>(const __nv_bfloat16* p, float (&v)[16]) {
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const uint4 u = reinterpret_cast<const uint4*>(p)[j];
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[e]));
      v[8 * j + 2 * e] = f.x;
      v[8 * j + 2 * e + 1] = f.y;
    }
  }
}
__device__ __forceinline__ void store_out(float* p, float x) { *p = x; }
__device__ __forceinline__ void store_out(__nv_bfloat16* p, float x) { *p = __float2bfloat16_rn(x); }

// Byte offsets of one pipeline slot: a state's codes and scales, the step's q, k, v rows, and a
// small header (skip flag, the state's index in the pool).  Every piece is 16-byte aligned.
template <class T>
struct MxSlot {
  static constexpr uint32_t CODES = 0;
  static constexpr uint32_t SCALES = DK * DV;
  static constexpr uint32_t Q = SCALES + MX_SCALE_BYTES;
  static constexpr uint32_t K = Q + DK * (uint32_t)sizeof(T);
  static constexpr uint32_t V = K + DK * (uint32_t)sizeof(T);
  static constexpr uint32_t META = V + DV * (uint32_t)sizeof(T);
  static constexpr uint32_t BYTES = (META + 16 + 127) / 128 * 128;
  static constexpr uint32_t LOAD_BYTES = META;  // the bulk copies of one state
};
template <class T>
struct MxSmem {
  static constexpr uint32_t PART = 2 * MxSlot<T>::BYTES;           // readout partials [16][192] fp32
  static constexpr uint32_t BARS = PART + MX_GROUPS * DV * 4;      // two mbarriers
  static constexpr uint32_t MISC = BARS + 16;                      // abort flag, gate
  static constexpr uint32_t BYTES = MISC + 16;
};
constexpr int MX_CTAS_PER_SM = 4;
constexpr unsigned long long MX_DRAIN_NS = 1000000000ull;

__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_u32(dst)),
               "l"(src), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}
__device__ __forceinline__ void bulk_store(void* dst, const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(smem_u32(src)),
               "r"(bytes)
               : "memory");
}

// Persistent CTAs, each stepping the states blockIdx.x, blockIdx.x + gridDim.x, ... through a
// two-slot pipeline: while the CTA updates the state in one slot, the next state's codes,
// scales and q, k, v rows land in the other (bulk copies issued by thread 0 and counted by the
// slot's mbarrier); the updated codes and scales are written back in place in shared memory and
// leave with one bulk store, and the slot is refilled once that store has read it.  Every wait
// is bounded: past `wait_ns` the CTA records GLA_ERR_TIMEOUT, drains its copies in flight and
// returns.
template <class T>
__global__ void __launch_bounds__(MX_THREADS, MX_CTAS_PER_SM)
decode_step_mxfp8_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                         const float* __restrict__ log_lambda, float scale, uint8_t* __restrict__ codes,
                         uint8_t* __restrict__ scales, const int32_t* __restrict__ slot, int pool_rows,
                         T* __restrict__ o, long long total, int H, const float* __restrict__ aug, unsigned* err,
                         unsigned long long wait_ns) {
  using SL = MxSlot<T>;
  using SM = MxSmem<T>;
  extern __shared__ __align__(128) uint8_t mx_smem[];
  float(*s_part)[DV] = reinterpret_cast<float(*)[DV]>(mx_smem + SM::PART);
  uint64_t* full = reinterpret_cast<uint64_t*>(mx_smem + SM::BARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(mx_smem + SM::MISC);
  float* s_gate = reinterpret_cast<float*>(mx_smem + SM::MISC + 4);

  const int tid = threadIdx.x;
  const int p = tid % MX_PIECES;
  const int g = tid / MX_PIECES;
  if (tid == 0) {
    mbar_init(&full[0], 1);
    mbar_init(&full[1], 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

  // Thread 0: the loads of state j into slot s (or, for a pool slot out of range, an error, the
  // skip flag and a bare arrival that completes the slot's phase).
  auto issue = [&](long long j, int s) {
    uint8_t* sb = mx_smem + s * SL::BYTES;
    const int n = (int)(j / H), h = (int)(j % H);
    const int row = slot ? slot[n] : n;
    long long* meta = reinterpret_cast<long long*>(sb + SL::META);
    if (row < 0 || row >= pool_rows) {
      raise_error(err, ERR_SHAPE);
      meta[0] = -1;
      mbar_arrive(&full[s]);
      return;
    }
    const long long st = (long long)row * H + h;
    meta[0] = st;
    mbar_expect_tx(&full[s], SL::LOAD_BYTES);
    bulk_load(sb + SL::CODES, codes + st * (DK * DV), DK * DV, &full[s]);
    bulk_load(sb + SL::SCALES, scales + st * MX_SCALE_BYTES, MX_SCALE_BYTES, &full[s]);
    bulk_load(sb + SL::Q, q + j * DK, DK * sizeof(T), &full[s]);
    bulk_load(sb + SL::K, k + j * DK, DK * sizeof(T), &full[s]);
    bulk_load(sb + SL::V, v + j * DV, DV * sizeof(T), &full[s]);
  };

  const long long stride = gridDim.x;
  long long j = blockIdx.x;
  int issued = 0;  // states whose loads thread 0 has issued (iterations 0 .. issued - 1)
  if (tid == 0) {
    if (j < total) issue(j, 0), ++issued;
    if (j + stride < total) issue(j + stride, 1), ++issued;
  }
  int it = 0;
  for (; j < total; j += stride, ++it) {
    const int s = it & 1;
    // A thread whose wait gave up skips the state's work; the first barrier below is also the
    // vote, so every thread of the CTA then leaves the loop together.
    // (warp-uniform, so that the block's shuffles always see every lane)
    const bool ok = __all_sync(0xffffffffu, mbar_wait(&full[s], (uint32_t)(it >> 1) & 1u, wait_ns, abort_flag));
    uint8_t* sb = mx_smem + s * SL::BYTES;
    const long long st = ok ? *reinterpret_cast<const long long*>(sb + SL::META) : -1;
    const T* sq = reinterpret_cast<const T*>(sb + SL::Q);
    const T* sk = reinterpret_cast<const T*>(sb + SL::K);
    const T* sv = reinterpret_cast<const T*>(sb + SL::V);
    const int h = (int)(j % H);
    if (st >= 0) {
      float vv[16];
      load16(sv + 16 * p, vv);
      const float lam = expf(log_lambda[h]);
      float acc[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) acc[e] = 0.f;
#pragma unroll 2
      for (int i = 0; i < MX_ROWS; ++i) {
        const int a = g + MX_GROUPS * i;
        const float ka = to_f(sk[a]), qa = scale * to_f(sq[a]);
        uint4* cp = reinterpret_cast<uint4*>(sb + SL::CODES) + a * MX_PIECES + p;
        uint8_t* scp = sb + SL::SCALES + a * MX_BLOCKS + (p >> 1);
        // x = fma(lambda, code * scale, k_a v) as in the fp32-state step.  The scale is a power
        // of two, so lambda * scale is exact while it is a normal fp32 number (or lambda is 0),
        // and fma(lambda * scale, code, k_a v) is then the same value with one multiply less.
        const float sc = e8m0_to_f(*scp);
        const float lsc = lam * sc;
        float x[16];
        const bool fold = lsc >= 1.17549435e-38f || lam == 0.f;
        if (fold)
          dequantise16(*cp, 1.f, x);  // (no multiply: the scale rides in lambda)
        else
          dequantise16(*cp, sc, x);
        const uint64_t l2 = fold ? f2b(lsc, lsc) : f2b(lam, lam), k2 = f2b(ka, ka), q2 = f2b(qa, qa);
#pragma unroll
        for (int e = 0; e < 16; e += 2) {
          b2f(pfma(l2, f2b(x[e], x[e + 1]), pmul(k2, f2b(vv[e], vv[e + 1]))), x[e], x[e + 1]);
          b2f(pfma(q2, f2b(x[e], x[e + 1]), f2b(acc[e], acc[e + 1])), acc[e], acc[e + 1]);
        }
        const int se = mx_shared_exp(block_max(x));
        *cp = quantise16(x, se);  // in place: this thread's own 16 bytes
        // (both lanes of the block read this byte above, before the shuffle in block_max)
        if ((p & 1) == 0) *scp = (uint8_t)(se + 127);
      }
#pragma unroll
      for (int e = 0; e < 16; e += 4)
        *reinterpret_cast<float4*>(&s_part[g][16 * p + e]) = make_float4(acc[e], acc[e + 1], acc[e + 2], acc[e + 3]);
      if (aug && tid < 32) {  // gate = sigmoid(q . (a_h * k)), q unscaled
        float gt = 0.f;
#pragma unroll
        for (int d = tid; d < DK; d += 32) gt = fmaf(to_f(sq[d]) * aug[h * DK + d], to_f(sk[d]), gt);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) gt += __shfl_xor_sync(0xffffffffu, gt, off);
        if (tid == 0) *s_gate = 1.f / (1.f + expf(-gt));
      }
    }
    fence_async_smem_mx();  // the new codes and scales are read next by the bulk store
    if (__syncthreads_or(!ok)) break;
    if (st >= 0) {
      if (tid == 0) {
        bulk_store(codes + st * (DK * DV), sb + SL::CODES, DK * DV);
        bulk_store(scales + st * MX_SCALE_BYTES, sb + SL::SCALES, MX_SCALE_BYTES);
        asm volatile("cp.async.bulk.commit_group;" ::: "memory");
      }
      float t = 0.f;  // output column tid (tid < 192 = d_v)
#pragma unroll
      for (int r = 0; r < MX_GROUPS; ++r) t += s_part[r][tid];
      if (aug) t = fmaf(*s_gate, to_f(sv[tid]), t);
      store_out(o + j * DV + tid, t);
    }
    __syncthreads();  // slot s and the partials are free again
    if (tid == 0 && j + 2 * stride < total) {
      asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");  // the store has read slot s
      issue(j + 2 * stride, s);
      ++issued;
    }
  }
  if (tid == 0) {
    // after a timeout: no copy into shared memory may still be in flight when the CTA exits
    for (int i = it; i < issued; ++i) mbar_wait_drain(&full[i & 1], (uint32_t)(i >> 1) & 1u, MX_DRAIN_NS, err);
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
    if (*abort_flag) raise_error(err, ERR_TIMEOUT);
  }
}

}  // namespace

cudaError_t launch_mxfp8_quantise(const float* x, uint8_t* codes, uint8_t* scales, long long rows,
                                  cudaStream_t stream) {
  const long long pieces = rows * MX_PIECES;
  if (pieces == 0) return cudaSuccess;
  long long blocks = (pieces + 255) / 256;
  if (blocks > 152 * 16) blocks = 152 * 16;
  mxfp8_quantise_kernel<<<(unsigned)blocks, 256, 0, stream>>>(reinterpret_cast<const float4*>(x),
                                                              reinterpret_cast<uint4*>(codes), scales, pieces);
  return cudaGetLastError();
}

cudaError_t launch_mxfp8_dequantise(const uint8_t* codes, const uint8_t* scales, float* x, long long rows,
                                    cudaStream_t stream) {
  const long long pieces = rows * MX_PIECES;
  if (pieces == 0) return cudaSuccess;
  long long blocks = (pieces + 255) / 256;
  if (blocks > 152 * 16) blocks = 152 * 16;
  mxfp8_dequantise_kernel<<<(unsigned)blocks, 256, 0, stream>>>(reinterpret_cast<const uint4*>(codes), scales,
                                                                reinterpret_cast<float4*>(x), pieces);
  return cudaGetLastError();
}

cudaError_t launch_decode_step_mxfp8(int dtype_f32, const void* q, const void* k, const void* v,
                                     const float* log_lambda, float scale, uint8_t* codes, uint8_t* scales,
                                     const int32_t* slot, int pool_rows, void* o, int N, int H,
                                     const float* aug, unsigned* err, unsigned long long wait_ns,
                                     cudaStream_t stream) {
  const long long total = (long long)N * H;
  if (total == 0) return cudaSuccess;
  int dev = 0, sms = 152;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const long long ctas = std::min(total, (long long)sms * MX_CTAS_PER_SM);
  using BF = __nv_bfloat16;
  static bool attr_set[2] = {false, false};
  cudaError_t e;
  if (dtype_f32) {
    if (!attr_set[1]) {
      if ((e = cudaFuncSetAttribute(decode_step_mxfp8_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)MxSmem<float>::BYTES)) != cudaSuccess)
        return e;
      attr_set[1] = true;
    }
    decode_step_mxfp8_kernel<float><<<(unsigned)ctas, MX_THREADS, MxSmem<float>::BYTES, stream>>>(
        (const float*)q, (const float*)k, (const float*)v, log_lambda, scale, codes, scales, slot, pool_rows,
        (float*)o, total, H, aug, err, wait_ns);
  } else {
    if (!attr_set[0]) {
      if ((e = cudaFuncSetAttribute(decode_step_mxfp8_kernel<BF>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)MxSmem<BF>::BYTES)) != cudaSuccess)
        return e;
      attr_set[0] = true;
    }
    decode_step_mxfp8_kernel<BF><<<(unsigned)ctas, MX_THREADS, MxSmem<BF>::BYTES, stream>>>(
        (const BF*)q, (const BF*)k, (const BF*)v, log_lambda, scale, codes, scales, slot, pool_rows, (BF*)o,
        total, H, aug, err, wait_ns);
  }
  return cudaGetLastError();
}

}  // namespace gla
