// Chunked GLA forward on the 5th-generation tensor cores (bf16 operands, fp32 accumulation and
// state): TMA -> shared memory -> tcgen05.mma -> tensor memory -> register epilogue.
//
// "Beyond the KV cache" (Laplace 3B on Trainium2), section "Challenge 1: Using native PyTorch on
// Trainium for GLA": within each 128-token chunk the output is decay-masked linear attention plus
// the contribution of the state carried from earlier chunks; the state then advances with the
// decay compounded over the chunk, and only that advance is sequential.  Per chunk of L tokens
// (local i, j; S = state before the chunk, s = scale):
//     A   = Q K^T                                   (MMA1: 128 x 128 x 96)
//     P   = s * lambda^(i-j) * A  for j <= i, else 0  (decay-mask warps, bf16, kept in TMEM)
//     O   = P V  +  diag(s lambda^(i+1)) (Q S)       (MMA2: 128 x 64 x 128, MMA3: 128 x 64 x 96)
//     S'  = lambda^L S + K^T Vt,  Vt_j = lambda^(L-1-j) v_j   (MMA4: 128(96) x 64 x 128)
// The decay is never split into lambda^i * lambda^-j, so lambda = 0.5 cannot overflow.
// Operands that carry the state are split into two bf16 terms, x = hi + lo with hi = bf16(x),
// lo = bf16(x - hi), and multiplied twice into the same fp32 accumulator: the state copy S in
// MMA3 and the decayed values Vt in MMA4.  That keeps about 16 significant bits on the state
// path; only P is a single bf16 rounding.
//
// Work split: one CTA per (sequence, head, 64-column tile of d_v); the three tiles of a head
// repeat the cheap Q K^T but share nothing else, which triples the CTA count for the 152 SMs.
// Each tcgen05.mma costs about 100 cycles to issue regardless of N <= 128, so the kernel keeps
// the instruction count low (28 per chunk: the hi/lo halves ride in one N = 128 MMA) and issues
// from three threads in parallel, one per independent accumulator chain.
// Warp roles (384 threads, 1 CTA per SM):
//   warp 0      TMA producer: Q, K, V chunk tiles into a 2-stage ring (72 KB per stage).
//   warp 1      allocates tensor memory; one lane issues MMA1 (Q K^T).
//   warp 2      one lane issues MMA4 (K^T [Vt_hi | Vt_lo]) and MMA3 (Q [S_hi | S_lo]).
//   warp 3      one lane issues MMA2 (P V, P read from tensor memory).
//   warps 4-7   per chunk: Vt = lambda^(L-1-j) V (hi and lo, zero past the sequence end), then
//               the decay mask A (TMEM) -> P (bf16 pairs, back into TMEM).  A is released as
//               soon as it is in registers, so the next chunk's Q K^T overlaps this one's P.
//   warps 8-11  epilogue: U (TMEM) -> S = lambda^L S + U in fp32 registers -> bf16 hi/lo copy of
//               S for the next chunk's Q S; O (TMEM: intra, inter hi, inter lo) -> o (bf16).
// Tensor memory (512 columns): A [0,128), P [128,192), O_intra [192,256), O_inter hi|lo
// [256,384), U hi|lo [384,512).  Every mbarrier wait is bounded (see gla_common.cuh); on a
// timeout the CTA records GLA_ERR_TIMEOUT, drains its copies and MMAs, frees tensor memory and
// returns.
#include <cuda.h>

#include "gla_common.cuh"

namespace gla {
namespace {

constexpr int TN = 64;             // d_v columns per CTA
constexpr int NTILE = DV / TN;     // 3
constexpr int NTHREADS = 384;

// ---- shared memory map (byte offsets from a 1024-byte aligned base) -------------------------
constexpr uint32_t SZ_Q0 = 128 * 128;        // d_k 0..63, K-major, 128B swizzle
constexpr uint32_t SZ_Q1 = 128 * 64;         // d_k 64..95, K-major, 64B swizzle
constexpr uint32_t SZ_K = 2 * 128 * 128;     // d_k 0..63 | 64..127 (96..127 zero-filled by TMA)
constexpr uint32_t SZ_V = 128 * 128;         // 64 d_v columns, 128B swizzle
constexpr uint32_t ST_Q0 = 0;
constexpr uint32_t ST_K = ST_Q0 + SZ_Q0;
constexpr uint32_t ST_V = ST_K + SZ_K;
constexpr uint32_t ST_Q1 = ST_V + SZ_V;
constexpr uint32_t SZ_STAGE = ST_Q1 + SZ_Q1;  // 73728
constexpr uint32_t OFF_VT = 2 * SZ_STAGE;    // Vt hi, then Vt lo (SZ_V each)
constexpr uint32_t OFF_SP = OFF_VT + 2 * SZ_V;
constexpr uint32_t SZ_SPH = 96 * 128;        // bf16 S tile: 96 rows (d_k) x 64 columns
constexpr uint32_t SZ_SP = 2 * SZ_SPH;       // one buffer: hi then lo
constexpr uint32_t OFF_PW = OFF_SP + 2 * SZ_SP;
constexpr uint32_t OFF_BAR = OFF_PW + 2 * 129 * 4 + 8;
enum {
  B_FULL = 0, B_EMPTY = 2, B_VT_FULL = 4, B_VT_EMPTY, B_A_FULL, B_A_EMPTY, B_P_FULL, B_P_EMPTY,
  B_U_FULL, B_U_EMPTY, B_SP_FULL, B_SP_EMPTY = B_SP_FULL + 2, B_O_FULL = B_SP_EMPTY + 2, B_O_EMPTY,
  B_DRAIN, NBAR = B_DRAIN + 3
};
constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
constexpr uint32_t SMEM_BYTES = OFF_MISC + 16 + 1024;
static_assert(SMEM_BYTES <= 232448, "shared memory budget");

// ---- tensor memory columns ------------------------------------------------------------------
constexpr uint32_t TM_A = 0, TM_P = 128, TM_OI = 192, TM_OE = 256, TM_U = 384, TMEM_COLS = 512;

constexpr unsigned long long DRAIN_NS = 1000000000ull;  // drain waits on the exit path

// ---- tcgen05 descriptors --------------------------------------------------------------------
// Instruction descriptor, kind::f16: D f32 (bits 4-5 = 1), A and B bf16 (bits 7-9, 10-12 = 1),
// A/B major-ness (bit 15/16: 0 K-major, 1 MN-major), N >> 3 (bits 17-22), M >> 4 (bits 24-28).
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, int a_mn, int b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
constexpr uint32_t LAYOUT_SW128 = 2, LAYOUT_SW64 = 4;

// Shared-memory matrix descriptor: start address, leading / stride byte offsets (>> 4), fixed
// version bits 46-47 = 1, swizzle layout in bits 61-63.
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo, uint32_t layout) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo & 0x3FFFFu) >> 4) << 16) |
         ((uint64_t)((sbo & 0x3FFFFu) >> 4) << 32) | (1ull << 46) | ((uint64_t)layout << 61);
}

// K-major operand made of 128-row, 128B-swizzled panels of 64 bf16 along K: step kk (16 along K).
__device__ __forceinline__ uint64_t desc_kmajor_sw128(uint32_t base, int kk) {
  return sdesc(base + (uint32_t)(kk >> 2) * 16384u + (uint32_t)(kk & 3) * 32u, 16, 1024, LAYOUT_SW128);
}
// Q: panel 0 (128B swizzle) for d_k 0..63, panel 1 (64B swizzle) for d_k 64..95.
__device__ __forceinline__ uint64_t desc_q(uint32_t stage, int kk) {
  if (kk < 4) return sdesc(stage + ST_Q0 + (uint32_t)kk * 32u, 16, 1024, LAYOUT_SW128);
  return sdesc(stage + ST_Q1 + (uint32_t)(kk - 4) * 32u, 16, 512, LAYOUT_SW64);
}
// MN-major operand: rows along K (8-row groups 1024 B apart), 64-element MN blocks `lbo` apart.
__device__ __forceinline__ uint64_t desc_mn_sw128(uint32_t base, int kk, uint32_t lbo) {
  return sdesc(base + (uint32_t)kk * 2048u, lbo, 1024, LAYOUT_SW128);
}

// ---- PTX wrappers ---------------------------------------------------------------------------
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint64_t* bar, int x,
                                            int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(
          dst),
      "l"((uint64_t)map), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void umma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(
          d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(acc));
}

// Same, with the A operand (M lanes x K/2 columns of bf16 pairs) read from tensor memory.
__device__ __forceinline__ void umma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}" ::"r"(
          d_tmem),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc));
}

__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

#define GLA_R8(b) "=r"(r[b]), "=r"(r[b + 1]), "=r"(r[b + 2]), "=r"(r[b + 3]), "=r"(r[b + 4]), "=r"(r[b + 5]), \
                  "=r"(r[b + 6]), "=r"(r[b + 7])
// 16 columns at each of three tensor-memory addresses of this thread's lane (one wait).
__device__ __forceinline__ void tmem_ld16x3(uint32_t ta, uint32_t tb, uint32_t tc, uint32_t (&r)[48]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%48];\n"
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%49];\n"
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47}, [%50];\n"
      "tcgen05.wait::ld.sync.aligned;"
      : GLA_R8(0), GLA_R8(8), GLA_R8(16), GLA_R8(24), GLA_R8(32), GLA_R8(40)
      : "r"(ta), "r"(tb), "r"(tc)
      : "memory");
}
// 16 columns at each of two tensor-memory addresses of this thread's lane (one wait).
__device__ __forceinline__ void tmem_ld16x2(uint32_t ta, uint32_t tb, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%32];\n"
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%33];\n"
      "tcgen05.wait::ld.sync.aligned;"
      : GLA_R8(0), GLA_R8(8), GLA_R8(16), GLA_R8(24)
      : "r"(ta), "r"(tb)
      : "memory");
}
// 32 columns of this thread's lane.
__device__ __forceinline__ void tmem_ld32(uint32_t ta, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
      "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
      "tcgen05.wait::ld.sync.aligned;"
      : GLA_R8(0), GLA_R8(8), GLA_R8(16), GLA_R8(24)
      : "r"(ta)
      : "memory");
}
#undef GLA_R8

// 16 consecutive 32-bit columns of this thread's tensor-memory lane.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Packed two-wide fp32 arithmetic (one instruction for both lanes of a float2).
__device__ __forceinline__ uint64_t f2u(float2 v) {
  return (uint64_t)__float_as_uint(v.x) | ((uint64_t)__float_as_uint(v.y) << 32);
}
__device__ __forceinline__ float2 u2f(uint64_t u) {
  return make_float2(__uint_as_float((uint32_t)u), __uint_as_float((uint32_t)(u >> 32)));
}
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(f2u(a)), "l"(f2u(b)));
  return u2f(r);
}
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(f2u(a)), "l"(f2u(b)));
  return u2f(r);
}
__device__ __forceinline__ float2 sub2(float2 a, float2 b) {
  uint64_t r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(f2u(a)), "l"(f2u(b)));
  return u2f(r);
}
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(f2u(a)), "l"(f2u(b)), "l"(f2u(c)));
  return u2f(r);
}
__device__ __forceinline__ float2 bf2_to_f2(uint32_t w) {
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}
__device__ __forceinline__ float2 ld_f2(const uint32_t* r, int x) {
  return make_float2(__uint_as_float(r[x]), __uint_as_float(r[x + 1]));
}

// x ~ hi + lo with hi = bf16(x), lo = bf16(x - hi); returns the two packed pairs.
__device__ __forceinline__ void split_bf16x2(float2 x, uint32_t& hi, uint32_t& lo) {
  hi = pack_bf16(x.x, x.y);
  const float2 r = sub2(x, bf2_to_f2(hi));
  lo = pack_bf16(r.x, r.y);
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

// Warp-uniform bounded wait: every lane waits (and so acquires), then the warp agrees.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, const ChunkArgs& a, volatile int* abort_flag) {
  const bool ok = mbar_wait(bar, parity, a.wait_ns, abort_flag, a.err);
  return __all_sync(0xffffffffu, ok);
}

struct TmaMaps {
  CUtensorMap q0, q1, k, v;
};

__global__ void __launch_bounds__(NTHREADS, 1) tc_fwd_kernel(const __grid_constant__ TmaMaps maps, const ChunkArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  const uint32_t sbase = (raw_u32 + 1023u) & ~1023u;
  uint8_t* sm = smem_raw + (sbase - raw_u32);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + OFF_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + OFF_MISC + 4);
  float* pw = reinterpret_cast<float*>(sm + OFF_PW);  // lambda^d, d = 0..128
  float* pws = pw + 129;                               // scale * lambda^d

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int n, h, tile;
  unit_of_block(a, NTILE, n, h, tile);
  long long tb, te;
  seq_range(a, n, tb, te);
  const int len = (int)(te - tb);
  const int nc = (len + CHUNK - 1) / CHUNK;
  const int col0 = tile * TN;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NBAR; ++i) {
      uint32_t cnt = 1;
      if (i == B_EMPTY || i == B_EMPTY + 1) cnt = 3;
      if (i == B_O_FULL) cnt = 2;
      if (i == B_VT_FULL || i == B_A_EMPTY || i == B_P_FULL || i == B_U_EMPTY || i == B_SP_FULL ||
          i == B_SP_FULL + 1 || i == B_O_EMPTY)
        cnt = 128;
      mbar_init(&bars[i], cnt);
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    fence_async_smem();
  }
  if (threadIdx.x < 129) {
    const float ll = a.log_lambda[h];
    const float p = threadIdx.x == 0 ? 1.f : expf((float)threadIdx.x * ll);
    pw[threadIdx.x] = p;
    pws[threadIdx.x] = a.scale * p;
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(TMEM_COLS));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  if (warp == 0 && lane == 0) {
    asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&maps.q0) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&maps.q1) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&maps.k) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&maps.v) : "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int issued[2] = {0, 0};
      for (int c = 0; c < nc; ++c) {
        const int s = c & 1;
        const uint32_t ph = (uint32_t)(c >> 1) & 1u;
        if (!mbar_wait(&bars[B_EMPTY + s], ph ^ 1u, a.wait_ns, abort_flag, a.err)) break;
        const uint32_t st = sbase + (uint32_t)s * SZ_STAGE;
        uint64_t* full = &bars[B_FULL + s];
        mbar_expect_tx(full, SZ_STAGE);
        const int tok = (int)(tb + (long long)c * CHUNK);
        tma_load_3d(st + ST_Q0, &maps.q0, full, 0, h, tok);
        tma_load_3d(st + ST_Q1, &maps.q1, full, 64, h, tok);
        tma_load_3d(st + ST_K, &maps.k, full, 0, h, tok);
        tma_load_3d(st + ST_K + 16384u, &maps.k, full, 64, h, tok);
        tma_load_3d(st + ST_V, &maps.v, full, col0, h, tok);
        ++issued[s];
      }
      // Never leave a copy in flight into shared memory that is about to be released.
      for (int s = 0; s < 2; ++s)
        if (issued[s]) mbar_wait(&bars[B_FULL + s], (uint32_t)(issued[s] - 1) & 1u, DRAIN_NS, nullptr, a.err);
    }
    __syncwarp();
  } else if (warp < 4) {
    // ------------------------------------------------------------------ MMA issuers
    if (lane == 0) {
      constexpr uint32_t ID_QK = idesc_bf16(128, 128, 0, 0);  // A = Q K^T
      constexpr uint32_t ID_PV = idesc_bf16(128, TN, 0, 1);   // O_intra = P V
      constexpr uint32_t ID_W = idesc_bf16(128, 2 * TN, 1, 1);  // U = K^T [Vt_hi | Vt_lo]
      constexpr uint32_t ID_QS = idesc_bf16(128, 2 * TN, 0, 1); // O_inter = Q [S_hi | S_lo]
      const uint32_t vt = sbase + OFF_VT;
      for (int c = 0; c < nc; ++c) {
        const int s = c & 1;
        const uint32_t ph = (uint32_t)(c >> 1) & 1u, pc = (uint32_t)c & 1u;
        const uint32_t st = sbase + (uint32_t)s * SZ_STAGE;
        if (!mbar_wait(&bars[B_FULL + s], ph, a.wait_ns, abort_flag, a.err)) break;
        if (warp == 1) {
          if (!mbar_wait(&bars[B_A_EMPTY], pc ^ 1u, a.wait_ns, abort_flag, a.err)) break;
          tc_fence_after();
          for (int kk = 0; kk < 6; ++kk)
            umma(tmem + TM_A, desc_q(st, kk), desc_kmajor_sw128(st + ST_K, kk), ID_QK, kk > 0);
          umma_commit(&bars[B_A_FULL]);
          umma_commit(&bars[B_EMPTY + s]);
        } else if (warp == 3) {
          if (!mbar_wait(&bars[B_P_FULL], pc, a.wait_ns, abort_flag, a.err)) break;
          if (!mbar_wait(&bars[B_O_EMPTY], pc ^ 1u, a.wait_ns, abort_flag, a.err)) break;
          tc_fence_after();
          for (int kk = 0; kk < 8; ++kk)
            umma_ts(tmem + TM_OI, tmem + TM_P + 8u * kk, desc_mn_sw128(st + ST_V, kk, 8192), ID_PV, kk > 0);
          umma_commit(&bars[B_P_EMPTY]);
          umma_commit(&bars[B_O_FULL]);
          umma_commit(&bars[B_EMPTY + s]);
        } else {
          if (!mbar_wait(&bars[B_VT_FULL], pc, a.wait_ns, abort_flag, a.err)) break;
          if (!mbar_wait(&bars[B_U_EMPTY], pc ^ 1u, a.wait_ns, abort_flag, a.err)) break;
          tc_fence_after();
          for (int kk = 0; kk < 8; ++kk)
            umma(tmem + TM_U, desc_mn_sw128(st + ST_K, kk, 16384), desc_mn_sw128(vt, kk, SZ_V), ID_W, kk > 0);
          umma_commit(&bars[B_U_FULL]);
          umma_commit(&bars[B_VT_EMPTY]);
          const int b = c & 1;
          const uint32_t fb = (uint32_t)(c >> 1) & 1u;
          if (!mbar_wait(&bars[B_SP_FULL + b], fb, a.wait_ns, abort_flag, a.err)) break;
          if (!mbar_wait(&bars[B_O_EMPTY], pc ^ 1u, a.wait_ns, abort_flag, a.err)) break;
          tc_fence_after();
          const uint32_t spb = sbase + OFF_SP + (uint32_t)b * SZ_SP;
          for (int kk = 0; kk < 6; ++kk)
            umma(tmem + TM_OE, desc_q(st, kk), desc_mn_sw128(spb, kk, SZ_SPH), ID_QS, kk > 0);
          umma_commit(&bars[B_SP_EMPTY + b]);
          umma_commit(&bars[B_O_FULL]);
          umma_commit(&bars[B_EMPTY + s]);
        }
      }
      // All MMAs (and their barrier arrivals) finish before tensor memory is released.
      uint64_t* drain = &bars[B_DRAIN + (warp - 1)];
      umma_commit(drain);
      mbar_wait(drain, 0, DRAIN_NS, nullptr, a.err);
    }
    __syncwarp();
  } else if (warp < 8) {
    // ------------------------------------------------------------------ Vt, then decay mask A -> P
    const int i = threadIdx.x - 128;  // query row = tensor-memory lane; also the Vt row
    const int q = warp & 3;           // this warp's lanes are rows 32q .. 32q + 31
    const uint32_t lane_addr = tmem + ((uint32_t)(q << 5) << 16);
    const float lam = pw[1];
    const float2 lam2 = make_float2(lam * lam, lam * lam);
    {  // P columns of groups past this warp's rows stay zero for the whole kernel: write them once
      uint32_t z[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) z[e] = 0u;
      for (int g = q + 1; g < 4; ++g) tmem_st16(lane_addr + TM_P + 16u * g, z);
      asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
    }
    for (int c = 0; c < nc; ++c) {
      const int s = c & 1;
      const uint32_t ph = (uint32_t)(c >> 1) & 1u, pc = (uint32_t)c & 1u;
      const int L = min(CHUNK, len - c * CHUNK);
      if (!warp_wait(&bars[B_FULL + s], ph, a, abort_flag)) break;
      if (!warp_wait(&bars[B_VT_EMPTY], pc ^ 1u, a, abort_flag)) break;
      {  // Vt row i = lambda^(L-1-i) v_i, split into hi and lo
        const uint8_t* vsrc = sm + s * SZ_STAGE + ST_V;
        uint8_t* vhi = sm + OFF_VT;
        uint8_t* vlo = sm + OFF_VT + SZ_V;
        const float fi = i < L ? pw[L - 1 - i] : 0.f;
        const float2 f = make_float2(fi, fi);
#pragma unroll
        for (int p = 0; p < 8; ++p) {
          const int off = i * 128 + ((p ^ (i & 7)) << 4);  // same permutation on both sides
          const uint4 x = *reinterpret_cast<const uint4*>(vsrc + off);
          const uint32_t w[4] = {x.x, x.y, x.z, x.w};
          uint32_t hi[4], lo[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) split_bf16x2(mul2(bf2_to_f2(w[e]), f), hi[e], lo[e]);
          *reinterpret_cast<uint4*>(vhi + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
          *reinterpret_cast<uint4*>(vlo + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
        }
        fence_async_smem();
        mbar_arrive(&bars[B_VT_FULL]);
      }
      if (!warp_wait(&bars[B_A_FULL], pc, a, abort_flag)) break;
      if (!warp_wait(&bars[B_P_EMPTY], pc ^ 1u, a, abort_flag)) break;
      tc_fence_after();
      // P row i = s lambda^(i-j) A_ij for j <= i and i < L, one 32-column group at a time, each
      // stored straight back to tensor memory.  Below the diagonal group the factors come from one
      // table read and a multiplicative chain toward larger i - j (the values only shrink, so an
      // underflow to zero loses nothing); the diagonal group reads the table per element.
      for (int g = 0; g <= q; ++g) {
        uint32_t r[32];
        tmem_ld32(lane_addr + TM_A + 32u * g, r);
        if (g == q) {
          tc_fence_before();
          mbar_arrive(&bars[B_A_EMPTY]);
        }
        uint32_t pkg[16];
        const int d0 = i - 32 * g;  // i - j at the group's first column
        if (g < q) {
          // f = (pws[d0 - 2e], pws[d0 - 2e - 1]), from e = 15 down to e = 0
          float2 f = i < L ? make_float2(pws[d0 - 30], pws[d0 - 31]) : make_float2(0.f, 0.f);
#pragma unroll
          for (int e = 15; e >= 0; --e) {
            if (e < 15) f = mul2(f, lam2);
            const float2 pv = mul2(f, ld_f2(r, 2 * e));
            pkg[e] = pack_bf16(pv.x, pv.y);
          }
        } else {
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const int d = d0 - 2 * e;
            const float f0 = (d >= 0 && i < L) ? pws[max(d, 0)] : 0.f;
            const float f1 = (d >= 1 && i < L) ? pws[max(d - 1, 0)] : 0.f;
            pkg[e] = pack_bf16(f0 * __uint_as_float(r[2 * e]), f1 * __uint_as_float(r[2 * e + 1]));
          }
        }
        tmem_st16(lane_addr + TM_P + 16u * g, pkg);
      }
      asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
      tc_fence_before();
      mbar_arrive(&bars[B_P_FULL]);
    }
  } else {
    // ------------------------------------------------------------------ epilogue
    const int r_ = ((warp & 3) << 5) + lane;  // d_k row of S and U; query row of O
    const uint32_t lane_addr = tmem + ((uint32_t)((warp & 3) << 5) << 16);
    const long long sbase_g = (((long long)n * a.H + h) * DK + r_) * DV + col0;
    float S[TN];
#pragma unroll
    for (int x = 0; x < TN; ++x) S[x] = 0.f;
    if (a.h0 && r_ < DK) {
      const float4* src = reinterpret_cast<const float4*>(a.h0 + sbase_g);
#pragma unroll
      for (int x = 0; x < TN / 4; ++x) {
        const float4 v4 = src[x];
        S[4 * x] = v4.x;
        S[4 * x + 1] = v4.y;
        S[4 * x + 2] = v4.z;
        S[4 * x + 3] = v4.w;
      }
    }
    auto write_sprev = [&](int buf) {
      if (r_ < DK) {
        const uint32_t row = sbase + OFF_SP + (uint32_t)buf * SZ_SP + (uint32_t)r_ * 128u;
#pragma unroll
        for (int cc = 0; cc < 8; ++cc) {
          uint32_t hi[4], lo[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) split_bf16x2(make_float2(S[8 * cc + 2 * e], S[8 * cc + 2 * e + 1]), hi[e], lo[e]);
          const uint32_t off = (uint32_t)((cc ^ (r_ & 7)) << 4);
          st_shared_v4(row + off, hi[0], hi[1], hi[2], hi[3]);
          st_shared_v4(row + SZ_SPH + off, lo[0], lo[1], lo[2], lo[3]);
        }
      }
      fence_async_smem();
      mbar_arrive(&bars[B_SP_FULL + buf]);
    };
    write_sprev(0);
    bool aborted = false;
    for (int c = 0; c < nc; ++c) {
      const uint32_t pc = (uint32_t)c & 1u;
      const int L = min(CHUNK, len - c * CHUNK);
      // S <- lambda^L S + U_hi + U_lo
      if (!warp_wait(&bars[B_U_FULL], pc, a, abort_flag)) { aborted = true; break; }
      tc_fence_after();
      const float lamL = pw[L];
#pragma unroll
      for (int qq = 0; qq < 4; ++qq) {
        uint32_t u[32];  // [0, 16): hi columns, [16, 32): lo columns of this quarter
        tmem_ld16x2(lane_addr + TM_U + 16u * qq, lane_addr + TM_U + TN + 16u * qq, u);
#pragma unroll
        for (int x = 0; x < 16; x += 2) {
          const float2 sv = fma2(make_float2(lamL, lamL), make_float2(S[16 * qq + x], S[16 * qq + x + 1]),
                                 add2(ld_f2(u, x), ld_f2(u, 16 + x)));
          S[16 * qq + x] = sv.x;
          S[16 * qq + x + 1] = sv.y;
        }
      }
      tc_fence_before();
      mbar_arrive(&bars[B_U_EMPTY]);
      if (c + 1 < nc) {
        const int b2 = (c + 1) & 1;
        const uint32_t f2 = (uint32_t)((c + 1) >> 1) & 1u;
        if (!warp_wait(&bars[B_SP_EMPTY + b2], f2 ^ 1u, a, abort_flag)) { aborted = true; break; }
        write_sprev(b2);
      }
      // o = O_intra + s lambda^(i+1) (O_inter_hi + O_inter_lo)
      if (!warp_wait(&bars[B_O_FULL], pc, a, abort_flag)) { aborted = true; break; }
      tc_fence_after();
      const float f = pws[r_ + 1];
      uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(a.o) +
                                            ((tb + (long long)c * CHUNK + r_) * a.H + h) * (long long)DV + col0);
#pragma unroll
      for (int qq = 0; qq < 4; ++qq) {
        uint32_t ov[48];  // 16 intra, 16 inter-hi, 16 inter-lo columns
        tmem_ld16x3(lane_addr + TM_OI + 16u * qq, lane_addr + TM_OE + 16u * qq,
                    lane_addr + TM_OE + TN + 16u * qq, ov);
        if (qq == 3) {
          tc_fence_before();
          mbar_arrive(&bars[B_O_EMPTY]);
        }
        uint32_t ob[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int x = 2 * e;
          const float2 ovx = fma2(make_float2(f, f), add2(ld_f2(ov, 16 + x), ld_f2(ov, 32 + x)), ld_f2(ov, x));
          ob[e] = pack_bf16(ovx.x, ovx.y);
        }
        if (r_ < L) {
          dst[2 * qq] = make_uint4(ob[0], ob[1], ob[2], ob[3]);
          dst[2 * qq + 1] = make_uint4(ob[4], ob[5], ob[6], ob[7]);
        }
      }
    }
    if (!aborted && a.hT && r_ < DK) {
      float4* dst = reinterpret_cast<float4*>(a.hT + sbase_g);
#pragma unroll
      for (int x = 0; x < TN / 4; ++x) dst[x] = make_float4(S[4 * x], S[4 * x + 1], S[4 * x + 2], S[4 * x + 3]);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS));
  }
}

// ---- host side ------------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// 3-D view [T_total, H, d] of a token-major bf16 tensor; box = (box_x columns, 1 head, 128 tokens).
bool make_map(CUtensorMap* m, const void* base, int d, int H, long long T, int box_x, CUtensorMapSwizzle sw) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)H, (cuuint64_t)T};
  const cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)H * d * 2};
  const cuuint32_t box[3] = {(cuuint32_t)box_x, 1, (cuuint32_t)CHUNK};
  const cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_tc_fwd(const ChunkArgs& a, cudaStream_t stream) {
  const long long blocks = (long long)a.n_seq * a.H * NTILE;
  if (blocks == 0) return cudaSuccess;
  const long long T_total = a.cu_seqlens ? (long long)a.T : (long long)a.n_seq * a.T;
  TmaMaps maps;
  memset(&maps, 0, sizeof(maps));
  if (T_total > 0) {
    if (!make_map(&maps.q0, a.q, DK, a.H, T_total, 64, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map(&maps.q1, a.q, DK, a.H, T_total, 32, CU_TENSOR_MAP_SWIZZLE_64B) ||
        !make_map(&maps.k, a.k, DK, a.H, T_total, 64, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map(&maps.v, a.v, DV, a.H, T_total, 64, CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  }
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(tc_fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  tc_fwd_kernel<<<(unsigned)blocks, NTHREADS, SMEM_BYTES, stream>>>(maps, a);
  return cudaGetLastError();
}

}  // namespace gla
