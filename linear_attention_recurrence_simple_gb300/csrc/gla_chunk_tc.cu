// Chunked GLA scans on the 5th-generation tensor cores (bf16 operands, fp32 accumulation and
// state): TMA -> shared memory -> tcgen05.mma -> tensor memory -> register epilogue.  One kernel
// template serves the forward and the three backward scans.
//
// "Beyond the KV cache" (Laplace 3B on Trainium2), section "Challenge 1: Using native PyTorch on
// Trainium for GLA": within each 128-token chunk the output is decay-masked linear attention plus
// the contribution of the state carried from earlier chunks; the state then advances with the
// decay compounded over the chunk, and only that advance is sequential.  Forward, per chunk of L
// tokens (local i, j; S = state before the chunk, s = scale):
//     A   = Q K^T                                   (MMA1)
//     P   = s lambda^(i-j) A  for j <= i, else 0      (decay-mask warps, bf16, kept in TMEM)
//     O   = P V  +  diag(s lambda^(i+1)) (Q S)       (MMA2, MMA3)
//     S'  = lambda^L S + K^T Vt,  Vt_j = lambda^(L-1-j) v_j   (MMA4)
// Section "Challenge 3" (the backward differentiates through the sequential state updates): the
// adjoint of the recurrence, with R = dL/dS flowing in from the next chunk (R = dhT for the last),
// gives per chunk
//     dq_i = s sum_{j<=i} lambda^(i-j) (dO_i.v_j) k_j + s lambda^(i+1) S dO_i        (forward scan)
//     dk_i = s sum_{j>=i} lambda^(j-i) (dO_j.v_i) q_j + lambda^(L-1-i) R v_i          (reverse scan)
//     dv_i = s sum_{j>=i} lambda^(j-i) (q_j.k_i) dO_j + lambda^(L-1-i) R^T k_i        (reverse scan)
//     R'   = lambda^L R + Q^T dOt,  dOt_j = s lambda^(j+1) dO_j,   dh0 = R after the first chunk.
// Each is the forward's pattern with other operands (X Y^T masked, times Z; X times the carried
// state; K4^T times the weighted Z4):
//     mode   X      Y      Z      K4  Z4   mask   inter factor      state weight     output
//     FWD    q      k      v_t    k   v_t  j<=i   s lambda^(i+1)    lambda^(L-1-j)   o_t (bf16), hT
//     DV     k      q      dO_t   q   dO_t j>=i   lambda^(L-1-i)    s lambda^(j+1)   dv_t (bf16), dh0
//     DQ     dO_t   v_t    k      k   v_t  j<=i   s lambda^(i+1)    lambda^(L-1-j)   dq partial (fp32 add)
//     DK     v_t    dO_t   q      q   dO_t j>=i   lambda^(L-1-i)    s lambda^(j+1)   dk partial (fp32 add)
// (_t = this CTA's 64-column tile of d_v).  dq and dk contract over all of d_v, so the three tile
// CTAs of a head add fp32 partials into an accumulator (vector red.add), converted to bf16 after.
// The decay is never split into lambda^i * lambda^-j, so lambda = 0.5 cannot overflow.  Operands
// that carry the state are split into two bf16 terms, x = hi + lo with hi = bf16(x),
// lo = bf16(x - hi): the state copy in MMA3 and the weighted Z4 in MMA4, about 16 significant
// bits on the state path; only P is a single bf16 rounding.
//
// Work split: a work unit is a (sequence, head, 64-column tile of d_v); 1 CTA per SM (all of
// tensor memory, ~224 KB of shared memory).  Equal-length forward batches run one persistent CTA
// per SM over a work list built in the prologue; with a final-state output the list is balanced
// (the chunks of all (sequence, head) pairs cut into equal ranges, one per group of three CTAs,
// a pair straddling two ranges handed over through its final-state tile; see the kernel).
// Varlen batches and the backward scans run one CTA per unit.  One thread issues at most one
// tcgen05.mma (M = 128, K = 16) per ~70 cycles whatever N <= 128 is (measured), so the kernel
// keeps the instruction count low (hi/lo halves ride in one N = 128 MMA where N allows) and issues
// from three threads in parallel, one per accumulator chain.  Warp roles:
//   warp 0      TMA producer: X, Y, Z chunk tiles into a 2-stage ring.
//   warp 1      allocates tensor memory; one lane issues MMA1 (X Y^T), then MMA3 (X times the
//               state copy), whose inputs are ready long before the weighted Z4 that MMA4 waits for.
//   warp 2      one lane issues MMA4 (K4^T [Z4t_hi | Z4t_lo]).
//   warp 3      one lane issues MMA2 (P Z, P read from tensor memory).
//   warps 4-7   decay mask A (TMEM) -> P (bf16 pairs, back into TMEM).  A is released as soon as
//               it is in registers, so the next chunk's MMA1 overlaps this one's P.
//   warps 8-11  epilogue: U (TMEM) -> state = lambda^L state + U in fp32 registers -> bf16 hi/lo
//               copy for the next chunk's MMA3; O (TMEM) -> output row.  In the backward scans
//               (640 threads) warps 8-11 keep the state part and warps 16-19 take the output part.
//   warps 12-15 the weighted Z4 for MMA4 (hi and lo, zero past the sequence end).
// Registers: setmaxnreg in each role redistributes exactly the registers the CTA launches with
// (forward: 128 each, then 72 control, 184 mask, 184 epilogue, 72 Z4; backward: 96 each, then
// 64, 120, 136, 64, 96 output).
// Tensor memory (512 columns): A [0,128), P [128,192), then O_intra, O_inter and U [384,512).
// Every mbarrier wait is bounded (see gla_common.cuh); on a timeout the CTA records
// GLA_ERR_TIMEOUT, drains its copies and MMAs, frees tensor memory and returns.
#include <cuda.h>
#include <string.h>

#include <algorithm>
#include <atomic>
#include <mutex>
#include <type_traits>

#include "gla_common.cuh"

namespace gla {

// MODE_FWDA: the forward with the self-augmentation step (see the decay mask).  MODE_FWDS: the
// forward's final states only (no outputs): the producer loads k and the v tile, MMA4 and the
// epilogue's state update run, everything that builds outputs is left out.
enum ScanMode { MODE_FWD = 0, MODE_DV = 1, MODE_DQ = 2, MODE_DK = 3, MODE_FWDA = 4, MODE_FWDS = 5 };

namespace {

constexpr int TN = 64;             // d_v columns per CTA
constexpr int NTILE = DV / TN;     // 3

template <int MODE>
struct Cfg {
  static constexpr bool REVERSE = MODE == MODE_DV || MODE == MODE_DK;  // reverse scan, j >= i mask
  static constexpr bool NARROW = MODE == MODE_DQ || MODE == MODE_DK;   // X, Y are 64-wide d_v tiles
  static constexpr bool FWD = MODE == MODE_FWD || MODE == MODE_FWDA || MODE == MODE_FWDS;
  static constexpr bool AUG = MODE == MODE_FWDA;
  static constexpr bool STATES = MODE == MODE_FWDS;
  // Warp roles: 16 warps with one epilogue warpgroup (forward), or 20 with the epilogue's state
  // and output parts in two warpgroups (backward scans).  Per-thread registers of each warpgroup
  // after setmaxnreg add up to the launch count times the number of warpgroups (the host checks
  // the compiled count before the first launch: any other split could wait forever).
  static constexpr bool SPLIT = !FWD;
  static constexpr int THREADS = SPLIT ? 640 : 512;
  static constexpr int REG_LAUNCH = SPLIT ? 96 : 128;
  static constexpr int REG_CTRL = SPLIT ? 64 : 72, REG_MASK = SPLIT ? 120 : 184, REG_STATE = SPLIT ? 136 : 184;
  static constexpr int REG_Z4 = SPLIT ? 64 : 72, REG_OUT = SPLIT ? 96 : 0;
  static_assert(REG_CTRL + REG_MASK + REG_STATE + REG_Z4 + REG_OUT == THREADS / 128 * REG_LAUNCH, "register split");
  static_assert(THREADS * REG_LAUNCH <= 65536, "launch registers");
  // shared memory of one stage (byte offsets; each tile 1024-aligned)
  //   wide:   X panel 0 (16 KB) | Y 2 panels (32 KB) | Z tile (16 KB) | X panel 1 (8 KB, 64B swizzle)
  //   narrow: X tile (16 KB) | Y tile (16 KB) | Z 2 panels (32 KB)
  //   states only: Y 2 panels (32 KB) | Z tile (16 KB); no X, so three stages fit in the space of two
  static constexpr int NSTAGE = STATES ? 3 : 2;  // depth of the TMA ring
  static constexpr uint32_t ST_X = 0;
  static constexpr uint32_t ST_X1 = NARROW ? 0 : 65536;
  static constexpr uint32_t ST_Y = STATES ? 0 : 16384;
  static constexpr uint32_t ST_Z = NARROW || STATES ? 32768 : 49152;
  static constexpr uint32_t ST_K4 = NARROW ? ST_Z : ST_Y;
  static constexpr uint32_t ST_Z4 = NARROW ? ST_Y : ST_Z;
  static constexpr uint32_t SZ_STAGE = NARROW ? 65536 : (STATES ? 49152 : 73728);
  static constexpr int K1 = NARROW ? 4 : 6;       // K steps of MMA1 and MMA3 (d_v tile / d_k)
  static constexpr int OW = NARROW ? DK : TN;     // output columns per CTA
  // tensor memory columns
  static constexpr uint32_t TM_A = 0, TM_P = 128, TM_OI = 192, TM_OE = NARROW ? 288 : 256, TM_U = 384;
};

constexpr uint32_t SZ_TILE64 = 128 * 128;       // one 128-row, 128-byte-row tile
constexpr uint32_t SZ_SPH = 96 * 128;           // bf16 state tile: 96 rows (d_k) x 64 columns
constexpr uint32_t SZ_SP = 2 * SZ_SPH;          // hi then lo
enum {
  B_FULL = 0, B_EMPTY = 3, B_VT_FULL = 6, B_VT_EMPTY = 8, B_A_FULL = 10, B_A_EMPTY, B_P_FULL, B_P_EMPTY,
  B_U_FULL, B_U_EMPTY, B_SP_FULL, B_SP_EMPTY, B_O_FULL, B_O_EMPTY,
  B_ZR, B_P_HALF = B_ZR + 2, B_TBL_FULL, B_TBL_EMPTY = B_TBL_FULL + 2, B_ST_FULL = B_TBL_EMPTY + 2,
  B_HANDOVER, B_DRAIN, NBAR = B_DRAIN + 3
};
constexpr int PW_FLOATS = 2 * 129;  // lambda^d and scale * lambda^d, d = 0..128
constexpr int MAX_ITEMS = 32;       // work units per CTA (the host sizes the grid to keep within it)
constexpr uint32_t RED_ROW = 208;                 // 192 bytes of fp32 + 16 (bank spread)
constexpr uint32_t RED_WARP_BYTES = 32 * RED_ROW;
template <int MODE>
struct Smem {
  // weighted Z4 copies (hi and lo): two buffers in the states-only scan, whose next chunk's
  // weighting then overlaps this chunk's MMA4 (it has no state copy and no output staging)
  static constexpr uint32_t NVT = Cfg<MODE>::STATES ? 2 : 1;
  static constexpr uint32_t OFF_VT = Cfg<MODE>::NSTAGE * Cfg<MODE>::SZ_STAGE;
  static constexpr uint32_t OFF_SP = OFF_VT + NVT * 2 * SZ_TILE64;
  // output staging: wide, the bf16 output tile for the TMA store; narrow, one region per epilogue
  // warp (32 rows x 48 fp32, rows padded to 208 bytes) that turns row-wise sums into adds of
  // contiguous row segments
  static constexpr uint32_t OFF_OST = OFF_SP + (Cfg<MODE>::STATES ? 0 : SZ_SP);
  static constexpr uint32_t OFF_PW =
      OFF_OST + (Cfg<MODE>::STATES ? 0 : (Cfg<MODE>::NARROW ? 4u * RED_WARP_BYTES : SZ_TILE64));
  // two decay tables (per unit parity), then (self-augmentation) two copies of the head's aug_balance
  static constexpr uint32_t OFF_AUG = Cfg<MODE>::AUG ? (OFF_PW + 2 * PW_FLOATS * 4 + 8 + 15) / 16 * 16
                                                      : OFF_PW + 2 * PW_FLOATS * 4 + 8;
  static constexpr uint32_t OFF_BAR = OFF_AUG + (Cfg<MODE>::AUG ? 2 * DK * 4 : 0);
  static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr uint32_t OFF_ITEMS = OFF_MISC + 16;  // the CTA's work list (see the kernel)
  static constexpr uint32_t BYTES = OFF_ITEMS + MAX_ITEMS * 32 + 1024;
  static_assert(BYTES <= 232448, "shared memory budget");
};
constexpr uint32_t TMEM_COLS = 512;

constexpr unsigned long long DRAIN_NS = 1000000000ull;  // drain waits on the exit path

// ---- tcgen05 descriptors --------------------------------------------------------------------
// Instruction descriptor, kind::f16: D f32 (bits 4-5 = 1), A and B bf16 (bits 7-9, 10-12 = 1),
// A/B major-ness (bit 15/16: 0 K-major, 1 MN-major), N >> 3 (bits 17-22), M >> 4 (bits 24-28).
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, int a_mn, int b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
constexpr uint32_t LAYOUT_SW128 = 2, LAYOUT_SW64 = 4;

// Shared-memory matrix descriptor, kept as its two 32-bit words: lo = start address >> 4
// (bits 0-13) | leading byte offset >> 4 (bits 16-29); hi = stride byte offset >> 4 | the fixed
// version bit (bit 46 of the descriptor) | swizzle layout (bits 61-63).
// Stepping along K or to another panel only adds (bytes >> 4) to lo, so each MMA of a K loop costs
// one integer add in the issuing thread (the issue rate of a thread depends on that work).
struct SDesc {
  uint32_t lo, hi;
};
__device__ __forceinline__ SDesc sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo, uint32_t layout) {
  return {((saddr & 0x3FFFFu) >> 4) | (((lbo & 0x3FFFFu) >> 4) << 16),
          ((sbo & 0x3FFFFu) >> 4) | (1u << 14) | (layout << 29)};
}
__device__ __forceinline__ SDesc operator+(SDesc d, uint32_t bytes) { return {d.lo + (bytes >> 4), d.hi}; }

// ---- PTX wrappers ---------------------------------------------------------------------------
// Brings a box of a tensor into L2 (no shared memory written, nothing to wait for).
__device__ __forceinline__ void tma_prefetch_3d(const CUtensorMap* map, int x, int y, int z) {
  asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"((uint64_t)map), "r"(x), "r"(y),
               "r"(z)
               : "memory");
}
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint64_t* bar, int x,
                                            int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(
          dst),
      "l"((uint64_t)map), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint64_t* bar, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          dst),
      "l"((uint64_t)map), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// Shared -> global tile store (bulk-group completion), and the wait for this thread's bulk groups
// to have read shared memory (the global writes are complete by the end of the grid).
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, uint32_t src, int x, int y, int z) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"((uint64_t)map),
               "r"(x), "r"(y), "r"(z), "r"(src)
               : "memory");
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_gpu(unsigned* p, unsigned v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ void umma(uint32_t d_tmem, SDesc a, SDesc b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n .reg .b64 da, db;\n mov.b64 da, {%1, %2};\n mov.b64 db, {%3, %4};\n"
      " setp.ne.b32 p, %6, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %5, p;\n}" ::"r"(d_tmem),
      "r"(a.lo), "r"(a.hi), "r"(b.lo), "r"(b.hi), "r"(idesc), "r"(acc));
}
// Same, with the A operand (M lanes x K/2 columns of bf16 pairs) read from tensor memory.
__device__ __forceinline__ void umma_ts(uint32_t d_tmem, uint32_t a_tmem, SDesc b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n .reg .b64 db;\n mov.b64 db, {%2, %3};\n setp.ne.b32 p, %5, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], db, %4, p;\n}" ::"r"(d_tmem),
      "r"(a_tmem), "r"(b.lo), "r"(b.hi), "r"(idesc), "r"(acc));
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

__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

// Warp-uniform bounded wait: every lane waits (and so acquires), then the warp agrees.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, const ChunkArgs& a, volatile int* abort_flag) {
  const bool ok = mbar_wait(bar, parity, a.wait_ns, abort_flag);
  return __all_sync(0xffffffffu, ok);
}

// 32 bytes to a 32-byte aligned global address.
__device__ __forceinline__ void st_global_v8(void* p, const uint32_t (&v)[8]) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(v[0]), "r"(v[1]), "r"(v[2]),
               "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
               : "memory");
}

__device__ __forceinline__ void red_add_v4(float* p, float a, float b, float c, float d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(a), "f"(b), "f"(c), "f"(d) : "memory");
}

struct TmaMaps {
  CUtensorMap x, x1, y, z, o;  // o: the bf16 output (wide modes), 32-row boxes (one per epilogue warp)
  CUtensorMap s;                // fp32 final state (forward hand-over loads), 32-column x 96-row boxes
};

// What a scan kernel needs besides its tensor maps: sequence layout and decay (in `a`), the
// initial state, the final-state output, and the output (bf16 rows, or fp32 partial sums).
struct ScanParams {
  ChunkArgs a;
  const float* s0;  // [n_seq, H, 96, 192] initial state (h0 or dhT), or null = zeros
  float* s_out;     // final state (hT or dh0), or null
  void* out;        // FWD / DV: bf16 [T, H, 192];  DQ / DK: fp32 [T, H, 96] accumulator
  int balanced = 0;  // chunk ranges split evenly over the CTAs (forward, equal lengths, s_out given)
  int flag_set = 0;  // which set of hand-over flags a balanced launch uses
  unsigned epoch = 0;  // the value a raised flag holds in this launch (never 0)
};

// Hand-over flags of balanced launches: flag b of a set is raised (to the launch's epoch) by CTA b
// once the piece of a unit it ran first (the unit's first chunks) has left its state in the unit's
// final-state tile, and lowered again (to 0) by CTA b + NTILE, which runs the unit's remaining
// chunks from that state.  Launches use the sets in turn, so up to FLAG_SETS balanced launches may
// run at the same time; a flag left raised by a launch that gave up holds another epoch (and the
// host lowers them all when it reads the error).
constexpr int FLAG_SETS = 16, FLAG_MAX_CTAS = 1024;
__device__ unsigned g_handover[FLAG_SETS * FLAG_MAX_CTAS];

// Per-warpgroup register budgets (every warp of the warpgroup executes the same instruction).
template <int N>
__device__ __forceinline__ void setmaxnreg_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}
template <int N>
__device__ __forceinline__ void setmaxnreg_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}

template <int MODE>
__global__ void __launch_bounds__(Cfg<MODE>::THREADS, 1) tc_scan_kernel(const __grid_constant__ TmaMaps maps, const ScanParams prm) {
  using C = Cfg<MODE>;
  using SMM = Smem<MODE>;
  const ChunkArgs& a = prm.a;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  const uint32_t sbase = (raw_u32 + 1023u) & ~1023u;
  uint8_t* sm = smem_raw + (sbase - raw_u32);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + SMM::OFF_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + SMM::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + SMM::OFF_MISC + 4);
  // Decay tables of a work unit (lambda^d and scale * lambda^d, d = 0..128), two buffers used by
  // alternate units of this CTA.
  float* const pw_base = reinterpret_cast<float*>(sm + SMM::OFF_PW);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // Extents of the caller's buffers, for the debug-bounds build's index checks: (token, head) rows
  // of q, k, v, o and the gradients; rows of the [n_seq, H, 96, 192] states.
  [[maybe_unused]] const long long tokens = a.cu_seqlens ? (long long)a.T : (long long)a.n_seq * a.T;
  [[maybe_unused]] const long long rows_total = tokens * a.H, state_rows = (long long)a.n_seq * a.H * DK;
  // Persistent CTAs: this CTA runs work units blockIdx.x, blockIdx.x + gridDim.x, ... (a unit is a
  // (sequence, head, 64-column tile of d_v)); the chunk pipeline runs on across unit boundaries,
  // so a unit's first loads overlap the previous unit's last chunks.  Barrier phases count the
  // CTA's chunks over all its units (gk).
  // The CTA's work list is built once, in shared memory, by the lanes of warp 0 in the prologue;
  // every role then reads its next item from it.  An item is a unit (sequence, head, 64-column
  // tile of d_v) or a piece of one (processing steps [it0, it1) of its chunks).
  //   plain:    units blockIdx.x, blockIdx.x + gridDim.x, ..., each whole;
  //   balanced: CTAs work in groups of NTILE, one per d_v tile, so that the tiles of a
  //             (sequence, head) run at the same time and share its Q and K through L2.  The
  //             pairs' chunks, concatenated in order, are cut into one equal contiguous range
  //             per group, and each CTA of group t runs range t for its tile.  A pair that
  //             straddles ranges t and t + 1 is run in two pieces: its first chunks by group t
  //             as its first item (a "tail" piece: the final state goes to the unit's final-state
  //             tile and raises the CTA's hand-over flag), the rest by group t + 1 as its last
  //             item (a "head" piece: it starts from that state once the flag of the same tile's
  //             CTA in group t is up).  All CTAs are resident (cooperative launch), so the wait
  //             ends.
  const int n_units = a.n_seq * a.H * NTILE;  // below 2^31 (checked on the host)
  struct Unit {
    int n, h, tile, len, nc;
    long long tb;
    int it0, it1;     // processing steps [it0, it1) of the unit's chunks
    bool head, tail;  // balanced pieces (see below)
  };
  struct ItemInfo {  // 32 bytes
    long long tb;
    int n, h, tile, len, it0, it1;  // tile | 256 (head piece) | 512 (tail piece)
  };
  ItemInfo* const items = reinterpret_cast<ItemInfo*>(sm + SMM::OFF_ITEMS);
  int* const n_items_smem = reinterpret_cast<int*>(sm + SMM::OFF_MISC + 8);
  auto unit_at = [&](int k) {
    const ItemInfo& t = items[k];
    Unit w;
    w.tb = t.tb;
    w.n = t.n;
    w.h = t.h;
    w.tile = t.tile & 255;
    w.head = (t.tile & 256) != 0;
    w.tail = (t.tile & 512) != 0;
    w.len = t.len;
    w.nc = (w.len + CHUNK - 1) / CHUNK;
    w.it0 = t.it0;
    w.it1 = t.it1;
    return w;
  };

  if (threadIdx.x == 0) {
    for (int i = 0; i < NBAR; ++i) {
      uint32_t cnt = 1;
      if (i >= B_EMPTY && i < B_EMPTY + C::NSTAGE) cnt = C::STATES ? 1 : 3;  // the MMA issuers that read a stage
      if (i == B_TBL_FULL || i == B_TBL_FULL + 1) cnt = 128;   // the Z4 warps write a unit's table
      if (i == B_TBL_EMPTY || i == B_TBL_EMPTY + 1) cnt = C::SPLIT ? 512 : (C::STATES ? 256 : 384);  // its readers
      if (i == B_O_FULL) cnt = 2;
      if (i == B_ST_FULL) cnt = 128;  // the epilogue threads' final-state rows are visible (tail piece)
      if (i == B_VT_FULL || i == B_VT_FULL + 1 || i == B_A_EMPTY || i == B_P_FULL || i == B_P_HALF || i == B_U_EMPTY || i == B_SP_FULL ||
          i == B_O_EMPTY || i == B_ZR || i == B_ZR + 1)
        cnt = 128;
      mbar_init(&bars[i], cnt);
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    fence_async_smem();
  }
  if (warp == 0) {
    int n_it, pu0 = 0, pk0 = 0, pu1 = 0, pk1 = 0, ncu = 1;
    const int my_tile = (int)blockIdx.x % NTILE;
    if (prm.balanced) {  // equal lengths; each range spans at least one pair's chunks (host-checked)
      // 32-bit arithmetic: the host keeps the chunk total below 2^31
      const unsigned groups = gridDim.x / NTILE, grp = blockIdx.x / NTILE;
      ncu = (a.T + CHUNK - 1) / CHUNK;
      const unsigned ctot = (unsigned)(n_units / NTILE) * (unsigned)ncu, cq = ctot / groups, cr = ctot % groups;
      const unsigned g0 = cq * grp + cr * grp / groups, g1 = cq * (grp + 1) + cr * (grp + 1) / groups;
      pu0 = (int)(g0 / (unsigned)ncu);
      pk0 = (int)(g0 - (unsigned)pu0 * (unsigned)ncu);
      pu1 = (int)(g1 / (unsigned)ncu);
      pk1 = (int)(g1 - (unsigned)pu1 * (unsigned)ncu);
      n_it = grp < groups ? (pk1 > 0) + (pu1 - pu0) : 0;  // tail piece, whole pairs, head piece
    } else {
      n_it = (int)blockIdx.x < n_units ? (n_units - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
    }
    n_it = min(n_it, MAX_ITEMS);
    for (int k = lane; k < n_it; k += 32) {
      int u, it0 = 0, it1 = -1, flags = 0;
      if (!prm.balanced) {
        u = (int)blockIdx.x + k * (int)gridDim.x;
      } else if (pk1 > 0 && k == 0) {
        u = pu1 * NTILE + my_tile;
        it1 = pk1;
        flags = 512;
      } else if (k - (pk1 > 0) < pu1 - pu0 - (pk0 > 0)) {
        u = (pu0 + (pk0 > 0) + k - (pk1 > 0)) * NTILE + my_tile;
      } else {
        u = pu0 * NTILE + my_tile;
        it0 = pk0;
        flags = 256;
      }
      ItemInfo t;
      unit_of(a, NTILE, u, t.n, t.h, t.tile);
      t.tile |= flags;
      long long te;
      seq_range(a, t.n, t.tb, te);
      t.len = (int)(te - t.tb);
      t.it0 = it0;
      t.it1 = it1 >= 0 ? it1 : (t.len + CHUNK - 1) / CHUNK;
      items[k] = t;
    }
    if (lane == 0) *n_items_smem = n_it;
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(TMEM_COLS));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  if (warp == 0 && lane == 0) {
    asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&maps.x) : "memory");
    if (!C::NARROW) asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&maps.x1) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&maps.y) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&maps.z) : "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int n_items = *n_items_smem;

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    setmaxnreg_dec<C::REG_CTRL>();
    if (lane == 0) {
      int issued[C::NSTAGE] = {};
      int gk = 0;
      bool stop = false;
      for (int u = 0; u < n_items && !stop; ++u) {
       const Unit w = unit_at(u);
       const int h = w.h, col0 = w.tile * TN;
       for (int it = w.it0; it < w.it1; ++it, ++gk) {
        const int c = C::REVERSE ? w.nc - 1 - it : it;
        const int s = gk % C::NSTAGE;
        const uint32_t ph = (uint32_t)(gk / C::NSTAGE) & 1u;
        if (!mbar_wait(&bars[B_EMPTY + s], ph ^ 1u, a.wait_ns, abort_flag)) { stop = true; break; }
        const uint32_t st = sbase + (uint32_t)s * C::SZ_STAGE;
        uint64_t* full = &bars[B_FULL + s];
        mbar_expect_tx(full, C::SZ_STAGE);
        const int tok = (int)(w.tb + (long long)c * CHUNK);
        (void)GLA_IN_BOUNDS(tok >= 0 && tok < tokens && h >= 0 && h < a.H, a.err);
        if (C::NARROW) {
          tma_load_3d(st + C::ST_X, &maps.x, full, col0, h, tok);
          tma_load_3d(st + C::ST_Y, &maps.y, full, col0, h, tok);
          tma_load_3d(st + C::ST_Z, &maps.z, full, 0, h, tok);
          tma_load_3d(st + C::ST_Z + 16384u, &maps.z, full, 64, h, tok);
        } else {
          if (!C::STATES) {
            tma_load_3d(st + C::ST_X, &maps.x, full, 0, h, tok);
            tma_load_3d(st + C::ST_X1, &maps.x1, full, 64, h, tok);
          }
          tma_load_3d(st + C::ST_Y, &maps.y, full, 0, h, tok);
          tma_load_3d(st + C::ST_Y + 16384u, &maps.y, full, 64, h, tok);
          tma_load_3d(st + C::ST_Z, &maps.z, full, col0, h, tok);
        }
        // The same boxes of the unit's chunk two steps on go into L2 now, so that their load,
        // issued once a stage frees up, does not wait for DRAM.
        if (it + 2 < w.it1) {
          const int tp = (int)(w.tb + (long long)(C::REVERSE ? w.nc - 3 - it : it + 2) * CHUNK);
          if (C::NARROW) {
            tma_prefetch_3d(&maps.x, col0, h, tp);
            tma_prefetch_3d(&maps.y, col0, h, tp);
            tma_prefetch_3d(&maps.z, 0, h, tp);
            tma_prefetch_3d(&maps.z, 64, h, tp);
          } else {
            if (!C::STATES) {
              tma_prefetch_3d(&maps.x, 0, h, tp);
              tma_prefetch_3d(&maps.x1, 64, h, tp);
            }
            tma_prefetch_3d(&maps.y, 0, h, tp);
            tma_prefetch_3d(&maps.y, 64, h, tp);
            tma_prefetch_3d(&maps.z, col0, h, tp);
          }
        }
        ++issued[s];
       }
      }
      // Never leave a copy in flight into shared memory that is about to be released.
      for (int s = 0; s < C::NSTAGE; ++s)
        if (issued[s]) mbar_wait_drain(&bars[B_FULL + s], (uint32_t)(issued[s] - 1) & 1u, DRAIN_NS, a.err);
    }
    __syncwarp();
  } else if (warp < 4) {
    // ------------------------------------------------------------------ MMA issuers
    setmaxnreg_dec<C::REG_CTRL>();
    if (lane == 0) {
      constexpr uint32_t ID_A = idesc_bf16(128, 128, 0, 0);           // A = X Y^T
      constexpr uint32_t ID_PZ = idesc_bf16(128, C::OW, 0, 1);        // O_intra = P Z
      constexpr uint32_t ID_U = idesc_bf16(128, 2 * TN, 1, 1);        // U = K4^T [Z4t_hi | Z4t_lo]
      constexpr uint32_t ID_E = C::NARROW ? idesc_bf16(128, DK, 0, 0)  // O_inter = X S^T (hi, lo)
                                          : idesc_bf16(128, 2 * TN, 0, 1);  // O_inter = X [S_hi | S_lo]
      // Operand descriptors (K steps and panels are constant offsets from these):
      //   X: K-major (wide: 64-column 128B-swizzled panel + 32-column 64B panel; narrow: one panel)
      //   Y: K-major (wide: two 128B panels);  Z, K4, weighted Z4: MN-major
      //   state copy: MN-major [hi | lo] (wide) or K-major (narrow)
      const SDesc dvt = sdesc(sbase + SMM::OFF_VT, SZ_TILE64, 1024, LAYOUT_SW128);
      int gk = 0, nu = 0;  // chunks; units with chunks (states only: one U per unit)
      bool stop = C::STATES && warp != 2;  // states only: MMA4 alone
      for (int u = 0; u < n_items && !stop; ++u) {
       const Unit wi = unit_at(u);
       for (int it = wi.it0; it < wi.it1; ++it, ++gk) {
        const int s = gk % C::NSTAGE;
        const uint32_t ph = (uint32_t)(gk / C::NSTAGE) & 1u, pc = (uint32_t)gk & 1u;
        const uint32_t st = sbase + (uint32_t)s * C::SZ_STAGE;
        const SDesc dx = sdesc(st + C::ST_X, 16, 1024, LAYOUT_SW128);
        const SDesc dx1 = sdesc(st + C::ST_X1, 16, 512, LAYOUT_SW64);
        // K step kk of X: 16 columns = 32 bytes along the panel row
        auto x_step = [&](int kk) {
          return C::NARROW ? dx + (uint32_t)kk * 32u : (kk < 4 ? dx + (uint32_t)kk * 32u : dx1 + (uint32_t)(kk - 4) * 32u);
        };
        if (!mbar_wait(&bars[B_FULL + s], ph, a.wait_ns, abort_flag)) { stop = true; break; }
        if (warp == 1) {
          if (!mbar_wait(&bars[B_A_EMPTY], pc ^ 1u, a.wait_ns, abort_flag)) { stop = true; break; }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < C::K1; ++kk) {
            const SDesc dy = sdesc(st + C::ST_Y, 16, 1024, LAYOUT_SW128);
            const SDesc db = C::NARROW ? dy + (uint32_t)kk * 32u
                                       : dy + (uint32_t)(kk >> 2) * 16384u + (uint32_t)(kk & 3) * 32u;
            umma(tmem + C::TM_A, x_step(kk), db, ID_A, kk > 0);
          }
          umma_commit(&bars[B_A_FULL]);
          // the state before this chunk (one buffer: the epilogue overwrites it after this MMA3)
          const uint32_t spb = sbase + SMM::OFF_SP;
          const SDesc dsp = C::NARROW ? sdesc(spb, 16, 1024, LAYOUT_SW128) : sdesc(spb, SZ_SPH, 1024, LAYOUT_SW128);
          if (!mbar_wait(&bars[B_SP_FULL], pc, a.wait_ns, abort_flag)) { stop = true; break; }
          if (!mbar_wait(&bars[B_O_EMPTY], pc ^ 1u, a.wait_ns, abort_flag)) { stop = true; break; }
          tc_fence_after();
          if (C::NARROW) {
            // state tile as a K-major B operand: N = 96 rows (d_k), K = this tile's 64 columns
#pragma unroll
            for (int part = 0; part < 2; ++part)
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                umma(tmem + C::TM_OE, x_step(kk), dsp + (uint32_t)part * SZ_SPH + (uint32_t)kk * 32u, ID_E,
                     part + kk > 0);
          } else {
            // state tile as an MN-major B operand: K = 96 rows (d_k), N = [hi | lo] x 64 columns
#pragma unroll
            for (int kk = 0; kk < 6; ++kk)
              umma(tmem + C::TM_OE, x_step(kk), dsp + (uint32_t)kk * 2048u, ID_E, kk > 0);
          }
          umma_commit(&bars[B_SP_EMPTY]);
          umma_commit(&bars[B_O_FULL]);
          umma_commit(&bars[B_EMPTY + s]);
        } else if (warp == 3) {
          if (C::REVERSE && !mbar_wait(&bars[B_ZR + s], ph, a.wait_ns, abort_flag)) { stop = true; break; }
          if (!mbar_wait(&bars[C::REVERSE ? B_P_HALF : B_P_FULL], pc, a.wait_ns, abort_flag)) { stop = true; break; }
          if (!mbar_wait(&bars[B_O_EMPTY], pc ^ 1u, a.wait_ns, abort_flag)) { stop = true; break; }
          tc_fence_after();
          const SDesc dz = sdesc(st + C::ST_Z, C::NARROW ? 16384u : 8192u, 1024, LAYOUT_SW128);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            umma_ts(tmem + C::TM_OI, tmem + C::TM_P + 8u * kk, dz + (uint32_t)kk * 2048u, ID_PZ, kk > 0);
          if (C::REVERSE && !mbar_wait(&bars[B_P_FULL], pc, a.wait_ns, abort_flag)) { stop = true; break; }
          tc_fence_after();
#pragma unroll
          for (int kk = 4; kk < 8; ++kk)
            umma_ts(tmem + C::TM_OI, tmem + C::TM_P + 8u * kk, dz + (uint32_t)kk * 2048u, ID_PZ, 1);
          umma_commit(&bars[B_P_EMPTY]);
          umma_commit(&bars[B_O_FULL]);
          umma_commit(&bars[B_EMPTY + s]);
        } else {
          const int vb = SMM::NVT == 2 ? (gk & 1) : 0;  // weighted Z4 buffer and its phase
          const uint32_t vph = SMM::NVT == 2 ? (uint32_t)(gk >> 1) & 1u : pc;
          if (!mbar_wait(&bars[B_VT_FULL + vb], vph, a.wait_ns, abort_flag)) { stop = true; break; }
          // states only: U accumulates over the unit's chunks, read once after the last
          const bool u_first = !C::STATES || it == wi.it0, u_last = !C::STATES || it + 1 == wi.it1;
          if (u_first && !mbar_wait(&bars[B_U_EMPTY], (C::STATES ? (uint32_t)nu & 1u : pc) ^ 1u, a.wait_ns,
                                    abort_flag)) { stop = true; break; }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            umma(tmem + C::TM_U, sdesc(st + C::ST_K4, 16384, 1024, LAYOUT_SW128) + (uint32_t)kk * 2048u,
                 dvt + (uint32_t)vb * 2u * SZ_TILE64 + (uint32_t)kk * 2048u, ID_U, kk > 0 || !u_first);
          if (u_last) umma_commit(&bars[B_U_FULL]);
          umma_commit(&bars[B_VT_EMPTY + vb]);
          umma_commit(&bars[B_EMPTY + s]);
        }
       }
       if (C::STATES) nu += wi.it1 > wi.it0;
      }
      // All MMAs (and their barrier arrivals) finish before tensor memory is released.
      uint64_t* drain = &bars[B_DRAIN + (warp - 1)];
      umma_commit(drain);
      mbar_wait_drain(drain, 0, DRAIN_NS, a.err);
    }
    __syncwarp();
  } else if (warp < 8) {
    // ------------------------------------------------------------------ decay mask
    setmaxnreg_inc<C::REG_MASK>();
    if constexpr (!C::STATES) {
    const int i = threadIdx.x - 128;  // query row = tensor-memory lane
    const int q = warp & 3;           // this warp's lanes are rows 32q .. 32q + 31
    const uint32_t lane_addr = tmem + ((uint32_t)(q << 5) << 16);
    {  // P groups on the far side of this warp's diagonal stay zero for the whole kernel
      uint32_t z[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) z[e] = 0u;
      for (int g = 0; g < 4; ++g)
        if (C::REVERSE ? g < q : g > q) tmem_st16(lane_addr + C::TM_P + 16u * g, z);
      asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
    }
    int gk = 0, ku = 0;
    bool stop = false;
    for (int u = 0; u < n_items && !stop; ++u, ++ku) {
     const Unit wi = unit_at(u);
     const int tbuf = ku & 1;
     if (!warp_wait(&bars[B_TBL_FULL + tbuf], (uint32_t)(ku >> 1) & 1u, a, abort_flag)) break;
     const float* pws = pw_base + tbuf * PW_FLOATS + 129;  // scale * lambda^d of this unit's head
     const float lam = pw_base[tbuf * PW_FLOATS + 1];
     const float2 lam2 = make_float2(lam * lam, lam * lam);
     // Decay factors of the diagonal group for this lane: s lambda^(i-j) (forward, j <= i) or
     // s lambda^(j-i) (reverse, j >= i), zero across the diagonal; element pair e is columns
     // 32q + 2e and 32q + 2e + 1.
     float2 dgf[16];
#pragma unroll
     for (int e = 0; e < 16; ++e) {
       const int d0 = C::REVERSE ? 2 * e - lane : lane - 2 * e;
       const int d1 = C::REVERSE ? d0 + 1 : d0 - 1;
       dgf[e] = make_float2(d0 >= 0 ? pws[max(d0, 0)] : 0.f, d1 >= 0 ? pws[max(d1, 0)] : 0.f);
     }
     for (int it = wi.it0; it < wi.it1; ++it, ++gk) {
      const uint32_t pc = (uint32_t)gk & 1u;
      // Self-augmentation: row i's output gains sigmoid(q_i . (a_h * k_i)) v_i, which is that
      // gate added to P's diagonal entry (i, i) before MMA2.  The gate is read from the stage's
      // q and k rows (held until MMA2 is done), while MMA1 runs.
      float sig = 0.f;
      if constexpr (C::AUG) {
        if (!warp_wait(&bars[B_FULL + gk % C::NSTAGE], (uint32_t)(gk / C::NSTAGE) & 1u, a, abort_flag)) { stop = true; break; }
        const uint32_t st = sbase + (uint32_t)(gk % C::NSTAGE) * C::SZ_STAGE;
        const uint32_t avs = sbase + SMM::OFF_AUG + (uint32_t)tbuf * DK * 4u;
        // q: columns 0..63 in a 128B-swizzled panel, 64..95 in a 64B-swizzled one; k: two
        // 128B-swizzled panels.  16-byte piece p of a row holds columns 8p .. 8p + 7.  The sum
        // runs in four independent parts.
        float gp[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 2
        for (int p = 0; p < 12; ++p) {
          const uint4 qv = ld_shared_v4(p < 8 ? st + C::ST_X + (uint32_t)i * 128u + ((uint32_t)(p ^ (i & 7)) << 4)
                                              : st + C::ST_X1 + (uint32_t)i * 64u + ((uint32_t)((p - 8) ^ ((i >> 1) & 3)) << 4));
          const uint4 kv = ld_shared_v4(st + C::ST_Y + (uint32_t)(p >> 3) * 16384u + (uint32_t)i * 128u +
                                        ((uint32_t)((p & 7) ^ (i & 7)) << 4));
          const uint4 a0 = ld_shared_v4(avs + (uint32_t)p * 32u), a1 = ld_shared_v4(avs + (uint32_t)p * 32u + 16u);
          const uint32_t qw[4] = {qv.x, qv.y, qv.z, qv.w}, kw[4] = {kv.x, kv.y, kv.z, kv.w};
          const uint32_t aw[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 qf = bf2_to_f2(qw[e]), kf = bf2_to_f2(kw[e]);
            gp[e] = fmaf(qf.x * __uint_as_float(aw[2 * e]), kf.x, gp[e]);
            gp[e] = fmaf(qf.y * __uint_as_float(aw[2 * e + 1]), kf.y, gp[e]);
          }
        }
        sig = 1.f / (1.f + expf(-((gp[0] + gp[1]) + (gp[2] + gp[3]))));
      }
      if (!warp_wait(&bars[B_A_FULL], pc, a, abort_flag)) { stop = true; break; }
      if (!warp_wait(&bars[B_P_EMPTY], pc ^ 1u, a, abort_flag)) { stop = true; break; }
      tc_fence_after();
      // P row i, one 32-column group at a time, stored straight back to tensor memory.
      //   forward scans: s lambda^(i-j) A_ij for j <= i;  reverse scans: s lambda^(j-i) A_ij for j >= i.
      // Nothing is masked at the sequence end of a partial chunk: forward rows i >= L only reach
      // output rows that are never stored (j <= i < L bounds the rows that are), and in the reverse
      // scans the Z4 warps zero the rows j >= L of Z, which columns j >= L of P multiply.  Off the
      // diagonal group the factors come from one table read and a multiplicative chain toward
      // larger |i - j| (values only shrink, so an underflow to zero loses nothing); the diagonal
      // group uses the lane's factors, read from the table once per unit.
      // Reverse scans: P columns 0..63 (groups 0, 1, scaled first by the row blocks with the most
      // groups) are announced on their own, so that MMA2 can take its first four K steps while the
      // later groups are scaled.  (In the forward scans this measured slower.)
      const int g_first = C::REVERSE ? q : 0, g_last = C::REVERSE ? 3 : q;
      if (C::REVERSE && g_first > 1) mbar_arrive(&bars[B_P_HALF]);
      for (int g = g_first; g <= g_last; ++g) {
        uint32_t r[32];
        tmem_ld32(lane_addr + C::TM_A + 32u * g, r);
        if (g == g_last) {
          tc_fence_before();
          mbar_arrive(&bars[B_A_EMPTY]);
        }
        uint32_t pkg[16];
        if (g != q) {
          if (!C::REVERSE) {
            const int d0 = i - 32 * g;  // i - j at the group's first column (>= 1 here)
            float2 f = make_float2(pws[d0 - 30], pws[d0 - 31]);
#pragma unroll
            for (int e = 15; e >= 0; --e) {
              if (e < 15) f = mul2(f, lam2);
              const float2 pv = mul2(f, ld_f2(r, 2 * e));
              pkg[e] = pack_bf16(pv.x, pv.y);
            }
          } else {
            const int d0 = 32 * g - i;  // j - i at the group's first column (>= 1 here)
            float2 f = make_float2(pws[d0], pws[d0 + 1]);
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              if (e > 0) f = mul2(f, lam2);
              const float2 pv = mul2(f, ld_f2(r, 2 * e));
              pkg[e] = pack_bf16(pv.x, pv.y);
            }
          }
        } else {
          // diagonal group: the lane's own factors (fixed for the kernel)
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            float2 pv = mul2(dgf[e], ld_f2(r, 2 * e));
            if (C::AUG && e == (lane >> 1)) {  // the diagonal entry (column i) carries the gate
              if (lane & 1)
                pv.y += sig;
              else
                pv.x += sig;
            }
            pkg[e] = pack_bf16(pv.x, pv.y);
          }
        }
        tmem_st16(lane_addr + C::TM_P + 16u * g, pkg);
        if (C::REVERSE && g == 1) {
          asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
          tc_fence_before();
          mbar_arrive(&bars[B_P_HALF]);
        }
      }
      asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
      tc_fence_before();
      mbar_arrive(&bars[B_P_FULL]);
     }
     mbar_arrive(&bars[B_TBL_EMPTY + tbuf]);
    }
    }
  } else if (warp >= 12 && warp < 16) {
    // ------------------------------------------------------------------ weighted Z4 (hi and lo)
    setmaxnreg_dec<C::REG_Z4>();
    const int t = threadIdx.x - 384;  // row of the chunk
    int gk = 0, ku = 0;
    bool stop = false;
    for (int u = 0; u < n_items && !stop; ++u, ++ku) {
     const Unit w = unit_at(u);
     // This unit's decay table, into the buffer that unit ku - 2 used (once all its readers are done).
     const int tbuf = ku & 1;
     float* pw = pw_base + tbuf * PW_FLOATS;
     float* pws = pw + 129;
     if (ku >= 2 && !warp_wait(&bars[B_TBL_EMPTY + tbuf], (uint32_t)((ku - 2) >> 1) & 1u, a, abort_flag)) break;
     if (GLA_IN_BOUNDS(w.h >= 0 && w.h < a.H, a.err)) {
       const float ll = a.log_lambda[w.h];
       for (int d = t; d <= 128; d += 128) {
         const float pv = d == 0 ? 1.f : expf((float)d * ll);
         pw[d] = pv;
         pws[d] = a.scale * pv;
       }
       if (C::AUG && t < DK)
         reinterpret_cast<float*>(sm + SMM::OFF_AUG)[tbuf * DK + t] = a.aug[w.h * DK + t];
     }
     mbar_arrive(&bars[B_TBL_FULL + tbuf]);
     if (!warp_wait(&bars[B_TBL_FULL + tbuf], (uint32_t)(ku >> 1) & 1u, a, abort_flag)) break;
     for (int it = w.it0; it < w.it1; ++it, ++gk) {
      const int c = C::REVERSE ? w.nc - 1 - it : it;
      const int s = gk % C::NSTAGE;
      const uint32_t ph = (uint32_t)(gk / C::NSTAGE) & 1u, pc = (uint32_t)gk & 1u;
      const int L = min(CHUNK, w.len - c * CHUNK);
      if (!warp_wait(&bars[B_FULL + s], ph, a, abort_flag)) { stop = true; break; }
      const int vb = SMM::NVT == 2 ? (gk & 1) : 0;  // weighted Z4 buffer and its phase
      const uint32_t vph = SMM::NVT == 2 ? (uint32_t)(gk >> 1) & 1u : pc;
      if (!warp_wait(&bars[B_VT_EMPTY + vb], vph ^ 1u, a, abort_flag)) { stop = true; break; }
      const uint8_t* zsrc = sm + s * C::SZ_STAGE + C::ST_Z4;
      uint8_t* zhi = sm + SMM::OFF_VT + vb * 2 * SZ_TILE64;
      uint8_t* zlo = zhi + SZ_TILE64;
      {  // Z4t row j = w_j z_j; w_j = 0 past the sequence end
        const int j = t;
        float wj = j < L ? (C::REVERSE ? pws[j + 1] : pw[L - 1 - j]) : 0.f;
        // states only: weights relative to the unit's end (lambda^(len - 1 - position)), so that
        // MMA4 accumulates the whole unit's update in tensor memory
        if constexpr (C::STATES) wj *= expf((float)(w.len - c * CHUNK - L) * a.log_lambda[w.h]);
        const float2 f = make_float2(wj, wj);
        auto weigh = [&](int p) {
          const int off = j * 128 + ((p ^ (j & 7)) << 4);  // same permutation on both sides
          const uint4 x = *reinterpret_cast<const uint4*>(zsrc + off);
          const uint32_t w[4] = {x.x, x.y, x.z, x.w};
          uint32_t hi[4], lo[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) split_bf16x2(mul2(bf2_to_f2(w[e]), f), hi[e], lo[e]);
          *reinterpret_cast<uint4*>(zhi + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
          *reinterpret_cast<uint4*>(zlo + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
        };
        if constexpr (C::STATES) {  // (its own code: unrolled, all loads in flight together)
#pragma unroll
          for (int p = 0; p < 8; ++p) weigh(p);
        } else {
#pragma unroll 1
          for (int p = 0; p < 8; ++p) weigh(p);
        }
        if (C::REVERSE && j >= L) {
          // Reverse scans: rows of Z past the sequence end are zeroed, so MMA2 needs no column mask
          // on P (the mask warps leave P's columns j >= L unmasked).
          uint8_t* zrow = sm + s * C::SZ_STAGE + C::ST_Z + j * 128;
#pragma unroll 1
          for (int p = 0; p < (C::NARROW ? 16 : 8); ++p)
            *reinterpret_cast<uint4*>(zrow + (p >> 3) * 16384 + (((p & 7) ^ (j & 7)) << 4)) = make_uint4(0, 0, 0, 0);
        }
      }
      fence_async_smem();
      mbar_arrive(&bars[B_VT_FULL + vb]);
      if (C::REVERSE) mbar_arrive(&bars[B_ZR + s]);
     }
     mbar_arrive(&bars[B_TBL_EMPTY + tbuf]);
    }
  } else {
    // ------------------------------------------------------------------ epilogue
    // The running state of the unit's 96 x 64 tile (fp32 registers, thread r_ = d_k row):
    // S <- lambda^L S + U_hi + U_lo per chunk, its bf16 hi/lo copy for MMA3 and the final state;
    // and the output rows of each chunk from O_intra and O_inter (thread r_ = query row).  One
    // body, instantiated as a single role (forward: warps 8-11 do both, in the order update of
    // chunk it, copy for chunk it + 1, output of chunk it) or as two (backward: warps 8-11 the
    // state, warps 16-19 the output).
    auto epilogue = [&](auto do_state_t, auto do_out_t) {
      constexpr bool DO_STATE = decltype(do_state_t)::value, DO_OUT = decltype(do_out_t)::value;
      const int r_ = ((warp & 3) << 5) + lane;  // d_k row of the state and U; query row of O
      const uint32_t lane_addr = tmem + ((uint32_t)((warp & 3) << 5) << 16);
      const uint32_t spb = sbase + SMM::OFF_SP;
      const bool out32 = (reinterpret_cast<uintptr_t>(prm.out) & 31u) == 0;
      float S[TN];
      auto write_sprev = [&]() {
        if (r_ < DK) {
          const uint32_t row = sbase + SMM::OFF_SP + (uint32_t)r_ * 128u;
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
        mbar_arrive(&bars[B_SP_FULL]);
      };
      bool aborted = false;
      bool head_pending = false;  // a head piece's state load is in flight (thread r_ = 0)
      int nst = 0;  // full chunks stored through the staging tile
      int gk = 0, ku = 0, nu = 0;  // nu: units with chunks (states only: one U per unit)
      for (int u = 0; u < n_items && !aborted; ++u, ++ku) {
       const Unit w = unit_at(u);
       const int h = w.h, col0 = w.tile * TN, nc = w.nc, tbuf = ku & 1;
       if (!warp_wait(&bars[B_TBL_FULL + tbuf], (uint32_t)(ku >> 1) & 1u, a, abort_flag)) { aborted = true; break; }
       const float* pw = pw_base + tbuf * PW_FLOATS;
       const float* pws = pw + 129;
       const int srow0 = (w.n * a.H + h) * DK;  // the unit's first state row
       if constexpr (DO_STATE) {
#pragma unroll
         for (int x = 0; x < TN; ++x) S[x] = 0.f;
         if (C::FWD && w.head) {
           // (the hand-over tile lands in the state-copy buffer: the last MMA3 must have read it)
           if (gk > 0 && !warp_wait(&bars[B_SP_EMPTY], (uint32_t)(gk - 1) & 1u, a, abort_flag)) { aborted = true; break; }
           // The same tile's CTA of the previous group ran this unit's first chunks and left the
           // state in its final-state tile.  Thread r_ = 0 waits for that CTA's flag, lowers it
           // for the next launch and loads the tile into the (free) state-copy buffer by TMA; each
           // thread then takes its fp32 row from there (the row covers exactly the bytes of its
           // own hi and lo copy rows, so the copy written next overwrites nothing of another's).
           if (r_ == 0) {
             unsigned* flag = &g_handover[prm.flag_set * FLAG_MAX_CTAS + blockIdx.x - NTILE];
             unsigned long long t0 = ~0ull;
             bool seen = true;
             if (!GLA_IN_BOUNDS(prm.flag_set < FLAG_SETS && blockIdx.x >= NTILE && blockIdx.x < FLAG_MAX_CTAS + NTILE,
                                a.err)) {
               *abort_flag = 1;
               seen = false;
             }
             while (seen && ld_acquire_gpu(flag) != prm.epoch) {
               const unsigned long long tn = global_timer_ns();
               if (t0 == ~0ull) {
                 t0 = tn;
               } else if (*abort_flag || tn - t0 > a.wait_ns) {
                 *abort_flag = 1;
                 seen = false;
                 break;
               }
             }
             if (seen) {
               *reinterpret_cast<volatile unsigned*>(flag) = 0u;
               asm volatile("fence.proxy.async.global;" ::: "memory");
               head_pending = true;
               mbar_expect_tx(&bars[B_HANDOVER], 2 * SZ_SPH);
               tma_load_2d(spb, &maps.s, &bars[B_HANDOVER], col0, srow0);
               tma_load_2d(spb + SZ_SPH, &maps.s, &bars[B_HANDOVER], col0 + 32, srow0);
             }
           }
           if (!warp_wait(&bars[B_HANDOVER], 0u, a, abort_flag)) { aborted = true; break; }
           head_pending = false;
           if (r_ < DK) {
#pragma unroll
             for (int x = 0; x < TN / 4; ++x) {
               const uint4 v = ld_shared_v4(spb + (uint32_t)(x >> 3) * SZ_SPH + (uint32_t)r_ * 128u +
                                            ((uint32_t)((x & 7) ^ (r_ & 7)) << 4));
               S[4 * x] = __uint_as_float(v.x);
               S[4 * x + 1] = __uint_as_float(v.y);
               S[4 * x + 2] = __uint_as_float(v.z);
               S[4 * x + 3] = __uint_as_float(v.w);
             }
           }
         } else if (prm.s0 && r_ < DK && GLA_IN_BOUNDS(srow0 + r_ < state_rows && col0 + TN <= DV, a.err)) {
           const float4* src = reinterpret_cast<const float4*>(prm.s0 + ((long long)srow0 + r_) * DV + col0);
#pragma unroll
           for (int x = 0; x < TN / 4; ++x) {
             const float4 v4 = src[x];
             S[4 * x] = v4.x;
             S[4 * x + 1] = v4.y;
             S[4 * x + 2] = v4.z;
             S[4 * x + 3] = v4.w;
           }
         }
       }
       for (int it = w.it0 - 1; it < w.it1; ++it) {
        const int g = gk + (it - w.it0);  // the CTA's chunk count
        const uint32_t pc = (uint32_t)g & 1u;
        const int c = it < w.it0 ? 0 : (C::REVERSE ? nc - 1 - it : it);
        const int L = min(CHUNK, w.len - c * CHUNK);
        if constexpr (DO_STATE) {
          if (it >= w.it0 && (!C::STATES || it + 1 == w.it1)) {
            // state <- lambda^L state + U_hi + U_lo (states only: once per unit, L = its length)
            if (!warp_wait(&bars[B_U_FULL], C::STATES ? (uint32_t)nu & 1u : pc, a, abort_flag)) { aborted = true; break; }
            tc_fence_after();
            const float lamL = C::STATES ? expf((float)w.len * a.log_lambda[h]) : pw[L];
#pragma unroll
            for (int qq = 0; qq < 4; ++qq) {
              uint32_t u[32];  // [0, 16): hi columns, [16, 32): lo columns of this quarter
              tmem_ld16x2(lane_addr + C::TM_U + 16u * qq, lane_addr + C::TM_U + TN + 16u * qq, u);
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
          }
          if (!C::STATES && it + 1 < w.it1) {  // after MMA3 of this chunk has read the previous copy
            if (g >= 0 && !warp_wait(&bars[B_SP_EMPTY], pc, a, abort_flag)) { aborted = true; break; }
            write_sprev();
          }
        }
        if (it < w.it0) continue;
        if constexpr (DO_OUT && !C::STATES) {
          // out row = O_intra + g * O_inter;  g = s lambda^(i+1) (forward scans) or lambda^(L-1-i)
          if (!warp_wait(&bars[B_O_FULL], pc, a, abort_flag)) { aborted = true; break; }
          tc_fence_after();
          const float gf = C::REVERSE ? (r_ < L ? pw[L - 1 - r_] : 0.f) : pws[r_ + 1];
          const long long orow = (w.tb + (long long)c * CHUNK + r_) * a.H + h;
          if (!C::NARROW) {
            // Full chunks go through the staging tile, each warp's 32 rows with that warp's own TMA
            // store (no per-row stores on the load/store pipe, and no barrier across the warps: lane 0
            // waits for its previous store to have read the rows before they are rewritten); a partial
            // last chunk is stored row by row so that nothing past the sequence end is written.
            const bool staged = L == CHUNK;
            if (staged && nst > 0) {
              if (lane == 0) bulk_wait_read_all();
              __syncwarp();
            }
            uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(prm.out) + orow * DV + col0);
            const uint32_t srow = sbase + SMM::OFF_OST + (uint32_t)r_ * 128u;
#pragma unroll
            for (int qq = 0; qq < 4; ++qq) {
              uint32_t ov[48];  // 16 intra, 16 inter-hi, 16 inter-lo columns
              tmem_ld16x3(lane_addr + C::TM_OI + 16u * qq, lane_addr + C::TM_OE + 16u * qq,
                          lane_addr + C::TM_OE + TN + 16u * qq, ov);
              if (qq == 3) {
                tc_fence_before();
                mbar_arrive(&bars[B_O_EMPTY]);
              }
              uint32_t ob[8];
#pragma unroll
              for (int e = 0; e < 8; ++e) {
                const int x = 2 * e;
                const float2 ovx = fma2(make_float2(gf, gf), add2(ld_f2(ov, 16 + x), ld_f2(ov, 32 + x)), ld_f2(ov, x));
                ob[e] = pack_bf16(ovx.x, ovx.y);
              }
              if (staged) {  // 16-byte pieces 2qq, 2qq + 1 of the row, in the 128B-swizzled layout
                st_shared_v4(srow + ((uint32_t)((2 * qq) ^ (r_ & 7)) << 4), ob[0], ob[1], ob[2], ob[3]);
                st_shared_v4(srow + ((uint32_t)((2 * qq + 1) ^ (r_ & 7)) << 4), ob[4], ob[5], ob[6], ob[7]);
              } else if (r_ < L && GLA_IN_BOUNDS(orow >= 0 && orow < rows_total, a.err)) {
                if (out32) {  // one full 32-byte sector per store
                  st_global_v8(dst + 2 * qq, ob);
                } else {
                  dst[2 * qq] = make_uint4(ob[0], ob[1], ob[2], ob[3]);
                  dst[2 * qq + 1] = make_uint4(ob[4], ob[5], ob[6], ob[7]);
                }
              }
            }
            if (staged) {
              fence_async_smem();
              __syncwarp();
              if (lane == 0 && GLA_IN_BOUNDS(w.tb + (long long)c * CHUNK + 32 * (warp & 3) + 32 <= tokens, a.err))
                tma_store_3d(&maps.o, sbase + SMM::OFF_OST + (uint32_t)(warp & 3) * 4096u, col0, h,
                             (int)(w.tb + (long long)c * CHUNK) + 32 * (warp & 3));
              ++nst;
            }
          } else {
            // fp32 partial sums for the accumulator, 48 columns at a time: each thread writes its row
            // into the warp's region, then the warp adds contiguous 16-byte pieces (12 per row), so one
            // red.add instruction covers about three rows' segments instead of 32 rows.
            const uint32_t wreg = sbase + SMM::OFF_OST + (uint32_t)(warp & 3) * RED_WARP_BYTES;
            const long long row0 = (w.tb + (long long)c * CHUNK + ((warp & 3) << 5)) * a.H + h;  // lane 0's row
#pragma unroll
            for (int half = 0; half < 2; ++half) {
#pragma unroll
              for (int q3 = 0; q3 < 3; ++q3) {
                const int qq = 3 * half + q3;
                uint32_t ov[32];  // 16 intra, 16 inter columns
                tmem_ld16x2(lane_addr + C::TM_OI + 16u * qq, lane_addr + C::TM_OE + 16u * qq, ov);
                if (qq == 5) {
                  tc_fence_before();
                  mbar_arrive(&bars[B_O_EMPTY]);
                }
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  const float2 v0 = fma2(make_float2(gf, gf), ld_f2(ov, 16 + 4 * e), ld_f2(ov, 4 * e));
                  const float2 v1 = fma2(make_float2(gf, gf), ld_f2(ov, 18 + 4 * e), ld_f2(ov, 4 * e + 2));
                  st_shared_v4(wreg + (uint32_t)lane * RED_ROW + (uint32_t)(4 * q3 + e) * 16u, __float_as_uint(v0.x),
                               __float_as_uint(v0.y), __float_as_uint(v1.x), __float_as_uint(v1.y));
                }
              }
              __syncwarp();
#pragma unroll 2
              for (int k = 0; k < 12; ++k) {
                const int pidx = k * 32 + lane, row = pidx / 12, pc = pidx - row * 12;
                if (((warp & 3) << 5) + row < L && GLA_IN_BOUNDS(row0 + (long long)row * a.H < rows_total, a.err)) {
                  const uint4 v = ld_shared_v4(wreg + (uint32_t)row * RED_ROW + (uint32_t)pc * 16u);
                  red_add_v4(reinterpret_cast<float*>(prm.out) + (row0 + (long long)row * a.H) * DK + 48 * half + 4 * pc,
                             __uint_as_float(v.x), __uint_as_float(v.y), __uint_as_float(v.z), __uint_as_float(v.w));
                }
              }
              __syncwarp();
            }
          }
        }
       }
       if (aborted) break;
       nu += w.it1 > w.it0;
       if constexpr (DO_STATE) {
         if (C::FWD && prm.s_out) {
           // Forward: each thread stores its final-state row straight from registers (no staging,
           // nothing to wait for); a tail piece raises its hand-over flag once every row is visible.
           if (r_ < DK && GLA_IN_BOUNDS(srow0 + r_ < state_rows, a.err)) {
             float* dst = prm.s_out + ((long long)srow0 + r_) * DV + col0;
             if ((reinterpret_cast<uintptr_t>(prm.s_out) & 31u) == 0) {
#pragma unroll
               for (int x = 0; x < TN / 8; ++x) {
                 const uint32_t v[8] = {__float_as_uint(S[8 * x]),     __float_as_uint(S[8 * x + 1]),
                                        __float_as_uint(S[8 * x + 2]), __float_as_uint(S[8 * x + 3]),
                                        __float_as_uint(S[8 * x + 4]), __float_as_uint(S[8 * x + 5]),
                                        __float_as_uint(S[8 * x + 6]), __float_as_uint(S[8 * x + 7])};
                 st_global_v8(dst + 8 * x, v);
               }
             } else {
#pragma unroll
               for (int x = 0; x < TN / 4; ++x)
                 reinterpret_cast<float4*>(dst)[x] = make_float4(S[4 * x], S[4 * x + 1], S[4 * x + 2], S[4 * x + 3]);
             }
           }
           if (w.tail) {  // the next group's CTA continues this unit from the stored state
             __threadfence();
             mbar_arrive(&bars[B_ST_FULL]);
             if (r_ == 0) {
               if (mbar_wait(&bars[B_ST_FULL], 0u, a.wait_ns, abort_flag) &&
                   GLA_IN_BOUNDS(prm.flag_set < FLAG_SETS && blockIdx.x < FLAG_MAX_CTAS, a.err))
                 st_release_gpu(&g_handover[prm.flag_set * FLAG_MAX_CTAS + blockIdx.x], prm.epoch);
             }
           }
         }
         if (!C::FWD && prm.s_out && r_ < DK && GLA_IN_BOUNDS(srow0 + r_ < state_rows, a.err)) {
           float4* dst = reinterpret_cast<float4*>(prm.s_out + ((long long)srow0 + r_) * DV + col0);
#pragma unroll
           for (int x = 0; x < TN / 4; ++x) dst[x] = make_float4(S[4 * x], S[4 * x + 1], S[4 * x + 2], S[4 * x + 3]);
         }
       }
       mbar_arrive(&bars[B_TBL_EMPTY + tbuf]);
       gk += w.it1 - w.it0;
      }
      if (lane == 0) bulk_wait_read_all();  // this warp's last tile store has read shared memory
      if (r_ == 0 && head_pending) mbar_wait_drain(&bars[B_HANDOVER], 0u, DRAIN_NS, a.err);  // after an abort
    };
    if constexpr (!C::SPLIT) {
      setmaxnreg_inc<C::REG_STATE>();
      epilogue(std::true_type(), std::true_type());
    } else if (warp < 12) {
      setmaxnreg_inc<C::REG_STATE>();
      epilogue(std::true_type(), std::false_type());
    } else {
      setmaxnreg_dec<C::REG_OUT>();
      epilogue(std::false_type(), std::true_type());
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS));
  }
  if (threadIdx.x == 0 && *abort_flag) raise_error(a.err, ERR_TIMEOUT);
}

// fp32 partial-sum accumulator [T, H, 96] -> bf16 output (dq or dk).
__global__ void acc_to_bf16_kernel(const float4* __restrict__ acc, uint2* __restrict__ out, long long n4) {
  for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < n4; e += (long long)gridDim.x * blockDim.x) {
    const float4 a = acc[e];
    out[e] = make_uint2(pack_bf16(a.x, a.y), pack_bf16(a.z, a.w));
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
bool make_map(CUtensorMap* m, const void* base, int d, int H, long long T, int box_x, CUtensorMapSwizzle sw,
              int box_t = CHUNK) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)H, (cuuint64_t)T};
  const cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)H * d * 2};
  const cuuint32_t box[3] = {(cuuint32_t)box_x, 1, (cuuint32_t)box_t};
  const cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D view [n_seq * H * 96, 192] of an fp32 state tensor [n_seq, H, 96, 192]; box = 32 columns x
// 96 rows (half of a unit's tile), 128B swizzle.
bool make_state_map(CUtensorMap* m, const void* base, long long rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)DV, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)DV * 4};
  const cuuint32_t box[2] = {32, (cuuint32_t)DK};
  const cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// max_ctas > 0 makes the CTAs persistent: max_ctas of them (more if a CTA would get more than
// MAX_ITEMS units), each running every gridDim.x-th work unit; 0 launches one CTA per unit and
// leaves the order to the block scheduler.
template <int MODE>
cudaError_t launch_scan(const void* X, const void* Y, const void* Z, const ScanParams& p, cudaStream_t stream,
                        int max_ctas) {
  using C = Cfg<MODE>;
  const ChunkArgs& a = p.a;
  long long blocks = (long long)a.n_seq * a.H * NTILE;  // work units
  if (blocks == 0) return cudaSuccess;
  if (max_ctas > 0 && blocks > max_ctas) blocks = std::max((long long)max_ctas, (blocks + MAX_ITEMS - 1) / MAX_ITEMS);
  const long long T_total = a.cu_seqlens ? (long long)a.T : (long long)a.n_seq * a.T;
  TmaMaps maps;
  memset(&maps, 0, sizeof(maps));
  if (T_total > 0) {
    const int dx = C::NARROW ? DV : DK, dz = C::NARROW ? DK : DV;
    if (!make_map(&maps.x, X, dx, a.H, T_total, 64, CU_TENSOR_MAP_SWIZZLE_128B) ||
        (!C::NARROW && !make_map(&maps.x1, X, DK, a.H, T_total, 32, CU_TENSOR_MAP_SWIZZLE_64B)) ||
        !make_map(&maps.y, Y, dx, a.H, T_total, 64, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map(&maps.z, Z, dz, a.H, T_total, 64, CU_TENSOR_MAP_SWIZZLE_128B) ||
        (!C::NARROW && !C::STATES && !make_map(&maps.o, p.out, DV, a.H, T_total, 64, CU_TENSOR_MAP_SWIZZLE_128B, 32)))
      return cudaErrorInvalidValue;
  }
  const long long state_rows = (long long)a.n_seq * a.H * DK;
  if (Cfg<MODE>::FWD && p.s_out && !make_state_map(&maps.s, p.s_out, state_rows))
    return cudaErrorInvalidValue;
  static bool attr_set = false;
  if (!attr_set) {
    // The warpgroups' setmaxnreg split redistributes exactly the registers the CTA is launched
    // with; with any other compiled count an increase could wait forever, so refuse to launch.
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, tc_scan_kernel<MODE>);
    if (e != cudaSuccess) return e;
    if (fa.numRegs != C::REG_LAUNCH) return cudaErrorInvalidConfiguration;
    e = cudaFuncSetAttribute(tc_scan_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Smem<MODE>::BYTES);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  // A balanced launch needs all its CTAs resident at once (a CTA may wait for its predecessor's
  // flag), which a cooperative launch guarantees or refuses; refused, it runs plain instead.
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = dim3((unsigned)blocks);
  cfg.blockDim = dim3(C::THREADS);
  cfg.dynamicSmemBytes = Smem<MODE>::BYTES;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  if (p.balanced) {
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, tc_scan_kernel<MODE>, maps, p) == cudaSuccess) return cudaSuccess;
    (void)cudaGetLastError();
    ScanParams plain = p;
    plain.balanced = 0;
    cfg.attrs = nullptr;
    cfg.numAttrs = 0;
    return cudaLaunchKernelEx(&cfg, tc_scan_kernel<MODE>, maps, plain);
  }
  return cudaLaunchKernelEx(&cfg, tc_scan_kernel<MODE>, maps, p);
}

}  // namespace

size_t tc_bwd_acc_bytes(long long T_total, int H) { return (size_t)T_total * H * DK * sizeof(float); }

cudaError_t launch_tc_fwd(const ChunkArgs& a, cudaStream_t stream) {
  ScanParams p;
  p.a = a;
  p.s0 = a.h0;
  p.s_out = a.hT;
  p.out = a.o;
  // Equal-length batches: one persistent CTA per SM (a unit's first loads overlap the previous
  // unit's last chunks).  Packed varlen batches: one CTA per unit, so that the block scheduler
  // hands the next (longest-first) unit to whichever SM frees up.
  // With at least as many units as SMs and a final-state output to hand states over through, the
  // chunks are split evenly over the persistent CTAs (balanced), so no SM idles while others run
  // a last round of whole units.
  int max_ctas = 0;
  if (!a.cu_seqlens) {
    int dev = 0;
    max_ctas = 152;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&max_ctas, cudaDevAttrMultiProcessorCount, dev);
    const long long units = (long long)a.n_seq * a.H * NTILE;
    if (a.hT && a.T > 0 && units / NTILE >= max_ctas / NTILE && max_ctas <= FLAG_MAX_CTAS &&
        units / NTILE * ((a.T + CHUNK - 1) / CHUNK) < (1ll << 31)) {
      static std::atomic<unsigned> launches{0};
      const unsigned n = launches.fetch_add(1u);
      p.balanced = 1;
      p.flag_set = (int)(n % FLAG_SETS);
      p.epoch = n / FLAG_SETS % 0xFFFFFFFu + 1u;
    }
  }
  if (a.aug) return launch_scan<MODE_FWDA>(a.q, a.k, a.v, p, stream, max_ctas);
  return launch_scan<MODE_FWD>(a.q, a.k, a.v, p, stream, max_ctas);
}

// The forward's final states only (hT; no outputs), one CTA per unit.  Refused (an error) when
// the states-only kernel did not compile to the register count its role split needs.
cudaError_t launch_tc_fwd_states(const ChunkArgs& a, cudaStream_t stream) {
  // packed sequences only: one CTA per whole unit (the states-only weights are relative to the
  // unit's end, so a unit is never split into pieces)
  if (!a.cu_seqlens) return cudaErrorInvalidValue;
  ScanParams p;
  p.a = a;
  p.s0 = a.h0;
  p.s_out = a.hT;
  p.out = nullptr;
  return launch_scan<MODE_FWDS>(a.q, a.k, a.v, p, stream, 0);
}

// After a wait gave up, a hand-over flag may have been left raised; lower them all.
cudaError_t tc_clear_handover(cudaStream_t stream) {
  void* p = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&p, g_handover);
  if (e != cudaSuccess) return e;
  return cudaMemsetAsync(p, 0, sizeof(g_handover), stream);
}

namespace {
// Two side streams per device for the backward's independent scans (created on first use).
constexpr int kMaxDevices = 64;
std::mutex g_stream_mu;
cudaStream_t g_side[kMaxDevices][2];

cudaError_t side_streams(cudaStream_t (&out)[2]) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_stream_mu);
  for (int i = 0; i < 2; ++i) {
    if (!g_side[dev][i]) {
      e = cudaStreamCreateWithFlags(&g_side[dev][i], cudaStreamNonBlocking);
      if (e != cudaSuccess) return e;
    }
    out[i] = g_side[dev][i];
  }
  return cudaSuccess;
}
}  // namespace

// Backward in bf16: dv and dh0 directly; dq and dk through fp32 partial sums in acc_q / acc_k
// (each tc_bwd_acc_bytes, 16-byte aligned), each rounded to bf16 once its scan is done.  The three
// scans are independent: DV runs on the caller's stream, and DK and DQ (each with its zeroing and
// its rounding pass) on two side streams forked from it and joined back with events, so their
// kernels fill each other's idle SMs.
cudaError_t launch_tc_bwd(const ChunkArgs& a, float* acc_q, float* acc_k, cudaStream_t stream) {
  const long long T_total = a.cu_seqlens ? (long long)a.T : (long long)a.n_seq * a.T;
  const size_t acc = tc_bwd_acc_bytes(T_total, a.H);
  const long long n4 = T_total * a.H * DK / 4;
  cudaError_t e;
  cudaStream_t side[2];
  if ((e = side_streams(side)) != cudaSuccess) return e;
  int dev = 0, sms = 152;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  long long conv_blocks = (n4 + 255) / 256;
  if (conv_blocks > (long long)sms * 8) conv_blocks = (long long)sms * 8;
  // One side stream per accumulator: zero it, run its scan, round it to bf16.
  auto partial_scan = [&](cudaStream_t st, float* acc_p, void* out, bool dk_scan) -> cudaError_t {
    cudaError_t r;
    if (acc && (r = cudaMemsetAsync(acc_p, 0, acc, st)) != cudaSuccess) return r;
    ScanParams p;
    p.a = a;
    p.s_out = nullptr;
    p.out = acc_p;
    if (dk_scan) {
      p.s0 = a.dhT;
      r = launch_scan<MODE_DK>(a.v, a.dO, a.q, p, st, 0);
    } else {
      p.s0 = a.h0;
      r = launch_scan<MODE_DQ>(a.dO, a.v, a.k, p, st, 0);
    }
    if (r != cudaSuccess) return r;
    if (n4 > 0) {
      acc_to_bf16_kernel<<<(unsigned)conv_blocks, 256, 0, st>>>(reinterpret_cast<const float4*>(acc_p),
                                                                reinterpret_cast<uint2*>(out), n4);
      r = cudaGetLastError();
    }
    return r;
  };
  cudaEvent_t ev[3] = {nullptr, nullptr, nullptr};
  for (int i = 0; i < 3; ++i)
    if ((e = cudaEventCreateWithFlags(&ev[i], cudaEventDisableTiming)) != cudaSuccess) break;
  if (e == cudaSuccess) e = cudaEventRecord(ev[0], stream);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(side[0], ev[0], 0);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(side[1], ev[0], 0);
  if (e == cudaSuccess) e = partial_scan(side[0], acc_k, a.dk, true);
  if (e == cudaSuccess) e = partial_scan(side[1], acc_q, a.o, false);  // a.o carries dq here
  if (e == cudaSuccess) {
    ScanParams p;
    p.a = a;
    p.s0 = a.dhT;
    p.s_out = a.hT;  // dh0
    p.out = a.dv;
    e = launch_scan<MODE_DV>(a.k, a.q, a.dO, p, stream, 0);
  }
  if (e == cudaSuccess) e = cudaEventRecord(ev[1], side[0]);
  if (e == cudaSuccess) e = cudaEventRecord(ev[2], side[1]);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(stream, ev[1], 0);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(stream, ev[2], 0);
  for (int i = 0; i < 3; ++i)
    if (ev[i]) cudaEventDestroy(ev[i]);
  return e;
}

}  // namespace gla
