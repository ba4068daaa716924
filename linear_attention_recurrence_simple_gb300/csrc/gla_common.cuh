// Device-side helpers shared by the GLA kernels: element conversion, the sticky error word,
// bounded waits, and the argument block every chunked kernel receives.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace gla {

constexpr int DK = 96;
constexpr int DV = 192;
constexpr int CHUNK = 128;

// Positive codes stored in the device error word (the host negates them into gla_status).
constexpr unsigned ERR_SHAPE = 2;
constexpr unsigned ERR_TIMEOUT = 8;
constexpr unsigned ERR_BOUNDS = 9;

// Everything a chunked forward or backward kernel needs; passed by value.
struct ChunkArgs {
  const void* q;
  const void* k;
  const void* v;
  const void* dO;          // backward only
  const float* log_lambda;
  const float* h0;         // may be null
  const float* aug;        // forward only: aug_balance [H, 96] (self-augmentation), or null
  const float* dhT;        // backward only; may be null
  void* o;                 // forward output (or dq in the backward)
  void* dk;                // backward only
  void* dv;                // backward only
  float* hT;               // forward final state / backward dh0; may be null
  const int32_t* cu_seqlens;  // null: fixed length T
  const int32_t* order;       // longest-first sequence order (packed calls), or null
  float scale;
  int n_seq;
  int T;                   // per-sequence length (fixed) or packed total
  int H;
  unsigned* err;           // device error word
  unsigned long long wait_ns;  // limit of every bounded wait
};

// The decode step's fused per-tier Head RMSNorm + SiLU gate: g [N, H, 192] (dtype of o), the
// tier gains weight [n_tiers, 192] fp32, the head-to-tier map tier [H] int32, eps.
struct DecodeNormGate {
  const void* g;
  const float* w;
  const int32_t* tier;
  int n_tiers;
  float eps;
};

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }

template <class T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

__device__ __forceinline__ void raise_error(unsigned* word, unsigned code) {
  atomicCAS(word, 0u, code);
}

// Index checks of the debug-bounds build (compiled with -DGLA_DEBUG_BOUNDS, a stand-in for a
// memory checker): `ok` states that an access stays inside its buffer; when it does not, the
// error word records ERR_BOUNDS and the caller skips the access.  In the release build the check
// is the constant true and the condition is never evaluated.
#ifdef GLA_DEBUG_BOUNDS
constexpr bool kDebugBounds = true;
#define GLA_IN_BOUNDS(ok, err) (::gla::in_bounds_check((ok), (err)))
__device__ __forceinline__ bool in_bounds_check(bool ok, unsigned* err) {
  if (!ok) raise_error(err, ERR_BOUNDS);
  return ok;
}
#else
constexpr bool kDebugBounds = false;
#define GLA_IN_BOUNDS(ok, err) true
#endif

// Token range [begin, end) of sequence n.  Packed offsets are read on the device, so they are
// clamped here to 0 <= begin <= end <= T (the packed total), which keeps every access inside the
// caller's buffers whatever the offsets hold; an offset that needed clamping (decreasing, negative
// or past T) records ERR_SHAPE in the error word.
__device__ __forceinline__ void seq_range(const ChunkArgs& a, int n, long long& begin, long long& end) {
  if (a.cu_seqlens) {
    const long long b = a.cu_seqlens[n], e = a.cu_seqlens[n + 1];
    begin = min(max(b, 0ll), (long long)a.T);
    end = min(max(e, begin), (long long)a.T);
    if (begin != b || end != e) raise_error(a.err, ERR_SHAPE);
  } else {
    begin = (long long)n * a.T;
    end = begin + a.T;
  }
}

// Splits a 1-D work-unit index into (sequence, head, tile) with the sequence slowest, so that
// with a longest-first order the longest sequences start first.
__device__ __forceinline__ void unit_of(const ChunkArgs& a, int tiles, int b, int& n, int& h, int& tile) {
  const unsigned per_seq = (unsigned)a.H * (unsigned)tiles;  // the host keeps unit counts below 2^31
  const int rank = (int)((unsigned)b / per_seq);
  const int rem = (int)((unsigned)b - (unsigned)rank * per_seq);
  h = rem / tiles;
  tile = rem % tiles;
  n = a.order && GLA_IN_BOUNDS(rank < a.n_seq, a.err) ? a.order[rank] : rank;
  if (!GLA_IN_BOUNDS(n >= 0 && n < a.n_seq, a.err)) n = 0;
}
// Debug-bounds build: a unit's (sequence, head) and a chunk's rows [t0, t0 + L) lie inside the
// caller's buffers (always true in the release build).
__device__ __forceinline__ bool unit_in_bounds([[maybe_unused]] const ChunkArgs& a, [[maybe_unused]] int n,
                                               [[maybe_unused]] int h) {
  return GLA_IN_BOUNDS(n >= 0 && n < a.n_seq && h >= 0 && h < a.H, a.err);
}
__device__ __forceinline__ bool rows_in_bounds([[maybe_unused]] const ChunkArgs& a, [[maybe_unused]] long long t0,
                                               [[maybe_unused]] int L) {
  return GLA_IN_BOUNDS(t0 >= 0 && L >= 0 && t0 + L <= (a.cu_seqlens ? (long long)a.T : (long long)a.n_seq * a.T),
                       a.err);
}
__device__ __forceinline__ void unit_of_block(const ChunkArgs& a, int tiles, int& n, int& h, int& tile) {
  unit_of(a, tiles, (int)blockIdx.x, n, h, tile);
}

__device__ __forceinline__ unsigned long long global_timer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ------------------------------------------------------------------------------------------
// mbarrier helpers (shared::cta).  Every wait is bounded: it repeats try_wait, reads the global
// timer after each, and gives up after `limit_ns` (or as soon as *abort is set).
// ------------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("{\n .reg .b64 st;\n mbarrier.arrive.shared::cta.b64 st, [%0];\n}" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("{\n .reg .b64 st;\n mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n}" ::"r"(
                   smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

// One try_wait (the hardware may suspend the thread for a short, system-dependent time before it
// returns false).  A suspend-time hint was measured slower once the load/store pipe stopped
// backing up: a wait whose phase has already completed then cost ~250 cycles.
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait of a CTA role.  It gives up once `limit_ns` has passed since its first failed
// try_wait, or as soon as another role has given up (*abort set), and then sets *abort and returns
// false; the kernel reports ERR_TIMEOUT once, at exit, when *abort is set.  Kept small because
// every wait site is inlined into the warp-specialised kernels, whose speed depends on their code
// fitting the instruction caches.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, unsigned long long limit_ns,
                                          volatile int* abort) {
  unsigned long long t0 = ~0ull;
  while (!mbar_try_wait(bar, parity)) {
    const unsigned long long t = global_timer_ns();
    if (t0 == ~0ull) {
      t0 = t;
    } else if (*abort || t - t0 > limit_ns) {
      *abort = 1;
      return false;
    }
  }
  return true;
}

// Bounded wait on the exit path (no abort flag): raises ERR_TIMEOUT itself.
__device__ __forceinline__ void mbar_wait_drain(uint64_t* bar, uint32_t parity, unsigned long long limit_ns,
                                                unsigned* err) {
  const unsigned long long t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > limit_ns) {
      raise_error(err, ERR_TIMEOUT);
      return;
    }
  }
}

}  // namespace gla
