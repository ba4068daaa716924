// gla_chunk_fwd_noalloc: the chunked forward without any device allocation or workspace.
//
// Some callers cannot allocate device memory per call: a serving engine that hands all of the
// GPU's memory to its own pool at start-up and plans every byte in advance, or host code running
// where no allocator is reachable.  gla_chunk_fwd asks such callers for a workspace (the
// longest-first schedule of packed sequences); this variant keeps that schedule instead in a
// fixed array in device memory that the library owns, so the caller passes only inputs and outputs.
//
// The array holds GLA_NOALLOC_MAX_SEQS int32 entries (64 KB) and every GPU that loads the library
// keeps it until the process exits.  All calls on a device share it: the schedule kernel rewrites
// the entries a call uses before the forward kernel reads them, so nothing needs clearing, but two
// calls that overlap on the GPU (different streams, no ordering between them) race on it.
#include <mutex>

#include "gla.h"
#include "gla_common.cuh"

namespace gla {
cudaError_t launch_simt_fwd(const ChunkArgs& a, cudaStream_t stream);
cudaError_t launch_tc_fwd(const ChunkArgs& a, cudaStream_t stream);
cudaError_t launch_lpt_order(const int32_t* cu_seqlens, int n_seq, int32_t* order, cudaStream_t stream);
int current_device_state(unsigned** err, unsigned long long* wait_ns);
int check_chunk_sizes(int n_seq, int T, int H, int dk, int dv, int dtype, const int32_t* cu_seqlens,
                      long long* tokens);
}  // namespace gla

namespace {

static __device__ __align__(256) int32_t g_noalloc_order[GLA_NOALLOC_MAX_SEQS];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
int32_t* g_order_ptr[kMaxDevices];

// Device address of g_noalloc_order on the current device, looked up once per device (the name
// is only a host-side stand-in for the array; a kernel must be given the address below).
int order_scratch(int32_t** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GLA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_order_ptr[dev]) {
    int32_t* p = nullptr;
    if (cudaGetSymbolAddress((void**)&p, g_noalloc_order) != cudaSuccess || !p) return GLA_ERR_LAUNCH;
    g_order_ptr[dev] = p;
  }
  *out = g_order_ptr[dev];
  return GLA_OK;
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

}  // namespace

extern "C" int gla_chunk_fwd_noalloc(const void* q, const void* k, const void* v, const float* log_lambda,
                                     const float* h0, float scale, void* o, float* hT,
                                     const int32_t* cu_seqlens, int n_seq, int T, int H, int dk, int dv,
                                     int dtype, gla_stream_t stream) {
  // the same size checks as gla_chunk_fwd (the device indexing is 32-bit)
  long long tokens = 0;
  int rc = gla::check_chunk_sizes(n_seq, T, H, dk, dv, dtype, cu_seqlens, &tokens);
  if (rc) return rc;
  if (cu_seqlens && n_seq > GLA_NOALLOC_MAX_SEQS) return GLA_ERR_WORKSPACE;
  if (n_seq == 0) return GLA_OK;
  if (!log_lambda) return GLA_ERR_NULL;
  if (tokens > 0 && (!q || !k || !v || !o)) return GLA_ERR_NULL;
  for (const void* p : {(const void*)q, (const void*)k, (const void*)v, (const void*)o,
                        (const void*)h0, (const void*)hT, (const void*)log_lambda})
    if (p && !aligned16(p)) return GLA_ERR_ALIGN;
  unsigned* err;
  unsigned long long wait_ns;
  rc = gla::current_device_state(&err, &wait_ns);
  if (rc) return rc;

  gla::ChunkArgs a = {};
  a.q = q;
  a.k = k;
  a.v = v;
  a.log_lambda = log_lambda;
  a.h0 = h0;
  a.o = o;
  a.hT = hT;
  a.cu_seqlens = cu_seqlens;
  a.scale = scale;
  a.n_seq = n_seq;
  a.T = T;
  a.H = H;
  a.err = err;
  a.wait_ns = wait_ns;
  cudaStream_t s = (cudaStream_t)stream;
  if (cu_seqlens) {
    int32_t* order = nullptr;
    rc = order_scratch(&order);
    if (rc) return rc;
    if (gla::launch_lpt_order(cu_seqlens, n_seq, order, s) != cudaSuccess) return GLA_ERR_LAUNCH;
    a.order = order;
  }
  const cudaError_t e = dtype == GLA_F32 ? gla::launch_simt_fwd(a, s) : gla::launch_tc_fwd(a, s);
  return e == cudaSuccess ? GLA_OK : GLA_ERR_LAUNCH;
}
