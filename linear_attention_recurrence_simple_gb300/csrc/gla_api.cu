// C ABI of libgla.so: argument validation, kernel choice, launches on the caller's stream, and
// the per-device sticky error word.  Nothing here allocates device memory.
#include <mutex>

#include "gla.h"
#include "gla_common.cuh"

namespace gla {
cudaError_t launch_decode_step(int dtype_f32, int state_bf16, const void* q, const void* k, const void* v,
                               const float* log_lambda, float scale, void* state,
                               const int32_t* slot, int pool_rows, void* o, int N, int H,
                               const float* aug, unsigned* err, cudaStream_t stream,
                               const DecodeNormGate* ngp);
cudaError_t launch_simt_fwd(const ChunkArgs& a, cudaStream_t stream);
cudaError_t launch_simt_bwd(int dtype_f32, const ChunkArgs& a, cudaStream_t stream);
cudaError_t launch_tc_fwd(const ChunkArgs& a, cudaStream_t stream);
cudaError_t launch_tc_bwd(const ChunkArgs& a, float* acc_q, float* acc_k, cudaStream_t stream);
size_t tc_bwd_acc_bytes(long long T_total, int H);
cudaError_t tc_clear_handover(cudaStream_t stream);
int check_chunk_sizes(int n_seq, int T, int H, int dk, int dv, int dtype, const int32_t* cu_seqlens,
                      long long* tokens);
cudaError_t launch_mxfp8_quantise(const float* x, uint8_t* codes, uint8_t* scales, long long rows,
                                  cudaStream_t stream);
cudaError_t launch_mxfp8_dequantise(const uint8_t* codes, const uint8_t* scales, float* x, long long rows,
                                    cudaStream_t stream);
cudaError_t launch_decode_step_mxfp8(int dtype_f32, const void* q, const void* k, const void* v,
                                     const float* log_lambda, float scale, uint8_t* codes, uint8_t* scales,
                                     const int32_t* slot, int pool_rows, void* o, int N, int H,
                                     const float* aug, unsigned* err, unsigned long long wait_ns,
                                     cudaStream_t stream);
cudaError_t launch_head_norm_gate(int dtype_f32, const void* o, const void* g, const float* w,
                                  const int32_t* tier, int n_tiers, float eps, void* y, long long rows,
                                  int H, unsigned* err, cudaStream_t stream);
}  // namespace gla

namespace {

// Sticky error word, one per device (each device that loads the module gets its own copy).
__device__ unsigned g_error_word;

constexpr int kMaxDevices = 64;
constexpr int kSortMaxSeqs = 16384;  // longest-first ordering up to this many sequences
std::mutex g_mu;
unsigned* g_err_ptr[kMaxDevices];
int g_dev_ok[kMaxDevices];  // 0 unknown, 1 sm_103, -1 other
unsigned long long g_wait_ns[kMaxDevices];

// Ranks sequence i by (length descending, index ascending); order[rank] = i.
__global__ void lpt_order_kernel(const int32_t* __restrict__ cu, int n_seq, int32_t* __restrict__ order) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n_seq) return;
  if (n_seq > kSortMaxSeqs) {
    order[i] = i;
    return;
  }
  const int li = cu[i + 1] - cu[i];
  int rank = 0;
  for (int j = 0; j < n_seq; ++j) {
    const int lj = cu[j + 1] - cu[j];
    rank += (lj > li) || (lj == li && j < i);
  }
  order[rank] = i;
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

// Current device, its sm_103 check, and its error-word address.
int device_state(int* dev_out, unsigned** err_out, unsigned long long* wait_out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GLA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_dev_ok[dev] == 0) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
      return GLA_ERR_UNSUPPORTED;
    }
    g_dev_ok[dev] = (major == 10 && minor == 3) ? 1 : -1;
  }
  if (g_dev_ok[dev] != 1) return GLA_ERR_UNSUPPORTED;
  if (!g_err_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_error_word) != cudaSuccess) return GLA_ERR_LAUNCH;
    g_err_ptr[dev] = (unsigned*)p;
  }
  if (g_wait_ns[dev] == 0) g_wait_ns[dev] = 2000000000ull;
  *dev_out = dev;
  *err_out = g_err_ptr[dev];
  *wait_out = g_wait_ns[dev];
  return GLA_OK;
}

// Checks shared by the forward and backward; fills the sequence/schedule part of `a`.
int check_chunk_call(int n_seq, int T, int H, int dk, int dv, int dtype, const int32_t* cu_seqlens,
                     void* workspace, size_t ws_bytes, long long* tokens) {
  const int rc = gla::check_chunk_sizes(n_seq, T, H, dk, dv, dtype, cu_seqlens, tokens);
  if (rc) return rc;
  if (cu_seqlens) {
    if (n_seq > 0) {
      if (!workspace) return GLA_ERR_WORKSPACE;
      if (ws_bytes < gla_workspace_bytes(n_seq, H)) return GLA_ERR_WORKSPACE;
      if (!aligned16(workspace)) return GLA_ERR_ALIGN;
    }
  }
  return GLA_OK;
}

int to_status(cudaError_t e) { return e == cudaSuccess ? GLA_OK : GLA_ERR_LAUNCH; }

}  // namespace

namespace gla {
// Size, dtype and layout checks of every chunked call (with or without a workspace): dtype,
// d_k / d_v, non-negative sizes, the 32-bit limits of the device indexing (state rows (sequence,
// head, d_k row), work units and token coordinates), and the alignment of cu_seqlens.  Sets the
// token count.
int check_chunk_sizes(int n_seq, int T, int H, int dk, int dv, int dtype, const int32_t* cu_seqlens,
                      long long* tokens) {
  if (dtype != GLA_BF16 && dtype != GLA_F32) return GLA_ERR_DTYPE;
  if (dk != GLA_DK || dv != GLA_DV) return GLA_ERR_UNSUPPORTED;
  if (n_seq < 0 || T < 0 || H < 1) return GLA_ERR_SHAPE;
  *tokens = cu_seqlens ? (long long)T : (long long)n_seq * T;
  if ((long long)n_seq * H * GLA_DK >= (1ll << 31) || *tokens >= (1ll << 31)) return GLA_ERR_SHAPE;
  if (cu_seqlens && ((uintptr_t)cu_seqlens & 3u)) return GLA_ERR_ALIGN;
  return GLA_OK;
}
// Internal accessors for the allocation-free entry point (gla_noalloc.cu); the entry points
// above do not go through them.
int current_device_state(unsigned** err, unsigned long long* wait_ns) {
  int dev;
  return device_state(&dev, err, wait_ns);
}
cudaError_t launch_lpt_order(const int32_t* cu_seqlens, int n_seq, int32_t* order, cudaStream_t stream) {
  lpt_order_kernel<<<(n_seq + 255) / 256, 256, 0, stream>>>(cu_seqlens, n_seq, order);
  return cudaGetLastError();
}
}  // namespace gla

extern "C" {

size_t gla_workspace_bytes(int n_seq, int H) {
  (void)H;
  if (n_seq < 0) return 0;
  return 256 + (((size_t)n_seq * sizeof(int32_t) + 255) / 256) * 256;
}

size_t gla_bwd_workspace_bytes(int n_seq, int T, int H, int packed, int dtype) {
  if (n_seq < 0 || T < 0 || H < 1) return 0;
  size_t bytes = packed ? gla_workspace_bytes(n_seq, H) : 0;
  if (dtype == GLA_BF16) {
    const long long T_total = packed ? (long long)T : (long long)n_seq * T;
    const size_t acc = ((gla::tc_bwd_acc_bytes(T_total, H) + 255) / 256) * 256;
    bytes = (bytes ? bytes : 256) + 2 * acc;
  }
  return bytes;
}

static int chunk_fwd(const void* q, const void* k, const void* v, const float* log_lambda,
                     const float* h0, float scale, const float* aug, void* o, float* hT,
                     const int32_t* cu_seqlens, int n_seq, int T, int H, int dk, int dv, int dtype,
                     void* workspace, size_t ws_bytes, gla_stream_t stream) {
  long long tokens = 0;
  int rc = check_chunk_call(n_seq, T, H, dk, dv, dtype, cu_seqlens, workspace, ws_bytes, &tokens);
  if (rc) return rc;
  if (n_seq == 0) return GLA_OK;
  if (!log_lambda) return GLA_ERR_NULL;
  if (tokens > 0 && (!q || !k || !v || !o)) return GLA_ERR_NULL;
  for (const void* p : {(const void*)q, (const void*)k, (const void*)v, (const void*)o,
                        (const void*)h0, (const void*)hT, (const void*)log_lambda, (const void*)aug})
    if (p && !aligned16(p)) return GLA_ERR_ALIGN;
  int dev;
  unsigned* err;
  unsigned long long wait_ns;
  rc = device_state(&dev, &err, &wait_ns);
  if (rc) return rc;

  gla::ChunkArgs a = {};
  a.q = q;
  a.k = k;
  a.v = v;
  a.log_lambda = log_lambda;
  a.h0 = h0;
  a.aug = aug;
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
    int32_t* order = (int32_t*)((char*)workspace + 256);
    lpt_order_kernel<<<(n_seq + 255) / 256, 256, 0, s>>>(cu_seqlens, n_seq, order);
    if (cudaGetLastError() != cudaSuccess) return GLA_ERR_LAUNCH;
    a.order = order;
  }
  if (dtype == GLA_F32) return to_status(gla::launch_simt_fwd(a, s));
  return to_status(gla::launch_tc_fwd(a, s));
}

int gla_chunk_fwd(const void* q, const void* k, const void* v, const float* log_lambda,
                  const float* h0, float scale, void* o, float* hT, const int32_t* cu_seqlens,
                  int n_seq, int T, int H, int dk, int dv, int dtype, void* workspace,
                  size_t ws_bytes, gla_stream_t stream) {
  return chunk_fwd(q, k, v, log_lambda, h0, scale, nullptr, o, hT, cu_seqlens, n_seq, T, H, dk, dv,
                   dtype, workspace, ws_bytes, stream);
}

int gla_chunk_fwd_aug(const void* q, const void* k, const void* v, const float* log_lambda,
                      const float* h0, float scale, const float* aug, void* o, float* hT,
                      const int32_t* cu_seqlens, int n_seq, int T, int H, int dk, int dv, int dtype,
                      void* workspace, size_t ws_bytes, gla_stream_t stream) {
  if (!aug) return GLA_ERR_NULL;
  return chunk_fwd(q, k, v, log_lambda, h0, scale, aug, o, hT, cu_seqlens, n_seq, T, H, dk, dv,
                   dtype, workspace, ws_bytes, stream);
}

int gla_chunk_bwd(const void* q, const void* k, const void* v, const float* log_lambda,
                  const float* h0, float scale, const void* dO, const float* dhT, void* dq,
                  void* dk, void* dv, float* dh0, const int32_t* cu_seqlens, int n_seq, int T,
                  int H, int dk_size, int dv_size, int dtype, void* workspace, size_t ws_bytes,
                  gla_stream_t stream) {
  long long tokens = 0;
  int rc = check_chunk_call(n_seq, T, H, dk_size, dv_size, dtype, cu_seqlens, workspace, ws_bytes,
                            &tokens);
  if (rc) return rc;
  if (n_seq == 0) return GLA_OK;
  const size_t ws_need = gla_bwd_workspace_bytes(n_seq, T, H, cu_seqlens != nullptr, dtype);
  if (ws_need > 0 && (!workspace || ws_bytes < ws_need)) return GLA_ERR_WORKSPACE;
  if (workspace && !aligned16(workspace)) return GLA_ERR_ALIGN;
  if (!log_lambda) return GLA_ERR_NULL;
  if (tokens > 0 && (!q || !k || !v || !dO || !dq || !dk || !dv)) return GLA_ERR_NULL;
  for (const void* p : {(const void*)q, (const void*)k, (const void*)v, (const void*)dO,
                        (const void*)dq, (const void*)dk, (const void*)dv, (const void*)h0,
                        (const void*)dhT, (const void*)dh0, (const void*)log_lambda})
    if (p && !aligned16(p)) return GLA_ERR_ALIGN;
  int dev;
  unsigned* err;
  unsigned long long wait_ns;
  rc = device_state(&dev, &err, &wait_ns);
  if (rc) return rc;

  gla::ChunkArgs a = {};
  a.q = q;
  a.k = k;
  a.v = v;
  a.dO = dO;
  a.log_lambda = log_lambda;
  a.h0 = h0;
  a.dhT = dhT;
  a.o = dq;
  a.dk = dk;
  a.dv = dv;
  a.hT = dh0;
  a.cu_seqlens = cu_seqlens;
  a.scale = scale;
  a.n_seq = n_seq;
  a.T = T;
  a.H = H;
  a.err = err;
  a.wait_ns = wait_ns;
  cudaStream_t s = (cudaStream_t)stream;
  char* ws = (char*)workspace;
  if (cu_seqlens) {
    int32_t* order = (int32_t*)(ws + 256);
    lpt_order_kernel<<<(n_seq + 255) / 256, 256, 0, s>>>(cu_seqlens, n_seq, order);
    if (cudaGetLastError() != cudaSuccess) return GLA_ERR_LAUNCH;
    a.order = order;
  }
  if (dtype == GLA_F32) return to_status(gla::launch_simt_bwd(1, a, s));
  const size_t head = cu_seqlens ? gla_workspace_bytes(n_seq, H) : 256;
  const size_t acc = ((gla::tc_bwd_acc_bytes(tokens, H) + 255) / 256) * 256;
  float* acc_q = (float*)(ws + head);
  float* acc_k = (float*)(ws + head + acc);
  return to_status(gla::launch_tc_bwd(a, acc_q, acc_k, s));
}

static int decode_step(const void* q, const void* k, const void* v, const float* log_lambda,
                       float scale, const float* aug, void* state, int state_bf16, const int32_t* slot,
                       int pool_rows, void* o, int N, int H, int dk, int dv, int dtype,
                       gla_stream_t stream, const gla::DecodeNormGate* ngp = nullptr) {
  if (dtype != GLA_BF16 && dtype != GLA_F32) return GLA_ERR_DTYPE;
  if (dk != GLA_DK || dv != GLA_DV) return GLA_ERR_UNSUPPORTED;
  if (N < 0 || H < 1 || pool_rows < 0) return GLA_ERR_SHAPE;
  if (!slot && pool_rows < N) return GLA_ERR_SHAPE;
  if (N == 0) return GLA_OK;
  if (!q || !k || !v || !log_lambda || !state || !o) return GLA_ERR_NULL;
  for (const void* p : {(const void*)q, (const void*)k, (const void*)v, (const void*)o,
                        (const void*)state, (const void*)log_lambda})
    if (!aligned16(p)) return GLA_ERR_ALIGN;
  if (aug && !aligned16(aug)) return GLA_ERR_ALIGN;
  if (slot && ((uintptr_t)slot & 3u)) return GLA_ERR_ALIGN;
  int dev;
  unsigned* err;
  unsigned long long wait_ns;
  int rc = device_state(&dev, &err, &wait_ns);
  if (rc) return rc;
  return to_status(gla::launch_decode_step(dtype == GLA_F32, state_bf16, q, k, v, log_lambda, scale, state,
                                           slot, pool_rows, o, N, H, aug, err, (cudaStream_t)stream, ngp));
}

int gla_decode_step(const void* q, const void* k, const void* v, const float* log_lambda,
                    float scale, float* state, const int32_t* slot, int pool_rows, void* o, int N,
                    int H, int dk, int dv, int dtype, gla_stream_t stream) {
  return decode_step(q, k, v, log_lambda, scale, nullptr, state, 0, slot, pool_rows, o, N, H, dk, dv,
                     dtype, stream);
}

int gla_decode_step_aug(const void* q, const void* k, const void* v, const float* log_lambda,
                        float scale, const float* aug, float* state, const int32_t* slot,
                        int pool_rows, void* o, int N, int H, int dk, int dv, int dtype,
                        gla_stream_t stream) {
  if (!aug) return GLA_ERR_NULL;
  return decode_step(q, k, v, log_lambda, scale, aug, state, 0, slot, pool_rows, o, N, H, dk, dv, dtype,
                     stream);
}

int gla_decode_step_bf16_state(const void* q, const void* k, const void* v, const float* log_lambda,
                               float scale, const float* aug, void* state, const int32_t* slot,
                               int pool_rows, void* o, int N, int H, int dk, int dv, int dtype,
                               gla_stream_t stream) {
  return decode_step(q, k, v, log_lambda, scale, aug, state, 1, slot, pool_rows, o, N, H, dk, dv, dtype,
                     stream);
}

int gla_decode_step_norm_gate(const void* q, const void* k, const void* v, const float* log_lambda,
                              float scale, const float* aug, float* state, const int32_t* slot,
                              int pool_rows, const void* g, const float* weight, const int32_t* tier,
                              int n_tiers, float eps, void* y, int N, int H, int dk, int dv, int dtype,
                              gla_stream_t stream) {
  if (dtype != GLA_BF16 && dtype != GLA_F32) return GLA_ERR_DTYPE;
  if (dk != GLA_DK || dv != GLA_DV) return GLA_ERR_UNSUPPORTED;
  if (n_tiers < 1 || !(eps >= 0.f)) return GLA_ERR_SHAPE;
  if (N > 0) {
    if (!g || !weight || !tier) return GLA_ERR_NULL;
    if (!aligned16(g) || !aligned16(weight)) return GLA_ERR_ALIGN;
    if ((uintptr_t)tier & 3u) return GLA_ERR_ALIGN;
  }
  const gla::DecodeNormGate ng = {g, weight, tier, n_tiers, eps};
  return decode_step(q, k, v, log_lambda, scale, aug, state, 0, slot, pool_rows, y, N, H, dk, dv, dtype,
                     stream, &ng);
}

int gla_decode_step_mxfp8_state(const void* q, const void* k, const void* v, const float* log_lambda,
                                float scale, const float* aug, uint8_t* state_codes, uint8_t* state_scales,
                                const int32_t* slot, int pool_rows, void* o, int N, int H, int dk, int dv,
                                int dtype, gla_stream_t stream) {
  if (dtype != GLA_BF16 && dtype != GLA_F32) return GLA_ERR_DTYPE;
  if (dk != GLA_DK || dv != GLA_DV) return GLA_ERR_UNSUPPORTED;
  if (N < 0 || H < 1 || pool_rows < 0) return GLA_ERR_SHAPE;
  if (!slot && pool_rows < N) return GLA_ERR_SHAPE;
  if (N == 0) return GLA_OK;
  if (!q || !k || !v || !log_lambda || !state_codes || !state_scales || !o) return GLA_ERR_NULL;
  for (const void* p : {(const void*)q, (const void*)k, (const void*)v, (const void*)o,
                        (const void*)state_codes, (const void*)state_scales, (const void*)log_lambda})
    if (!aligned16(p)) return GLA_ERR_ALIGN;
  if (aug && !aligned16(aug)) return GLA_ERR_ALIGN;
  if (slot && ((uintptr_t)slot & 3u)) return GLA_ERR_ALIGN;
  int dev;
  unsigned* err;
  unsigned long long wait_ns;
  int rc = device_state(&dev, &err, &wait_ns);
  if (rc) return rc;
  return to_status(gla::launch_decode_step_mxfp8(dtype == GLA_F32, q, k, v, log_lambda, scale, state_codes,
                                                 state_scales, slot, pool_rows, o, N, H, aug, err, wait_ns,
                                                 (cudaStream_t)stream));
}

int gla_state_to_mxfp8(const float* x, uint8_t* codes, uint8_t* scales, long long rows, gla_stream_t stream) {
  if (rows < 0 || rows > (1ll << 40)) return GLA_ERR_SHAPE;
  if (rows == 0) return GLA_OK;
  if (!x || !codes || !scales) return GLA_ERR_NULL;
  if (!aligned16(x) || !aligned16(codes) || !aligned16(scales)) return GLA_ERR_ALIGN;
  int dev;
  unsigned* err;
  unsigned long long wait_ns;
  int rc = device_state(&dev, &err, &wait_ns);
  if (rc) return rc;
  return to_status(gla::launch_mxfp8_quantise(x, codes, scales, rows, (cudaStream_t)stream));
}

int gla_state_from_mxfp8(const uint8_t* codes, const uint8_t* scales, float* x, long long rows,
                         gla_stream_t stream) {
  if (rows < 0 || rows > (1ll << 40)) return GLA_ERR_SHAPE;
  if (rows == 0) return GLA_OK;
  if (!x || !codes || !scales) return GLA_ERR_NULL;
  if (!aligned16(x) || !aligned16(codes) || !aligned16(scales)) return GLA_ERR_ALIGN;
  int dev;
  unsigned* err;
  unsigned long long wait_ns;
  int rc = device_state(&dev, &err, &wait_ns);
  if (rc) return rc;
  return to_status(gla::launch_mxfp8_dequantise(codes, scales, x, rows, (cudaStream_t)stream));
}

int gla_head_norm_gate(const void* o, const void* g, const float* weight, const int32_t* tier,
                       int n_tiers, float eps, void* y, long long rows, int H, int dv, int dtype,
                       gla_stream_t stream) {
  if (dtype != GLA_BF16 && dtype != GLA_F32) return GLA_ERR_DTYPE;
  if (dv != GLA_DV) return GLA_ERR_UNSUPPORTED;
  if (rows < 0 || H < 1 || n_tiers < 1 || !(eps >= 0.f) || rows > (1ll << 40)) return GLA_ERR_SHAPE;
  if (H > 4096) return GLA_ERR_UNSUPPORTED;  // with rows <= 2^40, element offsets stay below 2^60
  if (rows == 0) return GLA_OK;
  if (!o || !g || !weight || !tier || !y) return GLA_ERR_NULL;
  for (const void* p : {o, g, (const void*)weight, (const void*)y})
    if (!aligned16(p)) return GLA_ERR_ALIGN;
  if ((uintptr_t)tier & 3u) return GLA_ERR_ALIGN;
  int dev;
  unsigned* err;
  unsigned long long wait_ns;
  int rc = device_state(&dev, &err, &wait_ns);
  if (rc) return rc;
  return to_status(gla::launch_head_norm_gate(dtype == GLA_F32, o, g, weight, tier, n_tiers, eps, y, rows,
                                              H, err, (cudaStream_t)stream));
}

int gla_get_device_error(gla_stream_t stream) {
  int dev;
  unsigned* err;
  unsigned long long wait_ns;
  int rc = device_state(&dev, &err, &wait_ns);
  if (rc) return rc;
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return GLA_ERR_LAUNCH;
  unsigned word = 0;
  if (cudaMemcpyFromSymbol(&word, g_error_word, sizeof(word)) != cudaSuccess) return GLA_ERR_LAUNCH;
  if (word) {
    const unsigned zero = 0;
    if (cudaMemcpyToSymbol(g_error_word, &zero, sizeof(zero)) != cudaSuccess) return GLA_ERR_LAUNCH;
    if (gla::tc_clear_handover((cudaStream_t)stream) != cudaSuccess ||
        cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess)
      return GLA_ERR_LAUNCH;
  }
  return -(int)word;
}

int gla_set_wait_limit_ns(unsigned long long ns) {
  int dev;
  unsigned* err;
  unsigned long long wait_ns;
  int rc = device_state(&dev, &err, &wait_ns);
  if (rc) return rc;
  std::lock_guard<std::mutex> lock(g_mu);
  g_wait_ns[dev] = ns ? ns : 1ull;
  return GLA_OK;
}

int gla_debug_bounds(void) { return gla::kDebugBounds ? 1 : 0; }

const char* gla_status_string(int status) {
  switch (status) {
    case GLA_OK: return "GLA_OK";
    case GLA_ERR_NULL: return "GLA_ERR_NULL: a required pointer is NULL";
    case GLA_ERR_SHAPE: return "GLA_ERR_SHAPE: bad size, cu_seqlens or pool slot";
    case GLA_ERR_DTYPE: return "GLA_ERR_DTYPE: unknown dtype";
    case GLA_ERR_ALIGN: return "GLA_ERR_ALIGN: pointer not 16-byte aligned";
    case GLA_ERR_UNSUPPORTED: return "GLA_ERR_UNSUPPORTED: only d_k=96, d_v=192 on sm_103";
    case GLA_ERR_WORKSPACE: return "GLA_ERR_WORKSPACE: workspace missing or too small";
    case GLA_ERR_LAUNCH: return "GLA_ERR_LAUNCH: the CUDA runtime refused a launch";
    case GLA_ERR_TIMEOUT: return "GLA_ERR_TIMEOUT: a bounded device wait gave up";
    case GLA_ERR_BOUNDS: return "GLA_ERR_BOUNDS: a device index check of the debug-bounds build failed";
    default: return "unknown gla_status";
  }
}

}  // extern "C"
