// Sequence-split forward for long sequences (no counterpart in the paper).
//
// "Beyond the KV cache", section "Challenge 1": within a chunk the work is parallel and only the
// state's advance from chunk to chunk is sequential.  A sequence's chunks therefore split into
// segments whose work runs in parallel once each segment knows the state it starts from:
//   1. every segment runs the chunked forward from a zero state, final states only (bf16: the
//      tensor-core scan's states-only mode, which loads k and v and runs the state update
//      alone); its final state is U_i = sum_j lambda^(L_i-1-j) k_j v_j^T over its L_i tokens;
//   2. a short scan per (sequence, head) chains them: S_in[first] = h0,
//      S_in[i+1] = lambda^(L_i) S_in[i] + U_i, and hT = lambda^(L_last) S_in[last] + U_last;
//   3. every segment runs the chunked forward again from S_in[i], writing the outputs.
// A sequence whose chunks sit on one CTA (one unit per (sequence, head, d_v tile)) then spreads
// over as many CTAs as it has segments, at the price of a second pass over k and v (in fp32 mode
// step 1 is the full forward, whose outputs step 3 overwrites).  The host plans the segments from
// a host copy of the sequence offsets; the device arrays it needs go into the caller's workspace.
#include <algorithm>
#include <vector>

#include "gla.h"
#include "gla_common.cuh"

namespace gla {
int current_device_state(unsigned** err, unsigned long long* wait_ns);
cudaError_t launch_lpt_order(const int32_t* cu_seqlens, int n_seq, int32_t* order, cudaStream_t stream);
cudaError_t launch_tc_fwd_states(const ChunkArgs& a, cudaStream_t stream);

namespace {

constexpr int SPLIT_THREADS = 256;

// One CTA per (sequence, head) and quarter of the 96 x 192 state: walks the sequence's segments
// in order (step 2 above).  seg_first[n] .. seg_first[n + 1] - 1 are sequence n's segments.
__global__ void __launch_bounds__(SPLIT_THREADS)
split_scan_kernel(const float* __restrict__ U, const float* __restrict__ h0, const int32_t* __restrict__ seg_cu,
                  const int32_t* __restrict__ seg_first, const float* __restrict__ log_lambda, float* __restrict__ S_in,
                  float* __restrict__ hT, int H) {
  constexpr int STATE = DK * DV, PART = STATE / 4;
  const int nh = blockIdx.x / 4, part = blockIdx.x % 4;
  const int n = nh / H, h = nh % H;
  const float ll = log_lambda[h];
  const int i0 = seg_first[n], i1 = seg_first[n + 1];
  for (int e = part * PART + (int)threadIdx.x; e < (part + 1) * PART; e += SPLIT_THREADS) {
    float s = h0 ? h0[(long long)nh * STATE + e] : 0.f;
    for (int i = i0; i < i1; ++i) {
      const long long at = ((long long)i * H + h) * STATE + e;
      S_in[at] = s;
      s = fmaf(expf((float)(seg_cu[i + 1] - seg_cu[i]) * ll), s, U[at]);
    }
    if (hT) hT[(long long)nh * STATE + e] = s;
  }
}

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

struct SplitPlan {
  std::vector<int32_t> seg_cu, seg_first;
  int M = 0;
};

// Segments of at most seg_chunks chunks (chunk-aligned within each sequence); an empty sequence
// keeps one empty segment, which passes h0 through.
int plan_split(const int32_t* cu, int n_seq, int seg_chunks, SplitPlan* p) {
  p->seg_cu.assign(1, cu[0]);
  p->seg_first.assign(1, 0);
  for (int n = 0; n < n_seq; ++n) {
    const long long a = cu[n], b = cu[n + 1];
    if (b < a) return GLA_ERR_SHAPE;
    const long long step = (long long)seg_chunks * GLA_CHUNK;
    if (b == a) {
      p->seg_cu.push_back((int32_t)b);
    } else {
      for (long long t = a + step; ; t += step) {
        p->seg_cu.push_back((int32_t)std::min(t, b));
        if (t >= b) break;
      }
    }
    p->seg_first.push_back((int32_t)p->seg_cu.size() - 1);
  }
  p->M = (int)p->seg_cu.size() - 1;
  return GLA_OK;
}

struct SplitLayout {
  size_t seg_cu, seg_first, lpt, U, S_in, total;
};

SplitLayout split_layout(int M, int n_seq, int H) {
  SplitLayout l;
  const size_t state = (size_t)M * H * DK * DV * sizeof(float);
  l.seg_cu = 0;
  l.seg_first = l.seg_cu + align256((size_t)(M + 1) * sizeof(int32_t));
  l.lpt = l.seg_first + align256((size_t)(n_seq + 1) * sizeof(int32_t));
  l.U = l.lpt + align256(gla_workspace_bytes(M, H));
  l.S_in = l.U + align256(state);
  l.total = l.S_in + align256(state);
  return l;
}

}  // namespace
}  // namespace gla

extern "C" {

size_t gla_split_workspace_bytes(const int32_t* cu_seqlens_host, int n_seq, int H, int seg_chunks) {
  if (!cu_seqlens_host || n_seq < 0 || H < 1 || seg_chunks < 1) return 0;
  gla::SplitPlan plan;
  if (gla::plan_split(cu_seqlens_host, n_seq, seg_chunks, &plan) != GLA_OK) return 0;
  return gla::split_layout(plan.M, n_seq, H).total;
}

int gla_chunk_fwd_split(const void* q, const void* k, const void* v, const float* log_lambda,
                        const float* h0, float scale, const float* aug, void* o, float* hT,
                        const int32_t* cu_seqlens_host, int n_seq, int T, int H, int dk, int dv,
                        int dtype, int seg_chunks, void* workspace, size_t ws_bytes,
                        gla_stream_t stream) {
  if (dtype != GLA_BF16 && dtype != GLA_F32) return GLA_ERR_DTYPE;
  if (dk != GLA_DK || dv != GLA_DV) return GLA_ERR_UNSUPPORTED;
  if (n_seq < 0 || T < 0 || H < 1 || seg_chunks < 1) return GLA_ERR_SHAPE;
  if (n_seq == 0) return GLA_OK;
  if (!cu_seqlens_host) return GLA_ERR_NULL;
  if (cu_seqlens_host[0] != 0 || cu_seqlens_host[n_seq] != T) return GLA_ERR_SHAPE;
  gla::SplitPlan plan;
  int rc = gla::plan_split(cu_seqlens_host, n_seq, seg_chunks, &plan);
  if (rc) return rc;
  if ((long long)plan.M * H * GLA_DK >= (1ll << 31)) return GLA_ERR_SHAPE;
  const gla::SplitLayout l = gla::split_layout(plan.M, n_seq, H);
  if (!workspace || ws_bytes < l.total) return GLA_ERR_WORKSPACE;
  if (((uintptr_t)workspace & 255u) != 0) return GLA_ERR_ALIGN;
  if (!log_lambda || (T > 0 && (!q || !k || !v || !o))) return GLA_ERR_NULL;
  char* ws = (char*)workspace;
  int32_t* seg_cu = (int32_t*)(ws + l.seg_cu);
  int32_t* seg_first = (int32_t*)(ws + l.seg_first);
  float* U = (float*)(ws + l.U);
  float* S_in = (float*)(ws + l.S_in);
  cudaStream_t s = (cudaStream_t)stream;
  // The plan goes to the device (pageable copies: staged before the calls return).
  if (cudaMemcpyAsync(seg_cu, plan.seg_cu.data(), plan.seg_cu.size() * sizeof(int32_t),
                      cudaMemcpyHostToDevice, s) != cudaSuccess ||
      cudaMemcpyAsync(seg_first, plan.seg_first.data(), plan.seg_first.size() * sizeof(int32_t),
                      cudaMemcpyHostToDevice, s) != cudaSuccess)
    return GLA_ERR_LAUNCH;
  // 1. segment states from zero
  bool states_done = false;
  if (dtype == GLA_BF16) {
    for (const void* p : {q, k, v, (const void*)o, (const void*)log_lambda})
      if (((uintptr_t)p & 15u) != 0) return GLA_ERR_ALIGN;
    unsigned* err;
    unsigned long long wait_ns;
    if ((rc = gla::current_device_state(&err, &wait_ns)) != GLA_OK) return rc;
    int32_t* order = (int32_t*)(ws + l.lpt + 256);
    if (gla::launch_lpt_order(seg_cu, plan.M, order, s) != cudaSuccess) return GLA_ERR_LAUNCH;
    gla::ChunkArgs a = {};
    a.q = q;
    a.k = k;
    a.v = v;
    a.log_lambda = log_lambda;
    a.hT = U;
    a.cu_seqlens = seg_cu;
    a.order = order;
    a.scale = scale;
    a.n_seq = plan.M;
    a.T = T;
    a.H = H;
    a.err = err;
    a.wait_ns = wait_ns;
    states_done = gla::launch_tc_fwd_states(a, s) == cudaSuccess;
    if (!states_done) (void)cudaGetLastError();  // refused: the full forward below instead
  }
  if (!states_done) {  // (the outputs written here are overwritten by step 3)
    rc = gla_chunk_fwd(q, k, v, log_lambda, nullptr, scale, o, U, seg_cu, plan.M, T, H, dk, dv, dtype,
                       ws + l.lpt, l.U - l.lpt, stream);
    if (rc) return rc;
  }
  // 2. chain the segment states
  gla::split_scan_kernel<<<(unsigned)((long long)n_seq * H * 4), gla::SPLIT_THREADS, 0, s>>>(
      U, h0, seg_cu, seg_first, log_lambda, S_in, hT, H);
  if (cudaGetLastError() != cudaSuccess) return GLA_ERR_LAUNCH;
  // 3. the outputs, each segment from its starting state
  if (aug)
    return gla_chunk_fwd_aug(q, k, v, log_lambda, S_in, scale, aug, o, nullptr, seg_cu, plan.M, T, H, dk,
                             dv, dtype, ws + l.lpt, l.U - l.lpt, stream);
  return gla_chunk_fwd(q, k, v, log_lambda, S_in, scale, o, nullptr, seg_cu, plan.M, T, H, dk, dv, dtype,
                       ws + l.lpt, l.U - l.lpt, stream);
}

}  // extern "C"
