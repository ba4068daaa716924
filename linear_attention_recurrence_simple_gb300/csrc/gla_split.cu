// Sequence-split forward for long sequences (no counterpart in the paper).
//
// "Beyond the KV cache", section "Challenge 1": within a chunk the work is parallel and only the
// state's advance from chunk to chunk is sequential.  A sequence's chunks therefore split into
// segments whose work runs in parallel once each segment knows the state it starts from:
//   1. every segment runs the chunked forward from a zero state, final states only (bf16: the
//      tensor-core scan's states-only mode, which loads k and v and accumulates the weighted
//      products in tensor memory); its final state is U_i = sum_j lambda^(L_i-1-j) k_j v_j^T
//      over its L_i tokens;
//   2. a short scan per (sequence, head) chains them: S_in[first] = h0,
//      S_in[i+1] = lambda^(L_i) S_in[i] + U_i, and hT = lambda^(L_last) S_in[last] + U_last;
//   3. every segment runs the chunked forward again from S_in[i], writing the outputs.
// A sequence whose chunks sit on one CTA (one unit per (sequence, head, d_v tile)) then spreads
// over as many CTAs as it has segments, at the price of a second pass over k and v (in fp32 mode
// step 1 is the full forward, whose outputs step 3 overwrites).  The host plans the segments from
// a host copy of the sequence offsets (seg_chunks = 0: the length from a cost model of the packed
// forward, or no split at all); the device arrays it needs go into the caller's workspace.
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
constexpr int STATE4 = DK * DV / 4;            // float4 entries of one state
constexpr int SCAN_CTAS_PER_STATE = STATE4 / SPLIT_THREADS;  // 18
static_assert(STATE4 % SPLIT_THREADS == 0, "a state is a whole number of CTAs");
constexpr int SCAN_AHEAD = 4;                  // segments whose loads are issued together

// One thread per 4 consecutive entries of one (sequence, head)'s 96 x 192 state: walks the
// sequence's segments in order (step 2 above), issuing the loads of SCAN_AHEAD segments before
// their links of the chain.  seg_first[n] .. seg_first[n + 1] - 1 are sequence n's segments.
__global__ void __launch_bounds__(SPLIT_THREADS)
split_scan_kernel(const float4* __restrict__ U, const float4* __restrict__ h0, const int32_t* __restrict__ seg_cu,
                  const int32_t* __restrict__ seg_first, const float* __restrict__ log_lambda,
                  float4* __restrict__ S_in, float4* __restrict__ hT, int H, [[maybe_unused]] int n_seq,
                  [[maybe_unused]] int M, [[maybe_unused]] unsigned* err) {
  const long long nh = blockIdx.x / SCAN_CTAS_PER_STATE;
  const int e = (int)(blockIdx.x % SCAN_CTAS_PER_STATE) * SPLIT_THREADS + (int)threadIdx.x;
  const int n = (int)(nh / H), h = (int)(nh % H);
  if (!GLA_IN_BOUNDS(n < n_seq && e < STATE4, err)) return;
  const float ll = log_lambda[h];
  const int i0 = seg_first[n], i1 = seg_first[n + 1];
  if (!GLA_IN_BOUNDS(0 <= i0 && i0 <= i1 && i1 <= M, err)) return;  // sequence n's segments
  float4 s = h0 ? h0[nh * STATE4 + e] : make_float4(0.f, 0.f, 0.f, 0.f);
  for (int i = i0; i < i1; i += SCAN_AHEAD) {
    float4 u[SCAN_AHEAD];
    float d[SCAN_AHEAD];
#pragma unroll
    for (int j = 0; j < SCAN_AHEAD; ++j) {
      if (i + j < i1) {
        u[j] = U[((long long)(i + j) * H + h) * STATE4 + e];
        d[j] = expf((float)(seg_cu[i + j + 1] - seg_cu[i + j]) * ll);
      }
    }
#pragma unroll
    for (int j = 0; j < SCAN_AHEAD; ++j) {
      if (i + j < i1) {
        S_in[((long long)(i + j) * H + h) * STATE4 + e] = s;
        s = make_float4(fmaf(d[j], s.x, u[j].x), fmaf(d[j], s.y, u[j].y), fmaf(d[j], s.z, u[j].z),
                        fmaf(d[j], s.w, u[j].w));
      }
    }
  }
  if (hT) hT[nh * STATE4 + e] = s;
}

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

struct SplitPlan {
  std::vector<int32_t> seg_cu, seg_first;
  int M = 0;
};

// Cost model of the automatic segment length (seg_chunks = 0).  The packed forward runs one CTA
// per unit, (segment, head, d_v tile), one CTA per SM, longest units first; a unit takes its
// chunk count plus a start-up cost, in chunk times.  The split runs two such passes (the
// states-only pass at about half the full one), the plain forward one.  Costs are
// kept in quarter chunk times (integers).
constexpr int PLAN_SMS = 152;             // SMs of a GB300
constexpr long long UNIT_OVERHEAD = 12;   // 3 chunk times per unit: pipeline fill and drain
constexpr long long SPLIT_PASSES_X4 = 6;  // both passes of the split: 6/4 of a full pass

using UnitGroups = std::vector<std::pair<int, long long>>;  // (chunks, units), any order

// Estimated makespan of units placed longest-first on PLAN_SMS SMs, each on the least loaded.
// A full round of PLAN_SMS equal units puts one on every SM, and the r < PLAN_SMS left over go
// to the r least loaded SMs (exact while the loads differ by less than one unit): the loads stay
// sorted by merging the r raised entries back into the rest.
long long lpt_makespan(UnitGroups g) {
  std::sort(g.begin(), g.end(), [](const auto& a, const auto& b) { return a.first > b.first; });
  long long load[PLAN_SMS] = {}, tmp[PLAN_SMS];
  long long base = 0;
  for (size_t i = 0; i < g.size();) {
    long long count = 0;
    const int len = g[i].first;
    for (; i < g.size() && g[i].first == len; ++i) count += g[i].second;
    const long long cost = 4ll * len + UNIT_OVERHEAD;
    base += count / PLAN_SMS * cost;
    const int r = (int)(count % PLAN_SMS);
    if (r == 0) continue;
    for (int i = 0; i < r; ++i) load[i] += cost;
    std::merge(load, load + r, load + r, load + PLAN_SMS, tmp);
    std::copy(tmp, tmp + PLAN_SMS, load);
  }
  return base + load[PLAN_SMS - 1];
}

// Chunks per segment for seg_chunks = 0: the plain forward's estimate against the split's for
// segment lengths that cut the longest sequence into 2 .. 64 equal parts; 0 when no split is
// estimated faster (every sequence then stays one segment).
int choose_seg_chunks(const int32_t* cu, int n_seq, int H) {
  const long long units = 3ll * H;  // (head, d_v tile) units per segment
  std::vector<int> c(n_seq);
  int c_max = 0;
  long long chunks = 0, segs = 0;
  UnitGroups plain;
  for (int n = 0; n < n_seq; ++n) {
    c[n] = (int)(((long long)cu[n + 1] - cu[n] + GLA_CHUNK - 1) / GLA_CHUNK);
    c_max = std::max(c_max, c[n]);
    if (c[n] > 0) {
      plain.push_back({c[n], units});
      chunks += c[n];
      ++segs;
    }
  }
  if (c_max < 2) return 0;
  long long best = lpt_makespan(plain);
  // A pass over segs' segments takes at least an even spread of all their costs over the SMs.
  auto bound = [&](long long n_segs) {
    return SPLIT_PASSES_X4 * ((units * (4 * chunks + n_segs * UNIT_OVERHEAD)) / PLAN_SMS) / 4;
  };
  if (bound(segs) >= best) return 0;
  int best_len = 0, prev = 0;
  UnitGroups g;
  for (int parts = 2; parts <= std::min(c_max, 64); ++parts) {
    const int len = (c_max + parts - 1) / parts;
    if (len == prev) continue;
    prev = len;
    long long n_segs = 0;
    g.clear();
    for (int n = 0; n < n_seq; ++n) {
      if (c[n] >= len) g.push_back({len, units * (c[n] / len)});
      if (c[n] % len) g.push_back({c[n] % len, units});
      n_segs += (c[n] + len - 1) / len;
    }
    if (bound(n_segs) >= best || SPLIT_PASSES_X4 * (4ll * len + UNIT_OVERHEAD) / 4 >= best) continue;
    const long long t = SPLIT_PASSES_X4 * lpt_makespan(g) / 4;
    if (t < best) {
      best = t;
      best_len = len;
    }
  }
  return best_len;
}

// Segments of at most seg_chunks chunks (chunk-aligned within each sequence; 0: chosen by
// choose_seg_chunks); an empty sequence keeps one empty segment, which passes h0 through.
int plan_split(const int32_t* cu, int n_seq, int H, int seg_chunks, SplitPlan* p) {
  for (int n = 0; n < n_seq; ++n)
    if (cu[n + 1] < cu[n]) return GLA_ERR_SHAPE;
  if (seg_chunks == 0) {
    seg_chunks = choose_seg_chunks(cu, n_seq, H);
    if (seg_chunks == 0) seg_chunks = 1 << 24;  // one segment per sequence
  }
  p->seg_cu.assign(1, cu[0]);
  p->seg_first.assign(1, 0);
  for (int n = 0; n < n_seq; ++n) {
    const long long a = cu[n], b = cu[n + 1];
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

// With one segment per sequence (M == n_seq) the call is the plain forward: no segment states.
SplitLayout split_layout(int M, int n_seq, int H) {
  SplitLayout l;
  const size_t state = (size_t)M * H * DK * DV * sizeof(float);
  l.seg_cu = 0;
  l.seg_first = l.seg_cu + align256((size_t)(M + 1) * sizeof(int32_t));
  l.lpt = l.seg_first + align256((size_t)(n_seq + 1) * sizeof(int32_t));
  l.U = l.lpt + align256(gla_workspace_bytes(M, H));
  l.S_in = l.U + align256(state);
  l.total = M == n_seq ? l.U : l.S_in + align256(state);
  return l;
}

}  // namespace
}  // namespace gla

extern "C" {

size_t gla_split_workspace_bytes(const int32_t* cu_seqlens_host, int n_seq, int H, int seg_chunks) {
  if (!cu_seqlens_host || n_seq < 0 || H < 1 || seg_chunks < 0) return 0;
  gla::SplitPlan plan;
  if (gla::plan_split(cu_seqlens_host, n_seq, H, seg_chunks, &plan) != GLA_OK) return 0;
  return gla::split_layout(plan.M, n_seq, H).total;
}

int gla_split_choose_seg_chunks(const int32_t* cu_seqlens_host, int n_seq, int H) {
  if (!cu_seqlens_host) return GLA_ERR_NULL;
  if (n_seq < 0 || H < 1) return GLA_ERR_SHAPE;
  for (int n = 0; n < n_seq; ++n)
    if (cu_seqlens_host[n + 1] < cu_seqlens_host[n]) return GLA_ERR_SHAPE;
  return gla::choose_seg_chunks(cu_seqlens_host, n_seq, H);
}

int gla_chunk_fwd_split(const void* q, const void* k, const void* v, const float* log_lambda,
                        const float* h0, float scale, const float* aug, void* o, float* hT,
                        const int32_t* cu_seqlens_host, int n_seq, int T, int H, int dk, int dv,
                        int dtype, int seg_chunks, void* workspace, size_t ws_bytes,
                        gla_stream_t stream) {
  if (dtype != GLA_BF16 && dtype != GLA_F32) return GLA_ERR_DTYPE;
  if (dk != GLA_DK || dv != GLA_DV) return GLA_ERR_UNSUPPORTED;
  if (n_seq < 0 || T < 0 || H < 1 || seg_chunks < 0) return GLA_ERR_SHAPE;
  if (n_seq == 0) return GLA_OK;
  if (!cu_seqlens_host) return GLA_ERR_NULL;
  if (cu_seqlens_host[0] != 0 || cu_seqlens_host[n_seq] != T) return GLA_ERR_SHAPE;
  gla::SplitPlan plan;
  int rc = gla::plan_split(cu_seqlens_host, n_seq, H, seg_chunks, &plan);
  if (rc) return rc;
  if ((long long)plan.M * H * GLA_DK >= (1ll << 31)) return GLA_ERR_SHAPE;
  const gla::SplitLayout l = gla::split_layout(plan.M, n_seq, H);
  if (!workspace || ws_bytes < l.total) return GLA_ERR_WORKSPACE;
  if (((uintptr_t)workspace & 255u) != 0) return GLA_ERR_ALIGN;
  if (!log_lambda || (T > 0 && (!q || !k || !v || !o))) return GLA_ERR_NULL;
  for (const void* p : {q, k, v, (const void*)o, (const void*)log_lambda, (const void*)h0, (const void*)hT,
                        (const void*)aug})
    if (((uintptr_t)p & 15u) != 0) return GLA_ERR_ALIGN;
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
  if (plan.M == n_seq) {  // one segment per sequence: the plain forward
    if (aug)
      return gla_chunk_fwd_aug(q, k, v, log_lambda, h0, scale, aug, o, hT, seg_cu, n_seq, T, H, dk, dv,
                               dtype, ws + l.lpt, l.U - l.lpt, stream);
    return gla_chunk_fwd(q, k, v, log_lambda, h0, scale, o, hT, seg_cu, n_seq, T, H, dk, dv, dtype,
                         ws + l.lpt, l.U - l.lpt, stream);
  }
  // 1. segment states from zero
  bool states_done = false;
  if (dtype == GLA_BF16) {
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
  unsigned* scan_err = nullptr;
  {
    unsigned long long wait_ns;
    if ((rc = gla::current_device_state(&scan_err, &wait_ns)) != GLA_OK) return rc;
  }
  gla::split_scan_kernel<<<(unsigned)((long long)n_seq * H * gla::SCAN_CTAS_PER_STATE), gla::SPLIT_THREADS, 0,
                           s>>>((const float4*)U, (const float4*)h0, seg_cu, seg_first, log_lambda,
                                (float4*)S_in, (float4*)hT, H, n_seq, plan.M, scan_err);
  if (cudaGetLastError() != cudaSuccess) return GLA_ERR_LAUNCH;
  // 3. the outputs, each segment from its starting state
  if (aug)
    return gla_chunk_fwd_aug(q, k, v, log_lambda, S_in, scale, aug, o, nullptr, seg_cu, plan.M, T, H, dk,
                             dv, dtype, ws + l.lpt, l.U - l.lpt, stream);
  return gla_chunk_fwd(q, k, v, log_lambda, S_in, scale, o, nullptr, seg_cu, plan.M, T, H, dk, dv, dtype,
                       ws + l.lpt, l.U - l.lpt, stream);
}

}  // extern "C"
