// The chunked forward with host-memory inputs and outputs: the copies to and from the device
// are pipelined with the compute inside the library, so that a caller streaming host data makes
// one call per batch.
//
// "Beyond the KV cache" (Laplace 3B on Trainium2), section "Challenge 1: Using native PyTorch on
// Trainium for GLA": the forward of a batch is independent per sequence, and within a sequence
// the chunk scan carries only the state from one chunk to the next.  So the batch is cut into
// pieces that can move and run one after another: sub-batches of whole sequences, or, with more
// pieces than sequences, each sequence cut at chunk boundaries into consecutive parts, a part
// starting from the state the previous one left (its h0 = that part's final state, the very
// value the uncut scan carries across the cut, so the results equal the single call's).  Piece i
// is copied in on one stream while piece i - 1 runs on the caller's stream and piece i - 2 is
// copied out on a third; events order the three.
#include <mutex>
#include <vector>

#include "gla.h"
#include "gla_common.cuh"

namespace {

constexpr int kMaxDev = 64;

struct HostPipe {
  cudaStream_t in = nullptr, out = nullptr;
  std::vector<cudaEvent_t> events;  // reused by successive calls (a wait binds the record it sees)
};
std::mutex g_pipe_mu;  // held while a call issues its work: one caller uses the pool at a time
HostPipe g_pipe[kMaxDev];

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

// The device workspace: staged q, k, v and o for the whole batch, the final states and the
// initial states, and two buffers of states handed from one part of a sequence to the next.
struct HostLayout {
  size_t q, k, v, o, hT, h0, mid0, mid1, total;
};
HostLayout host_layout(int n_seq, int T, int H, int dtype) {
  const size_t el = dtype == GLA_F32 ? 4 : 2;
  const size_t rows = (size_t)n_seq * (size_t)T * (size_t)H;
  const size_t st = align256((size_t)n_seq * H * GLA_DK * GLA_DV * sizeof(float));
  HostLayout l;
  l.q = 0;
  l.k = l.q + align256(rows * GLA_DK * el);
  l.v = l.k + align256(rows * GLA_DK * el);
  l.o = l.v + align256(rows * GLA_DV * el);
  l.hT = l.o + align256(rows * GLA_DV * el);
  l.h0 = l.hT + st;
  l.mid0 = l.h0 + st;
  l.mid1 = l.mid0 + st;
  l.total = l.mid1 + st;
  return l;
}

}  // namespace

extern "C" {

size_t gla_chunk_fwd_host_workspace_bytes(int n_seq, int T, int H, int dtype) {
  if (n_seq < 0 || T < 0 || H < 1 || (dtype != GLA_BF16 && dtype != GLA_F32)) return 0;
  return host_layout(n_seq, T, H, dtype).total;
}

int gla_chunk_fwd_host(const void* q, const void* k, const void* v, const float* log_lambda,
                       const float* h0, float scale, void* o, float* hT, int n_seq, int T, int H,
                       int dk, int dv, int dtype, int pieces, void* workspace, size_t ws_bytes,
                       gla_stream_t stream) {
  if (dtype != GLA_BF16 && dtype != GLA_F32) return GLA_ERR_DTYPE;
  if (dk != GLA_DK || dv != GLA_DV) return GLA_ERR_UNSUPPORTED;
  if (n_seq < 0 || T < 0 || H < 1 || pieces < 1) return GLA_ERR_SHAPE;
  if ((long long)n_seq * T * H * GLA_DV >= (1ll << 40)) return GLA_ERR_SHAPE;
  if (n_seq == 0) return GLA_OK;
  if (!log_lambda) return GLA_ERR_NULL;
  if (T > 0 && (!q || !k || !v || !o)) return GLA_ERR_NULL;
  const HostLayout l = host_layout(n_seq, T, H, dtype);
  if (!workspace || ws_bytes < l.total) return GLA_ERR_WORKSPACE;
  if (((uintptr_t)workspace & 255u) != 0 || ((uintptr_t)log_lambda & 15u) != 0) return GLA_ERR_ALIGN;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return GLA_ERR_LAUNCH;

  // The pieces: sub-batches of whole sequences, or each sequence cut into `cuts` parts of a
  // whole number of chunks (the largest such count up to pieces / n_seq).
  int cuts = 1;
  if (pieces > n_seq && T > 0) {
    cuts = pieces / n_seq;
    while (cuts > 1 && (T % cuts != 0 || (T / cuts) % GLA_CHUNK != 0)) --cuts;
  }
  const int subs = cuts > 1 ? n_seq : (pieces < n_seq ? pieces : n_seq);
  const int n_pieces = subs * cuts;

  char* ws = static_cast<char*>(workspace);
  const size_t el = dtype == GLA_F32 ? 4 : 2;
  const size_t st_bytes = (size_t)H * GLA_DK * GLA_DV * sizeof(float);  // one sequence's states
  float* d_hT = reinterpret_cast<float*>(ws + l.hT);
  float* d_h0 = reinterpret_cast<float*>(ws + l.h0);
  float* d_mid[2] = {reinterpret_cast<float*>(ws + l.mid0), reinterpret_cast<float*>(ws + l.mid1)};
  const cudaStream_t comp = (cudaStream_t)stream;

  std::lock_guard<std::mutex> lock(g_pipe_mu);
  HostPipe& pp = g_pipe[dev];
  if (!pp.in && cudaStreamCreateWithFlags(&pp.in, cudaStreamNonBlocking) != cudaSuccess) return GLA_ERR_LAUNCH;
  if (!pp.out && cudaStreamCreateWithFlags(&pp.out, cudaStreamNonBlocking) != cudaSuccess) return GLA_ERR_LAUNCH;
  const size_t need_events = 2 * (size_t)n_pieces + 2;
  while (pp.events.size() < need_events) {
    cudaEvent_t e;
    if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) return GLA_ERR_LAUNCH;
    pp.events.push_back(e);
  }
  cudaEvent_t* ev = pp.events.data();
  bool ok = cudaEventRecord(ev[0], comp) == cudaSuccess && cudaStreamWaitEvent(pp.in, ev[0], 0) == cudaSuccess &&
            cudaStreamWaitEvent(pp.out, ev[0], 0) == cudaSuccess;
  if (ok && h0) ok = cudaMemcpyAsync(d_h0, h0, (size_t)n_seq * st_bytes, cudaMemcpyDefault, pp.in) == cudaSuccess;
  int rc = GLA_OK;
  for (int p = 0; ok && rc == GLA_OK && p < n_pieces; ++p) {
    // piece p: sequences [a, b), tokens [t0, t1) of each, part j of the cut
    const int j = p % cuts, s = p / cuts;
    const int a = cuts > 1 ? s : (int)((long long)n_seq * s / subs);
    const int b = cuts > 1 ? s + 1 : (int)((long long)n_seq * (s + 1) / subs);
    const int t0 = (int)((long long)T * j / cuts), t1 = (int)((long long)T * (j + 1) / cuts);
    const int len = t1 - t0;
    const bool last = t1 == T;
    // copy in: rows (n, t) of sequences a..b-1 at tokens t0..t1-1 (contiguous for one sequence,
    // or for whole sequences)
    // (no rows at all when T = 0: then q, k, v and o may be NULL and nothing is copied)
    const size_t row0 = ((size_t)a * T + t0) * H, nrows = (size_t)(b - a) * len * H;
    if (nrows > 0)
      ok = cudaMemcpyAsync(ws + l.q + row0 * GLA_DK * el, (const char*)q + row0 * GLA_DK * el, nrows * GLA_DK * el,
                           cudaMemcpyDefault, pp.in) == cudaSuccess &&
           cudaMemcpyAsync(ws + l.k + row0 * GLA_DK * el, (const char*)k + row0 * GLA_DK * el, nrows * GLA_DK * el,
                           cudaMemcpyDefault, pp.in) == cudaSuccess &&
           cudaMemcpyAsync(ws + l.v + row0 * GLA_DV * el, (const char*)v + row0 * GLA_DV * el, nrows * GLA_DV * el,
                           cudaMemcpyDefault, pp.in) == cudaSuccess;
    ok = ok && cudaEventRecord(ev[1 + 2 * p], pp.in) == cudaSuccess &&
         cudaStreamWaitEvent(comp, ev[1 + 2 * p], 0) == cudaSuccess;
    if (!ok) break;
    // compute: the piece as a fixed-length batch of b - a sequences of len tokens
    const float* p_h0 = j > 0 ? d_mid[(j - 1) & 1] + (size_t)a * (st_bytes / 4) : (h0 ? d_h0 + (size_t)a * (st_bytes / 4) : nullptr);
    float* p_hT = last ? (hT ? d_hT + (size_t)a * (st_bytes / 4) : nullptr) : d_mid[j & 1] + (size_t)a * (st_bytes / 4);
    if (cuts > 1) {
      // one sequence: its rows at tokens t0.. form a [1, len, H, d] batch
      rc = gla_chunk_fwd(ws + l.q + row0 * GLA_DK * el, ws + l.k + row0 * GLA_DK * el, ws + l.v + row0 * GLA_DV * el,
                         log_lambda, p_h0, scale, ws + l.o + row0 * GLA_DV * el, p_hT, nullptr, 1, len, H, dk, dv,
                         dtype, nullptr, 0, stream);
    } else {
      rc = gla_chunk_fwd(ws + l.q + row0 * GLA_DK * el, ws + l.k + row0 * GLA_DK * el, ws + l.v + row0 * GLA_DV * el,
                         log_lambda, p_h0, scale, ws + l.o + row0 * GLA_DV * el, p_hT, nullptr, b - a, T, H, dk, dv,
                         dtype, nullptr, 0, stream);
    }
    if (rc != GLA_OK) break;
    // copy out: the piece's o rows, and the final states once a sequence is done
    ok = cudaEventRecord(ev[2 + 2 * p], comp) == cudaSuccess && cudaStreamWaitEvent(pp.out, ev[2 + 2 * p], 0) == cudaSuccess;
    if (ok && nrows > 0)
      ok = cudaMemcpyAsync((char*)o + row0 * GLA_DV * el, ws + l.o + row0 * GLA_DV * el, nrows * GLA_DV * el,
                           cudaMemcpyDefault, pp.out) == cudaSuccess;
    if (ok && last && hT)
      ok = cudaMemcpyAsync(hT + (size_t)a * (st_bytes / 4), p_hT, (size_t)(b - a) * st_bytes, cudaMemcpyDefault,
                           pp.out) == cudaSuccess;
  }
  // the caller's stream completes after the last copy out (also after a failure part-way, so
  // that nothing issued is left unordered)
  const bool joined = cudaEventRecord(ev[2 * n_pieces + 1], pp.out) == cudaSuccess &&
                      cudaStreamWaitEvent(comp, ev[2 * n_pieces + 1], 0) == cudaSuccess;
  if (rc != GLA_OK) return rc;
  return ok && joined ? GLA_OK : GLA_ERR_LAUNCH;
}

}  // extern "C"
