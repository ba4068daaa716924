// Simple GLA mixer: plain fp64 CPU oracle.  TEST INFRASTRUCTURE ONLY.
//
// Only the tests, the package's smoke check and the benchmark's CPU-baseline leg load this
// file.  The GPU library shares no code, header or constant with it, and it never calls the
// GPU library.  Everything here is written for a reader checking it against the source by eye:
// straight loops over tokens, fp64 throughout, no blocking and no reordering beyond what the
// definitions state.
//
// Source: "Beyond the KV cache: Training and serving i14's Laplace 3B linear attention model
// on AWS Trainium2 with native PyTorch" (AWS blog post and its Spanish and Chinese copies),
//   - section "i14 and the Laplace 3B architecture", paragraph "GLA mixer": each head keeps a
//     d_k x d_v state S_t, decayed by the fixed per-head factor lambda_h and written with the
//     rank-1 outer product k_t v_t^T ("GLA recurrent-state update equation"); the readout
//     queries the state ("GLA state-readout equation").  The equation images are missing from
//     the text; the readings used are
//         S_t = lambda_h * S_{t-1} + k_t v_t^T,        o_t = S_t^T (scale * q_t),
//     with the readout taken after the update, S_0 = h0 (zeros when absent), hT = S_T.
//   - section "Challenge 1: Using native PyTorch on Trainium for GLA": the chunked form
//     (intra-chunk masked linear attention plus the running state, state advanced with the
//     decay compounded over the chunk).  Its equation images are missing too; the chunked
//     function below is derived from the recurrence and used only to show chunk-size
//     invariance of the definition.
//   - section "Challenge 3" (backward through the sequential state updates): the page only says
//     that autograd differentiates the 16 sequential updates; the backward below is the adjoint
//     of the recurrence above.  lambda is fixed, not learned, so there is no lambda gradient.
//
// Layouts (all C order): q, k [T_total, H, dk]; v, o, dO [T_total, H, dv];
// h0, hT, dhT, dh0 [n_seq, H, dk, dv]; sequence n owns tokens cu_seqlens[n] .. cu_seqlens[n+1]-1.
// Inputs are fp32 arrays (bf16 inputs arrive as their exact fp32 values); results are fp64.
// log_lambda is the natural log of lambda_h, one fp32 per head; lambda_h = exp(log_lambda[h])
// evaluated in double.

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <functional>
#include <thread>
#include <vector>

namespace {

// Runs body(n, h) for every (sequence, head) pair on `nthreads` threads (0 = all cores).
void for_each_unit(int n_seq, int H, int nthreads, const std::function<void(int, int)>& body) {
  const long total = (long)n_seq * H;
  if (nthreads <= 0) nthreads = (int)std::thread::hardware_concurrency();
  if (nthreads <= 0) nthreads = 1;
  if (nthreads > total) nthreads = (int)(total > 0 ? total : 1);
  std::atomic<long> next(0);
  auto worker = [&]() {
    for (long u = next.fetch_add(1); u < total; u = next.fetch_add(1)) body((int)(u / H), (int)(u % H));
  };
  if (nthreads == 1) { worker(); return; }
  std::vector<std::thread> pool;
  for (int i = 0; i < nthreads; ++i) pool.emplace_back(worker);
  for (auto& t : pool) t.join();
}

int check_common(const int32_t* cu_seqlens, int n_seq, int H, int dk, int dv) {
  if (!cu_seqlens || n_seq < 0 || H <= 0 || dk <= 0 || dv <= 0) return -1;
  if (cu_seqlens[0] != 0) return -2;
  for (int n = 0; n < n_seq; ++n)
    if (cu_seqlens[n + 1] < cu_seqlens[n]) return -2;
  return 0;
}

}  // namespace

extern "C" {

int oracle_hardware_threads(void) { return (int)std::thread::hardware_concurrency(); }

// Forward: the per-token recurrence, read literally.
int oracle_fwd(const float* q, const float* k, const float* v, const float* log_lambda,
               const float* h0, double scale, const int32_t* cu_seqlens, int n_seq, int H,
               int dk, int dv, double* o, double* hT, int nthreads) {
  int rc = check_common(cu_seqlens, n_seq, H, dk, dv);
  if (rc) return rc;
  for_each_unit(n_seq, H, nthreads, [&](int n, int h) {
    const double lam = std::exp((double)log_lambda[h]);
    std::vector<double> S((size_t)dk * dv, 0.0);
    if (h0) {
      const float* src = h0 + ((size_t)n * H + h) * dk * dv;
      for (size_t e = 0; e < S.size(); ++e) S[e] = (double)src[e];
    }
    std::vector<double> sq(dk);
    for (int t = cu_seqlens[n]; t < cu_seqlens[n + 1]; ++t) {
      const float* kt = k + ((size_t)t * H + h) * dk;
      const float* vt = v + ((size_t)t * H + h) * dv;
      const float* qt = q + ((size_t)t * H + h) * dk;
      // S_t = lambda * S_{t-1} + k_t v_t^T
      for (int a = 0; a < dk; ++a)
        for (int b = 0; b < dv; ++b)
          S[(size_t)a * dv + b] = lam * S[(size_t)a * dv + b] + (double)kt[a] * (double)vt[b];
      // o_t = S_t^T (scale * q_t)
      for (int a = 0; a < dk; ++a) sq[a] = scale * (double)qt[a];
      double* ot = o + ((size_t)t * H + h) * dv;
      for (int b = 0; b < dv; ++b) {
        double acc = 0.0;
        for (int a = 0; a < dk; ++a) acc += S[(size_t)a * dv + b] * sq[a];
        ot[b] = acc;
      }
    }
    if (hT) std::memcpy(hT + ((size_t)n * H + h) * dk * dv, S.data(), S.size() * sizeof(double));
  });
  return 0;
}

// Forward in chunks of C tokens, fp64.  Used only to show that the chunked decomposition the
// GPU path uses reaches the recurrence's result for any chunk size.  Within a chunk of L
// tokens (local index i, j = 0..L-1; the state before the chunk is S):
//   o_i   = scale * lambda^(i+1) * S^T q_i + scale * sum_{j<=i} lambda^(i-j) (q_i . k_j) v_j
//   S_new = lambda^L * S + sum_j lambda^(L-1-j) k_j v_j^T
int oracle_fwd_chunked(const float* q, const float* k, const float* v, const float* log_lambda,
                       const float* h0, double scale, const int32_t* cu_seqlens, int n_seq, int H,
                       int dk, int dv, int C, double* o, double* hT, int nthreads) {
  int rc = check_common(cu_seqlens, n_seq, H, dk, dv);
  if (rc) return rc;
  if (C <= 0) return -1;
  for_each_unit(n_seq, H, nthreads, [&](int n, int h) {
    const double lam = std::exp((double)log_lambda[h]);
    std::vector<double> S((size_t)dk * dv, 0.0), Snew((size_t)dk * dv);
    if (h0) {
      const float* src = h0 + ((size_t)n * H + h) * dk * dv;
      for (size_t e = 0; e < S.size(); ++e) S[e] = (double)src[e];
    }
    for (int t0 = cu_seqlens[n]; t0 < cu_seqlens[n + 1]; t0 += C) {
      const int L = std::min(C, cu_seqlens[n + 1] - t0);
      auto Q = [&](int i, int a) { return (double)q[((size_t)(t0 + i) * H + h) * dk + a]; };
      auto K = [&](int i, int a) { return (double)k[((size_t)(t0 + i) * H + h) * dk + a]; };
      auto V = [&](int i, int b) { return (double)v[((size_t)(t0 + i) * H + h) * dv + b]; };
      for (int i = 0; i < L; ++i) {
        double* oi = o + ((size_t)(t0 + i) * H + h) * dv;
        const double inter = scale * std::pow(lam, i + 1);
        for (int b = 0; b < dv; ++b) {
          double acc = 0.0;
          for (int a = 0; a < dk; ++a) acc += Q(i, a) * S[(size_t)a * dv + b];
          oi[b] = inter * acc;
        }
        for (int j = 0; j <= i; ++j) {
          double qk = 0.0;
          for (int a = 0; a < dk; ++a) qk += Q(i, a) * K(j, a);
          const double w = scale * std::pow(lam, i - j) * qk;
          for (int b = 0; b < dv; ++b) oi[b] += w * V(j, b);
        }
      }
      const double lamL = std::pow(lam, L);
      for (int a = 0; a < dk; ++a)
        for (int b = 0; b < dv; ++b) {
          double acc = lamL * S[(size_t)a * dv + b];
          for (int j = 0; j < L; ++j) acc += std::pow(lam, L - 1 - j) * K(j, a) * V(j, b);
          Snew[(size_t)a * dv + b] = acc;
        }
      S.swap(Snew);
    }
    if (hT) std::memcpy(hT + ((size_t)n * H + h) * dk * dv, S.data(), S.size() * sizeof(double));
  });
  return 0;
}

// One decode step for N independent states, in place: S <- lambda S + k v^T; o = S^T (scale q).
// q, k [N, H, dk]; v [N, H, dv]; state [N, H, dk, dv] (fp64, updated); o [N, H, dv].
int oracle_decode_step(const float* q, const float* k, const float* v, const float* log_lambda,
                       double scale, double* state, double* o, int N, int H, int dk, int dv,
                       int nthreads) {
  if (N < 0 || H <= 0 || dk <= 0 || dv <= 0) return -1;
  for_each_unit(N, H, nthreads, [&](int n, int h) {
    const double lam = std::exp((double)log_lambda[h]);
    double* S = state + ((size_t)n * H + h) * dk * dv;
    const float* kt = k + ((size_t)n * H + h) * dk;
    const float* vt = v + ((size_t)n * H + h) * dv;
    const float* qt = q + ((size_t)n * H + h) * dk;
    for (int a = 0; a < dk; ++a)
      for (int b = 0; b < dv; ++b)
        S[(size_t)a * dv + b] = lam * S[(size_t)a * dv + b] + (double)kt[a] * (double)vt[b];
    double* ot = o + ((size_t)n * H + h) * dv;
    for (int b = 0; b < dv; ++b) {
      double acc = 0.0;
      for (int a = 0; a < dk; ++a) acc += S[(size_t)a * dv + b] * (scale * (double)qt[a]);
      ot[b] = acc;
    }
  });
  return 0;
}

// Self-augmentation (section "i14 and the Laplace 3B architecture", the paragraph after the
// state readout): each head's output gains a gated copy of the token's own value,
//     add_t = sigmoid(q_t . (a_h (*) k_t)) * v_t,
// where (*) is the element-wise product and a_h (aug_balance) is the head's learned rescaling of
// the key's d_k channels; a = 0 gives sigmoid(0) = 1/2, the half-strength copy of the value the
// page describes at initialisation.  The equation image is missing from the text; the readings
// used: the query enters unscaled (the readout's scale is not applied to the gate), a holds one
// d_k vector per head, and the term is added to the readout o_t.  Rows are tokens of a forward
// call or sequences of a decode step: q, k [rows, H, dk]; v, add [rows, H, dv]; aug [H, dk].
int oracle_self_aug(const float* q, const float* k, const float* v, const float* aug, long long rows,
                    int H, int dk, int dv, double* add) {
  if (rows < 0 || H <= 0 || dk <= 0 || dv <= 0) return -1;
  for (long long t = 0; t < rows; ++t)
    for (int h = 0; h < H; ++h) {
      const float* qt = q + ((size_t)t * H + h) * dk;
      const float* kt = k + ((size_t)t * H + h) * dk;
      const float* vt = v + ((size_t)t * H + h) * dv;
      const float* ah = aug + (size_t)h * dk;
      double g = 0.0;
      for (int c = 0; c < dk; ++c) g += (double)qt[c] * ((double)ah[c] * (double)kt[c]);
      const double gate = 1.0 / (1.0 + std::exp(-g));
      double* out = add + ((size_t)t * H + h) * dv;
      for (int b = 0; b < dv; ++b) out[b] = gate * (double)vt[b];
    }
  return 0;
}

// Per-tier Head RMSNorm and SiLU output gate (same section, the end of the paragraph after the
// readout, and the architecture table's "Head RMSNorm (per tier)"): each head's output row is
// RMS-normalised, scaled by the gain of the head's decay tier (the heads of a tier share one
// Head RMSNorm), and gated element-wise by SiLU(g_t), the gate stream of the QKVG projection:
//     y_{t,h} = o_{t,h} / sqrt(mean_c o_{t,h,c}^2 + eps) (*) w_{tier(h)} (*) SiLU(g_{t,h}),
//     SiLU(x) = x * sigmoid(x).
// Readings: the RMS runs over one head's d_v channels; the tier of each head and eps are inputs
// (the pages state neither).  o, g, y [rows, H, dv]; w [n_tiers, dv]; tier [H].
int oracle_head_norm_gate(const float* o, const float* g, const float* w, const int32_t* tier,
                          int n_tiers, double eps, long long rows, int H, int dv, double* y) {
  if (rows < 0 || H <= 0 || dv <= 0 || n_tiers <= 0 || eps < 0) return -1;
  for (int h = 0; h < H; ++h)
    if (tier[h] < 0 || tier[h] >= n_tiers) return -1;
  for (long long t = 0; t < rows; ++t)
    for (int h = 0; h < H; ++h) {
      const float* ot = o + ((size_t)t * H + h) * dv;
      const float* gt = g + ((size_t)t * H + h) * dv;
      const float* wt = w + (size_t)tier[h] * dv;
      double ss = 0.0;
      for (int c = 0; c < dv; ++c) ss += (double)ot[c] * (double)ot[c];
      const double inv = 1.0 / std::sqrt(ss / dv + eps);
      double* yt = y + ((size_t)t * H + h) * dv;
      for (int c = 0; c < dv; ++c) {
        const double gc = (double)gt[c];
        const double silu = gc / (1.0 + std::exp(-gc));
        yt[c] = (double)ot[c] * inv * (double)wt[c] * silu;
      }
    }
  return 0;
}

// A value rounded to the nearest bf16 (8 significant bits, ties to even), fp64 in and out;
// zeros and non-finite values pass through.  Written from the format's definition.
double round_to_bf16(double x) {
  if (x == 0.0 || !std::isfinite(x)) return x;
  int e;
  const double m = std::frexp(x, &e);  // x = m 2^e, 0.5 <= |m| < 1
  const double r = std::nearbyint(std::ldexp(m, 8));  // 8 significant bits; default rounding
  return std::ldexp(r, e - 8);                         // mode: to nearest, ties to even
}

// One decode step with the state stored in bf16 (not on the pages: a storage variant that
// halves the state traffic).  The update and the readout are those of oracle_decode_step,
// computed from the stored (bf16-valued) state; the readout uses the updated state before it
// is rounded, and the stored state is the update rounded to bf16.  state holds bf16 values in
// fp64 and is updated in place.  (The self-augmentation term does not touch the state: a
// caller adds oracle_self_aug's output to o.)
int oracle_decode_step_bf16_state(const float* q, const float* k, const float* v, const float* log_lambda,
                                  double scale, double* state, double* o, int N, int H, int dk, int dv) {
  if (N < 0 || H <= 0 || dk <= 0 || dv <= 0) return -1;
  std::vector<double> S((size_t)dk * dv);
  for (int n = 0; n < N; ++n)
    for (int h = 0; h < H; ++h) {
      const double lam = std::exp((double)log_lambda[h]);
      double* St = state + ((size_t)n * H + h) * dk * dv;
      const float* kt = k + ((size_t)n * H + h) * dk;
      const float* vt = v + ((size_t)n * H + h) * dv;
      const float* qt = q + ((size_t)n * H + h) * dk;
      for (int a = 0; a < dk; ++a)
        for (int b = 0; b < dv; ++b)
          S[(size_t)a * dv + b] = lam * St[(size_t)a * dv + b] + (double)kt[a] * (double)vt[b];
      double* ot = o + ((size_t)n * H + h) * dv;
      for (int b = 0; b < dv; ++b) {
        double acc = 0.0;
        for (int a = 0; a < dk; ++a) acc += S[(size_t)a * dv + b] * (scale * (double)qt[a]);
        ot[b] = acc;
      }
      for (size_t e = 0; e < S.size(); ++e) St[e] = round_to_bf16(S[e]);
    }
  return 0;
}

int oracle_round_to_bf16(const double* x, double* y, long long n) {
  for (long long i = 0; i < n; ++i) y[i] = round_to_bf16(x[i]);
  return 0;
}

// ---- MXFP8 decode state (not on the pages: a storage variant that quarters the state stream) ----
// Format: OCP "Microscaling Formats (MX) Specification" v1.0, MXFP8 with E4M3 elements: every
// block of 32 consecutive elements of a state row shares one E8M0 scale X = 2^(byte - 127).
// E4M3 (OCP "8-bit Floating Point Specification"): sign, 4 exponent bits (bias 7), 3 mantissa
// bits; no infinities; S.1111.111 is NaN; the largest finite value is 0.1111.110 = 448;
// exponent field 0 holds the subnormals m/8 * 2^-6.
double e4m3_value(uint8_t c) {
  const int sign = c >> 7, e = (c >> 3) & 15, m = c & 7;
  if (e == 15 && m == 7) return std::nan("");
  const double mag = e == 0 ? std::ldexp((double)m, -9) : std::ldexp(8.0 + m, e - 10);
  return sign ? -mag : mag;
}

// A finite value to E4M3: round to nearest, ties to even, magnitudes from 448 up saturate to 448
// (the conversion with saturation of the MX specification).
uint8_t e4m3_code(double y) {
  const uint8_t sign = std::signbit(y) ? 0x80 : 0;
  const double a = std::fabs(y);
  if (a >= 448.0) return sign | 0x7E;
  int ex = 0;
  if (a > 0) std::frexp(a, &ex);
  const int E = std::max(ex - 1, -6);                         // a in [2^E, 2^(E+1)), or subnormal
  const double r = std::nearbyint(std::ldexp(a, 3 - E));      // multiples of 2^(E-3); default
  const double val = std::ldexp(r, E - 3);                    // rounding: to nearest, ties to even
  if (val == 0.0) return sign;
  std::frexp(val, &ex);
  const int Ev = ex - 1;                                      // (a carry may have raised it)
  if (Ev < -6) return sign | (uint8_t)std::ldexp(val, 9);     // subnormal: m 2^-9
  const int m = (int)std::ldexp(val, 3 - Ev) - 8;
  return sign | (uint8_t)(((Ev + 7) << 3) | m);
}

// One block of n (32) values.  Shared exponent: the MX specification's floor(log2(max |x|)) - 8
// (8 = the exponent of E4M3's largest power of two), raised by one when the block maximum
// would then exceed 448 (the specification would saturate it to 448, an error of up to 12.5 %),
// i.e. the smallest exponent at which the whole block is representable; clamped to E8M0's
// [-127, 127] (-127 for an all-zero block).  Elements x / 2^shared_exp converted as above.
void mxfp8_block(const float* x, int n, uint8_t* codes, uint8_t* scale_byte) {
  double mx = 0.0;
  for (int i = 0; i < n; ++i) mx = std::max(mx, std::fabs((double)x[i]));
  int se = -127;
  if (mx > 0) {
    int ex;
    std::frexp(mx, &ex);
    se = ex - 1 - 8;
    if (std::ldexp(mx, -se) > 448.0) se += 1;
    se = std::min(std::max(se, -127), 127);
  }
  *scale_byte = (uint8_t)(se + 127);
  for (int i = 0; i < n; ++i) codes[i] = e4m3_code(std::ldexp((double)x[i], -se));
}

double e8m0_value(uint8_t b) { return b == 255 ? std::nan("") : std::ldexp(1.0, (int)b - 127); }

// rows x cols (cols a multiple of 32) fp32 values -> codes [rows, cols], scales [rows, cols/32].
int oracle_mxfp8_quantize(const float* x, long long rows, int cols, uint8_t* codes, uint8_t* scales) {
  if (rows < 0 || cols <= 0 || cols % 32) return -1;
  for (long long r = 0; r < rows; ++r)
    for (int b = 0; b < cols / 32; ++b)
      mxfp8_block(x + r * cols + 32 * b, 32, codes + r * cols + 32 * b, scales + r * (cols / 32) + b);
  return 0;
}

int oracle_mxfp8_dequantize(const uint8_t* codes, const uint8_t* scales, long long rows, int cols, double* x) {
  if (rows < 0 || cols <= 0 || cols % 32) return -1;
  for (long long r = 0; r < rows; ++r)
    for (int c = 0; c < cols; ++c)
      x[r * cols + c] = e4m3_value(codes[r * cols + c]) * e8m0_value(scales[r * (cols / 32) + c / 32]);
  return 0;
}

// One decode step with an MXFP8-stored state [N, H, dk, dv] (codes) + [N, H, dk, dv/32]
// (scales), in place.  The state is widened exactly, updated and read out in fp64 as in
// oracle_decode_step (the readout from the update before any rounding); the update is then
// rounded to fp32, the precision in which the GPU path takes its quantisation decisions, and
// stored as MXFP8 row by row.  pre (optional, [N, H, dk, dv]) receives those fp32 values.
int oracle_decode_step_mxfp8_state(const float* q, const float* k, const float* v, const float* log_lambda,
                                   double scale, uint8_t* codes, uint8_t* scales, double* o, int N, int H,
                                   int dk, int dv, float* pre) {
  if (N < 0 || H <= 0 || dk <= 0 || dv <= 0 || dv % 32) return -1;
  std::vector<double> S((size_t)dk * dv);
  std::vector<float> X((size_t)dk * dv);
  for (int n = 0; n < N; ++n)
    for (int h = 0; h < H; ++h) {
      const double lam = std::exp((double)log_lambda[h]);
      uint8_t* Ct = codes + ((size_t)n * H + h) * dk * dv;
      uint8_t* Bt = scales + ((size_t)n * H + h) * dk * (dv / 32);
      const float* kt = k + ((size_t)n * H + h) * dk;
      const float* vt = v + ((size_t)n * H + h) * dv;
      const float* qt = q + ((size_t)n * H + h) * dk;
      for (int a = 0; a < dk; ++a)
        for (int b = 0; b < dv; ++b) {
          const double s_ab = e4m3_value(Ct[(size_t)a * dv + b]) * e8m0_value(Bt[(size_t)a * (dv / 32) + b / 32]);
          S[(size_t)a * dv + b] = lam * s_ab + (double)kt[a] * (double)vt[b];
        }
      double* ot = o + ((size_t)n * H + h) * dv;
      for (int b = 0; b < dv; ++b) {
        double acc = 0.0;
        for (int a = 0; a < dk; ++a) acc += S[(size_t)a * dv + b] * (scale * (double)qt[a]);
        ot[b] = acc;
      }
      for (size_t e = 0; e < S.size(); ++e) X[e] = (float)S[e];
      for (int a = 0; a < dk; ++a)
        for (int b = 0; b < dv / 32; ++b)
          mxfp8_block(&X[(size_t)a * dv + 32 * b], 32, Ct + (size_t)a * dv + 32 * b, Bt + (size_t)a * (dv / 32) + b);
      if (pre) std::memcpy(pre + ((size_t)n * H + h) * dk * dv, X.data(), X.size() * sizeof(float));
    }
  return 0;
}

// Backward of oracle_fwd (the adjoint of the recurrence), given dO = dL/do and dhT = dL/dhT.
// With G_t = dL/dS_t (all later uses included) and R_t = lambda * G_{t+1} (R_T = dhT):
//   G_t  = R_t + scale * q_t dO_t^T
//   dq_t = scale * S_t dO_t            (S_t is the forward state after token t)
//   dk_t = G_t v_t,   dv_t = G_t^T k_t
//   dh0  = lambda * G_1               (= dhT for an empty sequence)
// dhT and h0 may be null (zeros); dh0 may be null (not written).
int oracle_bwd(const float* q, const float* k, const float* v, const float* log_lambda,
               const float* h0, double scale, const float* dO, const float* dhT,
               const int32_t* cu_seqlens, int n_seq, int H, int dk, int dv, double* dq,
               double* dk_out, double* dv_out, double* dh0, int nthreads) {
  int rc = check_common(cu_seqlens, n_seq, H, dk, dv);
  if (rc) return rc;
  for_each_unit(n_seq, H, nthreads, [&](int n, int h) {
    const double lam = std::exp((double)log_lambda[h]);
    const size_t DS = (size_t)dk * dv;
    // Pass 1, forward in time: rebuild S_t and read dq_t off it.
    std::vector<double> S(DS, 0.0);
    if (h0) {
      const float* src = h0 + ((size_t)n * H + h) * DS;
      for (size_t e = 0; e < DS; ++e) S[e] = (double)src[e];
    }
    for (int t = cu_seqlens[n]; t < cu_seqlens[n + 1]; ++t) {
      const float* kt = k + ((size_t)t * H + h) * dk;
      const float* vt = v + ((size_t)t * H + h) * dv;
      const float* gt = dO + ((size_t)t * H + h) * dv;
      for (int a = 0; a < dk; ++a)
        for (int b = 0; b < dv; ++b)
          S[(size_t)a * dv + b] = lam * S[(size_t)a * dv + b] + (double)kt[a] * (double)vt[b];
      double* dqt = dq + ((size_t)t * H + h) * dk;
      for (int a = 0; a < dk; ++a) {
        double acc = 0.0;
        for (int b = 0; b < dv; ++b) acc += S[(size_t)a * dv + b] * (double)gt[b];
        dqt[a] = scale * acc;
      }
    }
    // Pass 2, backward in time: carry R = lambda * G_{t+1}.
    std::vector<double> R(DS, 0.0), G(DS);
    if (dhT) {
      const float* src = dhT + ((size_t)n * H + h) * DS;
      for (size_t e = 0; e < DS; ++e) R[e] = (double)src[e];
    }
    for (int t = cu_seqlens[n + 1] - 1; t >= cu_seqlens[n]; --t) {
      const float* qt = q + ((size_t)t * H + h) * dk;
      const float* kt = k + ((size_t)t * H + h) * dk;
      const float* vt = v + ((size_t)t * H + h) * dv;
      const float* gt = dO + ((size_t)t * H + h) * dv;
      for (int a = 0; a < dk; ++a)
        for (int b = 0; b < dv; ++b)
          G[(size_t)a * dv + b] = R[(size_t)a * dv + b] + scale * (double)qt[a] * (double)gt[b];
      double* dkt = dk_out + ((size_t)t * H + h) * dk;
      for (int a = 0; a < dk; ++a) {
        double acc = 0.0;
        for (int b = 0; b < dv; ++b) acc += G[(size_t)a * dv + b] * (double)vt[b];
        dkt[a] = acc;
      }
      double* dvt = dv_out + ((size_t)t * H + h) * dv;
      for (int b = 0; b < dv; ++b) {
        double acc = 0.0;
        for (int a = 0; a < dk; ++a) acc += G[(size_t)a * dv + b] * (double)kt[a];
        dvt[b] = acc;
      }
      for (size_t e = 0; e < DS; ++e) R[e] = lam * G[e];
    }
    if (dh0) std::memcpy(dh0 + ((size_t)n * H + h) * DS, R.data(), DS * sizeof(double));
  });
  return 0;
}

}  // extern "C"
