// Chunked GLA kernels on the CUDA cores: the all-fp32 forward (GLA_F32 mode) and the backward.
//
// "Beyond the KV cache" (Laplace 3B on Trainium2), section "Challenge 1: Using native PyTorch on
// Trainium for GLA": inside a chunk the output is masked linear attention plus the contribution
// of the carried state, and the state then advances with the decay compounded over the chunk.
// With local indices i, j in a chunk of L tokens and S the state before it:
//     o_i   = scale * lambda^(i+1) * S^T q_i + sum_{j<=i} scale * lambda^(i-j) (q_i . k_j) v_j
//     S'    = lambda^L S + sum_j lambda^(L-1-j) k_j v_j^T
// The decay is never split into lambda^i * lambda^-j: every power is looked up from a per-head
// table lambda^d, d = 0..SC, so lambda = 0.5 (the pages' head 0) cannot overflow.
//
// The backward ("Challenge 3": the backward pass differentiates through the sequential state
// updates) is the adjoint of the recurrence, also in chunks:
//   dq (forward in time):   dq_i = scale lambda^(i+1) S dO_i + sum_{j<=i} scale lambda^(i-j) (dO_i.v_j) k_j
//   reverse in time, carrying R = dL/dS flowing in from the next chunk (R = dhT for the last):
//     dk_i = lambda^(L-1-i) R v_i   + sum_{j>=i} scale lambda^(j-i) (dO_j . v_i) q_j
//     dv_i = lambda^(L-1-i) R^T k_i + sum_{j>=i} scale lambda^(j-i) (q_j . k_i) dO_j
//     R'   = lambda^L R + scale * sum_j lambda^(j+1) q_j dO_j^T ;   dh0 = R after the first chunk.
//
// These kernels use 64-token chunks so that their fp32 tiles fit in shared memory; the chunk size
// does not change the result.  One CTA of 256 threads runs the chunk scan of one (sequence,
// head, column tile).  Rows past the end of a sequence are loaded as zeros, so they add nothing.
#include <type_traits>

#include "gla_common.cuh"

namespace gla {
namespace {

constexpr int SC = 64;          // chunk length of these kernels
constexpr int NT = 256;         // threads per CTA

template <class T>
__device__ __forceinline__ void load_rows(float* dst, int pitch, const T* src, long long t0, int L,
                                          int H, int h, int width, int col0, int ncols) {
  for (int e = threadIdx.x; e < SC * ncols; e += NT) {
    const int i = e / ncols, c = e % ncols;
    dst[i * pitch + c] = i < L ? to_f(src[((t0 + i) * H + h) * (long long)width + col0 + c]) : 0.f;
  }
}

__device__ __forceinline__ void fill_powers(float* pw, float ll) {
  for (int d = threadIdx.x; d <= SC; d += NT) pw[d] = d == 0 ? 1.f : expf((float)d * ll);
}

// ------------------------------------------------------------------------------------------
// Forward.  Tile = 64 columns of d_v (3 tiles).  Each chunk is four small matrix products on
// register tiles: P = Q K^T (64 x 64 over d_k), O_intra = P V (64 x 64 over the chunk),
// O_inter = Q S (64 x 64 over d_k), and S' = lambda^L S + (w K)^T V (96 x 64 over the chunk).
// Thread (ty, tx) = (t / 16, t % 16) owns the rows ty + 16a (a < 4; a < 6 of the state) and, in
// P, the columns tx + 16b, elsewhere the 4 adjacent columns 4tx .. 4tx + 3.  Rows strided by 16
// put a quarter warp's 8 threads on 8 consecutive rows, so with the padded pitches below their
// float4 loads along a row fall in 8 different bank groups; about 8 fused multiply-adds per
// shared-memory load.
// ------------------------------------------------------------------------------------------
constexpr int FWD_TILE = 64;
constexpr int FWD_TILES = DV / FWD_TILE;
constexpr int QP = DK + 4;        // row pitch of q and k (floats; rows stay 16-byte aligned)
constexpr int VP = FWD_TILE + 4;  // row pitch of the v tile, P and the state tile
constexpr size_t FWD_SMEM = sizeof(float) * (2 * SC * QP + 2 * SC * VP + DK * VP + 2 * SC + 8);

__device__ __forceinline__ float4 ld4(const float* p) { return *reinterpret_cast<const float4*>(p); }

// A chunk's rows of q and k (96 values) and of the v tile (64) from fp32 inputs: 16-byte loads,
// all issued before the first store (16 per thread), rows past the end as zeros.  Other input
// types go through load_rows.
__device__ __forceinline__ void load_chunk_f32(float* Qs, float* Ks, float* Vs, const float* q, const float* k,
                                               const float* v, long long t0, int L, int H, int h, int col0,
                                               int qp, int vp) {
  constexpr int QV = DK / 4, VV = 64 / 4;  // float4 per q / k row, per v tile row
  float4 rq[QV * SC / NT], rk[QV * SC / NT], rv[VV * SC / NT];
#pragma unroll
  for (int m = 0; m < QV * SC / NT; ++m) {
    const int e = threadIdx.x + NT * m, i = e / QV, c = e % QV;
    const long long row = (t0 + (i < L ? i : 0)) * H + h;
    rq[m] = i < L ? ld4(q + row * DK + 4 * c) : make_float4(0.f, 0.f, 0.f, 0.f);
    rk[m] = i < L ? ld4(k + row * DK + 4 * c) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
#pragma unroll
  for (int m = 0; m < VV * SC / NT; ++m) {
    const int e = threadIdx.x + NT * m, i = e / VV, c = e % VV;
    const long long row = (t0 + (i < L ? i : 0)) * H + h;
    rv[m] = i < L ? ld4(v + row * DV + col0 + 4 * c) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
#pragma unroll
  for (int m = 0; m < QV * SC / NT; ++m) {
    const int e = threadIdx.x + NT * m, i = e / QV, c = e % QV;
    *reinterpret_cast<float4*>(Qs + i * qp + 4 * c) = rq[m];
    *reinterpret_cast<float4*>(Ks + i * qp + 4 * c) = rk[m];
  }
#pragma unroll
  for (int m = 0; m < VV * SC / NT; ++m) {
    const int e = threadIdx.x + NT * m, i = e / VV, c = e % VV;
    *reinterpret_cast<float4*>(Vs + i * vp + 4 * c) = rv[m];
  }
}
// The next chunk's rows into L2 while this one computes (one 128-byte line per thread and call).
__device__ __forceinline__ void prefetch_chunk(const void* base, long long t0, int L, int H, int h, int width,
                                               int esize, int col0, int ncols) {
  const int lines = (ncols * esize + 127) / 128;
  for (int e = threadIdx.x; e < L * lines; e += NT) {
    const int i = e / lines, c = e % lines;
    const char* p = (const char*)base + (((t0 + i) * H + h) * (long long)width + col0) * esize + 128 * c;
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
  }
}
__device__ __forceinline__ void st4(float* p, float4 x) { *reinterpret_cast<float4*>(p) = x; }
__device__ __forceinline__ void store4o(float* p, float4 x) { st4(p, x); }
__device__ __forceinline__ void store4o(__nv_bfloat16* p, float4 x) {
  p[0] = __float2bfloat16_rn(x.x);
  p[1] = __float2bfloat16_rn(x.y);
  p[2] = __float2bfloat16_rn(x.z);
  p[3] = __float2bfloat16_rn(x.w);
}

// REVERSE: the dv scan of the backward on the same tiles (reverse in time, carrying R = dL/dS):
//   X = k, Y = q, Z = dO;  P[i][j] = scale lambda^(j-i) X_i . Y_j (j >= i);
//   dv_i = sum_j P[i][j] Z_j + lambda^(L-1-i) R^T X_i;  R <- lambda^L R + scale sum_j lambda^(j+1) Y_j Z_j^T
// (R starts from dhT; dh0 comes from the dk scan).
template <class T, bool REVERSE>
__global__ void __launch_bounds__(NT, 2) simt_wide_kernel(ChunkArgs a) {
  extern __shared__ __align__(16) float sm[];
  float* Qs = sm;                 // [SC][QP]
  float* Ks = Qs + SC * QP;       // [SC][QP]
  float* Vs = Ks + SC * QP;       // [SC][VP]   column tile of v
  float* Ps = Vs + SC * VP;       // [SC][VP]   decayed, masked scale*q.k (plus the gate)
  float* Ss = Ps + SC * VP;       // [DK][VP]   state tile
  float* pw = Ss + DK * VP;       // [SC + 1]   lambda^d
  float* gs = pw + SC + 4;        // [SC]       self-augmentation gates of the chunk's rows
  const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
  int n, h, tile;
  unit_of_block(a, FWD_TILES, n, h, tile);
  long long tb, te;
  seq_range(a, n, tb, te);
  if (!unit_in_bounds(a, n, h)) return;  // (debug-bounds build; uniform over the CTA)
  const int col0 = tile * FWD_TILE;
  const T* q = (const T*)(REVERSE ? a.k : a.q);   // X: the score's row operand (and the readout's)
  const T* k = (const T*)(REVERSE ? a.q : a.k);   // Y: its column operand (and the state's row factor)
  const T* v = (const T*)(REVERSE ? a.dO : a.v);  // Z: the tile's operand
  T* o = (T*)(REVERSE ? a.dv : a.o);
  const float* s0 = REVERSE ? a.dhT : a.h0;
  const bool aug = !REVERSE && a.aug;
  const long long sbase = ((long long)n * a.H + h) * DK * DV;

  fill_powers(pw, a.log_lambda[h]);
  for (int e = tid; e < DK * FWD_TILE; e += NT) {
    const int r = e / FWD_TILE, c = e % FWD_TILE;
    Ss[r * VP + c] = s0 ? s0[sbase + (long long)r * DV + col0 + c] : 0.f;
  }
  __syncthreads();

  const long long nchunks = (te - tb + SC - 1) / SC;
  for (long long m0 = 0; m0 < nchunks; ++m0) {
    const long long t0 = tb + (REVERSE ? nchunks - 1 - m0 : m0) * SC;
    const int L = (int)(te - t0 < SC ? te - t0 : SC);
    if (!rows_in_bounds(a, t0, L)) break;  // (debug-bounds build; uniform over the CTA)
    if constexpr (std::is_same<T, float>::value) {
      load_chunk_f32(Qs, Ks, Vs, q, k, v, t0, L, a.H, h, col0, QP, VP);
    } else {
      load_rows(Qs, QP, q, t0, L, a.H, h, DK, 0, DK);
      load_rows(Ks, QP, k, t0, L, a.H, h, DK, 0, DK);
      load_rows(Vs, VP, v, t0, L, a.H, h, DV, col0, FWD_TILE);
    }
    __syncthreads();
    if (m0 + 1 < nchunks) {  // the next chunk's rows into L2 during this chunk's arithmetic
      const long long tn = REVERSE ? t0 - SC : t0 + SC;
      const int Ln = (int)(te - tn < SC ? te - tn : SC);
      prefetch_chunk(q, tn, Ln, a.H, h, DK, (int)sizeof(T), 0, DK);
      prefetch_chunk(k, tn, Ln, a.H, h, DK, (int)sizeof(T), 0, DK);
      prefetch_chunk(v, tn, Ln, a.H, h, DV, (int)sizeof(T), col0, FWD_TILE);
    }
    if (aug) {  // gate of row i: sigmoid(q_i . (a_h * k_i)), q unscaled; added to P[i][i] below
      if (tid < SC) {
        float g = 0.f;
        for (int c = 0; c < DK; ++c) g = fmaf(Qs[tid * QP + c] * a.aug[h * DK + c], Ks[tid * QP + c], g);
        gs[tid] = 1.f / (1.f + expf(-g));
      }
      __syncthreads();
    }
    {  // P[i][j] = scale lambda^|i-j| X_i . Y_j on the causal side (j <= i, or j >= i reversed)
      float acc[4][4];
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[r][c] = 0.f;
#pragma unroll 2
      for (int kk = 0; kk < DK; kk += 4) {
        float4 qv[4], kv[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) qv[r] = ld4(Qs + (ty + 16 * r) * QP + kk);
#pragma unroll
        for (int c = 0; c < 4; ++c) kv[c] = ld4(Ks + (tx + 16 * c) * QP + kk);
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            acc[r][c] = fmaf(qv[r].x, kv[c].x, acc[r][c]);
            acc[r][c] = fmaf(qv[r].y, kv[c].y, acc[r][c]);
            acc[r][c] = fmaf(qv[r].z, kv[c].z, acc[r][c]);
            acc[r][c] = fmaf(qv[r].w, kv[c].w, acc[r][c]);
          }
      }
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int i = ty + 16 * r, j = tx + 16 * c;
          const bool on = REVERSE ? j >= i : j <= i;
          float p = on ? acc[r][c] * (a.scale * pw[REVERSE ? j - i : i - j]) : 0.f;
          if (aug && j == i) p += gs[i];
          Ps[i * VP + j] = p;
        }
    }
    __syncthreads();
    {  // o_i = sum_j P[i][j] v_j + scale lambda^(i+1) S^T q_i  (this tile's 64 columns)
      float oi[4][4], oe[4][4];
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int c = 0; c < 4; ++c) oi[r][c] = oe[r][c] = 0.f;
      for (int j = 0; j < L; ++j) {
        const float4 vv = ld4(Vs + j * VP + 4 * tx);
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const float p = Ps[(ty + 16 * r) * VP + j];
          oi[r][0] = fmaf(p, vv.x, oi[r][0]);
          oi[r][1] = fmaf(p, vv.y, oi[r][1]);
          oi[r][2] = fmaf(p, vv.z, oi[r][2]);
          oi[r][3] = fmaf(p, vv.w, oi[r][3]);
        }
      }
#pragma unroll 2
      for (int kk = 0; kk < DK; kk += 4) {
        float4 qv[4], sv[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) qv[r] = ld4(Qs + (ty + 16 * r) * QP + kk);
#pragma unroll
        for (int m = 0; m < 4; ++m) sv[m] = ld4(Ss + (kk + m) * VP + 4 * tx);
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const float qm[4] = {qv[r].x, qv[r].y, qv[r].z, qv[r].w};
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            oe[r][0] = fmaf(qm[m], sv[m].x, oe[r][0]);
            oe[r][1] = fmaf(qm[m], sv[m].y, oe[r][1]);
            oe[r][2] = fmaf(qm[m], sv[m].z, oe[r][2]);
            oe[r][3] = fmaf(qm[m], sv[m].w, oe[r][3]);
          }
        }
      }
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int i = ty + 16 * r;
        if (i < L) {
          const float f = REVERSE ? pw[L - 1 - i] : a.scale * pw[i + 1];
          store4o(o + ((t0 + i) * a.H + h) * (long long)DV + col0 + 4 * tx,
                  make_float4(fmaf(f, oe[r][0], oi[r][0]), fmaf(f, oe[r][1], oi[r][1]),
                              fmaf(f, oe[r][2], oi[r][2]), fmaf(f, oe[r][3], oi[r][3])));
        }
      }
    }
    __syncthreads();
    {  // S <- lambda^L S + sum_j lambda^(L-1-j) k_j v_j^T  (rows ty + 16a of d_k, columns 4tx..)
      float acc[6][4];
      const float lamL = pw[L];
#pragma unroll
      for (int r = 0; r < 6; ++r) {
        const float4 sv = ld4(Ss + (ty + 16 * r) * VP + 4 * tx);
        acc[r][0] = lamL * sv.x;
        acc[r][1] = lamL * sv.y;
        acc[r][2] = lamL * sv.z;
        acc[r][3] = lamL * sv.w;
      }
      for (int j = 0; j < L; ++j) {
        const float w = REVERSE ? a.scale * pw[j + 1] : pw[L - 1 - j];
        const float4 vv = ld4(Vs + j * VP + 4 * tx);
        const float4 wv = make_float4(w * vv.x, w * vv.y, w * vv.z, w * vv.w);
#pragma unroll
        for (int r = 0; r < 6; ++r) {
          const float kj = Ks[j * QP + ty + 16 * r];
          acc[r][0] = fmaf(kj, wv.x, acc[r][0]);
          acc[r][1] = fmaf(kj, wv.y, acc[r][1]);
          acc[r][2] = fmaf(kj, wv.z, acc[r][2]);
          acc[r][3] = fmaf(kj, wv.w, acc[r][3]);
        }
      }
#pragma unroll
      for (int r = 0; r < 6; ++r) st4(Ss + (ty + 16 * r) * VP + 4 * tx, make_float4(acc[r][0], acc[r][1], acc[r][2], acc[r][3]));
    }
    __syncthreads();
  }
  if (!REVERSE && a.hT) {
    for (int e = tid; e < DK * FWD_TILE; e += NT) {
      const int r = e / FWD_TILE, c = e % FWD_TILE;
      a.hT[sbase + (long long)r * DV + col0 + c] = Ss[r * VP + c];
    }
  }
}

// ------------------------------------------------------------------------------------------
// Backward, dq (forward in time) and dk with dh0 (reverse in time): one scan template over a tile
// of 32 rows of d_k, carrying the matching 32 rows of a d_k x d_v state, with scores over all of
// d_v.  With X the score's row operand, Y its column operand and Z the tile's operand:
//   dq:  X = dO, Y = v, Z = k;   P[i][j] = scale lambda^(i-j) X_i . Y_j (j <= i);
//        out_i = sum_j P[i][j] Z_j + scale lambda^(i+1) S X_i;  S <- lambda^L S + sum_j lambda^(L-1-j) Z_j Y_j^T
//   dk:  X = v, Y = dO, Z = q;   P[i][j] = scale lambda^(j-i) X_i . Y_j (j >= i);
//        out_i = sum_j P[i][j] Z_j + lambda^(L-1-i) R X_i;      R <- lambda^L R + scale sum_j lambda^(j+1) Z_j Y_j^T
// (S, R: the tile's 32 rows; R starts from dhT and leaves as dh0.)  The chunk's products run on
// register tiles as in the forward: thread (ty, tx) owns P rows ty + 16a, columns tx + 16b;
// output rows ty + 16a, tile columns tx and tx + 16; state rows ty and ty + 16, columns
// 4tx + 64m.
// ------------------------------------------------------------------------------------------
constexpr int BQ_TILE = 32;
constexpr int BQ_TILES = DK / BQ_TILE;
constexpr int XP = DV + 4;        // row pitch of X and Y (192 values) and of the state rows
constexpr int ZP = BQ_TILE + 4;   // row pitch of the Z tile
constexpr int PP = SC + 4;        // row pitch of P
constexpr size_t BQ_SMEM = sizeof(float) * (2 * SC * XP + SC * ZP + BQ_TILE * XP + SC * PP + SC + 8);

// A chunk's rows [t0, t0 + L) of columns [col0, col0 + NCOLS) of a [T, H, width] input into shared
// memory rows of pitch `pitch`: fp32 inputs with 16-byte loads, all issued before the first store;
// rows past the end as zeros.
template <int NCOLS, class T>
__device__ __forceinline__ void load_rows4(float* dst, int pitch, const T* src, long long t0, int L, int H, int h,
                                           int width, int col0) {
  if constexpr (std::is_same<T, float>::value) {
    constexpr int PER = SC * NCOLS / 4 / NT;  // float4 per thread
    static_assert(PER * NT * 4 == SC * NCOLS, "whole float4 per thread");
    float4 r[PER];
#pragma unroll
    for (int m = 0; m < PER; ++m) {
      const int e = threadIdx.x + NT * m, i = e / (NCOLS / 4), c = e % (NCOLS / 4);
      const long long row = (t0 + (i < L ? i : 0)) * H + h;
      r[m] = i < L ? ld4(src + row * width + col0 + 4 * c) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int m = 0; m < PER; ++m) {
      const int e = threadIdx.x + NT * m, i = e / (NCOLS / 4), c = e % (NCOLS / 4);
      st4(dst + i * pitch + 4 * c, r[m]);
    }
  } else {
    load_rows(dst, pitch, src, t0, L, H, h, width, col0, NCOLS);
  }
}
template <class T, bool REVERSE>
__global__ void __launch_bounds__(NT, 1) simt_bwd_narrow_kernel(ChunkArgs a) {
  extern __shared__ __align__(16) float sm[];
  float* Xs = sm;                  // [SC][XP]
  float* Ys = Xs + SC * XP;        // [SC][XP]
  float* Zs = Ys + SC * XP;        // [SC][ZP]   the d_k tile of Z
  float* Ss = Zs + SC * ZP;        // [BQ_TILE][XP]  the carried state's tile rows
  float* Ps = Ss + BQ_TILE * XP;   // [SC][PP]
  float* pw = Ps + SC * PP;        // [SC + 1]
  const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
  int n, h, tile;
  unit_of_block(a, BQ_TILES, n, h, tile);
  long long tb, te;
  seq_range(a, n, tb, te);
  if (!unit_in_bounds(a, n, h)) return;  // (debug-bounds build; uniform over the CTA)
  const int row0 = tile * BQ_TILE;
  const T* X = (const T*)(REVERSE ? a.v : a.dO);
  const T* Y = (const T*)(REVERSE ? a.dO : a.v);
  const T* Z = (const T*)(REVERSE ? a.q : a.k);
  T* out = (T*)(REVERSE ? a.dk : a.o);
  const float* s0 = REVERSE ? a.dhT : a.h0;
  const long long sbase = ((long long)n * a.H + h) * DK * DV;

  fill_powers(pw, a.log_lambda[h]);
  for (int e = tid; e < BQ_TILE * DV; e += NT) {
    const int r = e / DV, c = e % DV;
    Ss[r * XP + c] = s0 ? s0[sbase + (long long)(row0 + r) * DV + c] : 0.f;
  }
  __syncthreads();
  const long long nchunks = (te - tb + SC - 1) / SC;
  for (long long m0 = 0; m0 < nchunks; ++m0) {
    const long long t0 = tb + (REVERSE ? nchunks - 1 - m0 : m0) * SC;
    const int L = (int)(te - t0 < SC ? te - t0 : SC);
    if (!rows_in_bounds(a, t0, L)) break;  // (debug-bounds build; uniform over the CTA)
    load_rows4<DV>(Xs, XP, X, t0, L, a.H, h, DV, 0);
    load_rows4<DV>(Ys, XP, Y, t0, L, a.H, h, DV, 0);
    load_rows4<BQ_TILE>(Zs, ZP, Z, t0, L, a.H, h, DK, row0);
    __syncthreads();
    if (m0 + 1 < nchunks) {  // the next chunk's rows into L2 during this chunk's arithmetic
      const long long tn = REVERSE ? t0 - SC : t0 + SC;
      const int Ln = (int)(te - tn < SC ? te - tn : SC);
      prefetch_chunk(X, tn, Ln, a.H, h, DV, (int)sizeof(T), 0, DV);
      prefetch_chunk(Y, tn, Ln, a.H, h, DV, (int)sizeof(T), 0, DV);
      prefetch_chunk(Z, tn, Ln, a.H, h, DK, (int)sizeof(T), row0, BQ_TILE);
    }
    {  // P[i][j] = scale lambda^|i-j| X_i . Y_j on the causal side (j <= i, or j >= i reversed)
      float acc[4][4];
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[r][c] = 0.f;
#pragma unroll 2
      for (int kk = 0; kk < DV; kk += 4) {
        float4 xv[4], yv[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) xv[r] = ld4(Xs + (ty + 16 * r) * XP + kk);
#pragma unroll
        for (int c = 0; c < 4; ++c) yv[c] = ld4(Ys + (tx + 16 * c) * XP + kk);
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            acc[r][c] = fmaf(xv[r].x, yv[c].x, acc[r][c]);
            acc[r][c] = fmaf(xv[r].y, yv[c].y, acc[r][c]);
            acc[r][c] = fmaf(xv[r].z, yv[c].z, acc[r][c]);
            acc[r][c] = fmaf(xv[r].w, yv[c].w, acc[r][c]);
          }
      }
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int i = ty + 16 * r, j = tx + 16 * c;
          const bool on = REVERSE ? j >= i : j <= i;
          Ps[i * PP + j] = on ? acc[r][c] * (a.scale * pw[REVERSE ? j - i : i - j]) : 0.f;
        }
    }
    __syncthreads();
    {  // out_i = sum_j P[i][j] Z_j + g_i (state rows) . X_i for the tile's columns tx, tx + 16
      float oi[4][2], oe[4][2];
#pragma unroll
      for (int r = 0; r < 4; ++r) oi[r][0] = oi[r][1] = oe[r][0] = oe[r][1] = 0.f;
      for (int j = 0; j < L; ++j) {
        const float z0 = Zs[j * ZP + tx], z1 = Zs[j * ZP + tx + 16];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const float p = Ps[(ty + 16 * r) * PP + j];
          oi[r][0] = fmaf(p, z0, oi[r][0]);
          oi[r][1] = fmaf(p, z1, oi[r][1]);
        }
      }
#pragma unroll 2
      for (int kk = 0; kk < DV; kk += 4) {
        float4 xv[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) xv[r] = ld4(Xs + (ty + 16 * r) * XP + kk);
        const float4 s0v = ld4(Ss + tx * XP + kk), s1v = ld4(Ss + (tx + 16) * XP + kk);
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          oe[r][0] = fmaf(xv[r].x, s0v.x, fmaf(xv[r].y, s0v.y, fmaf(xv[r].z, s0v.z, fmaf(xv[r].w, s0v.w, oe[r][0]))));
          oe[r][1] = fmaf(xv[r].x, s1v.x, fmaf(xv[r].y, s1v.y, fmaf(xv[r].z, s1v.z, fmaf(xv[r].w, s1v.w, oe[r][1]))));
        }
      }
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int i = ty + 16 * r;
        if (i < L) {
          const float f = REVERSE ? pw[L - 1 - i] : a.scale * pw[i + 1];
          T* row = out + ((t0 + i) * a.H + h) * (long long)DK + row0;
          row[tx] = from_f<T>(fmaf(f, oe[r][0], oi[r][0]));
          row[tx + 16] = from_f<T>(fmaf(f, oe[r][1], oi[r][1]));
        }
      }
    }
    __syncthreads();
    {  // state rows ty, ty + 16: lambda^L S + sum_j w_j Z_j[row] Y_j
      float acc[2][3][4];
      const float lamL = pw[L];
#pragma unroll
      for (int r = 0; r < 2; ++r)
#pragma unroll
        for (int m = 0; m < 3; ++m) {
          const float4 sv = ld4(Ss + (ty + 16 * r) * XP + 4 * tx + 64 * m);
          acc[r][m][0] = lamL * sv.x;
          acc[r][m][1] = lamL * sv.y;
          acc[r][m][2] = lamL * sv.z;
          acc[r][m][3] = lamL * sv.w;
        }
      for (int j = 0; j < L; ++j) {
        const float w = REVERSE ? a.scale * pw[j + 1] : pw[L - 1 - j];
        const float z0 = w * Zs[j * ZP + ty], z1 = w * Zs[j * ZP + ty + 16];
#pragma unroll
        for (int m = 0; m < 3; ++m) {
          const float4 yv = ld4(Ys + j * XP + 4 * tx + 64 * m);
          acc[0][m][0] = fmaf(z0, yv.x, acc[0][m][0]);
          acc[0][m][1] = fmaf(z0, yv.y, acc[0][m][1]);
          acc[0][m][2] = fmaf(z0, yv.z, acc[0][m][2]);
          acc[0][m][3] = fmaf(z0, yv.w, acc[0][m][3]);
          acc[1][m][0] = fmaf(z1, yv.x, acc[1][m][0]);
          acc[1][m][1] = fmaf(z1, yv.y, acc[1][m][1]);
          acc[1][m][2] = fmaf(z1, yv.z, acc[1][m][2]);
          acc[1][m][3] = fmaf(z1, yv.w, acc[1][m][3]);
        }
      }
#pragma unroll
      for (int r = 0; r < 2; ++r)
#pragma unroll
        for (int m = 0; m < 3; ++m)
          st4(Ss + (ty + 16 * r) * XP + 4 * tx + 64 * m, make_float4(acc[r][m][0], acc[r][m][1], acc[r][m][2], acc[r][m][3]));
    }
    __syncthreads();
  }
  if (REVERSE && a.hT) {  // dh0
    for (int e = tid; e < BQ_TILE * DV; e += NT) {
      const int r = e / DV, c = e % DV;
      a.hT[sbase + (long long)(row0 + r) * DV + c] = Ss[r * XP + c];
    }
  }
}

template <class K>
cudaError_t launch(K kernel, int tiles, size_t smem, const ChunkArgs& a, cudaStream_t stream) {
  const long long blocks = (long long)a.n_seq * a.H * tiles;
  if (blocks == 0) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kernel<<<(unsigned)blocks, NT, smem, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_simt_fwd(const ChunkArgs& a, cudaStream_t stream) {
  return launch(simt_wide_kernel<float, false>, FWD_TILES, FWD_SMEM, a, stream);
}

// The fp32 mode's backward (bf16 inputs go through the tensor-core scans).
cudaError_t launch_simt_bwd(int dtype_f32, const ChunkArgs& a, cudaStream_t stream) {
  if (!dtype_f32) return cudaErrorInvalidValue;
  cudaError_t e = launch(simt_bwd_narrow_kernel<float, false>, BQ_TILES, BQ_SMEM, a, stream);
  if (e == cudaSuccess) e = launch(simt_bwd_narrow_kernel<float, true>, BQ_TILES, BQ_SMEM, a, stream);
  if (e == cudaSuccess) e = launch(simt_wide_kernel<float, true>, FWD_TILES, FWD_SMEM, a, stream);
  return e;
}

}  // namespace gla
