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
constexpr int PK = DK + 1;      // padded row pitches (bank-conflict-free column walks)
constexpr int PV = DV + 1;
constexpr int PT = 65;

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

template <class T>
__global__ void __launch_bounds__(NT, 2) simt_fwd_kernel(ChunkArgs a) {
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
  const T* q = (const T*)a.q;
  const T* k = (const T*)a.k;
  const T* v = (const T*)a.v;
  T* o = (T*)a.o;
  const long long sbase = ((long long)n * a.H + h) * DK * DV;

  fill_powers(pw, a.log_lambda[h]);
  for (int e = tid; e < DK * FWD_TILE; e += NT) {
    const int r = e / FWD_TILE, c = e % FWD_TILE;
    Ss[r * VP + c] = a.h0 ? a.h0[sbase + (long long)r * DV + col0 + c] : 0.f;
  }
  __syncthreads();

  for (long long t0 = tb; t0 < te; t0 += SC) {
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
    if (t0 + SC < te) {  // the next chunk's rows into L2 during this chunk's arithmetic
      const int Ln = (int)(te - t0 - SC < SC ? te - t0 - SC : SC);
      prefetch_chunk(q, t0 + SC, Ln, a.H, h, DK, (int)sizeof(T), 0, DK);
      prefetch_chunk(k, t0 + SC, Ln, a.H, h, DK, (int)sizeof(T), 0, DK);
      prefetch_chunk(v, t0 + SC, Ln, a.H, h, DV, (int)sizeof(T), col0, FWD_TILE);
    }
    if (a.aug) {  // gate of row i: sigmoid(q_i . (a_h * k_i)), q unscaled; added to P[i][i] below
      if (tid < SC) {
        float g = 0.f;
        for (int c = 0; c < DK; ++c) g = fmaf(Qs[tid * QP + c] * a.aug[h * DK + c], Ks[tid * QP + c], g);
        gs[tid] = 1.f / (1.f + expf(-g));
      }
      __syncthreads();
    }
    {  // P[i][j] = scale lambda^(i-j) q_i . k_j for j <= i, else 0
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
          float p = j <= i ? acc[r][c] * (a.scale * pw[i - j]) : 0.f;
          if (a.aug && j == i) p += gs[i];
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
          const float f = a.scale * pw[i + 1];
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
        const float w = pw[L - 1 - j];
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
  if (a.hT) {
    for (int e = tid; e < DK * FWD_TILE; e += NT) {
      const int r = e / FWD_TILE, c = e % FWD_TILE;
      a.hT[sbase + (long long)r * DV + col0 + c] = Ss[r * VP + c];
    }
  }
}

// ------------------------------------------------------------------------------------------
// Backward, dq: forward-in-time scan.  Tile = 32 rows of d_k (3 tiles); needs all of d_v.
// ------------------------------------------------------------------------------------------
constexpr int BQ_TILE = 32;
constexpr int BQ_TILES = DK / BQ_TILE;
constexpr int PQ = BQ_TILE + 1;
constexpr size_t BQ_SMEM = sizeof(float) * (2 * SC * PV + SC * PQ + BQ_TILE * PV + SC * PT + SC + 1);

template <class T>
__global__ void __launch_bounds__(NT) simt_bwd_dq_kernel(ChunkArgs a) {
  extern __shared__ float sm[];
  float* Vs = sm;                 // [SC][PV]
  float* Gs = Vs + SC * PV;       // [SC][PV]   dO
  float* Ks = Gs + SC * PV;       // [SC][PQ]   k, d_k tile
  float* Ss = Ks + SC * PQ;       // [BQ_TILE][PV]  forward state rows of the tile
  float* Ps = Ss + BQ_TILE * PV;  // [SC][PT]
  float* pw = Ps + SC * PT;
  const int tid = threadIdx.x;
  int n, h, tile;
  unit_of_block(a, BQ_TILES, n, h, tile);
  long long tb, te;
  seq_range(a, n, tb, te);
  if (!unit_in_bounds(a, n, h)) return;  // (debug-bounds build; uniform over the CTA)
  const int row0 = tile * BQ_TILE;
  const T* k = (const T*)a.k;
  const T* v = (const T*)a.v;
  const T* dO = (const T*)a.dO;
  T* dq = (T*)a.o;
  const long long sbase = ((long long)n * a.H + h) * DK * DV;

  fill_powers(pw, a.log_lambda[h]);
  for (int e = tid; e < BQ_TILE * DV; e += NT) {
    const int r = e / DV, c = e % DV;
    Ss[r * PV + c] = a.h0 ? a.h0[sbase + (long long)(row0 + r) * DV + c] : 0.f;
  }
  __syncthreads();
  for (long long t0 = tb; t0 < te; t0 += SC) {
    const int L = (int)(te - t0 < SC ? te - t0 : SC);
    if (!rows_in_bounds(a, t0, L)) break;  // (debug-bounds build; uniform over the CTA)
    load_rows(Vs, PV, v, t0, L, a.H, h, DV, 0, DV);
    load_rows(Gs, PV, dO, t0, L, a.H, h, DV, 0, DV);
    load_rows(Ks, PQ, k, t0, L, a.H, h, DK, row0, BQ_TILE);
    __syncthreads();
    {  // P[i][j] = scale lambda^(i-j) dO_i.v_j, j <= i
      const int i = tid / 4;
      for (int m = 0; m < SC / 4; ++m) {
        const int j = (tid % 4) + 4 * m;
        float acc = 0.f;
        if (j <= i) {
#pragma unroll 8
          for (int c = 0; c < DV; ++c) acc = fmaf(Gs[i * PV + c], Vs[j * PV + c], acc);
          acc *= a.scale * pw[i - j];
        }
        Ps[i * PT + j] = acc;
      }
    }
    __syncthreads();
    {  // dq_i = sum_j P[i][j] k_j + scale lambda^(i+1) S dO_i     (8 outputs per thread)
      const int i = tid / 4, cb = tid % 4;
      float intra[8], inter[8];
#pragma unroll
      for (int m = 0; m < 8; ++m) intra[m] = inter[m] = 0.f;
      for (int j = 0; j <= i; ++j) {
        const float p = Ps[i * PT + j];
#pragma unroll
        for (int m = 0; m < 8; ++m) intra[m] = fmaf(p, Ks[j * PQ + cb + 4 * m], intra[m]);
      }
      for (int c = 0; c < DV; ++c) {
        const float g = Gs[i * PV + c];
#pragma unroll
        for (int m = 0; m < 8; ++m) inter[m] = fmaf(g, Ss[(cb + 4 * m) * PV + c], inter[m]);
      }
      if (i < L) {
        const float f = a.scale * pw[i + 1];
        T* row = dq + ((t0 + i) * a.H + h) * (long long)DK + row0;
#pragma unroll
        for (int m = 0; m < 8; ++m) row[cb + 4 * m] = from_f<T>(fmaf(f, inter[m], intra[m]));
      }
    }
    __syncthreads();
    for (int e = tid; e < BQ_TILE * DV; e += NT) {
      const int r = e / DV, c = e % DV;
      float acc = pw[L] * Ss[r * PV + c];
      for (int j = 0; j < L; ++j) acc = fmaf(pw[L - 1 - j] * Ks[j * PQ + r], Vs[j * PV + c], acc);
      Ss[r * PV + c] = acc;
    }
    __syncthreads();
  }
}

// ------------------------------------------------------------------------------------------
// Backward, dk and dh0: reverse-in-time scan.  Tile = 32 rows of d_k; carry R[rows, all d_v].
// ------------------------------------------------------------------------------------------
template <class T>
__global__ void __launch_bounds__(NT) simt_bwd_dk_kernel(ChunkArgs a) {
  extern __shared__ float sm[];
  float* Vs = sm;                 // [SC][PV]
  float* Gs = Vs + SC * PV;       // [SC][PV]   dO
  float* Qs = Gs + SC * PV;       // [SC][PQ]   q, d_k tile
  float* Rs = Qs + SC * PQ;       // [BQ_TILE][PV]
  float* Bs = Rs + BQ_TILE * PV;  // [SC][PT]   B[i][j] = scale lambda^(j-i) dO_j.v_i, j >= i
  float* pw = Bs + SC * PT;
  const int tid = threadIdx.x;
  int n, h, tile;
  unit_of_block(a, BQ_TILES, n, h, tile);
  long long tb, te;
  seq_range(a, n, tb, te);
  if (!unit_in_bounds(a, n, h)) return;  // (debug-bounds build; uniform over the CTA)
  const int row0 = tile * BQ_TILE;
  const T* q = (const T*)a.q;
  const T* v = (const T*)a.v;
  const T* dO = (const T*)a.dO;
  T* dk = (T*)a.dk;
  const long long sbase = ((long long)n * a.H + h) * DK * DV;

  fill_powers(pw, a.log_lambda[h]);
  for (int e = tid; e < BQ_TILE * DV; e += NT) {
    const int r = e / DV, c = e % DV;
    Rs[r * PV + c] = a.dhT ? a.dhT[sbase + (long long)(row0 + r) * DV + c] : 0.f;
  }
  __syncthreads();
  const long long nchunks = (te - tb + SC - 1) / SC;
  for (long long m0 = nchunks - 1; m0 >= 0; --m0) {
    const long long t0 = tb + m0 * SC;
    const int L = (int)(te - t0 < SC ? te - t0 : SC);
    if (!rows_in_bounds(a, t0, L)) break;  // (debug-bounds build; uniform over the CTA)
    load_rows(Vs, PV, v, t0, L, a.H, h, DV, 0, DV);
    load_rows(Gs, PV, dO, t0, L, a.H, h, DV, 0, DV);
    load_rows(Qs, PQ, q, t0, L, a.H, h, DK, row0, BQ_TILE);
    __syncthreads();
    {
      const int i = tid / 4;
      for (int m = 0; m < SC / 4; ++m) {
        const int j = (tid % 4) + 4 * m;
        float acc = 0.f;
        if (j >= i) {
#pragma unroll 8
          for (int c = 0; c < DV; ++c) acc = fmaf(Gs[j * PV + c], Vs[i * PV + c], acc);
          acc *= a.scale * pw[j - i];
        }
        Bs[i * PT + j] = acc;
      }
    }
    __syncthreads();
    {  // dk_i = sum_{j>=i} B[i][j] q_j + lambda^(L-1-i) R v_i
      const int i = tid / 4, cb = tid % 4;
      if (i < L) {
        float intra[8], inter[8];
#pragma unroll
        for (int m = 0; m < 8; ++m) intra[m] = inter[m] = 0.f;
        for (int j = i; j < SC; ++j) {
          const float b = Bs[i * PT + j];
#pragma unroll
          for (int m = 0; m < 8; ++m) intra[m] = fmaf(b, Qs[j * PQ + cb + 4 * m], intra[m]);
        }
        for (int c = 0; c < DV; ++c) {
          const float vc = Vs[i * PV + c];
#pragma unroll
          for (int m = 0; m < 8; ++m) inter[m] = fmaf(vc, Rs[(cb + 4 * m) * PV + c], inter[m]);
        }
        const float f = pw[L - 1 - i];
        T* row = dk + ((t0 + i) * a.H + h) * (long long)DK + row0;
#pragma unroll
        for (int m = 0; m < 8; ++m) row[cb + 4 * m] = from_f<T>(fmaf(f, inter[m], intra[m]));
      }
    }
    __syncthreads();
    // R <- lambda^L R + scale sum_j lambda^(j+1) q_j dO_j^T
    for (int e = tid; e < BQ_TILE * DV; e += NT) {
      const int r = e / DV, c = e % DV;
      float acc = pw[L] * Rs[r * PV + c];
      for (int j = 0; j < L; ++j) acc = fmaf(a.scale * pw[j + 1] * Qs[j * PQ + r], Gs[j * PV + c], acc);
      Rs[r * PV + c] = acc;
    }
    __syncthreads();
  }
  if (a.hT) {  // dh0
    for (int e = tid; e < BQ_TILE * DV; e += NT) {
      const int r = e / DV, c = e % DV;
      a.hT[sbase + (long long)(row0 + r) * DV + c] = Rs[r * PV + c];
    }
  }
}

// ------------------------------------------------------------------------------------------
// Backward, dv: reverse-in-time scan.  Tile = 64 columns of d_v; carry R[all d_k, columns].
// ------------------------------------------------------------------------------------------
constexpr int BV_TILE = 64;
constexpr int BV_TILES = DV / BV_TILE;
constexpr size_t BV_SMEM = sizeof(float) * (2 * SC * PK + SC * PT + DK * PT + SC * PT + SC + 1);

template <class T>
__global__ void __launch_bounds__(NT) simt_bwd_dv_kernel(ChunkArgs a) {
  extern __shared__ float sm[];
  float* Qs = sm;                 // [SC][PK]
  float* Ks = Qs + SC * PK;       // [SC][PK]
  float* Gs = Ks + SC * PK;       // [SC][PT]  dO column tile
  float* Rs = Gs + SC * PT;       // [DK][PT]
  float* Bs = Rs + DK * PT;       // [SC][PT]  B[i][j] = scale lambda^(j-i) q_j.k_i, j >= i
  float* pw = Bs + SC * PT;
  const int tid = threadIdx.x;
  int n, h, tile;
  unit_of_block(a, BV_TILES, n, h, tile);
  long long tb, te;
  seq_range(a, n, tb, te);
  if (!unit_in_bounds(a, n, h)) return;  // (debug-bounds build; uniform over the CTA)
  const int col0 = tile * BV_TILE;
  const T* q = (const T*)a.q;
  const T* k = (const T*)a.k;
  const T* dO = (const T*)a.dO;
  T* dv = (T*)a.dv;
  const long long sbase = ((long long)n * a.H + h) * DK * DV;

  fill_powers(pw, a.log_lambda[h]);
  for (int e = tid; e < DK * BV_TILE; e += NT) {
    const int r = e / BV_TILE, c = e % BV_TILE;
    Rs[r * PT + c] = a.dhT ? a.dhT[sbase + (long long)r * DV + col0 + c] : 0.f;
  }
  __syncthreads();
  const long long nchunks = (te - tb + SC - 1) / SC;
  for (long long m0 = nchunks - 1; m0 >= 0; --m0) {
    const long long t0 = tb + m0 * SC;
    const int L = (int)(te - t0 < SC ? te - t0 : SC);
    if (!rows_in_bounds(a, t0, L)) break;  // (debug-bounds build; uniform over the CTA)
    load_rows(Qs, PK, q, t0, L, a.H, h, DK, 0, DK);
    load_rows(Ks, PK, k, t0, L, a.H, h, DK, 0, DK);
    load_rows(Gs, PT, dO, t0, L, a.H, h, DV, col0, BV_TILE);
    __syncthreads();
    {
      const int i = tid / 4;
      for (int m = 0; m < SC / 4; ++m) {
        const int j = (tid % 4) + 4 * m;
        float acc = 0.f;
        if (j >= i) {
#pragma unroll 8
          for (int c = 0; c < DK; ++c) acc = fmaf(Qs[j * PK + c], Ks[i * PK + c], acc);
          acc *= a.scale * pw[j - i];
        }
        Bs[i * PT + j] = acc;
      }
    }
    __syncthreads();
    {  // dv_i = sum_{j>=i} B[i][j] dO_j + lambda^(L-1-i) R^T k_i
      const int i = tid / 4, cb = tid % 4;
      if (i < L) {
        float intra[16], inter[16];
#pragma unroll
        for (int m = 0; m < 16; ++m) intra[m] = inter[m] = 0.f;
        for (int j = i; j < SC; ++j) {
          const float b = Bs[i * PT + j];
#pragma unroll
          for (int m = 0; m < 16; ++m) intra[m] = fmaf(b, Gs[j * PT + cb + 4 * m], intra[m]);
        }
        for (int c = 0; c < DK; ++c) {
          const float kc = Ks[i * PK + c];
#pragma unroll
          for (int m = 0; m < 16; ++m) inter[m] = fmaf(kc, Rs[c * PT + cb + 4 * m], inter[m]);
        }
        const float f = pw[L - 1 - i];
        T* row = dv + ((t0 + i) * a.H + h) * (long long)DV + col0;
#pragma unroll
        for (int m = 0; m < 16; ++m) row[cb + 4 * m] = from_f<T>(fmaf(f, inter[m], intra[m]));
      }
    }
    __syncthreads();
    for (int e = tid; e < DK * BV_TILE; e += NT) {
      const int r = e / BV_TILE, c = e % BV_TILE;
      float acc = pw[L] * Rs[r * PT + c];
      for (int j = 0; j < L; ++j) acc = fmaf(a.scale * pw[j + 1] * Qs[j * PK + r], Gs[j * PT + c], acc);
      Rs[r * PT + c] = acc;
    }
    __syncthreads();
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
  return launch(simt_fwd_kernel<float>, FWD_TILES, FWD_SMEM, a, stream);
}

cudaError_t launch_simt_bwd(int dtype_f32, const ChunkArgs& a, cudaStream_t stream) {
  cudaError_t e;
  if (dtype_f32) {
    e = launch(simt_bwd_dq_kernel<float>, BQ_TILES, BQ_SMEM, a, stream);
    if (e == cudaSuccess) e = launch(simt_bwd_dk_kernel<float>, BQ_TILES, BQ_SMEM, a, stream);
    if (e == cudaSuccess) e = launch(simt_bwd_dv_kernel<float>, BV_TILES, BV_SMEM, a, stream);
  } else {
    e = launch(simt_bwd_dq_kernel<__nv_bfloat16>, BQ_TILES, BQ_SMEM, a, stream);
    if (e == cudaSuccess) e = launch(simt_bwd_dk_kernel<__nv_bfloat16>, BQ_TILES, BQ_SMEM, a, stream);
    if (e == cudaSuccess) e = launch(simt_bwd_dv_kernel<__nv_bfloat16>, BV_TILES, BV_SMEM, a, stream);
  }
  return e;
}

}  // namespace gla
