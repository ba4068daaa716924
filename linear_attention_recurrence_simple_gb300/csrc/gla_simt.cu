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
// Forward.  Tile = 64 columns of d_v (3 tiles).
// ------------------------------------------------------------------------------------------
constexpr int FWD_TILE = 64;
constexpr int FWD_TILES = DV / FWD_TILE;
constexpr size_t FWD_SMEM = sizeof(float) * (2 * SC * PK + 2 * SC * PT + DK * PT + SC + 1);

template <class T>
__global__ void __launch_bounds__(NT) simt_fwd_kernel(ChunkArgs a) {
  extern __shared__ float sm[];
  float* Qs = sm;                 // [SC][PK]
  float* Ks = Qs + SC * PK;       // [SC][PK]
  float* Vs = Ks + SC * PK;       // [SC][PT]   column tile of v
  float* Ps = Vs + SC * PT;       // [SC][PT]   decayed, masked scale*q.k
  float* Ss = Ps + SC * PT;       // [DK][PT]   state tile
  float* pw = Ss + DK * PT;       // [SC + 1]
  const int tid = threadIdx.x;
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
    Ss[r * PT + c] = a.h0 ? a.h0[sbase + (long long)r * DV + col0 + c] : 0.f;
  }
  __syncthreads();

  for (long long t0 = tb; t0 < te; t0 += SC) {
    const int L = (int)(te - t0 < SC ? te - t0 : SC);
    if (!rows_in_bounds(a, t0, L)) break;  // (debug-bounds build; uniform over the CTA)
    load_rows(Qs, PK, q, t0, L, a.H, h, DK, 0, DK);
    load_rows(Ks, PK, k, t0, L, a.H, h, DK, 0, DK);
    load_rows(Vs, PT, v, t0, L, a.H, h, DV, col0, FWD_TILE);
    __syncthreads();
    {  // P[i][j] = scale lambda^(i-j) q_i.k_j for j <= i; with aug_balance the diagonal also
       // carries the self-augmentation gate sigmoid(q_i . (a_h * k_i)), so that the row's output
       // gains that multiple of v_i
      const int i = tid / 4;
      for (int m = 0; m < SC / 4; ++m) {
        const int j = (tid % 4) + 4 * m;
        float acc = 0.f;
        if (j <= i) {
#pragma unroll 8
          for (int c = 0; c < DK; ++c) acc = fmaf(Qs[i * PK + c], Ks[j * PK + c], acc);
          acc *= a.scale * pw[i - j];
          if (a.aug && j == i) {
            float g = 0.f;
            for (int c = 0; c < DK; ++c) g = fmaf(Qs[i * PK + c] * a.aug[h * DK + c], Ks[i * PK + c], g);
            acc += 1.f / (1.f + expf(-g));
          }
        }
        Ps[i * PT + j] = acc;
      }
    }
    __syncthreads();
    {  // o_i = sum_j P[i][j] v_j + scale lambda^(i+1) S^T q_i
      const int i = tid / 4, cb = tid % 4;
      float intra[16], inter[16];
#pragma unroll
      for (int m = 0; m < 16; ++m) intra[m] = inter[m] = 0.f;
      for (int j = 0; j <= i; ++j) {
        const float p = Ps[i * PT + j];
#pragma unroll
        for (int m = 0; m < 16; ++m) intra[m] = fmaf(p, Vs[j * PT + cb + 4 * m], intra[m]);
      }
      for (int c = 0; c < DK; ++c) {
        const float qc = Qs[i * PK + c];
#pragma unroll
        for (int m = 0; m < 16; ++m) inter[m] = fmaf(qc, Ss[c * PT + cb + 4 * m], inter[m]);
      }
      if (i < L) {
        const float f = a.scale * pw[i + 1];
        T* orow = o + ((t0 + i) * a.H + h) * (long long)DV + col0;
#pragma unroll
        for (int m = 0; m < 16; ++m) orow[cb + 4 * m] = from_f<T>(fmaf(f, inter[m], intra[m]));
      }
    }
    __syncthreads();
    // S <- lambda^L S + sum_j lambda^(L-1-j) k_j v_j^T
    for (int e = tid; e < DK * FWD_TILE; e += NT) {
      const int r = e / FWD_TILE, c = e % FWD_TILE;
      float acc = pw[L] * Ss[r * PT + c];
      for (int j = 0; j < L; ++j) acc = fmaf(pw[L - 1 - j] * Ks[j * PK + r], Vs[j * PT + c], acc);
      Ss[r * PT + c] = acc;
    }
    __syncthreads();
  }
  if (a.hT) {
    for (int e = tid; e < DK * FWD_TILE; e += NT) {
      const int r = e / FWD_TILE, c = e % FWD_TILE;
      a.hT[sbase + (long long)r * DV + col0 + c] = Ss[r * PT + c];
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
