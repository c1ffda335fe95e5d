// qwm_calibrate: historical-query sensitivity and the PSAC principal basis.
//
// QuantWM Abstract: QSAC weighs channels by "historical Query sensitivity";
// PSAC corrects key errors "along the dominant Query subspace using low-rank
// projections".  roboind article, "Step 2": the energy of historical queries
// concentrates in a few directions.
//
// 1. gram_kernel: partial Gram matrices Q^T Q of row blocks (float32 FMA,
//    fixed order), one CTA per (head, row block).
// 2. eig_kernel, one CTA per head: sums the partials in a fixed order, writes
//    s_c = G_cc / n_h, then finds the top-r eigenvectors of G by block
//    subspace iteration on G^2 (start block = unit vectors of the largest
//    diagonal entries, modified Gram-Schmidt twice per step) with a two-pass
//    Rayleigh-Ritz (parallel cyclic Jacobi on the projected matrix, then once
//    more on the re-orthonormalised Ritz vectors, which restores
//    orthogonality to float32 precision).  When r + oversample exceeds 64 the
//    whole matrix goes through Jacobi instead.  Every loop has a fixed bound;
//    a miss of the residual tolerance sets QWM_DEV_NOT_CONVERGED.
// 3. weights_kernel: w_g = s_{32g} + ... + s_{32g+31}, left to right in
//    float32 (an input of the centroid decision).
#include <math.h>
#include <string.h>

#include <mutex>

#include "qwm_internal.cuh"

namespace qwm {
namespace {

constexpr int kRowsPerSplit = 128;
constexpr int kMaxSplits = 32;
constexpr int kEigThreads = 256;
constexpr int kCheckEvery = 2;       // A^2 iterations between Rayleigh-Ritz checks
constexpr float kResidualTol = 2e-6f;
constexpr float kShift = 9.5367431640625e-07f;   // 2^-20 of the mean eigenvalue

int splits_for(int64_t n_h) {
  const int s = (int)((n_h + kRowsPerSplit - 1) / kRowsPerSplit);
  return s < kMaxSplits ? s : kMaxSplits;
}

int eig_cols(const qwm_config& c) {
  int m = c.rank + c.oversample;
  if (m > c.head_dim || m > 64) m = c.head_dim;
  return m;
}

// ------------------------------------------------------------------ Gram
template <int D, typename T>
__global__ void __launch_bounds__(256) gram_kernel(const T* __restrict__ Q, int64_t n_h,
                                                   float* __restrict__ part, int splits,
                                                   int64_t rows_per_split) {
  constexpr int TI = D / 16;           // each thread owns a TI x TI block of G
  __shared__ float qs[32][D];
  const int h = blockIdx.x, sp = blockIdx.y;
  const int ty = threadIdx.x / 16, tx = threadIdx.x % 16;
  float acc[TI][TI];
#pragma unroll
  for (int i = 0; i < TI; ++i)
#pragma unroll
    for (int j = 0; j < TI; ++j) acc[i][j] = 0.f;
  const int64_t r0 = (int64_t)sp * rows_per_split;
  const int64_t r1 = min(n_h, r0 + rows_per_split);
  const T* qh = Q + (int64_t)h * n_h * D;
  for (int64_t rb = r0; rb < r1; rb += 32) {
    const int nr = (int)min((int64_t)32, r1 - rb);
    __syncthreads();
    for (int i = threadIdx.x; i < 32 * D; i += 256) {
      const int rr = i / D, cc = i % D;
      qs[rr][cc] = rr < nr ? load_elem(qh, (rb + rr) * D + cc) : 0.f;
    }
    __syncthreads();
    for (int rr = 0; rr < nr; ++rr) {
      float a[TI], b[TI];
#pragma unroll
      for (int i = 0; i < TI; ++i) {
        a[i] = qs[rr][ty * TI + i];
        b[i] = qs[rr][tx * TI + i];
      }
#pragma unroll
      for (int i = 0; i < TI; ++i)
#pragma unroll
        for (int j = 0; j < TI; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
  }
  float* out = part + ((int64_t)h * splits + sp) * D * D;
#pragma unroll
  for (int i = 0; i < TI; ++i)
#pragma unroll
    for (int j = 0; j < TI; ++j) out[(ty * TI + i) * D + tx * TI + j] = acc[i][j];
}

// ------------------------------------------------------------ block helpers
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Round-robin pairing of n_even indices at step k: pair 0 = (n-1, k), pair a
// = ((k+a) mod (n-1), (k-a) mod (n-1)).  Every index is in one pair per step,
// every pair meets once per sweep.
__device__ __forceinline__ void rr_pair(int ne, int k, int a, int* p, int* q) {
  const int m = ne - 1;
  if (a == 0) {
    *p = ne - 1;
    *q = k % m;
  } else {
    *p = (k + a) % m;
    *q = (k - a + m) % m;
  }
}

// Parallel cyclic Jacobi on the symmetric n x n matrix A (leading dim lda,
// float32), rotations accumulated into V (caller initialises it).  The
// rotation of pair (p, q) uses t = -sign(th)/(|th| + sqrt(th^2+1)),
// th = (A_pp - A_qq)/(2 A_pq), c = 1/sqrt(1+t^2), s = t c, which zeroes
// A'_pq; it is skipped when |A_pq| <= 2^-20 sqrt(|A_pp A_qq|) (float32
// rounding keeps smaller off-diagonals alive forever).  Each step
// updates every 2x2 block (pair a rows, pair b columns) in place.  Returns
// the sweeps used (at most max_sweeps).
__device__ int jacobi(float* A, int lda, float* V, int ldv, int n, int max_sweeps, float* rot,
                      int* prs) {
  const int ne = n + (n & 1), half = ne / 2;
  const int tid = threadIdx.x, nt = blockDim.x;
  int sweep = 0;
  for (; sweep < max_sweeps; ++sweep) {
    int rotated = 0;
    for (int k = 0; k < ne - 1; ++k) {
      for (int a = tid; a < half; a += nt) {
        int p, q;
        rr_pair(ne, k, a, &p, &q);
        float c = 1.f, s = 0.f;
        if (p < n && q < n) {
          const float app = A[p * lda + p], aqq = A[q * lda + q], apq = A[p * lda + q];
          if (apq != 0.f && fabsf(apq) > 9.5367431640625e-07f * sqrtf(fabsf(app * aqq))) {
            const float th = (app - aqq) / (2.f * apq);
            const float t = (th >= 0.f ? -1.f : 1.f) / (fabsf(th) + sqrtf(th * th + 1.f));
            c = 1.f / sqrtf(t * t + 1.f);
            s = t * c;
            rotated = 1;
          }
        }
        rot[2 * a] = c;
        rot[2 * a + 1] = s;
        prs[2 * a] = p;
        prs[2 * a + 1] = q;
      }
      __syncthreads();
      for (int idx = tid; idx < half * half; idx += nt) {
        const int a = idx / half, b = idx % half;
        const int p1 = prs[2 * a], q1 = prs[2 * a + 1], p2 = prs[2 * b], q2 = prs[2 * b + 1];
        const float c1 = rot[2 * a], s1 = rot[2 * a + 1], c2 = rot[2 * b], s2 = rot[2 * b + 1];
        const bool vp1 = p1 < n, vq1 = q1 < n, vp2 = p2 < n, vq2 = q2 < n;
        const float m00 = (vp1 && vp2) ? A[p1 * lda + p2] : 0.f;
        const float m01 = (vp1 && vq2) ? A[p1 * lda + q2] : 0.f;
        const float m10 = (vq1 && vp2) ? A[q1 * lda + p2] : 0.f;
        const float m11 = (vq1 && vq2) ? A[q1 * lda + q2] : 0.f;
        // T = J1^T M, J = [[c, s], [-s, c]]
        const float t00 = c1 * m00 - s1 * m10, t01 = c1 * m01 - s1 * m11;
        const float t10 = s1 * m00 + c1 * m10, t11 = s1 * m01 + c1 * m11;
        // R = T J2
        if (vp1 && vp2) A[p1 * lda + p2] = t00 * c2 - t01 * s2;
        if (vp1 && vq2) A[p1 * lda + q2] = t00 * s2 + t01 * c2;
        if (vq1 && vp2) A[q1 * lda + p2] = t10 * c2 - t11 * s2;
        if (vq1 && vq2) A[q1 * lda + q2] = t10 * s2 + t11 * c2;
      }
      for (int idx = tid; idx < n * half; idx += nt) {
        const int i = idx / half, a = idx % half;
        const int p = prs[2 * a], q = prs[2 * a + 1];
        if (p < n && q < n) {
          const float c = rot[2 * a], s = rot[2 * a + 1];
          const float vp = V[i * ldv + p], vq = V[i * ldv + q];
          V[i * ldv + p] = c * vp - s * vq;
          V[i * ldv + q] = s * vp + c * vq;
        }
      }
      __syncthreads();
    }
    if (!__syncthreads_or(rotated)) break;
  }
  return sweep + 1;
}

// Modified Gram-Schmidt, twice, on the m <= 64 columns of X (d rows, leading
// dim ldx).  Column k lives in the registers of warp k % 8 (d/32 values per
// lane); the owner of column j normalises it and publishes it through a
// double-buffered shared row, then every warp projects its later columns
// against it: one block barrier per column and pass.
template <int D>
__device__ void mgs2(float* X, int ldx, int m, float* colbuf /* [2][D] */) {
  constexpr int J = D / 32;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  float v[8][J];
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const int k = warp + 8 * c;
#pragma unroll
    for (int j = 0; j < J; ++j) v[c][j] = k < m ? X[(lane + 32 * j) * ldx + k] : 0.f;
  }
  int step = 0;
  for (int pass = 0; pass < 2; ++pass) {
    for (int j = 0; j < m; ++j, ++step) {
      float* cb = colbuf + (step & 1) * D;
      if (warp == (j & 7)) {
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          if (c == (j >> 3)) {
            float s2 = 0.f;
#pragma unroll
            for (int jj = 0; jj < J; ++jj) s2 = fmaf(v[c][jj], v[c][jj], s2);
            s2 = warp_sum(s2);
            const float inv = s2 > 0.f ? 1.f / sqrtf(s2) : 0.f;
#pragma unroll
            for (int jj = 0; jj < J; ++jj) {
              v[c][jj] *= inv;
              cb[lane + 32 * jj] = v[c][jj];
            }
          }
        }
      }
      __syncthreads();
      float u[J];
#pragma unroll
      for (int jj = 0; jj < J; ++jj) u[jj] = cb[lane + 32 * jj];
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const int k = warp + 8 * c;
        if (k > j && k < m) {
          float dt = 0.f;
#pragma unroll
          for (int jj = 0; jj < J; ++jj) dt = fmaf(u[jj], v[c][jj], dt);
          dt = warp_sum(dt);
#pragma unroll
          for (int jj = 0; jj < J; ++jj) v[c][jj] = fmaf(-dt, u[jj], v[c][jj]);
        }
      }
    }
  }
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const int k = warp + 8 * c;
    if (k < m) {
#pragma unroll
      for (int j = 0; j < J; ++j) X[(lane + 32 * j) * ldx + k] = v[c][j];
    }
  }
  __syncthreads();
}

// Full-matrix Modified Gram-Schmidt, twice (the m = d path), with block
// barriers; used once per calibration.
__device__ void mgs2_block(float* X, int ldx, int d, int m, float* tmp) {
  const int tid = threadIdx.x, nt = blockDim.x, lane = tid & 31, warp = tid >> 5, nw = nt >> 5;
  for (int pass = 0; pass < 2; ++pass) {
    for (int j = 0; j < m; ++j) {
      if (warp == 0) {
        float s = 0.f;
        for (int i = lane; i < d; i += 32) s = fmaf(X[i * ldx + j], X[i * ldx + j], s);
        s = warp_sum(s);
        if (lane == 0) tmp[0] = s > 0.f ? 1.f / sqrtf(s) : 0.f;
      }
      __syncthreads();
      const float inv = tmp[0];
      for (int i = tid; i < d; i += nt) X[i * ldx + j] *= inv;
      __syncthreads();
      for (int k = j + 1 + warp; k < m; k += nw) {
        float s = 0.f;
        for (int i = lane; i < d; i += 32) s = fmaf(X[i * ldx + j], X[i * ldx + k], s);
        s = warp_sum(s);
        for (int i = lane; i < d; i += 32) X[i * ldx + k] = fmaf(-s, X[i * ldx + j], X[i * ldx + k]);
      }
      __syncthreads();
    }
  }
}

// W (d x m) = A (d x d) X (d x m).  A thread computes rows ri, ri+32,
// ri+64, ri+96 (those below d) of 4 consecutive columns: the 32 lanes of a
// warp read 32 different rows of A (conflict-free with its odd leading dim)
// and the same entries of X (broadcast).
__device__ void matmul_ax(const float* A, int lda, const float* X, int ldx, float* W, int ldw, int d,
                          int m) {
  const int cgroups = (m + 3) / 4;
  for (int tile = threadIdx.x; tile < 32 * cgroups; tile += blockDim.x) {
    const int ri = tile % 32, cg = tile / 32;
    float acc[4][4];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int b = 0; b < 4; ++b) acc[a][b] = 0.f;
    for (int l = 0; l < d; ++l) {
      float xa[4], ar[4];
#pragma unroll
      for (int b = 0; b < 4; ++b) xa[b] = (4 * cg + b < m) ? X[l * ldx + 4 * cg + b] : 0.f;
#pragma unroll
      for (int a = 0; a < 4; ++a) ar[a] = (ri + 32 * a < d) ? A[(ri + 32 * a) * lda + l] : 0.f;
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b) acc[a][b] = fmaf(ar[a], xa[b], acc[a][b]);
    }
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int b = 0; b < 4; ++b)
        if (ri + 32 * a < d && 4 * cg + b < m) W[(ri + 32 * a) * ldw + 4 * cg + b] = acc[a][b];
  }
  __syncthreads();
}

// H (m x m) = X^T W, symmetrised
__device__ void project(const float* X, int ldx, const float* W, int ldw, float* H, int ldh, int d,
                        int m) {
  for (int idx = threadIdx.x; idx < m * m; idx += blockDim.x) {
    const int a = idx / m, b = idx % m;
    if (b < a) continue;
    float s1 = 0.f, s2 = 0.f;
    for (int i = 0; i < d; ++i) {
      s1 = fmaf(X[i * ldx + a], W[i * ldw + b], s1);
      s2 = fmaf(X[i * ldx + b], W[i * ldw + a], s2);
    }
    const float s = 0.5f * (s1 + s2);
    H[a * ldh + b] = s;
    H[b * ldh + a] = s;
  }
  __syncthreads();
}

// X (d x m) <- X V[:, order] with order the descending sort of diag(H);
// theta[k] receives the sorted Ritz values.  Works row by row through a
// per-warp buffer.
__device__ void rotate_sorted(float* X, int ldx, int d, int m, const float* V, int ldv,
                              const float* H, int ldh, float* theta, int* order, float* wbuf) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = blockDim.x >> 5;
  for (int i = tid; i < m; i += blockDim.x) {
    const float hi = H[i * ldh + i];
    int rank = 0;
    for (int j = 0; j < m; ++j) {
      const float hj = H[j * ldh + j];
      rank += (hj > hi) || (hj == hi && j < i);
    }
    order[rank] = i;
  }
  __syncthreads();
  for (int k = tid; k < m; k += blockDim.x) theta[k] = H[order[k] * ldh + order[k]];
  float* buf = wbuf + warp * 128;
  for (int i = warp; i < d; i += nw) {
    for (int k = lane; k < m; k += 32) {
      const int col = order[k];
      float s = 0.f;
      for (int a = 0; a < m; ++a) s = fmaf(X[i * ldx + a], V[a * ldv + col], s);
      buf[k] = s;
    }
    __syncwarp();
    for (int k = lane; k < m; k += 32) X[i * ldx + k] = buf[k];
    __syncwarp();
  }
  __syncthreads();
}

__device__ void set_identity(float* V, int ldv, int m) {
  for (int idx = threadIdx.x; idx < m * m; idx += blockDim.x)
    V[(idx / m) * ldv + idx % m] = (idx / m == idx % m) ? 1.f : 0.f;
  __syncthreads();
}

// Buffers of the eigen-solver for one head, as float offsets.  A2 = A^2 is
// kept only on the subspace path (m < d).
struct EigLayout {
  int ldg, ldm, m;
  size_t g, g2, x, w, h, v, floats;
};

__host__ __device__ inline EigLayout eig_layout(int d, int m) {
  EigLayout L;
  L.m = m;
  L.ldg = d + 1;
  L.ldm = m + 1;
  L.g = 0;
  L.g2 = L.g + (size_t)d * L.ldg;
  L.x = L.g2 + (m < d ? (size_t)d * L.ldg : 0);
  L.w = L.x + (size_t)d * L.ldm;
  L.h = L.w + (size_t)d * L.ldm;
  L.v = L.h + (size_t)m * L.ldm;
  L.floats = L.v + (size_t)m * L.ldm;
  return L;
}

template <int D>
__global__ void __launch_bounds__(kEigThreads, 1)
eig_kernel(const float* __restrict__ part, int splits, int64_t n_h, int r, int m, int max_iter,
           float* __restrict__ s_out, float* __restrict__ U_out, float* __restrict__ lam_out,
           float* __restrict__ energy_out, int32_t* __restrict__ iters_out,
           uint32_t* __restrict__ status, float* __restrict__ gws, int use_smem) {
  extern __shared__ __align__(16) float smem[];
  __shared__ float rot[2 * 66 + 130];
  __shared__ int prs[2 * 66 + 130];
  __shared__ float tmp[4];
  __shared__ float theta[128];
  __shared__ int order[128];
  __shared__ float wbuf[(kEigThreads / 32) * 128];
  __shared__ float red[kEigThreads / 32];
  const int h = blockIdx.x, tid = threadIdx.x;
  const EigLayout L = eig_layout(D, m);
  float* base = use_smem ? smem : gws + (size_t)h * L.floats;
  float* A = base + L.g;
  float* A2 = base + L.g2;
  float* X = base + L.x;
  float* W = base + L.w;
  float* Hm = base + L.h;
  float* V = base + L.v;

  // sum partial Gram matrices in split order
  for (int idx = tid; idx < D * D; idx += blockDim.x) {
    float s = 0.f;
    for (int sp = 0; sp < splits; ++sp) s += part[((int64_t)h * splits + sp) * D * D + idx];
    A[(idx / D) * L.ldg + idx % D] = s;
  }
  __syncthreads();
  // sensitivity and trace
  float tr_part = 0.f;
  for (int c = tid; c < D; c += blockDim.x) {
    const float gcc = A[c * L.ldg + c];
    s_out[h * D + c] = __fdiv_rn(gcc, (float)n_h);
    tr_part += gcc;
  }
  tr_part = warp_sum(tr_part);
  if ((tid & 31) == 0) red[tid >> 5] = tr_part;
  __syncthreads();
  if (tid == 0) {
    float t = 0.f;
    for (int i = 0; i < (int)(blockDim.x >> 5); ++i) t += red[i];
    tmp[1] = t;
  }
  __syncthreads();
  const float trace = tmp[1];
  if (r == 0) {
    if (tid == 0) {
      energy_out[h] = 0.f;
      iters_out[h] = 0;
    }
    return;
  }
  // scale to unit mean eigenvalue and shift: eigenvectors unchanged
  const float scale = trace > 0.f ? (float)D / trace : 1.f;
  for (int idx = tid; idx < D * D; idx += blockDim.x) {
    const int i = idx / D, j = idx % D;
    A[i * L.ldg + j] = A[i * L.ldg + j] * scale + (i == j ? kShift : 0.f);
  }
  __syncthreads();

  int iters = 0;
  bool converged = false;
  const bool full = (m == D);
  if (full) {
    // Jacobi on the whole (scaled) matrix
    for (int idx = tid; idx < D * D; idx += blockDim.x)
      Hm[(idx / D) * L.ldm + idx % D] = A[(idx / D) * L.ldg + idx % D];
    set_identity(X, L.ldm, D);
    set_identity(V, L.ldm, D);
    iters = jacobi(Hm, L.ldm, V, L.ldm, D, 16, rot, prs);
    // X <- V sorted
    set_identity(X, L.ldm, D);
    rotate_sorted(X, L.ldm, D, D, V, L.ldm, Hm, L.ldm, theta, order, wbuf);
  } else {
    // start block: unit vectors at the m largest diagonal entries
    for (int i = tid; i < D; i += blockDim.x) {
      const float gi = A[i * L.ldg + i];
      int rank = 0;
      for (int j = 0; j < D; ++j) {
        const float gj = A[j * L.ldg + j];
        rank += (gj > gi) || (gj == gi && j < i);
      }
      for (int k = 0; k < m; ++k) X[i * L.ldm + k] = (rank == k) ? 1.f : 0.f;
    }
    __syncthreads();
  }

  if (!full) matmul_ax(A, L.ldg, A, L.ldg, A2, L.ldg, D, D);   // iterate on A^2
  while (true) {
    if (!full) {
      for (int t = 0; t < kCheckEvery && iters < max_iter; ++t, ++iters) {
        matmul_ax(A2, L.ldg, X, L.ldm, W, L.ldm, D, m);
        for (int idx = tid; idx < D * m; idx += blockDim.x)
          X[(idx / m) * L.ldm + idx % m] = W[(idx / m) * L.ldm + idx % m];
        __syncthreads();
        mgs2<D>(X, L.ldm, m, wbuf);
      }
      // Rayleigh-Ritz on A, first pass
      matmul_ax(A, L.ldg, X, L.ldm, W, L.ldm, D, m);
      project(X, L.ldm, W, L.ldm, Hm, L.ldm, D, m);
      set_identity(V, L.ldm, m);
      jacobi(Hm, L.ldm, V, L.ldm, m, 12, rot, prs);
      rotate_sorted(X, L.ldm, D, m, V, L.ldm, Hm, L.ldm, theta, order, wbuf);
    }
    // second pass on the re-orthonormalised Ritz vectors
    if (full) mgs2_block(X, L.ldm, D, m, tmp);
    else mgs2<D>(X, L.ldm, m, wbuf);
    matmul_ax(A, L.ldg, X, L.ldm, W, L.ldm, D, m);
    project(X, L.ldm, W, L.ldm, Hm, L.ldm, D, m);
    set_identity(V, L.ldm, m);
    jacobi(Hm, L.ldm, V, L.ldm, m, 4, rot, prs);
    rotate_sorted(X, L.ldm, D, m, V, L.ldm, Hm, L.ldm, theta, order, wbuf);
    rotate_sorted(W, L.ldm, D, m, V, L.ldm, Hm, L.ldm, theta, order, wbuf);
    // residuals of the leading r Ritz pairs
    float worst = 0.f;
    for (int k = tid >> 5; k < r; k += blockDim.x >> 5) {
      float s = 0.f;
      for (int i = tid & 31; i < D; i += 32) {
        const float e = W[i * L.ldm + k] - theta[k] * X[i * L.ldm + k];
        s = fmaf(e, e, s);
      }
      s = warp_sum(s);
      worst = fmaxf(worst, sqrtf(s));
    }
    if ((tid & 31) == 0) red[tid >> 5] = worst;
    __syncthreads();
    if (tid == 0) {
      float wv = 0.f;
      for (int i = 0; i < (int)(blockDim.x >> 5); ++i) wv = fmaxf(wv, red[i]);
      tmp[2] = wv;
    }
    __syncthreads();
    converged = tmp[2] <= kResidualTol * fabsf(theta[0]);
    if (full || converged || iters >= max_iter) break;
  }

  // outputs: U rows with the sign rule, eigenvalues unscaled and unshifted
  for (int k = tid >> 5; k < r; k += blockDim.x >> 5) {
    const int lane = tid & 31;
    float best = -1.f;
    int bi = D;
    for (int i = lane; i < D; i += 32) {
      const float a = fabsf(X[i * L.ldm + k]);
      if (a > best || (a == best && i < bi)) {
        best = a;
        bi = i;
      }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      const float ob = __shfl_xor_sync(0xffffffffu, best, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (ob > best || (ob == best && oi < bi)) {
        best = ob;
        bi = oi;
      }
    }
    const float sgn = X[bi * L.ldm + k] < 0.f ? -1.f : 1.f;
    for (int i = lane; i < D; i += 32) U_out[((int64_t)h * r + k) * D + i] = sgn * X[i * L.ldm + k];
    if (lane == 0) lam_out[h * r + k] = (theta[k] - kShift) / scale;
  }
  __syncthreads();
  if (tid == 0) {
    float e = 0.f;
    for (int k = 0; k < r; ++k) e += (theta[k] - kShift) / scale;
    energy_out[h] = trace > 0.f ? e / trace : 0.f;
    iters_out[h] = iters;
    if (!converged && !full) atomicOr(status, QWM_DEV_NOT_CONVERGED);
  }
}

__global__ void weights_kernel(const float* __restrict__ s, float* __restrict__ w, int HG) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= HG) return;
  const float* p = s + (int64_t)i * kGroup;
  float acc = p[0];
  for (int c = 1; c < kGroup; ++c) acc = __fadd_rn(acc, p[c]);
  w[i] = acc;
}

}  // namespace

size_t gram_workspace_bytes(const qwm_config& c) {
  const size_t part = (size_t)c.heads * splits_for(c.max_hist) * c.head_dim * c.head_dim * 4;
  const EigLayout L = eig_layout(c.head_dim, eig_cols(c));
  return part + 256 + (size_t)c.heads * L.floats * 4;
}

cudaError_t launch_gram(const qwm_ctx* c, const void* q, int64_t n_h, cudaStream_t st) {
  const int sp = splits_for(n_h);
  const int64_t rps = (n_h + sp - 1) / sp;
  dim3 grid(c->cfg.heads, sp);
  float* part = (float*)c->ws;
  if (c->cfg.head_dim == 128) {
    if (c->cfg.dtype == QWM_BF16) gram_kernel<128, __nv_bfloat16><<<grid, 256, 0, st>>>((const __nv_bfloat16*)q, n_h, part, sp, rps);
    else gram_kernel<128, float><<<grid, 256, 0, st>>>((const float*)q, n_h, part, sp, rps);
  } else {
    if (c->cfg.dtype == QWM_BF16) gram_kernel<64, __nv_bfloat16><<<grid, 256, 0, st>>>((const __nv_bfloat16*)q, n_h, part, sp, rps);
    else gram_kernel<64, float><<<grid, 256, 0, st>>>((const float*)q, n_h, part, sp, rps);
  }
  return cudaGetLastError();
}

cudaError_t launch_eig(const qwm_ctx* c, int64_t n_h, int32_t version, cudaStream_t st) {
  const int D = c->cfg.head_dim, H = c->cfg.heads, r = c->cfg.rank;
  const int m = eig_cols(c->cfg);
  const EigLayout L = eig_layout(D, m);
  const size_t part_bytes = (size_t)H * splits_for(c->cfg.max_hist) * D * D * 4;
  float* gws = (float*)(c->ws + ((part_bytes + 255) & ~size_t(255)));
  const size_t bytes = L.floats * 4;
  const int use_smem = bytes <= 210 * 1024;
  const size_t smem = use_smem ? bytes : 0;
  float* U = c->basis + (size_t)version * H * (r > 0 ? r : 1) * D;   // version = basis slot
  const int sp = splits_for(n_h);
  cudaError_t e;
  if (D == 128) {
    e = cudaFuncSetAttribute(eig_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    eig_kernel<128><<<H, kEigThreads, smem, st>>>((const float*)c->ws, sp, n_h, r, m, c->cfg.max_iter,
                                                  c->s, U, c->lambda, c->energy, c->iters, c->status,
                                                  gws, use_smem);
  } else {
    e = cudaFuncSetAttribute(eig_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    eig_kernel<64><<<H, kEigThreads, smem, st>>>((const float*)c->ws, sp, n_h, r, m, c->cfg.max_iter,
                                                 c->s, U, c->lambda, c->energy, c->iters, c->status,
                                                 gws, use_smem);
  }
  return cudaGetLastError();
}

cudaError_t launch_group_weights(const qwm_ctx* c, cudaStream_t st) {
  const int HG = c->cfg.heads * c->G;
  weights_kernel<<<(HG + 127) / 128, 128, 0, st>>>(c->s, c->w, HG);
  return cudaGetLastError();
}

}  // namespace qwm

// ---------------------------------------------------------------------------
// Calibration without any device allocation.
//
// Some callers cannot allocate device memory at all: a plugin whose host
// application owns every byte of device memory through its own pool, or a code
// path that must not call cudaMalloc/cudaFree because those calls can
// synchronise the device.  For them the Gram partial sums of one calibration
// live in the file-scope array below instead of a caller workspace.  Every GPU
// that loads this library holds the array (8 MiB) until the process exits.
// ---------------------------------------------------------------------------
namespace qwm {
namespace {

constexpr size_t kStaticScratchBytes = size_t(8) << 20;
static __device__ __align__(256) float g_calib_scratch[kStaticScratchBytes / sizeof(float)];

constexpr int kMaxDevices = 64;
static float* g_scratch_ptr[kMaxDevices];
static std::mutex g_scratch_mu;

// Device address of the scratch array on the current device, looked up once
// per device (host code cannot use the symbol itself as a device address).
cudaError_t static_scratch(float** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_calib_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = static_cast<float*>(p);
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace qwm

extern "C" qwm_status qwm_calibrate_static(int32_t heads, int32_t head_dim, int32_t rank, int32_t dtype,
                                           int32_t max_iter, int32_t oversample, const void* d_q_hist,
                                           int64_t n_h, float* d_s, float* d_U, float* d_lambda,
                                           float* d_energy, uint32_t* d_status, void* stream) {
  using namespace qwm;
  if (heads < 1 || rank < 0 || rank > head_dim || max_iter < 1 || oversample < 0 || n_h < 1)
    return QWM_ERR_INVALID_ARG;
  if (head_dim != 64 && head_dim != 128) return QWM_ERR_UNSUPPORTED;
  if (dtype != QWM_F32 && dtype != QWM_BF16) return QWM_ERR_INVALID_ARG;
  if (!d_q_hist || !d_s || !d_energy || (rank > 0 && (!d_U || !d_lambda))) return QWM_ERR_INVALID_ARG;
  const size_t D = head_dim, H = heads;
  qwm_config cfg;
  memset(&cfg, 0, sizeof(cfg));
  cfg.heads = heads;
  cfg.head_dim = head_dim;
  cfg.rank = rank;
  cfg.oversample = oversample;
  const int m = eig_cols(cfg);
  const EigLayout L = eig_layout(head_dim, m);
  const bool use_smem = L.floats * 4 <= 210 * 1024;
  // scratch: [64 status/iteration words][spill of the eigen-solver][partials]
  const size_t cap = kStaticScratchBytes / sizeof(float);
  const size_t head_words = 64 + H;
  const size_t spill = use_smem ? 0 : H * L.floats;
  const size_t per_split = H * D * D;
  if (head_words + spill + per_split > cap) return QWM_ERR_CAPACITY;   // too many heads for 8 MiB
  int splits = splits_for(n_h);
  const int fit = (int)((cap - head_words - spill) / per_split);
  if (splits > fit) splits = fit;
  const int64_t rps = (n_h + splits - 1) / splits;
  float* scratch = nullptr;
  if (static_scratch(&scratch) != cudaSuccess) return QWM_ERR_CUDA;
  uint32_t* status_words = reinterpret_cast<uint32_t*>(scratch);
  int32_t* iters = reinterpret_cast<int32_t*>(scratch + 64);
  float* gws = scratch + head_words;
  float* part = gws + spill;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint32_t* status = d_status ? d_status : status_words;
  if (!d_status && cudaMemsetAsync(status_words, 0, 4, st) != cudaSuccess) return QWM_ERR_CUDA;
  dim3 grid(heads, splits);
  if (head_dim == 128) {
    if (dtype == QWM_BF16) gram_kernel<128, __nv_bfloat16><<<grid, 256, 0, st>>>((const __nv_bfloat16*)d_q_hist, n_h, part, splits, rps);
    else gram_kernel<128, float><<<grid, 256, 0, st>>>((const float*)d_q_hist, n_h, part, splits, rps);
  } else {
    if (dtype == QWM_BF16) gram_kernel<64, __nv_bfloat16><<<grid, 256, 0, st>>>((const __nv_bfloat16*)d_q_hist, n_h, part, splits, rps);
    else gram_kernel<64, float><<<grid, 256, 0, st>>>((const float*)d_q_hist, n_h, part, splits, rps);
  }
  if (cudaGetLastError() != cudaSuccess) return QWM_ERR_CUDA;
  const size_t smem = use_smem ? L.floats * 4 : 0;
  float* lam = rank > 0 ? d_lambda : d_energy;   // not written when rank == 0
  float* U = rank > 0 ? d_U : d_energy;
  cudaError_t e;
  if (head_dim == 128) {
    e = cudaFuncSetAttribute(eig_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess)
      eig_kernel<128><<<heads, kEigThreads, smem, st>>>(part, splits, n_h, rank, m, max_iter, d_s, U, lam,
                                                         d_energy, iters, status, gws, use_smem ? 1 : 0);
  } else {
    e = cudaFuncSetAttribute(eig_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess)
      eig_kernel<64><<<heads, kEigThreads, smem, st>>>(part, splits, n_h, rank, m, max_iter, d_s, U, lam,
                                                        d_energy, iters, status, gws, use_smem ? 1 : 0);
  }
  if (e != cudaSuccess || cudaGetLastError() != cudaSuccess) return QWM_ERR_CUDA;
  return QWM_OK;
}
