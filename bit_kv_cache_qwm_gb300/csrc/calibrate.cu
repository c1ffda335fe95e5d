// qwm_calibrate: historical-query sensitivity and the PSAC principal basis.
//
// QuantWM Abstract: QSAC weighs channels by "historical Query sensitivity";
// PSAC corrects key errors "along the dominant Query subspace using low-rank
// projections".  roboind article, "Step 2": the energy of historical queries
// concentrates in a few directions.
//
// 1. gram_kernel: partial Gram matrices Q^T Q of 128-row blocks (float32
//    FMA, fixed order), one CTA per (head, row block).
// 2. gram_sum_kernel: adds the partials in split order (many CTAs) and writes
//    s_c = G_cc / n_h.
// 3. square_kernel: A^2 = (G scale + 2^-20 I)^2 tile by tile (the scale makes
//    the mean eigenvalue 1).
// 4. eig_kernel, one CTA per head: the top-r eigenvectors of G by block
//    subspace iteration on A^2 (start block = unit vectors of the largest
//    diagonal entries; modified Gram-Schmidt once per step, twice before a
//    convergence check), a Rayleigh-Ritz check after kFirstCheck steps and
//    then every kCheckEvery (parallel cyclic Jacobi on the projected matrix),
//    and on the converged Ritz vectors one more Gram-Schmidt pass and
//    Rayleigh-Ritz pass, which restores orthogonality to float32 precision.
//    When r + oversample exceeds 64 the whole matrix goes through Jacobi
//    instead.  Every loop has a fixed bound; a miss of the residual tolerance
//    sets QWM_DEV_NOT_CONVERGED.
// 5. weights_kernel: w_g = s_{32g} + ... + s_{32g+31}, left to right in
//    float32 (an input of the centroid decision).
#include <math.h>
#include <string.h>

#include <mutex>

#include <cuda.h>

#include "qwm_internal.cuh"

namespace qwm {
namespace {

constexpr int kRowsPerSplit = 128;
constexpr int kMaxSplits = 32;
constexpr int kEigThreads = 256;
// A^2 iterations before the first Rayleigh-Ritz check, and between later
// checks.  A check costs about as much as three A^2 steps (the first, from
// unrotated vectors, five Jacobi sweeps), and the kernel takes as long as its
// slowest head: on the synthetic calibrations (1,024 to 4,096 historical
// queries, r = 16, 16 extra columns) the slowest head converges after 5 to 6
// steps, so one check at 6 replaces checks at 4 and 6.
constexpr int kFirstCheck = 6;
constexpr int kCheckEvery = 2;
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

// The eigen-solver works on A = G * scale + shift * I (unit mean eigenvalue,
// eigenvectors unchanged); every kernel forms A through this expression.
__device__ __forceinline__ float scaled_entry(float g, float scale, bool diag) {
  return __fmaf_rn(g, scale, diag ? kShift : 0.f);
}

// trace(G) in a fixed order (thread c holds G_cc, warp butterfly, then the
// warp partials left to right), so that every kernel derives the same scale.
// G row-major d x d; blockDim.x >= D.
template <int D>
__device__ float gram_trace(const float* G, float* red /* [blockDim/32] */) {
  const int tid = threadIdx.x;
  float t = tid < D ? G[(size_t)tid * (D + 1)] : 0.f;
  t = warp_sum(t);
  if ((tid & 31) == 0) red[tid >> 5] = t;
  __syncthreads();
  float tr = 0.f;
  for (int i = 0; i < (int)(blockDim.x >> 5); ++i) tr += red[i];
  __syncthreads();
  return tr;
}

__device__ __forceinline__ float scale_of(float trace, int d) { return trace > 0.f ? (float)d / trace : 1.f; }

// ------------------------------------------------- Gram sum and A^2 kernels
// Sums each head's split partials in split order into split 0, which then
// holds G, and writes s_c = G_cc / n_h.  A thread owns 4 consecutive entries.
__global__ void __launch_bounds__(256) gram_sum_kernel(float* __restrict__ part, int splits, int d,
                                                       int64_t n_h, float* __restrict__ s_out) {
  const int h = blockIdx.x;
  const int dd = d * d;
  const int q4 = blockIdx.y * blockDim.x + threadIdx.x;
  if (q4 * 4 >= dd) return;
  float4* p = reinterpret_cast<float4*>(part + (size_t)h * splits * dd) + q4;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int sp = 0; sp < splits; ++sp) {
    const float4 v = p[(size_t)sp * (dd / 4)];
    acc.x += v.x;
    acc.y += v.y;
    acc.z += v.z;
    acc.w += v.w;
  }
  *p = acc;
  const float e[4] = {acc.x, acc.y, acc.z, acc.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int idx = q4 * 4 + i;
    if (idx / d == idx % d) s_out[(size_t)h * d + idx % d] = __fdiv_rn(e[i], (float)n_h);
  }
}

// One 32 x 32 tile of A^2 per CTA (grid: heads x (D/32)^2), A formed from G
// on the fly: A2_ij = sum_l A_il A_lj, float32 FMA in l order.
template <int D>
__global__ void __launch_bounds__(256) square_kernel(const float* __restrict__ part, int splits,
                                                     float* __restrict__ A2) {
  constexpr int T = D / 32;
  __shared__ float ai[32][D + 1];
  __shared__ float aj[32][D + 1];
  __shared__ float red[8];
  const int h = blockIdx.x, ti = blockIdx.y / T, tj = blockIdx.y % T, tid = threadIdx.x;
  const float* G = part + (size_t)h * splits * D * D;
  const float scale = scale_of(gram_trace<D>(G, red), D);
  for (int idx = tid; idx < 32 * D; idx += blockDim.x) {
    const int rr = idx / D, l = idx % D;
    const int gi = 32 * ti + rr, gj = 32 * tj + rr;
    ai[rr][l] = scaled_entry(G[(size_t)gi * D + l], scale, gi == l);
    aj[rr][l] = scaled_entry(G[(size_t)gj * D + l], scale, gj == l);
  }
  __syncthreads();
  const int i = tid >> 3, j0 = (tid & 7) * 4;
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 8
  for (int l = 0; l < D; ++l) {
    const float a = ai[i][l];
#pragma unroll
    for (int b = 0; b < 4; ++b) acc[b] = fmaf(a, aj[j0 + b][l], acc[b]);
  }
  float* out = A2 + ((size_t)h * D + 32 * ti + i) * D + 32 * tj + j0;
  *reinterpret_cast<float4*>(out) = make_float4(acc[0], acc[1], acc[2], acc[3]);
}

// ------------------------------------------------------------------ Jacobi
// Round-robin pairing of ne (even) indices at step k: pair 0 = (ne-1, k),
// pair a = ((k+a) mod (ne-1), (k-a) mod (ne-1)).  Every index is in one pair
// per step, every pair meets once per sweep.
__device__ __forceinline__ void rr_pair(int ne, int k, int a, int* p, int* q) {
  const int mm = ne - 1;
  if (a == 0) {
    *p = mm;
    *q = k;
  } else {
    int pp = k + a, qq = k - a;
    if (pp >= mm) pp -= mm;
    if (qq < 0) qq += mm;
    *p = pp;
    *q = qq;
  }
}

// A rotation of pair (p, q) is due when |A_pq| > 2^-20 sqrt(|A_pp A_qq|),
// tested as A_pq^2 > 2^-40 |A_pp A_qq|: float32 rounding keeps smaller
// off-diagonals alive forever.
__device__ __forceinline__ bool rotation_due(float apq, float app, float aqq) {
  return apq * apq > 9.094947017729282e-13f * fabsf(app * aqq);
}

// The rotation of pair (p, q) of the symmetric matrix A: t = -sign(th) /
// (|th| + sqrt(th^2 + 1)), th = (A_pp - A_qq) / (2 A_pq), c = 1/sqrt(1+t^2),
// s = t c; J = [[c, s], [-s, c]] zeroes A'_pq of J^T A J.  Skipped (c = 1,
// s = 0, false) for the padding index (>= n) or when no rotation is due.
// Fast reciprocal and reciprocal square root: their few-ulp errors leave
// c^2 + s^2 within about 1e-7 of 1, and the final Rayleigh-Ritz pass runs on
// re-orthonormalised vectors.
__device__ __forceinline__ bool jacobi_rotation(const float* A, int lda, int n, int p, int q, float* c,
                                                float* s) {
  *c = 1.f;
  *s = 0.f;
  if (p >= n || q >= n) return false;
  const float app = A[p * lda + p], aqq = A[q * lda + q], apq = A[p * lda + q];
  if (!rotation_due(apq, app, aqq)) return false;
  const float th = __fdividef(app - aqq, 2.f * apq);
  const float r2 = fmaf(th, th, 1.f);
  const float t = __fdividef(th >= 0.f ? -1.f : 1.f, fabsf(th) + r2 * rsqrtf(r2));
  *c = rsqrtf(fmaf(t, t, 1.f));
  *s = t * *c;
  return true;
}

// R = J1^T M J2 for the 2 x 2 block M = A[(p1, q1), (p2, q2)].
__device__ __forceinline__ void rotate_block(const float* A, float* B, int ld, int n, int p1, int q1, float c1,
                                             float s1, int p2, int q2, float c2, float s2) {
  const bool vp1 = p1 < n, vq1 = q1 < n, vp2 = p2 < n, vq2 = q2 < n;
  const float m00 = (vp1 && vp2) ? A[p1 * ld + p2] : 0.f;
  const float m01 = (vp1 && vq2) ? A[p1 * ld + q2] : 0.f;
  const float m10 = (vq1 && vp2) ? A[q1 * ld + p2] : 0.f;
  const float m11 = (vq1 && vq2) ? A[q1 * ld + q2] : 0.f;
  const float t00 = c1 * m00 - s1 * m10, t01 = c1 * m01 - s1 * m11;
  const float t10 = s1 * m00 + c1 * m10, t11 = s1 * m01 + c1 * m11;
  if (vp1 && vp2) B[p1 * ld + p2] = t00 * c2 - t01 * s2;
  if (vp1 && vq2) B[p1 * ld + q2] = t00 * s2 + t01 * c2;
  if (vq1 && vp2) B[q1 * ld + p2] = t10 * c2 - t11 * s2;
  if (vq1 && vq2) B[q1 * ld + q2] = t10 * s2 + t11 * c2;
}

// True when some off-diagonal entry of the symmetric n x n matrix A is still
// above the rotation threshold (the same test as jacobi_rotation).  Block-wide.
__device__ bool offdiag_alive(const float* A, int lda, int n) {
  int alive = 0;
  for (int idx = threadIdx.x; idx < n * n; idx += blockDim.x) {
    const int p = idx / n, q = idx - p * n;
    if (q <= p) continue;
    alive |= rotation_due(A[p * lda + q], A[p * lda + p], A[q * lda + q]);
  }
  return __syncthreads_or(alive) != 0;
}

// Parallel cyclic Jacobi for n <= 64 (at most 32 pairs a step), rotations
// accumulated into V (caller initialises it).  In each step lane l of every
// warp derives the rotation of pair l from the current matrix and the warp
// exchanges them by shuffles; the matrix is double-buffered (every thread
// writes its rotated 2 x 2 blocks into the other buffer and rotates its
// entries of V in place), so a step costs one block barrier.  The annihilated
// entries of each rotated pair are set to zero.  A sweep starts only while
// some off-diagonal entry is above the threshold.  Returns the buffer holding
// the result.
constexpr int kJacMaxBlk = 4;   // (32 pairs)^2 / 256 threads
constexpr int kJacMaxV = 8;     // 64 rows x 32 pairs / 256 threads

__device__ float* jacobi_db(float* Ha, float* Hb, int ldh, float* V, int ldv, int n, int max_sweeps,
                            int* sweeps) {
  const int ne = n + (n & 1), half = ne >> 1, mm = ne - 1;
  const int tid = threadIdx.x, nt = blockDim.x, lane = tid & 31;
  const int nblk = half * half, nvi = n * half;
  const int nbit = (nblk + nt - 1) / nt, nvit = (nvi + nt - 1) / nt;   // block-uniform trip counts
  // this thread's blocks (a, b) and V entries (row i, pair a), fixed for the call
  int ba[kJacMaxBlk], bb[kJacMaxBlk], vi[kJacMaxV], va[kJacMaxV];
#pragma unroll
  for (int it = 0; it < kJacMaxBlk; ++it) {
    const int idx = tid + it * nt;
    ba[it] = idx < nblk ? idx / half : -1;
    bb[it] = idx < nblk ? idx - (idx / half) * half : 0;
  }
#pragma unroll
  for (int it = 0; it < kJacMaxV; ++it) {
    const int idx = tid + it * nt;
    vi[it] = idx < nvi ? idx / half : -1;
    va[it] = idx < nvi ? idx - (idx / half) * half : 0;
  }
  float* cur = Ha;
  float* nxt = Hb;
  int sweep = 0;
  for (; sweep < max_sweeps; ++sweep) {
    if (!offdiag_alive(cur, ldh, n)) break;
    for (int k = 0; k < mm; ++k) {
      float c = 1.f, s = 0.f;
      int p = ne, q = ne;
      if (lane < half) {
        rr_pair(ne, k, lane, &p, &q);
        jacobi_rotation(cur, ldh, n, p, q, &c, &s);
      }
#pragma unroll
      for (int it = 0; it < kJacMaxBlk; ++it) {
        if (it >= nbit) break;
        const int a = ba[it] < 0 ? 0 : ba[it], b = bb[it];
        const float c1 = __shfl_sync(0xffffffffu, c, a), s1 = __shfl_sync(0xffffffffu, s, a);
        const float c2 = __shfl_sync(0xffffffffu, c, b), s2 = __shfl_sync(0xffffffffu, s, b);
        const int p1 = __shfl_sync(0xffffffffu, p, a), q1 = __shfl_sync(0xffffffffu, q, a);
        const int p2 = __shfl_sync(0xffffffffu, p, b), q2 = __shfl_sync(0xffffffffu, q, b);
        if (ba[it] >= 0) {
          rotate_block(cur, nxt, ldh, n, p1, q1, c1, s1, p2, q2, c2, s2);
          if (a == b && s1 != 0.f) {
            nxt[p1 * ldh + q1] = 0.f;
            nxt[q1 * ldh + p1] = 0.f;
          }
        }
      }
#pragma unroll
      for (int it = 0; it < kJacMaxV; ++it) {
        if (it >= nvit) break;
        const int a = va[it];
        const float c1 = __shfl_sync(0xffffffffu, c, a), s1 = __shfl_sync(0xffffffffu, s, a);
        const int p1 = __shfl_sync(0xffffffffu, p, a), q1 = __shfl_sync(0xffffffffu, q, a);
        if (vi[it] >= 0 && s1 != 0.f) {
          const int i = vi[it];
          const float vp = V[i * ldv + p1], vq = V[i * ldv + q1];
          V[i * ldv + p1] = c1 * vp - s1 * vq;
          V[i * ldv + q1] = s1 * vp + c1 * vq;
        }
      }
      __syncthreads();
      float* t = cur;
      cur = nxt;
      nxt = t;
    }
  }
  *sweeps = sweep;
  return cur;
}

// The same sweeps for larger n, in place: the rotations of a step go through
// a shared table (rot: 2 floats, prs: 2 ints per pair), two barriers a step.
__device__ int jacobi_table(float* A, int lda, float* V, int ldv, int n, int max_sweeps, float* rot,
                            int* prs) {
  const int ne = n + (n & 1), half = ne / 2;
  const int tid = threadIdx.x, nt = blockDim.x;
  int sweep = 0;
  for (; sweep < max_sweeps; ++sweep) {
    int rotated = 0;
    for (int k = 0; k < ne - 1; ++k) {
      for (int a = tid; a < half; a += nt) {
        int p, q;
        float c, s;
        rr_pair(ne, k, a, &p, &q);
        rotated |= jacobi_rotation(A, lda, n, p, q, &c, &s);
        rot[2 * a] = c;
        rot[2 * a + 1] = s;
        prs[2 * a] = p;
        prs[2 * a + 1] = q;
      }
      __syncthreads();
      for (int idx = tid; idx < half * half; idx += nt) {
        const int a = idx / half, b = idx % half;
        const int p1 = prs[2 * a], q1 = prs[2 * a + 1], p2 = prs[2 * b], q2 = prs[2 * b + 1];
        // in place: each 2 x 2 block is read and written by one thread only
        rotate_block(A, A, lda, n, p1, q1, rot[2 * a], rot[2 * a + 1], p2, q2, rot[2 * b], rot[2 * b + 1]);
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

__device__ float* jacobi(float* Ha, float* Hb, int ldh, float* V, int ldv, int n, int max_sweeps, float* rot,
                         int* prs, int* sweeps) {
  if (n <= 64) return jacobi_db(Ha, Hb, ldh, V, ldv, n, max_sweeps, sweeps);
  *sweeps = jacobi_table(Ha, ldh, V, ldv, n, max_sweeps, rot, prs);
  return Ha;
}

// --------------------------------------------------------- Gram-Schmidt
template <int J>
__device__ __forceinline__ void normalise_publish(float (&v)[J], float* cb, int lane) {
  float s2 = 0.f;
#pragma unroll
  for (int jj = 0; jj < J; ++jj) s2 = fmaf(v[jj], v[jj], s2);
  s2 = warp_sum(s2);
  const float inv = s2 > 0.f ? 1.f / sqrtf(s2) : 0.f;
#pragma unroll
  for (int jj = 0; jj < J; ++jj) {
    v[jj] *= inv;
    cb[lane + 32 * jj] = v[jj];
  }
}

// 1/sqrt(x) for x > 0: the hardware estimate and one Newton step.
__device__ __forceinline__ float rsqrt_nr(float x) {
  const float y = rsqrtf(x);
  return y * fmaf(-0.5f * x * y, y, 1.5f);
}

// Modified Gram-Schmidt, twice, on the m <= 8C columns of Xin (d rows,
// leading dim ldx), result in Xout (which may be Xin).  Column k lives in the
// registers of warp k % 8 (d/32 values per lane).  In step j every warp
// projects all its later columns against the published column j; the owner
// of column j+1, then final, normalises it and publishes it through a
// double-buffered shared row: one block barrier per column and pass.  The
// squared norm of column j+1 rides in the same interleaved warp reductions as
// the projection coefficients, and the norm after the update follows from
// ||v - f u||^2 = ||v||^2 - f^2 (u a unit vector); where that difference
// cancels (below 1e-4 ||v||^2) the norm is summed again from the vector.
template <int D, int C>
__device__ void mgs2(const float* Xin, float* Xout, int ldx, int m, float* colbuf /* [2][D] */, int passes) {
  constexpr int J = D / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float v[C][J];
#pragma unroll
  for (int c = 0; c < C; ++c) {
    const int k = warp + 8 * c;
#pragma unroll
    for (int j = 0; j < J; ++j) v[c][j] = k < m ? Xin[(lane + 32 * j) * ldx + k] : 0.f;
  }
  if (warp == 0) normalise_publish<J>(v[0], colbuf, lane);
  int step = 0;
  for (int pass = 0; pass < passes; ++pass) {
    for (int j = 0; j < m; ++j, ++step) {
      int nx = j + 1;
      if (nx == m) nx = pass + 1 < passes ? 0 : -1;
      const int sel = nx >= 0 ? nx >> 3 : 0;
      const bool owner = nx >= 0 && warp == (nx & 7);
      __syncthreads();
      const float* cb = colbuf + (step & 1) * D;
      float u[J];
#pragma unroll
      for (int jj = 0; jj < J; ++jj) u[jj] = cb[lane + 32 * jj];
      // register selects of slot sel (an indexed register array would live
      // in local memory)
      float w[J];
#pragma unroll
      for (int jj = 0; jj < J; ++jj) w[jj] = v[0][jj];
#pragma unroll
      for (int c = 1; c < C; ++c)
#pragma unroll
        for (int jj = 0; jj < J; ++jj) w[jj] = c == sel ? v[c][jj] : w[jj];
      float dt[C + 1];
#pragma unroll
      for (int c = 0; c < C; ++c) {
        dt[c] = 0.f;
#pragma unroll
        for (int jj = 0; jj < J; ++jj) dt[c] = fmaf(u[jj], v[c][jj], dt[c]);
      }
      dt[C] = 0.f;
#pragma unroll
      for (int jj = 0; jj < J; ++jj) dt[C] = fmaf(w[jj], w[jj], dt[C]);
#pragma unroll
      for (int o = 16; o; o >>= 1)
#pragma unroll
        for (int c = 0; c <= C; ++c) dt[c] += __shfl_xor_sync(0xffffffffu, dt[c], o);
      float fsel = 0.f;
#pragma unroll
      for (int c = 0; c < C; ++c) {
        const int k = warp + 8 * c;
        const float f = (k > j && k < m) ? dt[c] : 0.f;
        fsel = c == sel ? f : fsel;
#pragma unroll
        for (int jj = 0; jj < J; ++jj) v[c][jj] = fmaf(-f, u[jj], v[c][jj]);
      }
      if (owner) {
#pragma unroll
        for (int jj = 0; jj < J; ++jj) w[jj] = v[0][jj];
#pragma unroll
        for (int c = 1; c < C; ++c)
#pragma unroll
          for (int jj = 0; jj < J; ++jj) w[jj] = c == sel ? v[c][jj] : w[jj];
        float n2 = fmaf(-fsel, fsel, dt[C]);
        if (__any_sync(0xffffffffu, !(n2 > 1e-4f * dt[C]))) {
          n2 = 0.f;
#pragma unroll
          for (int jj = 0; jj < J; ++jj) n2 = fmaf(w[jj], w[jj], n2);
          n2 = warp_sum(n2);
        }
        const float inv = n2 > 0.f ? rsqrt_nr(n2) : 0.f;
        float* nb = colbuf + ((step + 1) & 1) * D;
#pragma unroll
        for (int jj = 0; jj < J; ++jj) {
          w[jj] *= inv;
          nb[lane + 32 * jj] = w[jj];
        }
#pragma unroll
        for (int c = 0; c < C; ++c)
#pragma unroll
          for (int jj = 0; jj < J; ++jj) v[c][jj] = c == sel ? w[jj] : v[c][jj];
      }
    }
  }
#pragma unroll
  for (int c = 0; c < C; ++c) {
    const int k = warp + 8 * c;
    if (k < m) {
#pragma unroll
      for (int j = 0; j < J; ++j) Xout[(lane + 32 * j) * ldx + k] = v[c][j];
    }
  }
  __syncthreads();
}

// Modified Gram-Schmidt, twice, in place, for m > 64 columns (the whole-
// matrix path; used once per calibration).
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

// passes = 2 (MGS twice: orthogonal to float32 precision) before a
// Rayleigh-Ritz pass; 1 between checks, where the basis only has to stay well
// conditioned, and on Ritz vectors that are orthonormal up to rounding.
template <int D>
__device__ void orthonormalise(const float* Xin, float* Xout, int ldx, int m, float* colbuf, float* tmp,
                               int passes) {
  if (m <= 32) mgs2<D, 4>(Xin, Xout, ldx, m, colbuf, passes);
  else if (m <= 64) mgs2<D, 8>(Xin, Xout, ldx, m, colbuf, passes);
  else mgs2_block(Xout, ldx, D, m, tmp);   // whole-matrix path: Xin == Xout
}

// ------------------------------------------------------------ small products
// W (D x m) = B X for a symmetric D x D matrix B, read by rows (B_li = B_il).
// A thread computes rows ri, ri+32, ... of 4 consecutive columns: the lanes
// of a warp read 32 consecutive entries of a row of B and the same entries of
// X (broadcast).  kScaledG: B is the Gram matrix G in global memory and A is
// formed entry by entry.
template <int D, bool kScaledG>
__device__ void mm_bx(const float* B, int ldb, float scale, const float* X, int ldx, float* W, int ldw, int m) {
  constexpr int R = D / 32;
  const int ntiles = 32 * ((m + 3) >> 2);
  for (int tile = threadIdx.x; tile < ntiles; tile += blockDim.x) {
    const int ri = tile & 31, c0 = (tile >> 5) * 4;
    float acc[R][4];
#pragma unroll
    for (int a = 0; a < R; ++a)
#pragma unroll
      for (int b = 0; b < 4; ++b) acc[a][b] = 0.f;
#pragma unroll 4
    for (int l = 0; l < D; ++l) {
      float xb[4], br[R];
#pragma unroll
      for (int b = 0; b < 4; ++b) xb[b] = c0 + b < m ? X[l * ldx + c0 + b] : 0.f;
#pragma unroll
      for (int a = 0; a < R; ++a) {
        const int i = ri + 32 * a;
        if constexpr (kScaledG) br[a] = scaled_entry(__ldg(B + (size_t)l * ldb + i), scale, l == i);
        else br[a] = B[l * ldb + i];
      }
#pragma unroll
      for (int a = 0; a < R; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b) acc[a][b] = fmaf(br[a], xb[b], acc[a][b]);
    }
#pragma unroll
    for (int a = 0; a < R; ++a)
#pragma unroll
      for (int b = 0; b < 4; ++b)
        if (c0 + b < m) W[(ri + 32 * a) * ldw + c0 + b] = acc[a][b];
  }
  __syncthreads();
}

// Y (D x m) = X V[:, order]: the Ritz vectors in descending Ritz value order.
// Same tiling as mm_bx; the lanes read 32 different rows of X (odd leading
// dimension: no bank conflicts) and the same entries of V.
template <int D>
__device__ void mm_rot(const float* X, int ldx, const float* V, int ldv, const int* order, float* Y, int ldy,
                       int m) {
  constexpr int R = D / 32;
  const int ntiles = 32 * ((m + 3) >> 2);
  for (int tile = threadIdx.x; tile < ntiles; tile += blockDim.x) {
    const int ri = tile & 31, c0 = (tile >> 5) * 4;
    int oc[4];
#pragma unroll
    for (int b = 0; b < 4; ++b) oc[b] = c0 + b < m ? order[c0 + b] : 0;
    float acc[R][4];
#pragma unroll
    for (int a = 0; a < R; ++a)
#pragma unroll
      for (int b = 0; b < 4; ++b) acc[a][b] = 0.f;
#pragma unroll 4
    for (int k = 0; k < m; ++k) {
      float xr[R], vb[4];
#pragma unroll
      for (int a = 0; a < R; ++a) xr[a] = X[(ri + 32 * a) * ldx + k];
#pragma unroll
      for (int b = 0; b < 4; ++b) vb[b] = V[k * ldv + oc[b]];
#pragma unroll
      for (int a = 0; a < R; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b) acc[a][b] = fmaf(xr[a], vb[b], acc[a][b]);
    }
#pragma unroll
    for (int a = 0; a < R; ++a)
#pragma unroll
      for (int b = 0; b < 4; ++b)
        if (c0 + b < m) Y[(ri + 32 * a) * ldy + c0 + b] = acc[a][b];
  }
  __syncthreads();
}

// H (m x m) = (X^T W + W^T X) / 2.  P = X^T W first (a thread computes a
// 2 x 2 block of P, four dot products over the d rows in row order), then
// H_ab = (P_ab + P_ba) / 2.  P goes through the scratch matrix Pm.
__device__ void project(const float* X, int ldx, const float* W, int ldw, float* H, float* Pm, int ldh, int d,
                        int m) {
  const int nb = (m + 1) >> 1;
  for (int blk = threadIdx.x; blk < nb * nb; blk += blockDim.x) {
    const int a0 = 2 * (blk / nb), b0 = 2 * (blk % nb);
    const bool a1 = a0 + 1 < m, b1 = b0 + 1 < m;
    float s00 = 0.f, s01 = 0.f, s10 = 0.f, s11 = 0.f;
    for (int i = 0; i < d; ++i) {
      const float x0 = X[i * ldx + a0], x1 = a1 ? X[i * ldx + a0 + 1] : 0.f;
      const float w0 = W[i * ldw + b0], w1 = b1 ? W[i * ldw + b0 + 1] : 0.f;
      s00 = fmaf(x0, w0, s00);
      s01 = fmaf(x0, w1, s01);
      s10 = fmaf(x1, w0, s10);
      s11 = fmaf(x1, w1, s11);
    }
    Pm[a0 * ldh + b0] = s00;
    if (b1) Pm[a0 * ldh + b0 + 1] = s01;
    if (a1) Pm[(a0 + 1) * ldh + b0] = s10;
    if (a1 && b1) Pm[(a0 + 1) * ldh + b0 + 1] = s11;
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < m * m; idx += blockDim.x) {
    const int a = idx / m, b = idx % m;
    H[a * ldh + b] = 0.5f * (Pm[a * ldh + b] + Pm[b * ldh + a]);
  }
  __syncthreads();
}

// order = indices of diag(H) in descending order (ties: lower index first),
// theta = the sorted diagonal.
__device__ void sort_diag(const float* H, int ldh, int m, float* theta, int* order) {
  for (int i = threadIdx.x; i < m; i += blockDim.x) {
    const float hi = H[i * ldh + i];
    int rank = 0;
    for (int j = 0; j < m; ++j) {
      const float hj = H[j * ldh + j];
      rank += (hj > hi) || (hj == hi && j < i);
    }
    order[rank] = i;
  }
  __syncthreads();
  for (int k = threadIdx.x; k < m; k += blockDim.x) theta[k] = H[order[k] * ldh + order[k]];
  __syncthreads();
}

__device__ void set_identity(float* V, int ldv, int m) {
  for (int idx = threadIdx.x; idx < m * m; idx += blockDim.x)
    V[(idx / m) * ldv + idx % m] = (idx / m == idx % m) ? 1.f : 0.f;
  __syncthreads();
}

// Buffers of the eigen-solver for one head, as float offsets: A^2 (subspace
// path only), A itself when the whole set still fits in shared memory (else
// the Rayleigh-Ritz products read G from global memory), the d x m blocks X,
// W, T and the m x m matrices H0, H1, V.
constexpr size_t kEigSmemLimit = 220 * 1024;

struct EigLayout {
  int ldx, ldh, m;
  bool a_region;
  size_t a2, a, x, w, t, h0, h1, v, floats;
};

__host__ __device__ inline EigLayout eig_layout(int d, int m) {
  EigLayout L;
  L.m = m;
  L.ldx = m + 1;
  L.ldh = m + 1;
  const size_t sq = (size_t)d * (d + 1);
  const size_t rest = 3 * (size_t)d * L.ldx + 3 * (size_t)m * L.ldh;
  L.a_region = m < d && (2 * sq + rest) * 4 <= kEigSmemLimit;
  L.a2 = 0;
  L.a = L.a2 + (m < d ? sq : 0);
  L.x = L.a + (L.a_region ? sq : 0);
  L.w = L.x + (size_t)d * L.ldx;
  L.t = L.w + (size_t)d * L.ldx;
  L.h0 = L.t + (size_t)d * L.ldx;
  L.h1 = L.h0 + (size_t)m * L.ldh;
  L.v = L.h1 + (size_t)m * L.ldh;
  L.floats = L.v + (size_t)m * L.ldh;
  return L;
}

// One CTA per head: the top-r eigenvectors of A = G * scale + shift.
//   m < d: block subspace iteration on A^2 (from the square kernel, held in
//     shared memory) from unit vectors at the m largest diagonal entries,
//     orthonormalised by MGS every step (twice before a check); after
//     kFirstCheck steps and then every kCheckEvery steps a Rayleigh-Ritz pass
//     on A (Jacobi on X^T A X) and the residual test of the leading r Ritz
//     pairs.
//   m = d: Jacobi on the whole matrix.
// Then the final Ritz vectors are re-orthonormalised and put through one more
// Rayleigh-Ritz pass, which restores orthogonality to float32 precision.
template <int D>
__global__ void __launch_bounds__(kEigThreads, 1)
eig_kernel(const float* __restrict__ part, int splits, const float* __restrict__ A2g, int r, int m,
           int max_iter, float* __restrict__ U_out, float* __restrict__ lam_out, float* __restrict__ energy_out,
           int32_t* __restrict__ iters_out, uint32_t* __restrict__ status, float* __restrict__ gws,
           int use_smem) {
  extern __shared__ __align__(16) float smem[];
  __shared__ float rot[2 * (D / 2)];
  __shared__ int prs[2 * (D / 2)];
  __shared__ float colbuf[2 * D];
  __shared__ float theta[D];
  __shared__ int order[D];
  __shared__ float red[kEigThreads / 32];
  __shared__ float tmp[2];
  const int h = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const float* G = part + (size_t)h * splits * D * D;
  const float trace = gram_trace<D>(G, red);
  if (r == 0) {
    if (tid == 0) {
      energy_out[h] = 0.f;
      iters_out[h] = 0;
    }
    return;
  }
  const float scale = scale_of(trace, D);
  const EigLayout L = eig_layout(D, m);
  const int ldx = L.ldx, ldh = L.ldh;
  float* base = use_smem ? smem : gws + (size_t)h * L.floats;
  float* X = base + L.x;
  float* W = base + L.w;
  float* T = base + L.t;
  float* H0 = base + L.h0;
  float* H1 = base + L.h1;
  float* V = base + L.v;
  float* As = base + L.a;
  // W = A X for the Rayleigh-Ritz passes
  auto times_a = [&](const float* Xs, float* Ws) {
    if (L.a_region) mm_bx<D, false>(As, D + 1, 1.f, Xs, ldx, Ws, ldx, m);
    else mm_bx<D, true>(G, D, scale, Xs, ldx, Ws, ldx, m);
  };
  int iters = 0, sweeps = 0;
  bool converged = false;
  if (m == D) {
    for (int idx = tid; idx < D * D; idx += blockDim.x) {
      const int i = idx / D, j = idx % D;
      H0[i * ldh + j] = scaled_entry(G[idx], scale, i == j);
    }
    set_identity(V, ldh, D);
    const float* Hc = jacobi(H0, H1, ldh, V, ldh, D, 16, rot, prs, &iters);
    sort_diag(Hc, ldh, D, theta, order);
    for (int idx = tid; idx < D * D; idx += blockDim.x) X[(idx / D) * ldx + idx % D] = V[(idx / D) * ldh + order[idx % D]];
    __syncthreads();
    converged = true;
  } else {
    float* A2s = base + L.a2;
    const float* a2h = A2g + (size_t)h * D * D;
    for (int idx = tid; idx < D * D; idx += blockDim.x) A2s[(idx / D) * (D + 1) + idx % D] = a2h[idx];
    if (L.a_region)
      for (int idx = tid; idx < D * D; idx += blockDim.x) {
        const int i = idx / D, j = idx % D;
        As[i * (D + 1) + j] = scaled_entry(G[idx], scale, i == j);
      }
    // start block: unit vectors at the m largest diagonal entries of G
    for (int i = tid; i < D; i += blockDim.x) {
      const float gi = G[i * (D + 1)];
      int rank = 0;
      for (int j = 0; j < D; ++j) {
        const float gj = G[j * (D + 1)];
        rank += (gj > gi) || (gj == gi && j < i);
      }
      for (int k = 0; k < m; ++k) X[i * ldx + k] = (rank == k) ? 1.f : 0.f;
    }
    __syncthreads();
    while (true) {
      for (int t = 0, n = iters == 0 ? kFirstCheck : kCheckEvery; t < n && iters < max_iter; ++t, ++iters) {
        mm_bx<D, false>(A2s, D + 1, 1.f, X, ldx, W, ldx, m);
        const bool last = t + 1 == n || iters + 1 == max_iter;   // a check follows
        orthonormalise<D>(W, X, ldx, m, colbuf, tmp, last ? 2 : 1);
      }
      // Rayleigh-Ritz on A and the residuals of the leading r Ritz pairs
      times_a(X, W);
      project(X, ldx, W, ldx, H0, H1, ldh, D, m);
      set_identity(V, ldh, m);
      const float* Hc = jacobi(H0, H1, ldh, V, ldh, m, 12, rot, prs, &sweeps);
      sort_diag(Hc, ldh, m, theta, order);
      mm_rot<D>(X, ldx, V, ldh, order, T, ldx, m);
      float* t = X;
      X = T;
      T = t;
      mm_rot<D>(W, ldx, V, ldh, order, T, ldx, m);
      t = W;
      W = T;
      T = t;
      float worst = 0.f;
      for (int k = warp; k < r; k += kEigThreads / 32) {
        float s = 0.f;
        for (int i = lane; i < D; i += 32) {
          const float e = W[i * ldx + k] - theta[k] * X[i * ldx + k];
          s = fmaf(e, e, s);
        }
        worst = fmaxf(worst, sqrtf(warp_sum(s)));
      }
      if (lane == 0) red[warp] = worst;
      __syncthreads();
      float wv = 0.f;
      for (int i = 0; i < kEigThreads / 32; ++i) wv = fmaxf(wv, red[i]);
      __syncthreads();
      converged = wv <= kResidualTol * fabsf(theta[0]);
      if (converged || iters >= max_iter) break;
    }
  }
  // re-orthonormalise and one more Rayleigh-Ritz pass
  orthonormalise<D>(X, X, ldx, m, colbuf, tmp, 1);
  times_a(X, W);
  project(X, ldx, W, ldx, H0, H1, ldh, D, m);
  set_identity(V, ldh, m);
  const float* Hc = jacobi(H0, H1, ldh, V, ldh, m, 4, rot, prs, &sweeps);
  sort_diag(Hc, ldh, m, theta, order);
  mm_rot<D>(X, ldx, V, ldh, order, T, ldx, m);
  X = T;

  // outputs: U rows with the sign rule, eigenvalues unscaled and unshifted
  for (int k = warp; k < r; k += kEigThreads / 32) {
    float best = -1.f;
    int bi = D;
    for (int i = lane; i < D; i += 32) {
      const float a = fabsf(X[i * ldx + k]);
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
    const float sgn = X[bi * ldx + k] < 0.f ? -1.f : 1.f;
    for (int i = lane; i < D; i += 32) U_out[((int64_t)h * r + k) * D + i] = sgn * X[i * ldx + k];
    if (lane == 0) lam_out[h * r + k] = (theta[k] - kShift) / scale;
  }
  __syncthreads();
  if (tid == 0) {
    float e = 0.f;
    for (int k = 0; k < r; ++k) e += (theta[k] - kShift) / scale;
    energy_out[h] = trace > 0.f ? e / trace : 0.f;
    iters_out[h] = iters;
    if (!converged) atomicOr(status, QWM_DEV_NOT_CONVERGED);
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

// Calibration workspace (byte offsets): the Gram partials of every split
// (split 0 of each head ends up holding G), A^2 of every head (subspace path)
// and the eigen-solver's buffers when they do not fit in shared memory.
struct CalibWs {
  size_t part, a2, spill, bytes;
  bool use_smem;
};

CalibWs calib_ws(int H, int d, int m, int splits) {
  auto al = [](size_t x) { return (x + 255) & ~size_t(255); };
  const EigLayout L = eig_layout(d, m);
  CalibWs w;
  w.use_smem = L.floats * 4 <= kEigSmemLimit;
  w.part = 0;
  w.a2 = al(w.part + (size_t)H * splits * d * d * 4);
  w.spill = al(w.a2 + (m < d ? (size_t)H * d * d * 4 : 0));
  w.bytes = al(w.spill + (w.use_smem ? 0 : (size_t)H * L.floats * 4));
  return w;
}

size_t gram_workspace_bytes(const qwm_config& c) {
  return calib_ws(c.heads, c.head_dim, eig_cols(c), splits_for(c.max_hist)).bytes;
}

template <int D>
cudaError_t gram_and_sum(int H, int dtype, const void* q, int64_t n_h, float* part, int splits, int64_t rps,
                         float* s_out, cudaStream_t st) {
  dim3 grid(H, splits);
  if (dtype == QWM_BF16) gram_kernel<D, __nv_bfloat16><<<grid, 256, 0, st>>>((const __nv_bfloat16*)q, n_h, part, splits, rps);
  else gram_kernel<D, float><<<grid, 256, 0, st>>>((const float*)q, n_h, part, splits, rps);
  gram_sum_kernel<<<dim3(H, D * D / 1024), 256, 0, st>>>(part, splits, D, n_h, s_out);
  return cudaGetLastError();
}

template <int D>
cudaError_t square_only(int H, int r, int m, const float* part, int splits, float* a2, cudaStream_t st) {
  if (r > 0 && m < D) square_kernel<D><<<dim3(H, (D / 32) * (D / 32)), 256, 0, st>>>(part, splits, a2);
  return cudaGetLastError();
}

template <int D>
cudaError_t eig_only(int H, int r, int m, int max_iter, const float* part, int splits, float* a2, float* gws,
                     bool use_smem, float* U, float* lam, float* energy, int32_t* iters, uint32_t* status,
                     cudaStream_t st) {
  const size_t smem = use_smem ? eig_layout(D, m).floats * 4 : 0;
  cudaError_t e = cudaFuncSetAttribute(eig_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  eig_kernel<D><<<H, kEigThreads, smem, st>>>(part, splits, a2, r, m, max_iter, U, lam, energy, iters, status,
                                             gws, use_smem ? 1 : 0);
  return cudaGetLastError();
}

template <int D>
cudaError_t square_and_eig(int H, int r, int m, int max_iter, const float* part, int splits, float* a2, float* gws,
                           bool use_smem, float* U, float* lam, float* energy, int32_t* iters, uint32_t* status,
                           cudaStream_t st) {
  cudaError_t e = square_only<D>(H, r, m, part, splits, a2, st);
  if (e != cudaSuccess) return e;
  return eig_only<D>(H, r, m, max_iter, part, splits, a2, gws, use_smem, U, lam, energy, iters, status, st);
}

cudaError_t launch_gram(const qwm_ctx* c, const void* q, int64_t n_h, cudaStream_t st) {
  const int sp = splits_for(n_h);
  const int64_t rps = (n_h + sp - 1) / sp;
  float* part = (float*)c->ws;
  if (c->cfg.head_dim == 128) return gram_and_sum<128>(c->cfg.heads, c->cfg.dtype, q, n_h, part, sp, rps, c->s, st);
  return gram_and_sum<64>(c->cfg.heads, c->cfg.dtype, q, n_h, part, sp, rps, c->s, st);
}

cudaError_t launch_square(const qwm_ctx* c, int64_t n_h, cudaStream_t st) {
  const int D = c->cfg.head_dim, H = c->cfg.heads, r = c->cfg.rank;
  const int m = eig_cols(c->cfg);
  const CalibWs w = calib_ws(H, D, m, splits_for(c->cfg.max_hist));
  const float* part = (const float*)c->ws;
  float* a2 = (float*)(c->ws + w.a2);
  const int sp = splits_for(n_h);
  if (D == 128) return square_only<128>(H, r, m, part, sp, a2, st);
  return square_only<64>(H, r, m, part, sp, a2, st);
}

cudaError_t launch_eig(const qwm_ctx* c, int64_t n_h, int32_t version, cudaStream_t st) {
  const int D = c->cfg.head_dim, H = c->cfg.heads, r = c->cfg.rank;
  const int m = eig_cols(c->cfg);
  const CalibWs w = calib_ws(H, D, m, splits_for(c->cfg.max_hist));
  const float* part = (const float*)c->ws;
  float* a2 = (float*)(c->ws + w.a2);
  float* gws = (float*)(c->ws + w.spill);
  float* U = c->basis + (size_t)version * H * (r > 0 ? r : 1) * D;   // version = basis slot
  const int sp = splits_for(n_h);
  if (D == 128)
    return eig_only<128>(H, r, m, c->cfg.max_iter, part, sp, a2, gws, w.use_smem, U, c->lambda, c->energy,
                         c->iters, c->status, st);
  return eig_only<64>(H, r, m, c->cfg.max_iter, part, sp, a2, gws, w.use_smem, U, c->lambda, c->energy,
                      c->iters, c->status, st);
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
struct ScratchAddr {
  unsigned long long ctx_id;   // driver context the address belongs to
  float* ptr;
};
static ScratchAddr g_scratch_addr[kMaxDevices];
static std::mutex g_scratch_mu;

// The driver's id of the current context (unique for the life of the
// process, unlike the context handle, which a new context may reuse), or 0
// when none is current.  Found through the runtime's driver entry points, so
// the library does not link the driver library itself.
typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);
unsigned long long current_ctx_id() {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static bool looked_up = false;
  if (!looked_up) {
    cudaDriverEntryPointQueryResult q1, q2;
    void* f1 = nullptr;
    void* f2 = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f1, 12000, cudaEnableDefault, &q1) == cudaSuccess &&
        cudaGetDriverEntryPointByVersion("cuCtxGetId", &f2, 12000, cudaEnableDefault, &q2) == cudaSuccess &&
        q1 == cudaDriverEntryPointSuccess && q2 == cudaDriverEntryPointSuccess) {
      get_current = reinterpret_cast<CtxGetCurrentFn>(f1);
      get_id = reinterpret_cast<CtxGetIdFn>(f2);
    }
    looked_up = true;
  }
  CUcontext c = nullptr;
  unsigned long long id = 0;
  if (!get_current || get_current(&c) != CUDA_SUCCESS || !c || get_id(c, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// Device address of the scratch array in the current context.  It is looked
// up once per device and context (host code cannot use the symbol itself as a
// device address); a new context on the device (after cudaDeviceReset, for
// instance) has a new id, so its first call looks the address up again.
cudaError_t static_scratch(float** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  const unsigned long long id = current_ctx_id();
  ScratchAddr& a = g_scratch_addr[dev];
  if (!a.ptr || id == 0 || a.ctx_id != id) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_calib_scratch);   // makes the primary context current if none was
    if (e != cudaSuccess) return e;
    a.ptr = static_cast<float*>(p);
    a.ctx_id = current_ctx_id();
  }
  *out = a.ptr;
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
  // scratch (floats): [status word, iteration counts, padded to 64][A^2][spill][partials]
  const CalibWs w1 = calib_ws(heads, head_dim, m, 1);
  const size_t cap = kStaticScratchBytes / sizeof(float);
  const size_t head_words = (1 + H + 63) & ~size_t(63);
  const size_t a2_words = (w1.spill - w1.a2) / sizeof(float);
  const size_t spill_words = (w1.bytes - w1.spill) / sizeof(float);
  const size_t per_split = H * D * D;
  const size_t fixed = head_words + a2_words + spill_words;
  if (fixed + per_split > cap) return QWM_ERR_CAPACITY;   // too many heads for 8 MiB
  int splits = splits_for(n_h);
  const int fit = (int)((cap - fixed) / per_split);
  if (splits > fit) splits = fit;
  const int64_t rps = (n_h + splits - 1) / splits;
  float* scratch = nullptr;
  if (static_scratch(&scratch) != cudaSuccess) return QWM_ERR_CUDA;
  uint32_t* status_words = reinterpret_cast<uint32_t*>(scratch);
  int32_t* iters = reinterpret_cast<int32_t*>(scratch + 1);
  float* a2 = scratch + head_words;
  float* gws = a2 + a2_words;
  float* part = gws + spill_words;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint32_t* status = d_status ? d_status : status_words;
  if (!d_status && cudaMemsetAsync(status_words, 0, 4, st) != cudaSuccess) return QWM_ERR_CUDA;
  float* lam = rank > 0 ? d_lambda : d_energy;   // not written when rank == 0
  float* U = rank > 0 ? d_U : d_energy;
  cudaError_t e;
  if (head_dim == 128) {
    e = gram_and_sum<128>(heads, dtype, d_q_hist, n_h, part, splits, rps, d_s, st);
    if (e == cudaSuccess)
      e = square_and_eig<128>(heads, rank, m, max_iter, part, splits, a2, gws, w1.use_smem, U, lam, d_energy, iters,
                              status, st);
  } else {
    e = gram_and_sum<64>(heads, dtype, d_q_hist, n_h, part, splits, rps, d_s, st);
    if (e == cudaSuccess)
      e = square_and_eig<64>(heads, rank, m, max_iter, part, splits, a2, gws, w1.use_smem, U, lam, d_energy, iters,
                             status, st);
  }
  return e == cudaSuccess ? QWM_OK : QWM_ERR_CUDA;
}
