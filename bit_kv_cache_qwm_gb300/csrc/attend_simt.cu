// qwm_attend, CUDA-core kernel: the float32 path (and a cross-check of the
// tensor-core kernels for any dtype and any rank 0 <= r <= d).
//
// Attention over the packed cache with PSAC compensation (QuantWM Abstract:
// PSAC "restores the remaining Key errors along the dominant Query subspace
// using low-rank projections"; roboind article, "Step 2"):
//   l_n = q . k_hat_n + (q U_t^T) . e_n,   O = softmax(scale * l) V_hat.
//
// A CTA of 8 warps owns 32 query rows of one head; each warp owns 4 rows.
// Every 128-slot tile is dequantised once per CTA into shared memory
// (k_hat = centroid + zero + code*scale and v_hat = zero + code*scale in
// float32, e in the stored float16).  A lane computes the logits of 4 keys
// with a compensated float32 dot product (Ogita, Rump and Oishi, "Accurate
// sum and dot product", SIAM J. Sci. Comput. 26(6), 2005, algorithm Dot2:
// every product split exactly into a float32 pair by a fused multiply-add,
// the running sum kept with its rounding error), as accurate as a dot product
// in twice the float32 precision, so rounding of the logit stays far below the
// float32 tolerance of the output; softmax
// weights, their sums and the output accumulate in float32 with the running
// maximum subtracted in float64.  q U_t^T is recomputed whenever the basis
// version of the tile changes.
#include <math.h>

#include "qwm_internal.cuh"

namespace qwm {
namespace {

constexpr int kRowsPerWarp = 4;
constexpr int kWarps = 8;
constexpr int kRows = kRowsPerWarp * kWarps;

// one term of Dot2: (hi, lo) += x * y, with the product and the sum split
// exactly (the _rn intrinsics keep the compiler from contracting them)
__device__ __forceinline__ void dot2_step(float x, float y, float& hi, float& lo) {
  const float p = __fmul_rn(x, y);
  const float pe = __fmaf_rn(x, y, -p);          // x * y - p exactly
  const float s = __fadd_rn(hi, p);
  const float z = __fsub_rn(s, hi);
  const float se = __fadd_rn(__fsub_rn(hi, __fsub_rn(s, z)), __fsub_rn(p, z));   // hi + p - s exactly
  hi = s;
  lo = __fadd_rn(lo, __fadd_rn(se, pe));
}

template <int D, typename T>
__global__ void __launch_bounds__(kWarps * 32)
attend_simt_kernel(const T* __restrict__ Q, int64_t M, float scale, T* __restrict__ O,
                   const uint8_t* __restrict__ cache, int64_t max_tiles, TileOffsets off,
                   int64_t n_tiles, const int2* __restrict__ tiles, const T* __restrict__ cent,
                   int nC, const float* __restrict__ basis, int max_versions, int H, int r, int ib,
                   uint32_t* status) {
  constexpr int G = D / kGroup;
  constexpr int J = D / 32;
  extern __shared__ __align__(16) float sm[];
  const int rp = r + 1;
  float* kh = sm;                          // [128][D+1]
  float* vh = kh + kTile * (D + 1);        // [128][D]
  __half* es = reinterpret_cast<__half*>(vh + kTile * D);   // [128][r+1] (fp16, as stored)
  float* qs = vh + kTile * D + (kTile * rp + 1) / 2;         // [kRows][D]
  float* zs = qs + kRows * D;              // [kRows][r]

  const int h = blockIdx.y;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t row0 = (int64_t)blockIdx.x * kRows;

  for (int i = threadIdx.x; i < kRows * D; i += blockDim.x) {
    const int64_t row = row0 + i / D;
    qs[i] = row < M ? load_elem(Q, ((int64_t)h * M + row) * D + i % D) : 0.f;
  }

  double mrow[kRowsPerWarp];
  float lrow[kRowsPerWarp], o[kRowsPerWarp][J];
#pragma unroll
  for (int a = 0; a < kRowsPerWarp; ++a) {
    mrow[a] = -INFINITY;
    lrow[a] = 0.f;
#pragma unroll
    for (int j = 0; j < J; ++j) o[a][j] = 0.f;
  }

  int cur_version = -1;
  const T* ch = cent + (int64_t)h * nC * D;
  for (int64_t t = 0; t < n_tiles; ++t) {
    const int2 meta = tiles[t];
    const int nv = meta.y;
    const uint8_t* tb = cache + ((int64_t)h * max_tiles + t) * off.bytes;
    __syncthreads();
    // ---- dequantise the tile ----
    for (int i = threadIdx.x; i < kTile * G; i += blockDim.x) {
      const int slot = i / G, g = i % G;
      const int idx = cent_index(ib == 1 ? tb[off.idx + slot] : reinterpret_cast<const uint16_t*>(tb + off.idx)[slot], nC, status);
      const uint2 kc = *reinterpret_cast<const uint2*>(tb + off.kcode + slot * (D / 4) + g * 8);
      const uint2 vc = *reinterpret_cast<const uint2*>(tb + off.vcode + slot * (D / 4) + g * 8);
      const __half2 kq = *reinterpret_cast<const __half2*>(tb + off.kqp + (slot * G + g) * 4);
      const __half2 vq = *reinterpret_cast<const __half2*>(tb + off.vqp + (slot * G + g) * 4);
      const float kz = __low2float(kq), ks = __high2float(kq);
      const float vz = __low2float(vq), vs = __high2float(vq);
#pragma unroll 8
      for (int c = 0; c < 32; ++c) {
        const uint32_t kw = c < 16 ? kc.x : kc.y, vw = c < 16 ? vc.x : vc.y;
        const int sh = 2 * (c & 15);
        const float kcode = (float)((kw >> sh) & 3u), vcode = (float)((vw >> sh) & 3u);
        const float cval = load_elem(ch, (int64_t)idx * D + g * 32 + c);
        kh[slot * (D + 1) + g * 32 + c] = cval + (kz + kcode * ks);
        vh[slot * D + g * 32 + c] = vz + vcode * vs;
      }
    }
    for (int i = threadIdx.x; i < kTile * r; i += blockDim.x) {
      const int slot = i / r, m = i % r;
      es[slot * rp + m] = reinterpret_cast<const __half*>(tb + off.e)[slot * r + m];
    }
    // ---- q U^T for a new basis version ----
    if (meta.x != cur_version && r > 0) {
      cur_version = meta.x;
      const float* U = basis + ((int64_t)cur_version * H + h) * r * D;
      for (int i = threadIdx.x; i < kRows * r; i += blockDim.x) {
        const int a = i / r, m = i % r;
        double s = 0.0;
        for (int c = 0; c < D; ++c) s += (double)qs[a * D + c] * (double)U[m * D + c];
        zs[a * r + m] = (float)s;
      }
    }
    __syncthreads();
    // ---- logits, online softmax, accumulation ----
#pragma unroll 1
    for (int a = 0; a < kRowsPerWarp; ++a) {
      const int lr = warp * kRowsPerWarp + a;
      const float* q = qs + lr * D;
      const float* z = zs + lr * r;
      double lg[4];
      double tmax = -INFINITY;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int key = lane + 32 * k;
        float hi = 0.f, lo = 0.f;
        const float* kr = kh + key * (D + 1);
        for (int c = 0; c < D; ++c) dot2_step(q[c], kr[c], hi, lo);
        const __half* er = es + key * rp;
        for (int m = 0; m < r; ++m) dot2_step(z[m], __half2float(er[m]), hi, lo);
        lg[k] = key < nv ? (double)hi + (double)lo : -INFINITY;
        tmax = fmax(tmax, lg[k]);
      }
#pragma unroll
      for (int sh = 16; sh; sh >>= 1) tmax = fmax(tmax, __shfl_xor_sync(0xffffffffu, tmax, sh));
      if (tmax == -INFINITY) continue;     // tile holds no valid key
      const double mnew = fmax(mrow[a], tmax);
      const float corr = mrow[a] == -INFINITY ? 0.f : expf((float)((double)scale * (mrow[a] - mnew)));
      mrow[a] = mnew;
      float p[4];
      float psum = 0.f;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        p[k] = lg[k] == -INFINITY ? 0.f : expf((float)((double)scale * (lg[k] - mnew)));
        psum += p[k];
      }
#pragma unroll
      for (int sh = 16; sh; sh >>= 1) psum += __shfl_xor_sync(0xffffffffu, psum, sh);
      lrow[a] = lrow[a] * corr + psum;
#pragma unroll
      for (int j = 0; j < J; ++j) o[a][j] *= corr;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        for (int src = 0; src < 32; ++src) {
          const float pk = __shfl_sync(0xffffffffu, p[k], src);
          const float* vr = vh + (32 * k + src) * D;
#pragma unroll
          for (int j = 0; j < J; ++j) o[a][j] = fmaf(pk, vr[lane + 32 * j], o[a][j]);
        }
      }
    }
  }
  // ---- normalise and store ----
#pragma unroll
  for (int a = 0; a < kRowsPerWarp; ++a) {
    const int64_t row = row0 + warp * kRowsPerWarp + a;
    if (row >= M) continue;
    const float inv = lrow[a] > 0.f ? 1.f / lrow[a] : 0.f;
#pragma unroll
    for (int j = 0; j < J; ++j) {
      const float v = o[a][j] * inv;
      T* dst = O + ((int64_t)h * M + row) * D + lane + 32 * j;
      if constexpr (sizeof(T) == 4) *reinterpret_cast<float*>(dst) = v;
      else *reinterpret_cast<__nv_bfloat16*>(dst) = __float2bfloat16_rn(v);
    }
  }
}

template <int D, typename T>
cudaError_t launch_t(const qwm_ctx* c, const void* q, int64_t M, float scale, void* out,
                     cudaStream_t st) {
  const int r = c->cfg.rank;
  const size_t smem = ((size_t)kTile * (D + 1) + (size_t)kTile * D + ((size_t)kTile * (r + 1) + 1) / 2 +
                       (size_t)kRows * D + (size_t)kRows * (r > 0 ? r : 1)) * 4;
  auto kern = attend_simt_kernel<D, T>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)((M + kRows - 1) / kRows), (unsigned)c->cfg.heads);
  kern<<<grid, kWarps * 32, smem, st>>>((const T*)q, M, scale, (T*)out, c->cache, c->lay.max_tiles,
                                        tile_offsets(c->lay), c->n_tiles, c->tiles,
                                        (const T*)c->centroids, c->cfg.n_centroids, c->basis,
                                        c->cfg.max_versions, c->cfg.heads, r, c->ib, c->status);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attend_simt(const qwm_ctx* c, const void* q, int64_t M, float scale, void* out,
                               cudaStream_t st) {
  const bool bf = c->cfg.dtype == QWM_BF16;
  if (c->cfg.head_dim == 128)
    return bf ? launch_t<128, __nv_bfloat16>(c, q, M, scale, out, st)
              : launch_t<128, float>(c, q, M, scale, out, st);
  return bf ? launch_t<64, __nv_bfloat16>(c, q, M, scale, out, st)
            : launch_t<64, float>(c, q, M, scale, out, st);
}

}  // namespace qwm
