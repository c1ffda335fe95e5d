// qwm_kmeans: Lloyd's k-means that builds the high-precision centroids QSAC
// assigns keys to (roboind article on QuantWM, "Step 1": "each Key is
// assigned to a clustering center ... the center retaining high accuracy").
//
// Per iteration:
//   assign   nearest centroid in float32 squared Euclidean distance (lowest
//            index on a tie).  Same thread layout as the append kernel: thread
//            (key, 32-channel group), centroids staged in shared memory as
//            float32, partial distances combined with two shuffles.
//   update   float64 sums of the assigned keys (atomics) and counts, then
//            centroid = float32(sum / count); a centroid without keys keeps its
//            position.
// The result is rounded to the configured dtype (nearest even).
#include "qwm_internal.cuh"

namespace qwm {
namespace {

constexpr unsigned kFullMask = 0xffffffffu;

template <int D, typename T>
__global__ void km_init_kernel(const T* __restrict__ keys, int64_t n, const int32_t* __restrict__ rows,
                               int nC, float* __restrict__ cf) {
  const int h = blockIdx.y;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < (int64_t)nC * D;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int j = (int)(i / D), c = (int)(i % D);
    int64_t r = rows[(int64_t)h * nC + j];
    r = r < 0 ? 0 : (r >= n ? n - 1 : r);
    cf[((int64_t)h * nC + j) * D + c] = load_elem(keys, ((int64_t)h * n + r) * D + c);
  }
}

template <int D, typename T>
__global__ void __launch_bounds__(kTile * (D / kGroup))
km_assign_kernel(const T* __restrict__ keys, int64_t n, const float* __restrict__ cf, int nC,
                 int32_t* __restrict__ assign) {
  constexpr int G = D / kGroup;
  constexpr int NT = kTile * G;
  constexpr int TPW = 32 / G;
  constexpr int CH = 16384 / D;
  extern __shared__ __align__(16) float cs[];   // [CH][D]
  const int h = blockIdx.y;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int gi = lane / TPW, ti = lane % TPW;
  const int t = warp * TPW + ti;
  const int64_t tok = (int64_t)blockIdx.x * kTile + t;
  const bool valid = tok < n;
  float kx[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) kx[i] = valid ? load_elem(keys, ((int64_t)h * n + tok) * D + gi * kGroup + i) : 0.f;
  float best = INFINITY;
  int bj = 0;
  const float* ch = cf + (int64_t)h * nC * D;
  for (int c0 = 0; c0 < nC; c0 += CH) {
    const int cn = min(CH, nC - c0);
    __syncthreads();
    for (int i = threadIdx.x; i < cn * D; i += NT) cs[i] = ch[(int64_t)c0 * D + i];
    __syncthreads();
#pragma unroll 1
    for (int j = 0; j < cn; ++j) {
      const float4* cp = reinterpret_cast<const float4*>(cs + j * D + gi * kGroup);
      float s0 = 0.f, s1 = 0.f;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const float4 a = cp[q];
        const float d0 = kx[4 * q] - a.x, d1 = kx[4 * q + 1] - a.y;
        const float d2 = kx[4 * q + 2] - a.z, d3 = kx[4 * q + 3] - a.w;
        s0 = fmaf(d0, d0, s0);
        s1 = fmaf(d1, d1, s1);
        s0 = fmaf(d2, d2, s0);
        s1 = fmaf(d3, d3, s1);
      }
      float s = s0 + s1;
      s += __shfl_xor_sync(kFullMask, s, TPW);
      if (G == 4) s += __shfl_xor_sync(kFullMask, s, 2 * TPW);
      if (s < best) {
        best = s;
        bj = c0 + j;
      }
    }
  }
  if (valid && gi == 0) assign[(int64_t)h * n + tok] = bj;
}

template <int D, typename T>
__global__ void km_accumulate_kernel(const T* __restrict__ keys, int64_t n, const int32_t* __restrict__ assign,
                                     int nC, double* __restrict__ sums, int32_t* __restrict__ counts) {
  const int h = blockIdx.y;
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;   // over n * D
  if (i >= n * D) return;
  const int64_t tok = i / D;
  const int c = (int)(i % D);
  const int a = assign[(int64_t)h * n + tok];
  atomicAdd(&sums[((int64_t)h * nC + a) * D + c], (double)load_elem(keys, ((int64_t)h * n + tok) * D + c));
  if (c == 0) atomicAdd(&counts[(int64_t)h * nC + a], 1);
}

template <int D>
__global__ void km_finalize_kernel(const double* __restrict__ sums, const int32_t* __restrict__ counts,
                                   int nC, float* __restrict__ cf) {
  const int h = blockIdx.y;
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (int64_t)nC * D) return;
  const int j = (int)(i / D);
  const int cnt = counts[(int64_t)h * nC + j];
  if (cnt > 0) cf[(int64_t)h * nC * D + i] = (float)(sums[(int64_t)h * nC * D + i] / (double)cnt);
}

template <typename T>
__global__ void km_output_kernel(const float* __restrict__ cf, int64_t total, T* __restrict__ out) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= total) return;
  if constexpr (sizeof(T) == 4) out[i] = cf[i];
  else out[i] = __float2bfloat16_rn(cf[i]);
}

struct KmLayout {
  size_t cf, sums, counts, assign, bytes;
};

KmLayout km_layout(int64_t H, int64_t d, int64_t C, int64_t n) {
  KmLayout L;
  auto al = [](size_t x) { return (x + 255) & ~size_t(255); };
  L.cf = 0;
  L.sums = al(L.cf + (size_t)H * C * d * 4);
  L.counts = al(L.sums + (size_t)H * C * d * 8);
  L.assign = al(L.counts + (size_t)H * C * 4);
  L.bytes = al(L.assign + (size_t)H * n * 4);
  return L;
}

template <int D, typename T>
cudaError_t run(int H, int nC, const void* keys, int64_t n, const int32_t* rows, int iters, void* out,
                uint8_t* ws, cudaStream_t st) {
  const KmLayout L = km_layout(H, D, nC, n);
  float* cf = (float*)(ws + L.cf);
  double* sums = (double*)(ws + L.sums);
  int32_t* counts = (int32_t*)(ws + L.counts);
  int32_t* assign = (int32_t*)(ws + L.assign);
  const T* k = (const T*)keys;
  km_init_kernel<D, T><<<dim3((unsigned)((nC * D + 255) / 256), H), 256, 0, st>>>(k, n, rows, nC, cf);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  constexpr int CH = 16384 / D;
  const size_t smem = (size_t)CH * D * 4;
  e = cudaFuncSetAttribute(km_assign_kernel<D, T>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  for (int it = 0; it < iters; ++it) {
    km_assign_kernel<D, T><<<dim3((unsigned)((n + kTile - 1) / kTile), H), kTile * (D / kGroup), smem, st>>>(
        k, n, cf, nC, assign);
    e = cudaMemsetAsync(sums, 0, (size_t)H * nC * D * 8, st);
    if (e == cudaSuccess) e = cudaMemsetAsync(counts, 0, (size_t)H * nC * 4, st);
    if (e != cudaSuccess) return e;
    km_accumulate_kernel<D, T><<<dim3((unsigned)((n * D + 255) / 256), H), 256, 0, st>>>(k, n, assign, nC, sums,
                                                                                         counts);
    km_finalize_kernel<D><<<dim3((unsigned)((nC * D + 255) / 256), H), 256, 0, st>>>(sums, counts, nC, cf);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  const int64_t total = (int64_t)H * nC * D;
  km_output_kernel<T><<<(unsigned)((total + 255) / 256), 256, 0, st>>>(cf, total, (T*)out);
  return cudaGetLastError();
}

}  // namespace
}  // namespace qwm

extern "C" size_t qwm_kmeans_workspace_bytes(int32_t heads, int32_t head_dim, int32_t n_centroids, int64_t n) {
  if (heads < 1 || head_dim < 1 || n_centroids < 1 || n < 1) return 0;
  return qwm::km_layout(heads, head_dim, n_centroids, n).bytes;
}

extern "C" qwm_status qwm_kmeans(int32_t heads, int32_t head_dim, int32_t dtype, int32_t n_centroids,
                                 const void* d_keys, int64_t n, const int32_t* d_init_rows, int32_t iters,
                                 void* d_centroids, void* d_workspace, void* stream) {
  using namespace qwm;
  if (heads < 1 || n_centroids < 1 || n_centroids > 1024 || n < 1 || iters < 0) return QWM_ERR_INVALID_ARG;
  if (head_dim != 64 && head_dim != 128) return QWM_ERR_UNSUPPORTED;
  if (dtype != QWM_F32 && dtype != QWM_BF16) return QWM_ERR_INVALID_ARG;
  if (!d_keys || !d_init_rows || !d_centroids || !d_workspace) return QWM_ERR_INVALID_ARG;
  if ((uintptr_t)d_workspace & 255) return QWM_ERR_INVALID_ARG;
  if (fault_injected("launch")) return QWM_ERR_CUDA;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* ws = (uint8_t*)d_workspace;
  cudaError_t e;
  if (head_dim == 128)
    e = dtype == QWM_BF16 ? run<128, __nv_bfloat16>(heads, n_centroids, d_keys, n, d_init_rows, iters, d_centroids, ws, st)
                          : run<128, float>(heads, n_centroids, d_keys, n, d_init_rows, iters, d_centroids, ws, st);
  else
    e = dtype == QWM_BF16 ? run<64, __nv_bfloat16>(heads, n_centroids, d_keys, n, d_init_rows, iters, d_centroids, ws, st)
                          : run<64, float>(heads, n_centroids, d_keys, n, d_init_rows, iters, d_centroids, ws, st);
  return e == cudaSuccess ? QWM_OK : QWM_ERR_CUDA;
}
