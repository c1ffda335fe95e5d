// Host side of the libqwm C ABI: argument checks, layout, bookkeeping of
// segments and basis versions, launches.  No torch, no allocation of device
// memory: every device buffer belongs to the caller.
#include <math.h>
#include <string.h>

#include <new>

#include "qwm_internal.cuh"
#include "tcgen05_util.cuh"

using namespace qwm;

namespace {

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

qwm_status check_config(const qwm_config* c) {
  if (!c) return QWM_ERR_INVALID_ARG;
  if (c->heads < 1 || c->group != kGroup) return QWM_ERR_INVALID_ARG;
  if (c->head_dim != 64 && c->head_dim != 128) return QWM_ERR_UNSUPPORTED;
  if (c->rank < 0 || c->rank > c->head_dim) return QWM_ERR_INVALID_ARG;
  if (c->n_centroids < 1 || c->n_centroids > 1024) return QWM_ERR_INVALID_ARG;
  if (c->dtype != QWM_F32 && c->dtype != QWM_BF16) return QWM_ERR_INVALID_ARG;
  if (c->max_tokens < 1 || c->max_versions < 1 || c->max_iter < 1 || c->oversample < 0 ||
      c->max_hist < 1)
    return QWM_ERR_INVALID_ARG;
  return QWM_OK;
}

cudaStream_t S(void* p) { return reinterpret_cast<cudaStream_t>(p); }

qwm_status cuda_status(cudaError_t e) { return e == cudaSuccess ? QWM_OK : QWM_ERR_CUDA; }

// The caller's stream waits for the eigen-solver of the last calibration (a
// no-op once it has finished).
cudaError_t join_eig(const qwm_ctx* x, cudaStream_t s) {
  return x->eig_pending ? cudaStreamWaitEvent(s, x->ev_eig, 0) : cudaSuccess;
}

void release_streams(qwm_ctx* x) {
  if (x->side) cudaStreamSynchronize(x->side);
  if (x->ev_fork) cudaEventDestroy(x->ev_fork);
  if (x->ev_eig) cudaEventDestroy(x->ev_eig);
  if (x->side) cudaStreamDestroy(x->side);
  x->side = nullptr;
  x->ev_fork = x->ev_eig = nullptr;
}

}  // namespace

extern "C" const char* qwm_status_string(qwm_status s) {
  switch (s) {
    case QWM_OK: return "ok";
    case QWM_ERR_INVALID_ARG: return "invalid argument";
    case QWM_ERR_UNSUPPORTED: return "unsupported configuration";
    case QWM_ERR_CAPACITY: return "capacity exhausted (cache tiles or basis versions)";
    case QWM_ERR_NOT_CALIBRATED: return "not calibrated (calibrate and set centroids first)";
    case QWM_ERR_NOT_CONVERGED: return "eigen-solver did not converge within max_iter";
    case QWM_ERR_CUDA: return "CUDA error";
    case QWM_ERR_OOM: return "out of host memory";
    case QWM_ERR_DEVICE: return "device status bits set";
  }
  return "unknown status";
}

extern "C" qwm_status qwm_sizes(const qwm_config* c, qwm_layout* out) {
  qwm_status st = check_config(c);
  if (st != QWM_OK) return st;
  if (!out) return QWM_ERR_INVALID_ARG;
  qwm_layout L;
  memset(&L, 0, sizeof(L));
  const int64_t d = c->head_dim, G = d / kGroup, r = c->rank, H = c->heads;
  const int64_t ib = c->n_centroids <= 256 ? 1 : 2;
  const int64_t esz = c->dtype == QWM_F32 ? 4 : 2;
  L.off_idx = 0;
  L.off_kcode = L.off_idx + kTile * ib;
  L.off_kqp = L.off_kcode + kTile * d / 4;
  L.off_e = L.off_kqp + kTile * G * 4;
  L.off_vcode = L.off_e + kTile * r * 2;
  L.off_vqp = L.off_vcode + kTile * d / 4;
  L.tile_bytes = L.off_vqp + kTile * G * 4;
  L.bytes_per_token = L.tile_bytes / kTile;
  L.max_tiles = (c->max_tokens + kTile - 1) / kTile;
  L.cache_bytes = (size_t)H * L.max_tiles * L.tile_bytes;
  size_t o = 0;
  L.st_status = o;    o = align256(o + 64 * 4);
  L.st_s = o;         o = align256(o + H * d * 4);
  L.st_w = o;         o = align256(o + H * G * 4);
  L.st_lambda = o;    o = align256(o + H * (r > 0 ? r : 1) * 4);
  L.st_energy = o;    o = align256(o + H * 4);
  L.st_centroids = o; o = align256(o + (size_t)H * c->n_centroids * d * esz);
  L.st_basis = o;     o = align256(o + (size_t)c->max_versions * H * (r > 0 ? r : 1) * d * 4);
  L.st_tiles = o;     o = align256(o + (size_t)L.max_tiles * 8);
  L.st_iters = o;     o = align256(o + H * 4);
  if (c->dtype == QWM_BF16) {
    L.st_centroids_f32 = o;
    o = align256(o + (size_t)H * c->n_centroids * d * 4);
  } else {
    L.st_centroids_f32 = L.st_centroids;
  }
  if (c->dtype == QWM_BF16 && d == 128) {
    L.st_centroids_f16 = o;
    o = align256(o + (size_t)H * c->n_centroids * d * 2);
  } else {
    L.st_centroids_f16 = L.st_centroids;
  }
  L.state_bytes = o;
  L.workspace_bytes = align256(small_workspace_offset(*c) + small_workspace_bytes(*c));
  *out = L;
  return QWM_OK;
}

extern "C" qwm_status qwm_create(const qwm_config* c, void* d_cache, void* d_state,
                                 void* d_workspace, qwm_ctx** out) {
  if (!out) return QWM_ERR_INVALID_ARG;
  *out = nullptr;
  qwm_layout L;
  qwm_status st = qwm_sizes(c, &L);
  if (st != QWM_OK) return st;
  if (!d_cache || !d_state || !d_workspace) return QWM_ERR_INVALID_ARG;
  if (((uintptr_t)d_cache | (uintptr_t)d_state | (uintptr_t)d_workspace) & 255)
    return QWM_ERR_INVALID_ARG;
  if (fault_injected("oom")) return QWM_ERR_OOM;
  qwm_ctx* x = new (std::nothrow) qwm_ctx();
  if (!x) return QWM_ERR_OOM;
  x->cfg = *c;
  x->lay = L;
  if (cudaGetDevice(&x->device) != cudaSuccess) {
    delete x;
    return QWM_ERR_CUDA;
  }
  x->G = c->head_dim / kGroup;
  x->ib = c->n_centroids <= 256 ? 1 : 2;
  x->esz = c->dtype == QWM_F32 ? 4 : 2;
  x->cache = (uint8_t*)d_cache;
  x->state = (uint8_t*)d_state;
  x->ws = (uint8_t*)d_workspace;
  x->status = (uint32_t*)(x->state + L.st_status);
  x->s = (float*)(x->state + L.st_s);
  x->w = (float*)(x->state + L.st_w);
  x->lambda = (float*)(x->state + L.st_lambda);
  x->energy = (float*)(x->state + L.st_energy);
  x->centroids = (void*)(x->state + L.st_centroids);
  x->cent32 = reinterpret_cast<float*>(x->state + L.st_centroids_f32);
  x->cent16 = reinterpret_cast<__half*>(x->state + L.st_centroids_f16);
  x->cent16_flag = x->status + 1;   // the word after the status word
  x->cent16_ok = false;
  x->basis = (float*)(x->state + L.st_basis);
  x->tiles = (int2*)(x->state + L.st_tiles);
  x->iters = (int32_t*)(x->state + L.st_iters);
  x->n_tokens = 0;
  x->n_tiles = 0;
  x->version = -1;
  x->slot = -1;
  x->centroids_set = false;
  x->attend_kernel = 0;
  x->assign = 0;
  // the eigen-solver's stream has the highest priority: its few CTAs are
  // dispatched before those of the quantisation that becomes ready with it
  int lo_prio = 0, hi_prio = 0;
  if (cudaMemset(d_state, 0, L.state_bytes) != cudaSuccess ||
      cudaDeviceSynchronize() != cudaSuccess ||
      cudaDeviceGetStreamPriorityRange(&lo_prio, &hi_prio) != cudaSuccess ||
      cudaStreamCreateWithPriority(&x->side, cudaStreamNonBlocking, hi_prio) != cudaSuccess ||
      cudaEventCreateWithFlags(&x->ev_fork, cudaEventDisableTiming) != cudaSuccess ||
      cudaEventCreateWithFlags(&x->ev_eig, cudaEventDisableTiming) != cudaSuccess) {
    release_streams(x);
    delete x;
    return QWM_ERR_CUDA;
  }
  *out = x;
  return QWM_OK;
}

// One warp waits (the attention kernels' bounded mbarrier wait) on a barrier
// nothing arrives at: the wait runs out after `limit` SM cycles, sets the
// timeout bit and the kernel returns.
__global__ void wait_timeout_kernel(long long limit, uint32_t* status) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ volatile int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    tcx::bar_init(&bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  tcx::bar_wait(&bar, 0u, &abort_flag, status, limit);
}

extern "C" qwm_status qwm_selftest_wait_timeout(int64_t limit_cycles, uint32_t* d_status, void* stream) {
  if (!d_status || limit_cycles < 1 || limit_cycles > ((int64_t)1 << 32)) return QWM_ERR_INVALID_ARG;
  wait_timeout_kernel<<<1, 32, 0, S(stream)>>>((long long)limit_cycles, d_status);
  return cuda_status(cudaGetLastError());
}

extern "C" qwm_status qwm_destroy(qwm_ctx* ctx) {
  if (ctx) release_streams(ctx);
  delete ctx;
  return QWM_OK;
}

// float32 copy of the bf16 centroids (exact), read by the attention kernels
static __global__ void bf16_to_f32_kernel(const __nv_bfloat16* __restrict__ in, float* __restrict__ out, int64_t n) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) out[i] = __bfloat162float(in[i]);
}

// float16 copy of the bf16 centroids at d = 128 with the channels of every
// 16-channel block in the order 0, 8, 1, 9, ..., 7, 15 (the operand order of
// attention kernel 6); a value that rounds beyond the float16 range sets
// *flag.  bf16 has 8 significant bits, so every centroid inside the range is
// copied exactly (down to 2^-17; smaller magnitudes round to a multiple of
// 2^-24).
static __global__ void bf16_to_f16_blocks_kernel(const __nv_bfloat16* __restrict__ in, __half* __restrict__ out,
                                                 int64_t n, uint32_t* flag) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const int p = (int)(i & 127), q = p & 15;
  const int ch = (p & ~15) + (q >> 1) + 8 * (q & 1);
  const __half hv = __float2half_rn(__bfloat162float(in[(i & ~(int64_t)127) + ch]));
  if (__hisinf(hv)) atomicOr(flag, 1u);
  out[i] = hv;
}

extern "C" qwm_status qwm_set_centroids(qwm_ctx* x, const void* d_centroids, void* stream) {
  if (!x || !d_centroids) return QWM_ERR_INVALID_ARG;
  if (fault_injected("launch")) return QWM_ERR_CUDA;
  size_t bytes = (size_t)x->cfg.heads * x->cfg.n_centroids * x->cfg.head_dim * x->esz;
  cudaError_t e = cudaMemcpyAsync(x->centroids, d_centroids, bytes, cudaMemcpyDeviceToDevice, S(stream));
  const int64_t n = (int64_t)x->cfg.heads * x->cfg.n_centroids * x->cfg.head_dim;
  if (e == cudaSuccess && x->cfg.dtype == QWM_BF16) {
    bf16_to_f32_kernel<<<(unsigned)((n + 255) / 256), 256, 0, S(stream)>>>(
        (const __nv_bfloat16*)x->centroids, x->cent32, n);
    e = cudaGetLastError();
  }
  bool f16_ok = false;
  if (e == cudaSuccess && x->cfg.dtype == QWM_BF16 && x->cfg.head_dim == 128) {
    uint32_t flag = 1;
    e = cudaMemsetAsync(x->cent16_flag, 0, 4, S(stream));
    if (e == cudaSuccess) {
      bf16_to_f16_blocks_kernel<<<(unsigned)((n + 255) / 256), 256, 0, S(stream)>>>(
          (const __nv_bfloat16*)x->centroids, x->cent16, n, x->cent16_flag);
      e = cudaGetLastError();
    }
    if (e == cudaSuccess) e = cudaMemcpyAsync(&flag, x->cent16_flag, 4, cudaMemcpyDeviceToHost, S(stream));
    if (e == cudaSuccess) e = cudaStreamSynchronize(S(stream));
    f16_ok = e == cudaSuccess && flag == 0;
  }
  if (e != cudaSuccess) return QWM_ERR_CUDA;
  x->cent16_ok = f16_ok;
  x->centroids_set = true;
  return QWM_OK;
}

// A new basis version takes the lowest basis slot that no live segment uses;
// with none free the call fails.  The current version's slot may be taken
// when no segment refers to it: the new basis replaces it, and an append
// still reading it is ordered before the overwrite on the caller's stream.
static qwm_status next_version(qwm_ctx* x, int32_t* v_out, int32_t* slot_out) {
  for (int32_t s = 0; s < x->cfg.max_versions; ++s) {
    bool used = false;
    for (const auto& g : x->segs) used = used || g.slot == s;
    if (!used) {
      *v_out = x->version + 1;
      *slot_out = s;
      return QWM_OK;
    }
  }
  return QWM_ERR_CAPACITY;
}

extern "C" qwm_status qwm_calibrate(qwm_ctx* x, const void* d_q, int64_t n_h, void* stream) {
  if (!x || !d_q || n_h < 1 || n_h > x->cfg.max_hist) return QWM_ERR_INVALID_ARG;
  NvtxRange range("qwm_calibrate");
  int32_t v, slot;
  qwm_status st = next_version(x, &v, &slot);
  if (st != QWM_OK) return st;
  if (fault_injected("launch")) return QWM_ERR_CUDA;
  // Gram sums and A^2 on the caller's stream (after the previous
  // eigen-solver has read the buffers this overwrites), then the eigen-solver
  // on the side stream and the group weights on the caller's: the
  // eigen-solver is ready before the quantisation of the next append, so its
  // CTAs get SMs first (a quantisation CTA and an eigen-solver CTA do not fit
  // on one SM together)
  cudaStream_t s = S(stream);
  cudaError_t e = join_eig(x, s);
  if (e == cudaSuccess) e = launch_gram(x, d_q, n_h, s);
  if (e == cudaSuccess) e = launch_square(x, n_h, s);
  if (e == cudaSuccess) e = cudaEventRecord(x->ev_fork, s);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(x->side, x->ev_fork, 0);
  if (e == cudaSuccess) e = launch_eig(x, n_h, slot, x->side);
  if (e == cudaSuccess) e = cudaEventRecord(x->ev_eig, x->side);
  if (e == cudaSuccess) e = launch_group_weights(x, s);
  if (e != cudaSuccess) return QWM_ERR_CUDA;
  x->eig_pending = true;
  x->version = v;
  x->slot = slot;
  return QWM_OK;
}

extern "C" qwm_status qwm_set_calibration(qwm_ctx* x, const float* h_s, const float* h_U,
                                          void* stream) {
  if (!x || !h_s || (x->cfg.rank > 0 && !h_U)) return QWM_ERR_INVALID_ARG;
  int32_t v, slot;
  qwm_status st = next_version(x, &v, &slot);
  if (st != QWM_OK) return st;
  if (fault_injected("launch")) return QWM_ERR_CUDA;
  const size_t H = x->cfg.heads, d = x->cfg.head_dim, r = x->cfg.rank;
  cudaStream_t s = S(stream);
  cudaError_t e = join_eig(x, s);
  if (e == cudaSuccess) e = cudaMemcpyAsync(x->s, h_s, H * d * 4, cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess && r > 0) {
    float* dst = x->basis + (size_t)slot * H * r * d;
    e = cudaMemcpyAsync(dst, h_U, H * r * d * 4, cudaMemcpyHostToDevice, s);
  }
  if (e == cudaSuccess) e = cudaMemsetAsync(x->lambda, 0, H * (r > 0 ? r : 1) * 4, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(x->energy, 0, H * 4, s);
  if (e == cudaSuccess) e = launch_group_weights(x, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return QWM_ERR_CUDA;
  x->version = v;
  x->slot = slot;
  return QWM_OK;
}

extern "C" qwm_status qwm_get_calibration(qwm_ctx* x, float* h_s, float* h_U, float* h_lambda,
                                          float* h_energy, void* stream) {
  if (!x) return QWM_ERR_INVALID_ARG;
  if (x->version < 0) return QWM_ERR_NOT_CALIBRATED;
  const size_t H = x->cfg.heads, d = x->cfg.head_dim, r = x->cfg.rank;
  cudaStream_t s = S(stream);
  cudaError_t e = join_eig(x, s);
  if (e == cudaSuccess && h_s) e = cudaMemcpyAsync(h_s, x->s, H * d * 4, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess && h_U && r > 0)
    e = cudaMemcpyAsync(h_U, x->basis + (size_t)x->slot * H * r * d,
                        H * r * d * 4, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess && h_lambda && r > 0)
    e = cudaMemcpyAsync(h_lambda, x->lambda, H * r * 4, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess && h_energy)
    e = cudaMemcpyAsync(h_energy, x->energy, H * 4, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  return cuda_status(e);
}

extern "C" qwm_status qwm_append(qwm_ctx* x, const void* d_k, const void* d_v, int64_t n,
                                 void* stream) {
  if (!x || n < 0) return QWM_ERR_INVALID_ARG;
  if (n == 0) return QWM_OK;
  if (!d_k || !d_v) return QWM_ERR_INVALID_ARG;
  if (x->version < 0 || !x->centroids_set) return QWM_ERR_NOT_CALIBRATED;
  const int64_t tiles = (n + kTile - 1) / kTile;
  if (x->n_tiles + tiles > x->lay.max_tiles) return QWM_ERR_CAPACITY;
  if (fault_injected("launch")) return QWM_ERR_CUDA;
  NvtxRange range("qwm_append");
  // quantisation (group weights only), then the PSAC coefficients once the
  // basis of the current calibration is there
  cudaStream_t s = S(stream);
  cudaError_t e = launch_append(x, d_k, d_v, n, x->n_tiles, x->slot, s);
  if (e == cudaSuccess && x->cfg.rank > 0) e = join_eig(x, s);
  if (e == cudaSuccess) e = launch_append_e(x, d_k, n, x->n_tiles, x->slot, s);
  if (e != cudaSuccess) return QWM_ERR_CUDA;
  SegmentRec r;
  r.first_tile = x->n_tiles;
  r.n_tiles = tiles;
  r.n_tokens = n;
  r.version = x->version;
  r.slot = x->slot;
  x->segs.push_back(r);
  x->n_tiles += tiles;
  x->n_tokens += n;
  return QWM_OK;
}

extern "C" qwm_status qwm_attend(qwm_ctx* x, const void* d_q, int64_t M, float scale, void* d_out,
                                 void* stream) {
  if (!x || M < 0) return QWM_ERR_INVALID_ARG;
  if (M == 0) return QWM_OK;
  if (!d_q || !d_out) return QWM_ERR_INVALID_ARG;
  if (x->n_tokens == 0) return QWM_ERR_INVALID_ARG;
  if (M > (int64_t)1 << 31) return QWM_ERR_INVALID_ARG;
  if (!(scale > 0.f)) scale = 1.0f / sqrtf((float)x->cfg.head_dim);
  int k = qwm_attend_kernel_for(x, M);
  if (k == 5 && !attend_small_supported(x, M)) return QWM_ERR_UNSUPPORTED;
  if (k == 2 && !attend_mma_supported(x)) return QWM_ERR_UNSUPPORTED;
  if (k == 3 && !attend_tc_supported(x)) return QWM_ERR_UNSUPPORTED;
  if (k == 4 && !attend_tc2_supported(x)) return QWM_ERR_UNSUPPORTED;
  if (k == 6 && !attend_tc3_supported(x)) return QWM_ERR_UNSUPPORTED;
  if (k == 7 && !attend_tc3_few_supported(x, M)) return QWM_ERR_UNSUPPORTED;
  if (fault_injected("launch")) return QWM_ERR_CUDA;
  NvtxRange range("qwm_attend");
  cudaStream_t s = S(stream);
  cudaError_t e = join_eig(x, s);   // the basis of the last calibration
  if (e != cudaSuccess) return QWM_ERR_CUDA;
  e = k == 5   ? launch_attend_small(x, d_q, M, scale, d_out, x->ws + small_workspace_offset(x->cfg), s)
      : k == 7 ? launch_attend_tc3_few(x, d_q, M, scale, d_out, x->ws + small_workspace_offset(x->cfg), s)
      : k == 6 ? launch_attend_tc3(x, d_q, M, scale, d_out, s)
      : k == 4 ? launch_attend_tc2(x, d_q, M, scale, d_out, s)
      : k == 3 ? launch_attend_tc(x, d_q, M, scale, d_out, s)
      : k == 2 ? launch_attend_mma(x, d_q, M, scale, d_out, s)
               : launch_attend_simt(x, d_q, M, scale, d_out, s);
  return cuda_status(e);
}

extern "C" qwm_status qwm_rewind(qwm_ctx* x, int32_t n_segments) {
  if (!x || n_segments < 0 || n_segments > (int32_t)x->segs.size()) return QWM_ERR_INVALID_ARG;
  x->segs.resize(n_segments);
  x->n_tiles = 0;
  x->n_tokens = 0;
  for (const auto& s : x->segs) {
    x->n_tiles += s.n_tiles;
    x->n_tokens += s.n_tokens;
  }
  return QWM_OK;
}

extern "C" qwm_status qwm_peek_status_bits(qwm_ctx* x, uint32_t* bits, void* stream) {
  if (!x || !bits) return QWM_ERR_INVALID_ARG;
  cudaStream_t s = S(stream);
  uint32_t h = 0;
  cudaError_t e = join_eig(x, s);
  if (e == cudaSuccess) e = cudaMemcpyAsync(&h, x->status, 4, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(x->status, 0, 4, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return QWM_ERR_CUDA;
  *bits = h;
  return QWM_OK;
}

extern "C" qwm_status qwm_get_status(qwm_ctx* x, void* stream) {
  uint32_t bits = 0;
  qwm_status st = qwm_peek_status_bits(x, &bits, stream);
  if (st != QWM_OK) return st;
  if (bits & QWM_DEV_NOT_CONVERGED) return QWM_ERR_NOT_CONVERGED;
  if (bits) return QWM_ERR_DEVICE;
  return QWM_OK;
}

extern "C" qwm_status qwm_set_assignment(qwm_ctx* x, int32_t mode) {
  if (!x || mode < 0 || mode > 1) return QWM_ERR_INVALID_ARG;
  x->assign = mode;
  return QWM_OK;
}

extern "C" qwm_status qwm_dequantize(qwm_ctx* x, float* d_khat, float* d_vhat, float* d_e, void* stream) {
  if (!x || !d_khat || !d_vhat || (x->cfg.rank > 0 && !d_e)) return QWM_ERR_INVALID_ARG;
  if (!x->centroids_set) return QWM_ERR_NOT_CALIBRATED;
  if (fault_injected("launch")) return QWM_ERR_CUDA;
  cudaError_t e = join_eig(x, S(stream));
  if (e == cudaSuccess) e = launch_dequantize(x, d_khat, d_vhat, d_e, S(stream));
  return cuda_status(e);
}

extern "C" qwm_status qwm_set_attend_kernel(qwm_ctx* x, int32_t k) {
  if (!x || k < 0 || k > 7) return QWM_ERR_INVALID_ARG;
  x->attend_kernel = k;
  return QWM_OK;
}

extern "C" int32_t qwm_attend_kernel_for(const qwm_ctx* x, int64_t M) {
  if (!x) return -1;
  if (x->attend_kernel != 0) return x->attend_kernel;
  // few rows: kernel 5 decodes every tile once per 16-row block, kernel 7
  // once for up to 64 rows at a higher cost per tile; kernel 7 wins from the
  // second row block on
  if (attend_small_supported(x, M)) return (M > 16 && attend_tc3_few_supported(x, M)) ? 7 : 5;
  return qwm_resolved_attend_kernel(x);
}

extern "C" int32_t qwm_resolved_attend_kernel(const qwm_ctx* x) {
  if (!x) return -1;
  if (x->attend_kernel != 0) return x->attend_kernel;
  if (attend_tc3_supported(x)) return 6;
  if (attend_tc2_supported(x)) return 4;
  if (attend_tc_supported(x)) return 3;
  return attend_mma_supported(x) ? 2 : 1;
}

extern "C" int64_t qwm_num_tokens(const qwm_ctx* x) { return x ? x->n_tokens : -1; }
extern "C" int64_t qwm_num_tiles(const qwm_ctx* x) { return x ? x->n_tiles : -1; }
extern "C" int32_t qwm_num_segments(const qwm_ctx* x) { return x ? (int32_t)x->segs.size() : -1; }
extern "C" int32_t qwm_version(const qwm_ctx* x) { return x ? x->version : -1; }
