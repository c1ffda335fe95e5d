// Internal declarations shared by the host glue and the kernels of libqwm.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include <nvtx3/nvToolsExt.h>

#include <vector>

#include "qwm.h"

namespace qwm {

constexpr int kTile = 128;   // token slots per cache tile
constexpr int kGroup = 32;   // channels per quantisation group

struct SegmentRec {
  int64_t first_tile;
  int64_t n_tiles;
  int64_t n_tokens;
  int32_t version;
  int32_t slot;     // basis slot holding that version's U
};

}  // namespace qwm

struct qwm_ctx {
  qwm_config cfg;
  qwm_layout lay;
  int device;
  int G;          // groups per head
  int ib;         // index bytes per slot
  int esz;        // element size of the configured dtype
  uint8_t* cache;
  uint8_t* state;
  uint8_t* ws;
  // typed views into the state buffer
  uint32_t* status;
  float* s;
  float* w;
  float* lambda;
  float* energy;
  void* centroids;
  float* cent32;    // float32 copy of the centroids (bf16 configs)
  __half* cent16;   // float16 copy, block channel order 0, 8, 1, 9, ... (bf16, d = 128)
  uint32_t* cent16_flag;   // device word: a centroid outside the float16 range
  bool cent16_ok;   // every centroid fits float16 (kernel 6 applies)
  float* basis;     // [max_versions][H][r][d]
  int2* tiles;      // [max_tiles] (version, valid)
  int32_t* iters;   // [H] eigen-solver iterations of the last calibrate
  // host bookkeeping
  int64_t n_tokens;
  int64_t n_tiles;
  int32_t version;       // -1 before the first calibration
  int32_t slot;          // basis slot of the current version
  bool centroids_set;
  int32_t attend_kernel;
  int32_t assign;        // 0 QSAC, 1 nearest centroid
  std::vector<qwm::SegmentRec> segs;
  // The eigen-solver of a calibration runs on `side`, forked from the
  // caller's stream after the Gram sums and group weights (ev_fork) and joined
  // (ev_eig) by every later call that reads the basis, the eigen-solver's
  // outputs, its workspace or the status word; append's quantisation, which
  // needs only the group weights, runs before the join.
  cudaStream_t side = nullptr;
  cudaEvent_t ev_fork = nullptr, ev_eig = nullptr;
  bool eig_pending = false;
};

namespace qwm {

// Host-side fault injection for tests of the error paths, read at every call
// (no GPU fault is involved): QWM_FAULT_INJECT=oom makes qwm_create fail as if
// the host allocation of the context had failed, before any CUDA call;
// QWM_FAULT_INJECT=launch makes qwm_set_centroids, qwm_calibrate,
// qwm_set_calibration, qwm_append, qwm_attend, qwm_dequantize and qwm_kmeans
// return QWM_ERR_CUDA after their argument checks and before any launch, with
// the context unchanged.
inline bool fault_injected(const char* what) {
  const char* v = getenv("QWM_FAULT_INJECT");
  return v != nullptr && strcmp(v, what) == 0;
}

// An NVTX range around one call of the ABI (recorded only when a profiler is
// attached).
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

// ---- launchers (each returns cudaGetLastError() of its launch) ----
cudaError_t launch_append(const qwm_ctx* c, const void* k, const void* v, int64_t n,
                          int64_t tile0, int32_t version, cudaStream_t st);
cudaError_t launch_append_e(const qwm_ctx* c, const void* k, int64_t n, int64_t tile0, int32_t slot,
                            cudaStream_t st);
cudaError_t launch_gram(const qwm_ctx* c, const void* q, int64_t n_h, cudaStream_t st);
cudaError_t launch_square(const qwm_ctx* c, int64_t n_h, cudaStream_t st);
cudaError_t launch_eig(const qwm_ctx* c, int64_t n_h, int32_t version, cudaStream_t st);
cudaError_t launch_group_weights(const qwm_ctx* c, cudaStream_t st);
cudaError_t launch_dequantize(const qwm_ctx* c, float* khat, float* vhat, float* e, cudaStream_t st);
cudaError_t launch_attend_simt(const qwm_ctx* c, const void* q, int64_t M, float scale, void* out,
                               cudaStream_t st);
cudaError_t launch_attend_mma(const qwm_ctx* c, const void* q, int64_t M, float scale, void* out,
                              cudaStream_t st);
bool attend_mma_supported(const qwm_ctx* c);
cudaError_t launch_attend_tc(const qwm_ctx* c, const void* q, int64_t M, float scale, void* out,
                             cudaStream_t st);
bool attend_tc_supported(const qwm_ctx* c);
bool attend_tc2_supported(const qwm_ctx* c);
cudaError_t launch_attend_tc2(const qwm_ctx* c, const void* q, int64_t M, float scale, void* out,
                              cudaStream_t st);
bool attend_tc3_supported(const qwm_ctx* c);
cudaError_t launch_attend_tc3(const qwm_ctx* c, const void* q, int64_t M, float scale, void* out,
                              cudaStream_t st);
size_t gram_workspace_bytes(const qwm_config& cfg);
// few-row attention (M <= 64): its workspace follows the calibration's
size_t small_workspace_bytes(const qwm_config& cfg);
bool attend_small_supported(const qwm_ctx* c, int64_t M);
cudaError_t launch_attend_small(const qwm_ctx* c, const void* q, int64_t M, float scale, void* out,
                                uint8_t* ws, cudaStream_t st);
inline size_t small_workspace_offset(const qwm_config& cfg) {
  return (gram_workspace_bytes(cfg) + 255) & ~size_t(255);
}
// the few-row kernels' partial results: rows of kPartRowFloats floats
// (O[128] unnormalised, running maximum, sum, pad), at most
// small_max_parts() row blocks x KV splits per head, merged per query row by
// launch_small_combine
constexpr int kPartRowFloats = 132;
int small_max_parts();
float* small_part_buffer(const qwm_config& cfg, uint8_t* ws);
cudaError_t launch_small_combine(const qwm_ctx* c, int64_t M, int n_split, uint8_t* ws, void* out,
                                 cudaStream_t st);
// kernel 7: kernel 6 with one 128-row query tile per CTA and the KV range
// split over CTAs (M <= 64), merged by the few-row combine kernel
bool attend_tc3_few_supported(const qwm_ctx* c, int64_t M);
cudaError_t launch_attend_tc3_few(const qwm_ctx* c, const void* q, int64_t M, float scale, void* out,
                                  uint8_t* ws, cudaStream_t st);

// ---- device helpers ----
// The centroid index of a cache slot as read from the cache bytes.  A build
// with QWM_DEBUG_BOUNDS checks it against the centroid count: an index out of
// range sets the status bit QWM_DEV_BOUNDS and is replaced by 0, so no read
// beyond the centroid table follows.  Other builds use it as stored (append
// writes only indices below the count).
__device__ __forceinline__ int cent_index(int idx, int nC, uint32_t* status) {
#ifdef QWM_DEBUG_BOUNDS
  if ((unsigned)idx >= (unsigned)nC) {
    atomicOr(status, QWM_DEV_BOUNDS);
    return 0;
  }
#else
  (void)nC;
  (void)status;
#endif
  return idx;
}
__device__ __forceinline__ float load_elem(const float* p, int64_t i) { return p[i]; }
__device__ __forceinline__ float load_elem(const __nv_bfloat16* p, int64_t i) {
  return __bfloat162float(p[i]);
}

// Tile section offsets (bytes) for one configuration.
struct TileOffsets {
  int idx, kcode, kqp, e, vcode, vqp, bytes;
};

inline TileOffsets tile_offsets(const qwm_layout& L) {
  TileOffsets t;
  t.idx = (int)L.off_idx;
  t.kcode = (int)L.off_kcode;
  t.kqp = (int)L.off_kqp;
  t.e = (int)L.off_e;
  t.vcode = (int)L.off_vcode;
  t.vqp = (int)L.off_vqp;
  t.bytes = (int)L.tile_bytes;
  return t;
}

}  // namespace qwm
