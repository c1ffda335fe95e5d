/*
 * libqwm -- the QuantWM 2-bit KV cache on one GB300 GPU (sm_103a).
 *
 * C ABI of the data-parallel hot path of QuantWM ("QuantWM: Temporally
 * Consistent 2-Bit KV Cache Quantization for World Models and Video
 * Generation", Abstract; the roboind article on QuantWM, sections "Step 1" and
 * "Step 2"):
 *
 *   qwm_calibrate  historical-query sensitivity s_c = mean q_c^2 and the PSAC
 *                  basis U_r (top-r eigenvectors of Q_hist^T Q_hist);
 *   qwm_append     QSAC centroid choice, INT2 quantisation and 2-bit packing of
 *                  the key residual and of the value, PSAC coefficients
 *                  e = U_r (k - k_hat);
 *   qwm_attend     softmax attention of a query chunk over every cached token,
 *                  logit = q.k_hat + (q U_r^T).e.
 *
 * Conventions shared by every call
 *   - The caller owns every device buffer (cache, state, workspace, inputs,
 *     outputs); the library owns only the host handle qwm_ctx.
 *   - Device pointers are plain CUDA device addresses on the device that was
 *     current at qwm_create.  Tensors are dense and row-major:
 *     keys, values, queries and outputs are [heads][rows][head_dim] in the
 *     configured dtype (float32 or bfloat16).
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Compute calls are asynchronous on that stream; calls on one
 *     context must be ordered (one stream, or events between streams).  One
 *     exception: the eigen-solver of qwm_calibrate runs on a stream the
 *     context owns (see qwm_calibrate); every later call that reads what it
 *     writes makes its own stream wait for it first.
 *   - Errors found on the host (arguments, sizes, capacity, call order) are
 *     returned before any launch and leave the context unchanged.  A CUDA
 *     launch error returns QWM_ERR_CUDA.  Conditions found on the device (an
 *     eigen-solver that did not converge, a float16 parameter that saturated)
 *     set bits of a device status word read by qwm_get_status.
 *   - Every entry point is thread-compatible: one context must not be used by
 *     two host threads at once.
 */
#ifndef QWM_H
#define QWM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  QWM_OK = 0,
  QWM_ERR_INVALID_ARG = 1,     /* null pointer, bad size or shape             */
  QWM_ERR_UNSUPPORTED = 2,     /* valid but not built (e.g. head_dim 96)      */
  QWM_ERR_CAPACITY = 3,        /* cache tiles or basis versions exhausted     */
  QWM_ERR_NOT_CALIBRATED = 4,  /* append/attend before calibrate/centroids    */
  QWM_ERR_NOT_CONVERGED = 5,   /* device: eigen-solver hit its iteration cap  */
  QWM_ERR_CUDA = 6,            /* a CUDA runtime call or launch failed        */
  QWM_ERR_OOM = 7,             /* host allocation failed                      */
  QWM_ERR_DEVICE = 8           /* device: other status bits set (see below)   */
} qwm_status;

typedef enum { QWM_F32 = 0, QWM_BF16 = 1 } qwm_dtype;

/* Test hooks, read from the environment at every call:
 *   QWM_FAULT_INJECT=oom     qwm_create returns QWM_ERR_OOM after its argument
 *                            checks, before any CUDA call, creating nothing;
 *   QWM_FAULT_INJECT=launch  qwm_set_centroids, qwm_calibrate,
 *                            qwm_set_calibration, qwm_append, qwm_attend,
 *                            qwm_dequantize and qwm_kmeans return QWM_ERR_CUDA
 *                            after their argument checks and before launching
 *                            anything; the context is left unchanged.
 * A library built with -DQWM_DEBUG_BOUNDS (libqwm_dbg.so) checks every
 * centroid index it reads from the cache against n_centroids; one out of range
 * sets QWM_DEV_BOUNDS in the status word and is read as 0.
 * qwm_calibrate, qwm_append and qwm_attend each open an NVTX range of their
 * own name (recorded only under a profiler). */

/* device status word bits (qwm_get_status / qwm_peek_status_bits) */
#define QWM_DEV_NOT_CONVERGED 0x1u  /* calibrate: residual above tolerance at max_iter */
#define QWM_DEV_SATURATED     0x2u  /* append: a float16 zero or scale saturated at 65504 */
#define QWM_DEV_TIMEOUT       0x4u  /* a bounded device wait ran out; the kernel left early */
#define QWM_DEV_BOUNDS        0x8u  /* QWM_DEBUG_BOUNDS builds only: a cache slot named a
                                       centroid index >= n_centroids (read as 0) */

typedef struct {
  int32_t heads;         /* H >= 1                                              */
  int32_t head_dim;      /* d: 64 or 128                                        */
  int32_t group;         /* channels per quantisation group: must be 32         */
  int32_t rank;          /* PSAC rank r, 0 <= r <= d                            */
  int32_t n_centroids;   /* C, 1 <= C <= 1024                                   */
  int32_t dtype;         /* qwm_dtype of keys, values, queries, centroids, out  */
  int64_t max_tokens;    /* cache capacity in token slots (rounded up to 128);
                            every append starts a new 128-slot tile             */
  int32_t max_versions;  /* basis slots: versions alive at once, the current
                            one included (>= 1)                                 */
  int32_t max_iter;      /* eigen-solver iteration cap (>= 1)                   */
  int32_t oversample;    /* extra subspace columns of the eigen-solver (>= 0)   */
  int32_t max_hist;      /* largest n_h a calibrate call may pass (>= 1)        */
} qwm_config;

/* Sizes and byte offsets derived from a config (qwm_sizes). */
typedef struct {
  size_t cache_bytes;      /* H * max_tiles * tile_bytes                        */
  size_t state_bytes;      /* calibration, centroids, bases, tile table, status */
  size_t workspace_bytes;  /* calibrate scratch, then the few-row attention's   */
                           /* partial results (bf16, d = 128)                    */
  size_t tile_bytes;       /* bytes of one 128-slot tile of one head            */
  size_t bytes_per_token;  /* tile_bytes / 128                                  */
  int64_t max_tiles;       /* tiles per head                                    */
  /* offsets of the sections inside one tile */
  size_t off_idx, off_kcode, off_kqp, off_e, off_vcode, off_vqp;
  /* offsets of the arrays inside the state buffer */
  size_t st_status, st_s, st_w, st_lambda, st_energy, st_centroids, st_basis, st_tiles, st_iters;
  size_t st_centroids_f32;  /* float32 copy of bf16 centroids (= st_centroids for f32) */
  size_t st_centroids_f16;  /* float16 copy of bf16 centroids at d = 128, the channels of
                               every 16-channel block in the order 0, 8, 1, 9, ..., 7, 15
                               (= st_centroids when unused)                         */
} qwm_layout;

typedef struct qwm_ctx qwm_ctx;

/* Human-readable name of a status code (static string). */
const char* qwm_status_string(qwm_status s);

/* Validate `cfg` and compute every size and offset.  No CUDA call.
 * Cache layout: [H][max_tiles][tile_bytes]; one tile holds 128 token slots as
 *   idx   u8 (C <= 256) or u16       [128]
 *   kcode 2-bit K residual codes     [128][d/4]   channel c in byte c/4, bits 2(c%4)
 *   kqp   fp16 (zero, scale) of K    [128][d/32][2]
 *   e     fp16 PSAC coefficients     [128][r]
 *   vcode 2-bit V codes              [128][d/4]
 *   vqp   fp16 (zero, scale) of V    [128][d/32][2]
 * State tile table: int32 pairs (basis slot, valid slots) per tile; a basis
 * slot holds the U of one live basis version. */
qwm_status qwm_sizes(const qwm_config* cfg, qwm_layout* out);

/* Bind a context to caller-owned device buffers of at least the sizes from
 * qwm_sizes (256-byte aligned).  Zeroes the state buffer (synchronously).
 * The buffers must outlive the context.  *out receives the handle. */
qwm_status qwm_create(const qwm_config* cfg, void* d_cache, void* d_state, void* d_workspace,
                      qwm_ctx** out);

/* Release the host handle (device buffers stay with the caller); waits for
 * the context's own stream first.  NULL is a no-op. */
qwm_status qwm_destroy(qwm_ctx* ctx);

/* Self-test of the bounded device waits: one warp waits on an mbarrier that
 * nothing arrives at, with the wait of the attention kernels limited to
 * limit_cycles SM cycles (1 .. 2^32); when it runs out it ORs QWM_DEV_TIMEOUT
 * into *d_status (a caller-owned, caller-zeroed device word) and the kernel
 * returns, leaving the CUDA context usable.  Asynchronous on `stream`. */
qwm_status qwm_selftest_wait_timeout(int64_t limit_cycles, uint32_t* d_status, void* stream);

/* Copy the high-precision centroids [H][C][d] (configured dtype, device) into
 * the state.  QSAC chooses among these ("each Key is assigned to a
 * clustering center ... the center retaining high accuracy", roboind
 * article, "Step 1").  Asynchronous on `stream`, except for bf16 caches at
 * d = 128: there the call also builds the float16 copy that attention
 * kernel 6 reads and waits for `stream` once to learn whether every centroid
 * fits the float16 range (|C| < 65520); when one does not, kernel 6 is not
 * used for this context. */
qwm_status qwm_set_centroids(qwm_ctx* ctx, const void* d_centroids, void* stream);

/* Calibrate from n_h historical queries [H][n_h][d] (device, configured dtype):
 * s_c = mean q_c^2, group weights w_g = sum of s over the group, and the PSAC
 * basis U_r = top-r eigenvectors of Q_hist^T Q_hist (rows, descending
 * eigenvalue; the largest-magnitude entry of each is positive) by block
 * subspace iteration with Rayleigh-Ritz ("the energy of historical queries
 * tends to be concentrated in a few directions", roboind article "Step 2").
 * Opens a new basis version: later appends store coefficients in it.
 * Needs 1 <= n_h <= max_hist.  Asynchronous; non-convergence within max_iter
 * sets QWM_DEV_NOT_CONVERGED and keeps the best basis found.
 * Streams: the Gram sums, s and the group weights are computed on `stream`;
 * the eigen-solver then runs on a stream owned by the context, after them.
 * Later calls on the context that read its results (the coefficient step of
 * qwm_append, qwm_attend, qwm_calibrate, qwm_set_calibration,
 * qwm_get_calibration, qwm_get_status, qwm_peek_status_bits,
 * qwm_dequantize) make their stream wait for it, so the quantisation of the
 * next qwm_append, which needs only the group weights, overlaps it.  Code
 * that reads the basis in the state buffer directly must first issue one of
 * those calls on its stream.  Under CUDA graph capture, end the capture
 * after such a call (it joins the context's stream back into the graph). */
qwm_status qwm_calibrate(qwm_ctx* ctx, const void* d_q_hist, int64_t n_h, void* stream);

/* Calibration for callers that cannot allocate device memory.  (The QuantWM
 * pages have no counterpart of this entry point; it only changes where the
 * scratch lives.)  Some callers cannot call cudaMalloc at all: a plugin whose
 * host application owns all device memory through its own pool, or a code
 * path that must not allocate or free because cudaMalloc/cudaFree may
 * synchronise the device.  This call needs no context and no workspace: it
 * computes the same sensitivity s [H][d], basis U [H][r][d], eigenvalues
 * lambda [H][r] and energy [H] as qwm_calibrate (all float32, caller-owned
 * device buffers; U and lambda may be NULL when rank is 0) from q_hist
 * [H][n_h][d] (dtype QWM_F32 or QWM_BF16), with its scratch (Gram partial
 * sums, A^2, eigen-solver buffers) in one 8 MiB array compiled into the
 * library, which every GPU that loads the library keeps until the process
 * exits.
 *   - Limit: one split of partial sums (H*d*d floats) plus A^2 (H*d*d floats)
 *     must fit in 8 MiB; when rank + oversample > 64 the whole-matrix solver
 *     needs no A^2 but spills 6*d*(d+1) floats per head at d = 128.  Larger
 *     requests return QWM_ERR_CAPACITY before any launch.  That is up to 63
 *     heads at d = 128 (18 when rank + oversample > 64) and 255 at d = 64.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress) once for that device and its current context;
 *     make that first call before any stream capture.  A new context on the
 *     device (after cudaDeviceReset, for instance) has a new driver id, and
 *     the first call in it looks the address up again (also before any
 *     capture).  No call allocates or frees memory.
 *   - All calls share the one array: calls that overlap on the GPU (two
 *     streams, or two host threads) race and corrupt each other's results;
 *     order them.  Nothing in the array needs to start at zero except the
 *     status word, which the call clears itself.
 *   - d_status (optional, caller-zeroed) receives QWM_DEV_NOT_CONVERGED when
 *     the eigen-solver hits max_iter.  With d_status NULL that bit goes to a
 *     word of the shared array and is not reported: a caller that needs to
 *     know about non-convergence passes d_status.  Asynchronous on `stream`. */
qwm_status qwm_calibrate_static(int32_t heads, int32_t head_dim, int32_t rank, int32_t dtype,
                                int32_t max_iter, int32_t oversample, const void* d_q_hist,
                                int64_t n_h, float* d_s, float* d_U, float* d_lambda,
                                float* d_energy, uint32_t* d_status, void* stream);

/* Install a calibration computed elsewhere: s [H][d] and U [H][r][d] (host
 * float32).  Opens a new basis version like qwm_calibrate.  Synchronous. */
qwm_status qwm_set_calibration(qwm_ctx* ctx, const float* h_s, const float* h_U, void* stream);

/* Read the current calibration back (host float32, any pointer may be NULL):
 * s [H][d], U [H][r][d], lambda [H][r], energy [H] = sum(lambda)/trace.
 * Synchronous. */
qwm_status qwm_get_calibration(qwm_ctx* ctx, float* h_s, float* h_U, float* h_lambda,
                               float* h_energy, void* stream);

/* Append one chunk of n tokens: keys and values [H][n][d] (device).  For each
 * key: QSAC j* = argmin_j sum_g w_g (range_g(k - C_j)/3)^2/12 (float32
 * decision, lowest j on a tie), the residual k - C_j* and the value are
 * quantised per 32-channel group to INT2 with fp16 zero = min and
 * scale = range/3, packed 4 codes a byte, and e = U_r (k - k_hat) is stored
 * as r fp16 values (QuantWM Abstract; roboind article "Step 1", "Step 2").
 * Occupies ceil(n/128) new tiles; slots past n in the last tile are zeroed
 * and masked in attention.  n = 0 is a no-op.  Needs a calibration and
 * centroids.  Asynchronous: the quantisation runs at once on `stream`, the
 * coefficients e after the eigen-solver of the last qwm_calibrate (two
 * kernels; the second rebuilds k - k_hat from the tile with the same float32
 * operations). */
qwm_status qwm_append(qwm_ctx* ctx, const void* d_k, const void* d_v, int64_t n, void* stream);

/* Attention of M query rows [H][M][d] over every cached token:
 *   O = softmax(scale * (q.k_hat_n + (q U_t(n)^T).e_n)) V_hat
 * with U_t(n) the basis version the token was appended under ("the current
 * Query matching score with the Historical Key determines how the model
 * allocates attention", roboind article, "The key to a smaller error").
 * softmax_scale <= 0 selects 1/sqrt(d).  Output [H][M][d] in the configured
 * dtype (device).  The cache must hold at least one token.  Asynchronous. */
qwm_status qwm_attend(qwm_ctx* ctx, const void* d_q, int64_t M, float softmax_scale, void* d_out,
                      void* stream);

/* Drop every segment (append call) after the first n_segments, freeing their
 * tiles.  Host bookkeeping only; no device work. */
qwm_status qwm_rewind(qwm_ctx* ctx, int32_t n_segments);

/* Synchronise `stream`, read and clear the device status word.  Returns
 * QWM_ERR_NOT_CONVERGED or QWM_ERR_DEVICE when bits were set, else QWM_OK. */
qwm_status qwm_get_status(qwm_ctx* ctx, void* stream);

/* Same as qwm_get_status but returns the raw bits in *bits. */
qwm_status qwm_peek_status_bits(qwm_ctx* ctx, uint32_t* bits, void* stream);

/* Lloyd's k-means that builds the centroids QSAC assigns keys to ("each Key is
 * assigned to a clustering center", roboind article, "Step 1").  keys
 * [H][n][d] (dtype), d_init_rows [H][C] int32 (device; the starting keys,
 * e.g. the first C entries of a seeded permutation), `iters` iterations:
 * assignment to the nearest centroid in float32 squared distance (lowest
 * index on a tie), update to the float64 mean of the assigned keys rounded to
 * float32, an empty cluster keeps its centroid.  Output [H][C][d] in dtype
 * (nearest even), ready for qwm_set_centroids.  d_workspace: at least
 * qwm_kmeans_workspace_bytes(...) bytes, 256-byte aligned, caller-owned.
 * Asynchronous. */
size_t qwm_kmeans_workspace_bytes(int32_t heads, int32_t head_dim, int32_t n_centroids, int64_t n);
qwm_status qwm_kmeans(int32_t heads, int32_t head_dim, int32_t dtype, int32_t n_centroids,
                      const void* d_keys, int64_t n, const int32_t* d_init_rows, int32_t iters,
                      void* d_centroids, void* d_workspace, void* stream);

/* Centroid assignment of later appends: 0 = QSAC (default; the
 * sensitivity-weighted residual-range score), 1 = nearest centroid (squared
 * distance), the baseline the roboind article's "Step 1" describes for QVG and
 * that QSAC replaces.  For comparisons (the attention-shift diagnostics). */
qwm_status qwm_set_assignment(qwm_ctx* ctx, int32_t mode);

/* The cache in float32 for analysis: k_hat [H][n_tiles*128][d] =
 * C[j] + zero + code*scale, v_hat [H][n_tiles*128][d] = zero + code*scale,
 * e [H][n_tiles*128][r] (the stored fp16 coefficients; may be NULL when
 * r = 0), slot s of tile t at row t*128 + s; pad slots are zero.  Caller-owned
 * device buffers.  Asynchronous. */
qwm_status qwm_dequantize(qwm_ctx* ctx, float* d_khat, float* d_vhat, float* d_e, void* stream);

/* Attention kernel choice: 0 = automatic (bf16 and d = 128: for M <= 64 and
 * r <= 32 kernel 5, or kernel 7 when 16 < M and kernel 6 applies; else kernel
 * 6 when r <= 16 and the centroids fit float16, kernel 4 when r <= 16, kernel
 * 3 when r <= 32; otherwise kernel 2 where it applies, else kernel 1), 1 =
 * float32 CUDA-core kernel, 2 = bf16
 * mma.sync kernel, 3 = bf16 tcgen05 kernel with 128 query rows per CTA, 4 =
 * bf16 tcgen05 kernel with 256 query rows per CTA (r <= 16; the key as two
 * bf16 terms), 5 = bf16 kernel for at most 64 query rows (split over the
 * cache tiles, partial results in the context workspace, merged by a second
 * kernel), 6 = tcgen05 kernel with 256 query rows per CTA and the key split
 * into its float16 centroid row and float16 residual (r <= 16, centroids
 * within the float16 range; queries are scaled per row by a power of two
 * into that range), 7 = kernel 6 with one 128-row query tile per CTA and the
 * cache tiles split over CTAs, merged by kernel 5's second kernel (M <= 64;
 * partial results in the context workspace).  An explicit choice the
 * configuration (or M) does not support makes qwm_attend return
 * QWM_ERR_UNSUPPORTED. */
qwm_status qwm_set_attend_kernel(qwm_ctx* ctx, int32_t kernel);

/* The attention kernel qwm_attend runs for more than 64 query rows (1 to 4,
 * or 6; automatic resolved). */
int32_t qwm_resolved_attend_kernel(const qwm_ctx* ctx);

/* The attention kernel qwm_attend runs for M query rows (1 to 7). */
int32_t qwm_attend_kernel_for(const qwm_ctx* ctx, int64_t M);

int64_t qwm_num_tokens(const qwm_ctx* ctx);    /* valid tokens cached        */
int64_t qwm_num_tiles(const qwm_ctx* ctx);     /* tiles in use per head      */
int32_t qwm_num_segments(const qwm_ctx* ctx);  /* append calls kept          */
int32_t qwm_version(const qwm_ctx* ctx);       /* current basis version, -1 before any */

#ifdef __cplusplus
}
#endif
#endif /* QWM_H */
