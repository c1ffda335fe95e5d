// qwm_dequantize: the cache's dequantised keys, values and PSAC coefficients
// as float32, for analysis (the attention-shift diagnostics).
//
// k_hat = C[j] + zero_g + code_c * scale_g and v_hat = zero_g + code_c *
// scale_g on every channel c of group g (roboind article on QuantWM, "Step 1":
// centre plus 2-bit residual; values quantised the same way), e = the stored
// float16 coefficients ("Step 2").  Float32 in the order
// f32(C + f32(zero + f32(code * scale))).  Pad slots become zeros.
#include "qwm_internal.cuh"

namespace qwm {
namespace {

// one CTA per (tile, head), thread = slot
template <typename T>
__global__ void __launch_bounds__(kTile) dequantize_kernel(const uint8_t* __restrict__ cache, int64_t max_tiles,
                                                          TileOffsets off, const int2* __restrict__ tiles,
                                                          const T* __restrict__ cent, int nC, int d, int r, int ib,
                                                          float* __restrict__ khat, float* __restrict__ vhat,
                                                          float* __restrict__ e, int64_t n_tiles) {
  const int64_t tile = blockIdx.x;
  const int h = blockIdx.y, t = threadIdx.x;
  const int G = d / kGroup;
  const uint8_t* tb = cache + ((int64_t)h * max_tiles + tile) * off.bytes;
  const bool valid = t < tiles[tile].y;
  const int64_t row = ((int64_t)h * n_tiles + tile) * kTile + t;
  float* kr = khat + row * d;
  float* vr = vhat + row * d;
  int idx = ib == 1 ? tb[off.idx + t] : reinterpret_cast<const uint16_t*>(tb + off.idx)[t];
  if (idx >= nC) idx = 0;
  const T* cj = cent + ((int64_t)h * nC + idx) * d;
  for (int c = 0; c < d; ++c) {
    const int g = c / kGroup;
    const uint32_t kqp = *reinterpret_cast<const uint32_t*>(tb + off.kqp + (t * G + g) * 4);
    const uint32_t vqp = *reinterpret_cast<const uint32_t*>(tb + off.vqp + (t * G + g) * 4);
    const uint32_t kc = (tb[off.kcode + t * (d / 4) + c / 4] >> (2 * (c % 4))) & 3u;
    const uint32_t vc = (tb[off.vcode + t * (d / 4) + c / 4] >> (2 * (c % 4))) & 3u;
    const float kz = __half2float(__ushort_as_half((unsigned short)(kqp & 0xffffu)));
    const float ks = __half2float(__ushort_as_half((unsigned short)(kqp >> 16)));
    const float vz = __half2float(__ushort_as_half((unsigned short)(vqp & 0xffffu)));
    const float vs = __half2float(__ushort_as_half((unsigned short)(vqp >> 16)));
    const float rk = __fadd_rn(kz, __fmul_rn((float)kc, ks));
    kr[c] = valid ? __fadd_rn(load_elem(cj, c), rk) : 0.f;
    vr[c] = valid ? __fadd_rn(vz, __fmul_rn((float)vc, vs)) : 0.f;
  }
  if (r > 0) {
    const __half* es = reinterpret_cast<const __half*>(tb + off.e) + (int64_t)t * r;
    float* er = e + row * r;
    for (int m = 0; m < r; ++m) er[m] = valid ? __half2float(es[m]) : 0.f;
  }
}

}  // namespace

cudaError_t launch_dequantize(const qwm_ctx* c, float* khat, float* vhat, float* e, cudaStream_t st) {
  if (c->n_tiles == 0) return cudaSuccess;
  dim3 grid((unsigned)c->n_tiles, (unsigned)c->cfg.heads);
  const TileOffsets off = tile_offsets(c->lay);
  if (c->cfg.dtype == QWM_BF16)
    dequantize_kernel<__nv_bfloat16><<<grid, kTile, 0, st>>>(c->cache, c->lay.max_tiles, off, c->tiles,
                                                             (const __nv_bfloat16*)c->centroids, c->cfg.n_centroids,
                                                             c->cfg.head_dim, c->cfg.rank, c->ib, khat, vhat, e,
                                                             c->n_tiles);
  else
    dequantize_kernel<float><<<grid, kTile, 0, st>>>(c->cache, c->lay.max_tiles, off, c->tiles,
                                                     (const float*)c->centroids, c->cfg.n_centroids, c->cfg.head_dim,
                                                     c->cfg.rank, c->ib, khat, vhat, e, c->n_tiles);
  return cudaGetLastError();
}

}  // namespace qwm
