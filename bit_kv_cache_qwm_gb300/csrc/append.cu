// qwm_append: QSAC centroid choice, INT2 quantisation and 2-bit packing of the
// key residual and of the value in one pass (append_kernel), then the PSAC
// coefficients (append_e_kernel).  The split lets the quantisation, which
// needs only the group weights of the new calibration, run while the
// eigen-solver of that calibration still computes the basis the coefficients
// need; the second kernel rebuilds k - k_hat from the tile's bytes with the
// same float32 operations the first one used, so e does not depend on it.
//
// QuantWM Abstract: QSAC "jointly considers historical Query sensitivity and
// residual ranges to select INT2-friendly Key centroids"; roboind article,
// "Step 1": each key is assigned to a high-precision centre and the residual
// is quantised to 2 bits; "Step 2": the key error is kept along the dominant
// query directions.
//
// One CTA encodes one 128-slot cache tile of one head.  Thread (token t,
// group g) holds the 32 channels of group g of key t in registers; the four
// (two for d = 64) group threads of a token sit in lanes TPW apart of one warp
// and combine their partial scores with two shuffles.  Centroids are staged,
// negated, in shared memory as float32, 64 KiB at a time; every lane of a
// quarter-warp reads the same address, so the loads are broadcasts, and the
// group slices of a row are padded to start 4 banks apart.  The
// score of a centroid is formed exactly as the decision definition states:
// f32 residual, exact max/min (their evaluation order does not matter), R*R,
// w*R^2, fixed tree sum, strict < in ascending index order so the lowest
// index wins a tie.  NEAREST replaces the score by the squared distance (the
// nearest-centroid baseline): per group a float32 sum of f32(rho*rho) in
// channel order, the same tree over groups.
#include "qwm_internal.cuh"

namespace qwm {
namespace {

constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
__device__ __forceinline__ float min3(float a, float b, float c) {
  float d;
  asm("min.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

template <typename T>
__device__ __forceinline__ void load32(const T* p, float* x);

template <>
__device__ __forceinline__ void load32<float>(const float* p, float* x) {
  const float4* q = reinterpret_cast<const float4*>(p);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    float4 v = __ldg(q + i);
    x[4 * i] = v.x; x[4 * i + 1] = v.y; x[4 * i + 2] = v.z; x[4 * i + 3] = v.w;
  }
}

template <>
__device__ __forceinline__ void load32<__nv_bfloat16>(const __nv_bfloat16* p, float* x) {
  const uint4* q = reinterpret_cast<const uint4*>(p);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint4 v = __ldg(q + i);
    uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      x[8 * i + 2 * j] = __uint_as_float(w[j] << 16);
      x[8 * i + 2 * j + 1] = __uint_as_float(w[j] & 0xffff0000u);
    }
  }
}

// float16 with saturation at +-65504; sets *sat when it saturated.
__device__ __forceinline__ __half f16_sat(float x, bool* sat) {
  __half h = __float2half_rn(x);
  if (__hisinf(h)) {
    *sat = true;
    h = __float2half_rn(x > 0.f ? 65504.f : -65504.f);
  }
  return h;
}

// Per-group asymmetric INT2: zero = f16(min), scale = f16(f32(range/3)),
// code = clamp(rint(f32(f32(x - zero) / scale)), 0, 3) (0 when scale = 0).
// Packs 32 codes into 8 bytes, returns (zero | scale << 16), and the
// dequantised values zero + code*scale in xhat.
__device__ __forceinline__ uint32_t quantize32(const float* x, uint2* packed, float* xhat, bool* sat) {
  float mx = x[0], mn = x[0];
#pragma unroll
  for (int i = 1; i < 31; i += 2) {
    mx = max3(mx, x[i], x[i + 1]);
    mn = min3(mn, x[i], x[i + 1]);
  }
  mx = fmaxf(mx, x[31]);
  mn = fminf(mn, x[31]);
  const float R = __fsub_rn(mx, mn);
  const __half zh = f16_sat(mn, sat);
  const __half sh = f16_sat(__fdiv_rn(R, 3.0f), sat);
  const float zf = __half2float(zh), sf = __half2float(sh);
  uint32_t lo = 0, hi = 0;
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    uint32_t c = 0;
    if (sf != 0.f) {
      float t = rintf(__fdiv_rn(__fsub_rn(x[i], zf), sf));
      t = fminf(fmaxf(t, 0.f), 3.f);
      c = (uint32_t)t;
    }
    xhat[i] = __fadd_rn(zf, __fmul_rn((float)c, sf));
    if (i < 16) lo |= c << (2 * i);
    else hi |= c << (2 * (i - 16));
  }
  packed->x = lo;
  packed->y = hi;
  return (uint32_t)__half_as_ushort(zh) | ((uint32_t)__half_as_ushort(sh) << 16);
}

template <int D, typename T, bool NEAREST>
__global__ void __launch_bounds__(kTile * (D / kGroup))
append_kernel(const T* __restrict__ K, const T* __restrict__ V, int64_t n,
              const T* __restrict__ cent, int nC, const float* __restrict__ w,
              uint8_t* __restrict__ cache, int64_t max_tiles,
              TileOffsets off, int64_t tile0, int32_t version, int2* __restrict__ tiles,
              uint32_t* __restrict__ status, int ib) {
  constexpr int G = D / kGroup;
  constexpr int NT = kTile * G;
  constexpr int TPW = 32 / G;            // tokens per warp
  constexpr int CH = 16384 / D;          // centroids staged per pass
  constexpr int GS = kGroup + 4;         // padded group stride: the G group slices of a
  constexpr int RS = G * GS;             // row start 4 banks apart (conflict-free LDS.128)
  extern __shared__ __align__(16) float smem[];
  float* cs = smem;                      // [CH][G][GS] negated centroids

  const int h = blockIdx.y;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int gi = lane / TPW, ti = lane % TPW;
  const int t = warp * TPW + ti;                       // slot in the tile
  const int64_t tok = (int64_t)blockIdx.x * kTile + t; // token in the chunk
  const bool valid = tok < n;

  float kx[32];
  if (valid) load32<T>(K + ((int64_t)h * n + tok) * D + gi * kGroup, kx);
  else {
#pragma unroll
    for (int i = 0; i < 32; ++i) kx[i] = 0.f;
  }
  const float wg = w[h * G + gi];

  // ---- QSAC: exhaustive sensitivity-weighted range score ----
  float best = __int_as_float(0x7f800000);
  int bj = 0;
  const T* ch = cent + (int64_t)h * nC * D;
  for (int c0 = 0; c0 < nC; c0 += CH) {
    const int cn = min(CH, nC - c0);
    __syncthreads();
    for (int i = threadIdx.x; i < cn * D; i += NT)
      cs[(i / D) * RS + ((i % D) / kGroup) * GS + (i % kGroup)] = -load_elem(ch + (int64_t)c0 * D, i);
    __syncthreads();
    if constexpr (NEAREST) {
#pragma unroll 1
      for (int j = 0; j < cn; ++j) {
        const float* cr = cs + j * RS + gi * GS;
        float acc = 0.f;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float dlt = __fadd_rn(kx[i], cr[i]);
          acc = __fadd_rn(acc, __fmul_rn(dlt, dlt));
        }
        float S;
        if (G == 4) {
          const float u = __fadd_rn(acc, __shfl_xor_sync(kFull, acc, TPW));
          S = __fadd_rn(u, __shfl_xor_sync(kFull, u, 2 * TPW));
        } else {
          S = __fadd_rn(acc, __shfl_xor_sync(kFull, acc, TPW));
        }
        if (S < best) {
          best = S;
          bj = c0 + j;
        }
      }
    } else {
    // two centroids per step, each with even/odd partial max/min: eight
    // independent dependency chains per thread
#pragma unroll 1
    for (int j = 0; j < cn; j += 2) {
      const bool two = j + 1 < cn;
      const float4* ca = reinterpret_cast<const float4*>(cs + j * RS + gi * GS);
      const float4* cb = reinterpret_cast<const float4*>(cs + (two ? j + 1 : j) * RS + gi * GS);
      float ax0 = -INFINITY, ax1 = -INFINITY, an0 = INFINITY, an1 = INFINITY;
      float bx0 = -INFINITY, bx1 = -INFINITY, bn0 = INFINITY, bn1 = INFINITY;
#pragma unroll
      for (int q = 0; q < 8; q += 2) {
        const float4 a0 = ca[q], a1 = ca[q + 1], b0 = cb[q], b1 = cb[q + 1];
        const float2 k01 = make_float2(kx[4 * q], kx[4 * q + 1]), k23 = make_float2(kx[4 * q + 2], kx[4 * q + 3]);
        const float2 k45 = make_float2(kx[4 * q + 4], kx[4 * q + 5]), k67 = make_float2(kx[4 * q + 6], kx[4 * q + 7]);
        const float2 ra0 = __fadd2_rn(k01, make_float2(a0.x, a0.y)), ra1 = __fadd2_rn(k23, make_float2(a0.z, a0.w));
        const float2 ra2 = __fadd2_rn(k45, make_float2(a1.x, a1.y)), ra3 = __fadd2_rn(k67, make_float2(a1.z, a1.w));
        const float2 rb0 = __fadd2_rn(k01, make_float2(b0.x, b0.y)), rb1 = __fadd2_rn(k23, make_float2(b0.z, b0.w));
        const float2 rb2 = __fadd2_rn(k45, make_float2(b1.x, b1.y)), rb3 = __fadd2_rn(k67, make_float2(b1.z, b1.w));
        ax0 = max3(ax0, ra0.x, ra0.y); an0 = min3(an0, ra0.x, ra0.y);
        ax1 = max3(ax1, ra1.x, ra1.y); an1 = min3(an1, ra1.x, ra1.y);
        bx0 = max3(bx0, rb0.x, rb0.y); bn0 = min3(bn0, rb0.x, rb0.y);
        bx1 = max3(bx1, rb1.x, rb1.y); bn1 = min3(bn1, rb1.x, rb1.y);
        ax0 = max3(ax0, ra2.x, ra2.y); an0 = min3(an0, ra2.x, ra2.y);
        ax1 = max3(ax1, ra3.x, ra3.y); an1 = min3(an1, ra3.x, ra3.y);
        bx0 = max3(bx0, rb2.x, rb2.y); bn0 = min3(bn0, rb2.x, rb2.y);
        bx1 = max3(bx1, rb3.x, rb3.y); bn1 = min3(bn1, rb3.x, rb3.y);
      }
      const float Ra = __fsub_rn(fmaxf(ax0, ax1), fminf(an0, an1));
      const float Rb = __fsub_rn(fmaxf(bx0, bx1), fminf(bn0, bn1));
      const float ta = __fmul_rn(wg, __fmul_rn(Ra, Ra));
      const float tb = __fmul_rn(wg, __fmul_rn(Rb, Rb));
      float Sa, Sb;
      if (G == 4) {
        const float ua = __fadd_rn(ta, __shfl_xor_sync(kFull, ta, TPW));
        const float ub = __fadd_rn(tb, __shfl_xor_sync(kFull, tb, TPW));
        Sa = __fadd_rn(ua, __shfl_xor_sync(kFull, ua, 2 * TPW));
        Sb = __fadd_rn(ub, __shfl_xor_sync(kFull, ub, 2 * TPW));
      } else {
        Sa = __fadd_rn(ta, __shfl_xor_sync(kFull, ta, TPW));
        Sb = __fadd_rn(tb, __shfl_xor_sync(kFull, tb, TPW));
      }
      if (Sa < best) {
        best = Sa;
        bj = c0 + j;
      }
      if (two && Sb < best) {
        best = Sb;
        bj = c0 + j + 1;
      }
    }
    }
  }

  // ---- residual of the chosen centroid, INT2 ----
  float cj[32];
  load32<T>(ch + (int64_t)bj * D + gi * kGroup, cj);
#pragma unroll
  for (int i = 0; i < 32; ++i) cj[i] = __fsub_rn(kx[i], cj[i]);   // residual rho
  bool sat = false;
  uint2 kpk;
  float rh[32];
  const uint32_t kqp = quantize32(cj, &kpk, rh, &sat);

  const int64_t tile = tile0 + blockIdx.x;
  uint8_t* base = cache + ((int64_t)h * max_tiles + tile) * off.bytes;

  // ---- value ----
  float vx[32];
  if (valid) load32<T>(V + ((int64_t)h * n + tok) * D + gi * kGroup, vx);
  else {
#pragma unroll
    for (int i = 0; i < 32; ++i) vx[i] = 0.f;
  }
  uint2 vpk;
  const uint32_t vqp = quantize32(vx, &vpk, rh, &sat);

  // ---- stores (pad slots get zeros) ----
  if (gi == 0) {
    if (ib == 1) base[off.idx + t] = valid ? (uint8_t)bj : 0;
    else reinterpret_cast<uint16_t*>(base + off.idx)[t] = valid ? (uint16_t)bj : 0;
  }
  const uint2 z2 = make_uint2(0, 0);
  *reinterpret_cast<uint2*>(base + off.kcode + t * (D / 4) + gi * 8) = valid ? kpk : z2;
  *reinterpret_cast<uint32_t*>(base + off.kqp + (t * G + gi) * 4) = valid ? kqp : 0u;
  *reinterpret_cast<uint2*>(base + off.vcode + t * (D / 4) + gi * 8) = valid ? vpk : z2;
  *reinterpret_cast<uint32_t*>(base + off.vqp + (t * G + gi) * 4) = valid ? vqp : 0u;
  if (valid && sat) atomicOr(status, QWM_DEV_SATURATED);
  if (h == 0 && threadIdx.x == 0) {
    const int64_t left = n - (int64_t)blockIdx.x * kTile;
    tiles[tile] = make_int2(version, (int)(left < kTile ? left : kTile));
  }
}

// PSAC coefficients of the tiles append_kernel just wrote: thread (token t,
// group g) as there, k - k_hat rebuilt from the key, the stored centroid
// index and the stored codes, zero and scale (rho = f32(k - C), k_hat's
// residual = f32(zero + f32(code * scale)), delta = f32(rho - that): the same
// operations append_kernel's quantiser performs), then e_m = U_m . delta as a
// float32 fma chain over the group's 32 channels and a fixed two-shuffle tree
// over the groups, rounded once to fp16.  Pad slots get 0.
template <int D, typename T>
__global__ void __launch_bounds__(kTile * (D / kGroup))
append_e_kernel(const T* __restrict__ K, int64_t n, const T* __restrict__ cent, int nC,
                const float* __restrict__ U, int r, uint8_t* __restrict__ cache, int64_t max_tiles,
                TileOffsets off, int64_t tile0, int ib) {
  constexpr int G = D / kGroup;
  constexpr int NT = kTile * G;
  constexpr int TPW = 32 / G;
  constexpr int US = kGroup + 4;                // group slices of a basis row 4 banks apart
  extern __shared__ __align__(16) float us[];   // [r][G][US] PSAC basis rows
  const int h = blockIdx.y;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int gi = lane / TPW, ti = lane % TPW;
  const int t = warp * TPW + ti;
  const int64_t tok = (int64_t)blockIdx.x * kTile + t;
  const bool valid = tok < n;
  for (int i = threadIdx.x; i < r * D; i += NT)
    us[(i / kGroup) * US + (i % kGroup)] = U[(int64_t)h * r * D + i];
  const int64_t tile = tile0 + blockIdx.x;
  uint8_t* base = cache + ((int64_t)h * max_tiles + tile) * off.bytes;
  float kx[32], cj[32];
  if (valid) load32<T>(K + ((int64_t)h * n + tok) * D + gi * kGroup, kx);
  else {
#pragma unroll
    for (int i = 0; i < 32; ++i) kx[i] = 0.f;
  }
  const int bj = ib == 1 ? base[off.idx + t] : reinterpret_cast<const uint16_t*>(base + off.idx)[t];
  load32<T>(cent + ((int64_t)h * nC + bj) * D + gi * kGroup, cj);
  const uint2 kpk = *reinterpret_cast<const uint2*>(base + off.kcode + t * (D / 4) + gi * 8);
  const uint32_t kqp = *reinterpret_cast<const uint32_t*>(base + off.kqp + (t * G + gi) * 4);
  const float zf = __half2float(__ushort_as_half((unsigned short)(kqp & 0xffffu)));
  const float sf = __half2float(__ushort_as_half((unsigned short)(kqp >> 16)));
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const uint32_t c = ((i < 16 ? kpk.x : kpk.y) >> (2 * (i & 15))) & 3u;
    const float rho = __fsub_rn(kx[i], cj[i]);
    cj[i] = __fsub_rn(rho, __fadd_rn(zf, __fmul_rn((float)c, sf)));   // k - k_hat
  }
  __syncthreads();   // us ready
  __half* eout = reinterpret_cast<__half*>(base + off.e) + (int64_t)t * r;
  for (int m = 0; m < r; ++m) {
    const float4* um = reinterpret_cast<const float4*>(us + (m * G + gi) * US);
    float p = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float4 u4 = um[i];
      p = fmaf(u4.x, cj[4 * i], p);
      p = fmaf(u4.y, cj[4 * i + 1], p);
      p = fmaf(u4.z, cj[4 * i + 2], p);
      p = fmaf(u4.w, cj[4 * i + 3], p);
    }
    p += __shfl_xor_sync(kFull, p, TPW);
    if (G == 4) p += __shfl_xor_sync(kFull, p, 2 * TPW);
    if (gi == (m % G)) eout[m] = valid ? __float2half_rn(p) : __float2half_rn(0.f);
  }
}

template <int D, typename T>
cudaError_t launch_e_t(const qwm_ctx* c, const void* k, int64_t n, int64_t tile0, int32_t slot,
                       cudaStream_t st) {
  const int r = c->cfg.rank, H = c->cfg.heads;
  const size_t smem = (size_t)r * (D / kGroup) * (kGroup + 4) * 4;
  auto kern = append_e_kernel<D, T>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)((n + kTile - 1) / kTile), (unsigned)H);
  const float* U = c->basis + (size_t)slot * H * r * D;
  kern<<<grid, kTile * (D / kGroup), smem, st>>>((const T*)k, n, (const T*)c->centroids, c->cfg.n_centroids,
                                                 U, r, c->cache, c->lay.max_tiles, tile_offsets(c->lay), tile0,
                                                 c->ib);
  return cudaGetLastError();
}

template <int D, typename T>
cudaError_t launch_t(const qwm_ctx* c, const void* k, const void* v, int64_t n, int64_t tile0,
                     int32_t version, cudaStream_t st) {
  const int H = c->cfg.heads, nC = c->cfg.n_centroids;
  constexpr int CH = 16384 / D;
  const size_t smem = (size_t)CH * (D / kGroup) * (kGroup + 4) * 4;
  auto kern = c->assign == 1 ? append_kernel<D, T, true> : append_kernel<D, T, false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)((n + kTile - 1) / kTile), (unsigned)H);
  kern<<<grid, kTile * (D / kGroup), smem, st>>>(
      (const T*)k, (const T*)v, n, (const T*)c->centroids, nC, c->w, c->cache,
      c->lay.max_tiles, tile_offsets(c->lay), tile0, version, c->tiles, c->status, c->ib);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_append_e(const qwm_ctx* c, const void* k, int64_t n, int64_t tile0, int32_t slot,
                            cudaStream_t st) {
  if (c->cfg.rank == 0) return cudaSuccess;
  const bool bf = c->cfg.dtype == QWM_BF16;
  if (c->cfg.head_dim == 128)
    return bf ? launch_e_t<128, __nv_bfloat16>(c, k, n, tile0, slot, st) : launch_e_t<128, float>(c, k, n, tile0, slot, st);
  return bf ? launch_e_t<64, __nv_bfloat16>(c, k, n, tile0, slot, st) : launch_e_t<64, float>(c, k, n, tile0, slot, st);
}

cudaError_t launch_append(const qwm_ctx* c, const void* k, const void* v, int64_t n, int64_t tile0,
                          int32_t version, cudaStream_t st) {
  const bool bf = c->cfg.dtype == QWM_BF16;
  if (c->cfg.head_dim == 128)
    return bf ? launch_t<128, __nv_bfloat16>(c, k, v, n, tile0, version, st)
              : launch_t<128, float>(c, k, v, n, tile0, version, st);
  return bf ? launch_t<64, __nv_bfloat16>(c, k, v, n, tile0, version, st)
            : launch_t<64, float>(c, k, v, n, tile0, version, st);
}

}  // namespace qwm
