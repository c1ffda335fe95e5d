// qwm_attend, tensor-core kernel with warp-level mma.sync (bf16/fp16 inputs,
// float32 accumulation) for head_dim 128 and PSAC rank r <= 32.
//
// Attention over the packed cache with PSAC compensation (QuantWM Abstract;
// roboind article, "Step 2"):
//   l_n = q . k_hat_n + (q U_t^T) . e_n,   O = softmax(scale * l) V_hat.
//
// CTA = 8 warps = 128 query rows of one head; warp w owns rows 16w..16w+15
// and keeps its Q fragments in registers for the whole pass.  For every
// 128-slot tile (double-buffered with cp.async, one tile ahead):
//   - all 256 threads dequantise the tile once into shared memory:
//     k_hat = C[idx] + zero + code*scale in float32, stored as two bf16
//     terms hi = bf16(k_hat), lo = bf16(k_hat - hi) so that q.k_hat keeps
//     ~16 significant bits (a single bf16 k_hat moves large logits by
//     ~0.4% and flips near-tied softmax rows); v_hat in fp16; e padded to
//     16 or 32 fp16 columns.  Rows are stored with a 16-byte-chunk XOR
//     swizzle so ldmatrix reads are conflict-free.
//   - each warp computes S = Q khi^T + Q klo^T + Zhi E^T + Zlo E^T with
//     m16n8k16 MMAs (Z = q U_t^T, split in two fp16 terms, recomputed when the
//     tile's basis version changes), masks pad slots, runs the online softmax
//     in the exp2 domain, and accumulates O += P V_hat (P and V_hat fp16).
#include <math.h>

#include "qwm_internal.cuh"

namespace qwm {
namespace {

constexpr int kWarpsA = 8;
constexpr int kRowsA = 16 * kWarpsA;
constexpr int kD = 128;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

// byte offset of element (row, col) of a [rows][128] 16-bit tile, swizzled
__device__ __forceinline__ int swz(int row, int col) {
  return row * 256 + ((((col >> 3) ^ (row & 7))) << 4) + ((col & 7) << 1);
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void mma_bf16(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void mma_f16(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src));
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;"); }
__device__ __forceinline__ void cp_wait1() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }

struct MmaArgs {
  const __nv_bfloat16* Q;
  __nv_bfloat16* O;
  int64_t M;
  float scale_log2;
  const uint8_t* cache;
  int64_t max_tiles;
  TileOffsets off;
  int64_t n_tiles;
  const int2* tiles;
  const __nv_bfloat16* cent;
  int nC;
  const float* basis;
  int max_versions;
  int H;
  int r;
  int ib;
  uint32_t* status;
};

// RP: e / Z columns after padding (16 or 32); CS: centroids staged in smem
template <int RP, bool CS>
__global__ void __launch_bounds__(kWarpsA * 32, 1) attend_mma_kernel(const MmaArgs a) {
  constexpr int G = kD / kGroup;
  constexpr int NT = kWarpsA * 32;
  extern __shared__ __align__(128) uint8_t sm[];
  const int TB = a.off.bytes;
  uint8_t* tbuf = sm;                                  // [2][TB]
  uint8_t* khi = sm + 2 * TB;                          // [128][128] bf16, swizzled
  uint8_t* klo = khi + 32768;
  uint8_t* vhs = klo + 32768;                          // [128][128] fp16, swizzled
  __half* es = reinterpret_cast<__half*>(vhs + 32768); // [128][RP]
  uint8_t* cs = reinterpret_cast<uint8_t*>(es + 128 * RP);  // [C][128] bf16, swizzled
  uint8_t* uhi = khi;                                  // [RP][128] bf16 (aliases khi)
  uint8_t* ulo = klo;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, t4 = lane & 3;
  const int h = blockIdx.y;
  const int64_t row0 = (int64_t)blockIdx.x * kRowsA + warp * 16;

  // ---- centroids of this head into shared memory ----
  const __nv_bfloat16* ch = a.cent + (int64_t)h * a.nC * kD;
  if (CS) {
    for (int i = tid; i < a.nC * 16; i += NT) {
      const int j = i >> 4, c = i & 15;
      const uint4 v = *reinterpret_cast<const uint4*>(ch + (int64_t)j * kD + c * 8);
      *reinterpret_cast<uint4*>(cs + swz(j, c * 8)) = v;
    }
  }
  // ---- Q fragments (A operand, rows row0 + g, row0 + g + 8) ----
  uint32_t qf[8][4];
  {
    const __nv_bfloat16* q0 = a.Q + ((int64_t)h * a.M + row0 + g) * kD;
    const __nv_bfloat16* q1 = q0 + 8 * kD;
    const bool v0 = row0 + g < a.M, v1 = row0 + g + 8 < a.M;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      const int c = ks * 16 + 2 * t4;
      qf[ks][0] = v0 ? *reinterpret_cast<const uint32_t*>(q0 + c) : 0u;
      qf[ks][1] = v1 ? *reinterpret_cast<const uint32_t*>(q1 + c) : 0u;
      qf[ks][2] = v0 ? *reinterpret_cast<const uint32_t*>(q0 + c + 8) : 0u;
      qf[ks][3] = v1 ? *reinterpret_cast<const uint32_t*>(q1 + c + 8) : 0u;
    }
  }

  float o[16][4];
#pragma unroll
  for (int j = 0; j < 16; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
  float mrow[2] = {-INFINITY, -INFINITY}, lrow[2] = {0.f, 0.f};
  constexpr int KZ = RP > 0 ? RP / 16 : 1;
  uint32_t zf[2][KZ][4];        // [hi/lo][k16 step][A regs]
  int cur_version = -1;

  const uint8_t* tiles_h = a.cache + (int64_t)h * a.max_tiles * TB;
  auto prefetch = [&](int64_t t) {
    if (t < a.n_tiles) {
      const uint8_t* src = tiles_h + t * TB;
      uint8_t* dst = tbuf + (t & 1) * TB;
      for (int i = tid; i < TB / 16; i += NT) cp_async16(smem_u32(dst + i * 16), src + i * 16);
    }
    cp_commit();
  };
  prefetch(0);

  for (int64_t t = 0; t < a.n_tiles; ++t) {
    prefetch(t + 1);
    cp_wait1();
    __syncthreads();   // tile t landed; previous tile's smem readers are done
    const int2 meta = a.tiles[t];
    const int nv = meta.y;
    const uint8_t* tb = tbuf + (t & 1) * TB;

    // ---- Z = q U_t^T for a new basis version (two fp16 terms) ----
    if constexpr (RP > 0) if (meta.x != cur_version) {
      cur_version = meta.x;
      const float* U = a.basis + ((int64_t)cur_version * a.H + h) * a.r * kD;
      for (int i = tid; i < RP * kD; i += NT) {
        const int m = i / kD, c = i % kD;
        const float u = m < a.r ? U[m * kD + c] : 0.f;
        const __nv_bfloat16 hi = __float2bfloat16_rn(u);
        const __nv_bfloat16 lo = __float2bfloat16_rn(u - __bfloat162float(hi));
        *reinterpret_cast<__nv_bfloat16*>(uhi + swz(m, c)) = hi;
        *reinterpret_cast<__nv_bfloat16*>(ulo + swz(m, c)) = lo;
      }
      __syncthreads();
      float z[RP / 8][4];
#pragma unroll
      for (int j = 0; j < RP / 8; ++j) z[j][0] = z[j][1] = z[j][2] = z[j][3] = 0.f;
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
#pragma unroll
        for (int j = 0; j < RP / 8; j += 2) {
          const int mi = lane >> 3;
          const int row = 8 * (j + (mi >> 1)) + (lane & 7);
          const int col = 16 * ks + 8 * (mi & 1);
          uint32_t b0, b1, b2, b3;
          ldsm_x4(smem_u32(uhi + swz(row, col)), b0, b1, b2, b3);
          mma_bf16(z[j], qf[ks], b0, b1);
          mma_bf16(z[j + 1], qf[ks], b2, b3);
          ldsm_x4(smem_u32(ulo + swz(row, col)), b0, b1, b2, b3);
          mma_bf16(z[j], qf[ks], b0, b1);
          mma_bf16(z[j + 1], qf[ks], b2, b3);
        }
      }
#pragma unroll
      for (int kk = 0; kk < RP / 16; ++kk) {
        const float* za = z[2 * kk];
        const float* zb = z[2 * kk + 1];
        float hi[8], lo[8];
        const float zz[8] = {za[0], za[1], za[2], za[3], zb[0], zb[1], zb[2], zb[3]};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          hi[i] = __half2float(__float2half_rn(zz[i]));
          lo[i] = zz[i] - hi[i];
        }
        zf[0][kk][0] = pack_f16(hi[0], hi[1]);
        zf[0][kk][1] = pack_f16(hi[2], hi[3]);
        zf[0][kk][2] = pack_f16(hi[4], hi[5]);
        zf[0][kk][3] = pack_f16(hi[6], hi[7]);
        zf[1][kk][0] = pack_f16(lo[0], lo[1]);
        zf[1][kk][1] = pack_f16(lo[2], lo[3]);
        zf[1][kk][2] = pack_f16(lo[4], lo[5]);
        zf[1][kk][3] = pack_f16(lo[6], lo[7]);
      }
      __syncthreads();   // uhi/ulo alias khi/klo
    }

    // ---- dequantise the tile ----
    {
      const int key = tid & 127, half = tid >> 7;
      const int idx = cent_index(a.ib == 1 ? tb[a.off.idx + key]
                                           : reinterpret_cast<const uint16_t*>(tb + a.off.idx)[key],
                                 a.nC, a.status);
      const uint4 kc = *reinterpret_cast<const uint4*>(tb + a.off.kcode + key * 32 + half * 16);
      const uint4 vc = *reinterpret_cast<const uint4*>(tb + a.off.vcode + key * 32 + half * 16);
      const uint32_t kw[4] = {kc.x, kc.y, kc.z, kc.w};
      const uint32_t vw[4] = {vc.x, vc.y, vc.z, vc.w};
#pragma unroll
      for (int gg = 0; gg < 2; ++gg) {
        const int grp = half * 2 + gg;
        const __half2 kq = *reinterpret_cast<const __half2*>(tb + a.off.kqp + (key * G + grp) * 4);
        const __half2 vq = *reinterpret_cast<const __half2*>(tb + a.off.vqp + (key * G + grp) * 4);
        const float kz = __low2float(kq), ks = __high2float(kq);
        const float vz = __low2float(vq), vs = __high2float(vq);
#pragma unroll
        for (int c8 = 0; c8 < 4; ++c8) {
          const int col = grp * 32 + c8 * 8;
          uint4 craw;
          if (CS) craw = *reinterpret_cast<const uint4*>(cs + swz(idx, col));
          else craw = __ldg(reinterpret_cast<const uint4*>(ch + (int64_t)idx * kD + col));
          const uint32_t cw[4] = {craw.x, craw.y, craw.z, craw.w};
          const uint32_t kbits = (kw[gg * 2 + (c8 >> 1)] >> (16 * (c8 & 1))) & 0xffffu;
          const uint32_t vbits = (vw[gg * 2 + (c8 >> 1)] >> (16 * (c8 & 1))) & 0xffffu;
          uint32_t ph[4], pl[4], pv[4];
#pragma unroll
          for (int e2 = 0; e2 < 4; ++e2) {
            float kh2[2], vh2[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
              const int e = 2 * e2 + u;
              const float code_k = (float)((kbits >> (2 * e)) & 3u);
              const float code_v = (float)((vbits >> (2 * e)) & 3u);
              const float cval = __uint_as_float(u ? (cw[e2] & 0xffff0000u) : (cw[e2] << 16));
              kh2[u] = cval + fmaf(code_k, ks, kz);
              vh2[u] = fmaf(code_v, vs, vz);
            }
            const __nv_bfloat162 hb = __floats2bfloat162_rn(kh2[0], kh2[1]);
            const float2 hf = __bfloat1622float2(hb);
            ph[e2] = *reinterpret_cast<const uint32_t*>(&hb);
            pl[e2] = pack_bf16(kh2[0] - hf.x, kh2[1] - hf.y);
            pv[e2] = pack_f16(vh2[0], vh2[1]);
          }
          *reinterpret_cast<uint4*>(khi + swz(key, col)) = make_uint4(ph[0], ph[1], ph[2], ph[3]);
          *reinterpret_cast<uint4*>(klo + swz(key, col)) = make_uint4(pl[0], pl[1], pl[2], pl[3]);
          *reinterpret_cast<uint4*>(vhs + swz(key, col)) = make_uint4(pv[0], pv[1], pv[2], pv[3]);
        }
      }
      if constexpr (RP > 0) {
        const __half* esrc = reinterpret_cast<const __half*>(tb + a.off.e) + key * a.r;
        for (int m = half; m < RP; m += 2) es[key * RP + m] = m < a.r ? esrc[m] : __float2half_rn(0.f);
      }
    }
    __syncthreads();

    // ---- two halves of 64 keys ----
#pragma unroll 1
    for (int hk = 0; hk < 2; ++hk) {
      if (hk * 64 >= nv) break;
      float s[8][4];
#pragma unroll
      for (int j = 0; j < 8; ++j) s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.f;
      const int mi = lane >> 3;
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
#pragma unroll
        for (int j = 0; j < 8; j += 2) {
          const int row = hk * 64 + 8 * (j + (mi >> 1)) + (lane & 7);
          const int col = 16 * ks + 8 * (mi & 1);
          uint32_t b0, b1, b2, b3;
          ldsm_x4(smem_u32(khi + swz(row, col)), b0, b1, b2, b3);
          mma_bf16(s[j], qf[ks], b0, b1);
          mma_bf16(s[j + 1], qf[ks], b2, b3);
          ldsm_x4(smem_u32(klo + swz(row, col)), b0, b1, b2, b3);
          mma_bf16(s[j], qf[ks], b0, b1);
          mma_bf16(s[j + 1], qf[ks], b2, b3);
        }
      }
      if constexpr (RP > 0) {
#pragma unroll
        for (int kk = 0; kk < RP / 16; ++kk) {
#pragma unroll
          for (int j = 0; j < 8; j += 2) {
            const int row = hk * 64 + 8 * (j + (mi >> 1)) + (lane & 7);
            const int col = 16 * kk + 8 * (mi & 1);
            uint32_t b0, b1, b2, b3;
            ldsm_x4(smem_u32(es + row * RP + col), b0, b1, b2, b3);
            mma_f16(s[j], zf[0][kk], b0, b1);
            mma_f16(s[j + 1], zf[0][kk], b2, b3);
            mma_f16(s[j], zf[1][kk], b0, b1);
            mma_f16(s[j + 1], zf[1][kk], b2, b3);
          }
        }
      }
      // mask, scale to the exp2 domain, online softmax
      float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int key = hk * 64 + 8 * j + 2 * t4;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int kk = key + (u & 1);
          const float v = kk < nv ? s[j][u] * a.scale_log2 : -INFINITY;
          s[j][u] = v;
          mx[u >> 1] = fmaxf(mx[u >> 1], v);
        }
      }
      float corr[2];
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        mx[i] = fmaxf(mx[i], __shfl_xor_sync(0xffffffffu, mx[i], 1));
        mx[i] = fmaxf(mx[i], __shfl_xor_sync(0xffffffffu, mx[i], 2));
        const float mnew = fmaxf(mrow[i], mx[i]);
        corr[i] = ex2(mrow[i] - mnew);
        mrow[i] = mnew;
      }
      float ps[2] = {0.f, 0.f};
      uint32_t pf[4][4];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float p0 = ex2(s[j][0] - mrow[0]), p1 = ex2(s[j][1] - mrow[0]);
        const float p2 = ex2(s[j][2] - mrow[1]), p3 = ex2(s[j][3] - mrow[1]);
        ps[0] += p0 + p1;
        ps[1] += p2 + p3;
        pf[j >> 1][(j & 1) * 2 + 0] = pack_f16(p0, p1);
        pf[j >> 1][(j & 1) * 2 + 1] = pack_f16(p2, p3);
      }
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        ps[i] += __shfl_xor_sync(0xffffffffu, ps[i], 1);
        ps[i] += __shfl_xor_sync(0xffffffffu, ps[i], 2);
        lrow[i] = lrow[i] * corr[i] + ps[i];
      }
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        o[j][0] *= corr[0];
        o[j][1] *= corr[0];
        o[j][2] *= corr[1];
        o[j][3] *= corr[1];
      }
      // O += P V_hat over the 64 keys (4 k16 steps)
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
        for (int j = 0; j < 16; j += 2) {
          const int row = hk * 64 + 16 * kk + 8 * (mi & 1) + (lane & 7);
          const int col = 8 * (j + (mi >> 1));
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(smem_u32(vhs + swz(row, col)), b0, b1, b2, b3);
          mma_f16(o[j], pf[kk], b0, b1);
          mma_f16(o[j + 1], pf[kk], b2, b3);
        }
      }
    }
  }
  cp_wait1();   // drain the (empty) last prefetch group

  // ---- normalise and store ----
  const float inv0 = lrow[0] > 0.f ? 1.f / lrow[0] : 0.f;
  const float inv1 = lrow[1] > 0.f ? 1.f / lrow[1] : 0.f;
  __nv_bfloat16* o0 = a.O + ((int64_t)h * a.M + row0 + g) * kD;
  __nv_bfloat16* o1 = o0 + 8 * kD;
  const bool v0 = row0 + g < a.M, v1 = row0 + g + 8 < a.M;
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const int c = 8 * j + 2 * t4;
    if (v0) *reinterpret_cast<uint32_t*>(o0 + c) = pack_bf16(o[j][0] * inv0, o[j][1] * inv0);
    if (v1) *reinterpret_cast<uint32_t*>(o1 + c) = pack_bf16(o[j][2] * inv1, o[j][3] * inv1);
  }
}

size_t mma_smem(const qwm_ctx* c, int RP, bool cs) {
  return 2 * c->lay.tile_bytes + 3 * 32768 + (size_t)128 * RP * 2 + (cs ? (size_t)c->cfg.n_centroids * 256 : 0);
}

template <int RP, bool CS>
cudaError_t launch_rp(const qwm_ctx* c, const MmaArgs& a, int64_t M, cudaStream_t st) {
  const size_t smem = mma_smem(c, RP, CS);
  auto kern = attend_mma_kernel<RP, CS>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)((M + kRowsA - 1) / kRowsA), (unsigned)c->cfg.heads);
  kern<<<grid, kWarpsA * 32, smem, st>>>(a);
  return cudaGetLastError();
}

}  // namespace

bool attend_mma_supported(const qwm_ctx* c) {
  return c->cfg.dtype == QWM_BF16 && c->cfg.head_dim == kD && c->cfg.rank <= 32;
}

cudaError_t launch_attend_mma(const qwm_ctx* c, const void* q, int64_t M, float scale, void* out,
                              cudaStream_t st) {
  MmaArgs a;
  a.Q = (const __nv_bfloat16*)q;
  a.O = (__nv_bfloat16*)out;
  a.M = M;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.cache = c->cache;
  a.max_tiles = c->lay.max_tiles;
  a.off = tile_offsets(c->lay);
  a.n_tiles = c->n_tiles;
  a.tiles = c->tiles;
  a.cent = (const __nv_bfloat16*)c->centroids;
  a.nC = c->cfg.n_centroids;
  a.basis = c->basis;
  a.max_versions = c->cfg.max_versions;
  a.H = c->cfg.heads;
  a.r = c->cfg.rank;
  a.ib = c->ib;
  a.status = c->status;
  const int RP = a.r == 0 ? 0 : (a.r <= 16 ? 16 : 32);
  const bool cs = c->cfg.n_centroids <= 256;
  if (RP == 0) return cs ? launch_rp<0, true>(c, a, M, st) : launch_rp<0, false>(c, a, M, st);
  if (RP == 16) return cs ? launch_rp<16, true>(c, a, M, st) : launch_rp<16, false>(c, a, M, st);
  return cs ? launch_rp<32, true>(c, a, M, st) : launch_rp<32, false>(c, a, M, st);
}

}  // namespace qwm
