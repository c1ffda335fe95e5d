// qwm_attend for few query rows (M <= 64): split KV over many CTAs, the logit
// taken apart into exact pieces so that the 2-bit codes never have to be
// turned into k_hat.
//
// Attention over the packed cache with PSAC compensation (QuantWM Abstract;
// roboind article, "Step 2"):
//   l_n = q . k_hat_n + (q U_t^T) . e_n,   O = softmax(scale * l) V_hat,
// with k_hat_n = C[j_n] + zero_g + code_c * scale_g on every channel c of
// group g.  Hence, for a query row q,
//   q . k_hat_n = q . C[j_n]                              (QC, once per row)
//               + sum_g zero_g(n) * sum_{c in g} q_c       (zero term)
//               + sum_g scale_g(n) * sum_{c in g} q_c code_c(n),
// and the last sums are products of q (fp16) with the codes 0..3, exact in
// fp16, on the tensor cores (mma.sync m16n8k16, float32 accumulation): one
// product per 32-channel group, scaled afterwards by that key's group scale.
//
// Channel orders.  In a packed code word (16 channels, channel c at bits
// 2c..2c+1) channels c and c+8 lie 16 bits apart, so one shift and one mask
// put their codes into the two fp16 halves of a register.  The k slots of
// every m16n8k16 step are therefore filled with channel pairs (c, c+8): slots
// (2t, 2t+1) hold channels (t, t+8) and slots (2t+8, 2t+9) channels (t+4,
// t+12) of the step's 16 channels, for Q's A fragments and the codes' B
// fragments alike (a sum over k does not depend on the order of k).  v_hat
// is stored with the same pairing along its 128 columns (physical columns
// 16b+2i, 16b+2i+1 hold dims 16b+i, 16b+i+8), so O comes out of the PV
// product in that column order and is put back in order when written.
//
// Kernels (one head h, one block of 16 query rows mb):
//   qc_kernel         QC[row][j] = q_row . C[j] for every centroid (bf16
//                     operands, exact products, float32 sums) into the
//                     workspace.
//   attend_small      CTA = (mb, split, h), 4 warps, a contiguous range of
//                     tiles (bulk-copied into a 2-stage shared ring); warp w
//                     takes keys 32w..32w+31 of every tile: code products,
//                     PSAC term Z E^T (Z = q U_t^T in two fp16 terms), QC
//                     gather, online softmax in the exp2 domain, v_hat of its
//                     keys in fp16 (its own shared region), O += P V_hat.  The
//                     four warps' partials are merged in shared memory and the
//                     CTA's unnormalised O, maximum and sum go to the
//                     workspace.
//   combine           O = sum_s O_s 2^(m_s - m) / sum_s l_s 2^(m_s - m).
// Waits are bounded by the SM clock; a timeout sets device status bit 0x4.
#include <math.h>

#include "qwm_internal.cuh"

namespace qwm {
namespace {

constexpr int kD = 128;
constexpr int kSmallWarps = 4;
constexpr int kSmallThreads = kSmallWarps * 32;
constexpr int kMaxRowBlocks = 4;        // M <= 64
constexpr int kMaxParts = 64;           // row blocks x splits per head
constexpr int kPartLd = 132;            // floats per partial row: O[128], m, l, pad
static_assert(kPartLd == kPartRowFloats, "partial rows shared with the few-row mode of kernel 6");
constexpr long long kWaitCycles = 1ll << 31;
constexpr uint32_t kDevTimeout = 0x4u;

__device__ __forceinline__ uint32_t su32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

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
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// the codes at bits 0-1 and 16-17 of w as an exact fp16 pair (low, high
// half): 1024 + c is exact in fp16 (0x6400 | c), minus 1024
__device__ __forceinline__ uint32_t codes_pair16(uint32_t w) {
  const uint32_t m = (w & 0x00030003u) | 0x64006400u;
  const __half2 r = __hsub2(*reinterpret_cast<const __half2*>(&m), __float2half2_rn(1024.f));
  return *reinterpret_cast<const uint32_t*>(&r);
}
// byte offset of element (row, col) of a [rows][128] fp16 tile with a 16-byte
// chunk XOR swizzle (conflict-free ldmatrix)
__device__ __forceinline__ int swz(int row, int col) {
  return row * 256 + ((((col >> 3) ^ (row & 7))) << 4) + ((col & 7) << 1);
}

__device__ __forceinline__ void bar_init(uint64_t* b, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(su32(b)), "r"(count));
}
__device__ __forceinline__ void bar_expect_tx(uint64_t* b, uint32_t bytes) {
  asm volatile("{\n.reg .b64 st;\nmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n}"
               ::"r"(su32(b)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void bar_arrive(uint64_t* b) {
  asm volatile("{\n.reg .b64 st;\nmbarrier.arrive.shared::cta.b64 st, [%0];\n}" ::"r"(su32(b)) : "memory");
}
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               ::"r"(su32(dst)), "l"(src), "r"(bytes), "r"(su32(bar)) : "memory");
}
// bounded wait for the phase with parity `par`; false on timeout (flagged)
__device__ __forceinline__ bool bar_wait(uint64_t* b, uint32_t par, uint32_t* status) {
  const long long t0 = clock64();
  while (true) {
    uint32_t done;
    asm volatile("{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
                 "selp.u32 %0, 1, 0, p;\n}"
                 : "=r"(done) : "r"(su32(b)), "r"(par) : "memory");
    if (done) return true;
    if (clock64() - t0 > kWaitCycles) {
      atomicOr(status, kDevTimeout);
      return false;
    }
  }
}

struct SmallArgs {
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
  int nC, nCp;          // centroids, padded to a multiple of 8
  const float* basis;
  int H, r, ib;
  int n_mb, n_split;
  float* qc;            // [H][n_mb][16][nCp]
  float* part;          // [H][n_mb][n_split][16][kPartLd]
  uint32_t* status;
};

// ---------------------------------------------------------------- QC
// grid (n_mb, H), 4 warps; warp w takes centroid blocks of 8, w, w+4, ...
__global__ void __launch_bounds__(kSmallThreads) qc_kernel(const SmallArgs a) {
  const int mb = blockIdx.x, h = blockIdx.y, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int64_t r0 = (int64_t)mb * 16 + g, r1 = r0 + 8;
  const __nv_bfloat16* q0 = a.Q + ((int64_t)h * a.M + r0) * kD;
  const __nv_bfloat16* q1 = a.Q + ((int64_t)h * a.M + r1) * kD;
  uint32_t qf[8][4];
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) {
    const int c = 16 * ks + 2 * t;
    qf[ks][0] = r0 < a.M ? *reinterpret_cast<const uint32_t*>(q0 + c) : 0u;
    qf[ks][1] = r1 < a.M ? *reinterpret_cast<const uint32_t*>(q1 + c) : 0u;
    qf[ks][2] = r0 < a.M ? *reinterpret_cast<const uint32_t*>(q0 + c + 8) : 0u;
    qf[ks][3] = r1 < a.M ? *reinterpret_cast<const uint32_t*>(q1 + c + 8) : 0u;
  }
  const __nv_bfloat16* ch = a.cent + (int64_t)h * a.nC * kD;
  float* out = a.qc + ((int64_t)h * a.n_mb + mb) * 16 * a.nCp;
  for (int jb = warp; jb < a.nCp / 8; jb += kSmallWarps) {
    const int n = 8 * jb + g;                       // this lane's centroid (B column)
    const __nv_bfloat16* crow = ch + (int64_t)n * kD;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      const int c = 16 * ks + 2 * t;
      const uint32_t b0 = n < a.nC ? __ldg(reinterpret_cast<const uint32_t*>(crow + c)) : 0u;
      const uint32_t b1 = n < a.nC ? __ldg(reinterpret_cast<const uint32_t*>(crow + c + 8)) : 0u;
      mma_bf16(acc, qf[ks], b0, b1);
    }
    const int col = 8 * jb + 2 * t;
    *reinterpret_cast<float2*>(out + g * a.nCp + col) = make_float2(acc[0], acc[1]);
    *reinterpret_cast<float2*>(out + (g + 8) * a.nCp + col) = make_float2(acc[2], acc[3]);
  }
}

// ---------------------------------------------------------------- attend
template <int RP>
__global__ void __launch_bounds__(kSmallThreads) attend_small_kernel(const SmallArgs a) {
  constexpr int G = kD / kGroup;
  const int mb = blockIdx.x, split = blockIdx.y, h = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
  const uint32_t TB = (uint32_t)a.off.bytes;
  extern __shared__ __align__(128) uint8_t sm[];
  uint8_t* ring = sm;                                      // [2][TB]
  uint8_t* vs = sm + 2 * TB;                               // [4 warps][32 keys][128] fp16, swizzled
  // QC rows with a stride of nCp + 4 floats: the 8 rows a gather reads for
  // one key then fall into 8 different bank groups
  const int qld = a.nCp + 4;
  float* qcs = reinterpret_cast<float*>(vs + kSmallWarps * 8192);   // [16][qld]
  float* zs = qcs + 16 * qld;                              // [16][32]
  float* red = reinterpret_cast<float*>(sm);               // [4][16][kPartLd], after the loop
  __shared__ __align__(8) uint64_t full[2], empty[2];
  __shared__ int ok_sh;

  const int64_t t_begin = a.n_tiles * split / a.n_split;
  const int64_t nt = a.n_tiles * (split + 1) / a.n_split - t_begin;
  const uint8_t* tiles_h = a.cache + (int64_t)h * a.max_tiles * a.off.bytes;
  if (tid == 0) {
    ok_sh = 1;
    for (int i = 0; i < 2; ++i) {
      bar_init(&full[i], 1);
      bar_init(&empty[i], kSmallWarps);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (tid == 0) {
    for (int64_t u = 0; u < 2 && u < nt; ++u) {
      bar_expect_tx(&full[u], TB);
      bulk_g2s(ring + u * TB, tiles_h + (t_begin + u) * TB, TB, &full[u]);
    }
  }
  // QC rows of this block
  const float* qcg = a.qc + ((int64_t)h * a.n_mb + mb) * 16 * a.nCp;
  for (int i = tid; i < 16 * a.nCp / 4; i += kSmallThreads) {
    const int row = i / (a.nCp / 4), c4 = i - row * (a.nCp / 4);
    reinterpret_cast<float4*>(qcs + row * qld)[c4] = reinterpret_cast<const float4*>(qcg)[i];
  }
  // Q as fp16 A fragments (the code products) and the per-group row sums
  const int64_t r0 = (int64_t)mb * 16 + g, r1 = r0 + 8;
  const __nv_bfloat16* q0 = a.Q + ((int64_t)h * a.M + r0) * kD;
  const __nv_bfloat16* q1 = a.Q + ((int64_t)h * a.M + r1) * kD;
  uint32_t qf[8][4];
  float qsum[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
  auto qpair = [&](const __nv_bfloat16* qr, bool in, int c) {   // channels (c, c+8)
    return in ? make_float2(__bfloat162float(qr[c]), __bfloat162float(qr[c + 8])) : make_float2(0.f, 0.f);
  };
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) {
    const int c = 16 * ks + t;
    float2 x[4];
    x[0] = qpair(q0, r0 < a.M, c);
    x[1] = qpair(q1, r1 < a.M, c);
    x[2] = qpair(q0, r0 < a.M, c + 4);
    x[3] = qpair(q1, r1 < a.M, c + 4);
#pragma unroll
    for (int i = 0; i < 4; ++i) qf[ks][i] = pack_f16(x[i].x, x[i].y);
    qsum[0][ks >> 1] += (x[0].x + x[0].y) + (x[2].x + x[2].y);
    qsum[1][ks >> 1] += (x[1].x + x[1].y) + (x[3].x + x[3].y);
  }
#pragma unroll
  for (int i = 0; i < 2; ++i)
#pragma unroll
    for (int grp = 0; grp < 4; ++grp) {
      qsum[i][grp] += __shfl_xor_sync(0xffffffffu, qsum[i][grp], 1);
      qsum[i][grp] += __shfl_xor_sync(0xffffffffu, qsum[i][grp], 2);
    }
  uint32_t zf[2][RP > 0 ? RP / 16 : 1][4];   // Z = q U^T as two fp16 terms
  float o[16][4];
#pragma unroll
  for (int j = 0; j < 16; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
  float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
  const float c2 = a.scale_log2;
  int cur_slot = -1;
  bool ok = true;
  uint8_t* vw = vs + warp * 8192;
  __syncthreads();

  for (int64_t u = 0; u < nt; ++u) {
    const int st = (int)(u & 1);
    const int64_t tt = t_begin + u;
    const uint8_t* tb = ring + st * TB;
    const int nv = a.tiles[tt].y, slot = a.tiles[tt].x;
    const bool got = bar_wait(&full[st], (uint32_t)((u >> 1) & 1), a.status);
    if (!__syncthreads_and(got && ok)) { ok = false; break; }
    if constexpr (RP > 0) {
      if (slot != cur_slot) {
        cur_slot = slot;
        // Z[row][i] = q_row . U_i (float32), thread = (row, 4 components)
        const float* U = a.basis + ((int64_t)slot * a.H + h) * a.r * kD;
        for (int e = tid; e < 16 * (RP / 4); e += kSmallThreads) {
          const int row = e / (RP / 4), i0 = 4 * (e % (RP / 4));
          const int64_t gr = (int64_t)mb * 16 + row;
          float z[4] = {0.f, 0.f, 0.f, 0.f};
          if (gr < a.M) {
            const __nv_bfloat16* qr = a.Q + ((int64_t)h * a.M + gr) * kD;
            for (int c = 0; c < kD; ++c) {
              const float qv = __bfloat162float(qr[c]);
#pragma unroll
              for (int k = 0; k < 4; ++k)
                if (i0 + k < a.r) z[k] = fmaf(qv, __ldg(U + (int64_t)(i0 + k) * kD + c), z[k]);
            }
          }
#pragma unroll
          for (int k = 0; k < 4; ++k) zs[row * 32 + i0 + k] = z[k];
        }
        __syncthreads();
#pragma unroll
        for (int ks = 0; ks < RP / 16; ++ks) {
          const int c = 16 * ks + 2 * t;
          const float v[4][2] = {{zs[g * 32 + c], zs[g * 32 + c + 1]}, {zs[(g + 8) * 32 + c], zs[(g + 8) * 32 + c + 1]},
                                 {zs[g * 32 + c + 8], zs[g * 32 + c + 9]}, {zs[(g + 8) * 32 + c + 8], zs[(g + 8) * 32 + c + 9]}};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const __half h0 = __float2half_rn(v[i][0]), h1 = __float2half_rn(v[i][1]);
            const __half2 hh = __halves2half2(h0, h1);
            zf[0][ks][i] = *reinterpret_cast<const uint32_t*>(&hh);
            zf[1][ks][i] = pack_f16(v[i][0] - __half2float(h0), v[i][1] - __half2float(h1));
          }
        }
        __syncthreads();
      }
    }
    // ---- logits of keys 32w .. 32w+31: four blocks of 8 ----
    float lg[4][4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int kb = 32 * warp + 8 * j;            // first key of the block
      const int kn = kb + g;                        // this lane's B column (key)
      const uint4 c0 = *reinterpret_cast<const uint4*>(tb + a.off.kcode + kn * 32);
      const uint4 c1 = *reinterpret_cast<const uint4*>(tb + a.off.kcode + kn * 32 + 16);
      const uint32_t cw[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
      float sg[4][4];
#pragma unroll
      for (int grp = 0; grp < 4; ++grp) {
        sg[grp][0] = sg[grp][1] = sg[grp][2] = sg[grp][3] = 0.f;
#pragma unroll
        for (int ks = 0; ks < 2; ++ks) {
          // channels 32grp + 16ks + (t, t+8) and (t+4, t+12): word 2grp + ks
          // shifted by 2t, bits 0/16 and 8/24
          const uint32_t wv = cw[2 * grp + ks] >> (2 * t);
          mma_f16(sg[grp], qf[2 * grp + ks], codes_pair16(wv), codes_pair16(wv >> 8));
        }
      }
      float se[4] = {0.f, 0.f, 0.f, 0.f};
      if constexpr (RP > 0) {
        const __half* erow = reinterpret_cast<const __half*>(tb + a.off.e) + kn * a.r;
#pragma unroll
        for (int ks = 0; ks < RP / 16; ++ks) {
          const int c = 16 * ks + 2 * t;
          uint32_t b0, b1;
          if (a.r == RP) {   // 4-byte aligned pairs
            b0 = *reinterpret_cast<const uint32_t*>(erow + c);
            b1 = *reinterpret_cast<const uint32_t*>(erow + c + 8);
          } else {
            const __half zero = __float2half_rn(0.f);
            const __half2 e0 = __halves2half2(c < a.r ? erow[c] : zero, c + 1 < a.r ? erow[c + 1] : zero);
            const __half2 e1 = __halves2half2(c + 8 < a.r ? erow[c + 8] : zero, c + 9 < a.r ? erow[c + 9] : zero);
            b0 = *reinterpret_cast<const uint32_t*>(&e0);
            b1 = *reinterpret_cast<const uint32_t*>(&e1);
          }
          mma_f16(se, zf[0][ks], b0, b1);
          mma_f16(se, zf[1][ks], b0, b1);
        }
      }
      // this lane's entries: rows g, g+8; keys kb + 2t, kb + 2t + 1
#pragma unroll
      for (int kk = 0; kk < 2; ++kk) {
        const int key = kb + 2 * t + kk;
        const int idx = cent_index(a.ib == 1 ? tb[a.off.idx + key] : reinterpret_cast<const uint16_t*>(tb + a.off.idx)[key],
                                   a.nC, a.status);
        const uint4 qp = *reinterpret_cast<const uint4*>(tb + a.off.kqp + key * G * 4);
        const uint32_t qw[4] = {qp.x, qp.y, qp.z, qp.w};
        float v0 = qcs[g * qld + idx] + se[kk], v1 = qcs[(g + 8) * qld + idx] + se[2 + kk];
#pragma unroll
        for (int grp = 0; grp < 4; ++grp) {
          const float zr = __half2float(__ushort_as_half((unsigned short)(qw[grp] & 0xffffu)));
          const float sc = __half2float(__ushort_as_half((unsigned short)(qw[grp] >> 16)));
          v0 = fmaf(sc, sg[grp][kk], fmaf(zr, qsum[0][grp], v0));
          v1 = fmaf(sc, sg[grp][2 + kk], fmaf(zr, qsum[1][grp], v1));
        }
        const bool valid = key < nv;
        lg[j][kk] = valid ? v0 : -INFINITY;
        lg[j][2 + kk] = valid ? v1 : -INFINITY;
      }
    }
    // ---- online softmax (exp2 domain) ----
    float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      mx[0] = fmaxf(mx[0], fmaxf(lg[j][0], lg[j][1]));
      mx[1] = fmaxf(mx[1], fmaxf(lg[j][2], lg[j][3]));
    }
    // lazy rescale: a row's reference maximum moves only when the tile's
    // maximum exceeds it by more than 2^8 (P <= 2^8 stays within fp16), so O
    // is rescaled on few tiles
    float mref[2];
    bool need[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      mx[i] = fmaxf(mx[i], __shfl_xor_sync(0xffffffffu, mx[i], 1));
      mx[i] = fmaxf(mx[i], __shfl_xor_sync(0xffffffffu, mx[i], 2));
      const float mnew = fmaxf(m_run[i], mx[i] * c2);
      need[i] = mnew > m_run[i] + 8.f;       // also when m_run is -inf and mnew finite
    }
    if (__any_sync(0xffffffffu, need[0] || need[1])) {
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const float mnew = fmaxf(m_run[i], mx[i] * c2);
        const float corr = !need[i] ? 1.f : (m_run[i] == -INFINITY ? 0.f : ex2(m_run[i] - mnew));
        l_run[i] *= corr;
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) {
          o[jj][2 * i] *= corr;
          o[jj][2 * i + 1] *= corr;
        }
        if (need[i]) m_run[i] = mnew;
      }
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) mref[i] = m_run[i] == -INFINITY ? 0.f : m_run[i];
    uint32_t pf[2][4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      float p[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        p[e] = ex2(fmaf(lg[j][e], c2, -mref[e >> 1]));
        l_run[e >> 1] += p[e];
      }
      // P fragment of keys 16(j/2) .. +15: tile j gives columns 2t (a0, a1),
      // tile j+1 columns 2t+8 (a2, a3)
      pf[j >> 1][(j & 1) * 2] = pack_f16(p[0], p[1]);
      pf[j >> 1][(j & 1) * 2 + 1] = pack_f16(p[2], p[3]);
    }
    // ---- v_hat of this warp's 32 keys (lane = key) ----
    {
      const int key = 32 * warp + lane;
      const uint4 c0 = *reinterpret_cast<const uint4*>(tb + a.off.vcode + key * 32);
      const uint4 c1 = *reinterpret_cast<const uint4*>(tb + a.off.vcode + key * 32 + 16);
      const uint4 qp = *reinterpret_cast<const uint4*>(tb + a.off.vqp + key * G * 4);
      const uint32_t vw4[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
      const uint32_t qw[4] = {qp.x, qp.y, qp.z, qp.w};
#pragma unroll
      for (int grp = 0; grp < 4; ++grp) {
        const __half2 vz2 = __half2half2(__ushort_as_half((unsigned short)(qw[grp] & 0xffffu)));
        const __half2 vs2 = __half2half2(__ushort_as_half((unsigned short)(qw[grp] >> 16)));
#pragma unroll
        for (int b2 = 0; b2 < 2; ++b2) {
          // 16-dim block b = 2grp + b2: physical columns 16b + 2i, 16b + 2i + 1
          // hold dims 16b + i and 16b + i + 8 (codes at bits 2i and 2i + 16)
          const int b = 2 * grp + b2;
          const uint32_t wv = vw4[b];
          uint32_t w[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const uint32_t cu = codes_pair16(wv >> (2 * i));
            const __half2 hh = __hfma2(*reinterpret_cast<const __half2*>(&cu), vs2, vz2);   // zero + code*scale
            w[i] = *reinterpret_cast<const uint32_t*>(&hh);
          }
          *reinterpret_cast<uint4*>(vw + swz(lane, 16 * b)) = make_uint4(w[0], w[1], w[2], w[3]);
          *reinterpret_cast<uint4*>(vw + swz(lane, 16 * b + 8)) = make_uint4(w[4], w[5], w[6], w[7]);
        }
      }
    }
    __syncwarp();
    // ---- O += P V_hat over the 32 keys (2 k16 steps) ----
    {
      const int mi = lane >> 3;
#pragma unroll
      for (int kk = 0; kk < 2; ++kk) {
#pragma unroll
        for (int j = 0; j < 16; j += 2) {
          const int row = 16 * kk + 8 * (mi & 1) + (lane & 7);
          const int col = 8 * (j + (mi >> 1));
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(su32(vw + swz(row, col)), b0, b1, b2, b3);
          mma_f16(o[j], pf[kk], b0, b1);
          mma_f16(o[j + 1], pf[kk], b2, b3);
        }
      }
    }
    __syncwarp();
    // this warp is done with ring stage st; thread 0 refills it with tile u + 2
    if (lane == 0) bar_arrive(&empty[st]);
    if (tid == 0 && u + 2 < nt) {
      if (bar_wait(&empty[st], (uint32_t)((u >> 1) & 1), a.status)) {
        bar_expect_tx(&full[st], TB);
        bulk_g2s(ring + st * TB, tiles_h + (tt + 2) * TB, TB, &full[st]);
      } else {
        ok_sh = 0;
      }
    }
    ok = ok && ok_sh;
  }
  // ---- merge the four warps' partials, write this CTA's partial ----
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    l_run[i] += __shfl_xor_sync(0xffffffffu, l_run[i], 1);
    l_run[i] += __shfl_xor_sync(0xffffffffu, l_run[i], 2);
  }
  __syncthreads();   // ring and v_hat buffers are free (no copy is in flight)
  float* rw = red + warp * 16 * kPartLd;
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    // physical columns 8j + 2t, 8j + 2t + 1: dims d and d + 8 of block j / 2
    const int d = 16 * (j >> 1) + 4 * (j & 1) + t;
    rw[g * kPartLd + d] = o[j][0];
    rw[g * kPartLd + d + 8] = o[j][1];
    rw[(g + 8) * kPartLd + d] = o[j][2];
    rw[(g + 8) * kPartLd + d + 8] = o[j][3];
  }
  if (t == 0) {
    rw[g * kPartLd + 128] = m_run[0];
    rw[g * kPartLd + 129] = l_run[0];
    rw[(g + 8) * kPartLd + 128] = m_run[1];
    rw[(g + 8) * kPartLd + 129] = l_run[1];
  }
  __syncthreads();
  if (!__syncthreads_and(ok)) return;
  {
    // thread = (row, 16 channels)
    const int row = tid >> 3, c0 = 16 * (tid & 7);
    float mw[kSmallWarps], mm = -INFINITY;
#pragma unroll
    for (int w = 0; w < kSmallWarps; ++w) {
      mw[w] = red[(w * 16 + row) * kPartLd + 128];
      mm = fmaxf(mm, mw[w]);
    }
    float f[kSmallWarps], l = 0.f;
#pragma unroll
    for (int w = 0; w < kSmallWarps; ++w) {
      f[w] = mw[w] == -INFINITY ? 0.f : ex2(mw[w] - mm);
      l = fmaf(red[(w * 16 + row) * kPartLd + 129], f[w], l);
    }
    float* dst = a.part + ((((int64_t)h * a.n_mb + mb) * a.n_split + split) * 16 + row) * kPartLd;
#pragma unroll
    for (int c = 0; c < 16; c += 4) {
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int w = 0; w < kSmallWarps; ++w) {
        const float4 v = *reinterpret_cast<const float4*>(red + (w * 16 + row) * kPartLd + c0 + c);
        acc.x = fmaf(v.x, f[w], acc.x);
        acc.y = fmaf(v.y, f[w], acc.y);
        acc.z = fmaf(v.z, f[w], acc.z);
        acc.w = fmaf(v.w, f[w], acc.w);
      }
      *reinterpret_cast<float4*>(dst + c0 + c) = acc;
    }
    if ((tid & 7) == 0) {
      dst[128] = mm;
      dst[129] = l;
    }
  }
}

// ---------------------------------------------------------------- combine
// grid (M, H), one warp per query row: lane = 4 channels
__global__ void __launch_bounds__(32) combine_kernel(const SmallArgs a) {
  const int64_t row = blockIdx.x;
  const int h = blockIdx.y, lane = threadIdx.x;
  const int mb = (int)(row >> 4), ri = (int)(row & 15);
  const float* base = a.part + (((int64_t)h * a.n_mb + mb) * a.n_split * 16 + ri) * kPartLd;
  float mm = -INFINITY;
  for (int s = 0; s < a.n_split; ++s) mm = fmaxf(mm, base[(int64_t)s * 16 * kPartLd + 128]);
  float l = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s = 0; s < a.n_split; ++s) {
    const float* p = base + (int64_t)s * 16 * kPartLd;
    const float ms = p[128];
    const float f = ms == -INFINITY ? 0.f : ex2(ms - mm);
    l = fmaf(p[129], f, l);
    const float4 v = *reinterpret_cast<const float4*>(p + 4 * lane);
    acc.x = fmaf(v.x, f, acc.x);
    acc.y = fmaf(v.y, f, acc.y);
    acc.z = fmaf(v.z, f, acc.z);
    acc.w = fmaf(v.w, f, acc.w);
  }
  const float inv = l > 0.f ? 1.f / l : 0.f;
  __nv_bfloat16* dst = a.O + ((int64_t)h * a.M + row) * kD + 4 * lane;
  const __nv_bfloat162 b0 = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
  const __nv_bfloat162 b1 = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
  uint2 w;
  w.x = *reinterpret_cast<const uint32_t*>(&b0);
  w.y = *reinterpret_cast<const uint32_t*>(&b1);
  *reinterpret_cast<uint2*>(dst) = w;
}

size_t small_smem(const qwm_ctx* c) {
  const int nCp = (c->cfg.n_centroids + 7) & ~7;
  return 2 * (size_t)c->lay.tile_bytes + kSmallWarps * 8192 + 16 * (size_t)(nCp + 4) * 4 + 16 * 32 * 4;
}

// splits per row block: among 2, 3 or 4 waves of the resident CTA slots (SMs x
// CTAs per SM, from the occupancy of the kernel instance), the split count
// whose CTAs fill their waves best (the fewest waves on a tie); at least 2
// tiles per split and row blocks x splits <= kMaxParts
int small_splits(const qwm_ctx* c, int n_mb, const void* kern, size_t smem) {
  int dev = 0, sms = 152, per_sm = 2;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  int occ = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kSmallThreads, smem) == cudaSuccess && occ > 0)
    per_sm = occ;
  const int64_t units = (int64_t)c->cfg.heads * n_mb, slots = (int64_t)sms * per_sm;
  const int64_t by_tiles = c->n_tiles / 2 > 0 ? c->n_tiles / 2 : 1;
  const int64_t cap = by_tiles < kMaxParts / n_mb ? by_tiles : kMaxParts / n_mb;
  int64_t best = 1;
  double best_fill = -1.0;
  for (int waves = 2; waves <= 4; ++waves) {
    int64_t s = waves * slots / units;
    if (s > cap) s = cap;
    if (s < 1) s = 1;
    const int64_t ctas = s * units, used = (ctas + slots - 1) / slots;
    const double fill = (double)ctas / (double)(used * slots);
    if (fill > best_fill + 1e-9) {
      best_fill = fill;
      best = s;
    }
  }
  return (int)best;
}

template <int RP>
cudaError_t launch_small_rp(const qwm_ctx* c, SmallArgs& a, cudaStream_t st) {
  const size_t smem = small_smem(c);
  auto kern = attend_small_kernel<RP>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  a.n_split = small_splits(c, a.n_mb, reinterpret_cast<const void*>(kern), smem);
  qc_kernel<<<dim3(a.n_mb, a.H), kSmallThreads, 0, st>>>(a);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  kern<<<dim3(a.n_mb, a.n_split, a.H), kSmallThreads, smem, st>>>(a);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  combine_kernel<<<dim3((unsigned)a.M, a.H), 32, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace

size_t small_workspace_bytes(const qwm_config& cfg) {
  if (cfg.dtype != QWM_BF16 || cfg.head_dim != kD) return 0;
  const size_t nCp = (cfg.n_centroids + 7) & ~7;
  const size_t qc = (size_t)cfg.heads * kMaxRowBlocks * 16 * nCp * 4;
  const size_t part = (size_t)cfg.heads * kMaxParts * 16 * kPartLd * 4;
  return ((qc + 255) & ~size_t(255)) + part;
}

int small_max_parts() { return kMaxParts; }

float* small_part_buffer(const qwm_config& cfg, uint8_t* ws) {
  const size_t nCp = (cfg.n_centroids + 7) & ~7;
  const size_t qc_bytes = (size_t)cfg.heads * kMaxRowBlocks * 16 * nCp * 4;
  return reinterpret_cast<float*>(ws + ((qc_bytes + 255) & ~size_t(255)));
}

cudaError_t launch_small_combine(const qwm_ctx* c, int64_t M, int n_split, uint8_t* ws, void* out,
                                 cudaStream_t st) {
  SmallArgs a = {};
  a.O = (__nv_bfloat16*)out;
  a.M = M;
  a.H = c->cfg.heads;
  a.n_mb = (int)((M + 15) / 16);
  a.n_split = n_split;
  a.part = small_part_buffer(c->cfg, ws);
  combine_kernel<<<dim3((unsigned)M, a.H), 32, 0, st>>>(a);
  return cudaGetLastError();
}

bool attend_small_supported(const qwm_ctx* c, int64_t M) {
  return c->cfg.dtype == QWM_BF16 && c->cfg.head_dim == kD && c->cfg.rank <= 32 && M >= 1 &&
         M <= 16 * kMaxRowBlocks && small_smem(c) <= 227 * 1024;
}

cudaError_t launch_attend_small(const qwm_ctx* c, const void* q, int64_t M, float scale, void* out,
                                uint8_t* ws, cudaStream_t st) {
  SmallArgs a;
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
  a.nCp = (a.nC + 7) & ~7;
  a.basis = c->basis;
  a.H = c->cfg.heads;
  a.r = c->cfg.rank;
  a.ib = c->ib;
  a.n_mb = (int)((M + 15) / 16);
  a.n_split = 1;
  const size_t qc_bytes = (size_t)a.H * kMaxRowBlocks * 16 * a.nCp * 4;
  a.qc = reinterpret_cast<float*>(ws);
  a.part = reinterpret_cast<float*>(ws + ((qc_bytes + 255) & ~size_t(255)));
  a.status = c->status;
  const int RP = a.r == 0 ? 0 : (a.r <= 16 ? 16 : 32);
  return RP == 0 ? launch_small_rp<0>(c, a, st) : RP == 16 ? launch_small_rp<16>(c, a, st) : launch_small_rp<32>(c, a, st);
}

}  // namespace qwm
