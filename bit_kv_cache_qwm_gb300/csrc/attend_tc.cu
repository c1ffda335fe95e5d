// qwm_attend, sm_103a tensor-core kernel: tcgen05.mma with TMEM accumulators.
//
// Attention over the packed cache with PSAC compensation (QuantWM Abstract;
// roboind article, "Step 2"):
//   l_n = q . k_hat_n + (q U_t^T) . e_n,   O = softmax(scale * l) V_hat.
//
// One CTA owns 128 query rows of one head and streams every 128-slot tile of
// that head.  Warp roles:
//   warps 0-3   softmax: thread i owns query row i (TMEM lane i).  Writes its
//               Q row into TMEM once (the A operand of QK^T).  Reads S
//               from TMEM, online softmax in the exp2 domain with a lazy
//               rescale (O is corrected only when the running maximum grows
//               by more than 2^8), writes P (fp16) into TMEM, final 1/l and
//               store of O.
//   warps 4-11  producers: one thread bulk-copies every packed tile
//               (cp.async.bulk, mbarrier complete_tx) into a 2-stage shared
//               ring two tiles ahead; all of them dequantise from shared
//               memory k_hat into two bf16 terms (hi + lo, SW128 K-major,
//               rows = keys), v_hat into fp16 (the same layout, read by the PV
//               MMA as an MN-major operand), e
//               into a no-swizzle K-major fp16 tile; recompute Z = q U_t^T as
//               two fp16 terms when the tile's basis slot changes.
//   warp 12     MMA issuer (one lane) and TMEM owner:
//               S[t&1]  = Q khi^T + Q klo^T + Zhi E^T + Zlo E^T   (M=N=128)
//               and O += P V_hat (A = P in TMEM).  The issuer probes the
//               ready barriers without blocking and issues whatever is ready,
//               in order within each stream (S of a tile before its PV).
// TMEM columns: S0 [0,128), S1 [128,256), O [256,384), P [384,448),
// Q [448,512) (bf16 pairs).
// Synchronisation: mbarriers (kA_ready, kB_ready, v_ready, p_ready, s_free[2],
// q_ready arrived by threads; sA_done[2], sB_done[2], pv_done by
// tcgen05.commit; full[2] by the bulk copies).  Every wait is bounded by
// the SM clock; a timeout sets a device status bit and every role leaves its
// loop, the TMEM is freed and the kernel returns.
#include <math.h>

#include "qwm_internal.cuh"
#include "tcgen05_util.cuh"

namespace qwm {
namespace {

using namespace tcx;

constexpr int kD = 128;
constexpr int kSoftWarps = 4, kProdWarps = 8;
constexpr int kThreads = (kSoftWarps + kProdWarps + 1) * 32;   // 416
constexpr int kProdThreads = kProdWarps * 32;
constexpr uint32_t kColS0 = 0, kColO = 256, kColP = 384, kColQ = 448;

constexpr uint32_t kIdescQK = (1u << 4) | (1u << 7) | (1u << 10) | (16u << 17) | (8u << 24);  // bf16 x bf16 -> f32
constexpr uint32_t kIdescF16 = (1u << 4) | (16u << 17) | (8u << 24);                           // f16 x f16 -> f32
constexpr uint32_t kIdescPV = kIdescF16 | (1u << 16);                                          // B MN-major


// Two 2-bit codes (bits 0-1 and 2-3 of n) as exact floats: 2^23 + c has c in
// the low mantissa bits, so (2^23 | c) - 2^23 = c with no rounding.
__device__ __forceinline__ float2 codes_f2(uint32_t n) {
  const float2 m = make_float2(__uint_as_float(0x4B000000u | (n & 3u)), __uint_as_float(0x4B000000u | ((n >> 2) & 3u)));
  return __fadd2_rn(m, make_float2(-8388608.f, -8388608.f));
}
// The same for fp16 pairs: 1024 + c is exact in fp16 (0x6400 | c).
__device__ __forceinline__ __half2 codes_h2(uint32_t n) {
  const uint32_t w = 0x64006400u | (n & 3u) | (((n >> 2) & 3u) << 16);
  return __hsub2(*reinterpret_cast<const __half2*>(&w), __float2half2_rn(1024.f));
}
// Two 2-bit codes at bits p and p+2 of a 16-bit word n as exact floats,
// without shifts: the code's bits are the low mantissa bits of a float whose
// exponent makes bit p weigh 1 (2^(23-p) + c), minus 2^(23-p).
template <int P>
__device__ __forceinline__ float2 codes_at(uint32_t n) {
  constexpr uint32_t e0 = (uint32_t)(127 + 23 - P) << 23, e1 = (uint32_t)(127 + 21 - P) << 23;
  const float2 m = make_float2(__uint_as_float((n & (3u << P)) | e0), __uint_as_float((n & (12u << P)) | e1));
  return __fadd2_rn(m, make_float2(-__uint_as_float(e0), -__uint_as_float(e1)));
}
// k_hat as two bf16 terms: hi = k_hat with the low 16 bits of its float32
// pattern cleared (the truncation to 8 significant bits, exactly a bf16),
// lo = the remainder k_hat - hi (exact in float32, below one bf16 ulp of hi)
// rounded to bf16; |k_hat - hi - lo| < 2^-16 |k_hat|.  The hi pair is one
// byte permute of the two float32 patterns.
__device__ __forceinline__ void split_bf16x2(float2 kv, uint32_t& hi, uint32_t& lo) {
  const float2 ht = make_float2(__uint_as_float(__float_as_uint(kv.x) & 0xffff0000u),
                                __uint_as_float(__float_as_uint(kv.y) & 0xffff0000u));
  const float2 rem = __fadd2_rn(kv, make_float2(-ht.x, -ht.y));
  const __nv_bfloat162 lb = __floats2bfloat162_rn(rem.x, rem.y);
  hi = __byte_perm(__float_as_uint(kv.x), __float_as_uint(kv.y), 0x7632);
  lo = *reinterpret_cast<const uint32_t*>(&lb);
}
// The e row of `key` (r fp16 coefficients, zero-padded to RP) into the
// no-swizzle K-major core-matrix layout of the PSAC B operand.  With r == RP
// the rows are 16-byte aligned in the packed tile and copy as vectors.
template <int RP>
__device__ __forceinline__ void store_e_row(const uint8_t* e_base, int key, int r, uint8_t* Es) {
  const __half* esrc = reinterpret_cast<const __half*>(e_base) + key * r;
  uint8_t* dst = Es + (key >> 3) * (RP / 8) * 128 + (key & 7) * 16;
  if (r == RP) {
#pragma unroll
    for (int j = 0; j < RP / 8; ++j)
      *reinterpret_cast<uint4*>(dst + j * 128) = reinterpret_cast<const uint4*>(esrc)[j];
    return;
  }
#pragma unroll
  for (int j = 0; j < RP / 8; ++j) {
    uint32_t w[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int m0 = 8 * j + 2 * e;
      const __half e0 = m0 < r ? esrc[m0] : __float2half_rn(0.f);
      const __half e1 = m0 + 1 < r ? esrc[m0 + 1] : __float2half_rn(0.f);
      const __half2 ee = __halves2half2(e0, e1);
      w[e] = *reinterpret_cast<const uint32_t*>(&ee);
    }
    *reinterpret_cast<uint4*>(dst + j * 128) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}
__device__ __forceinline__ void prod_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kProdThreads) : "memory"); }
// AND of a predicate over the 256 producer threads (named barrier 1): every
// producer takes the same branch after a bounded wait, so none is left behind
// at a later producer barrier.
__device__ __forceinline__ bool prod_all(bool v) {
  uint32_t r;
  asm volatile("{\n.reg .pred p, q;\nsetp.ne.u32 p, %1, 0;\nbar.red.and.pred q, 1, %2, p;\n"
               "selp.u32 %0, 1, 0, q;\n}"
               : "=r"(r) : "r"((uint32_t)v), "n"(kProdThreads) : "memory");
  return r != 0;
}

// byte offset of (row, k) in a [128 rows][128 k] 16-bit tile stored as two
// SW128 K-major atoms of 64 k each (chunk = 8 elements)
__device__ __forceinline__ int sw128_off(int row, int chunk16) {
  return (chunk16 >> 3) * 16384 + (row >> 3) * 1024 + (row & 7) * 128 + (((chunk16 & 7) ^ (row & 7)) << 4);
}
// centroid rows in smem: [C][256 B], 16-byte chunks XOR-swizzled by row & 7
__device__ __forceinline__ int cswz(int row, int chunk) { return row * 256 + ((chunk ^ (row & 7)) << 4); }

struct TcArgs {
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
  const float* cent32;   // float32 copy of the centroids
  int nC;
  const float* basis;
  int H;
  int r;
  int ib;
  uint32_t* status;
};

template <int RP, bool CS>
__global__ void __launch_bounds__(kThreads, 1) attend_tc_kernel(const TcArgs a) {
  constexpr int G = kD / kGroup;
  extern __shared__ __align__(1024) uint8_t sm_raw[];
  uint8_t* sm = sm_raw + ((1024 - (su32(sm_raw) & 1023)) & 1023);
  uint8_t* Khi = sm;                     // 32 KB
  uint8_t* Klo = sm + 32768;             // 32 KB
  uint8_t* Vt = sm + 65536;              // 32 KB
  uint8_t* Es = sm + 98304;              // 128 x RP fp16, core matrices
  uint8_t* Zh = Es + 128 * RP * 2;       // 128 x RP fp16
  uint8_t* Zl = Zh + 128 * RP * 2;
  uint8_t* Ring = Zl + 128 * RP * 2;     // 2 x tile bytes (packed tiles)
  uint8_t* Cs = Ring + 2 * a.off.bytes;  // C x 256 B (CS only)
  __shared__ __align__(8) uint64_t bars[14];
  __shared__ uint32_t tmem_base_sh;
  __shared__ volatile int abort_sh;
  uint64_t* kA_ready = &bars[0];  // keys 0-63 of k_hat (and their e) written
  uint64_t* kB_ready = &bars[1];  // keys 64-127
  uint64_t* v_ready = &bars[2];
  uint64_t* p_ready = &bars[3];
  uint64_t* pv_done = &bars[4];
  uint64_t* sA_done = &bars[5];   // [2] per S buffer: first half of S(t) computed
  uint64_t* sB_done = &bars[7];   // [2] whole S(t) computed
  uint64_t* s_free = &bars[9];    // [2]
  uint64_t* full = &bars[11];     // [2] packed tile landed in ring stage
  uint64_t* q_ready = &bars[13];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h = blockIdx.y;
  const int64_t row0 = (int64_t)blockIdx.x * 128;
  const int64_t nt = a.n_tiles;

  if (tid == 0) {
    abort_sh = 0;
    bar_init(kA_ready, kProdThreads);
    bar_init(kB_ready, kProdThreads);
    bar_init(v_ready, kProdThreads);
    bar_init(p_ready, 128);
    bar_init(pv_done, 1);
    for (int i = 0; i < 2; ++i) {
      bar_init(&sA_done[i], 1);
      bar_init(&sB_done[i], 1);
      bar_init(&s_free[i], 128);
      bar_init(&full[i], 1);
    }
    bar_init(q_ready, 128);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 12) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(su32(&tmem_base_sh)));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = tmem_base_sh;

  if (warp < kSoftWarps) {
    // ------------------------------------------------------------ softmax
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    const float c2 = a.scale_log2;
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    {
      // this thread's Q row into TMEM columns [448, 512) as bf16 pairs
      const int64_t grow = row0 + tid;
      const uint4* src = reinterpret_cast<const uint4*>(a.Q + ((int64_t)h * a.M + grow) * kD);
      for (int hf = 0; hf < 2; ++hf) {
        uint32_t v[32];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          uint4 x = make_uint4(0, 0, 0, 0);
          if (grow < a.M) x = src[8 * hf + i];
          v[4 * i] = x.x; v[4 * i + 1] = x.y; v[4 * i + 2] = x.z; v[4 * i + 3] = x.w;
        }
        tmem_st32(tmem + lane_base + kColQ + 32 * hf, v);
      }
      tmem_wait_st();
      fence_before();
      bar_arrive(q_ready);
    }
    for (int64_t t = 0; t < nt && ok; ++t) {
      const int b = (int)(t & 1);
      const int nv = a.tiles[t].y;
      if (!warp_all(bar_wait(&sB_done[b], (uint32_t)((t >> 1) & 1), &abort_sh, a.status))) { ok = false; break; }
      fence_after();
      const uint32_t sbase = tmem + lane_base + kColS0 + 128u * b;
      float mx = -INFINITY;
      const bool ragged = nv < 128;
      for (int cb = 0; cb < 2; ++cb) {
        uint32_t v[64];
        tmem_ld64(sbase + 64 * cb, v);
        tmem_wait_ld();
        if (!ragged) {
#pragma unroll
          for (int i = 0; i < 64; i += 2) mx = max3f(mx, __uint_as_float(v[i]), __uint_as_float(v[i + 1]));
        } else {
#pragma unroll
          for (int i = 0; i < 64; ++i)
            if (64 * cb + i < nv) mx = fmaxf(mx, __uint_as_float(v[i]));
        }
      }
      const float mnew = fmaxf(m_run, mx * c2);
      if (t > 0) {
        if (!warp_all(bar_wait(pv_done, (uint32_t)((t - 1) & 1), &abort_sh, a.status))) { ok = false; break; }
        fence_after();
      }
      // lazy rescale: only rows whose maximum grew by more than 2^8 change,
      // but the TMEM traffic is issued by the whole warp (factor 1 elsewhere)
      const bool need = mnew > m_run + 8.f;
      if (t > 0 && __any_sync(0xffffffffu, need)) {
        const float corr = need ? ex2(m_run - mnew) : 1.f;
        for (int cb = 0; cb < 4; ++cb) {
          uint32_t v[32];
          tmem_ld32(tmem + lane_base + kColO + 32 * cb, v);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * corr);
          tmem_st32(tmem + lane_base + kColO + 32 * cb, v);
        }
        l_run *= corr;
      }
      if (need) m_run = mnew;
      float2 psum2 = make_float2(0.f, 0.f);
      const float2 c2v = make_float2(c2, c2), mv = make_float2(-m_run, -m_run);
      for (int cb = 0; cb < 2; ++cb) {
        uint32_t v[64], pk[32];
        tmem_ld64(sbase + 64 * cb, v);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float2 arg = __ffma2_rn(make_float2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1])), c2v, mv);
          float2 pp = make_float2(ex2(arg.x), ex2(arg.y));
          if (ragged) {
            const int k0 = 64 * cb + 2 * i;
            pp.x = k0 < nv ? pp.x : 0.f;
            pp.y = k0 + 1 < nv ? pp.y : 0.f;
          }
          psum2 = __fadd2_rn(psum2, pp);
          const __half2 hp = __floats2half2_rn(pp.x, pp.y);
          pk[i] = *reinterpret_cast<const uint32_t*>(&hp);
        }
        tmem_st32(tmem + lane_base + kColP + 32 * cb, pk);
      }
      const float psum = psum2.x + psum2.y;
      tmem_wait_st();
      l_run += psum;
      fence_before();
      bar_arrive(&s_free[b]);
      bar_arrive(p_ready);
    }
    // epilogue: every lane loads (warp-collective), valid rows store
    if (ok && nt > 0) ok = warp_all(bar_wait(pv_done, (uint32_t)((nt - 1) & 1), &abort_sh, a.status));
    fence_after();
    const int64_t row = row0 + tid;
    if (ok) {
      const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
      __nv_bfloat16* dst = a.O + ((int64_t)h * a.M + row) * kD;
      for (int cb = 0; cb < 4; ++cb) {
        uint32_t v[32];
        tmem_ld32(tmem + lane_base + kColO + 32 * cb, v);
        tmem_wait_ld();
        if (row < a.M) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const __nv_bfloat162 bb = __floats2bfloat162_rn(__uint_as_float(v[8 * q + 2 * e]) * inv,
                                                              __uint_as_float(v[8 * q + 2 * e + 1]) * inv);
              w[e] = *reinterpret_cast<const uint32_t*>(&bb);
            }
            *reinterpret_cast<uint4*>(dst + 32 * cb + 8 * q) = make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
      }
    }
  } else if (warp < kSoftWarps + kProdWarps) {
    // ------------------------------------------------------------ producers
    const int p = tid - kSoftWarps * 32;      // 0..255
    const __nv_bfloat16* ch = a.cent + (int64_t)h * a.nC * kD;
    if (CS) {
      for (int i = p; i < a.nC * 16; i += kProdThreads) {
        const int j = i >> 4, c = i & 15;
        *reinterpret_cast<uint4*>(Cs + cswz(j, c)) = *reinterpret_cast<const uint4*>(ch + (int64_t)j * kD + 8 * c);
      }
    }
    int cur_slot = -1;
    bool ok = true;
    const uint32_t TB = (uint32_t)a.off.bytes;
    const uint8_t* tiles_h = a.cache + (int64_t)h * a.max_tiles * a.off.bytes;
    if (p == 0) {
      for (int64_t u = 0; u < 2 && u < nt; ++u) {
        bar_expect_tx(&full[u], TB);
        bulk_g2s(Ring + u * TB, tiles_h + u * TB, TB, &full[u]);
      }
    }
    prod_sync();
    for (int64_t t = 0; t < nt && ok; ++t) {
      const uint8_t* tb = Ring + (t & 1) * TB;
      const int slot = a.tiles[t].x;
      if (!prod_all(bar_wait(&full[t & 1], (uint32_t)((t >> 1) & 1), &abort_sh, a.status))) { ok = false; break; }
      for (int hk = 0; hk < 2; ++hk) {
        // half hk (keys 64hk .. 64hk+63) of S(t-1) must be computed before
        // its k_hat rows are overwritten
        if (t > 0) {
          uint64_t* prev = hk == 0 ? &sA_done[(t - 1) & 1] : &sB_done[(t - 1) & 1];
          if (!prod_all(bar_wait(prev, (uint32_t)(((t - 1) >> 1) & 1), &abort_sh, a.status))) { ok = false; break; }
        }
        if constexpr (RP > 0) {
          if (hk == 0 && slot != cur_slot) {
            cur_slot = slot;
            // Z and all of khi are read by both halves of S(t-1)
            if (t > 0 && !prod_all(bar_wait(&sB_done[(t - 1) & 1], (uint32_t)(((t - 1) >> 1) & 1), &abort_sh, a.status))) { ok = false; break; }
            // stage U (fp32 [r][128]) in the free khi buffer, then Z = q U^T
            float* Us = reinterpret_cast<float*>(Khi);
            const float* U = a.basis + ((int64_t)slot * a.H + h) * a.r * kD;
            for (int i = p; i < RP * kD; i += kProdThreads) Us[i] = (i / kD) < a.r ? U[i] : 0.f;
            prod_sync();
            if (p < 128) {
              float z[RP];
#pragma unroll
              for (int i = 0; i < RP; ++i) z[i] = 0.f;
              const int64_t grow = row0 + p;
              const uint4* qrow = reinterpret_cast<const uint4*>(a.Q + ((int64_t)h * a.M + grow) * kD);
              for (int c8 = 0; c8 < 16; ++c8) {
                const uint4 qv = grow < a.M ? qrow[c8] : make_uint4(0, 0, 0, 0);
                const uint32_t qw[4] = {qv.x, qv.y, qv.z, qv.w};
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                  const float qf = __uint_as_float(e & 1 ? (qw[e >> 1] & 0xffff0000u) : (qw[e >> 1] << 16));
                  const int c = 8 * c8 + e;
#pragma unroll
                  for (int i = 0; i < RP; ++i) z[i] = fmaf(qf, Us[i * kD + c], z[i]);
                }
              }
#pragma unroll
              for (int j = 0; j < RP / 8; ++j) {
                uint32_t hw[4], lw[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  const __half h0 = __float2half_rn(z[8 * j + 2 * e]), h1 = __float2half_rn(z[8 * j + 2 * e + 1]);
                  const __half2 hh = __halves2half2(h0, h1);
                  const __half2 ll = __floats2half2_rn(z[8 * j + 2 * e] - __half2float(h0),
                                                       z[8 * j + 2 * e + 1] - __half2float(h1));
                  hw[e] = *reinterpret_cast<const uint32_t*>(&hh);
                  lw[e] = *reinterpret_cast<const uint32_t*>(&ll);
                }
                const int off = ((p >> 3) * (RP / 8) + j) * 128 + (p & 7) * 16;
                *reinterpret_cast<uint4*>(Zh + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
                *reinterpret_cast<uint4*>(Zl + off) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
              }
            }
            prod_sync();
          }
        }
        // ---- k_hat (hi, lo) of 64 keys: thread = (key, 32-channel group) ----
        {
          const int key = hk * 64 + (p >> 2), grp = p & 3;
          const int idx = cent_index(a.ib == 1 ? tb[a.off.idx + key] : reinterpret_cast<const uint16_t*>(tb + a.off.idx)[key], a.nC, a.status);
          const uint2 kc = *reinterpret_cast<const uint2*>(tb + a.off.kcode + key * 32 + grp * 8);
          const uint32_t qp = *reinterpret_cast<const uint32_t*>(tb + a.off.kqp + (key * G + grp) * 4);
          const float kz = __half2float(__ushort_as_half((unsigned short)(qp & 0xffffu)));
          const float ks = __half2float(__ushort_as_half((unsigned short)(qp >> 16)));
          const float2 kz2 = make_float2(kz, kz), ks2 = make_float2(ks, ks);
#pragma unroll
          for (int c8 = 0; c8 < 4; ++c8) {
            // chunk order rotated by the group: the 8 lanes of a store phase
            // (2 keys x 4 groups) then hit 8 different bank groups
            const int cl = (c8 + grp) & 3;
            const int chunk = grp * 4 + cl;          // 8-channel chunk 0..15
            uint4 craw;
            if (CS) craw = *reinterpret_cast<const uint4*>(Cs + cswz(idx, chunk));
            else craw = __ldg(reinterpret_cast<const uint4*>(ch + (int64_t)idx * kD + 8 * chunk));
            const uint32_t cw[4] = {craw.x, craw.y, craw.z, craw.w};
            const uint32_t bits = ((cl >> 1) ? kc.y : kc.x) >> (16 * (cl & 1)) & 0xffffu;
            uint32_t ph[4], pl[4];
#pragma unroll
            for (int e2 = 0; e2 < 4; ++e2) {
              const float2 cd = codes_f2(bits >> (4 * e2));
              const float2 rq = __ffma2_rn(cd, ks2, kz2);                      // zero + code*scale
              const float2 cc = make_float2(__uint_as_float(cw[e2] << 16), __uint_as_float(cw[e2] & 0xffff0000u));
              const float2 kv = __fadd2_rn(cc, rq);                            // + centroid
              split_bf16x2(kv, ph[e2], pl[e2]);
            }
            const int off = sw128_off(key, chunk);
            *reinterpret_cast<uint4*>(Khi + off) = make_uint4(ph[0], ph[1], ph[2], ph[3]);
            *reinterpret_cast<uint4*>(Klo + off) = make_uint4(pl[0], pl[1], pl[2], pl[3]);
          }
          if constexpr (RP > 0) {
            if (p < 64) store_e_row<RP>(tb + a.off.e, hk * 64 + p, a.r, Es);
          }
        }
        fence_async_smem();
        bar_arrive(hk == 0 ? kA_ready : kB_ready);
      }
      if (!ok) break;
      // ---- v_hat^T ----
      if (t > 0) {
        if (!prod_all(bar_wait(pv_done, (uint32_t)((t - 1) & 1), &abort_sh, a.status))) { ok = false; break; }
      }
      {
        // v_hat rows (thread = key, 64 channels), stored like k_hat; the PV
        // MMA reads this tile as an MN-major B operand
        const int key = p & 127, half = p >> 7;
        const uint4 vc = *reinterpret_cast<const uint4*>(tb + a.off.vcode + key * 32 + half * 16);
        const uint2 vq = *reinterpret_cast<const uint2*>(tb + a.off.vqp + (key * G + 2 * half) * 4);
        const uint32_t vw[4] = {vc.x, vc.y, vc.z, vc.w};
#pragma unroll
        for (int gg = 0; gg < 2; ++gg) {
          const uint32_t qp = gg ? vq.y : vq.x;
          const __half2 vz2 = __half2half2(__ushort_as_half((unsigned short)(qp & 0xffffu)));
          const __half2 vs2 = __half2half2(__ushort_as_half((unsigned short)(qp >> 16)));
#pragma unroll
          for (int c8 = 0; c8 < 4; ++c8) {
            const int chunk = half * 8 + gg * 4 + c8;
            const uint32_t bits = (vw[gg * 2 + (c8 >> 1)] >> (16 * (c8 & 1))) & 0xffffu;
            uint32_t w[4];
#pragma unroll
            for (int e2 = 0; e2 < 4; ++e2) {
              const __half2 hh = __hfma2(codes_h2(bits >> (4 * e2)), vs2, vz2);   // zero + code*scale
              w[e2] = *reinterpret_cast<const uint32_t*>(&hh);
            }
            *reinterpret_cast<uint4*>(Vt + sw128_off(key, chunk)) = make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
      }
      fence_async_smem();
      bar_arrive(v_ready);
      // every producer is done with ring stage t & 1: refill it with tile t + 2
      prod_sync();
      if (p == 0 && t + 2 < nt) {
        bar_expect_tx(&full[t & 1], TB);
        bulk_g2s(Ring + (t & 1) * TB, tiles_h + (t + 2) * TB, TB, &full[t & 1]);
      }
    }
  } else {
    // ------------------------------------------------------------ MMA issuer
    const bool leader = lane == 0;
    bool ok = true;
    const uint32_t kh = su32(Khi), kl = su32(Klo), vt = su32(Vt);
    const uint32_t ea = su32(Es), za = su32(Zh), zl = su32(Zl);
    constexpr uint32_t kSbo = (RP / 8) * 128;
    ok = warp_all(bar_wait(q_ready, 0u, &abort_sh, a.status));
    fence_after();
    // Issue whatever is ready, in tile order per stream: S(t) first half,
    // S(t) second half, O += P(t) V(t).  The leader alone probes readiness
    // without blocking and issues; the other lanes wait at the end.
    if (leader && ok) {
      int64_t nA = 0, nB = 0, nP = 0;
      long long last = clock64();
      while (nP < nt) {
        bool did = false;
        if (nA < nt) {
          const int b = (int)(nA & 1);
          if (bar_test(kA_ready, (uint32_t)(nA & 1)) && bar_test(kB_ready, (uint32_t)(nA & 1)) &&
              (nA < 2 || bar_test(&s_free[b], (uint32_t)(((nA >> 1) - 1) & 1)))) {
            fence_after();
            // full N = 128 MMAs: N = 64 halves run at a fraction of the rate
            const uint32_t d = tmem + kColS0 + 128u * b;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const uint32_t ko = (j >> 2) * 16384 + (j & 3) * 32;
              mma_ts(d, tmem + kColQ + 8 * j, desc_sw128(kh + ko), kIdescQK, j > 0);
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const uint32_t ko = (j >> 2) * 16384 + (j & 3) * 32;
              mma_ts(d, tmem + kColQ + 8 * j, desc_sw128(kl + ko), kIdescQK, 1);
            }
            if constexpr (RP > 0) {
#pragma unroll
              for (int kk = 0; kk < RP / 16; ++kk) {
                mma_ss(d, desc_none(za + 256 * kk, 128, kSbo), desc_none(ea + 256 * kk, 128, kSbo), kIdescF16, 1);
                mma_ss(d, desc_none(zl + 256 * kk, 128, kSbo), desc_none(ea + 256 * kk, 128, kSbo), kIdescF16, 1);
              }
            }
            commit(&sA_done[b]);
            commit(&sB_done[b]);
            ++nA;
            ++nB;
            did = true;
          }
        }
        if (nP < nB && bar_test(p_ready, (uint32_t)(nP & 1)) && bar_test(v_ready, (uint32_t)(nP & 1))) {
          fence_after();
#pragma unroll
          for (int j = 0; j < 8; ++j)
            mma_ts(tmem + kColO, tmem + kColP + 8 * j, desc_sw128_mn(vt + 2048 * j), kIdescPV,
                   (nP > 0 || j > 0) ? 1u : 0u);
          commit(pv_done);
          ++nP;
          did = true;
        }
        if (did) {
          last = clock64();
        } else if (abort_sh) {
          ok = false;
          break;
        } else if (clock64() - last > kWaitCycles) {
          abort_sh = 1;
          atomicOr(a.status, kDevTimeout);
          ok = false;
          break;
        }
      }
      // wait for the last PV before the TMEM can be released (bounded)
      if (ok && nt > 0) bar_wait(pv_done, (uint32_t)((nt - 1) & 1), &abort_sh, a.status);
    }
    __syncwarp();
  }

  fence_before();
  __syncthreads();
  fence_after();
  if (warp == 12) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem));
}


// ---------------------------------------------------------------------------
// Two query tiles per CTA.  The k_hat, e and v_hat tiles a CTA dequantises
// feed two M = 128 MMAs (query rows 0-127 and 128-255 of the CTA), which
// halves the dequantisation per flop.  Warp roles:
//   warps 0-3 / 4-7  softmax of query tile a / b (thread = row; TMEM lane =
//                    row).  Load their Q rows into shared memory once (the
//                    A operand of QK^T), online softmax as in the one-tile
//                    kernel, P (fp16) written over the first 64 columns of
//                    their own S buffer.
//   warps 8-14       producers: k_hat (hi, lo), e, v_hat and Z = q U_t^T for
//                    both query tiles; centroids read through L2.
//   warp 15          MMA issuer and TMEM owner: S_g(t) = Q_g khi^T + Q_g
//                    klo^T + Zhi_g E^T + Zlo_g E^T, O_g += P_g V_hat, for
//                    g = a, b; S_g(t+1) is issued after PV_g(t), so the
//                    tensor pipe's in-order execution keeps P_g(t) intact
//                    until PV_g(t) has read it.
// TMEM columns: S_a [0,128), S_b [128,256), O_a [256,384), O_b [384,512).
// Split KV: with gridDim.z = 2 the two CTAs of a cluster take the two halves
// of the tile range for the same query rows; rank 1 sends its unnormalised
// O, running maximum and sum to rank 0 through distributed shared memory
// (into buffers rank 0 no longer needs) and rank 0 merges them:
// m = max(m0, m1), O = (O0 2^(m0-m) + O1 2^(m1-m)) / (l0 2^(m0-m) + l1 2^(m1-m)).
// 16 warps: 4 per SM sub-partition, which leaves 128 registers a thread
constexpr int kSoft2Warps = 8, kProd2Warps = 7;
constexpr int kThreads2 = (kSoft2Warps + kProd2Warps + 1) * 32;   // 512
constexpr int kMmaWarp2 = kSoft2Warps + kProd2Warps;             // 15
constexpr uint32_t kColOa = 256;

__device__ __forceinline__ void prod2_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kProd2Warps * 32) : "memory"); }
__device__ __forceinline__ bool prod2_all(bool v) {
  uint32_t r;
  asm volatile("{\n.reg .pred p, q;\nsetp.ne.u32 p, %1, 0;\nbar.red.and.pred q, 1, %2, p;\n"
               "selp.u32 %0, 1, 0, q;\n}"
               : "=r"(r) : "r"((uint32_t)v), "n"(kProd2Warps * 32) : "memory");
  return r != 0;
}

constexpr int kRecvLd = 132;   // floats per row of a received partial: O[128], m, l, ok, pad

template <int RP>
__global__ void __launch_bounds__(kThreads2, 1) attend_tc2_kernel(const TcArgs a) {
  constexpr int G = kD / kGroup;
  constexpr int kZBytes = 128 * RP * 2;
  extern __shared__ __align__(1024) uint8_t sm_raw[];
  uint8_t* sm = sm_raw + ((1024 - (su32(sm_raw) & 1023)) & 1023);
  uint8_t* Qs = sm;                       // 2 x 32 KB: Q_a, Q_b (SW128 K-major)
  uint8_t* Khi = sm + 65536;              // 32 KB
  uint8_t* Klo = sm + 98304;              // 32 KB
  uint8_t* Vt = sm + 131072;              // 32 KB
  uint8_t* Es = sm + 163840;              // 128 x RP fp16, core matrices
  uint8_t* Zs = Es + kZBytes;             // [tile g][hi, lo] 128 x RP fp16
  uint8_t* Ring = Zs + 4 * kZBytes;       // 2 x tile bytes (packed tiles)
  __shared__ __align__(8) uint64_t bars[11];
  __shared__ uint32_t tmem_base_sh;
  __shared__ volatile int abort_sh;
  uint64_t* k_ready = &bars[0];   // k_hat, e (and Z) of tile t written
  uint64_t* v_ready = &bars[1];
  uint64_t* s_done = &bars[2];    // [2] S_g(t) computed
  uint64_t* p_ready = &bars[4];   // [2] P_g(t) written
  uint64_t* pv_done = &bars[6];   // [2] O_g += P_g(t) V(t) done
  uint64_t* full = &bars[8];      // [2] packed tile landed in ring stage
  uint64_t* q_ready = &bars[10];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h = blockIdx.y;
  const int64_t row0 = (int64_t)blockIdx.x * 256;
  // this CTA's share of the tile range (split KV across the cluster)
  const int nsplit = (int)gridDim.z;
  const int split = nsplit > 1 ? (int)cluster_rank() : 0;
  const int64_t t_begin = a.n_tiles * split / nsplit;
  const int64_t nt = a.n_tiles * (split + 1) / nsplit - t_begin;
  constexpr int kProdThreads2 = kProd2Warps * 32;
  float m_run = -INFINITY, l_run = 0.f;   // softmax row state, used by the epilogue
  bool sm_ok = false;

  if (tid == 0) {
    abort_sh = 0;
    bar_init(k_ready, kProdThreads2);
    bar_init(v_ready, kProdThreads2);
    for (int g = 0; g < 2; ++g) {
      bar_init(&s_done[g], 1);
      bar_init(&p_ready[g], 128);
      bar_init(&pv_done[g], 1);
      bar_init(&full[g], 1);
    }
    bar_init(q_ready, 256);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == kMmaWarp2) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(su32(&tmem_base_sh)));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = tmem_base_sh;

  if (warp < kSoft2Warps) {
    // ------------------------------------------------------------ softmax
    const int g = warp >> 2, i = tid & 127;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t colS = 128u * g, colO = kColOa + 128u * g;
    const float c2 = a.scale_log2;
    bool ok = true;
    const int64_t grow = row0 + 128 * g + i;
    {
      // this thread's Q row into the SW128 K-major A tile of query tile g
      const uint4* src = reinterpret_cast<const uint4*>(a.Q + ((int64_t)h * a.M + grow) * kD);
      uint8_t* qt = Qs + g * 32768;
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        const uint4 x = grow < a.M ? src[c] : make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4*>(qt + sw128_off(i, c)) = x;
      }
      fence_async_smem();
      bar_arrive(q_ready);
    }
    for (int64_t t = 0; t < nt && ok; ++t) {
      const int nv = a.tiles[t_begin + t].y;
      if (!warp_all(bar_wait(&s_done[g], (uint32_t)(t & 1), &abort_sh, a.status))) { ok = false; break; }
      fence_after();
      const uint32_t sbase = tmem + lane_base + colS;
      float mx = -INFINITY;
      const bool ragged = nv < 128;
      for (int cb = 0; cb < 2; ++cb) {
        uint32_t v[64];
        tmem_ld64(sbase + 64 * cb, v);
        tmem_wait_ld();
        if (!ragged) {
#pragma unroll
          for (int k = 0; k < 64; k += 2) mx = max3f(mx, __uint_as_float(v[k]), __uint_as_float(v[k + 1]));
        } else {
#pragma unroll
          for (int k = 0; k < 64; ++k)
            if (64 * cb + k < nv) mx = fmaxf(mx, __uint_as_float(v[k]));
        }
      }
      const float mnew = fmaxf(m_run, mx * c2);
      // PV_g(t-1) has read P_g(t-1) and finished O_g before either changes
      if (t > 0) {
        if (!warp_all(bar_wait(&pv_done[g], (uint32_t)((t - 1) & 1), &abort_sh, a.status))) { ok = false; break; }
        fence_after();
      }
      const bool need = mnew > m_run + 8.f;
      if (t > 0 && __any_sync(0xffffffffu, need)) {
        const float corr = need ? ex2(m_run - mnew) : 1.f;
        for (int cb = 0; cb < 4; ++cb) {
          uint32_t v[32];
          tmem_ld32(tmem + lane_base + colO + 32 * cb, v);
          tmem_wait_ld();
#pragma unroll
          for (int k = 0; k < 32; ++k) v[k] = __float_as_uint(__uint_as_float(v[k]) * corr);
          tmem_st32(tmem + lane_base + colO + 32 * cb, v);
        }
        l_run *= corr;
      }
      if (need) m_run = mnew;
      float2 psum2 = make_float2(0.f, 0.f);
      const float2 c2v = make_float2(c2, c2), mv = make_float2(-m_run, -m_run);
      for (int cb = 0; cb < 2; ++cb) {
        uint32_t v[64], pk[32];
        tmem_ld64(sbase + 64 * cb, v);
        tmem_wait_ld();
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          const float2 arg = __ffma2_rn(make_float2(__uint_as_float(v[2 * k]), __uint_as_float(v[2 * k + 1])), c2v, mv);
          float2 pp = make_float2(ex2(arg.x), ex2(arg.y));
          if (ragged) {
            const int k0 = 64 * cb + 2 * k;
            pp.x = k0 < nv ? pp.x : 0.f;
            pp.y = k0 + 1 < nv ? pp.y : 0.f;
          }
          psum2 = __fadd2_rn(psum2, pp);
          const __half2 hp = __floats2half2_rn(pp.x, pp.y);
          pk[k] = *reinterpret_cast<const uint32_t*>(&hp);
        }
        // P over S columns already read (pair 32cb.. from columns 64cb..)
        tmem_st32(sbase + 32 * cb, pk);
      }
      l_run += psum2.x + psum2.y;
      tmem_wait_st();
      fence_before();
      bar_arrive(&p_ready[g]);
    }
    if (ok && nt > 0) ok = warp_all(bar_wait(&pv_done[g], (uint32_t)((nt - 1) & 1), &abort_sh, a.status));
    fence_after();
    sm_ok = ok;
  } else if (warp < kMmaWarp2) {
    // ------------------------------------------------------------ producers
    const int p = tid - kSoft2Warps * 32;      // 0..223
    int cur_slot = -1;
    bool ok = true;
    const uint32_t TB = (uint32_t)a.off.bytes;
    const uint8_t* tiles_h = a.cache + (int64_t)h * a.max_tiles * a.off.bytes;
    if (p == 0) {
      for (int64_t u = 0; u < 2 && u < nt; ++u) {
        bar_expect_tx(&full[u], TB);
        bulk_g2s(Ring + u * TB, tiles_h + (t_begin + u) * TB, TB, &full[u]);
      }
    }
    prod2_sync();
    for (int64_t t = 0; t < nt && ok; ++t) {
      const uint8_t* tb = Ring + (t & 1) * TB;
      const int slot = a.tiles[t_begin + t].x;
      if (!prod2_all(bar_wait(&full[t & 1], (uint32_t)((t >> 1) & 1), &abort_sh, a.status))) { ok = false; break; }
      // S_a(t-1) and S_b(t-1) have read k_hat, e and Z
      if (t > 0) {
        const uint32_t par = (uint32_t)((t - 1) & 1);
        if (!prod2_all(bar_wait(&s_done[0], par, &abort_sh, a.status) &&
                       bar_wait(&s_done[1], par, &abort_sh, a.status))) { ok = false; break; }
      }
      if constexpr (RP > 0) {
        if (slot != cur_slot) {
          cur_slot = slot;
          // stage U (fp32 [r][128]) in the free khi buffer, then Z = q U^T
          // for the CTA's 256 query rows (thread = row)
          float* Us = reinterpret_cast<float*>(Khi);
          const float* U = a.basis + ((int64_t)slot * a.H + h) * a.r * kD;
          for (int k = p; k < RP * kD; k += kProdThreads2) Us[k] = (k / kD) < a.r ? U[k] : 0.f;
          prod2_sync();
          for (int zr = p; zr < 256; zr += kProdThreads2) {
          float z[RP];
#pragma unroll
          for (int k = 0; k < RP; ++k) z[k] = 0.f;
          const int64_t grow = row0 + zr;
          const uint4* qrow = reinterpret_cast<const uint4*>(a.Q + ((int64_t)h * a.M + grow) * kD);
          for (int c8 = 0; c8 < 16; ++c8) {
            const uint4 qv = grow < a.M ? qrow[c8] : make_uint4(0, 0, 0, 0);
            const uint32_t qw[4] = {qv.x, qv.y, qv.z, qv.w};
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const float qf = __uint_as_float(e & 1 ? (qw[e >> 1] & 0xffff0000u) : (qw[e >> 1] << 16));
              const int c = 8 * c8 + e;
#pragma unroll
              for (int k = 0; k < RP; ++k) z[k] = fmaf(qf, Us[k * kD + c], z[k]);
            }
          }
          const int gq = zr >> 7, iq = zr & 127;
          uint8_t* zh = Zs + (2 * gq) * kZBytes;
          uint8_t* zl = zh + kZBytes;
#pragma unroll
          for (int j = 0; j < RP / 8; ++j) {
            uint32_t hw[4], lw[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const __half h0 = __float2half_rn(z[8 * j + 2 * e]), h1 = __float2half_rn(z[8 * j + 2 * e + 1]);
              const __half2 hh = __halves2half2(h0, h1);
              const __half2 ll = __floats2half2_rn(z[8 * j + 2 * e] - __half2float(h0),
                                                   z[8 * j + 2 * e + 1] - __half2float(h1));
              hw[e] = *reinterpret_cast<const uint32_t*>(&hh);
              lw[e] = *reinterpret_cast<const uint32_t*>(&ll);
            }
            const int off = ((iq >> 3) * (RP / 8) + j) * 128 + (iq & 7) * 16;
            *reinterpret_cast<uint4*>(zh + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
            *reinterpret_cast<uint4*>(zl + off) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
          }
          }
          prod2_sync();
        }
      }
      // ---- k_hat (hi, lo): item = (key, 32-channel group) ----
#pragma unroll 1
      for (int item = p; item < 512; item += kProdThreads2) {
        const int key = item >> 2, grp = item & 3;
        const int idx = cent_index(a.ib == 1 ? tb[a.off.idx + key] : reinterpret_cast<const uint16_t*>(tb + a.off.idx)[key], a.nC, a.status);
        const uint2 kc = *reinterpret_cast<const uint2*>(tb + a.off.kcode + key * 32 + grp * 8);
        const uint32_t qp = *reinterpret_cast<const uint32_t*>(tb + a.off.kqp + (key * G + grp) * 4);
        const float kz = __half2float(__ushort_as_half((unsigned short)(qp & 0xffffu)));
        const float ks = __half2float(__ushort_as_half((unsigned short)(qp >> 16)));
        const float2 kz2 = make_float2(kz, kz), ks2 = make_float2(ks, ks);
        const float* c32 = a.cent32 + ((int64_t)h * a.nC + idx) * kD;
        float4 craw[8];
#pragma unroll
        for (int c8 = 0; c8 < 4; ++c8) {
          const int chunk = grp * 4 + ((c8 + grp) & 3);
          craw[2 * c8] = __ldg(reinterpret_cast<const float4*>(c32 + 8 * chunk));
          craw[2 * c8 + 1] = __ldg(reinterpret_cast<const float4*>(c32 + 8 * chunk + 4));
        }
#pragma unroll
        for (int c8 = 0; c8 < 4; ++c8) {
          // chunk order rotated by the group: the 8 lanes of a store phase
          // (2 keys x 4 groups) then hit 8 different bank groups
          const int cl = (c8 + grp) & 3;
          const int chunk = grp * 4 + cl;
          const float2 cc4[4] = {make_float2(craw[2 * c8].x, craw[2 * c8].y), make_float2(craw[2 * c8].z, craw[2 * c8].w),
                                 make_float2(craw[2 * c8 + 1].x, craw[2 * c8 + 1].y),
                                 make_float2(craw[2 * c8 + 1].z, craw[2 * c8 + 1].w)};
          const uint32_t bits = ((cl >> 1) ? kc.y : kc.x) >> (16 * (cl & 1)) & 0xffffu;
          const float2 cds[4] = {codes_at<0>(bits), codes_at<4>(bits), codes_at<8>(bits), codes_at<12>(bits)};
          uint32_t ph[4], pl[4];
#pragma unroll
          for (int e2 = 0; e2 < 4; ++e2) {
            const float2 rq = __ffma2_rn(cds[e2], ks2, kz2);                 // zero + code*scale
            const float2 kv = __fadd2_rn(cc4[e2], rq);                       // + centroid
            split_bf16x2(kv, ph[e2], pl[e2]);
          }
          const int off = sw128_off(key, chunk);
          *reinterpret_cast<uint4*>(Khi + off) = make_uint4(ph[0], ph[1], ph[2], ph[3]);
          *reinterpret_cast<uint4*>(Klo + off) = make_uint4(pl[0], pl[1], pl[2], pl[3]);
        }
      }
      if constexpr (RP > 0) {
        if (p < 128) {
          // e rows: thread = key
          store_e_row<RP>(tb + a.off.e, p, a.r, Es);
        }
      }
      fence_async_smem();
      bar_arrive(k_ready);
      // ---- v_hat: PV_a(t-1) and PV_b(t-1) have read the previous one ----
      if (t > 0) {
        const uint32_t par = (uint32_t)((t - 1) & 1);
        if (!prod2_all(bar_wait(&pv_done[0], par, &abort_sh, a.status) &&
                       bar_wait(&pv_done[1], par, &abort_sh, a.status))) { ok = false; break; }
      }
      for (int item = p; item < 256; item += kProdThreads2) {
        const int key = item & 127, half = item >> 7;
        const uint4 vc = *reinterpret_cast<const uint4*>(tb + a.off.vcode + key * 32 + half * 16);
        const uint2 vq = *reinterpret_cast<const uint2*>(tb + a.off.vqp + (key * G + 2 * half) * 4);
        const uint32_t vw[4] = {vc.x, vc.y, vc.z, vc.w};
#pragma unroll
        for (int gg = 0; gg < 2; ++gg) {
          const uint32_t qv = gg ? vq.y : vq.x;
          const __half2 vz2 = __half2half2(__ushort_as_half((unsigned short)(qv & 0xffffu)));
          const __half2 vs2 = __half2half2(__ushort_as_half((unsigned short)(qv >> 16)));
#pragma unroll
          for (int c8 = 0; c8 < 4; ++c8) {
            const int chunk = half * 8 + gg * 4 + c8;
            const uint32_t bits = (vw[gg * 2 + (c8 >> 1)] >> (16 * (c8 & 1))) & 0xffffu;
            uint32_t w[4];
#pragma unroll
            for (int e2 = 0; e2 < 4; ++e2) {
              const __half2 hh = __hfma2(codes_h2(bits >> (4 * e2)), vs2, vz2);   // zero + code*scale
              w[e2] = *reinterpret_cast<const uint32_t*>(&hh);
            }
            *reinterpret_cast<uint4*>(Vt + sw128_off(key, chunk)) = make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
      }
      fence_async_smem();
      bar_arrive(v_ready);
      // every producer is done with ring stage t & 1: refill it with tile t + 2
      prod2_sync();
      if (p == 0 && t + 2 < nt) {
        bar_expect_tx(&full[t & 1], TB);
        bulk_g2s(Ring + (t & 1) * TB, tiles_h + (t_begin + t + 2) * TB, TB, &full[t & 1]);
      }
    }
  } else {
    // ------------------------------------------------------------ MMA issuer
    const bool leader = lane == 0;
    bool ok = true;
    const uint32_t qs = su32(Qs), kh = su32(Khi), kl = su32(Klo), vt = su32(Vt);
    const uint32_t ea = su32(Es), zs = su32(Zs);
    constexpr uint32_t kSbo = (RP / 8) * 128;
    ok = warp_all(bar_wait(q_ready, 0u, &abort_sh, a.status));
    fence_after();
    // streams: S_a, S_b, PV_a, PV_b.  S_g(n) needs k_hat(n) and PV_g(n-1)
    // issued; PV_g(n) needs S_g(n) issued, P_g(n) and v_hat(n).  The leader
    // alone polls and issues (the other lanes wait at the end), so the loop
    // costs as few issue slots as possible on the sub-partition it shares
    // with softmax and producer warps.
    if (leader && ok) {
      int64_t nS[2] = {0, 0}, nP[2] = {0, 0};
      long long last = clock64();
      while (nP[0] < nt || nP[1] < nt) {
        bool did = false;
#pragma unroll
        for (int g = 0; g < 2; ++g) {
          const int64_t n = nS[g];
          if (n < nt && nP[g] == n && bar_test(k_ready, (uint32_t)(n & 1))) {
            fence_after();
            const uint32_t d = tmem + 128u * g, qa = qs + 32768u * g;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const uint32_t ko = (j >> 2) * 16384 + (j & 3) * 32;
              mma_ss(d, desc_sw128(qa + ko), desc_sw128(kh + ko), kIdescQK, j > 0);
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const uint32_t ko = (j >> 2) * 16384 + (j & 3) * 32;
              mma_ss(d, desc_sw128(qa + ko), desc_sw128(kl + ko), kIdescQK, 1);
            }
            if constexpr (RP > 0) {
              const uint32_t zh = zs + 2u * g * kZBytes, zl = zh + kZBytes;
#pragma unroll
              for (int kk = 0; kk < RP / 16; ++kk) {
                mma_ss(d, desc_none(zh + 256 * kk, 128, kSbo), desc_none(ea + 256 * kk, 128, kSbo), kIdescF16, 1);
                mma_ss(d, desc_none(zl + 256 * kk, 128, kSbo), desc_none(ea + 256 * kk, 128, kSbo), kIdescF16, 1);
              }
            }
            commit(&s_done[g]);
            ++nS[g];
            did = true;
          }
        }
#pragma unroll
        for (int g = 0; g < 2; ++g) {
          const int64_t n = nP[g];
          if (n < nS[g] && bar_test(&p_ready[g], (uint32_t)(n & 1)) && bar_test(v_ready, (uint32_t)(n & 1))) {
            fence_after();
            const uint32_t ps = tmem + 128u * g;
#pragma unroll
            for (int j = 0; j < 8; ++j)
              mma_ts(tmem + kColOa + 128u * g, ps + 8 * j, desc_sw128_mn(vt + 2048 * j), kIdescPV,
                     (n > 0 || j > 0) ? 1u : 0u);
            commit(&pv_done[g]);
            ++nP[g];
            did = true;
          }
        }
        if (did) {
          last = clock64();
        } else if (abort_sh) {
          ok = false;
          break;
        } else if (clock64() - last > kWaitCycles) {
          abort_sh = 1;
          atomicOr(a.status, kDevTimeout);
          ok = false;
          break;
        }
      }
      // the last PVs complete before the TMEM is released (bounded)
      if (ok && nt > 0) {
        bar_wait(&pv_done[0], (uint32_t)((nt - 1) & 1), &abort_sh, a.status);
        bar_wait(&pv_done[1], (uint32_t)((nt - 1) & 1), &abort_sh, a.status);
      }
    }
    __syncwarp();
  }

  fence_before();
  __syncthreads();
  fence_after();
  // ------------------------------------------------------------ epilogue
  {
    const int g = (warp >> 2) & 1, i = tid & 127;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t colO = kColOa + 128u * g;
    const int64_t grow = row0 + 128 * g + i;
    const bool softmax = warp < kSoft2Warps;
    float* recv = reinterpret_cast<float*>(sm) + (128 * g + i) * kRecvLd;   // rank 0's buffers, now free
    float f0 = 1.f, f1 = 0.f, inv = 0.f;
    bool store = softmax && sm_ok;
    if (nsplit > 1) {
      cluster_sync();   // both CTAs are past their tiles
      if (softmax && split == 1) {
        const uint32_t dst = map_rank(su32(recv), 0);
        for (int cb = 0; cb < 4; ++cb) {
          uint32_t v[32];
          tmem_ld32(tmem + lane_base + colO + 32 * cb, v);
          tmem_wait_ld();
#pragma unroll
          for (int q = 0; q < 8; ++q) st_cluster_v4(dst + (32 * cb + 4 * q) * 4, v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
        }
        st_cluster_v4(dst + 128 * 4, __float_as_uint(m_run), __float_as_uint(l_run), sm_ok ? 1u : 0u, 0u);
      }
      cluster_sync();   // the partials of rank 1 have landed
      store = store && split == 0;
      if (store) {
        const float m1 = recv[128], l1 = recv[129];
        store = __float_as_uint(recv[130]) != 0u;
        const float mm = fmaxf(m_run, m1);
        f0 = m_run == -INFINITY ? 0.f : ex2(m_run - mm);
        f1 = m1 == -INFINITY ? 0.f : ex2(m1 - mm);
        const float l = l_run * f0 + l1 * f1;
        inv = l > 0.f ? 1.f / l : 0.f;
      }
    } else {
      inv = l_run > 0.f ? 1.f / l_run : 0.f;
    }
    // every lane of a softmax warp loads (warp-collective); valid rows store
    if (softmax && __any_sync(0xffffffffu, store)) {
      __nv_bfloat16* dst = a.O + ((int64_t)h * a.M + grow) * kD;
      for (int cb = 0; cb < 4; ++cb) {
        uint32_t v[32];
        tmem_ld32(tmem + lane_base + colO + 32 * cb, v);
        tmem_wait_ld();
        if (store && grow < a.M) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int c = 32 * cb + 8 * q + 2 * e;
              float o0 = __uint_as_float(v[8 * q + 2 * e]) * f0, o1 = __uint_as_float(v[8 * q + 2 * e + 1]) * f0;
              if (nsplit > 1) {
                o0 = fmaf(recv[c], f1, o0);
                o1 = fmaf(recv[c + 1], f1, o1);
              }
              const __nv_bfloat162 bb = __floats2bfloat162_rn(o0 * inv, o1 * inv);
              w[e] = *reinterpret_cast<const uint32_t*>(&bb);
            }
            *reinterpret_cast<uint4*>(dst + 32 * cb + 8 * q) = make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
      }
    }
  }
  fence_before();
  __syncthreads();
  fence_after();
  if (warp == kMmaWarp2) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem));
}

size_t tc_smem(const qwm_ctx* c, int RP, bool cs) {
  return 1024 + 3 * 32768 + 3 * (size_t)128 * RP * 2 + 2 * c->lay.tile_bytes +
         (cs ? (size_t)c->cfg.n_centroids * 256 : 0);
}

template <int RP, bool CS>
cudaError_t launch_rp(const qwm_ctx* c, const TcArgs& a, int64_t M, cudaStream_t st) {
  const size_t smem = tc_smem(c, RP, CS);
  auto kern = attend_tc_kernel<RP, CS>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)((M + 127) / 128), (unsigned)c->cfg.heads);
  kern<<<grid, kThreads, smem, st>>>(a);
  return cudaGetLastError();
}

size_t tc2_smem(const qwm_ctx* c, int RP) {
  return 1024 + 5 * 32768 + 5 * (size_t)128 * RP * 2 + 2 * c->lay.tile_bytes;
}

// KV splits per query-row pair: 2 (a cluster of two CTAs) when that cuts
// the number of full waves over the SMs, else 1
int tc2_splits(const qwm_ctx* c, int64_t M) {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      sms < 1)
    return 1;
  const int64_t units = ((M + 255) / 256) * c->cfg.heads;
  const int64_t w1 = (units + sms - 1) / sms;         // waves with one split
  const int64_t w2x2 = (2 * units + sms - 1) / sms;   // twice the waves with two splits
  return (c->n_tiles >= 2 && w2x2 < 2 * w1) ? 2 : 1;
}

template <int RP>
cudaError_t launch_tc2(const qwm_ctx* c, const TcArgs& a, int64_t M, cudaStream_t st) {
  const size_t smem = tc2_smem(c, RP);
  auto kern = attend_tc2_kernel<RP>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int ns = tc2_splits(c, M);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((M + 255) / 256), (unsigned)c->cfg.heads, (unsigned)ns);
  cfg.blockDim = dim3(kThreads2, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = (unsigned)ns;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kern, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

TcArgs tc_args(const qwm_ctx* c, const void* q, int64_t M, float scale, void* out) {
  TcArgs a;
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
  a.cent32 = c->cent32;
  a.nC = c->cfg.n_centroids;
  a.basis = c->basis;
  a.H = c->cfg.heads;
  a.r = c->cfg.rank;
  a.ib = c->ib;
  a.status = c->status;
  return a;
}

}  // namespace

bool attend_tc_supported(const qwm_ctx* c) {
  return c->cfg.dtype == QWM_BF16 && c->cfg.head_dim == kD && c->cfg.rank <= 32;
}

bool attend_tc2_supported(const qwm_ctx* c) {
  return c->cfg.dtype == QWM_BF16 && c->cfg.head_dim == kD && c->cfg.rank <= 16 &&
         tc2_smem(c, c->cfg.rank == 0 ? 0 : 16) <= 227 * 1024;
}

cudaError_t launch_attend_tc(const qwm_ctx* c, const void* q, int64_t M, float scale, void* out,
                             cudaStream_t st) {
  const TcArgs a = tc_args(c, q, M, scale, out);
  const int RP = a.r == 0 ? 0 : (a.r <= 16 ? 16 : 32);
  const bool cs = c->cfg.n_centroids <= 256;
  if (RP == 0) return cs ? launch_rp<0, true>(c, a, M, st) : launch_rp<0, false>(c, a, M, st);
  if (RP == 16) return cs ? launch_rp<16, true>(c, a, M, st) : launch_rp<16, false>(c, a, M, st);
  return cs ? launch_rp<32, true>(c, a, M, st) : launch_rp<32, false>(c, a, M, st);
}

cudaError_t launch_attend_tc2(const qwm_ctx* c, const void* q, int64_t M, float scale, void* out,
                              cudaStream_t st) {
  const TcArgs a = tc_args(c, q, M, scale, out);
  return a.r == 0 ? launch_tc2<0>(c, a, M, st) : launch_tc2<16>(c, a, M, st);
}

}  // namespace qwm
