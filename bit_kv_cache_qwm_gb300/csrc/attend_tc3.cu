// qwm_attend, sm_103a tensor-core kernel with the key split into centroid and
// residual (kernel 6, the default for bf16 caches at d = 128, r <= 16).
//
// Attention over the packed cache with PSAC compensation (QuantWM Abstract;
// roboind article, "Step 2"):
//   l_n = q . k_hat_n + (q U_t^T) . e_n,   O = softmax(scale * l) V_hat,
// with k_hat_n = C[j_n] + rho_hat_n, rho_hat = zero + code * scale per group.
// The logit is taken apart along that sum, all in float16 MMAs with float32
// accumulation:
//   q . k_hat = q . C[j]        (the bf16 centroid row, exact in float16)
//             + q . rho_hat     (the dequantised residual, one float16 rounding)
// so the only rounding of the key is that of the residual, whose range is a
// fraction of the key's (the centroid carries the rest).  Q enters as float16
// scaled per row by a power of two that keeps its largest entry below 2^15
// (exact; the softmax multiplies the logits back).  Every float16 operand
// holds the channels of each 16-channel block in the order
// 0, 8, 1, 9, ..., 7, 15, so that one shift and one mask of a packed 32-bit
// code word give the two 2-bit codes of a float16 pair; Q, the centroid
// table and V_hat use the same order and the output is put back in channel
// order when it is stored.
//
// One CTA owns 256 query rows (two M = 128 tiles a, b) of one head and
// streams its 128-key tiles (the few-row mode, kernel 7: one tile of 128
// rows, the tiles of the cache split over gridDim.z CTAs whose partial
// results a second kernel merges).  Warp roles (16 warps):
//   warps 0-3 / 4-7  softmax of query tile a / b: thread = row = TMEM lane.
//                    Write the row's scaled float16 Q into a SW128 K-major
//                    shared tile once (the A operand of the S MMAs), then per
//                    tile: online softmax in the exp2 domain with a lazy
//                    rescale of O (only when the running maximum grows by
//                    more than 2^8), P in float16 over the first 64 columns
//                    of S, then arrive on the tile's "P written" barrier.
//   warps 8-11       key producers, per tile: gather the centroid rows (B1,
//                    asynchronous 16-byte copies) once the centroid parts of
//                    the previous tile are done, then write the residuals
//                    (B2), the e rows and Z = q U_t^T (float16) when a tile's
//                    basis slot changes (double-buffered, so a basis change
//                    never waits) once its S MMAs are done.
//   warps 12-14      value producers: one thread bulk-copies every packed
//                    tile into a 2-stage shared ring (a stage is refilled
//                    once both groups are done with it); per tile all write
//                    V_hat once the previous tile's PV MMAs are done.  The
//                    two groups run their loops independently, so the value
//                    dequantisation of a tile overlaps the key work of the
//                    next.
//   warp 15          MMA issuer and TMEM owner: per tile t, in a fixed order,
//                    for g = a, b: O_g += P_g(t-1) V_hat(t-1) (A = P in
//                    TMEM), S_g = Q_g B1^T (centroid part); then S_g +=
//                    Q_g B2^T + Z_g E^T (residual and PSAC parts).  The whole
//                    warp waits, one elected lane issues.  The centroid part
//                    only needs B1, so it runs on the tensor pipe while the
//                    producers still compute B2.  S_g(t) is issued after
//                    PV_g(t-1), so the tensor pipe's in-order execution keeps
//                    P_g(t-1) intact until PV_g(t-1) has read it.
// Handoffs between threads (P written, V_hat written, B1 gathered, B2
// written) use named barriers: an mbarrier wait goes through the shared-memory pipe,
// which the MMAs' operand reads and the producers' stores keep busy (a wait
// on a completed mbarrier then takes hundreds of cycles).  The tensor pipe's
// completions (S done, PV done, B1 free) arrive on mbarriers.
// TMEM columns: S_a [0,128), S_b [128,256), O_a [256,384), O_b [384,512).
// Split KV: with gridDim.z = 2 the two CTAs of a cluster take the two halves
// of the tile range for the same rows; rank 1 sends its unnormalised O,
// running maximum and sum to rank 0 through distributed shared memory and
// rank 0 merges them (log-sum-exp).
// Every mbarrier wait is bounded by the SM clock; a timeout sets a device
// status bit and every role leaves its loop (a role that leaves arrives once
// more on the named barriers it feeds, and a role that waits on one reads the
// abort flag after each wait and stops before the next), the TMEM is freed
// and the kernel returns.
#include <math.h>

#include "qwm_internal.cuh"
#include "tcgen05_util.cuh"

namespace qwm {
namespace {

using namespace tcx;

constexpr int kD = 128;
// 16 warps: 4 per SM sub-partition, which leaves 128 registers a thread
constexpr int kSoftW = 8, kKeyW = 4, kValW = 3;
constexpr int kThreads3 = (kSoftW + kKeyW + kValW + 1) * 32;   // 512
constexpr int kMmaW = kSoftW + kKeyW + kValW;                  // 15
constexpr int kKeyT = kKeyW * 32, kValT = kValW * 32;          // 128, 96
constexpr uint32_t kColO = 256;
// float16 x float16 -> float32, M = 128, N = 128: S (both operands K-major)
// and PV (MN-major B)
constexpr uint32_t kIdescS = (1u << 4) | (16u << 17) | (8u << 24);
constexpr uint32_t kIdescPV = kIdescS | (1u << 16);
// shared-memory layout (bytes from the 1 KiB aligned base)
constexpr int kTileOp = 32768;                // one 128 x 128 float16 operand tile
constexpr int kOffB1 = 2 * kTileOp;           // after Q_a, Q_b
constexpr int kOffB2 = kOffB1 + kTileOp;
constexpr int kOffV = kOffB2 + kTileOp;
constexpr int kOffE = kOffV + kTileOp;        // 128 keys x 16 coefficients
constexpr int kZBuf = 128 * 16 * 2;           // 128 rows x 16 (one query tile)
constexpr int kOffZ = kOffE + kZBuf;
constexpr int kOffU = kOffZ + 4 * kZBuf;      // [Z buffer][query tile]
constexpr int kOffQsc = kOffU + 16 * kD * 4;
constexpr int kOffZsel = kOffQsc + 256 * 4;
constexpr int kOffRing = kOffZsel + 64;
constexpr int kRecvLd = 132;                  // floats per row of a received partial: O[128], m, l, ok, pad
static_assert(kRecvLd == kPartRowFloats, "the few-row mode writes rows of the combine kernel's partials");

struct Tc3Args {
  const __nv_bfloat16* Q;
  __nv_bfloat16* O;
  int64_t M;
  float scale_log2;
  const uint8_t* cache;
  int64_t max_tiles;
  TileOffsets off;
  int64_t n_tiles;
  const int2* tiles;
  const __half* cent16;   // [H][C][128] float16, channel order of the blocks above
  int nC;
  const float* basis;
  int H;
  int r;
  int ib;
  uint32_t* status;
  // few-row mode: the KV range split over gridDim.z CTAs (no cluster), each
  // writing its unnormalised O, running maximum and sum for every row below
  // M to part[((h n_mb + row / 16) n_split + split) 16 + row % 16][kRecvLd]
  float* part;
  int n_mb;
};

// named barriers of the key producers (1; KT threads) and the value producers (2)
template <int KT>
__device__ __forceinline__ void key_sync3() { asm volatile("bar.sync 1, %0;" ::"n"(KT) : "memory"); }
__device__ __forceinline__ void val_sync3() { asm volatile("bar.sync 2, %0;" ::"n"(kValT) : "memory"); }
// named barrier "V_hat of the tile written" (5): the value producers arrive,
// the MMA warp waits.  A named barrier does not pass through the
// shared-memory pipe, which the MMAs' operand reads and the producers' stores
// keep busy, so the handoff costs tens of cycles instead of hundreds.
__device__ __forceinline__ void vready_arrive() { asm volatile("bar.arrive 5, %0;" ::"n"(kValT + 32) : "memory"); }
__device__ __forceinline__ void vready_sync() { asm volatile("bar.sync 5, %0;" ::"n"(kValT + 32) : "memory"); }
// The MMA warp's other inputs arrive on named barriers too: "P_g of keys 0-63
// written" (11 + g), "P_g of keys 64-95 written" (13 + g) and "P_g written"
// (7 + g; the four softmax warps of tile g arrive, and PV_g runs in three
// parts as its keys' P is ready), "B1 gathered" (9) and "B2, e, Z written"
// (10; the key producers arrive).  Whoever arrives does so once
// per tile, and once more for the tile it was on if it gives up; the MMA warp
// reads the abort flag after each tile's last wait and stops at the next, so
// no named-barrier wait is left without its arrival.
constexpr int kNbP = 7, kNbKc = 9, kNbKr = 10, kNbP1 = 11, kNbP2 = 13;
__device__ __forceinline__ void nbar_arrive(int id, int n) { asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(n) : "memory"); }
__device__ __forceinline__ void nbar_sync(int id, int n) { asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory"); }
// named barriers of the softmax warps of query tile g (3 + g; 128 threads)
__device__ __forceinline__ bool soft_all3(int g, bool v) {
  uint32_t r;
  asm volatile("{\n.reg .pred p, q;\nsetp.ne.u32 p, %1, 0;\nbar.red.and.pred q, %2, 128, p;\n"
               "selp.u32 %0, 1, 0, q;\n}"
               : "=r"(r) : "r"((uint32_t)v), "r"(3 + g) : "memory");
  return r != 0;
}
template <int KT>
__device__ __forceinline__ bool key_all3(bool v) {
  uint32_t r;
  asm volatile("{\n.reg .pred p, q;\nsetp.ne.u32 p, %1, 0;\nbar.red.and.pred q, 1, %2, p;\n"
               "selp.u32 %0, 1, 0, q;\n}"
               : "=r"(r) : "r"((uint32_t)v), "n"(KT) : "memory");
  return r != 0;
}
__device__ __forceinline__ bool val_all3(bool v) {
  uint32_t r;
  asm volatile("{\n.reg .pred p, q;\nsetp.ne.u32 p, %1, 0;\nbar.red.and.pred q, 2, %2, p;\n"
               "selp.u32 %0, 1, 0, q;\n}"
               : "=r"(r) : "r"((uint32_t)v), "n"(kValT) : "memory");
  return r != 0;
}

// byte offset of 16-byte chunk `chunk` (0..15) of row `row` (0..127) in a
// 128 x 128 16-bit tile stored as two SW128 K-major atoms of 64 elements
__device__ __forceinline__ int op_off(int row, int chunk) {
  return (chunk >> 3) * 16384 + (row >> 3) * 1024 + (row & 7) * 128 + (((chunk & 7) ^ (row & 7)) << 4);
}

// zero + code * scale for the codes of channels (c, c + 8) of a 16-channel
// block, which sit 16 bits apart in the block's 32-bit code word w: one
// shift and one mask give both codes as the low mantissa bits of 1024 + code
// (exact in float16), then one subtraction and one fused multiply-add.
template <int I>
__device__ __forceinline__ uint32_t dq_pair(uint32_t w, __half2 s2, __half2 z2) {
  const uint32_t t = ((w >> (2 * I)) & 0x00030003u) | 0x64006400u;
  const __half2 c = __hsub2(*reinterpret_cast<const __half2*>(&t), __float2half2_rn(1024.f));
  const __half2 r = __hfma2(c, s2, z2);
  return *reinterpret_cast<const uint32_t*>(&r);
}

// The 16 channels of block b (code word w, group parameters qp) into chunks
// 2b and 2b + 1 of `row`.  The first store of blocks 4-7 goes to the odd
// chunk, so the 8 lanes of a store phase (one row, blocks 0-7) hit 8
// different bank groups.
__device__ __forceinline__ void dq_block(uint8_t* tile, int row, int b, uint32_t w, uint32_t qp) {
  const __half2 z2 = __half2half2(__ushort_as_half((unsigned short)(qp & 0xffffu)));
  const __half2 s2 = __half2half2(__ushort_as_half((unsigned short)(qp >> 16)));
  const uint4 lo = make_uint4(dq_pair<0>(w, s2, z2), dq_pair<1>(w, s2, z2), dq_pair<2>(w, s2, z2), dq_pair<3>(w, s2, z2));
  const uint4 hi = make_uint4(dq_pair<4>(w, s2, z2), dq_pair<5>(w, s2, z2), dq_pair<6>(w, s2, z2), dq_pair<7>(w, s2, z2));
  if (b < 4) {
    *reinterpret_cast<uint4*>(tile + op_off(row, 2 * b)) = lo;
    *reinterpret_cast<uint4*>(tile + op_off(row, 2 * b + 1)) = hi;
  } else {
    *reinterpret_cast<uint4*>(tile + op_off(row, 2 * b + 1)) = hi;
    *reinterpret_cast<uint4*>(tile + op_off(row, 2 * b)) = lo;
  }
}

__device__ __forceinline__ float bf16_at(const uint4* x, int ch) {
  const uint4 v = x[ch >> 3];
  const int e = (ch & 7) >> 1;
  const uint32_t w = e == 0 ? v.x : e == 1 ? v.y : e == 2 ? v.z : v.w;
  return __uint_as_float((ch & 1) ? (w & 0xffff0000u) : (w << 16));
}

// online-softmax step of one row over the 16 Q keys key0 .. key0 + 16 Q - 1
// of a tile held in v[0 .. 16 Q - 1]: P (float16 pairs) into TMEM columns
// key0 / 2 .. of the row's S buffer; returns the sum of the P values
// (FULL: all 128 keys of the tile are valid, no per-key test)
template <int Q, bool FULL>
__device__ __forceinline__ float exp_keys(const uint32_t* v, int key0, int nv, float2 c2v, float2 mv,
                                          uint32_t taddr) {
  float2 ps = make_float2(0.f, 0.f);
#pragma unroll
  for (int q = 0; q < Q; ++q) {
    uint32_t pk[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int k0 = 16 * q + 2 * k, key = key0 + k0;
      const float2 arg = __ffma2_rn(make_float2(__uint_as_float(v[k0]), __uint_as_float(v[k0 + 1])), c2v, mv);
      float2 pp = make_float2(ex2(arg.x), ex2(arg.y));
      if (!FULL) {
        pp.x = key < nv ? pp.x : 0.f;
        pp.y = key + 1 < nv ? pp.y : 0.f;
      }
      ps = __fadd2_rn(ps, pp);
      const __half2 hp = __floats2half2_rn(pp.x, pp.y);
      pk[k] = *reinterpret_cast<const uint32_t*>(&hp);
    }
    tmem_st8(taddr + key0 / 2 + 8 * q, pk);
  }
  return ps.x + ps.y;
}

// NQ: query tiles of 128 rows per CTA (2; 1 in the few-row mode)
template <int RP, int NQ>
__global__ void __launch_bounds__(kThreads3, 1) attend_tc3_kernel(const Tc3Args a) {
  extern __shared__ __align__(1024) uint8_t sm_raw[];
  uint8_t* sm = sm_raw + ((1024 - (su32(sm_raw) & 1023)) & 1023);
  uint8_t* Qs = sm;
  uint8_t* B1 = sm + kOffB1;
  uint8_t* B2 = sm + kOffB2;
  uint8_t* Vt = sm + kOffV;
  uint8_t* Es = sm + kOffE;
  uint8_t* ZS = sm + kOffZ;
  float* US = reinterpret_cast<float*>(sm + kOffU);
  float* QSC = reinterpret_cast<float*>(sm + kOffQsc);
  uint8_t* Ring = sm + kOffRing;
  __shared__ __align__(8) uint64_t bars[15];
  __shared__ uint32_t tmem_base_sh;
  __shared__ volatile int abort_sh;
  uint64_t* b1_free = &bars[3];    // the centroid parts of S_a(t) and S_b(t) done
  uint64_t* s_done = &bars[4];     // [2] S_g(t) complete
  uint64_t* pv_done = &bars[8];    // [2] O_g += P_g(t) V(t) done
  uint64_t* full = &bars[10];      // [2] packed tile landed in ring stage
  uint64_t* q_ready = &bars[12];
  uint64_t* ring_free = &bars[13];  // [2] the key producers are done with the ring stage

  const int tid = threadIdx.x, warp = tid >> 5;
  const int h = blockIdx.y;
  const int64_t row0 = (int64_t)blockIdx.x * 128 * NQ;
  // key producers: warps 4 NQ .. 11 (with one query tile the second tile's
  // softmax warps join them)
  constexpr int KT = kKeyT + 128 * (2 - NQ);
  const bool partial = a.part != nullptr;
  const int nsplit = (int)gridDim.z;
  const int split = partial ? (int)blockIdx.z : (nsplit > 1 ? (int)cluster_rank() : 0);
  const int t_begin = (int)(a.n_tiles * split / nsplit);
  const int nt = (int)(a.n_tiles * (split + 1) / nsplit) - t_begin;
  float m_run = -INFINITY, l_run = 0.f;      // softmax row state, used by the epilogue
  bool sm_ok = false;

  if (tid == 0) {
    abort_sh = 0;
    bar_init(&ring_free[0], 1);
    bar_init(&ring_free[1], 1);
    bar_init(b1_free, 1);
    for (int g = 0; g < 2; ++g) {
      bar_init(&s_done[g], 1);
      bar_init(&pv_done[g], 1);
      bar_init(&full[g], 1);
    }
    bar_init(q_ready, 128 * NQ);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == kMmaW) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(su32(&tmem_base_sh)));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = tmem_base_sh;

  if (warp < 4 * NQ) {
    // ------------------------------------------------------------ softmax
    const int g = warp >> 2, i = tid & 127;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t colS = 128u * g;
    const int64_t grow = row0 + 128 * g + i;
    float c2;
    {
      // Q row -> float16 x 2^-e (largest entry below 2^15) in the pair order
      // of the operands, into the SW128 K-major A tile of query tile g
      const uint4* src = reinterpret_cast<const uint4*>(a.Q + ((int64_t)h * a.M + grow) * kD);
      float mx = 0.f;
      if (grow < a.M) {
#pragma unroll 4
        for (int c = 0; c < 16; ++c) {
          const uint4 xv = src[c];
          const uint32_t w[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
          for (int e = 0; e < 4; ++e)
            mx = max3f(mx, fabsf(__uint_as_float(w[e] << 16)), fabsf(__uint_as_float(w[e] & 0xffff0000u)));
        }
      }
      const int ex = (int)((__float_as_uint(mx) >> 23) & 0xffu) - 127;
      const int e = ex > 14 ? ex - 14 : 0;
      const float qs = __uint_as_float((uint32_t)(127 - e) << 23);   // 2^-e
      QSC[128 * g + i] = qs;
      c2 = a.scale_log2 * __uint_as_float((uint32_t)(127 + e) << 23);
      uint8_t* qt = Qs + g * kTileOp;
#pragma unroll
      for (int b = 0; b < 8; ++b) {
        // channels 16 b .. 16 b + 15 -> chunks 2 b, 2 b + 1
        uint4 x[2];
        x[0] = grow < a.M ? src[2 * b] : make_uint4(0, 0, 0, 0);
        x[1] = grow < a.M ? src[2 * b + 1] : make_uint4(0, 0, 0, 0);
        uint32_t w[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const __half2 hh = __floats2half2_rn(bf16_at(x, k) * qs, bf16_at(x, k + 8) * qs);
          w[k] = *reinterpret_cast<const uint32_t*>(&hh);
        }
        *reinterpret_cast<uint4*>(qt + op_off(i, 2 * b)) = make_uint4(w[0], w[1], w[2], w[3]);
        *reinterpret_cast<uint4*>(qt + op_off(i, 2 * b + 1)) = make_uint4(w[4], w[5], w[6], w[7]);
      }
      fence_async_smem();
      bar_arrive(q_ready);
    }
    bool ok = true;
    int t = 0;
    for (; t < nt && ok; ++t) {
      const int nv = a.tiles[t_begin + t].y;
      // one warp of the group polls the mbarrier (each poll is a trip through
      // the busy shared-memory pipe); the vote hands the result to the others
      if (!soft_all3(g, (warp & 3) != 0 || bar_wait(&s_done[g], (uint32_t)(t & 1), &abort_sh, a.status))) {
        ok = false;
        break;
      }
      fence_after();
      const uint32_t sbase = tmem + lane_base + colS;
      // keys 64-127: their maximum; then keys 0-63, which stay in registers
      uint32_t v[64];
      tmem_ld64(sbase + 64, v);
      tmem_wait_ld();
      float mx0 = -INFINITY, mx1 = -INFINITY;
      if (nv >= 128) {
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          mx0 = max3f(mx0, __uint_as_float(v[4 * k]), __uint_as_float(v[4 * k + 1]));
          mx1 = max3f(mx1, __uint_as_float(v[4 * k + 2]), __uint_as_float(v[4 * k + 3]));
        }
      } else {
#pragma unroll
        for (int k = 0; k < 64; ++k)
          if (64 + k < nv) mx0 = fmaxf(mx0, __uint_as_float(v[k]));
      }
      tmem_ld64(sbase, v);
      tmem_wait_ld();
      if (nv >= 64) {
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          mx0 = max3f(mx0, __uint_as_float(v[4 * k]), __uint_as_float(v[4 * k + 1]));
          mx1 = max3f(mx1, __uint_as_float(v[4 * k + 2]), __uint_as_float(v[4 * k + 3]));
        }
      } else {
#pragma unroll
        for (int k = 0; k < 64; ++k)
          if (k < nv) mx0 = fmaxf(mx0, __uint_as_float(v[k]));
      }
      const float mnew = fmaxf(m_run, fmaxf(mx0, mx1) * c2);
      // S_g(t) follows PV_g(t-1) in the tensor pipe's order, so O_g is complete
      const bool need = mnew > m_run + 8.f;
      if (t > 0 && __any_sync(0xffffffffu, need)) {
        const float corr = need ? ex2(m_run - mnew) : 1.f;
        const uint32_t colO = kColO + 128u * g;
        // in 16-column pieces: the 64 S values stay in registers meanwhile
#pragma unroll 1
        for (int cb = 0; cb < 8; ++cb) {
          uint32_t o[16];
          tmem_ld16(tmem + lane_base + colO + 16 * cb, o);
          tmem_wait_ld();
#pragma unroll
          for (int k = 0; k < 16; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * corr);
          tmem_st16(tmem + lane_base + colO + 16 * cb, o);
        }
        l_run *= corr;
      }
      if (need) m_run = mnew;
      const float2 c2v = make_float2(c2, c2), mv = make_float2(-m_run, -m_run);
      // keys 0-63 first (they are in registers; their P goes over S columns
      // 0-31, already read), then keys 64-127 again from TMEM (S columns
      // 64-127, untouched), whose P goes over columns 32-63
      float psum = nv >= 128 ? exp_keys<4, true>(v, 0, nv, c2v, mv, sbase) : exp_keys<4, false>(v, 0, nv, c2v, mv, sbase);
      // P of keys 0-63 written: the MMA warp may start PV_g(t) on them
      tmem_wait_st();
      fence_before();
      nbar_arrive(kNbP1 + g, 160);
#pragma unroll 1
      for (int hq = 0; hq < 2; ++hq) {
        uint32_t w[32];
        tmem_ld32(sbase + 64 + 32 * hq, w);
        tmem_wait_ld();
        psum += nv >= 128 ? exp_keys<2, true>(w, 64 + 32 * hq, nv, c2v, mv, sbase)
                          : exp_keys<2, false>(w, 64 + 32 * hq, nv, c2v, mv, sbase);
        if (hq == 0) {
          // P of keys 64-95 written too
          tmem_wait_st();
          fence_before();
          nbar_arrive(kNbP2 + g, 160);
        }
      }
      tmem_wait_st();
      l_run += psum;
      fence_before();
      // P_g(t) written: the MMA warp issues PV_g(t) once the tile's four
      // warps have arrived
      nbar_arrive(kNbP + g, 160);
    }
    // a group that gave up before writing P_g(t) still lets the MMA warp pass
    // its wait for it
    if (!ok && t < nt) {
      nbar_arrive(kNbP1 + g, 160);
      nbar_arrive(kNbP2 + g, 160);
      nbar_arrive(kNbP + g, 160);
    }
    if (ok && nt > 0) ok = warp_all(bar_wait(&pv_done[g], (uint32_t)((nt - 1) & 1), &abort_sh, a.status));
    fence_after();
    sm_ok = ok;
  } else if (warp < kSoftW + kKeyW) {
    // ------------------------------------------------------------ key producers
    const int p = tid - 128 * NQ, kw = p >> 5;   // 0 .. KT - 1, its warp in the group
    const uint32_t TB = (uint32_t)a.off.bytes;
    const __half* c16 = a.cent16 + (int64_t)h * a.nC * kD;
    int cur_slot = -1, zb = 1;
    bool ok = true;
    // Z needs the per-row scales of Q the softmax warps publish
    bool kc_due = true;   // the tile's "B1 gathered" arrival is still due
    if constexpr (RP > 0) ok = key_all3<KT>(bar_wait(q_ready, 0u, &abort_sh, a.status));
    for (int t = 0; t < nt && ok; ++t) {
      kc_due = true;
      const uint8_t* tb = Ring + (t & 1) * TB;
      const uint32_t pp = (uint32_t)((t - 1) & 1);
      // one warp of the group polls each mbarrier; the vote hands the result on
      if (!key_all3<KT>(kw != 0 || bar_wait(&full[t & 1], (uint32_t)((t >> 1) & 1), &abort_sh, a.status))) {
        ok = false;
        break;
      }
      // ---- B1: the centroid parts of S_a(t-1) and S_b(t-1) have read it
      if (t > 0 && !key_all3<KT>(kw != 0 || bar_wait(b1_free, pp, &abort_sh, a.status))) {
        ok = false;
        break;
      }
      {
        // thread: one 16-byte chunk of NK consecutive keys, their indices in
        // one or two 16-byte loads (a warp covers whole 256-byte centroid rows)
        constexpr int NK = 2048 / KT;
        const int chunk = p & 15, k0 = NK * (p >> 4);
        uint32_t iw[NK / 2];
        if (a.ib == 1) {
#pragma unroll
          for (int q = 0; q < NK / 16 + (NK < 16); ++q) {
            if constexpr (NK >= 16) {
              const uint4 w = *reinterpret_cast<const uint4*>(tb + a.off.idx + k0 + 16 * q);
              iw[4 * q] = w.x, iw[4 * q + 1] = w.y, iw[4 * q + 2] = w.z, iw[4 * q + 3] = w.w;
            } else {
              const uint2 w = *reinterpret_cast<const uint2*>(tb + a.off.idx + k0);
              iw[0] = w.x, iw[1] = w.y;
            }
          }
        } else {
#pragma unroll
          for (int q = 0; q < NK / 8; ++q) {
            const uint4 w = *reinterpret_cast<const uint4*>(tb + a.off.idx + 2 * k0 + 16 * q);
            iw[4 * q] = w.x, iw[4 * q + 1] = w.y, iw[4 * q + 2] = w.z, iw[4 * q + 3] = w.w;
          }
        }
        const __half* csrc = c16 + 8 * chunk;
#pragma unroll
        for (int k = 0; k < NK; ++k) {
          const int raw = a.ib == 1 ? (int)((iw[k >> 2] >> (8 * (k & 3))) & 0xffu)
                                    : (int)((iw[k >> 1] >> (16 * (k & 1))) & 0xffffu);
          const int idx = cent_index(raw, a.nC, a.status);
          cp_async16(B1 + op_off(k0 + k, chunk), csrc + (int64_t)idx * kD);
        }
      }
      cp_async_wait_all();
      fence_async_smem();
      nbar_arrive(kNbKc, KT + 32);
      kc_due = false;
      // ---- B2, e, Z: S_a(t-1) and S_b(t-1) are complete
      if (t > 0 && !key_all3<KT>(kw != 0 || (bar_wait(&s_done[0], pp, &abort_sh, a.status) &&
                                             (NQ == 1 || bar_wait(&s_done[1], pp, &abort_sh, a.status))))) {
        ok = false;
        break;
      }
      if constexpr (RP > 0) {
        const int bslot = a.tiles[t_begin + t].x;
        if (bslot != cur_slot) {
          // a new basis: Z = q U_t^T into the other Z buffer, whose last
          // reader (two basis changes ago) is complete
          cur_slot = bslot;
          zb ^= 1;
          const float* Ug = a.basis + ((int64_t)bslot * a.H + h) * a.r * kD;
          for (int k = p; k < 16 * kD; k += KT) US[k] = (k / kD) < a.r ? Ug[k] : 0.f;
          key_sync3<KT>();
          for (int zr = p; zr < 128 * NQ; zr += KT) {
            float z[16];
#pragma unroll
            for (int k = 0; k < 16; ++k) z[k] = 0.f;
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
                for (int k = 0; k < 16; ++k) z[k] = fmaf(qf, US[k * kD + c], z[k]);
              }
            }
            const float qsc = QSC[zr];
            const int rr = zr & 127;
            uint8_t* zt = ZS + (zb * 2 + (zr >> 7)) * kZBuf;
#pragma unroll
            for (int j = 0; j < 2; ++j) {
              uint32_t w[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const __half2 hz = __floats2half2_rn(z[8 * j + 2 * e] * qsc, z[8 * j + 2 * e + 1] * qsc);
                w[e] = *reinterpret_cast<const uint32_t*>(&hz);
              }
              *reinterpret_cast<uint4*>(zt + ((rr >> 3) * 2 + j) * 128 + (rr & 7) * 16) =
                  make_uint4(w[0], w[1], w[2], w[3]);
            }
          }
        }
        if (p < 128) {
          // e row of key p: r float16 values, zero-padded to 16, as two core
          // matrices of a no-swizzle K-major tile
          uint8_t* dst = Es + (p >> 3) * 256 + (p & 7) * 16;
          const __half* esrc = reinterpret_cast<const __half*>(tb + a.off.e) + p * a.r;
          if (a.r == 16) {
            *reinterpret_cast<uint4*>(dst) = reinterpret_cast<const uint4*>(esrc)[0];
            *reinterpret_cast<uint4*>(dst + 128) = reinterpret_cast<const uint4*>(esrc)[1];
          } else {
#pragma unroll
            for (int j = 0; j < 2; ++j) {
              uint32_t w[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int m0 = 8 * j + 2 * e;
                const __half2 ee = __halves2half2(m0 < a.r ? esrc[m0] : __float2half_rn(0.f),
                                                  m0 + 1 < a.r ? esrc[m0 + 1] : __float2half_rn(0.f));
                w[e] = *reinterpret_cast<const uint32_t*>(&ee);
              }
              *reinterpret_cast<uint4*>(dst + 128 * j) = make_uint4(w[0], w[1], w[2], w[3]);
            }
          }
        }
      }
#pragma unroll 1
      for (int it = p; it < 1024; it += KT) {
        const int key = it >> 3, b = it & 7;
        const uint32_t w = *reinterpret_cast<const uint32_t*>(tb + a.off.kcode + key * 32 + 4 * b);
        const uint32_t qp = *reinterpret_cast<const uint32_t*>(tb + a.off.kqp + (key * 4 + (b >> 1)) * 4);
        dq_block(B2, key, b, w, qp);
      }
      fence_async_smem();
      nbar_arrive(kNbKr, KT + 32);
      // the key producers are done with ring stage t & 1
      key_sync3<KT>();
      if (p == 0) bar_arrive(&ring_free[t & 1]);
    }
    // a group that gave up arrives once more for the tile it was on
    if (!ok && nt > 0) {
      if (kc_due) nbar_arrive(kNbKc, KT + 32);
      nbar_arrive(kNbKr, KT + 32);
    }
  } else if (warp < kMmaW) {
    // ------------------------------------------------------------ value producers
    const int p = tid - (kSoftW + kKeyW) * 32, vw = p >> 5;   // 0..95, its warp in the group
    const uint32_t TB = (uint32_t)a.off.bytes;
    const uint8_t* tiles_h = a.cache + (int64_t)h * a.max_tiles * a.off.bytes;
    bool ok = true;
    if (p == 0) {
      for (int u = 0; u < 2 && u < nt; ++u) {
        bar_expect_tx(&full[u], TB);
        bulk_g2s(Ring + u * TB, tiles_h + (int64_t)(t_begin + u) * TB, TB, &full[u]);
      }
    }
    for (int t = 0; t < nt && ok; ++t) {
      const uint8_t* tb = Ring + (t & 1) * TB;
      const uint32_t pp = (uint32_t)((t - 1) & 1);
      if (!val_all3(vw != 0 || bar_wait(&full[t & 1], (uint32_t)((t >> 1) & 1), &abort_sh, a.status))) {
        ok = false;
        break;
      }
      // ---- V_hat: PV_a(t-1) and PV_b(t-1) have read the previous one
      if (t > 0 && !val_all3(vw != 0 || (bar_wait(&pv_done[0], pp, &abort_sh, a.status) &&
                                         (NQ == 1 || bar_wait(&pv_done[1], pp, &abort_sh, a.status))))) {
        ok = false;
        break;
      }
#pragma unroll 1
      for (int it = p; it < 1024; it += kValT) {
        const int key = it >> 3, b = it & 7;
        const uint32_t w = *reinterpret_cast<const uint32_t*>(tb + a.off.vcode + key * 32 + 4 * b);
        const uint32_t qp = *reinterpret_cast<const uint32_t*>(tb + a.off.vqp + (key * 4 + (b >> 1)) * 4);
        dq_block(Vt, key, b, w, qp);
      }
      fence_async_smem();
      vready_arrive();
      // refill ring stage t & 1 with tile t + 2 once both producer groups are done with it
      val_sync3();
      if (p == 0 && t + 2 < nt) {
        if (bar_wait(&ring_free[t & 1], (uint32_t)((t >> 1) & 1), &abort_sh, a.status)) {
          bar_expect_tx(&full[t & 1], TB);
          bulk_g2s(Ring + (t & 1) * TB, tiles_h + (int64_t)(t_begin + t + 2) * TB, TB, &full[t & 1]);
        }
      }
    }
    // a group that gave up before arriving for its current tile arrives once
    // more, so that a softmax warp waiting for that tile's V_hat is released
    if (!ok) vready_arrive();
  } else {
    // ------------------------------------------------------------ MMA issuer
    bool ok = warp_all(bar_wait(q_ready, 0u, &abort_sh, a.status));
    fence_after();
    // per tile t, in a fixed order: for each query tile g, PV_g(t-1) (P_g(t-1)
    // written by the softmax warps of tile g, V_hat(t-1) written) and then
    // the centroid part S1_g(t) (B1(t) gathered), so that S_g(t) follows
    // PV_g(t-1) in the tensor pipe and P_g(t-1), which lies over S_g, is read
    // before it is overwritten; then the residual and PSAC parts S2_a(t),
    // S2_b(t) (B2(t), e and Z written).  All waits are named barriers; the
    // whole warp waits, one elected lane issues.
    if (ok) {
      const uint32_t qs0 = su32(Qs), b1 = su32(B1), b2 = su32(B2);
      const uint32_t es = su32(Es), zs0 = su32(ZS), vt = su32(Vt);
      // the Z buffer of each tile follows the key producers' rule: it flips
      // whenever the tile's basis slot differs from the previous tile's
      int cur_slot = -1, zb = 1, ab_read = 0;
      int bs_next = nt > 0 ? a.tiles[t_begin].x : 0;
      for (int t = 0; t <= nt; ++t) {
        if (__any_sync(0xffffffffu, ab_read != 0)) break;
        const int bslot = bs_next;
        if (t + 1 < nt) bs_next = a.tiles[t_begin + t + 1].x;
        if (t < nt) {
          nbar_sync(kNbKc, KT + 32);
          fence_after();
        }
        if (t > 0) {
          // the first half of PV_g(t-1) (keys 0-63) as soon as their P is
          // written, while the softmax still works on keys 64-127
#pragma unroll
          for (int g = 0; g < NQ; ++g) {
            nbar_sync(kNbP1 + g, 160);
            if (g == 0) vready_sync();
            fence_after();
            if (elect_one()) {
#pragma unroll
              for (int j = 0; j < 4; ++j)
                mma_ts(tmem + kColO + 128u * g, tmem + 128u * g + 8 * j, desc_sw128_mn(vt + 2048 * j), kIdescPV,
                       (t > 1 || j > 0) ? 1u : 0u);
            }
            __syncwarp();
          }
        }
        if (t > 0) {
          // keys 64-95
#pragma unroll
          for (int g = 0; g < NQ; ++g) {
            nbar_sync(kNbP2 + g, 160);
            fence_after();
            if (elect_one()) {
#pragma unroll
              for (int j = 4; j < 6; ++j)
                mma_ts(tmem + kColO + 128u * g, tmem + 128u * g + 8 * j, desc_sw128_mn(vt + 2048 * j), kIdescPV, 1u);
            }
            __syncwarp();
          }
        }
#pragma unroll
        for (int g = 0; g < NQ; ++g) {
          if (t > 0) {
            nbar_sync(kNbP + g, 160);
            fence_after();
            if (elect_one()) {
#pragma unroll
              for (int j = 6; j < 8; ++j)
                mma_ts(tmem + kColO + 128u * g, tmem + 128u * g + 8 * j, desc_sw128_mn(vt + 2048 * j), kIdescPV, 1u);
              commit(&pv_done[g]);
            }
            __syncwarp();
          }
          if (t < nt) {
            const uint32_t d = tmem + 128u * g, qa = qs0 + kTileOp * g;
            if (elect_one()) {
#pragma unroll
              for (int j = 0; j < 8; ++j) {
                const uint32_t ko = (j >> 2) * 16384 + (j & 3) * 32;
                mma_ss(d, desc_sw128(qa + ko), desc_sw128(b1 + ko), kIdescS, j > 0);
              }
            }
            __syncwarp();
          }
        }
        if (t == nt) break;
        if (elect_one()) commit(b1_free);
        __syncwarp();
        nbar_sync(kNbKr, KT + 32);
        ab_read = abort_sh;   // after this tile's last wait; used before the next tile's first
        fence_after();
        if (RP > 0 && bslot != cur_slot) {
          cur_slot = bslot;
          zb ^= 1;
        }
#pragma unroll
        for (int g = 0; g < NQ; ++g) {
          const uint32_t d = tmem + 128u * g, qa = qs0 + kTileOp * g;
          if (elect_one()) {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const uint32_t ko = (j >> 2) * 16384 + (j & 3) * 32;
              mma_ss(d, desc_sw128(qa + ko), desc_sw128(b2 + ko), kIdescS, 1);
            }
            if constexpr (RP > 0)
              mma_ss(d, desc_none(zs0 + (zb * 2 + g) * kZBuf, 128, 256), desc_none(es, 128, 256), kIdescS, 1);
            commit(&s_done[g]);
          }
          __syncwarp();
        }
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
    const uint32_t colO = kColO + 128u * g;
    const int64_t grow = row0 + 128 * g + i;
    const bool softmax = warp < 4 * NQ;
    float* recv = reinterpret_cast<float*>(sm) + (128 * g + i) * kRecvLd;   // rank 0's buffers, now free
    float f0 = 1.f, f1 = 0.f, inv = 0.f;
    bool store = softmax && sm_ok && !partial;
    if (partial) {
      // few-row mode: this split's unnormalised O in channel order, its
      // running maximum and sum (a split that gave up reports no weight)
      if (softmax) {
        float* pr = nullptr;
        if (grow < a.M)
          pr = a.part + ((((int64_t)h * a.n_mb + (grow >> 4)) * nsplit + split) * 16 + (grow & 15)) * kRecvLd;
        for (int cb = 0; cb < 4; ++cb) {
          uint32_t v[32];
          tmem_ld32(tmem + lane_base + colO + 32 * cb, v);
          tmem_wait_ld();
          if (pr) {
#pragma unroll
            for (int k = 0; k < 32; ++k) {
              const int q = k & 15, ch = 16 * (2 * cb + (k >> 4)) + (q >> 1) + 8 * (q & 1);
              pr[ch] = sm_ok && nt > 0 ? __uint_as_float(v[k]) : 0.f;
            }
          }
        }
        if (pr) {
          pr[128] = sm_ok && nt > 0 ? m_run : -INFINITY;
          pr[129] = sm_ok && nt > 0 ? l_run : 0.f;
        }
      }
    } else if (nsplit > 1) {
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
    // every lane of a softmax warp loads (warp-collective); valid rows store.
    // Column p of O holds channel 16 (p / 16) + (p % 16) / 2 + 8 (p % 2).
    if (softmax && __any_sync(0xffffffffu, store)) {
      __nv_bfloat16* dst = a.O + ((int64_t)h * a.M + grow) * kD;
      for (int cb = 0; cb < 4; ++cb) {
        uint32_t v[32];
        tmem_ld32(tmem + lane_base + colO + 32 * cb, v);
        tmem_wait_ld();
        if (store && grow < a.M) {
          float o[32];
#pragma unroll
          for (int k = 0; k < 32; ++k) {
            o[k] = __uint_as_float(v[k]) * f0;
            if (nsplit > 1) o[k] = fmaf(recv[32 * cb + k], f1, o[k]);
            o[k] *= inv;
          }
#pragma unroll
          for (int jb = 0; jb < 2; ++jb) {
            const float* ob = o + 16 * jb;
            uint32_t lo[4], hi[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const __nv_bfloat162 l2 = __floats2bfloat162_rn(ob[4 * e], ob[4 * e + 2]);
              const __nv_bfloat162 h2 = __floats2bfloat162_rn(ob[4 * e + 1], ob[4 * e + 3]);
              lo[e] = *reinterpret_cast<const uint32_t*>(&l2);
              hi[e] = *reinterpret_cast<const uint32_t*>(&h2);
            }
            __nv_bfloat16* blk = dst + 16 * (2 * cb + jb);
            *reinterpret_cast<uint4*>(blk) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
            *reinterpret_cast<uint4*>(blk + 8) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
          }
        }
      }
    }
  }
  fence_before();
  __syncthreads();
  fence_after();
  if (warp == kMmaW) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem));
}

size_t tc3_smem(const qwm_ctx* c) { return 1024 + kOffRing + 2 * c->lay.tile_bytes; }

// KV splits per query-row pair: 2 (a cluster of two CTAs) when that cuts
// the number of full waves over the SMs, else 1
int tc3_splits(const qwm_ctx* c, int64_t M) {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      sms < 1)
    return 1;
  const int64_t units = ((M + 255) / 256) * c->cfg.heads;
  const int64_t w1 = (units + sms - 1) / sms;
  const int64_t w2x2 = (2 * units + sms - 1) / sms;
  return (c->n_tiles >= 2 && w2x2 < 2 * w1) ? 2 : 1;
}

// few-row mode: KV splits per head, the split count whose CTAs (one per SM)
// fill 2 to 4 waves best, at most one split per tile and within the
// partial buffer (row blocks of 16 x splits <= small_max_parts())
int tc3_few_splits(const qwm_ctx* c, int n_mb) {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      sms < 1)
    sms = 152;
  const int64_t units = c->cfg.heads;
  int64_t cap = small_max_parts() / n_mb;
  if (cap > c->n_tiles) cap = c->n_tiles;
  if (cap < 1) cap = 1;
  int64_t best = 1;
  double best_fill = -1.0;
  for (int waves = 2; waves <= 4; ++waves) {
    int64_t sp = waves * (int64_t)sms / units;
    if (sp > cap) sp = cap;
    if (sp < 1) sp = 1;
    const int64_t ctas = sp * units, used = (ctas + sms - 1) / sms;
    const double fill = (double)ctas / (double)(used * sms);
    if (fill > best_fill + 1e-9) {
      best_fill = fill;
      best = sp;
    }
  }
  return (int)best;
}

template <int RP, int NQ>
cudaError_t launch_tc3(const qwm_ctx* c, const Tc3Args& a, int64_t M, int ns, cudaStream_t st) {
  const size_t smem = tc3_smem(c);
  auto kern = attend_tc3_kernel<RP, NQ>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((M + 128 * NQ - 1) / (128 * NQ)), (unsigned)c->cfg.heads, (unsigned)ns);
  cfg.blockDim = dim3(kThreads3, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = (unsigned)ns;
  cfg.attrs = attr;
  cfg.numAttrs = a.part == nullptr ? 1 : 0;   // the few-row mode's splits meet in the combine kernel
  e = cudaLaunchKernelEx(&cfg, kern, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

Tc3Args tc3_args(const qwm_ctx* c, const void* q, int64_t M, float scale, void* out) {
  Tc3Args a;
  a.Q = (const __nv_bfloat16*)q;
  a.O = (__nv_bfloat16*)out;
  a.M = M;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.cache = c->cache;
  a.max_tiles = c->lay.max_tiles;
  a.off = tile_offsets(c->lay);
  a.n_tiles = c->n_tiles;
  a.tiles = c->tiles;
  a.cent16 = c->cent16;
  a.nC = c->cfg.n_centroids;
  a.basis = c->basis;
  a.H = c->cfg.heads;
  a.r = c->cfg.rank;
  a.ib = c->ib;
  a.status = c->status;
  a.part = nullptr;
  a.n_mb = 0;
  return a;
}

}  // namespace

bool attend_tc3_supported(const qwm_ctx* c) {
  return c->cfg.dtype == QWM_BF16 && c->cfg.head_dim == kD && c->cfg.rank <= 16 && c->cent16_ok &&
         c->lay.max_tiles < (int64_t(1) << 30) && tc3_smem(c) <= 227 * 1024;
}

cudaError_t launch_attend_tc3(const qwm_ctx* c, const void* q, int64_t M, float scale, void* out,
                              cudaStream_t st) {
  const Tc3Args a = tc3_args(c, q, M, scale, out);
  const int ns = tc3_splits(c, M);
  return a.r == 0 ? launch_tc3<0, 2>(c, a, M, ns, st) : launch_tc3<16, 2>(c, a, M, ns, st);
}

bool attend_tc3_few_supported(const qwm_ctx* c, int64_t M) {
  return attend_tc3_supported(c) && M >= 1 && M <= 64 && small_workspace_bytes(c->cfg) > 0;
}

cudaError_t launch_attend_tc3_few(const qwm_ctx* c, const void* q, int64_t M, float scale, void* out, uint8_t* ws,
                                  cudaStream_t st) {
  Tc3Args a = tc3_args(c, q, M, scale, out);
  a.n_mb = (int)((M + 15) / 16);
  a.part = small_part_buffer(c->cfg, ws);
  const int ns = tc3_few_splits(c, a.n_mb);
  cudaError_t e = a.r == 0 ? launch_tc3<0, 1>(c, a, M, ns, st) : launch_tc3<16, 1>(c, a, M, ns, st);
  if (e != cudaSuccess) return e;
  return launch_small_combine(c, M, ns, ws, out, st);
}

}  // namespace qwm
