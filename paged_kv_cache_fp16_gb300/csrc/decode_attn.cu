// Decode attention that reads the packed q8/q6/q4 pages directly.
//
// The pages compute attention over a quantized cache by dequantizing it to fp16 and running
// SDPA (MTPLX pull request #267, "feat(kv-cache): add q6 paged KV quantization", description:
// no kernel consumes the packed bytes).  This kernel computes the same function without
// materialising fp16 in memory: each thread unpacks the codes it needs straight into
// tensor-core fragments, scales them to the same fp16 k_hat = fp16(c * scale) and
// v_hat = fp16(c * scale) the dequantizer produces, and accumulates in float32.
//
// Decomposition (one CTA per (layer, sequence, KV head, token split); 4 warps, each warp one
// 16-token tile at a time):
//   S^T[16 tok x 8 heads] = K_hat[16 x 256] . Q^T[256 x 8]   16 x mma.m16n8k16 (tokens as M, so
//                                                            the 6 query heads of a GQA group pad
//                                                            to N = 8 instead of M = 16)
//   online softmax over the tile (log2 domain, lazy rescale)
//   P^T via movmatrix (the S^T accumulator layout transposed into the B-operand layout)
//   O^T[256 x 8] += V_hat^T[256 x 16] . P^T[16 x 8]          16 x mma.m16n8k16
// The contraction index order is free, so the head dimension is permuted such that every thread
// unpacks whole 24-bit q6 quads (or q4/q8 words) it reads itself: no dequantized tile is ever
// staged.  The 4 warps' (m, l, O) are merged in shared memory, each split writes one partial,
// and a second kernel merges the splits (log-sum-exp).
//
// Loads: when page_size is a multiple of 16, a tile is 16 contiguous rows of one page, so each
// warp streams its tiles through a ring of shared-memory stages with the bulk-copy engine
// (cp.async.bulk: the page's K codes, V codes, K scales and V scales, completing on one mbarrier
// per stage); waits are bounded and report KVQ_DEVERR_TIMEOUT instead of hanging.  Other page
// sizes gather rows with plain loads.
#include <mutex>
#include <vector>

#include <type_traits>

#include <cuda_runtime.h>
#include <cuda_fp16.h>

#include "kvq_device.cuh"
#include "kvq_internal.h"
#include "kvq_math.cuh"
#include "kvq_warp.cuh"

namespace kvq {
namespace {

constexpr int kD = 256;
constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kTile = 16;
constexpr int kRec = kD + 4;   // workspace record per (split, head): O[256], m, l, pad, pad
#define kNegInf (-__int_as_float(0x7f800000))
#define kMaxFloor (-1e30f)   // floor of the running max; a max still at it saw no valid token

struct LayerPools {
  const uint8_t* kc;
  const uint16_t* ks;
  const uint8_t* vc;
  const uint16_t* vs;
  int64_t k_pages, v_pages;
};

struct AttnArgs {
  LayerPools L[KVQ_MAX_TENSORS];
  const uint16_t* q;
  float* out;
  float* ws;
  const int32_t* pt;
  const int32_t* lens;
  int32_t* err;
  // fused append: the new token of every sequence, fp16 [nseq][H][D] per layer (else unused)
  const uint16_t* knew[KVQ_MAX_TENSORS];
  const uint16_t* vnew[KVQ_MAX_TENSORS];
  int n_layers, nseq, H, G, Hq, ps, max_pages, n_splits, tiles_per_cta;
  int len_add;     // tokens attended beyond lens[s]: 1 with the fused append, else 0
  float qk_scale;  // softmax_scale * log2(e)
};

// Side channels of the decode attention (fp16 sinks and outliers), per layer; zero when unused.
struct AttnSide {
  const uint16_t* kov[KVQ_MAX_TENSORS];   // K outlier values, fp16 [pages][H][ps][k]
  const uint8_t* koi[KVQ_MAX_TENSORS];    // K outlier positions
  const uint16_t* vov[KVQ_MAX_TENSORS];
  const uint8_t* voi[KVQ_MAX_TENSORS];
  const uint16_t* ksink[KVQ_MAX_TENSORS]; // fp16 [max_seqs][n_sink][H][D]
  const uint16_t* vsink[KVQ_MAX_TENSORS];
  int k, n_sink;
};

template <int BITS> struct Wd;
// Stage counts: with the query fragments in shared memory (q6, q4) the staged kernel holds 128
// registers, so shared memory decides the CTAs per SM: 4 for q6 (2 stages) and q4 (3); q8 (2
// stages, fragments in registers) runs 3.
template <> struct Wd<8> { static constexpr int kPd = 256, kKWords = 16, kVWords = 8, kStages = 2; };
template <> struct Wd<6> { static constexpr int kPd = 192, kKWords = 12, kVWords = 6, kStages = 2; };
template <> struct Wd<4> { static constexpr int kPd = 128, kKWords = 8, kVWords = 4, kStages = 3; };

// shared-memory stage: [K codes 16 x pd][V codes 16 x pd][K scales 16 x 2][V scales 16 x 2]
template <int BITS> __host__ __device__ constexpr int stage_bytes() { return 2 * kTile * Wd<BITS>::kPd + 4 * kTile; }
template <int BITS> __host__ __device__ constexpr int warp_bytes() { return Wd<BITS>::kStages * stage_bytes<BITS>(); }
template <int BITS> __host__ __device__ constexpr int tma_smem_bytes() {
  return kWarps * warp_bytes<BITS>() + kWarps * Wd<BITS>::kStages * 16;  // + barriers, flags
}

// Shared-memory layout of the staged kernel: the stage ring, the barriers and flags, and the query
// B fragments every warp of the CTA shares (4 KB: 32 registers per thread saved).  With side
// channels a stage also holds the tile's K and V outlier values (fp16 [16][k]) and positions
// (uint8 [16][k]), sized by k at launch (side_stage_extra); two stages per warp; then each warp's
// sparse residual tile: half a tile's columns, fp16 [16 tokens][128] with a 272-byte row stride
// (conflict-free ldmatrix), all zero between uses.  At q6/q4 and k = 3 a CTA takes 74 KB, so
// three CTAs fit on an SM.
template <int BITS, bool SIDE>
struct Lay {
  static constexpr int kStages = SIDE ? 2 : Wd<BITS>::kStages;
  static constexpr int kBase = stage_bytes<BITS>();   // bytes of the four page copies
  // without side channels (with them the stages grow by side_stage_extra(k) at run time, and
  // kRing is the smallest ring, k = 0)
  static constexpr int kStage = kBase;
  static constexpr int kWarpBytes = kStages * kStage;
  static constexpr int kRing = kWarps * kWarpBytes;
  static constexpr int kQf = kRing + kWarps * kStages * 16;   // query B fragments [16][32] uint2
  static constexpr int kQfEnd = kQf + 16 * 32 * 8;
  static constexpr int kOtStride = kD + 16;                  // bytes per half-tile row (128 fp16)
  static constexpr int kOtBytes = kTile * kOtStride;         // one warp's residual half-tile
  static constexpr int kTotal = kQfEnd;                      // without side channels
};

// Bytes a stage adds for k outliers per row: K and V values (fp16 [16][k], rounded up to 16 bytes)
// and positions (uint8 [16][k]).
__host__ __device__ constexpr int side_stage_extra(int k) {
  return 2 * ((32 * k + 15) / 16 * 16) + 2 * 16 * k;
}

// Shared memory of the side-channel kernel for k outliers per row.
template <int BITS>
__host__ __device__ constexpr int side_smem_bytes(int k) {
  return kWarps * Lay<BITS, true>::kStages * (Lay<BITS, true>::kBase + side_stage_extra(k)) +
         kWarps * Lay<BITS, true>::kStages * 16 + 16 * 32 * 8 + kWarps * Lay<BITS, true>::kOtBytes;
}

constexpr int kMergeBytes = kWarps * 8 * kD * 4 + 2 * kWarps * 8 * 4;

// PRMT selector picking bytes (b0, b1) of the first and (b0, b1) of the second source word.
__host__ __device__ constexpr uint32_t sel4(int a0, int a1, int b0, int b1) {
  return static_cast<uint32_t>(a0 | (a1 << 4) | (b0 << 8) | (b1 << 12));
}

// Exact fp16 codes of elements 8*GI + k (lo[k]) and 8*GI + k + 4 (hi[k]), k = 0..3, of the
// thread's packed V bytes, paired across two tokens: low half token A, high half token B.
// (The d order matches the output mapping of tile_pv.)
template <int BITS, int GI>
__device__ __forceinline__ void cross_group(const uint32_t* wa, const uint32_t* wb, uint32_t lo[4],
                                            uint32_t hi[4]) {
  if constexpr (BITS == 6) {
#pragma unroll
    for (int qd = 0; qd < 2; ++qd) {           // quads 2*GI (-> lo) and 2*GI + 1 (-> hi)
      const int b = 6 * GI + 3 * qd;           // byte offset of the quad (compile-time)
      const int w = b / 4, intra = b % 4;
      uint32_t xa, xb;
      int i0;
      if (intra <= 1) {
        xa = wa[w]; xb = wb[w]; i0 = intra;
      } else {                                 // the quad straddles two words: align it first
        xa = __funnelshift_r(wa[w], wa[w + 1], 8 * intra);
        xb = __funnelshift_r(wb[w], wb[w + 1], 8 * intra);
        i0 = 0;
      }
      const uint32_t p1 = prmt(xa, xb, sel4(i0, i0 + 1, 4 + i0, 5 + i0));      // A.b0 A.b1 B.b0 B.b1
      const uint32_t p2 = prmt(xa, xb, sel4(i0 + 1, i0 + 2, 5 + i0, 6 + i0));  // A.b1 A.b2 B.b1 B.b2
      uint32_t* o = qd ? hi : lo;
      o[0] = hfma2u((p1 & 0x003F003Fu) | 0x64006400u, kH1, kHm1056);
      o[1] = hfma2u(((p1 >> 2) & 0x03F003F0u) | 0x64006400u, kH16th, kHm96);
      o[2] = hfma2u((p2 & 0x03F003F0u) | 0x64006400u, kH16th, kHm96);
      o[3] = hfma2u(((p2 >> 8) & 0x00FC00FCu) | 0x64006400u, kHQuarter, kHm288);
    }
  } else if constexpr (BITS == 8) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      lo[k] = hfma2u((prmt(wa[2 * GI], wb[2 * GI], sel4(k, k, 4 + k, 4 + k)) & 0x00FF00FFu) ^
                         0x64806480u, kH1, kHm1152);
      hi[k] = hfma2u((prmt(wa[2 * GI + 1], wb[2 * GI + 1], sel4(k, k, 4 + k, 4 + k)) &
                      0x00FF00FFu) ^ 0x64806480u, kH1, kHm1152);
    }
  } else {
    uint32_t pb[4];
#pragma unroll
    for (int b = 0; b < 4; ++b) pb[b] = prmt(wa[GI], wb[GI], sel4(b, b, 4 + b, 4 + b));
    // each 16-bit lane holds the byte twice: its low nibble at bits 0-3 (1024 + u) and its high
    // nibble at bits 4-7 (1024 + 16u, scale 1/16) -- no shifts
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      if (k & 1) {
        lo[k] = hfma2u((pb[k >> 1] & 0x00F000F0u) | 0x64006400u, kH16th, kHm72);
        hi[k] = hfma2u((pb[2 + (k >> 1)] & 0x00F000F0u) | 0x64006400u, kH16th, kHm72);
      } else {
        lo[k] = hfma2u((pb[k >> 1] & 0x000F000Fu) | 0x64006400u, kH1, kHm1032);
        hi[k] = hfma2u((pb[2 + (k >> 1)] & 0x000F000Fu) | 0x64006400u, kH1, kHm1032);
      }
    }
  }
}

// ------------------------------------------------------------------------------ tile compute
// One 16-token tile: K words of rows g, g+8 (thread's 64 head-dim elements) with their fp16
// scales; V words of tokens 2c, 2c+1, 2c+8, 2c+9 (thread's 32 head-dim elements) with their
// scales (0 for masked tokens).  V is read only after Q.K^T so the two share registers.
template <int BITS>
struct KRegs {
  uint32_t kw[2][Wd<BITS>::kKWords];
  uint32_t ks2[2];   // the rows' fp16 scales, twice (half2): k_hat = fp16(code * scale)
  float vsc[2];      // the rows' V scales (0 if masked), folded into P for the P.V product
  bool kval[2];
};

// The same tile with the K words left in the stage: the unpack reads each group's words from
// shared memory as it goes, so no copy of them is held across Q.K^T.  Taken by the side-channel
// kernel (2.35 -> 2.19 ms at q6: it frees the registers its side passes need) and at q8 (-0.7 %);
// the plain q6 and q4 kernels measured 0.5 % and 0.3 % slower with it.
template <int BITS>
struct KStage {
  const uint32_t* kw[2];   // the rows' packed K words in the stage
  uint32_t ks2[2];
  float vsc[2];
  bool kval[2];
};

template <int BITS>
struct VRegs {
  uint32_t vw[4][Wd<BITS>::kVWords];
};

// Q.K^T of one tile and the online-softmax update; returns P^T as the two B-operand registers.
// Where a thread's query B fragments come from: registers, or the CTA's shared copy.
struct QFragRegs {
  const uint32_t (*qf)[2];
  __device__ __forceinline__ uint2 pair(int ks) const { return make_uint2(qf[ks][0], qf[ks][1]); }
};
struct QFragSmem {
  uint32_t addr;   // shared address of this lane's fragments; k-step ks at addr + 256 * ks
  __device__ __forceinline__ uint2 pair(int ks) const {
    uint2 r;
    asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(r.x), "=r"(r.y) : "r"(addr + 256 * ks));
    return r;
  }
};

// The tile softmax's 2^x: the hardware's approximate exponential for q6/q4 (1.305 -> 1.271 ms and
// 1.145 -> 1.106 ms on the 16-layer decode), the library exp2f for q8, whose kernel measured
// 2.3 % slower with the approximate one (1.488 vs 1.454 ms).
template <int BITS>
__device__ __forceinline__ float softmax_exp2(float x) {
  if constexpr (BITS == 8) return exp2f(x);
  else return ex2_fast(x);
}

// With SIDE, kc[4] (same layout as the scores) is added to the dense scores -- the outlier and
// sink terms of the keys -- and p[4] is returned for the value side terms.
template <int BITS, bool SIDE = false, typename QF, typename KT>
__device__ __forceinline__ void tile_qk_softmax(const KT& T, const QF& Q,
                                                float (&acc)[16][4], float& m0, float& m1,
                                                float& l0, float& l1, float qk_scale,
                                                uint32_t& pb0, uint32_t& pb1,
                                                const float* kc = nullptr,
                                                float* p_out = nullptr) {
  // ---------------- S^T = K_hat . Q^T, one accumulation chain (four independent chains measured
  // 3.3 % slower at q6: their 12 registers cost the 128-register kernel more than the chain's
  // latency).  K_hat is the dequantizer's fp16(code * scale), one half2 multiply of the exact
  // codes by the row's fp16 scale: keys carry outlier channels, and scaling the scores of the
  // exact codes instead (one fp32 multiply per score) moves them by the fp16 rounding of those
  // large elements -- enough to take N(0, 1) caches with x10 channels outside the tolerance
  float sacc[4] = {};
#define KVQ_QK_GROUP(GI)                                                                \
  {                                                                                     \
    uint32_t p0[4], p1[4];                                                              \
    unpack_group<BITS, GI>(T.kw[0], p0);                                                \
    unpack_group<BITS, GI>(T.kw[1], p1);                                                \
    _Pragma("unroll") for (int i = 0; i < 4; ++i) {                                     \
      p0[i] = hmul2u(p0[i], T.ks2[0]);                                                  \
      p1[i] = hmul2u(p1[i], T.ks2[1]);                                                  \
    }                                                                                   \
    const uint2 qa = Q.pair(2 * GI), qb = Q.pair(2 * GI + 1);                           \
    mma16816(sacc, p0[0], p1[0], p0[1], p1[1], qa.x, qa.y);                             \
    mma16816(sacc, p0[2], p1[2], p0[3], p1[3], qb.x, qb.y);                             \
  }
  KVQ_QK_GROUP(0) KVQ_QK_GROUP(1) KVQ_QK_GROUP(2) KVQ_QK_GROUP(3)
  KVQ_QK_GROUP(4) KVQ_QK_GROUP(5) KVQ_QK_GROUP(6) KVQ_QK_GROUP(7)
#undef KVQ_QK_GROUP

  // ---------------- online softmax (log2 domain); sacc: [tok g | g+8][head 2c | 2c+1]
  float sc[4];
  if constexpr (SIDE) {
    sc[0] = T.kval[0] ? (sacc[0] + kc[0]) * qk_scale : kNegInf;
    sc[1] = T.kval[0] ? (sacc[1] + kc[1]) * qk_scale : kNegInf;
    sc[2] = T.kval[1] ? (sacc[2] + kc[2]) * qk_scale : kNegInf;
    sc[3] = T.kval[1] ? (sacc[3] + kc[3]) * qk_scale : kNegInf;
  } else {
    sc[0] = T.kval[0] ? sacc[0] * qk_scale : kNegInf;
    sc[1] = T.kval[0] ? sacc[1] * qk_scale : kNegInf;
    sc[2] = T.kval[1] ? sacc[2] * qk_scale : kNegInf;
    sc[3] = T.kval[1] ? sacc[3] * qk_scale : kNegInf;
  }
  float tm0 = fmaxf(sc[0], sc[2]), tm1 = fmaxf(sc[1], sc[3]);
#pragma unroll
  for (int o = 4; o < 32; o <<= 1) {
    tm0 = fmaxf(tm0, __shfl_xor_sync(kFullMask, tm0, o));
    tm1 = fmaxf(tm1, __shfl_xor_sync(kFullMask, tm1, o));
  }
  // the running max never drops below a finite floor (far below any score fp16 inputs can
  // give), so no exponential below needs a guard against -inf - -inf
  const float n0 = fmaxf(fmaxf(m0, tm0), kMaxFloor), n1 = fmaxf(fmaxf(m1, tm1), kMaxFloor);
  const float al0 = softmax_exp2<BITS>(m0 - n0);
  const float al1 = softmax_exp2<BITS>(m1 - n1);
  float p[4];
  p[0] = softmax_exp2<BITS>(sc[0] - n0);
  p[2] = softmax_exp2<BITS>(sc[2] - n0);
  p[1] = softmax_exp2<BITS>(sc[1] - n1);
  p[3] = softmax_exp2<BITS>(sc[3] - n1);
  l0 = l0 * al0 + (p[0] + p[2]);
  l1 = l1 * al1 + (p[1] + p[3]);
  m0 = n0;
  m1 = n1;
  if (__any_sync(kFullMask, al0 != 1.f || al1 != 1.f)) {
#pragma unroll
    for (int mt = 0; mt < 16; ++mt) {
      acc[mt][0] *= al0; acc[mt][1] *= al1; acc[mt][2] *= al0; acc[mt][3] *= al1;
    }
  }
  // P times each token's V scale: O = sum_t (p_t s_t) c_t, so the V operand is the exact integer
  // codes (the normaliser l keeps the unscaled p)
  pb0 = movtrans(pack_h2(p[0] * T.vsc[0], p[1] * T.vsc[0]));   // tokens 2c, 2c+1 ; head g
  pb1 = movtrans(pack_h2(p[2] * T.vsc[1], p[3] * T.vsc[1]));   // tokens 8+2c, 8+2c+1 ; head g
  if constexpr (SIDE) {
#pragma unroll
    for (int k = 0; k < 4; ++k) p_out[k] = p[k];
  }
}


// O^T += V_hat^T . P^T for one tile.
template <int BITS>
__device__ __forceinline__ void tile_pv(const VRegs<BITS>& T, uint32_t pb0, uint32_t pb1,
                                        float (&acc)[16][4]) {
  // ---------------- O^T += C_V^T . (P S_V)^T on the exact integer codes
#define KVQ_PV_GROUP(GI)                                                                \
  {                                                                                     \
    uint32_t lab[4], hab[4], lcd[4], hcd[4];                                            \
    cross_group<BITS, GI>(T.vw[0], T.vw[1], lab, hab);                                  \
    cross_group<BITS, GI>(T.vw[2], T.vw[3], lcd, hcd);                                  \
    _Pragma("unroll") for (int k = 0; k < 4; ++k) {                                     \
      mma16816(acc[4 * GI + k], lab[k], hab[k], lcd[k], hcd[k], pb0, pb1);              \
    }                                                                                   \
  }
  KVQ_PV_GROUP(0) KVQ_PV_GROUP(1) KVQ_PV_GROUP(2) KVQ_PV_GROUP(3)
#undef KVQ_PV_GROUP
}

// Q^T B-fragments for head g of this KV head's group (zero for padding heads).
__device__ __forceinline__ void load_q_frags(const AttnArgs& a, int ls, int h, int g, int c,
                                             bool any, uint32_t (&qf)[16][2]) {
  uint32_t qw[32];
  if (g < a.G && any) {
    const uint16_t* qp = a.q + ((static_cast<int64_t>(ls) * a.Hq) + h * a.G + g) * kD + 64 * c;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint4 v = ld_nc_v4(qp + 8 * i);
      qw[4 * i] = v.x; qw[4 * i + 1] = v.y; qw[4 * i + 2] = v.z; qw[4 * i + 3] = v.w;
    }
  } else {
#pragma unroll
    for (int i = 0; i < 32; ++i) qw[i] = 0;
  }
#pragma unroll
  for (int gi = 0; gi < 8; ++gi)
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      qf[2 * gi + j][0] = prmt(qw[4 * gi + j], qw[4 * gi + j + 2], 0x5410u);
      qf[2 * gi + j][1] = prmt(qw[4 * gi + j], qw[4 * gi + j + 2], 0x7632u);
    }
}

// Merge the CTA's warps in shared memory and write the split's partial record.  The warps' O^T
// accumulators go to sm_o[warp][head][d] with the low five bits of d XOR-ed by sw(head, d) =
// (d >> 5) | (head >> 1) << 3, a bijection within each 32-element block: the 32 lanes of a warp
// store (head 2c or 2c + 1, d = 32 g + ...) for the 32 (g, c) pairs at once, which without the
// swizzle all fall in one bank (a 32-way conflict per store; the merge had cost 3 % of the decode).
__device__ __forceinline__ int merge_slot(int j, int d) {
  return j * kD + (d ^ ((d >> 5) | ((j >> 1) << 3)));
}

__device__ __forceinline__ void cta_merge_write(const AttnArgs& a, float* sm, int ls, int h,
                                                int split, int warp, int g, int c,
                                                const float (&acc)[16][4], float m0, float m1,
                                                float l0, float l1) {
  if (m0 == kMaxFloor) m0 = kNegInf;   // no valid token: an empty partial for the merges
  if (m1 == kMaxFloor) m1 = kNegInf;
  float* sm_o = sm;                                              // [warp][8 * kD], swizzled
  float (*sm_m)[8] = reinterpret_cast<float (*)[8]>(sm + kWarps * 8 * kD);
  float (*sm_l)[8] = reinterpret_cast<float (*)[8]>(sm + kWarps * 8 * kD + kWarps * 8);
#pragma unroll
  for (int o = 4; o < 32; o <<= 1) {
    l0 += __shfl_xor_sync(kFullMask, l0, o);
    l1 += __shfl_xor_sync(kFullMask, l1, o);
  }
  if (g == 0) {
    sm_m[warp][2 * c] = m0; sm_m[warp][2 * c + 1] = m1;
    sm_l[warp][2 * c] = l0; sm_l[warp][2 * c + 1] = l1;
  }
  float* wo = sm_o + warp * 8 * kD;
#pragma unroll
  for (int mt = 0; mt < 16; ++mt) {
    const int gi = mt >> 2, k = mt & 3;
    const int d = 32 * g + 8 * gi + k;
    wo[merge_slot(2 * c, d)] = acc[mt][0];
    wo[merge_slot(2 * c + 1, d)] = acc[mt][1];
    wo[merge_slot(2 * c, d + 4)] = acc[mt][2];
    wo[merge_slot(2 * c + 1, d + 4)] = acc[mt][3];
  }
  __syncthreads();
  float* rec = a.ws + ((static_cast<int64_t>(ls) * a.H + h) * a.n_splits + split) * 8 * kRec;
  // a thread's elements move through the heads in order: the warps' weights exp2(m_w - M) of
  // a head are computed once, when its first element comes up
  int jc = -1;
  float f[kWarps], M = kNegInf;
  for (int i = threadIdx.x; i < a.G * kD; i += kThreads) {
    const int jh = i / kD, d = i - jh * kD;
    if (jh != jc) {
      jc = jh;
      M = kNegInf;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) M = fmaxf(M, sm_m[w][jh]);
#pragma unroll
      for (int w = 0; w < kWarps; ++w)
        f[w] = (sm_m[w][jh] == kNegInf) ? 0.f : exp2f(sm_m[w][jh] - M);
    }
    const int slot = merge_slot(jh, d);
    float O = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) O += sm_o[w * 8 * kD + slot] * f[w];
    rec[jh * kRec + d] = O;
    if (d == 0) {
      float Lsum = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) Lsum += sm_l[w][jh] * f[w];
      rec[jh * kRec + kD] = M;
      rec[jh * kRec + kD + 1] = Lsum;
    }
  }
}

// ------------------------------------------------------------------------------ TMA kernel
// Fused append, first part: this lane's 16 elements of the new K (lanes 0-15) or V (lanes 16-31)
// row of (layer, sequence s, KV head h), loaded at the start of the kernel so their latency
// overlaps the block's set-up.
__device__ __forceinline__ void append_load(const AttnArgs& a, int layer, int s, int h, int lane,
                                            uint4& x0, uint4& x1) {
  const uint16_t* src = (lane >= 16 ? a.vnew[layer] : a.knew[layer]) +
                        (static_cast<int64_t>(s) * a.H + h) * kD + (lane & 15) * 16;
  x0 = ld_nc_v4(src);
  x1 = ld_nc_v4(src + 8);
}

// Fused append, second part: quantize the loaded rows exactly as kvq_quant_pack_paged does and
// store them at physical row `prow` of the pools (lanes 0-15 the K row, lanes 16-31 the V row, one
// 16-element unit per lane).
template <int BITS>
__device__ __forceinline__ void append_rows(const LayerPools& P, int64_t prow, int lane,
                                            const uint4& x0, const uint4& x1) {
  constexpr int kQm = SymQ<BITS>::kQmax;
  constexpr int kB = SymQ<BITS>::kBias;
  constexpr int kM = SymQ<BITS>::kMask;
  constexpr int kPd = Wd<BITS>::kPd;
  const bool is_v = lane >= 16;
  const int u = lane & 15;
  const __half2 m2 = __hmax2(absmax8(x0), absmax8(x1));
  float amax = fmaxf(__low2float(m2), __high2float(m2));
#pragma unroll
  for (int o = 8; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kFullMask, amax, o));
  const uint16_t sbits = f2h(row_scale_f32<kQm>(amax));
  const float sc = h2f(sbits);
  const float y = (sc == 0.f) ? 0.f : __frcp_rn(sc);
  const float se = (sc == 0.f) ? 1.f : sc;
  const bool clip = sc < 6.103515625e-05f;   // 2^-14, smallest normal fp16
  uint32_t pk[4];
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    const uint4& vv = hh ? x1 : x0;
    const uint32_t w[4] = {vv.x, vv.y, vv.z, vv.w};
    uint32_t f[8];
#pragma unroll
    for (int e = 0; e < 8; ++e)
      f[e] = quant_field<kQm, kB, kM>(h2f(static_cast<uint16_t>(w[e >> 1] >> (16 * (e & 1)))),
                                      se, y, clip);
    pack8<BITS>(f, pk[2 * hh], pk[2 * hh + 1]);
  }
  uint8_t* gcodes = const_cast<uint8_t*>(is_v ? P.vc : P.kc);
  uint16_t* gscales = const_cast<uint16_t*>(is_v ? P.vs : P.ks);
  const int off = u * SymQ<BITS>::kUnitBytes;
  store_unit<BITS>(gcodes + prow * kPd + off, pk[0], pk[1], pk[2], pk[3]);
  if (u == 0) gscales[prow] = sbits;
}

// The side-channel kernel's order of a tile's tokens: its k-th fragment row holds token
// tok_order(k), an involution that swaps the neighbours 4<->5, 6<->7, 12<->13, 14<->15.  The
// output sums over the tile's tokens, so any fixed order is exact.  At q6 (192-byte rows, 16
// banks apart) the four lanes that read tokens 2c + delta of one V column group then meet rows of
// both parities (2-way instead of 4-way bank conflicts) and the K reads stay conflict-free: the
// side-channel kernel, latency-bound at 12 warps per SM, gains 5 % (2.52 -> 2.40 ms); the plain
// kernel, issue-bound, measured 1 % slower with it and keeps the natural order.
__device__ __forceinline__ int tok_order(int k) { return k ^ ((k >> 2) & 1); }

// Column of element d in a residual tile.  Keys follow the score product's k-order: the dense
// path's k-step 2*GI + h pairs, for thread c, elements 64c + 8*GI + {0, 4, 1, 5} (h = 0) or
// {2, 6, 3, 7} (h = 1) at k = 2c, 2c+1, 2c+8, 2c+9.  Values follow the value product's m-order:
// block 4*GI + k holds d = 32*m' + 8*GI + k at row m' and d + 4 at row m' + 8.
template <bool KEY>
__device__ __forceinline__ int side_col(int d) {
  const int o = d & 7;
  if constexpr (KEY)
    return 16 * (2 * ((d & 63) >> 3) + ((o >> 1) & 1)) + 2 * (d >> 6) + ((o >> 2) & 1) +
           8 * (o & 1);
  else
    return 16 * (4 * ((d & 31) >> 3) + (o & 3)) + (d >> 5) + 8 * (o >> 2);
}

// One lane's side entries of a tile, read from the stage before it is handed back: the outliers
// of token row r = lane >> 1 (entries lane & 1, + 2, ...) when the row is live and not a sink,
// each as bits 0-7 its residual-tile column (side_col), 8-11 its residual-tile row
// (tok_order(r)), 12 valid, 16-31 the fp16 value.
template <bool KEY, int NE>
__device__ __forceinline__ void side_collect(const uint8_t* idx, const uint16_t* val, int k,
                                             int n_sink, int tb, int len, int lane,
                                             uint32_t (&ent)[NE]) {
  const int row = lane >> 1;
  const bool live = tb + row < len && tb + row >= n_sink;
#pragma unroll
  for (int i = 0; i < NE; ++i) {
    const int j = (lane & 1) + 2 * i;
    ent[i] = 0;
    if (live && j < k)
      ent[i] = (static_cast<uint32_t>(val[row * k + j]) << 16) | 0x1000u |
               static_cast<uint32_t>(tok_order(row) << 8) |
               static_cast<uint32_t>(side_col<KEY>(idx[row * k + j]));
  }
}

// Write (or clear) half `hf` of the tile's K or V side terms -- residual-tile columns
// [128 hf, 128 hf + 128) -- into the warp's half-tile: the lane's entries, and in the sequence's
// first tile the sink rows' exact fp16 values from the sink buffer [seq][n_sink][H][256].
template <bool KEY, int NE>
__device__ __forceinline__ void side_half(uint16_t* ot, const uint32_t (&ent)[NE],
                                          int hf, bool clear, int n_sink, const uint16_t* sink,
                                          int s, int H, int h, int tb, int len, int lane) {
  constexpr int kRowH = (kD + 16) / 2;   // halves per half-tile row
#pragma unroll
  for (int i = 0; i < NE; ++i) {
    const uint32_t e = ent[i];
    if ((e & 0x1000u) && static_cast<int>((e >> 7) & 1u) == hf)
      ot[((e >> 8) & 15u) * kRowH + (e & 127u)] = clear ? static_cast<uint16_t>(0)
                                                        : static_cast<uint16_t>(e >> 16);
  }
  if (tb < n_sink) {   // only the first tile: n_sink <= 16 = kTile
    const int nr = min(min(n_sink - tb, kTile), len - tb);
    for (int e = lane; e < nr * kD; e += 32) {
      const int r = e / kD, d = e - r * kD;
      const int col = side_col<KEY>(d);
      if ((col >> 7) == hf)
        ot[tok_order(r) * kRowH + (col & 127)] =
            clear ? static_cast<uint16_t>(0)
                  : sink[((static_cast<int64_t>(s) * n_sink + tb + r) * H + h) * kD + d];
    }
  }
}

// With side channels q6/q4 fit 3 CTAs per SM (168 registers, 74 KB at k = 3); q8 keeps 2.
template <int BITS, bool APPEND, bool SIDE, int NE = KVQ_MAX_OUTLIERS / 2>
__global__ void __launch_bounds__(kThreads, SIDE ? (BITS == 8 ? 2 : 3) : (BITS == 8 ? 3 : 4)) decode_attn_tma_kernel(const AttnArgs a,
                                                                      const AttnSide sd) {
  using W = Wd<BITS>;
  using Ly = Lay<BITS, SIDE>;
  constexpr int S = Ly::kStages;
  constexpr int kPd = W::kPd;
  extern __shared__ __align__(128) uint8_t smem[];

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2;
  const int c = lane & 3;
  const int split = blockIdx.x;
  const int h = blockIdx.y;
  const int ls = blockIdx.z;
  const int layer = ls / a.nseq;
  const int s = ls - layer * a.nseq;
  const LayerPools P = a.L[layer];
  // with APPEND the new token at position lens[s] is attended too
  const int len = __ldg(a.lens + s) + (APPEND ? 1 : 0);
  const int n_tiles = (len + kTile - 1) / kTile;
  const int tile0 = split * a.tiles_per_cta;
  // a split that starts past the sequence's end has no work and writes no partial (the merge
  // reads only the splits that hold tokens): with ragged lengths the grid is sized by the longest
  // sequence, so this keeps the short ones from costing more than a block launch
  if (tile0 >= n_tiles) return;
  const int tile1 = min(n_tiles, tile0 + a.tiles_per_cta);
  const int n_mine = (tile1 - tile0 - warp + kWarps - 1) > 0
                         ? (tile1 - tile0 - warp + kWarps - 1) / kWarps : 0;
  // fused append: the warp whose last tile holds the new token loads its rows and page id now
  bool append_here = false;
  int append_page = -1, append_slot = 0;
  uint4 nx0 = make_uint4(0, 0, 0, 0), nx1 = nx0;
  if constexpr (APPEND) {
    const int ta = (len - 1) / kTile;
    append_here = len > 0 && ta >= tile0 && ta < tile1 && (ta - tile0) % kWarps == warp;
    if (append_here) {
      append_load(a, layer, s, h, lane, nx0, nx1);
      const int pos = len - 1;
      const int lp = pos / a.ps;
      append_slot = pos - lp * a.ps;
      if (lp < a.max_pages) append_page = __ldg(a.pt + static_cast<int64_t>(s) * a.max_pages + lp);
    }
  }

  // stage size: the four page copies, plus the tile's outlier values and positions with side
  // channels (sized by k; compile-time constants without them)
  const uint32_t kStageBytes = SIDE ? Ly::kBase + side_stage_extra(sd.k) : Ly::kStage;
  const uint32_t kvov = Ly::kBase + (SIDE ? (32 * sd.k + 15) / 16 * 16 : 0);   // V values
  const uint32_t kkoi = kvov + (kvov - Ly::kBase);                              // K positions
  const uint32_t kvoi = kkoi + 16 * (SIDE ? sd.k : 0);                          // V positions
  const uint32_t ring = kWarps * S * kStageBytes;
  uint8_t* wbase = smem + warp * S * kStageBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + ring) + warp * S;
  int* flags = reinterpret_cast<int*>(smem + ring + kWarps * S * 8) + warp * S;
  const uint32_t qf_off = ring + kWarps * S * 16;
  // SIDE: this warp's residual half-tile (fp16 [16][128], stride Ly::kOtStride), zeroed once;
  // each tile's side terms are written into it half by half, consumed by tensor-core products
  // and cleared again
  uint16_t* ot = nullptr;
  if constexpr (SIDE) {
    ot = reinterpret_cast<uint16_t*>(smem + qf_off + 16 * 32 * 8 + warp * Ly::kOtBytes);
    for (int i = lane; i < Ly::kOtBytes / 16; i += 32)
      reinterpret_cast<uint4*>(ot)[i] = make_uint4(0, 0, 0, 0);
    __syncwarp();
  }

  if (lane == 0) {
    for (int i = 0; i < S; ++i) mbar_init(&bars[i], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncwarp();

  // Page ids and in-page slots of this warp's tiles, 32 at a time: lane i holds those of tile
  // 32 * blk + i, so the per-tile issue needs two shuffles instead of a dependent global load and
  // a division by the page size in one lane (0.85 % of the 16-layer decode).  All lanes call it.
  int pg_blk = -1, pg_val = -1, sl_val = 0;
  auto page_of = [&](int j, int& slot) -> int {
    const int blk = j >> 5;
    if (blk != pg_blk) {   // warp-uniform
      pg_blk = blk;
      pg_val = -1;
      sl_val = 0;
      const int jl = blk * 32 + lane;
      if (jl < n_mine) {
        const int tok = (tile0 + warp + jl * kWarps) * kTile;
        const int lp = tok / a.ps;
        sl_val = tok - lp * a.ps;
        if (lp < a.max_pages) pg_val = __ldg(a.pt + static_cast<int64_t>(s) * a.max_pages + lp);
      }
    }
    slot = __shfl_sync(kFullMask, sl_val, j & 31);
    return __shfl_sync(kFullMask, pg_val, j & 31);
  };

  // Issue the loads of this warp's j-th tile (page id `page`, first slot `slot0`) into stage
  // j % S (lane 0 only).
  auto issue = [&](int j, int page, int slot0) {
    const int st = j % S;
    const bool ok = page >= 0 && page < P.k_pages && page < P.v_pages;
    flags[st] = ok ? 1 : 0;
    uint8_t* dst = wbase + st * kStageBytes;
    if (ok) {
      const int64_t row = (static_cast<int64_t>(page) * a.H + h) * a.ps + slot0;
      const int nk = SIDE ? sd.k : 0;
      mbar_expect_tx(&bars[st], Ly::kBase + 96 * nk);   // 32k + 32k + 16k + 16k bytes of side data
      bulk_g2s(dst, P.kc + row * kPd, kTile * kPd, &bars[st]);
      bulk_g2s(dst + kTile * kPd, P.vc + row * kPd, kTile * kPd, &bars[st]);
      bulk_g2s(dst + 2 * kTile * kPd, P.ks + row, 2 * kTile, &bars[st]);
      bulk_g2s(dst + 2 * kTile * kPd + 2 * kTile, P.vs + row, 2 * kTile, &bars[st]);
      if constexpr (SIDE) {
        if (nk > 0) {   // the tile's outliers: 16 rows x k values (fp16) and positions (uint8)
          bulk_g2s(dst + Ly::kBase, sd.kov[layer] + row * nk, 32 * nk, &bars[st]);
          bulk_g2s(dst + kvov, sd.vov[layer] + row * nk, 32 * nk, &bars[st]);
          bulk_g2s(dst + kkoi, sd.koi[layer] + row * nk, 16 * nk, &bars[st]);
          bulk_g2s(dst + kvoi, sd.voi[layer] + row * nk, 16 * nk, &bars[st]);
        }
      }
    } else {
      report(a.err, KVQ_DEVERR_PAGE_RANGE);
      mbar_arrive(&bars[st]);
    }
  };

  if constexpr (APPEND) {
    // The new token (position len - 1) sits in the sequence's last tile, which exactly one warp
    // of the grid streams.  That warp quantizes the new rows into the pages before it issues any
    // copy, so its copy of the tile reads them from global memory (each lane orders its stores
    // before the bulk copies with a proxy fence); the tile loop itself has no append code.  The
    // new rows and the tail's page id were loaded at the start of the kernel.
    if (append_here) {   // warp-uniform
      if (append_page >= 0 && append_page < P.k_pages && append_page < P.v_pages)
        append_rows<BITS>(P, (static_cast<int64_t>(append_page) * a.H + h) * a.ps + append_slot,
                          lane, nx0, nx1);   // else the tile's issue reports it
      asm volatile("fence.proxy.async.global;" ::: "memory");
      __syncwarp();
    }
  }

  for (int j = 0; j < S && j < n_mine; ++j) {
    int slot;
    const int page = page_of(j, slot);
    if (lane == 0) issue(j, page, slot);
  }

  // The query fragments: for q6/q4 computed once per CTA (warp 0) into shared memory, which
  // frees the registers for a fourth CTA per SM; q8's stages allow only three, so it keeps them
  // in registers.
  constexpr bool kQShared = BITS != 8;
  using QSrc = typename std::conditional<kQShared, QFragSmem, QFragRegs>::type;
  const uint32_t qaddr = smem_u32(smem + qf_off) + 8 * lane;
  uint32_t qf[kQShared ? 1 : 16][2];
  if constexpr (kQShared) {
    if (warp == 0) {
      uint32_t qt[16][2];
      load_q_frags(a, ls, h, g, c, len > 0, qt);
#pragma unroll
      for (int ks = 0; ks < 16; ++ks)
        asm volatile("st.shared.v2.u32 [%0], {%1,%2};" ::"r"(qaddr + 256 * ks), "r"(qt[ks][0]),
                     "r"(qt[ks][1])
                     : "memory");
    }
    __syncthreads();
  } else {
    load_q_frags(a, ls, h, g, c, len > 0, reinterpret_cast<uint32_t (&)[16][2]>(qf));
  }
  QSrc Q;
  if constexpr (kQShared) Q = QFragSmem{qaddr};
  else Q = QFragRegs{qf};
  float acc[16][4];
#pragma unroll
  for (int mt = 0; mt < 16; ++mt)
#pragma unroll
    for (int k = 0; k < 4; ++k) acc[mt][k] = 0.f;
  float m0 = kNegInf, m1 = kNegInf, l0 = 0.f, l1 = 0.f;
  bool timed_out = false;
  int issued = (S < n_mine) ? S : n_mine;

  for (int j = 0; j < n_mine; ++j) {
    const int st = j % S;
    const uint32_t parity = static_cast<uint32_t>((j / S) & 1);
    const bool arrived = mbar_wait_stage(&bars[st], parity);
    if (__any_sync(kFullMask, !arrived)) {   // warp-uniform exit
      timed_out = true;
      break;
    }
    uint8_t* sk = wbase + st * kStageBytes;
    uint8_t* sv = sk + kTile * kPd;
    uint16_t* sks = reinterpret_cast<uint16_t*>(sk + 2 * kTile * kPd);
    uint16_t* svs = sks + kTile;
    const bool ok = flags[st] != 0;
    const int tb = (tile0 + warp + j * kWarps) * kTile;
    constexpr bool kStageK = SIDE || BITS == 8;
    typename std::conditional<kStageK, KStage<BITS>, KRegs<BITS>>::type K;
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      // fragment row g + 8r holds this token (side channels: in tok_order)
      const int row = SIDE ? tok_order(g + 8 * r) : g + 8 * r;
      K.kval[r] = ok && tb + row < len;
      K.ks2[r] = (SIDE && tb + row < sd.n_sink) ? 0u                      // sinks: exact below
                                                : static_cast<uint32_t>(sks[row]) * 0x10001u;
      K.vsc[r] = (K.kval[r] && !(SIDE && tb + row < sd.n_sink)) ? h2f(svs[row]) : 0.f;
      const uint8_t* krow = sk + row * kPd + c * (4 * W::kKWords);
      if constexpr (kStageK) {
        K.kw[r] = reinterpret_cast<const uint32_t*>(krow);
      } else {
        const uint4* src = reinterpret_cast<const uint4*>(krow);
#pragma unroll
        for (int i = 0; i < W::kKWords / 4; ++i) {
          const uint4 v = src[i];
          K.kw[r][4 * i] = v.x; K.kw[r][4 * i + 1] = v.y;
          K.kw[r][4 * i + 2] = v.z; K.kw[r][4 * i + 3] = v.w;
        }
      }
    }
    uint32_t pb0, pb1;
    float sp[4];   // SIDE: the tile's probabilities (unscaled), for the value side terms
    uint32_t vent[NE];   // SIDE: this lane's value entries (side_collect)
    const bool side_work = SIDE && (sd.k > 0 || (tb == 0 && sd.n_sink > 0));   // warp-uniform
    if constexpr (SIDE) {
      // Key terms the codes do not carry: the outliers (q[pos] * value) and, for sink rows, the
      // whole exact fp16 row (their dense scale is zeroed above).  With the query fragments in
      // shared memory (q6, q4) each thread adds its two tokens' outliers to its four scores
      // directly, reading q[head][pos] from the fragments; sink rows (a sequence's first tile)
      // and q8 go through a tensor-core product of the residual half-tile with the fragments,
      // columns in the dense path's MMA k-order.
      float so[4] = {0.f, 0.f, 0.f, 0.f};
      if (side_work) {
        side_collect<false, NE>(sk + kvoi, reinterpret_cast<const uint16_t*>(sk + kvov), sd.k,
                                sd.n_sink, tb, len, lane, vent);
        uint32_t kent[NE];
        bool mma_pass = true;
        if constexpr (kQShared) {
          // q[n][d] sits in k-step ks = 2 ((d >> 3) & 7) + ((d >> 1) & 1) of lane 4n + (d >> 6),
          // word d & 1, half (d >> 2) & 1; this thread's heads are n = 2c and 2c + 1
          const uint8_t* koi = sk + kkoi;
          const uint16_t* kov = reinterpret_cast<const uint16_t*>(sk + Ly::kBase);
          const uint8_t* qh = smem + qf_off + 64 * c;
#pragma unroll
          for (int r = 0; r < 2; ++r) {
            const int row = tok_order(g + 8 * r);
            if (tb + row < len && tb + row >= sd.n_sink) {
#pragma unroll
              for (int j = 0; j < 2 * NE; ++j) {
                if (j >= sd.k) break;
                const int d = koi[row * sd.k + j];
                const float v = h2f(kov[row * sd.k + j]);
                const uint8_t* qa = qh + 256 * (2 * ((d >> 3) & 7) + ((d >> 1) & 1)) +
                                    8 * (d >> 6) + 4 * (d & 1) + 2 * ((d >> 2) & 1);
                so[2 * r] = fmaf(h2f(*reinterpret_cast<const uint16_t*>(qa)), v, so[2 * r]);
                so[2 * r + 1] =
                    fmaf(h2f(*reinterpret_cast<const uint16_t*>(qa + 32)), v, so[2 * r + 1]);
              }
            }
          }
#pragma unroll
          for (int i = 0; i < NE; ++i) kent[i] = 0u;   // the pass below carries sink rows only
          mma_pass = tb < sd.n_sink;                    // warp-uniform
        } else {
          side_collect<true, NE>(sk + kkoi, reinterpret_cast<const uint16_t*>(sk + Ly::kBase),
                                 sd.k, sd.n_sink, tb, len, lane, kent);
        }
        if (mma_pass) {
          const uint32_t ob = smem_u32(ot) + (lane & 15) * Ly::kOtStride + 16 * (lane >> 4);
          float so4[4][4] = {};   // four independent accumulation chains
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {   // k-steps 8 hf .. 8 hf + 7
            side_half<true, NE>(ot, kent, hf, false, sd.n_sink, sd.ksink[layer], s, a.H, h, tb,
                                len, lane);
            __syncwarp();
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
              uint32_t af[4];
              ldsm_x4(ob + 32 * ks, af);
              const uint2 qb = Q.pair(8 * hf + ks);
              mma16816(so4[ks & 3], af[0], af[1], af[2], af[3], qb.x, qb.y);
            }
            __syncwarp();
            side_half<true, NE>(ot, kent, hf, true, sd.n_sink, sd.ksink[layer], s, a.H, h, tb,
                                len, lane);
            __syncwarp();
          }
#pragma unroll
          for (int k4 = 0; k4 < 4; ++k4)
            so[k4] += (so4[0][k4] + so4[1][k4]) + (so4[2][k4] + so4[3][k4]);
        }
      }
      tile_qk_softmax<BITS, true>(K, Q, acc, m0, m1, l0, l1, a.qk_scale, pb0, pb1, so, sp);
    } else {
      tile_qk_softmax<BITS>(K, Q, acc, m0, m1, l0, l1, a.qk_scale, pb0, pb1);
    }
    VRegs<BITS> V;
#pragma unroll
    for (int qi = 0; qi < 4; ++qi) {
      const int row = SIDE ? tok_order(2 * c + (qi & 1) + 8 * (qi >> 1))
                           : 2 * c + (qi & 1) + 8 * (qi >> 1);
      const uint8_t* src = sv + row * kPd + g * (4 * W::kVWords);
      if constexpr (W::kVWords % 4 == 0) {
#pragma unroll
        for (int i = 0; i < W::kVWords / 4; ++i) {
          const uint4 v = reinterpret_cast<const uint4*>(src)[i];
          V.vw[qi][4 * i] = v.x; V.vw[qi][4 * i + 1] = v.y;
          V.vw[qi][4 * i + 2] = v.z; V.vw[qi][4 * i + 3] = v.w;
        }
      } else {
#pragma unroll
        for (int i = 0; i < W::kVWords / 2; ++i) {
          const uint2 v = reinterpret_cast<const uint2*>(src)[i];
          V.vw[qi][2 * i] = v.x; V.vw[qi][2 * i + 1] = v.y;
        }
      }
    }
    // every byte of the stage has been read: hand it back to the copy engine
    int next_slot = 0;
    const int next_page = (j + S < n_mine) ? page_of(j + S, next_slot) : -1;   // warp-uniform
    __syncwarp();
    if (lane == 0 && j + S < n_mine) {
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      issue(j + S, next_page, next_slot);
      ++issued;
    }
    tile_pv<BITS>(V, pb0, pb1, acc);
    if constexpr (SIDE) {
      if (side_work) {
        // value terms: O^T += R_V^T . P^T with the unscaled probabilities (the residual tile holds
        // real fp16 values), into the same accumulators and running-max domain as the codes
        const uint32_t pv0 = movtrans(pack_h2(sp[0], sp[1]));
        const uint32_t pv1 = movtrans(pack_h2(sp[2], sp[3]));
        const uint32_t ob = smem_u32(ot) + ((lane & 7) + 8 * (lane >> 4)) * Ly::kOtStride +
                            16 * ((lane >> 3) & 1);
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {   // blocks 8 hf .. 8 hf + 7
          side_half<false, NE>(ot, vent, hf, false, sd.n_sink, sd.vsink[layer], s, a.H, h, tb, len,
                               lane);
          __syncwarp();
#pragma unroll
          for (int b = 0; b < 8; ++b) {
            uint32_t af[4];
            ldsm_x4_trans(ob + 32 * b, af);
            mma16816(acc[8 * hf + b], af[0], af[1], af[2], af[3], pv0, pv1);
          }
          __syncwarp();
          side_half<false, NE>(ot, vent, hf, true, sd.n_sink, sd.vsink[layer], s, a.H, h, tb, len,
                               lane);
          __syncwarp();
        }
      }
    }
  }

  if (timed_out) {
    // drain the copies still in flight (bounded) before the shared memory is released: the
    // phases of one stage complete in order, so its last issued phase is the one to wait for
    if (lane == 0) {
      report(a.err, KVQ_DEVERR_TIMEOUT);
      for (int j = issued - S > 0 ? issued - S : 0; j < issued; ++j)
        mbar_wait_bounded(&bars[j % S], static_cast<uint32_t>((j / S) & 1));
    }
    m0 = m1 = kNegInf;
    l0 = l1 = 0.f;
  }
  __syncthreads();  // every warp is done with its stages: reuse them for the merge
  cta_merge_write(a, reinterpret_cast<float*>(smem), ls, h, split, warp, g, c, acc, m0, m1, l0,
                  l1);
}

// ------------------------------------------------------------------------------ gather kernel
// Any page size: each thread loads the rows of its tokens with plain loads.
template <int BITS>
__global__ void __launch_bounds__(kThreads, 3) decode_attn_gather_kernel(const AttnArgs a) {
  using W = Wd<BITS>;
  __shared__ __align__(16) float sm[kMergeBytes / 4];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2;
  const int c = lane & 3;
  const int split = blockIdx.x;
  const int h = blockIdx.y;
  const int ls = blockIdx.z;
  const int layer = ls / a.nseq;
  const int s = ls - layer * a.nseq;
  const LayerPools P = a.L[layer];
  const int len = __ldg(a.lens + s);
  const int n_tiles = (len + kTile - 1) / kTile;
  const int tile0 = split * a.tiles_per_cta;
  if (tile0 >= n_tiles) return;   // no work and no partial, as in the staged kernel
  const int tile1 = min(n_tiles, tile0 + a.tiles_per_cta);

  uint32_t qf[16][2];
  load_q_frags(a, ls, h, g, c, len > 0, qf);
  float acc[16][4];
#pragma unroll
  for (int mt = 0; mt < 16; ++mt)
#pragma unroll
    for (int k = 0; k < 4; ++k) acc[mt][k] = 0.f;
  float m0 = kNegInf, m1 = kNegInf, l0 = 0.f, l1 = 0.f;

  for (int tile = tile0 + warp; tile < tile1; tile += kWarps) {
    const int tb = tile * kTile;
    KRegs<BITS> K;
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int t = tb + g + 8 * r;
      int64_t row = -1;
      if (t < len) row = locate_row(a.pt, a.max_pages, a.ps, a.H, P.k_pages, s, t, h, a.err);
      K.kval[r] = row >= 0;
      K.ks2[r] = 0u;
      K.vsc[r] = 0.f;
      if (t < len) {
        const int64_t vrow = locate_row(a.pt, a.max_pages, a.ps, a.H, P.v_pages, s, t, h, a.err);
        if (vrow >= 0) K.vsc[r] = h2f(ld_nc_u16(P.vs + vrow));
      }
#pragma unroll
      for (int i = 0; i < W::kKWords; ++i) K.kw[r][i] = 0;
      if (row >= 0) {
        const uint8_t* src = P.kc + row * W::kPd + c * (4 * W::kKWords);
#pragma unroll
        for (int i = 0; i < W::kKWords / 4; ++i) {
          const uint4 v = ld_nc_v4(src + 16 * i);
          K.kw[r][4 * i] = v.x; K.kw[r][4 * i + 1] = v.y;
          K.kw[r][4 * i + 2] = v.z; K.kw[r][4 * i + 3] = v.w;
        }
        K.ks2[r] = static_cast<uint32_t>(ld_nc_u16(P.ks + row)) * 0x10001u;
      }
    }
    uint32_t pb0, pb1;
    tile_qk_softmax<BITS>(K, QFragRegs{qf}, acc, m0, m1, l0, l1, a.qk_scale, pb0, pb1);
    VRegs<BITS> V;
#pragma unroll
    for (int qi = 0; qi < 4; ++qi) {
      const int t = tb + 2 * c + (qi & 1) + 8 * (qi >> 1);
      int64_t row = -1;
      if (t < len) row = locate_row(a.pt, a.max_pages, a.ps, a.H, P.v_pages, s, t, h, a.err);
#pragma unroll
      for (int i = 0; i < W::kVWords; ++i) V.vw[qi][i] = 0;
      if (row >= 0) {
        const uint8_t* src = P.vc + row * W::kPd + g * (4 * W::kVWords);
        if constexpr (W::kVWords % 4 == 0) {
#pragma unroll
          for (int i = 0; i < W::kVWords / 4; ++i) {
            const uint4 v = ld_nc_v4(src + 16 * i);
            V.vw[qi][4 * i] = v.x; V.vw[qi][4 * i + 1] = v.y;
            V.vw[qi][4 * i + 2] = v.z; V.vw[qi][4 * i + 3] = v.w;
          }
        } else {
#pragma unroll
          for (int i = 0; i < W::kVWords / 2; ++i) {
            const uint2 v = ld_nc_v2(src + 8 * i);
            V.vw[qi][2 * i] = v.x; V.vw[qi][2 * i + 1] = v.y;
          }
        }
      }
    }
    tile_pv<BITS>(V, pb0, pb1, acc);
  }
  cta_merge_write(a, sm, ls, h, split, warp, g, c, acc, m0, m1, l0, l1);
}

// One CTA per (query head, layer * nseq + seq); thread d merges the splits of element d.  Only
// the splits that start inside the sequence wrote a partial.
__global__ void __launch_bounds__(kD) decode_merge_kernel(const AttnArgs a) {
  const int j = blockIdx.x;
  const int ls = blockIdx.y;
  const int h = j / a.G, jj = j - h * a.G;
  const int d = threadIdx.x;
  const int len = __ldg(a.lens + (ls % a.nseq)) + a.len_add;
  const int n_tiles = (len + kTile - 1) / kTile;
  const int n_live = min(a.n_splits, (n_tiles + a.tiles_per_cta - 1) / a.tiles_per_cta);
  const float* base = a.ws + ((static_cast<int64_t>(ls) * a.H + h) * a.n_splits) * 8 * kRec +
                      jj * kRec;
  float M = kNegInf;
  for (int sp = 0; sp < n_live; ++sp) M = fmaxf(M, base[sp * 8 * kRec + kD]);
  float O = 0.f, L = 0.f;
  if (M != kNegInf) {
    for (int sp = 0; sp < n_live; ++sp) {
      const float* r = base + sp * 8 * kRec;
      const float m = r[kD];
      if (m == kNegInf) continue;
      const float f = exp2f(m - M);
      O += r[d] * f;
      L += r[kD + 1] * f;
    }
  }
  a.out[(static_cast<int64_t>(ls) * a.Hq + j) * kD + d] = (L > 0.f) ? O / L : 0.f;
}

int tiles_per_cta_for(int n_layers, int nseq, int H, int max_seq_len) {
  const int tiles = (max_seq_len + kTile - 1) / kTile;
  const int sms = sm_count() > 0 ? sm_count() : 152;
  const int64_t units = static_cast<int64_t>(n_layers) * nseq * H;
  // aim for >= 2 resident waves (3 CTAs per SM), at most 256 tiles (4096 tokens) per CTA (the
  // entry point without a workspace may raise a CTA's tiles above 256 to fit its partials in its
  // static scratch; no kernel sizes storage by the tiles per CTA)
  const int64_t want_splits = (6LL * sms + units - 1) / units;
  int64_t t = (tiles + want_splits - 1) / want_splits;
  if (t > 256) t = 256;
  t = ((t + kWarps - 1) / kWarps) * kWarps;
  if (t < kWarps) t = kWarps;
  return static_cast<int>(t);
}

template <int BITS, bool APPEND, bool SIDE, int NE>
cudaError_t launch_tma(const AttnArgs& a, dim3 grid, cudaStream_t cs, const AttnSide& sd) {
  const int smem = SIDE ? side_smem_bytes<BITS>(sd.k) : Lay<BITS, SIDE>::kTotal;
  static_assert(Lay<BITS, SIDE>::kRing >= kMergeBytes, "merge buffer must fit in the stage ring");
  cudaError_t e = cudaFuncSetAttribute(decode_attn_tma_kernel<BITS, APPEND, SIDE, NE>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  decode_attn_tma_kernel<BITS, APPEND, SIDE, NE><<<grid, kThreads, smem, cs>>>(a, sd);
  return cudaSuccess;
}

// With side channels each lane holds the outlier entries j = (lane & 1) + 2i, i < NE, of its
// token row: NE = 2 serves up to 4 outliers per row (the pages' 0.01 gives 3 at D = 256) with
// half the entry loops of NE = 4 (up to 8).
template <int BITS, bool APPEND = false, bool SIDE = false>
cudaError_t launch_attn(const AttnArgs& a, dim3 grid, bool tma, cudaStream_t cs,
                        const AttnSide& sd = AttnSide{}) {
  if (tma) {
    cudaError_t e;
    if constexpr (SIDE)
      e = sd.k <= 4 ? launch_tma<BITS, APPEND, SIDE, 2>(a, grid, cs, sd)
                    : launch_tma<BITS, APPEND, SIDE, 4>(a, grid, cs, sd);
    else
      e = launch_tma<BITS, APPEND, SIDE, 4>(a, grid, cs, sd);
    if (e != cudaSuccess) return e;
  } else {
    decode_attn_gather_kernel<BITS><<<grid, kThreads, 0, cs>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace
}  // namespace kvq

extern "C" size_t kvq_decode_attn_workspace(int n_layers, int nseq, int num_kv_heads,
                                            int num_q_heads, int head_dim, int page_size,
                                            int max_seq_len) {
  (void)num_q_heads; (void)head_dim; (void)page_size;
  if (n_layers < 1 || nseq < 1 || num_kv_heads < 1 || max_seq_len < 0) return 0;
  const int tpc = kvq::tiles_per_cta_for(n_layers, nseq, num_kv_heads, max_seq_len);
  const int tiles = (max_seq_len + kvq::kTile - 1) / kvq::kTile;
  const int n_splits = tiles > 0 ? (tiles + tpc - 1) / tpc : 1;
  return static_cast<size_t>(n_layers) * nseq * num_kv_heads * n_splits * 8 * kvq::kRec *
         sizeof(float);
}

namespace kvq {
namespace {

// Validation and kernel arguments shared by every decode entry point (knew/vnew non-NULL: the
// fused append; k_sides/v_sides non-NULL: side channels).  Fills `a` and `sd` except where the
// split partials go and the split plan (ws, tiles_per_cta, n_splits), which each entry sets.
kvq_status prepare_attn(const char* fn, const kvq_pool* k_pools, const kvq_pool* v_pools,
                        int n_layers, const uint16_t* const* knew, const uint16_t* const* vnew,
                        const kvq_side* k_sides, const kvq_side* v_sides, const uint16_t* q,
                        int num_q_heads, const int32_t* page_table, int max_pages,
                        const int32_t* seq_lens, int nseq, int max_seq_len, float softmax_scale,
                        float* out, int32_t* dev_err, AttnArgs& a, AttnSide& sd) {
  const bool append = knew != nullptr || vnew != nullptr;
  const bool side = k_sides != nullptr || v_sides != nullptr;
  if (n_layers < 1 || n_layers > KVQ_MAX_TENSORS)
    return fail(KVQ_ERR_RANGE, "%s: n_layers %d not in [1, %d]", fn, n_layers, KVQ_MAX_TENSORS);
  kvq_status st = check_pools_uniform(k_pools, n_layers, fn);
  if (st != KVQ_OK) return st;
  st = check_pools_uniform(v_pools, n_layers, fn);
  if (st != KVQ_OK) return st;
  const kvq_pool& k0 = k_pools[0];
  const kvq_pool& v0 = v_pools[0];
  if (v0.bits != k0.bits || v0.num_heads != k0.num_heads || v0.head_dim != k0.head_dim ||
      v0.page_size != k0.page_size)
    return fail(KVQ_ERR_SHAPE, "%s: K and V pools differ in shape", fn);
  if (k0.head_dim != kD)
    return fail(KVQ_ERR_SHAPE, "%s: head_dim %d unsupported (256 only)", fn, k0.head_dim);
  const int H = k0.num_heads;
  if (num_q_heads < H || num_q_heads % H || num_q_heads / H > 8)
    return fail(KVQ_ERR_SHAPE, "%s: num_q_heads %d must be a multiple of %d, at most 8 per KV "
                "head", fn, num_q_heads, H);
  if ((append || side) && k0.page_size % kTile)
    return fail(KVQ_ERR_SHAPE, "%s: page_size %d must be a multiple of 16", fn, k0.page_size);
  sd = AttnSide{};
  if (side) {
    if (!k_sides || !v_sides) return fail(KVQ_ERR_NULL, "%s: NULL side array", fn);
    const int k = k_sides[0].n_outlier, ns = k_sides[0].n_sink;
    if (k < 0 || k > KVQ_MAX_OUTLIERS || ns < 0 || ns > KVQ_MAX_SINKS)
      return fail(KVQ_ERR_RANGE, "%s: n_outlier %d / n_sink %d out of range", fn, k, ns);
    for (int i = 0; i < n_layers; ++i) {
      for (const kvq_side* sp : {&k_sides[i], &v_sides[i]}) {
        if (sp->n_outlier != k || sp->n_sink != ns)
          return fail(KVQ_ERR_SHAPE, "%s: sides differ in n_outlier/n_sink", fn);
        if (k > 0 && (!sp->out_val || !sp->out_idx))
          return fail(KVQ_ERR_NULL, "%s: side of layer %d has no outlier arrays", fn, i);
        if (ns > 0 && !sp->sink)
          return fail(KVQ_ERR_NULL, "%s: side of layer %d has no sink buffer", fn, i);
        if ((k > 0 && (!aligned16(sp->out_val) || !aligned16(sp->out_idx))) ||
            (ns > 0 && !aligned16(sp->sink)))
          return fail(KVQ_ERR_ALIGN, "%s: side arrays must be 16-byte aligned", fn);
        if (ns > 0 && sp->max_seqs < nseq)
          return fail(KVQ_ERR_RANGE, "%s: sink buffer holds %d sequences, call has %d", fn,
                      sp->max_seqs, nseq);
      }
      sd.kov[i] = k_sides[i].out_val;
      sd.koi[i] = k_sides[i].out_idx;
      sd.vov[i] = v_sides[i].out_val;
      sd.voi[i] = v_sides[i].out_idx;
      sd.ksink[i] = k_sides[i].sink;
      sd.vsink[i] = v_sides[i].sink;
    }
    sd.k = k;
    sd.n_sink = ns;
  }
  if (nseq < 1 || max_pages < 1 || max_seq_len < 0)
    return fail(KVQ_ERR_RANGE, "%s: bad nseq/max_pages/max_seq_len", fn);
  if (static_cast<int64_t>(max_seq_len) > static_cast<int64_t>(max_pages) * k0.page_size)
    return fail(KVQ_ERR_RANGE, "%s: max_seq_len exceeds max_pages * page_size", fn);
  if (!q || !page_table || !seq_lens || !out) return fail(KVQ_ERR_NULL, "%s: NULL pointer", fn);
  if (!aligned16(q) || !aligned16(out))
    return fail(KVQ_ERR_ALIGN, "%s: q/out must be 16-byte aligned", fn);
  if (append) {
    if (!knew || !vnew) return fail(KVQ_ERR_NULL, "%s: NULL new-token array", fn);
    for (int i = 0; i < n_layers; ++i) {
      if (!knew[i] || !vnew[i]) return fail(KVQ_ERR_NULL, "%s: new K/V of layer %d is NULL", fn, i);
      if (!aligned16(knew[i]) || !aligned16(vnew[i]))
        return fail(KVQ_ERR_ALIGN, "%s: new K/V rows must be 16-byte aligned", fn);
    }
  }
  if (static_cast<int64_t>(n_layers) * nseq > 65535)
    return fail(KVQ_ERR_RANGE, "%s: n_layers * nseq > 65535", fn);

  for (int i = 0; i < KVQ_MAX_TENSORS; ++i) {
    if (i < n_layers)
      a.L[i] = LayerPools{k_pools[i].codes, k_pools[i].scales, v_pools[i].codes,
                          v_pools[i].scales, k_pools[i].num_pages, v_pools[i].num_pages};
    else
      a.L[i] = LayerPools{nullptr, nullptr, nullptr, nullptr, 0, 0};
    a.knew[i] = (append && i < n_layers) ? knew[i] : nullptr;
    a.vnew[i] = (append && i < n_layers) ? vnew[i] : nullptr;
  }
  a.q = q;
  a.out = out;
  a.ws = nullptr;
  a.pt = page_table;
  a.lens = seq_lens;
  a.err = dev_err;
  a.n_layers = n_layers;
  a.nseq = nseq;
  a.H = H;
  a.G = num_q_heads / H;
  a.Hq = num_q_heads;
  a.ps = k0.page_size;
  a.max_pages = max_pages;
  a.n_splits = 0;
  a.tiles_per_cta = 0;
  a.len_add = append ? 1 : 0;
  a.qk_scale = softmax_scale * 1.4426950408889634f;
  return KVQ_OK;
}

// Launches the attention kernel of the call's width and variant over (split, KV head,
// layer * nseq + seq), then the split merge.
kvq_status launch_decode(const char* fn, const AttnArgs& a, int bits, bool append, bool side,
                         const AttnSide& sd, cudaStream_t cs) {
  const dim3 grid(a.n_splits, a.H, a.n_layers * a.nseq);
  const bool tma = (a.ps % kTile) == 0;
  cudaError_t e;
  switch (bits) {
    case 8:
      e = side ? launch_attn<8, false, true>(a, grid, tma, cs, sd)
               : append ? launch_attn<8, true>(a, grid, tma, cs) : launch_attn<8>(a, grid, tma, cs);
      break;
    case 6:
      e = side ? launch_attn<6, false, true>(a, grid, tma, cs, sd)
               : append ? launch_attn<6, true>(a, grid, tma, cs) : launch_attn<6>(a, grid, tma, cs);
      break;
    default:
      e = side ? launch_attn<4, false, true>(a, grid, tma, cs, sd)
               : append ? launch_attn<4, true>(a, grid, tma, cs) : launch_attn<4>(a, grid, tma, cs);
      break;
  }
  if (e == cudaSuccess) {
    decode_merge_kernel<<<dim3(a.Hq, a.n_layers * a.nseq), kD, 0, cs>>>(a);
    e = cudaGetLastError();
  }
  if (e != cudaSuccess) return fail(KVQ_ERR_CUDA, "%s launch: %s", fn, cudaGetErrorString(e));
  return ok();
}

// The entry points with a caller-provided workspace for the split partials.
kvq_status decode_attn_entry(const char* fn, const kvq_pool* k_pools, const kvq_pool* v_pools,
                             int n_layers, const uint16_t* const* knew,
                             const uint16_t* const* vnew, const kvq_side* k_sides,
                             const kvq_side* v_sides, const uint16_t* q, int num_q_heads,
                             const int32_t* page_table, int max_pages, const int32_t* seq_lens,
                             int nseq, int max_seq_len, float softmax_scale, float* out,
                             void* workspace, size_t workspace_bytes, int32_t* dev_err,
                             cudaStream_t cs) {
  AttnArgs a;
  AttnSide sd;
  const kvq_status st = prepare_attn(fn, k_pools, v_pools, n_layers, knew, vnew, k_sides, v_sides,
                                     q, num_q_heads, page_table, max_pages, seq_lens, nseq,
                                     max_seq_len, softmax_scale, out, dev_err, a, sd);
  if (st != KVQ_OK) return st;
  if (!workspace) return fail(KVQ_ERR_NULL, "%s: NULL workspace", fn);
  if (!aligned16(workspace))
    return fail(KVQ_ERR_ALIGN, "%s: workspace must be 16-byte aligned", fn);
  const size_t need = kvq_decode_attn_workspace(n_layers, nseq, a.H, num_q_heads, kD, a.ps,
                                                max_seq_len);
  if (workspace_bytes < need)
    return fail(KVQ_ERR_WORKSPACE, "%s: workspace %zu < %zu bytes", fn, workspace_bytes, need);
  a.ws = static_cast<float*>(workspace);
  a.tiles_per_cta = tiles_per_cta_for(n_layers, nseq, a.H, max_seq_len);
  const int tiles = (max_seq_len + kTile - 1) / kTile;
  a.n_splits = tiles > 0 ? (tiles + a.tiles_per_cta - 1) / a.tiles_per_cta : 1;
  return launch_decode(fn, a, k_pools[0].bits, knew != nullptr || vnew != nullptr,
                       k_sides != nullptr || v_sides != nullptr, sd, cs);
}

}  // namespace
}  // namespace kvq

extern "C" kvq_status kvq_decode_attn(const kvq_pool* k_pools, const kvq_pool* v_pools,
                                      int n_layers, const uint16_t* q, int num_q_heads,
                                      const int32_t* page_table, int max_pages,
                                      const int32_t* seq_lens, int nseq, int max_seq_len,
                                      float softmax_scale, float* out, void* workspace,
                                      size_t workspace_bytes, int32_t* dev_err,
                                      kvq_stream_t stream) {
  return kvq::decode_attn_entry("kvq_decode_attn", k_pools, v_pools, n_layers, nullptr, nullptr,
                                nullptr, nullptr, q, num_q_heads, page_table, max_pages, seq_lens, nseq,
                                max_seq_len, softmax_scale, out, workspace, workspace_bytes,
                                dev_err, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" kvq_status kvq_append_decode_attn(const kvq_pool* k_pools, const kvq_pool* v_pools,
                                             int n_layers, const uint16_t* const* k_new,
                                             const uint16_t* const* v_new, const uint16_t* q,
                                             int num_q_heads, const int32_t* page_table,
                                             int max_pages, const int32_t* seq_lens, int nseq,
                                             int max_seq_len, float softmax_scale, float* out,
                                             void* workspace, size_t workspace_bytes,
                                             int32_t* dev_err, kvq_stream_t stream) {
  if (!k_new || !v_new)
    return kvq::fail(KVQ_ERR_NULL, "kvq_append_decode_attn: NULL new-token array");
  return kvq::decode_attn_entry("kvq_append_decode_attn", k_pools, v_pools, n_layers, k_new,
                                v_new, nullptr, nullptr, q, num_q_heads, page_table, max_pages, seq_lens, nseq,
                                max_seq_len, softmax_scale, out, workspace, workspace_bytes,
                                dev_err, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" kvq_status kvq_decode_attn_side(const kvq_pool* k_pools, const kvq_pool* v_pools,
                                           const kvq_side* k_sides, const kvq_side* v_sides,
                                           int n_layers, const uint16_t* q, int num_q_heads,
                                           const int32_t* page_table, int max_pages,
                                           const int32_t* seq_lens, int nseq, int max_seq_len,
                                           float softmax_scale, float* out, void* workspace,
                                           size_t workspace_bytes, int32_t* dev_err,
                                           kvq_stream_t stream) {
  if (!k_sides || !v_sides)
    return kvq::fail(KVQ_ERR_NULL, "kvq_decode_attn_side: NULL side array");
  return kvq::decode_attn_entry("kvq_decode_attn_side", k_pools, v_pools, n_layers, nullptr,
                                nullptr, k_sides, v_sides, q, num_q_heads, page_table, max_pages,
                                seq_lens, nseq, max_seq_len, softmax_scale, out, workspace,
                                workspace_bytes, dev_err, reinterpret_cast<cudaStream_t>(stream));
}

// ------------------------------------------------------------------------------------------------
// Decode attention without a caller-provided workspace.
//
// Some callers cannot call cudaMalloc at the point where they run attention: code embedded in a
// runtime whose own allocator owns all device memory, or a latency-critical serving loop that
// must not allocate (cudaMalloc can synchronize the device) once it is running.  For them the
// split partials live in a fixed array of device memory that belongs to this library: every GPU
// that loads the library holds it (32 MiB) until the process exits.
namespace kvq {
namespace {

constexpr size_t kNoAllocScratchBytes = static_cast<size_t>(32) << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of the scratch array for the current device.  The host-side name of the array
// is only a stand-in, so the address is looked up once per device (with that device current)
// and cached.
kvq_status noalloc_scratch(void** out) {
  static std::mutex mu;
  static std::vector<void*> cache;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess)
    return fail(KVQ_ERR_CUDA, "kvq_decode_attn_noalloc: cudaGetDevice: %s", cudaGetErrorString(e));
  std::lock_guard<std::mutex> lock(mu);
  if (static_cast<int>(cache.size()) <= dev) cache.resize(dev + 1, nullptr);
  if (cache[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr)
      return fail(KVQ_ERR_CUDA, "kvq_decode_attn_noalloc: cudaGetSymbolAddress: %s",
                  cudaGetErrorString(e));
    cache[dev] = p;
  }
  *out = cache[dev];
  return KVQ_OK;
}

}  // namespace
}  // namespace kvq

extern "C" kvq_status kvq_decode_attn_noalloc(const kvq_pool* k_pools, const kvq_pool* v_pools,
                                              int n_layers, const uint16_t* q, int num_q_heads,
                                              const int32_t* page_table, int max_pages,
                                              const int32_t* seq_lens, int nseq, int max_seq_len,
                                              float softmax_scale, float* out, int32_t* dev_err,
                                              kvq_stream_t stream) {
  using namespace kvq;
  const char* fn = "kvq_decode_attn_noalloc";
  AttnArgs a;
  AttnSide sd;
  kvq_status st = prepare_attn(fn, k_pools, v_pools, n_layers, nullptr, nullptr, nullptr, nullptr,
                               q, num_q_heads, page_table, max_pages, seq_lens, nseq, max_seq_len,
                               softmax_scale, out, dev_err, a, sd);
  if (st != KVQ_OK) return st;

  // One partial record per (layer, sequence, KV head, split); the split count is capped so that
  // all records fit in the static scratch (the splits then grow past the usual 256 tiles).
  const size_t per_split = static_cast<size_t>(n_layers) * nseq * a.H * 8 * kRec * sizeof(float);
  if (per_split > kNoAllocScratchBytes)
    return fail(KVQ_ERR_RANGE, "%s: %d layers x %d sequences x %d KV heads need %zu bytes of "
                "scratch, more than the %zu-byte static scratch; use kvq_decode_attn with a "
                "workspace", fn, n_layers, nseq, a.H, per_split, kNoAllocScratchBytes);
  const int tiles = (max_seq_len + kTile - 1) / kTile;
  const int max_splits = static_cast<int>(kNoAllocScratchBytes / per_split);
  int tpc = tiles_per_cta_for(n_layers, nseq, a.H, max_seq_len);
  int n_splits = tiles > 0 ? (tiles + tpc - 1) / tpc : 1;
  if (n_splits > max_splits) {
    tpc = (tiles + max_splits - 1) / max_splits;
    tpc = ((tpc + kWarps - 1) / kWarps) * kWarps;
    n_splits = (tiles + tpc - 1) / tpc;
  }
  void* ws = nullptr;
  st = noalloc_scratch(&ws);
  if (st != KVQ_OK) return st;
  a.ws = static_cast<float*>(ws);
  a.tiles_per_cta = tpc;
  a.n_splits = n_splits;
  return launch_decode(fn, a, k_pools[0].bits, false, false, sd,
                       reinterpret_cast<cudaStream_t>(stream));
}
