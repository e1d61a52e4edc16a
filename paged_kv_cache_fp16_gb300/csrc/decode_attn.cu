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
// unpacks whole 24-bit q6 quads (or q4/q8 words) it loaded itself: no shared-memory staging of
// the dequantized tile.  The 4 warps' (m, l, O) are merged in shared memory, each split writes
// one partial, and a second kernel merges the splits (log-sum-exp).
//
// The unpack turns each 6/4/8-bit field into an fp16 with a known exponent by OR-ing it into
// the mantissa of 1024 (0x6400), then one half2 FMA removes the 1024 and the bias exactly.
#include <cuda_runtime.h>
#include <cuda_fp16.h>

#include "kvq_device.cuh"
#include "kvq_internal.h"

namespace kvq {
namespace {

constexpr int kD = 256;
constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kTile = 16;
constexpr int kRec = kD + 4;   // workspace record per (split, head): O[256], m, l, pad, pad
#define kNegInf (-__int_as_float(0x7f800000))

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
  int n_layers, nseq, H, G, Hq, ps, max_pages, n_splits, tiles_per_cta;
  float qk_scale;  // softmax_scale * log2(e)
};

template <int BITS> struct Wd;
template <> struct Wd<8> { static constexpr int kPd = 256, kKWords = 16, kVWords = 8; };
template <> struct Wd<6> { static constexpr int kPd = 192, kKWords = 12, kVWords = 6; };
template <> struct Wd<4> { static constexpr int kPd = 128, kKWords = 8, kVWords = 4; };

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}

__device__ __forceinline__ uint32_t hfma2u(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t r;
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(c));
  return r;
}

__device__ __forceinline__ uint32_t hmul2u(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// fp16x2 constants
constexpr uint32_t kH1 = 0x3C003C00u;        // 1.0
constexpr uint32_t kH16th = 0x2C002C00u;     // 0.0625
constexpr uint32_t kHQuarter = 0x34003400u;  // 0.25
constexpr uint32_t kHm1056 = 0xE420E420u;    // -1056
constexpr uint32_t kHm96 = 0xD600D600u;      // -96
constexpr uint32_t kHm288 = 0xDC80DC80u;     // -288
constexpr uint32_t kHm1032 = 0xE408E408u;    // -1032
constexpr uint32_t kHm1152 = 0xE480E480u;    // -1152

// Eight consecutive elements e0..e7 (group `gi` of a thread's loaded words) -> four half2 holding
// the exact signed codes {e_k, e_{k+4}}, k = 0..3.
template <int BITS, int GI>
__device__ __forceinline__ void unpack_group(const uint32_t* w, uint32_t p[4]) {
  if constexpr (BITS == 6) {
    // two 24-bit quads at byte 6*GI: fields u0..u3 (quad 0) and u0'..u3' (quad 1)
    constexpr int b = 6 * GI;
    constexpr int w0 = b / 4;
    const uint32_t x = w[w0], y = w[w0 + 1];
    constexpr uint32_t s1 = (b % 4 == 0) ? 0x4310u : 0x6532u;  // [B0 B1 B3 B4]
    constexpr uint32_t s2 = (b % 4 == 0) ? 0x5421u : 0x7643u;  // [B1 B2 B4 B5]
    const uint32_t p1 = prmt(x, y, s1);
    const uint32_t p2 = prmt(x, y, s2);
    p[0] = hfma2u((p1 & 0x003F003Fu) | 0x64006400u, kH1, kHm1056);            // 1024 + u0
    p[1] = hfma2u(((p1 >> 2) & 0x03F003F0u) | 0x64006400u, kH16th, kHm96);     // 1024 + 16 u1
    p[2] = hfma2u((p2 & 0x03F003F0u) | 0x64006400u, kH16th, kHm96);            // 1024 + 16 u2
    p[3] = hfma2u(((p2 >> 8) & 0x00FC00FCu) | 0x64006400u, kHQuarter, kHm288); // 1024 + 4 u3
  } else if constexpr (BITS == 4) {
    const uint32_t x = w[GI];  // nibble n = element n
#pragma unroll
    for (int k = 0; k < 4; ++k)
      p[k] = hfma2u(((x >> (4 * k)) & 0x000F000Fu) | 0x64006400u, kH1, kHm1032);
  } else {
    const uint32_t x = w[2 * GI], y = w[2 * GI + 1];  // bytes e0..e3, e4..e7 (int8)
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint32_t sel = static_cast<uint32_t>(k | (k << 4) | ((4 + k) << 8) | ((4 + k) << 12));
      p[k] = hfma2u((prmt(x, y, sel) & 0x00FF00FFu) ^ 0x64806480u, kH1, kHm1152);  // 1024+c+128
    }
  }
}

__device__ __forceinline__ void mma16816(float c[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t movtrans(uint32_t x) {
  uint32_t r;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(r) : "r"(x));
  return r;
}

__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// Physical row of token `t` of sequence `s`, head h; -1 if out of range (error bit set).
__device__ __forceinline__ int64_t token_row(const AttnArgs& a, int s, int t, int h,
                                             int64_t num_pages) {
  return locate_row(a.pt, a.max_pages, a.ps, a.H, num_pages, s, t, h, a.err);
}

template <int BITS>
__global__ void __launch_bounds__(kThreads, 2) decode_attn_kernel(const AttnArgs a) {
  using W = Wd<BITS>;
  __shared__ float sm_o[kWarps][8][kD];
  __shared__ float sm_m[kWarps][8];
  __shared__ float sm_l[kWarps][8];

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2;   // fragment row group
  const int c = lane & 3;    // fragment column pair
  const int split = blockIdx.x;
  const int h = blockIdx.y;
  const int ls = blockIdx.z;             // layer * nseq + seq
  const int layer = ls / a.nseq;
  const int s = ls - layer * a.nseq;
  const LayerPools P = a.L[layer];
  const int len = __ldg(a.lens + s);
  const int n_tiles = (len + kTile - 1) / kTile;
  const int tile0 = split * a.tiles_per_cta;
  const int tile1 = min(n_tiles, tile0 + a.tiles_per_cta);

  // Q^T B-fragments for head g of this KV head's group (zero for padding heads).
  uint32_t qf[16][2];
  {
    uint32_t qw[32];
    if (g < a.G && len > 0) {
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

  float acc[16][4];
#pragma unroll
  for (int mt = 0; mt < 16; ++mt)
#pragma unroll
    for (int k = 0; k < 4; ++k) acc[mt][k] = 0.f;
  float m0 = kNegInf, m1 = kNegInf, l0 = 0.f, l1 = 0.f;

  for (int tile = tile0 + warp; tile < tile1; tile += kWarps) {
    const int tb = tile * kTile;
    // ---------------- S^T = K_hat . Q^T
    uint32_t kw[2][W::kKWords];
    uint32_t ksc[2];
    bool kval[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int t = tb + g + 8 * r;
      int64_t row = -1;
      if (t < len) row = token_row(a, s, t, h, P.k_pages);
      kval[r] = row >= 0;
      ksc[r] = 0;
#pragma unroll
      for (int i = 0; i < W::kKWords; ++i) kw[r][i] = 0;
      if (row >= 0) {
        const uint8_t* src = P.kc + row * W::kPd + c * (4 * W::kKWords);
#pragma unroll
        for (int i = 0; i < W::kKWords / 4; ++i) {
          const uint4 v = ld_nc_v4(src + 16 * i);
          kw[r][4 * i] = v.x; kw[r][4 * i + 1] = v.y; kw[r][4 * i + 2] = v.z; kw[r][4 * i + 3] = v.w;
        }
        const uint32_t sb = ld_nc_u16(P.ks + row);
        ksc[r] = sb | (sb << 16);
      }
    }
    float sacc[4] = {0.f, 0.f, 0.f, 0.f};
#define KVQ_QK_GROUP(GI)                                                              \
    {                                                                                 \
      uint32_t p0[4], p1[4];                                                          \
      unpack_group<BITS, GI>(kw[0], p0);                                              \
      unpack_group<BITS, GI>(kw[1], p1);                                              \
      _Pragma("unroll") for (int k = 0; k < 4; ++k) {                                 \
        p0[k] = hmul2u(p0[k], ksc[0]);                                                \
        p1[k] = hmul2u(p1[k], ksc[1]);                                                \
      }                                                                               \
      mma16816(sacc, p0[0], p1[0], p0[1], p1[1], qf[2 * GI][0], qf[2 * GI][1]);       \
      mma16816(sacc, p0[2], p1[2], p0[3], p1[3], qf[2 * GI + 1][0], qf[2 * GI + 1][1]); \
    }
    KVQ_QK_GROUP(0) KVQ_QK_GROUP(1) KVQ_QK_GROUP(2) KVQ_QK_GROUP(3)
    KVQ_QK_GROUP(4) KVQ_QK_GROUP(5) KVQ_QK_GROUP(6) KVQ_QK_GROUP(7)
#undef KVQ_QK_GROUP

    // ---------------- online softmax (log2 domain); sacc: [tok g | g+8][head 2c | 2c+1]
    float sc[4];
    sc[0] = kval[0] ? sacc[0] * a.qk_scale : kNegInf;
    sc[1] = kval[0] ? sacc[1] * a.qk_scale : kNegInf;
    sc[2] = kval[1] ? sacc[2] * a.qk_scale : kNegInf;
    sc[3] = kval[1] ? sacc[3] * a.qk_scale : kNegInf;
    float tm0 = fmaxf(sc[0], sc[2]), tm1 = fmaxf(sc[1], sc[3]);
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      tm0 = fmaxf(tm0, __shfl_xor_sync(kFullMask, tm0, o));
      tm1 = fmaxf(tm1, __shfl_xor_sync(kFullMask, tm1, o));
    }
    const float n0 = fmaxf(m0, tm0), n1 = fmaxf(m1, tm1);
    const float al0 = (n0 == kNegInf) ? 1.f : exp2f(m0 - n0);
    const float al1 = (n1 == kNegInf) ? 1.f : exp2f(m1 - n1);
    float p[4];
    p[0] = (n0 == kNegInf) ? 0.f : exp2f(sc[0] - n0);
    p[2] = (n0 == kNegInf) ? 0.f : exp2f(sc[2] - n0);
    p[1] = (n1 == kNegInf) ? 0.f : exp2f(sc[1] - n1);
    p[3] = (n1 == kNegInf) ? 0.f : exp2f(sc[3] - n1);
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
    const uint32_t pb0 = movtrans(pack_h2(p[0], p[1]));   // tokens 2c, 2c+1 ; head g
    const uint32_t pb1 = movtrans(pack_h2(p[2], p[3]));   // tokens 8+2c, 8+2c+1 ; head g

    // ---------------- O^T += V_hat^T . P^T ; thread tokens 2c, 2c+1, 2c+8, 2c+9, d in [32g, 32g+32)
    uint32_t vw[4][W::kVWords];
    uint32_t vsc[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int t = tb + 2 * c + (q & 1) + 8 * (q >> 1);
      int64_t row = -1;
      if (t < len) row = token_row(a, s, t, h, P.v_pages);
      vsc[q] = 0;
#pragma unroll
      for (int i = 0; i < W::kVWords; ++i) vw[q][i] = 0;
      if (row >= 0) {
        const uint8_t* src = P.vc + row * W::kPd + g * (4 * W::kVWords);
        if constexpr (W::kVWords % 4 == 0) {
#pragma unroll
          for (int i = 0; i < W::kVWords / 4; ++i) {
            const uint4 v = ld_nc_v4(src + 16 * i);
            vw[q][4 * i] = v.x; vw[q][4 * i + 1] = v.y; vw[q][4 * i + 2] = v.z; vw[q][4 * i + 3] = v.w;
          }
        } else {
#pragma unroll
          for (int i = 0; i < W::kVWords / 2; ++i) {
            const uint2 v = ld_nc_v2(src + 8 * i);
            vw[q][2 * i] = v.x; vw[q][2 * i + 1] = v.y;
          }
        }
        vsc[q] = ld_nc_u16(P.vs + row);
      }
    }
    const uint32_t sab = vsc[0] | (vsc[1] << 16), scd = vsc[2] | (vsc[3] << 16);
#define KVQ_PV_GROUP(GI)                                                                \
    {                                                                                   \
      uint32_t pa[4], pb[4], pc[4], pd[4];                                              \
      unpack_group<BITS, GI>(vw[0], pa);                                                \
      unpack_group<BITS, GI>(vw[1], pb);                                                \
      unpack_group<BITS, GI>(vw[2], pc);                                                \
      unpack_group<BITS, GI>(vw[3], pd);                                                \
      _Pragma("unroll") for (int k = 0; k < 4; ++k) {                                   \
        const uint32_t lab = hmul2u(prmt(pa[k], pb[k], 0x5410u), sab);                 \
        const uint32_t hab = hmul2u(prmt(pa[k], pb[k], 0x7632u), sab);                 \
        const uint32_t lcd = hmul2u(prmt(pc[k], pd[k], 0x5410u), scd);                 \
        const uint32_t hcd = hmul2u(prmt(pc[k], pd[k], 0x7632u), scd);                 \
        mma16816(acc[4 * GI + k], lab, hab, lcd, hcd, pb0, pb1);                        \
      }                                                                                 \
    }
    KVQ_PV_GROUP(0) KVQ_PV_GROUP(1) KVQ_PV_GROUP(2) KVQ_PV_GROUP(3)
#undef KVQ_PV_GROUP
  }

  // ---------------- merge the warps in shared memory
#pragma unroll
  for (int o = 4; o < 32; o <<= 1) {
    l0 += __shfl_xor_sync(kFullMask, l0, o);
    l1 += __shfl_xor_sync(kFullMask, l1, o);
  }
  if (g == 0) {
    sm_m[warp][2 * c] = m0; sm_m[warp][2 * c + 1] = m1;
    sm_l[warp][2 * c] = l0; sm_l[warp][2 * c + 1] = l1;
  }
#pragma unroll
  for (int mt = 0; mt < 16; ++mt) {
    const int gi = mt >> 2, k = mt & 3;
    const int d = 32 * g + 8 * gi + k;
    sm_o[warp][2 * c][d] = acc[mt][0];
    sm_o[warp][2 * c + 1][d] = acc[mt][1];
    sm_o[warp][2 * c][d + 4] = acc[mt][2];
    sm_o[warp][2 * c + 1][d + 4] = acc[mt][3];
  }
  __syncthreads();
  float* rec = a.ws + ((static_cast<int64_t>(ls) * a.H + h) * a.n_splits + split) * 8 * kRec;
  for (int i = threadIdx.x; i < a.G * kD; i += kThreads) {
    const int j = i / kD, d = i - j * kD;
    float M = kNegInf;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, sm_m[w][j]);
    float O = 0.f, Lsum = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float f = (sm_m[w][j] == kNegInf) ? 0.f : exp2f(sm_m[w][j] - M);
      O += sm_o[w][j][d] * f;
      Lsum += sm_l[w][j] * f;
    }
    rec[j * kRec + d] = O;
    if (d == 0) {
      rec[j * kRec + kD] = M;
      rec[j * kRec + kD + 1] = Lsum;
    }
  }
}

// One CTA per (layer, seq, query head); thread d merges the splits of output element d.
__global__ void __launch_bounds__(kD) decode_merge_kernel(const AttnArgs a) {
  const int j = blockIdx.x;        // query head
  const int ls = blockIdx.y;       // layer * nseq + seq
  const int h = j / a.G, jj = j - h * a.G;
  const int d = threadIdx.x;
  const float* base = a.ws + ((static_cast<int64_t>(ls) * a.H + h) * a.n_splits) * 8 * kRec +
                      jj * kRec;
  float M = kNegInf;
  for (int sp = 0; sp < a.n_splits; ++sp) M = fmaxf(M, base[sp * 8 * kRec + kD]);
  float O = 0.f, L = 0.f;
  if (M != kNegInf) {
    for (int sp = 0; sp < a.n_splits; ++sp) {
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
  // aim for >= 8 CTAs per SM over the whole grid, at most 64 tiles (1024 tokens) per CTA
  const int64_t want_splits = (8LL * sms + units - 1) / units;
  int64_t t = (tiles + want_splits - 1) / want_splits;
  if (t > 64) t = 64;
  t = ((t + kWarps - 1) / kWarps) * kWarps;
  if (t < kWarps) t = kWarps;
  return static_cast<int>(t);
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

extern "C" kvq_status kvq_decode_attn(const kvq_pool* k_pools, const kvq_pool* v_pools,
                                      int n_layers, const uint16_t* q, int num_q_heads,
                                      const int32_t* page_table, int max_pages,
                                      const int32_t* seq_lens, int nseq, int max_seq_len,
                                      float softmax_scale, float* out, void* workspace,
                                      size_t workspace_bytes, int32_t* dev_err,
                                      kvq_stream_t stream) {
  using namespace kvq;
  if (n_layers < 1 || n_layers > KVQ_MAX_TENSORS)
    return fail(KVQ_ERR_RANGE, "kvq_decode_attn: n_layers %d not in [1, %d]", n_layers,
                KVQ_MAX_TENSORS);
  kvq_status st = check_pools_uniform(k_pools, n_layers, "kvq_decode_attn(k)");
  if (st != KVQ_OK) return st;
  st = check_pools_uniform(v_pools, n_layers, "kvq_decode_attn(v)");
  if (st != KVQ_OK) return st;
  const kvq_pool& k0 = k_pools[0];
  const kvq_pool& v0 = v_pools[0];
  if (v0.bits != k0.bits || v0.num_heads != k0.num_heads || v0.head_dim != k0.head_dim ||
      v0.page_size != k0.page_size)
    return fail(KVQ_ERR_SHAPE, "kvq_decode_attn: K and V pools differ in shape");
  if (k0.head_dim != kD)
    return fail(KVQ_ERR_SHAPE, "kvq_decode_attn: head_dim %d unsupported (256 only)",
                k0.head_dim);
  const int H = k0.num_heads;
  if (num_q_heads < H || num_q_heads % H || num_q_heads / H > 8)
    return fail(KVQ_ERR_SHAPE, "kvq_decode_attn: num_q_heads %d must be a multiple of %d, "
                "at most 8 per KV head", num_q_heads, H);
  if (nseq < 1 || max_pages < 1 || max_seq_len < 0)
    return fail(KVQ_ERR_RANGE, "kvq_decode_attn: bad nseq/max_pages/max_seq_len");
  if (static_cast<int64_t>(max_seq_len) > static_cast<int64_t>(max_pages) * k0.page_size)
    return fail(KVQ_ERR_RANGE, "kvq_decode_attn: max_seq_len exceeds max_pages * page_size");
  if (!q || !page_table || !seq_lens || !out || !workspace)
    return fail(KVQ_ERR_NULL, "kvq_decode_attn: NULL pointer");
  if (!aligned16(q) || !aligned16(out) || !aligned16(workspace))
    return fail(KVQ_ERR_ALIGN, "kvq_decode_attn: q/out/workspace must be 16-byte aligned");
  const size_t need = kvq_decode_attn_workspace(n_layers, nseq, H, num_q_heads, kD,
                                                k0.page_size, max_seq_len);
  if (workspace_bytes < need)
    return fail(KVQ_ERR_WORKSPACE, "kvq_decode_attn: workspace %zu < %zu bytes",
                workspace_bytes, need);
  if (static_cast<int64_t>(n_layers) * nseq > 65535)
    return fail(KVQ_ERR_RANGE, "kvq_decode_attn: n_layers * nseq > 65535");

  AttnArgs a;
  for (int i = 0; i < KVQ_MAX_TENSORS; ++i) {
    if (i < n_layers)
      a.L[i] = LayerPools{k_pools[i].codes, k_pools[i].scales, v_pools[i].codes,
                          v_pools[i].scales, k_pools[i].num_pages, v_pools[i].num_pages};
    else
      a.L[i] = LayerPools{nullptr, nullptr, nullptr, nullptr, 0, 0};
  }
  a.q = q;
  a.out = out;
  a.ws = static_cast<float*>(workspace);
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
  a.tiles_per_cta = tiles_per_cta_for(n_layers, nseq, H, max_seq_len);
  const int tiles = (max_seq_len + kTile - 1) / kTile;
  a.n_splits = tiles > 0 ? (tiles + a.tiles_per_cta - 1) / a.tiles_per_cta : 1;
  a.qk_scale = softmax_scale * 1.4426950408889634f;

  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  const dim3 grid(a.n_splits, H, n_layers * nseq);
  switch (k0.bits) {
    case 8: decode_attn_kernel<8><<<grid, kThreads, 0, cs>>>(a); break;
    case 6: decode_attn_kernel<6><<<grid, kThreads, 0, cs>>>(a); break;
    default: decode_attn_kernel<4><<<grid, kThreads, 0, cs>>>(a); break;
  }
  decode_merge_kernel<<<dim3(num_q_heads, n_layers * nseq), kD, 0, cs>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(KVQ_ERR_CUDA, "decode attention launch: %s",
                                    cudaGetErrorString(e));
  return ok();
}
