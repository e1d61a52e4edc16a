// Packed KIVI storage (b-bit codes + fp16 scale and zero per group) and decode attention over it.
//
// VeloxQuant-MLX source page "veloxquant_mlx.cache.kivi_cache": the page keeps its KIVI cache in
// fp16 and estimates what a packed form would cost (module docstring, _quantized_bytes,
// _account_bytes): b-bit codes plus an fp16 (scale, zero) pair per group -- per (token group,
// channel) for keys, per (token, channel group) for values.  This file stores exactly that:
//   zero = gmin (an fp16 value already); scale = fp16(max(float32(gmax - gmin) / levels, eps));
//   c = clamp(rint(float32(x - gmin) / float32(scale)), 0, levels), 0 if the fp16 scale is 0;
//   codes LSB-first along the head dimension of each token row.
// Reconstruction for attention is one fp16 fused multiply-add c * scale + zero per element.
//
// kivi_pack: keys at head_dim 64 -- one warp per (layer, b, h, token group), each lane holding an
// 8-channel chunk of a quarter of the group's rows, min/max by shuffles; other head dims -- one
// thread per (layer, b, h, token group, 8-channel chunk), re-reading the rows (cache hits);
// values -- one thread per (layer, b, h, token, channel group) holding the group in registers.
// 2-bit codes come from fp16 compares against each group's code boundaries (kvq_kivi_cut.cuh);
// wider codes divide by the stored scale.
//
// kivi_decode_attn (head_dim 64): one CTA per (split, KV head, layer * batch); 4 warps, 16-token
// tiles; S^T = K_hat . Q^T and O^T += V_hat^T . P^T on mma.sync m16n8k16 as in the q8/q6/q4
// decode kernel.  Each thread's 2-bit codes for a tile arrive in one word per K row and one
// half-word per V token; a field placed in the mantissa of fp16 1024 becomes an exact fp16 code
// with one half2 FMA, and one more half2 FMA applies the group's scale and zero.  V fields of two
// tokens are paired in one word, so the V operand needs no re-pairing.  Tokens [n_packed, offset)
// come from the fp16 cache (the residual window).  Splits are merged by log-sum-exp.
#include <cmath>

#include <cuda_runtime.h>
#include <cuda_fp16.h>

#include "kvq_device.cuh"
#include "kvq_divu32.cuh"
#include "kvq_internal.h"
#include "kvq_kivi_cut.cuh"
#include "kvq_math.cuh"
#include "kvq_warp.cuh"

namespace kvq {
namespace {

constexpr int kThreads = 256;

struct KPArgs {
  kivi_packed c[KVQ_MAX_TENSORS];
  const uint16_t* k[KVQ_MAX_TENSORS];
  const uint16_t* v[KVQ_MAX_TENSORS];
  int n_layers, lo, hi;
  float eps, levels;
  // item decomposition without 64-bit divisions, when the per-layer item counts are < 2^31
  bool fast32;
  bool v8;                               // value tensors 32-byte aligned, head dim % 16 == 0
  DivU32 div_g, div_span, div_ngroups;   // by D / gs, hi - lo, (hi - lo) / gs
};

__device__ __forceinline__ __half2 as_h2(uint32_t w) { return *reinterpret_cast<__half2*>(&w); }
__device__ __forceinline__ uint32_t h2u(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }

// Group parameters as the pack uses them: zero, the stored fp16 scale and RN(1 / scale).
struct GP {
  float z, s, y;
  float t1, t2, t3;   // 2-bit fields: the thresholds of codes 1, 2, 3 on RN(x - zero)
};

__device__ __forceinline__ GP make_gp(float z, uint16_t s16) {
  GP g;
  g.z = z;
  g.s = h2f(s16);
  g.y = __frcp_rn(g.s);
  return g;
}

// The exact quotient, out of line: it runs only near ties.
__device__ __noinline__ float exact_quotient(float d, float s) { return __fdiv_rn(d, s); }

// Field of x: clamp(rint(RN(RN(x - zero) / scale)), 0, levels), 0 if the fp16 scale is 0.
// q0 = RN(d * RN(1 / s)) differs from RN(d / s) by less than 2^-22 * q0 (three roundings of
// relative size 2^-24; no overflow or underflow: s is an fp16 value >= 2^-24 and d an fp16
// difference).  Where q0 is farther than q0 * 2^-20 from the nearest half-integer both round to
// the same integer; elsewhere the IEEE quotient decides.
__device__ __forceinline__ uint32_t field(float x, const GP& g, float levels) {
  if (g.s == 0.f) return 0;
  const float d = __fsub_rn(x, g.z);
  float q = __fmul_rn(d, g.y);
  const float dist = fabsf(__fsub_rn(__fadd_rn(floorf(q), 0.5f), q));
  if (dist <= __fmul_rn(q, 9.5367431640625e-07f)) q = exact_quotient(d, g.s);  // 2^-20
  return static_cast<uint32_t>(fminf(fmaxf(rintf(q), 0.f), levels));
}

// 2-bit fields (levels = 3) as three compares.  With d = RN(x - zero) and q = RN(d / s), the code
// clamp(rint_half_even(q), 0, 3) is >= 1 iff q > 0.5, >= 2 iff q >= 1.5, >= 3 iff q > 2.5, i.e.
// (ties going to the even neighbour) iff the real quotient d / s exceeds 0.5 + 2^-25, reaches
// 1.5 - 2^-24, exceeds 2.5 + 2^-23.  None of s * (0.5 + 2^-25), s * (1.5 - 2^-24),
// s * (2.5 + 2^-23) is an fp32 value (the odd parts of the multipliers exceed 2^24), so each
// condition is d >= RU(s * m), and one fused multiply-add rounded upward gives RU(s * m) exactly
// from the exact power-of-two product s * 2^-k.  A zero scale gives code 0 everywhere.
__device__ __forceinline__ void set_thresholds3(GP& g) {
  if (g.s == 0.f) {
    g.t1 = g.t2 = g.t3 = __int_as_float(0x7f800000);
    return;
  }
  g.t1 = __fmaf_ru(g.s, 0.5f, g.s * 2.98023223876953125e-08f);      // s (0.5 + 2^-25)
  g.t2 = __fmaf_ru(g.s, 1.5f, -(g.s * 5.9604644775390625e-08f));    // s (1.5 - 2^-24)
  g.t3 = __fmaf_ru(g.s, 2.5f, g.s * 1.1920928955078125e-07f);       // s (2.5 + 2^-23)
}

// The code boundaries of two groups' 2-bit fields (fp16 compares replace three float compares).
__device__ __forceinline__ L3Cut gp_cut(const GP& a, const GP& b) {
  return l3_cut2(a.z, a.t1, a.t2, a.t3, b.z, b.t1, b.t2, b.t3);
}

// 8 fields of `bits` bits -> packed LSB-first (2 bits: 16 bits, 4 bits: 32 bits, 8: 64 bits).
template <int BITS>
__device__ __forceinline__ uint2 pack_fields8(const uint32_t f[8]) {
  uint32_t lo = 0, hi = 0;
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const int bit = e * BITS;
    if (bit < 32) lo |= f[e] << bit; else hi |= f[e] << (bit - 32);
  }
  return make_uint2(lo, hi);
}

template <int BITS>
__device__ __forceinline__ void store_fields8(uint8_t* p, const uint32_t f[8]) {
  const uint2 w = pack_fields8<BITS>(f);
  if constexpr (BITS == 2) *reinterpret_cast<uint16_t*>(p) = static_cast<uint16_t>(w.x);
  else if constexpr (BITS == 4) *reinterpret_cast<uint32_t*>(p) = w.x;
  else *reinterpret_cast<uint2*>(p) = w;
}

__device__ __forceinline__ void f8(const uint4& v, float f[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    f[2 * k] = h2f(static_cast<uint16_t>(w[k] & 0xffffu));
    f[2 * k + 1] = h2f(static_cast<uint16_t>(w[k] >> 16));
  }
}

__device__ __forceinline__ uint16_t scale16(float mn, float mx, float levels, float eps) {
  return f2h(fmaxf(__fdiv_rn(__fsub_rn(mx, mn), levels), eps));
}

template <int BITS>
__device__ void pack_keys_part(const KPArgs& a, int64_t first, int64_t stride) {
  const kivi_packed& c0 = a.c[0];
  const int B = c0.batch, H = c0.num_heads, S = c0.capacity, D = c0.head_dim, gs = c0.group_size;
  const int chunks = D / 8;
  const int n_groups = (a.hi - a.lo) / gs;
  const int64_t per_layer = static_cast<int64_t>(B) * H * n_groups * chunks;
  const int64_t items = per_layer * a.n_layers;
  const int cb = D * BITS / 8;  // code bytes per row
  for (int64_t it = first; it < items; it += stride) {
    const int layer = static_cast<int>(it / per_layer);
    int64_t r = it - layer * per_layer;
    const int ch = static_cast<int>(r % chunks);
    r /= chunks;
    const int g = static_cast<int>(r % n_groups);
    const int64_t bh = r / n_groups;
    const int t0 = a.lo + g * gs;
    const kivi_packed& C = a.c[layer];
    const uint4* src = reinterpret_cast<const uint4*>(a.k[layer] + (bh * S + t0) * D) + ch;
    const int row_v = D / 8;  // uint4 per row
    __half2 mn[4], mx[4];
    {
      const uint4 v0 = src[0];
      const uint32_t w0[4] = {v0.x, v0.y, v0.z, v0.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) mn[k] = mx[k] = as_h2(w0[k]);
    }
    for (int t = 1; t < gs; ++t) {
      const uint4 v = src[static_cast<int64_t>(t) * row_v];
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        mn[k] = __hmin2(mn[k], as_h2(w[k]));
        mx[k] = __hmax2(mx[k], as_h2(w[k]));
      }
    }
    GP gp[8];
    uint32_t sw[4], zw[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float z0 = __low2float(mn[k]), z1 = __high2float(mn[k]);
      const uint16_t s0 = scale16(z0, __low2float(mx[k]), a.levels, a.eps);
      const uint16_t s1 = scale16(z1, __high2float(mx[k]), a.levels, a.eps);
      gp[2 * k] = make_gp(z0, s0);
      gp[2 * k + 1] = make_gp(z1, s1);
      if constexpr (BITS == 2) {
        set_thresholds3(gp[2 * k]);
        set_thresholds3(gp[2 * k + 1]);
      }
      sw[k] = s0 | (static_cast<uint32_t>(s1) << 16);
      zw[k] = *reinterpret_cast<const uint32_t*>(&mn[k]);
    }
    const int64_t prow = (bh * (S / gs) + t0 / gs) * D + ch * 8;   // params [B][H][S/gs][D]
    *reinterpret_cast<uint4*>(C.k_scale + prow) = make_uint4(sw[0], sw[1], sw[2], sw[3]);
    *reinterpret_cast<uint4*>(C.k_zero + prow) = make_uint4(zw[0], zw[1], zw[2], zw[3]);
    uint8_t* dst = C.k_codes + (bh * S + t0) * cb + ch * BITS;     // 8 fields = BITS bytes
    if constexpr (BITS == 2) {
      L3Cut cut[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) cut[k] = gp_cut(gp[2 * k], gp[2 * k + 1]);
      for (int t = 0; t < gs; ++t) {
        const uint4 v = src[static_cast<int64_t>(t) * row_v];
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        *reinterpret_cast<uint16_t*>(dst + static_cast<int64_t>(t) * cb) =
            static_cast<uint16_t>(l3_codes8<4>(w, cut));
      }
    } else {
      for (int t = 0; t < gs; ++t) {
        float x[8];
        f8(src[static_cast<int64_t>(t) * row_v], x);
        uint32_t f[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) f[e] = field(x[e], gp[e], a.levels);
        store_fields8<BITS>(dst + static_cast<int64_t>(t) * cb, f);
      }
    }
  }
}

// Keys at head_dim 64: one warp per (layer, batch row, head, token group), every row read once.
// Lane l takes the 8-channel chunk l & 7 (16 bytes of a row) of the group's token quarter
// l >> 3 (GS / 4 rows) into registers; the per-channel fp16 min / max reduce over the quarter and
// then across the four quarters by shuffles, and each lane codes its own rows.  `first` and
// `stride` count warps, so the lanes of a warp always share an item.
template <int BITS, int GS>
__device__ void pack_keys_d64(const KPArgs& a, int64_t first, int64_t stride) {
  constexpr int kD64 = 64, kQ = GS / 4, kCb = kD64 * BITS / 8;
  const kivi_packed& c0 = a.c[0];
  const int B = c0.batch, H = c0.num_heads, S = c0.capacity;
  const int lane = threadIdx.x & 31, ch = lane & 7, tq = lane >> 3;
  const int n_groups = (a.hi - a.lo) / GS;
  const int64_t per_layer = static_cast<int64_t>(B) * H * n_groups;
  const int64_t items = per_layer * a.n_layers;
  // one item: (layer, batch row * H + head, token group)
  auto item = [&](int layer, int64_t bh, int g) {
    const int t0 = a.lo + g * GS;
    const kivi_packed& C = a.c[layer];
    const uint4* src =
        reinterpret_cast<const uint4*>(a.k[layer] + (bh * S + t0 + tq * kQ) * kD64) + ch;
    uint4 x[kQ];
#pragma unroll
    for (int i = 0; i < kQ; ++i) x[i] = src[i * (kD64 / 8)];
    uint32_t mn[4], mx[4];
    {
      const uint32_t w0[4] = {x[0].x, x[0].y, x[0].z, x[0].w};
#pragma unroll
      for (int k = 0; k < 4; ++k) mn[k] = mx[k] = w0[k];
    }
#pragma unroll
    for (int i = 1; i < kQ; ++i) {
      const uint32_t w[4] = {x[i].x, x[i].y, x[i].z, x[i].w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        mn[k] = h2u(__hmin2(as_h2(mn[k]), as_h2(w[k])));
        mx[k] = h2u(__hmax2(as_h2(mx[k]), as_h2(w[k])));
      }
    }
#pragma unroll
    for (int o = 8; o <= 16; o <<= 1) {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        mn[k] = h2u(__hmin2(as_h2(mn[k]), as_h2(__shfl_xor_sync(kFullMask, mn[k], o))));
        mx[k] = h2u(__hmax2(as_h2(mx[k]), as_h2(__shfl_xor_sync(kFullMask, mx[k], o))));
      }
    }
    // The four lanes of a chunk share its 8 channels' groups: lane tq derives the scales (and,
    // for 2 bits, the code boundaries) of channels 2 tq, 2 tq + 1 and the chunk's lanes exchange
    // them by shuffles.
    const uint32_t mn_w = tq == 0 ? mn[0] : tq == 1 ? mn[1] : tq == 2 ? mn[2] : mn[3];
    const uint32_t mx_w = tq == 0 ? mx[0] : tq == 1 ? mx[1] : tq == 2 ? mx[2] : mx[3];
    const float z0 = __low2float(as_h2(mn_w)), z1 = __high2float(as_h2(mn_w));
    const uint16_t s0 = scale16(z0, __low2float(as_h2(mx_w)), a.levels, a.eps);
    const uint16_t s1 = scale16(z1, __high2float(as_h2(mx_w)), a.levels, a.eps);
    uint32_t sw[4];
#pragma unroll
    for (int k = 0; k < 4; ++k)
      sw[k] = __shfl_sync(kFullMask, s0 | (static_cast<uint32_t>(s1) << 16), k * 8 + ch);
    if (tq == 0) {
      const int64_t prow = (bh * (S / GS) + t0 / GS) * kD64 + ch * 8;   // params [B][H][S/gs][D]
      *reinterpret_cast<uint4*>(C.k_scale + prow) = make_uint4(sw[0], sw[1], sw[2], sw[3]);
      *reinterpret_cast<uint4*>(C.k_zero + prow) = make_uint4(mn[0], mn[1], mn[2], mn[3]);
    }
    uint8_t* dst = C.k_codes + (bh * S + t0 + tq * kQ) * kCb + ch * BITS;   // 8 fields = BITS bytes
    if constexpr (BITS == 2) {
      GP g0 = make_gp(z0, s0), g1 = make_gp(z1, s1);
      set_thresholds3(g0);
      set_thresholds3(g1);
      const L3Cut mine = gp_cut(g0, g1);
      L3Cut cut[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        cut[k].x1 = __shfl_sync(kFullMask, mine.x1, k * 8 + ch);
        cut[k].x2 = __shfl_sync(kFullMask, mine.x2, k * 8 + ch);
        cut[k].x3 = __shfl_sync(kFullMask, mine.x3, k * 8 + ch);
      }
#pragma unroll
      for (int i = 0; i < kQ; ++i) {
        const uint32_t w[4] = {x[i].x, x[i].y, x[i].z, x[i].w};
        *reinterpret_cast<uint16_t*>(dst + static_cast<int64_t>(i) * kCb) =
            static_cast<uint16_t>(l3_codes8<4>(w, cut));
      }
    } else {
      GP gp[8];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        gp[2 * k] = make_gp(__low2float(as_h2(mn[k])), static_cast<uint16_t>(sw[k] & 0xffffu));
        gp[2 * k + 1] = make_gp(__high2float(as_h2(mn[k])), static_cast<uint16_t>(sw[k] >> 16));
      }
#pragma unroll
      for (int i = 0; i < kQ; ++i) {
        float xf[8];
        f8(x[i], xf);
        uint32_t f[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) f[e] = field(xf[e], gp[e], a.levels);
        store_fields8<BITS>(dst + static_cast<int64_t>(i) * kCb, f);
      }
    }
  };
  if (a.fast32) {   // running (layer, offset); offset / n_groups by multiply-high
    const uint32_t pl = static_cast<uint32_t>(per_layer);
    int layer = static_cast<int>(first / per_layer);
    uint32_t r = static_cast<uint32_t>(first - layer * per_layer);
    const int dl = static_cast<int>(stride / per_layer);
    const uint32_t dr = static_cast<uint32_t>(stride - dl * per_layer);
    for (int64_t it = first; it < items; it += stride) {
      const uint32_t bh = divu32(r, a.div_ngroups);
      item(layer, bh, static_cast<int>(r - bh * n_groups));
      r += dr;
      layer += dl;
      if (r >= pl) {
        r -= pl;
        ++layer;
      }
    }
  } else {
    for (int64_t it = first; it < items; it += stride) {
      const int layer = static_cast<int>(it / per_layer);
      const int64_t r = it - layer * per_layer;
      item(layer, r / n_groups, static_cast<int>(r % n_groups));
    }
  }
}

// One value item -- (layer, batch row * H + head, token, channel group) -- whose NV 16-byte
// vectors (the group's 8 NV channels) are already in registers: min / max, parameters, codes.
template <int BITS, int NV>
__device__ __forceinline__ void value_group(const KPArgs& a, int layer, int64_t bh, int t, int g,
                                            const uint4 (&vv)[NV]) {
  const kivi_packed& C = a.c[layer];
  const int S = C.capacity, D = C.head_dim, G = D / (8 * NV), cb = D * BITS / 8;
  __half2 mn = as_h2(vv[0].x), mx = mn;
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const uint32_t w[4] = {vv[k].x, vv[k].y, vv[k].z, vv[k].w};
#pragma unroll
    for (int j = 0; j < 4; ++j) { mn = __hmin2(mn, as_h2(w[j])); mx = __hmax2(mx, as_h2(w[j])); }
  }
  const float z = fminf(__low2float(mn), __high2float(mn));
  const uint16_t sb = scale16(z, fmaxf(__low2float(mx), __high2float(mx)), a.levels, a.eps);
  GP gp = make_gp(z, sb);
  if constexpr (BITS == 2) set_thresholds3(gp);
  const int64_t pidx = (bh * S + t) * G + g;                      // params [B][H][S][G]
  C.v_scale[pidx] = sb;
  C.v_zero[pidx] = f2h(z);
  uint8_t* dst = C.v_codes + (bh * S + t) * cb + g * NV * BITS;
  if constexpr (BITS == 2) {
    const L3Cut cut = l3_cut1(gp.z, gp.t1, gp.t2, gp.t3);
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      const uint32_t w[4] = {vv[k].x, vv[k].y, vv[k].z, vv[k].w};
      *reinterpret_cast<uint16_t*>(dst + k * BITS) = static_cast<uint16_t>(l3_codes8<1>(w, &cut));
    }
  } else {
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      float x[8];
      f8(vv[k], x);
      uint32_t f[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) f[e] = field(x[e], gp, a.levels);
      store_fields8<BITS>(dst + k * BITS, f);
    }
  }
}

// Values: one thread per item, groups of 8 NV channels.  The running loop loads the next item's
// vectors before it codes the current one, so every thread keeps a load in flight while it
// computes.
template <int BITS, int NV, bool V8>
__device__ void pack_values_part(const KPArgs& a, int64_t first, int64_t stride) {
  const kivi_packed& c0 = a.c[0];
  const int B = c0.batch, H = c0.num_heads, S = c0.capacity, D = c0.head_dim;
  const int G = D / (8 * NV);
  const int span = a.hi - a.lo;
  const int64_t per_layer = static_cast<int64_t>(B) * H * span * G;
  const int64_t items = per_layer * a.n_layers;
  auto load = [&](int layer, int64_t bh, int t, int g, uint4 (&vv)[NV]) {
    const uint4* src = reinterpret_cast<const uint4*>(a.v[layer] + (bh * S + t) * D) + g * NV;
    if constexpr (V8 && NV % 2 == 0) {   // 32-byte aligned: pairs of vectors in 256-bit loads
#pragma unroll
      for (int k = 0; k < NV; k += 2) ld_stream_v8(src + k, vv[k], vv[k + 1]);
    } else {
#pragma unroll
      for (int k = 0; k < NV; ++k) vv[k] = src[k];
    }
  };
  if (a.fast32) {   // running (layer, offset); offset / G and / span by multiply-high
    if (first >= items) return;
    const uint32_t pl = static_cast<uint32_t>(per_layer);
    int layer = static_cast<int>(first / per_layer);
    uint32_t r = static_cast<uint32_t>(first - layer * per_layer);
    const int dl = static_cast<int>(stride / per_layer);
    const uint32_t dr = static_cast<uint32_t>(stride - dl * per_layer);
    // position of the running item: (layer, bh, t, g)
    int cl = layer, ct, cg;
    uint32_t cbh;
    auto place = [&](uint32_t rr, uint32_t& bh, int& t, int& g) {
      const uint32_t q = divu32(rr, a.div_g);          // token row of the layer
      bh = divu32(q, a.div_span);
      t = a.lo + static_cast<int>(q - bh * span);
      g = static_cast<int>(rr - q * G);
    };
    place(r, cbh, ct, cg);
    uint4 cur[NV];
    load(cl, cbh, ct, cg, cur);
    for (int64_t it = first;; it += stride) {
      r += dr;
      layer += dl;
      if (r >= pl) {
        r -= pl;
        ++layer;
      }
      const bool more = it + stride < items;
      int nl = layer, nt = 0, ng = 0;
      uint32_t nbh = 0;
      uint4 nxt[NV];
      if (more) {
        place(r, nbh, nt, ng);
        load(nl, nbh, nt, ng, nxt);
      }
      value_group<BITS, NV>(a, cl, cbh, ct, cg, cur);
      if (!more) break;
      cl = nl; cbh = nbh; ct = nt; cg = ng;
#pragma unroll
      for (int k = 0; k < NV; ++k) cur[k] = nxt[k];
    }
  } else {
    for (int64_t it = first; it < items; it += stride) {
      const int layer = static_cast<int>(it / per_layer);
      int64_t r = it - layer * per_layer;
      const int g = static_cast<int>(r % G);
      r /= G;
      const int64_t bh = r / span;
      const int t = a.lo + static_cast<int>(r - bh * span);
      uint4 vv[NV];
      load(layer, bh, t, g, vv);
      value_group<BITS, NV>(a, layer, bh, t, g, vv);
    }
  }
}

// Keys and values in two launches, each with its own register allocation (the head_dim-64 key
// path holds a token quarter of its group in registers; the value path needs far fewer).  The
// head_dim-64 key kernel for groups of up to 32 tokens is built for 4 blocks per SM (64
// registers, 20 bytes spilled): 16-layer 2-bit pack 0.501 -> 0.494 ms against 3 blocks at 72.
template <int BITS, int GS>
__global__ void __launch_bounds__(kThreads, (GS > 0 && GS <= 32) ? 4 : 1)
    kivi_pack_keys_kernel(const KPArgs a) {
  if constexpr (GS > 0)   // head_dim 64: a warp per token group
    pack_keys_d64<BITS, GS>(a, (static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x) >> 5,
                            static_cast<int64_t>(gridDim.x) * (kThreads / 32));
  else
    pack_keys_part<BITS>(a, static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x,
                         static_cast<int64_t>(gridDim.x) * kThreads);
}

template <int BITS, int NV, bool V8>
__global__ void __launch_bounds__(kThreads) kivi_pack_values_kernel(const KPArgs a) {
  pack_values_part<BITS, NV, V8>(a, static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x,
                                 static_cast<int64_t>(gridDim.x) * kThreads);
}

// ================================================================================================
// Decode attention, head_dim 64.
constexpr int kAD = 64;
constexpr int kAWarps = 4;
constexpr int kAThreads = kAWarps * 32;
constexpr int kATile = 16;
constexpr int kChunk = 64;            // tokens per stage: four tiles
constexpr int kAStages = 3;           // stages per warp
constexpr int kARec = kAD + 4;        // workspace record: O[64], m, l, pad, pad
// stage layout (bytes): K codes | V codes | K scale | K zero | V scale | V zero
constexpr int kOffVC = kChunk * 16, kOffKS = 2 * kChunk * 16, kOffKZ = kOffKS + 512;
constexpr int kOffVS = kOffKZ + 512, kOffVZ = kOffVS + 512;
constexpr int kStageBytes = kOffVZ + 512;
constexpr int kAttnSmem = kAWarps * kAStages * kStageBytes + kAWarps * kAStages * 8;
#define kNegInfF (-__int_as_float(0x7f800000))
#define kMaxFloorF (-1e30f)   // floor of the running max; a max still at it saw no valid token

struct KAArgs {
  kivi_packed c[KVQ_MAX_TENSORS];
  const uint16_t* k[KVQ_MAX_TENSORS];
  const uint16_t* v[KVQ_MAX_TENSORS];
  const uint16_t* q;
  float* out;
  float* ws;
  int32_t* err;
  int n_layers, B, H, G, Hq, S, n_packed, offset, n_splits, tiles_per_cta;
  float qk_scale;
};

// Shared-memory loads at 32-bit shared-window addresses (no generic-address arithmetic).
__device__ __forceinline__ uint32_t lds_u32(uint32_t a) {
  uint32_t r;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(r) : "r"(a));
  return r;
}
__device__ __forceinline__ uint32_t lds_u16(uint32_t a) {
  uint16_t r;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(r) : "r"(a));
  return r;
}
__device__ __forceinline__ uint4 lds_v4(uint32_t a) {
  uint4 r;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "r"(a));
  return r;
}

// Exact fp16 codes {e_k, e_(k + 8)} of a word of sixteen 2-bit fields, k = 0..7 (the callers
// unroll k).  Fields 0-4 of each half already sit at mantissa bits 2k, 2k + 1 of fp16 1024, where
// they read as 1024 + 4^k u, so one fp16 FMA with scale 4^-k and offset -1024 * 4^-k gives u
// exactly; fields 5-7 are read the same way from w10 = w >> 10 (one shift per word).
__device__ __forceinline__ uint32_t code_pair2(uint32_t w, uint32_t w10, int k) {
  constexpr uint32_t kScale[5] = {0x3C003C00u, 0x34003400u, 0x2C002C00u, 0x24002400u,
                                  0x1C001C00u};   // 1, 1/4, 1/16, 1/64, 1/256
  constexpr uint32_t kOff[5] = {0xE400E400u, 0xDC00DC00u, 0xD400D400u, 0xCC00CC00u,
                                0xC400C400u};     // -1024, -256, -64, -16, -4
  const int j = k < 5 ? k : k - 5;
  const uint32_t src = k < 5 ? w : w10;
  return hfma2u((src & (0x00030003u << (2 * j))) | 0x64006400u, kScale[j], kOff[j]);
}

// One CTA: split `blockIdx.x` of KV head blockIdx.y of (layer, batch row) blockIdx.z, four warps.
// The CTA's tiles are cut into 64-token chunks dealt round-robin to the warps; each warp streams
// the packed bytes of its chunks through a private ring of kAStages shared-memory stages
// (cp.async.bulk completing on an mbarrier, bounded waits).  Tiles at or beyond n_packed read the
// fp16 residual cache with plain loads.
//
// Per thread and tile: K codes of rows g, g+8 for head-dim elements [16c, 16c + 16) (one word per
// row; pairs {e_k, e_k+8} drive the k-steps and the Q fragments use the same element order), V
// codes of tokens 2c, 2c+1, 2c+8, 2c+9 for elements [8g, 8g + 8) (one half-word per token, two
// tokens paired in one word so the V operand needs no re-pairing).  A field placed in the
// mantissa of fp16 1024 becomes an exact fp16 code with one half2 FMA, and one more half2 FMA
// applies the group's scale and zero (c * scale + zero, one rounding).
__global__ void __launch_bounds__(kAThreads, 4) kivi_attn_kernel(const KAArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  const int split = blockIdx.x, h = blockIdx.y, lb = blockIdx.z;
  const int layer = lb / a.B, b = lb - layer * a.B;
  const kivi_packed& C = a.c[layer];
  const int S = a.S, gs = C.group_size, G = kAD / gs;
  const int gsh = __ffs(gs) - 1;   // group sizes are powers of two: divisions by gs are shifts
  const int64_t bh = static_cast<int64_t>(b) * a.H + h;
  const int n_tiles = (a.offset + kATile - 1) / kATile;
  const int tile0 = split * a.tiles_per_cta;
  const int tile1 = min(n_tiles, tile0 + a.tiles_per_cta);
  const int n_chunks = (tile1 - tile0 + 3) / 4;
  const int n_mine = n_chunks > warp ? (n_chunks - warp + kAWarps - 1) / kAWarps : 0;

  uint8_t* wbase = smem + warp * kAStages * kStageBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kAWarps * kAStages * kStageBytes) +
                   warp * kAStages;
  if (lane == 0) {
    for (int i = 0; i < kAStages; ++i) mbar_init(&bars[i], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncwarp();

  const uint8_t* kc = C.k_codes + bh * S * 16;    // 16 bytes per row at D = 64, 2 bits
  const uint8_t* vc = C.v_codes + bh * S * 16;
  const uint16_t* ksc = C.k_scale + bh * (S / gs) * kAD;
  const uint16_t* kze = C.k_zero + bh * (S / gs) * kAD;
  const uint16_t* vsc = C.v_scale + bh * S * G;
  const uint16_t* vze = C.v_zero + bh * S * G;

  // Copy the packed tokens of this warp's j-th chunk into stage j % kAStages (lane 0 only);
  // a chunk with no packed token completes its phase with a plain arrive.
  auto issue = [&](int j) {
    const int st = j % kAStages;
    const int t0 = (tile0 + 4 * (warp + j * kAWarps)) * kATile;
    const int cnt = min(kChunk, max(0, a.n_packed - t0));   // a multiple of gs (and of 16)
    uint8_t* dst = wbase + st * kStageBytes;
    if (cnt > 0) {
      const uint32_t code = cnt * 16, kpar = (cnt >> gsh) * kAD * 2, vpar = cnt * G * 2;
      mbar_expect_tx(&bars[st], 2 * code + 2 * kpar + 2 * vpar);
      bulk_g2s(dst, kc + static_cast<int64_t>(t0) * 16, code, &bars[st]);
      bulk_g2s(dst + kOffVC, vc + static_cast<int64_t>(t0) * 16, code, &bars[st]);
      bulk_g2s(dst + kOffKS, ksc + (t0 >> gsh) * kAD, kpar, &bars[st]);
      bulk_g2s(dst + kOffKZ, kze + (t0 >> gsh) * kAD, kpar, &bars[st]);
      bulk_g2s(dst + kOffVS, vsc + static_cast<int64_t>(t0) * G, vpar, &bars[st]);
      bulk_g2s(dst + kOffVZ, vze + static_cast<int64_t>(t0) * G, vpar, &bars[st]);
    } else {
      mbar_arrive(&bars[st]);
    }
  };
  if (lane == 0)
    for (int j = 0; j < kAStages && j < n_mine; ++j) issue(j);

  // Q^T fragments: k-step ks uses elements 16c + 2ks + {0, 8} (b0) and 16c + 2ks + {1, 9} (b1)
  uint32_t qf[4][2];
  {
    uint32_t qw[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    if (g < a.G) {
      const uint16_t* qp = a.q + (static_cast<int64_t>(lb) * a.Hq + h * a.G + g) * kAD + 16 * c;
      const uint4 x0 = ld_nc_v4(qp), x1 = ld_nc_v4(qp + 8);
      qw[0] = x0.x; qw[1] = x0.y; qw[2] = x0.z; qw[3] = x0.w;
      qw[4] = x1.x; qw[5] = x1.y; qw[6] = x1.z; qw[7] = x1.w;
    }
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
      qf[ks][0] = prmt(qw[ks], qw[ks + 4], 0x5410u);   // low halves: e_2ks, e_2ks+8
      qf[ks][1] = prmt(qw[ks], qw[ks + 4], 0x7632u);   // high halves: e_2ks+1, e_2ks+9
    }
  }

  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int k = 0; k < 4; ++k) acc[i][k] = 0.f;
  float m0 = kNegInfF, m1 = kNegInfF, l0 = 0.f, l1 = 0.f;

  const uint16_t* kres = a.k[layer] + bh * S * kAD;
  const uint16_t* vres = a.v[layer] + bh * S * kAD;
  int kgroup = -1;
  uint32_t ks2[8], kz2[8];   // scale / zero pairs for the thread's K elements {e_k, e_k+8}
  bool timed_out = false;
  int issued = n_mine < kAStages ? n_mine : kAStages;

  for (int j = 0; j < n_mine; ++j) {
    const int st = j % kAStages;
    const bool arrived = mbar_wait_stage(&bars[st], static_cast<uint32_t>((j / kAStages) & 1));
    if (__any_sync(kFullMask, !arrived)) {   // warp-uniform exit
      timed_out = true;
      break;
    }
    const uint32_t sb = smem_u32(wbase + st * kStageBytes);   // the stage, shared window
    const int ctile = tile0 + 4 * (warp + j * kAWarps);
    const int t0 = ctile * kATile;
#pragma unroll 1
    for (int i = 0; i < 4; ++i) {
      if (ctile + i >= tile1) break;   // warp-uniform
      const int tb = t0 + i * kATile, lt = i * kATile;
      const bool packed = tb < a.n_packed;   // tiles never straddle (n_packed % 16 == 0)
      // ---------------- K fragments (rows g, g + 8)
      uint32_t kf[2][8];   // pairs {e_k, e_k+8}, k = 0..7
      bool kval[2];
#pragma unroll
      for (int r = 0; r < 2; ++r) kval[r] = tb + g + 8 * r < a.offset;
      if (packed) {
        const int grp = tb >> gsh;
        if (grp != kgroup) {   // group parameters of the thread's 16 channels (warp-uniform)
          kgroup = grp;
          const uint32_t sp = sb + kOffKS + ((tb - t0) >> gsh) * (kAD * 2) + 32 * c;
          const uint4 s0 = lds_v4(sp);
          const uint4 s1 = lds_v4(sp + 16);
          const uint4 z0 = lds_v4(sp + (kOffKZ - kOffKS));
          const uint4 z1 = lds_v4(sp + (kOffKZ - kOffKS) + 16);
          const uint32_t sw[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
          const uint32_t zw[8] = {z0.x, z0.y, z0.z, z0.w, z1.x, z1.y, z1.z, z1.w};
#pragma unroll
          for (int k = 0; k < 8; ++k) {   // element k is half (k & 1) of word k >> 1
            const uint32_t sel = (k & 1) ? 0x7632u : 0x5410u;
            ks2[k] = prmt(sw[k >> 1], sw[(k >> 1) + 4], sel);
            kz2[k] = prmt(zw[k >> 1], zw[(k >> 1) + 4], sel);
          }
        }
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          const uint32_t w = lds_u32(sb + (lt + g + 8 * r) * 16 + 4 * c);
          const uint32_t w10 = w >> 10;
#pragma unroll
          for (int k = 0; k < 8; ++k) kf[r][k] = hfma2u(code_pair2(w, w10, k), ks2[k], kz2[k]);
        }
      } else {
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          uint32_t hw[8] = {0, 0, 0, 0, 0, 0, 0, 0};
          if (kval[r]) {
            const uint16_t* rp = kres + static_cast<int64_t>(tb + g + 8 * r) * kAD + 16 * c;
            const uint4 x0 = *reinterpret_cast<const uint4*>(rp);
            const uint4 x1 = *reinterpret_cast<const uint4*>(rp + 8);
            hw[0] = x0.x; hw[1] = x0.y; hw[2] = x0.z; hw[3] = x0.w;
            hw[4] = x1.x; hw[5] = x1.y; hw[6] = x1.z; hw[7] = x1.w;
          }
#pragma unroll
          for (int k = 0; k < 8; ++k)
            kf[r][k] = prmt(hw[k >> 1], hw[(k >> 1) + 4], (k & 1) ? 0x7632u : 0x5410u);
        }
      }
      // ---------------- S^T = K_hat . Q^T ; k-step ks: A cols {2c,2c+1} = {e_2ks, e_2ks+8},
      // {2c+8, 2c+9} = {e_2ks+1, e_2ks+9}
      float sacc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        mma16816(sacc, kf[0][2 * ks], kf[1][2 * ks], kf[0][2 * ks + 1], kf[1][2 * ks + 1],
                 qf[ks][0], qf[ks][1]);
      float sc[4];
      sc[0] = kval[0] ? sacc[0] * a.qk_scale : kNegInfF;
      sc[1] = kval[0] ? sacc[1] * a.qk_scale : kNegInfF;
      sc[2] = kval[1] ? sacc[2] * a.qk_scale : kNegInfF;
      sc[3] = kval[1] ? sacc[3] * a.qk_scale : kNegInfF;
      float tm0 = fmaxf(sc[0], sc[2]), tm1 = fmaxf(sc[1], sc[3]);
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        tm0 = fmaxf(tm0, __shfl_xor_sync(kFullMask, tm0, o));
        tm1 = fmaxf(tm1, __shfl_xor_sync(kFullMask, tm1, o));
      }
      // a running max held above a finite floor: no exponential needs a -inf guard (0.285 ->
      // 0.281 ms at the 16-layer shape)
      const float n0 = fmaxf(fmaxf(m0, tm0), kMaxFloorF), n1 = fmaxf(fmaxf(m1, tm1), kMaxFloorF);
      const float al0 = ex2_fast(m0 - n0);
      const float al1 = ex2_fast(m1 - n1);
      float p[4];
      p[0] = ex2_fast(sc[0] - n0);
      p[2] = ex2_fast(sc[2] - n0);
      p[1] = ex2_fast(sc[1] - n1);
      p[3] = ex2_fast(sc[3] - n1);
      l0 = l0 * al0 + (p[0] + p[2]);
      l1 = l1 * al1 + (p[1] + p[3]);
      m0 = n0;
      m1 = n1;
      if (__any_sync(kFullMask, al0 != 1.f || al1 != 1.f)) {
#pragma unroll
        for (int mt = 0; mt < 4; ++mt) {
          acc[mt][0] *= al0; acc[mt][1] *= al1; acc[mt][2] *= al0; acc[mt][3] *= al1;
        }
      }
      const uint32_t pb0 = movtrans(pack_h2(p[0], p[1]));
      const uint32_t pb1 = movtrans(pack_h2(p[2], p[3]));
      // ---------------- V^T fragments: tokens (2c, 2c+1) and (2c+8, 2c+9), elements 8g + j
      uint32_t vf[2][8];   // [token pair][element j]: {A.e_j, B.e_j}
      if (packed) {
        const int gi = (8 * g) >> gsh;
#pragma unroll
        for (int pr = 0; pr < 2; ++pr) {
          const int ta = lt + 2 * c + 8 * pr;   // local token of A; B = A + 1 (all packed)
          const uint32_t w = lds_u16(sb + kOffVC + ta * 16 + 2 * g) |
                             (lds_u16(sb + kOffVC + (ta + 1) * 16 + 2 * g) << 16);
          const uint32_t s2 = lds_u16(sb + kOffVS + (ta * G + gi) * 2) |
                              (lds_u16(sb + kOffVS + ((ta + 1) * G + gi) * 2) << 16);
          const uint32_t z2 = lds_u16(sb + kOffVZ + (ta * G + gi) * 2) |
                              (lds_u16(sb + kOffVZ + ((ta + 1) * G + gi) * 2) << 16);
          const uint32_t w10 = w >> 10;
#pragma unroll
          for (int jj = 0; jj < 8; ++jj) vf[pr][jj] = hfma2u(code_pair2(w, w10, jj), s2, z2);
        }
      } else {
#pragma unroll
        for (int pr = 0; pr < 2; ++pr) {
          const int ta = tb + 2 * c + 8 * pr, tbb = ta + 1;
          uint4 xa = make_uint4(0, 0, 0, 0), xb = make_uint4(0, 0, 0, 0);
          if (ta < a.offset)
            xa = *reinterpret_cast<const uint4*>(vres + static_cast<int64_t>(ta) * kAD + 8 * g);
          if (tbb < a.offset)
            xb = *reinterpret_cast<const uint4*>(vres + static_cast<int64_t>(tbb) * kAD + 8 * g);
          const uint32_t wa[4] = {xa.x, xa.y, xa.z, xa.w}, wb[4] = {xb.x, xb.y, xb.z, xb.w};
#pragma unroll
          for (int jj = 0; jj < 8; ++jj)
            vf[pr][jj] = prmt(wa[jj >> 1], wb[jj >> 1], (jj & 1) ? 0x7632u : 0x5410u);
        }
      }
      // O^T += V_hat^T . P^T ; m-tile mt rows g -> element 8g + 2mt, g + 8 -> element 8g + 2mt + 1
#pragma unroll
      for (int mt = 0; mt < 4; ++mt)
        mma16816(acc[mt], vf[0][2 * mt], vf[0][2 * mt + 1], vf[1][2 * mt], vf[1][2 * mt + 1],
                 pb0, pb1);
    }
    // the stage is consumed: hand it back to the copy engine
    __syncwarp();
    if (lane == 0 && j + kAStages < n_mine) {
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      issue(j + kAStages);
      ++issued;
    }
  }

  if (timed_out) {
    // drain the copies still in flight (bounded) before the shared memory is reused: the phases
    // of one stage complete in order, so its last issued phase is the one to wait for
    if (lane == 0) {
      report(a.err, KVQ_DEVERR_TIMEOUT);
      for (int j = issued - kAStages > 0 ? issued - kAStages : 0; j < issued; ++j)
        mbar_wait_bounded(&bars[j % kAStages], static_cast<uint32_t>((j / kAStages) & 1));
    }
    m0 = m1 = kNegInfF;
    l0 = l1 = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int k = 0; k < 4; ++k) acc[i][k] = 0.f;
  }

  // ---------------- merge the warps, write the split's partial record
  if (m0 == kMaxFloorF) m0 = kNegInfF;   // no valid token: an empty partial for the merges
  if (m1 == kMaxFloorF) m1 = kNegInfF;
#pragma unroll
  for (int o = 4; o < 32; o <<= 1) {
    l0 += __shfl_xor_sync(kFullMask, l0, o);
    l1 += __shfl_xor_sync(kFullMask, l1, o);
  }
  __syncthreads();   // every warp is done with its stages: reuse them for the merge
  float (*sm_o)[8][kAD] = reinterpret_cast<float (*)[8][kAD]>(smem);
  float (*sm_m)[8] = reinterpret_cast<float (*)[8]>(smem + kAWarps * 8 * kAD * 4);
  float (*sm_l)[8] = reinterpret_cast<float (*)[8]>(smem + kAWarps * 8 * kAD * 4 + kAWarps * 32);
  if (g == 0) {
    sm_m[warp][2 * c] = m0; sm_m[warp][2 * c + 1] = m1;
    sm_l[warp][2 * c] = l0; sm_l[warp][2 * c + 1] = l1;
  }
  // slot of (head j, d) in a warp's [8][64] block: the low three bits of d XOR-ed by
  // (d >> 5) | (j >> 1) << 1, so the 32 lanes of each store (heads 2c or 2c + 1, d = 8 g + ...)
  // fall in 32 different banks
  auto slot = [](int j, int d) { return j * kAD + (d ^ ((d >> 5) | ((j >> 1) << 1))); };
  float* wo = &sm_o[warp][0][0];
#pragma unroll
  for (int mt = 0; mt < 4; ++mt) {
    const int d = 8 * g + 2 * mt;
    wo[slot(2 * c, d)] = acc[mt][0];
    wo[slot(2 * c + 1, d)] = acc[mt][1];
    wo[slot(2 * c, d + 1)] = acc[mt][2];
    wo[slot(2 * c + 1, d + 1)] = acc[mt][3];
  }
  __syncthreads();
  float* rec = a.ws + ((static_cast<int64_t>(lb) * a.H + h) * a.n_splits + split) * 8 * kARec;
  // the warps' weights exp2(m_w - M) of a head, computed once when its first element comes up
  int jc = -1;
  float f[kAWarps], M = kNegInfF;
  for (int i = threadIdx.x; i < a.G * kAD; i += kAThreads) {
    const int jh = i / kAD, d = i - jh * kAD;
    if (jh != jc) {
      jc = jh;
      M = kNegInfF;
#pragma unroll
      for (int w = 0; w < kAWarps; ++w) M = fmaxf(M, sm_m[w][jh]);
#pragma unroll
      for (int w = 0; w < kAWarps; ++w)
        f[w] = (sm_m[w][jh] == kNegInfF) ? 0.f : exp2f(sm_m[w][jh] - M);
    }
    float O = 0.f;
#pragma unroll
    for (int w = 0; w < kAWarps; ++w) O += (&sm_o[w][0][0])[slot(jh, d)] * f[w];
    rec[jh * kARec + d] = O;
    if (d == 0) {
      float Lsum = 0.f;
#pragma unroll
      for (int w = 0; w < kAWarps; ++w) Lsum += sm_l[w][jh] * f[w];
      rec[jh * kARec + kAD] = M;
      rec[jh * kARec + kAD + 1] = Lsum;
    }
  }
}

__global__ void __launch_bounds__(kAD) kivi_attn_merge_kernel(const KAArgs a) {
  const int j = blockIdx.x, lb = blockIdx.y;
  const int h = j / a.G, jj = j - h * a.G;
  const int d = threadIdx.x;
  const float* base = a.ws + ((static_cast<int64_t>(lb) * a.H + h) * a.n_splits) * 8 * kARec +
                      jj * kARec;
  float M = kNegInfF;
  for (int sp = 0; sp < a.n_splits; ++sp) M = fmaxf(M, base[sp * 8 * kARec + kAD]);
  float O = 0.f, L = 0.f;
  if (M != kNegInfF) {
    for (int sp = 0; sp < a.n_splits; ++sp) {
      const float* r = base + sp * 8 * kARec;
      if (r[kAD] == kNegInfF) continue;
      const float f = exp2f(r[kAD] - M);
      O += r[d] * f;
      L += r[kAD + 1] * f;
    }
  }
  a.out[(static_cast<int64_t>(lb) * a.Hq + j) * kAD + d] = (L > 0.f) ? O / L : 0.f;
}

// Tiles per CTA (a multiple of 16: four 64-token chunks, one per warp at least).  The number of
// splits per (layer, batch row, KV head), up to 16, minimises the estimated time: whole waves of
// resident CTAs (4 per SM) times the chunks per warp plus a fixed cost of about 1.5 chunks per CTA
// (ring fill, Q load, the partial record); fewer splits win ties.
int attn_tiles_per_cta(int n_layers, int B, int H, int offset) {
  const int tiles = (offset + kATile - 1) / kATile;
  const int chunks = (tiles + 3) / 4;
  const int sms = sm_count() > 0 ? sm_count() : 152;
  const double cap = 4.0 * sms;
  const double units = static_cast<double>(n_layers) * B * H;
  int best_cpc = 4;
  double best_t = 0.0;
  for (int s = 1; s <= 16; ++s) {
    int cpc = (chunks + s - 1) / s;
    cpc = ((cpc + kAWarps - 1) / kAWarps) * kAWarps;
    if (cpc < kAWarps) cpc = kAWarps;
    const int splits = chunks > 0 ? (chunks + cpc - 1) / cpc : 1;
    const double t = std::ceil(units * splits / cap) * (cpc / kAWarps + 1.5);
    if (s == 1 || t < best_t) {
      best_t = t;
      best_cpc = cpc;
    }
  }
  return best_cpc * 4;
}

kvq_status check_caches(const kivi_packed* c, int n, const char* fn) {
  if (!c) return fail(KVQ_ERR_NULL, "%s: cache array is NULL", fn);
  if (n < 1 || n > KVQ_MAX_TENSORS)
    return fail(KVQ_ERR_RANGE, "%s: n_layers %d not in [1, %d]", fn, n, KVQ_MAX_TENSORS);
  for (int i = 0; i < n; ++i) {
    const kivi_packed& p = c[i];
    if (p.bits != 2 && p.bits != 4 && p.bits != 8)
      return fail(KVQ_ERR_BITS, "%s: bits %d not in {2, 4, 8}", fn, p.bits);
    if (p.group_size != 8 && p.group_size != 16 && p.group_size != 32 && p.group_size != 64)
      return fail(KVQ_ERR_SHAPE, "%s: group_size %d not in {8, 16, 32, 64}", fn, p.group_size);
    if (p.head_dim < 8 || p.head_dim > 256 || p.head_dim % p.group_size || p.head_dim % 8)
      return fail(KVQ_ERR_SHAPE, "%s: head_dim %d must be a multiple of group_size, <= 256", fn,
                  p.head_dim);
    if (p.batch < 1 || p.num_heads < 1 || p.capacity < 1 || p.capacity % p.group_size)
      return fail(KVQ_ERR_RANGE, "%s: bad batch/heads/capacity (capacity a multiple of "
                  "group_size)", fn);
    if (!p.k_codes || !p.k_scale || !p.k_zero || !p.v_codes || !p.v_scale || !p.v_zero)
      return fail(KVQ_ERR_NULL, "%s: cache %d has a NULL array", fn, i);
    if (!aligned16(p.k_codes) || !aligned16(p.k_scale) || !aligned16(p.k_zero) ||
        !aligned16(p.v_codes) || !aligned16(p.v_scale) || !aligned16(p.v_zero))
      return fail(KVQ_ERR_ALIGN, "%s: cache %d arrays must be 16-byte aligned", fn, i);
    if (p.bits != c[0].bits || p.group_size != c[0].group_size || p.batch != c[0].batch ||
        p.num_heads != c[0].num_heads || p.capacity != c[0].capacity ||
        p.head_dim != c[0].head_dim)
      return fail(KVQ_ERR_SHAPE, "%s: cache %d differs from cache 0", fn, i);
  }
  return KVQ_OK;
}

}  // namespace
}  // namespace kvq

namespace kvq {
namespace {
// At most the blocks resident on the SMs at once (the kernels loop over their items), so no block
// waits for a second wave; `cache` holds the kernel's resident blocks per SM.
template <typename K>
int resident_grid(K kernel, int& cache, int64_t threads) {
  if (cache == 0) {
    int b = 0;
    const cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, kernel, kThreads, 0);
    cache = (e != cudaSuccess || b < 1) ? 1 : b;
  }
  const int sms = sm_count() > 0 ? sm_count() : 152;
  const int64_t need = (threads + kThreads - 1) / kThreads;
  const int64_t cap = static_cast<int64_t>(sms) * cache;
  return static_cast<int>(need > cap ? cap : (need < 1 ? 1 : need));
}

template <int BITS, int GS>
void launch_keys(const KPArgs& a, int64_t threads, cudaStream_t cs) {
  static int cache = 0;
  const int grid = resident_grid(kivi_pack_keys_kernel<BITS, GS>, cache, threads);
  kivi_pack_keys_kernel<BITS, GS><<<grid, kThreads, 0, cs>>>(a);
}

template <int BITS, int NV, bool V8>
void launch_values_w(const KPArgs& a, int64_t threads, cudaStream_t cs) {
  static int cache = 0;
  const int grid = resident_grid(kivi_pack_values_kernel<BITS, NV, V8>, cache, threads);
  kivi_pack_values_kernel<BITS, NV, V8><<<grid, kThreads, 0, cs>>>(a);
}

// Value groups of 16 or more channels load their fp16 vectors in pairs (256-bit accesses) when
// every value tensor is 32-byte aligned and the head dim a multiple of 16.
template <int BITS, int NV>
void launch_values(const KPArgs& a, int64_t threads, cudaStream_t cs) {
  if (NV % 2 == 0 && a.v8) launch_values_w<BITS, NV, true>(a, threads, cs);
  else launch_values_w<BITS, NV, false>(a, threads, cs);
}

template <int BITS>
void launch_pack(const KPArgs& a, int key_gs, int gs, int64_t key_threads, int64_t value_threads,
                 cudaStream_t cs) {
  switch (key_gs) {   // 0: any head_dim (a thread per key chunk); else head_dim 64, group gs
    case 8: launch_keys<BITS, 8>(a, key_threads, cs); break;
    case 16: launch_keys<BITS, 16>(a, key_threads, cs); break;
    case 32: launch_keys<BITS, 32>(a, key_threads, cs); break;
    case 64: launch_keys<BITS, 64>(a, key_threads, cs); break;
    default: launch_keys<BITS, 0>(a, key_threads, cs); break;
  }
  switch (gs) {   // value groups of gs channels: gs / 8 vectors
    case 8: launch_values<BITS, 1>(a, value_threads, cs); break;
    case 16: launch_values<BITS, 2>(a, value_threads, cs); break;
    case 32: launch_values<BITS, 4>(a, value_threads, cs); break;
    default: launch_values<BITS, 8>(a, value_threads, cs); break;
  }
}
}  // namespace
}  // namespace kvq

extern "C" kvq_status kivi_pack(const kivi_packed* caches, const uint16_t* const* k,
                                const uint16_t* const* v, int n_layers, int lo, int hi,
                                float eps, kvq_stream_t stream) {
  using namespace kvq;
  const char* fn = "kivi_pack";
  kvq_status st = check_caches(caches, n_layers, fn);
  if (st != KVQ_OK) return st;
  const kivi_packed& c0 = caches[0];
  if (lo < 0 || hi < lo || hi > c0.capacity || lo % c0.group_size || hi % c0.group_size)
    return fail(KVQ_ERR_SHAPE, "%s: need 0 <= lo <= hi <= capacity, both multiples of "
                "group_size (lo %d hi %d)", fn, lo, hi);
  if (!(eps >= 0.f)) return fail(KVQ_ERR_RANGE, "%s: eps must be >= 0", fn);
  if (!k || !v) return fail(KVQ_ERR_NULL, "%s: NULL tensor array", fn);
  for (int i = 0; i < n_layers; ++i) {
    if (!k[i] || !v[i]) return fail(KVQ_ERR_NULL, "%s: tensor of layer %d is NULL", fn, i);
    if (!aligned16(k[i]) || !aligned16(v[i]))
      return fail(KVQ_ERR_ALIGN, "%s: tensors must be 16-byte aligned", fn);
  }
  if (hi == lo) return ok();
  KPArgs a;
  for (int i = 0; i < KVQ_MAX_TENSORS; ++i) {
    a.c[i] = caches[i < n_layers ? i : 0];
    a.k[i] = i < n_layers ? k[i] : nullptr;
    a.v[i] = i < n_layers ? v[i] : nullptr;
  }
  a.n_layers = n_layers;
  a.lo = lo;
  a.hi = hi;
  a.eps = eps;
  a.levels = static_cast<float>((1 << c0.bits) - 1);
  a.v8 = c0.head_dim % 16 == 0;
  for (int i = 0; i < n_layers; ++i)
    if (reinterpret_cast<uintptr_t>(v[i]) % 32) a.v8 = false;
  {
    const int64_t span = hi - lo, G = c0.head_dim / c0.group_size;
    const int64_t bhc = static_cast<int64_t>(c0.batch) * c0.num_heads;
    a.fast32 = bhc * span * G < (1LL << 31) && bhc * (span / c0.group_size) < (1LL << 31);
    a.div_g = make_divu32(static_cast<uint32_t>(G));
    a.div_span = make_divu32(static_cast<uint32_t>(span));
    a.div_ngroups = make_divu32(static_cast<uint32_t>(span / c0.group_size));
  }
  // keys: a thread per (group, 8-channel chunk), or at head_dim 64 a warp per group
  const bool d64 = c0.head_dim == 64;
  const int64_t kitems = static_cast<int64_t>(n_layers) * c0.batch * c0.num_heads *
                         ((hi - lo) / c0.group_size) * (d64 ? 32 : c0.head_dim / 8);
  const int64_t vitems = static_cast<int64_t>(n_layers) * c0.batch * c0.num_heads * (hi - lo) *
                         (c0.head_dim / c0.group_size);
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  const int kgs = d64 ? c0.group_size : 0;
  switch (c0.bits) {
    case 2: launch_pack<2>(a, kgs, c0.group_size, kitems, vitems, cs); break;
    case 4: launch_pack<4>(a, kgs, c0.group_size, kitems, vitems, cs); break;
    default: launch_pack<8>(a, kgs, c0.group_size, kitems, vitems, cs); break;
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(KVQ_ERR_CUDA, "%s launch: %s", fn, cudaGetErrorString(e));
  return ok();
}

extern "C" size_t kivi_decode_attn_workspace(int n_layers, int batch, int num_heads,
                                             int num_q_heads, int head_dim, int offset) {
  (void)num_q_heads; (void)head_dim;
  if (n_layers < 1 || batch < 1 || num_heads < 1 || offset < 0) return 0;
  const int tpc = kvq::attn_tiles_per_cta(n_layers, batch, num_heads, offset);
  const int tiles = (offset + kvq::kATile - 1) / kvq::kATile;
  const int n_splits = tiles > 0 ? (tiles + tpc - 1) / tpc : 1;
  return static_cast<size_t>(n_layers) * batch * num_heads * n_splits * 8 * kvq::kARec *
         sizeof(float);
}

extern "C" kvq_status kivi_decode_attn(const kivi_packed* caches, const uint16_t* const* k,
                                       const uint16_t* const* v, int n_layers, const uint16_t* q,
                                       int num_q_heads, int n_packed, int offset,
                                       float softmax_scale, float* out, void* workspace,
                                       size_t workspace_bytes, int32_t* dev_err,
                                       kvq_stream_t stream) {
  using namespace kvq;
  const char* fn = "kivi_decode_attn";
  kvq_status st = check_caches(caches, n_layers, fn);
  if (st != KVQ_OK) return st;
  const kivi_packed& c0 = caches[0];
  if (c0.bits != 2 || c0.head_dim != kAD || c0.group_size % 16)
    return fail(KVQ_ERR_SHAPE, "%s: supports 2-bit codes, head_dim 64, group_size 16/32/64", fn);
  const int H = c0.num_heads;
  if (num_q_heads < H || num_q_heads % H || num_q_heads / H > 8)
    return fail(KVQ_ERR_SHAPE, "%s: num_q_heads %d must be a multiple of %d, at most 8 per KV "
                "head", fn, num_q_heads, H);
  if (n_packed < 0 || n_packed % c0.group_size || offset < n_packed || offset > c0.capacity)
    return fail(KVQ_ERR_RANGE, "%s: need 0 <= n_packed <= offset <= capacity, n_packed a "
                "multiple of group_size", fn);
  if (!k || !v || !q || !out || !workspace) return fail(KVQ_ERR_NULL, "%s: NULL pointer", fn);
  for (int i = 0; i < n_layers; ++i) {
    if (!k[i] || !v[i]) return fail(KVQ_ERR_NULL, "%s: fp16 cache of layer %d is NULL", fn, i);
    if (!aligned16(k[i]) || !aligned16(v[i]))
      return fail(KVQ_ERR_ALIGN, "%s: fp16 caches must be 16-byte aligned", fn);
  }
  if (!aligned16(q) || !aligned16(out) || !aligned16(workspace))
    return fail(KVQ_ERR_ALIGN, "%s: q/out/workspace must be 16-byte aligned", fn);
  const size_t need = kivi_decode_attn_workspace(n_layers, c0.batch, H, num_q_heads, kAD, offset);
  if (workspace_bytes < need)
    return fail(KVQ_ERR_WORKSPACE, "%s: workspace %zu < %zu bytes", fn, workspace_bytes, need);
  if (static_cast<int64_t>(n_layers) * c0.batch > 65535 || H > 65535)
    return fail(KVQ_ERR_RANGE, "%s: n_layers * batch and num_heads must be <= 65535", fn);
  KAArgs a;
  for (int i = 0; i < KVQ_MAX_TENSORS; ++i) {
    a.c[i] = caches[i < n_layers ? i : 0];
    a.k[i] = i < n_layers ? k[i] : nullptr;
    a.v[i] = i < n_layers ? v[i] : nullptr;
  }
  a.q = q;
  a.out = out;
  a.ws = static_cast<float*>(workspace);
  a.err = dev_err;
  a.n_layers = n_layers;
  a.B = c0.batch;
  a.H = H;
  a.G = num_q_heads / H;
  a.Hq = num_q_heads;
  a.S = c0.capacity;
  a.n_packed = n_packed;
  a.offset = offset;
  a.tiles_per_cta = attn_tiles_per_cta(n_layers, c0.batch, H, offset);
  const int tiles = (offset + kATile - 1) / kATile;
  a.n_splits = tiles > 0 ? (tiles + a.tiles_per_cta - 1) / a.tiles_per_cta : 1;
  a.qk_scale = softmax_scale * 1.4426950408889634f;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  static_assert(kAttnSmem >= kAWarps * 8 * kAD * 4 + 2 * kAWarps * 32,
                "the merge buffer must fit in the stage ring");
  cudaError_t e = cudaFuncSetAttribute(kivi_attn_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kAttnSmem);
  if (e != cudaSuccess) return fail(KVQ_ERR_CUDA, "%s: %s", fn, cudaGetErrorString(e));
  kivi_attn_kernel<<<dim3(a.n_splits, H, n_layers * c0.batch), kAThreads, kAttnSmem, cs>>>(a);
  kivi_attn_merge_kernel<<<dim3(num_q_heads, n_layers * c0.batch), kAD, 0, cs>>>(a);
  e = cudaGetLastError();
  if (e != cudaSuccess) return fail(KVQ_ERR_CUDA, "%s launch: %s", fn, cudaGetErrorString(e));
  return ok();
}
