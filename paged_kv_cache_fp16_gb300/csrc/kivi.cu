// KIVI asymmetric min/max group quantize -> dequantize, in place on fp16 [B][H][S][D] tensors.
//
// VeloxQuant-MLX source page "veloxquant_mlx.cache.kivi_cache": KIVIKVCache._quant_dequant_along
// (the float32 round trip), update_and_fetch (keys per channel with groups along tokens, values
// per token with groups along channels, applied to the newly aged token slice [lo, hi)).
// Per group: scale = max((gmax - gmin) / levels, eps); c = clamp(rint((x - gmin) / scale), 0,
// levels); y = fp16((c * scale) + gmin), every step an IEEE float32 operation with its own
// rounding (explicit __f*_rn intrinsics so the compiler cannot fuse the multiply-add).  A ragged
// last group reduces over its real elements only, which equals the page's padding by repetition.
//
// One launch covers all tensors: the first blocks take key groups, the rest value groups.
// Keys: one thread per (tensor, b, h, token group, channel pair) holds the pair's column of the
// group in registers (fp16 min/max as a tree); adjacent threads own adjacent pairs of a row, so
// every row access is contiguous across the warp.  Values: one thread per (row, channel group)
// holds the group in 16-byte vectors.  Groups that are not a multiple of 8 channels use a scalar
// kernel.  HBM-bound: 4 bytes per element.  The data are modified in place, so loads use the
// coherent path (no ld.global.nc).
//
// The code of an element needs rint(RN(d / scale)) with d = RN(x - gmin) >= 0.  With the group's
// y = RN(1 / scale), q0 = RN(d * y) is within 2.5 ulp of RN(d / scale); wherever q0 is farther
// than |q0| * 2^-20 (> 8 ulp) from every half-integer both round to the same integer, so q0 is
// used; otherwise (near or at a tie) the IEEE quotient is computed.  The result is identical to
// dividing every element.  With levels = 3 (2 bits) the code is three compares instead: it is
// >= 1, 2, 3 iff d / scale exceeds 0.5 + 2^-25, reaches 1.5 - 2^-24, exceeds 2.5 + 2^-23 (ties
// of RN(d / scale) at 0.5, 1.5, 2.5 go to the even neighbour), and since no scale * m is an
// fp32 value (the multipliers' odd parts exceed 2^24) each condition is d >= RU(scale * m),
// one upward-rounded FMA per group from the exact product scale * 2^-k.
#include <algorithm>

#include <cuda_runtime.h>

#include "kvq_device.cuh"
#include "kvq_divu32.cuh"
#include "kvq_internal.h"
#include "kvq_kivi_cut.cuh"

namespace kvq {
namespace {

constexpr int kThreads = 256;
constexpr int kKeepRows = 32;  // key group rows held in registers (longer groups are re-read)
constexpr int kMaxVecs = 8;    // value group vectors held in registers (<= 64 channels)

// Passed by value (kernel parameter space): the library allocates no device memory.
struct KiviArgs {
  uint16_t* x[KVQ_MAX_TENSORS];
  int key_list[KVQ_MAX_TENSORS];  // indices into x of the key tensors
  int val_list[KVQ_MAX_TENSORS];  // indices into x of the value tensors
  int n_keys, n_vals;
  int B, H, S, D, lo, hi, gs;
  int key_blocks;                 // blocks [0, key_blocks) do keys, the rest values
  float levels, eps;
};

struct Group {
  float mn, sc, y;   // gmin, scale, RN(1 / scale)
  float t1, t2, t3;  // levels = 3: thresholds of codes 1, 2, 3 on d = RN(x - gmin)
};

template <bool L3, bool RCP = true>
__device__ __forceinline__ Group make_group(float mn, float mx, float levels, float eps) {
  Group g;
  g.mn = mn;
  g.sc = fmaxf(__fdiv_rn(__fsub_rn(mx, mn), levels), eps);
  g.y = RCP ? __frcp_rn(g.sc) : 0.f;
  if constexpr (L3) {
    if (g.sc == 0.f) {   // eps = 0 and a constant group: every code is 0
      g.t1 = g.t2 = g.t3 = __int_as_float(0x7f800000);
    } else {
      g.t1 = __fmaf_ru(g.sc, 0.5f, g.sc * 2.98023223876953125e-08f);    // sc (0.5 + 2^-25)
      g.t2 = __fmaf_ru(g.sc, 1.5f, -(g.sc * 5.9604644775390625e-08f));  // sc (1.5 - 2^-24)
      g.t3 = __fmaf_ru(g.sc, 2.5f, g.sc * 1.1920928955078125e-07f);     // sc (2.5 + 2^-23)
    }
  }
  return g;
}

// The exact quotient, out of line: it runs only near ties, and keeping it out of the unrolled
// loops keeps the kernel's code small.
__device__ __noinline__ float exact_quotient(float d, float sc) { return __fdiv_rn(d, sc); }

template <bool L3>
__device__ __forceinline__ uint16_t roundtrip(float x, const Group& g, float levels) {
  const float d = __fsub_rn(x, g.mn);
  float c;
  if constexpr (L3) {
    c = d >= g.t3 ? 3.f : (d >= g.t2 ? 2.f : (d >= g.t1 ? 1.f : 0.f));
  } else {
    const float q0 = __fmul_rn(d, g.y);
    const float dist = fabsf(__fsub_rn(__fadd_rn(floorf(q0), 0.5f), q0));
    float q = q0;
    if (dist <= __fmul_rn(q0, 9.5367431640625e-07f)) q = exact_quotient(d, g.sc);  // 2^-20
    c = fminf(fmaxf(rintf(q), 0.f), levels);
  }
  return f2h(__fadd_rn(__fmul_rn(c, g.sc), g.mn));
}

template <bool L3>
__device__ __forceinline__ uint32_t roundtrip2(uint32_t w, const Group& g0, const Group& g1,
                                               float levels) {
  const uint32_t lo = roundtrip<L3>(h2f(static_cast<uint16_t>(w & 0xffffu)), g0, levels);
  const uint32_t hi = roundtrip<L3>(h2f(static_cast<uint16_t>(w >> 16)), g1, levels);
  return lo | (hi << 16);
}

__device__ __forceinline__ __half2 as_h2(uint32_t w) { return *reinterpret_cast<__half2*>(&w); }

// ------------------------------------------------------------------------------ keys
template <bool L3>
__device__ __forceinline__ void keys_part(const KiviArgs& a, int64_t first, int64_t stride) {
  const int span = a.hi - a.lo;
  const int n_groups = (span + a.gs - 1) / a.gs;
  const int pairs = a.D / 2;
  const int64_t bh_count = static_cast<int64_t>(a.B) * a.H;
  const int64_t items = static_cast<int64_t>(a.n_keys) * bh_count * n_groups * pairs;
  for (int64_t it = first; it < items; it += stride) {
    const int pr = static_cast<int>(it % pairs);
    const int64_t r1 = it / pairs;
    const int g = static_cast<int>(r1 % n_groups);
    const int64_t r2 = r1 / n_groups;
    const int64_t bh = r2 % bh_count;
    const int ti = a.key_list[r2 / bh_count];
    const int t0 = a.lo + g * a.gs;
    const int n = min(a.gs, a.hi - t0);
    uint32_t* base = reinterpret_cast<uint32_t*>(a.x[ti] + (bh * a.S + t0) * a.D) + pr;
    const int64_t stride_w = a.D / 2;   // in half2 words
    uint32_t keep[kKeepRows];
    keep[0] = base[0];
#pragma unroll
    for (int r = 1; r < kKeepRows; ++r)   // rows past the group repeat row 0 (min/max unchanged)
      keep[r] = (r < n) ? base[r * stride_w] : keep[0];
    // pairwise tree of fp16 min / max (exact)
    __half2 mn[kKeepRows / 2], mx[kKeepRows / 2];
#pragma unroll
    for (int r = 0; r < kKeepRows / 2; ++r) {
      mn[r] = __hmin2(as_h2(keep[2 * r]), as_h2(keep[2 * r + 1]));
      mx[r] = __hmax2(as_h2(keep[2 * r]), as_h2(keep[2 * r + 1]));
    }
#pragma unroll
    for (int w = kKeepRows / 4; w >= 1; w >>= 1)
#pragma unroll
      for (int r = 0; r < w; ++r) {
        mn[r] = __hmin2(mn[r], mn[r + w]);
        mx[r] = __hmax2(mx[r], mx[r + w]);
      }
    __half2 gmn = mn[0], gmx = mx[0];
    for (int r = kKeepRows; r < n; ++r) {
      const __half2 v = as_h2(base[r * stride_w]);
      gmn = __hmin2(gmn, v);
      gmx = __hmax2(gmx, v);
    }
    const Group g0 = make_group<L3>(__low2float(gmn), __low2float(gmx), a.levels, a.eps);
    const Group g1 = make_group<L3>(__high2float(gmn), __high2float(gmx), a.levels, a.eps);
#pragma unroll
    for (int r = 0; r < kKeepRows; ++r)
      if (r < n) base[r * stride_w] = roundtrip2<L3>(keep[r], g0, g1, a.levels);
    for (int r = kKeepRows; r < n; ++r)
      base[r * stride_w] = roundtrip2<L3>(base[r * stride_w], g0, g1, a.levels);
  }
}

// ------------------------------------------------------------------------------ values
template <bool L3>
__device__ __forceinline__ void values_part(const KiviArgs& a, int64_t first, int64_t stride) {
  const int span = a.hi - a.lo;
  const int groups = (a.D + a.gs - 1) / a.gs;
  const int64_t rows_per_tensor = static_cast<int64_t>(a.B) * a.H * span;
  const int64_t items = rows_per_tensor * a.n_vals * groups;
  for (int64_t it = first; it < items; it += stride) {
    const int g = static_cast<int>(it % groups);
    const int64_t row = it / groups;
    const int64_t vi = row / rows_per_tensor;
    const int64_t r = row - vi * rows_per_tensor;
    const int64_t bh = r / span;
    const int t = a.lo + static_cast<int>(r - bh * span);
    const int c0 = g * a.gs;
    const int nv = (min(a.D, c0 + a.gs) - c0) / 8;   // 16-byte vectors in this group
    uint4* p = reinterpret_cast<uint4*>(a.x[a.val_list[vi]] + (bh * a.S + t) * a.D + c0);
    uint4 v[kMaxVecs];
    v[0] = p[0];
#pragma unroll
    for (int k = 1; k < kMaxVecs; ++k) v[k] = (k < nv) ? p[k] : v[0];  // repeats keep min/max
    __half2 mn[kMaxVecs], mx[kMaxVecs];
#pragma unroll
    for (int k = 0; k < kMaxVecs; ++k) {
      mn[k] = __hmin2(__hmin2(as_h2(v[k].x), as_h2(v[k].y)), __hmin2(as_h2(v[k].z), as_h2(v[k].w)));
      mx[k] = __hmax2(__hmax2(as_h2(v[k].x), as_h2(v[k].y)), __hmax2(as_h2(v[k].z), as_h2(v[k].w)));
    }
#pragma unroll
    for (int w = kMaxVecs / 2; w >= 1; w >>= 1)
#pragma unroll
      for (int k = 0; k < w; ++k) {
        mn[k] = __hmin2(mn[k], mn[k + w]);
        mx[k] = __hmax2(mx[k], mx[k + w]);
      }
    const Group gr = make_group<L3>(fminf(__low2float(mn[0]), __high2float(mn[0])),
                                fmaxf(__low2float(mx[0]), __high2float(mx[0])), a.levels, a.eps);
#pragma unroll
    for (int k = 0; k < kMaxVecs; ++k) {
      if (k >= nv) continue;
      p[k] = make_uint4(roundtrip2<L3>(v[k].x, gr, gr, a.levels),
                        roundtrip2<L3>(v[k].y, gr, gr, a.levels),
                        roundtrip2<L3>(v[k].z, gr, gr, a.levels),
                        roundtrip2<L3>(v[k].w, gr, gr, a.levels));
    }
  }
}

// Keys and values of every tensor in one launch (block-uniform split).
template <bool L3>
__global__ void __launch_bounds__(kThreads, 3) kivi_kernel(const KiviArgs a) {
  if (static_cast<int>(blockIdx.x) < a.key_blocks)
    keys_part<L3>(a, static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x,
              static_cast<int64_t>(a.key_blocks) * kThreads);
  else
    values_part<L3>(a, static_cast<int64_t>(blockIdx.x - a.key_blocks) * kThreads + threadIdx.x,
                static_cast<int64_t>(gridDim.x - a.key_blocks) * kThreads);
}

// Values whose groups are not a multiple of 8 channels (or longer than 64): one thread per
// (row, channel group), scalar loads.
template <bool L3>
__global__ void __launch_bounds__(kThreads) kivi_values_scalar_kernel(const KiviArgs a) {
  const int span = a.hi - a.lo;
  const int groups = (a.D + a.gs - 1) / a.gs;
  const int64_t rows_per_tensor = static_cast<int64_t>(a.B) * a.H * span;
  const int64_t items = rows_per_tensor * a.n_vals * groups;
  for (int64_t it = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; it < items;
       it += static_cast<int64_t>(gridDim.x) * kThreads) {
    const int g = static_cast<int>(it % groups);
    const int64_t row = it / groups;
    const int64_t vi = row / rows_per_tensor;
    const int64_t r = row - vi * rows_per_tensor;
    const int64_t bh = r / span;
    const int t = a.lo + static_cast<int>(r - bh * span);
    uint16_t* p = a.x[a.val_list[vi]] + (bh * a.S + t) * a.D;
    const int c0 = g * a.gs, c1 = min(a.D, c0 + a.gs);
    float mn = __int_as_float(0x7f800000), mx = -mn;
    for (int c = c0; c < c1; ++c) { const float v = h2f(p[c]); mn = fminf(mn, v); mx = fmaxf(mx, v); }
    const Group gr = make_group<L3>(mn, mx, a.levels, a.eps);
    for (int c = c0; c < c1; ++c) p[c] = roundtrip<L3>(h2f(p[c]), gr, a.levels);
  }
}

// ------------------------------------------------------------------------------ 2 bits
// levels = 3 with key groups of at most 32 tokens and value groups of 8..64 channels (8 | gs): one
// thread per item (a key channel pair of one token group, or a value channel group of one row),
// no grid-stride loop, the flat item index split with multiply-high division.  Key and value
// blocks are interleaved in proportion to their counts (pattern of period pk + pv), so every wave
// of the grid streams both.  A group's four reconstructions fp16(RN(RN(c * scale) + gmin)),
// c = 0..3, are computed once, and so are the group's three code boundaries as fp16 values; each
// pair of elements then costs three packed fp16 compares and three bit selects.
struct L3Plan {
  DivU32 period;      // pk + pv
  DivU32 pairs;       // D / 2
  DivU32 key_groups;  // token groups of the span
  DivU32 bh;          // B * H
  DivU32 val_groups;  // channel groups per row
  DivU32 span;        // hi - lo
  int pk, pv;
  uint32_t key_items, val_items;
};

__device__ __forceinline__ uint32_t recon_bits(const Group& g, float c) {
  return f2h(__fadd_rn(__fmul_rn(c, g.sc), g.mn));
}

__device__ __forceinline__ L3Cut l3_cut(const Group& a, const Group& b) {
  return l3_cut2(a.mn, a.t1, a.t2, a.t3, b.mn, b.t1, b.t2, b.t3);
}

__device__ __forceinline__ L3Cut l3_cut(const Group& g) { return l3_cut1(g.mn, g.t1, g.t2, g.t3); }

// A value group of NV 16-byte vectors (8 * NV channels): load, fp16 min/max tree, the 2-bit
// round trip, store.  V8: the group is 32-byte aligned and moves in 256-bit accesses.
template <int NV, bool V8>
__device__ __forceinline__ void l3_value_group(uint4* pv, float levels, float eps) {
  uint4 v[NV];
  if constexpr (V8 && NV % 2 == 0) {
#pragma unroll
    for (int k = 0; k < NV; k += 2) ld_v8(pv + k, v[k], v[k + 1]);
  } else {
#pragma unroll
    for (int k = 0; k < NV; ++k) v[k] = pv[k];
  }
  __half2 mn = __hmin2(__hmin2(as_h2(v[0].x), as_h2(v[0].y)), __hmin2(as_h2(v[0].z), as_h2(v[0].w)));
  __half2 mx = __hmax2(__hmax2(as_h2(v[0].x), as_h2(v[0].y)), __hmax2(as_h2(v[0].z), as_h2(v[0].w)));
#pragma unroll
  for (int k = 1; k < NV; ++k) {
    mn = __hmin2(mn, __hmin2(__hmin2(as_h2(v[k].x), as_h2(v[k].y)),
                             __hmin2(as_h2(v[k].z), as_h2(v[k].w))));
    mx = __hmax2(mx, __hmax2(__hmax2(as_h2(v[k].x), as_h2(v[k].y)),
                             __hmax2(as_h2(v[k].z), as_h2(v[k].w))));
  }
  const Group gr = make_group<true, false>(fminf(__low2float(mn), __high2float(mn)),
                                           fmaxf(__low2float(mx), __high2float(mx)), levels, eps);
  const uint32_t r0 = recon_bits(gr, 0.f), r1 = recon_bits(gr, 1.f);
  const uint32_t r2 = recon_bits(gr, 2.f), r3 = recon_bits(gr, 3.f);
  const uint32_t rr0 = r0 | (r0 << 16), rr1 = r1 | (r1 << 16);
  const uint32_t rr2 = r2 | (r2 << 16), rr3 = r3 | (r3 << 16);
  const L3Cut cut = l3_cut(gr);
  uint4 o[NV];
#pragma unroll
  for (int k = 0; k < NV; ++k)
    o[k] = make_uint4(l3_cut_word(v[k].x, cut, rr0, rr1, rr2, rr3),
                      l3_cut_word(v[k].y, cut, rr0, rr1, rr2, rr3),
                      l3_cut_word(v[k].z, cut, rr0, rr1, rr2, rr3),
                      l3_cut_word(v[k].w, cut, rr0, rr1, rr2, rr3));
  if constexpr (V8 && NV % 2 == 0) {
#pragma unroll
    for (int k = 0; k < NV; k += 2) st_v8(pv + k, o[k], o[k + 1]);
  } else {
#pragma unroll
    for (int k = 0; k < NV; ++k) pv[k] = o[k];
  }
}

// One key item: the column pair (channels 2 pr, 2 pr + 1) of one token group in registers, its
// two groups' fp16 min / max as a tree, parameters, code boundaries and reconstructions, then the
// round trip of every row.  SW > 0: a full group of kKeepRows rows SW words apart -- the loads
// and stores take immediate offsets and no row predicate (the workload's head_dim 64, group 32);
// SW = 0: n rows sw words apart.
template <int SW>
__device__ __forceinline__ void l3_key_group(uint32_t* base, int n, int64_t sw,
                                             const KiviArgs& a) {
  const int64_t stride = SW > 0 ? SW : sw;
  uint32_t keep[kKeepRows];
  keep[0] = base[0];
#pragma unroll
  for (int r = 1; r < kKeepRows; ++r) keep[r] = (SW > 0 || r < n) ? base[r * stride] : keep[0];
  __half2 mn[kKeepRows / 2], mx[kKeepRows / 2];
#pragma unroll
  for (int r = 0; r < kKeepRows / 2; ++r) {
    mn[r] = __hmin2(as_h2(keep[2 * r]), as_h2(keep[2 * r + 1]));
    mx[r] = __hmax2(as_h2(keep[2 * r]), as_h2(keep[2 * r + 1]));
  }
#pragma unroll
  for (int w = kKeepRows / 4; w >= 1; w >>= 1)
#pragma unroll
    for (int r = 0; r < w; ++r) {
      mn[r] = __hmin2(mn[r], mn[r + w]);
      mx[r] = __hmax2(mx[r], mx[r + w]);
    }
  const Group g0 = make_group<true, false>(__low2float(mn[0]), __low2float(mx[0]), a.levels,
                                           a.eps);
  const Group g1 = make_group<true, false>(__high2float(mn[0]), __high2float(mx[0]), a.levels,
                                           a.eps);
  // the four reconstructions of both channels, as half2 (low: channel 2 pr, high: 2 pr + 1)
  const uint32_t rr0 = recon_bits(g0, 0.f) | (recon_bits(g1, 0.f) << 16);
  const uint32_t rr1 = recon_bits(g0, 1.f) | (recon_bits(g1, 1.f) << 16);
  const uint32_t rr2 = recon_bits(g0, 2.f) | (recon_bits(g1, 2.f) << 16);
  const uint32_t rr3 = recon_bits(g0, 3.f) | (recon_bits(g1, 3.f) << 16);
  const L3Cut cut = l3_cut(g0, g1);
#pragma unroll
  for (int r = 0; r < kKeepRows; ++r) {
    if (SW == 0 && r >= n) break;
    base[r * stride] = l3_cut_word(keep[r], cut, rr0, rr1, rr2, rr3);
  }
}

// Built for 4 blocks per SM (64 registers, no spills): 32 warps per SM keep more loads in flight
// than 3 blocks at 76 registers did (128-token flush of 16 layers, back to back from a CUDA graph:
// 23.8 against 24.6 us when that choice was made).
template <bool V8>
__global__ void __launch_bounds__(kThreads, 4) kivi_l3_kernel(const KiviArgs a, const L3Plan p) {
  const uint32_t b = blockIdx.x;
  const uint32_t q = divu32(b, p.period);
  const int o = static_cast<int>(b - q * static_cast<uint32_t>(p.pk + p.pv));
  if (o < p.pk) {
    // ---------------------------------------------------------------- keys
    const uint32_t it = (q * p.pk + o) * kThreads + threadIdx.x;
    if (it >= p.key_items) return;
    const uint32_t r1 = divu32(it, p.pairs);
    const int pr = static_cast<int>(it - r1 * static_cast<uint32_t>(a.D / 2));
    const uint32_t r2 = divu32(r1, p.key_groups);
    const int g = static_cast<int>(r1 - r2 * static_cast<uint32_t>((a.hi - a.lo + a.gs - 1) / a.gs));
    const uint32_t ki = divu32(r2, p.bh);
    const int64_t bh = r2 - ki * static_cast<uint32_t>(a.B * a.H);
    const int t0 = a.lo + g * a.gs;
    const int n = min(a.gs, a.hi - t0);
    uint32_t* base = reinterpret_cast<uint32_t*>(a.x[a.key_list[ki]] + (bh * a.S + t0) * a.D) + pr;
    if (n == kKeepRows && a.D == 64) l3_key_group<32>(base, n, 32, a);
    else l3_key_group<0>(base, n, a.D / 2, a);
  } else {
    // ---------------------------------------------------------------- values
    const uint32_t it = (q * p.pv + (o - p.pk)) * kThreads + threadIdx.x;
    if (it >= p.val_items) return;
    const int groups = (a.D + a.gs - 1) / a.gs;
    const uint32_t row = divu32(it, p.val_groups);
    const int gi = static_cast<int>(it - row * static_cast<uint32_t>(groups));
    const uint32_t r2 = divu32(row, p.span);
    const int t = a.lo + static_cast<int>(row - r2 * static_cast<uint32_t>(a.hi - a.lo));
    const uint32_t vi = divu32(r2, p.bh);
    const int64_t bh = r2 - vi * static_cast<uint32_t>(a.B * a.H);
    const int c0 = gi * a.gs;
    const int nv = (min(a.D, c0 + a.gs) - c0) / 8;   // 16-byte vectors in this group
    uint4* pv = reinterpret_cast<uint4*>(a.x[a.val_list[vi]] + (bh * a.S + t) * a.D + c0);
    if (nv == 4) {   // groups of 32 channels: no padding, no bounds
      l3_value_group<4, V8>(pv, a.levels, a.eps);
      return;
    }
    if (nv == 2) {
      l3_value_group<2, V8>(pv, a.levels, a.eps);
      return;
    }
    if (nv == 1) {
      l3_value_group<1, V8>(pv, a.levels, a.eps);
      return;
    }
    // other group widths: up to 8 vectors, padded with the first (min / max unchanged)
    uint4 v[kMaxVecs];
    v[0] = pv[0];
#pragma unroll
    for (int k = 1; k < kMaxVecs; ++k) v[k] = (k < nv) ? pv[k] : v[0];
    __half2 mn = __hmin2(__hmin2(as_h2(v[0].x), as_h2(v[0].y)), __hmin2(as_h2(v[0].z), as_h2(v[0].w)));
    __half2 mx = __hmax2(__hmax2(as_h2(v[0].x), as_h2(v[0].y)), __hmax2(as_h2(v[0].z), as_h2(v[0].w)));
#pragma unroll
    for (int k = 1; k < kMaxVecs; ++k) {
      mn = __hmin2(mn, __hmin2(__hmin2(as_h2(v[k].x), as_h2(v[k].y)),
                               __hmin2(as_h2(v[k].z), as_h2(v[k].w))));
      mx = __hmax2(mx, __hmax2(__hmax2(as_h2(v[k].x), as_h2(v[k].y)),
                               __hmax2(as_h2(v[k].z), as_h2(v[k].w))));
    }
    const Group gr = make_group<true, false>(fminf(__low2float(mn), __high2float(mn)),
                                             fmaxf(__low2float(mx), __high2float(mx)), a.levels,
                                             a.eps);
    const uint32_t c0r = recon_bits(gr, 0.f), c1r = recon_bits(gr, 1.f);
    const uint32_t c2r = recon_bits(gr, 2.f), c3r = recon_bits(gr, 3.f);
    const uint32_t rr0 = c0r | (c0r << 16), rr1 = c1r | (c1r << 16);
    const uint32_t rr2 = c2r | (c2r << 16), rr3 = c3r | (c3r << 16);
    const L3Cut cut = l3_cut(gr);
#pragma unroll
    for (int k = 0; k < kMaxVecs; ++k) {
      if (k >= nv) break;
      pv[k] = make_uint4(l3_cut_word(v[k].x, cut, rr0, rr1, rr2, rr3),
                         l3_cut_word(v[k].y, cut, rr0, rr1, rr2, rr3),
                         l3_cut_word(v[k].z, cut, rr0, rr1, rr2, rr3),
                         l3_cut_word(v[k].w, cut, rr0, rr1, rr2, rr3));
    }
  }
}

int blocks_for_threads(int64_t threads, int cap) {
  int64_t b = (threads + kThreads - 1) / kThreads;
  if (b > cap) b = cap;
  return static_cast<int>(b < 1 ? 1 : b);
}

}  // namespace
}  // namespace kvq

extern "C" kvq_status kivi_quant_dequant(uint16_t* const* x, const int32_t* is_key,
                                         int n_tensors, int B, int H, int S, int D, int lo,
                                         int hi, int group_size, int levels, float eps,
                                         kvq_stream_t stream) {
  using namespace kvq;
  if (n_tensors < 1 || n_tensors > KVQ_MAX_TENSORS)
    return fail(KVQ_ERR_RANGE, "kivi_quant_dequant: n_tensors %d not in [1, %d]", n_tensors,
                KVQ_MAX_TENSORS);
  if (B < 1 || H < 1 || S < 1)
    return fail(KVQ_ERR_RANGE, "kivi_quant_dequant: B, H, S must be >= 1");
  if (D < 8 || D > 256 || D % 8)
    return fail(KVQ_ERR_SHAPE, "kivi_quant_dequant: D %d must be a multiple of 8 in [8, 256]", D);
  if (lo < 0 || hi < lo || hi > S)
    return fail(KVQ_ERR_SHAPE, "kivi_quant_dequant: need 0 <= lo <= hi <= S (lo %d hi %d S %d)",
                lo, hi, S);
  if (group_size < 1 || levels < 1)
    return fail(KVQ_ERR_SHAPE, "kivi_quant_dequant: group_size and levels must be >= 1");
  if (!(eps >= 0.f)) return fail(KVQ_ERR_RANGE, "kivi_quant_dequant: eps must be >= 0");
  if (!x || !is_key) return fail(KVQ_ERR_NULL, "kivi_quant_dequant: NULL array");
  for (int i = 0; i < n_tensors; ++i) {
    if (!x[i]) return fail(KVQ_ERR_NULL, "kivi_quant_dequant: tensor %d is NULL", i);
    if (!aligned16(x[i]))
      return fail(KVQ_ERR_ALIGN, "kivi_quant_dequant: tensor %d not 16-byte aligned", i);
  }
  if (hi == lo) return ok();

  KiviArgs a;
  a.B = B; a.H = H; a.S = S; a.D = D; a.lo = lo; a.hi = hi; a.gs = group_size;
  a.levels = static_cast<float>(levels);
  a.eps = eps;
  a.n_keys = a.n_vals = 0;
  for (int i = 0; i < KVQ_MAX_TENSORS; ++i) {
    a.x[i] = i < n_tensors ? x[i] : nullptr;
    a.key_list[i] = a.val_list[i] = 0;
  }
  for (int i = 0; i < n_tensors; ++i) {
    if (is_key[i]) a.key_list[a.n_keys++] = i; else a.val_list[a.n_vals++] = i;
  }
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const int span = hi - lo;
  const int sms = sm_count() > 0 ? sm_count() : 152;
  const int cap = sms * 3;
  const int64_t key_items = static_cast<int64_t>(a.n_keys) * B * H *
                            ((span + group_size - 1) / group_size) * (D / 2);
  const int64_t val_rows = static_cast<int64_t>(a.n_vals) * B * H * span;
  const int64_t val_items = val_rows * ((D + group_size - 1) / group_size);
  const bool vec_values = group_size % 8 == 0 && group_size <= 8 * kMaxVecs;
  const int kb = a.n_keys > 0 ? blocks_for_threads(key_items, cap) : 0;
  const int vb = (a.n_vals > 0 && vec_values) ? blocks_for_threads(val_items, cap) : 0;
  a.key_blocks = kb;
  const bool l3 = levels == 3;   // 2 bits: codes by thresholds
  const int key_groups = (span + group_size - 1) / group_size;
  if (l3 && group_size <= kKeepRows && (a.n_vals == 0 || vec_values) &&
      key_items + val_items > 0 && key_items < (1LL << 31) && val_items < (1LL << 31)) {
    // one thread per item, key and value blocks interleaved
    L3Plan p;
    const int64_t nkb = (key_items + kThreads - 1) / kThreads;
    const int64_t nvb = (val_items + kThreads - 1) / kThreads;
    if (nkb == 0) { p.pk = 0; p.pv = 1; }
    else if (nvb == 0) { p.pk = 1; p.pv = 0; }
    else if (nvb >= nkb) { p.pk = 1; p.pv = static_cast<int>((nvb + nkb / 2) / nkb); }
    else { p.pv = 1; p.pk = static_cast<int>((nkb + nvb / 2) / nvb); }
    if (p.pk + p.pv > 64) {   // very lopsided: plain halves (rare shapes)
      p.pk = nkb > 0 ? 1 : 0;
      p.pv = nvb > 0 ? 1 : 0;
    }
    int64_t periods = 0;
    if (p.pk > 0) periods = (nkb + p.pk - 1) / p.pk;
    if (p.pv > 0) periods = std::max<int64_t>(periods, (nvb + p.pv - 1) / p.pv);
    p.period = make_divu32(static_cast<uint32_t>(p.pk + p.pv));
    p.pairs = make_divu32(static_cast<uint32_t>(D / 2));
    p.key_groups = make_divu32(static_cast<uint32_t>(key_groups));
    p.bh = make_divu32(static_cast<uint32_t>(B * H));
    p.val_groups = make_divu32(static_cast<uint32_t>((D + group_size - 1) / group_size));
    p.span = make_divu32(static_cast<uint32_t>(span));
    p.key_items = static_cast<uint32_t>(key_items);
    p.val_items = static_cast<uint32_t>(val_items);
    const int64_t blocks = periods * (p.pk + p.pv);
    if (blocks < (1LL << 31)) {
      // 256-bit value accesses when every tensor is 32-byte aligned (value groups are 16 or 32
      // channels at 16-channel offsets: D and group_size are multiples of 8 here, so check both)
      bool v8 = D % 16 == 0 && group_size % 16 == 0;
      for (int i = 0; i < n_tensors; ++i)
        if (reinterpret_cast<uintptr_t>(x[i]) % 32) v8 = false;
      if (v8) kivi_l3_kernel<true><<<static_cast<unsigned>(blocks), kThreads, 0, st>>>(a, p);
      else kivi_l3_kernel<false><<<static_cast<unsigned>(blocks), kThreads, 0, st>>>(a, p);
      const cudaError_t e = cudaGetLastError();
      if (e != cudaSuccess) return fail(KVQ_ERR_CUDA, "kivi launch: %s", cudaGetErrorString(e));
      return ok();
    }
  }
  if (kb + vb > 0) {
    if (l3) kivi_kernel<true><<<kb + vb, kThreads, 0, st>>>(a);
    else kivi_kernel<false><<<kb + vb, kThreads, 0, st>>>(a);
  }
  if (a.n_vals > 0 && !vec_values) {
    a.key_blocks = 0;
    const int nb = blocks_for_threads(val_items, sms * 8);
    if (l3) kivi_values_scalar_kernel<true><<<nb, kThreads, 0, st>>>(a);
    else kivi_values_scalar_kernel<false><<<nb, kThreads, 0, st>>>(a);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(KVQ_ERR_CUDA, "kivi launch: %s", cudaGetErrorString(e));
  return ok();
}
