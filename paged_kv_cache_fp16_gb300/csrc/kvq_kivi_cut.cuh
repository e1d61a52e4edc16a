// 2-bit KIVI codes (levels = 3) by fp16 compares against per-group code boundaries.
//
// VeloxQuant-MLX source page "veloxquant_mlx.cache.kivi_cache", KIVIKVCache._quant_dequant_along:
// the code of x in a group with minimum z is clamp(rint(RN(d / scale)), 0, 3), d = RN(x - z).  As
// three compares it counts the thresholds t1 < t2 < t3 that d reaches (the threshold form of the
// two KIVI sources).  d is nondecreasing in x, so d(x) >= t holds exactly for the fp16 x at or
// above one boundary X(t): the smallest fp16 value that reaches t.  Finding X(t) costs a few float
// evaluations per group; every pair of elements then costs one packed fp16 compare (HSET2) per
// threshold, with no conversion to float and no subtraction.
//
// Order keys map the non-NaN fp16 bit patterns monotonically onto 0x03ff (-inf) .. 0xfc00 (+inf),
// -0 just below +0 (both give the same d, so no boundary separates them).  A NaN element compares
// false against every boundary, as its NaN difference fails every threshold.
#pragma once

#include <cstdint>

#include <cuda_fp16.h>

#include "kvq_device.cuh"

namespace kvq {
namespace {

constexpr uint32_t kKeyNegInf = 0x03ffu, kKeyPosInf = 0xfc00u;
constexpr uint32_t kNeverReached = 0x7fffu;   // a NaN: no fp16 compare with it is true

__device__ __forceinline__ uint32_t hkey(uint32_t b) { return b ^ ((b & 0x8000u) ? 0xffffu : 0x8000u); }
__device__ __forceinline__ uint32_t hbits(uint32_t k) { return k ^ ((k & 0x8000u) ? 0x8000u : 0xffffu); }

__device__ __forceinline__ bool reaches(uint32_t k, float z, float t) {
  return __fsub_rn(h2f(static_cast<uint16_t>(hbits(k))), z) >= t;
}

// fp16 bits of the smallest non-NaN fp16 X with RN(X - z) >= t, or kNeverReached.  The guess
// fp16(z + t) is almost always the answer or its neighbour; otherwise a bisection over the order
// keys whose bracket keeps !reaches(lo) and reaches(hi) (-inf reaches no t > -inf).  The
// bisection runs where many fp16 values share one float difference, e.g. a boundary at zero.
__device__ __forceinline__ uint32_t first_reaching(float z, float t) {
  uint32_t k = hkey(f2h(__fadd_rn(z, t)));
  k = min(max(k, kKeyNegInf + 1u), kKeyPosInf);
  uint32_t lo, hi;
  if (reaches(k, z, t)) {
    if (!reaches(k - 1u, z, t)) return hbits(k);
    lo = kKeyNegInf;
    hi = k - 1u;
  } else {
    if (k == kKeyPosInf) return kNeverReached;
    if (reaches(k + 1u, z, t)) return hbits(k + 1u);
    if (!reaches(kKeyPosInf, z, t)) return kNeverReached;
    lo = k + 1u;
    hi = kKeyPosInf;
  }
  while (hi - lo > 1u) {
    const uint32_t m = (lo + hi) >> 1;
    if (reaches(m, z, t)) hi = m; else lo = m;
  }
  return hbits(hi);
}

// Two searches at once, one per half (low: a, high: b), on packed operations: the guess is
// fp16(z + t) rounded up, which is the answer unless fp16(z + t) is exactly representable after a
// float32 sum that rounded down, or many fp16 values share the difference at the boundary; the
// guess and its lower neighbour are checked for both halves with one packed float32 subtraction
// each, and a half that does not settle takes the scalar search.
__device__ __forceinline__ uint32_t hkey2(uint32_t b) {
  return b ^ 0x80008000u ^ (((b >> 15) & 0x00010001u) * 0x7fffu);
}
__device__ __forceinline__ uint32_t hbits2(uint32_t k) {
  return k ^ 0xffffffffu ^ (((k >> 15) & 0x00010001u) * 0x7fffu);
}

// RN32(x - z) >= t for the fp16 values of both halves of `bits`: bit 0 (low half), bit 1 (high).
__device__ __forceinline__ uint32_t reaches2(uint32_t bits, uint64_t nz, float ta, float tb) {
  const float2 x = __half22float2(*reinterpret_cast<const __half2*>(&bits));
  uint64_t xx, d;
  asm("mov.b64 %0, {%1, %2};" : "=l"(xx) : "f"(x.x), "f"(x.y));
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(xx), "l"(nz));
  float da, db;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(da), "=f"(db) : "l"(d));
  return static_cast<uint32_t>(da >= ta) | (static_cast<uint32_t>(db >= tb) << 1);
}

__device__ __forceinline__ uint32_t first_reaching2(float za, float ta, float zb, float tb) {
  uint64_t zz, tt, g, nz;
  asm("mov.b64 %0, {%1, %2};" : "=l"(zz) : "f"(za), "f"(zb));
  asm("mov.b64 %0, {%1, %2};" : "=l"(tt) : "f"(ta), "f"(tb));
  asm("mov.b64 %0, {%1, %2};" : "=l"(nz) : "f"(-za), "f"(-zb));
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(g) : "l"(zz), "l"(tt));
  float ga, gb;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(ga), "=f"(gb) : "l"(g));
  const uint32_t hb = (static_cast<uint32_t>(__half_as_ushort(__float2half_ru(gb))) << 16) |
                      __half_as_ushort(__float2half_ru(ga));
  const uint32_t k = __vmaxu2(__vminu2(hkey2(hb), 0xfc00fc00u), 0x04000400u);
  const uint32_t r0 = reaches2(hbits2(k), nz, ta, tb);
  const uint32_t rm = reaches2(hbits2(k - 0x00010001u), nz, ta, tb);
  const uint32_t ok = r0 & ~rm;   // bit i: half i settled at its guess
  uint32_t out = hbits2(k);
  if (ok != 3u) {   // rare: the scalar search for the half that did not settle
    if (!(ok & 1u)) out = (out & 0xffff0000u) | first_reaching(za, ta);
    if (!(ok & 2u)) out = (out & 0x0000ffffu) | (first_reaching(zb, tb) << 16);
  }
  return out;
}

// The three code boundaries of two groups as half2 words (low half: group a, high half: group b).
// They nest: x >= X3 implies x >= X2 implies x >= X1.
struct L3Cut {
  uint32_t x1, x2, x3;
};

__device__ __forceinline__ L3Cut l3_cut2(float za, float a1, float a2, float a3, float zb,
                                         float b1, float b2, float b3) {
  L3Cut c;
  c.x1 = first_reaching2(za, a1, zb, b1);
  c.x2 = first_reaching2(za, a2, zb, b2);
  c.x3 = first_reaching2(za, a3, zb, b3);
  return c;
}

__device__ __forceinline__ L3Cut l3_cut1(float z, float t1, float t2, float t3) {
  L3Cut c;   // three scalar searches (a packed pair measured slower here)
  c.x1 = first_reaching(z, t1) * 0x10001u;
  c.x2 = first_reaching(z, t2) * 0x10001u;
  c.x3 = first_reaching(z, t3) * 0x10001u;
  return c;
}

__device__ __forceinline__ __half2 cut_h2(uint32_t w) { return *reinterpret_cast<__half2*>(&w); }

// Round trip of both elements of a word: the code masks by fp16 compare, then the group's fp16
// reconstructions rr0..rr3 (half2, same halves as w) by bit select.
__device__ __forceinline__ uint32_t l3_cut_word(uint32_t w, const L3Cut& c, uint32_t rr0,
                                                uint32_t rr1, uint32_t rr2, uint32_t rr3) {
  const __half2 x = cut_h2(w);
  const uint32_t m1 = __hge2_mask(x, cut_h2(c.x1));
  const uint32_t m2 = __hge2_mask(x, cut_h2(c.x2));
  const uint32_t m3 = __hge2_mask(x, cut_h2(c.x3));
  uint32_t r = (rr0 & ~m1) | (rr1 & m1);
  r = (r & ~m2) | (rr2 & m2);
  return (r & ~m3) | (rr3 & m3);
}

// 2-bit codes of the 8 fp16 elements of w[0..3] (element e = half e & 1 of word e >> 1), packed
// LSB-first: element e at bits 2e, 2e + 1.  c[k] holds the boundaries of word k's two elements.
// Since the masks nest, code bit 1 is the second mask and code bit 0 the parity of the three.
template <int NC>
__device__ __forceinline__ uint32_t l3_codes8(const uint32_t w[4], const L3Cut* c) {
  uint32_t acc = 0;   // element 2k: bits 4k, 4k + 1; element 2k + 1: bits 16 + 4k + 2, + 3
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const L3Cut& ck = c[NC == 1 ? 0 : k];
    const __half2 x = cut_h2(w[k]);
    const uint32_t m1 = __hge2_mask(x, cut_h2(ck.x1));
    const uint32_t m2 = __hge2_mask(x, cut_h2(ck.x2));
    const uint32_t m3 = __hge2_mask(x, cut_h2(ck.x3));
    acc |= (m1 ^ m2 ^ m3) & ((0x1u << (4 * k)) | (0x4u << (16 + 4 * k)));
    acc |= m2 & ((0x2u << (4 * k)) | (0x8u << (16 + 4 * k)));
  }
  return (acc & 0xffffu) | (acc >> 16);
}

}  // namespace
}  // namespace kvq
