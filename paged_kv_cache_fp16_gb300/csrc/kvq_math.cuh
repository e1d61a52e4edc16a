// Device arithmetic shared by the quantize, dequantize and attention kernels.
#pragma once

#include <cstdint>
#include <cuda_fp16.h>

namespace kvq {

// ---------------------------------------------------------------------------------------------
// Quotient x / s, correctly rounded, from a per-row reciprocal.
//
// Markstein's correction (P. Markstein, "Computation of elementary functions on the IBM RISC
// System/6000 processor", IBM J. Res. Dev. 34(1), 1990): with y = RN(1/s) and q0 = RN(x * y)
// (within one ulp of x/s), the remainder r = x - s*q0 is exact in one fused multiply-add and
// q1 = RN(q0 + r*y) is the correctly rounded quotient.  The row's scale s is shared by all its
// elements, so y is computed once per row (__frcp_rn, IEEE round to nearest) and each element
// costs one multiply and two FMAs.  tests/test_gpu_division_exhaustive.py checks q1 against
// IEEE division for every finite fp16 x and every positive fp16 s.
__device__ __forceinline__ float div_by_row_scale(float x, float s, float y) {
  const float q0 = __fmul_rn(x, y);
  const float r = __fmaf_rn(-q0, s, x);
  return __fmaf_rn(r, y, q0);
}

// fp16 row scale fp16_rne(float32(amax) / qmax) without a division instruction: the same
// Markstein step with the constant y = RN(1/qmax) gives the correctly rounded float32 quotient
// for every fp16 amax (checked exhaustively with the quotient above), then one rounding to fp16.
template <int QMAX>
__device__ __forceinline__ float row_scale_f32(float amax) {
  constexpr float y = 1.0f / static_cast<float>(QMAX);  // RN(1/qmax), folded at compile time
  return div_by_row_scale(amax, static_cast<float>(QMAX), y);
}

// Round half to even and bias in one add: for |q| < 2^22, RN(q + 1.5 * 2^23 + bias) has an
// ulp of 1, so its low mantissa bits hold rint(q) + bias (1.5 * 2^23 is even, so ties go to the
// even integer exactly as rint does).  The field is then the low BITS bits of the sum's pattern:
// c + bias for q6/q4, and the int8 two's-complement byte of c for q8 (bias 0).
template <int BIAS>
__device__ __forceinline__ uint32_t rint_biased_bits(float q) {
  return __float_as_uint(__fadd_rn(q, 12582912.0f + static_cast<float>(BIAS)));
}

// One element of the symmetric quantizer: the stored field of clamp(rint(x / s), -QMAX, QMAX)
// (+ BIAS, or the int8 byte for q8), given the row's se = s (1 if s == 0), y = RN(1/s) (0 if
// s == 0) and clip = (s is subnormal in fp16).  For a normal fp16 s = fp16(amax / QMAX) every
// |x| <= amax gives |x / s| <= QMAX * (1 + 2^-10) < QMAX + 1/2, so the clamp can only act on
// rows with a subnormal scale and is skipped elsewhere.
template <int QMAX, int BIAS, int MASK>
__device__ __forceinline__ uint32_t quant_field(float x, float se, float y, bool clip) {
  float q = div_by_row_scale(x, se, y);
  if (clip) q = fminf(fmaxf(q, -static_cast<float>(QMAX)), static_cast<float>(QMAX));
  return rint_biased_bits<BIAS>(q) & static_cast<uint32_t>(MASK);
}

// The same with the clamp decided at compile time: a row with a normal fp16 scale never needs it,
// so a kernel can branch once per row instead of testing per element.
template <int QMAX, int BIAS, int MASK, bool CLIP>
__device__ __forceinline__ uint32_t quant_field_c(float x, float se, float y) {
  float q = div_by_row_scale(x, se, y);
  if constexpr (CLIP) q = fminf(fmaxf(q, -static_cast<float>(QMAX)), static_cast<float>(QMAX));
  return rint_biased_bits<BIAS>(q) & static_cast<uint32_t>(MASK);
}

// Two elements of the quantizer at once without the clamp (rows whose fp16 scale is normal):
// the quotient and the rounding add of quant_field_c<..., false> with Blackwell's packed float32
// instructions (mul/fma/add.rn.f32x2), whose two lanes are each the IEEE float32 operation of the
// scalar path -- four instructions per pair instead of eight.  Returns the two raw sums
// (rint_biased_bits); tests/cuda/division_check.cu compares them with the scalar path for every
// finite fp16 x and positive fp16 s.
__device__ __forceinline__ uint64_t f32x2_of(float lo, float hi) {
  return static_cast<uint64_t>(__float_as_uint(lo)) |
         (static_cast<uint64_t>(__float_as_uint(hi)) << 32);
}

template <int BIAS>
__device__ __forceinline__ uint2 quant_raw2(float xa, float xb, float se, float y) {
  const uint64_t x = f32x2_of(xa, xb), yy = f32x2_of(y, y), ns = f32x2_of(-se, -se);
  constexpr float kMagic = 12582912.0f + static_cast<float>(BIAS);
  const uint64_t mg = f32x2_of(kMagic, kMagic);
  uint64_t q0, r, q1, t;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(q0) : "l"(x), "l"(yy));        // q0 = RN(x * y)
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(q0), "l"(ns), "l"(x));   // x - q0 * s
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(q1) : "l"(r), "l"(yy), "l"(q0));  // q0 + r * y
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(t) : "l"(q1), "l"(mg));           // rint + bias
  return make_uint2(static_cast<uint32_t>(t), static_cast<uint32_t>(t >> 32));
}

// ---------------------------------------------------------------------------------------------
// Packed fields -> exact fp16 codes.  A field u placed in the low mantissa bits of 1024 (fp16
// 0x6400) reads as 1024 + u (or 1024 + 16u / 1024 + 4u when it sits higher); one half2 FMA then
// removes the offset and the bias exactly (every intermediate is a small integer).

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
constexpr uint32_t kHm1056 = 0xE420E420u;    // -1056 = -(1024 + 32)
constexpr uint32_t kHm96 = 0xD600D600u;      // -96   = -(64 + 32)
constexpr uint32_t kHm288 = 0xDC80DC80u;     // -288  = -(256 + 32)
constexpr uint32_t kHm1032 = 0xE408E408u;    // -1032 = -(1024 + 8)
constexpr uint32_t kHm72 = 0xD480D480u;      // -72   = -(64 + 8)
constexpr uint32_t kHm1152 = 0xE480E480u;    // -1152 = -(1024 + 128)

// Eight consecutive elements e0..e7 of a packed row -> four half2 holding the exact signed codes
// {e_k, e_{k+4}}, k = 0..3.  The bytes of the group start at byte 6*GI (q6), word GI (q4) or
// word 2*GI (q8) of `w`.
template <int BITS, int GI>
__device__ __forceinline__ void unpack_group(const uint32_t* w, uint32_t p[4]) {
  if constexpr (BITS == 6) {
    // two 24-bit little-endian quads: fields u0..u3 then u0'..u3'
    constexpr int b = 6 * GI;
    constexpr int w0 = b / 4;
    const uint32_t x = w[w0], y = w[w0 + 1];
    constexpr uint32_t s1 = (b % 4 == 0) ? 0x4310u : 0x6532u;  // bytes [B0 B1 B3 B4]
    constexpr uint32_t s2 = (b % 4 == 0) ? 0x5421u : 0x7643u;  // bytes [B1 B2 B4 B5]
    const uint32_t p1 = prmt(x, y, s1);
    const uint32_t p2 = prmt(x, y, s2);
    p[0] = hfma2u((p1 & 0x003F003Fu) | 0x64006400u, kH1, kHm1056);            // 1024 + u0
    p[1] = hfma2u(((p1 >> 2) & 0x03F003F0u) | 0x64006400u, kH16th, kHm96);     // 1024 + 16 u1
    p[2] = hfma2u((p2 & 0x03F003F0u) | 0x64006400u, kH16th, kHm96);            // 1024 + 16 u2
    p[3] = hfma2u(((p2 >> 8) & 0x00FC00FCu) | 0x64006400u, kHQuarter, kHm288); // 1024 + 4 u3
  } else if constexpr (BITS == 4) {
    // nibble n = element n; nibbles 1 and 5 (3 and 7 after one shift) already sit at mantissa
    // bits 4-7, where they read as 1024 + 16u (scale 1/16), so one shift serves all four pairs
    const uint32_t x = w[GI], y = w[GI] >> 8;
    p[0] = hfma2u((x & 0x000F000Fu) | 0x64006400u, kH1, kHm1032);      // 1024 + u
    p[1] = hfma2u((x & 0x00F000F0u) | 0x64006400u, kH16th, kHm72);     // 1024 + 16 u
    p[2] = hfma2u((y & 0x000F000Fu) | 0x64006400u, kH1, kHm1032);
    p[3] = hfma2u((y & 0x00F000F0u) | 0x64006400u, kH16th, kHm72);
  } else {
    const uint32_t x = w[2 * GI], y = w[2 * GI + 1];  // int8 bytes e0..e3, e4..e7
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint32_t sel = static_cast<uint32_t>(k | (k << 4) | ((4 + k) << 8) | ((4 + k) << 12));
      p[k] = hfma2u((prmt(x, y, sel) & 0x00FF00FFu) ^ 0x64806480u, kH1, kHm1152);
    }
  }
}

// ---------------------------------------------------------------------------------------------
// Symmetric row quantizer: per width the clip bound, field bias and mask, and the packed bytes of
// one 16-element unit.
template <int BITS> struct SymQ;
template <> struct SymQ<8> { static constexpr int kQmax = 127, kBias = 0, kMask = 0xff, kUnitBytes = 16; };
template <> struct SymQ<6> { static constexpr int kQmax = 31, kBias = 32, kMask = 0x3f, kUnitBytes = 12; };
template <> struct SymQ<4> { static constexpr int kQmax = 7, kBias = 8, kMask = 0x0f, kUnitBytes = 8; };


__device__ __forceinline__ __half2 habs2u(uint32_t w) {
  return __habs2(*reinterpret_cast<const __half2*>(&w));
}

__device__ __forceinline__ __half2 absmax8(const uint4& v) {
  return __hmax2(__hmax2(habs2u(v.x), habs2u(v.y)), __hmax2(habs2u(v.z), habs2u(v.w)));
}

// 8 fields (each < 2^BITS) -> packed little-endian bits: q6 two 24-bit words, q4 one word,
// q8 two words.
template <int BITS>
__device__ __forceinline__ void pack8(const uint32_t f[8], uint32_t& a, uint32_t& b) {
  if constexpr (BITS == 6) {
    a = f[0] | (f[1] << 6) | (f[2] << 12) | (f[3] << 18);
    b = f[4] | (f[5] << 6) | (f[6] << 12) | (f[7] << 18);
  } else if constexpr (BITS == 4) {
    a = 0;
#pragma unroll
    for (int k = 0; k < 8; ++k) a |= f[k] << (4 * k);
    b = 0;
  } else {
    a = f[0] | (f[1] << 8) | (f[2] << 16) | (f[3] << 24);
    b = f[4] | (f[5] << 8) | (f[6] << 16) | (f[7] << 24);
  }
}

// Store one unit (16 elements) of packed codes.  With D % 16 == 0 the row stride packed_dim is
// a multiple of 12 / 16 / 8 bytes (q6 / q8 / q4), so a unit is 4- / 16- / 8-byte aligned.
template <int BITS>
__device__ __forceinline__ void store_unit(uint8_t* p, const uint32_t a0, const uint32_t b0,
                                           const uint32_t a1, const uint32_t b1) {
  if constexpr (BITS == 6) {
    // fields 0..7 -> 24-bit words a0, b0; fields 8..15 -> a1, b1; 12 bytes = 3 words
    *reinterpret_cast<uint32_t*>(p) = a0 | (b0 << 24);
    *reinterpret_cast<uint32_t*>(p + 4) = (b0 >> 8) | (a1 << 16);
    *reinterpret_cast<uint32_t*>(p + 8) = (a1 >> 16) | (b1 << 8);
  } else if constexpr (BITS == 4) {
    *reinterpret_cast<uint2*>(p) = make_uint2(a0, a1);
  } else {
    *reinterpret_cast<uint4*>(p) = make_uint4(a0, b0, a1, b1);
  }
}

// ---------------------------------------------------------------------------------------------
// Packing fields from the quantizer's raw rounding sums with integer multiply-adds (the FMA pipe)
// instead of masks and shifts (the integer-logic pipe).
__device__ __forceinline__ uint32_t mad_u32(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t r;
  asm("mad.lo.u32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(c));
  return r;
}

// The quantizer's raw sum RN(q + 1.5 * 2^23 + B): its pattern is kMagic + B + c for the code c
// (every term a small integer), so with B + c in [0, 2^BITS) the field is the pattern minus
// kMagic.  q8 takes B = 128 here (fields c + 128) and flips each byte's top bit after packing.
constexpr uint32_t kMagic = 0x4B400000u;   // bits of 1.5 * 2^23
template <int BITS> constexpr int raw_bias() { return BITS == 8 ? 128 : SymQ<BITS>::kBias; }

template <int QMAX, int B, bool CLIP>
__device__ __forceinline__ uint32_t quant_raw(float x, float se, float y) {
  float q = div_by_row_scale(x, se, y);
  if constexpr (CLIP) q = fminf(fmaxf(q, -static_cast<float>(QMAX)), static_cast<float>(QMAX));
  return rint_biased_bits<B>(q);
}

// 8 raw sums -> the packed fields (pack8's layout): the fields are the digits of a base-2^BITS
// number, so one multiply-add per field builds it from the raw patterns and a constant removes
// the kMagic terms (all arithmetic mod 2^32).
template <int BITS>
__device__ __forceinline__ void pack8_raw(const uint32_t r[8], uint32_t& a, uint32_t& b) {
  if constexpr (BITS == 6) {
    constexpr uint32_t kOff = kMagic * (1u + 64u + 4096u + 262144u);
    a = mad_u32(mad_u32(mad_u32(r[3], 64u, r[2]), 64u, r[1]), 64u, r[0]) - kOff;
    b = mad_u32(mad_u32(mad_u32(r[7], 64u, r[6]), 64u, r[5]), 64u, r[4]) - kOff;
  } else if constexpr (BITS == 4) {
    uint32_t t = r[7];
    uint32_t off = 1u;
#pragma unroll
    for (int k = 6; k >= 0; --k) {
      t = mad_u32(t, 16u, r[k]);
      off = off * 16u + 1u;
    }
    a = t - kMagic * off;
    b = 0;
  } else {
    constexpr uint32_t kOff = kMagic * (1u + 256u + 65536u + 16777216u);
    a = (mad_u32(mad_u32(mad_u32(r[3], 256u, r[2]), 256u, r[1]), 256u, r[0]) - kOff) ^ 0x80808080u;
    b = (mad_u32(mad_u32(mad_u32(r[7], 256u, r[6]), 256u, r[5]), 256u, r[4]) - kOff) ^ 0x80808080u;
  }
}

}  // namespace kvq
