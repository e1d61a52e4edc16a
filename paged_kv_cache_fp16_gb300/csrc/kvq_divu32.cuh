// Division of 32-bit unsigned integers by a divisor fixed for a launch, used to split flat
// work-item indices without 64-bit division.
#pragma once

#include <cstdint>

namespace kvq {

// Division of 32-bit unsigned integers by an invariant divisor d >= 1 with one multiply-high and
// shifts (T. Granlund and P. L. Montgomery, "Division by invariant integers using
// multiplication", PLDI 1994, the unsigned N-bit method): with l = ceil(log2 d) and
// m = floor(2^32 (2^l - d) / d) + 1, q = (t + ((n - t) >> min(l, 1))) >> max(l - 1, 0) for
// t = mulhi(m, n) is floor(n / d) for every 32-bit n.
struct DivU32 {
  uint32_t m, s1, s2;
};

inline DivU32 make_divu32(uint32_t d) {
  uint32_t l = 0;
  while ((1ull << l) < d) ++l;
  DivU32 r;
  r.m = static_cast<uint32_t>(((1ull << 32) * ((1ull << l) - d)) / d + 1);
  r.s1 = l < 1 ? l : 1;
  r.s2 = l > 1 ? l - 1 : 0;
  return r;
}

__device__ __forceinline__ uint32_t divu32(uint32_t n, const DivU32& f) {
  const uint32_t t = __umulhi(n, f.m);
  return (t + ((n - t) >> f.s1)) >> f.s2;
}

}  // namespace kvq
