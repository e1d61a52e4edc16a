// Exhaustive check of the quantizer's per-element arithmetic (test only).
//
// For every finite fp16 x and every positive finite fp16 scale s it compares
//   (1) the per-row-reciprocal quotient (Markstein correction) with IEEE float32 division,
//   (2) the stored field of q8/q6/q4 with clamp(rint_half_even(x / s), -qmax, qmax) + bias computed
//       from IEEE division, on the inputs the quantizer can see: all x when s is subnormal, and
//       |x| <= qmax * s * (1 + 2^-9) when s is normal (a superset of |x| <= amax, since
//       s = fp16(amax / qmax)), and
//   (3) the division-free row scale amax / qmax with IEEE division for every fp16 amax.
#include <cstdint>
#include <cstdio>
#include <cuda_runtime.h>
#include <cuda_fp16.h>

#include "kvq_math.cuh"

namespace {

template <int QMAX, int BIAS, int MASK>
__device__ bool field_ok(float x, float s, float ref_q, float se, float y, bool clip) {
  if (s >= 6.103515625e-05f && fabsf(x) > static_cast<float>(QMAX) * s * (1.0f + 1.0f / 512.0f))
    return true;  // unreachable pair
  const float c = fminf(fmaxf(rintf(ref_q), -static_cast<float>(QMAX)), static_cast<float>(QMAX));
  const uint32_t want = static_cast<uint32_t>(static_cast<int>(c) + BIAS) & MASK;
  return kvq::quant_field<QMAX, BIAS, MASK>(x, se, y, clip) == want;
}

__global__ void check_kernel(unsigned long long* bad) {
  const unsigned long long n = 65536ull * 0x7BFFull;  // x: all 16-bit patterns, s: 0x0001..0x7BFF
  unsigned long long nq = 0, n8 = 0, n6 = 0, n4 = 0;
  for (unsigned long long i = blockIdx.x * (unsigned long long)blockDim.x + threadIdx.x; i < n;
       i += (unsigned long long)gridDim.x * blockDim.x) {
    const uint16_t xb = static_cast<uint16_t>(i & 0xffff);
    if ((xb & 0x7c00) == 0x7c00) continue;  // inf / nan
    const uint16_t sb = static_cast<uint16_t>(1 + (i >> 16));
    const float x = __half2float(__ushort_as_half(xb));
    const float s = __half2float(__ushort_as_half(sb));
    const float y = __frcp_rn(s);
    const float ref = __fdiv_rn(x, s);
    if (kvq::div_by_row_scale(x, s, y) != ref) ++nq;
    // the packed two-element path equals the scalar raw sums (biases of q8 / q6 / q4)
    {
      const uint2 p0 = kvq::quant_raw2<0>(x, -x, s, y), p32 = kvq::quant_raw2<32>(x, -x, s, y);
      const uint2 p8 = kvq::quant_raw2<8>(x, -x, s, y);
      const float qa = kvq::div_by_row_scale(x, s, y), qb = kvq::div_by_row_scale(-x, s, y);
      if (p0.x != kvq::rint_biased_bits<0>(qa) || p0.y != kvq::rint_biased_bits<0>(qb) ||
          p32.x != kvq::rint_biased_bits<32>(qa) || p32.y != kvq::rint_biased_bits<32>(qb) ||
          p8.x != kvq::rint_biased_bits<8>(qa) || p8.y != kvq::rint_biased_bits<8>(qb))
        ++nq;
    }
    const bool clip = s < 6.103515625e-05f;
    if (!field_ok<127, 0, 0xff>(x, s, ref, s, y, clip)) ++n8;
    if (!field_ok<31, 32, 0x3f>(x, s, ref, s, y, clip)) ++n6;
    if (!field_ok<7, 8, 0x0f>(x, s, ref, s, y, clip)) ++n4;
  }
  if (nq) atomicAdd(bad + 0, nq);
  if (n8) atomicAdd(bad + 1, n8);
  if (n6) atomicAdd(bad + 2, n6);
  if (n4) atomicAdd(bad + 3, n4);
}

__global__ void scale_kernel(unsigned long long* bad) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;   // all positive finite fp16 amax
  if (i < 1 || i > 0x7BFF) return;
  const float amax = __half2float(__ushort_as_half(static_cast<uint16_t>(i)));
  if (kvq::row_scale_f32<127>(amax) != __fdiv_rn(amax, 127.f)) atomicAdd(bad + 4, 1ull);
  if (kvq::row_scale_f32<31>(amax) != __fdiv_rn(amax, 31.f)) atomicAdd(bad + 4, 1ull);
  if (kvq::row_scale_f32<7>(amax) != __fdiv_rn(amax, 7.f)) atomicAdd(bad + 4, 1ull);
}

}  // namespace

extern "C" int run_division_check(unsigned long long* host_bad) {
  unsigned long long* d = nullptr;
  if (cudaMalloc(&d, 5 * sizeof(unsigned long long)) != cudaSuccess) return 1;
  cudaMemset(d, 0, 5 * sizeof(unsigned long long));
  check_kernel<<<4096, 256>>>(d);
  scale_kernel<<<(0x7C00 + 255) / 256, 256>>>(d);
  cudaError_t e = cudaDeviceSynchronize();
  if (e == cudaSuccess) e = cudaMemcpy(host_bad, d, 5 * sizeof(unsigned long long),
                                       cudaMemcpyDeviceToHost);
  cudaFree(d);
  return e == cudaSuccess ? 0 : 2;
}
