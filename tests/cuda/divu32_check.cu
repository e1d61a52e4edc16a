// Check of the library's division by an invariant divisor (test only).
//
// kvq_divu32.cuh divides 32-bit unsigned integers by a divisor fixed for a launch with one
// multiply-high and shifts (Granlund and Montgomery's unsigned method); the kernels use it to
// split flat work-item and row indices.  This compares it with the integer division n / d:
//   (1) every n in [0, 2^32) for a set of divisors (the small ones the kernels meet -- head
//       counts, page sizes, tokens per work item -- powers of two and their neighbours, and the
//       largest 32-bit divisors);
//   (2) every divisor in [1, 65536] on numerators around each multiple scale: k d - 1, k d and
//       k d + d - 1 for k = floor((2^32 - 1) / d) >> j, j = 0 .. 31, and 0 .. 255.
#include <cstdint>
#include <cuda_runtime.h>

#include "kvq_divu32.cuh"

namespace {

__global__ void all_numerators(const kvq::DivU32* f, const uint32_t* d, int nd,
                               unsigned long long* bad) {
  const unsigned long long n_all = 1ull << 32;
  for (int k = 0; k < nd; ++k) {
    unsigned long long nb = 0;
    for (unsigned long long i = blockIdx.x * (unsigned long long)blockDim.x + threadIdx.x;
         i < n_all; i += (unsigned long long)gridDim.x * blockDim.x) {
      const uint32_t n = static_cast<uint32_t>(i);
      if (kvq::divu32(n, f[k]) != n / d[k]) ++nb;
    }
    if (nb) atomicAdd(bad, nb);
  }
}

__global__ void all_small_divisors(const kvq::DivU32* f, unsigned long long* bad) {
  const uint32_t d = blockIdx.x + 1;   // 1 .. 65536
  const kvq::DivU32 fd = f[blockIdx.x];
  unsigned long long nb = 0;
  const uint32_t kmax = 0xffffffffu / d;
  for (int t = threadIdx.x; t < 32 * 3 + 256; t += blockDim.x) {
    uint32_t n;
    if (t < 96) {
      const uint32_t k = kmax >> (t / 3);
      const uint64_t base = static_cast<uint64_t>(k) * d;
      const uint64_t v = (t % 3 == 0) ? (base ? base - 1 : 0) : (t % 3 == 1 ? base : base + d - 1);
      n = static_cast<uint32_t>(v > 0xffffffffull ? 0xffffffffull : v);
    } else {
      n = static_cast<uint32_t>(t - 96);
    }
    if (kvq::divu32(n, fd) != n / d) ++nb;
  }
  if (nb) atomicAdd(bad + 1, nb);
}

}  // namespace

extern "C" int run_divu32_check(unsigned long long* bad_out) {
  const uint32_t ds[] = {1u, 2u, 3u, 4u, 5u, 6u, 7u, 8u, 9u, 12u, 15u, 16u, 17u, 24u, 31u, 32u,
                         33u, 64u, 100u, 128u, 255u, 256u, 1000u, 4096u, 65535u, 65536u, 65537u,
                         262143u, 262144u, 1000003u, 0x7fffffffu, 0x80000000u, 0x80000001u,
                         0xfffffffeu, 0xffffffffu};
  const int nd = static_cast<int>(sizeof(ds) / sizeof(ds[0]));
  kvq::DivU32 fs[sizeof(ds) / sizeof(ds[0])];
  for (int i = 0; i < nd; ++i) fs[i] = kvq::make_divu32(ds[i]);
  kvq::DivU32* small = new kvq::DivU32[65536];
  for (uint32_t d = 1; d <= 65536; ++d) small[d - 1] = kvq::make_divu32(d);

  kvq::DivU32 *d_fs = nullptr, *d_small = nullptr;
  uint32_t* d_ds = nullptr;
  unsigned long long* d_bad = nullptr;
  int rc = 0;
  if (cudaMalloc(&d_fs, sizeof(fs)) != cudaSuccess ||
      cudaMalloc(&d_ds, sizeof(ds)) != cudaSuccess ||
      cudaMalloc(&d_small, 65536 * sizeof(kvq::DivU32)) != cudaSuccess ||
      cudaMalloc(&d_bad, 2 * sizeof(unsigned long long)) != cudaSuccess) {
    rc = 1;
  } else {
    cudaMemcpy(d_fs, fs, sizeof(fs), cudaMemcpyHostToDevice);
    cudaMemcpy(d_ds, ds, sizeof(ds), cudaMemcpyHostToDevice);
    cudaMemcpy(d_small, small, 65536 * sizeof(kvq::DivU32), cudaMemcpyHostToDevice);
    cudaMemset(d_bad, 0, 2 * sizeof(unsigned long long));
    all_numerators<<<152 * 8, 256>>>(d_fs, d_ds, nd, d_bad);
    all_small_divisors<<<65536, 128>>>(d_small, d_bad);
    if (cudaDeviceSynchronize() != cudaSuccess) rc = 2;
    cudaMemcpy(bad_out, d_bad, 2 * sizeof(unsigned long long), cudaMemcpyDeviceToHost);
  }
  cudaFree(d_fs);
  cudaFree(d_ds);
  cudaFree(d_small);
  cudaFree(d_bad);
  delete[] small;
  return rc;
}
