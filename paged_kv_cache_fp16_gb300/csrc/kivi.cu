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
// Keys: one thread per (tensor, b, h, token group, channel pair) walks the group's tokens with the
// pair's values in registers; adjacent threads own adjacent pairs of a row (coalesced rows).
// Values: one thread per (row, channel group) holds the group in 16-byte vectors.  Groups that
// are not a multiple of 8 channels use a scalar kernel.  HBM-bound: 4 bytes per element.
// The data are modified in place, so loads use the coherent path (no ld.global.nc).
#include <cuda_runtime.h>

#include "kvq_device.cuh"
#include "kvq_internal.h"

namespace kvq {
namespace {

constexpr int kThreads = 256;

// Passed by value (kernel parameter space): the library allocates no device memory.
struct KiviArgs {
  uint16_t* x[KVQ_MAX_TENSORS];
  int key_list[KVQ_MAX_TENSORS];  // indices into x of the key tensors
  int val_list[KVQ_MAX_TENSORS];  // indices into x of the value tensors
  int n_keys, n_vals;
  int B, H, S, D, lo, hi, gs;
  float levels, eps;
};

__device__ __forceinline__ void to_f8(const uint4& v, float f[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    f[2 * k] = h2f(static_cast<uint16_t>(w[k] & 0xffffu));
    f[2 * k + 1] = h2f(static_cast<uint16_t>(w[k] >> 16));
  }
}

__device__ __forceinline__ float group_scale(float mn, float mx, float levels, float eps) {
  return fmaxf(__fdiv_rn(__fsub_rn(mx, mn), levels), eps);
}

__device__ __forceinline__ uint16_t roundtrip(float x, float mn, float scale, float levels) {
  const float c = fminf(fmaxf(rintf(__fdiv_rn(__fsub_rn(x, mn), scale)), 0.f), levels);
  return f2h(__fadd_rn(__fmul_rn(c, scale), mn));
}

__device__ __forceinline__ uint4 roundtrip8(const float f[8], const float mn[8],
                                            const float sc[8], float levels) {
  uint32_t w[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    w[k] = static_cast<uint32_t>(roundtrip(f[2 * k], mn[2 * k], sc[2 * k], levels)) |
           (static_cast<uint32_t>(roundtrip(f[2 * k + 1], mn[2 * k + 1], sc[2 * k + 1], levels))
            << 16);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// ------------------------------------------------------------------------------ keys
// One thread per (key tensor, b, h, token group, channel pair): it walks the group's tokens, keeps
// the pair's values in registers (up to kKeepRows tokens; longer groups are read twice), reduces
// min/max per channel without any cross-thread step, and writes the round trip back.  Adjacent
// threads own adjacent channel pairs of the same token row, so every load and store of a row is
// contiguous across the warp.
constexpr int kKeepRows = 32;

__global__ void __launch_bounds__(kThreads) kivi_keys_kernel(const KiviArgs a) {
  const int span = a.hi - a.lo;
  const int n_groups = (span + a.gs - 1) / a.gs;
  const int pairs = a.D / 2;
  const int64_t bh_count = static_cast<int64_t>(a.B) * a.H;
  const int64_t items = static_cast<int64_t>(a.n_keys) * bh_count * n_groups * pairs;
  for (int64_t it = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; it < items;
       it += static_cast<int64_t>(gridDim.x) * kThreads) {
    const int pr = static_cast<int>(it % pairs);
    const int64_t r1 = it / pairs;
    const int g = static_cast<int>(r1 % n_groups);
    const int64_t r2 = r1 / n_groups;
    const int64_t bh = r2 % bh_count;
    const int ti = a.key_list[r2 / bh_count];
    const int t0 = a.lo + g * a.gs;
    const int n = min(a.gs, a.hi - t0);
    uint32_t* base = reinterpret_cast<uint32_t*>(a.x[ti] + (bh * a.S + t0) * a.D) + pr;
    const int stride = a.D / 2;   // in half2 words
    uint32_t keep[kKeepRows];
    // fp16 +-inf as the identities (inputs are finite)
    __half2 mn = __halves2half2(__ushort_as_half(0x7c00), __ushort_as_half(0x7c00));
    __half2 mx = __halves2half2(__ushort_as_half(0xfc00), __ushort_as_half(0xfc00));
#pragma unroll
    for (int r = 0; r < kKeepRows; ++r) {
      keep[r] = 0;
      if (r < n) {
        keep[r] = base[static_cast<int64_t>(r) * stride];
        const __half2 v = *reinterpret_cast<const __half2*>(&keep[r]);
        mn = __hmin2(mn, v);
        mx = __hmax2(mx, v);
      }
    }
    for (int r = kKeepRows; r < n; ++r) {
      const uint32_t w = base[static_cast<int64_t>(r) * stride];
      const __half2 v = *reinterpret_cast<const __half2*>(&w);
      mn = __hmin2(mn, v);
      mx = __hmax2(mx, v);
    }
    // fp16 min/max are exact; the group arithmetic is float32
    const float mn0 = __low2float(mn), mn1 = __high2float(mn);
    const float sc0 = group_scale(mn0, __low2float(mx), a.levels, a.eps);
    const float sc1 = group_scale(mn1, __high2float(mx), a.levels, a.eps);
    auto rt = [&](uint32_t w) -> uint32_t {
      const uint32_t lo = roundtrip(h2f(static_cast<uint16_t>(w & 0xffffu)), mn0, sc0, a.levels);
      const uint32_t hi = roundtrip(h2f(static_cast<uint16_t>(w >> 16)), mn1, sc1, a.levels);
      return lo | (hi << 16);
    };
#pragma unroll
    for (int r = 0; r < kKeepRows; ++r)
      if (r < n) base[static_cast<int64_t>(r) * stride] = rt(keep[r]);
    for (int r = kKeepRows; r < n; ++r)
      base[static_cast<int64_t>(r) * stride] = rt(base[static_cast<int64_t>(r) * stride]);
  }
}

// ------------------------------------------------------------------------------ values
// One thread per (value tensor, row, channel group) for groups of a multiple of 8 channels
// (16-byte vectors, at most 64 channels held in registers); the group's min/max, scale and round
// trip stay in the thread.
constexpr int kMaxVecs = 8;

__global__ void __launch_bounds__(kThreads) kivi_values_kernel(const KiviArgs a) {
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
    const int c0 = g * a.gs;
    const int nv = (min(a.D, c0 + a.gs) - c0) / 8;   // 16-byte vectors in this group
    uint4* p = reinterpret_cast<uint4*>(a.x[a.val_list[vi]] + (bh * a.S + t) * a.D + c0);
    uint4 v[kMaxVecs];
    __half2 mn = __halves2half2(__ushort_as_half(0x7c00), __ushort_as_half(0x7c00));
    __half2 mx = __halves2half2(__ushort_as_half(0xfc00), __ushort_as_half(0xfc00));
#pragma unroll
    for (int k = 0; k < kMaxVecs; ++k) {
      v[k] = make_uint4(0, 0, 0, 0);
      if (k < nv) {
        v[k] = p[k];
        const uint32_t w[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const __half2 h = *reinterpret_cast<const __half2*>(&w[e]);
          mn = __hmin2(mn, h);
          mx = __hmax2(mx, h);
        }
      }
    }
    const float mnf = fminf(__low2float(mn), __high2float(mn));
    const float sc = group_scale(mnf, fmaxf(__low2float(mx), __high2float(mx)), a.levels, a.eps);
#pragma unroll
    for (int k = 0; k < kMaxVecs; ++k) {
      if (k >= nv) continue;
      float f[8], mn8[8], sc8[8];
      to_f8(v[k], f);
#pragma unroll
      for (int e = 0; e < 8; ++e) { mn8[e] = mnf; sc8[e] = sc; }
      p[k] = roundtrip8(f, mn8, sc8, a.levels);
    }
  }
}

// Any group size: one thread per (row, channel group), scalar loads.
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
    const float sc = group_scale(mn, mx, a.levels, a.eps);
    for (int c = c0; c < c1; ++c) p[c] = roundtrip(h2f(p[c]), mn, sc, a.levels);
  }
}


int grid_cap() {
  const int sms = sm_count();
  return (sms > 0 ? sms : 1) * (2048 / kThreads);
}

int blocks_for_threads(int64_t threads) {
  int64_t b = (threads + kThreads - 1) / kThreads;
  const int cap = grid_cap();
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
  if (a.n_keys > 0) {
    const int64_t items = static_cast<int64_t>(a.n_keys) * B * H *
                          ((span + group_size - 1) / group_size) * (D / 2);
    kivi_keys_kernel<<<blocks_for_threads(items), kThreads, 0, st>>>(a);
  }
  if (a.n_vals > 0) {
    const int64_t rows = static_cast<int64_t>(a.n_vals) * B * H * span;
    const int64_t items = rows * ((D + group_size - 1) / group_size);
    if (group_size % 8 == 0 && group_size <= 8 * kMaxVecs)
      kivi_values_kernel<<<blocks_for_threads(items), kThreads, 0, st>>>(a);
    else
      kivi_values_scalar_kernel<<<blocks_for_threads(items), kThreads, 0, st>>>(a);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(KVQ_ERR_CUDA, "kivi launch: %s", cudaGetErrorString(e));
  return ok();
}
