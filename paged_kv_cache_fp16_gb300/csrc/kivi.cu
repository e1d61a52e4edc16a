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
// Keys: one warp per (tensor, b, h, token group); each lane owns a 16-byte chunk of 8 channels,
// a group's rows are spread over the warp, per-channel min/max are reduced across the lanes that
// share a chunk, and the tile is kept in registers between the two passes when it fits.
// Values: each lane owns a chunk of one row; channel groups made of a power-of-two number of
// whole chunks reduce with a segmented shuffle.  Other group sizes use a scalar kernel with one
// thread per (row, channel group).  All of this is HBM-bound: 4 bytes per element (read + write).
// The data are modified in place, so loads use the coherent path (no ld.global.nc).
#include <cuda_runtime.h>

#include "kvq_device.cuh"
#include "kvq_internal.h"

namespace kvq {
namespace {

constexpr int kThreads = 256;
constexpr int kKeepChunks = 8;  // per-lane register cache for the key tile (8 x 16 B)

// Passed by value (kernel parameter space): the library allocates no device memory.
struct KiviArgs {
  uint16_t* x[KVQ_MAX_TENSORS];
  int key_list[KVQ_MAX_TENSORS];  // indices into x of the key tensors
  int val_list[KVQ_MAX_TENSORS];  // indices into x of the value tensors
  int n_keys, n_vals;
  int B, H, S, D, lo, hi, gs, chunks, lpr_log2;
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
// Work item: (key tensor index among the call's tensors, b, h, group g).
__global__ void __launch_bounds__(kThreads) kivi_keys_kernel(const KiviArgs a) {
  const int lane = threadIdx.x & 31;
  const int lpr = 1 << a.lpr_log2;
  const int rps = 32 >> a.lpr_log2;
  const int chunk = lane & (lpr - 1);
  const int sub = lane >> a.lpr_log2;
  const bool lane_on = chunk < a.chunks;
  const int span = a.hi - a.lo;
  const int n_groups = (span + a.gs - 1) / a.gs;
  const int64_t items = static_cast<int64_t>(a.n_keys) * a.B * a.H * n_groups;
  const int64_t warp = (static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x) >> 5;
  const int64_t n_warps = (static_cast<int64_t>(gridDim.x) * kThreads) >> 5;

  for (int64_t it = warp; it < items; it += n_warps) {
    const int g = static_cast<int>(it % n_groups);
    const int64_t bh_all = it / n_groups;
    const int bh = static_cast<int>(bh_all % (static_cast<int64_t>(a.B) * a.H));
    const int ti = a.key_list[bh_all / (static_cast<int64_t>(a.B) * a.H)];
    const int t0 = a.lo + g * a.gs;
    const int n = min(a.gs, a.hi - t0);
    uint16_t* base = a.x[ti] + (static_cast<int64_t>(bh) * a.S + t0) * a.D + chunk * 8;
    const int steps = (n + rps - 1) / rps;

    float mn[8], mx[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) { mn[k] = __int_as_float(0x7f800000); mx[k] = -mn[k]; }
    uint4 keep[kKeepChunks];
#pragma unroll
    for (int j = 0; j < kKeepChunks; ++j) keep[j] = make_uint4(0, 0, 0, 0);
    for (int j = 0; j < steps; ++j) {
      const int row = j * rps + sub;
      if (lane_on && row < n) {
        const uint4 v = *reinterpret_cast<const uint4*>(base + static_cast<int64_t>(row) * a.D);
        float f[8];
        to_f8(v, f);
#pragma unroll
        for (int k = 0; k < 8; ++k) { mn[k] = fminf(mn[k], f[k]); mx[k] = fmaxf(mx[k], f[k]); }
#pragma unroll
        for (int q = 0; q < kKeepChunks; ++q) if (q == j) keep[q] = v;
      }
    }
    // lanes sharing a chunk differ in the bits above lpr_log2
    for (int o = lpr; o < 32; o <<= 1) {
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        mn[k] = fminf(mn[k], __shfl_xor_sync(kFullMask, mn[k], o));
        mx[k] = fmaxf(mx[k], __shfl_xor_sync(kFullMask, mx[k], o));
      }
    }
    float sc[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) sc[k] = group_scale(mn[k], mx[k], a.levels, a.eps);
    if (!lane_on) continue;
    for (int j = 0; j < steps; ++j) {
      const int row = j * rps + sub;
      if (row >= n) continue;
      uint4 v;
      if (j < kKeepChunks) {
        v = keep[0];
#pragma unroll
        for (int q = 1; q < kKeepChunks; ++q) if (q == j) v = keep[q];
      } else {
        v = *reinterpret_cast<const uint4*>(base + static_cast<int64_t>(row) * a.D);
      }
      float f[8];
      to_f8(v, f);
      *reinterpret_cast<uint4*>(base + static_cast<int64_t>(row) * a.D) =
          roundtrip8(f, mn, sc, a.levels);
    }
  }
}

// ------------------------------------------------------------------------------ values
// One lane per 16-byte chunk of a row; channel groups of (1 << glog2) chunks starting at
// channel 0.  Work item: one warp step of rows over all value tensors.
__global__ void __launch_bounds__(kThreads) kivi_values_kernel(const KiviArgs a, int glog2) {
  const int lane = threadIdx.x & 31;
  const int lpr = 1 << a.lpr_log2;
  const int rps = 32 >> a.lpr_log2;
  const int chunk = lane & (lpr - 1);
  const int sub = lane >> a.lpr_log2;
  const int span = a.hi - a.lo;
  const int64_t rows_per_tensor = static_cast<int64_t>(a.B) * a.H * span;
  const int64_t total_rows = rows_per_tensor * a.n_vals;
  const int64_t n_steps = (total_rows + rps - 1) / rps;
  const int64_t warp = (static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x) >> 5;
  const int64_t n_warps = (static_cast<int64_t>(gridDim.x) * kThreads) >> 5;
  const int gl = 1 << glog2;

  for (int64_t st = warp; st < n_steps; st += n_warps) {
    const int64_t row = st * rps + sub;
    const bool on = row < total_rows && chunk < a.chunks;
    uint16_t* p = nullptr;
    float f[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) f[k] = 0.f;
    float mn = __int_as_float(0x7f800000), mx = -mn;
    if (on) {
      const int64_t vi = row / rows_per_tensor;
      const int64_t r = row - vi * rows_per_tensor;
      const int64_t bh = r / span;
      const int t = a.lo + static_cast<int>(r - bh * span);
      p = a.x[a.val_list[vi]] + (bh * a.S + t) * a.D + chunk * 8;
      to_f8(*reinterpret_cast<const uint4*>(p), f);
#pragma unroll
      for (int k = 0; k < 8; ++k) { mn = fminf(mn, f[k]); mx = fmaxf(mx, f[k]); }
    }
    for (int o = 1; o < gl; o <<= 1) {
      mn = fminf(mn, __shfl_xor_sync(kFullMask, mn, o));
      mx = fmaxf(mx, __shfl_xor_sync(kFullMask, mx, o));
    }
    if (!on) continue;
    const float sc = group_scale(mn, mx, a.levels, a.eps);
    float mn8[8], sc8[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) { mn8[k] = mn; sc8[k] = sc; }
    *reinterpret_cast<uint4*>(p) = roundtrip8(f, mn8, sc8, a.levels);
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

int ceil_log2(int v) {
  int l = 0;
  while ((1 << l) < v) ++l;
  return l;
}

int grid_cap() {
  const int sms = sm_count();
  return (sms > 0 ? sms : 1) * (2048 / kThreads);
}

int blocks_for_warps(int64_t warps) {
  int64_t b = (warps + (kThreads / 32) - 1) / (kThreads / 32);
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
  a.chunks = D / 8;
  a.lpr_log2 = ceil_log2(a.chunks);
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
    const int64_t items = static_cast<int64_t>(a.n_keys) * B * H * ((span + group_size - 1) / group_size);
    kivi_keys_kernel<<<blocks_for_warps(items), kThreads, 0, st>>>(a);
  }
  if (a.n_vals > 0) {
    // fast path: a group is a power-of-two number of whole 16-byte chunks (or the whole row)
    int glog2 = -1;
    const int lpr = 1 << a.lpr_log2;
    if (group_size >= lpr * 8) {
      glog2 = a.lpr_log2;
    } else if (group_size % 8 == 0 && (group_size / 8 & (group_size / 8 - 1)) == 0) {
      glog2 = ceil_log2(group_size / 8);
    }
    const int64_t rows = static_cast<int64_t>(a.n_vals) * B * H * span;
    if (glog2 >= 0) {
      const int rps = 32 >> a.lpr_log2;
      kivi_values_kernel<<<blocks_for_warps((rows + rps - 1) / rps), kThreads, 0, st>>>(a, glog2);
    } else {
      const int64_t items = rows * ((D + group_size - 1) / group_size);
      kivi_values_scalar_kernel<<<blocks_for_warps((items + 31) / 32), kThreads, 0, st>>>(a);
    }
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(KVQ_ERR_CUDA, "kivi launch: %s", cudaGetErrorString(e));
  return ok();
}
