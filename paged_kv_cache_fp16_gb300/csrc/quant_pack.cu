// Symmetric per-token-per-head quantize + pack into pages, and the inverse gather + dequantize.
//
// MTPLX pull request #267, "feat(kv-cache): add q6 paged KV quantization", description: one fp16
// scale per (token, KV head) row, qmax 127/31/7 (bit-width table paragraph), q6 codes biased by
// +32 and packed four per three bytes little-endian (byte-layout formula), packed_dim(D, 6) =
// 3D/4.  The q6 pack is written here as one 24-bit little-endian word per four fields,
// w = u0 | u1 << 6 | u2 << 12 | u3 << 18, whose three bytes are exactly the page's byte0..2.
//
// Thread layout: each lane owns one 16-byte chunk (8 elements) of a row; a row spans
// next_pow2(D/8) lanes, so a warp covers 32 / that rows per step.  Loads and stores of a row
// are contiguous across its lanes (coalesced), the row max is a segmented warp-shuffle
// reduction, and codes are packed in registers.  Persistent grid, several steps in flight per
// warp.  The work is HBM-bound: per row 2D bytes in, packed_dim + 2 bytes out.
#include <cuda_runtime.h>

#include "kvq_device.cuh"
#include "kvq_internal.h"

namespace kvq {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;

struct PackArgs {
  const uint16_t* x[KVQ_MAX_TENSORS];  // quant: inputs; dequant: outputs (cast back)
  PoolRef pool[KVQ_MAX_TENSORS];
  const int32_t* page_table;
  const int32_t* cu;
  const int32_t* start;
  int32_t* err;
  int64_t rows_per_tensor;  // total_tokens * H
  int n_tensors, H, D, page_size, pd, max_pages, nseq;
  int lpr_log2;             // lanes per row = 1 << lpr_log2
  int chunks;               // D / 8
};

template <int BITS> struct Q;
template <> struct Q<8> { static constexpr int kQmax = 127; static constexpr int kBias = 0; };
template <> struct Q<6> { static constexpr int kQmax = 31; static constexpr int kBias = 32; };
template <> struct Q<4> { static constexpr int kQmax = 7; static constexpr int kBias = 8; };

__device__ __forceinline__ void unpack_half8(const uint4& v, float f[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    f[2 * k] = h2f(static_cast<uint16_t>(w[k] & 0xffffu));
    f[2 * k + 1] = h2f(static_cast<uint16_t>(w[k] >> 16));
  }
}

// Row address data shared by quant and dequant: the physical row, or -1.
__device__ __forceinline__ int64_t row_target(const PackArgs& a, int t, int64_t r) {
  const int token = static_cast<int>(r / a.H);
  const int h = static_cast<int>(r - static_cast<int64_t>(token) * a.H);
  const int s = find_seq(a.cu, a.nseq, token);
  const int64_t pos = static_cast<int64_t>(__ldg(a.start + s)) + (token - __ldg(a.cu + s));
  return locate_row(a.page_table, a.max_pages, a.page_size, a.H, a.pool[t].num_pages, s, pos, h,
                    a.err);
}

// Store 8 packed codes of one chunk.  `m` = row * chunks + chunk indexes the chunk's byte
// position m * (8 * BITS / 8) within the pool's code array.
template <int BITS>
__device__ __forceinline__ void store_codes(uint8_t* codes, int64_t m, const int c[8]) {
  if constexpr (BITS == 8) {
    uint32_t w0 = 0, w1 = 0;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      w0 |= (static_cast<uint32_t>(c[k]) & 0xffu) << (8 * k);
      w1 |= (static_cast<uint32_t>(c[k + 4]) & 0xffu) << (8 * k);
    }
    *reinterpret_cast<uint2*>(codes + m * 8) = make_uint2(w0, w1);
  } else if constexpr (BITS == 4) {
    uint32_t w = 0;
#pragma unroll
    for (int k = 0; k < 8; ++k) w |= static_cast<uint32_t>(c[k] + Q<4>::kBias) << (4 * k);
    *reinterpret_cast<uint32_t*>(codes + m * 4) = w;
  } else {
    uint32_t w0 = 0, w1 = 0;  // two 24-bit little-endian words
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      w0 |= static_cast<uint32_t>(c[k] + Q<6>::kBias) << (6 * k);
      w1 |= static_cast<uint32_t>(c[k + 4] + Q<6>::kBias) << (6 * k);
    }
    const uint32_t lo = w0 | (w1 << 24);   // bytes 0..3
    const uint16_t hi = static_cast<uint16_t>(w1 >> 8);  // bytes 4..5
    uint8_t* p = codes + m * 6;
    if ((m & 1) == 0) {  // 6m % 4 == 0
      *reinterpret_cast<uint32_t*>(p) = lo;
      *reinterpret_cast<uint16_t*>(p + 4) = hi;
    } else {             // 6m % 4 == 2
      *reinterpret_cast<uint16_t*>(p) = static_cast<uint16_t>(lo & 0xffffu);
      *reinterpret_cast<uint32_t*>(p + 2) = (lo >> 16) | (static_cast<uint32_t>(hi) << 16);
    }
  }
}

template <int BITS>
__device__ __forceinline__ void load_codes(const uint8_t* codes, int64_t m, int c[8]) {
  if constexpr (BITS == 8) {
    const uint2 w = ld_nc_v2(codes + m * 8);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      c[k] = static_cast<int>(static_cast<int8_t>((w.x >> (8 * k)) & 0xffu));
      c[k + 4] = static_cast<int>(static_cast<int8_t>((w.y >> (8 * k)) & 0xffu));
    }
  } else if constexpr (BITS == 4) {
    const uint32_t w = ld_nc_u32(codes + m * 4);
#pragma unroll
    for (int k = 0; k < 8; ++k) c[k] = static_cast<int>((w >> (4 * k)) & 0xfu) - Q<4>::kBias;
  } else {
    const uint8_t* p = codes + m * 6;
    uint32_t lo, hi;
    if ((m & 1) == 0) {
      lo = ld_nc_u32(p);
      hi = ld_nc_u16(p + 4);
    } else {
      const uint32_t a = ld_nc_u16(p), b = ld_nc_u32(p + 2);
      lo = a | (b << 16);
      hi = b >> 16;
    }
    const uint32_t w0 = lo & 0xffffffu;
    const uint32_t w1 = (lo >> 24) | (hi << 8);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      c[k] = static_cast<int>((w0 >> (6 * k)) & 63u) - Q<6>::kBias;
      c[k + 4] = static_cast<int>((w1 >> (6 * k)) & 63u) - Q<6>::kBias;
    }
  }
}

template <int BITS>
__global__ void __launch_bounds__(kThreads) quant_pack_kernel(const PackArgs a) {
  constexpr float kQ = static_cast<float>(Q<BITS>::kQmax);
  const int lane = threadIdx.x & 31;
  const int lpr = 1 << a.lpr_log2;
  const int rps = 32 >> a.lpr_log2;
  const int chunk = lane & (lpr - 1);
  const int sub = lane >> a.lpr_log2;
  const int64_t total_rows = static_cast<int64_t>(a.n_tensors) * a.rows_per_tensor;
  const int64_t n_steps = (total_rows + rps - 1) / rps;
  const int64_t warp = (static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x) >> 5;
  const int64_t n_warps = (static_cast<int64_t>(gridDim.x) * kThreads) >> 5;

  for (int64_t step0 = warp * kUnroll; step0 < n_steps; step0 += n_warps * kUnroll) {
    uint4 v[kUnroll];
    int64_t row[kUnroll];
    bool act[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      row[u] = (step0 + u) * rps + sub;
      act[u] = row[u] < total_rows && chunk < a.chunks;
      v[u] = make_uint4(0, 0, 0, 0);
      if (act[u]) {
        const int t = static_cast<int>(row[u] / a.rows_per_tensor);
        const int64_t r = row[u] - static_cast<int64_t>(t) * a.rows_per_tensor;
        v[u] = ld_stream_v4(a.x[t] + r * a.D + chunk * 8);
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      float f[8];
      unpack_half8(v[u], f);
      float amax = 0.f;
#pragma unroll
      for (int k = 0; k < 8; ++k) amax = fmaxf(amax, fabsf(f[k]));
      for (int o = lpr >> 1; o >= 1; o >>= 1)
        amax = fmaxf(amax, __shfl_xor_sync(kFullMask, amax, o));
      if (!act[u]) continue;
      const int t = static_cast<int>(row[u] / a.rows_per_tensor);
      const int64_t r = row[u] - static_cast<int64_t>(t) * a.rows_per_tensor;
      const int64_t prow = row_target(a, t, r);
      if (prow < 0) continue;
      const uint16_t sbits = f2h(__fdiv_rn(amax, kQ));
      const float s = h2f(sbits);
      int c[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        float q = 0.f;
        if (s != 0.f) q = fminf(fmaxf(rintf(__fdiv_rn(f[k], s)), -kQ), kQ);
        c[k] = static_cast<int>(q);
      }
      store_codes<BITS>(a.pool[t].codes, prow * a.chunks + chunk, c);
      if (chunk == 0) a.pool[t].scales[prow] = sbits;
    }
  }
}

template <int BITS>
__global__ void __launch_bounds__(kThreads) dequant_kernel(const PackArgs a) {
  const int lane = threadIdx.x & 31;
  const int lpr = 1 << a.lpr_log2;
  const int rps = 32 >> a.lpr_log2;
  const int chunk = lane & (lpr - 1);
  const int sub = lane >> a.lpr_log2;
  const int64_t total_rows = static_cast<int64_t>(a.n_tensors) * a.rows_per_tensor;
  const int64_t n_steps = (total_rows + rps - 1) / rps;
  const int64_t warp = (static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x) >> 5;
  const int64_t n_warps = (static_cast<int64_t>(gridDim.x) * kThreads) >> 5;

  for (int64_t step0 = warp * kUnroll; step0 < n_steps; step0 += n_warps * kUnroll) {
    int c[kUnroll][8];
    float s[kUnroll];
    int64_t dst[kUnroll];   // element offset of the output chunk, or -1
    int tt[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t row = (step0 + u) * rps + sub;
      dst[u] = -1;
      tt[u] = 0;
      s[u] = 0.f;
#pragma unroll
      for (int k = 0; k < 8; ++k) c[u][k] = 0;
      if (row < total_rows && chunk < a.chunks) {
        const int t = static_cast<int>(row / a.rows_per_tensor);
        const int64_t r = row - static_cast<int64_t>(t) * a.rows_per_tensor;
        const int64_t prow = row_target(a, t, r);
        if (prow >= 0) {
          load_codes<BITS>(a.pool[t].codes, prow * a.chunks + chunk, c[u]);
          s[u] = h2f(ld_nc_u16(a.pool[t].scales + prow));
          dst[u] = r * a.D + chunk * 8;
          tt[u] = t;
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      if (dst[u] < 0) continue;
      uint32_t w[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint32_t lo = f2h(__fmul_rn(static_cast<float>(c[u][2 * k]), s[u]));
        const uint32_t hi = f2h(__fmul_rn(static_cast<float>(c[u][2 * k + 1]), s[u]));
        w[k] = lo | (hi << 16);
      }
      uint16_t* out = const_cast<uint16_t*>(a.x[tt[u]]) + dst[u];
      *reinterpret_cast<uint4*>(out) = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
}

int ceil_log2(int v) {
  int l = 0;
  while ((1 << l) < v) ++l;
  return l;
}

// Persistent grid: enough blocks for the work, at most what is resident on all SMs at once.
template <int BITS, bool QUANT>
int grid_for(int64_t n_steps) {
  static int blocks_per_sm = 0;
  if (blocks_per_sm == 0) {
    int b = 0;
    cudaError_t e = QUANT ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                                &b, quant_pack_kernel<BITS>, kThreads, 0)
                          : cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                                &b, dequant_kernel<BITS>, kThreads, 0);
    blocks_per_sm = (e != cudaSuccess || b < 1) ? 1 : b;
  }
  const int64_t warps_needed = (n_steps + kUnroll - 1) / kUnroll;
  const int64_t blocks_needed = (warps_needed + (kThreads / 32) - 1) / (kThreads / 32);
  const int sms = sm_count();
  const int64_t cap = static_cast<int64_t>(sms > 0 ? sms : 1) * blocks_per_sm;
  int64_t g = blocks_needed < cap ? blocks_needed : cap;
  return static_cast<int>(g < 1 ? 1 : g);
}

kvq_status prepare(PackArgs& a, const kvq_pool* pools, const uint16_t* const* x, int n_tensors,
                   const int32_t* page_table, int max_pages, const int32_t* cu,
                   const int32_t* start, int nseq, int total_tokens, int32_t* err,
                   const char* what) {
  if (n_tensors < 1 || n_tensors > KVQ_MAX_TENSORS)
    return fail(KVQ_ERR_RANGE, "%s: n_tensors %d not in [1, %d]", what, n_tensors,
                KVQ_MAX_TENSORS);
  kvq_status st = check_pools_uniform(pools, n_tensors, what);
  if (st != KVQ_OK) return st;
  if (nseq < 0 || total_tokens < 0 || max_pages < 1)
    return fail(KVQ_ERR_RANGE, "%s: bad nseq %d / total_tokens %d / max_pages %d", what, nseq,
                total_tokens, max_pages);
  if (total_tokens > 0 && nseq < 1)
    return fail(KVQ_ERR_RANGE, "%s: tokens given but no sequences", what);
  if (!x) return fail(KVQ_ERR_NULL, "%s: tensor array is NULL", what);
  if (total_tokens > 0 && (!page_table || !cu || !start))
    return fail(KVQ_ERR_NULL, "%s: page_table/cu/start_pos is NULL", what);
  for (int i = 0; i < n_tensors; ++i) {
    if (!x[i] && total_tokens > 0) return fail(KVQ_ERR_NULL, "%s: tensor %d is NULL", what, i);
    if (!aligned16(x[i])) return fail(KVQ_ERR_ALIGN, "%s: tensor %d not 16-byte aligned", what, i);
  }
  const kvq_pool& p0 = pools[0];
  a.n_tensors = n_tensors;
  a.H = p0.num_heads;
  a.D = p0.head_dim;
  a.page_size = p0.page_size;
  a.pd = kvq_packed_dim(p0.head_dim, p0.bits);
  a.max_pages = max_pages;
  a.nseq = nseq;
  a.chunks = p0.head_dim / 8;
  a.lpr_log2 = ceil_log2(a.chunks);
  a.rows_per_tensor = static_cast<int64_t>(total_tokens) * p0.num_heads;
  a.page_table = page_table;
  a.cu = cu;
  a.start = start;
  a.err = err;
  for (int i = 0; i < KVQ_MAX_TENSORS; ++i) {
    a.x[i] = i < n_tensors ? x[i] : nullptr;
    a.pool[i] = i < n_tensors ? PoolRef{pools[i].codes, pools[i].scales, pools[i].num_pages}
                              : PoolRef{nullptr, nullptr, 0};
  }
  return KVQ_OK;
}

}  // namespace

// explicit launchers (kernel templates cannot be template-template args portably)
static kvq_status launch_quant(const PackArgs& a, int bits, cudaStream_t stream) {
  const int rps = 32 >> a.lpr_log2;
  const int64_t n_steps = (static_cast<int64_t>(a.n_tensors) * a.rows_per_tensor + rps - 1) / rps;
  if (n_steps == 0) return ok();
  switch (bits) {
    case 8: quant_pack_kernel<8><<<grid_for<8, true>(n_steps), kThreads, 0, stream>>>(a); break;
    case 6: quant_pack_kernel<6><<<grid_for<6, true>(n_steps), kThreads, 0, stream>>>(a); break;
    default: quant_pack_kernel<4><<<grid_for<4, true>(n_steps), kThreads, 0, stream>>>(a); break;
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(KVQ_ERR_CUDA, "quant_pack launch: %s", cudaGetErrorString(e));
  return ok();
}

static kvq_status launch_dequant(const PackArgs& a, int bits, cudaStream_t stream) {
  const int rps = 32 >> a.lpr_log2;
  const int64_t n_steps = (static_cast<int64_t>(a.n_tensors) * a.rows_per_tensor + rps - 1) / rps;
  if (n_steps == 0) return ok();
  switch (bits) {
    case 8: dequant_kernel<8><<<grid_for<8, false>(n_steps), kThreads, 0, stream>>>(a); break;
    case 6: dequant_kernel<6><<<grid_for<6, false>(n_steps), kThreads, 0, stream>>>(a); break;
    default: dequant_kernel<4><<<grid_for<4, false>(n_steps), kThreads, 0, stream>>>(a); break;
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(KVQ_ERR_CUDA, "dequant launch: %s", cudaGetErrorString(e));
  return ok();
}

}  // namespace kvq

extern "C" kvq_status kvq_quant_pack_paged(const kvq_pool* pools, const uint16_t* const* x,
                                           int n_tensors, const int32_t* page_table,
                                           int max_pages, const int32_t* cu_new_tokens,
                                           const int32_t* start_pos, int nseq,
                                           int total_new_tokens, int32_t* dev_err,
                                           kvq_stream_t stream) {
  kvq::PackArgs a;
  kvq_status st = kvq::prepare(a, pools, x, n_tensors, page_table, max_pages, cu_new_tokens,
                               start_pos, nseq, total_new_tokens, dev_err,
                               "kvq_quant_pack_paged");
  if (st != KVQ_OK) return st;
  return kvq::launch_quant(a, pools[0].bits, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" kvq_status kvq_dequant_paged(const kvq_pool* pools, uint16_t* const* out,
                                        int n_tensors, const int32_t* page_table, int max_pages,
                                        const int32_t* cu_tokens, const int32_t* start_pos,
                                        int nseq, int total_tokens, int32_t* dev_err,
                                        kvq_stream_t stream) {
  kvq::PackArgs a;
  kvq_status st = kvq::prepare(a, pools, const_cast<const uint16_t* const*>(out), n_tensors,
                               page_table, max_pages, cu_tokens, start_pos, nseq, total_tokens,
                               dev_err, "kvq_dequant_paged");
  if (st != KVQ_OK) return st;
  return kvq::launch_dequant(a, pools[0].bits, reinterpret_cast<cudaStream_t>(stream));
}
