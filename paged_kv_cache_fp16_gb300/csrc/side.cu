// fp16 side channels on the symmetric quantizer: attention sinks and dense-and-sparse outliers.
//
// VeloxQuant-MLX API docs, "veloxquant_mlx.cache.kvquant_cache module": per-vector
// dense-and-sparse outlier isolation with an fp16 side channel (value + position index), and
// Attention Sink-Aware quantization (the first n_sink tokens of a sequence kept in exact fp16).
// Applied here to the symmetric per-token-per-head quantizer of MTPLX pull request #267:
//   a row's k largest-magnitude elements (ties: the lower position) are stored as fp16 value +
//   uint8 position, ascending by position; the rest of the row (outliers set to 0) is quantized
//   as usual, so its scale comes from the (k+1)-th largest magnitude and the outlier positions
//   hold code 0; dequantization writes the values back.  Rows at positions < n_sink are also
//   copied exactly into a [seq][n_sink][H][D] fp16 buffer that dequantization reads instead.
//
// A warp takes 32 consecutive rows: lane i locates row i (page-table lookups in parallel), then
// the warp walks them one row at a time, lane l holding elements [8l, 8l + 8).  Selection: each
// element's key is ((|x| bits << 8) | (255 - position)) + 1 -- unique within the row, larger for
// a larger magnitude and, among equal magnitudes, for the lower position; padding lanes hold 0 --
// and k + 1 rounds of a warp max (redux) pick the outliers, then the largest remaining magnitude,
// which is the dense row's amax; lane j keeps the j-th outlier and stores it at its rank among
// the k positions (ascending order without a sort).  The scale and code arithmetic are the
// quant-pack kernel's.
#include <cuda_runtime.h>
#include <cuda_fp16.h>

#include "kvq_device.cuh"
#include "kvq_internal.h"
#include "kvq_math.cuh"

namespace kvq {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

struct SideRef {
  uint16_t* out_val;
  uint8_t* out_idx;
  uint16_t* sink;
};

struct SideArgs {
  const uint16_t* x[KVQ_MAX_TENSORS];   // quant: inputs; dequant: outputs
  PoolRef pool[KVQ_MAX_TENSORS];
  SideRef side[KVQ_MAX_TENSORS];
  const int32_t* page_table;
  const int32_t* cu;
  const int32_t* start;
  int32_t* err;
  int n_tensors, total_tokens, H, D, page_size, pd, max_pages, nseq, k, n_sink;
};

// Bytes of the packed fields of 8 consecutive elements (lane l's share of a row).
template <int BITS> constexpr int lane_bytes() { return BITS; }

template <int BITS>
__device__ __forceinline__ void store_lane(uint8_t* p, uint32_t a, uint32_t b) {
  if constexpr (BITS == 6) {   // two 24-bit words -> 6 bytes, 2-byte aligned
    uint16_t* q = reinterpret_cast<uint16_t*>(p);
    q[0] = static_cast<uint16_t>(a & 0xffffu);
    q[1] = static_cast<uint16_t>((a >> 16) | ((b & 0xffu) << 8));
    q[2] = static_cast<uint16_t>(b >> 8);
  } else if constexpr (BITS == 4) {
    *reinterpret_cast<uint32_t*>(p) = a;
  } else {
    *reinterpret_cast<uint2*>(p) = make_uint2(a, b);
  }
}

template <int BITS>
__device__ __forceinline__ uint64_t load_lane(const uint8_t* p) {
  if constexpr (BITS == 6) {
    const uint16_t* q = reinterpret_cast<const uint16_t*>(p);
    return static_cast<uint64_t>(q[0]) | (static_cast<uint64_t>(q[1]) << 16) |
           (static_cast<uint64_t>(q[2]) << 32);
  } else if constexpr (BITS == 4) {
    return *reinterpret_cast<const uint32_t*>(p);
  } else {
    const uint2 w = *reinterpret_cast<const uint2*>(p);
    return static_cast<uint64_t>(w.x) | (static_cast<uint64_t>(w.y) << 32);
  }
}

__device__ __forceinline__ int64_t shfl_i64(int64_t v, int src) {
  const int lo = __shfl_sync(kFullMask, static_cast<int>(v & 0xffffffffLL), src);
  const int hi = __shfl_sync(kFullMask, static_cast<int>(v >> 32), src);
  return (static_cast<int64_t>(hi) << 32) | static_cast<uint32_t>(lo);
}

// Row r of the call's [total_tokens][H] rows -> (sequence, position, physical row or -1).
__device__ __forceinline__ int64_t row_place(const SideArgs& a, int64_t num_pages, int r, int& s,
                                             int64_t& pos) {
  const int tok = r / a.H, h = r - tok * a.H;
  s = find_seq(a.cu, a.nseq, tok);
  pos = static_cast<int64_t>(__ldg(a.start + s)) + (tok - __ldg(a.cu + s));
  return locate_row(a.page_table, a.max_pages, a.page_size, a.H, num_pages, s, pos, h, a.err);
}

template <int BITS>
__global__ void __launch_bounds__(kThreads) quant_pack_side_kernel(const SideArgs a) {
  constexpr int kQm = SymQ<BITS>::kQmax;
  constexpr int kB = SymQ<BITS>::kBias;
  constexpr int kM = SymQ<BITS>::kMask;
  const int t = blockIdx.y;
  const PoolRef pool = a.pool[t];
  const SideRef sd = a.side[t];
  const int lane = threadIdx.x & 31;
  const int rows = a.total_tokens * a.H;
  const bool live = 8 * lane < a.D;
  const int n_blocks = (rows + 31) / 32;
  for (int blk = blockIdx.x * kWarps + (threadIdx.x >> 5); blk < n_blocks;
       blk += gridDim.x * kWarps) {
    // lane i locates row 32 * blk + i; the warp then walks the 32 rows
    int my_s = 0;
    int64_t my_pos = 0, my_prow = -1;
    if (32 * blk + lane < rows)
      my_prow = row_place(a, pool.num_pages, 32 * blk + lane, my_s, my_pos);
    const int nr = min(32, rows - 32 * blk);
    for (int i = 0; i < nr; ++i) {
      const int r = 32 * blk + i;
      const int64_t prow = shfl_i64(my_prow, i);
      if (prow < 0) continue;   // warp-uniform
      const int s = __shfl_sync(kFullMask, my_s, i);
      const int64_t pos = shfl_i64(my_pos, i);
      const int h = r % a.H;
      uint4 xv = make_uint4(0, 0, 0, 0);
      if (live) xv = ld_stream_v4(a.x[t] + static_cast<int64_t>(r) * a.D + 8 * lane);
      const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
      uint32_t key[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const uint32_t bits = (xw[e >> 1] >> (16 * (e & 1))) & 0xffffu;
        key[e] = live ? ((((bits & 0x7fffu) << 8) | (255u - (8 * lane + e))) + 1u) : 0u;
      }
      // k rounds of a warp max pick the outliers (lane j keeps the j-th), round k the dense amax
      uint32_t my_opos = 0xffffu, my_oval = 0;
      float amax = 0.f;
      for (int j = 0; j <= a.k; ++j) {
        uint32_t m = key[0];
#pragma unroll
        for (int e = 1; e < 8; ++e) m = max(m, key[e]);
        const uint32_t w = __reduce_max_sync(kFullMask, m);
        if (j == a.k) {
          amax = (w == 0u) ? 0.f : h2f(static_cast<uint16_t>((w - 1u) >> 8));
          break;
        }
        uint32_t v = 0;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          if (key[e] == w) {
            v = (xw[e >> 1] >> (16 * (e & 1))) & 0xffffu;
            key[e] = 0u;   // taken: it also leaves the dense row
          }
        }
        const uint32_t val = __reduce_or_sync(kFullMask, v);
        if (lane == j) {
          my_opos = 255u - ((w - 1u) & 0xffu);
          my_oval = val;
        }
      }
      const uint16_t sbits = f2h(row_scale_f32<kQm>(amax));
      const float sc = h2f(sbits);
      const float y = (sc == 0.f) ? 0.f : __frcp_rn(sc);
      const float se = (sc == 0.f) ? 1.f : sc;
      const bool clip = sc < 6.103515625e-05f;   // 2^-14, smallest normal fp16
      if (live) {
        uint32_t f[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const bool dense = key[e] != 0u;
          const float xe = dense ? h2f(static_cast<uint16_t>(xw[e >> 1] >> (16 * (e & 1)))) : 0.f;
          f[e] = quant_field<kQm, kB, kM>(xe, se, y, clip);
        }
        uint32_t pa, pb;
        pack8<BITS>(f, pa, pb);
        store_lane<BITS>(pool.codes + prow * a.pd + lane * lane_bytes<BITS>(), pa, pb);
      }
      if (lane == 0) pool.scales[prow] = sbits;
      if (a.k > 0) {
        // ascending positions: lane j < k stores its outlier at its rank among the k positions
        uint32_t rank = 0;
        for (int j = 0; j < a.k; ++j) rank += __shfl_sync(kFullMask, my_opos, j) < my_opos ? 1u : 0u;
        if (lane < a.k) {
          sd.out_idx[prow * a.k + rank] = static_cast<uint8_t>(my_opos);
          sd.out_val[prow * a.k + rank] = static_cast<uint16_t>(my_oval);
        }
      }
      if (pos < a.n_sink && live)
        *reinterpret_cast<uint4*>(sd.sink + ((static_cast<int64_t>(s) * a.n_sink + pos) * a.H + h) *
                                                a.D + 8 * lane) = xv;
    }
  }
}

template <int BITS>
__global__ void __launch_bounds__(kThreads) dequant_side_kernel(const SideArgs a) {
  constexpr int kB = SymQ<BITS>::kBias;
  constexpr uint32_t kM = SymQ<BITS>::kMask;
  const int t = blockIdx.y;
  uint16_t* out = const_cast<uint16_t*>(a.x[t]);
  const PoolRef pool = a.pool[t];
  const SideRef sd = a.side[t];
  const int lane = threadIdx.x & 31;
  const int rows = a.total_tokens * a.H;
  const bool live = 8 * lane < a.D;
  const int n_blocks = (rows + 31) / 32;
  for (int blk = blockIdx.x * kWarps + (threadIdx.x >> 5); blk < n_blocks;
       blk += gridDim.x * kWarps) {
    int my_s = 0;
    int64_t my_pos = 0, my_prow = -1;
    if (32 * blk + lane < rows)
      my_prow = row_place(a, pool.num_pages, 32 * blk + lane, my_s, my_pos);
    const int nr = min(32, rows - 32 * blk);
    for (int i = 0; i < nr; ++i) {
      const int r = 32 * blk + i;
      const int64_t prow = shfl_i64(my_prow, i);
      if (prow < 0) continue;   // warp-uniform
      const int s = __shfl_sync(kFullMask, my_s, i);
      const int64_t pos = shfl_i64(my_pos, i);
      if (!live) continue;
      const int h = r % a.H;
      uint4 res;
      if (pos < a.n_sink) {
        res = *reinterpret_cast<const uint4*>(
            sd.sink + ((static_cast<int64_t>(s) * a.n_sink + pos) * a.H + h) * a.D + 8 * lane);
      } else {
        const uint64_t fw = load_lane<BITS>(pool.codes + prow * a.pd + lane * lane_bytes<BITS>());
        const float sc = h2f(pool.scales[prow]);
        uint32_t o[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const uint32_t fld = static_cast<uint32_t>(fw >> (BITS * e)) & kM;
          const int c = (BITS == 8) ? static_cast<int>(static_cast<int8_t>(fld))
                                    : static_cast<int>(fld) - kB;
          o[e] = f2h(static_cast<float>(c) * sc);   // exact product, one rounding to fp16
        }
        for (int j = 0; j < a.k; ++j) {
          const uint32_t d = sd.out_idx[prow * a.k + j];
          const uint32_t v = sd.out_val[prow * a.k + j];
#pragma unroll
          for (int e = 0; e < 8; ++e)
            if (d == static_cast<uint32_t>(8 * lane + e)) o[e] = v;
        }
        res = make_uint4(o[0] | (o[1] << 16), o[2] | (o[3] << 16), o[4] | (o[5] << 16),
                         o[6] | (o[7] << 16));
      }
      *reinterpret_cast<uint4*>(out + static_cast<int64_t>(r) * a.D + 8 * lane) = res;
    }
  }
}

kvq_status check_sides(const kvq_pool* pools, const kvq_side* sides, int n, int nseq,
                       const char* fn) {
  if (!sides) return fail(KVQ_ERR_NULL, "%s: side array is NULL", fn);
  const int k = sides[0].n_outlier, ns = sides[0].n_sink;
  if (k < 0 || k > KVQ_MAX_OUTLIERS || k >= pools[0].head_dim)
    return fail(KVQ_ERR_RANGE, "%s: n_outlier %d not in [0, %d] (and < head_dim)", fn, k,
                KVQ_MAX_OUTLIERS);
  if (ns < 0 || ns > KVQ_MAX_SINKS)
    return fail(KVQ_ERR_RANGE, "%s: n_sink %d not in [0, %d]", fn, ns, KVQ_MAX_SINKS);
  for (int i = 0; i < n; ++i) {
    const kvq_side& sd = sides[i];
    if (sd.n_outlier != k || sd.n_sink != ns)
      return fail(KVQ_ERR_SHAPE, "%s: side %d differs from side 0 in n_outlier/n_sink", fn, i);
    if (k > 0 && (!sd.out_val || !sd.out_idx))
      return fail(KVQ_ERR_NULL, "%s: side %d has no outlier arrays", fn, i);
    if (ns > 0 && !sd.sink) return fail(KVQ_ERR_NULL, "%s: side %d has no sink buffer", fn, i);
    if ((k > 0 && (!aligned16(sd.out_val) || !aligned16(sd.out_idx))) ||
        (ns > 0 && !aligned16(sd.sink)))
      return fail(KVQ_ERR_ALIGN, "%s: side %d arrays must be 16-byte aligned", fn, i);
    if (ns > 0 && sd.max_seqs < nseq)
      return fail(KVQ_ERR_RANGE, "%s: side %d sink buffer holds %d sequences, call has %d", fn,
                  i, sd.max_seqs, nseq);
  }
  return KVQ_OK;
}

kvq_status side_call(bool quant, const kvq_pool* pools, const kvq_side* sides,
                     const uint16_t* const* x, int n_tensors, const int32_t* page_table,
                     int max_pages, const int32_t* cu, const int32_t* start, int nseq,
                     int total, int32_t* dev_err, kvq_stream_t stream, const char* fn) {
  if (n_tensors < 1 || n_tensors > KVQ_MAX_TENSORS)
    return fail(KVQ_ERR_RANGE, "%s: n_tensors %d not in [1, %d]", fn, n_tensors, KVQ_MAX_TENSORS);
  kvq_status st = check_pools_uniform(pools, n_tensors, fn);
  if (st != KVQ_OK) return st;
  const kvq_pool& p0 = pools[0];
  if (p0.head_dim % 16 || p0.head_dim > 256)
    return fail(KVQ_ERR_SHAPE, "%s: head_dim %d must be a multiple of 16, <= 256", fn,
                p0.head_dim);
  if (nseq < 0 || total < 0 || max_pages < 1)
    return fail(KVQ_ERR_RANGE, "%s: bad nseq/total/max_pages", fn);
  st = check_sides(pools, sides, n_tensors, nseq, fn);
  if (st != KVQ_OK) return st;
  if (!x || !page_table || !cu || !start) return fail(KVQ_ERR_NULL, "%s: NULL pointer", fn);
  for (int i = 0; i < n_tensors; ++i) {
    if (!x[i]) return fail(KVQ_ERR_NULL, "%s: tensor %d is NULL", fn, i);
    if (!aligned16(x[i])) return fail(KVQ_ERR_ALIGN, "%s: tensor %d not 16-byte aligned", fn, i);
  }
  if (total == 0 || nseq == 0) return ok();
  if (static_cast<int64_t>(total) * p0.num_heads > 0x7fffffffLL)
    return fail(KVQ_ERR_RANGE, "%s: too many rows", fn);
  SideArgs a;
  for (int i = 0; i < KVQ_MAX_TENSORS; ++i) {
    const int j = i < n_tensors ? i : 0;
    a.x[i] = x[j];
    a.pool[i] = PoolRef{pools[j].codes, pools[j].scales, pools[j].num_pages};
    a.side[i] = SideRef{sides[j].out_val, sides[j].out_idx, sides[j].sink};
  }
  a.page_table = page_table;
  a.cu = cu;
  a.start = start;
  a.err = dev_err;
  a.n_tensors = n_tensors;
  a.total_tokens = total;
  a.H = p0.num_heads;
  a.D = p0.head_dim;
  a.page_size = p0.page_size;
  a.pd = kvq_packed_dim(p0.head_dim, p0.bits);
  a.max_pages = max_pages;
  a.nseq = nseq;
  a.k = sides[0].n_outlier;
  a.n_sink = sides[0].n_sink;
  const int sms = sm_count() > 0 ? sm_count() : 152;
  const int64_t rows = static_cast<int64_t>(total) * a.H;
  int64_t blocks = ((rows + 31) / 32 + kWarps - 1) / kWarps;
  const int64_t cap = (8LL * sms + n_tensors - 1) / n_tensors;
  if (blocks > cap) blocks = cap;
  const dim3 grid(static_cast<unsigned>(blocks), n_tensors);
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  switch (p0.bits) {
    case 8:
      if (quant) quant_pack_side_kernel<8><<<grid, kThreads, 0, cs>>>(a);
      else dequant_side_kernel<8><<<grid, kThreads, 0, cs>>>(a);
      break;
    case 6:
      if (quant) quant_pack_side_kernel<6><<<grid, kThreads, 0, cs>>>(a);
      else dequant_side_kernel<6><<<grid, kThreads, 0, cs>>>(a);
      break;
    default:
      if (quant) quant_pack_side_kernel<4><<<grid, kThreads, 0, cs>>>(a);
      else dequant_side_kernel<4><<<grid, kThreads, 0, cs>>>(a);
      break;
  }
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(KVQ_ERR_CUDA, "%s launch: %s", fn, cudaGetErrorString(e));
  return ok();
}

}  // namespace
}  // namespace kvq

extern "C" kvq_status kvq_quant_pack_paged_side(const kvq_pool* pools, const kvq_side* sides,
                                                const uint16_t* const* x, int n_tensors,
                                                const int32_t* page_table, int max_pages,
                                                const int32_t* cu_new_tokens,
                                                const int32_t* start_pos, int nseq,
                                                int total_new_tokens, int32_t* dev_err,
                                                kvq_stream_t stream) {
  return kvq::side_call(true, pools, sides, x, n_tensors, page_table, max_pages, cu_new_tokens,
                        start_pos, nseq, total_new_tokens, dev_err, stream,
                        "kvq_quant_pack_paged_side");
}

extern "C" kvq_status kvq_dequant_paged_side(const kvq_pool* pools, const kvq_side* sides,
                                             uint16_t* const* out, int n_tensors,
                                             const int32_t* page_table, int max_pages,
                                             const int32_t* cu_tokens, const int32_t* start_pos,
                                             int nseq, int total_tokens, int32_t* dev_err,
                                             kvq_stream_t stream) {
  return kvq::side_call(false, pools, sides, const_cast<const uint16_t* const*>(out), n_tensors,
                        page_table, max_pages, cu_tokens, start_pos, nseq, total_tokens, dev_err,
                        stream, "kvq_dequant_paged_side");
}
