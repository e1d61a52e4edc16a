// Symmetric per-token-per-head quantize + pack into pages, and the inverse gather + dequantize.
//
// MTPLX pull request #267, "feat(kv-cache): add q6 paged KV quantization", description: one fp16
// scale per (token, KV head) row, qmax 127/31/7 (bit-width table paragraph), q6 codes biased by
// +32 and packed four per three bytes little-endian (byte-layout formula), packed_dim(D, 6) =
// 3D/4.  The q6 pack is written here as one 24-bit little-endian word per four fields,
// w = u0 | u1 << 6 | u2 << 12 | u3 << 18, whose three bytes are exactly the page's byte0..2.
//
// Thread layout: a warp takes a block of 8 new tokens (all their heads: rows contiguous in the
// input); lanes 0..7 look up the page of one token each and broadcast it by shuffle.  Each lane
// owns one 16-byte chunk (8 elements) of a row; a row spans next_pow2(D/8) lanes, so a warp
// covers 32 / that rows per step, with 8 steps of loads in flight.  Row loads and stores are
// contiguous across lanes (coalesced), the row max is an fp16 max plus a segmented shuffle, and
// codes are packed in registers.  Per element: the quotient by the row's scale from a per-row
// reciprocal with one Markstein correction (exact), then one add that rounds half to even and
// leaves the biased field in the low bits.  HBM-bound: per row 2D bytes in, packed_dim + 2 out.
#include <cuda_runtime.h>

#include "kvq_device.cuh"
#include "kvq_internal.h"
#include "kvq_math.cuh"

namespace kvq {
namespace {

constexpr int kThreads = 256;
constexpr int kWarpsPerBlock = kThreads / 32;
constexpr int kTok = 8;     // tokens per warp work item (all heads of each)
constexpr int kUnroll = 8;  // row steps with loads in flight per lane

struct PackArgs {
  const uint16_t* x[KVQ_MAX_TENSORS];  // quant: inputs; dequant: outputs (cast back)
  PoolRef pool[KVQ_MAX_TENSORS];
  const int32_t* page_table;
  const int32_t* cu;
  const int32_t* start;
  int32_t* err;
  int n_tensors, total_tokens, H, D, page_size, pd, max_pages, nseq;
  int lpr_log2;             // lanes per row = 1 << lpr_log2
  int chunks;               // D / 8
};

template <int BITS> struct Q;
template <> struct Q<8> { static constexpr int kQmax = 127, kBias = 0, kMask = 0xff; };
template <> struct Q<6> { static constexpr int kQmax = 31, kBias = 32, kMask = 0x3f; };
template <> struct Q<4> { static constexpr int kQmax = 7, kBias = 8, kMask = 0x0f; };

// Physical row of head 0 of new token `tok` ((page * H) * page_size + slot), or -1.
__device__ __forceinline__ long long token_base(const PackArgs& a, int64_t num_pages, int tok) {
  const int s = find_seq(a.cu, a.nseq, tok);
  const int64_t pos = static_cast<int64_t>(__ldg(a.start + s)) + (tok - __ldg(a.cu + s));
  return locate_row(a.page_table, a.max_pages, a.page_size, a.H, num_pages, s, pos, 0, a.err);
}

__device__ __forceinline__ long long shfl_ll(long long v, int src) {
  const int lo = __shfl_sync(kFullMask, static_cast<int>(v & 0xffffffffLL), src);
  const int hi = __shfl_sync(kFullMask, static_cast<int>(v >> 32), src);
  return (static_cast<long long>(hi) << 32) | static_cast<unsigned int>(lo);
}

__device__ __forceinline__ float half2_absmax(const uint4& v) {
  const __half2 a = __habs2(*reinterpret_cast<const __half2*>(&v.x));
  const __half2 b = __habs2(*reinterpret_cast<const __half2*>(&v.y));
  const __half2 c = __habs2(*reinterpret_cast<const __half2*>(&v.z));
  const __half2 d = __habs2(*reinterpret_cast<const __half2*>(&v.w));
  const __half2 m = __hmax2(__hmax2(a, b), __hmax2(c, d));
  return fmaxf(__low2float(m), __high2float(m));
}

// Store the 8 fields of one chunk; `m` = physical row * chunks + chunk, so the chunk's bytes
// start at m * BITS (8 fields of BITS bits).
template <int BITS>
__device__ __forceinline__ void store_fields(uint8_t* codes, int64_t m, const uint32_t f[8]) {
  if constexpr (BITS == 8) {
    const uint32_t w0 = f[0] | (f[1] << 8) | (f[2] << 16) | (f[3] << 24);
    const uint32_t w1 = f[4] | (f[5] << 8) | (f[6] << 16) | (f[7] << 24);
    *reinterpret_cast<uint2*>(codes + m * 8) = make_uint2(w0, w1);
  } else if constexpr (BITS == 4) {
    uint32_t w = 0;
#pragma unroll
    for (int k = 0; k < 8; ++k) w |= f[k] << (4 * k);
    *reinterpret_cast<uint32_t*>(codes + m * 4) = w;
  } else {
    // two 24-bit little-endian words w = u0 | u1 << 6 | u2 << 12 | u3 << 18
    const uint32_t w0 = f[0] | (f[1] << 6) | (f[2] << 12) | (f[3] << 18);
    const uint32_t w1 = f[4] | (f[5] << 6) | (f[6] << 12) | (f[7] << 18);
    const uint32_t lo = w0 | (w1 << 24);                  // bytes 0..3
    const uint32_t hi = w1 >> 8;                          // bytes 4..5
    uint8_t* p = codes + m * 6;
    if ((m & 1) == 0) {  // 6m % 4 == 0
      *reinterpret_cast<uint32_t*>(p) = lo;
      *reinterpret_cast<uint16_t*>(p + 4) = static_cast<uint16_t>(hi);
    } else {             // 6m % 4 == 2
      *reinterpret_cast<uint16_t*>(p) = static_cast<uint16_t>(lo & 0xffffu);
      *reinterpret_cast<uint32_t*>(p + 2) = (lo >> 16) | (hi << 16);
    }
  }
}

// Load the packed bytes of one chunk as words for unpack_group<BITS, 0>.
template <int BITS>
__device__ __forceinline__ void load_fields(const uint8_t* codes, int64_t m, uint32_t w[2]) {
  if constexpr (BITS == 8) {
    const uint2 v = ld_nc_v2(codes + m * 8);
    w[0] = v.x;
    w[1] = v.y;
  } else if constexpr (BITS == 4) {
    w[0] = ld_nc_u32(codes + m * 4);
    w[1] = 0;
  } else {
    const uint8_t* p = codes + m * 6;
    if ((m & 1) == 0) {
      w[0] = ld_nc_u32(p);
      w[1] = ld_nc_u16(p + 4);
    } else {
      const uint32_t a = ld_nc_u16(p), b = ld_nc_u32(p + 2);
      w[0] = a | (b << 16);
      w[1] = b >> 16;
    }
  }
}

template <int BITS>
__global__ void __launch_bounds__(kThreads) quant_pack_kernel(const PackArgs a) {
  constexpr float kQ = static_cast<float>(Q<BITS>::kQmax);
  const int t = blockIdx.y;
  const uint16_t* __restrict__ x = a.x[t];
  const PoolRef pool = a.pool[t];
  const int lane = threadIdx.x & 31;
  const int lpr = 1 << a.lpr_log2;
  const int rps = 32 >> a.lpr_log2;
  const int chunk = lane & (lpr - 1);
  const int sub = lane >> a.lpr_log2;
  const int H = a.H;
  const int n_items = (a.total_tokens + kTok - 1) / kTok;
  const int n_warps = gridDim.x * kWarpsPerBlock;

  for (int item = blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5); item < n_items;
       item += n_warps) {
    const int tok0 = item * kTok;
    const int ntok = min(kTok, a.total_tokens - tok0);
    long long base = -1;
    if (lane < ntok) base = token_base(a, pool.num_pages, tok0 + lane);
    const int nrows = ntok * H;
    const uint16_t* xi = x + static_cast<int64_t>(tok0) * H * a.D + chunk * 8;
    for (int r0 = 0; r0 < nrows; r0 += rps * kUnroll) {
      uint4 v[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int row = r0 + u * rps + sub;
        v[u] = make_uint4(0, 0, 0, 0);
        if (row < nrows && chunk < a.chunks)
          v[u] = ld_stream_v4(xi + static_cast<int64_t>(row) * a.D);
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int row = r0 + u * rps + sub;
        float amax = half2_absmax(v[u]);
        for (int o = lpr >> 1; o >= 1; o >>= 1)
          amax = fmaxf(amax, __shfl_xor_sync(kFullMask, amax, o));
        const int k = row / H;
        const long long b = shfl_ll(base, k < kTok ? k : 0);
        if (row >= nrows || chunk >= a.chunks || b < 0) continue;
        const int64_t prow = b + static_cast<int64_t>(row - k * H) * a.page_size;
        const uint16_t sbits = f2h(__fdiv_rn(amax, kQ));
        const float s = h2f(sbits);
        // s == 0: y = 0 gives a zero quotient (codes 0); subnormal s: clip to +-qmax
        const float y = (s == 0.f) ? 0.f : __frcp_rn(s);
        const float se = (s == 0.f) ? 1.f : s;
        const bool clip = s < 6.103515625e-05f;   // 2^-14, smallest normal fp16
        const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
        uint32_t f[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float xe = h2f(static_cast<uint16_t>(w[e >> 1] >> (16 * (e & 1))));
          f[e] = quant_field<Q<BITS>::kQmax, Q<BITS>::kBias, Q<BITS>::kMask>(xe, se, y, clip);
        }
        store_fields<BITS>(pool.codes, prow * a.chunks + chunk, f);
        if (chunk == 0) pool.scales[prow] = sbits;
      }
    }
  }
}

template <int BITS>
__global__ void __launch_bounds__(kThreads) dequant_kernel(const PackArgs a) {
  const int t = blockIdx.y;
  uint16_t* __restrict__ out = const_cast<uint16_t*>(a.x[t]);
  const PoolRef pool = a.pool[t];
  const int lane = threadIdx.x & 31;
  const int lpr = 1 << a.lpr_log2;
  const int rps = 32 >> a.lpr_log2;
  const int chunk = lane & (lpr - 1);
  const int sub = lane >> a.lpr_log2;
  const int H = a.H;
  const int n_items = (a.total_tokens + kTok - 1) / kTok;
  const int n_warps = gridDim.x * kWarpsPerBlock;

  for (int item = blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5); item < n_items;
       item += n_warps) {
    const int tok0 = item * kTok;
    const int ntok = min(kTok, a.total_tokens - tok0);
    long long base = -1;
    if (lane < ntok) base = token_base(a, pool.num_pages, tok0 + lane);
    const int nrows = ntok * H;
    uint16_t* oi = out + static_cast<int64_t>(tok0) * H * a.D + chunk * 8;
    for (int r0 = 0; r0 < nrows; r0 += rps * kUnroll) {
      uint32_t w[kUnroll][2];
      uint32_t sc[kUnroll];
      bool act[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int row = r0 + u * rps + sub;
        const int k = row / H;
        const long long b = shfl_ll(base, k < kTok ? k : 0);
        act[u] = row < nrows && chunk < a.chunks && b >= 0;
        w[u][0] = w[u][1] = 0;
        sc[u] = 0;
        if (act[u]) {
          const int64_t prow = b + static_cast<int64_t>(row - k * H) * a.page_size;
          load_fields<BITS>(pool.codes, prow * a.chunks + chunk, w[u]);
          sc[u] = ld_nc_u16(pool.scales + prow);
        }
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        if (!act[u]) continue;
        const int row = r0 + u * rps + sub;
        uint32_t p[4];
        unpack_group<BITS, 0>(w[u], p);          // {e_k, e_{k+4}}
        const uint32_t s2 = sc[u] | (sc[u] << 16);
        // exact codes times the fp16 scale: one rounding, the same as fp16(float(c) * scale)
        const uint32_t o0 = hmul2u(prmt(p[0], p[1], 0x5410u), s2);   // e0 e1
        const uint32_t o1 = hmul2u(prmt(p[2], p[3], 0x5410u), s2);   // e2 e3
        const uint32_t o2 = hmul2u(prmt(p[0], p[1], 0x7632u), s2);   // e4 e5
        const uint32_t o3 = hmul2u(prmt(p[2], p[3], 0x7632u), s2);   // e6 e7
        *reinterpret_cast<uint4*>(oi + static_cast<int64_t>(row) * a.D) =
            make_uint4(o0, o1, o2, o3);
      }
    }
  }
}

int ceil_log2(int v) {
  int l = 0;
  while ((1 << l) < v) ++l;
  return l;
}

// Persistent grid: blockIdx.y = tensor; per tensor enough blocks for its token blocks, with all
// tensors together at most what is resident on the SMs at once.
template <int BITS, bool QUANT>
dim3 grid_for(int n_tensors, int total_tokens) {
  static int blocks_per_sm = 0;
  if (blocks_per_sm == 0) {
    int b = 0;
    cudaError_t e = QUANT ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                                &b, quant_pack_kernel<BITS>, kThreads, 0)
                          : cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                                &b, dequant_kernel<BITS>, kThreads, 0);
    blocks_per_sm = (e != cudaSuccess || b < 1) ? 1 : b;
  }
  const int64_t items = (static_cast<int64_t>(total_tokens) + kTok - 1) / kTok;
  const int64_t need = (items + kWarpsPerBlock - 1) / kWarpsPerBlock;
  const int sms = sm_count();
  const int64_t cap = static_cast<int64_t>(sms > 0 ? sms : 1) * blocks_per_sm;
  int64_t per = (cap + n_tensors - 1) / n_tensors;
  if (per > need) per = need;
  if (per < 1) per = 1;
  return dim3(static_cast<unsigned>(per), static_cast<unsigned>(n_tensors));
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
  a.total_tokens = total_tokens;
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
  if (a.total_tokens == 0) return ok();
  switch (bits) {
    case 8: quant_pack_kernel<8><<<grid_for<8, true>(a.n_tensors, a.total_tokens), kThreads, 0, stream>>>(a); break;
    case 6: quant_pack_kernel<6><<<grid_for<6, true>(a.n_tensors, a.total_tokens), kThreads, 0, stream>>>(a); break;
    default: quant_pack_kernel<4><<<grid_for<4, true>(a.n_tensors, a.total_tokens), kThreads, 0, stream>>>(a); break;
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(KVQ_ERR_CUDA, "quant_pack launch: %s", cudaGetErrorString(e));
  return ok();
}

static kvq_status launch_dequant(const PackArgs& a, int bits, cudaStream_t stream) {
  if (a.total_tokens == 0) return ok();
  switch (bits) {
    case 8: dequant_kernel<8><<<grid_for<8, false>(a.n_tensors, a.total_tokens), kThreads, 0, stream>>>(a); break;
    case 6: dequant_kernel<6><<<grid_for<6, false>(a.n_tensors, a.total_tokens), kThreads, 0, stream>>>(a); break;
    default: dequant_kernel<4><<<grid_for<4, false>(a.n_tensors, a.total_tokens), kThreads, 0, stream>>>(a); break;
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
