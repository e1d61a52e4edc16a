// Symmetric per-token-per-head quantize + pack into pages, and the inverse gather + dequantize.
//
// MTPLX pull request #267, "feat(kv-cache): add q6 paged KV quantization", description: one fp16
// scale per (token, KV head) row, qmax 127/31/7 (bit-width table paragraph), q6 codes biased by
// +32 and packed four per three bytes little-endian (byte-layout formula), packed_dim(D, 6) =
// 3D/4.  The q6 pack is written here as one 24-bit little-endian word per four fields,
// w = u0 | u1 << 6 | u2 << 12 | u3 << 18, whose three bytes are exactly the page's byte0..2.
//
// Thread layout: a warp takes a block of 8 new tokens (all their heads: rows contiguous in the
// input); lanes 0..7 look up the page of one token each and broadcast it by shuffle.  A row is
// cut into 16-element units (32 input bytes; 16 / 12 / 8 packed bytes for q8 / q6 / q4, so every
// lane's packed access is aligned and uniform); 8 lanes share a row (fewer for short rows), so
// one warp instruction serves 4 rows and the per-row scalar work (scale, reciprocal, address)
// is amortized over them.  Lane j of a row takes units j and j + 8, so each load or store
// instruction covers a contiguous span of every row (coalesced).  The row max is an fp16 max
// plus a segmented shuffle, and codes are packed in registers.  Per element: the quotient by the row's scale from a per-row
// reciprocal with one Markstein correction (exact), then one add that rounds half to even and
// leaves the biased field in the low bits.  HBM-bound: per row 2D bytes in, packed_dim + 2 out.
#include <type_traits>

#include <cuda_runtime.h>

#include "kvq_device.cuh"
#include "kvq_internal.h"
#include "kvq_divu32.cuh"
#include "kvq_math.cuh"
#include "kvq_rowwise.cuh"

namespace kvq {
namespace {

constexpr int kThreads = 256;
constexpr int kWarpsPerBlock = kThreads / 32;
constexpr int kTok = 8;     // most tokens per warp work item (all heads of each)
// quant-pack: warp steps with loads in flight.  q8 takes 3 (80 registers, 3 blocks per SM): 4.30
// -> 4.21 ms on the 16-layer workload; q6 and q4 keep 2 (64 registers, 4 blocks; 3 steps, or a
// minimum of 3 or 4 blocks per SM declared in the launch bounds, measured 1-12 % slower there).
template <int BITS> constexpr int qp_unroll() { return BITS == 8 ? 3 : 2; }
// dequant: its loads are smaller than the quantizer's, so more warp steps stay in flight.  The
// kernel is built for at least 3 blocks per SM (up to 85 registers), q4 for 4.  q6 takes 6 steps
// (80 registers, 3 blocks): more bytes in flight per SM than 4 steps at 4 blocks (64 registers,
// which also spilled), 4.09 -> 3.90 ms on the 16-layer workload (5 steps 3.94, 7 steps spill,
// 4.16).  q4 takes 4 steps at 4 blocks (60 registers; 3.770 ms against 3.800 at 3 blocks, 5 and 6
// steps 3.82 and 3.785), q8 4 steps at 3 blocks (74 registers; 4.44 ms against 4.54 with 2 steps
// at 4 blocks, 4.50 with 3).
template <int BITS> constexpr int dq_unroll() { return BITS == 6 ? 6 : 4; }

struct PackArgs {
  const uint16_t* x[KVQ_MAX_TENSORS];  // quant: inputs; dequant: outputs (cast back)
  PoolRef pool[KVQ_MAX_TENSORS];
  const int32_t* page_table;
  const int32_t* cu;
  const int32_t* start;
  int32_t* err;
  int n_tensors, total_tokens, H, D, page_size, pd, max_pages, nseq;
  int units;     // 16-element units per row: ceil(D / 16)
  int lpr_log2;  // lanes per row = 1 << lpr_log2 = min(next_pow2(units), 8)
  int tpi;       // tokens per work item, 1..kTok (fewer for calls too small to fill the GPU)
  bool v8;       // every fp16 tensor 32-byte aligned: its 16-element units move in one 256-bit access
  DivU32 div_h;  // by the head count: a row's token
};

// Physical row of head 0 of new token `tok` ((page * H) * page_size + slot), or -1.
__device__ __forceinline__ long long token_base(const PackArgs& a, int64_t num_pages, int tok) {
  const int s = find_seq(a.cu, a.nseq, a.total_tokens, tok);
  const int64_t pos = static_cast<int64_t>(__ldg(a.start + s)) + (tok - __ldg(a.cu + s));
  return locate_row(a.page_table, a.max_pages, a.page_size, a.H, num_pages, s, pos, 0, a.err);
}

__device__ __forceinline__ long long shfl_ll(long long v, int src) {
  const int lo = __shfl_sync(kFullMask, static_cast<int>(v & 0xffffffffLL), src);
  const int hi = __shfl_sync(kFullMask, static_cast<int>(v >> 32), src);
  return (static_cast<long long>(hi) << 32) | static_cast<unsigned int>(lo);
}

template <int BITS, int UPL, bool V8>
__global__ void __launch_bounds__(kThreads) quant_pack_kernel(const PackArgs a) {
  constexpr int kUnroll = qp_unroll<BITS>();
  constexpr int kQm = SymQ<BITS>::kQmax;
  constexpr int kB = SymQ<BITS>::kBias;
  constexpr int kM = SymQ<BITS>::kMask;
  const int t = blockIdx.y;
  const uint16_t* __restrict__ x = a.x[t];
  const PoolRef pool = a.pool[t];
  const int lane = threadIdx.x & 31;
  const int lpr = 1 << a.lpr_log2;
  const int rps = 32 >> a.lpr_log2;
  const int lr = lane & (lpr - 1);       // lane within the row
  const int sub = lane >> a.lpr_log2;    // row within the step
  const int H = a.H, D = a.D;
  const int n_items = (a.total_tokens + a.tpi - 1) / a.tpi;
  const int n_warps = gridDim.x * kWarpsPerBlock;

  for (int item = blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5); item < n_items;
       item += n_warps) {
    const int tok0 = item * a.tpi;
    const int ntok = min(a.tpi, a.total_tokens - tok0);
    long long base = -1;
    if (lane < ntok) base = token_base(a, pool.num_pages, tok0 + lane);
    const int nrows = ntok * H;
    const uint16_t* xi = x + static_cast<int64_t>(tok0) * H * D;
    for (int r0 = 0; r0 < nrows; r0 += rps * kUnroll) {
      uint4 v[kUnroll][UPL][2];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int row = r0 + u * rps + sub;
#pragma unroll
        for (int j = 0; j < UPL; ++j) {
          const int unit = lr + j * lpr;
          const int e0 = unit * 16;
          v[u][j][0] = v[u][j][1] = make_uint4(0, 0, 0, 0);
          if (row < nrows && e0 < D) {
            const uint16_t* src = xi + static_cast<int64_t>(row) * D + e0;
            if constexpr (V8) {
              ld_stream_v8(src, v[u][j][0], v[u][j][1]);
            } else {
              v[u][j][0] = ld_stream_v4(src);
              v[u][j][1] = ld_stream_v4(src + 8);
            }
          }
        }
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int row = r0 + u * rps + sub;
        __half2 m2 = absmax8(v[u][0][0]);
        m2 = __hmax2(m2, absmax8(v[u][0][1]));
#pragma unroll
        for (int j = 1; j < UPL; ++j) m2 = __hmax2(m2, __hmax2(absmax8(v[u][j][0]), absmax8(v[u][j][1])));
        float amax = fmaxf(__low2float(m2), __high2float(m2));
        for (int o = lpr >> 1; o >= 1; o >>= 1)
          amax = fmaxf(amax, __shfl_xor_sync(kFullMask, amax, o));
        const int k = static_cast<int>(divu32(static_cast<uint32_t>(row), a.div_h));
        const long long b = shfl_ll(base, k < kTok ? k : 0);
        if (row >= nrows || b < 0) continue;
        const int64_t prow = b + static_cast<int64_t>(row - k * H) * a.page_size;
        const uint16_t sbits = f2h(row_scale_f32<kQm>(amax));
        const float s = h2f(sbits);
        // s == 0: y = 0 gives a zero quotient (codes 0); subnormal s: clip to +-qmax
        const float y = (s == 0.f) ? 0.f : __frcp_rn(s);
        const float se = (s == 0.f) ? 1.f : s;
        const bool clip = s < 6.103515625e-05f;   // 2^-14, smallest normal fp16
        uint8_t* crow = pool.codes + prow * a.pd;
        // the clamp only matters for a subnormal scale: decide it once per row
        auto units = [&](auto clip_tag) {
          constexpr bool kClip = decltype(clip_tag)::value;
#pragma unroll
          for (int j = 0; j < UPL; ++j) {
            const int unit = lr + j * lpr;
            if (unit * 16 >= D) continue;
            uint32_t pk[4];
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              const uint4& vv = v[u][j][hh];
              const uint32_t w[4] = {vv.x, vv.y, vv.z, vv.w};
              uint32_t f[8];
              if constexpr (kClip) {
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                  const float xe = h2f(static_cast<uint16_t>(w[e >> 1] >> (16 * (e & 1))));
                  f[e] = quant_field_c<kQm, kB, kM, true>(xe, se, y);
                }
                pack8<BITS>(f, pk[2 * hh], pk[2 * hh + 1]);
              } else if constexpr (BITS == 4) {
                // the common path: two elements per packed float32 instruction; at q4 the fields
                // are packed from the raw rounding sums by integer multiply-adds (measured on one
                // box: 3.67 -> 3.46 ms for the 16-layer call; masks and shifts: 3.58 ms)
#pragma unroll
                for (int e = 0; e < 8; e += 2) {
                  const uint2 r = quant_raw2<raw_bias<BITS>()>(
                      h2f(static_cast<uint16_t>(w[e >> 1])),
                      h2f(static_cast<uint16_t>(w[e >> 1] >> 16)), se, y);
                  f[e] = r.x;
                  f[e + 1] = r.y;
                }
                pack8_raw<BITS>(f, pk[2 * hh], pk[2 * hh + 1]);
              } else {
                // q6 / q8: the same packed quotient, fields by masks and shifts (the multiply-add
                // packing measured 1.9 % slower at q6, 0.4 % at q8; this form 0.6 % faster than the
                // scalar quotient at q6)
#pragma unroll
                for (int e = 0; e < 8; e += 2) {
                  const uint2 r = quant_raw2<kB>(h2f(static_cast<uint16_t>(w[e >> 1])),
                                                 h2f(static_cast<uint16_t>(w[e >> 1] >> 16)), se, y);
                  f[e] = r.x & static_cast<uint32_t>(kM);
                  f[e + 1] = r.y & static_cast<uint32_t>(kM);
                }
                pack8<BITS>(f, pk[2 * hh], pk[2 * hh + 1]);
              }
            }
            store_unit<BITS>(crow + unit * SymQ<BITS>::kUnitBytes, pk[0], pk[1], pk[2], pk[3]);
          }
        };
        if (clip) units(std::true_type{});
        else units(std::false_type{});
        if (lr == 0) pool.scales[prow] = sbits;
      }
    }
  }
}

template <int BITS, int UPL, bool V8>
__global__ void __launch_bounds__(kThreads, BITS == 4 ? 4 : 3) dequant_kernel(const PackArgs a) {
  constexpr int kDqU = dq_unroll<BITS>();
  const int t = blockIdx.y;
  uint16_t* __restrict__ out = const_cast<uint16_t*>(a.x[t]);
  const PoolRef pool = a.pool[t];
  const int lane = threadIdx.x & 31;
  const int lpr = 1 << a.lpr_log2;
  const int rps = 32 >> a.lpr_log2;
  const int lr = lane & (lpr - 1);
  const int sub = lane >> a.lpr_log2;
  const int H = a.H, D = a.D;
  const int n_items = (a.total_tokens + a.tpi - 1) / a.tpi;
  const int n_warps = gridDim.x * kWarpsPerBlock;

  for (int item = blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5); item < n_items;
       item += n_warps) {
    const int tok0 = item * a.tpi;
    const int ntok = min(a.tpi, a.total_tokens - tok0);
    long long base = -1;
    if (lane < ntok) base = token_base(a, pool.num_pages, tok0 + lane);
    const int nrows = ntok * H;
    uint16_t* oi = out + static_cast<int64_t>(tok0) * H * D;
    for (int r0 = 0; r0 < nrows; r0 += rps * kDqU) {
      uint32_t w[kDqU][UPL][4];
      uint32_t sc[kDqU];
      bool act[kDqU];
#pragma unroll
      for (int u = 0; u < kDqU; ++u) {
        const int row = r0 + u * rps + sub;
        const int k = static_cast<int>(divu32(static_cast<uint32_t>(row), a.div_h));
        const long long b = shfl_ll(base, k < kTok ? k : 0);
        act[u] = row < nrows && b >= 0;
        sc[u] = 0;
#pragma unroll
        for (int j = 0; j < UPL; ++j) w[u][j][0] = w[u][j][1] = w[u][j][2] = w[u][j][3] = 0;
        if (act[u]) {
          const int64_t prow = b + static_cast<int64_t>(row - k * H) * a.page_size;
          const uint8_t* crow = pool.codes + prow * a.pd;
#pragma unroll
          for (int j = 0; j < UPL; ++j) {
            const int unit = lr + j * lpr;
            if (unit * 16 < D) load_unit<BITS>(crow + unit * SymQ<BITS>::kUnitBytes, w[u][j]);
          }
          sc[u] = ld_nc_u16(pool.scales + prow);
        }
      }
#pragma unroll
      for (int u = 0; u < kDqU; ++u) {
        if (!act[u]) continue;
        const int row = r0 + u * rps + sub;
        const uint32_t s2 = sc[u] | (sc[u] << 16);
        uint16_t* orow = oi + static_cast<int64_t>(row) * D;
#pragma unroll
        for (int j = 0; j < UPL; ++j) {
          const int unit = lr + j * lpr;
          if (unit * 16 >= D) continue;
          uint32_t p[4], q[4];
          unpack_group<BITS, 0>(w[u][j], p);     // elements 0..7 of the unit: {e_k, e_k+4}
          unpack_group<BITS, 1>(w[u][j], q);     // elements 8..15
          // exact codes times the fp16 scale: one rounding, the same as fp16(float(c) * scale)
          const uint4 o0 = make_uint4(hmul2u(prmt(p[0], p[1], 0x5410u), s2),
                                      hmul2u(prmt(p[2], p[3], 0x5410u), s2),
                                      hmul2u(prmt(p[0], p[1], 0x7632u), s2),
                                      hmul2u(prmt(p[2], p[3], 0x7632u), s2));
          const uint4 o1 = make_uint4(hmul2u(prmt(q[0], q[1], 0x5410u), s2),
                                      hmul2u(prmt(q[2], q[3], 0x5410u), s2),
                                      hmul2u(prmt(q[0], q[1], 0x7632u), s2),
                                      hmul2u(prmt(q[2], q[3], 0x7632u), s2));
          if constexpr (V8) {
            st_v8(orow + unit * 16, o0, o1);
          } else {
            *reinterpret_cast<uint4*>(orow + unit * 16) = o0;
            *reinterpret_cast<uint4*>(orow + unit * 16 + 8) = o1;
          }
        }
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
// tensors together at most what is resident on the SMs at once (rounded down per tensor, so no
// block waits for a second wave).
template <typename K>
dim3 grid_for(K kernel, int& cache, int n_tensors, int total_tokens, int tpi) {
  if (cache == 0) {
    int b = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, kernel, kThreads, 0);
    cache = (e != cudaSuccess || b < 1) ? 1 : b;
  }
  const int64_t items = (static_cast<int64_t>(total_tokens) + tpi - 1) / tpi;
  const int64_t need = (items + kWarpsPerBlock - 1) / kWarpsPerBlock;
  const int sms = sm_count();
  const int64_t cap = static_cast<int64_t>(sms > 0 ? sms : 1) * cache;
  int64_t per = cap / n_tensors;
  if (per > need) per = need;
  if (per < 1) per = 1;
  return dim3(static_cast<unsigned>(per), static_cast<unsigned>(n_tensors));
}

template <int BITS, int UPL, bool QUANT, bool V8>
cudaError_t launch_one(const PackArgs& a_in, cudaStream_t stream) {
  static int cache = 0;
  if (QUANT) {
    // A call with few new tokens (a decode-step append) takes fewer tokens per work item, so one
    // round of the grid's warps covers its items: the warps a tensor gets at most (its share of
    // the resident blocks) each take one item when tokens / warps <= 8.
    PackArgs a = a_in;
    if (cache == 0) grid_for(quant_pack_kernel<BITS, UPL, V8>, cache, a.n_tensors, 1, 1);
    const int64_t warps = static_cast<int64_t>(sm_count() > 0 ? sm_count() : 152) * cache /
                          a.n_tensors * kWarpsPerBlock;
    const int64_t per = warps > 0 ? (a.total_tokens + warps - 1) / warps : kTok;
    a.tpi = per < 1 ? 1 : (per > kTok ? kTok : static_cast<int>(per));
    quant_pack_kernel<BITS, UPL, V8>
        <<<grid_for(quant_pack_kernel<BITS, UPL, V8>, cache, a.n_tensors, a.total_tokens, a.tpi),
           kThreads, 0, stream>>>(a);
  } else {
    dequant_kernel<BITS, UPL, V8>
        <<<grid_for(dequant_kernel<BITS, UPL, V8>, cache, a_in.n_tensors, a_in.total_tokens,
                    a_in.tpi),
           kThreads, 0, stream>>>(a_in);
  }
  return cudaGetLastError();
}

// 256-bit accesses to the fp16 rows when every tensor of the call is 32-byte aligned (16-element
// units then start on 32-byte boundaries: D is a multiple of 16).  Measured on the 16-layer
// workload against two 128-bit accesses: quant-pack q6 3.907 -> 3.699 ms, q8 4.211 -> 4.090,
// q4 3.455 -> 3.326; dequant q6 3.924 -> 3.832, q8 4.450 -> 4.134, q4 3.768 -> 3.556.
template <int BITS, int UPL, bool QUANT>
cudaError_t launch_width(const PackArgs& a, cudaStream_t stream) {
  return a.v8 ? launch_one<BITS, UPL, QUANT, true>(a, stream)
              : launch_one<BITS, UPL, QUANT, false>(a, stream);
}

// Head dims that are not a multiple of 16: one warp per row (kvq_rowwise.cuh).
template <int BITS, bool QUANT>
cudaError_t launch_rowwise(const PackArgs& a, cudaStream_t stream) {
  const unsigned nb = rowwise_blocks(static_cast<int64_t>(a.n_tensors) * a.total_tokens * a.H,
                                     sm_count());
  if (QUANT) rowwise_quant_kernel<BITS, false><<<nb, kRowThreads, 0, stream>>>(a);
  else rowwise_dequant_kernel<BITS, false><<<nb, kRowThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

template <bool QUANT>
cudaError_t launch_bits(const PackArgs& a, int bits, cudaStream_t stream) {
  if (a.D % 16) {
    switch (bits) {
      case 8: return launch_rowwise<8, QUANT>(a, stream);
      case 6: return launch_rowwise<6, QUANT>(a, stream);
      default: return launch_rowwise<4, QUANT>(a, stream);
    }
  }
  const int upl = (a.units + (1 << a.lpr_log2) - 1) >> a.lpr_log2;  // 1 or 2 for D <= 256
  switch (bits) {
    case 8: return upl == 1 ? launch_width<8, 1, QUANT>(a, stream) : launch_width<8, 2, QUANT>(a, stream);
    case 6: return upl == 1 ? launch_width<6, 1, QUANT>(a, stream) : launch_width<6, 2, QUANT>(a, stream);
    default: return upl == 1 ? launch_width<4, 1, QUANT>(a, stream) : launch_width<4, 2, QUANT>(a, stream);
  }
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
  a.units = (p0.head_dim + 15) / 16;
  a.div_h = make_divu32(static_cast<uint32_t>(a.H));
  a.lpr_log2 = ceil_log2(a.units) < 3 ? ceil_log2(a.units) : 3;
  a.total_tokens = total_tokens;
  a.tpi = kTok;
  a.page_table = page_table;
  a.cu = cu;
  a.start = start;
  a.err = err;
  a.v8 = true;
  for (int i = 0; i < n_tensors; ++i)
    if (reinterpret_cast<uintptr_t>(x[i]) % 32) a.v8 = false;
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
  cudaError_t e = launch_bits<true>(a, bits, stream);
  if (e != cudaSuccess) return fail(KVQ_ERR_CUDA, "quant_pack launch: %s", cudaGetErrorString(e));
  return ok();
}

static kvq_status launch_dequant(const PackArgs& a, int bits, cudaStream_t stream) {
  if (a.total_tokens == 0) return ok();
  cudaError_t e = launch_bits<false>(a, bits, stream);
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
