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
// Thread layout (the plain quant-pack kernel's): a warp takes a block of 8 new tokens (all their
// heads); lanes 0..7 locate one token each and broadcast it by shuffle.  A row is cut into
// 16-element units, 8 lanes share a row (fewer for short rows) and lane j of a row holds units j
// and j + 8, so one warp instruction serves 4 rows.
//
// Selection.  For k <= 3 by magnitude first: each lane sorts its elements' magnitudes two at a
// time (fp16 pairs through min/max networks) into its 4 largest, tags each (magnitude << 3) |
// lane so equal magnitudes of different lanes differ, and k + 1 rounds of a max over the row's
// lanes give the k-th largest magnitude M and the (k+1)-th, T, the dense row's amax (counted
// with multiplicity).  When M > T the outliers are exactly the elements with |x| > T, one half2
// compare per pair of elements.  When M == T (a tie at the threshold) positions decide: if any
// row of the warp step has one, the step selects again by keys.  Element x at position p has
// the key (|x| bits << 8) | (255 - p) (one byte permute per element): unique in the row, larger
// for a larger magnitude and, among equal magnitudes, for the lower position.  Each lane keeps
// its DEPTH largest keys (sorting networks, bitonic merges; DEPTH >= k + 1, or the lane's own
// remaining maximum is recomputed for the last round) and k + 1 rounds of a max over the row's
// lanes give the (k+1)-th largest key; an element is an outlier iff its key exceeds it.  k > 3
// always selects by keys.  Outliers are zeroed in the dense row, whose scale and codes are the
// quant-pack kernel's arithmetic (the fields packed by integer multiply-adds from the rounding
// sums, which keeps them off the integer-logic pipe).  Each lane notes its outliers in a bit
// mask; an outlier's place among the row's k (ascending by position) is the count of outliers
// before it, from the lanes' counts scanned over the row; the lane stores its own outliers, the
// fp16 values (with their signs) read back from the input row.
#include <type_traits>

#include <cuda_runtime.h>
#include <cuda_fp16.h>

#include "kvq_device.cuh"
#include "kvq_internal.h"
#include "kvq_math.cuh"
#include "kvq_divu32.cuh"
#include "kvq_rowwise.cuh"

namespace kvq {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kTok = 8;   // new tokens per warp work item (all their heads)
constexpr int kQU = 1;    // quant-pack: warp steps with loads in flight
constexpr int kDU = 2;    // dequant: warp steps with loads in flight

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
  int units;     // 16-element units per row: D / 16
  int lpr_log2;  // lanes per row = 1 << lpr_log2 = min(next_pow2(units), 8)
  bool v8;       // every fp16 tensor 32-byte aligned: its 16-element units move in one 256-bit access
  bool items32;  // work items (tensor, token block) index in 32 bits: split by div_items
  bool seq32;    // nseq * total_tokens < 2^32: the sequence guess takes div_total
  DivU32 div_h, div_items;   // by the head count and the token blocks per tensor
  DivU32 div_ps, div_total;  // by the page size, by the token count (sequence guesses)
};

// Work item g -> its tensor (the item within the tensor is g - tensor * n_items).
__device__ __forceinline__ int item_tensor(const SideArgs& a, int64_t g, int n_items) {
  return a.items32 ? static_cast<int>(divu32(static_cast<uint32_t>(g), a.div_items))
                   : static_cast<int>(g / n_items);
}

// New token `tok` -> physical row of its head 0 ((page * H) * page_size + slot) or -1, with its
// sequence and position (the position clamped to int: it is only compared with n_sink).
__device__ __forceinline__ long long token_place(const SideArgs& a, int64_t num_pages, int tok,
                                                 int& s, int& pos) {
  s = a.seq32 ? find_seq(a.cu, a.nseq, tok, a.div_total)
              : find_seq(a.cu, a.nseq, a.total_tokens, tok);
  const int64_t p = static_cast<int64_t>(__ldg(a.start + s)) + (tok - __ldg(a.cu + s));
  pos = p > 0x7fffffffLL ? 0x7fffffff : static_cast<int>(p);
  return locate_row(a.page_table, a.max_pages, a.page_size, a.H, num_pages, s, p, 0, a.err,
                    a.div_ps);
}

__device__ __forceinline__ long long shfl_ll(long long v, int src) {
  const int lo = __shfl_sync(kFullMask, static_cast<int>(v & 0xffffffffLL), src);
  const int hi = __shfl_sync(kFullMask, static_cast<int>(v >> 32), src);
  return (static_cast<long long>(hi) << 32) | static_cast<unsigned int>(lo);
}

// ---------------------------------------------------------------------------- selection keys
// Compare-exchange: a >= b afterwards; P: in each half of a pair of non-negative fp16 values
// (for those, the fp16 order is the order of their bit patterns).
// |x| of both halves of an fp16 pair, as an fp16 operation (the compares can take it as an
// operand modifier).
__device__ __forceinline__ uint32_t habs_u(uint32_t x) {
  __half2 h = __habs2(*reinterpret_cast<const __half2*>(&x));
  return *reinterpret_cast<const uint32_t*>(&h);
}

template <bool P = false>
__device__ __forceinline__ void cx(uint32_t& a, uint32_t& b) {
  if constexpr (P) {
    uint32_t hi, lo;
    asm("max.f16x2 %0, %1, %2;" : "=r"(hi) : "r"(a), "r"(b));
    asm("min.f16x2 %0, %1, %2;" : "=r"(lo) : "r"(a), "r"(b));
    a = hi;
    b = lo;
  } else {
    const uint32_t hi = max(a, b);
    b = min(a, b);
    a = hi;
  }
}

template <bool P = false>
__device__ __forceinline__ uint32_t max_of(uint32_t a, uint32_t b) {
  if constexpr (P) {
    uint32_t d;
    asm("max.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
  } else {
    return max(a, b);
  }
}

template <bool P = false>
__device__ __forceinline__ void sort4(uint32_t& a, uint32_t& b, uint32_t& c, uint32_t& d) {
  cx<P>(a, b); cx<P>(c, d); cx<P>(a, c); cx<P>(b, d); cx<P>(b, c);
}

// A bitonic sequence t[0..N) -> descending (half-cleaners of Batcher's bitonic sorter).
template <int N, bool P = false>
__device__ __forceinline__ void bitonic_desc(uint32_t* t) {
#pragma unroll
  for (int len = N / 2; len >= 1; len /= 2) {
#pragma unroll
    for (int i = 0; i < N; ++i)
      if ((i & len) == 0) cx<P>(t[i], t[i + len]);
  }
}

// Keys of 8 consecutive elements (4 words of fp16 pairs); cb = 255 - position of the first.
__device__ __forceinline__ void keys8(const uint4& v, uint32_t cb, uint32_t k[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  const uint32_t c0 = cb | ((cb - 1u) << 16);   // bytes [255-p, 0, 255-(p+1), 0]
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t m = w[i] & 0x7fff7fffu;       // |x| of both halves
    const uint32_t c = c0 - 0x00020002u * static_cast<uint32_t>(i);
    k[2 * i] = prmt(m, c, 0x5104u);              // [255-p, |x| lo byte, |x| hi byte, 0]
    k[2 * i + 1] = prmt(m, c, 0x7326u);
  }
}

// k[0..8) -> k[0..DEPTH) = its DEPTH largest, descending (DEPTH 4 or 8).
template <int DEPTH>
__device__ __forceinline__ void top_of8(uint32_t k[8]) {
  sort4(k[0], k[1], k[2], k[3]);
  sort4(k[4], k[5], k[6], k[7]);
  if constexpr (DEPTH == 4) {
    // the 4 largest of two descending lists: max(a_i, b_{3-i}) is bitonic
#pragma unroll
    for (int i = 0; i < 4; ++i) k[i] = max(k[i], k[7 - i]);
    bitonic_desc<4>(k);
  } else {
    uint32_t t[8] = {k[0], k[1], k[2], k[3], k[7], k[6], k[5], k[4]};   // down then up
    bitonic_desc<8>(t);
#pragma unroll
    for (int i = 0; i < 8; ++i) k[i] = t[i];
  }
}

// run = the DEPTH largest of two descending lists run, g.
template <int DEPTH, bool P = false>
__device__ __forceinline__ void merge_top(uint32_t* run, const uint32_t* g) {
#pragma unroll
  for (int i = 0; i < DEPTH; ++i) run[i] = max_of<P>(run[i], g[DEPTH - 1 - i]);
  bitonic_desc<DEPTH, P>(run);
}

// Exact selection by keys: thr = the row's (k+1)-th largest key, last = its k-th (0 if k = 0).
// Each lane keeps its DEPTH largest keys; k + 1 rounds of a max over the row's lanes take the
// winners, the lane that held each popping it from its list (all lanes take part).
template <int UPL, int DEPTH>
__device__ __forceinline__ void key_select(const uint4 (&v)[UPL][2], int lr, int lpr, int D,
                                           int k, uint32_t& thr, uint32_t& last) {
  uint32_t top[DEPTH];
#pragma unroll
  for (int i = 0; i < DEPTH; ++i) top[i] = 0u;
#pragma unroll
  for (int j = 0; j < UPL; ++j) {
    const int unit = lr + j * lpr;
    if (unit * 16 >= D) continue;
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      uint32_t g[8];
      keys8(v[j][hh], 255u - static_cast<uint32_t>(16 * unit + 8 * hh), g);
      top_of8<DEPTH>(g);
      if (j == 0 && hh == 0) {
#pragma unroll
        for (int i = 0; i < DEPTH; ++i) top[i] = g[i];
      } else {
        merge_top<DEPTH>(top, g);
      }
    }
  }
  thr = 0u;
  last = 0u;
#pragma unroll
  for (int j = 0; j <= KVQ_MAX_OUTLIERS; ++j) {
    if (j > k) break;
    uint32_t m = top[0];
    if (j >= DEPTH && j == k) {
      // this lane may have given all DEPTH listed keys: its largest key below the last
      // outlier's, rebuilt from the elements
      m = 0u;
#pragma unroll
      for (int jj = 0; jj < UPL; ++jj) {
        const int unit = lr + jj * lpr;
        if (unit * 16 >= D) continue;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          uint32_t g[8];
          keys8(v[jj][hh], 255u - static_cast<uint32_t>(16 * unit + 8 * hh), g);
#pragma unroll
          for (int e = 0; e < 8; ++e) m = max(m, g[e] < last ? g[e] : 0u);
        }
      }
    }
#pragma unroll
    for (int o = 4; o >= 1; o >>= 1)
      if (o < lpr) m = max(m, __shfl_xor_sync(kFullMask, m, o));
    if (j == k) {
      thr = m;
      break;
    }
    last = m;
    const bool pop = top[0] == m;
#pragma unroll
    for (int i = 0; i + 1 < DEPTH; ++i) top[i] = pop ? top[i + 1] : top[i];
    top[DEPTH - 1] = pop ? 0u : top[DEPTH - 1];
  }
}

// Selection by magnitude alone (k <= 3): T = the row's (k+1)-th largest magnitude and M = its
// k-th (fp16 bits, counted with multiplicity; M = 0 if k = 0).  Each lane sorts its magnitudes
// two at a time (fp16 pairs) into the 4 largest of its lower and of its upper halves, merges the two lists, tags each entry (magnitude << 3) | lane so that equal
// magnitudes of different lanes differ, and k + 1 rounds of a max over the row's lanes take the
// winners.  When M > T the outliers are exactly the elements with |x| > T; when M == T (a tie
// at the threshold) positions decide, and the keys are needed.
template <int UPL>
__device__ __forceinline__ void magnitude_select(const uint4 (&v)[UPL][2], int lr, int lpr,
                                                 int D, int k, uint32_t& T, uint32_t& M) {
  uint32_t run[4] = {0u, 0u, 0u, 0u};
#pragma unroll
  for (int j = 0; j < UPL; ++j) {
    if ((lr + j * lpr) * 16 >= D) continue;
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      uint32_t g[4] = {habs_u(v[j][hh].x), habs_u(v[j][hh].y), habs_u(v[j][hh].z),
                       habs_u(v[j][hh].w)};
      sort4<true>(g[0], g[1], g[2], g[3]);
      if (j == 0 && hh == 0) {
#pragma unroll
        for (int i = 0; i < 4; ++i) run[i] = g[i];
      } else {
        merge_top<4, true>(run, g);
      }
    }
  }
  // the lower-half list against the upper-half list reversed: a bitonic sequence per half
  uint32_t top[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) top[i] = max_of<true>(run[i], prmt(run[3 - i], 0u, 0x1032u));
  bitonic_desc<4, true>(top);
#pragma unroll
  for (int i = 0; i < 4; ++i) top[i] = ((top[i] & 0x7fffu) << 3) | static_cast<uint32_t>(lr);
  uint32_t thr = 0u, last = 0u;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    if (j > k) break;
    uint32_t m = top[0];
#pragma unroll
    for (int o = 4; o >= 1; o >>= 1)
      if (o < lpr) m = max(m, __shfl_xor_sync(kFullMask, m, o));
    if (j == k) {
      thr = m;
      break;
    }
    last = m;
    const bool pop = top[0] == m;
    // at most k <= 3 pops: the last entry never needs clearing (after three pops it is the head)
#pragma unroll
    for (int i = 0; i < 3; ++i) top[i] = pop ? top[i + 1] : top[i];
  }
  T = thr >> 3;
  M = last >> 3;
}

// ------------------------------------------------------------------------------ quant-pack
template <int BITS, int UPL, int DEPTH, bool V8>
__global__ void __launch_bounds__(kThreads, 4) quant_pack_side_kernel(const SideArgs a) {
  constexpr int kQm = SymQ<BITS>::kQmax;
  const int lane = threadIdx.x & 31;
  const int lpr = 1 << a.lpr_log2;
  const int rps = 32 >> a.lpr_log2;
  const int lr = lane & (lpr - 1);
  const int sub = lane >> a.lpr_log2;
  const int H = a.H, D = a.D, k = a.k;
  const int n_items = (a.total_tokens + kTok - 1) / kTok;
  const int64_t n_work = static_cast<int64_t>(a.n_tensors) * n_items;
  const int n_warps = gridDim.x * kWarps;

  for (int64_t g = blockIdx.x * kWarps + (threadIdx.x >> 5); g < n_work; g += n_warps) {
    const int t = item_tensor(a, g, n_items);
    const int item = static_cast<int>(g - static_cast<int64_t>(t) * n_items);
    const uint16_t* __restrict__ x = a.x[t];
    const PoolRef pool = a.pool[t];
    const SideRef sd = a.side[t];
    const int tok0 = item * kTok;
    const int ntok = min(kTok, a.total_tokens - tok0);
    long long base = -1;
    int my_s = 0, my_pos = 0;
    if (lane < ntok) base = token_place(a, pool.num_pages, tok0 + lane, my_s, my_pos);
    const int nrows = ntok * H;
    const uint16_t* xi = x + static_cast<int64_t>(tok0) * H * D;
    for (int r0 = 0; r0 < nrows; r0 += rps * kQU) {
      uint4 v[kQU][UPL][2];
#pragma unroll
      for (int u = 0; u < kQU; ++u) {
        const int row = r0 + u * rps + sub;
#pragma unroll
        for (int j = 0; j < UPL; ++j) {
          const int e0 = (lr + j * lpr) * 16;
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
      for (int u = 0; u < kQU; ++u) {
        const int row = r0 + u * rps + sub;
        const int kt = static_cast<int>(divu32(static_cast<uint32_t>(row), a.div_h));
        const int src = kt < kTok ? kt : 0;
        const long long b = shfl_ll(base, src);
        const int s = __shfl_sync(kFullMask, my_s, src);
        const int pos = __shfl_sync(kFullMask, my_pos, src);
        // T = the dense row's amax (fp16 bits); by_key: outliers decided by key, not |x| > T
        uint32_t T, thr = 0u;
        bool by_key;
        if constexpr (DEPTH == 4) {
          uint32_t M;
          magnitude_select<UPL>(v[u], lr, lpr, D, k, T, M);
          by_key = false;
          if (__any_sync(kFullMask, k > 0 && M == T && row < nrows)) {
            uint32_t last;
            key_select<UPL, 4>(v[u], lr, lpr, D, k, thr, last);
            T = thr >> 8;
            by_key = k > 0 && (last >> 8) == T;
          }
        } else {
          uint32_t last;
          key_select<UPL, DEPTH>(v[u], lr, lpr, D, k, thr, last);
          T = thr >> 8;
          by_key = k > 0 && (last >> 8) == T;
        }
        const bool valid = row < nrows && b >= 0;
        const int h = row - kt * H;
        const int64_t prow = b + static_cast<int64_t>(h) * a.page_size;
        const uint16_t sbits = f2h(row_scale_f32<kQm>(h2f(static_cast<uint16_t>(T))));
        const float sc = h2f(sbits);
        const float y = (sc == 0.f) ? 0.f : __frcp_rn(sc);
        const float se = (sc == 0.f) ? 1.f : sc;
        const bool clip = sc < 6.103515625e-05f;   // 2^-14, smallest normal fp16
        const uint32_t T2 = T | (T << 16);
        uint8_t* crow = pool.codes + prow * a.pd;
        // the lane's outliers: bit 16 j + 8 hh + e for element e of half hh of its unit j
        uint32_t omask = 0u;
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
              uint32_t w[4] = {vv.x, vv.y, vv.z, vv.w};
              // outliers (|x| > T, or at a tie key > thr) as 0xffff per half, zeroed
              uint32_t gt[4];
              if (!by_key) {
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                  gt[i] = __hgt2_mask(__habs2(*reinterpret_cast<const __half2*>(&w[i])),
                                      *reinterpret_cast<const __half2*>(&T2));
                }
              } else {
                uint32_t g[8];
                keys8(vv, 255u - static_cast<uint32_t>(16 * unit + 8 * hh), g);
#pragma unroll
                for (int i = 0; i < 4; ++i)
                  gt[i] = (g[2 * i] > thr ? 0x0000ffffu : 0u) |
                          (g[2 * i + 1] > thr ? 0xffff0000u : 0u);
              }
#pragma unroll
              for (int i = 0; i < 4; ++i) w[i] &= ~gt[i];
              // one flag byte per element, then one bit per element in the product's top byte
              const uint32_t fx = prmt(gt[0], gt[1], 0x7531u), fy = prmt(gt[2], gt[3], 0x7531u);
              const uint32_t fb = ((fx & 0x08040201u) | (fy & 0x80402010u)) * 0x01010101u;
              const int gi = 2 * j + hh;
              omask = prmt(omask, fb, (0x3210u & ~(0xfu << (4 * gi))) | (7u << (4 * gi)));
              uint32_t f[8];
              if constexpr (kClip) {
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                  const float xe = h2f(static_cast<uint16_t>(w[e >> 1] >> (16 * (e & 1))));
                  f[e] = quant_raw<kQm, raw_bias<BITS>(), true>(xe, se, y);
                }
              } else {   // two elements per packed float32 instruction
#pragma unroll
                for (int e = 0; e < 8; e += 2) {
                  const uint2 r = quant_raw2<raw_bias<BITS>()>(
                      h2f(static_cast<uint16_t>(w[e >> 1])),
                      h2f(static_cast<uint16_t>(w[e >> 1] >> 16)), se, y);
                  f[e] = r.x;
                  f[e + 1] = r.y;
                }
              }
              pack8_raw<BITS>(f, pk[2 * hh], pk[2 * hh + 1]);
            }
            if (valid)
              store_unit<BITS>(crow + unit * SymQ<BITS>::kUnitBytes, pk[0], pk[1], pk[2], pk[3]);
          }
        };
        if (clip) units(std::true_type{});
        else units(std::false_type{});
        if (valid && lr == 0) pool.scales[prow] = sbits;
        // outliers, ascending by position: an outlier's rank is the count of the row's outliers
        // in earlier units (the units j * lpr + i, i < lpr, precede those of j + 1) plus those
        // before it in its own unit; the counts per j scanned over the row's lanes
        const uint32_t cnt = static_cast<uint32_t>(__popc(omask & 0xffffu)) |
                             (static_cast<uint32_t>(__popc(omask >> 16)) << 16);
        uint32_t incl = cnt;
#pragma unroll
        for (int o = 1; o < 8; o <<= 1) {
          if (o >= lpr) break;
          const uint32_t n = __shfl_up_sync(kFullMask, incl, o, lpr);
          if (lr >= o) incl += n;
        }
        const uint32_t tot = __shfl_sync(kFullMask, incl, lpr - 1, lpr);
        const uint32_t ex = incl - cnt;
        if (valid) {
          for (uint32_t mk = omask; mk != 0u; mk &= mk - 1u) {
            const int n = __ffs(static_cast<int>(mk)) - 1;
            const bool hi = n >= 16;
            const uint32_t before = omask & ((1u << n) - 1u) & (hi ? 0xffff0000u : 0x0000ffffu);
            const uint32_t rank = (hi ? (tot & 0xffffu) + (ex >> 16) : (ex & 0xffffu)) +
                                  static_cast<uint32_t>(__popc(before));
            const int p = 16 * (lr + (hi ? lpr : 0)) + (n & 15);
            if (rank < static_cast<uint32_t>(k)) {
              const uint16_t val = __ldg(xi + static_cast<int64_t>(row) * D + p);
              sd.out_idx[prow * k + rank] = static_cast<uint8_t>(p);
              sd.out_val[prow * k + rank] = val;
            }
          }
        }
        if (valid && pos < a.n_sink) {
          uint16_t* dst = sd.sink + ((static_cast<int64_t>(s) * a.n_sink + pos) * H + h) * D;
#pragma unroll
          for (int j = 0; j < UPL; ++j) {
            const int e0 = (lr + j * lpr) * 16;
            if (e0 >= D) continue;
            *reinterpret_cast<uint4*>(dst + e0) = v[u][j][0];
            *reinterpret_cast<uint4*>(dst + e0 + 8) = v[u][j][1];
          }
        }
      }
    }
  }
}

// -------------------------------------------------------------------------------- dequant
// The plain dequant kernel's layout and arithmetic (fp16(c * scale), one rounding); then, after a
// warp barrier that orders the stores, the row's lane j < k writes outlier j over its position.
// Rows at positions < n_sink are copied from the sink buffer instead.
template <int BITS, int UPL, bool V8>
__global__ void __launch_bounds__(kThreads) dequant_side_kernel(const SideArgs a) {
  const int lane = threadIdx.x & 31;
  const int lpr = 1 << a.lpr_log2;
  const int rps = 32 >> a.lpr_log2;
  const int lr = lane & (lpr - 1);
  const int sub = lane >> a.lpr_log2;
  const int H = a.H, D = a.D, k = a.k;
  const int n_items = (a.total_tokens + kTok - 1) / kTok;
  const int64_t n_work = static_cast<int64_t>(a.n_tensors) * n_items;
  const int n_warps = gridDim.x * kWarps;

  for (int64_t g = blockIdx.x * kWarps + (threadIdx.x >> 5); g < n_work; g += n_warps) {
    const int t = item_tensor(a, g, n_items);
    const int item = static_cast<int>(g - static_cast<int64_t>(t) * n_items);
    uint16_t* __restrict__ out = const_cast<uint16_t*>(a.x[t]);
    const PoolRef pool = a.pool[t];
    const SideRef sd = a.side[t];
    const int tok0 = item * kTok;
    const int ntok = min(kTok, a.total_tokens - tok0);
    long long base = -1, sink_row = -1;   // sink_row: index of head 0's row in the sink buffer
    if (lane < ntok) {
      int s, pos;
      base = token_place(a, pool.num_pages, tok0 + lane, s, pos);
      if (pos < a.n_sink) sink_row = (static_cast<long long>(s) * a.n_sink + pos) * H;
    }
    const int nrows = ntok * H;
    uint16_t* oi = out + static_cast<int64_t>(tok0) * H * D;
    for (int r0 = 0; r0 < nrows; r0 += rps * kDU) {
      uint32_t w[kDU][UPL][4];
      uint32_t sc[kDU], ov[kDU];   // scale; outlier lr: position | value << 16
      bool act[kDU], dense[kDU];
#pragma unroll
      for (int u = 0; u < kDU; ++u) {
        const int row = r0 + u * rps + sub;
        const int kt = static_cast<int>(divu32(static_cast<uint32_t>(row), a.div_h));
        const int src = kt < kTok ? kt : 0;
        const long long b = shfl_ll(base, src);
        const bool snk = __shfl_sync(kFullMask, static_cast<int>(sink_row >= 0), src) != 0;
        act[u] = row < nrows && b >= 0;
        dense[u] = act[u] && !snk;
        sc[u] = ov[u] = 0;
#pragma unroll
        for (int j = 0; j < UPL; ++j) w[u][j][0] = w[u][j][1] = w[u][j][2] = w[u][j][3] = 0;
        if (dense[u]) {
          const int64_t prow = b + static_cast<int64_t>(row - kt * H) * a.page_size;
          const uint8_t* crow = pool.codes + prow * a.pd;
#pragma unroll
          for (int j = 0; j < UPL; ++j) {
            const int unit = lr + j * lpr;
            if (unit * 16 < D) load_unit<BITS>(crow + unit * SymQ<BITS>::kUnitBytes, w[u][j]);
          }
          sc[u] = ld_nc_u16(pool.scales + prow);
          if (lr < k)
            ov[u] = __ldg(sd.out_idx + prow * k + lr) |
                    (static_cast<uint32_t>(ld_nc_u16(sd.out_val + prow * k + lr)) << 16);
        }
      }
#pragma unroll
      for (int u = 0; u < kDU; ++u) {
        const int row = r0 + u * rps + sub;
        const int kt = static_cast<int>(divu32(static_cast<uint32_t>(row), a.div_h));
        const long long srow = shfl_ll(sink_row, kt < kTok ? kt : 0);
        if (!act[u]) continue;
        uint16_t* orow = oi + static_cast<int64_t>(row) * D;
        if (!dense[u]) {
          const uint16_t* sp = sd.sink + (srow + (row - kt * H)) * D;
#pragma unroll
          for (int j = 0; j < UPL; ++j) {
            const int e0 = (lr + j * lpr) * 16;
            if (e0 >= D) continue;
            *reinterpret_cast<uint4*>(orow + e0) = ld_nc_v4(sp + e0);
            *reinterpret_cast<uint4*>(orow + e0 + 8) = ld_nc_v4(sp + e0 + 8);
          }
          continue;
        }
        const uint32_t s2 = sc[u] | (sc[u] << 16);
#pragma unroll
        for (int j = 0; j < UPL; ++j) {
          const int unit = lr + j * lpr;
          if (unit * 16 >= D) continue;
          uint32_t p[4], q[4];
          unpack_group<BITS, 0>(w[u][j], p);
          unpack_group<BITS, 1>(w[u][j], q);
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
      // the dense stores of every lane come before the outlier stores over them
      __syncwarp();
#pragma unroll
      for (int u = 0; u < kDU; ++u) {
        const int row = r0 + u * rps + sub;
        uint16_t* orow = oi + static_cast<int64_t>(row) * D;
        if (dense[u] && lr < k) {
          const uint32_t d = ov[u] & 0xffu;
          if (d < static_cast<uint32_t>(D)) orow[d] = static_cast<uint16_t>(ov[u] >> 16);
        }
        if (k > lpr) {   // more outliers than lanes per row (short rows): lane lr also takes lr + lpr, ...
          const int kt = static_cast<int>(divu32(static_cast<uint32_t>(row), a.div_h));
          const long long b = shfl_ll(base, kt < kTok ? kt : 0);
          if (dense[u]) {
            const int64_t prow = b + static_cast<int64_t>(row - kt * H) * a.page_size;
            for (int j = lr + lpr; j < k; j += lpr) {
              const uint32_t d = __ldg(sd.out_idx + prow * k + j);
              if (d < static_cast<uint32_t>(D)) orow[d] = ld_nc_u16(sd.out_val + prow * k + j);
            }
          }
        }
      }
    }
  }
}

// Persistent 1-D grid over all (tensor, token block) work items: at most the blocks that are
// resident on the SMs at once, so no block waits for a second wave.
template <typename K>
unsigned side_grid(K kernel, int& cache, int n_tensors, int total_tokens) {
  if (cache == 0) {
    int b = 0;
    const cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, kernel, kThreads, 0);
    cache = (e != cudaSuccess || b < 1) ? 1 : b;
  }
  const int64_t items = (static_cast<int64_t>(total_tokens) + kTok - 1) / kTok * n_tensors;
  const int64_t need = (items + kWarps - 1) / kWarps;
  const int sms = sm_count();
  const int64_t cap = static_cast<int64_t>(sms > 0 ? sms : 1) * cache;
  return static_cast<unsigned>(need < cap ? (need > 0 ? need : 1) : cap);
}

template <int BITS, int UPL, int DEPTH, bool V8>
void launch_quant_w(const SideArgs& a, cudaStream_t cs) {
  static int cache = 0;
  auto kern = quant_pack_side_kernel<BITS, UPL, DEPTH, V8>;
  kern<<<side_grid(kern, cache, a.n_tensors, a.total_tokens), kThreads, 0, cs>>>(a);
}

template <int BITS, int UPL, bool V8>
void launch_dequant_w(const SideArgs& a, cudaStream_t cs) {
  static int cache = 0;
  auto kern = dequant_side_kernel<BITS, UPL, V8>;
  kern<<<side_grid(kern, cache, a.n_tensors, a.total_tokens), kThreads, 0, cs>>>(a);
}

// 256-bit accesses to the fp16 rows when every tensor of the call is 32-byte aligned.
template <int BITS, int UPL, int DEPTH>
void launch_quant(const SideArgs& a, cudaStream_t cs) {
  a.v8 ? launch_quant_w<BITS, UPL, DEPTH, true>(a, cs) : launch_quant_w<BITS, UPL, DEPTH, false>(a, cs);
}

template <int BITS, int UPL>
void launch_dequant(const SideArgs& a, cudaStream_t cs) {
  a.v8 ? launch_dequant_w<BITS, UPL, true>(a, cs) : launch_dequant_w<BITS, UPL, false>(a, cs);
}

template <int BITS>
void launch_side(bool quant, const SideArgs& a, cudaStream_t cs) {
  const int upl = (a.units + (1 << a.lpr_log2) - 1) >> a.lpr_log2;   // 1 or 2 for D <= 256
  if (quant) {
    const bool deep = a.k > 3;
    if (upl == 1) deep ? launch_quant<BITS, 1, 8>(a, cs) : launch_quant<BITS, 1, 4>(a, cs);
    else deep ? launch_quant<BITS, 2, 8>(a, cs) : launch_quant<BITS, 2, 4>(a, cs);
  } else {
    upl == 1 ? launch_dequant<BITS, 1>(a, cs) : launch_dequant<BITS, 2>(a, cs);
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
  a.v8 = true;
  for (int i = 0; i < n_tensors; ++i)
    if (reinterpret_cast<uintptr_t>(x[i]) % 32) a.v8 = false;
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
  a.units = p0.head_dim / 16;
  a.div_h = make_divu32(static_cast<uint32_t>(a.H));
  a.div_ps = make_divu32(static_cast<uint32_t>(a.page_size));
  a.seq32 = static_cast<int64_t>(total) * nseq < (1LL << 32);
  a.div_total = make_divu32(static_cast<uint32_t>(total));
  {
    const int64_t n_items = (static_cast<int64_t>(total) + kTok - 1) / kTok;
    a.items32 = n_items * n_tensors <= 0xffffffffLL;
    a.div_items = make_divu32(static_cast<uint32_t>(n_items));
  }
  a.lpr_log2 = 0;
  while ((1 << a.lpr_log2) < a.units && a.lpr_log2 < 3) ++a.lpr_log2;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  if (a.D % 16) {   // head dims that are not a multiple of 16: one warp per row
    const unsigned nb = rowwise_blocks(static_cast<int64_t>(n_tensors) * total * a.H, sm_count());
    switch (p0.bits) {
      case 8:
        if (quant) rowwise_quant_kernel<8, true><<<nb, kRowThreads, 0, cs>>>(a);
        else rowwise_dequant_kernel<8, true><<<nb, kRowThreads, 0, cs>>>(a);
        break;
      case 6:
        if (quant) rowwise_quant_kernel<6, true><<<nb, kRowThreads, 0, cs>>>(a);
        else rowwise_dequant_kernel<6, true><<<nb, kRowThreads, 0, cs>>>(a);
        break;
      default:
        if (quant) rowwise_quant_kernel<4, true><<<nb, kRowThreads, 0, cs>>>(a);
        else rowwise_dequant_kernel<4, true><<<nb, kRowThreads, 0, cs>>>(a);
        break;
    }
  } else {
    switch (p0.bits) {
      case 8: launch_side<8>(quant, a, cs); break;
      case 6: launch_side<6>(quant, a, cs); break;
      default: launch_side<4>(quant, a, cs); break;
    }
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
