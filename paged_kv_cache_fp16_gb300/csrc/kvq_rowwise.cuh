// Quant-pack and dequant for head dims that are not a multiple of 16 (plain and with fp16 side
// channels).
//
// MTPLX pull request #267, "feat(kv-cache): add q6 paged KV quantization", packed_dim sentence:
// q6 needs only D % 4 == 0 (four fields per three bytes), q4 D % 2 == 0, q8 any D.  The fast
// kernels cut a row into 16-element units; these take every other D <= 256 the pages allow.  One
// warp per row; lane i owns the row's packing groups i, i + 32, ... (a q6 quad: four fields in
// three bytes; a q4 pair in one byte; a q8 byte), so every packed byte has one writer.  The scale,
// the fields, the outlier keys and the reconstruction are the same device arithmetic as the fast
// kernels (row_scale_f32, quant_field, fp16(code * scale)), so the results are bit-identical to
// theirs and to the oracle.  Loads and stores are scalar: the rows are not 16-byte aligned.
//
// The including file provides the argument struct (fields x, pool, page_table, cu, start, err,
// n_tensors, total_tokens, H, D, page_size, pd, max_pages, nseq; with side channels also side,
// k, n_sink) -- PackArgs in quant_pack.cu, SideArgs in side.cu.
#pragma once

#include <cstdint>
#include <cuda_fp16.h>

#include "kvq_device.cuh"
#include "kvq_math.cuh"

namespace kvq {

constexpr int kRowThreads = 256;
constexpr int kRowWarps = kRowThreads / 32;

template <int BITS> struct RowGroup;
template <> struct RowGroup<8> { static constexpr int kElems = 1, kBytes = 1; };
template <> struct RowGroup<6> { static constexpr int kElems = 4, kBytes = 3; };
template <> struct RowGroup<4> { static constexpr int kElems = 2, kBytes = 1; };

// Groups a lane owns at most: D / elems / 32 for D <= 256 (q8: 8, q4: 4, q6: 2).
template <int BITS> constexpr int row_slots() { return 256 / RowGroup<BITS>::kElems / 32; }

// Row r of the call -> tensor t, token tok, head h; physical row (or -1), sequence, position.
template <typename Args>
__device__ __forceinline__ int64_t row_place(const Args& a, int64_t r, int& t, int& tok, int& h,
                                             int& s, int64_t& pos) {
  const int64_t per_t = static_cast<int64_t>(a.total_tokens) * a.H;
  t = static_cast<int>(r / per_t);
  const int64_t rr = r - t * per_t;
  tok = static_cast<int>(rr / a.H);
  h = static_cast<int>(rr - static_cast<int64_t>(tok) * a.H);
  s = find_seq(a.cu, a.nseq, a.total_tokens, tok);
  pos = static_cast<int64_t>(__ldg(a.start + s)) + (tok - __ldg(a.cu + s));
  return locate_row(a.page_table, a.max_pages, a.page_size, a.H, a.pool[t].num_pages, s, pos, h,
                    a.err);
}

// Quantize + pack one row per warp.  SIDE: the row's k largest magnitudes (ties to the lower
// position) go to the side channel as (fp16 value, uint8 position) ascending by position, the
// dense row has them zeroed, and rows at positions < n_sink are copied into the sink buffer.
template <int BITS, bool SIDE, typename Args>
__global__ void __launch_bounds__(kRowThreads) rowwise_quant_kernel(const Args a) {
  using RG = RowGroup<BITS>;
  constexpr int kE = RG::kElems, kNB = RG::kBytes, kSlots = row_slots<BITS>();
  constexpr int kQm = SymQ<BITS>::kQmax, kB = SymQ<BITS>::kBias, kM = SymQ<BITS>::kMask;
  const int lane = threadIdx.x & 31;
  const int D = a.D;
  const int n_groups = D / kE;
  const int64_t n_rows = static_cast<int64_t>(a.n_tensors) * a.total_tokens * a.H;
  for (int64_t r = static_cast<int64_t>(blockIdx.x) * kRowWarps + (threadIdx.x >> 5); r < n_rows;
       r += static_cast<int64_t>(gridDim.x) * kRowWarps) {
    int t, tok, h, s;
    int64_t pos;
    const int64_t prow = row_place(a, r, t, tok, h, s, pos);   // warp-uniform
    if (prow < 0) continue;
    const uint16_t* xr = a.x[t] + (static_cast<int64_t>(tok) * a.H + h) * D;
    uint16_t xb[kSlots][kE];
#pragma unroll
    for (int j = 0; j < kSlots; ++j) {
      const int g = lane + 32 * j;
#pragma unroll
      for (int e = 0; e < kE; ++e) xb[j][e] = g < n_groups ? __ldg(xr + g * kE + e) : 0;
    }
    if constexpr (SIDE) {
      if (pos < a.n_sink) {   // the exact row for the sink buffer
        uint16_t* sk = a.side[t].sink + ((static_cast<int64_t>(s) * a.n_sink + pos) * a.H + h) * D;
#pragma unroll
        for (int j = 0; j < kSlots; ++j) {
          const int g = lane + 32 * j;
#pragma unroll
          for (int e = 0; e < kE; ++e)
            if (g < n_groups) sk[g * kE + e] = xb[j][e];
        }
      }
      // k rounds of the row's largest remaining key: (|x| bits << 8) | (255 - position)
      uint32_t sel[kSlots] = {};   // bit e: element e of slot j is an outlier
      uint32_t okey[KVQ_MAX_OUTLIERS];
      for (int i = 0; i < a.k; ++i) {
        uint32_t best = 0;
#pragma unroll
        for (int j = 0; j < kSlots; ++j) {
          const int g = lane + 32 * j;
#pragma unroll
          for (int e = 0; e < kE; ++e) {
            const uint32_t key = ((static_cast<uint32_t>(xb[j][e]) & 0x7fffu) << 8) |
                                 static_cast<uint32_t>(255 - (g * kE + e));
            if (g < n_groups && !((sel[j] >> e) & 1u) && key > best) best = key;
          }
        }
        best = __reduce_max_sync(kFullMask, best);
        if (i < KVQ_MAX_OUTLIERS) okey[i] = best;
        const int p = 255 - static_cast<int>(best & 0xffu);   // the winner's position
        const int gw = p / kE;
        if ((gw & 31) == lane) {
#pragma unroll
          for (int j = 0; j < kSlots; ++j)
            if (j == (gw >> 5)) sel[j] |= 1u << (p - gw * kE);
        }
      }
      // the outliers ascending by position: lane i < k stores the key of rank-i position
      if (lane < a.k) {
        const int pi = 255 - static_cast<int>(okey[lane] & 0xffu);
        int rank = 0;
        for (int i = 0; i < a.k; ++i) rank += (255 - static_cast<int>(okey[i] & 0xffu)) < pi;
        const int64_t o = prow * a.k + rank;
        a.side[t].out_idx[o] = static_cast<uint8_t>(pi);
        a.side[t].out_val[o] = __ldg(xr + pi);
      }
#pragma unroll
      for (int j = 0; j < kSlots; ++j)
#pragma unroll
        for (int e = 0; e < kE; ++e)
          if ((sel[j] >> e) & 1u) xb[j][e] = 0;
    }
    float amax = 0.f;
#pragma unroll
    for (int j = 0; j < kSlots; ++j)
#pragma unroll
      for (int e = 0; e < kE; ++e) amax = fmaxf(amax, fabsf(h2f(xb[j][e])));
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kFullMask, amax, o));
    const uint16_t sbits = f2h(row_scale_f32<kQm>(amax));
    const float sc = h2f(sbits);
    const float y = (sc == 0.f) ? 0.f : __frcp_rn(sc);
    const float se = (sc == 0.f) ? 1.f : sc;
    const bool clip = sc < 6.103515625e-05f;   // 2^-14, smallest normal fp16
    uint8_t* crow = a.pool[t].codes + prow * a.pd;
#pragma unroll
    for (int j = 0; j < kSlots; ++j) {
      const int g = lane + 32 * j;
      if (g >= n_groups) continue;
      uint32_t w = 0;
#pragma unroll
      for (int e = 0; e < kE; ++e)
        w |= quant_field<kQm, kB, kM>(h2f(xb[j][e]), se, y, clip) << (BITS * e);
#pragma unroll
      for (int b = 0; b < kNB; ++b) crow[g * kNB + b] = static_cast<uint8_t>(w >> (8 * b));
    }
    if (lane == 0) a.pool[t].scales[prow] = sbits;
  }
}

// Gather + unpack + dequantize one row per warp.  SIDE: rows at positions < n_sink are the sink
// buffer's exact rows; other rows get their outliers written over the dense reconstruction.
template <int BITS, bool SIDE, typename Args>
__global__ void __launch_bounds__(kRowThreads) rowwise_dequant_kernel(const Args a) {
  using RG = RowGroup<BITS>;
  constexpr int kE = RG::kElems, kNB = RG::kBytes, kSlots = row_slots<BITS>();
  constexpr int kB = SymQ<BITS>::kBias, kM = SymQ<BITS>::kMask;
  const int lane = threadIdx.x & 31;
  const int D = a.D;
  const int n_groups = D / kE;
  const int64_t n_rows = static_cast<int64_t>(a.n_tensors) * a.total_tokens * a.H;
  for (int64_t r = static_cast<int64_t>(blockIdx.x) * kRowWarps + (threadIdx.x >> 5); r < n_rows;
       r += static_cast<int64_t>(gridDim.x) * kRowWarps) {
    int t, tok, h, s;
    int64_t pos;
    const int64_t prow = row_place(a, r, t, tok, h, s, pos);   // warp-uniform
    if (prow < 0) continue;
    uint16_t* orow = const_cast<uint16_t*>(a.x[t]) + (static_cast<int64_t>(tok) * a.H + h) * D;
    if constexpr (SIDE) {
      if (pos < a.n_sink) {
        const uint16_t* sk =
            a.side[t].sink + ((static_cast<int64_t>(s) * a.n_sink + pos) * a.H + h) * D;
        for (int e = lane; e < D; e += 32) orow[e] = sk[e];
        continue;
      }
    }
    const float sc = h2f(ld_nc_u16(a.pool[t].scales + prow));
    const uint8_t* crow = a.pool[t].codes + prow * a.pd;
#pragma unroll
    for (int j = 0; j < kSlots; ++j) {
      const int g = lane + 32 * j;
      if (g >= n_groups) continue;
      uint32_t w = 0;
#pragma unroll
      for (int b = 0; b < kNB; ++b) w |= static_cast<uint32_t>(__ldg(crow + g * kNB + b)) << (8 * b);
#pragma unroll
      for (int e = 0; e < kE; ++e) {
        const int f = static_cast<int>((w >> (BITS * e)) & static_cast<uint32_t>(kM));
        const int c = BITS == 8 ? static_cast<int>(static_cast<int8_t>(f)) : f - kB;
        orow[g * kE + e] = f2h(static_cast<float>(c) * sc);   // exact product, one rounding
      }
    }
    if constexpr (SIDE) {
      __syncwarp();   // the dense stores of the row before the outliers overwrite theirs
      if (lane < a.k) {
        const int64_t o = prow * a.k + lane;
        orow[a.side[t].out_idx[o]] = a.side[t].out_val[o];
      }
    }
  }
}

// Grid of the row kernels: one warp per row, at most 16 blocks of 8 warps per SM.
inline unsigned rowwise_blocks(int64_t rows, int sms) {
  int64_t b = (rows + kRowWarps - 1) / kRowWarps;
  const int64_t cap = static_cast<int64_t>(sms > 0 ? sms : 152) * 16;
  if (b > cap) b = cap;
  return static_cast<unsigned>(b < 1 ? 1 : b);
}

}  // namespace kvq
