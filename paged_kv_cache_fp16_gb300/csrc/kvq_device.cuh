// Device-side helpers shared by the libkvq kernels.
#pragma once

#include <cstdint>
#include <cuda_fp16.h>

#include "kvq.h"
#include "kvq_divu32.cuh"

namespace kvq {

constexpr unsigned kFullMask = 0xffffffffu;

// A pool as the kernels see it (bits/H/D/page_size are uniform per call and passed separately).
struct PoolRef {
  uint8_t* codes;
  uint16_t* scales;
  int64_t num_pages;
};

__device__ __forceinline__ void report(int32_t* err, int bit) {
  if (err) atomicOr(err, bit);
}

// Streaming 16-byte load that does not allocate in L1 (input read exactly once).
__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// The same for 32 bytes in one 256-bit access (the address must be 32-byte aligned).
__device__ __forceinline__ void ld_stream_v8(const void* p, uint4& lo, uint4& hi) {
  asm volatile("ld.global.nc.L1::no_allocate.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(lo.x), "=r"(lo.y), "=r"(lo.z), "=r"(lo.w), "=r"(hi.x), "=r"(hi.y),
                 "=r"(hi.z), "=r"(hi.w)
               : "l"(p));
}

// 32-byte coherent load in one 256-bit access (data the same launch also writes).
__device__ __forceinline__ void ld_v8(const void* p, uint4& lo, uint4& hi) {
  asm volatile("ld.global.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(lo.x), "=r"(lo.y), "=r"(lo.z), "=r"(lo.w), "=r"(hi.x), "=r"(hi.y),
                 "=r"(hi.z), "=r"(hi.w)
               : "l"(p)
               : "memory");
}

// 32-byte store in one 256-bit access (the address must be 32-byte aligned).
__device__ __forceinline__ void st_v8(void* p, const uint4& lo, const uint4& hi) {
  asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(lo.x),
               "r"(lo.y), "r"(lo.z), "r"(lo.w), "r"(hi.x), "r"(hi.y), "r"(hi.z), "r"(hi.w)
               : "memory");
}

__device__ __forceinline__ uint4 ld_nc_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

__device__ __forceinline__ uint2 ld_nc_v2(const void* p) {
  uint2 r;
  asm volatile("ld.global.nc.v2.u32 {%0,%1}, [%2];" : "=r"(r.x), "=r"(r.y) : "l"(p));
  return r;
}

__device__ __forceinline__ uint32_t ld_nc_u32(const void* p) {
  uint32_t r;
  asm volatile("ld.global.nc.u32 %0, [%1];" : "=r"(r) : "l"(p));
  return r;
}

__device__ __forceinline__ uint16_t ld_nc_u16(const void* p) {
  uint16_t r;
  asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(r) : "l"(p));
  return r;
}

// Largest s in [0, nseq) with cu[s] <= i.  For a well-formed cu (non-decreasing, cu[0] = 0,
// i < cu[nseq] = total) this is the sequence that owns new-token row i; for any cu it stays in
// range.  The guess g = i * nseq / total is checked first (cu[g] <= i < cu[g + 1], two loads in
// parallel): it is exact whenever the sequences add equal numbers of tokens (a decode-step
// append, a uniform prefill), which saves the binary search's chain of dependent loads; otherwise
// the search runs on the side of g that holds the answer.
// The search from a guess g in [0, nseq).
__device__ __forceinline__ int find_seq_from(const int32_t* __restrict__ cu, int nseq, int i,
                                             int g) {
  int lo = 0, hi = nseq - 1;
  if (nseq > 1) {
    const int c0 = __ldg(cu + g), c1 = __ldg(cu + g + 1);
    if (c0 <= i && (g == nseq - 1 || i < c1)) return g;
    if (c0 > i) hi = g - 1;
    else lo = g + 1;
  }
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (__ldg(cu + mid) <= i) lo = mid; else hi = mid - 1;
  }
  return lo;
}

__device__ __forceinline__ int find_seq(const int32_t* __restrict__ cu, int nseq, int total,
                                        int i) {
  int g = 0;
  if (total > 0 && nseq > 1) {
    g = static_cast<int>((static_cast<int64_t>(i) * nseq) / total);
    g = g < 0 ? 0 : (g > nseq - 1 ? nseq - 1 : g);
  }
  return find_seq_from(cu, nseq, i, g);
}

// The same with the guess's division by a divider made on the host (`div_total` divides by
// total; valid when nseq * total < 2^32, 0 <= i < total).
__device__ __forceinline__ int find_seq(const int32_t* __restrict__ cu, int nseq, int i,
                                        const DivU32& div_total) {
  int g = static_cast<int>(divu32(static_cast<uint32_t>(i) * static_cast<uint32_t>(nseq),
                                  div_total));
  g = g > nseq - 1 ? nseq - 1 : g;
  return find_seq_from(cu, nseq, i, g);
}

// Physical row index ((page * H + h) * page_size + slot) of slot `slot` of logical page `lp` of
// sequence `s`, or -1 (and the error bit) if the logical or physical page is out of range.
__device__ __forceinline__ int64_t locate_row_at(const int32_t* __restrict__ page_table,
                                                 int max_pages, int page_size, int num_heads,
                                                 int64_t num_pages, int s, int64_t lp, int slot,
                                                 int h, int32_t* err) {
  if (lp >= max_pages) { report(err, KVQ_DEVERR_PAGE_RANGE); return -1; }
  int page = __ldg(page_table + static_cast<int64_t>(s) * max_pages + lp);
  if (page < 0 || page >= num_pages) { report(err, KVQ_DEVERR_PAGE_RANGE); return -1; }
  return (static_cast<int64_t>(page) * num_heads + h) * page_size + slot;
}

// Physical row index ((page * H + h) * page_size + slot) of token `pos` of sequence `s`,
// or -1 (and the error bit) if the logical or physical page is out of range.
__device__ __forceinline__ int64_t locate_row(const int32_t* __restrict__ page_table,
                                              int max_pages, int page_size, int num_heads,
                                              int64_t num_pages, int s, int64_t pos, int h,
                                              int32_t* err) {
  if (pos < 0) { report(err, KVQ_DEVERR_PAGE_RANGE); return -1; }
  const int64_t lp = pos / page_size;
  return locate_row_at(page_table, max_pages, page_size, num_heads, num_pages, s, lp,
                       static_cast<int>(pos - lp * page_size), h, err);
}

// The same with the division by the page size made by a divider (`div_ps`; 0 <= pos < 2^32).
__device__ __forceinline__ int64_t locate_row(const int32_t* __restrict__ page_table,
                                              int max_pages, int page_size, int num_heads,
                                              int64_t num_pages, int s, int64_t pos, int h,
                                              int32_t* err, const DivU32& div_ps) {
  if (pos < 0 || pos > 0xffffffffLL) { report(err, KVQ_DEVERR_PAGE_RANGE); return -1; }
  const uint32_t lp = divu32(static_cast<uint32_t>(pos), div_ps);
  return locate_row_at(page_table, max_pages, page_size, num_heads, num_pages, s, lp,
                       static_cast<int>(static_cast<uint32_t>(pos) - lp * page_size), h, err);
}

// Load one 16-element unit of packed codes (12 / 8 / 16 bytes for q6 / q4 / q8) into the words
// that unpack_group<BITS, 0> and <BITS, 1> read.
template <int BITS>
__device__ __forceinline__ void load_unit(const uint8_t* p, uint32_t w[4]) {
  if constexpr (BITS == 6) {
    w[0] = ld_nc_u32(p);
    w[1] = ld_nc_u32(p + 4);
    w[2] = ld_nc_u32(p + 8);
    w[3] = 0;
  } else if constexpr (BITS == 4) {
    const uint2 v = ld_nc_v2(p);
    w[0] = v.x; w[1] = v.y; w[2] = w[3] = 0;
  } else {
    const uint4 v = ld_nc_v4(p);
    w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
  }
}

__device__ __forceinline__ float h2f(uint16_t b) { return __half2float(__ushort_as_half(b)); }
__device__ __forceinline__ uint16_t f2h(float f) { return __half_as_ushort(__float2half_rn(f)); }

}  // namespace kvq
