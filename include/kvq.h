/*
 * kvq.h -- C ABI of libkvq: quantized paged KV cache kernels for NVIDIA GB300 (sm_103a).
 *
 * Operations (each defined on the page cited at its declaration):
 *   kvq_quant_pack_paged   symmetric per-token-per-head quantize + pack into paged storage
 *   kvq_dequant_paged      gather + unpack + dequantize back to fp16
 *   kivi_quant_dequant     KIVI asymmetric group quantize->dequantize, in place
 *   kvq_decode_attn        decode attention that reads the packed pages directly
 *   kvq_append_decode_attn one decode step: append the new token, then attend, in one launch
 *   kivi_pack, kivi_decode_attn   packed KIVI storage and decode attention over it
 *   kivi_update, kivi_trim, kivi_packed_update, kivi_packed_trim   the KIVI cache protocol
 *   kvq_*_side             fp16 attention sinks and outlier side channel on the symmetric path
 * plus host helpers: packed_dim, the KIVI residual boundary, and a page allocator.
 *
 * Conventions shared by every entry point
 *   - The caller owns all memory.  The library never allocates or frees device memory and never
 *     synchronizes a stream.  Pointers documented "device" must be device (or managed) memory;
 *     "host" pointers are read before the call returns.
 *   - fp16 values are passed as their 16-bit patterns (uint16_t).
 *   - Every GPU entry point validates its arguments on the host first and returns a status
 *     without launching anything if they are invalid.  Otherwise it enqueues its kernels on
 *     `stream` (NULL = the legacy default stream) and returns KVQ_OK, or KVQ_ERR_CUDA if a launch
 *     was rejected.  Asynchronous device faults surface at the caller's next synchronization.
 *   - Kernels that read a page table check every page id they use against the pool size.  An id
 *     outside [0, num_pages) or a logical page beyond max_pages is skipped (nothing is read or
 *     written for that row) and, if `dev_err` is non-NULL, bit KVQ_DEVERR_PAGE_RANGE is OR-ed
 *     into *dev_err (device int32, caller zeroes it).  The kernels never trap.
 *   - kvq_last_error() returns a thread-local message describing the last non-OK status.
 */
#ifndef KVQ_H
#define KVQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define KVQ_API __attribute__((visibility("default")))
#else
#define KVQ_API
#endif

/* Same object as cudaStream_t. */
typedef struct CUstream_st* kvq_stream_t;

typedef enum kvq_status {
  KVQ_OK = 0,
  KVQ_ERR_BITS = 1,      /* bit width not in {8, 6, 4} (the explicit width table)            */
  KVQ_ERR_SHAPE = 2,     /* head_dim / heads / group / range shape not supported              */
  KVQ_ERR_NULL = 3,      /* a required pointer is NULL                                        */
  KVQ_ERR_ALIGN = 4,     /* a device pointer is not 16-byte aligned                           */
  KVQ_ERR_RANGE = 5,     /* a count or index is out of range                                  */
  KVQ_ERR_CUDA = 6,      /* a CUDA launch or query failed                                     */
  KVQ_ERR_NOMEM = 7,     /* the host page allocator has too few free pages                    */
  KVQ_ERR_WORKSPACE = 8  /* the caller's workspace is too small                               */
} kvq_status;

/* Bits OR-ed into the optional device error word. */
#define KVQ_DEVERR_PAGE_RANGE 1  /* a page id or logical page was out of range (row skipped)   */
#define KVQ_DEVERR_TIMEOUT 2     /* a bounded wait for an asynchronous copy gave up (the
                                    affected output is invalid; the kernel returned normally)  */

/* Maximum number of tensors one quant/dequant/KIVI call may batch, and of layers per decode
 * attention call. */
#define KVQ_MAX_TENSORS 64

/*
 * One page pool: the packed storage of one (layer, K-or-V) tensor.
 *   codes  : device uint8  [num_pages][num_heads][page_size][packed_dim(head_dim, bits)]
 *   scales : device fp16   [num_pages][num_heads][page_size]  (one scale per token per head)
 * Token `pos` of sequence `s` lives in physical page page_table[s * max_pages + pos / page_size],
 * slot pos % page_size.  Both arrays must be 16-byte aligned.  Within one page, the rows of one
 * head are contiguous (page_size * packed_dim bytes).
 */
typedef struct kvq_pool {
  int32_t bits;       /* 8, 6 or 4 */
  int32_t num_heads;  /* KV heads H */
  int32_t head_dim;   /* D <= 256 with kvq_packed_dim(D, bits) > 0: any D at q8, even at q4,
                         a multiple of 4 at q6 (the decode attention takes D = 256 only) */
  int32_t page_size;  /* tokens per page, >= 1 */
  int64_t num_pages;
  uint8_t* codes;
  uint16_t* scales;
} kvq_pool;

/* ---------------------------------------------------------------------------------------------
 * Host helpers
 * ------------------------------------------------------------------------------------------ */

/* Library version string. */
KVQ_API const char* kvq_version(void);

/* Thread-local message for the last non-OK status returned on this thread ("" if none). */
KVQ_API const char* kvq_last_error(void);

/* Name of a status code. */
KVQ_API const char* kvq_status_string(kvq_status status);

/*
 * The address under which kernels read page-locked host memory (cudaHostAlloc, or
 * cudaHostRegister with the mapped flag; on systems with unified addressing all page-locked memory
 * is mapped).  Any entry point documented to take "device" input may be given this address: its
 * kernels then read the host memory directly over the host link (NVLink-C2C on Grace systems)
 * instead of the caller copying it to the device first.  A device or managed pointer is returned
 * as is; other memory is refused with KVQ_ERR_RANGE (no kernel ever sees an unmapped address).
 * No counterpart on the pages: a host-memory convenience of this library.
 */
KVQ_API kvq_status kvq_host_device_view(const void* host_ptr, void** device_ptr);

/*
 * Bytes per packed row.  MTPLX pull request #267, "feat(kv-cache): add q6 paged KV
 * quantization", description, packed_dim sentence: packed_dim(D, 6) = D*3/4 and q6 needs
 * D % 4 == 0; q8 stores one code per byte, q4 two per byte (D % 2 == 0).
 * Returns -1 for an unknown width or an unsupported D (no error state is set).
 */
KVQ_API int kvq_packed_dim(int head_dim, int bits);

/*
 * KIVI residual-window boundary.  VeloxQuant-MLX source page "veloxquant_mlx.cache.kivi_cache",
 * KIVIKVCache._quantization_boundary: the tokens older than the newest `residual_length`,
 * snapped down to a multiple of `group_size`: ((max(0, offset - residual_length)) / group_size)
 * * group_size.  Returns -1 if group_size < 1 or residual_length < 0.
 */
KVQ_API int kivi_boundary(int offset, int residual_length, int group_size);

/*
 * Host page allocator over page ids [0, num_pages) (a LIFO free list; not thread-safe).
 * The pages themselves are the caller's kvq_pool memory; this only hands out ids.
 * MTPLX pull request #267, description: cache allocation is width-generic through packed_dim --
 * the allocator deals in pages, never in bytes.
 */
typedef struct kvq_allocator kvq_allocator;

/* Returns NULL on bad size or host allocation failure. */
KVQ_API kvq_allocator* kvq_alloc_create(int64_t num_pages);
KVQ_API void kvq_alloc_destroy(kvq_allocator* a);
KVQ_API int64_t kvq_alloc_free_count(const kvq_allocator* a);

/* Take n page ids into out_ids (host int32[n]).  All or nothing: KVQ_ERR_NOMEM if fewer than n
 * are free (nothing taken). */
KVQ_API kvq_status kvq_alloc_pages(kvq_allocator* a, int64_t n, int32_t* out_ids);

/* Return n page ids.  KVQ_ERR_RANGE (nothing returned) if an id is out of range, not currently
 * allocated, or repeated in `ids`. */
KVQ_API kvq_status kvq_free_pages(kvq_allocator* a, int64_t n, const int32_t* ids);

/*
 * Map the pages that an append of new_tokens[s] tokens at position cur_len[s] needs, for every
 * sequence s: every logical page in [cur_len[s] / page_size, ceil((cur_len[s] + new_tokens[s]) /
 * page_size)) whose entry in the host table page_table[s * max_pages + p] is negative gets a
 * fresh page id.  Entries already >= 0 are kept (a partially filled tail page is appended into).
 * All or nothing: on KVQ_ERR_NOMEM or KVQ_ERR_RANGE (a page beyond max_pages) the table is left
 * unchanged.  The caller then copies the table to the device.
 */
KVQ_API kvq_status kvq_table_reserve(kvq_allocator* a, int32_t* page_table, int max_pages, int page_size,
                             const int32_t* cur_len, const int32_t* new_tokens, int nseq);

/* ---------------------------------------------------------------------------------------------
 * Quantize + pack into pages
 * ------------------------------------------------------------------------------------------ */

/*
 * MTPLX pull request #267, "feat(kv-cache): add q6 paged KV quantization", description:
 * symmetric per-token-per-head quantizer with one fp16 scale per row, qmax 127 / 31 / 7 for
 * 8 / 6 / 4 bits (bit-width table paragraph); q6 codes biased by +32 and packed four per three
 * bytes, byte0 = u0 | (u1 & 3) << 6, byte1 = (u1 >> 2) | (u2 & 15) << 4,
 * byte2 = (u2 >> 4) | (u3 & 63) << 2 (byte-layout formula).
 *
 * Per row x (one token, one KV head, D fp16):
 *   scale = fp16_rne(float32(max_d |x_d|) / qmax)           (IEEE float32 divide)
 *   c_d   = clamp(rint_half_even(float32(x_d) / float32(scale)), -qmax, qmax), or 0 if scale == 0
 *   q8: byte = int8 two's complement of c; q6: u = c + 32, 4 -> 3 bytes as above;
 *   q4: u = c + 8, element 2i in the low nibble of byte i.
 *
 * pools      host array [n_tensors]: the destination pools (all with the same bits, num_heads,
 *            head_dim, page_size).
 * x          host array [n_tensors] of device pointers, each fp16 [total_new_tokens][H][D],
 *            16-byte aligned: the new rows of every sequence, sequence s owning rows
 *            cu_new_tokens[s] .. cu_new_tokens[s+1]-1, which are its tokens start_pos[s],
 *            start_pos[s]+1, ...
 * page_table device int32 [nseq][max_pages], shared by every tensor of the call.
 * cu_new_tokens device int32 [nseq+1], non-decreasing, cu[0] = 0, cu[nseq] = total_new_tokens.
 * start_pos  device int32 [nseq].
 * dev_err    optional device int32 error word (see the file header).
 * Rows are independent; a row's packed bytes and scale are written whole.  Two rows of one call
 * mapping to the same (page, slot) race (a caller error).
 * Head dims that are not a multiple of 16 run a one-warp-per-row kernel (same arithmetic).
 * Errors: KVQ_ERR_BITS, KVQ_ERR_SHAPE (kvq_packed_dim(D, bits) < 1, D > 256, mismatched pools),
 * KVQ_ERR_NULL, KVQ_ERR_ALIGN, KVQ_ERR_RANGE (n_tensors not in [1, KVQ_MAX_TENSORS], nseq < 0,
 * total_new_tokens < 0, max_pages < 1), KVQ_ERR_CUDA.
 */
KVQ_API kvq_status kvq_quant_pack_paged(const kvq_pool* pools, const uint16_t* const* x, int n_tensors,
                                const int32_t* page_table, int max_pages,
                                const int32_t* cu_new_tokens, const int32_t* start_pos, int nseq,
                                int total_new_tokens, int32_t* dev_err, kvq_stream_t stream);

/* ---------------------------------------------------------------------------------------------
 * Gather + unpack + dequantize
 * ------------------------------------------------------------------------------------------ */

/*
 * MTPLX pull request #267, description: dequantization runs over the active window; the inverse
 * of kvq_quant_pack_paged: x_hat_d = fp16_rne(float32(c_d) * float32(scale)) (the product is
 * exact in float32).
 *
 * Same addressing as kvq_quant_pack_paged: out[i] (host array of device pointers, each fp16
 * [total_tokens][H][D], 16-byte aligned) receives rows cu_tokens[s] .. cu_tokens[s+1]-1 =
 * tokens start_pos[s], start_pos[s]+1, ... of sequence s.  Rows whose page id is out of range
 * are left untouched.  Errors as for kvq_quant_pack_paged.
 */
KVQ_API kvq_status kvq_dequant_paged(const kvq_pool* pools, uint16_t* const* out, int n_tensors,
                             const int32_t* page_table, int max_pages, const int32_t* cu_tokens,
                             const int32_t* start_pos, int nseq, int total_tokens,
                             int32_t* dev_err, kvq_stream_t stream);

/* ---------------------------------------------------------------------------------------------
 * KIVI group quantize -> dequantize, in place
 * ------------------------------------------------------------------------------------------ */

/*
 * VeloxQuant-MLX source page "veloxquant_mlx.cache.kivi_cache", KIVIKVCache._quant_dequant_along
 * and update_and_fetch.  For every tensor i, the token slice [lo, hi) of x[i] (device fp16
 * [B][H][S][D], 16-byte aligned, modified in place) is round-tripped in float32:
 *   keys   (is_key[i] != 0): per channel, groups of group_size tokens starting at lo;
 *   values (is_key[i] == 0): per token, groups of group_size channels starting at channel 0;
 *   a ragged last group uses only its real elements (the page pads it with its last element,
 *   which leaves min and max unchanged);
 *   scale = max((gmax - gmin) / levels, eps); c = clamp(rint_half_even((x - gmin) / scale), 0,
 *   levels); y = fp16_rne((c * scale) + gmin) with two roundings (no fused multiply-add).
 * is_key     host int32 [n_tensors].
 * levels     2^b - 1 for b-bit KIVI (the page's default b = 2 gives 3); >= 1.
 * eps        the page's 1e-8 (as float32).
 * Use kivi_boundary() for hi and the previous frontier for lo (update_and_fetch).
 * Errors: KVQ_ERR_SHAPE (D % 8, D > 256, 0 <= lo <= hi <= S violated, group_size < 1,
 * levels < 1), KVQ_ERR_NULL, KVQ_ERR_ALIGN, KVQ_ERR_RANGE (n_tensors, B, H, S), KVQ_ERR_CUDA.
 * An empty slice (lo == hi) launches nothing and returns KVQ_OK.
 */
KVQ_API kvq_status kivi_quant_dequant(uint16_t* const* x, const int32_t* is_key, int n_tensors, int B,
                              int H, int S, int D, int lo, int hi, int group_size, int levels,
                              float eps, kvq_stream_t stream);

/* ---------------------------------------------------------------------------------------------
 * Decode attention over packed pages
 * ------------------------------------------------------------------------------------------ */

/*
 * Attention for one decode query per sequence over that sequence's whole packed cache, reading
 * the packed pages directly (MTPLX pull request #267, description: the reference path instead
 * dequantizes to fp16 and runs SDPA; this computes the same function without materialising fp16).
 * For layer l, sequence s, query head j (KV head h = j / (Hq / H)):
 *   s_t = softmax_scale * sum_d q[l][s][j][d] * k_hat_t[d],   t in [0, seq_lens[s])
 *   out[l][s][j][:] = sum_t softmax(s)_t * v_hat_t[:]    (float32 accumulation)
 * where k_hat, v_hat are the fp16 dequantized rows of k_pools[l], v_pools[l].
 * k_pools, v_pools host arrays [n_layers] (same bits/H/D/page_size for all).
 * q          device fp16 [n_layers][nseq][num_q_heads][D], 16-byte aligned.
 * out        device float32 [n_layers][nseq][num_q_heads][D]; a sequence of length 0 gets 0.
 * page_table device int32 [nseq][max_pages] (shared by all layers); seq_lens device int32 [nseq].
 * max_seq_len host upper bound on seq_lens (sizes the split over tokens).
 * workspace  device scratch of at least kvq_decode_attn_workspace(...) bytes, 16-byte aligned;
 *            its contents need no initialisation and are garbage afterwards.
 * Errors: KVQ_ERR_SHAPE (num_q_heads % H, num_q_heads / H > 8, D != 256 for now), KVQ_ERR_BITS,
 * KVQ_ERR_NULL, KVQ_ERR_ALIGN, KVQ_ERR_RANGE, KVQ_ERR_WORKSPACE, KVQ_ERR_CUDA.
 */
KVQ_API size_t kvq_decode_attn_workspace(int n_layers, int nseq, int num_kv_heads, int num_q_heads,
                                 int head_dim, int page_size, int max_seq_len);

KVQ_API kvq_status kvq_decode_attn(const kvq_pool* k_pools, const kvq_pool* v_pools, int n_layers,
                           const uint16_t* q, int num_q_heads, const int32_t* page_table,
                           int max_pages, const int32_t* seq_lens, int nseq, int max_seq_len,
                           float softmax_scale, float* out, void* workspace,
                           size_t workspace_bytes, int32_t* dev_err, kvq_stream_t stream);

/*
 * One decode step with the append fused in: for every sequence s, quantize its new token's K and
 * V rows (k_new[l], v_new[l]: device fp16 [nseq][H][256] per layer, 16-byte aligned) exactly as
 * kvq_quant_pack_paged would, store them at position seq_lens[s] of the pools (page
 * page_table[s][seq_lens[s] / page_size], which the caller has mapped, e.g. with
 * kvq_table_reserve), and attend over the seq_lens[s] + 1 tokens that result -- one launch (plus
 * the split merge).  MTPLX pull request #267, description: quantize on write, and attention over
 * the active window; the pages run the two as separate steps (write, then dequantize + SDPA).
 * seq_lens holds the lengths BEFORE the append and is not modified: the caller advances it.
 * max_seq_len bounds seq_lens[s] + 1.  The page size must be a multiple of 16.  Other arguments,
 * the workspace (kvq_decode_attn_workspace with that max_seq_len) and the errors are those of
 * kvq_decode_attn; the pools are written, so they must not be read by other work in flight.
 */
KVQ_API kvq_status kvq_append_decode_attn(const kvq_pool* k_pools, const kvq_pool* v_pools,
                                          int n_layers, const uint16_t* const* k_new,
                                          const uint16_t* const* v_new, const uint16_t* q,
                                          int num_q_heads, const int32_t* page_table,
                                          int max_pages, const int32_t* seq_lens, int nseq,
                                          int max_seq_len, float softmax_scale, float* out,
                                          void* workspace, size_t workspace_bytes,
                                          int32_t* dev_err, kvq_stream_t stream);

/* ---------------------------------------------------------------------------------------------
 * fp16 side channels: attention sinks and dense-and-sparse outliers
 * ------------------------------------------------------------------------------------------ */

#define KVQ_MAX_OUTLIERS 8
#define KVQ_MAX_SINKS 16

/*
 * VeloxQuant-MLX API docs, "veloxquant_mlx.cache.kvquant_cache module": per-vector
 * dense-and-sparse outlier isolation with an fp16 side channel (value + position index), and
 * Attention Sink-Aware quantization (the first n_sink tokens of a sequence restored to exact
 * fp16), applied to the symmetric quantizer above.  One kvq_side accompanies one kvq_pool:
 *   a row's n_outlier largest-magnitude elements (ties: the lower position) are stored as fp16
 *   value + uint8 position, ascending by position, in out_val / out_idx at the row's physical
 *   index; the rest of the row (outliers set to 0) is quantized as usual -- its scale comes from
 *   the (n_outlier + 1)-th largest magnitude and the outlier positions hold code 0;
 *   rows at positions < n_sink are also copied exactly into sink, which dequantization and
 *   attention read instead of the pages.
 * The page's fraction 0.01 gives n_outlier = ceil(0.01 * head_dim) (3 at 256).
 */
typedef struct kvq_side {
  int32_t n_outlier;  /* outliers per row, 0..KVQ_MAX_OUTLIERS, < head_dim */
  int32_t n_sink;     /* sink tokens per sequence, 0..KVQ_MAX_SINKS */
  int32_t max_seqs;   /* sequences the sink buffer holds (>= nseq of every call) */
  uint16_t* out_val;  /* fp16 [num_pages][H][page_size][n_outlier], 16-byte aligned */
  uint8_t* out_idx;   /* uint8 [num_pages][H][page_size][n_outlier], 16-byte aligned */
  uint16_t* sink;     /* fp16 [max_seqs][n_sink][H][D], 16-byte aligned */
} kvq_side;

/*
 * kvq_quant_pack_paged with the side channels: same arguments plus sides[i] for pools[i]
 * (uniform n_outlier and n_sink).  Any head_dim a pool accepts.  Errors: those of
 * kvq_quant_pack_paged, KVQ_ERR_RANGE (n_outlier, n_sink, max_seqs < nseq).
 */
KVQ_API kvq_status kvq_quant_pack_paged_side(const kvq_pool* pools, const kvq_side* sides,
                                             const uint16_t* const* x, int n_tensors,
                                             const int32_t* page_table, int max_pages,
                                             const int32_t* cu_new_tokens,
                                             const int32_t* start_pos, int nseq,
                                             int total_new_tokens, int32_t* dev_err,
                                             kvq_stream_t stream);

/* kvq_dequant_paged with the side channels: outliers written back, sink rows exact. */
KVQ_API kvq_status kvq_dequant_paged_side(const kvq_pool* pools, const kvq_side* sides,
                                          uint16_t* const* out, int n_tensors,
                                          const int32_t* page_table, int max_pages,
                                          const int32_t* cu_tokens, const int32_t* start_pos,
                                          int nseq, int total_tokens, int32_t* dev_err,
                                          kvq_stream_t stream);

/*
 * kvq_decode_attn over pools with side channels: the keys and values of a row are the dense
 * reconstruction with its outliers written back, and the sink positions (< n_sink) use the exact
 * fp16 rows of the sink buffer.  k_sides[l] / v_sides[l] accompany k_pools[l] / v_pools[l]
 * (uniform n_outlier and n_sink; max_seqs >= nseq).  The page size must be a multiple of 16.
 * Other arguments, the workspace and the errors are those of kvq_decode_attn.
 */
KVQ_API kvq_status kvq_decode_attn_side(const kvq_pool* k_pools, const kvq_pool* v_pools,
                                        const kvq_side* k_sides, const kvq_side* v_sides,
                                        int n_layers, const uint16_t* q, int num_q_heads,
                                        const int32_t* page_table, int max_pages,
                                        const int32_t* seq_lens, int nseq, int max_seq_len,
                                        float softmax_scale, float* out, void* workspace,
                                        size_t workspace_bytes, int32_t* dev_err,
                                        kvq_stream_t stream);

/* ---------------------------------------------------------------------------------------------
 * Packed KIVI storage and decode attention over it
 * ------------------------------------------------------------------------------------------ */

/*
 * VeloxQuant-MLX source page "veloxquant_mlx.cache.kivi_cache": the page keeps the KIVI cache in
 * fp16 and estimates the bytes of a packed form (module docstring, _quantized_bytes,
 * _account_bytes): b-bit codes plus an fp16 (scale, zero) pair per group -- per (token group,
 * channel) for keys, per (token, channel group) for values.  This is that packed form, for one
 * layer of a [batch][heads][capacity][head_dim] cache:
 *   k_codes [B][H][capacity][D*bits/8]   k_scale, k_zero fp16 [B][H][capacity/gs][D]
 *   v_codes [B][H][capacity][D*bits/8]   v_scale, v_zero fp16 [B][H][capacity][D/gs]
 * zero = the group minimum (an fp16 value), scale = fp16(max((max - min) / levels, eps)) with
 * levels = 2^bits - 1, code = clamp(rint((x - zero) / scale), 0, levels) (0 when the fp16 scale
 * is 0), stored LSB-first along the head dimension.  Its size is exactly the page's estimate.
 * All arrays 16-byte aligned; bits in {2, 4, 8}; group_size in {8, 16, 32, 64}; head_dim a
 * multiple of group_size, at most 256; capacity a multiple of group_size.
 */
typedef struct kivi_packed {
  int32_t bits;
  int32_t group_size;
  int32_t batch;
  int32_t num_heads;
  int32_t capacity;
  int32_t head_dim;
  uint8_t* k_codes;
  uint16_t* k_scale;
  uint16_t* k_zero;
  uint8_t* v_codes;
  uint16_t* v_scale;
  uint16_t* v_zero;
} kivi_packed;

/*
 * Pack tokens [lo, hi) of every layer's fp16 K and V (k[l], v[l]: device fp16 [B][H][capacity]
 * [D], 16-byte aligned; the same layout the in-place KIVI cache uses) into caches[l].  lo and hi
 * are multiples of group_size (the residual boundary of kivi_boundary always is).  eps is the
 * page's 1e-8.  Errors: KVQ_ERR_BITS, KVQ_ERR_SHAPE, KVQ_ERR_NULL, KVQ_ERR_ALIGN, KVQ_ERR_RANGE,
 * KVQ_ERR_CUDA.
 */
KVQ_API kvq_status kivi_pack(const kivi_packed* caches, const uint16_t* const* k,
                             const uint16_t* const* v, int n_layers, int lo, int hi, float eps,
                             kvq_stream_t stream);

/*
 * Decode attention of one query per batch row over a KIVI cache whose tokens [0, n_packed) are
 * packed in caches[l] and tokens [n_packed, offset) are still fp16 in k[l], v[l] (the residual
 * window).  q device fp16 [n_layers][B][num_q_heads][D]; out device float32, same shape; query
 * head j uses KV head j / (num_q_heads / H); the reconstruction of a packed element is
 * c * scale + zero in fp16 (one fused rounding), accumulation in float32.  Supports bits 2,
 * head_dim 64, group_size 16/32/64, at most 8 query heads per KV head; n_packed a multiple of
 * group_size; 0 <= n_packed <= offset <= capacity.  workspace: kivi_decode_attn_workspace(...)
 * bytes, 16-byte aligned, no initialisation needed.  dev_err (device int32, may be NULL) gets
 * KVQ_DEVERR_TIMEOUT OR-ed in if a staged copy never completed (the affected split then counts
 * no tokens).  Errors: KVQ_ERR_BITS, KVQ_ERR_SHAPE (bits, head_dim, group_size, num_q_heads),
 * KVQ_ERR_NULL, KVQ_ERR_ALIGN, KVQ_ERR_RANGE (n_packed, offset, grid limits), KVQ_ERR_WORKSPACE,
 * KVQ_ERR_CUDA.
 */
KVQ_API size_t kivi_decode_attn_workspace(int n_layers, int batch, int num_heads, int num_q_heads,
                                          int head_dim, int offset);

KVQ_API kvq_status kivi_decode_attn(const kivi_packed* caches, const uint16_t* const* k,
                                    const uint16_t* const* v, int n_layers, const uint16_t* q,
                                    int num_q_heads, int n_packed, int offset,
                                    float softmax_scale, float* out, void* workspace,
                                    size_t workspace_bytes, int32_t* dev_err,
                                    kvq_stream_t stream);

/* ---------------------------------------------------------------------------------------------
 * The KIVI cache protocol: update (append + flush) and trim (frontier rollback)
 * ------------------------------------------------------------------------------------------ */

/*
 * VeloxQuant-MLX source page "veloxquant_mlx.cache.kivi_cache": KIVIKVCache.update_and_fetch,
 * _quantization_boundary, trim and _rollback_frontier.  A kivi_state (host memory, owned by the
 * caller) tracks one cache of n_layers layers that append and trim together: `offset` tokens
 * held in [B][H][capacity][D] fp16 K and V caches, the first `n_quantized` of them quantized.
 * bits 2/4/8 give levels 2^bits - 1; eps is the page's 1e-8.  Fill it with kivi_state_init
 * (offset 0); the calls below advance it only when they succeed.
 */
typedef struct kivi_state {
  int32_t batch;
  int32_t num_heads;
  int32_t head_dim;         /* multiple of 8, <= 256 */
  int32_t capacity;
  int32_t bits;             /* 2, 4 or 8 */
  int32_t group_size;
  int32_t residual_length;  /* the page's residual window R (128 by default) */
  float eps;
  int32_t offset;           /* tokens held */
  int32_t n_quantized;      /* the quantization frontier */
} kivi_state;

KVQ_API kvq_status kivi_state_init(kivi_state* st, int batch, int num_heads, int head_dim,
                                   int capacity, int bits, int group_size, int residual_length);

/*
 * update_and_fetch for the page's in-place cache: copy the n_new new tokens of every layer
 * (k_new[l], v_new[l]: device fp16 [B][H][n_new][D], 16-byte aligned) into k_cache[l],
 * v_cache[l] at st->offset (one launch for all layers), then round-trip the tokens
 * [n_quantized, kivi_boundary(offset + n_new)) in place (kivi_quant_dequant, one launch), and
 * advance the state.  n_layers <= 32.  Errors: those of kivi_quant_dequant, KVQ_ERR_RANGE if the
 * tokens do not fit.  The "fetch" is the caches' first st->offset tokens.
 */
KVQ_API kvq_status kivi_update(kivi_state* st, uint16_t* const* k_cache, uint16_t* const* v_cache,
                               const uint16_t* const* k_new, const uint16_t* const* v_new,
                               int n_layers, int n_new, kvq_stream_t stream);

/*
 * trim for the page's in-place cache: drop the last n tokens (at most offset) and pull the
 * frontier down to min(n_quantized, (offset / group_size) * group_size).  Host only: the rows
 * between the new frontier and the new offset keep their round-tripped values in the cache and
 * are quantized again by the next flush (the double rounding the page bounds by one step).
 * Returns the number of tokens dropped.
 */
KVQ_API int kivi_trim(kivi_state* st, int n);

/*
 * update_and_fetch with the quantized region packed (kivi_packed, one per layer, matching the
 * state): append as kivi_update, then kivi_pack tokens [n_quantized, boundary) from the fp16
 * caches.  Attention: kivi_decode_attn(n_packed = st->n_quantized, offset = st->offset).
 */
KVQ_API kvq_status kivi_packed_update(kivi_state* st, const kivi_packed* caches,
                                      uint16_t* const* k_cache, uint16_t* const* v_cache,
                                      const uint16_t* const* k_new, const uint16_t* const* v_new,
                                      int n_layers, int n_new, kvq_stream_t stream);

/*
 * trim with the quantized region packed: as kivi_trim, and the rows that leave the packed region
 * ([new frontier, min(old frontier, new offset))) get their round-tripped values written into
 * the fp16 caches (kivi_unpack), as the page's in-place cache holds them.  *trimmed (may be
 * NULL) receives the number of tokens dropped.
 */
KVQ_API kvq_status kivi_packed_trim(kivi_state* st, const kivi_packed* caches,
                                    uint16_t* const* k_cache, uint16_t* const* v_cache,
                                    int n_layers, int n, int* trimmed, kvq_stream_t stream);

/*
 * Write the reconstruction fp16(float32(c * scale) + zero) of packed tokens [lo, hi) of every
 * layer into k[l], v[l] (device fp16 [B][H][capacity][D]).  Errors: KVQ_ERR_BITS, KVQ_ERR_SHAPE,
 * KVQ_ERR_NULL, KVQ_ERR_ALIGN, KVQ_ERR_RANGE, KVQ_ERR_CUDA.
 */
KVQ_API kvq_status kivi_unpack(const kivi_packed* caches, uint16_t* const* k, uint16_t* const* v,
                               int n_layers, int lo, int hi, kvq_stream_t stream);

/*
 * Decode attention for callers that cannot allocate device memory (no counterpart on the pages:
 * it is an addition of this library).  Same arguments, semantics and errors as kvq_decode_attn,
 * minus the workspace: the split partials go to a scratch array of 32 MiB that the library owns
 * in device memory, which every GPU that loads the library holds until the process exits.
 * Meant for code that cannot call cudaMalloc where it runs attention -- for example inside a
 * runtime whose allocator owns all device memory, or a serving loop that must not allocate
 * (cudaMalloc may synchronize the device) once it is running.  It calls no allocation routine.
 *   - The first call on a device looks up the scratch array's device address (cached per
 *     device); make that first call before any stream capture.
 *   - All calls share the one array: calls whose kernels overlap on the GPU (other streams,
 *     other threads) race on it and must be serialized by the caller.  Nothing in it needs to be
 *     cleared between calls: every partial a call reads was written earlier by that same call.
 *   - To fit the array, the number of splits over tokens is capped (each split of each
 *     (layer, sequence, KV head) unit takes 8,320 bytes), so a split may then cover more than
 *     the usual 256 tiles (4,096 tokens); a problem with more than 4,032
 *     n_layers * nseq * num_kv_heads units does not fit even with one split each and returns
 *     KVQ_ERR_RANGE with the byte counts in kvq_last_error().
 */
KVQ_API kvq_status kvq_decode_attn_noalloc(const kvq_pool* k_pools, const kvq_pool* v_pools,
                                           int n_layers, const uint16_t* q, int num_q_heads,
                                           const int32_t* page_table, int max_pages,
                                           const int32_t* seq_lens, int nseq, int max_seq_len,
                                           float softmax_scale, float* out, int32_t* dev_err,
                                           kvq_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* KVQ_H */
