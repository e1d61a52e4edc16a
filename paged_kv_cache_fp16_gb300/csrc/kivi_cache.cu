// The KIVI cache protocol on the device: update_and_fetch (append the new tokens, then quantize the
// tokens that left the residual window) and trim (drop the last tokens and pull the quantization
// frontier back), for the page's in-place fp16 cache and for the packed form.
//
// VeloxQuant-MLX source page "veloxquant_mlx.cache.kivi_cache": KIVIKVCache.update_and_fetch,
// _quantization_boundary, trim and _rollback_frontier.  The state (offset, frontier) is a host
// struct the caller owns; one state covers all layers, which append and trim together.
//
// kivi_append_kernel: one launch copies every layer's new K and V tokens ([B][H][n][D]) into the
// caches ([B][H][capacity][D]) at the offset, 16 bytes per thread step (HBM-bound copy).
// kivi_unpack_kernel<BITS>: the rows a trim moves out of the packed region get their
// round-tripped values written back into the fp16 window, fp16(float32(c * scale) + zero) -- the
// reconstruction of the page's round trip -- one thread per (tensor, row, 8-element chunk).
// The flush itself reuses kivi_quant_dequant (in place) or kivi_pack (packed).
#include <cuda_runtime.h>
#include <cuda_fp16.h>

#include "kvq_device.cuh"
#include "kvq_internal.h"

namespace kvq {
namespace {

constexpr int kThreads = 256;

struct AppendArgs {
  uint16_t* dst[KVQ_MAX_TENSORS];        // caches: K of layer l at 2l, V at 2l + 1
  const uint16_t* src[KVQ_MAX_TENSORS];  // new tokens, same order
  int n_tensors, B, H, S, D, offset, n_new;
};

__global__ void __launch_bounds__(kThreads) kivi_append_kernel(const AppendArgs a) {
  const int vec = a.D / 8;                                      // 16-byte vectors per row
  const int64_t per_tensor = static_cast<int64_t>(a.B) * a.H * a.n_new * vec;
  const int64_t items = per_tensor * a.n_tensors;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
  for (int64_t it = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; it < items;
       it += stride) {
    const int t = static_cast<int>(it / per_tensor);
    int64_t r = it - t * per_tensor;
    const int v = static_cast<int>(r % vec);
    r /= vec;
    const int tok = static_cast<int>(r % a.n_new);
    const int64_t bh = r / a.n_new;
    const uint4 x = reinterpret_cast<const uint4*>(a.src[t] + (bh * a.n_new + tok) * a.D)[v];
    reinterpret_cast<uint4*>(a.dst[t] + (bh * a.S + a.offset + tok) * a.D)[v] = x;
  }
}

struct UnpackArgs {
  kivi_packed c[KVQ_MAX_TENSORS];
  uint16_t* k[KVQ_MAX_TENSORS];
  uint16_t* v[KVQ_MAX_TENSORS];
  int n_layers, lo, hi;
};

template <int BITS>
__global__ void __launch_bounds__(kThreads) kivi_unpack_kernel(const UnpackArgs a) {
  const kivi_packed& c0 = a.c[0];
  const int B = c0.batch, H = c0.num_heads, S = c0.capacity, D = c0.head_dim, gs = c0.group_size;
  const int chunks = D / 8, G = D / gs, cb = D * BITS / 8;
  const int span = a.hi - a.lo;
  const int64_t per_tensor = static_cast<int64_t>(B) * H * span * chunks;
  const int64_t items = per_tensor * 2 * a.n_layers;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
  constexpr uint32_t kMask = (1u << BITS) - 1;
  for (int64_t it = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; it < items;
       it += stride) {
    const int tensor = static_cast<int>(it / per_tensor);
    const int layer = tensor >> 1;
    const bool is_v = tensor & 1;
    int64_t r = it - tensor * per_tensor;
    const int ch = static_cast<int>(r % chunks);
    r /= chunks;
    const int64_t bh = r / span;
    const int t = a.lo + static_cast<int>(r - bh * span);
    const kivi_packed& C = a.c[layer];
    const uint8_t* codes = (is_v ? C.v_codes : C.k_codes) + (bh * S + t) * cb + ch * BITS;
    uint32_t lo = 0, hi = 0;   // 8 fields, LSB-first
    if constexpr (BITS == 2) lo = *reinterpret_cast<const uint16_t*>(codes);
    else if constexpr (BITS == 4) lo = *reinterpret_cast<const uint32_t*>(codes);
    else {
      const uint2 w = *reinterpret_cast<const uint2*>(codes);
      lo = w.x;
      hi = w.y;
    }
    float s[8], z[8];
    if (!is_v) {   // per channel of the token group t / gs
      const int64_t p = (bh * (S / gs) + t / gs) * D + ch * 8;
      const uint4 sw = *reinterpret_cast<const uint4*>(C.k_scale + p);
      const uint4 zw = *reinterpret_cast<const uint4*>(C.k_zero + p);
      const uint32_t sv[4] = {sw.x, sw.y, sw.z, sw.w}, zv[4] = {zw.x, zw.y, zw.z, zw.w};
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        s[e] = h2f(static_cast<uint16_t>(sv[e >> 1] >> (16 * (e & 1))));
        z[e] = h2f(static_cast<uint16_t>(zv[e >> 1] >> (16 * (e & 1))));
      }
    } else {       // per channel group of the token (gs >= 8: one group per chunk)
      const int64_t p = (bh * S + t) * G + (ch * 8) / gs;
      const float s1 = h2f(C.v_scale[p]), z1 = h2f(C.v_zero[p]);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        s[e] = s1;
        z[e] = z1;
      }
    }
    uint32_t out[4];
#pragma unroll
    for (int e = 0; e < 8; e += 2) {
      uint16_t y[2];
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int bit = (e + k) * BITS;
        const uint32_t f = (bit < 32 ? (lo >> bit) : (hi >> (bit - 32))) & kMask;
        y[k] = f2h(__fadd_rn(__fmul_rn(static_cast<float>(f), s[e + k]), z[e + k]));
      }
      out[e >> 1] = y[0] | (static_cast<uint32_t>(y[1]) << 16);
    }
    uint16_t* dst = (is_v ? a.v[layer] : a.k[layer]) + (bh * S + t) * D + ch * 8;
    *reinterpret_cast<uint4*>(dst) = make_uint4(out[0], out[1], out[2], out[3]);
  }
}

int grid_for(int64_t items) {
  const int sms = sm_count() > 0 ? sm_count() : 152;
  int64_t b = (items + kThreads - 1) / kThreads;
  const int64_t cap = static_cast<int64_t>(sms) * 8;
  return static_cast<int>(b > cap ? cap : (b < 1 ? 1 : b));
}

kvq_status check_state(const kivi_state* st, const char* fn) {
  if (!st) return fail(KVQ_ERR_NULL, "%s: state is NULL", fn);
  if (st->bits != 2 && st->bits != 4 && st->bits != 8)
    return fail(KVQ_ERR_BITS, "%s: bits %d not in {2, 4, 8}", fn, st->bits);
  if (st->batch < 1 || st->num_heads < 1 || st->capacity < 1 || st->group_size < 1 ||
      st->residual_length < 0 || st->head_dim < 8 || st->head_dim > 256 || st->head_dim % 8)
    return fail(KVQ_ERR_SHAPE, "%s: bad state shape", fn);
  if (st->offset < 0 || st->offset > st->capacity || st->n_quantized < 0 ||
      st->n_quantized > st->offset)
    return fail(KVQ_ERR_RANGE, "%s: state offset %d / frontier %d out of range", fn, st->offset,
                st->n_quantized);
  return KVQ_OK;
}

kvq_status check_tensors(uint16_t* const* kc, uint16_t* const* vc, const uint16_t* const* kn,
                         const uint16_t* const* vn, int n_layers, int max_layers, const char* fn) {
  if (n_layers < 1 || n_layers > max_layers)
    return fail(KVQ_ERR_RANGE, "%s: n_layers %d not in [1, %d]", fn, n_layers, max_layers);
  if (!kc || !vc) return fail(KVQ_ERR_NULL, "%s: NULL cache array", fn);
  if ((kn == nullptr) != (vn == nullptr)) return fail(KVQ_ERR_NULL, "%s: NULL new-token array", fn);
  for (int i = 0; i < n_layers; ++i) {
    if (!kc[i] || !vc[i]) return fail(KVQ_ERR_NULL, "%s: cache of layer %d is NULL", fn, i);
    if (!aligned16(kc[i]) || !aligned16(vc[i]))
      return fail(KVQ_ERR_ALIGN, "%s: caches must be 16-byte aligned", fn);
    if (kn) {
      if (!kn[i] || !vn[i]) return fail(KVQ_ERR_NULL, "%s: new tokens of layer %d NULL", fn, i);
      if (!aligned16(kn[i]) || !aligned16(vn[i]))
        return fail(KVQ_ERR_ALIGN, "%s: new tokens must be 16-byte aligned", fn);
    }
  }
  return KVQ_OK;
}

kvq_status check_caches_match(const kivi_state* st, const kivi_packed* c, int n_layers,
                              const char* fn) {
  if (!c) return fail(KVQ_ERR_NULL, "%s: packed cache array is NULL", fn);
  const int gs = st->group_size;
  if ((gs != 8 && gs != 16 && gs != 32 && gs != 64) || st->head_dim % gs || st->capacity % gs)
    return fail(KVQ_ERR_SHAPE, "%s: packed group_size %d must be 8/16/32/64 and divide head_dim "
                "and capacity", fn, gs);
  for (int i = 0; i < n_layers; ++i) {
    const kivi_packed& p = c[i];
    if (p.bits != st->bits || p.group_size != st->group_size || p.batch != st->batch ||
        p.num_heads != st->num_heads || p.capacity != st->capacity ||
        p.head_dim != st->head_dim)
      return fail(KVQ_ERR_SHAPE, "%s: packed cache %d does not match the state", fn, i);
    if (!p.k_codes || !p.k_scale || !p.k_zero || !p.v_codes || !p.v_scale || !p.v_zero)
      return fail(KVQ_ERR_NULL, "%s: packed cache %d has a NULL array", fn, i);
    if (!aligned16(p.k_codes) || !aligned16(p.k_scale) || !aligned16(p.k_zero) ||
        !aligned16(p.v_codes) || !aligned16(p.v_scale) || !aligned16(p.v_zero))
      return fail(KVQ_ERR_ALIGN, "%s: packed cache %d arrays must be 16-byte aligned", fn, i);
  }
  return KVQ_OK;
}

kvq_status append(const kivi_state* st, uint16_t* const* kc, uint16_t* const* vc,
                  const uint16_t* const* kn, const uint16_t* const* vn, int n_layers, int n_new,
                  cudaStream_t cs, const char* fn) {
  if (n_new == 0) return KVQ_OK;
  AppendArgs a;
  for (int i = 0; i < KVQ_MAX_TENSORS; ++i) {
    const int l = i >> 1;
    a.dst[i] = (l < n_layers) ? ((i & 1) ? vc[l] : kc[l]) : nullptr;
    a.src[i] = (l < n_layers) ? ((i & 1) ? vn[l] : kn[l]) : nullptr;
  }
  a.n_tensors = 2 * n_layers;
  a.B = st->batch;
  a.H = st->num_heads;
  a.S = st->capacity;
  a.D = st->head_dim;
  a.offset = st->offset;
  a.n_new = n_new;
  const int64_t items = static_cast<int64_t>(a.n_tensors) * a.B * a.H * n_new * (a.D / 8);
  kivi_append_kernel<<<grid_for(items), kThreads, 0, cs>>>(a);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(KVQ_ERR_CUDA, "%s: append launch: %s", fn, cudaGetErrorString(e));
  return KVQ_OK;
}

kvq_status unpack(const kivi_packed* caches, uint16_t* const* k, uint16_t* const* v, int n_layers,
                  int lo, int hi, cudaStream_t cs, const char* fn) {
  if (hi <= lo) return KVQ_OK;
  UnpackArgs a;
  for (int i = 0; i < KVQ_MAX_TENSORS; ++i) {
    a.c[i] = caches[i < n_layers ? i : 0];
    a.k[i] = i < n_layers ? k[i] : nullptr;
    a.v[i] = i < n_layers ? v[i] : nullptr;
  }
  a.n_layers = n_layers;
  a.lo = lo;
  a.hi = hi;
  const kivi_packed& c0 = caches[0];
  const int64_t items = static_cast<int64_t>(2) * n_layers * c0.batch * c0.num_heads * (hi - lo) *
                        (c0.head_dim / 8);
  const int grid = grid_for(items);
  switch (c0.bits) {
    case 2: kivi_unpack_kernel<2><<<grid, kThreads, 0, cs>>>(a); break;
    case 4: kivi_unpack_kernel<4><<<grid, kThreads, 0, cs>>>(a); break;
    default: kivi_unpack_kernel<8><<<grid, kThreads, 0, cs>>>(a); break;
  }
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(KVQ_ERR_CUDA, "%s: unpack launch: %s", fn, cudaGetErrorString(e));
  return KVQ_OK;
}

}  // namespace
}  // namespace kvq

extern "C" kvq_status kivi_state_init(kivi_state* st, int batch, int num_heads, int head_dim,
                                      int capacity, int bits, int group_size,
                                      int residual_length) {
  using namespace kvq;
  if (!st) return fail(KVQ_ERR_NULL, "kivi_state_init: state is NULL");
  kivi_state s;
  s.batch = batch;
  s.num_heads = num_heads;
  s.head_dim = head_dim;
  s.capacity = capacity;
  s.bits = bits;
  s.group_size = group_size;
  s.residual_length = residual_length;
  s.eps = 1e-8f;
  s.offset = 0;
  s.n_quantized = 0;
  const kvq_status r = check_state(&s, "kivi_state_init");
  if (r != KVQ_OK) return r;
  *st = s;
  return ok();
}

extern "C" kvq_status kivi_update(kivi_state* st, uint16_t* const* k_cache, uint16_t* const* v_cache,
                                  const uint16_t* const* k_new, const uint16_t* const* v_new,
                                  int n_layers, int n_new, kvq_stream_t stream) {
  using namespace kvq;
  const char* fn = "kivi_update";
  kvq_status r = check_state(st, fn);
  if (r != KVQ_OK) return r;
  r = check_tensors(k_cache, v_cache, k_new, v_new, n_layers, KVQ_MAX_TENSORS / 2, fn);
  if (r != KVQ_OK) return r;
  if (n_new > 0 && (!k_new || !v_new)) return fail(KVQ_ERR_NULL, "%s: NULL new-token array", fn);
  if (n_new < 0 || n_new > st->capacity - st->offset)
    return fail(KVQ_ERR_RANGE, "%s: %d new tokens do not fit (offset %d, capacity %d)", fn, n_new,
                st->offset, st->capacity);
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  r = append(st, k_cache, v_cache, k_new, v_new, n_layers, n_new, cs, fn);
  if (r != KVQ_OK) return r;
  const int offset = st->offset + n_new;
  const int boundary = kivi_boundary(offset, st->residual_length, st->group_size);
  if (boundary > st->n_quantized) {
    uint16_t* x[KVQ_MAX_TENSORS];
    int32_t is_key[KVQ_MAX_TENSORS];
    for (int l = 0; l < n_layers; ++l) {
      x[2 * l] = k_cache[l];
      is_key[2 * l] = 1;
      x[2 * l + 1] = v_cache[l];
      is_key[2 * l + 1] = 0;
    }
    r = kivi_quant_dequant(x, is_key, 2 * n_layers, st->batch, st->num_heads, st->capacity,
                           st->head_dim, st->n_quantized, boundary, st->group_size,
                           (1 << st->bits) - 1, st->eps, stream);
    if (r != KVQ_OK) return r;
    st->n_quantized = boundary;
  }
  st->offset = offset;
  return ok();
}

extern "C" int kivi_trim(kivi_state* st, int n) {
  if (!st || n <= 0 || st->offset <= 0) return 0;
  const int trimmed = n < st->offset ? n : st->offset;
  st->offset -= trimmed;
  const int snapped = (st->offset / st->group_size) * st->group_size;
  if (snapped < st->n_quantized) st->n_quantized = snapped;
  return trimmed;
}

extern "C" kvq_status kivi_packed_update(kivi_state* st, const kivi_packed* caches,
                                         uint16_t* const* k_cache, uint16_t* const* v_cache,
                                         const uint16_t* const* k_new,
                                         const uint16_t* const* v_new, int n_layers, int n_new,
                                         kvq_stream_t stream) {
  using namespace kvq;
  const char* fn = "kivi_packed_update";
  kvq_status r = check_state(st, fn);
  if (r != KVQ_OK) return r;
  r = check_tensors(k_cache, v_cache, k_new, v_new, n_layers, KVQ_MAX_TENSORS / 2, fn);
  if (r != KVQ_OK) return r;
  r = check_caches_match(st, caches, n_layers, fn);
  if (r != KVQ_OK) return r;
  if (n_new > 0 && (!k_new || !v_new)) return fail(KVQ_ERR_NULL, "%s: NULL new-token array", fn);
  if (n_new < 0 || n_new > st->capacity - st->offset)
    return fail(KVQ_ERR_RANGE, "%s: %d new tokens do not fit (offset %d, capacity %d)", fn, n_new,
                st->offset, st->capacity);
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  r = append(st, k_cache, v_cache, k_new, v_new, n_layers, n_new, cs, fn);
  if (r != KVQ_OK) return r;
  const int offset = st->offset + n_new;
  const int boundary = kivi_boundary(offset, st->residual_length, st->group_size);
  if (boundary > st->n_quantized) {
    r = kivi_pack(caches, k_cache, v_cache, n_layers, st->n_quantized, boundary, st->eps,
                  stream);
    if (r != KVQ_OK) return r;
    st->n_quantized = boundary;
  }
  st->offset = offset;
  return ok();
}

extern "C" kvq_status kivi_packed_trim(kivi_state* st, const kivi_packed* caches,
                                       uint16_t* const* k_cache, uint16_t* const* v_cache,
                                       int n_layers, int n, int* trimmed, kvq_stream_t stream) {
  using namespace kvq;
  const char* fn = "kivi_packed_trim";
  kvq_status r = check_state(st, fn);
  if (r != KVQ_OK) return r;
  r = check_tensors(k_cache, v_cache, nullptr, nullptr, n_layers, KVQ_MAX_TENSORS, fn);
  if (r != KVQ_OK) return r;
  r = check_caches_match(st, caches, n_layers, fn);
  if (r != KVQ_OK) return r;
  const int cut = (n <= 0) ? 0 : (n < st->offset ? n : st->offset);
  const int offset = st->offset - cut;
  const int snapped = (offset / st->group_size) * st->group_size;
  const int new_nq = snapped < st->n_quantized ? snapped : st->n_quantized;
  const int hi = st->n_quantized < offset ? st->n_quantized : offset;
  if (cut > 0 && hi > new_nq) {
    r = unpack(caches, k_cache, v_cache, n_layers, new_nq, hi,
               reinterpret_cast<cudaStream_t>(stream), fn);
    if (r != KVQ_OK) return r;
  }
  if (cut > 0) {
    st->offset = offset;
    st->n_quantized = new_nq;
  }
  if (trimmed) *trimmed = cut;
  return ok();
}

extern "C" kvq_status kivi_unpack(const kivi_packed* caches, uint16_t* const* k,
                                  uint16_t* const* v, int n_layers, int lo, int hi,
                                  kvq_stream_t stream) {
  using namespace kvq;
  const char* fn = "kivi_unpack";
  if (!caches) return fail(KVQ_ERR_NULL, "%s: packed cache array is NULL", fn);
  if (n_layers < 1 || n_layers > KVQ_MAX_TENSORS)
    return fail(KVQ_ERR_RANGE, "%s: n_layers %d not in [1, %d]", fn, n_layers, KVQ_MAX_TENSORS);
  kivi_state st;
  const kivi_packed& c0 = caches[0];
  st.batch = c0.batch;
  st.num_heads = c0.num_heads;
  st.head_dim = c0.head_dim;
  st.capacity = c0.capacity;
  st.bits = c0.bits;
  st.group_size = c0.group_size;
  st.residual_length = 0;
  st.eps = 0.f;
  st.offset = c0.capacity;
  st.n_quantized = 0;
  kvq_status r = check_state(&st, fn);
  if (r != KVQ_OK) return r;
  r = check_caches_match(&st, caches, n_layers, fn);
  if (r != KVQ_OK) return r;
  r = check_tensors(k, v, nullptr, nullptr, n_layers, KVQ_MAX_TENSORS, fn);
  if (r != KVQ_OK) return r;
  if (lo < 0 || hi < lo || hi > c0.capacity)
    return fail(KVQ_ERR_SHAPE, "%s: need 0 <= lo <= hi <= capacity (lo %d hi %d)", fn, lo, hi);
  r = unpack(caches, k, v, n_layers, lo, hi, reinterpret_cast<cudaStream_t>(stream), fn);
  if (r != KVQ_OK) return r;
  return ok();
}
