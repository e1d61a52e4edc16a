// Host side of libkvq: error state, validation helpers, packed_dim, the KIVI boundary and the
// page allocator.  The only CUDA calls here are the SM-count query and the pointer queries of
// kvq_host_device_view.
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include <cuda_runtime.h>

#include "kvq_internal.h"

namespace kvq {

namespace {
thread_local char g_last_error[512] = {0};
}

kvq_status fail(kvq_status st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  int n = std::snprintf(g_last_error, sizeof(g_last_error), "%s: ", kvq_status_string(st));
  if (n > 0 && n < static_cast<int>(sizeof(g_last_error)))
    std::vsnprintf(g_last_error + n, sizeof(g_last_error) - n, fmt, ap);
  va_end(ap);
  return st;
}

kvq_status ok() {
  g_last_error[0] = 0;
  return KVQ_OK;
}

kvq_status check_pool(const kvq_pool& p, const char* what) {
  if (qmax_of(p.bits) < 0) return fail(KVQ_ERR_BITS, "%s: bits %d not in {8, 6, 4}", what, p.bits);
  if (p.head_dim > 256 || kvq_packed_dim(p.head_dim, p.bits) < 1)
    return fail(KVQ_ERR_SHAPE, "%s: head_dim %d not supported at %d bits (at most 256; q6 needs "
                "a multiple of 4, q4 of 2)", what, p.head_dim, p.bits);
  if (p.num_heads < 1) return fail(KVQ_ERR_SHAPE, "%s: num_heads %d < 1", what, p.num_heads);
  if (p.page_size < 1) return fail(KVQ_ERR_SHAPE, "%s: page_size %d < 1", what, p.page_size);
  if (p.num_pages < 1 || p.num_pages > INT32_MAX)
    return fail(KVQ_ERR_RANGE, "%s: num_pages %lld out of range", what,
                static_cast<long long>(p.num_pages));
  if (!p.codes || !p.scales) return fail(KVQ_ERR_NULL, "%s: codes/scales pointer is NULL", what);
  if (!aligned16(p.codes) || !aligned16(p.scales))
    return fail(KVQ_ERR_ALIGN, "%s: codes/scales must be 16-byte aligned", what);
  return KVQ_OK;
}

kvq_status check_pools_uniform(const kvq_pool* pools, int n, const char* what) {
  if (!pools) return fail(KVQ_ERR_NULL, "%s: pool array is NULL", what);
  for (int i = 0; i < n; ++i) {
    kvq_status st = check_pool(pools[i], what);
    if (st != KVQ_OK) return st;
    if (pools[i].bits != pools[0].bits || pools[i].num_heads != pools[0].num_heads ||
        pools[i].head_dim != pools[0].head_dim || pools[i].page_size != pools[0].page_size)
      return fail(KVQ_ERR_SHAPE, "%s: pool %d differs from pool 0 in bits/heads/dim/page_size",
                  what, i);
  }
  return KVQ_OK;
}

int sm_count() {
  static std::mutex mu;
  static std::vector<int> cache;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (static_cast<int>(cache.size()) <= dev) cache.resize(dev + 1, 0);
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cache[dev] = n;
  }
  return cache[dev];
}

}  // namespace kvq

extern "C" {

const char* kvq_version(void) { return "libkvq 0.1.0 (sm_103a)"; }

const char* kvq_last_error(void) { return kvq::g_last_error; }

const char* kvq_status_string(kvq_status status) {
  switch (status) {
    case KVQ_OK: return "KVQ_OK";
    case KVQ_ERR_BITS: return "KVQ_ERR_BITS";
    case KVQ_ERR_SHAPE: return "KVQ_ERR_SHAPE";
    case KVQ_ERR_NULL: return "KVQ_ERR_NULL";
    case KVQ_ERR_ALIGN: return "KVQ_ERR_ALIGN";
    case KVQ_ERR_RANGE: return "KVQ_ERR_RANGE";
    case KVQ_ERR_CUDA: return "KVQ_ERR_CUDA";
    case KVQ_ERR_NOMEM: return "KVQ_ERR_NOMEM";
    case KVQ_ERR_WORKSPACE: return "KVQ_ERR_WORKSPACE";
  }
  return "KVQ_ERR_UNKNOWN";
}

kvq_status kvq_host_device_view(const void* host_ptr, void** device_ptr) {
  using namespace kvq;
  if (!host_ptr || !device_ptr) return fail(KVQ_ERR_NULL, "kvq_host_device_view: NULL pointer");
  cudaPointerAttributes attr;
  cudaError_t e = cudaPointerGetAttributes(&attr, host_ptr);
  if (e != cudaSuccess)
    return fail(KVQ_ERR_CUDA, "kvq_host_device_view: cudaPointerGetAttributes: %s",
                cudaGetErrorString(e));
  if (attr.type == cudaMemoryTypeDevice || attr.type == cudaMemoryTypeManaged) {
    *device_ptr = const_cast<void*>(host_ptr);
    return ok();
  }
  if (attr.type != cudaMemoryTypeHost)
    return fail(KVQ_ERR_RANGE, "kvq_host_device_view: not page-locked host memory (allocate it "
                "with cudaHostAlloc or register it with cudaHostRegister)");
  void* d = nullptr;
  e = cudaHostGetDevicePointer(&d, const_cast<void*>(host_ptr), 0);
  if (e != cudaSuccess || d == nullptr)
    return fail(KVQ_ERR_CUDA, "kvq_host_device_view: cudaHostGetDevicePointer: %s",
                cudaGetErrorString(e));
  *device_ptr = d;
  return ok();
}

int kvq_packed_dim(int head_dim, int bits) {
  if (head_dim < 1) return -1;
  switch (bits) {
    case 8: return head_dim;
    case 6: return head_dim % 4 ? -1 : head_dim / 4 * 3;
    case 4: return head_dim % 2 ? -1 : head_dim / 2;
    default: return -1;
  }
}

int kivi_boundary(int offset, int residual_length, int group_size) {
  if (group_size < 1 || residual_length < 0) return -1;
  long long aged = static_cast<long long>(offset) - residual_length;
  if (aged < 0) aged = 0;
  return static_cast<int>((aged / group_size) * group_size);
}

// ------------------------------------------------------------------------------------------------
// Page allocator: a LIFO free list plus an "allocated" bitmap for double-free detection.
struct kvq_allocator {
  std::vector<int32_t> free_list;
  std::vector<uint8_t> in_use;
};

kvq_allocator* kvq_alloc_create(int64_t num_pages) {
  if (num_pages < 1 || num_pages > INT32_MAX) return nullptr;
  kvq_allocator* a = new (std::nothrow) kvq_allocator;
  if (!a) return nullptr;
  try {
    a->free_list.resize(static_cast<size_t>(num_pages));
    a->in_use.assign(static_cast<size_t>(num_pages), 0);
  } catch (...) {
    delete a;
    return nullptr;
  }
  // Hand out low ids first: the list is popped from the back.
  for (int64_t i = 0; i < num_pages; ++i)
    a->free_list[static_cast<size_t>(i)] = static_cast<int32_t>(num_pages - 1 - i);
  return a;
}

void kvq_alloc_destroy(kvq_allocator* a) { delete a; }

int64_t kvq_alloc_free_count(const kvq_allocator* a) {
  return a ? static_cast<int64_t>(a->free_list.size()) : -1;
}

kvq_status kvq_alloc_pages(kvq_allocator* a, int64_t n, int32_t* out_ids) {
  if (!a) return kvq::fail(KVQ_ERR_NULL, "allocator is NULL");
  if (n < 0) return kvq::fail(KVQ_ERR_RANGE, "negative page count");
  if (n > 0 && !out_ids) return kvq::fail(KVQ_ERR_NULL, "out_ids is NULL");
  if (static_cast<int64_t>(a->free_list.size()) < n)
    return kvq::fail(KVQ_ERR_NOMEM, "%lld pages requested, %zu free",
                     static_cast<long long>(n), a->free_list.size());
  for (int64_t i = 0; i < n; ++i) {
    int32_t id = a->free_list.back();
    a->free_list.pop_back();
    a->in_use[static_cast<size_t>(id)] = 1;
    out_ids[i] = id;
  }
  return kvq::ok();
}

kvq_status kvq_free_pages(kvq_allocator* a, int64_t n, const int32_t* ids) {
  if (!a) return kvq::fail(KVQ_ERR_NULL, "allocator is NULL");
  if (n < 0) return kvq::fail(KVQ_ERR_RANGE, "negative page count");
  if (n > 0 && !ids) return kvq::fail(KVQ_ERR_NULL, "ids is NULL");
  const int64_t total = static_cast<int64_t>(a->in_use.size());
  // validate everything first (all or nothing); mark with 2 to catch repeats
  int64_t i = 0;
  kvq_status st = KVQ_OK;
  for (; i < n; ++i) {
    int32_t id = ids[i];
    if (id < 0 || id >= total || a->in_use[static_cast<size_t>(id)] != 1) {
      st = kvq::fail(KVQ_ERR_RANGE, "page id %d is out of range, free, or repeated", id);
      break;
    }
    a->in_use[static_cast<size_t>(id)] = 2;
  }
  if (st != KVQ_OK) {
    for (int64_t j = 0; j < i; ++j) a->in_use[static_cast<size_t>(ids[j])] = 1;
    return st;
  }
  for (int64_t j = 0; j < n; ++j) {
    a->in_use[static_cast<size_t>(ids[j])] = 0;
    a->free_list.push_back(ids[j]);
  }
  return kvq::ok();
}

kvq_status kvq_table_reserve(kvq_allocator* a, int32_t* page_table, int max_pages, int page_size,
                             const int32_t* cur_len, const int32_t* new_tokens, int nseq) {
  if (!a || !page_table || !cur_len || !new_tokens)
    return kvq::fail(KVQ_ERR_NULL, "NULL argument to kvq_table_reserve");
  if (max_pages < 1 || page_size < 1 || nseq < 0)
    return kvq::fail(KVQ_ERR_RANGE, "bad max_pages/page_size/nseq");
  // count what is needed, checking ranges, before touching anything
  int64_t need = 0;
  for (int s = 0; s < nseq; ++s) {
    if (cur_len[s] < 0 || new_tokens[s] < 0)
      return kvq::fail(KVQ_ERR_RANGE, "negative length for sequence %d", s);
    int64_t end = static_cast<int64_t>(cur_len[s]) + new_tokens[s];
    if (new_tokens[s] == 0) continue;
    int64_t p0 = cur_len[s] / page_size, p1 = (end + page_size - 1) / page_size;
    if (p1 > max_pages)
      return kvq::fail(KVQ_ERR_RANGE, "sequence %d needs %lld pages > max_pages %d", s,
                       static_cast<long long>(p1), max_pages);
    for (int64_t p = p0; p < p1; ++p)
      if (page_table[static_cast<int64_t>(s) * max_pages + p] < 0) ++need;
  }
  if (need > static_cast<int64_t>(a->free_list.size()))
    return kvq::fail(KVQ_ERR_NOMEM, "%lld pages needed, %zu free", static_cast<long long>(need),
                     a->free_list.size());
  for (int s = 0; s < nseq; ++s) {
    if (new_tokens[s] == 0) continue;
    int64_t end = static_cast<int64_t>(cur_len[s]) + new_tokens[s];
    int64_t p0 = cur_len[s] / page_size, p1 = (end + page_size - 1) / page_size;
    for (int64_t p = p0; p < p1; ++p) {
      int32_t& e = page_table[static_cast<int64_t>(s) * max_pages + p];
      if (e < 0) {
        int32_t id = a->free_list.back();
        a->free_list.pop_back();
        a->in_use[static_cast<size_t>(id)] = 1;
        e = id;
      }
    }
  }
  return kvq::ok();
}

}  // extern "C"
