// Internal declarations shared by the libkvq translation units (host side).
#pragma once

#include <cstdint>
#include <cstddef>

#include "kvq.h"

namespace kvq {

// Records `msg` (printf-style) as this thread's last error and returns `st`.
kvq_status fail(kvq_status st, const char* fmt, ...);
// Clears this thread's last error and returns KVQ_OK.
kvq_status ok();

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline int qmax_of(int bits) {
  switch (bits) {
    case 8: return 127;
    case 6: return 31;
    case 4: return 7;
    default: return -1;
  }
}

// Checks one pool's description and pointers.  `what` names it in the message.
kvq_status check_pool(const kvq_pool& p, const char* what);

// Checks that every pool of an array matches the first one's bits/H/D/page_size.
kvq_status check_pools_uniform(const kvq_pool* pools, int n, const char* what);

// Number of SMs of the current device (cached per device).
int sm_count();

}  // namespace kvq
