// Host-side helpers shared by the libkvq entry points.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kvq.h"

namespace kvq {

// Record an error message for kvq_last_error_string() and return `st`.
kvq_status_t fail(kvq_status_t st, const char* fmt, ...);
// Clear the calling thread's last error.
void clear_error();
// Map a CUDA error (from a launch) to a status, recording its text.
kvq_status_t cuda_status(cudaError_t e, const char* where);
// Streaming multiprocessors of the current device (cached per device).
int sm_count();
inline bool aligned(const void* p, unsigned a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
// The failure-path test hook of kvq_debug_set_stall_ns (0 = off).
uint64_t stall_ns();

// Bytes between the pages of consecutive (block, KV head) pairs in the K and
// the V cache.  Separate caches: a K page and a V page (k_page, v_page bytes).
// Paired layout (v_cache == k_cache + k_page: each pair's K page followed by
// its V page in one allocation): both advance by k_page + v_page.
struct PageStrides {
  int64_t k, v;
  bool paired;
};
inline PageStrides page_strides(const void* k_cache, const void* v_cache, int64_t k_page, int64_t v_page) {
  const bool paired = static_cast<const uint8_t*>(v_cache) == static_cast<const uint8_t*>(k_cache) + k_page;
  return paired ? PageStrides{k_page + v_page, k_page + v_page, true} : PageStrides{k_page, v_page, false};
}

}  // namespace kvq
