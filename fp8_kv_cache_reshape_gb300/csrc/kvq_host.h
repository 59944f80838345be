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

}  // namespace kvq
