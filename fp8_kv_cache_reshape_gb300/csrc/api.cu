// libkvq: version, per-thread error text, device queries.
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <mutex>

#include "kvq_host.h"

namespace kvq {

static thread_local char g_err[512] = "";

kvq_status_t fail(kvq_status_t st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return st;
}

void clear_error() { g_err[0] = '\0'; }

kvq_status_t cuda_status(cudaError_t e, const char* where) {
  if (e == cudaSuccess) return KVQ_OK;
  return fail(KVQ_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

int sm_count() {
  static std::mutex mu;
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  std::lock_guard<std::mutex> lk(mu);
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    cache[dev] = n;
  }
  return cache[dev];
}

static std::atomic<uint64_t> g_stall_ns{0};
uint64_t stall_ns() { return g_stall_ns.load(std::memory_order_relaxed); }

}  // namespace kvq

extern "C" void kvq_debug_set_stall_ns(uint64_t ns) { kvq::g_stall_ns.store(ns, std::memory_order_relaxed); }

extern "C" int kvq_version(void) { return 10000; }

extern "C" const char* kvq_last_error_string(void) { return kvq::g_err; }
