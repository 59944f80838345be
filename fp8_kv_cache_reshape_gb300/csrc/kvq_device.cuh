// Device helpers for libkvq (sm_103a): inline PTX for mbarriers, bulk
// (TMA) copies, ldmatrix / movmatrix / mma.sync, and the cache layout rules
// of include/kvq.h.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <stdint.h>
#include <cstring>

#include "../../include/kvq.h"

#define KVQ_DEVINL __device__ __forceinline__

namespace kvq {

constexpr int kPage = 16;                 // tokens per page
constexpr int kScaleTailBytes = 2 * kPage * 4;  // per-token V page: P K scales, then P V scales (float32)
constexpr unsigned kWaitPolls = 1u << 26;        // try_wait polls before a wait is declared stuck
constexpr uint64_t kWaitNs = 2000000000ull;      // ... or 2 s of wall time, whichever comes first

// ------------------------------------------------------------ layout rules ---
// Byte offset of 16-byte chunk j of row t inside a K page whose rows are
// `row_bytes` long (64, 128 or 256).  Matches the TMA 64B/128B swizzle
// patterns, so a page can be staged with one contiguous bulk copy and read
// by ldmatrix without bank conflicts.
KVQ_DEVINL int k_chunk_offset(int t, int j, int row_bytes) {
  int pj;
  if (row_bytes == 128) pj = j ^ (t & 7);
  else if (row_bytes == 64) pj = j ^ ((t >> 1) & 3);
  else pj = (j & 8) | ((j ^ t) & 7);  // 256-byte rows: each half like a 128-byte row
  return t * row_bytes + (pj << 4);
}
// Byte offset of 16-byte chunk j of token t in an FP8 K page.  D <= 128: row
// t, chunk swizzled as above.  D = 256: two 2 KiB half-pages (dims 0-127,
// 128-255), each 16 rows of 128 bytes with the 128-byte-row swizzle, so that
// each half is a canonical SWIZZLE_128B K-major operand for tcgen05.mma.
KVQ_DEVINL int fp8_k_offset(int t, int j, int D) {
  if (D == 256) return (j >> 3) * (kPage * 128) + t * 128 + (((j & 7) ^ (t & 7)) << 4);
  return k_chunk_offset(t, j, D);
}
__host__ __device__ __forceinline__ int fp8_v_slot(int t) {  // rho in include/kvq.h
  return t < 8 ? (((t >> 1) << 2) | (t & 1)) : ((((t - 8) >> 1) << 2) | 2 | (t & 1));
}
// Byte offset of token t in row d of a BF16 V page (rows of 16 bf16 = 32 B).
KVQ_DEVINL int bf16_v_offset(int d, int t) {
  int half = (t >> 3) ^ ((d >> 2) & 1);
  return d * 32 + half * 16 + (t & 7) * 2;
}

// ------------------------------------------------------------- status word ---
KVQ_DEVINL void set_status(int* st, int bits) {
  if (st) atomicOr(st, bits);
}

// ---------------------------------------------------------------- smem / mbarrier
KVQ_DEVINL uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
KVQ_DEVINL void mbar_init(uint64_t* bar, unsigned count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
KVQ_DEVINL void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
KVQ_DEVINL void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}
KVQ_DEVINL void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
KVQ_DEVINL void mbar_arrive(uint64_t* bar) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(smem_u32(bar))
               : "memory");
}
KVQ_DEVINL void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(
                   smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
KVQ_DEVINL bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
KVQ_DEVINL uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Bounded wait: true when the phase completed; false after kWaitPolls polls,
// limit_ns nanoseconds (kWaitNs by default), or as soon as *abort_flag (if
// given) becomes nonzero.
KVQ_DEVINL bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag = nullptr,
                          uint64_t limit_ns = kWaitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (unsigned i = 1; i < kWaitPolls; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63) == 0) {
      if (abort_flag && *abort_flag) return false;
      if (globaltimer_ns() - t0 > limit_ns) return false;
    }
  }
  return false;
}
// Test hook of the failure path: when stall_ns > 0, a wait of at most stall_ns
// on `bar`, a barrier that nothing arrives on; it fails exactly like a stuck
// pipeline wait.  Returns true (no stall) when stall_ns == 0.
KVQ_DEVINL bool stall_wait(uint64_t* bar, uint64_t stall_ns, volatile int* abort_flag) {
  return stall_ns == 0 || mbar_wait(bar, 0, abort_flag, stall_ns);
}

// One contiguous global -> shared bulk copy that completes `bytes` of
// transaction count on `bar`.  dst, src 16-byte aligned; bytes % 16 == 0.
KVQ_DEVINL void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}
KVQ_DEVINL uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
// L2 policy for data that other CTAs read again soon (kept over evict-first lines).
KVQ_DEVINL uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// A 32-bit load cached in L2 only (no L1 line is left behind).
KVQ_DEVINL int ld_l2only_s32(const int32_t* src) {
  int v;
  asm volatile("ld.global.cg.s32 %0, [%1];" : "=r"(v) : "l"(src) : "memory");
  return v;
}
// Hint: bring `bytes` at src into L2 (no data returned, no completion to wait
// for).  src 16-byte aligned; bytes % 16 == 0.
KVQ_DEVINL void prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// Programmatic dependent launch: wait until the preceding grid's memory is visible.
KVQ_DEVINL void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Allow the programmatic dependent grid to be scheduled (it still waits for
// this grid's completion in grid_dependency_wait()).
KVQ_DEVINL void grid_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// max(a, b, c) in one instruction (sm_100 and later); NaN inputs are ignored as by fmaxf.
KVQ_DEVINL float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
KVQ_DEVINL void named_bar_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}
KVQ_DEVINL void named_bar_arrive(int id, int threads) {
  asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(threads) : "memory");
}
// Per-warpgroup register budget (all four warps of the warpgroup execute it).
template <int N>
KVQ_DEVINL void setmaxnreg_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <int N>
KVQ_DEVINL void setmaxnreg_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

// ---------------------------------------------------------- tensor-core ops ---
KVQ_DEVINL void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
KVQ_DEVINL uint32_t movmatrix_t(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}
// D = A(16x16, row) * B(16x8, col) + C, f16 inputs, f32 accumulators.
KVQ_DEVINL void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                        uint32_t b1, const float (&c)[4]) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%10,%11,%12,%13};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]), "f"(c[2]), "f"(c[3]));
}
KVQ_DEVINL void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                         uint32_t b1, const float (&c)[4]) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%10,%11,%12,%13};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]), "f"(c[2]), "f"(c[3]));
}

// Two float32 -> two E4M3 codes (lo -> low byte), RNE, saturating.
KVQ_DEVINL uint32_t f32x2_to_e4m3x2(float lo, float hi) {
  return static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3));
}
// Four E4M3 codes in one register -> two f16x2 registers (bytes 0,1 -> lo;
// bytes 2,3 -> hi); exact.
KVQ_DEVINL void e4m3x4_to_f16x2x2(uint32_t x, uint32_t& lo, uint32_t& hi) {
  asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, a;\n\tcvt.rn.f16x2.e4m3x2 %1, b;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(x));
}
// Four E5M2 codes in one register -> two f16x2 registers, as above; exact.
KVQ_DEVINL void e5m2x4_to_f16x2x2(uint32_t x, uint32_t& lo, uint32_t& hi) {
  asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %2;\n\t"
      "cvt.rn.f16x2.e5m2x2 %0, a;\n\tcvt.rn.f16x2.e5m2x2 %1, b;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(x));
}
template <bool E5>
KVQ_DEVINL void fp8x4_to_f16x2x2(uint32_t x, uint32_t& lo, uint32_t& hi) {
  if constexpr (E5) {
    e5m2x4_to_f16x2x2(x, lo, hi);
  } else {
    e4m3x4_to_f16x2x2(x, lo, hi);
  }
}
KVQ_DEVINL uint32_t pack_f16x2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}
KVQ_DEVINL uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}
// Two float32 FMAs in one instruction: (a.x*b.x + c.x, a.y*b.y + c.y).
KVQ_DEVINL float2 ffma2(float2 a, float2 b, float2 c) {
  unsigned long long ra, rb, rc, rd;
  memcpy(&ra, &a, 8);
  memcpy(&rb, &b, 8);
  memcpy(&rc, &c, 8);
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(rd) : "l"(ra), "l"(rb), "l"(rc));
  float2 d;
  memcpy(&d, &rd, 8);
  return d;
}
// Two float32 additions in one instruction.
KVQ_DEVINL float2 fadd2(float2 a, float2 b) {
  unsigned long long ra, rb, rd;
  memcpy(&ra, &a, 8);
  memcpy(&rb, &b, 8);
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(rd) : "l"(ra), "l"(rb));
  float2 d;
  memcpy(&d, &rd, 8);
  return d;
}
// 2^k for an integer-valued k <= 127, exactly (0 for k < -126, -inf or NaN):
// the rescale between two integer softmax stabilizers.
KVQ_DEVINL float exp2_int(float k) {
  if (!(k >= -126.f)) return 0.f;
  return __uint_as_float(static_cast<uint32_t>(127 + static_cast<int>(k)) << 23);
}
// E4M3 1.0 in all four bytes: the A operand of an MMA that sums the columns of B.
constexpr uint32_t kE4m3OnesX4 = 0x38383838u;
KVQ_DEVINL float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// float32 -> E4M3, round-to-nearest-even, saturating to +-448.
KVQ_DEVINL uint8_t f32_to_e4m3(float x) {
  return static_cast<uint8_t>(__nv_cvt_float_to_fp8(x, __NV_SATFINITE, __NV_E4M3));
}
// float32 -> E5M2, round-to-nearest-even, saturating to +-57344.
KVQ_DEVINL uint8_t f32_to_e5m2(float x) {
  return static_cast<uint8_t>(__nv_cvt_float_to_fp8(x, __NV_SATFINITE, __NV_E5M2));
}
template <bool E5>
KVQ_DEVINL uint8_t f32_to_fp8(float x) {
  if constexpr (E5)
    return f32_to_e5m2(x);
  else
    return f32_to_e4m3(x);
}

}  // namespace kvq
