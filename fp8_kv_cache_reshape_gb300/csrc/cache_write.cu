// kvq_reshape_and_cache and kvq_quantize_query.
//
// Quantization follows "FP8 quantization and long-context inference"
// (section 1.1: q = round(x / scale)) and "FP8 and KV cache" ("Dynamic or
// static scale": values whose quotient exceeds 448 saturate to 448): one IEEE
// float32 division, then one saturating round-to-nearest-even conversion.
// Per-KV-head scales follow "The state of FP8 KV-cache and attention
// quantization in vLLM" ("Kernel and vLLM improvements", per-head scales: the
// cache-write kernel takes an array of scales instead of a scalar).
//
// One CTA handles a group of 16 consecutive tokens of one KV head.  When the
// group's slots fill exactly one page (the common case: prefill chunks and
// cache fills) the V page is transposed in shared memory and written as full
// 16-byte rows; otherwise every token is scattered on its own.
#include "kvq_device.cuh"
#include "kvq_host.h"

namespace kvq {

namespace {

// 16 bf16 (two 16-byte loads) -> 16 floats.
KVQ_DEVINL void load16_bf16(const __nv_bfloat16* src, float (&x)[16]) {
  const uint4* s = reinterpret_cast<const uint4*>(src);
  uint4 a = __ldg(s), b = __ldg(s + 1);
  const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    x[2 * i] = __uint_as_float(w[i] << 16);
    x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

template <bool E5>
KVQ_DEVINL uint4 quant16(const float (&x)[16], float s) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t b0 = f32_to_fp8<E5>(__fdiv_rn(x[4 * i + 0], s));
    uint32_t b1 = f32_to_fp8<E5>(__fdiv_rn(x[4 * i + 1], s));
    uint32_t b2 = f32_to_fp8<E5>(__fdiv_rn(x[4 * i + 2], s));
    uint32_t b3 = f32_to_fp8<E5>(__fdiv_rn(x[4 * i + 3], s));
    w[i] = b0 | (b1 << 8) | (b2 << 16) | (b3 << 24);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// FP8 cache write (E4M3, or E5M2 when E5 is set).  grid = (ceil(T / 16), Hkv), block = 128.
// PT: per-token dynamic scales -- each (token, head) is quantized with
// amax_d |x| / (format maximum) of its own values, and the K and V scales are
// stored in the token's slot of the scale tail of its V page (a per-token V
// page is the P x D codes followed by P K scales and P V scales, float32;
// k_scale / v_scale are unused).
template <int D, bool E5, bool PT>
__global__ void __launch_bounds__(128) reshape_and_cache_fp8_kernel(
    const __nv_bfloat16* __restrict__ k, const __nv_bfloat16* __restrict__ v,
    const int64_t* __restrict__ slot_mapping, uint8_t* __restrict__ k_cache, uint8_t* __restrict__ v_cache,
    const float* __restrict__ k_scale, const float* __restrict__ v_scale, int T, int Hkv, int64_t num_slots,
    int64_t kstr, int64_t vstr, int* dev_status) {
  // kstr, vstr: bytes between consecutive (block, head) pages of each cache
  constexpr int CH = D / 16;          // 16-byte chunks per row
  constexpr int PAGE_BYTES = kPage * D;
  __shared__ __align__(16) uint8_t vt[D * kPage];  // transposed V page
  __shared__ int64_t slots[kPage];
  __shared__ int fast;

  const int g0 = blockIdx.x * kPage;
  const int h = blockIdx.y;
  const int tid = threadIdx.x;
  if (tid < kPage) {
    int t = g0 + tid;
    slots[tid] = (t < T) ? slot_mapping[t] : -1;
  }
  __syncthreads();
  if (tid == 0) {
    int64_t s0 = slots[0];
    bool ok = (g0 + kPage <= T) && s0 >= 0 && (s0 % kPage) == 0 && s0 + kPage <= num_slots;
    for (int i = 1; ok && i < kPage; ++i) ok = (slots[i] == s0 + i);
    fast = ok ? 1 : 0;
    for (int i = 0; i < kPage; ++i)
      if (slots[i] >= num_slots) set_status(dev_status, KVQ_DEV_BAD_SLOT);
  }
  __syncthreads();
  if constexpr (PT) {
    // one (token, 16-byte chunk) per thread; a token's CH chunks sit in CH
    // consecutive lanes, so its maximum is a CH-lane shuffle reduction
    static_assert(kPage * CH <= 128 && (CH & (CH - 1)) == 0, "one item per thread, CH a power of two");
    constexpr float kFmtMax = E5 ? 57344.f : 448.f;
    if (tid < kPage * CH) {  // whole warps: kPage * CH is a multiple of 32
      const int t = tid / CH, j = tid % CH;
      const int64_t slot = slots[t];
      const bool valid = slot >= 0 && slot < num_slots;
      float xk[16], xv[16];
      if (valid) {
        const size_t src = (static_cast<size_t>(g0 + t) * Hkv + h) * D + j * 16;
        load16_bf16(k + src, xk);
        load16_bf16(v + src, xv);
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) xk[i] = xv[i] = 0.f;
      }
      float ak = 0.f, av = 0.f;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        ak = fmaxf(ak, fabsf(xk[i]));
        av = fmaxf(av, fabsf(xv[i]));
      }
#pragma unroll
      for (int o = 1; o < CH; o <<= 1) {
        ak = fmaxf(ak, __shfl_xor_sync(0xffffffffu, ak, o));
        av = fmaxf(av, __shfl_xor_sync(0xffffffffu, av, o));
      }
      const float skt = ak > 0.f ? __fdiv_rn(ak, kFmtMax) : 1.f;  // an all-zero token keeps scale 1
      const float svt = av > 0.f ? __fdiv_rn(av, kFmtMax) : 1.f;
      if (valid) {
        const int64_t blk = slot / kPage;
        const int off = static_cast<int>(slot % kPage);
        const size_t page = (static_cast<size_t>(blk) * Hkv + h) * kstr;
        const size_t vpage = (static_cast<size_t>(blk) * Hkv + h) * vstr;
        if (j == 0) {  // the scale tail: K scales, then V scales, one per token slot
          float* tail = reinterpret_cast<float*>(v_cache + vpage + PAGE_BYTES);
          tail[off] = skt;
          tail[kPage + off] = svt;
        }
        *reinterpret_cast<uint4*>(k_cache + page + fp8_k_offset(off, j, D)) = quant16<E5>(xk, skt);
        const uint4 qv = quant16<E5>(xv, svt);
        const uint8_t* qb = reinterpret_cast<const uint8_t*>(&qv);
        const int slot_in_row = fp8_v_slot(off);
        if (fast) {
#pragma unroll
          for (int i = 0; i < 16; ++i) vt[(j * 16 + i) * kPage + slot_in_row] = qb[i];
        } else {
          uint8_t* vp = v_cache + vpage + slot_in_row;
#pragma unroll
          for (int i = 0; i < 16; ++i) vp[(j * 16 + i) * kPage] = qb[i];
        }
      }
    }
  }
  const float sk = PT ? 1.f : k_scale[h], sv = PT ? 1.f : v_scale[h];

  for (int u = tid; u < (PT ? 0 : kPage * CH); u += blockDim.x) {
    const int t = u / CH, j = u % CH;
    const int64_t slot = slots[t];
    if (slot < 0 || slot >= num_slots) continue;
    const int64_t blk = slot / kPage;
    const int off = static_cast<int>(slot % kPage);
    const size_t src = (static_cast<size_t>(g0 + t) * Hkv + h) * D + j * 16;
    const size_t page = (static_cast<size_t>(blk) * Hkv + h) * kstr;
    const size_t vpage = (static_cast<size_t>(blk) * Hkv + h) * vstr;
    float x[16];
    load16_bf16(k + src, x);
    *reinterpret_cast<uint4*>(k_cache + page + fp8_k_offset(off, j, D)) = quant16<E5>(x, sk);
    load16_bf16(v + src, x);
    uint4 qv = quant16<E5>(x, sv);
    const uint8_t* qb = reinterpret_cast<const uint8_t*>(&qv);
    const int slot_in_row = fp8_v_slot(off);
    if (fast) {
#pragma unroll
      for (int i = 0; i < 16; ++i) vt[(j * 16 + i) * kPage + slot_in_row] = qb[i];
    } else {
      uint8_t* vp = v_cache + vpage + slot_in_row;
#pragma unroll
      for (int i = 0; i < 16; ++i) vp[(j * 16 + i) * kPage] = qb[i];
    }
  }
  if (fast) {
    __syncthreads();
    const int64_t blk = slots[0] / kPage;
    uint8_t* vp = v_cache + (static_cast<size_t>(blk) * Hkv + h) * vstr;
    for (int d = tid; d < D; d += blockDim.x)
      *reinterpret_cast<uint4*>(vp + d * kPage) = *reinterpret_cast<const uint4*>(vt + d * kPage);
  }
}

// BF16 cache write (bit copy into the BF16 page format).
template <int D>
__global__ void __launch_bounds__(128) reshape_and_cache_bf16_kernel(
    const uint16_t* __restrict__ k, const uint16_t* __restrict__ v, const int64_t* __restrict__ slot_mapping,
    uint8_t* __restrict__ k_cache, uint8_t* __restrict__ v_cache, int T, int Hkv, int64_t num_slots,
    int64_t kstr, int64_t vstr, int* dev_status) {
  constexpr int ROWB = D * 2;
  constexpr int CH = ROWB / 16;  // 8 bf16 per chunk
  const int g0 = blockIdx.x * kPage;
  const int h = blockIdx.y;
  for (int u = threadIdx.x; u < kPage * CH; u += blockDim.x) {
    const int t = u / CH, j = u % CH;
    if (g0 + t >= T) continue;
    const int64_t slot = slot_mapping[g0 + t];
    if (slot < 0) continue;
    if (slot >= num_slots) {
      if (j == 0) set_status(dev_status, KVQ_DEV_BAD_SLOT);
      continue;
    }
    const int64_t blk = slot / kPage;
    const int off = static_cast<int>(slot % kPage);
    const size_t src = (static_cast<size_t>(g0 + t) * Hkv + h) * D + j * 8;
    uint8_t* page_k = k_cache + (static_cast<size_t>(blk) * Hkv + h) * kstr;
    uint8_t* page_v = v_cache + (static_cast<size_t>(blk) * Hkv + h) * vstr;
    *reinterpret_cast<uint4*>(page_k + k_chunk_offset(off, j, ROWB)) =
        __ldg(reinterpret_cast<const uint4*>(k + src));
    uint4 vv = __ldg(reinterpret_cast<const uint4*>(v + src));
    const uint16_t* ve = reinterpret_cast<const uint16_t*>(&vv);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int d = j * 8 + i;
      *reinterpret_cast<uint16_t*>(page_v + bf16_v_offset(d, off)) = ve[i];
    }
  }
}

// Query quantization: 16 elements per thread, scalar tail.
__global__ void __launch_bounds__(256) quantize_query_kernel(const __nv_bfloat16* __restrict__ q,
                                                             uint8_t* __restrict__ q8,
                                                             const float* __restrict__ q_scale, int64_t n) {
  const float s = *q_scale;
  const int64_t nvec = n / 16;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < nvec;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    float x[16];
    load16_bf16(q + i * 16, x);
    *reinterpret_cast<uint4*>(q8 + i * 16) = quant16<false>(x, s);
  }
  if (blockIdx.x == 0) {
    for (int64_t i = nvec * 16 + threadIdx.x; i < n; i += blockDim.x)
      q8[i] = f32_to_e4m3(__fdiv_rn(__bfloat162float(q[i]), s));
  }
}

}  // namespace

}  // namespace kvq

using namespace kvq;

extern "C" kvq_status_t kvq_reshape_and_cache(const void* k, const void* v, const int64_t* slot_mapping,
                                              void* k_cache, void* v_cache, const float* k_scale,
                                              const float* v_scale, int T, int Hkv, int D, int P,
                                              int64_t num_blocks, kvq_dtype_t cache_dtype, int* dev_status,
                                              kvq_stream_t stream) {
  clear_error();
  if (T < 0 || Hkv < 1 || num_blocks < 1) return fail(KVQ_ERR_INVALID_ARG, "reshape_and_cache: bad sizes");
  if (P != kPage) return fail(KVQ_ERR_UNSUPPORTED, "reshape_and_cache: page size %d (only 16)", P);
  if (cache_dtype != KVQ_DTYPE_FP8_E4M3 && cache_dtype != KVQ_DTYPE_FP8_E5M2 && cache_dtype != KVQ_DTYPE_BF16)
    return fail(KVQ_ERR_INVALID_ARG, "reshape_and_cache: bad cache dtype");
  const bool fp8 = cache_dtype != KVQ_DTYPE_BF16;
  if (D != 64 && D != 128 && !(fp8 && D == 256))
    return fail(KVQ_ERR_UNSUPPORTED, "reshape_and_cache: head_dim %d (64 or 128; 256 for FP8)", D);
  if (T == 0) return KVQ_OK;
  if (!k || !v || !slot_mapping || !k_cache || !v_cache)
    return fail(KVQ_ERR_INVALID_ARG, "reshape_and_cache: null pointer");
  if (fp8 && (!k_scale || !v_scale))
    return fail(KVQ_ERR_INVALID_ARG, "reshape_and_cache: FP8 needs k_scale and v_scale");
  if (!aligned(k, 16) || !aligned(v, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
      !aligned(slot_mapping, 8))
    return fail(KVQ_ERR_INVALID_ARG, "reshape_and_cache: pointers must be 16-byte aligned");
  if (Hkv > 65535) return fail(KVQ_ERR_UNSUPPORTED, "reshape_and_cache: too many KV heads");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  dim3 grid((T + kPage - 1) / kPage, Hkv);
  const int64_t num_slots = num_blocks * kPage;
  const int64_t page_b = static_cast<int64_t>(kPage) * D * (fp8 ? 1 : 2);
  const PageStrides ps = page_strides(k_cache, v_cache, page_b, page_b);
  if (fp8) {
    auto kb = static_cast<const __nv_bfloat16*>(k);
    auto vb = static_cast<const __nv_bfloat16*>(v);
    auto kc = static_cast<uint8_t*>(k_cache);
    auto vc = static_cast<uint8_t*>(v_cache);
    auto launch = [&](auto kernel) {
      kernel<<<grid, 128, 0, s>>>(kb, vb, slot_mapping, kc, vc, k_scale, v_scale, T, Hkv, num_slots, ps.k, ps.v,
                                  dev_status);
    };
    const bool e5 = cache_dtype == KVQ_DTYPE_FP8_E5M2;
    if (D == 256)
      e5 ? launch(reshape_and_cache_fp8_kernel<256, true, false>)
         : launch(reshape_and_cache_fp8_kernel<256, false, false>);
    else if (D == 128)
      e5 ? launch(reshape_and_cache_fp8_kernel<128, true, false>)
         : launch(reshape_and_cache_fp8_kernel<128, false, false>);
    else
      e5 ? launch(reshape_and_cache_fp8_kernel<64, true, false>) : launch(reshape_and_cache_fp8_kernel<64, false, false>);
  } else {
    auto kb = static_cast<const uint16_t*>(k);
    auto vb = static_cast<const uint16_t*>(v);
    auto kc = static_cast<uint8_t*>(k_cache);
    auto vc = static_cast<uint8_t*>(v_cache);
    if (D == 128)
      reshape_and_cache_bf16_kernel<128><<<grid, 128, 0, s>>>(kb, vb, slot_mapping, kc, vc, T, Hkv, num_slots,
                                                              ps.k, ps.v, dev_status);
    else
      reshape_and_cache_bf16_kernel<64><<<grid, 128, 0, s>>>(kb, vb, slot_mapping, kc, vc, T, Hkv, num_slots,
                                                             ps.k, ps.v, dev_status);
  }
  return cuda_status(cudaGetLastError(), "reshape_and_cache launch");
}

extern "C" kvq_status_t kvq_reshape_and_cache_per_token(const void* k, const void* v, const int64_t* slot_mapping,
                                                        void* k_cache, void* v_cache, int T, int Hkv, int D, int P,
                                                        int64_t num_blocks, kvq_dtype_t cache_dtype,
                                                        int* dev_status, kvq_stream_t stream) {
  clear_error();
  if (T < 0 || Hkv < 1 || num_blocks < 1) return fail(KVQ_ERR_INVALID_ARG, "reshape_and_cache_per_token: bad sizes");
  if (P != kPage) return fail(KVQ_ERR_UNSUPPORTED, "reshape_and_cache_per_token: page size %d (only 16)", P);
  if (D != 64 && D != 128) return fail(KVQ_ERR_UNSUPPORTED, "reshape_and_cache_per_token: head_dim %d", D);
  if (cache_dtype != KVQ_DTYPE_FP8_E4M3 && cache_dtype != KVQ_DTYPE_FP8_E5M2)
    return fail(KVQ_ERR_INVALID_ARG, "reshape_and_cache_per_token: cache dtype must be E4M3 or E5M2");
  if (T == 0) return KVQ_OK;
  if (!k || !v || !slot_mapping || !k_cache || !v_cache)
    return fail(KVQ_ERR_INVALID_ARG, "reshape_and_cache_per_token: null pointer");
  if (!aligned(k, 16) || !aligned(v, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
      !aligned(slot_mapping, 8))
    return fail(KVQ_ERR_INVALID_ARG, "reshape_and_cache_per_token: misaligned pointer");
  if (Hkv > 65535) return fail(KVQ_ERR_UNSUPPORTED, "reshape_and_cache_per_token: too many KV heads");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  dim3 grid((T + kPage - 1) / kPage, Hkv);
  const int64_t num_slots = num_blocks * kPage;
  auto kb = static_cast<const __nv_bfloat16*>(k);
  auto vb = static_cast<const __nv_bfloat16*>(v);
  auto kc = static_cast<uint8_t*>(k_cache);
  auto vc = static_cast<uint8_t*>(v_cache);
  const int64_t page_b = static_cast<int64_t>(kPage) * D;
  const PageStrides ps = page_strides(k_cache, v_cache, page_b, page_b + kScaleTailBytes);
  auto launch = [&](auto kernel) {
    kernel<<<grid, 128, 0, s>>>(kb, vb, slot_mapping, kc, vc, nullptr, nullptr, T, Hkv, num_slots, ps.k, ps.v,
                                dev_status);
  };
  const bool e5 = cache_dtype == KVQ_DTYPE_FP8_E5M2;
  if (D == 128)
    e5 ? launch(reshape_and_cache_fp8_kernel<128, true, true>) : launch(reshape_and_cache_fp8_kernel<128, false, true>);
  else
    e5 ? launch(reshape_and_cache_fp8_kernel<64, true, true>) : launch(reshape_and_cache_fp8_kernel<64, false, true>);
  return cuda_status(cudaGetLastError(), "reshape_and_cache_per_token launch");
}

extern "C" kvq_status_t kvq_quantize_query(const void* q, uint8_t* q8, const float* q_scale, int64_t n,
                                           kvq_stream_t stream) {
  clear_error();
  if (n < 0) return fail(KVQ_ERR_INVALID_ARG, "quantize_query: n < 0");
  if (n == 0) return KVQ_OK;
  if (!q || !q8 || !q_scale) return fail(KVQ_ERR_INVALID_ARG, "quantize_query: null pointer");
  if (!aligned(q, 16) || !aligned(q8, 16))
    return fail(KVQ_ERR_INVALID_ARG, "quantize_query: pointers must be 16-byte aligned");
  const int64_t nvec = n / 16;
  int64_t blocks = (nvec + 255) / 256;
  const int64_t cap = static_cast<int64_t>(sm_count()) * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  quantize_query_kernel<<<static_cast<unsigned>(blocks), 256, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const __nv_bfloat16*>(q), q8, q_scale, n);
  return cuda_status(cudaGetLastError(), "quantize_query launch");
}
