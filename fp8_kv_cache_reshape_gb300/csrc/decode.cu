// kvq_paged_decode_attention: split-KV paged decode over the FP8 (or BF16)
// cache, plus the log-sum-exp combine.
//
// Method: "The state of FP8 KV-cache and attention quantization in vLLM"
//  - "Performance benchmarks": decode cost is the per-token KV read (the ITL
//    slope), so the kernel streams pages at HBM speed and reads FP8 directly;
//  - "Problems we found" / "Kernel and vLLM improvements", two-level
//    accumulation: the P.V contraction runs over the whole context; here every
//    page's MMA result lands in fresh FP32 registers and is then added into a
//    running FP32 sum, and page ranges are merged in FP32 by the combine;
//  - "Skip layers": sliding-window layers read only the window's pages and
//    may keep a BF16 cache.
//
// Partial kernel (persistent): work item = (sequence, KV head, page range).
// Warp NW is the producer: it reads block ids and streams each page (K page +
// V page, one contiguous bulk copy each) into a ring of NST shared-memory
// stages guarded by mbarriers.  Warps 0..NW-1 consume pages round-robin.  Per
// page a consumer computes S^T = K Q^T (16 tokens x 8 query heads, M = tokens)
// with mma.m16n8k16 (f16 inputs: E4M3 converts to f16 exactly), updates an
// online softmax in base 2, transposes P in registers with movmatrix, and
// computes O^T += V^T P^T (M = dims) into fresh FP32 fragments.  At the end of
// an item the NW warp states are merged through shared memory and one
// normalized partial output + log2-sum-exp is written per query head.
#include <cfloat>
#include <cmath>

#include "kvq_device.cuh"
#include "kvq_host.h"

namespace kvq {

namespace {

constexpr float kLog2e = 1.4426950408889634f;

struct DecodeParams {
  const void* q;
  const uint8_t* k_cache;
  const uint8_t* v_cache;
  const float* k_scale;
  const float* v_scale;
  const int32_t* block_table;
  const int32_t* seq_lens;
  float* o_part;    // [B][Hq][S][D]
  float* lse_part;  // [B][Hq][S], log2 units
  int B, Hq, Hkv, g, max_blocks;
  int64_t num_blocks;
  float sm_scale;
  int window;
  int num_splits;
  int pages_per_split;
  int num_items;
  int* dev_status;
};

template <int D, bool FP8>
struct Geo {
  static constexpr int ESZ = FP8 ? 1 : 2;
  static constexpr int ROWB = D * ESZ;        // bytes of one K row
  static constexpr int PAGE = kPage * ROWB;   // bytes of one K page (= one V page)
  static constexpr int STAGE = 2 * PAGE;
  static constexpr int MT = D / 16;           // 16-row tiles of O^T
  static constexpr int KS = D / 16;           // 16-dim k-steps of QK
};

template <int D, bool FP8, int NW, int NST>
constexpr size_t decode_smem_bytes() {
  return size_t(NST) * Geo<D, FP8>::STAGE + 2 * NST * sizeof(uint64_t) + NST * sizeof(int) +
         (2 * NW * 8 + NW * 8 * D) * sizeof(float) + 16;
}

struct ItemRange {
  int b, kvh, split;
  int lo, hi;     // attended token positions [lo, hi)
  int pg0, n;     // first page and page count of this split
};

KVQ_DEVINL ItemRange item_range(const DecodeParams& p, int item, bool report) {
  ItemRange r;
  const int S = p.num_splits;
  const int bh = item / S;
  r.split = item - bh * S;
  r.b = bh / p.Hkv;
  r.kvh = bh - r.b * p.Hkv;
  int L = p.seq_lens[r.b];
  const int cap = p.max_blocks * kPage;
  if (L < 0 || L > cap) {
    if (report) set_status(p.dev_status, KVQ_DEV_BAD_SEQLEN);
    L = L < 0 ? 0 : cap;
  }
  r.hi = L;
  r.lo = (p.window > 0 && L > p.window) ? L - p.window : 0;
  const int first = r.lo / kPage;
  const int last = (L + kPage - 1) / kPage;
  r.pg0 = first + r.split * p.pages_per_split;
  int pg1 = r.pg0 + p.pages_per_split;
  if (pg1 > last) pg1 = last;
  r.n = pg1 > r.pg0 ? pg1 - r.pg0 : 0;
  return r;
}

template <int D, bool FP8, int NW, int NST>
__global__ void __launch_bounds__((NW + 1) * 32) decode_partial_kernel(const __grid_constant__ DecodeParams p) {
  using G = Geo<D, FP8>;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* stages = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + size_t(NST) * G::STAGE);
  uint64_t* empty = full + NST;
  int* stage_bad = reinterpret_cast<int*>(empty + NST);
  float* mbuf = reinterpret_cast<float*>(stage_bad + NST);  // [NW][8]
  float* lbuf = mbuf + NW * 8;                              // [NW][8]
  float* obuf = lbuf + NW * 8;                              // [NW][8][D]
  volatile int* abort_flag = reinterpret_cast<volatile int*>(obuf + NW * 8 * D);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < NST; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();

  if (warp == NW) {
    // ------------------------------------------------------------ producer --
    const uint64_t pol = policy_evict_first();
    uint32_t it = 0;
    bool aborted = false;
    for (int item = blockIdx.x; item < p.num_items && !aborted; item += gridDim.x) {
      const ItemRange r = item_range(p, item, lane == 0 && threadIdx.x == NW * 32);
      const int32_t* bt = p.block_table + static_cast<size_t>(r.b) * p.max_blocks + r.pg0;
      for (int base = 0; base < r.n && !aborted; base += 32) {
        const int cnt = min(32, r.n - base);
        int blk = 0, bad = 0;
        if (lane < cnt) {
          blk = __ldg(bt + base + lane);
          if (blk < 0 || static_cast<int64_t>(blk) >= p.num_blocks) {
            bad = 1;
            blk = 0;
            set_status(p.dev_status, KVQ_DEV_BAD_BLOCK);
          }
        }
        for (int j = 0; j < cnt; ++j, ++it) {
          const int bj = __shfl_sync(0xffffffffu, blk, j);
          const int badj = __shfl_sync(0xffffffffu, bad, j);
          int ok = 1;
          if (lane == 0) {
            const int st = it % NST;
            const uint32_t ph = (it / NST) & 1;
            if (*abort_flag || !mbar_wait(&empty[st], ph ^ 1, abort_flag)) {
              ok = 0;
            } else {
              stage_bad[st] = badj;
              mbar_arrive_expect_tx(&full[st], G::STAGE);
              const size_t page = (static_cast<size_t>(bj) * p.Hkv + r.kvh) * G::PAGE;
              uint8_t* sk = stages + size_t(st) * G::STAGE;
              bulk_g2s(sk, p.k_cache + page, G::PAGE, &full[st], pol);
              bulk_g2s(sk + G::PAGE, p.v_cache + page, G::PAGE, &full[st], pol);
            }
          }
          ok = __shfl_sync(0xffffffffu, ok, 0);
          if (!ok) {
            aborted = true;
            break;
          }
        }
      }
    }
    if (aborted && lane == 0) {
      set_status(p.dev_status, KVQ_DEV_TIMEOUT);
      *abort_flag = 1;
      // let copies already issued land before the CTA exits
      const uint32_t first = it > NST ? it - NST : 0;
      for (uint32_t k = first; k < it; ++k) mbar_wait(&full[k % NST], (k / NST) & 1);
    }
    return;
  }

  // ------------------------------------------------------------- consumers --
  const int r = lane >> 2;   // fragment row group
  const int c = lane & 3;    // fragment column pair
  const float NEG_INF = -INFINITY;
  // per-lane ldmatrix offsets for the K page (constant per page)
  int koff[G::KS / (FP8 ? 2 : 1)];
  {
    const int tok = (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
    for (int i = 0; i < G::KS / (FP8 ? 2 : 1); ++i) {
      const int ch = FP8 ? (2 * i + (lane >> 4)) : (2 * i + (lane >> 4));
      koff[i] = k_chunk_offset(tok, ch, G::ROWB);
    }
  }
  int voff[FP8 ? (G::MT / 2) : G::MT];
  if constexpr (FP8) {
#pragma unroll
    for (int i = 0; i < G::MT / 2; ++i) voff[i] = (32 * i + lane) * kPage;
  } else {
#pragma unroll
    for (int i = 0; i < G::MT; ++i) {
      const int row = 16 * i + (lane & 7) + ((lane >> 3) & 1) * 8;
      const int half = lane >> 4;
      voff[i] = row * 32 + 16 * (half ^ ((row >> 2) & 1));
    }
  }

  uint32_t it0 = 0;
  for (int item = blockIdx.x; item < p.num_items; item += gridDim.x) {
    const ItemRange rg = item_range(p, item, false);
    // query fragments of head (kvh * g + r); heads >= g are zero padding
    uint32_t qf[G::KS][2];
    {
      const bool live = r < p.g;
      const uint16_t* qrow = static_cast<const uint16_t*>(p.q) +
                             (static_cast<size_t>(rg.b) * p.Hq + rg.kvh * p.g + (live ? r : 0)) * D;
#pragma unroll
      for (int kk = 0; kk < G::KS; ++kk) {
        if constexpr (FP8) {
          const uint2 w = live ? __ldg(reinterpret_cast<const uint2*>(qrow + kk * 16 + 4 * c)) : make_uint2(0, 0);
          const float x0 = __uint_as_float(w.x << 16), x1 = __uint_as_float(w.x & 0xFFFF0000u);
          const float x2 = __uint_as_float(w.y << 16), x3 = __uint_as_float(w.y & 0xFFFF0000u);
          qf[kk][0] = pack_f16x2(x0, x1);
          qf[kk][1] = pack_f16x2(x2, x3);
        } else {
          qf[kk][0] = live ? __ldg(reinterpret_cast<const uint32_t*>(qrow + kk * 16 + 2 * c)) : 0u;
          qf[kk][1] = live ? __ldg(reinterpret_cast<const uint32_t*>(qrow + kk * 16 + 8 + 2 * c)) : 0u;
        }
      }
    }
    float coef;
    if constexpr (FP8) coef = __fmul_rn(__fmul_rn(p.k_scale[rg.kvh], p.sm_scale), kLog2e);
    else coef = __fmul_rn(p.sm_scale, kLog2e);

    float m[2] = {NEG_INF, NEG_INF};
    float l[2] = {0.f, 0.f};
    float O[G::MT][4];
#pragma unroll
    for (int i = 0; i < G::MT; ++i) O[i][0] = O[i][1] = O[i][2] = O[i][3] = 0.f;

    int i = (warp - static_cast<int>(it0 % NW) + NW) % NW;
    if (*abort_flag) i = rg.n;  // abandoned: skip the pages, keep the barriers in step
    for (; i < rg.n; i += NW) {
      const uint32_t itg = it0 + i;
      const int st = itg % NST;
      if (!mbar_wait(&full[st], (itg / NST) & 1, abort_flag)) {
        if (lane == 0) {
          set_status(p.dev_status, KVQ_DEV_TIMEOUT);
          *abort_flag = 1;
        }
        break;
      }
      const uint8_t* sk = stages + size_t(st) * G::STAGE;
      const uint32_t kb = smem_u32(sk);
      const uint32_t vb = kb + G::PAGE;
      const int tok0 = (rg.pg0 + i) * kPage;
      const bool edge = stage_bad[st] || tok0 < rg.lo || tok0 + kPage > rg.hi;

      // ---- S^T = K Q^T : 16 tokens x 8 heads ----
      float s[4] = {0.f, 0.f, 0.f, 0.f};
      if constexpr (FP8) {
#pragma unroll
        for (int kk = 0; kk < G::KS; kk += 2) {
          uint32_t x0, x1, x2, x3;
          ldsm_x4(kb + koff[kk / 2], x0, x1, x2, x3);
          mma_f16(s, e4m3x2_to_f16x2(x0 & 0xFFFF), e4m3x2_to_f16x2(x1 & 0xFFFF), e4m3x2_to_f16x2(x0 >> 16),
                  e4m3x2_to_f16x2(x1 >> 16), qf[kk][0], qf[kk][1], s);
          mma_f16(s, e4m3x2_to_f16x2(x2 & 0xFFFF), e4m3x2_to_f16x2(x3 & 0xFFFF), e4m3x2_to_f16x2(x2 >> 16),
                  e4m3x2_to_f16x2(x3 >> 16), qf[kk + 1][0], qf[kk + 1][1], s);
        }
      } else {
#pragma unroll
        for (int kk = 0; kk < G::KS; ++kk) {
          uint32_t x0, x1, x2, x3;
          ldsm_x4(kb + koff[kk], x0, x1, x2, x3);
          mma_bf16(s, x0, x1, x2, x3, qf[kk][0], qf[kk][1], s);
        }
      }
      // ---- scale, mask, online softmax (base 2) ----
      bool ok0 = true, ok1 = true;  // tokens r and r + 8 of this page
      uint32_t vmask_lo = 0xFFFFFFFFu, vmask_hi = 0xFFFFFFFFu;
#pragma unroll
      for (int e = 0; e < 4; ++e) s[e] *= coef;
      if (edge) {
        const bool bad = stage_bad[st] != 0;
        auto live = [&](int t) { return !bad && tok0 + t >= rg.lo && tok0 + t < rg.hi; };
        ok0 = live(r);
        ok1 = live(r + 8);
        if (!ok0) s[0] = s[1] = NEG_INF;
        if (!ok1) s[2] = s[3] = NEG_INF;
        // V fragment lanes hold tokens 2c, 2c+1 (low) and 2c+8, 2c+9 (high)
        const bool t0 = live(2 * c), t1 = live(2 * c + 1), t8 = live(2 * c + 8), t9 = live(2 * c + 9);
        if constexpr (FP8) {
          vmask_lo = (t0 ? 0x000000FFu : 0u) | (t1 ? 0x0000FF00u : 0u) | (t8 ? 0x00FF0000u : 0u) |
                     (t9 ? 0xFF000000u : 0u);
        } else {
          vmask_lo = (t0 ? 0x0000FFFFu : 0u) | (t1 ? 0xFFFF0000u : 0u);
          vmask_hi = (t8 ? 0x0000FFFFu : 0u) | (t9 ? 0xFFFF0000u : 0u);
        }
      }
      float mx0 = fmaxf(s[0], s[2]), mx1 = fmaxf(s[1], s[3]);
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
      }
      const float mn0 = fmaxf(m[0], mx0), mn1 = fmaxf(m[1], mx1);
      const float base0 = (mn0 == NEG_INF) ? 0.f : mn0;
      const float base1 = (mn1 == NEG_INF) ? 0.f : mn1;
      const float al0 = ex2(m[0] - base0), al1 = ex2(m[1] - base1);  // rescale of the running sums
      m[0] = mn0;
      m[1] = mn1;
      const float p0 = ex2(s[0] - base0), p1 = ex2(s[1] - base1), p2 = ex2(s[2] - base0), p3 = ex2(s[3] - base1);
      l[0] = l[0] * al0 + (p0 + p2);
      l[1] = l[1] * al1 + (p1 + p3);

      // ---- O^T += V^T P^T : dims x 8 heads, fresh FP32 per page ----
      if constexpr (FP8) {
        // P as the sum of two f16 terms (hi + lo): ~22 significant bits
        const uint32_t h0 = pack_f16x2(p0, p1), h1 = pack_f16x2(p2, p3);
        const float2 f0 = __half22float2(*reinterpret_cast<const __half2*>(&h0));
        const float2 f1 = __half22float2(*reinterpret_cast<const __half2*>(&h1));
        const uint32_t pb0 = movmatrix_t(h0);  // tokens 2c, 2c+1 of head r
        const uint32_t pb1 = movmatrix_t(h1);  // tokens 2c+8, 2c+9 of head r
        const uint32_t pl0 = movmatrix_t(pack_f16x2(p0 - f0.x, p1 - f0.y));
        const uint32_t pl1 = movmatrix_t(pack_f16x2(p2 - f1.x, p3 - f1.y));
#pragma unroll
        for (int mt = 0; mt < G::MT; mt += 2) {
          uint32_t y0, y1, y2, y3;
          ldsm_x4(vb + voff[mt / 2], y0, y1, y2, y3);
          y0 &= vmask_lo;
          y1 &= vmask_lo;
          y2 &= vmask_lo;
          y3 &= vmask_lo;
          float t[4] = {0.f, 0.f, 0.f, 0.f};
          const uint32_t va0 = e4m3x2_to_f16x2(y0 & 0xFFFF), va1 = e4m3x2_to_f16x2(y1 & 0xFFFF);
          const uint32_t va2 = e4m3x2_to_f16x2(y0 >> 16), va3 = e4m3x2_to_f16x2(y1 >> 16);
          mma_f16(t, va0, va1, va2, va3, pb0, pb1, t);
          mma_f16(t, va0, va1, va2, va3, pl0, pl1, t);
          O[mt][0] = fmaf(O[mt][0], al0, t[0]);
          O[mt][1] = fmaf(O[mt][1], al1, t[1]);
          O[mt][2] = fmaf(O[mt][2], al0, t[2]);
          O[mt][3] = fmaf(O[mt][3], al1, t[3]);
          float u[4] = {0.f, 0.f, 0.f, 0.f};
          const uint32_t vb0 = e4m3x2_to_f16x2(y2 & 0xFFFF), vb1 = e4m3x2_to_f16x2(y3 & 0xFFFF);
          const uint32_t vb2 = e4m3x2_to_f16x2(y2 >> 16), vb3 = e4m3x2_to_f16x2(y3 >> 16);
          mma_f16(u, vb0, vb1, vb2, vb3, pb0, pb1, u);
          mma_f16(u, vb0, vb1, vb2, vb3, pl0, pl1, u);
          O[mt + 1][0] = fmaf(O[mt + 1][0], al0, u[0]);
          O[mt + 1][1] = fmaf(O[mt + 1][1], al1, u[1]);
          O[mt + 1][2] = fmaf(O[mt + 1][2], al0, u[2]);
          O[mt + 1][3] = fmaf(O[mt + 1][3], al1, u[3]);
        }
      } else {
        // P as the sum of two bf16 terms (hi + lo) keeps ~16 significant bits
        const uint32_t h0 = pack_bf16x2(p0, p1), h1 = pack_bf16x2(p2, p3);
        const float r0 = p0 - __uint_as_float(h0 << 16), r1 = p1 - __uint_as_float(h0 & 0xFFFF0000u);
        const float r2 = p2 - __uint_as_float(h1 << 16), r3 = p3 - __uint_as_float(h1 & 0xFFFF0000u);
        const uint32_t ph0 = movmatrix_t(h0), ph1 = movmatrix_t(h1);
        const uint32_t pl0 = movmatrix_t(pack_bf16x2(r0, r1)), pl1 = movmatrix_t(pack_bf16x2(r2, r3));
#pragma unroll
        for (int mt = 0; mt < G::MT; ++mt) {
          uint32_t y0, y1, y2, y3;
          ldsm_x4(vb + voff[mt], y0, y1, y2, y3);
          y0 &= vmask_lo;
          y1 &= vmask_lo;
          y2 &= vmask_hi;
          y3 &= vmask_hi;
          float t[4] = {0.f, 0.f, 0.f, 0.f};
          mma_bf16(t, y0, y1, y2, y3, ph0, ph1, t);
          mma_bf16(t, y0, y1, y2, y3, pl0, pl1, t);
          O[mt][0] = fmaf(O[mt][0], al0, t[0]);
          O[mt][1] = fmaf(O[mt][1], al1, t[1]);
          O[mt][2] = fmaf(O[mt][2], al0, t[2]);
          O[mt][3] = fmaf(O[mt][3], al1, t[3]);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st]);
    }
    it0 += rg.n;

    // ---- merge the NW warp states of this item ----
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      l[0] += __shfl_xor_sync(0xffffffffu, l[0], o);
      l[1] += __shfl_xor_sync(0xffffffffu, l[1], o);
    }
    if (r == 0) {
      mbuf[warp * 8 + 2 * c] = m[0];
      mbuf[warp * 8 + 2 * c + 1] = m[1];
      lbuf[warp * 8 + 2 * c] = l[0];
      lbuf[warp * 8 + 2 * c + 1] = l[1];
    }
    float* ow = obuf + warp * 8 * D;
#pragma unroll
    for (int mt = 0; mt < G::MT; ++mt) {
      const int d = mt * 16 + r;
      ow[(2 * c) * D + d] = O[mt][0];
      ow[(2 * c + 1) * D + d] = O[mt][1];
      ow[(2 * c) * D + d + 8] = O[mt][2];
      ow[(2 * c + 1) * D + d + 8] = O[mt][3];
    }
    named_bar_sync(1, NW * 32);
    const float vs = FP8 ? p.v_scale[rg.kvh] : 1.f;
    const size_t row0 = static_cast<size_t>(rg.b) * p.Hq + rg.kvh * p.g;
    for (int e = warp * 32 + lane; e < p.g * D; e += NW * 32) {
      const int h = e / D, d = e - h * D;
      float M = NEG_INF;
#pragma unroll
      for (int w = 0; w < NW; ++w) M = fmaxf(M, mbuf[w * 8 + h]);
      float o = 0.f, lse = NEG_INF;
      if (M != NEG_INF) {
        float den = 0.f, num = 0.f;
#pragma unroll
        for (int w = 0; w < NW; ++w) {
          const float f = ex2(mbuf[w * 8 + h] - M);
          den += f * lbuf[w * 8 + h];
          num += f * obuf[(w * 8 + h) * D + d];
        }
        o = num / den * vs;
        lse = M + __log2f(den);
      }
      const size_t idx = (row0 + h) * p.num_splits + rg.split;
      p.o_part[idx * D + d] = o;
      if (d == 0) p.lse_part[idx] = lse;
    }
    named_bar_sync(1, NW * 32);
  }
}

// out[row][d] = sum_s 2^(lse_s - M) o_s[d] / sum_s 2^(lse_s - M), row = (b, hq).
template <int D>
__global__ void __launch_bounds__(D) decode_combine_kernel(const float* __restrict__ o_part,
                                                           const float* __restrict__ lse_part,
                                                           __nv_bfloat16* __restrict__ out, int S) {
  const int row = blockIdx.x;
  const int d = threadIdx.x;
  const float* lp = lse_part + static_cast<size_t>(row) * S;
  float M = -INFINITY;
  for (int s = 0; s < S; ++s) M = fmaxf(M, lp[s]);
  float acc = 0.f, den = 0.f;
  if (M != -INFINITY) {
    const float* op = o_part + static_cast<size_t>(row) * S * D + d;
    for (int s = 0; s < S; ++s) {
      const float w = ex2(lp[s] - M);
      den += w;
      acc = fmaf(w, op[static_cast<size_t>(s) * D], acc);
    }
    acc = acc / den;
  }
  out[static_cast<size_t>(row) * D + d] = __float2bfloat16_rn(acc);
}

constexpr int kNW = 4;     // consumer warps per CTA
constexpr int kCtasPerSm = 2;

template <int D, bool FP8>
constexpr int stages_for() {  // about 64 KiB of pages in flight per CTA
  return (65536 / Geo<D, FP8>::STAGE) > 32 ? 32 : (65536 / Geo<D, FP8>::STAGE);
}

int decode_pages(int P, int max_blocks, int window) {
  int pages = max_blocks;
  if (window > 0) {
    const int w = (window + P - 1) / P + 1;
    if (w < pages) pages = w;
  }
  return pages < 1 ? 1 : pages;
}

void split_plan(int B, int Hkv, int P, int max_blocks, int window, int num_splits, int* S_out, int* pps_out) {
  const int pages = decode_pages(P, max_blocks, window);
  int S;
  if (num_splits > 0) {
    S = num_splits;
  } else {
    const long target = 4L * kCtasPerSm * sm_count();
    const long pairs = static_cast<long>(B) * Hkv;
    S = static_cast<int>((target + pairs - 1) / pairs);
    const int max_s = (pages + 15) / 16;
    if (S > max_s) S = max_s;
  }
  if (S > pages) S = pages;
  if (S < 1) S = 1;
  const int pps = (pages + S - 1) / S;
  S = (pages + pps - 1) / pps;
  *S_out = S;
  *pps_out = pps;
}

template <int D, bool FP8>
kvq_status_t launch_decode(const DecodeParams& p, __nv_bfloat16* out, cudaStream_t s) {
  constexpr int NST = stages_for<D, FP8>();
  constexpr size_t smem = decode_smem_bytes<D, FP8, kNW, NST>();
  auto kern = decode_partial_kernel<D, FP8, kNW, NST>;
  static int configured_mask = 0;  // devices whose attribute is set
  int dev = 0;
  cudaGetDevice(&dev);
  if (!(configured_mask & (1 << (dev & 31)))) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return cuda_status(e, "decode: set shared memory size");
    configured_mask |= 1 << (dev & 31);
  }
  int grid = kCtasPerSm * sm_count();
  if (grid > p.num_items) grid = p.num_items;
  kern<<<grid, (kNW + 1) * 32, smem, s>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_status(e, "decode partial launch");
  decode_combine_kernel<D><<<p.B * p.Hq, D, 0, s>>>(p.o_part, p.lse_part, out, p.num_splits);
  return cuda_status(cudaGetLastError(), "decode combine launch");
}

}  // namespace

}  // namespace kvq

using namespace kvq;

extern "C" int kvq_decode_num_splits(int B, int Hkv, int P, int max_blocks, int window, int num_splits) {
  if (B < 1 || Hkv < 1 || P < 1 || max_blocks < 1 || num_splits < 0) return 0;
  int S, pps;
  split_plan(B, Hkv, P, max_blocks, window, num_splits, &S, &pps);
  return S;
}

extern "C" size_t kvq_decode_workspace_size(int B, int Hq, int Hkv, int D, int P, int max_blocks, int window,
                                            int num_splits) {
  if (B < 1 || Hq < 1 || Hkv < 1 || D < 1 || P < 1 || max_blocks < 1 || num_splits < 0) return 0;
  int S, pps;
  split_plan(B, Hkv, P, max_blocks, window, num_splits, &S, &pps);
  const size_t rows = static_cast<size_t>(B) * Hq * S;
  const size_t o_bytes = rows * D * sizeof(float);
  return o_bytes + ((rows * sizeof(float) + 15) / 16) * 16;
}

extern "C" kvq_status_t kvq_paged_decode_attention(const void* q, const void* k_cache, const void* v_cache,
                                                   const float* k_scale, const float* v_scale,
                                                   const int32_t* block_table, const int32_t* seq_lens, void* out,
                                                   int B, int Hq, int Hkv, int D, int P, int max_blocks,
                                                   int64_t num_blocks, float sm_scale, int window,
                                                   kvq_dtype_t cache_dtype, int num_splits, void* workspace,
                                                   size_t workspace_bytes, int* dev_status, kvq_stream_t stream) {
  clear_error();
  if (B < 1 || Hq < 1 || Hkv < 1 || max_blocks < 1 || num_blocks < 1 || num_splits < 0)
    return fail(KVQ_ERR_INVALID_ARG, "paged_decode: bad sizes");
  if (Hq % Hkv != 0) return fail(KVQ_ERR_INVALID_ARG, "paged_decode: Hq %% Hkv != 0");
  if (window == 0 || window < -1) return fail(KVQ_ERR_INVALID_ARG, "paged_decode: window must be -1 or > 0");
  if (!(sm_scale > 0.f) || !(sm_scale < FLT_MAX)) return fail(KVQ_ERR_INVALID_ARG, "paged_decode: bad sm_scale");
  if (P != kPage) return fail(KVQ_ERR_UNSUPPORTED, "paged_decode: page size %d (only 16)", P);
  if (D != 64 && D != 128) return fail(KVQ_ERR_UNSUPPORTED, "paged_decode: head_dim %d", D);
  if (Hq / Hkv > 8) return fail(KVQ_ERR_UNSUPPORTED, "paged_decode: GQA ratio %d > 8", Hq / Hkv);
  if (cache_dtype != KVQ_DTYPE_FP8_E4M3 && cache_dtype != KVQ_DTYPE_BF16)
    return fail(KVQ_ERR_INVALID_ARG, "paged_decode: bad cache dtype");
  if (!q || !k_cache || !v_cache || !block_table || !seq_lens || !out || !workspace)
    return fail(KVQ_ERR_INVALID_ARG, "paged_decode: null pointer");
  if (cache_dtype == KVQ_DTYPE_FP8_E4M3 && (!k_scale || !v_scale))
    return fail(KVQ_ERR_INVALID_ARG, "paged_decode: FP8 needs k_scale and v_scale");
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(workspace, 16) ||
      !aligned(out, 4))
    return fail(KVQ_ERR_INVALID_ARG, "paged_decode: misaligned pointer");
  int S, pps;
  split_plan(B, Hkv, P, max_blocks, window, num_splits, &S, &pps);
  const size_t need = kvq_decode_workspace_size(B, Hq, Hkv, D, P, max_blocks, window, num_splits);
  if (workspace_bytes < need)
    return fail(KVQ_ERR_INVALID_ARG, "paged_decode: workspace %zu bytes < %zu needed", workspace_bytes, need);
  const long items = static_cast<long>(B) * Hkv * S;
  if (items > 0x7FFFFFFFL || static_cast<long>(B) * Hq > 0x7FFFFFFFL)
    return fail(KVQ_ERR_UNSUPPORTED, "paged_decode: problem too large");

  DecodeParams prm;
  prm.q = q;
  prm.k_cache = static_cast<const uint8_t*>(k_cache);
  prm.v_cache = static_cast<const uint8_t*>(v_cache);
  prm.k_scale = k_scale;
  prm.v_scale = v_scale;
  prm.block_table = block_table;
  prm.seq_lens = seq_lens;
  prm.o_part = static_cast<float*>(workspace);
  prm.lse_part = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) +
                                          static_cast<size_t>(B) * Hq * S * D * sizeof(float));
  prm.B = B;
  prm.Hq = Hq;
  prm.Hkv = Hkv;
  prm.g = Hq / Hkv;
  prm.max_blocks = max_blocks;
  prm.num_blocks = num_blocks;
  prm.sm_scale = sm_scale;
  prm.window = window;
  prm.num_splits = S;
  prm.pages_per_split = pps;
  prm.num_items = static_cast<int>(items);
  prm.dev_status = dev_status;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  auto o = static_cast<__nv_bfloat16*>(out);
  const bool fp8 = cache_dtype == KVQ_DTYPE_FP8_E4M3;
  if (D == 128) return fp8 ? launch_decode<128, true>(prm, o, s) : launch_decode<128, false>(prm, o, s);
  return fp8 ? launch_decode<64, true>(prm, o, s) : launch_decode<64, false>(prm, o, s);
}
