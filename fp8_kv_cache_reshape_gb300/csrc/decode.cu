// kvq_paged_decode_attention: split-KV paged decode over the FP8 (or BF16)
// cache, plus the log-sum-exp combine.
//
// Method: "The state of FP8 KV-cache and attention quantization in vLLM"
//  - "Performance benchmarks": decode cost is the per-token KV read (the ITL
//    slope), so the kernel streams pages at HBM speed and reads FP8 directly;
//  - "Problems we found" / "Kernel and vLLM improvements", two-level
//    accumulation: the P.V contraction runs over the whole context; here each
//    pair of pages' MMA result lands in fresh FP32 registers and is then added
//    into a running FP32 sum, and page ranges are merged in FP32;
//  - "Skip layers": sliding-window layers read only the window's pages and
//    may keep a BF16 cache.
//
// Partial kernel (persistent): work item = (sequence, KV head, page range).
// Warp NW is the producer: it reads block ids and streams pages (one
// contiguous bulk copy per K page and per V page, two pages per stage) into a
// ring of NST shared-memory stages guarded by mbarriers.  Warps 0..NW-1
// consume stages round-robin; each ring slot belongs to one warp.  FP8
// cache: a consumer copies its whole stage into registers with ldmatrix and
// releases the slot at once; the FP8 codes are converted to f16 in registers
// (exact) and S^T = K Q^T (16 tokens x 8 query heads, M = tokens) runs on
// mma.m16n8k16 f16 with q as f16(q * 2^k); one online-softmax update (base 2)
// covers the stage's 32 tokens; P is rounded to f16 and transposed in
// registers (movmatrix), and O^T = V^T P^T (M = dims, K = the tokens of each
// page) goes into fresh FP32 fragments that are then added into the running
// output.  (On this GPU an E4M3 mma.sync costs about as many issue slots per
// instruction as an f16 one plus the operand conversion, and its latency is
// higher: the conversion done once per fragment here is cheaper.)  BF16
// cache: the same flow on bf16 MMAs.
// At the end of an item each consumer warp writes its own normalized partial
// output and log2-sum-exp per query head (no cross-warp merge).  Items are
// ordered so that consecutive CTAs serve different (sequence, KV head)
// pairs.  A combine kernel, launched as a programmatic dependent of the
// partial kernel, merges the S x NW partials of each query head in one pass.
#include <cfloat>
#include <cmath>
#include <mutex>

#include "kvq_device.cuh"
#include "kvq_host.h"

namespace kvq {

namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr int PPS = 2;  // pages per pipeline stage

struct DecodeParams {
  const void* q;
  const uint8_t* k_cache;
  const uint8_t* v_cache;
  const float* k_scale;
  const float* v_scale;
  const int32_t* block_table;
  const int32_t* seq_lens;
  float* o_part;    // [B][Hq][S][NW][D]
  float* lse_part;  // [B][Hq][S][NW], log2 units
  // direct: one page range per (sequence, KV head) and one item per CTA; the
  // CTA merges its consumer warps' partials in shared memory and writes the
  // bf16 output itself (no combine kernel)
  __nv_bfloat16* out;
  int direct;
  // bytes between consecutive (block, KV head) pages of the K and V caches;
  // paired: each pair's K page is followed by its V page (one copy moves both)
  int64_t k_str, v_str;
  int paired;
  int B, Hq, Hkv, g, max_blocks;
  int64_t num_blocks;
  float sm_scale;
  int window;
  int num_splits;
  int num_items;
  // balanced plan (ragged batches): per KV head, the batch's attended pages
  // laid end to end are cut into num_slots = B * S equal slots; a slot's part
  // inside one sequence is a segment, whose partials sit at segment id
  // slot + b of [Hq][kseg][NW] (kseg = num_slots + B - 1)
  int balanced;
  int num_slots;
  int kseg;
  int* dev_status;
  // Append (optional, k_new != nullptr): the new token of each sequence,
  // bf16 [B][Hkv][D], is written into its cache slot slot_new[b] (-1: none)
  // exactly as kvq_reshape_and_cache writes it, by the CTA that reads the
  // sequence's last page, before it reads it.
  const uint16_t* k_new;
  const uint16_t* v_new;
  const int64_t* slot_new;
  uint8_t* k_cache_w;
  uint8_t* v_cache_w;
  // failure-path test hook (kvq_debug_set_stall_ns): > 0 makes consumer warp
  // 0 wait up to this long on a barrier nothing arrives on before its first
  // stage, which fails like a stuck pipeline wait
  uint64_t stall_ns;
};

template <int D, bool FP8>
struct Geo {
  static constexpr int ESZ = FP8 ? 1 : 2;
  static constexpr int ROWB = D * ESZ;        // bytes of one K row
  static constexpr int PAGE = kPage * ROWB;   // bytes of one K page (= one V page)
  static constexpr int STAGE = 2 * PPS * PAGE;
  static constexpr int MT = D / 16;           // 16-row tiles of O^T
  static constexpr int KS = D / 16;           // 16-dim k-steps of QK
};

constexpr int kNW = 4;     // consumer warps per CTA
// Resident CTAs per SM: 3, and 4 at head dim 64, whose stages carry half the
// bytes for the same per-stage work (the softmax of 32 tokens), so more
// consumer warps per SM keep the pages streaming.
template <int D>
constexpr int ctas_per_sm() {
  return D == 64 ? 4 : 3;
}
inline int ctas_per_sm_of(int D) { return D == 64 ? ctas_per_sm<64>() : ctas_per_sm<128>(); }

// As many pages in flight per CTA as fit beside ctas_per_sm() CTAs on one SM
// (228 KiB of shared memory per SM, 1 KiB of it reserved per CTA, a few
// hundred bytes of barriers), in a multiple of kNW stages: the consumers
// take stages round-robin, so with NST % NW == 0 every ring slot is always
// consumed by the same warp, which waits on the slot's phases in order.  (If
// two warps shared a slot, a warp could test a slot whose previous fill has
// not landed yet, and a parity wait would then see the phase before it as
// complete.)
// Per-token scales (PT): a V page carries its scale tail (16 K scales, 16 V
// scales) and moves with it in one copy; a stage is [K0][K1][V0 tail0][V1 tail1].
template <int D, bool FP8, bool PT>
constexpr int stage_stride() {
  return Geo<D, FP8>::STAGE + (PT ? PPS * kScaleTailBytes : 0);
}
// bytes of one V page in the cache and in a stage
template <int D, bool FP8, bool PT>
constexpr int v_stride() {
  return Geo<D, FP8>::PAGE + (PT ? kScaleTailBytes : 0);
}

constexpr int kSmemPerSm = 228 * 1024;
template <int D>
constexpr int ring_budget() {
  return kSmemPerSm / ctas_per_sm<D>() - 1024 - 512;
}
// Dynamic shared memory that lets at most n CTAs reside on an SM (n + 1
// would overrun the SM's budget with the 1 KB each CTA reserves).
constexpr int spread_smem(int n) { return kSmemPerSm / (n + 1) - 1024 + 16; }
template <int D, bool FP8, bool PT = false>
constexpr int stages_for() {
  constexpr int fit = ring_budget<D>() / stage_stride<D, FP8, PT>();
  constexpr int n = fit > 32 ? 32 : fit;
  return (n / kNW) * kNW < kNW ? kNW : (n / kNW) * kNW;
}

template <int D, bool FP8, int NST, bool PT = false>
constexpr size_t decode_smem_bytes() {
  return size_t(NST) * stage_stride<D, FP8, PT>() + (2 * NST + 1) * sizeof(uint64_t) + NST * sizeof(int) + 16;
}
// ctas_per_sm() CTAs of every instantiation fit on one SM
static_assert(ctas_per_sm<128>() * (decode_smem_bytes<128, true, stages_for<128, true>()>() + 1024) <= kSmemPerSm, "smem");
static_assert(ctas_per_sm<64>() * (decode_smem_bytes<64, true, stages_for<64, true>()>() + 1024) <= kSmemPerSm, "smem");
static_assert(ctas_per_sm<128>() * (decode_smem_bytes<128, false, stages_for<128, false>()>() + 1024) <= kSmemPerSm, "smem");
static_assert(ctas_per_sm<64>() * (decode_smem_bytes<64, false, stages_for<64, false>()>() + 1024) <= kSmemPerSm, "smem");
static_assert(ctas_per_sm<128>() * (decode_smem_bytes<128, true, stages_for<128, true, true>(), true>() + 1024) <= kSmemPerSm,
              "smem");
static_assert(ctas_per_sm<64>() * (decode_smem_bytes<64, true, stages_for<64, true, true>(), true>() + 1024) <= kSmemPerSm,
              "smem");

struct ItemRange {
  int b, kvh, split;
  int lo, hi;     // attended token positions [lo, hi)
  int pg0, n;     // first page and page count of this split (balanced plan:
                  // of this segment of slot `split`)
};

// The pages [first, last) that a sequence of L cached tokens attends to, cut
// into S near-equal ranges of pps pages (so that shorter sequences still
// spread over all splits).
struct SplitPages {
  int first, last, pps;
};

KVQ_DEVINL SplitPages split_pages(int L, int window, int S) {
  SplitPages sp;
  const int lo = (window > 0 && L > window) ? L - window : 0;
  sp.first = lo / kPage;
  sp.last = (L + kPage - 1) / kPage;
  sp.pps = (sp.last - sp.first + S - 1) / S;
  return sp;
}

// seq_lens[b], clamped to what the block table holds (reported once)
KVQ_DEVINL int seq_len_of(const int32_t* seq_lens, int b, int max_blocks, int* dev_status, bool report) {
  int L = seq_lens[b];
  const int cap = max_blocks * kPage;
  if (L < 0 || L > cap) {
    if (report) set_status(dev_status, KVQ_DEV_BAD_SEQLEN);
    L = L < 0 ? 0 : cap;
  }
  return L;
}

KVQ_DEVINL ItemRange item_range(const DecodeParams& p, int item, bool report) {
  ItemRange r;
  const int S = p.num_splits;
  // consecutive items belong to different (sequence, KV head) pairs, so each
  // pair's ranges run on CTAs spread over the whole GPU
  const int NG = p.B * p.Hkv;
  const int bh = item % NG;
  r.split = item / NG;
  r.b = bh / p.Hkv;
  r.kvh = bh - r.b * p.Hkv;
  const int L = seq_len_of(p.seq_lens, r.b, p.max_blocks, p.dev_status, report);
  r.hi = L;
  r.lo = (p.window > 0 && L > p.window) ? L - p.window : 0;
  const SplitPages sp = split_pages(L, p.window, S);
  r.pg0 = sp.first + r.split * sp.pps;
  int pg1 = r.pg0 + sp.pps;
  if (pg1 > sp.last) pg1 = sp.last;
  r.n = pg1 > r.pg0 ? pg1 - r.pg0 : 0;
  return r;
}

// Balanced plan: lane b (< B <= 32) of a warp holds sequence b's length,
// first attended page, attended page count and the inclusive prefix of the
// page counts over the batch.  spec: a hint read before the preceding kernel
// has completed (L2-only loads, nothing reported).
struct BatchScan {
  int L, first, pages, incl, total;
};
KVQ_DEVINL BatchScan batch_scan_of(const int32_t* seq_lens, int B, int max_blocks, int window, int lane, bool spec,
                                    int* report_to) {
  BatchScan bs;
  int L = 0;
  if (lane < B) {
    L = spec ? ld_l2only_s32(seq_lens + lane) : seq_lens[lane];
    const int cap = max_blocks * kPage;
    if (L < 0 || L > cap) {
      if (report_to) set_status(report_to, KVQ_DEV_BAD_SEQLEN);
      L = L < 0 ? 0 : cap;
    }
  }
  const SplitPages sp = split_pages(L, window, 1);
  bs.L = L;
  bs.first = sp.first;
  bs.pages = lane < B ? sp.last - sp.first : 0;
  int x = bs.pages;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  bs.incl = x;
  bs.total = __shfl_sync(0xffffffffu, x, 31);
  return bs;
}
KVQ_DEVINL BatchScan batch_scan(const DecodeParams& p, int lane, bool spec, bool report) {
  return batch_scan_of(p.seq_lens, p.B, p.max_blocks, p.window, lane, spec, report ? p.dev_status : nullptr);
}
// Slots that hold pages: all num_slots, or one per page when the batch has
// fewer pages (every used slot then holds at least one page, so the segment
// ids of a sequence's slots are all written).
KVQ_DEVINL int used_slots(int num_slots, int total) { return total < num_slots ? total : num_slots; }
// The slot holding stream page x (0 <= x < T, N = used slots): the largest s
// with floor(s * T / N) <= x.
KVQ_DEVINL int slot_of(int64_t x, int64_t T, int64_t N) { return static_cast<int>(((x + 1) * N + T - 1) / T) - 1; }

// The segments of one item, in stream order: one ItemRange per item in the
// per-sequence plan; in the balanced plan the parts of the item's slot inside
// each sequence it covers (none for an empty slot).  Warp-uniform.  The
// batch scan is taken again at each step rather than kept (registers).
struct SegCursor {
  int item;
  int pos, end;  // balanced: the slot's remaining stream pages [pos, end)
  int b;         // balanced: the next sequence to look at; per-sequence: 1 once returned
};
template <bool BAL>
KVQ_DEVINL SegCursor seg_begin(const DecodeParams& p, int item, int lane, bool spec) {
  SegCursor c;
  c.item = item;
  c.pos = c.end = c.b = 0;
  if constexpr (BAL) {
    const BatchScan bs = batch_scan(p, lane, spec, false);
    const int64_t T = bs.total;
    const int64_t N = used_slots(p.num_slots, bs.total);
    const int slot = item / p.Hkv;
    if (slot < N) {
      c.pos = static_cast<int>(slot * T / N);
      c.end = static_cast<int>((slot + 1) * T / N);
    }
    // first sequence whose pages reach past pos
    c.b = __popc(__ballot_sync(0xffffffffu, lane < p.B && bs.incl <= c.pos));
  }
  return c;
}
template <bool BAL>
KVQ_DEVINL bool seg_next(const DecodeParams& p, SegCursor& c, ItemRange& r, int lane, bool spec, bool report) {
  if constexpr (!BAL) {
    if (c.b) return false;
    r = item_range(p, c.item, report);
    c.b = 1;
    return true;
  }
  if (c.pos >= c.end) return false;
  const BatchScan bs = batch_scan(p, lane, spec, report);
  while (c.pos < c.end && c.b < p.B) {
    const int incl = __shfl_sync(0xffffffffu, bs.incl, c.b);
    const int pages = __shfl_sync(0xffffffffu, bs.pages, c.b);
    if (incl <= c.pos) {  // sequence b ends before pos (or is empty)
      ++c.b;
      continue;
    }
    const int start = incl - pages;  // sequence b's first stream page
    const int stop = min(c.end, incl);
    const int L = __shfl_sync(0xffffffffu, bs.L, c.b);
    const int kvh = c.item % p.Hkv, slot = c.item / p.Hkv;
    r.b = c.b;
    r.kvh = kvh;
    r.split = slot;
    r.hi = L;
    r.lo = (p.window > 0 && L > p.window) ? L - p.window : 0;
    r.pg0 = __shfl_sync(0xffffffffu, bs.first, c.b) + (c.pos - start);
    r.n = stop - c.pos;
    c.pos = stop;
    if (stop == incl) ++c.b;
    return true;
  }
  return false;
}

// Every segment of this CTA's items (item = blockIdx.x, + gridDim.x, ...).
template <bool BAL>
struct SegWalk {
  SegCursor c;
  KVQ_DEVINL SegWalk(const DecodeParams& p, int lane) {
    c.item = blockIdx.x;
    c.pos = c.end = c.b = 0;
    if (c.item < p.num_items) c = seg_begin<BAL>(p, c.item, lane, false);
  }
  KVQ_DEVINL bool next(const DecodeParams& p, int lane, ItemRange& r, bool report) {
    while (c.item < p.num_items) {
      if (seg_next<BAL>(p, c, r, lane, false, report)) return true;
      const int item = c.item + gridDim.x;
      c.item = item;
      if (item < p.num_items) c = seg_begin<BAL>(p, item, lane, false);
    }
    return false;
  }
};
// The per-sequence plan: one segment per item.
template <>
struct SegWalk<false> {
  int item;
  bool started;
  KVQ_DEVINL SegWalk(const DecodeParams&, int) : item(blockIdx.x), started(false) {}
  KVQ_DEVINL bool next(const DecodeParams& p, int, ItemRange& r, bool report) {
    if (started) item += gridDim.x;
    started = true;
    if (item >= p.num_items) return false;
    r = item_range(p, item, report);
    return true;
  }
};

// Before the preceding kernel has completed: bring the first pages of this
// CTA's first item into L2, so that its first stages arrive at L2 rather
// than HBM latency once it may start.  The sequence length and block ids are
// read only for this hint (they may still change and are read again after
// the wait; loads cached in L2 only leave no stale L1 line), clamped so that
// every address stays inside the block table and the caches.  A page the
// preceding kernel writes after the hint is updated in L2 like any other.
template <int D, bool FP8, bool PT, bool BAL>
KVQ_DEVINL void prefetch_first_pages(const DecodeParams& p, int lane, int max_pages) {
  using G = Geo<D, FP8>;
  constexpr int VS = v_stride<D, FP8, PT>();
  int b, kvh, pg0, n;
  if constexpr (BAL) {
    SegCursor cur = seg_begin<true>(p, blockIdx.x, lane, true);
    ItemRange r;
    if (!seg_next<true>(p, cur, r, lane, true, false)) return;
    b = r.b;
    kvh = r.kvh;
    pg0 = r.pg0;
    n = r.n;
  } else {
    const int NG = p.B * p.Hkv;
    const int item = blockIdx.x;
    const int bh = item % NG;
    b = bh / p.Hkv;
    kvh = bh - b * p.Hkv;
    int L = ld_l2only_s32(p.seq_lens + b);
    L = min(max(L, 0), p.max_blocks * kPage);
    const SplitPages sp = split_pages(L, p.window, p.num_splits);
    pg0 = sp.first + (item / NG) * sp.pps;
    n = min(sp.pps, sp.last - pg0);
  }
  n = min(n, max_pages);
  if (lane >= n) return;
  const int blk = ld_l2only_s32(p.block_table + static_cast<size_t>(b) * p.max_blocks + pg0 + lane);
  if (blk < 0 || static_cast<int64_t>(blk) >= p.num_blocks) return;
  const size_t pair = static_cast<size_t>(blk) * p.Hkv + kvh;
  if (p.paired) {
    prefetch_l2(p.k_cache + pair * p.k_str, G::PAGE + VS);
  } else {
    prefetch_l2(p.k_cache + pair * p.k_str, G::PAGE);
    prefetch_l2(p.v_cache + pair * p.v_str, VS);
  }
}

// Stage info word written by the producer: bit 0/1 = page 0/1 present,
// bit 2/3 = page 0/1 had an invalid block id (fully masked).
constexpr int kPresent0 = 1, kPresent1 = 2, kBad0 = 4, kBad1 = 8;

// E5: the FP8 cache holds E5M2 codes (the MMAs take them as their A operand).
// PT: per-token scales, in the scale tail of each V page (FP8 only;
// p.k_scale and p.v_scale are unused).
// SL: single-level accumulation (an ablation of the two-level scheme): the
// P.V MMAs accumulate into the running sum O * alpha directly instead of a
// fresh FP32 tile per stage (FP8, per-head scales only).
// AP: the append entry point's instantiation (the new token's cache write);
// the plain decode is compiled without it.
template <int D, bool FP8, int NW, int NST, bool E5, bool PT, bool SL, bool AP = false, bool BAL = false>
__global__ void __launch_bounds__((NW + 1) * 32, ctas_per_sm<D>()) decode_partial_kernel(const __grid_constant__ DecodeParams p) {
  using G = Geo<D, FP8>;
  static_assert(NST % NW == 0 && NST >= NW, "each ring slot must belong to one consumer warp");
  static_assert(FP8 || !PT, "per-token scales apply to FP8 caches");
  static_assert(!SL || (FP8 && !PT), "the single-level ablation covers the per-head FP8 path");
  static_assert(!BAL || (D == 128 && FP8 && !E5 && !PT && !SL), "the balanced plan covers the E4M3 per-head path");
  constexpr int STRIDE = stage_stride<D, FP8, PT>();
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* stages = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + size_t(NST) * STRIDE);
  uint64_t* empty = full + NST;
  uint64_t* stall_bar = empty + NST;  // nothing arrives on it (test hook)
  int* stage_info = reinterpret_cast<int*>(stall_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(stage_info + NST);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < NST; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    mbar_init(stall_bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  // launched as a programmatic dependent: the setup above overlaps the
  // preceding kernel, and nothing in global memory is touched before it has
  // completed.  The combine kernel may launch once every CTA is past that
  // point, so it too sees the preceding kernel's writes.  Without a combine
  // (direct output) the next kernel launches as the CTAs exit: its CTAs
  // waiting beside this grid's slowest ones would slow them.
  // the last consumer warp issues the hint: its first stage comes last, and
  // the producer's own chain is not lengthened where nothing runs before.
  // Direct-output calls (one short range per pair) gain nothing from it.
  if (warp == NW - 1 && !p.direct && blockIdx.x < p.num_items) {
    prefetch_first_pages<D, FP8, PT, BAL>(p, lane, PPS * NW);
  }
  grid_dependency_wait();
  if (!p.direct) grid_launch_dependents();

  if (warp == NW) {
    // ------------------------------------------------------------ producer --
    const uint64_t pol = policy_evict_first();
    uint32_t it = 0;  // stage counter
    bool aborted = false;
    SegWalk<BAL> walk(p, lane);
    // faults in the lengths: reported by lane 0 per item, or (balanced) by the
    // lane of each sequence in CTA 0
    const bool report = BAL ? blockIdx.x == 0 : lane == 0;
    for (ItemRange r; !aborted && walk.next(p, lane, r, report);) {
      const int32_t* bt = p.block_table + static_cast<size_t>(r.b) * p.max_blocks + r.pg0;
      // append: this item holds the page of the sequence's last token
      const int last_pg = (r.hi - 1) / kPage;
      const bool append = AP && r.hi > 0 && last_pg >= r.pg0 && last_pg < r.pg0 + r.n;
      constexpr int EPL = D / 32;  // elements of the new K (and V) row per lane
      uint16_t kx[EPL], vx[EPL];
      int64_t slot = -1;
      if (AP && append) {  // loads in flight while the item's first pages are issued
        slot = p.slot_new[r.b];
        const size_t src = (static_cast<size_t>(r.b) * p.Hkv + r.kvh) * D + lane * EPL;
#pragma unroll
        for (int e = 0; e < EPL; ++e) {
          kx[e] = p.k_new[src + e];
          vx[e] = p.v_new[src + e];
        }
      }
      // the whole warp; then the page may be copied.  blk_last: the block id
      // the table gives for the page of the sequence's last token
      auto write_new_token = [&](int blk_last) {
        if (slot < 0) return;
        const int64_t num_slots = p.num_blocks * kPage;
        // the slot must be the last token's slot under the block table (the
        // page this CTA reads back); any other slot is not written
        if (slot >= num_slots || slot / kPage != blk_last || static_cast<int>(slot % kPage) != (r.hi - 1) % kPage) {
          if (lane == 0) set_status(p.dev_status, KVQ_DEV_BAD_SLOT);
          return;
        }
        const int off = static_cast<int>(slot % kPage);
        const size_t pair = static_cast<size_t>(slot / kPage) * p.Hkv + r.kvh;
        uint8_t* kp = p.k_cache_w + pair * p.k_str;
        uint8_t* vp = p.v_cache_w + pair * p.v_str;
        const int d0 = lane * EPL;
        if constexpr (FP8) {
          const float sk = p.k_scale[r.kvh], sv = p.v_scale[r.kvh];
          uint32_t kw = 0;
#pragma unroll
          for (int e = 0; e < EPL; ++e) {
            const float xk = __uint_as_float(static_cast<uint32_t>(kx[e]) << 16);
            const float xv = __uint_as_float(static_cast<uint32_t>(vx[e]) << 16);
            kw |= f32_to_fp8<E5>(__fdiv_rn(xk, sk)) << (8 * e);
            vp[(d0 + e) * kPage + fp8_v_slot(off)] = static_cast<uint8_t>(f32_to_fp8<E5>(__fdiv_rn(xv, sv)));
          }
          // dims d0 .. d0 + EPL - 1 sit in one 16-byte chunk of the swizzled K row
          uint8_t* kd = kp + fp8_k_offset(off, d0 / 16, D) + d0 % 16;
          if constexpr (EPL == 4) {
            *reinterpret_cast<uint32_t*>(kd) = kw;
          } else {
            *reinterpret_cast<uint16_t*>(kd) = static_cast<uint16_t>(kw);
          }
        } else {
          // BF16: a bit copy; dims d0 .. d0 + EPL - 1 sit in one 16-byte chunk of the K row
          uint16_t* kd = reinterpret_cast<uint16_t*>(kp + k_chunk_offset(off, d0 / 8, G::ROWB) + (d0 % 8) * 2);
#pragma unroll
          for (int e = 0; e < EPL; ++e) {
            kd[e] = kx[e];
            *reinterpret_cast<uint16_t*>(vp + bf16_v_offset(d0 + e, off)) = vx[e];
          }
        }
        fence_proxy_async_global();  // the stores, before the bulk copy of the page reads them
      };
      // block ids: one coalesced load per 32 pages, issued a batch ahead so
      // that its latency hides behind the copies of the current batch
      auto load_ids = [&](int base) { return (base + lane < r.n) ? __ldg(bt + base + lane) : 0; };
      int blk_next = load_ids(0);
      for (int base = 0; base < r.n && !aborted; base += 32) {
        const int cnt = min(32, r.n - base);
        int blk = blk_next, bad = 0;
        if (base + 32 < r.n) blk_next = load_ids(base + 32);
        if (lane < cnt && (blk < 0 || static_cast<int64_t>(blk) >= p.num_blocks)) {
          bad = 1;
          blk = 0;
          set_status(p.dev_status, KVQ_DEV_BAD_BLOCK);
        }
        for (int j = 0; j < cnt; j += PPS, ++it) {
          const int b0 = __shfl_sync(0xffffffffu, blk, j);
          const int d0 = __shfl_sync(0xffffffffu, bad, j);
          const int b1 = __shfl_sync(0xffffffffu, blk, (j + 1) & 31);
          const int d1 = __shfl_sync(0xffffffffu, bad, (j + 1) & 31);
          const bool two = j + 1 < cnt;
          if constexpr (AP) {
            const int pg = r.pg0 + base + j;
            if (append && (pg == last_pg || (two && pg + 1 == last_pg))) {
              write_new_token(pg == last_pg ? (d0 ? -1 : b0) : (d1 ? -1 : b1));
              __syncwarp();
            }
          }
          // one stage = pages j, j + 1 laid out [K0][V0][K1][V1] (per-token
          // scales: each V page with its scale tail): a bulk copy per K page
          // and per V page, or over a paired cache one per page pair
          auto issue_pages = [&](int st) {
            constexpr int VS = v_stride<D, FP8, PT>();
            int info = kPresent0 | (d0 ? kBad0 : 0);
            if (two) info |= kPresent1 | (d1 ? kBad1 : 0);
            stage_info[st] = info;
            mbar_arrive_expect_tx(&full[st], (two ? 2u : 1u) * static_cast<uint32_t>(G::PAGE + VS));
            uint8_t* sk = stages + size_t(st) * STRIDE;
            const size_t pg0 = static_cast<size_t>(b0) * p.Hkv + r.kvh;
            const size_t pg1 = static_cast<size_t>(b1) * p.Hkv + r.kvh;
            if (p.paired) {
              bulk_g2s(sk, p.k_cache + pg0 * p.k_str, G::PAGE + VS, &full[st], pol);
              if (two) bulk_g2s(sk + G::PAGE + VS, p.k_cache + pg1 * p.k_str, G::PAGE + VS, &full[st], pol);
            } else {
              bulk_g2s(sk, p.k_cache + pg0 * p.k_str, G::PAGE, &full[st], pol);
              bulk_g2s(sk + G::PAGE, p.v_cache + pg0 * p.v_str, VS, &full[st], pol);
              if (two) {
                bulk_g2s(sk + G::PAGE + VS, p.k_cache + pg1 * p.k_str, G::PAGE, &full[st], pol);
                bulk_g2s(sk + 2 * G::PAGE + VS, p.v_cache + pg1 * p.v_str, VS, &full[st], pol);
              }
            }
          };
          int ok = 1;
          if (lane == 0) {
            const int st = it % NST;
            if (*abort_flag || !mbar_wait(&empty[st], ((it / NST) & 1) ^ 1, abort_flag)) {
              ok = 0;
            } else {
              issue_pages(st);
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
  // per-lane ldmatrix byte offsets inside a K page and a V page
  int koff[FP8 ? G::KS / 2 : G::KS];
  {
    const int tok = (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
    for (int i = 0; i < (FP8 ? G::KS / 2 : G::KS); ++i) koff[i] = k_chunk_offset(tok, 2 * i + (lane >> 4), G::ROWB);
  }
  // V offsets.  FP8: matrix 0/1 = page 0 rows (16 mt + 0..7 / 8..15), matrix
  // 2/3 = the same rows of page 1.  BF16: one m-tile of one page per x4.
  // stage layout [K0][V0][K1][V1]: K1 at k1off, V0 at v0off, V1 at v0off + v1d
  constexpr int VSZ = v_stride<D, FP8, PT>();
  constexpr int k1off = G::PAGE + VSZ;
  constexpr int v0off = G::PAGE;
  constexpr int v1d = G::PAGE + VSZ;
  const int vofs = (lane >> 4) * v1d + (lane & 15) * kPage;  // FP8: + 256 per m-tile
  int voff[FP8 ? 1 : G::MT];
  if constexpr (FP8) {
    voff[0] = vofs;
  } else {
#pragma unroll
    for (int i = 0; i < G::MT; ++i) {
      const int row = 16 * i + (lane & 7) + ((lane >> 3) & 1) * 8;
      voff[i] = row * 32 + 16 * ((lane >> 4) ^ ((row >> 2) & 1));
    }
  }

  if (warp == 0 && !stall_wait(stall_bar, p.stall_ns, abort_flag)) {
    if (lane == 0) {
      set_status(p.dev_status, KVQ_DEV_TIMEOUT);
      *abort_flag = 1;
    }
  }
  uint32_t it0 = 0;
  SegWalk<BAL> walk(p, lane);
  for (ItemRange rg; walk.next(p, lane, rg, false);) {
    // ---- query fragments of head (kvh * g + r); heads >= g are zero padding ----
    // FP8 cache: f16(q * sigma), sigma = 2^(7 - floor(log2 max|q|)) per head (a
    // bf16 value times a power of two: exact unless it falls below f16's
    // normal range), for the f16 MMAs; word 2w holds dims d, d + 1 and word
    // 2w + 1 dims d + 2, d + 3 for d = 32 (w / 2) + 16 (w % 2) + 4c.  BF16: q
    // as stored.
    constexpr int QW = D / 8;  // 32-bit words of q per lane
    uint32_t qh[QW];
    float coef0, coef1;  // score coefficient of heads 2c and 2c + 1
    {
      const bool live = r < p.g;
      const uint16_t* qrow = static_cast<const uint16_t*>(p.q) +
                             (static_cast<size_t>(rg.b) * p.Hq + rg.kvh * p.g + (live ? r : 0)) * D;
      if constexpr (FP8) {
        constexpr int NL = D / 16;  // loads of four dims per lane
        float x[NL][4];
        float mx = 0.f;
#pragma unroll
        for (int w = 0; w < NL; ++w) {
          const int dim = (w >> 1) * 32 + (w & 1) * 16 + 4 * c;
          const uint2 u = live ? __ldg(reinterpret_cast<const uint2*>(qrow + dim)) : make_uint2(0, 0);
          x[w][0] = __uint_as_float(u.x << 16);
          x[w][1] = __uint_as_float(u.x & 0xFFFF0000u);
          x[w][2] = __uint_as_float(u.y << 16);
          x[w][3] = __uint_as_float(u.y & 0xFFFF0000u);
#pragma unroll
          for (int e = 0; e < 4; ++e) mx = fmaxf(mx, fabsf(x[w][e]));
        }
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        int e2 = mx > 0.f ? static_cast<int>((__float_as_uint(mx) >> 23) & 0xFF) - 127 : 0;
        e2 = e2 < -100 ? -100 : e2;
        const float sigma = __uint_as_float(static_cast<uint32_t>(127 + 7 - e2) << 23);   // 2^(7 - e2)
        const float inv_sigma = __uint_as_float(static_cast<uint32_t>(127 - 7 + e2) << 23);
#pragma unroll
        for (int w = 0; w < NL; ++w) {
          qh[2 * w] = pack_f16x2(x[w][0] * sigma, x[w][1] * sigma);
          qh[2 * w + 1] = pack_f16x2(x[w][2] * sigma, x[w][3] * sigma);
        }
        // per-head K scale folded in here; per-token K scales multiply each score later
        const float cf = PT ? __fmul_rn(p.sm_scale, kLog2e) : __fmul_rn(__fmul_rn(p.k_scale[rg.kvh], p.sm_scale), kLog2e);
        // 1/sigma of heads 2c and 2c + 1 lives in lanes 8c and 8c + 4
        coef0 = cf * __shfl_sync(0xffffffffu, inv_sigma, 8 * c);
        coef1 = cf * __shfl_sync(0xffffffffu, inv_sigma, 8 * c + 4);
      } else {
#pragma unroll
        for (int kk = 0; kk < G::KS; ++kk) {
          qh[2 * kk] = live ? __ldg(reinterpret_cast<const uint32_t*>(qrow + kk * 16 + 2 * c)) : 0u;
          qh[2 * kk + 1] = live ? __ldg(reinterpret_cast<const uint32_t*>(qrow + kk * 16 + 8 + 2 * c)) : 0u;
        }
        coef0 = coef1 = __fmul_rn(p.sm_scale, kLog2e);
      }
    }

    float m[2] = {NEG_INF, NEG_INF};
    float l[2] = {0.f, 0.f};
    float O[G::MT][4];
#pragma unroll
    for (int i = 0; i < G::MT; ++i) O[i][0] = O[i][1] = O[i][2] = O[i][3] = 0.f;

    const int nst_item = (rg.n + PPS - 1) / PPS;  // stages of this item
    int i = (warp - static_cast<int>(it0 % NW) + NW) % NW;
    if (*abort_flag) i = nst_item;  // abandoned: skip the pages, keep the barriers in step
    for (; i < nst_item; i += NW) {
      const uint32_t itg = it0 + i;
      const int st = itg % NST;
      if (!mbar_wait(&full[st], (itg / NST) & 1, abort_flag)) {
        if (lane == 0) {
          set_status(p.dev_status, KVQ_DEV_TIMEOUT);
          *abort_flag = 1;
        }
        break;
      }
      const uint32_t kb = smem_u32(stages + size_t(st) * STRIDE);
      const uint32_t vb = kb + v0off;
      const int info = stage_info[st];
      const bool two = (info & kPresent1) != 0;
      const int tok0 = (rg.pg0 + i * PPS) * kPage;  // first token of page 0
      const int tok_end = tok0 + (two ? 2 : 1) * kPage;
      const bool edge = (info & (kBad0 | kBad1)) || tok0 < rg.lo || tok_end > rg.hi;
      // token liveness (edge stages): inside [lo, hi), present, valid block id
      auto live = [&](int pg, int t) {
        const int tok = tok0 + pg * kPage + t;
        const bool badp = pg == 0 ? (info & kBad0) : (info & kBad1);
        const bool present = pg == 0 || two;
        return present && !badp && tok >= rg.lo && tok < rg.hi;
      };

      float s0[4], s1[4];
      float p00, p01, p02, p03, p10, p11, p12, p13, al0, al1;
      // online softmax over the stage's 32 tokens (base 2)
      auto softmax = [&]() {
        float mx0 = fmaxf(fmaxf(s0[0], s0[2]), fmaxf(s1[0], s1[2]));
        float mx1 = fmaxf(fmaxf(s0[1], s0[3]), fmaxf(s1[1], s1[3]));
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
          mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
          mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
        }
        const float mn0 = fmaxf(m[0], mx0), mn1 = fmaxf(m[1], mx1);
        // probabilities come out scaled by 2^8 (exact): P fills the E4M3 range
        // and the running maximum itself is exactly 256
        const float base0 = ((mn0 == NEG_INF) ? 0.f : mn0) - 8.f;
        const float base1 = ((mn1 == NEG_INF) ? 0.f : mn1) - 8.f;
        al0 = ex2(m[0] - base0 - 8.f);  // rescale of the running sums
        al1 = ex2(m[1] - base1 - 8.f);
        m[0] = mn0;
        m[1] = mn1;
        p00 = ex2(s0[0] - base0); p01 = ex2(s0[1] - base1); p02 = ex2(s0[2] - base0); p03 = ex2(s0[3] - base1);
        p10 = ex2(s1[0] - base0); p11 = ex2(s1[1] - base1); p12 = ex2(s1[2] - base0); p13 = ex2(s1[3] - base1);
        l[0] = l[0] * al0 + ((p00 + p02) + (p10 + p12));
        l[1] = l[1] * al1 + ((p01 + p03) + (p11 + p13));
      };

      if constexpr (FP8) {
        // per-token scales (PT) of this lane's tokens r and r + 8 of both pages
        float sk00 = 1.f, sk01 = 1.f, sk10 = 1.f, sk11 = 1.f, sv00 = 0.f, sv01 = 0.f, sv10 = 0.f, sv11 = 0.f;
        if constexpr (PT) {  // the scale tails after each V page: 16 K scales, then 16 V scales
          const uint8_t* v0 = stages + size_t(st) * STRIDE + v0off;
          const float* t0 = reinterpret_cast<const float*>(v0 + G::PAGE);
          const float* t1 = reinterpret_cast<const float*>(v0 + v1d + G::PAGE);
          sk00 = t0[r];
          sk01 = t0[r + 8];
          sv00 = t0[kPage + r];
          sv01 = t0[kPage + r + 8];
          sk10 = t1[r];
          sk11 = t1[r + 8];
          sv10 = t1[kPage + r];
          sv11 = t1[kPage + r + 8];
        }
        // ---- S^T = K Q^T on f16 MMAs: the K codes converted in registers (exact).
        // An ldmatrix of 32 dims holds, per lane, dims 4c..4c+3 (x0: row r, x1:
        // row r + 8) and 16 + 4c..16 + 4c + 3 (x2, x3) of the chunk; each half
        // is one m16n8k16 with its k order permuted (k 2c, 2c + 1 <- dims 4c,
        // 4c + 1; k 2c + 8, 2c + 9 <- dims 4c + 2, 4c + 3), q permuted alike.
        // Two independent accumulation chains, one per half ----
        auto qk = [&](uint32_t kp, float (&s)[4], float ska, float skb) {  // ska, skb: tokens r, r + 8
          float a[4] = {0.f, 0.f, 0.f, 0.f}, b[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int kk = 0; kk < D / 32; ++kk) {
            uint32_t x0, x1, x2, x3;
            ldsm_x4(kp + koff[kk], x0, x1, x2, x3);
            uint32_t l0, h0, l1, h1, l2, h2, l3, h3;
            fp8x4_to_f16x2x2<E5>(x0, l0, h0);
            fp8x4_to_f16x2x2<E5>(x1, l1, h1);
            fp8x4_to_f16x2x2<E5>(x2, l2, h2);
            fp8x4_to_f16x2x2<E5>(x3, l3, h3);
            mma_f16(a, l0, l1, h0, h1, qh[4 * kk], qh[4 * kk + 1], a);
            mma_f16(b, l2, l3, h2, h3, qh[4 * kk + 2], qh[4 * kk + 3], b);
          }
          s[0] = (a[0] + b[0]) * coef0;
          s[1] = (a[1] + b[1]) * coef1;
          s[2] = (a[2] + b[2]) * coef0;
          s[3] = (a[3] + b[3]) * coef1;
          if constexpr (PT) {
            s[0] *= ska;
            s[1] *= ska;
            s[2] *= skb;
            s[3] *= skb;
          }
        };
        qk(kb, s0, sk00, sk01);
        if (two) qk(kb + k1off, s1, sk10, sk11);
        else s1[0] = s1[1] = s1[2] = s1[3] = NEG_INF;
        // ---- V fragments to registers, then release the ring slot ----
        uint32_t va[G::MT][4];
#pragma unroll
        for (int mt = 0; mt < G::MT; ++mt) ldsm_x4(vb + vofs + mt * 256, va[mt][0], va[mt][1], va[mt][2], va[mt][3]);
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);
        // masks (edge stages only): scores of dead tokens -> -inf, their V codes -> 0
        if (edge) {
          if (!live(0, r)) s0[0] = s0[1] = NEG_INF;
          if (!live(0, r + 8)) s0[2] = s0[3] = NEG_INF;
          if (!live(1, r)) s1[0] = s1[1] = NEG_INF;
          if (!live(1, r + 8)) s1[2] = s1[3] = NEG_INF;
          // lane word c of a V row holds tokens 2c, 2c+1, 2c+8, 2c+9
          auto vmask = [&](int pg) {
            return (live(pg, 2 * c) ? 0x000000FFu : 0u) | (live(pg, 2 * c + 1) ? 0x0000FF00u : 0u) |
                   (live(pg, 2 * c + 8) ? 0x00FF0000u : 0u) | (live(pg, 2 * c + 9) ? 0xFF000000u : 0u);
          };
          const uint32_t m0 = vmask(0), m1 = vmask(1);
#pragma unroll
          for (int mt = 0; mt < G::MT; ++mt) {
            va[mt][0] &= m0;
            va[mt][1] &= m0;
            va[mt][2] &= m1;
            va[mt][3] &= m1;
          }
        } else if (!two) {
#pragma unroll
          for (int mt = 0; mt < G::MT; ++mt) va[mt][2] = va[mt][3] = 0u;
        }
        // PT: V scales enter P as weights sv / c with c = 2^ceil(log2 m), m the
        // stage's largest live V scale (so P stays in E4M3's range and 1 / c is
        // exact); the stage's P.V is scaled by c
        float cst = 1.f, w00 = 1.f, w01 = 1.f, w10 = 1.f, w11 = 1.f;
        if constexpr (PT) {
          if (!two) sv10 = sv11 = 0.f;
          if (edge) {
            if (!live(0, r)) sv00 = 0.f;
            if (!live(0, r + 8)) sv01 = 0.f;
            if (!live(1, r)) sv10 = 0.f;
            if (!live(1, r + 8)) sv11 = 0.f;
          }
          float mv = fmaxf(fmaxf(sv00, sv01), fmaxf(sv10, sv11));
#pragma unroll
          for (int o = 4; o < 32; o <<= 1) mv = fmaxf(mv, __shfl_xor_sync(0xffffffffu, mv, o));
          // exponent of 2^ceil(log2 mv), within the normal range
          const uint32_t mb = __float_as_uint(mv);
          int ec = static_cast<int>(mb >> 23) - 127 + ((mb & 0x7FFFFFu) != 0u ? 1 : 0);
          ec = ec < -126 ? -126 : (ec > 126 ? 126 : ec);
          cst = mv > 0.f ? __uint_as_float(static_cast<uint32_t>(127 + ec) << 23) : 0.f;
          const float rc = mv > 0.f ? __uint_as_float(static_cast<uint32_t>(127 - ec) << 23) : 0.f;
          w00 = sv00 * rc;
          w01 = sv01 * rc;
          w10 = sv10 * rc;
          w11 = sv11 * rc;
        }
        softmax();
        float g0 = 1.f, g1 = 1.f;  // PT: factor of the stage's P.V of heads 2c, 2c + 1
        if constexpr (PT) {  // l above summed the unweighted p
          p00 *= w00; p01 *= w00; p02 *= w01; p03 *= w01;
          p10 *= w10; p11 *= w10; p12 *= w11; p13 *= w11;
          // Weights below 1 push probabilities toward f16's lower end, where they
          // lose bits.  Per head, a power of two f moves the stage's
          // largest weighted probability into [128, 256); P.V is then scaled by c / f.
          float pm0 = fmaxf(fmaxf(p00, p02), fmaxf(p10, p12));
          float pm1 = fmaxf(fmaxf(p01, p03), fmaxf(p11, p13));
#pragma unroll
          for (int o = 4; o < 32; o <<= 1) {
            pm0 = fmaxf(pm0, __shfl_xor_sync(0xffffffffu, pm0, o));
            pm1 = fmaxf(pm1, __shfl_xor_sync(0xffffffffu, pm1, o));
          }
          auto pow2_exp = [](float x) {  // e with 2^e <= x < 2^(e+1), clamped to [-119, 127]
            const int e = x > 0.f ? static_cast<int>((__float_as_uint(x) >> 23) & 0xFF) - 127 : 7;
            return e < -119 ? -119 : e;
          };
          const int e0 = pow2_exp(pm0), e1 = pow2_exp(pm1);
          const float f0 = __uint_as_float(static_cast<uint32_t>(127 + 7 - e0) << 23);  // 2^(7 - e0)
          const float f1 = __uint_as_float(static_cast<uint32_t>(127 + 7 - e1) << 23);
          g0 = cst * __uint_as_float(static_cast<uint32_t>(127 - 7 + e0) << 23);  // c / f0, exact
          g1 = cst * __uint_as_float(static_cast<uint32_t>(127 - 7 + e1) << 23);
          p00 *= f0; p01 *= f1; p02 *= f0; p03 *= f1;
          p10 *= f0; p11 *= f1; p12 *= f0; p13 *= f1;
        }
        // ---- P^T fragments: f16 pairs transposed, tokens 2c, 2c + 1 (pa0) and
        // 2c + 8, 2c + 9 (pa1) of head r: the B operand of the f16 P.V MMAs ----
        const uint32_t pa0 = movmatrix_t(pack_f16x2(p00, p01)), pa1 = movmatrix_t(pack_f16x2(p02, p03));  // page 0
        const uint32_t pb0 = movmatrix_t(pack_f16x2(p10, p11)), pb1 = movmatrix_t(pack_f16x2(p12, p13));  // page 1
        // ---- O^T += V^T P^T: per m-tile one m16n8k16 per page on the V codes
        // converted in registers (a lane's word holds tokens 2c, 2c + 1, 2c + 8,
        // 2c + 9 of its dimension: the A operand's k order), fresh FP32 per stage ----
#pragma unroll
        for (int mt = 0; mt < G::MT; ++mt) {
          uint32_t v0l, v0h, v1l, v1h, v2l, v2h, v3l, v3h;
          fp8x4_to_f16x2x2<E5>(va[mt][0], v0l, v0h);
          fp8x4_to_f16x2x2<E5>(va[mt][1], v1l, v1h);
          fp8x4_to_f16x2x2<E5>(va[mt][2], v2l, v2h);
          fp8x4_to_f16x2x2<E5>(va[mt][3], v3l, v3h);
          if constexpr (SL) {  // the MMAs add this stage into O * alpha themselves
            float c4[4] = {O[mt][0] * al0, O[mt][1] * al1, O[mt][2] * al0, O[mt][3] * al1};
            mma_f16(c4, v0l, v1l, v0h, v1h, pa0, pa1, c4);
            mma_f16(O[mt], v2l, v3l, v2h, v3h, pb0, pb1, c4);
            continue;
          }
          float t[4] = {0.f, 0.f, 0.f, 0.f};
          mma_f16(t, v0l, v1l, v0h, v1h, pa0, pa1, t);
          mma_f16(t, v2l, v3l, v2h, v3h, pb0, pb1, t);
          if constexpr (PT) {
            O[mt][0] = fmaf(t[0], g0, O[mt][0] * al0);
            O[mt][1] = fmaf(t[1], g1, O[mt][1] * al1);
            O[mt][2] = fmaf(t[2], g0, O[mt][2] * al0);
            O[mt][3] = fmaf(t[3], g1, O[mt][3] * al1);
          } else {
            O[mt][0] = fmaf(O[mt][0], al0, t[0]);
            O[mt][1] = fmaf(O[mt][1], al1, t[1]);
            O[mt][2] = fmaf(O[mt][2], al0, t[2]);
            O[mt][3] = fmaf(O[mt][3], al1, t[3]);
          }
        }
      } else {
        // ---- BF16 cache: S^T via bf16 MMA straight from shared memory ----
        auto qk = [&](uint32_t kp, float (&s)[4]) {
          float a[4] = {0.f, 0.f, 0.f, 0.f}, b[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int kk = 0; kk < G::KS; kk += 2) {
            uint32_t x0, x1, x2, x3, y0, y1, y2, y3;
            ldsm_x4(kp + koff[kk], x0, x1, x2, x3);
            ldsm_x4(kp + koff[kk + 1], y0, y1, y2, y3);
            mma_bf16(a, x0, x1, x2, x3, qh[2 * kk], qh[2 * kk + 1], a);
            mma_bf16(b, y0, y1, y2, y3, qh[2 * kk + 2], qh[2 * kk + 3], b);
          }
          s[0] = (a[0] + b[0]) * coef0;
          s[1] = (a[1] + b[1]) * coef1;
          s[2] = (a[2] + b[2]) * coef0;
          s[3] = (a[3] + b[3]) * coef1;
        };
        qk(kb, s0);
        if (two) qk(kb + k1off, s1);
        else s1[0] = s1[1] = s1[2] = s1[3] = NEG_INF;
        uint32_t vm0_lo = 0xFFFFFFFFu, vm0_hi = 0xFFFFFFFFu, vm1_lo = 0xFFFFFFFFu, vm1_hi = 0xFFFFFFFFu;
        if (edge) {
          if (!live(0, r)) s0[0] = s0[1] = NEG_INF;
          if (!live(0, r + 8)) s0[2] = s0[3] = NEG_INF;
          if (!live(1, r)) s1[0] = s1[1] = NEG_INF;
          if (!live(1, r + 8)) s1[2] = s1[3] = NEG_INF;
          // V fragments hold tokens 2c, 2c+1 (low pair) and 2c+8, 2c+9 (high pair)
          vm0_lo = (live(0, 2 * c) ? 0x0000FFFFu : 0u) | (live(0, 2 * c + 1) ? 0xFFFF0000u : 0u);
          vm0_hi = (live(0, 2 * c + 8) ? 0x0000FFFFu : 0u) | (live(0, 2 * c + 9) ? 0xFFFF0000u : 0u);
          vm1_lo = (live(1, 2 * c) ? 0x0000FFFFu : 0u) | (live(1, 2 * c + 1) ? 0xFFFF0000u : 0u);
          vm1_hi = (live(1, 2 * c + 8) ? 0x0000FFFFu : 0u) | (live(1, 2 * c + 9) ? 0xFFFF0000u : 0u);
        }
        softmax();
        // P as the sum of two bf16 terms (hi + lo), ~16 significant bits
        auto split = [&](float x, float y, uint32_t& hi, uint32_t& lo) {
          hi = pack_bf16x2(x, y);
          lo = pack_bf16x2(x - __uint_as_float(hi << 16), y - __uint_as_float(hi & 0xFFFF0000u));
          hi = movmatrix_t(hi);
          lo = movmatrix_t(lo);
        };
        uint32_t ha0, la0, ha1, la1, hb0, lb0, hb1, lb1;
        split(p00, p01, ha0, la0);
        split(p02, p03, ha1, la1);
        split(p10, p11, hb0, lb0);
        split(p12, p13, hb1, lb1);
#pragma unroll
        for (int mt = 0; mt < G::MT; ++mt) {
          float t[4] = {0.f, 0.f, 0.f, 0.f};
          {
            uint32_t y0, y1, y2, y3;
            ldsm_x4(vb + voff[mt], y0, y1, y2, y3);
            y0 &= vm0_lo;
            y1 &= vm0_lo;
            y2 &= vm0_hi;
            y3 &= vm0_hi;
            mma_bf16(t, y0, y1, y2, y3, ha0, ha1, t);
            mma_bf16(t, y0, y1, y2, y3, la0, la1, t);
          }
          if (two) {
            uint32_t y0, y1, y2, y3;
            ldsm_x4(vb + v1d + voff[mt], y0, y1, y2, y3);
            y0 &= vm1_lo;
            y1 &= vm1_lo;
            y2 &= vm1_hi;
            y3 &= vm1_hi;
            mma_bf16(t, y0, y1, y2, y3, hb0, hb1, t);
            mma_bf16(t, y0, y1, y2, y3, lb0, lb1, t);
          }
          O[mt][0] = fmaf(O[mt][0], al0, t[0]);
          O[mt][1] = fmaf(O[mt][1], al1, t[1]);
          O[mt][2] = fmaf(O[mt][2], al0, t[2]);
          O[mt][3] = fmaf(O[mt][3], al1, t[3]);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);
      }
    }
    it0 += nst_item;

    // ---- this warp's partial result for the segment (no cross-warp merge) ----
    // partial ((b * Hq + head) * S + split) * NW + warp, or in the balanced
    // plan (head * kseg + slot + b) * NW + warp; l and O are in units of 2^8 p,
    // the log-sum-exp in units of p
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      l[0] += __shfl_xor_sync(0xffffffffu, l[0], o);
      l[1] += __shfl_xor_sync(0xffffffffu, l[1], o);
    }
    if (p.direct) {
      // The ring is idle once every consumer warp is past its last stage (this
      // CTA's only item).  Each warp leaves (m, l, O) per query head there;
      // then the 128 consumer threads merge the four in FP32 and write out.
      // An abandoned call (timeout) writes nothing: bulk copies may still land.
      constexpr int WS = 16 + 8 * D;  // floats per warp: m[8], l[8], O[8][D]
      float* xw = reinterpret_cast<float*>(stages);
      named_bar_sync(1, NW * 32);
      if (!*abort_flag) {
        float* mine = xw + warp * WS;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int h = 2 * c + hh;
          if (r == 0) {
            mine[h] = m[hh];
            mine[8 + h] = l[hh];
          }
#pragma unroll
          for (int mt = 0; mt < G::MT; ++mt) {
            mine[16 + h * D + mt * 16 + r] = O[mt][hh];
            mine[16 + h * D + mt * 16 + r + 8] = O[mt][hh + 2];
          }
        }
      }
      named_bar_sync(1, NW * 32);
      if (!*abort_flag) {
        const float vs = (FP8 && !PT) ? p.v_scale[rg.kvh] : 1.f;  // PT: V scales are inside O
        __nv_bfloat16* dst = p.out + (static_cast<size_t>(rg.b) * p.Hq + rg.kvh * p.g) * D;
        for (int idx = threadIdx.x; idx < p.g * D; idx += NW * 32) {
          const int h = idx / D, d = idx - h * D;
          float M = -INFINITY;
#pragma unroll
          for (int w = 0; w < NW; ++w) M = fmaxf(M, xw[w * WS + h]);
          float num = 0.f, den = 0.f;
          if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < NW; ++w) {
              const float f = ex2(xw[w * WS + h] - M);  // 0 for a warp that saw no token
              den = fmaf(f, xw[w * WS + 8 + h], den);
              num = fmaf(f, xw[w * WS + 16 + h * D + d], num);
            }
          }
          dst[idx] = __float2bfloat16_rn(den > 0.f ? num / den * vs : 0.f);
        }
      }
      continue;  // one item per CTA in this mode
    }
    {
      const float vs = (FP8 && !PT) ? p.v_scale[rg.kvh] : 1.f;  // PT: V scales are inside O
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int h = 2 * c + hh;
        if (h < p.g) {
          const bool any = l[hh] > 0.f;
          const float f = any ? vs / l[hh] : 0.f;
          const size_t hq = static_cast<size_t>(rg.kvh) * p.g + h;
          const size_t idx = BAL ? ((hq * p.kseg + rg.split + rg.b) * NW + warp)
                                 : (((static_cast<size_t>(rg.b) * p.Hq + hq) * p.num_splits + rg.split) * NW + warp);
          float* dst = p.o_part + idx * D;
#pragma unroll
          for (int mt = 0; mt < G::MT; ++mt) {
            dst[mt * 16 + r] = O[mt][hh] * f;
            dst[mt * 16 + r + 8] = O[mt][hh + 2] * f;
          }
          if (r == 0) p.lse_part[idx] = any ? m[hh] + __log2f(l[hh]) - 8.f : -INFINITY;
        }
      }
    }
  }
}

// out[row][d] = sum_s 2^(lse_s - M) o_s[d] / sum_s 2^(lse_s - M) over the
// S' partials of row = (b, hq).  Grid (rows, D / 32), NW warps per CTA
// (chosen so that NW * kCombinePer covers S'): warp w takes partials w,
// w + NW, ... (lane = dimension) and loads their log-sum-exps and outputs
// together (one round trip), merges them against its own maximum, and the
// warps' results are merged through shared memory.
constexpr int kCombinePer = 8;  // partials per warp and pass
// Where a row's partials sit: per-sequence plan, S consecutive partials per
// row (row * S); balanced plan, the row's segments in its query head's block.
struct CombinePlan {
  int S;  // partials per row (per-sequence plan)
  int balanced;
  const int32_t* seq_lens;
  int B, Hq, max_blocks, window, num_slots, kseg;
};
template <int NW>
__global__ void __launch_bounds__(NW * 32) decode_combine_kernel(const float* __restrict__ o_part,
                                                                 const float* __restrict__ lse_part,
                                                                 __nv_bfloat16* __restrict__ out,
                                                                 const CombinePlan cp, int D) {
  static_assert(NW >= 1 && NW <= 32, "one lane per warp in the final merge");
  __shared__ float m_s[NW];
  __shared__ float den_s[NW];
  __shared__ float acc_s[NW][33];
  const int row = blockIdx.x;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  size_t first = static_cast<size_t>(row) * cp.S;
  int S = cp.S;
  if (cp.balanced) {
    // the sequence lengths were final before any partial CTA passed its wait,
    // and this grid launches only after that; L2-only loads see them
    const BatchScan bs = batch_scan_of(cp.seq_lens, cp.B, cp.max_blocks, cp.window, lane, true, nullptr);
    const int b = row / cp.Hq, hq = row - b * cp.Hq;
    const int incl = __shfl_sync(0xffffffffu, bs.incl, b);
    const int pages = __shfl_sync(0xffffffffu, bs.pages, b);
    int k0 = 0, cnt = 0;
    if (pages > 0) {
      const int N = used_slots(cp.num_slots, bs.total);
      k0 = slot_of(incl - pages, bs.total, N) + b;
      cnt = slot_of(incl - 1, bs.total, N) + b - k0 + 1;
    }
    first = (static_cast<size_t>(hq) * cp.kseg + k0) * kNW;
    S = cnt * kNW;
  }
  grid_dependency_wait();  // the partial kernel's writes are visible past this point
  // the next call's partial kernel may now start its setup (not earlier: its
  // CTAs would wait beside this call's partial CTAs, the slowest of which
  // set the call's time)
  grid_launch_dependents();
  const int d = blockIdx.y * 32 + lane;
  const float* lp = lse_part + first;
  const float* op = o_part + first * D + d;
  float m = -INFINITY, den = 0.f, acc = 0.f;
  for (int s0 = wid; s0 < S; s0 += NW * kCombinePer) {
    float l[kCombinePer], o[kCombinePer];
#pragma unroll
    for (int i = 0; i < kCombinePer; ++i) {
      const int s = s0 + i * NW;
      l[i] = s < S ? __ldg(lp + s) : -INFINITY;
      o[i] = s < S ? __ldg(op + s * D) : 0.f;  // S * D < 2^31: at most 65535 x 4 partials of 128 dims
    }
    float mn = m;
#pragma unroll
    for (int i = 0; i < kCombinePer; ++i) mn = fmaxf(mn, l[i]);
    if (mn != -INFINITY) {
      const float a = ex2(m - mn);  // m = -inf gives 0
      den *= a;
      acc *= a;
#pragma unroll
      for (int i = 0; i < kCombinePer; ++i) {
        const float w = ex2(l[i] - mn);
        den += w;
        acc = fmaf(w, o[i], acc);
      }
      m = mn;
    }
  }
  if (lane == 0) {
    m_s[wid] = m;
    den_s[wid] = den;
  }
  acc_s[wid][lane] = acc;
  __syncthreads();
  if (wid == 0) {
    const float mw = lane < NW ? m_s[lane] : -INFINITY;
    float M = mw;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float t = 0.f, dd = 0.f;
    if (M != -INFINITY) {
      // this lane's factor for warp `lane`, then a per-warp broadcast
      const float f = mw == -INFINITY ? 0.f : ex2(mw - M);
      dd = lane < NW ? den_s[lane] * f : 0.f;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) dd += __shfl_xor_sync(0xffffffffu, dd, o);
#pragma unroll 8
      for (int k = 0; k < NW; ++k) t = fmaf(__shfl_sync(0xffffffffu, f, k), acc_s[k][lane], t);
    }
    out[static_cast<size_t>(row) * D + d] = __float2bfloat16_rn(dd > 0.f ? t / dd : 0.f);
  }
}

int decode_pages(int P, int max_blocks, int window) {
  int pages = max_blocks;
  if (window > 0) {
    const int w = (window + P - 1) / P + 1;
    if (w < pages) pages = w;
  }
  return pages < 1 ? 1 : pages;
}

void split_plan(int B, int Hkv, int D, int P, int max_blocks, int window, int num_splits, int* S_out, int* pps_out) {
  const int pages = decode_pages(P, max_blocks, window);
  int S;
  if (num_splits > 0) {
    S = num_splits;
  } else {
    // at most one item per resident CTA: a second, partial wave of items would
    // take as long as the first
    const long target = static_cast<long>(ctas_per_sm_of(D)) * sm_count();
    const long pairs = static_cast<long>(B) * Hkv;
    S = static_cast<int>(target / pairs);
    // at least 4 pages (two stages) per split: short contexts run fastest cut
    // fine (512 tokens: 5.2 us at 8 splits against 7.2 us at 2)
    const int max_s = (pages + 3) / 4;
    if (S > max_s) S = max_s;
    // one range each, with direct output and no combine, where splitting
    // shortens no warp's work (at most one stage per consumer warp), or where
    // a few pages spread over many pairs (sliding-window layers: 4.8 against
    // 6.0 us)
    if (pages <= PPS * kNW || (pages <= 16 && pairs >= 32)) S = 1;
  }
  if (S > pages) S = pages;
  if (S < 1) S = 1;
  const int pps = (pages + S - 1) / S;
  S = (pages + pps - 1) / pps;
  *S_out = S;
  *pps_out = pps;
}

// The balanced plan (pages of the batch cut into equal slots) applies to
// ragged-capable batches that are split at all and fit one warp's scan.
bool balanced_plan(int B, int S) { return B > 1 && B <= 32 && S > 1; }

// Partials (one per consumer warp) a call writes: per-sequence plan B * Hq
// * S; balanced plan Hq * (B * S + B - 1) (segment ids slot + b).
size_t partial_count(int B, int Hq, int S) {
  if (balanced_plan(B, S)) return static_cast<size_t>(Hq) * (static_cast<size_t>(B) * S + B - 1) * kNW;
  return static_cast<size_t>(B) * Hq * S * kNW;
}

template <int D, bool FP8, bool E5 = false, bool PT = false, bool SL = false, bool AP = false, bool BAL = false>
kvq_status_t launch_decode(const DecodeParams& p, __nv_bfloat16* out, cudaStream_t s) {
  constexpr int NST = stages_for<D, FP8, PT>();
  constexpr size_t smem = decode_smem_bytes<D, FP8, NST, PT>();
  auto kern = decode_partial_kernel<D, FP8, kNW, NST, E5, PT, SL, AP, BAL>;
  static int configured_mask = 0;  // devices whose attribute is set
  int dev = 0;
  cudaGetDevice(&dev);
  if (!(configured_mask & (1 << (dev & 31)))) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, spread_smem(1));
    if (e != cudaSuccess) return cuda_status(e, "decode: set shared memory size");
    configured_mask |= 1 << (dev & 31);
  }
  const int sms = sm_count();
  constexpr int CPS = ctas_per_sm<D>();
  int grid = CPS * sms;
  DecodeParams q = p;
  q.out = out;
  // one page range per (sequence, KV head) and every item in its own CTA: the
  // CTAs write the output themselves
  q.direct = (p.num_splits == 1 && p.num_items <= grid) ? 1 : 0;
  if (grid > p.num_items) grid = p.num_items;
  // A grid smaller than the resident capacity asks for enough shared memory
  // that at most ceil(grid / SMs) CTAs fit on one SM: its CTAs then spread
  // over the SMs even when they are placed while the preceding kernel still
  // holds some of them (programmatic launch, below).
  const int per_sm = (grid + sms - 1) / sms;
  size_t dyn = smem;
  if (per_sm < CPS && static_cast<size_t>(spread_smem(per_sm)) > dyn) dyn = spread_smem(per_sm);
  // both kernels are programmatic dependents of what precedes them on the
  // stream: their launch and setup overlap its tail
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3((kNW + 1) * 32);
  cfg.dynamicSmemBytes = dyn;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, q);
  if (e != cudaSuccess) return cuda_status(e, "decode partial launch");
  if (q.direct) return KVQ_OK;
  cfg.gridDim = dim3(p.B * p.Hq, D / 32);
  cfg.dynamicSmemBytes = 0;
  CombinePlan cp;
  cp.S = p.num_splits * kNW;
  cp.balanced = p.balanced;
  cp.seq_lens = p.seq_lens;
  cp.B = p.B;
  cp.Hq = p.Hq;
  cp.max_blocks = p.max_blocks;
  cp.window = p.window;
  cp.num_slots = p.num_slots;
  cp.kseg = p.kseg;
  // warps per combine CTA: enough for a row's partials in one pass (balanced:
  // a sequence of average length spans about S + 1 segments)
  const int parts = (p.num_splits + (p.balanced ? 2 : 0)) * kNW;
  const float* op = p.o_part;
  const float* lp = p.lse_part;
  if (parts <= 4 * kCombinePer) {
    cfg.blockDim = dim3(4 * 32);
    e = cudaLaunchKernelEx(&cfg, decode_combine_kernel<4>, op, lp, out, cp, D);
  } else if (parts <= 8 * kCombinePer) {
    cfg.blockDim = dim3(8 * 32);
    e = cudaLaunchKernelEx(&cfg, decode_combine_kernel<8>, op, lp, out, cp, D);
  } else if (parts <= 16 * kCombinePer) {
    cfg.blockDim = dim3(16 * 32);
    e = cudaLaunchKernelEx(&cfg, decode_combine_kernel<16>, op, lp, out, cp, D);
  } else {
    cfg.blockDim = dim3(32 * 32);
    e = cudaLaunchKernelEx(&cfg, decode_combine_kernel<32>, op, lp, out, cp, D);
  }
  return cuda_status(e, "decode combine launch");
}

}  // namespace

}  // namespace kvq

using namespace kvq;

extern "C" int kvq_decode_num_splits(int B, int Hkv, int D, int P, int max_blocks, int window, int num_splits) {
  if (B < 1 || Hkv < 1 || D < 1 || P < 1 || max_blocks < 1 || num_splits < 0) return 0;
  int S, pps;
  split_plan(B, Hkv, D, P, max_blocks, window, num_splits, &S, &pps);
  return S;
}

extern "C" size_t kvq_decode_workspace_size(int B, int Hq, int Hkv, int D, int P, int max_blocks, int window,
                                            int num_splits) {
  if (B < 1 || Hq < 1 || Hkv < 1 || D < 1 || P < 1 || max_blocks < 1 || num_splits < 0) return 0;
  int S, pps;
  split_plan(B, Hkv, D, P, max_blocks, window, num_splits, &S, &pps);
  const size_t rows = partial_count(B, Hq, S);  // one partial per consumer warp
  const size_t o_bytes = rows * D * sizeof(float);
  return o_bytes + ((rows * sizeof(float) + 15) / 16) * 16;
}

namespace {

// The new token of each sequence for the append entry point.
struct AppendArgs {
  const void* k_new;
  const void* v_new;
  const int64_t* slot_new;
};

// Shared by the per-head and the per-token entry points.  per_token: the
// scales sit in the tail of each V page; k_scale and v_scale are unused.
kvq_status_t paged_decode(const void* q, const void* k_cache, const void* v_cache, const float* k_scale,
                          const float* v_scale, const int32_t* block_table, const int32_t* seq_lens, void* out, int B,
                          int Hq, int Hkv, int D, int P, int max_blocks, int64_t num_blocks, float sm_scale, int window,
                          kvq_dtype_t cache_dtype, int num_splits, void* workspace, size_t workspace_bytes,
                          int* dev_status, kvq_stream_t stream, bool per_token, bool single_level = false,
                          const AppendArgs* app = nullptr) {
  if (B < 1 || Hq < 1 || Hkv < 1 || max_blocks < 1 || num_blocks < 1 || num_splits < 0)
    return fail(KVQ_ERR_INVALID_ARG, "paged_decode: bad sizes");
  if (Hq % Hkv != 0) return fail(KVQ_ERR_INVALID_ARG, "paged_decode: Hq %% Hkv != 0");
  if (window == 0 || window < -1) return fail(KVQ_ERR_INVALID_ARG, "paged_decode: window must be -1 or > 0");
  if (!(sm_scale > 0.f) || !(sm_scale < FLT_MAX)) return fail(KVQ_ERR_INVALID_ARG, "paged_decode: bad sm_scale");
  if (P != kPage) return fail(KVQ_ERR_UNSUPPORTED, "paged_decode: page size %d (only 16)", P);
  if (D != 64 && D != 128) return fail(KVQ_ERR_UNSUPPORTED, "paged_decode: head_dim %d", D);
  if (Hq / Hkv > 8) return fail(KVQ_ERR_UNSUPPORTED, "paged_decode: GQA ratio %d > 8", Hq / Hkv);
  if (cache_dtype != KVQ_DTYPE_FP8_E4M3 && cache_dtype != KVQ_DTYPE_FP8_E5M2 && cache_dtype != KVQ_DTYPE_BF16)
    return fail(KVQ_ERR_INVALID_ARG, "paged_decode: bad cache dtype");
  const bool fp8 = cache_dtype != KVQ_DTYPE_BF16;
  if (!q || !k_cache || !v_cache || !block_table || !seq_lens || !out || !workspace)
    return fail(KVQ_ERR_INVALID_ARG, "paged_decode: null pointer");
  if (fp8 && !per_token && (!k_scale || !v_scale))
    return fail(KVQ_ERR_INVALID_ARG, "paged_decode: FP8 needs k_scale and v_scale");
  if (per_token && !fp8) return fail(KVQ_ERR_INVALID_ARG, "paged_decode: per-token scales need an FP8 cache");
  if (app && (per_token || single_level))
    return fail(KVQ_ERR_UNSUPPORTED, "paged_decode_append: per-head scales and two-level accumulation only");
  if (app && (!app->k_new || !app->v_new || !app->slot_new))
    return fail(KVQ_ERR_INVALID_ARG, "paged_decode_append: null pointer");
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(workspace, 16) ||
      !aligned(out, 4))
    return fail(KVQ_ERR_INVALID_ARG, "paged_decode: misaligned pointer");
  int S, pps;
  split_plan(B, Hkv, D, P, max_blocks, window, num_splits, &S, &pps);
  const size_t need = kvq_decode_workspace_size(B, Hq, Hkv, D, P, max_blocks, window, num_splits);
  if (workspace_bytes < need)
    return fail(KVQ_ERR_INVALID_ARG, "paged_decode: workspace %zu bytes < %zu needed", workspace_bytes, need);
  const long items = static_cast<long>(B) * Hkv * S;
  if (items > 0x7FFFFFFFL || static_cast<long>(B) * Hq > 0x7FFFFFFFL || S > 65535)
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
  prm.lse_part = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + partial_count(B, Hq, S) * D * sizeof(float));
  prm.B = B;
  prm.Hq = Hq;
  prm.Hkv = Hkv;
  prm.g = Hq / Hkv;
  prm.max_blocks = max_blocks;
  prm.num_blocks = num_blocks;
  prm.sm_scale = sm_scale;
  prm.window = window;
  prm.num_splits = S;
  prm.num_items = static_cast<int>(items);
  // the balanced plan is compiled for the E4M3 per-head two-level path at
  // head_dim 128; other paths keep one range per (sequence, KV head, split)
  prm.balanced = (balanced_plan(B, S) && D == 128 && cache_dtype == KVQ_DTYPE_FP8_E4M3 && !per_token &&
                  !single_level) ? 1 : 0;
  prm.num_slots = B * S;
  prm.kseg = B * S + B - 1;
  prm.dev_status = dev_status;
  prm.k_new = app ? static_cast<const uint16_t*>(app->k_new) : nullptr;
  prm.v_new = app ? static_cast<const uint16_t*>(app->v_new) : nullptr;
  prm.slot_new = app ? app->slot_new : nullptr;
  prm.k_cache_w = app ? static_cast<uint8_t*>(const_cast<void*>(k_cache)) : nullptr;
  prm.v_cache_w = app ? static_cast<uint8_t*>(const_cast<void*>(v_cache)) : nullptr;
  prm.stall_ns = stall_ns();
  {
    const int64_t page_b = static_cast<int64_t>(kPage) * D * (fp8 ? 1 : 2);
    const PageStrides ps = page_strides(k_cache, v_cache, page_b, page_b + (per_token ? kScaleTailBytes : 0));
    prm.k_str = ps.k;
    prm.v_str = ps.v;
    prm.paired = ps.paired ? 1 : 0;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  auto o = static_cast<__nv_bfloat16*>(out);
  const bool e5 = cache_dtype == KVQ_DTYPE_FP8_E5M2;
  if (single_level) {
    if (cache_dtype != KVQ_DTYPE_FP8_E4M3 || per_token)
      return fail(KVQ_ERR_UNSUPPORTED, "paged_decode: single-level accumulation covers E4M3 per-head caches");
    return D == 128 ? launch_decode<128, true, false, false, true>(prm, o, s)
                    : launch_decode<64, true, false, false, true>(prm, o, s);
  }
  if (per_token) {
    if (D == 128)
      return e5 ? launch_decode<128, true, true, true>(prm, o, s) : launch_decode<128, true, false, true>(prm, o, s);
    return e5 ? launch_decode<64, true, true, true>(prm, o, s) : launch_decode<64, true, false, true>(prm, o, s);
  }
  if (app) {
    if (e5)
      return D == 128 ? launch_decode<128, true, true, false, false, true>(prm, o, s)
                      : launch_decode<64, true, true, false, false, true>(prm, o, s);
    if (D == 128) {
      if (prm.balanced) return launch_decode<128, true, false, false, false, true, true>(prm, o, s);
      return fp8 ? launch_decode<128, true, false, false, false, true>(prm, o, s)
                 : launch_decode<128, false, false, false, false, true>(prm, o, s);
    }
    return fp8 ? launch_decode<64, true, false, false, false, true>(prm, o, s)
               : launch_decode<64, false, false, false, false, true>(prm, o, s);
  }
  if (e5) return D == 128 ? launch_decode<128, true, true>(prm, o, s) : launch_decode<64, true, true>(prm, o, s);
  if (D == 128) {
    if (prm.balanced) return launch_decode<128, true, false, false, false, false, true>(prm, o, s);
    return fp8 ? launch_decode<128, true>(prm, o, s) : launch_decode<128, false>(prm, o, s);
  }
  return fp8 ? launch_decode<64, true>(prm, o, s) : launch_decode<64, false>(prm, o, s);
}

}  // namespace

extern "C" kvq_status_t kvq_paged_decode_attention(const void* q, const void* k_cache, const void* v_cache,
                                                   const float* k_scale, const float* v_scale,
                                                   const int32_t* block_table, const int32_t* seq_lens, void* out,
                                                   int B, int Hq, int Hkv, int D, int P, int max_blocks,
                                                   int64_t num_blocks, float sm_scale, int window,
                                                   kvq_dtype_t cache_dtype, int num_splits, void* workspace,
                                                   size_t workspace_bytes, int* dev_status, kvq_stream_t stream) {
  clear_error();
  return paged_decode(q, k_cache, v_cache, k_scale, v_scale, block_table, seq_lens, out, B, Hq, Hkv, D, P,
                      max_blocks, num_blocks, sm_scale, window, cache_dtype, num_splits, workspace, workspace_bytes,
                      dev_status, stream, false);
}

extern "C" kvq_status_t kvq_paged_decode_attention_append(
    const void* q, const void* k_new, const void* v_new, const int64_t* slot_new, void* k_cache, void* v_cache,
    const float* k_scale, const float* v_scale, const int32_t* block_table, const int32_t* seq_lens, void* out, int B,
    int Hq, int Hkv, int D, int P, int max_blocks, int64_t num_blocks, float sm_scale, int window,
    kvq_dtype_t cache_dtype, int num_splits, void* workspace, size_t workspace_bytes, int* dev_status,
    kvq_stream_t stream) {
  clear_error();
  const AppendArgs app{k_new, v_new, slot_new};
  return paged_decode(q, k_cache, v_cache, k_scale, v_scale, block_table, seq_lens, out, B, Hq, Hkv, D, P,
                      max_blocks, num_blocks, sm_scale, window, cache_dtype, num_splits, workspace, workspace_bytes,
                      dev_status, stream, false, false, &app);
}

extern "C" kvq_status_t kvq_paged_decode_attention_acc(
    const void* q, const void* k_cache, const void* v_cache, const float* k_scale, const float* v_scale,
    const int32_t* block_table, const int32_t* seq_lens, void* out, int B, int Hq, int Hkv, int D, int P,
    int max_blocks, int64_t num_blocks, float sm_scale, int window, kvq_dtype_t cache_dtype, int num_splits,
    void* workspace, size_t workspace_bytes, int* dev_status, kvq_stream_t stream, kvq_accumulation_t accumulation) {
  clear_error();
  if (accumulation != KVQ_ACC_TWO_LEVEL && accumulation != KVQ_ACC_SINGLE_LEVEL)
    return fail(KVQ_ERR_INVALID_ARG, "paged_decode: bad accumulation mode");
  return paged_decode(q, k_cache, v_cache, k_scale, v_scale, block_table, seq_lens, out, B, Hq, Hkv, D, P,
                      max_blocks, num_blocks, sm_scale, window, cache_dtype, num_splits, workspace, workspace_bytes,
                      dev_status, stream, false, accumulation == KVQ_ACC_SINGLE_LEVEL);
}

extern "C" kvq_status_t kvq_paged_decode_attention_per_token(
    const void* q, const void* k_cache, const void* v_cache, const int32_t* block_table, const int32_t* seq_lens,
    void* out, int B, int Hq, int Hkv, int D, int P, int max_blocks, int64_t num_blocks, float sm_scale, int window,
    kvq_dtype_t cache_dtype, int num_splits, void* workspace, size_t workspace_bytes, int* dev_status,
    kvq_stream_t stream) {
  clear_error();
  return paged_decode(q, k_cache, v_cache, nullptr, nullptr, block_table, seq_lens, out, B, Hq, Hkv, D, P,
                      max_blocks, num_blocks, sm_scale, window, cache_dtype, num_splits, workspace, workspace_bytes,
                      dev_status, stream, true);
}

// ---------------------------------------------------------------------------
// Decode without a caller-provided workspace.
//
// Some callers cannot allocate device memory at the point where they run
// decode: code inside a region that must not call cudaMalloc (a memory-pool
// policy, a real-time loop, a plugin that has no access to its host engine's
// allocator).  For them the split-KV partials live in one fixed array that is
// part of this library's device image.  Every GPU that loads the library
// holds the array until the process exits.

namespace {

constexpr size_t kStaticScratchBytes = size_t(4) << 20;  // 4 MiB
static __device__ __align__(256) unsigned char g_decode_scratch[kStaticScratchBytes];

// The array's device address as seen from host code, per device, valid for
// the context it was looked up in: a new context on the device (after
// cudaDeviceReset, or another context made current) loads the module again,
// possibly elsewhere, so the address is looked up again when the current
// context differs from the one it was taken in.
struct ScratchAddr {
  void* ctx = nullptr;
  void* ptr = nullptr;
};
std::mutex g_scratch_mu;
ScratchAddr g_scratch_addr[64];

// cuCtxGetCurrent through the runtime's driver entry point (no link-time
// dependency on the driver library).
typedef int (*CtxGetCurrentFn)(void**);
CtxGetCurrentFn ctx_get_current() {
  static CtxGetCurrentFn fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 4000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      f = nullptr;
    return reinterpret_cast<CtxGetCurrentFn>(f);
  }();
  return fn;
}

}  // namespace

extern "C" size_t kvq_decode_static_scratch_bytes(void) { return kStaticScratchBytes; }

extern "C" kvq_status_t kvq_paged_decode_attention_static_scratch(
    const void* q, const void* k_cache, const void* v_cache, const float* k_scale, const float* v_scale,
    const int32_t* block_table, const int32_t* seq_lens, void* out, int B, int Hq, int Hkv, int D, int P,
    int max_blocks, int64_t num_blocks, float sm_scale, int window, kvq_dtype_t cache_dtype, int num_splits,
    int* dev_status, kvq_stream_t stream) {
  clear_error();
  if (B < 1 || Hq < 1 || Hkv < 1 || D < 1 || P < 1 || max_blocks < 1 || num_splits < 0)
    return fail(KVQ_ERR_INVALID_ARG, "paged_decode_static_scratch: bad sizes");
  const size_t need = kvq_decode_workspace_size(B, Hq, Hkv, D, P, max_blocks, window, num_splits);
  if (need > kStaticScratchBytes)
    return fail(KVQ_ERR_UNSUPPORTED,
                "paged_decode_static_scratch: needs %zu bytes of scratch, the static array holds %zu "
                "(use kvq_paged_decode_attention with a workspace, or fewer splits)",
                need, kStaticScratchBytes);
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_status(e, "paged_decode_static_scratch: cudaGetDevice");
  if (dev < 0 || dev >= 64) return fail(KVQ_ERR_UNSUPPORTED, "paged_decode_static_scratch: device %d", dev);
  CtxGetCurrentFn get_ctx = ctx_get_current();
  if (!get_ctx) return fail(KVQ_ERR_CUDA, "paged_decode_static_scratch: cuCtxGetCurrent unavailable");
  void* ctx = nullptr;
  if (get_ctx(&ctx) != 0 || ctx == nullptr) {
    // no context yet on this thread: cudaSetDevice creates the device's primary context
    e = cudaSetDevice(dev);
    if (e != cudaSuccess) return cuda_status(e, "paged_decode_static_scratch: cudaSetDevice");
    if (get_ctx(&ctx) != 0 || ctx == nullptr)
      return fail(KVQ_ERR_CUDA, "paged_decode_static_scratch: no current CUDA context");
  }
  void* ptr = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    ScratchAddr& a = g_scratch_addr[dev];
    if (a.ptr == nullptr || a.ctx != ctx) {
      // first call on this device (or in a new context): host code must use
      // the array's device address, not its host-side name
      void* addr = nullptr;
      e = cudaGetSymbolAddress(&addr, g_decode_scratch);
      if (e != cudaSuccess) return cuda_status(e, "paged_decode_static_scratch: cudaGetSymbolAddress");
      a.ptr = addr;
      a.ctx = ctx;
    }
    ptr = a.ptr;
  }
  return kvq_paged_decode_attention(q, k_cache, v_cache, k_scale, v_scale, block_table, seq_lens, out, B, Hq, Hkv,
                                    D, P, max_blocks, num_blocks, sm_scale, window, cache_dtype, num_splits, ptr,
                                    kStaticScratchBytes, dev_status, stream);
}
