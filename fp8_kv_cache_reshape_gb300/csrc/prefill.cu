// kvq_prefill_attention: chunked causal prefill over the paged FP8 cache on
// FP8 tensor cores (tcgen05.mma kind::f8f6f4, accumulators in tensor memory).
//
// Method: "The state of FP8 KV-cache and attention quantization in vLLM"
//  - "Kernel and vLLM improvements": QK^T and score.V both run in FP8 (e4m3);
//    two-level accumulation: partial P.V sums are promoted into real FP32;
//  - "Large head dimension limitations": the cost of the second level in
//    prefill (register pressure / extra passes);
// "FP8 and KV cache", "How to enable it in the engine": the query is
// quantized to FP8 too (kvq_quantize_query).
//
// One CTA = 128 query rows of one sequence x one query head; CTAs start
// heaviest query tile first.  Keys come in tiles of 128 (8 pages).  Warp
// roles (by warpgroup; setmaxnreg gives the softmax warpgroups 184 registers
// and the others fewer):
//  warps 12, 14  producers of the even / odd key tiles: block ids (read a
//             group of 4 tiles ahead) -> one bulk copy per K page and V page
//             into a 4-stage ring, each producer owning two of the stages
//             (pages of unknown / out-of-range blocks are zero filled and
//             masked).  Two issuing warps, because a page-sized bulk copy
//             costs the issuing warp tens of cycles;
//  warp 13    TMEM owner and MMA issuer: S_j = Q K_j^T into one of two TMEM
//             score buffers, then O_j = P_j V_j (P_j from TMEM, V_j from
//             shared memory) into a fresh TMEM accumulator O_tile (first
//             level);
//  warps 0-7  two threads per query row (warps w and w + 4 share TMEM lane
//             quarter w % 4), each owning 64 of the 128 columns of S_j:
//             online softmax in base 2 (the two halves exchange their tile
//             maxima through shared memory), P_j = e4m3(2^(s - m) * 256)
//             written back to TMEM over the first 16 of the thread's own S_j
//             columns, and the tile's rescale factor alpha_j;
//  warps 8-11 correction: O_run = O_run * alpha_j + O_tile_j in FP32 (second
//             level; O_run has its own TMEM columns), one thread per query
//             row, off the softmax warps' path; then the output rows.
// With single-level accumulation (SL) the P.V MMAs add into one TMEM sum O
// that the correction warps rescale in place.
// Shared-memory operands use the UMMA canonical K-major layouts: Q and K with
// the 128-byte swizzle (K pages are stored pre-swizzled by the cache format),
// V pages ([d][16 token slots]) without swizzle.
#include <cfloat>
#include <cmath>

#include "kvq_device.cuh"
#include "kvq_host.h"

namespace kvq {

namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr int TQ = 128;           // query rows per CTA
constexpr int TK = 128;           // keys per tile (8 pages)
constexpr int NPROD = 2;          // producer warps; tile j comes from producer j % NPROD
constexpr int PLANE = 128;        // bytes of one K-major operand row: 128 dims of FP8, 128-byte swizzle
// Warp roles, in warpgroups (setmaxnreg works per warpgroup):
//   warps 0 .. NSOFT-1  softmax, NPART per TMEM lane quarter (NPART threads
//                       per query row, TK / NPART columns of S each);
//   the next 4 warps    correction: the second accumulation level;
//   the last 4 warps    producer 0, MMA issuer, producer 1 (and one idle).
constexpr int NSOFT = 8;
constexpr int NPART = NSOFT / 4;
// P_j goes to tensor memory, over the first columns of each part's slice of
// S_j (already read by the thread that owns them), and P.V takes its A
// operand from there.
static_assert(NPART == 2, "P in TMEM: 16 columns of 4 keys per thread");
constexpr int NCORR = 4;
constexpr int W_CORR = NSOFT;
constexpr int W_PROD0 = NSOFT + NCORR, W_MMA = W_PROD0 + 1, W_PROD1 = W_PROD0 + 2;
constexpr int NTHREADS = (NSOFT + NCORR + 4) * 32;
// Registers per thread: the launch gives every thread the same count; the
// control and correction warpgroups then give some back and the softmax
// warpgroups take them (the sum must stay within the launch's allocation).
constexpr int REG_LAUNCH = (65536 / NTHREADS) / 8 * 8;
constexpr int REG_SOFT = 184, REG_CORR = 88, REG_CTRL = 56;  // all 65,536 of the launch
static_assert(NSOFT * 32 * REG_SOFT + NCORR * 32 * REG_CORR + 128 * REG_CTRL <= NTHREADS * REG_LAUNCH,
              "register split");
// TMEM: S0 | S1 | O_tile | O_run at head_dim 128 (128 columns each); at 256,
// S0 | S1 | O (single-level accumulation: O_tile and O_run do not both fit).
constexpr uint32_t TMEM_COLS = 512;

// Shared-memory plan for one head dimension.  Q and the K tile are stored as
// HD / 128 planes of 128-byte rows (dims 128h .. 128h + 127), each a canonical
// SWIZZLE_128B K-major operand; V pages stay [d][16 slots].
// PT: per-token scales; each V page carries its scale tail (16 K scales, 16 V
// scales) and lands with it, so V pages sit VPAGE_B = PAGE_B + 128 bytes
// apart in the stage (the P.V operand's stride along the keys says so).
template <int HD_, bool PT = false>
struct Geo {
  static constexpr int HD = HD_;
  static constexpr int NKV = HD == 128 ? 4 : 2;  // K/V stages (2 x 64 KiB at head_dim 256)
  static_assert(NKV % NPROD == 0, "each stage belongs to one producer, which refills it in tile order");
  static constexpr int PAGE_B = kPage * HD;      // bytes per page (K or V codes)
  static constexpr int VPAGE_B = PAGE_B + (PT ? kScaleTailBytes : 0);  // a V page in the stage
  static constexpr int TILE_B = TK * HD;         // bytes per K tile
  static constexpr int TILE_V = (TK / kPage) * VPAGE_B;  // bytes per V tile
  static constexpr int PLANE_Q = TQ * PLANE;     // one plane of Q
  static constexpr int PLANE_K = TK * PLANE;     // one plane of a K tile
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_KV = OFF_Q + TQ * HD;
  static constexpr int STAGE_B = TILE_B + TILE_V;  // K tile + V tile
  static constexpr int OFF_BAR = OFF_KV + NKV * STAGE_B;
  static constexpr int OFF_XCH = OFF_BAR + 512;  // row max exchange [2 tiles][NPART][TQ]
  static constexpr int OFF_ALPHA = OFF_XCH + 2 * NPART * TQ * 4;  // [4][TQ] rescale factors, softmax -> correction
  // PT: [4] the tiles' V-scale bounds C_t (softmax -> correction), then the
  // largest V scale of each part's keys [2 tiles][NPART] (softmax exchange)
  static constexpr int OFF_CT = OFF_ALPHA + 4 * TQ * 4;
  static constexpr int OFF_ONES = OFF_CT + 64;                     // E4M3 ones: the B operand of the row-sum MMA
  static constexpr int SMEM_BYTES = OFF_ONES + 1024 + 1024;        // + alignment slack
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory per CTA");
  static_assert(VPAGE_B % 16 == 0 && OFF_ONES % 16 == 0, "16-byte aligned operands");
};

struct PrefillParams {
  const uint8_t* q8;
  const float* q_scale;
  const uint8_t* k_cache;
  const uint8_t* v_cache;
  const float* k_scale;
  const float* v_scale;
  const int32_t* block_table;
  const int32_t* cu_seqlens_q;
  const int32_t* seq_lens;
  __nv_bfloat16* out;
  int B, Hq, Hkv, g, max_blocks;
  int64_t num_blocks;
  float sm_scale;
  int causal;
  int* dev_status;
  int64_t k_str, v_str;  // bytes between consecutive (block, KV head) pages of each cache
  // failure-path test hook (kvq_debug_set_stall_ns): > 0 makes the softmax
  // warps wait up to this long on a barrier nothing arrives on before the
  // first key tile, which fails like a stuck pipeline wait
  uint64_t stall_ns;
};

template <int NKV>
struct Bars {
  uint64_t q_full;
  // K and V of a stage land and are released separately: K once S = Q K^T
  // has been computed, V once P.V has, so the next K tile is copied while
  // this tile's softmax and P.V still run
  uint64_t k_full[NKV];
  uint64_t v_full[NKV];
  uint64_t k_empty[NKV];
  uint64_t v_empty[NKV];
  uint64_t s_full[2];
  uint64_t p_full[2];
  uint64_t o_full;  // P.V of the current tile is in O_tile
  uint64_t o_free;  // O_tile has been folded into O_run (correction warps)
  uint64_t rs_free;  // the row sums of tile j have been read: S_j's buffer may be rewritten
  uint64_t a_full[4];  // alpha of tile j is in slot j % 4 (softmax part 0 -> correction warps)
  uint64_t mma_done;
  uint64_t stall;  // nothing arrives on it (test hook)
  uint32_t tmem_base;
  int abort;
  uint32_t tile_bad[8];  // bit i: page i of tile j (slot j % 8) had a bad block id
};

// ------------------------------------------------------------ tcgen05 PTX ---
KVQ_DEVINL uint64_t desc_sw128(uint32_t saddr) {  // K-major, 128B swizzle, 8-row groups 1024 B apart
  uint64_t d = static_cast<uint64_t>((saddr >> 4) & 0x3FFF);
  d |= static_cast<uint64_t>(1) << 16;                 // leading offset (unused for swizzled K-major)
  d |= static_cast<uint64_t>(1024 >> 4) << 32;         // stride offset
  d |= static_cast<uint64_t>(1) << 46;                 // descriptor version
  d |= static_cast<uint64_t>(2) << 61;                 // SWIZZLE_128B
  return d;
}
KVQ_DEVINL uint64_t desc_interleave(uint32_t saddr, uint32_t lbo, uint32_t sbo) {  // K-major, no swizzle
  uint64_t d = static_cast<uint64_t>((saddr >> 4) & 0x3FFF);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFF) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFF) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  return d;
}
// kind::f8f6f4 instruction descriptor: D f32, A e4m3, B e4m3 (b_e5m2: e5m2),
// both K-major, M x N.  The element types of A and B are separate fields.
constexpr uint32_t idesc_e4m3(int M, int N, bool b_e5m2 = false) {
  return (1u << 4) | (0u << 7) | ((b_e5m2 ? 1u : 0u) << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}
KVQ_DEVINL void umma_f8(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// The same with the A operand in tensor memory (one row per TMEM lane, four
// FP8 elements of K per 32-bit column).
KVQ_DEVINL void umma_f8_ta(uint32_t tmem_d, uint32_t tmem_a, uint64_t bdesc, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n\t}" ::"r"(tmem_d),
      "r"(tmem_a), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
KVQ_DEVINL void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}
KVQ_DEVINL void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
KVQ_DEVINL void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
KVQ_DEVINL void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
KVQ_DEVINL void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
KVQ_DEVINL void tmem_ld16_async(uint32_t taddr, uint32_t (&v)[16]) {  // complete after tmem_wait_ld()
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]), "=r"(v[8]),
        "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
      : "r"(taddr));
}
KVQ_DEVINL void tmem_st16(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::
                   "r"(taddr),
               "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
               "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
               : "memory");
}
KVQ_DEVINL float tmem_ld1(uint32_t taddr) {  // one column of this warp's 32 lanes
  uint32_t v;
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];" : "=r"(v) : "r"(taddr));
  tmem_wait_ld();
  return __uint_as_float(v);
}
KVQ_DEVINL void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
      "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]), "=r"(v[8]),
        "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]),
        "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]),
        "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
      : "r"(taddr));
  tmem_wait_ld();
}
// tcgen05.ld without the wait; the registers are valid after tmem_wait_ld(),
// and tmem_pin32() after that wait keeps the compiler from using them earlier.
KVQ_DEVINL void tmem_ld32_nowait(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
      "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]), "=r"(v[8]),
        "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]),
        "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]),
        "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
      : "r"(taddr));
}
KVQ_DEVINL void tmem_pin32(uint32_t (&v)[32]) {
  asm volatile(""
               : "+r"(v[0]), "+r"(v[1]), "+r"(v[2]), "+r"(v[3]), "+r"(v[4]), "+r"(v[5]), "+r"(v[6]), "+r"(v[7]),
                 "+r"(v[8]), "+r"(v[9]), "+r"(v[10]), "+r"(v[11]), "+r"(v[12]), "+r"(v[13]), "+r"(v[14]),
                 "+r"(v[15]), "+r"(v[16]), "+r"(v[17]), "+r"(v[18]), "+r"(v[19]), "+r"(v[20]), "+r"(v[21]),
                 "+r"(v[22]), "+r"(v[23]), "+r"(v[24]), "+r"(v[25]), "+r"(v[26]), "+r"(v[27]), "+r"(v[28]),
                 "+r"(v[29]), "+r"(v[30]), "+r"(v[31]));
}

struct Job {
  int b, h, kvh, q0, nq, L, first_q;  // first_q: absolute position of the sequence's first new token
  int nkv;                             // key tiles this CTA visits
  bool valid;
};

KVQ_DEVINL Job make_job(const PrefillParams& p) {
  Job j;
  // grid (heads, query tiles, sequences), query tiles in reverse: the CTAs
  // start in order of decreasing work (later query tiles attend to more keys
  // under the causal mask), so the last, partial wave holds the lightest ones
  j.b = blockIdx.z;
  j.h = blockIdx.x;
  j.kvh = j.h / p.g;
  j.q0 = (gridDim.y - 1 - blockIdx.y) * TQ;
  const int c0 = p.cu_seqlens_q[j.b];
  const int c1 = p.cu_seqlens_q[j.b + 1];
  j.nq = c1 - c0;
  int L = p.seq_lens[j.b];
  const int cap = p.max_blocks * kPage;
  j.valid = j.q0 < j.nq;
  if (L < 0 || L > cap) {
    if (threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.y == 0) set_status(p.dev_status, KVQ_DEV_BAD_SEQLEN);
    L = L < 0 ? 0 : cap;
  }
  if (j.nq > L) {
    if (threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.y == 0) set_status(p.dev_status, KVQ_DEV_BAD_QROWS);
    j.valid = false;
  }
  j.L = L;
  j.first_q = L - j.nq;
  const int last_row = min(j.q0 + TQ, j.nq) - 1;
  const int kend = p.causal ? (j.first_q + last_row + 1) : L;  // keys [0, kend)
  j.nkv = j.valid ? (kend + TK - 1) / TK : 0;
  return j;
}

// SL: single-level accumulation (an ablation of the two-level scheme): P.V
// of every tile accumulates into one TMEM sum O, which the softmax warps
// rescale by alpha in place (skipped when alpha is 1 for the whole warp).
// Head dim 256 needs it: two-level would need 2 x 256 TMEM columns for O.
// E5: the caches hold E5M2 codes: K (the B operand of Q K^T) and V (the B
// operand of P.V) are E5M2, Q and P stay E4M3.
// PT: per-token scales in the V pages' tails.  Scores are s2 = raw *
// fl32(sk * b), b = fl32(fl32(q_scale * sm_scale) * log2 e); P.V runs on the
// weighted codes e4m3(fl32(2^(s2 - M + 8) * (sv / C_t))), C_t = 2^ceil(log2
// max sv) over the tile's cached keys, and the row sums on the unweighted
// codes e4m3(2^(s2 - M + 8)); the correction warps carry O_run / C_t, so
// every rescale stays a power of two.
template <int HD, bool SL, bool E5 = false, bool PT = false>
__global__ void __launch_bounds__(NTHREADS, 1) prefill_kernel(const __grid_constant__ PrefillParams p) {
  using G = Geo<HD, PT>;
  static_assert(HD == 128 || (HD == 256 && SL), "head_dim 256 runs with single-level accumulation");
  // K/V stage protocol.  Split: K and V of a stage land and are released
  // separately (K once S = Q K^T is computed and the softmax has read the
  // tile's page flags, V after P.V), so the next K tile is copied while this
  // tile's softmax and P.V run; the ring holds only two 64 KiB stages at head
  // dim 256, where this took 5.19 ms to 1.88 ms.  Combined: one barrier pair
  // per stage, both halves released after P.V -- per-token scales, whose
  // softmax reads the K scales from the V pages' tails (measured faster).
  constexpr bool SPLIT = !PT;
  static_assert(!PT || (HD == 128 && !SL), "per-token scales: head_dim 128, two-level accumulation");
  constexpr int NKV = G::NKV, PAGE_B = G::PAGE_B, TILE_B = G::TILE_B, STAGE_B = G::STAGE_B;
  constexpr int VPAGE_B = G::VPAGE_B;
  constexpr int OFF_Q = G::OFF_Q, OFF_KV = G::OFF_KV, OFF_XCH = G::OFF_XCH;
  using BarsN = Bars<NKV>;
  static_assert(sizeof(BarsN) <= 512, "barrier block");
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw + 1023) & ~1023u) - raw);
  const uint32_t sbase = smem_u32(smem);
  BarsN* bars = reinterpret_cast<BarsN*>(smem + G::OFF_BAR);
  volatile int* abort_flag = &bars->abort;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const Job job = make_job(p);
  if (!job.valid) return;  // uniform across the CTA

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, NSOFT * 32);
    for (int i = 0; i < NKV; ++i) {
      mbar_init(&bars->k_full[i], 1);
      mbar_init(&bars->v_full[i], 1);
      // split: released by the QK^T commit and by the softmax once every
      // softmax thread is past its wait on k_full (which then cannot move on)
      mbar_init(&bars->k_empty[i], SPLIT ? 2 : 1);
      mbar_init(&bars->v_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->s_full[i], 1);
      mbar_init(&bars->p_full[i], NSOFT * 32);
    }
    mbar_init(&bars->o_full, 1);
    mbar_init(&bars->o_free, NCORR * 32);
    mbar_init(&bars->rs_free, NCORR * 32);
    for (int i = 0; i < 4; ++i) mbar_init(&bars->a_full[i], NSOFT / NPART * 32);
    mbar_init(&bars->mma_done, 1);
    mbar_init(&bars->stall, 1);
    bars->abort = 0;
    fence_barrier_init();
  }
  if (warp == W_MMA) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&bars->tmem_base)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (threadIdx.x < 64) {  // 1 KiB of E4M3 1.0 for the row-sum MMA, before the tensor cores read it
    reinterpret_cast<uint4*>(smem + G::OFF_ONES)[threadIdx.x] =
        make_uint4(kE4m3OnesX4, kE4m3OnesX4, kE4m3OnesX4, kE4m3OnesX4);
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  const int nkv = job.nkv;
  // each warpgroup sets its register budget at the top of its own branch
  if (warp >= W_PROD0) {
    setmaxnreg_dec<REG_CTRL>();
    if (warp == W_PROD0 || warp == W_PROD1) {
      // ----------------------------------------------------------- producers --
      const int n_pages = (job.L + kPage - 1) / kPage;
      const int32_t* bt = p.block_table + static_cast<size_t>(job.b) * p.max_blocks;
      // Block ids come one warp-wide load per group of 4 tiles (32 pages), issued
      // a group ahead so that its latency hides behind the copies; lane
      // (j % 4) * 8 + i of `ids` holds the block of page i of tile j.
      auto load_ids = [&](int grp) {
        const int page = grp * 32 + lane;
        return page < n_pages ? __ldg(bt + page) : -1;
      };
      int ids = load_ids(0);
      int ids_next = load_ids(1);
      int cur_grp = 0;
      bool k_only = false;  // stopped between a tile's K and V copies
      int j = (warp == W_PROD0) ? 0 : 1;  // this producer's first tile
      for (; j < nkv; j += NPROD) {
        if ((j >> 2) != cur_grp) {  // steps of NPROD < 4 tiles: at most one group ahead
          cur_grp = j >> 2;
          ids = ids_next;
          ids_next = load_ids(cur_grp + 1);
        }
        const int st = j % NKV;
        const uint32_t free_parity = ((j / NKV) & 1) ^ 1;
        // split: K on k_full after k_empty, V below; combined: both halves on
        // v_full after v_empty
        uint64_t* k_bar = SPLIT ? &bars->k_full[st] : &bars->v_full[st];
        uint64_t* k_free = SPLIT ? &bars->k_empty[st] : &bars->v_empty[st];
        int ok = 1;
        if (lane == 0) ok = (!*abort_flag && mbar_wait(k_free, free_parity, abort_flag)) ? 1 : 0;
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        uint8_t* ks = smem + OFF_KV + st * STAGE_B;
        uint8_t* vs = ks + TILE_B;
        // lanes 0..7: one page each
        int blk = __shfl_sync(0xffffffffu, ids, ((j & 3) << 3) | (lane & 7));
        const int page = j * (TK / kPage) + lane;
        if (lane >= TK / kPage || page >= n_pages) {
          blk = -1;
        } else if (blk < 0 || static_cast<int64_t>(blk) >= p.num_blocks) {
          set_status(p.dev_status, KVQ_DEV_BAD_BLOCK);
          blk = -1;
        }
        const uint32_t load_mask = __ballot_sync(0xffffffffu, blk >= 0) & 0xFFu;
        const uint32_t bad_mask = __ballot_sync(0xffffffffu, lane < TK / kPage && page < n_pages && blk < 0) & 0xFFu;
        // zero-fill pages that are not loaded (past the end, or bad block ids):
        // K here, V once its half of the stage is free
        auto zero_v = [&]() {
          for (int pg = 0; pg < TK / kPage; ++pg) {
            if (load_mask & (1u << pg)) continue;
            uint4* vz = reinterpret_cast<uint4*>(vs + pg * VPAGE_B);
            for (int i = lane; i < VPAGE_B / 16; i += 32) vz[i] = make_uint4(0, 0, 0, 0);  // codes (and scales)
          }
        };
        if (load_mask != 0xFFu) {
          for (int pg = 0; pg < TK / kPage; ++pg) {
            if (load_mask & (1u << pg)) continue;
            for (int i = lane; i < PAGE_B / 16; i += 32) {
              // K: the page's kPage rows in each plane
              const int pl = i / (kPage * PLANE / 16), w = i % (kPage * PLANE / 16);
              reinterpret_cast<uint4*>(ks + pl * G::PLANE_K + pg * kPage * PLANE)[w] = make_uint4(0, 0, 0, 0);
            }
          }
          if constexpr (!SPLIT) zero_v();
          fence_proxy_async_smem();  // the zeros, before the tensor cores read the stage
        }
        __syncwarp();
        if (lane == 0) {
          bars->tile_bad[j & 7] = bad_mask;
          mbar_arrive_expect_tx(k_bar, static_cast<uint32_t>(SPLIT ? PAGE_B : PAGE_B + VPAGE_B) * __popc(load_mask));
        }
        __syncwarp();
        size_t pair_off = 0;
        if (lane < TK / kPage && blk >= 0) {
          pair_off = static_cast<size_t>(blk) * p.Hkv + job.kvh;
          const size_t off = pair_off * p.k_str;
          // one copy per plane (a K page of head dim 256 is stored as two half-pages)
#pragma unroll
          for (int pl = 0; pl < HD / PLANE; ++pl)
            bulk_g2s(ks + pl * G::PLANE_K + lane * kPage * PLANE, p.k_cache + off + pl * kPage * PLANE, kPage * PLANE,
                     k_bar, policy_evict_last());
          // combined: the V page (PT: with its scale tail) on the same barrier
          if constexpr (!SPLIT)
            bulk_g2s(vs + lane * VPAGE_B, p.v_cache + pair_off * p.v_str, VPAGE_B, k_bar, policy_evict_last());
        }
        if constexpr (SPLIT) {
          if (lane == 0) ok = (!*abort_flag && mbar_wait(&bars->v_empty[st], free_parity, abort_flag)) ? 1 : 0;
          ok = __shfl_sync(0xffffffffu, ok, 0);
          if (!ok) {
            k_only = true;
            break;
          }
          if (load_mask != 0xFFu) {
            zero_v();
            fence_proxy_async_smem();
          }
          __syncwarp();
          if (lane == 0) mbar_arrive_expect_tx(&bars->v_full[st], static_cast<uint32_t>(VPAGE_B) * __popc(load_mask));
          __syncwarp();
          if (lane < TK / kPage && blk >= 0)
            bulk_g2s(vs + lane * VPAGE_B, p.v_cache + pair_off * p.v_str, VPAGE_B, &bars->v_full[st], policy_evict_last());
        }
      }
      if (j < nkv && lane == 0) {  // abandoned: let this producer's issued copies land
        set_status(p.dev_status, KVQ_DEV_TIMEOUT);
        *abort_flag = 1;
        for (int k = j - NPROD; k >= 0 && k >= j - NKV; k -= NPROD) {
          if constexpr (SPLIT) mbar_wait(&bars->k_full[k % NKV], (k / NKV) & 1);
          mbar_wait(&bars->v_full[k % NKV], (k / NKV) & 1);
        }
        if (k_only) mbar_wait(&bars->k_full[j % NKV], (j / NKV) & 1);
      }
    } else if (warp == W_MMA) {
      // ------------------------------------------------------------ MMA issuer --
      constexpr uint32_t IDESC_S = idesc_e4m3(TQ, TK, E5);  // S = Q K^T: N = keys
      constexpr uint32_t IDESC_O = idesc_e4m3(TQ, HD, E5);  // O += P V: N = head dim
      const uint32_t q_s = sbase + OFF_Q;
      bool ok = true;
      auto wait = [&](uint64_t* bar, uint32_t parity) {
        if (ok && !mbar_wait(bar, parity, abort_flag)) {
          ok = false;
          if (lane == 0) {
            set_status(p.dev_status, KVQ_DEV_TIMEOUT);
            *abort_flag = 1;
          }
        }
        return ok;
      };
      auto issue_s = [&](int j) {  // S[j%2] = Q K_j^T
        const int st = j % NKV;
        if (!wait(SPLIT ? &bars->k_full[st] : &bars->v_full[st], (j / NKV) & 1)) return;
        tc_fence_after();
        if (lane == 0) {
          const uint32_t k_s = sbase + OFF_KV + st * STAGE_B;
          const uint32_t d = tmem + (j & 1) * TK;
#pragma unroll
          for (int kk = 0; kk < HD / 32; ++kk)  // 32 dims per MMA, four per 128-byte plane
            umma_f8(d, desc_sw128(q_s + (kk >> 2) * G::PLANE_Q + (kk & 3) * 32),
                    desc_sw128(k_s + (kk >> 2) * G::PLANE_K + (kk & 3) * 32), IDESC_S, kk > 0 ? 1u : 0u);
          umma_commit(&bars->s_full[j & 1]);
          if constexpr (SPLIT) umma_commit(&bars->k_empty[st]);  // the K half may be refilled
        }
        __syncwarp();
      };
      constexpr uint32_t IDESC_RS = idesc_e4m3(TQ, 16);  // row sums: N = 16 columns of ones
      const uint64_t ones_desc = desc_interleave(sbase + G::OFF_ONES, 128, 256);  // every byte 1.0
      if (wait(&bars->q_full, 0) && nkv > 0) issue_s(0);
      for (int j = 0; j < nkv && ok; ++j) {
        if (j + 1 < nkv) {
          // S_{j+1} goes into tile j - 1's buffer, which holds that tile's row sums until read
          if (j >= 1 && !wait(&bars->rs_free, (j - 1) & 1)) break;
          tc_fence_after();
          issue_s(j + 1);
        }
        if (!ok) break;
        if (!wait(&bars->p_full[j & 1], (j >> 1) & 1)) break;
        // two-level: O_tile of tile j - 1 has been read; SL: O has been rescaled for tile j
        if (j >= 1 && !wait(&bars->o_free, (j - 1) & 1)) break;
        // split: V_j (combined: it landed with K_j, before S_j)
        if (SPLIT && !wait(&bars->v_full[j % NKV], (j / NKV) & 1)) break;
        tc_fence_after();
        if (lane == 0) {
          const int st = j % NKV;
          const uint32_t v_s = sbase + OFF_KV + st * STAGE_B + TILE_B;
          const uint32_t d = tmem + 2 * TK;  // O_tile (SL: the running sum O)
          constexpr int KPP = TK / NPART / 32;  // 32-key steps per part
#pragma unroll
          for (int kk = 0; kk < TK / 32; ++kk) {  // 32 keys = 2 V pages per MMA
            const uint32_t acc = (kk > 0 || (SL && j > 0)) ? 1u : 0u;
            const uint64_t vdesc = desc_interleave(v_s + kk * 2 * VPAGE_B, VPAGE_B, 128);
            // P for keys 32kk .. 32kk + 31: 8 columns at the start of part pt's slice of S_j
            const int pt = kk / KPP;
            umma_f8_ta(d, tmem + (j & 1) * TK + pt * (TK / NPART) + 8 * (kk - pt * KPP), vdesc, IDESC_O, acc);
          }
          // the tile's row sums of the same P8 codes, sum_k P8[row][k] in each of 16
          // columns, into S_j's columns 32 .. 47 (already read by the softmax warps);
          // PT: of the unweighted codes, 16 columns after the weighted ones
          constexpr int RS_SRC = PT ? 16 : 0;
#pragma unroll
          for (int kk = 0; kk < TK / 32; ++kk) {
            const int pt = kk / KPP;
            umma_f8_ta(tmem + (j & 1) * TK + 32,
                       tmem + (j & 1) * TK + pt * (TK / NPART) + RS_SRC + 8 * (kk - pt * KPP), ones_desc, IDESC_RS,
                       kk > 0 ? 1u : 0u);
          }
          umma_commit(&bars->o_full);
          umma_commit(&bars->v_empty[st]);
        }
        __syncwarp();
      }
      // every MMA this thread issued has completed before TMEM is released
      if (lane == 0) umma_commit(&bars->mma_done);
      __syncwarp();
      mbar_wait(&bars->mma_done, 0);
    }
  } else if (warp >= W_CORR) {
    setmaxnreg_dec<REG_CORR>();
    // -------------------------------------------------- correction warps --
    // The rescale of the running sum, off the softmax warps' path, then the
    // output rows.  One thread per query row (TMEM lane), all HD columns.
    //  two-level: O_run = O_run * alpha_j + O_tile_j in FP32 for every key
    //             tile j (the second level), O_tile released for P.V j + 1;
    //  SL:        O = O * alpha_j in place (skipped when alpha_j is 1 for the
    //             whole warp) once P.V of tile j - 1 has landed, released for
    //             P.V of tile j, which adds into O.
    // The softmax warps cannot finish tile j + 3 before the release for tile
    // j (S_{j+3} is issued after P.V of tile j + 1, which waits for it), so
    // the four alpha slots and their barriers' parities never alias.
    const int quarter = warp & 3;
    const uint32_t t_lane = static_cast<uint32_t>(quarter * 32) << 16;
    const int row = quarter * 32 + lane;
    const uint32_t o_tile = tmem + t_lane + 2 * TK;  // SL: O
    const uint32_t o_run = o_tile + HD;              // two-level only
    const float* alpha_s = reinterpret_cast<const float*>(smem + G::OFF_ALPHA);
    const float* ct_s = reinterpret_cast<const float*>(smem + G::OFF_CT);  // PT: C_j of tile j in slot j % 4
    float c_prev = 1.f;                                                     // PT: C of the last tile folded
    // the row sum of the rounded probabilities, in units of 2^8 p: the tensor
    // core's sums of each tile's P8 codes (S_j's columns 32 .. 47), rescaled
    // like the output
    float l = 0.f;
    auto row_sum = [&](int j) {  // after o_full of tile j; then S_j's buffer may be rewritten
      const float rs = tmem_ld1(tmem + t_lane + (j & 1) * TK + 32);
      tc_fence_before();
      mbar_arrive(&bars->rs_free);
      return rs;
    };
    bool ok = true;
    auto wait_all = [&](uint64_t* bar, uint32_t parity) {
      if (!ok) return false;
      const bool got = mbar_wait(bar, parity, abort_flag);
      if (!__all_sync(0xffffffffu, got)) {
        ok = false;
        set_status(p.dev_status, KVQ_DEV_TIMEOUT);
        *abort_flag = 1;
      }
      return ok;
    };
    if constexpr (!SL) {
      {  // O_run = 0
        uint32_t z[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) z[i] = 0u;
#pragma unroll
        for (int c = 0; c < HD / 16; ++c) tmem_st16(o_run + 16 * c, z);
      }
      for (int j = 0; j < nkv && ok; ++j) {
        float alpha = 0.f;  // tile 0: O_run is zero
        float ratio = 1.f;  // PT: C_{j-1} / C_j, a power of two (O_run is kept in units of C_j)
        if (j > 0 || PT) {
          if (!wait_all(&bars->a_full[j & 3], (j >> 2) & 1)) break;
          if (j > 0) alpha = alpha_s[(j & 3) * TQ + row];
          if constexpr (PT) {
            const float c_j = ct_s[j & 3];
            ratio = c_prev / c_j;
            c_prev = c_j;
          }
        }
        if (!wait_all(&bars->o_full, j & 1)) break;  // P.V of tile j is in O_tile
        tc_fence_after();
        l = fmaf(l, alpha, row_sum(j));
        tmem_wait_st();  // this thread's previous O_run update
        const float am = PT ? alpha * ratio : alpha;
        const float2 a2 = make_float2(am, am);
        // 32 columns of O_tile and of O_run per tensor-memory round trip (its
        // latency, not the arithmetic, sets the pace of this fold, and P.V of
        // the next tile waits for the last O_tile load)
#pragma unroll
        for (int c = 0; c < HD / 32; ++c) {
          uint32_t t[2][16], o[2][16];
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            tmem_ld16_async(o_tile + 32 * c + 16 * u, t[u]);
            tmem_ld16_async(o_run + 32 * c + 16 * u, o[u]);
          }
          tmem_wait_ld();
          if (c == HD / 32 - 1) {  // all of O_tile has been read: P.V of the next tile may overwrite it
            tc_fence_before();
            mbar_arrive(&bars->o_free);
          }
#pragma unroll
          for (int u = 0; u < 2; ++u) {
#pragma unroll
            for (int i = 0; i < 16; i += 2) {
              const float2 r = ffma2(make_float2(__uint_as_float(o[u][i]), __uint_as_float(o[u][i + 1])), a2,
                                     make_float2(__uint_as_float(t[u][i]), __uint_as_float(t[u][i + 1])));
              o[u][i] = __float_as_uint(r.x);
              o[u][i + 1] = __float_as_uint(r.y);
            }
            tmem_st16(o_run + 32 * c + 16 * u, o[u]);
          }
        }
      }
    } else {
      for (int j = 1; j < nkv && ok; ++j) {
        if (!wait_all(&bars->o_full, (j - 1) & 1)) break;  // P.V of tile j - 1 has landed in O
        tc_fence_after();
        const float rs = row_sum(j - 1);
        if (!wait_all(&bars->a_full[j & 3], (j >> 2) & 1)) break;
        const float alpha = alpha_s[(j & 3) * TQ + row];
        l = (l + rs) * alpha;
        if (!__all_sync(0xffffffffu, alpha == 1.f)) {  // exact when skipped
#pragma unroll 4
          for (int c = 0; c < HD / 16; ++c) {
            uint32_t o[16];
            tmem_ld16_async(o_tile + 16 * c, o);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 16; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            tmem_st16(o_tile + 16 * c, o);
          }
          tmem_wait_st();
        }
        tc_fence_before();
        mbar_arrive(&bars->o_free);  // P.V of tile j may add into O
      }
      if (nkv >= 1 && wait_all(&bars->o_full, (nkv - 1) & 1)) {
        tc_fence_after();
        l += row_sum(nkv - 1);
      }
    }
    if (ok) {
      // out = O * v_scale / l (both in units of 2^8 p); PT: O_run is in units
      // of the last tile's C, and the V scales are inside it
      const float lt = l;
      const bool live_row = job.q0 + row < job.nq;
      const size_t out_row = (static_cast<size_t>(p.cu_seqlens_q[job.b]) + job.q0 + row) * p.Hq + job.h;
      const float f = (lt > 0.f) ? (PT ? c_prev : p.v_scale[job.kvh]) / lt : 0.f;
      tmem_wait_st();
      const uint32_t o_out = SL ? o_tile : o_run;
      uint4* dst = reinterpret_cast<uint4*>(p.out + out_row * HD);
#pragma unroll 2
      for (int c = 0; c < HD / 32; ++c) {
        uint32_t o[32];
        tmem_ld32(o_out + 32 * c, o);
        if (live_row) {
#pragma unroll
          for (int w = 0; w < 4; ++w) {
            uint4 u;
            u.x = pack_bf16x2(__uint_as_float(o[8 * w + 0]) * f, __uint_as_float(o[8 * w + 1]) * f);
            u.y = pack_bf16x2(__uint_as_float(o[8 * w + 2]) * f, __uint_as_float(o[8 * w + 3]) * f);
            u.z = pack_bf16x2(__uint_as_float(o[8 * w + 4]) * f, __uint_as_float(o[8 * w + 5]) * f);
            u.w = pack_bf16x2(__uint_as_float(o[8 * w + 6]) * f, __uint_as_float(o[8 * w + 7]) * f);
            dst[4 * c + w] = u;
          }
        }
      }
    }
  } else {
    setmaxnreg_inc<REG_SOFT>();
    // ------------------------------------------------------ softmax warps --
    const int part = warp >> 2;            // columns part*HC .. +HC-1 of S
    const int quarter = warp & 3;          // TMEM lanes 32*quarter .. +31
    const uint32_t t_lane = static_cast<uint32_t>(quarter * 32) << 16;
    const int row = quarter * 32 + lane;   // TMEM lane == query row
    constexpr int HC = TK / NPART;         // columns per thread
    float* xmax = reinterpret_cast<float*>(smem + OFF_XCH);   // [2 tiles][NPART][TQ]
    const bool live_row = job.q0 + row < job.nq;
    const int qpos = job.first_q + job.q0 + row;  // absolute position of this query
    const int kend = (p.causal && qpos + 1 < job.L) ? qpos + 1 : job.L;  // this row attends to keys [0, kend)
    const size_t out_row = (static_cast<size_t>(p.cu_seqlens_q[job.b]) + job.q0 + row) * p.Hq + job.h;

    // Q row (this thread's part) -> shared memory, 128-byte swizzled planes
    {
      const uint4* src = reinterpret_cast<const uint4*>(p.q8 + out_row * HD);
#pragma unroll
      for (int cc = 0; cc < HD / 16 / NPART; ++cc) {
        const int c = part * (HD / 16 / NPART) + cc;  // 16-byte chunk of the row
        const uint4 v = live_row ? __ldg(src + c) : make_uint4(0, 0, 0, 0);
        uint8_t* qs = smem + OFF_Q + (c >> 3) * G::PLANE_Q + row * PLANE;
        *reinterpret_cast<uint4*>(qs + (((c & 7) ^ (row & 7)) << 4)) = v;
      }
      fence_proxy_async_smem();
      mbar_arrive(&bars->q_full);
    }
    // PT: the K scales multiply each score before the maximum (c_j = fl32(sk_j *
    // bcoef)), and the exponent takes the scores as they are
    const float bcoef = __fmul_rn(__fmul_rn(*p.q_scale, p.sm_scale), kLog2e);
    const float coef =
        PT ? 1.f : __fmul_rn(__fmul_rn(__fmul_rn(*p.q_scale, p.k_scale[job.kvh]), p.sm_scale), kLog2e);
    float* ct_s = reinterpret_cast<float*>(smem + G::OFF_CT);  // PT: [4] C_j for the correction warps
    float* xv = ct_s + 4;                                       // PT: [2 tiles][NPART] largest V scales
    const int tail = job.L % kPage;          // valid tokens in the last page (0 = full)
    const int last_page = (job.L - 1) / kPage;

    float* alpha_s = reinterpret_cast<float*>(smem + G::OFF_ALPHA);  // [4][TQ], read by the correction warps
    // m: the running row maximum of the raw scores; M: the stabilizer, the
    // maximum of the base-2 scores rounded up to an integer, so that every
    // rescale 2^(M_old - M_new) is an exact power of two and the P8 codes do
    // not depend on how the keys are tiled (E4M3 rounding commutes with it)
    float m = -INFINITY, M = -INFINITY;
    bool ok = true;  // warp-uniform, since tcgen05.ld / st need every lane of the warp
    auto wait_all = [&](uint64_t* bar, uint32_t parity) {
      if (!ok) return false;
      const bool got = mbar_wait(bar, parity, abort_flag);
      if (!__all_sync(0xffffffffu, got)) {
        ok = false;
        set_status(p.dev_status, KVQ_DEV_TIMEOUT);
        *abort_flag = 1;
      }
      return ok;
    };

    if (!__all_sync(0xffffffffu, stall_wait(&bars->stall, p.stall_ns, abort_flag))) {
      ok = false;
      set_status(p.dev_status, KVQ_DEV_TIMEOUT);
      *abort_flag = 1;
    }
    // every softmax thread runs every tile's named barrier, also after a
    // failed wait, so no warp is left behind at bar.sync
    for (int j = 0; j < nkv; ++j) {
      const int st = j % NKV;
      const int key0 = j * TK + part * HC;
      const uint32_t sbuf = tmem + t_lane + (j & 1) * TK + part * HC;  // this thread's columns of S_j
      const bool tail_tile = tail != 0 && last_page / (TK / kPage) == j;  // holds the partial last page
      float sv[HC];
      float mx = -INFINITY;
      float vmx = 0.f;  // PT: the largest V scale of this thread's cached keys
      uint32_t bad = 0;  // pages of the tile with an invalid block id (zero-filled)
      // S_j; then the stage's barrier for the tile's page flags -- split: k_full,
      // which cannot move on before every softmax thread has passed this wait
      // (the softmax's arrive on k_empty below); combined: v_full -- and, split,
      // V_j where the last page's unused V slots are zeroed here
      if (wait_all(&bars->s_full[j & 1], (j >> 1) & 1) &&
          wait_all(SPLIT ? &bars->k_full[st] : &bars->v_full[st], (j / NKV) & 1) &&
          (!SPLIT || !tail_tile || wait_all(&bars->v_full[st], (j / NKV) & 1))) {
        tc_fence_after();
        bad = bars->tile_bad[j & 7];
        if (tail_tile) {
          // V rows (dims) row and row + 128 .. of the last page: slots past the sequence end
          for (int d = row + part * TQ; d < HD; d += NPART * TQ) {
            uint8_t* vrow = smem + OFF_KV + st * STAGE_B + TILE_B + (last_page % (TK / kPage)) * VPAGE_B + d * kPage;
            for (int t = tail; t < kPage; ++t) vrow[fp8_v_slot(t)] = 0;
          }
        }
        const bool need_mask = (key0 + HC > kend) || bad != 0;
        // raw scores (the positive scale is applied in the exponent below)
        {  // all 32-column loads in flight, one wait
          static_assert(HC % 32 == 0, "32-column loads");
          uint32_t v[HC / 32][32];
#pragma unroll
          for (int c = 0; c < HC / 32; ++c) tmem_ld32_nowait(sbuf + 32 * c, v[c]);
          tmem_wait_ld();
#pragma unroll
          for (int c = 0; c < HC / 32; ++c) {
            tmem_pin32(v[c]);
#pragma unroll
            for (int i = 0; i < 32; ++i) sv[32 * c + i] = __uint_as_float(v[c][i]);
          }
        }
        if constexpr (PT) {
          // the scale tails of this thread's pages: K scales scale the scores; the
          // largest V scale of the thread's cached keys goes to the exchange
          float vm = 0.f;
#pragma unroll
          for (int pg = 0; pg < HC / kPage; ++pg) {
            const float4* tl = reinterpret_cast<const float4*>(smem + OFF_KV + st * STAGE_B + TILE_B +
                                                               (part * (HC / kPage) + pg) * VPAGE_B + PAGE_B);
#pragma unroll
            for (int i4 = 0; i4 < 4; ++i4) {
              const float4 ks4 = tl[i4], vs4 = tl[4 + i4];
              const float kk[4] = {ks4.x, ks4.y, ks4.z, ks4.w}, vv[4] = {vs4.x, vs4.y, vs4.z, vs4.w};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int k = pg * 16 + 4 * i4 + e;
                sv[k] = __fmul_rn(sv[k], __fmul_rn(kk[e], bcoef));
                const bool cached = !tail_tile || key0 + k < job.L;  // slots past the end hold no scale
                vm = fmaxf(vm, cached ? vv[e] : 0.f);
              }
            }
          }
          vmx = vm;
        }
        if (need_mask) {  // last tiles only; static indices keep sv in registers
          const int lim = kend - key0;  // columns k < lim are causally visible
          const uint32_t badh = bad >> (part * (HC / kPage));
#pragma unroll
          for (int k = 0; k < HC; ++k)
            sv[k] = (k >= lim || ((badh >> (k / kPage)) & 1)) ? -INFINITY : sv[k];
        }
        // row maximum as a tree of three-input maxima, not a long chain
        static_assert(HC == 64 || HC == 32, "the max trees below cover 64 or 32 columns");
        if constexpr (HC == 64) {
          float m1[22], m2[8];
#pragma unroll
          for (int i = 0; i < 21; ++i) m1[i] = fmax3(sv[3 * i], sv[3 * i + 1], sv[3 * i + 2]);
          m1[21] = sv[63];
#pragma unroll
          for (int i = 0; i < 7; ++i) m2[i] = fmax3(m1[3 * i], m1[3 * i + 1], m1[3 * i + 2]);
          m2[7] = m1[21];
          mx = fmax3(fmax3(m2[0], m2[1], m2[2]), fmax3(m2[3], m2[4], m2[5]), fmaxf(m2[6], m2[7]));
        } else {
          float m1[11], m2[4];
#pragma unroll
          for (int i = 0; i < 10; ++i) m1[i] = fmax3(sv[3 * i], sv[3 * i + 1], sv[3 * i + 2]);
          m1[10] = fmaxf(sv[30], sv[31]);
#pragma unroll
          for (int i = 0; i < 3; ++i) m2[i] = fmax3(m1[3 * i], m1[3 * i + 1], m1[3 * i + 2]);
          m2[3] = fmaxf(m1[9], m1[10]);
          mx = fmax3(m2[0], m2[1], fmaxf(m2[2], m2[3]));
        }
      }
      xmax[((j & 1) * NPART + part) * TQ + row] = mx;
      if (PT && row == 0) xv[(j & 1) * NPART + part] = vmx;
      named_bar_sync(1, NSOFT * 32);
      // split: every softmax thread has read the tile's page flags and passed
      // k_full: the K half of the stage may be refilled once S_j is computed
      if (SPLIT && threadIdx.x == 0) mbar_arrive(&bars->k_empty[st]);
      if (ok) {
        // m and the maxima are raw scores; 2^(s - M) * 256 = 2^(raw * coef - (M - 8)),
        // the largest in (128, 256]
        float m_new = m;
#pragma unroll
        for (int pt = 0; pt < NPART; ++pt) m_new = fmaxf(m_new, xmax[((j & 1) * NPART + pt) * TQ + row]);
        const float M_new = (m_new == -INFINITY) ? -INFINITY : ceilf(m_new * coef);
        const float nb = (m_new == -INFINITY) ? 0.f : 8.f - M_new;
        const float alpha = exp2_int(M - M_new);  // 0 on the first tile
        // PT: C_j = 2^ceil(log2 max sv) over the tile's cached keys (1 if none)
        float c_inv = 1.f;
        if constexpr (PT) {
          float vmax = 0.f;
#pragma unroll
          for (int pt = 0; pt < NPART; ++pt) vmax = fmaxf(vmax, xv[(j & 1) * NPART + pt]);
          const uint32_t bits = __float_as_uint(vmax);
          int e = static_cast<int>(bits >> 23) - 127 + ((bits & 0x7FFFFFu) != 0u ? 1 : 0);
          e = vmax > 0.f ? (e < -126 ? -126 : e) : 0;
          c_inv = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);  // 2^-e, exact
          if (row == 0 && part == 0) ct_s[j & 3] = __uint_as_float(static_cast<uint32_t>(127 + e) << 23);
        }
        if (part == 0) {  // for the correction warps
          alpha_s[(j & 3) * TQ + row] = alpha;
          mbar_arrive(&bars->a_full[j & 3]);
        }
        const float2 coef2 = make_float2(coef, coef), nb2 = make_float2(nb, nb);
        uint32_t pw[4 * (HC / kPage)];           // this thread's P8 words (four keys each); PT: weighted
        uint32_t pu[PT ? 4 * (HC / kPage) : 1];  // PT: the unweighted words, for the row sums
#pragma unroll
        for (int pg = 0; pg < HC / kPage; ++pg) {  // pages of 16 keys
          float q[16];
#pragma unroll
          for (int t = 0; t < 16; t += 2) {
            const float2 e = ffma2(make_float2(sv[pg * 16 + t], sv[pg * 16 + t + 1]), coef2, nb2);
            q[t] = ex2(e.x);
            q[t + 1] = ex2(e.y);
          }
          // word w of a page holds keys 2w, 2w+1, 2w+8, 2w+9 (the V slot order)
          auto words = [&](const float (&x)[16], uint32_t* out4) {
#pragma unroll
            for (int ww = 0; ww < 4; ++ww)
              out4[ww] =
                  f32x2_to_e4m3x2(x[2 * ww], x[2 * ww + 1]) | (f32x2_to_e4m3x2(x[2 * ww + 8], x[2 * ww + 9]) << 16);
          };
          if constexpr (PT) {
            words(q, &pu[4 * pg]);
            const float4* tl = reinterpret_cast<const float4*>(smem + OFF_KV + st * STAGE_B + TILE_B +
                                                               (part * (HC / kPage) + pg) * VPAGE_B + PAGE_B);
            float qw[16];
#pragma unroll
            for (int i4 = 0; i4 < 4; ++i4) {
              const float4 vs4 = tl[4 + i4];
              const float vv[4] = {vs4.x, vs4.y, vs4.z, vs4.w};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int t = 4 * i4 + e;
                // sv / C_j is exact; slots past the sequence end hold no scale
                const float w = (tail_tile && key0 + pg * 16 + t >= job.L) ? 0.f : vv[e] * c_inv;
                qw[t] = __fmul_rn(q[t], w);
              }
            }
            words(qw, &pw[4 * pg]);
          } else {
            words(q, &pw[4 * pg]);
          }
        }
        m = m_new;
        M = M_new;
        tmem_st16(sbuf, pw);  // over the first 16 of this thread's 64 columns of S_j
        if constexpr (PT) tmem_st16(sbuf + 16, pu);  // the unweighted codes next to them
        tmem_wait_st();
        if (tail_tile) fence_proxy_async_smem();  // the zeroed V slots, before the tensor cores read them
        tc_fence_before();
        mbar_arrive(&bars->p_full[j & 1]);
      }
    }
    // the correction warps hold the row sums and write the output rows
  }

  tc_fence_before();
  __syncthreads();
  if (warp == W_MMA) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS) : "memory");
  }
}

}  // namespace

}  // namespace kvq

using namespace kvq;

namespace {

template <int HD, bool SL, bool E5 = false, bool PT = false>
kvq_status_t launch_prefill(const PrefillParams& prm, dim3 grid, cudaStream_t stream) {
  constexpr int smem = Geo<HD, PT>::SMEM_BYTES;
  static int configured_mask = 0;  // devices whose shared-memory attribute is set
  int dev = 0;
  cudaGetDevice(&dev);
  if (!(configured_mask & (1 << (dev & 31)))) {
    cudaError_t e =
        cudaFuncSetAttribute(prefill_kernel<HD, SL, E5, PT>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return cuda_status(e, "prefill: set shared memory size");
    configured_mask |= 1 << (dev & 31);
  }
  prefill_kernel<HD, SL, E5, PT><<<grid, NTHREADS, smem, stream>>>(prm);
  return cuda_status(cudaGetLastError(), "prefill launch");
}

kvq_status_t prefill(const uint8_t* q8, const float* q_scale, const void* k_cache, const void* v_cache,
                     const float* k_scale, const float* v_scale, const int32_t* block_table,
                     const int32_t* cu_seqlens_q, const int32_t* seq_lens, void* out, int B, int Hq, int Hkv, int D,
                     int P, int max_blocks, int64_t num_blocks, int max_q_tokens, float sm_scale, int causal,
                     int* dev_status, kvq_stream_t stream, int accumulation,
                     kvq_dtype_t cache_dtype = KVQ_DTYPE_FP8_E4M3, bool per_token = false) {
  if (B < 1 || Hq < 1 || Hkv < 1 || max_blocks < 1 || num_blocks < 1 || max_q_tokens < 0)
    return fail(KVQ_ERR_INVALID_ARG, "prefill: bad sizes");
  if (Hq % Hkv != 0) return fail(KVQ_ERR_INVALID_ARG, "prefill: Hq %% Hkv != 0");
  if (!(sm_scale > 0.f) || !(sm_scale < FLT_MAX)) return fail(KVQ_ERR_INVALID_ARG, "prefill: bad sm_scale");
  if (P != kPage) return fail(KVQ_ERR_UNSUPPORTED, "prefill: page size %d (only 16)", P);
  if (D != 128 && D != 256) return fail(KVQ_ERR_UNSUPPORTED, "prefill: head_dim %d (128 or 256)", D);
  // head_dim 256: single-level accumulation (two-level would need 2 x 256 TMEM
  // columns for O beside the score buffers); -1 = the default for the head dim
  if (D == 256 && accumulation == KVQ_ACC_TWO_LEVEL)
    return fail(KVQ_ERR_UNSUPPORTED, "prefill: head_dim 256 runs with single-level accumulation only");
  const bool single_level = D == 256 || accumulation == KVQ_ACC_SINGLE_LEVEL;
  if (cache_dtype != KVQ_DTYPE_FP8_E4M3 && cache_dtype != KVQ_DTYPE_FP8_E5M2)
    return fail(KVQ_ERR_UNSUPPORTED, "prefill: FP8 (E4M3 or E5M2) caches only");
  if (per_token && (D != 128 || single_level))
    return fail(KVQ_ERR_UNSUPPORTED, "prefill: per-token scales at head_dim 128 with two-level accumulation");
  if (max_q_tokens == 0) return KVQ_OK;
  if (!q8 || !q_scale || !k_cache || !v_cache || (!per_token && (!k_scale || !v_scale)) || !block_table ||
      !cu_seqlens_q || !seq_lens || !out)
    return fail(KVQ_ERR_INVALID_ARG, "prefill: null pointer");
  if (!aligned(q8, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16))
    return fail(KVQ_ERR_INVALID_ARG, "prefill: pointers must be 16-byte aligned");
  if (B > 65535 || (max_q_tokens + TQ - 1) / TQ > 65535) return fail(KVQ_ERR_UNSUPPORTED, "prefill: grid too large");
  PrefillParams prm;
  prm.q8 = q8;
  prm.q_scale = q_scale;
  prm.k_cache = static_cast<const uint8_t*>(k_cache);
  prm.v_cache = static_cast<const uint8_t*>(v_cache);
  prm.k_scale = k_scale;
  prm.v_scale = v_scale;
  prm.block_table = block_table;
  prm.cu_seqlens_q = cu_seqlens_q;
  prm.seq_lens = seq_lens;
  prm.out = static_cast<__nv_bfloat16*>(out);
  prm.B = B;
  prm.Hq = Hq;
  prm.Hkv = Hkv;
  prm.g = Hq / Hkv;
  prm.max_blocks = max_blocks;
  prm.num_blocks = num_blocks;
  prm.sm_scale = sm_scale;
  prm.causal = causal ? 1 : 0;
  prm.dev_status = dev_status;
  prm.stall_ns = stall_ns();
  {
    const int64_t page_b = static_cast<int64_t>(kPage) * D;
    const PageStrides ps = page_strides(k_cache, v_cache, page_b, page_b + (per_token ? kScaleTailBytes : 0));
    prm.k_str = ps.k;
    prm.v_str = ps.v;
  }
  dim3 grid(Hq, (max_q_tokens + TQ - 1) / TQ, B);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (per_token)
    return cache_dtype == KVQ_DTYPE_FP8_E5M2 ? launch_prefill<128, false, true, true>(prm, grid, st)
                                             : launch_prefill<128, false, false, true>(prm, grid, st);
  if (cache_dtype == KVQ_DTYPE_FP8_E5M2) {
    if (D == 256) return launch_prefill<256, true, true>(prm, grid, st);
    return single_level ? launch_prefill<128, true, true>(prm, grid, st)
                        : launch_prefill<128, false, true>(prm, grid, st);
  }
  if (D == 256) return launch_prefill<256, true>(prm, grid, st);
  return single_level ? launch_prefill<128, true>(prm, grid, st) : launch_prefill<128, false>(prm, grid, st);
}

}  // namespace

extern "C" kvq_status_t kvq_prefill_attention(const uint8_t* q8, const float* q_scale, const void* k_cache,
                                              const void* v_cache, const float* k_scale, const float* v_scale,
                                              const int32_t* block_table, const int32_t* cu_seqlens_q,
                                              const int32_t* seq_lens, void* out, int B, int Hq, int Hkv, int D,
                                              int P, int max_blocks, int64_t num_blocks, int max_q_tokens,
                                              float sm_scale, int causal, int* dev_status, kvq_stream_t stream) {
  clear_error();
  return prefill(q8, q_scale, k_cache, v_cache, k_scale, v_scale, block_table, cu_seqlens_q, seq_lens, out, B, Hq,
                 Hkv, D, P, max_blocks, num_blocks, max_q_tokens, sm_scale, causal, dev_status, stream, -1);
}

extern "C" kvq_status_t kvq_prefill_attention_dtype(const uint8_t* q8, const float* q_scale, const void* k_cache,
                                                    const void* v_cache, const float* k_scale, const float* v_scale,
                                                    const int32_t* block_table, const int32_t* cu_seqlens_q,
                                                    const int32_t* seq_lens, void* out, int B, int Hq, int Hkv,
                                                    int D, int P, int max_blocks, int64_t num_blocks,
                                                    int max_q_tokens, float sm_scale, int causal, int* dev_status,
                                                    kvq_stream_t stream, kvq_dtype_t cache_dtype) {
  clear_error();
  return prefill(q8, q_scale, k_cache, v_cache, k_scale, v_scale, block_table, cu_seqlens_q, seq_lens, out, B, Hq,
                 Hkv, D, P, max_blocks, num_blocks, max_q_tokens, sm_scale, causal, dev_status, stream, -1,
                 cache_dtype);
}

extern "C" kvq_status_t kvq_prefill_attention_acc(const uint8_t* q8, const float* q_scale, const void* k_cache,
                                                  const void* v_cache, const float* k_scale, const float* v_scale,
                                                  const int32_t* block_table, const int32_t* cu_seqlens_q,
                                                  const int32_t* seq_lens, void* out, int B, int Hq, int Hkv,
                                                  int D, int P, int max_blocks, int64_t num_blocks,
                                                  int max_q_tokens, float sm_scale, int causal, int* dev_status,
                                                  kvq_stream_t stream, kvq_accumulation_t accumulation) {
  clear_error();
  if (accumulation != KVQ_ACC_TWO_LEVEL && accumulation != KVQ_ACC_SINGLE_LEVEL)
    return fail(KVQ_ERR_INVALID_ARG, "prefill: bad accumulation mode");
  return prefill(q8, q_scale, k_cache, v_cache, k_scale, v_scale, block_table, cu_seqlens_q, seq_lens, out, B, Hq,
                 Hkv, D, P, max_blocks, num_blocks, max_q_tokens, sm_scale, causal, dev_status, stream,
                 static_cast<int>(accumulation));
}

extern "C" kvq_status_t kvq_prefill_attention_per_token(const uint8_t* q8, const float* q_scale, const void* k_cache,
                                                        const void* v_cache, const int32_t* block_table,
                                                        const int32_t* cu_seqlens_q, const int32_t* seq_lens,
                                                        void* out, int B, int Hq, int Hkv, int D, int P,
                                                        int max_blocks, int64_t num_blocks, int max_q_tokens,
                                                        float sm_scale, int causal, kvq_dtype_t cache_dtype,
                                                        int* dev_status, kvq_stream_t stream) {
  clear_error();
  return prefill(q8, q_scale, k_cache, v_cache, nullptr, nullptr, block_table, cu_seqlens_q, seq_lens, out, B, Hq,
                 Hkv, D, P, max_blocks, num_blocks, max_q_tokens, sm_scale, causal, dev_status, stream,
                 KVQ_ACC_TWO_LEVEL, cache_dtype, true);
}
