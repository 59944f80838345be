/*
 * kvq.h -- C ABI of libkvq: FP8 (E4M3) KV-cache quantization and attention
 * over a paged FP8 (or BF16) KV cache, for NVIDIA GB300 (sm_103a).
 *
 * The operations follow the statement of the method on these pages:
 *  [vLLM]   "The state of FP8 KV-cache and attention quantization in vLLM"
 *           (vLLM blog, 2026-04-22): sections "Problems we found",
 *           "Kernel and vLLM improvements" (two-level accumulation, skip
 *           layers, per-head scales, query quantization fusion),
 *           "Performance benchmarks".
 *  [FP8KV]  "FP8 and KV cache" (cooking-agi tutorial): sections "Dynamic or
 *           static scale", "KV cache", "How to enable it in the engine".
 *  [GTNT]   "FP8 quantization and long-context inference" (gtnt.cn),
 *           section 1.1 (scale = max_abs / 448, q = round(x / scale)) and
 *           section 6 (PagedAttention).
 *
 * Conventions for every call
 *  - All tensor arguments are DEVICE pointers owned by the caller; the
 *    library never allocates, frees or keeps them.  Scales are device
 *    pointers too, so calls can be captured in a CUDA graph.
 *  - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *    stream) and runs asynchronously; a KVQ_OK return means "validated and
 *    launched".
 *  - Host-side validation (null pointers, sizes, alignment, unsupported
 *    shapes) happens before any launch; on failure nothing is launched, a
 *    status is returned and kvq_last_error_string() describes it.
 *  - Faults only the device can see (a block id outside [0, num_blocks), a
 *    cache slot beyond the cache, a sequence longer than its block table, a
 *    pipeline wait that timed out) OR a KVQ_DEV_* bit into *dev_status
 *    (a device int the caller zeroes and reads back) and skip the offending
 *    work; kernels never trap.  dev_status may be NULL to ignore them.
 *  - bf16 tensors are passed as raw 16-bit storage (void*).
 *
 * Cache format (both caches have num_blocks blocks of Hkv pages each; one
 * page holds P = 16 tokens of one KV head; token slot s is block s / P,
 * offset t = s % P, following PagedAttention):
 *  - K cache, element [block][h][t][d]: a page is P rows of D elements; the
 *    16-byte chunks of row t are stored XOR-swizzled so that the page can be
 *    copied to shared memory as one contiguous block and read without bank
 *    conflicts: with 128-byte rows chunk j sits at chunk j ^ (t % 8); with
 *    64-byte rows at j ^ ((t / 2) % 4); with 256-byte rows (BF16, D = 128)
 *    each 128-byte half is swizzled as a 128-byte row.  Row bytes = D * esize.
 *    FP8 at D = 256 (prefill): the page is two 2 KiB half-pages, half h
 *    holding dims 128h .. 128h + 127 of the 16 tokens as 128-byte rows
 *    swizzled as above (byte (j / 8) * 2048 + t * 128 + ((j % 8) ^ (t % 8)) *
 *    16 for chunk j of token t), so each half is a tensor-core operand.
 *  - V cache, element [block][h][d][slot]: the page transposed, one row of P
 *    token slots per dimension d.  FP8: token t occupies slot rho(t) with
 *    rho = {0,1,4,5,8,9,12,13,2,3,6,7,10,11,14,15} (tokens 2c,2c+1,2c+8,2c+9
 *    share the 4-byte word c).  BF16: slot = t, and the two 16-byte halves of
 *    row d are swapped when (d / 4) is odd.
 *  - FP8 elements are E4M3 ("OCP FN": bias 7, max 448, min subnormal 2^-9,
 *    0x7F/0xFF NaN, no infinity) or E5M2 (KVQ_DTYPE_FP8_E5M2).  Page bytes =
 *    P * D * esize.
 *  - Separate or paired.  Two separate allocations [num_blocks][Hkv][K page]
 *    and [num_blocks][Hkv][V page], or one paired allocation
 *    [num_blocks][Hkv][K page | V page]: each (block, KV head) pair's K page
 *    directly followed by its V page (with per-token scales, the V page with
 *    its scale tail).  Every entry point takes a paired cache as k_cache =
 *    the allocation and v_cache = k_cache + K page bytes, and recognizes the
 *    layout from exactly that pointer relation (both caches then advance by
 *    K page + V page bytes per pair).  Results are bit-identical between the
 *    two layouts; decode moves a paired page pair with one bulk copy instead
 *    of two.
 *
 * Quantization (kvq_reshape_and_cache, kvq_quantize_query):
 *    code = e4m3_rne_satfinite( fl32(x / scale) )
 *  one IEEE float32 division, then one round-to-nearest-even conversion that
 *  saturates to +-448 ([FP8KV] "Dynamic or static scale": 180 / s = 672
 *  saturates to 448).  Dequantized value = decode(code) * scale.
 */
#ifndef KVQ_H
#define KVQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum kvq_status {
  KVQ_OK = 0,
  KVQ_ERR_INVALID_ARG = 1,   /* null pointer, bad size, misaligned pointer */
  KVQ_ERR_UNSUPPORTED = 2,   /* valid but not implemented (head_dim, page size, GQA ratio) */
  KVQ_ERR_CUDA = 3,          /* a CUDA runtime call failed (launch, attribute query) */
  KVQ_ERR_DEVICE_FAULT = 4   /* reserved for callers that fold *dev_status into a status */
} kvq_status_t;

typedef enum kvq_dtype {
  KVQ_DTYPE_FP8_E4M3 = 0,    /* 1-byte E4M3 codes with per-KV-head scales */
  KVQ_DTYPE_BF16 = 1,        /* unquantized bfloat16 ("skip layers") */
  KVQ_DTYPE_FP8_E5M2 = 2     /* 1-byte E5M2 codes with per-KV-head scales:
                                [FP8KV] "How to enable it in the engine" lists
                                fp8_e5m2 among the cache dtypes; [GTNT] section
                                1: 5 exponent bits, 2 mantissa bits, about
                                +-57344.  Bias 15, RNE, saturating to +-57344.
                                Prefill reads it through
                                kvq_prefill_attention_dtype. */
} kvq_dtype_t;

/*
 * How attention sums P.V over the keys.
 * [vLLM] "Problems we found" / "Kernel and vLLM improvements": FP8 tensor
 * cores can keep partial sums in less than FP32, which degrades long
 * contexts; two-level accumulation adds each tile's P.V, computed into a
 * fresh FP32 accumulator, into a running FP32 sum.  [FP8KV] training
 * section, "accumulation precision": DeepSeek-V3 promotes partial sums to
 * FP32 every 128 elements after measuring about 14 bits on H800.
 */
typedef enum kvq_accumulation {
  KVQ_ACC_TWO_LEVEL = 0,     /* the default of every call without an _acc suffix */
  KVQ_ACC_SINGLE_LEVEL = 1   /* ablation: the tensor cores add each tile into the
                                running sum themselves (rescaled by the online
                                softmax in place); E4M3 per-head caches only */
} kvq_accumulation_t;

/* Bits OR-ed into *dev_status by the kernels. */
#define KVQ_DEV_BAD_SLOT     0x1  /* slot >= num_blocks * P, or (append) not the last token's slot: not written */
#define KVQ_DEV_BAD_BLOCK    0x2  /* block id outside [0, num_blocks): page masked out */
#define KVQ_DEV_BAD_SEQLEN   0x4  /* seq_len < 0 or > max_blocks * P: clamped */
#define KVQ_DEV_TIMEOUT      0x8  /* a pipeline wait exceeded its bound: work abandoned */
#define KVQ_DEV_BAD_QROWS    0x10 /* prefill: new tokens exceed seq_len: rows skipped */

typedef void* kvq_stream_t;   /* cudaStream_t */

/* Library version (major * 10000 + minor * 100 + patch). */
int kvq_version(void);

/*
 * kvq_debug_set_stall_ns -- a test hook for the failure path of the bounded
 * pipeline waits (the pages have no counterpart; it exists so that the path
 * a stuck wait takes can be run without faulting or hanging a GPU).
 *
 * With ns > 0, every decode-partial and prefill kernel launched afterwards
 * (on any thread) makes one of its waits -- consumer warp 0 of each decode
 * CTA before its first stage; the softmax warps of each prefill CTA before
 * the first key tile -- a wait of at most ns nanoseconds on a barrier that
 * nothing arrives on.  It fails like any pipeline wait that exceeded its
 * bound: the kernel ORs KVQ_DEV_TIMEOUT into *dev_status, abandons its work
 * (the outputs are then meaningless), lets every bulk copy it issued land,
 * frees its tensor memory and returns; the context stays usable.  ns = 0
 * (the default) turns the hook off.  The setting is read at launch time, so
 * graphs captured while it was set keep it.
 */
void kvq_debug_set_stall_ns(uint64_t ns);

/* Text of the last host-side error on the calling thread ("" if none). */
const char* kvq_last_error_string(void);

/*
 * kvq_reshape_and_cache -- quantize new K/V tokens into the paged cache.
 * [vLLM] "Kernel and vLLM improvements", per-head scales: the cache-write
 * kernel takes an array of scales, one per KV head.  [FP8KV] "How to enable
 * it in the engine": scales per tensor or per head; uncalibrated = 1.0.
 *
 *  k, v          bf16 [T][Hkv][D], row-major, contiguous.
 *  slot_mapping  int64 [T]: cache slot of each token; a negative slot skips
 *                the token; a slot >= num_blocks * P sets KVQ_DEV_BAD_SLOT.
 *  k_cache       [num_blocks][Hkv][P][D] in the format above (written).
 *  v_cache       [num_blocks][Hkv][D][P] in the format above (written).
 *  k_scale,      float32 [Hkv] per-KV-head scales (FP8 only; may be NULL for
 *  v_scale       BF16).  Must be finite and > 0.
 *  T >= 0 (T == 0 launches nothing), Hkv >= 1, D in {64, 128} (and 256 for
 *  FP8 caches, which only kvq_prefill_attention reads), P == 16,
 *  num_blocks >= 1.  For BF16 the values are copied bit for bit.  FP8:
 *  code = encode(fl32(x / s[h])), one float32 division, then one
 *  round-to-nearest-even conversion saturating at the format's largest
 *  finite value (448 for E4M3, 57344 for E5M2).
 *  Only the bytes of the given slots are written; everything else in the
 *  caches is left as it was.  Slots must be distinct within one call.
 */
kvq_status_t kvq_reshape_and_cache(const void* k, const void* v, const int64_t* slot_mapping,
                                   void* k_cache, void* v_cache,
                                   const float* k_scale, const float* v_scale,
                                   int T, int Hkv, int D, int P, int64_t num_blocks,
                                   kvq_dtype_t cache_dtype, int* dev_status, kvq_stream_t stream);

/*
 * kvq_quantize_query -- per-tensor query quantization to E4M3.
 * [vLLM] "Kernel and vLLM improvements", query quantization fusion;
 * [FP8KV] "How to enable it in the engine": with FP8 attention the query is
 * quantized to FP8 too; one scale per tensor for Q.
 *
 *  q        bf16 [n] (any shape, contiguous).
 *  q8       uint8 [n] E4M3 codes (written).
 *  q_scale  float32 [1], finite and > 0.
 *  n >= 0; pointers 16-byte aligned when n > 0.
 */
kvq_status_t kvq_quantize_query(const void* q, uint8_t* q8, const float* q_scale, int64_t n,
                                kvq_stream_t stream);

/*
 * Split-KV plan for kvq_paged_decode_attention.  num_splits = 0 asks for the
 * library's choice for this GPU (one wave of resident CTAs: 3 per SM, 4 at
 * head dim D = 64; at least 4 pages per split; 1 split for at most 8 pages,
 * or at most 16 pages over 32 or more (sequence, KV head) pairs); the
 * function returns the number of splits that a call with the same arguments
 * will use (>= 1), or 0 on bad input.
 */
int kvq_decode_num_splits(int B, int Hkv, int D, int P, int max_blocks, int window, int num_splits);

/* Workspace bytes a decode call with these arguments needs (float32
 * partial outputs [B][Hq][S][4][D] and log-sum-exps [B][Hq][S][4]: one per
 * consumer warp of each of the S page ranges; for 2 to 32 sequences and
 * S > 1, [Hq][B * S + B - 1][4] partials, the ragged-batch plan's). */
size_t kvq_decode_workspace_size(int B, int Hq, int Hkv, int D, int P, int max_blocks,
                                 int window, int num_splits);

/*
 * kvq_paged_decode_attention -- one decode step of softmax(q K^T * sm_scale) V
 * over the paged cache, read directly in FP8 (or BF16).
 * [vLLM] "Performance benchmarks" (the decode cost is the per-token KV read,
 * the ITL slope), "Problems we found" / "Kernel and vLLM improvements"
 * (two-level FP32 accumulation: the P.V contraction runs over the context;
 * partial sums are promoted into real FP32 registers), "Skip layers"
 * (sliding-window layers keep a BF16 cache).
 *
 * Split-KV: each (sequence, KV head) is cut into num_splits ranges of pages;
 * a partial kernel writes per range (and per consumer warp within it, each
 * warp taking every fourth pair of pages) a normalized output and a
 * log-sum-exp to the workspace, and a combine kernel merges them (with one
 * range per sequence and KV head, all within one wave of the GPU, the
 * partial kernel merges its warps in shared memory and writes the output
 * itself):
 *   lse = log sum_i exp(lse_i),  out = sum_i exp(lse_i - lse) out_i.
 * Ragged batches (E4M3 cache, per-head scales, D = 128, 2 to 32 sequences,
 * S = num_splits > 1): per KV head the batch's attended pages are laid end
 * to end and cut into min(B * S, pages) equal slots instead, so that a long
 * sequence gets more ranges than a short one; a slot's part inside each
 * sequence it covers is merged like a range.  The plan is a function of
 * seq_lens alone: results are deterministic.
 * Both kernels are programmatic dependent launches: their launch and setup
 * overlap the preceding kernel on the stream, and neither reads anything it
 * uses from global memory before that kernel has completed (before it, the
 * partial kernel only hints L2 with its first pages).  A grid smaller than the GPU's
 * resident capacity asks for more shared memory per CTA than it uses, so
 * that its CTAs spread over the SMs; the combine's CTAs have as many warps
 * as the partials of a row need.
 * Accumulation: scores and P.V products are accumulated by tensor-core MMAs
 * into fresh FP32 registers per page of 16 tokens, then added into a running
 * FP32 sum (first level), and ranges are merged in FP32 (second level).
 *
 *  q            bf16 [B][Hq][D].  Query head h reads KV head h / (Hq / Hkv).
 *  k_cache,     the caches written by kvq_reshape_and_cache.
 *  v_cache
 *  k_scale,     float32 [Hkv] (FP8; ignored for BF16, may be NULL).
 *  v_scale
 *  block_table  int32 [B][max_blocks]: block id of each page of a sequence.
 *  seq_lens     int32 [B]: tokens in each sequence's cache (including the
 *               current token); 0 gives an all-zero output.
 *  out          bf16 [B][Hq][D] (written).
 *  window       -1 = full attention; W > 0 = the last W tokens
 *               [max(0, L - W), L) only (sliding-window layers).
 *  num_splits   0 = automatic, else the number of page ranges (>= 1).
 *  workspace    device buffer of kvq_decode_workspace_size(...) bytes,
 *               16-byte aligned, owned by the caller; contents on entry are
 *               ignored; calls sharing a workspace must not overlap.
 *  Supported: D in {64, 128}, P == 16, Hq % Hkv == 0, Hq / Hkv <= 8.
 *  Declared rounding: FP8 -- the K and V codes (E4M3 or E5M2) are converted
 *  to float16 in registers (exact) and both contractions run on float16
 *  MMAs with FP32 accumulation; per query head, sigma = 2^(7 - floor(log2
 *  max_d |q_d|)) and the query enters as qf = f16(fl32(q * sigma)) (RNE:
 *  exact for bf16 queries except elements that fall below float16's normal
 *  range, under 2^-21 of the head's maximum); scores s2 = fl32(sum_d qf_d
 *  k8_d) * c / sigma with c = fl32(fl32(k_scale * sm_scale) * log2(e));
 *  probabilities 2^(s2 - m) * 2^8 are rounded to float16 (11 significant
 *  bits) for the P.V MMA; the result is multiplied by v_scale.  BF16 -- scores use
 *  q and k exactly, c = fl32(sm_scale * log2(e)); probabilities are fed to
 *  the P.V MMA as the sum of two bfloat16 terms.  The output is rounded to
 *  bf16 once, at the end.
 */
kvq_status_t kvq_paged_decode_attention(const void* q, const void* k_cache, const void* v_cache,
                                        const float* k_scale, const float* v_scale,
                                        const int32_t* block_table, const int32_t* seq_lens,
                                        void* out, int B, int Hq, int Hkv, int D, int P,
                                        int max_blocks, int64_t num_blocks, float sm_scale,
                                        int window, kvq_dtype_t cache_dtype, int num_splits,
                                        void* workspace, size_t workspace_bytes,
                                        int* dev_status, kvq_stream_t stream);

/*
 * kvq_paged_decode_attention_append -- one decode step with the step's new
 * token written into the cache by the attention call itself: the result,
 * the cache bytes and the device status are those of kvq_reshape_and_cache
 * (one token per sequence, slot_mapping = slot_new) followed by
 * kvq_paged_decode_attention, in one launch of the partial kernel instead of
 * a separate cache-write kernel.  [vLLM] "Performance benchmarks" (a decode
 * step writes the new token and reads the whole context).
 *
 *  k_new, v_new  bf16 [B][Hkv][D]: the new token of each sequence, the last
 *                of its seq_lens[b] tokens.
 *  slot_new      int64 [B]: its cache slot (block * P + offset); -1 = no
 *                write; >= num_blocks * P sets KVQ_DEV_BAD_SLOT (no write).
 *                A sequence with seq_lens[b] = 0 has no last token: nothing
 *                is written for it.
 *  k_cache,      written (the new tokens' slots) and read.
 *  v_cache
 *  Other arguments as for kvq_paged_decode_attention.  The slot must be the
 *  last token's slot under block_table: block block_table[b][(L - 1) / P],
 *  offset (L - 1) % P (the page the call reads it back from); any other
 *  slot (or one in a page with an invalid block id) sets KVQ_DEV_BAD_SLOT
 *  and is not written.  Per-KV-head scales (FP8) or BF16 caches; two-level
 *  accumulation.
 */
kvq_status_t kvq_paged_decode_attention_append(const void* q, const void* k_new, const void* v_new,
                                               const int64_t* slot_new, void* k_cache, void* v_cache,
                                               const float* k_scale, const float* v_scale,
                                               const int32_t* block_table, const int32_t* seq_lens,
                                               void* out, int B, int Hq, int Hkv, int D, int P,
                                               int max_blocks, int64_t num_blocks, float sm_scale,
                                               int window, kvq_dtype_t cache_dtype, int num_splits,
                                               void* workspace, size_t workspace_bytes,
                                               int* dev_status, kvq_stream_t stream);

/*
 * kvq_paged_decode_attention_acc -- kvq_paged_decode_attention with an
 * explicit accumulation mode (kvq_accumulation_t above).  Two-level is the
 * call above; single-level feeds O * alpha to the P.V MMAs as their
 * accumulator input, so the tensor cores add each stage of 32 tokens into the
 * running sum.  Single-level: E4M3 cache, per-head scales only (else
 * KVQ_ERR_UNSUPPORTED).  It exists to measure what two-level costs and buys.
 */
kvq_status_t kvq_paged_decode_attention_acc(const void* q, const void* k_cache, const void* v_cache,
                                            const float* k_scale, const float* v_scale,
                                            const int32_t* block_table, const int32_t* seq_lens,
                                            void* out, int B, int Hq, int Hkv, int D, int P,
                                            int max_blocks, int64_t num_blocks, float sm_scale,
                                            int window, kvq_dtype_t cache_dtype, int num_splits,
                                            void* workspace, size_t workspace_bytes,
                                            int* dev_status, kvq_stream_t stream,
                                            kvq_accumulation_t accumulation);

/*
 * kvq_reshape_and_cache_per_token -- quantize new K/V tokens into the paged
 * cache with a dynamic scale per token and KV head.
 * [FP8KV] "Dynamic or static scale": with per-token scales each token's
 * largest value lands on the format's maximum (scales 3.2/448 and 180/448 in
 * the worked example), at the cost of one maximum per token; [GTNT] section
 * 2.2: per-token dynamic quantization computes a scale for every new token.
 *
 *  As kvq_reshape_and_cache (FP8 E4M3 or E5M2 only), except the V cache:
 *  v_cache   [num_blocks][Hkv] pages of P*D + 8*P bytes (written): the P x D
 *            codes in the V format above, then a scale tail of P K scales
 *            and P V scales, float32 -- tail[offset] is the K scale and
 *            tail[P + offset] the V scale of the token in slot offset,
 *            s = fl32(amax_d |x_d| / M) with M = 448 (E4M3) or 57344 (E5M2);
 *            a token whose values are all zero gets s = 1.  The scales ride
 *            on the V page so that decode fetches page and scales in one
 *            copy.  k_cache is as for kvq_reshape_and_cache.
 *  Each element is then code = encode(fl32(x / s)) as in
 *  kvq_reshape_and_cache.  Only the given slots' bytes and scales are
 *  written.
 */
kvq_status_t kvq_reshape_and_cache_per_token(const void* k, const void* v, const int64_t* slot_mapping,
                                             void* k_cache, void* v_cache, int T, int Hkv, int D, int P,
                                             int64_t num_blocks, kvq_dtype_t cache_dtype, int* dev_status,
                                             kvq_stream_t stream);

/*
 * kvq_paged_decode_attention_per_token -- kvq_paged_decode_attention over a
 * cache written by kvq_reshape_and_cache_per_token (same citations; the
 * per-token scales as above).
 *
 *  Arguments as for kvq_paged_decode_attention without k_scale and
 *  v_scale, with an FP8 (E4M3 or E5M2) cache in the per-token format (V
 *  pages of P*D + 8*P bytes, each with its scale tail).
 *  Declared rounding: the query terms and the per-head score coefficient as
 *  for kvq_paged_decode_attention with c = fl32(sm_scale * log2(e)); each
 *  score is then multiplied by its token's K scale.  V scales enter the
 *  probabilities: per stage of 32 tokens, with c = 2^ceil(log2 m), m the
 *  stage's largest V scale of a live token, and f a power of two per query
 *  head that moves the
 *  stage's largest weighted probability into [128, 256), P.V runs on
 *  p_j * (sv_j / c) * f, rounded to float16, and the stage's result is
 *  multiplied by c / f before it is added to the running FP32 sum.  The row sum uses the
 *  unweighted p_j.
 *  Workspace: kvq_decode_workspace_size() of the same arguments.
 */
kvq_status_t kvq_paged_decode_attention_per_token(const void* q, const void* k_cache, const void* v_cache,
                                                  const int32_t* block_table, const int32_t* seq_lens,
                                                  void* out, int B, int Hq, int Hkv, int D, int P,
                                                  int max_blocks, int64_t num_blocks, float sm_scale,
                                                  int window, kvq_dtype_t cache_dtype, int num_splits,
                                                  void* workspace, size_t workspace_bytes,
                                                  int* dev_status, kvq_stream_t stream);

/*
 * kvq_paged_decode_attention_static_scratch -- kvq_paged_decode_attention
 * for callers that cannot allocate device memory where they run decode (a
 * memory-pool policy that forbids new allocations, a real-time loop, a plugin
 * without access to its host engine's allocator).  The pages have no
 * counterpart: this entry point is about memory ownership only; the
 * computation, arguments and results are those of kvq_paged_decode_attention.
 *
 *  - The split-KV scratch lives in a fixed array of
 *    kvq_decode_static_scratch_bytes() bytes (4 MiB) inside the library's
 *    device image; every GPU that loads the library holds it until the
 *    process exits.  Nothing is allocated or freed by this call.
 *  - A call whose kvq_decode_workspace_size(...) exceeds the array returns
 *    KVQ_ERR_UNSUPPORTED and launches nothing.
 *  - The first call on each device looks up the array's device address
 *    (cudaGetSymbolAddress with that device current); make that first call
 *    before any stream capture on that device.  The address belongs to the
 *    CUDA context it was looked up in: a call made in another context on
 *    the device (after cudaDeviceReset, or with another context current)
 *    looks it up again, so that call too must come before any capture.
 *  - All calls on a device share the one array and it keeps the last call's
 *    contents.  Nothing in it needs to start at zero (each call writes every
 *    partial result before reading it), but calls that overlap on the GPU
 *    (different streams, or different host threads without ordering) race on
 *    it: order them on one stream.
 */
size_t kvq_decode_static_scratch_bytes(void);
kvq_status_t kvq_paged_decode_attention_static_scratch(const void* q, const void* k_cache, const void* v_cache,
                                                       const float* k_scale, const float* v_scale,
                                                       const int32_t* block_table, const int32_t* seq_lens,
                                                       void* out, int B, int Hq, int Hkv, int D, int P,
                                                       int max_blocks, int64_t num_blocks, float sm_scale,
                                                       int window, kvq_dtype_t cache_dtype, int num_splits,
                                                       int* dev_status, kvq_stream_t stream);

/*
 * kvq_prefill_attention -- chunked causal prefill over the FP8 cache on FP8
 * tensor cores.  [vLLM] "Kernel and vLLM improvements" (two-level
 * accumulation, prefill tile configurations), "Large head dimension
 * limitations" (two-level accumulation's cost in prefill); [FP8KV] "How to
 * enable it in the engine" (QK and score.V in FP8, query quantized to FP8).
 *
 * The new tokens must already be in the cache (kvq_reshape_and_cache).
 * Sequence b has nq_b = cu_seqlens_q[b+1] - cu_seqlens_q[b] new tokens, the
 * last nq_b of its L_b = seq_lens[b] cached tokens; query i of b sits at
 * position L_b - nq_b + i and attends to keys 0 .. L_b - nq_b + i (causal)
 * or to all L_b keys (causal = 0).
 *
 *  q8            uint8 [Tq][Hq][D] E4M3 codes (kvq_quantize_query), Tq =
 *                cu_seqlens_q[B].
 *  q_scale       float32 [1].
 *  k_cache, v_cache, k_scale, v_scale, block_table  as for decode (E4M3 caches;
 *                kvq_prefill_attention_dtype below reads E5M2 caches).
 *  cu_seqlens_q  int32 [B+1], non-decreasing, cu_seqlens_q[0] = 0.
 *  seq_lens      int32 [B].
 *  out           bf16 [Tq][Hq][D] (written).
 *  max_q_tokens  an upper bound of max_b nq_b (sizes the launch).
 *  Supported: D in {128, 256}, P == 16, Hq % Hkv == 0.  D = 256 runs with
 *  single-level accumulation (every tile's P8.V8 MMA adds into one
 *  tensor-memory sum rescaled in place): two-level would need two 256-column
 *  FP32 accumulators beside the score buffers, more than the 512 columns of
 *  tensor memory.
 *  Declared rounding: S = sum_d q8[d] k8[d] (exact products, FP32 sums),
 *  s2 = S * c with c = fl32(fl32(fl32(q_scale * k_scale) * sm_scale) *
 *  log2(e)); P8_j = e4m3_rne_sat(fl32(2^(s2_j - M) * 256)) with M the
 *  row's stabilizer, its maximum base-2 score rounded up to an integer
 *  (kept as a running value over the key tiles; every rescale 2^(M_old -
 *  M_new) is an exact power of two, with which E4M3 rounding commutes, so
 *  the result is that of the row's final M for any tiling, up to roundings
 *  of probabilities below 2^-14); out = v_scale * (sum_j P8_j V8_j) /
 *  (sum_j P8_j): the row sum adds the same rounded probabilities, summed by
 *  the tensor core.  Each KV tile's P8.V8 product goes into a fresh FP32
 *  tensor-memory accumulator that is then added in FP32 into the running
 *  output (two-level accumulation).
 */
kvq_status_t kvq_prefill_attention(const uint8_t* q8, const float* q_scale,
                                   const void* k_cache, const void* v_cache,
                                   const float* k_scale, const float* v_scale,
                                   const int32_t* block_table, const int32_t* cu_seqlens_q,
                                   const int32_t* seq_lens, void* out,
                                   int B, int Hq, int Hkv, int D, int P, int max_blocks,
                                   int64_t num_blocks, int max_q_tokens, float sm_scale,
                                   int causal, int* dev_status, kvq_stream_t stream);

/*
 * kvq_prefill_attention_dtype -- kvq_prefill_attention over a cache of the
 * given FP8 format: KVQ_DTYPE_FP8_E4M3 (the same as kvq_prefill_attention) or
 * KVQ_DTYPE_FP8_E5M2 ([FP8KV] "How to enable it in the engine": fp8_e5m2 is
 * one of the cache dtypes).  With E5M2 the K and V codes enter the tensor-core
 * products as E5M2 (the B operands of Q K^T and P.V); the query and P codes
 * stay E4M3; every other step and the declared rounding are those of
 * kvq_prefill_attention.  Any other dtype: KVQ_ERR_UNSUPPORTED.
 */
kvq_status_t kvq_prefill_attention_dtype(const uint8_t* q8, const float* q_scale,
                                         const void* k_cache, const void* v_cache,
                                         const float* k_scale, const float* v_scale,
                                         const int32_t* block_table, const int32_t* cu_seqlens_q,
                                         const int32_t* seq_lens, void* out,
                                         int B, int Hq, int Hkv, int D, int P, int max_blocks,
                                         int64_t num_blocks, int max_q_tokens, float sm_scale,
                                         int causal, int* dev_status, kvq_stream_t stream,
                                         kvq_dtype_t cache_dtype);

/*
 * kvq_prefill_attention_per_token -- kvq_prefill_attention over a cache
 * written by kvq_reshape_and_cache_per_token (V pages of P*D + 8*P bytes
 * with their scale tails).  [FP8KV] "Dynamic or static scale" (a scale per
 * token); [GTNT] section 2.2 (per-token dynamic scales for new tokens).
 *
 *  Arguments as for kvq_prefill_attention without k_scale and v_scale;
 *  cache_dtype KVQ_DTYPE_FP8_E4M3 or KVQ_DTYPE_FP8_E5M2; D = 128 (two-level
 *  accumulation).
 *  Declared rounding: per key, c_j = fl32(sk_j * b) with b = fl32(fl32(
 *  q_scale * sm_scale) * log2(e)) and s2_j = fl32(raw_j * c_j) (raw the
 *  FP32 dot product of the codes); M = ceil(max_j s2_j) as in
 *  kvq_prefill_attention.  The V scales run along the P.V contraction, so
 *  they enter the FP8 probabilities: per tile of 128 keys (aligned at key
 *  0), C = 2^ceil(log2 max sv_j) over the tile's cached keys and the P.V
 *  operand is e4m3(fl32(2^(s2_j - M + 8) * (sv_j / C))) (sv_j / C exact),
 *  while the row sum adds the unweighted codes e4m3(2^(s2_j - M + 8)); the
 *  tile's product is taken in units of C, and every rescale between tiles
 *  is a power of two.
 */
kvq_status_t kvq_prefill_attention_per_token(const uint8_t* q8, const float* q_scale,
                                             const void* k_cache, const void* v_cache,
                                             const int32_t* block_table, const int32_t* cu_seqlens_q,
                                             const int32_t* seq_lens, void* out,
                                             int B, int Hq, int Hkv, int D, int P, int max_blocks,
                                             int64_t num_blocks, int max_q_tokens, float sm_scale,
                                             int causal, kvq_dtype_t cache_dtype, int* dev_status,
                                             kvq_stream_t stream);

/*
 * kvq_prefill_attention_acc -- kvq_prefill_attention with an explicit
 * accumulation mode.  Single-level: every tile's P8.V8 MMA accumulates into
 * one tensor-memory sum, which is multiplied by alpha in place before the
 * next tile's MMA (skipped when alpha is 1 for all 32 rows of a warp, which
 * changes nothing).  It exists to measure what two-level costs and buys.
 */
kvq_status_t kvq_prefill_attention_acc(const uint8_t* q8, const float* q_scale,
                                       const void* k_cache, const void* v_cache,
                                       const float* k_scale, const float* v_scale,
                                       const int32_t* block_table, const int32_t* cu_seqlens_q,
                                       const int32_t* seq_lens, void* out,
                                       int B, int Hq, int Hkv, int D, int P, int max_blocks,
                                       int64_t num_blocks, int max_q_tokens, float sm_scale,
                                       int causal, int* dev_status, kvq_stream_t stream,
                                       kvq_accumulation_t accumulation);

#ifdef __cplusplus
}
#endif

#endif /* KVQ_H */
