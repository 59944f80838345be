// kvq_prefill_attention: chunked causal prefill on FP8 tensor cores.
#include "kvq_device.cuh"
#include "kvq_host.h"

using namespace kvq;

extern "C" kvq_status_t kvq_prefill_attention(const uint8_t* q8, const float* q_scale, const void* k_cache,
                                              const void* v_cache, const float* k_scale, const float* v_scale,
                                              const int32_t* block_table, const int32_t* cu_seqlens_q,
                                              const int32_t* seq_lens, void* out, int B, int Hq, int Hkv, int D,
                                              int P, int max_blocks, int64_t num_blocks, int max_q_tokens,
                                              float sm_scale, int causal, int* dev_status, kvq_stream_t stream) {
  clear_error();
  return fail(KVQ_ERR_UNSUPPORTED, "prefill_attention: not built yet");
}
