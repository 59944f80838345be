"""The byte and FLOP counts behind bench.py's roofline, against closed forms
worked out independently: the Llama-3.1-8B-shaped decode layer at 131,072
tokens (32 query / 8 KV heads, head dim 128) and the chunked prefill of
4,096 new causal tokens on 28,672 cached."""
import bench


def test_decode_bytes_of_the_128k_layer():
    kv = 131072 * 8 * 128 * 2          # FP8 K and V, one byte per element
    scales = 8 * 2 * 4                 # one float32 K and one V scale per KV head
    q_out = 32 * 128 * 2 * 2           # bf16 q read and out written
    assert bench.decode_bytes(131072) == kv + scales + q_out == 268_451_904


def test_decode_bytes_scale_with_batch_and_context():
    assert bench.decode_bytes(2 * 4096, batch=1) - bench.decode_bytes(4096) == 4096 * 8 * 128 * 2
    assert bench.decode_bytes(4096, batch=2) == 2 * bench.decode_bytes(4096) - 8 * 2 * 4


def test_cache_write_bytes_of_one_token():
    # bf16 K and V in (2 x 2 bytes per element), FP8 K and V out (2 x 1 byte)
    assert bench.cache_write_bytes(1) == 8 * 128 * 6 == 6144


def test_prefill_flops():
    # query i (0-based) of the 4,096 new ones attends to 28,672 + i + 1 keys
    pairs = sum(28672 + i + 1 for i in range(4096))
    assert pairs == 125_831_168
    assert bench.prefill_flops() == pairs * 32 * 4 * 128
    assert abs(bench.prefill_flops() - 2.0616e12) / 2.0616e12 < 1e-4
    assert bench.prefill_flops(d=256) == 2 * bench.prefill_flops()


def test_whole_job_value():
    # weak scaling: every rank's bytes over the slowest rank's time
    assert bench.job_value(1, 1e9, 10, 1000.0) == 10.0
    assert bench.job_value(4, 1e9, 10, 1000.0) == 40.0


def test_tiny_config_bytes():
    # 512 tokens x 1 KV head x 64 dims, K and V at one byte; 2 float32 scales;
    # q and out: 4 query heads x 64 dims in bf16
    assert bench.decode_bytes_lengths([512], 4, 1, 64) == 2 * 512 * 64 + 2 * 4 + 2 * 4 * 64 * 2 == 66_568


def test_concurrency_8_bytes_from_the_seeded_lengths():
    import workloads as W
    lengths = W.decode_lengths(W.CONC8)
    assert len(lengths) == 8 and all(16384 <= L <= 24576 for L in lengths)
    assert lengths == W.decode_case(W.CONC8).seq_lens.tolist()  # the same draw as the parity case
    expect = 2 * sum(lengths) * 8 * 128 + 8 * 2 * 4 + 8 * 32 * 128 * 2 * 2
    assert bench.decode_bytes_lengths(lengths, 32, 8, 128) == expect


def test_hybrid_step_bytes():
    full_kv = 2 * 8 * 32768 * 8 * 64            # 268,435,456: batch 8, 8 KV heads, head_dim 64, FP8
    sw_kv = 2 * 8 * 128 * 8 * 64 * 2            # 2,097,152: the 128-token windows in bf16
    q_out = 2 * 8 * 64 * 64 * 2                 # 64 query heads, q and out in bf16
    step, full, sw = bench.hybrid_step_bytes()
    assert full == full_kv + 8 * 2 * 4 + q_out == 268_566_592
    assert sw == sw_kv + q_out == 2_228_224      # no scales for a BF16 cache
    assert step == 12 * (full + sw)
    assert abs(step - 3.2495e9) / 3.2495e9 < 1e-4


def test_head_sharded_step_bytes_per_rank_are_those_of_one_gpu():
    # rank r of N holds 8 / N KV heads (32 / N query heads) of N sequences
    one = bench.decode_bytes(131072)
    for n in (2, 4, 8):
        kv = 2 * n * 131072 * (8 // n) * 128
        assert bench.decode_bytes(131072, batch=n, hq=32 // n, hkv=8 // n) == kv + 2 * (8 // n) * 4 + 2 * n * (32 // n) * 128 * 2
        assert abs(bench.decode_bytes(131072, batch=n, hq=32 // n, hkv=8 // n) - one) <= 64
