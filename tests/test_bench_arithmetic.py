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
