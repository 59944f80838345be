"""GPU parity of the per-token dynamic-scale calls against the float64
oracle: kvq_reshape_and_cache_per_token bit-exact on every cache byte and
every scale in the V pages' scale tails (unwritten slots keep their sentinel
/ NaN), and
kvq_paged_decode_attention_per_token within the decode tolerance against
the mirrored and the pure oracle.  Scale slots that no token wrote are NaN,
so a scale read for a masked token would show up in the output."""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import attention, kv_cache, layout
from oracle.kv_cache import FP8, FP8_E5M2
from tests.kvq_testlib import SENTINEL, assert_close, f32

pytestmark = pytest.mark.gpu


def _k():
    import fp8_kv_cache_reshape_gb300 as k
    return k


def oracle_per_token_cache(case):
    cfg = case.cfg
    kc = np.full((case.num_blocks, cfg.kv_heads, 16, cfg.head_dim), SENTINEL, np.uint8)
    vc = np.full((case.num_blocks, cfg.kv_heads, cfg.head_dim, 16), SENTINEL, np.uint8)
    sc = np.full((case.num_blocks, cfg.kv_heads, 2, 16), np.nan, np.float32)
    kv_cache.reshape_and_cache_per_token(f32(case.k), f32(case.v), case.slot_mapping.numpy(), kc, vc, sc,
                                         case.cache_dtype)
    return kc, vc, sc


def gpu_per_token_cache(case):
    k = _k()
    cfg = case.cfg
    kd, vd = k.alloc_kv_cache(case.num_blocks, cfg.kv_heads, cfg.head_dim, case.cache_dtype, fill=SENTINEL,
                              per_token=True)
    # unwritten scale slots hold NaN
    nan = np.full((case.num_blocks, cfg.kv_heads, 2, 16), np.nan, np.float32).view(np.uint8)
    vd.view(case.num_blocks, cfg.kv_heads, -1)[:, :, 16 * cfg.head_dim:] = \
        torch.from_numpy(nan.reshape(case.num_blocks, cfg.kv_heads, -1)).cuda()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    k.kvq_reshape_and_cache_per_token(case.k.cuda(), case.v.cuda(), case.slot_mapping.cuda(), kd, vd,
                                      case.cache_dtype, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return kd, vd


def gpu_decode(case, kd, vd, num_splits=0):
    k = _k()
    B, Hq, D = case.q.shape
    out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    k.kvq_paged_decode_attention_per_token(case.q.cuda(), kd, vd, case.block_table.cuda(),
                                           case.seq_lens.cuda(), out, num_blocks=case.num_blocks,
                                           sm_scale=case.sm_scale, window=case.window,
                                           cache_dtype=case.cache_dtype, num_splits=num_splits, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0, f"device status {int(st.item()):#x}"
    return f32(out)


def _bits(a):
    return np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)


@pytest.mark.parametrize("dtype", [FP8, FP8_E5M2])
@pytest.mark.parametrize("D,Hkv,lengths,scatter", [(128, 8, [1000, 333], False), (64, 8, [17, 16, 1], False),
                                                   (128, 2, [300], True)])
def test_cache_write_per_token_bit_exact(dtype, D, Hkv, lengths, scatter):
    cfg = W.DecodeConfig("pt", batch=len(lengths), q_heads=Hkv, kv_heads=Hkv, head_dim=D, context=max(lengths),
                         outliers=4 if D == 128 else 0)
    case = W.decode_case(cfg, lengths=lengths, cache_dtype=dtype)
    if scatter:  # slots in random order, some skipped (the scattered V path)
        g = torch.Generator().manual_seed(9)
        case.slot_mapping = case.slot_mapping[torch.randperm(case.slot_mapping.numel(), generator=g)].contiguous()
        case.slot_mapping[::5] = -1
    kd, vd = gpu_per_token_cache(case)
    kc, vc, sc = oracle_per_token_cache(case)
    ek, ev = layout.to_device_format_per_token(kc, vc, sc)
    assert np.array_equal(kd.cpu().numpy(), ek), "K cache bytes differ"
    code_bytes = 16 * D
    assert np.array_equal(vd.cpu().numpy()[:, :, :code_bytes], ev[:, :, :code_bytes]), "V cache bytes differ"
    _, _, got_sc = layout.from_device_format_per_token(kd.cpu().numpy(), vd.cpu().numpy(), D)
    assert np.array_equal(_bits(got_sc), _bits(sc)), "scales differ"


CASES = {
    "llama_small": (dict(batch=2, q_heads=32, kv_heads=8, head_dim=128, context=1000, outliers=4), [1000, 333], FP8, -1),
    "ragged_g4": (dict(batch=5, q_heads=8, kv_heads=2, head_dim=128, context=2049), [1, 16, 17, 250, 2049], FP8, -1),
    "gptoss_d64": (dict(batch=2, q_heads=64, kv_heads=8, head_dim=64, context=1500), [700, 1500], FP8, -1),
    "window_d64": (dict(batch=4, q_heads=64, kv_heads=8, head_dim=64, context=1000), [50, 128, 129, 1000], FP8, 128),
    "e5m2_llama": (dict(batch=2, q_heads=32, kv_heads=8, head_dim=128, context=1000, outliers=4), [1000, 333],
                   FP8_E5M2, -1),
    "e5m2_ragged_d64": (dict(batch=3, q_heads=16, kv_heads=2, head_dim=64, context=777), [777, 5, 300],
                        FP8_E5M2, -1),
}


def _check_decode(case, num_splits=0):
    kd, vd = gpu_per_token_cache(case)
    kc, vc, sc = oracle_per_token_cache(case)
    got = gpu_decode(case, kd, vd, num_splits=num_splits)
    args = (f32(case.q), kc, vc, sc, case.block_table.numpy(), case.seq_lens.numpy(), case.sm_scale)
    ref, _ = attention.paged_decode_per_token(*args, window=case.window, cache_dtype=case.cache_dtype, mode="mirror")
    pure, _ = attention.paged_decode_per_token(*args, window=case.window, cache_dtype=case.cache_dtype, mode="pure")
    assert_close(got, ref, what="vs mirrored oracle")
    assert_close(got, pure, what="vs pure oracle")
    return got


@pytest.mark.parametrize("name", list(CASES))
def test_decode_per_token_parity(name):
    kw, lengths, dtype, window = CASES[name]
    case = W.decode_case(W.DecodeConfig("pt_" + name, **kw), lengths=lengths, cache_dtype=dtype, window=window)
    _check_decode(case)


@pytest.mark.parametrize("splits", [1, 3, 64])
def test_decode_per_token_split_counts(splits):
    cfg = W.DecodeConfig("pt_splits", batch=2, q_heads=16, kv_heads=4, head_dim=128, context=900, outliers=4)
    case = W.decode_case(cfg, lengths=[900, 211], cache_dtype=FP8)
    _check_decode(case, num_splits=splits)


def test_decode_per_token_full_size_llama_128k():
    """One full Llama-3.1-8B layer at 131,072 tokens (8 KV heads, D 128,
    4 outlier channels) with per-token scales."""
    case = W.decode_case(W.LLAMA_128K, layer=3)
    kd, vd = gpu_per_token_cache(case)
    got = gpu_decode(case, kd, vd)
    kc, vc, sc = oracle_per_token_cache(case)
    ref, _ = attention.paged_decode_per_token(f32(case.q), kc, vc, sc, case.block_table.numpy(),
                                              case.seq_lens.numpy(), case.sm_scale, cache_dtype=FP8, mode="mirror")
    assert_close(got, ref, what="128K per-token vs mirrored oracle")
