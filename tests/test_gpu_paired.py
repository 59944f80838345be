"""The paired cache layout (each (block, KV head) pair's K page followed by
its V page in one allocation; v_cache = k_cache + one K page), which the
library recognizes from the pointers and moves with one copy per page in
decode.  Cache writes are bit-exact against the oracle's paired byte format;
decode and prefill read the same codes and run the same arithmetic in the
same order as over separate caches, so their results are bit-identical to
the separate layout's (and within the tolerance of the oracle)."""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import kv_cache, layout
from oracle.kv_cache import BF16, FP8, FP8_E5M2
from tests.kvq_testlib import SENTINEL, assert_close, f32, oracle_cache, oracle_decode, to_device_cache

pytestmark = pytest.mark.gpu

PAGE = 16


def _k():
    import fp8_kv_cache_reshape_gb300 as k
    return k


def paired_device(kc, vc, sc=None):
    """Device pair buffer and (k_cache, v_cache) views of it."""
    buf = torch.from_numpy(layout.to_device_format_paired(kc, vc, sc)).cuda()
    kpage = kc.shape[2] * kc.shape[3] * kc.dtype.itemsize
    return buf, buf.view(-1)[kpage:]


def decode(case, kd, vd, num_splits=0):
    k = _k()
    B, Hq, D = case.q.shape
    out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    k.kvq_paged_decode_attention(case.q.cuda(), kd, vd, case.k_scale.cuda(), case.v_scale.cuda(),
                                 case.block_table.cuda(), case.seq_lens.cuda(), out, num_blocks=case.num_blocks,
                                 sm_scale=case.sm_scale, window=case.window, cache_dtype=case.cache_dtype,
                                 num_splits=num_splits, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0, f"device status {int(st.item()):#x}"
    return f32(out)


CASES = {
    "llama_small": (dict(batch=2, q_heads=32, kv_heads=8, head_dim=128, context=1000, outliers=4), [1000, 333], FP8, -1),
    "gptoss_d64": (dict(batch=2, q_heads=64, kv_heads=8, head_dim=64, context=1500), [700, 1500], FP8, -1),
    "e5m2_ragged": (dict(batch=5, q_heads=8, kv_heads=2, head_dim=128, context=2049), [1, 16, 17, 250, 2049],
                    FP8_E5M2, -1),
    "window_bf16": (dict(batch=4, q_heads=64, kv_heads=8, head_dim=64, context=1000), [50, 128, 129, 1000], BF16, 128),
    "bf16_d128": (dict(batch=2, q_heads=32, kv_heads=8, head_dim=128, context=1300), [1300, 64], BF16, -1),
    "many_seqs_d64": (dict(batch=80, q_heads=16, kv_heads=8, head_dim=64, context=600),
                      [17 + (37 * i) % 583 for i in range(80)], FP8, -1),
}


@pytest.mark.parametrize("name", list(CASES))
def test_decode_over_a_paired_cache_equals_the_separate_layout(name):
    kw, lengths, dtype, window = CASES[name]
    case = W.decode_case(W.DecodeConfig("paired_" + name, **kw), lengths=lengths, cache_dtype=dtype, window=window)
    kc, vc = oracle_cache(case)
    kd, vd = to_device_cache(kc, vc)
    sep = decode(case, kd, vd)
    buf, vview = paired_device(kc, vc)
    got = decode(case, buf, vview)
    assert np.array_equal(got, sep), "paired and separate layouts differ"
    ref, _ = oracle_decode(case, kc, vc, mode="mirror")
    assert_close(got, ref, what=f"paired {name} vs mirrored oracle")


@pytest.mark.parametrize("dtype,D", [(FP8, 128), (FP8_E5M2, 64), (BF16, 64), (BF16, 128)])
def test_cache_write_into_a_paired_cache_bit_exact(dtype, D):
    k = _k()
    cfg = W.DecodeConfig("pw", batch=2, q_heads=8, kv_heads=8, head_dim=D, context=700)
    case = W.decode_case(cfg, lengths=[700, 313], cache_dtype=dtype)
    # scatter some slots (the V path that writes single bytes) and skip some
    g = torch.Generator().manual_seed(3)
    slots = case.slot_mapping[torch.randperm(case.slot_mapping.numel(), generator=g)].contiguous()
    slots[::7] = -1
    kd, vd = k.alloc_kv_cache(case.num_blocks, 8, D, cache_dtype=dtype, fill=SENTINEL, paired=True)
    k.kvq_reshape_and_cache(case.k.cuda(), case.v.cuda(), slots.cuda(), kd, vd, case.k_scale.cuda(),
                            case.v_scale.cuda(), cache_dtype=dtype)
    torch.cuda.synchronize()
    esize = 2 if dtype == BF16 else 1
    dt = np.uint16 if dtype == BF16 else np.uint8
    fill = SENTINEL if esize == 1 else (SENTINEL << 8) | SENTINEL
    kc = np.full((case.num_blocks, 8, PAGE, D), fill, dt)
    vc = np.full((case.num_blocks, 8, D, PAGE), fill, dt)
    kv_cache.reshape_and_cache(f32(case.k), f32(case.v), slots.numpy(), kc, vc, case.k_scale.numpy(),
                               case.v_scale.numpy(), dtype)
    assert np.array_equal(kd.cpu().numpy(), layout.to_device_format_paired(kc, vc))


@pytest.mark.parametrize("dtype", [FP8, FP8_E5M2])
def test_per_token_write_and_decode_over_a_paired_cache(dtype):
    k = _k()
    cfg = W.DecodeConfig("ppt", batch=2, q_heads=32, kv_heads=8, head_dim=128, context=1000, outliers=4)
    case = W.decode_case(cfg, lengths=[1000, 333], cache_dtype=dtype)
    kd, vd = k.alloc_kv_cache(case.num_blocks, 8, 128, cache_dtype=dtype, fill=SENTINEL, per_token=True, paired=True)
    # unwritten scale slots hold NaN (a read of one would show in the output)
    pair = kd.view(case.num_blocks, 8, -1)
    nan = torch.full((case.num_blocks, 8, 32), float("nan"), dtype=torch.float32)
    pair[:, :, 2 * 16 * 128:] = nan.view(torch.uint8).view(case.num_blocks, 8, -1).cuda()
    k.kvq_reshape_and_cache_per_token(case.k.cuda(), case.v.cuda(), case.slot_mapping.cuda(), kd, vd,
                                      cache_dtype=dtype)
    kc = np.full((case.num_blocks, 8, PAGE, 128), SENTINEL, np.uint8)
    vc = np.full((case.num_blocks, 8, 128, PAGE), SENTINEL, np.uint8)
    sc = np.full((case.num_blocks, 8, 2, PAGE), np.nan, np.float32)
    kv_cache.reshape_and_cache_per_token(f32(case.k), f32(case.v), case.slot_mapping.numpy(), kc, vc, sc, dtype)
    torch.cuda.synchronize()
    expect = layout.to_device_format_paired(kc, vc, sc)
    assert np.array_equal(kd.cpu().numpy(), expect), "paired per-token cache bytes differ"
    out = torch.empty(case.q.shape, dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    k.kvq_paged_decode_attention_per_token(case.q.cuda(), kd, vd, case.block_table.cuda(), case.seq_lens.cuda(),
                                           out, num_blocks=case.num_blocks, sm_scale=case.sm_scale,
                                           cache_dtype=dtype, dev_status=st)
    sep_k, sep_v = layout.to_device_format_per_token(kc, vc, sc)
    out_sep = torch.empty_like(out)
    k.kvq_paged_decode_attention_per_token(case.q.cuda(), torch.from_numpy(sep_k).cuda(),
                                           torch.from_numpy(sep_v).cuda(), case.block_table.cuda(),
                                           case.seq_lens.cuda(), out_sep, num_blocks=case.num_blocks,
                                           sm_scale=case.sm_scale, cache_dtype=dtype, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(out, out_sep), "paired and separate per-token decode differ"


def test_append_and_prefill_over_a_paired_cache_equal_the_separate_layout():
    k = _k()
    from tests import test_gpu_prefill as tp
    c = tp.build([256, 77], [384, 1000], Hq=16, Hkv=4, seed=5)
    kd, vd = to_device_cache(c["kc"], c["vc"])
    buf, vview = paired_device(c["kc"], c["vc"])

    def prefill(kcache, vcache):
        out = torch.full(c["q8"].shape, float("nan"), dtype=torch.bfloat16, device="cuda")
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        k.kvq_prefill_attention(torch.from_numpy(c["q8"]).cuda(), torch.tensor([c["qs"]], device="cuda"), kcache,
                                vcache, torch.from_numpy(c["ks"]).cuda(), torch.from_numpy(c["vs"]).cuda(),
                                torch.from_numpy(c["bt"]).cuda(), torch.from_numpy(c["cu"]).cuda(),
                                torch.from_numpy(c["lens"]).cuda(), out, max_q_tokens=256, num_blocks=c["nb"],
                                sm_scale=float(c["sm"]), dev_status=st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        return out

    assert torch.equal(prefill(buf, vview), prefill(kd, vd)), "paired and separate prefill differ"

    # decode with the new token's write, on both layouts
    cfg = W.DecodeConfig("pap", batch=3, q_heads=16, kv_heads=4, head_dim=128, context=900)
    case = W.decode_case(cfg, lengths=[900, 211, 17])
    kc, vc = oracle_cache(case)
    B = 3
    g = torch.Generator().manual_seed(11)
    k_new = torch.randn((B, 4, 128), generator=g).bfloat16()
    v_new = torch.randn((B, 4, 128), generator=g).bfloat16()
    last = case.seq_lens.long() - 1
    slot_new = torch.stack([case.block_table[b, last[b] // 16].long() * 16 + last[b] % 16 for b in range(B)])
    outs, caches = [], []
    for paired in (False, True):
        if paired:
            kd2, vd2 = paired_device(kc, vc)
        else:
            kd2, vd2 = to_device_cache(kc, vc)
        out = torch.empty(case.q.shape, dtype=torch.bfloat16, device="cuda")
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        k.kvq_paged_decode_attention_append(case.q.cuda(), k_new.cuda(), v_new.cuda(), slot_new.cuda(), kd2, vd2,
                                            case.k_scale.cuda(), case.v_scale.cuda(), case.block_table.cuda(),
                                            case.seq_lens.cuda(), out, num_blocks=case.num_blocks,
                                            sm_scale=case.sm_scale, dev_status=st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        outs.append(out)
        caches.append((kd2, vd2))
    assert torch.equal(outs[0], outs[1]), "paired and separate append decode differ"
    sep_bytes = np.concatenate([caches[0][0].cpu().numpy(), caches[0][1].cpu().numpy()], axis=2)
    assert np.array_equal(caches[1][0].cpu().numpy(), sep_bytes), "the new tokens landed differently"


@pytest.mark.parametrize("dtype", [FP8, FP8_E5M2])
def test_per_token_prefill_over_a_paired_cache_equals_the_separate_layout(dtype):
    from tests import test_gpu_prefill as tp
    c = tp.build_per_token([200, 64], [300, 900], Hq=16, Hkv=4, seed=2, cache_dtype=dtype)
    buf, vview = paired_device(c["kc"], c["vc"], c["sc"])
    got = tp.gpu_prefill_per_token(c, caches=(buf, vview))
    assert np.array_equal(got, tp.gpu_prefill_per_token(c), equal_nan=True), "paired and separate differ"
    rows = [(t, h) for t in range(0, got.shape[0], 7) for h in range(0, c["Hq"], 3)]
    tp.check_rows(got, tp.oracle_per_token(c, rows), rows, what=f"paired per-token prefill {dtype}")
