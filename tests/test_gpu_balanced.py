"""Decode of ragged batches under the balanced plan.  With 2 to 32 sequences
and more than one split, each KV head's attended pages are laid end to end
over the batch and cut into B x S equal slots: a long sequence gets more
page ranges than a short one, and a slot may span the end of one sequence
and the start of the next (its part in each is a segment with its own
partial).  Parity against the oracle with skewed lengths (empty, one token,
one page, long), automatic and explicit split counts, every cache type,
windows, per-token scales and the new token's write; 32 sequences (the
largest batch the plan covers) beside 33 (the per-sequence plan); and the
plan is deterministic: two runs and a page permutation give bit-identical
outputs."""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import attention
from oracle.kv_cache import BF16, FP8, FP8_E5M2
from tests.kvq_testlib import assert_close, f32, oracle_cache, oracle_decode, to_device_cache

pytestmark = pytest.mark.gpu

SKEWED = [40, 1, 4000, 16, 17, 2500, 7, 333]
# attended lengths: two sequences empty, the rest as built
SKEWED_ATTENDED = [0, 1, 4000, 16, 17, 2500, 0, 333]


def _k():
    import fp8_kv_cache_reshape_gb300 as k
    return k


def _decode(case, kd, vd, num_splits=0, block_table=None):
    k = _k()
    B, Hq, D = case.q.shape
    out = torch.full((B, Hq, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    bt = (case.block_table if block_table is None else block_table).cuda()
    k.kvq_paged_decode_attention(case.q.cuda(), kd, vd, case.k_scale.cuda(), case.v_scale.cuda(), bt,
                                 case.seq_lens.cuda(), out, num_blocks=case.num_blocks, sm_scale=case.sm_scale,
                                 window=case.window, cache_dtype=case.cache_dtype, num_splits=num_splits,
                                 dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0, f"device status {int(st.item()):#x}"
    return f32(out)


def _check(case, num_splits=0, what=""):
    kc, vc = oracle_cache(case)
    kd, vd = to_device_cache(kc, vc)
    got = _decode(case, kd, vd, num_splits=num_splits)
    ref, _ = oracle_decode(case, kc, vc, mode="mirror")
    pure, _ = oracle_decode(case, kc, vc, mode="pure")
    assert_close(got, ref, what=f"{what} vs mirrored oracle")
    assert_close(got, pure, what=f"{what} vs pure oracle")
    return got, (kc, vc, kd, vd)


@pytest.mark.parametrize("splits", [0, 3, 13])
@pytest.mark.parametrize("dtype,D", [(FP8, 128), (FP8, 64), (FP8_E5M2, 128), (BF16, 64)])
def test_skewed_batch_parity(dtype, D, splits):
    hq, hkv = (16, 4) if D == 128 else (32, 4)
    # no outlier channels: with sequences of a few tokens the unmirrored P
    # rounding on x20 channels is not averaged out (the plan is under test here)
    cfg = W.DecodeConfig("bal", batch=len(SKEWED), q_heads=hq, kv_heads=hkv, head_dim=D, context=max(SKEWED))
    case = W.decode_case(cfg, lengths=SKEWED, cache_dtype=dtype)
    case.seq_lens = torch.tensor(SKEWED_ATTENDED, dtype=torch.int32)
    got, _ = _check(case, splits, what=f"skewed {dtype} D={D} S={splits}")
    assert np.all(got[0] == 0) and np.all(got[6] == 0), "empty sequences must give 0"


@pytest.mark.parametrize("batch", [32, 33])
def test_largest_balanced_batch_and_the_next(batch):
    lengths = [1 + (97 * i) % 1500 for i in range(batch)]
    cfg = W.DecodeConfig(f"bal{batch}", batch=batch, q_heads=8, kv_heads=2, head_dim=128, context=max(lengths))
    case = W.decode_case(cfg, lengths=lengths)
    assert _k().kvq_decode_num_splits(batch, 2, case.block_table.shape[1], head_dim=128) > 1
    _check(case, what=f"B={batch}")


@pytest.mark.parametrize("dtype", [FP8, BF16])
def test_window_with_explicit_splits(dtype):
    cfg = W.DecodeConfig("balw", batch=5, q_heads=32, kv_heads=4, head_dim=64, context=3000)
    case = W.decode_case(cfg, lengths=[50, 128, 129, 1000, 3000], cache_dtype=dtype, window=128)
    _check(case, num_splits=3, what=f"window {dtype}")


@pytest.mark.parametrize("splits", [0, 4])
def test_per_token_scales_on_a_skewed_batch(splits):
    from tests import test_gpu_per_token as tpt
    cfg = W.DecodeConfig("balpt", batch=5, q_heads=16, kv_heads=4, head_dim=128, context=2000)
    case = W.decode_case(cfg, lengths=[2000, 17, 700, 1, 1500])
    kd, vd = tpt.gpu_per_token_cache(case)
    kc, vc, sc = tpt.oracle_per_token_cache(case)
    got = tpt.gpu_decode(case, kd, vd, num_splits=splits)
    args = (f32(case.q), kc, vc, sc, case.block_table.numpy(), case.seq_lens.numpy(), case.sm_scale)
    ref, _ = attention.paged_decode_per_token(*args, window=case.window, cache_dtype=case.cache_dtype, mode="mirror")
    assert_close(got, ref, what=f"per-token skewed S={splits}")


def test_new_tokens_write_on_a_skewed_batch():
    from tests import test_gpu_append as ta
    cfg = W.DecodeConfig("balap", batch=6, q_heads=16, kv_heads=4, head_dim=128, context=2049)
    case = W.decode_case(cfg, lengths=[1, 16, 17, 250, 2049, 900])
    kd, vd, last, ks, vs = ta._prepare(case)
    kd2, vd2 = kd.clone(), vd.clone()
    slot_new = case.slot_mapping[last].cuda()
    got, st = ta._append(case, kd, vd, last, ks, vs, slot_new)
    assert st == 0
    ref_out, st2 = ta._two_calls(case, kd2, vd2, last, ks, vs, slot_new)
    assert st2 == 0
    assert torch.equal(kd, kd2) and torch.equal(vd, vd2), "cache bytes differ from the two-call path"
    assert torch.equal(got.view(torch.int16), ref_out.view(torch.int16)), "output differs from the two-call path"
    kc, vc = oracle_cache(case)
    ref, _ = oracle_decode(case, kc, vc, mode="mirror")
    assert_close(f32(got), ref, what="append on a skewed batch")


def test_balanced_plan_is_deterministic_and_page_permutation_invariant():
    cfg = W.DecodeConfig("balperm", batch=4, q_heads=8, kv_heads=2, head_dim=128, context=1800)
    case = W.decode_case(cfg, lengths=[1800, 33, 900, 250])
    kc, vc = oracle_cache(case)
    kd, vd = to_device_cache(kc, vc)
    a = _decode(case, kd, vd, num_splits=5)
    assert np.array_equal(a, _decode(case, kd, vd, num_splits=5)), "two runs differ"
    nb = case.num_blocks
    perm = torch.randperm(nb, generator=torch.Generator().manual_seed(9))
    kd2 = torch.empty_like(kd)
    vd2 = torch.empty_like(vd)
    kd2[perm.cuda()] = kd
    vd2[perm.cuda()] = vd
    bt2 = perm[case.block_table.long()].to(torch.int32)
    assert np.array_equal(a, _decode(case, kd2, vd2, num_splits=5, block_table=bt2))
