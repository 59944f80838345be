"""The accumulation ablation: single-level accumulation (the tensor cores add
every tile into the running sum) against the default two-level scheme.

* parity: the single-level decode and prefill meet the same tolerance
  against the oracle as the two-level ones;
* the ablation itself: with two splits, each decode warp accumulates 4,096
  tokens of a 32K context; the single-level FP32 partials must agree with
  the two-level ones to within a median relative 2e-5 (the decode MMAs'
  own addition into the running sum measured 4.4e-6; a tensor-core
  accumulator that kept ~14 bits, as the pages report for FP8 on H800,
  would show up here);
* the modes that are not built are refused on the host."""
import numpy as np
import pytest
import torch

import workloads as W
from oracle.kv_cache import BF16, FP8, FP8_E5M2
from tests.kvq_testlib import assert_close, f32, oracle_cache, oracle_decode, to_device_cache
from tests import test_gpu_prefill as tp

pytestmark = pytest.mark.gpu


def _k():
    import fp8_kv_cache_reshape_gb300 as k
    return k


def decode(case, kd, vd, accumulation, num_splits=0, workspace=None):
    k = _k()
    out = torch.empty(case.q.shape, dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    k.kvq_paged_decode_attention(case.q.cuda(), kd, vd, case.k_scale.cuda(), case.v_scale.cuda(),
                                 case.block_table.cuda(), case.seq_lens.cuda(), out, num_blocks=case.num_blocks,
                                 sm_scale=case.sm_scale, window=case.window, cache_dtype=case.cache_dtype,
                                 num_splits=num_splits, workspace=workspace, dev_status=st, accumulation=accumulation)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return f32(out)


@pytest.mark.parametrize("kw,lengths", [
    (dict(batch=2, q_heads=32, kv_heads=8, head_dim=128, context=1000, outliers=4), [1000, 333]),
    (dict(batch=5, q_heads=8, kv_heads=2, head_dim=128, context=2049), [1, 16, 17, 250, 2049]),
    (dict(batch=2, q_heads=64, kv_heads=8, head_dim=64, context=1500), [700, 1500]),
])
def test_single_level_decode_parity(kw, lengths):
    case = W.decode_case(W.DecodeConfig("acc_dec", **kw), lengths=lengths)
    kc, vc = oracle_cache(case)
    kd, vd = to_device_cache(kc, vc)
    got = decode(case, kd, vd, "single_level")
    ref, _ = oracle_decode(case, kc, vc, mode="mirror")
    assert_close(got, ref, what="single-level decode vs mirrored oracle")


def test_single_level_partials_match_two_level_over_long_accumulation():
    k = _k()
    case = W.decode_case(W.LLAMA_128K, layer=2, lengths=[32768])
    kc, vc = oracle_cache(case)
    kd, vd = to_device_cache(kc, vc)
    B, Hq, D = case.q.shape
    # two page ranges, so that the partials go through the workspace (with one
    # range per sequence and KV head the kernel merges them in shared memory);
    # each consumer warp still accumulates 4,096 tokens
    need = k.kvq_decode_workspace_size(B, Hq, 8, D, case.block_table.shape[1], -1, 2)
    parts = {}
    for acc in ("two_level", "single_level"):
        ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
        decode(case, kd, vd, acc, num_splits=2, workspace=ws)
        parts[acc] = ws[: B * Hq * 2 * 4 * D * 4].view(torch.float32).cpu().numpy().astype(np.float64)
    a, b = parts["two_level"], parts["single_level"]
    assert np.all(np.isfinite(a)) and np.all(np.isfinite(b))
    diff = np.abs(a - b)
    # ~128 stage sums of O(1) values: well below 1e-4 of the partials' scale
    assert diff.max() <= 1e-4 * np.abs(a).max(), f"max |two - single| {diff.max():.3e}"
    # Two-level adds each stage's fresh FP32 tile in FP32 arithmetic; single-
    # level lets the f16 MMA add into the running sum itself, which on this GPU
    # is slightly coarser than an FP32 add (measured: median relative 4.4e-6
    # over 4,096 tokens per warp).  Far inside the output tolerance; a 14-bit
    # accumulator (the Hopper FP8 defect) would show as ~1e-4 and above.
    rel = np.median(diff / np.maximum(np.abs(a), 1e-3))
    print(f"[accumulation] median relative |two - single| {rel:.3e}, max {diff.max():.3e}")
    assert rel <= 2e-5


def test_single_level_prefill_parity():
    for nq, cached, seed in (([256], [384], 1), ([1, 130, 300], [0, 17, 1000], 3), ([77], [5000], 4)):
        c = tp.build(nq, cached, seed=seed)
        k = _k()
        kd, vd = to_device_cache(c["kc"], c["vc"])
        out = torch.full(c["q8"].shape, float("nan"), dtype=torch.bfloat16, device="cuda")
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        k.kvq_prefill_attention(torch.from_numpy(c["q8"]).cuda(), torch.tensor([c["qs"]], device="cuda"), kd, vd,
                                torch.from_numpy(c["ks"]).cuda(), torch.from_numpy(c["vs"]).cuda(),
                                torch.from_numpy(c["bt"]).cuda(), torch.from_numpy(c["cu"]).cuda(),
                                torch.from_numpy(c["lens"]).cuda(), out, max_q_tokens=int(np.max(np.diff(c["cu"]))),
                                num_blocks=c["nb"], sm_scale=float(c["sm"]), dev_status=st,
                                accumulation="single_level")
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        rng = np.random.default_rng(seed)
        rows = [(t, h) for t in range(c["q8"].shape[0]) for h in range(c["Hq"])]
        if len(rows) > 2000:
            rows = [rows[i] for i in rng.choice(len(rows), 2000, replace=False)]
        tp.check_all(f32(out), c, rows, what=f"single-level prefill nq={nq}")


@pytest.mark.parametrize("dtype", [BF16, FP8_E5M2])
def test_single_level_other_caches_unsupported(dtype):
    k = _k()
    case = W.decode_case(W.DecodeConfig("acc_uns", batch=1, q_heads=4, kv_heads=1, head_dim=64, context=64),
                         lengths=[64], cache_dtype=dtype)
    kc, vc = oracle_cache(case)
    kd, vd = to_device_cache(kc, vc)
    with pytest.raises(k.KvqError) as e:
        decode(case, kd, vd, "single_level")
    assert e.value.status == k.KVQ_ERR_UNSUPPORTED
