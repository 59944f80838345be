"""The failure path of the bounded pipeline waits, run without faulting or
hanging the GPU: kvq_debug_set_stall_ns makes one wait of each decode and
prefill CTA wait on a barrier that nothing arrives on, for at most 1 ms.
The wait runs out, the kernel reports KVQ_DEV_TIMEOUT in the status word,
lets its issued bulk copies land, frees its tensor memory and returns; the
next call, with the hook off, is correct against the oracle (the context
is still usable)."""
import numpy as np
import pytest
import torch

import workloads as W
from tests import test_gpu_prefill as tp
from tests.kvq_testlib import assert_close, f32, oracle_cache, oracle_decode, to_device_cache

pytestmark = pytest.mark.gpu

STALL_NS = 1_000_000  # 1 ms


def _k():
    import fp8_kv_cache_reshape_gb300 as k
    return k


@pytest.fixture
def stall_off_afterwards():
    yield
    _k().kvq_debug_set_stall_ns(0)


def test_decode_wait_timeout_is_reported_and_the_next_call_is_correct(stall_off_afterwards):
    k = _k()
    cfg = W.DecodeConfig("timeout_dec", batch=2, q_heads=32, kv_heads=8, head_dim=128, context=20000)
    case = W.decode_case(cfg, lengths=[20000, 777])
    kd, vd = to_device_cache(*oracle_cache(case))
    args = (case.q.cuda(), kd, vd, case.k_scale.cuda(), case.v_scale.cuda(), case.block_table.cuda(),
            case.seq_lens.cuda())
    out = torch.empty(case.q.shape, dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    k.kvq_debug_set_stall_ns(STALL_NS)
    k.kvq_paged_decode_attention(*args, out, num_blocks=case.num_blocks, sm_scale=case.sm_scale, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & k.KVQ_DEV_TIMEOUT, f"status {int(st.item()):#x}"
    k.kvq_debug_set_stall_ns(0)
    st.zero_()
    k.kvq_paged_decode_attention(*args, out, num_blocks=case.num_blocks, sm_scale=case.sm_scale, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert_close(f32(out), oracle_decode(case, *oracle_cache(case))[0], what="decode after a timed-out call")


def test_prefill_wait_timeout_is_reported_and_the_next_call_is_correct(stall_off_afterwards):
    k = _k()
    c = tp.build([300], [1000], Hq=8, Hkv=2, seed=21)
    k.kvq_debug_set_stall_ns(STALL_NS)
    out, st = tp.gpu_prefill(c, status=True)
    assert st & k.KVQ_DEV_TIMEOUT, f"status {st:#x}"
    k.kvq_debug_set_stall_ns(0)
    got = tp.gpu_prefill(c)  # asserts a zero status
    rows = [(t, h) for t in range(0, 300, 7) for h in range(8)]
    tp.check_all(got, c, rows, what="prefill after a timed-out call")
