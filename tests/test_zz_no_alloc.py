"""kvq_paged_decode_attention_static_scratch: decode for callers that cannot
allocate device memory where decode runs (an allocation-free region of a
serving loop, a memory-pool policy that forbids new allocations, a plugin
without access to its host's allocator).  Its split-KV scratch is a fixed
array inside the library's device image instead of a caller workspace.

The test calls the entry point through the C ABI twice in a row (two
different problems, so the second call runs over the first call's leftover
scratch) and checks each output against the workspace entry point's output.
Both calls run the same kernels with the same split plan on the same inputs
-- only the scratch memory differs -- and every partial result is written
before it is read, so the outputs must be bit-identical; a stale or
overlapping scratch region would show as a difference.  It also checks that a
problem needing more scratch than the array holds is rejected before any
launch.  This file sorts last so that a run stopping at the first failure
has already run every other test."""
import ctypes

import numpy as np
import pytest
import torch

import workloads as W
from tests.kvq_testlib import assert_close, f32, oracle_cache, oracle_decode, to_device_cache

pytestmark = pytest.mark.gpu


def _k():
    import fp8_kv_cache_reshape_gb300 as k
    return k


def _problem(name, lengths, q_heads=32, kv_heads=8, head_dim=128):
    cfg = W.DecodeConfig(name, batch=len(lengths), q_heads=q_heads, kv_heads=kv_heads, head_dim=head_dim,
                         context=max(lengths), outliers=4)
    case = W.decode_case(cfg, lengths=lengths)
    kc, vc = oracle_cache(case)
    kd, vd = to_device_cache(kc, vc)
    dev = dict(q=case.q.cuda(), kd=kd, vd=vd, ks=case.k_scale.cuda(), vs=case.v_scale.cuda(),
               bt=case.block_table.cuda(), sl=case.seq_lens.cuda())
    return case, dev


def _with_workspace(case, dev):
    k = _k()
    out = torch.empty(case.q.shape, dtype=torch.bfloat16, device="cuda")
    k.kvq_paged_decode_attention(dev["q"], dev["kd"], dev["vd"], dev["ks"], dev["vs"], dev["bt"], dev["sl"], out,
                                 num_blocks=case.num_blocks, sm_scale=case.sm_scale)
    torch.cuda.synchronize()
    return f32(out)


def _static_scratch_c_abi(case, dev):
    """Raw C-ABI call: device pointers and sizes only."""
    k = _k()
    B, Hq, D = case.q.shape
    out = torch.empty(case.q.shape, dtype=torch.bfloat16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = k.lib.kvq_paged_decode_attention_static_scratch(
        dev["q"].data_ptr(), dev["kd"].data_ptr(), dev["vd"].data_ptr(), dev["ks"].data_ptr(), dev["vs"].data_ptr(),
        dev["bt"].data_ptr(), dev["sl"].data_ptr(), out.data_ptr(), B, Hq, case.cfg.kv_heads, D, 16,
        case.block_table.shape[1], case.num_blocks, ctypes.c_float(case.sm_scale), -1, k.KVQ_DTYPE_FP8_E4M3, 0,
        status.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert rc == k.KVQ_OK, k.lib.kvq_last_error_string().decode()
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return f32(out)


def test_static_scratch_matches_workspace_entry_point_on_two_calls():
    first, dev1 = _problem("noalloc_a", [3000, 1234])
    second, dev2 = _problem("noalloc_b", [5000, 17, 640])
    ref1 = _with_workspace(first, dev1)
    ref2 = _with_workspace(second, dev2)
    got1 = _static_scratch_c_abi(first, dev1)
    got2 = _static_scratch_c_abi(second, dev2)
    assert np.array_equal(got1, ref1), f"first call: max |diff| {np.max(np.abs(got1 - ref1)):.3e}"
    assert np.array_equal(got2, ref2), f"second call: max |diff| {np.max(np.abs(got2 - ref2)):.3e}"
    # and both are decode results: within the attention tolerance of the oracle
    assert_close(got1, oracle_decode(first, *oracle_cache(first))[0], what="static scratch, first call")
    assert_close(got2, oracle_decode(second, *oracle_cache(second))[0], what="static scratch, second call")


def test_static_scratch_rejects_problems_larger_than_the_array():
    k = _k()
    limit = k.lib.kvq_decode_static_scratch_bytes()
    assert limit == 4 << 20
    need = k.lib.kvq_decode_workspace_size(64, 64, 8, 128, 16, 8192, -1, 16)
    assert need > limit
    dummy = torch.zeros(16, dtype=torch.uint8, device="cuda")
    p = dummy.data_ptr()
    rc = k.lib.kvq_paged_decode_attention_static_scratch(p, p, p, p, p, p, p, p, 64, 64, 8, 128, 16, 8192, 1 << 20,
                                                         ctypes.c_float(0.088), -1, k.KVQ_DTYPE_FP8_E4M3, 16, None,
                                                         torch.cuda.current_stream().cuda_stream)
    assert rc == k.KVQ_ERR_UNSUPPORTED
    assert b"static array" in k.lib.kvq_last_error_string()
