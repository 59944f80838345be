"""GPU parity of kvq_reshape_and_cache and kvq_quantize_query against the
oracle: bit-exact on every cache byte (sentinel-filled first) and every q8
byte."""
import math

import numpy as np
import pytest
import torch

import workloads as W
from oracle import kv_cache, layout
from oracle.kv_cache import FP8, FP8_E5M2, BF16
from tests.kvq_testlib import SENTINEL, f32, oracle_cache

pytestmark = pytest.mark.gpu

def _lib():
    import fp8_kv_cache_reshape_gb300 as k
    return k


def _run_gpu_write(case):
    k = _lib()
    cfg = case.cfg
    kd, vd = k.alloc_kv_cache(case.num_blocks, cfg.kv_heads, cfg.head_dim, case.cache_dtype, fill=SENTINEL)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    k.kvq_reshape_and_cache(case.k.cuda(), case.v.cuda(), case.slot_mapping.cuda(), kd, vd,
                            case.k_scale.cuda(), case.v_scale.cuda(), case.cache_dtype, dev_status=st)
    torch.cuda.synchronize()
    return kd.cpu().numpy(), vd.cpu().numpy(), int(st.item())


def _expected(case):
    kc, vc = oracle_cache(case)
    return layout.to_device_format(kc, vc)


@pytest.mark.parametrize("dtype", [FP8, FP8_E5M2, BF16])
@pytest.mark.parametrize("D,Hkv,lengths", [(128, 8, [1000, 333]), (64, 8, [17, 16, 1]), (64, 1, [512]),
                                           (256, 4, [300, 17])])
def test_cache_write_bit_exact(dtype, D, Hkv, lengths):
    if D == 256 and dtype == BF16:
        pytest.skip("head_dim 256 caches are FP8 only")
    cfg = W.DecodeConfig("t", batch=len(lengths), q_heads=Hkv, kv_heads=Hkv, head_dim=D, context=max(lengths),
                         outliers=4 if D == 128 else 0)
    case = W.decode_case(cfg, lengths=lengths, cache_dtype=dtype)
    gk, gv, st = _run_gpu_write(case)
    ek, ev = _expected(case)
    assert st == 0
    assert np.array_equal(gk, ek), "K cache bytes differ"
    assert np.array_equal(gv, ev), "V cache bytes differ"


@pytest.mark.parametrize("dtype", [FP8, FP8_E5M2, BF16])
def test_cache_write_scattered_slots_and_skips(dtype):
    """Slots in random order (slow path), negative slots skipped, ragged T."""
    cfg = W.DecodeConfig("t", batch=1, q_heads=8, kv_heads=8, head_dim=128, context=300)
    case = W.decode_case(cfg, lengths=[300], cache_dtype=dtype)
    g = torch.Generator().manual_seed(5)
    perm = torch.randperm(case.slot_mapping.numel(), generator=g)
    case.slot_mapping = case.slot_mapping[perm].contiguous()
    case.slot_mapping[::7] = -1
    gk, gv, st = _run_gpu_write(case)
    ek, ev = _expected(case)
    assert st == 0
    assert np.array_equal(gk, ek) and np.array_equal(gv, ev)


def test_cache_write_bad_slot_reported_and_skipped():
    cfg = W.DecodeConfig("t", batch=1, q_heads=2, kv_heads=2, head_dim=64, context=40)
    case = W.decode_case(cfg, lengths=[40])
    case.slot_mapping[3] = case.num_blocks * 16 + 5
    gk, gv, st = _run_gpu_write(case)
    assert st & 0x1
    ek, ev = _expected(case)  # the oracle skips the same token
    assert np.array_equal(gk, ek) and np.array_equal(gv, ev)


def test_cache_write_saturation_and_extremes():
    """Values far beyond 448 * scale saturate; tiny ones flush to signed zero."""
    cfg = W.DecodeConfig("t", batch=1, q_heads=1, kv_heads=1, head_dim=64, context=32, calibrated=False)
    case = W.decode_case(cfg, lengths=[32])
    k = case.k.float()
    k[0, 0, :8] = torch.tensor([1e4, -1e4, 449.0, -448.5, 1e-30, -1e-30, 0.0, -0.0])
    k[1, 0, :4] = torch.tensor([float(2 ** -10), float(3 * 2 ** -11), 464.0, 432.0])
    case.k = k.bfloat16()
    case.k_scale = torch.tensor([1.0])
    gk, gv, st = _run_gpu_write(case)
    ek, ev = _expected(case)
    assert np.array_equal(gk, ek) and np.array_equal(gv, ev)


def test_cache_write_e5m2_saturation_and_extremes():
    """E5M2: values beyond 57344 * scale saturate; values below half its
    smallest subnormal (2^-17) flush to signed zero; ties round to even."""
    cfg = W.DecodeConfig("t", batch=1, q_heads=1, kv_heads=1, head_dim=64, context=32, calibrated=False)
    case = W.decode_case(cfg, lengths=[32], cache_dtype=FP8_E5M2)
    k = case.k.float()
    k[0, 0, :8] = torch.tensor([1e6, -1e6, 61440.0, -57344.0, 1e-30, -1e-30, 0.0, -0.0])
    k[1, 0, :6] = torch.tensor([float(2 ** -17), float(3 * 2 ** -17), float(2 ** -16), 1.125, 1.375, 3.0])
    case.k = k.bfloat16()
    case.k_scale = torch.tensor([1.0])
    gk, gv, st = _run_gpu_write(case)
    ek, ev = _expected(case)
    assert np.array_equal(gk, ek) and np.array_equal(gv, ev)


@pytest.mark.parametrize("n", [5, 16, 4096 * 32 * 128 + 13])
def test_quantize_query_bit_exact(n):
    k = _lib()
    g = W.generator(77)
    q = W.randn_bf16((n,), g) * 3
    q = q.bfloat16()
    s = (q.float().abs().max() / 448).reshape(1)
    q8 = torch.empty(n, dtype=torch.uint8, device="cuda")
    k.kvq_quantize_query(q.cuda(), q8, s.cuda())
    torch.cuda.synchronize()
    exp = kv_cache.quantize_query(f32(q), np.float32(s.item()))
    assert np.array_equal(q8.cpu().numpy(), exp)


def test_cache_write_full_size_llama_128k():
    """The Llama-3.1-8B-shaped layer at 131,072 tokens (permuted pages,
    4 outlier channels x20, amax/448 scales): every byte of both caches."""
    case = W.decode_case(W.LLAMA_128K, layer=0)
    gk, gv, st = _run_gpu_write(case)
    ek, ev = _expected(case)
    assert st == 0
    assert np.array_equal(gk, ek) and np.array_equal(gv, ev)
