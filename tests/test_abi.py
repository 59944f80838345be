"""The C-ABI library loads and exports every symbol include/kvq.h declares
(no compute calls: this runs without a GPU)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kvq.h")
LIB = os.path.join(ROOT, "fp8_kv_cache_reshape_gb300", "libkvq.so")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kvq_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(LIB):
        import __graft_entry__
        __graft_entry__.build()
    return ctypes.CDLL(LIB)


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("kvq_reshape_and_cache", "kvq_quantize_query", "kvq_paged_decode_attention",
              "kvq_decode_workspace_size", "kvq_decode_num_splits", "kvq_prefill_attention",
              "kvq_last_error_string", "kvq_version"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_host_only_calls(lib):
    lib.kvq_version.restype = ctypes.c_int
    assert lib.kvq_version() >= 10000
    lib.kvq_last_error_string.restype = ctypes.c_char_p
    assert isinstance(lib.kvq_last_error_string(), bytes)


def test_host_validation_without_gpu(lib):
    """Argument checks run before any CUDA call and return their status."""
    f = lib.kvq_reshape_and_cache
    f.restype = ctypes.c_int
    p = ctypes.c_void_p
    f.argtypes = [p, p, p, p, p, p, p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                  ctypes.c_int64, ctypes.c_int, p, p]
    assert f(None, None, None, None, None, None, None, 4, 1, 96, 16, 8, 0, None, None) == 2  # head_dim 96
    assert f(None, None, None, None, None, None, None, 4, 1, 128, 32, 8, 0, None, None) == 2  # page 32
    assert f(None, None, None, None, None, None, None, 4, 1, 128, 16, 8, 0, None, None) == 1  # null pointers
    assert f(None, None, None, None, None, None, None, 0, 1, 128, 16, 8, 0, None, None) == 0  # nothing to do
    lib.kvq_last_error_string.restype = ctypes.c_char_p
    q = lib.kvq_quantize_query
    q.restype = ctypes.c_int
    q.argtypes = [p, p, p, ctypes.c_int64, p]
    assert q(None, None, None, -1, None) == 1
    assert q(None, None, None, 0, None) == 0


def test_per_token_entry_points_validate_without_gpu(lib):
    """The per-token calls refuse a BF16 cache, missing caches and misaligned
    pointers before any CUDA call."""
    p = ctypes.c_void_p
    i, i64, f32, sz = ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
    w = lib.kvq_reshape_and_cache_per_token
    w.restype = i
    w.argtypes = [p, p, p, p, p, i, i, i, i, i64, i, p, p]
    fake = ctypes.c_void_p(1 << 20)  # never dereferenced: the calls return first
    odd = ctypes.c_void_p((1 << 20) + 4)
    assert w(fake, fake, fake, fake, fake, 4, 1, 128, 16, 8, 1, None, None) == 1  # BF16 cache
    assert w(fake, fake, fake, fake, None, 4, 1, 128, 16, 8, 0, None, None) == 1  # no V cache
    assert w(fake, fake, fake, fake, odd, 4, 1, 128, 16, 8, 0, None, None) == 1  # V cache not 16-byte aligned
    assert w(fake, fake, fake, fake, fake, 4, 1, 96, 16, 8, 0, None, None) == 2  # head_dim 96
    assert w(None, None, None, None, None, 0, 1, 128, 16, 8, 2, None, None) == 0  # T = 0, E5M2
    d = lib.kvq_paged_decode_attention_per_token
    d.restype = i
    d.argtypes = [p, p, p, p, p, p, i, i, i, i, i, i, i64, f32, i, i, i, p, sz, p, p]
    args = [1, 8, 2, 128, 16, 4, 64, 0.088, -1]
    assert d(*[fake] * 6, *args, 1, 0, fake, 1 << 30, None, None) == 1  # BF16 cache
    assert d(fake, fake, None, *[fake] * 3, *args, 0, 0, fake, 1 << 30, None, None) == 1  # no V cache
    assert d(fake, fake, odd, *[fake] * 3, *args, 0, 0, fake, 1 << 30, None, None) == 1  # V cache misaligned
    assert d(*[fake] * 6, *args, 0, 0, fake, 16, None, None) == 1  # workspace too small


def test_append_entry_point_validates_without_gpu(lib):
    """The decode-with-append call refuses a missing new token or slot array
    before any CUDA call (all other arguments valid)."""
    p = ctypes.c_void_p
    i, i64, f32, sz = ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
    d = lib.kvq_paged_decode_attention_append
    d.restype = i
    d.argtypes = [p, p, p, p, p, p, p, p, p, p, p, i, i, i, i, i, i, i64, f32, i, i, i, p, sz, p, p]
    fake = ctypes.c_void_p(1 << 20)  # never dereferenced: the calls return first
    sizes = [1, 8, 2, 128, 16, 4, 64, 0.088, -1, 0, 0]  # B Hq Hkv D P max_blocks num_blocks sm window E4M3 splits
    assert d(fake, None, fake, fake, *([fake] * 7), *sizes, fake, 1 << 30, None, None) == 1  # no k_new
    assert d(fake, fake, fake, None, *([fake] * 7), *sizes, fake, 1 << 30, None, None) == 1  # no slot_new
    bad_d = list(sizes)
    bad_d[3] = 96
    assert d(fake, fake, fake, fake, *([fake] * 7), *bad_d, fake, 1 << 30, None, None) == 2  # head_dim 96


def test_per_token_prefill_validates_without_gpu(lib):
    """The per-token prefill refuses missing caches, a BF16 cache and head
    dim 256 before any CUDA call; an empty batch of new tokens is a no-op."""
    p = ctypes.c_void_p
    i, i64, f32 = ctypes.c_int, ctypes.c_int64, ctypes.c_float
    f = lib.kvq_prefill_attention_per_token
    f.restype = i
    f.argtypes = [p, p, p, p, p, p, p, p, i, i, i, i, i, i, i64, i, f32, i, i, p, p]
    fake = ctypes.c_void_p(1 << 20)  # never dereferenced: the calls return first
    dims = [1, 8, 2, 128, 16, 4, 64, 16, 0.088, 1]  # B Hq Hkv D P max_blocks num_blocks max_q sm causal
    assert f(fake, fake, fake, None, *[fake] * 4, *dims, 0, None, None) == 1  # no V cache
    assert f(*[fake] * 8, *dims, 1, None, None) == 2  # BF16 cache
    d256 = list(dims)
    d256[3] = 256
    assert f(*[fake] * 8, *d256, 0, None, None) == 2  # head dim 256
    empty = list(dims)
    empty[7] = 0
    assert f(*[None] * 8, *empty, 0, None, None) == 0
