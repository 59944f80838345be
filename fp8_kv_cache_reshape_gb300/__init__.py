"""Python binding of libkvq (include/kvq.h): FP8 E4M3 KV-cache quantization
and attention over a paged FP8 / BF16 KV cache on GB300 (sm_103a).

The functions below carry the C ABI's names and only marshal arguments:
shapes and device pointers are read from torch tensors, the current CUDA
stream is passed through, and a non-zero status raises KvqError with the
library's message.  Every step runs in the library's CUDA kernels; there is
no fallback.  PyTorch provides device memory and streams.

Build the library first (``python -c "import __graft_entry__ as g; g.build()"``
or ``python fp8_kv_cache_reshape_gb300/_build.py``); importing this module
without it raises ImportError.
"""
from __future__ import annotations

import ctypes
import math
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libkvq.so")

KVQ_OK = 0
KVQ_ERR_INVALID_ARG = 1
KVQ_ERR_UNSUPPORTED = 2
KVQ_ERR_CUDA = 3
KVQ_ERR_DEVICE_FAULT = 4

KVQ_DTYPE_FP8_E4M3 = 0
KVQ_DTYPE_BF16 = 1
KVQ_DTYPE_FP8_E5M2 = 2

KVQ_ACC_TWO_LEVEL = 0
KVQ_ACC_SINGLE_LEVEL = 1

KVQ_DEV_BAD_SLOT = 0x1
KVQ_DEV_BAD_BLOCK = 0x2
KVQ_DEV_BAD_SEQLEN = 0x4
KVQ_DEV_TIMEOUT = 0x8
KVQ_DEV_BAD_QROWS = 0x10

PAGE = 16

if not os.path.exists(LIB_PATH):
    raise ImportError(f"libkvq.so is not built ({LIB_PATH}); run fp8_kv_cache_reshape_gb300/_build.py")

lib = ctypes.CDLL(LIB_PATH)

_p = ctypes.c_void_p
_i = ctypes.c_int
_i64 = ctypes.c_int64
_f = ctypes.c_float
_sz = ctypes.c_size_t

lib.kvq_version.restype = _i
lib.kvq_version.argtypes = []
lib.kvq_last_error_string.restype = ctypes.c_char_p
lib.kvq_last_error_string.argtypes = []
lib.kvq_debug_set_stall_ns.restype = None
lib.kvq_debug_set_stall_ns.argtypes = [ctypes.c_uint64]
lib.kvq_reshape_and_cache.restype = _i
lib.kvq_reshape_and_cache.argtypes = [_p, _p, _p, _p, _p, _p, _p, _i, _i, _i, _i, _i64, _i, _p, _p]
lib.kvq_quantize_query.restype = _i
lib.kvq_quantize_query.argtypes = [_p, _p, _p, _i64, _p]
lib.kvq_decode_num_splits.restype = _i
lib.kvq_decode_num_splits.argtypes = [_i, _i, _i, _i, _i, _i, _i]
lib.kvq_decode_workspace_size.restype = _sz
lib.kvq_decode_workspace_size.argtypes = [_i, _i, _i, _i, _i, _i, _i, _i]
lib.kvq_paged_decode_attention.restype = _i
lib.kvq_paged_decode_attention.argtypes = [_p, _p, _p, _p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _i64, _f,
                                           _i, _i, _i, _p, _sz, _p, _p]
lib.kvq_decode_static_scratch_bytes.restype = _sz
lib.kvq_decode_static_scratch_bytes.argtypes = []
lib.kvq_paged_decode_attention_static_scratch.restype = _i
lib.kvq_paged_decode_attention_static_scratch.argtypes = [_p, _p, _p, _p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i,
                                                          _i64, _f, _i, _i, _i, _p, _p]
lib.kvq_reshape_and_cache_per_token.restype = _i
lib.kvq_reshape_and_cache_per_token.argtypes = [_p, _p, _p, _p, _p, _i, _i, _i, _i, _i64, _i, _p, _p]
lib.kvq_paged_decode_attention_per_token.restype = _i
lib.kvq_paged_decode_attention_per_token.argtypes = [_p, _p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _i64,
                                                     _f, _i, _i, _i, _p, _sz, _p, _p]
lib.kvq_paged_decode_attention_append.restype = _i
lib.kvq_paged_decode_attention_append.argtypes = [_p, _p, _p, _p, _p, _p, _p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i,
                                                  _i64, _f, _i, _i, _i, _p, _sz, _p, _p]
lib.kvq_paged_decode_attention_acc.restype = _i
lib.kvq_paged_decode_attention_acc.argtypes = lib.kvq_paged_decode_attention.argtypes + [_i]
lib.kvq_prefill_attention_acc.restype = _i
lib.kvq_prefill_attention_acc.argtypes = [_p, _p, _p, _p, _p, _p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _i64, _i,
                                          _f, _i, _p, _p, _i]
lib.kvq_prefill_attention_dtype.restype = _i
lib.kvq_prefill_attention_dtype.argtypes = [_p, _p, _p, _p, _p, _p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _i64, _i,
                                            _f, _i, _p, _p, _i]
lib.kvq_prefill_attention_per_token.restype = _i
lib.kvq_prefill_attention_per_token.argtypes = [_p, _p, _p, _p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _i64, _i,
                                                _f, _i, _i, _p, _p]
lib.kvq_prefill_attention.restype = _i
lib.kvq_prefill_attention.argtypes = [_p, _p, _p, _p, _p, _p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _i64, _i,
                                      _f, _i, _p, _p]


class KvqError(RuntimeError):
    def __init__(self, status: int, where: str):
        msg = lib.kvq_last_error_string().decode(errors="replace")
        super().__init__(f"{where}: status {status}: {msg}")
        self.status = status


def _check(status: int, where: str):
    if status != KVQ_OK:
        raise KvqError(status, where)


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("libkvq takes CUDA tensors only")
    if not t.is_contiguous():
        raise ValueError("libkvq takes contiguous tensors only")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _dtype_code(cache_dtype: str) -> int:
    if cache_dtype in ("fp8", "fp8_e4m3", KVQ_DTYPE_FP8_E4M3):
        return KVQ_DTYPE_FP8_E4M3
    if cache_dtype in ("bf16", "bfloat16", KVQ_DTYPE_BF16):
        return KVQ_DTYPE_BF16
    if cache_dtype in ("fp8_e5m2", KVQ_DTYPE_FP8_E5M2):
        return KVQ_DTYPE_FP8_E5M2
    raise ValueError(f"unknown cache dtype {cache_dtype!r}")


def _acc_code(accumulation) -> int:
    if accumulation in ("two_level", KVQ_ACC_TWO_LEVEL):
        return KVQ_ACC_TWO_LEVEL
    if accumulation in ("single_level", KVQ_ACC_SINGLE_LEVEL):
        return KVQ_ACC_SINGLE_LEVEL
    raise ValueError(f"unknown accumulation mode {accumulation!r}")


def version() -> int:
    return lib.kvq_version()


def kvq_debug_set_stall_ns(ns: int):
    """Failure-path test hook (include/kvq.h): > 0 makes later decode and
    prefill launches fail one bounded wait after `ns` nanoseconds; 0 = off."""
    lib.kvq_debug_set_stall_ns(int(ns))


# per-token scale tail of a V page: 16 K scales and 16 V scales, float32
SCALE_TAIL_BYTES = 2 * PAGE * 4


def alloc_kv_cache(num_blocks: int, kv_heads: int, head_dim: int, cache_dtype="fp8_e4m3",
                   device="cuda", fill=None, per_token=False, paired=False):
    """Allocate (k_cache, v_cache) as uint8 tensors in the library's paged
    format ([num_blocks][Hkv][P][D] and [num_blocks][Hkv][D][P] elements).
    per_token: each V page also carries its scale tail (FP8 only).
    paired: one allocation [num_blocks][Hkv][K page | V page]; k_cache is it
    and v_cache a flat view starting one K page in (the library recognizes
    the layout from the pointers and moves each pair with one copy)."""
    esz = 2 if _dtype_code(cache_dtype) == KVQ_DTYPE_BF16 else 1
    if per_token and esz != 1:
        raise ValueError("per-token scales need an FP8 cache")
    kpage = PAGE * head_dim * esz
    vpage = kpage + (SCALE_TAIL_BYTES if per_token else 0)
    make = (lambda shape: torch.empty(shape, dtype=torch.uint8, device=device)) if fill is None else \
        (lambda shape: torch.full(shape, fill, dtype=torch.uint8, device=device))
    if paired:
        buf = make((num_blocks, kv_heads, kpage + vpage))
        return buf, buf.view(-1)[kpage:]
    return make((num_blocks, kv_heads, kpage)), make((num_blocks, kv_heads, vpage))


def _is_paired(k_cache, v_cache, kpage):
    return v_cache.data_ptr() == k_cache.data_ptr() + kpage


def _num_blocks(k_cache, v_cache, Hkv, kpage):
    """Blocks of a cache from its K tensor: [num_blocks][Hkv][...] (separate
    or paired), or flat separate pages."""
    if k_cache.dim() >= 2 or _is_paired(k_cache, v_cache, kpage):
        return k_cache.shape[0]
    return k_cache.numel() // (Hkv * kpage)


def kvq_reshape_and_cache(k, v, slot_mapping, k_cache, v_cache, k_scale=None, v_scale=None,
                          cache_dtype="fp8_e4m3", dev_status=None, stream=None):
    """Quantize (or copy) new tokens k, v (bf16 [T][Hkv][D]) into the cache."""
    T, Hkv, D = k.shape
    dt = _dtype_code(cache_dtype)
    esz = 2 if dt == KVQ_DTYPE_BF16 else 1
    num_blocks = _num_blocks(k_cache, v_cache, Hkv, PAGE * D * esz)
    _check(lib.kvq_reshape_and_cache(_ptr(k), _ptr(v), _ptr(slot_mapping), _ptr(k_cache), _ptr(v_cache),
                                     _ptr(k_scale), _ptr(v_scale), T, Hkv, D, PAGE, num_blocks, dt,
                                     _ptr(dev_status), _stream(stream)), "kvq_reshape_and_cache")


def _check_per_token_cache(k_cache, v_cache, Hkv, D):
    kpage, vpage = PAGE * D, PAGE * D + SCALE_TAIL_BYTES
    if _is_paired(k_cache, v_cache, kpage):
        nb = k_cache.shape[0]
        ok = k_cache.numel() == nb * Hkv * (kpage + vpage)
    else:
        nb = k_cache.numel() // (Hkv * kpage)
        ok = k_cache.numel() == nb * Hkv * kpage and v_cache.numel() == nb * Hkv * vpage
    if not ok:
        raise ValueError("per-token caches must be alloc_kv_cache(..., per_token=True) tensors")
    return nb


def kvq_reshape_and_cache_per_token(k, v, slot_mapping, k_cache, v_cache, cache_dtype="fp8_e4m3",
                                    dev_status=None, stream=None):
    """Quantize new tokens k, v (bf16 [T][Hkv][D]) with one dynamic scale per
    token and head; the scales go to the scale tails of the V pages."""
    T, Hkv, D = k.shape
    num_blocks = _check_per_token_cache(k_cache, v_cache, Hkv, D)
    _check(lib.kvq_reshape_and_cache_per_token(_ptr(k), _ptr(v), _ptr(slot_mapping), _ptr(k_cache), _ptr(v_cache),
                                               T, Hkv, D, PAGE, num_blocks, _dtype_code(cache_dtype),
                                               _ptr(dev_status), _stream(stream)),
           "kvq_reshape_and_cache_per_token")


def kvq_quantize_query(q, q8, q_scale, stream=None):
    """q8 = E4M3(q / q_scale), per tensor."""
    _check(lib.kvq_quantize_query(_ptr(q), _ptr(q8), _ptr(q_scale), q.numel(), _stream(stream)),
           "kvq_quantize_query")


def kvq_decode_num_splits(B, Hkv, max_blocks, window=-1, num_splits=0, head_dim=128):
    return lib.kvq_decode_num_splits(B, Hkv, head_dim, PAGE, max_blocks, window, num_splits)


def kvq_decode_workspace_size(B, Hq, Hkv, D, max_blocks, window=-1, num_splits=0):
    return lib.kvq_decode_workspace_size(B, Hq, Hkv, D, PAGE, max_blocks, window, num_splits)


def kvq_paged_decode_attention(q, k_cache, v_cache, k_scale, v_scale, block_table, seq_lens, out,
                               num_blocks=None, sm_scale=None, window=-1, cache_dtype="fp8_e4m3",
                               num_splits=0, workspace=None, dev_status=None, stream=None, accumulation=None):
    """One decode step over the paged cache; writes out (bf16 [B][Hq][D]).

    workspace: a uint8 CUDA tensor of at least kvq_decode_workspace_size()
    bytes (allocated here when omitted).  accumulation: None (the default,
    two-level) or "two_level" / "single_level" through
    kvq_paged_decode_attention_acc."""
    B, Hq, D = q.shape
    max_blocks = block_table.shape[1]
    dt = _dtype_code(cache_dtype)
    Hkv = k_cache.shape[1] if k_cache.dim() >= 3 else None
    if Hkv is None:
        raise ValueError("k_cache must be [num_blocks][Hkv][...]")
    if num_blocks is None:
        num_blocks = k_cache.shape[0]
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(D)
    need = kvq_decode_workspace_size(B, Hq, Hkv, D, max_blocks, window, num_splits)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    args = (_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale), _ptr(block_table),
            _ptr(seq_lens), _ptr(out), B, Hq, Hkv, D, PAGE, max_blocks, num_blocks, float(sm_scale), window, dt,
            num_splits, _ptr(workspace), workspace.numel(), _ptr(dev_status), _stream(stream))
    if accumulation is None:
        _check(lib.kvq_paged_decode_attention(*args), "kvq_paged_decode_attention")
    else:
        _check(lib.kvq_paged_decode_attention_acc(*args, _acc_code(accumulation)), "kvq_paged_decode_attention_acc")
    return out


def kvq_paged_decode_attention_append(q, k_new, v_new, slot_new, k_cache, v_cache, k_scale, v_scale, block_table,
                                      seq_lens, out, num_blocks=None, sm_scale=None, window=-1,
                                      cache_dtype="fp8_e4m3", num_splits=0, workspace=None, dev_status=None,
                                      stream=None):
    """One decode step that also writes the step's new token (k_new, v_new:
    bf16 [B][Hkv][D], slot_new: int64 [B]) into the cache, as
    kvq_reshape_and_cache followed by kvq_paged_decode_attention would."""
    B, Hq, D = q.shape
    max_blocks = block_table.shape[1]
    Hkv = k_cache.shape[1]
    if num_blocks is None:
        num_blocks = k_cache.shape[0]
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(D)
    for t in (k_new, v_new):
        if t.dtype != torch.bfloat16 or tuple(t.shape) != (B, Hkv, D):
            raise ValueError("k_new / v_new must be bf16 [B][Hkv][D]")
    if slot_new.dtype != torch.int64 or slot_new.numel() != B:
        raise ValueError("slot_new must be int64 [B]")
    need = kvq_decode_workspace_size(B, Hq, Hkv, D, max_blocks, window, num_splits)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    _check(lib.kvq_paged_decode_attention_append(
        _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(slot_new), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale),
        _ptr(v_scale), _ptr(block_table), _ptr(seq_lens), _ptr(out), B, Hq, Hkv, D, PAGE, max_blocks, num_blocks,
        float(sm_scale), window, _dtype_code(cache_dtype), num_splits, _ptr(workspace), workspace.numel(),
        _ptr(dev_status), _stream(stream)), "kvq_paged_decode_attention_append")
    return out


def kvq_paged_decode_attention_per_token(q, k_cache, v_cache, block_table, seq_lens, out, num_blocks=None,
                                         sm_scale=None, window=-1, cache_dtype="fp8_e4m3", num_splits=0,
                                         workspace=None, dev_status=None, stream=None):
    """Decode over a cache written by kvq_reshape_and_cache_per_token."""
    B, Hq, D = q.shape
    max_blocks = block_table.shape[1]
    Hkv = k_cache.shape[1]
    if num_blocks is None:
        num_blocks = k_cache.shape[0]
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(D)
    need = kvq_decode_workspace_size(B, Hq, Hkv, D, max_blocks, window, num_splits)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    _check(lib.kvq_paged_decode_attention_per_token(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table),
        _ptr(seq_lens), _ptr(out), B, Hq, Hkv, D, PAGE, max_blocks, num_blocks, float(sm_scale), window,
        _dtype_code(cache_dtype), num_splits, _ptr(workspace), workspace.numel(), _ptr(dev_status),
        _stream(stream)), "kvq_paged_decode_attention_per_token")
    return out


def kvq_prefill_attention(q8, q_scale, k_cache, v_cache, k_scale, v_scale, block_table, cu_seqlens_q,
                          seq_lens, out, max_q_tokens, num_blocks=None, sm_scale=None, causal=True,
                          dev_status=None, stream=None, accumulation=None, cache_dtype="fp8_e4m3"):
    """Chunked causal prefill over the FP8 cache; writes out (bf16 [Tq][Hq][D]).
    accumulation: None (two-level) or "two_level" / "single_level" through
    kvq_prefill_attention_acc.  cache_dtype "fp8_e5m2" goes through
    kvq_prefill_attention_dtype (with the default accumulation)."""
    Tq, Hq, D = q8.shape
    B = cu_seqlens_q.numel() - 1
    Hkv = k_cache.shape[1]
    if num_blocks is None:
        num_blocks = k_cache.shape[0]
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(D)
    args = (_ptr(q8), _ptr(q_scale), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale),
            _ptr(block_table), _ptr(cu_seqlens_q), _ptr(seq_lens), _ptr(out), B, Hq, Hkv, D, PAGE,
            block_table.shape[1], num_blocks, int(max_q_tokens), float(sm_scale), 1 if causal else 0,
            _ptr(dev_status), _stream(stream))
    dt = _dtype_code(cache_dtype)
    if dt != KVQ_DTYPE_FP8_E4M3:
        if accumulation is not None:
            raise ValueError("an explicit accumulation mode takes an E4M3 cache")
        _check(lib.kvq_prefill_attention_dtype(*args, dt), "kvq_prefill_attention_dtype")
    elif accumulation is None:
        _check(lib.kvq_prefill_attention(*args), "kvq_prefill_attention")
    else:
        _check(lib.kvq_prefill_attention_acc(*args, _acc_code(accumulation)), "kvq_prefill_attention_acc")
    return out


def kvq_prefill_attention_per_token(q8, q_scale, k_cache, v_cache, block_table, cu_seqlens_q, seq_lens, out,
                                    max_q_tokens, num_blocks=None, sm_scale=None, causal=True,
                                    cache_dtype="fp8_e4m3", dev_status=None, stream=None):
    """Chunked causal prefill over a cache written by
    kvq_reshape_and_cache_per_token; writes out (bf16 [Tq][Hq][D])."""
    Tq, Hq, D = q8.shape
    B = cu_seqlens_q.numel() - 1
    Hkv = k_cache.shape[1]
    if num_blocks is None:
        num_blocks = k_cache.shape[0]
    _check_per_token_cache(k_cache, v_cache, Hkv, D)
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(D)
    _check(lib.kvq_prefill_attention_per_token(
        _ptr(q8), _ptr(q_scale), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), _ptr(cu_seqlens_q),
        _ptr(seq_lens), _ptr(out), B, Hq, Hkv, D, PAGE, block_table.shape[1], num_blocks, int(max_q_tokens),
        float(sm_scale), 1 if causal else 0, _dtype_code(cache_dtype), _ptr(dev_status), _stream(stream)),
        "kvq_prefill_attention_per_token")
    return out
