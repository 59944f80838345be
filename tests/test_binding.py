"""The Python binding checks its arguments before anything reaches the
library: CPU tensors, non-contiguous tensors, and wrongly shaped new tokens
for the append call are refused with ValueError (no GPU needed)."""
import pytest
import torch


def _k():
    import fp8_kv_cache_reshape_gb300 as k
    return k


def _decode_args(q):
    cache = torch.zeros(4, 2, 2048, dtype=torch.uint8)
    return (q, cache, cache.clone(), torch.ones(2), torch.ones(2), torch.zeros(2, 4, dtype=torch.int32),
            torch.ones(2, dtype=torch.int32), torch.empty_like(q))


def test_cpu_tensors_are_refused():
    k = _k()
    q = torch.zeros(2, 8, 128, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA"):
        k.kvq_paged_decode_attention(*_decode_args(q))


def test_non_contiguous_tensor_is_refused():
    k = _k()
    with pytest.raises(ValueError):
        k._ptr(torch.zeros(4, 4).t())


@pytest.mark.parametrize("bad", ["dtype", "shape", "slots"])
def test_append_new_token_shapes_are_checked(bad):
    k = _k()
    q = torch.zeros(2, 8, 128, dtype=torch.bfloat16)
    kn = torch.zeros(2, 2, 128, dtype=torch.float32 if bad == "dtype" else torch.bfloat16)
    if bad == "shape":
        kn = torch.zeros(2, 2, 64, dtype=torch.bfloat16)
    vn = torch.zeros(2, 2, 128, dtype=torch.bfloat16)
    slots = torch.zeros(3 if bad == "slots" else 2, dtype=torch.int64)
    q_, kc, vc, ks, vs, bt, sl, out = _decode_args(q)
    with pytest.raises(ValueError):
        k.kvq_paged_decode_attention_append(q_, kn, vn, slots, kc, vc, ks, vs, bt, sl, out)
