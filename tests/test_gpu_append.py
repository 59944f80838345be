"""kvq_paged_decode_attention_append: one decode step that writes the step's
new token into the cache itself.  Checked against

* the oracle: cache bytes bit-exact (the oracle's cache of every token, in
  the device page format) and the output within the decode tolerance of the
  mirrored oracle;
* the two-call path (kvq_reshape_and_cache of the new tokens, then
  kvq_paged_decode_attention): identical cache bytes and a bit-identical
  output;
* a sequence whose new token has no slot (-1): nothing written, the rest
  computed.
"""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import layout
from oracle.kv_cache import BF16, FP8, FP8_E5M2
from tests.kvq_testlib import SENTINEL, assert_close, f32, oracle_cache, oracle_decode

pytestmark = pytest.mark.gpu


def _k():
    import fp8_kv_cache_reshape_gb300 as k
    return k


def _split(case):
    """Indices of each sequence's last token (the step's new token) and of
    all the others (already cached)."""
    lens = case.seq_lens.tolist()
    offs = np.concatenate([[0], np.cumsum(lens)])
    last = torch.tensor([offs[b] + L - 1 for b, L in enumerate(lens)], dtype=torch.int64)
    mask = torch.ones(int(offs[-1]), dtype=torch.bool)
    mask[last] = False
    return last, torch.nonzero(mask).flatten()


def _prepare(case):
    k = _k()
    cfg = case.cfg
    kd, vd = k.alloc_kv_cache(case.num_blocks, cfg.kv_heads, cfg.head_dim, case.cache_dtype, fill=SENTINEL)
    last, rest = _split(case)
    ks, vs = case.k_scale.cuda(), case.v_scale.cuda()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    if rest.numel():
        k.kvq_reshape_and_cache(case.k[rest].cuda(), case.v[rest].cuda(), case.slot_mapping[rest].cuda(), kd, vd,
                                ks, vs, case.cache_dtype, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return kd, vd, last, ks, vs


def _two_calls(case, kd, vd, last, ks, vs, slot_new):
    k = _k()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    k.kvq_reshape_and_cache(case.k[last].cuda(), case.v[last].cuda(), slot_new, kd, vd, ks, vs, case.cache_dtype,
                            dev_status=st)
    out = torch.empty(case.q.shape, dtype=torch.bfloat16, device="cuda")
    k.kvq_paged_decode_attention(case.q.cuda(), kd, vd, ks, vs, case.block_table.cuda(), case.seq_lens.cuda(), out,
                                 num_blocks=case.num_blocks, sm_scale=case.sm_scale, window=case.window,
                                 cache_dtype=case.cache_dtype, dev_status=st)
    torch.cuda.synchronize()
    return out, int(st.item())


def _append(case, kd, vd, last, ks, vs, slot_new):
    k = _k()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.empty(case.q.shape, dtype=torch.bfloat16, device="cuda")
    k.kvq_paged_decode_attention_append(case.q.cuda(), case.k[last].cuda(), case.v[last].cuda(), slot_new, kd, vd,
                                        ks, vs, case.block_table.cuda(), case.seq_lens.cuda(), out,
                                        num_blocks=case.num_blocks, sm_scale=case.sm_scale, window=case.window,
                                        cache_dtype=case.cache_dtype, dev_status=st)
    torch.cuda.synchronize()
    return out, int(st.item())


CASES = {
    "llama_small": (dict(batch=2, q_heads=32, kv_heads=8, head_dim=128, context=1000, outliers=4), [1000, 333], FP8, -1),
    "ragged_g4": (dict(batch=5, q_heads=8, kv_heads=2, head_dim=128, context=2049), [1, 16, 17, 250, 2049], FP8, -1),
    "e5m2_d64": (dict(batch=3, q_heads=16, kv_heads=2, head_dim=64, context=777), [777, 5, 300], FP8_E5M2, -1),
    "window_bf16_d64": (dict(batch=4, q_heads=64, kv_heads=8, head_dim=64, context=1000), [50, 128, 129, 1000],
                        BF16, 128),
}


@pytest.mark.parametrize("name", list(CASES))
def test_append_matches_oracle_and_two_calls(name):
    kw, lengths, dtype, window = CASES[name]
    case = W.decode_case(W.DecodeConfig("app_" + name, **kw), lengths=lengths, cache_dtype=dtype, window=window)
    kd, vd, last, ks, vs = _prepare(case)
    kd2, vd2 = kd.clone(), vd.clone()
    slot_new = case.slot_mapping[last].cuda()
    got, st = _append(case, kd, vd, last, ks, vs, slot_new)
    assert st == 0
    ref_out, st2 = _two_calls(case, kd2, vd2, last, ks, vs, slot_new)
    assert st2 == 0
    assert torch.equal(kd, kd2) and torch.equal(vd, vd2), "cache bytes differ from the two-call path"
    assert torch.equal(got.view(torch.int16), ref_out.view(torch.int16)), "output differs from the two-call path"
    kc, vc = oracle_cache(case)
    ek, ev = layout.to_device_format(kc, vc)
    assert np.array_equal(kd.cpu().numpy(), ek) and np.array_equal(vd.cpu().numpy(), ev), "cache bytes vs oracle"
    ref, _ = oracle_decode(case, kc, vc, mode="mirror")
    assert_close(f32(got), ref, what="append vs mirrored oracle")


def test_append_without_slot_writes_nothing():
    kw, lengths, dtype, window = CASES["ragged_g4"]
    case = W.decode_case(W.DecodeConfig("app_noslot", **kw), lengths=lengths, cache_dtype=dtype, window=window)
    kd, vd, last, ks, vs = _prepare(case)
    kd2, vd2 = kd.clone(), vd.clone()
    slot_new = case.slot_mapping[last].clone()
    slot_new[3] = -1
    slot_new = slot_new.cuda()
    got, st = _append(case, kd, vd, last, ks, vs, slot_new)
    ref_out, st2 = _two_calls(case, kd2, vd2, last, ks, vs, slot_new)
    assert st == 0 and st2 == 0
    assert torch.equal(kd, kd2) and torch.equal(vd, vd2)
    assert torch.equal(got.view(torch.int16), ref_out.view(torch.int16))


@pytest.mark.parametrize("where", ["other_page", "wrong_offset"])
def test_append_slot_not_the_last_tokens_is_reported_and_not_written(where):
    """The new token's slot must be the last token's slot under the block
    table (the page the call reads back).  A slot elsewhere -- another page
    of the sequence, or the right page at another offset -- sets
    KVQ_DEV_BAD_SLOT and writes nothing; the result is that of the two-call
    path with that token skipped."""
    kw, lengths, dtype, window = CASES["ragged_g4"]
    case = W.decode_case(W.DecodeConfig("app_badslot", **kw), lengths=lengths, cache_dtype=dtype, window=window)
    kd, vd, last, ks, vs = _prepare(case)
    kd2, vd2 = kd.clone(), vd.clone()
    slot_new = case.slot_mapping[last].clone()
    b = 4  # 2,049 tokens: the last token is alone in page 128
    good = int(slot_new[b])
    if where == "other_page":
        slot_new[b] = int(case.slot_mapping[last[b] - 20])  # token 2,028 sits in page 126
    else:
        slot_new[b] = good - good % 16 + 5  # the right page, offset 5 instead of 0
    got, st = _append(case, kd, vd, last, ks, vs, slot_new.cuda())
    assert st & 0x1, f"status {st:#x}"
    skipped = slot_new.clone()
    skipped[b] = -1
    ref_out, st2 = _two_calls(case, kd2, vd2, last, ks, vs, skipped.cuda())
    assert st2 == 0
    assert torch.equal(kd, kd2) and torch.equal(vd, vd2), "a slot that is not the last token's was written"
    assert torch.equal(got.view(torch.int16), ref_out.view(torch.int16))
