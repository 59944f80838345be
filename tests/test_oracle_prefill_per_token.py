"""Pins of the oracle's prefill over per-token-scaled caches
(attention.prefill_per_token).

* A special case that reduces to the per-head path: when every token of a
  KV head has the same K scale and the same V scale, both powers of two,
  the per-token score coefficient equals the per-head one exactly, C_t is
  the V scale, the weighted and unweighted probability codes coincide, and
  the result is attention.prefill(mode="final") with those per-head scales,
  bit for bit -- over several 128-key groups, causal rows and GQA.
* Against the definition: with real per-token scales (the oracle's cache
  write of random tokens, a few ×20 outlier tokens), "final" stays within
  the rounding of the E4M3 probabilities of "pure" (the exact softmax over
  the dequantized values), and a scale attached to the wrong token would
  not: the same check fails for a cache whose V scales are shifted by one
  token.
* "mirror" (the tile walk with a running stabilizer) with power-of-two
  scales per head is per-head prefill's mirror; with real per-token scales
  it stays within the same rounding bound of pure.
* The last causal row attends to every cached key: it equals per-token
  decode over the same keys (pure modes, up to decode's float32 query),
  and its "final" result is within the same bound of it.
"""
import numpy as np
import pytest
import torch

from oracle import attention, kv_cache

P = 16


def _bf16(a):
    return torch.from_numpy(np.asarray(a, np.float32)).bfloat16().float().numpy()


def _case(nq, nc, Hq=4, Hkv=2, D=32, seed=0, outliers=0, qs=0.02, cache_dtype=kv_cache.FP8):
    rng = np.random.default_rng(seed)
    L = nq + nc
    pages = -(-L // P)
    nb = pages + 3
    bt = rng.permutation(nb)[:pages].astype(np.int32)[None, :]
    slots = bt[0][np.arange(L) // P].astype(np.int64) * P + np.arange(L) % P
    k = rng.standard_normal((L, Hkv, D))
    v = rng.standard_normal((L, Hkv, D))
    if outliers:
        idx = rng.choice(L, outliers, replace=False)
        k[idx] *= 20.0
        v[idx] *= 20.0
    k, v = _bf16(k), _bf16(v)
    kc = np.zeros((nb, Hkv, P, D), np.uint8)
    vc = np.zeros((nb, Hkv, D, P), np.uint8)
    sc = np.zeros((nb, Hkv, 2, P), np.float32)
    kv_cache.reshape_and_cache_per_token(k, v, slots, kc, vc, sc, cache_dtype)
    q8 = kv_cache.quantize_query(_bf16(rng.standard_normal((nq, Hq, D)) * 2.0), np.float32(qs))
    return dict(q8=q8, qs=np.float32(qs), kc=kc, vc=vc, sc=sc, bt=bt, cu=np.array([0, nq]),
                sl=np.array([L], np.int32), L=L, nq=nq, dtype=cache_dtype)


def _pt(c, sc=None, **kw):
    return attention.prefill_per_token(c["q8"], c["qs"], c["kc"], c["vc"], c["sc"] if sc is None else sc, c["bt"],
                                       c["cu"], c["sl"], 0.25, cache_dtype=c["dtype"], **kw)


def test_power_of_two_scales_per_head_reduce_to_per_head_prefill_bit_for_bit():
    c = _case(nq=150, nc=300, seed=1)
    Hkv = c["kc"].shape[1]
    ks = np.array([2.0 ** -6, 2.0 ** -5], np.float32)[:Hkv]
    vs = np.array([2.0 ** -7, 2.0 ** -4], np.float32)[:Hkv]
    sc = np.zeros_like(c["sc"])
    sc[:, :, 0, :] = ks[None, :, None]
    sc[:, :, 1, :] = vs[None, :, None]
    got = _pt(c, sc=sc, mode="final")
    ref = attention.prefill(c["q8"], c["qs"], c["kc"], c["vc"], ks, vs, c["bt"], c["cu"], c["sl"], 0.25,
                            mode="final")
    assert np.all(np.isfinite(got))
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("dtype", [kv_cache.FP8, kv_cache.FP8_E5M2])
def test_final_is_within_the_probability_rounding_of_pure(dtype):
    c = _case(nq=100, nc=320, seed=2, outliers=6, cache_dtype=dtype)
    fin = _pt(c, mode="final")
    pure = _pt(c, mode="pure")
    L, Hkv, D = c["L"], c["kc"].shape[1], c["kc"].shape[3]
    # every weight carries at most half an E4M3 ulp (2^-4 relative), in the
    # numerator and in the row sum: |final - pure| <= 2^-3 * max |v_hat|
    vmax = np.zeros(Hkv)
    for kv in range(Hkv):
        kk, vv = kv_cache.gather_tokens(c["kc"], c["vc"], c["bt"][0], np.arange(L), kv)
        sv = kv_cache.gather_scales(c["sc"][:, :, 1], c["bt"][0], np.arange(L), kv)
        vmax[kv] = np.max(np.abs(kv_cache.codec(dtype).decode(vv) * sv[:, None]))
    g = c["q8"].shape[1] // Hkv
    bound = 2.0 ** -3 * np.repeat(vmax, g)[None, :, None]
    err = np.abs(fin - pure)
    assert np.all(err <= bound), float(np.max(err / bound))
    assert err.mean() <= 2.0 ** -7 * vmax.max()
    # a V scale attached to its neighbour token breaks the bound
    bad = c["sc"].copy()
    bad[:, :, 1, :] = np.roll(bad[:, :, 1, :], 1, axis=-1)
    err_bad = np.abs(_pt(c, sc=bad, mode="final") - pure)
    assert err_bad.mean() > 4 * err.mean()


def test_last_row_equals_per_token_decode_over_the_same_keys():
    c = _case(nq=40, nc=500, Hq=8, Hkv=2, seed=3, outliers=3)
    t = c["nq"] - 1
    rows = [(t, h) for h in range(c["q8"].shape[1])]
    pure = _pt(c, mode="pure", rows=rows)[t]
    fin = _pt(c, mode="final", rows=rows)[t]
    q = c["q8"][t][None].astype(np.uint8)
    from oracle import e4m3
    qf = (e4m3.decode(q) * float(c["qs"])).astype(np.float32)
    dec, _ = attention.paged_decode_per_token(qf, c["kc"], c["vc"], c["sc"], c["bt"], c["sl"], 0.25, mode="pure")
    # the decode oracle takes q as float32 values (decode(q8) * q_scale rounded once)
    assert np.allclose(pure, dec[0], rtol=1e-6, atol=1e-9)
    vmax = np.max(np.abs(dec))
    assert np.max(np.abs(fin - dec[0])) <= 2.0 ** -3 * vmax + 1e-12


def test_mirror_with_power_of_two_scales_is_per_head_mirror_and_bounded_otherwise():
    c = _case(nq=150, nc=300, seed=4)
    Hkv = c["kc"].shape[1]
    ks = np.array([2.0 ** -6, 2.0 ** -5], np.float32)[:Hkv]
    vs = np.array([2.0 ** -7, 2.0 ** -4], np.float32)[:Hkv]
    sc = np.zeros_like(c["sc"])
    sc[:, :, 0, :] = ks[None, :, None]
    sc[:, :, 1, :] = vs[None, :, None]
    mir = _pt(c, sc=sc, mode="mirror")
    ref = attention.prefill(c["q8"], c["qs"], c["kc"], c["vc"], ks, vs, c["bt"], c["cu"], c["sl"], 0.25,
                            mode="mirror")
    assert np.all(np.isfinite(mir))
    assert np.allclose(mir, ref, rtol=1e-13, atol=0.0)  # float64 summation order only
    c2 = _case(nq=100, nc=320, seed=2, outliers=6)
    mir2 = _pt(c2, mode="mirror")
    pure2 = _pt(c2, mode="pure")
    assert np.all(np.isfinite(mir2))
    assert np.max(np.abs(mir2 - pure2)) <= 2.0 ** -3 * np.max(np.abs(pure2))
