"""Pins of the oracle's chunked prefill across several key tiles.

The mirrored prefill walks the keys in tiles (an online softmax: a running
integer stabilizer M = ceil(max s2), rescale a = 2^(M_old - M_new) of the
earlier numerator and row sum, P8 against the running M).  These tests tie
that loop to things it does not share code with:

* E4M3 rounding commutes with multiplication by a power of two wherever
  both values are normal -- checked on every code;
* without P rounding the loop is exact arithmetic on the same softmax, so
  every tile size (16, 128, one tile) gives the single-pass result, and the
  single-pass result equals the unquantized-P "pure" attention up to the
  float32 score coefficient -- a rescale applied to the row sum but not to the
  numerator, or a tile boundary off by one, breaks this at once;
* with P rounding every tile size still gives the single-pass ("final")
  result, because the rescales are exact powers of two;
* with the row maximum planted at key 0 the stabilizer is final from the
  first tile on, and with every key in one tile the loop is the single-pass
  formula, bit for bit;
* brute force: pure-Python loops over each key with math.exp2 and the
  brute-force E4M3 encoder (a scan of all 127 codes) at about 300 keys.
"Performance benchmarks" of "The state of FP8 KV-cache and attention
quantization in vLLM" names the online-softmax rescaling; the P8 reading
(x256 against an integer stabilizer, RNE, saturating) is this library's.
"""
import math

import numpy as np
import pytest
import torch

from oracle import attention, e4m3, kv_cache


def _bf16(a):
    return torch.from_numpy(np.asarray(a, np.float32)).bfloat16().float().numpy()


def _case(nq, nc, Hq=4, Hkv=2, D=16, P=16, seed=0, k=None, q8=None, qs=0.02, ks=(0.01, 0.02), vs=(0.015, 0.03),
          qmag=2.0):
    """A single-sequence prefill case built with the oracle's cache write;
    K may be given (bf16 values) and q8 may be given as codes."""
    rng = np.random.default_rng(seed)
    L = nq + nc
    pages = -(-L // P)
    nb = pages + 3
    bt = rng.permutation(nb)[:pages].astype(np.int32)[None, :]
    slots = bt[0][np.arange(L) // P].astype(np.int64) * P + np.arange(L) % P
    if k is None:
        k = _bf16(rng.standard_normal((L, Hkv, D)))
    v = _bf16(rng.standard_normal((L, Hkv, D)))
    kc = np.zeros((nb, Hkv, P, D), np.uint8)
    vc = np.zeros((nb, Hkv, D, P), np.uint8)
    ks = np.asarray(ks, np.float32)
    vs = np.asarray(vs, np.float32)
    kv_cache.reshape_and_cache(k, v, slots, kc, vc, ks, vs)
    if q8 is None:
        q8 = kv_cache.quantize_query(_bf16(rng.standard_normal((nq, Hq, D)) * qmag), np.float32(qs))
    return dict(q8=q8, qs=np.float32(qs), kc=kc, vc=vc, ks=ks, vs=vs, bt=bt, cu=np.array([0, nq]),
                sl=np.array([L], np.int32), L=L, nq=nq)


def _run(c, **kw):
    return attention.prefill(c["q8"], c["qs"], c["kc"], c["vc"], c["ks"], c["vs"], c["bt"], c["cu"], c["sl"],
                             0.25, **kw)


def _row_scores(c, t, h):
    """Base-2 scores of one row from the codes, independent of attention.prefill."""
    Hq, Hkv = c["q8"].shape[1], c["kc"].shape[1]
    kv = h // (Hq // Hkv)
    kk, _ = kv_cache.gather_tokens(c["kc"], c["vc"], c["bt"][0], np.arange(c["L"]), kv)
    n = c["L"] - c["nq"] + t + 1
    coef = float(attention.prefill_score_coef(c["qs"], c["ks"][kv], 0.25))
    return (e4m3.decode(kk[:n]) @ e4m3.decode(c["q8"][t, h])) * coef


def test_e4m3_rounding_commutes_with_powers_of_two_in_the_normal_range():
    """decode(encode(x * 2^k)) = decode(encode(x)) * 2^k when x and x * 2^k lie
    in [2^-6, 448): every float32 between neighbouring codes and at their
    midpoints rounds the same way after an exact binary shift."""
    vals = e4m3.decode(np.arange(0x08, 0x7E))  # normal codes below 448
    mids = 0.5 * (vals[:-1] + vals[1:])
    xs = np.concatenate([vals, mids, np.nextafter(mids, 0), np.nextafter(mids, 1e9)]).astype(np.float32)
    for k in range(-8, 9):
        y = (xs.astype(np.float64) * 2.0 ** k)
        ok = (xs >= 2.0 ** -6) & (y >= 2.0 ** -6) & (y < 448) & (xs < 448)
        a = e4m3.decode(e4m3.encode(y[ok].astype(np.float32)))
        b = e4m3.decode(e4m3.encode(xs[ok])) * 2.0 ** k
        assert np.array_equal(a, b), k


def test_tile_loop_without_p_rounding_is_the_single_pass_softmax():
    c = _case(nq=48, nc=400, seed=1)  # rows of 401 .. 448 keys: 26 .. 28 tiles of 16
    # the stabilizer does move between tiles in these rows
    moved = sum(np.ceil(np.max(_row_scores(c, t, h)[:16])) < np.ceil(np.max(_row_scores(c, t, h)))
                for t in (0, 20, 47) for h in range(4))
    assert moved >= 10
    single = _run(c, mode="final", quantize_p=False)
    pure = _run(c, mode="pure")
    for tile in (16, 128, 1000):
        loop = _run(c, mode="mirror", tile=tile, quantize_p=False)
        assert np.allclose(loop, single, rtol=1e-12, atol=1e-14), tile
    # the float32 score coefficient is the only difference from the pure definition
    assert np.max(np.abs(single - pure)) < 1e-5 * np.max(np.abs(pure))


def test_tile_loop_with_p_rounding_is_the_single_pass_result():
    """Every rescale is an exact power of two, so P8 against the running
    stabilizer, rescaled, is P8 against the final one wherever p * 256 is a
    normal E4M3 input (>= 2^-6): rows whose probabilities all stay there
    give the single-pass result for any tiling; in the others each key below
    2^-6 can differ by one subnormal step, 2^-9 / 256 in p, so the row moves
    by at most 2^-17 * (their count) * max|v_hat| / l with l > 1/2."""
    c = _case(nq=48, nc=400, seed=2, qmag=1.0)
    final = _run(c, mode="final")
    vmax = np.max(np.abs(e4m3.decode(c["vc"]))) * float(np.max(c["vs"]))
    n_exact = 0
    for tile in (16, 128, 1000):
        loop = _run(c, mode="mirror", tile=tile)
        for t in range(48):
            for h in range(4):
                sc = _row_scores(c, t, h)
                n_sub = int(np.sum(sc - np.ceil(np.max(sc)) + 8 < -6))
                if n_sub == 0:
                    assert np.allclose(loop[t, h], final[t, h], rtol=1e-12, atol=1e-14), (tile, t, h)
                    n_exact += 1
                else:
                    assert np.max(np.abs(loop[t, h] - final[t, h])) <= 2.0 ** -16 * n_sub * vmax, (tile, t, h)
    assert n_exact > 0.8 * 3 * 48 * 4
    # the stabilizer moves between tiles of 16 in these rows, and P rounding is live
    assert sum(np.ceil(np.max(_row_scores(c, t, 0)[:16])) < np.ceil(np.max(_row_scores(c, t, 0)))
               for t in range(48)) > 10
    assert not np.allclose(final, _run(c, mode="final", quantize_p=False), rtol=1e-6)


def test_tile_loop_with_the_maximum_at_key_zero_gives_the_final_max_codes():
    """Every row uses one query vector and key 0 equals it (scores q.k_j <=
    |q||k_j| < |q|^2 = score of key 0), so the running maximum is final from
    the first tile on and P8 against it is P8 against the final maximum."""
    rng = np.random.default_rng(7)
    nq, nc, Hq, Hkv, D = 32, 360, 4, 2, 16
    L = nq + nc
    qrow = _bf16(rng.standard_normal(D) * 0.9)  # score of key 0 about 3 nats above the rest
    qs = np.float32(np.abs(qrow).max() / 448)
    q8 = np.broadcast_to(kv_cache.quantize_query(qrow, qs), (nq, Hq, D)).copy()
    qhat = e4m3.decode(q8[0, 0]) * float(qs)
    k = _bf16(rng.standard_normal((L, Hkv, D)) * 0.6 * np.linalg.norm(qhat) / math.sqrt(D))
    k[0, :, :] = _bf16(qhat)[None, :]
    c = _case(nq, nc, Hq=Hq, Hkv=Hkv, D=D, k=k, q8=q8, qs=qs, ks=(np.abs(k).max() / 448,) * 2, seed=7)
    for t in (0, nq - 1):
        for h in (0, Hq - 1):
            s = _row_scores(c, t, h)
            assert np.argmax(s) == 0 and np.all(s[1:] < s[0])
            p = np.exp2(s - s[0])
            assert p[1:].sum() > 0.5  # the other keys carry real weight: a dropped key would show
    final = _run(c, mode="final")
    for tile in (16, 128):
        loop = _run(c, mode="mirror", tile=tile)
        assert np.allclose(loop, final, rtol=1e-12, atol=1e-14), tile


def test_one_tile_is_the_final_max_formula_bit_for_bit():
    c = _case(nq=20, nc=150, seed=3)
    assert np.array_equal(_run(c, mode="mirror", tile=4096), _run(c, mode="final"))


def _brute_row(c, t, h, tile=None):
    """One prefill row by pure-Python loops: base-2 scores from the codes,
    P8 by the brute-force encoder against the integer stabilizer (the
    running one when `tile` is given), normalized by the sum of the P8
    values."""
    Hq, Hkv = c["q8"].shape[1], c["kc"].shape[1]
    kv = h // (Hq // Hkv)
    D = c["q8"].shape[2]
    P = c["kc"].shape[2]
    n = c["L"] - c["nq"] + t + 1
    coef = float(attention.prefill_score_coef(c["qs"], c["ks"][kv], 0.25))
    qv = [e4m3.decode_code(int(x)) for x in c["q8"][t, h]]
    s, vrows = [], []
    for j in range(n):
        blk = int(c["bt"][0][j // P])
        krow = [e4m3.decode_code(int(c["kc"][blk, kv, j % P, d])) for d in range(D)]
        vrows.append([e4m3.decode_code(int(c["vc"][blk, kv, d, j % P])) for d in range(D)])
        s.append(sum(a * b for a, b in zip(qv, krow)) * coef)

    def p8(x):
        return e4m3.decode_code(e4m3.encode_bruteforce(float(np.float32(x * 256.0)))) / 256.0

    if tile is None:
        m = math.ceil(max(s))
        w = [p8(math.exp2(x - m)) for x in s]
        num = [sum(w[j] * vrows[j][d] for j in range(n)) for d in range(D)]
        return [x / sum(w) * float(c["vs"][kv]) for x in num]
    m, l, num = -math.inf, 0.0, [0.0] * D
    for t0 in range(0, n, tile):
        m_new = max(m, math.ceil(max(s[t0:t0 + tile])))
        a = math.exp2(m - m_new) if m != -math.inf else 0.0
        num = [x * a for x in num]
        l *= a
        for j in range(t0, min(n, t0 + tile)):
            w = p8(math.exp2(s[j] - m_new))
            l += w
            for d in range(D):
                num[d] += w * vrows[j][d]
        m = m_new
    return [x / l * float(c["vs"][kv]) for x in num]


@pytest.mark.parametrize("mode,tile", [("final", None), ("mirror", 128), ("mirror", 16)])
def test_bruteforce_about_300_keys(mode, tile):
    c = _case(nq=3, nc=297, Hq=2, Hkv=1, D=4, ks=(0.01,), vs=(0.02,), seed=11)
    got = _run(c, mode=mode, tile=tile or 128)
    for t in range(3):
        for h in range(2):
            assert np.allclose(got[t, h], _brute_row(c, t, h, tile), rtol=1e-11, atol=1e-13), (t, h)


def test_final_is_within_one_p8_rounding_of_pure():
    """Against unquantized P each p carries at most half an E4M3 ulp (2^-4 p)
    of rounding, so |final - pure| <= 2^-4 * max|v_hat| per element."""
    c = _case(nq=64, nc=500, seed=5)
    a = _run(c, mode="final")
    b = _run(c, mode="pure")
    vmax = np.max(np.abs(e4m3.decode(c["vc"]))) * float(np.max(c["vs"]))
    assert np.max(np.abs(a - b)) <= 2.0 ** -4 * vmax + 1e-6
    assert not np.allclose(a, b, rtol=1e-4)
