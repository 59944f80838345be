"""Attention over the paged FP8 (or BF16) KV cache, in float64.

Test infrastructure: only the tests, the smoke check and the bench's CPU
baseline may import this module.

What is computed
----------------
softmax(q . K^T * sm_scale) . V over the dequantized cache, per sequence and
query head, with query head h reading KV head h // (Hq / Hkv).

Sources
-------
* "The state of FP8 KV-cache and attention quantization in vLLM", section
  "Problems we found" / "Kernel and vLLM improvements", two-level
  accumulation: the contraction dimension of softmax(score) * V is the
  context length; partial sums must be promoted into real FP32 so that the
  error does not grow with context.  The oracle accumulates in float64.
* Same page, section "Performance benchmarks", single request: the FP8 FA3
  path uses online-softmax rescaling.
* Same page, "Skip layers": sliding-window layers attend to a fixed window
  (e.g. 128 tokens) and keep their cache in BF16.
* "FP8 and KV cache", section "How to enable it in the engine": with FP8
  attention the query is also quantized to FP8 (used by prefill).

Readings where the pages are silent
-----------------------------------
* The context length L counts the current token; decode attends to tokens
  [0, L), or to [max(0, L - W), L) with a window W.
* Chunked prefill: the nq new tokens of a sequence are the last nq of its L
  cached tokens; query i sits at position L - nq + i and (causal) attends to
  keys 0..L - nq + i.
* The softmax scale is an input (1/sqrt(D) by default in the callers).
* Prefill's softmax stabilizer is the row maximum of the base-2 scores
  rounded up to an integer, M = ceil(m): p_j = 2^(s2_j - M).  Any stabilizer gives the
  same softmax; an integer one makes every online-softmax rescale
  2^(M_old - M_new) an exact power of two, and rounding to E4M3 or float16
  commutes with powers of two, so the rounded probabilities -- and the
  result -- do not depend on how an implementation tiles or splits the keys.
* Prefill's probabilities feed an FP8 MMA: P8 = encode(fl32(p * 256)), 256
  a power of two the pages do not fix ("final"; "mirror" walks the keys in
  tiles with a running stabilizer, as the online softmax the vLLM page names
  for its FP8 attention kernel does, and equals "final").
* Where P is rounded for an FP8 MMA, the row sum l adds the same rounded
  values: the output is then a convex combination of the value rows with
  the weights the MMA actually applied (a lone dominant key reproduces its
  value row exactly, whatever its rounding).

Mirrored quantization points
----------------------------
``mode="mirror"`` rounds exactly where the CUDA path declares it rounds:
* decode: per query head, sigma = 2^(7 - floor(log2 max_d |q_d|)) (a power
  of two) and the query enters the MMA as qf = f16(fl32(q * sigma)) (RNE;
  exact for a bf16 q unless q * sigma falls below float16's normal range);
  scores are taken in base-2 units, s2 = (sum_d qf[d] * k8[d]) / sigma * c
  with c = fl32(fl32(k_scale * sm_scale) * log2(e));
  o = s_v * sum_j 2^(s2_j - m) v8_j / sum_j 2^(s2_j - m).  The kernel's
  rounding of P for the P.V MMA (2^(s2 - m) * 256 to float16, 11
  significant bits, taken against the running maximum) is not mirrored: it
  depends on how the context is cut into stages and splits; the tolerance
  carries it.  An E5M2 cache is mirrored the same way: its codes are
  decoded as E5M2.
* prefill: s2 = (sum_d q8[d] * k8[d]) * c with
  c = fl32(fl32(fl32(q_scale * k_scale) * sm_scale) * log2(e)), and P8 as
  above.
``mode="pure"`` uses the exact dequantized values and natural exponentials.
"""
from __future__ import annotations

import math

import numpy as np

from . import e4m3
from .kv_cache import FP8, BF16, FP8_TYPES, bf16_bits_to_f32, codec, gather_scales, gather_tokens

LOG2E_F32 = np.float32(1.4426950408889634)


def _f32(x):
    return np.float32(x)


def decode_score_coef(k_scale, sm_scale):
    """c = fl32(fl32(k_scale * sm_scale) * log2(e)), the decode kernels'
    declared float32 scale on q.k."""
    return np.float32(np.float32(_f32(k_scale) * _f32(sm_scale)) * LOG2E_F32)


def prefill_score_coef(q_scale, k_scale, sm_scale):
    """c = fl32(fl32(fl32(q_scale * k_scale) * sm_scale) * log2(e))."""
    a = np.float32(_f32(q_scale) * _f32(k_scale))
    b = np.float32(a * _f32(sm_scale))
    return np.float32(b * LOG2E_F32)


def _softmax_row(scores_base_e):
    """(p relative to the max, m, l) for one row of natural-log scores."""
    m = np.max(scores_base_e)
    p = np.exp(scores_base_e - m)
    return p, m, p.sum()


def query_f16(q_row):
    """The decode kernels' declared rounding of one query head: returns
    f16(fl32(q * sigma)) / sigma in float64, with sigma = 2^(7 -
    floor(log2 max|q|)) (exponent clamped at -100) and float16
    round-to-nearest-even (subnormals kept)."""
    q = np.asarray(q_row, dtype=np.float32)
    mx = float(np.max(np.abs(q))) if q.size else 0.0
    if mx == 0.0:
        return np.zeros(q.shape, dtype=np.float64)
    e = max(int(np.frexp(np.float32(mx))[1]) - 1, -100)
    sigma = np.float32(2.0 ** (7 - e))
    y = (q * sigma).astype(np.float32)
    return y.astype(np.float16).astype(np.float64) / float(sigma)


def stabilizer(s2):
    """The softmax stabilizer of base-2 scores: the row maximum rounded up to
    an integer, M = ceil(max_j s2_j).  p_j = 2^(s2_j - M) lies in (0, 1] with
    the largest in (1/2, 1]; any M gives the same softmax, and with an integer
    M every rescale between two stabilizers is an exact power of two."""
    return np.ceil(np.max(s2, axis=-1, keepdims=True))


def decode_positions(L, window):
    """Token positions a decode query at context length L attends to."""
    start = 0 if window is None or window < 0 else max(0, L - window)
    return np.arange(start, L, dtype=np.int64)


def paged_decode(q, k_cache, v_cache, k_scale, v_scale, block_table, seq_lens,
                 sm_scale, window=-1, cache_dtype=FP8, mode="mirror"):
    """One decode step: every sequence's query attends to its cached tokens.

    q: float32 [B][Hq][D] holding bf16 values.  k_cache / v_cache: the
    paged cache (see kv_cache).  Returns (out float64 [B][Hq][D],
    lse float64 [B][Hq] in natural-log units, -inf for an empty sequence).
    An empty sequence gives an all-zero output.
    """
    q = np.asarray(q, dtype=np.float32)
    B, Hq, D = q.shape
    Hkv = k_cache.shape[1]
    g = Hq // Hkv
    out = np.zeros((B, Hq, D), dtype=np.float64)
    lse = np.full((B, Hq), -np.inf, dtype=np.float64)
    for b in range(B):
        pos = decode_positions(int(seq_lens[b]), window)
        if pos.size == 0:
            continue
        for kv in range(Hkv):
            kk, vv = gather_tokens(k_cache, v_cache, block_table[b], pos, kv)
            if cache_dtype in FP8_TYPES:
                k_codes = codec(cache_dtype).decode(kk)  # [n][D]
                v_codes = codec(cache_dtype).decode(vv)
                sk = float(np.float32(k_scale[kv]))
                sv = float(np.float32(v_scale[kv]))
            else:
                k_codes = bf16_bits_to_f32(kk).astype(np.float64)
                v_codes = bf16_bits_to_f32(vv).astype(np.float64)
                sk = sv = 1.0
            for h in range(kv * g, (kv + 1) * g):
                qh = q[b, h].astype(np.float64)
                if mode == "mirror":
                    if cache_dtype in FP8_TYPES:  # f16 query for either cache format
                        qe = query_f16(q[b, h])
                        c = float(decode_score_coef(k_scale[kv], sm_scale))
                    else:
                        qe = qh
                        c = float(np.float32(_f32(sm_scale) * LOG2E_F32))
                    s2 = (k_codes @ qe) * c
                    m2 = np.max(s2)
                    p = np.exp2(s2 - m2)
                    l = p.sum()
                    out[b, h] = (p @ v_codes) / l * sv
                    lse[b, h] = (m2 + math.log2(l)) * math.log(2.0)
                else:
                    s = (k_codes * sk) @ qh * float(np.float32(sm_scale))
                    p, m, l = _softmax_row(s)
                    out[b, h] = (p @ (v_codes * sv)) / l
                    lse[b, h] = m + math.log(l)
    return out, lse


def paged_decode_per_token(q, k_cache, v_cache, kv_scale_cache, block_table, seq_lens,
                           sm_scale, window=-1, cache_dtype=FP8, mode="mirror"):
    """paged_decode over a cache written with per-token dynamic scales
    (kv_cache.reshape_and_cache_per_token; kv_scale_cache [nb][Hkv][2][P]):
    token j dequantizes as decode(k8_j) * sk_j and decode(v8_j) * sv_j.

    mirror: the query as in paged_decode; s2_j = (sum_d qf_d k8_jd) / sigma
    * c_j with c_j = fl32(fl32(sm_scale * log2(e)) * sk_j);
    o = sum_j 2^(s2_j - m) sv_j v8_j / sum_j 2^(s2_j - m).
    pure: exact dequantized values, natural exponentials.
    Returns (out float64 [B][Hq][D], lse float64 [B][Hq])."""
    q = np.asarray(q, dtype=np.float32)
    B, Hq, D = q.shape
    Hkv = k_cache.shape[1]
    g = Hq // Hkv
    fmt = codec(cache_dtype)
    out = np.zeros((B, Hq, D), dtype=np.float64)
    lse = np.full((B, Hq), -np.inf, dtype=np.float64)
    c0 = np.float32(_f32(sm_scale) * LOG2E_F32)
    for b in range(B):
        pos = decode_positions(int(seq_lens[b]), window)
        if pos.size == 0:
            continue
        for kv in range(Hkv):
            kk, vv = gather_tokens(k_cache, v_cache, block_table[b], pos, kv)
            k_codes, v_codes = fmt.decode(kk), fmt.decode(vv)
            sk = gather_scales(kv_scale_cache[:, :, 0], block_table[b], pos, kv).astype(np.float32)
            sv = gather_scales(kv_scale_cache[:, :, 1], block_table[b], pos, kv).astype(np.float64)
            for h in range(kv * g, (kv + 1) * g):
                if mode == "mirror":
                    c = (c0 * sk).astype(np.float32).astype(np.float64)
                    s2 = (k_codes @ query_f16(q[b, h])) * c
                    m2 = np.max(s2)
                    p = np.exp2(s2 - m2)
                    l = p.sum()
                    out[b, h] = (p * sv) @ v_codes / l
                    lse[b, h] = (m2 + math.log2(l)) * math.log(2.0)
                else:
                    s = (k_codes * sk.astype(np.float64)[:, None]) @ q[b, h].astype(np.float64)
                    s = s * float(np.float32(sm_scale))
                    p, m, l = _softmax_row(s)
                    out[b, h] = (p @ (v_codes * sv[:, None])) / l
                    lse[b, h] = m + math.log(l)
    return out, lse


def lse_merge(outs, lses):
    """Merge attention results over disjoint key sets (the split-KV combine):
    lse = log sum_i exp(lse_i); o = sum_i exp(lse_i - lse) o_i.  Parts with
    lse = -inf carry no weight; if all are empty the result is (0, -inf)."""
    outs = np.asarray(outs, dtype=np.float64)
    lses = np.asarray(lses, dtype=np.float64)
    m = np.max(lses)
    if not np.isfinite(m):
        return np.zeros(outs.shape[1:]), -np.inf
    w = np.exp(lses - m)
    tot = w.sum()
    return np.tensordot(w / tot, outs, axes=1), m + math.log(tot)


def _p8(p):
    """P quantized for the FP8 P.V product: decode(encode(fl32(p * 256))) / 256
    in float64 (256 is a power of two, so the scaling itself is exact)."""
    return e4m3.decode(e4m3.encode((p * 256.0).astype(np.float32))) / 256.0


def prefill(q8, q_scale, k_cache, v_cache, k_scale, v_scale, block_table,
            cu_seqlens_q, seq_lens, sm_scale, causal=True, mode="mirror",
            rows=None, tile=128, quantize_p=True, chunk=64, cache_dtype=FP8):
    """Chunked prefill over the FP8 cache (the new tokens are already cached).

    q8: uint8 [Tq][Hq][D] E4M3 codes.  cu_seqlens_q: int [B+1].  seq_lens:
    int [B], each counting the cached tokens including the new ones.
    rows: optional iterable of (token_index, head) pairs to evaluate; other
    rows of the result stay NaN (sampled checks at large sizes).
    cache_dtype: the cache's FP8 format (E4M3 or E5M2 codes; the query codes
    and the probabilities P8 are E4M3 either way).

    Modes (the scores of the mirrored modes are s2 = (sum_d q8_d k8_d) * c in
    base-2 units, c the float32 coefficient of prefill_score_coef):
    * "pure": softmax(q_hat . K_hat^T * sm_scale) . V_hat with the exact
      dequantized values and natural exponentials, no P quantization.
    * "final": P8_j = encode(fl32(2^(s2_j - M) * 256)) with M = ceil(max_j
      s2_j), the row's integer stabilizer -- one rounding per probability,
      independent of any tiling; o = s_v * sum_j decode(P8_j) v8_j /
      sum_j decode(P8_j): the output is normalized by the sum of the rounded
      probabilities it is a combination of.
    * "mirror": the online softmax: keys in tiles of `tile` in key order; per
      tile the running integer stabilizer M is updated, the earlier
      numerator and row sum (of the rounded P) are multiplied by
      a = 2^(M_old - M_new) (an exact power of two), and the tile's P8 is
      taken against the running M.
      E4M3 rounding commutes with powers of two (outside the subnormal
      range), so this equals "final" for every tile size.
    quantize_p=False keeps P unquantized in "final" / "mirror", numerator and
    row sum alike (used to pin the tile loop against the single-pass formula).
    Rows of one (sequence, KV head) are evaluated together, `chunk` at a
    time; a key past a row's causal limit has score -inf (p = 0).
    Returns out float64 [Tq][Hq][D].
    """
    if mode not in ("pure", "final", "mirror"):
        raise ValueError(f"unknown mode {mode!r}")
    q8 = np.asarray(q8, dtype=np.uint8)
    Tq, Hq, D = q8.shape
    Hkv = k_cache.shape[1]
    g = Hq // Hkv
    out = np.full((Tq, Hq, D), np.nan, dtype=np.float64)
    cu = np.asarray(cu_seqlens_q, dtype=np.int64)
    B = len(cu) - 1
    seq_of = np.zeros(Tq, dtype=np.int64)
    for b in range(B):
        seq_of[cu[b]:cu[b + 1]] = b
    if rows is None:
        rows = [(t, h) for t in range(Tq) for h in range(Hq)]
    by_seq_head = {}
    for t, h in rows:
        by_seq_head.setdefault((int(seq_of[t]), h // g), []).append((int(t), int(h)))
    qs = float(np.float32(q_scale))
    for (b, kv), items in by_seq_head.items():
        L = int(seq_lens[b])
        nq = int(cu[b + 1] - cu[b])
        kk, vv = gather_tokens(k_cache, v_cache, block_table[b], np.arange(L), kv)
        k_codes = codec(cache_dtype).decode(kk)   # [L][D]; the query and P codes are E4M3
        v_codes = codec(cache_dtype).decode(vv)
        sk = float(np.float32(k_scale[kv]))
        sv = float(np.float32(v_scale[kv]))
        c = float(prefill_score_coef(np.float32(q_scale), k_scale[kv], sm_scale))
        for r0 in range(0, len(items), chunk):
            part = items[r0:r0 + chunk]
            # keys 0 .. last[r] are visible to row r
            last = np.array([(L - nq + (t - int(cu[b]))) if causal else L - 1 for t, _ in part])
            n = int(last.max()) + 1
            qc = np.stack([e4m3.decode(q8[t, h]) for t, h in part])  # [R][D]
            visible = np.arange(n)[None, :] <= last[:, None]          # [R][n]
            if mode == "pure":
                s = (qc * qs) @ (k_codes[:n] * sk).T * float(np.float32(sm_scale))
                s = np.where(visible, s, -np.inf)
                m = np.max(s, axis=1, keepdims=True)
                p = np.exp(s - m)
                o = (p @ (v_codes[:n] * sv)) / p.sum(axis=1, keepdims=True)
            else:
                s2 = np.where(visible, (qc @ k_codes[:n].T) * c, -np.inf)
                q_of = _p8 if quantize_p else (lambda x: x)
                if mode == "final":
                    pq = q_of(np.exp2(s2 - stabilizer(s2)))
                    o = (pq @ v_codes[:n]) / pq.sum(axis=1, keepdims=True) * sv
                else:
                    R = len(part)
                    m_run = np.full(R, -np.inf)
                    l = np.zeros(R)
                    num = np.zeros((R, D))
                    for t0 in range(0, n, tile):  # online softmax over key tiles
                        seg = s2[:, t0:t0 + tile]
                        m_new = np.maximum(m_run, stabilizer(seg)[:, 0])
                        a = np.where(np.isfinite(m_run), np.exp2(m_run - m_new), 0.0)
                        pq = q_of(np.exp2(seg - m_new[:, None]))
                        num = num * a[:, None] + pq @ v_codes[t0:t0 + seg.shape[1]]
                        l = l * a + pq.sum(axis=1)
                        m_run = m_new
                    o = num / l[:, None] * sv
            for i, (t, h) in enumerate(part):
                out[t, h] = o[i]
    return out


def prefill_per_token_coef(q_scale, sm_scale):
    """b = fl32(fl32(q_scale * sm_scale) * log2(e)): the part of the score
    coefficient shared by all keys when K scales are per token."""
    return np.float32(np.float32(_f32(q_scale) * _f32(sm_scale)) * LOG2E_F32)


def pow2_ceil(x):
    """2^ceil(log2 x) for x > 0 (exact, from the float's exponent and
    mantissa); 1.0 for x <= 0."""
    x = float(x)
    if not x > 0.0:
        return 1.0
    m, e = math.frexp(x)  # x = m * 2^e, m in [1/2, 1)
    return math.ldexp(1.0, e - 1) if m == 0.5 else math.ldexp(1.0, e)


def prefill_per_token(q8, q_scale, k_cache, v_cache, kv_scale_cache, block_table,
                      cu_seqlens_q, seq_lens, sm_scale, causal=True, mode="final",
                      rows=None, tile=128, chunk=64, cache_dtype=FP8):
    """Chunked prefill over a cache written with per-token dynamic scales
    (kv_cache.reshape_and_cache_per_token; kv_scale_cache [nb][Hkv][2][P]):
    key j dequantizes as decode(k8_j) * sk_j and decode(v8_j) * sv_j.

    Sources: "FP8 and KV cache", section "Dynamic or static scale" (one
    scale per token); "FP8 quantization and long-context inference" (gtnt),
    section 2.2 (a scale for every new token); the prefill of "The state of
    FP8 KV-cache and attention quantization in vLLM" (FP8 QK^T and P.V).

    Modes:
    * "pure": softmax(q_hat . K_hat^T * sm_scale) . V_hat with the exact
      dequantized values and natural exponentials.
    * "final" (the reading the CUDA path declares): per key the score
      coefficient is c_j = fl32(sk_j * b), b = prefill_per_token_coef, and
      s2_j = (sum_d q8_d k8_jd) * c_j in base-2 units; M = ceil(max_j s2_j)
      (the integer stabilizer of prefill); p_j = 2^(s2_j - M).  The K scales
      are thus inside the scores; the V scales run along the P.V
      contraction, so they enter the FP8 probabilities: in each group of
      `tile` keys (aligned at key 0) with C_t = 2^ceil(log2 max sv_j) over
      the group's cached keys, the P.V operand is Pw_j = e4m3(fl32(fl32(p_j
      * 256) * (sv_j / C_t))) (sv_j / C_t exact: a power-of-two division),
      and the row sum takes the unweighted Pu_j = e4m3(fl32(p_j * 256)):
      o = sum_t C_t sum_{j in t} decode(Pw_j) v8_j / sum_j decode(Pu_j).
      With sv_j = C_t (all V scales of a group one power of two) Pw = Pu
      and this is prefill(mode="final") with the per-head scales.
    * "mirror": the same walked group by group in key order with the running
      integer stabilizer of the online softmax (the earlier numerator and row
      sum multiplied by 2^(M_old - M_new)).  The weights sv_j / C_t move many
      weighted probabilities into E4M3's subnormal range, where rounding does
      not commute with powers of two, so unlike the per-head case this is not
      "final": it is the reading of a one-pass kernel.
    Returns out float64 [Tq][Hq][D] (rows not in `rows` stay NaN).
    """
    if mode not in ("pure", "final", "mirror"):
        raise ValueError(f"unknown mode {mode!r}")
    q8 = np.asarray(q8, dtype=np.uint8)
    Tq, Hq, D = q8.shape
    Hkv = k_cache.shape[1]
    g = Hq // Hkv
    out = np.full((Tq, Hq, D), np.nan, dtype=np.float64)
    cu = np.asarray(cu_seqlens_q, dtype=np.int64)
    B = len(cu) - 1
    seq_of = np.zeros(Tq, dtype=np.int64)
    for b in range(B):
        seq_of[cu[b]:cu[b + 1]] = b
    if rows is None:
        rows = [(t, h) for t in range(Tq) for h in range(Hq)]
    by_seq_head = {}
    for t, h in rows:
        by_seq_head.setdefault((int(seq_of[t]), h // g), []).append((int(t), int(h)))
    qs = float(np.float32(q_scale))
    bcoef = np.float32(prefill_per_token_coef(q_scale, sm_scale))
    for (b, kv), items in by_seq_head.items():
        L = int(seq_lens[b])
        nq = int(cu[b + 1] - cu[b])
        pos = np.arange(L)
        kk, vv = gather_tokens(k_cache, v_cache, block_table[b], pos, kv)
        k_codes = codec(cache_dtype).decode(kk)
        v_codes = codec(cache_dtype).decode(vv)
        sk = gather_scales(kv_scale_cache[:, :, 0], block_table[b], pos, kv).astype(np.float32)
        sv = gather_scales(kv_scale_cache[:, :, 1], block_table[b], pos, kv).astype(np.float32)
        c = (sk * bcoef).astype(np.float32).astype(np.float64)          # [L]
        C = np.array([pow2_ceil(np.max(sv[t0:t0 + tile])) for t0 in range(0, L, tile)])
        w = (sv.astype(np.float64) / np.repeat(C, tile)[:L]).astype(np.float32)  # exact
        for r0 in range(0, len(items), chunk):
            part = items[r0:r0 + chunk]
            last = np.array([(L - nq + (t - int(cu[b]))) if causal else L - 1 for t, _ in part])
            n = int(last.max()) + 1
            qc = np.stack([e4m3.decode(q8[t, h]) for t, h in part])
            visible = np.arange(n)[None, :] <= last[:, None]
            if mode == "pure":
                s = (qc * qs) @ (k_codes[:n] * sk[:n, None].astype(np.float64)).T * float(np.float32(sm_scale))
                s = np.where(visible, s, -np.inf)
                m = np.max(s, axis=1, keepdims=True)
                p = np.exp(s - m)
                o = (p @ (v_codes[:n] * sv[:n, None].astype(np.float64))) / p.sum(axis=1, keepdims=True)
            else:
                s2 = np.where(visible, (qc @ k_codes[:n].T) * c[None, :n], -np.inf)

                def codes(seg, M, wseg):
                    p256 = (np.exp2(seg - M) * 256.0).astype(np.float32)
                    return (e4m3.decode(e4m3.encode(p256)),
                            e4m3.decode(e4m3.encode((p256 * wseg[None, :]).astype(np.float32))))
                if mode == "final":
                    pu, pw = codes(s2, stabilizer(s2), w[:n])
                    o = (pw * np.repeat(C, tile)[None, :n]) @ v_codes[:n] / pu.sum(axis=1, keepdims=True)
                else:
                    R = len(part)
                    m_run = np.full(R, -np.inf)
                    l = np.zeros(R)
                    num = np.zeros((R, D))
                    for gi, t0 in enumerate(range(0, n, tile)):
                        seg = s2[:, t0:t0 + tile]
                        m_new = np.maximum(m_run, stabilizer(seg)[:, 0])
                        a = np.where(np.isfinite(m_run), np.exp2(m_run - m_new), 0.0)
                        pu, pw = codes(seg, m_new[:, None], w[t0:t0 + seg.shape[1]])
                        num = num * a[:, None] + C[gi] * (pw @ v_codes[t0:t0 + seg.shape[1]])
                        l = l * a + pu.sum(axis=1)
                        m_run = m_new
                    o = num / l[:, None]
            for i, (t, h) in enumerate(part):
                out[t, h] = o[i]
    return out


def decode_reduced_accumulator(q, k_cache, v_cache, k_scale, v_scale, block_table,
                               seq_lens, sm_scale, mantissa_bits=14):
    """Planted-defect variant used only to show the long-context test is
    sensitive: the P.V sum is carried in one accumulator whose value is
    rounded to `mantissa_bits` significant bits after every addition, the
    single-level accumulation that "FP8 and KV cache" (training section,
    accumulation precision) reports for FP8 tensor cores (about 14 bits).
    FP8 cache, full attention only.  Returns out float64 [B][Hq][D]."""
    q = np.asarray(q, dtype=np.float32)
    B, Hq, D = q.shape
    Hkv = k_cache.shape[1]
    g = Hq // Hkv
    out = np.zeros((B, Hq, D), dtype=np.float64)

    def rnd(x):
        mant, ex = np.frexp(x)
        return np.ldexp(np.round(mant * 2.0 ** mantissa_bits) / 2.0 ** mantissa_bits, ex)

    for b in range(B):
        pos = decode_positions(int(seq_lens[b]), -1)
        for kv in range(Hkv):
            kk, vv = gather_tokens(k_cache, v_cache, block_table[b], pos, kv)
            k_codes = e4m3.decode(kk)
            v_codes = e4m3.decode(vv)
            sv = float(np.float32(v_scale[kv]))
            c = float(decode_score_coef(k_scale[kv], sm_scale))
            heads = slice(kv * g, (kv + 1) * g)
            s2 = (q[b, heads].astype(np.float64) @ k_codes.T) * c  # [g][n]
            p = np.exp2(s2 - np.max(s2, axis=1, keepdims=True))
            acc = np.zeros((g, D))
            for j in range(p.shape[1]):
                acc = rnd(acc + p[:, j, None] * v_codes[j][None, :])
            out[b, heads] = acc / p.sum(axis=1, keepdims=True) * sv
    return out
