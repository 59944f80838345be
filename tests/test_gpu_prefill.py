"""GPU parity of kvq_prefill_attention (tcgen05 FP8 MMA, TMEM accumulators)
against the float64 oracle on caches and query codes the oracle builds.

Every check holds the kernel to max-abs 1e-2 (+ 2^-8 |ref| where |ref| > 1)
and mean-abs 1e-3 against two oracle readings of the declared rounding
(exact q8 / K8 products, the float32 score coefficient, the integer
stabilizer M = ceil(max s2), P8 = e4m3(2^(s2 - M) * 256), the row sum over
the same rounded P8):
* "final": M of the whole row -- one rounding per probability, independent
  of how any implementation tiles the keys;
* "mirror": the running M of an online softmax over tiles of 128 keys, the
  order the kernel walks them in (equal to "final": the rescales are powers
  of two).
The unquantized-P ("pure") result is checked too, within the bound that one
E4M3 rounding of every probability allows.  Per-token-scaled caches
(kvq_prefill_attention_per_token) are checked against
attention.prefill_per_token's tile walk ("mirror": the V-scale weights move
probabilities into E4M3's subnormal range, where the running and the final
stabilizer round differently) and its exact softmax."""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import attention, kv_cache
from tests.kvq_testlib import MAX_ABS, MEAN_ABS, assert_close, f32, to_device_cache

pytestmark = pytest.mark.gpu


def _k():
    import fp8_kv_cache_reshape_gb300 as k
    return k


def build(nq_list, cached_list, Hq=32, Hkv=8, seed=0, sentinel=0xA5, D=128, cache_dtype=kv_cache.FP8):
    """Oracle caches for sequences of nq new + cached old tokens; q8 codes."""
    gen = W.generator(9000 + seed)
    lens = [a + b for a, b in zip(nq_list, cached_list)]
    bt, nb = W.paged_layout(lens, 16, gen)
    slots = torch.cat([W.slots_for(bt, b, torch.arange(L), 16) for b, L in enumerate(lens)])
    T = int(slots.numel())
    k = W.randn_bf16((T, Hkv, D), gen)
    v = W.randn_bf16((T, Hkv, D), gen)
    q = W.randn_bf16((sum(nq_list), Hq, D), gen)
    fmt_max = W.E5M2_MAX if cache_dtype == kv_cache.FP8_E5M2 else W.E4M3_MAX
    ks, vs = W.calibrate_amax(k, fmt_max), W.calibrate_amax(v, fmt_max)
    qs = np.float32(q.float().abs().max().item() / 448)
    kc = np.full((nb, Hkv, 16, D), sentinel, np.uint8)
    vc = np.full((nb, Hkv, D, 16), sentinel, np.uint8)
    kv_cache.reshape_and_cache(f32(k), f32(v), slots.numpy(), kc, vc, ks.numpy(), vs.numpy(), cache_dtype)
    q8 = kv_cache.quantize_query(f32(q), qs)
    cu = np.concatenate([[0], np.cumsum(nq_list)]).astype(np.int32)
    return dict(kc=kc, vc=vc, q8=q8, qs=qs, ks=ks.numpy(), vs=vs.numpy(), bt=bt.numpy(), nb=nb,
                cu=cu, lens=np.array(lens, np.int32), Hq=Hq, Hkv=Hkv, sm=1 / np.sqrt(float(D)), dtype=cache_dtype)


def gpu_prefill(c, causal=True, block_table=None, status=False):
    k = _k()
    kd, vd = to_device_cache(c["kc"], c["vc"])
    q8 = torch.from_numpy(c["q8"]).cuda()
    out = torch.full(c["q8"].shape, float("nan"), dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    bt = torch.from_numpy(c["bt"] if block_table is None else block_table).cuda()
    nq_max = int(np.max(np.diff(c["cu"])))
    k.kvq_prefill_attention(q8, torch.tensor([c["qs"]], device="cuda"), kd, vd, torch.from_numpy(c["ks"]).cuda(),
                            torch.from_numpy(c["vs"]).cuda(), bt, torch.from_numpy(c["cu"]).cuda(),
                            torch.from_numpy(c["lens"]).cuda(), out, max_q_tokens=nq_max, num_blocks=c["nb"],
                            sm_scale=float(c["sm"]), causal=causal, dev_status=st, cache_dtype=c["dtype"])
    torch.cuda.synchronize()
    if status:
        return f32(out), int(st.item())
    assert int(st.item()) == 0, f"device status {int(st.item()):#x}"
    return f32(out)


def oracle(c, rows=None, causal=True, mode="mirror"):
    return attention.prefill(c["q8"], c["qs"], c["kc"], c["vc"], c["ks"], c["vs"], c["bt"], c["cu"], c["lens"],
                             float(np.float32(c["sm"])), causal=causal, mode=mode, rows=rows,
                             cache_dtype=c.get("dtype", kv_cache.FP8))


def check_rows(got, ref, rows, what=""):
    g = np.stack([got[t, h] for t, h in rows])
    r = np.stack([ref[t, h] for t, h in rows])
    return assert_close(g, r, what=what)


def check_all(got, c, rows, causal=True, what="prefill"):
    """The kernel against the final-maximum and the running-maximum oracle."""
    check_rows(got, oracle(c, rows=rows, causal=causal, mode="final"), rows, what=f"{what} vs final-max oracle")
    check_rows(got, oracle(c, rows=rows, causal=causal), rows, what=f"{what} vs running-max oracle")


def check_rows_vs_pure(got, pure, rows, c):
    """Against unquantized P the kernel carries the FP8 rounding of P: each
    p is off by at most half an E4M3 ulp, 2^-4 p, so the output is off by at
    most 2^-4 max|v_hat| (all errors aligned); plus bf16 output rounding."""
    vmax = float(np.max(np.abs(W_decode(c["vc"]))) * np.max(c["vs"]))
    g = np.stack([got[t, h] for t, h in rows])
    r = np.stack([pure[t, h] for t, h in rows])
    err = np.abs(g - r)
    bound = 2.0 ** -4 * vmax + 2.0 ** -8 * np.abs(r)
    assert np.all(err <= bound), f"max err {err.max():.3e} vs 2^-4 max|v| = {2.0 ** -4 * vmax:.3e}"
    return float(err.max()), float(err.mean())


def W_decode(codes):
    from oracle import e4m3
    return e4m3.decode(codes[np.isfinite(e4m3.decode(codes))])


@pytest.mark.parametrize("nq,cached", [([256], [384]), ([128], [0]), ([1, 130, 300], [0, 17, 1000]),
                                       ([77], [5000])])
def test_prefill_parity(nq, cached):
    c = build(nq, cached, seed=len(nq) + cached[0])
    got = gpu_prefill(c)
    Tq = c["q8"].shape[0]
    rng = np.random.default_rng(1)
    rows = [(t, h) for t in range(Tq) for h in range(c["Hq"])]
    if len(rows) > 3000:
        rows = [rows[i] for i in rng.choice(len(rows), 3000, replace=False)]
    check_all(got, c, rows, what=f"nq={nq} cached={cached}")
    pure = oracle(c, rows=rows, mode="pure")
    # against unquantized P the mean error carries the zero-mean FP8 rounding
    # noise of P (about 2^-4/sqrt(3) of each term); the 1e-3 mean target is
    # met against the mirrored oracle above
    mx, mn = check_rows_vs_pure(got, pure, rows, c)
    assert mn <= 10 * MEAN_ABS


@pytest.mark.parametrize("nq,cached", [([256], [384]), ([1, 130, 300], [0, 17, 1000]), ([77], [2000])])
def test_prefill_head_dim_256(nq, cached):
    """Head dim 256 (single-level accumulation): two 128-dim planes per
    operand, P.V with N = 256; NaN-poisoned bytes outside the tokens."""
    c = build(nq, cached, Hq=8, Hkv=2, seed=11 + len(nq), sentinel=0x7F, D=256)
    got = gpu_prefill(c)
    Tq = c["q8"].shape[0]
    rng = np.random.default_rng(5)
    rows = [(t, h) for t in range(Tq) for h in range(c["Hq"])]
    if len(rows) > 2000:
        rows = [rows[i] for i in rng.choice(len(rows), 2000, replace=False)]
    check_all(got, c, rows, what=f"head_dim 256 nq={nq} cached={cached}")
    check_rows_vs_pure(got, oracle(c, rows=rows, mode="pure"), rows, c)


def test_prefill_non_causal():
    c = build([200], [300], Hq=8, Hkv=2, seed=5)
    got = gpu_prefill(c, causal=False)
    rows = [(t, h) for t in range(0, 200, 3) for h in range(8)]
    check_all(got, c, rows, causal=False, what="non-causal")


def test_prefill_nan_poisoned_cache_outside_tokens():
    """Every cache byte outside the sequences' tokens is an E4M3 NaN; partial
    last pages and spare pages must not leak into the result."""
    c = build([100, 37], [250, 3], Hq=8, Hkv=2, seed=7, sentinel=0x7F)
    got = gpu_prefill(c)
    rows = [(t, h) for t in range(137) for h in range(8)]
    check_all(got, c, rows, what="NaN-poisoned cache")


def test_prefill_bad_block_reported():
    c = build([64], [200], Hq=8, Hkv=2, seed=9)
    bt = c["bt"].copy()
    bt[0, 3] = c["nb"] + 100
    out, st = gpu_prefill(c, block_table=bt, status=True)
    assert st & 0x2
    got = gpu_prefill(c)  # the context stays usable
    rows = [(t, h) for t in range(0, 64, 5) for h in range(8)]
    check_all(got, c, rows, what="after a bad block id")


def test_prefill_full_size_sampled():
    """The chunked-prefill configuration: 4,096 new causal tokens on 28,672
    cached, 32/8 heads, head_dim 128; sampled rows across the whole chunk."""
    pc = W.prefill_case(W.PREFILL)
    k = _k()
    cfg = pc.cfg
    kd, vd = k.alloc_kv_cache(pc.num_blocks, cfg.kv_heads, cfg.head_dim, fill=0x7F)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    k.kvq_reshape_and_cache(pc.k.cuda(), pc.v.cuda(), pc.slot_mapping.cuda(), kd, vd, pc.k_scale.cuda(),
                            pc.v_scale.cuda(), dev_status=st)
    q8 = torch.empty(pc.q.shape, dtype=torch.uint8, device="cuda")
    k.kvq_quantize_query(pc.q.cuda(), q8, pc.q_scale.cuda())
    out = torch.empty(pc.q.shape, dtype=torch.bfloat16, device="cuda")
    k.kvq_prefill_attention(q8, pc.q_scale.cuda(), kd, vd, pc.k_scale.cuda(), pc.v_scale.cuda(),
                            pc.block_table.cuda(), pc.cu_seqlens_q.cuda(), pc.seq_lens.cuda(), out,
                            max_q_tokens=cfg.new_tokens, sm_scale=pc.sm_scale, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    # the oracle builds its own cache and q8 from the same inputs
    kc = np.zeros((pc.num_blocks, cfg.kv_heads, 16, 128), np.uint8)
    vc = np.zeros((pc.num_blocks, cfg.kv_heads, 128, 16), np.uint8)
    kv_cache.reshape_and_cache(f32(pc.k), f32(pc.v), pc.slot_mapping.numpy(), kc, vc, pc.k_scale.numpy(),
                               pc.v_scale.numpy())
    qs = np.float32(pc.q_scale.item())
    q8_ref = kv_cache.quantize_query(f32(pc.q), qs)
    assert np.array_equal(q8.cpu().numpy(), q8_ref)
    # every row of the first and the last 128-row query tile (the causal
    # diagonal at both ends, the last CTA wave) for all 32 heads, plus rows
    # spread over the chunk
    rng = np.random.default_rng(3)
    spread = sorted(set(int(t) for t in rng.choice(np.arange(128, 3968), 48, replace=False)))
    rows = [(t, h) for t in list(range(0, 128)) + list(range(3968, 4096)) for h in range(cfg.q_heads)]
    rows += [(t, h) for t in spread for h in range(0, cfg.q_heads, 3)]
    args = (q8_ref, qs, kc, vc, pc.k_scale.numpy(), pc.v_scale.numpy(), pc.block_table.numpy(),
            pc.cu_seqlens_q.numpy(), pc.seq_lens.numpy(), float(np.float32(pc.sm_scale)))
    got = f32(out)
    check_rows(got, attention.prefill(*args, rows=rows, mode="final"), rows, what="4K on 28K vs final-max oracle")
    check_rows(got, attention.prefill(*args, rows=rows), rows, what="4K on 28K vs running-max oracle")


def test_prefill_bad_lengths_reported():
    """A sequence with more new tokens than cached tokens is skipped
    (KVQ_DEV_BAD_QROWS) while the others are computed; a length beyond the
    block table is clamped (KVQ_DEV_BAD_SEQLEN); the context stays usable."""
    c = build([64, 40], [200, 10], Hq=8, Hkv=2, seed=13)
    good = dict(c)
    bad_rows = dict(c)
    bad_rows["lens"] = c["lens"].copy()
    bad_rows["lens"][1] = 30  # 40 new tokens but only 30 cached
    out, st = gpu_prefill(bad_rows, status=True)
    assert st & 0x10
    rows = [(t, h) for t in range(0, 64, 3) for h in range(8)]  # sequence 0 only
    check_all(out, good, rows, what="sequence 0 beside a skipped sequence")
    bad_len = dict(c)
    bad_len["lens"] = c["lens"].copy()
    bad_len["lens"][0] = c["bt"].shape[1] * 16 + 5
    out, st = gpu_prefill(bad_len, status=True)
    assert st & 0x4
    got = gpu_prefill(good)  # the context stays usable
    rows = [(t, h) for t in range(0, 104, 5) for h in range(8)]
    check_all(got, good, rows, what="after bad lengths")


@pytest.mark.parametrize("D,nq,cached", [(128, [256], [384]), (128, [1, 130, 300], [0, 17, 1000]),
                                         (256, [77], [2000])])
def test_prefill_over_an_e5m2_cache(D, nq, cached):
    """E5M2 K and V codes as the B operands of both products (query and P
    codes E4M3); NaN-poisoned bytes outside the tokens (0x7F is an E5M2 NaN
    too)."""
    c = build(nq, cached, Hq=8, Hkv=2, seed=40 + D + len(nq), sentinel=0x7F, D=D, cache_dtype=kv_cache.FP8_E5M2)
    got = gpu_prefill(c)
    Tq = c["q8"].shape[0]
    rng = np.random.default_rng(6)
    rows = [(t, h) for t in range(Tq) for h in range(c["Hq"])]
    if len(rows) > 2000:
        rows = [rows[i] for i in rng.choice(len(rows), 2000, replace=False)]
    check_all(got, c, rows, what=f"E5M2 cache head_dim {D} nq={nq}")


def build_per_token(nq_list, cached_list, Hq=32, Hkv=8, seed=0, outliers=4, cache_dtype=kv_cache.FP8):
    """Oracle per-token caches (NaN in unwritten scale slots) and q8 codes."""
    gen = W.generator(9500 + seed)
    lens = [a + b for a, b in zip(nq_list, cached_list)]
    bt, nb = W.paged_layout(lens, 16, gen)
    slots = torch.cat([W.slots_for(bt, b, torch.arange(L), 16) for b, L in enumerate(lens)])
    T, D = int(slots.numel()), 128
    k = W.randn_bf16((T, Hkv, D), gen)
    v = W.randn_bf16((T, Hkv, D), gen)
    if outliers:  # a few tokens x4 (their own scales absorb it; their tiles' other weights shrink)
        idx = torch.randperm(T, generator=gen)[:outliers]
        k[idx] = (k[idx].float() * 4).bfloat16()
        v[idx] = (v[idx].float() * 4).bfloat16()
    q = W.randn_bf16((sum(nq_list), Hq, D), gen)
    qs = np.float32(q.float().abs().max().item() / 448)
    kc = np.full((nb, Hkv, 16, D), 0xA5, np.uint8)
    vc = np.full((nb, Hkv, D, 16), 0xA5, np.uint8)
    sc = np.full((nb, Hkv, 2, 16), np.nan, np.float32)
    kv_cache.reshape_and_cache_per_token(f32(k), f32(v), slots.numpy(), kc, vc, sc, cache_dtype)
    q8 = kv_cache.quantize_query(f32(q), qs)
    cu = np.concatenate([[0], np.cumsum(nq_list)]).astype(np.int32)
    return dict(kc=kc, vc=vc, sc=sc, q8=q8, qs=qs, bt=bt.numpy(), nb=nb, cu=cu, lens=np.array(lens, np.int32),
                Hq=Hq, Hkv=Hkv, sm=1 / np.sqrt(float(D)), dtype=cache_dtype)


def gpu_prefill_per_token(c, caches=None):
    """caches: device (k_cache, v_cache) to read instead of separate ones."""
    from oracle import layout
    k = _k()
    if caches is None:
        kd_np, vd_np = layout.to_device_format_per_token(c["kc"], c["vc"], c["sc"])
        kd, vd = torch.from_numpy(kd_np).cuda(), torch.from_numpy(vd_np).cuda()
    else:
        kd, vd = caches
    out = torch.full(c["q8"].shape, float("nan"), dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    k.kvq_prefill_attention_per_token(torch.from_numpy(c["q8"]).cuda(), torch.tensor([c["qs"]], device="cuda"), kd,
                                      vd, torch.from_numpy(c["bt"]).cuda(), torch.from_numpy(c["cu"]).cuda(),
                                      torch.from_numpy(c["lens"]).cuda(), out,
                                      max_q_tokens=int(np.max(np.diff(c["cu"]))), num_blocks=c["nb"],
                                      sm_scale=float(c["sm"]), cache_dtype=c["dtype"], dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0, f"device status {int(st.item()):#x}"
    return f32(out)


def oracle_per_token(c, rows, mode="mirror"):
    return attention.prefill_per_token(c["q8"], c["qs"], c["kc"], c["vc"], c["sc"], c["bt"], c["cu"], c["lens"],
                                       float(np.float32(c["sm"])), mode=mode, rows=rows, cache_dtype=c["dtype"])


@pytest.mark.parametrize("dtype", [kv_cache.FP8, kv_cache.FP8_E5M2])
@pytest.mark.parametrize("nq,cached", [([256], [384]), ([1, 130, 300], [0, 17, 1000]), ([77], [3000])])
def test_prefill_over_a_per_token_cache(nq, cached, dtype):
    """Per-token K and V scales (a few tokens x4), ragged lengths, a partial
    last page whose unwritten scale slots hold NaN; against the declared
    reading (the tile walk, "mirror") and, within the probability rounding,
    the exact softmax."""
    c = build_per_token(nq, cached, seed=len(nq) + cached[0], cache_dtype=dtype)
    got = gpu_prefill_per_token(c)
    Tq = c["q8"].shape[0]
    rng = np.random.default_rng(7)
    rows = [(t, h) for t in range(Tq) for h in range(c["Hq"])]
    if len(rows) > 2000:
        rows = [rows[i] for i in rng.choice(len(rows), 2000, replace=False)]
    check_rows(got, oracle_per_token(c, rows), rows, what=f"per-token nq={nq} cached={cached} {dtype}")
    # against unquantized P: every weight within half an E4M3 ulp, numerator and row sum
    pure = oracle_per_token(c, rows, mode="pure")
    g = np.stack([got[t, h] for t, h in rows])
    r = np.stack([pure[t, h] for t, h in rows])
    vmax = np.max(np.abs(r))
    assert np.all(np.abs(g - r) <= 2.0 ** -3 * vmax + 2.0 ** -8 * np.abs(r))


def test_prefill_over_a_per_token_cache_full_size():
    """The prefill configuration (4,096 new tokens on 28,672 cached, 32/8
    heads) over a per-token cache: rows of the first and the last query tile
    (the causal diagonal and 32,768 keys) for every eighth head, against the
    tile walk."""
    c = build_per_token([4096], [28672], seed=21)
    got = gpu_prefill_per_token(c)
    rows = [(t, h) for t in list(range(0, 128, 9)) + list(range(3968, 4096, 9)) for h in range(0, 32, 8)]
    check_rows(got, oracle_per_token(c, rows), rows, what="per-token prefill 4K on 28K")
