"""Helpers shared by the tests: build caches with the oracle, move them to
the device in the library's page format, and measure errors.  Inputs come
from workloads/; expected values come only from oracle/."""
from __future__ import annotations

import numpy as np
import torch

from oracle import attention, kv_cache, layout
from oracle.kv_cache import FP8, BF16

SENTINEL = 0xA5

# Attention tolerance for unit-variance inputs: max-abs 1e-2 and mean-abs
# 1e-3, flat, for every element with |o| <= 1.  An element with |o| > 1 (in
# these workloads the x20 outlier channels, |o| up to ~60) gets 2^-8 |o| on
# top: the output is bfloat16 (8 significant bits), whose nearest value can
# be half an ulp, up to 2^-8 |o|, from the exact one; the decode kernels'
# declared rounding of P for the P.V MMA (float16, taken against a running
# maximum that depends on how the context is cut into stages and splits) is
# a smaller relative effect the oracle does not mirror.  Below |o| = 1 both
# stay inside the flat 1e-2.
MAX_ABS = 1e-2
MEAN_ABS = 1e-3
REL_ABOVE_ONE = 2.0 ** -8

# measured errors of the checks that ran in this process: (what, max, mean)
ERRORS = []


def bound(ref, max_abs=MAX_ABS):
    """The elementwise tolerance described above."""
    a = np.abs(np.asarray(ref, np.float64))
    return max_abs + np.where(a > 1.0, REL_ABOVE_ONE * a, 0.0)


def f32(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy()


def oracle_cache(case, sentinel=SENTINEL):
    """Logical oracle caches holding every token of the case."""
    cfg = case.cfg
    D, H = cfg.head_dim, cfg.kv_heads
    dt = np.uint16 if case.cache_dtype == BF16 else np.uint8
    fill = sentinel if dt == np.uint8 else (sentinel << 8) | sentinel
    kc = np.full((case.num_blocks, H, 16, D), fill, dt)
    vc = np.full((case.num_blocks, H, D, 16), fill, dt)
    kv_cache.reshape_and_cache(f32(case.k), f32(case.v), case.slot_mapping.numpy(), kc, vc,
                               case.k_scale.numpy(), case.v_scale.numpy(), case.cache_dtype)
    return kc, vc


def to_device_cache(kc, vc, device="cuda"):
    kd, vd = layout.to_device_format(kc, vc)
    return torch.from_numpy(kd).to(device), torch.from_numpy(vd).to(device)


def oracle_decode(case, kc, vc, mode="mirror", window=None):
    return attention.paged_decode(f32(case.q), kc, vc, case.k_scale.numpy(), case.v_scale.numpy(),
                                  case.block_table.numpy(), case.seq_lens.numpy(), case.sm_scale,
                                  window=case.window if window is None else window,
                                  cache_dtype=case.cache_dtype, mode=mode)


def errors(got: np.ndarray, ref: np.ndarray):
    d = np.abs(np.asarray(got, np.float64) - np.asarray(ref, np.float64))
    return float(d.max()), float(d.mean())


def assert_close(got, ref, max_abs=MAX_ABS, mean_abs=MEAN_ABS, what=""):
    """Elementwise |got - ref| <= bound(ref) (flat max_abs where |ref| <= 1)
    and mean |got - ref| <= mean_abs.  Records, prints and returns (max-abs,
    mean-abs)."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    mx, mn = errors(got, ref)
    ERRORS.append((what, mx, mn))
    small = np.abs(ref) <= 1.0
    mx_small = float(np.max(np.abs(got - ref)[small])) if np.any(small) else 0.0
    print(f"\n[errors] {what}: max-abs {mx:.3e} (|ref|<=1: {mx_small:.3e}) mean-abs {mn:.3e} (n={got.size})")
    bnd = bound(ref, max_abs)
    excess = np.abs(got - ref) - bnd
    worst = np.unravel_index(np.argmax(excess), excess.shape)
    assert np.all(excess <= 0), (f"{what}: |err| {abs(got[worst] - ref[worst]):.3e} > bound {bnd[worst]:.3e} "
                                 f"at {worst} (ref {ref[worst]:.4f}); max-abs {mx:.3e}")
    assert mn <= mean_abs, f"{what}: mean-abs {mn:.3e}"
    return mx, mn
