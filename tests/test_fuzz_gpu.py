"""A seeded random sweep of shapes through every kernel path, against the f64
oracle (a GB300 is needed).

Each case draws B, the GQA grouping, Sq, Skv (Sq may exceed Skv, lengths are
rarely tile multiples), the head width (a multiple of 8 up to 256), the dtype
and the mask, then runs the one-shot kernel, the split-KV path as the library
routes it, the persistent kernel over whole units and over the split-KV
schedule (heads up to 128 wide) and, for GQA groups of a multiple of 4 with
heads 72..128 wide, the CTA-pair kernel, each into a NaN-prefilled output
followed by a NaN guard.  Small cases compare every element, larger ones a sample of rows
the oracle computes one by one; the tolerance is the parity tests':
|o - o_ref| <= tol (1 + |o_ref|), tol = 2e-3 (f16), 8e-3 (bf16).
"""
import numpy as np
import pytest
import torch

import oracle
from causal_prefill_flash_gb300 import workloads as W

pytestmark = pytest.mark.gpu

TOL = {"f16": 2e-3, "bf16": 8e-3}
GUARD = 2048
N_CASES = 24
FULL_LIMIT = 2 * 10**9  # oracle multiply-adds above which rows are sampled


def _fa():
    import causal_prefill_flash_gb300 as fa
    return fa


def _draw(i):
    rng = np.random.default_rng(20251 + i)
    G = int(rng.choice([1, 1, 2, 3, 4, 8]))
    Hkv = int(rng.integers(1, 5))
    Hq = G * Hkv
    B = int(rng.integers(1, 4))
    Skv = int(rng.integers(1, 3000))
    Sq = int(rng.integers(1, Skv + 1)) if rng.random() < 0.7 else int(rng.integers(1, 1500))
    hd = int(rng.choice([8, 16, 32, 40, 64, 64, 72, 96, 120, 128, 128, 136, 192, 256]))
    dtype = "bf16" if rng.random() < 0.5 else "f16"
    causal = bool(rng.random() < 0.8)
    return B, Hq, Hkv, Sq, Skv, hd, dtype, causal


CASES = [_draw(i) for i in range(N_CASES)]


def _paths(hd, G):
    yield "oneshot", False, None
    if hd <= 128:
        yield "splitkv", True, None
        yield "persistent", False, "persistent"
        yield "persistent_ws", True, "persistent"
    if 64 < hd <= 128 and G % 4 == 0:
        yield "pair", False, "pair"


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}_H{}-{}_Sq{}_Skv{}_hd{}_{}_c{}".format(*c))
def test_random_shape_every_path(case):
    fa = _fa()
    B, Hq, Hkv, Sq, Skv, hd, dtype, causal = case
    w = W.Workload("fuzz", B, Hq, Hkv, Sq, Skv, hd, causal=causal, dtype=dtype, seed=Sq * 7 + Skv + hd)
    q, k, v = W.make_inputs(w)
    full = B * Hq * Sq * Skv * hd <= FULL_LIMIT
    if full:
        want = oracle.attention(q, k, v, causal=causal, scale=w.scale)
    else:
        rng = np.random.default_rng(Sq + Skv)
        rows = np.stack([rng.integers(0, B, 64), rng.integers(0, Hq, 64), rng.integers(0, Sq, 64)], axis=1)
        rows[0] = (0, 0, 0)
        rows[1] = (B - 1, Hq - 1, Sq - 1)
        want = oracle.attention_rows(q, k, v, rows, causal=causal, scale=w.scale)
    dq, dk, dv = q.cuda(), k.cuda(), v.cuda()
    for name, split, force in _paths(hd, Hq // Hkv):
        buf = torch.full((q.numel() + GUARD,), float("nan"), dtype=q.dtype, device="cuda")
        out = buf[: q.numel()].view(q.shape)
        if force:
            fa.debug_force_path(force)
        try:
            fa.attention(dq, dk, dv, causal=causal, scale=w.scale, out=out, split=split)
        finally:
            fa.debug_force_path("auto")
        torch.cuda.synchronize()
        assert fa.debug_status() == 0, f"{name}: kernel watchdog fired: {fa.debug_status():#x}"
        assert torch.isnan(buf[q.numel():]).all(), f"{name}: write past the output tensor"
        got = out.cpu().double().numpy()
        if not full:
            got = got[rows[:, 0], rows[:, 2], rows[:, 1]]
        err = np.abs(got - want)
        bad = ~(err <= TOL[dtype] * (1.0 + np.abs(want)))
        assert not bad.any(), f"{name}: {int(bad.sum())} of {err.size} out of tolerance, max err {np.nanmax(err):.3e}"
