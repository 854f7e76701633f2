"""The CTA-pair kernel (fa_prefill_pair_kernel: two CTAs on two SMs per unit of
four query heads of one KV head, paired tcgen05 MMAs with M = 256, each CTA
loading half of every K and V tile, P in shared memory) against the f64
oracle, through the C ABI with the kernel forced (it is not the library's
default).  Shapes cover GQA groups of 4 and 8, head widths 72..128, causal and
not, chunked prefill (Sq < Skv), rows that see no key (Sq > Skv), ragged tails
of both sequences, several batches, the per-row LSE, a K/V cache with spare
capacity, and shapes the kernel does not take (which run on the library's
choice).  Tolerance: |o - o_ref| <= tol (1 + |o_ref|), tol = 2e-3 (f16),
8e-3 (bf16); a NaN-filled guard after the output must stay untouched."""
import numpy as np
import pytest
import torch

import oracle
from causal_prefill_flash_gb300 import workloads as W

pytestmark = pytest.mark.gpu

TOL = {"f16": 2e-3, "bf16": 8e-3}
GUARD = 2048


def _fa():
    import causal_prefill_flash_gb300 as fa
    return fa


def _run(w, q, k, v):
    fa = _fa()
    buf = torch.full((q.numel() + GUARD,), float("nan"), dtype=q.dtype, device="cuda")
    out = buf[: q.numel()].view(q.shape)
    fa.attention(q.cuda(), k.cuda(), v.cuda(), causal=w.causal, scale=w.scale, out=out, split=False)
    torch.cuda.synchronize()
    assert fa.debug_status() == 0, f"kernel watchdog fired: {fa.debug_status():#x}"
    assert torch.isnan(buf[q.numel():]).all(), "write past the output tensor"
    return out


def _check(got, want, dtype):
    got = got.cpu().double().numpy()
    err = np.abs(got - want)
    bad = ~(err <= TOL[dtype] * (1.0 + np.abs(want)))
    assert not bad.any(), f"{int(bad.sum())} of {err.size} out of tolerance, max err {np.nanmax(err):.3e}"


@pytest.mark.parametrize("B,Hq,Hkv,Sq,Skv,hd,dtype,causal", [
    (1, 4, 1, 128, 128, 128, "bf16", True),
    (1, 4, 1, 128, 128, 128, "f16", False),
    (1, 8, 2, 300, 300, 128, "f16", True),       # ragged tail, two KV heads
    (2, 8, 1, 520, 700, 96, "bf16", True),       # chunked: Sq < Skv, G = 8
    (1, 4, 1, 200, 100, 128, "f16", True),       # rows that see no key
    (1, 4, 1, 257, 257, 72, "bf16", False),
    (1, 16, 4, 1000, 1000, 120, "bf16", True),
    (2, 8, 2, 129, 1031, 128, "f16", False),
    (1, 4, 1, 1, 1, 128, "bf16", True),          # one row, one key
])
def test_pair_kernel_matches_oracle(B, Hq, Hkv, Sq, Skv, hd, dtype, causal, force_pair):
    w = W.Workload("pair", B, Hq, Hkv, Sq, Skv, hd, causal=causal, dtype=dtype, seed=Sq * 3 + Skv + hd)
    q, k, v = W.make_inputs(w)
    _check(_run(w, q, k, v), oracle.attention(q, k, v, causal=causal, scale=w.scale), dtype)


def test_pair_kernel_large_score_range(force_pair):
    """Scores of std ~9 (Q, K of std 3): the online max moves often and far."""
    w = W.Workload("pair", 1, 8, 2, 700, 700, 128, causal=True, dtype="f16", seed=77, q_std=3.0, k_std=3.0)
    q, k, v = W.make_inputs(w)
    _check(_run(w, q, k, v), oracle.attention(q, k, v, causal=True, scale=w.scale), "f16")


def test_pair_kernel_gqa8192_rows(force_pair):
    """The 8192-token GQA prefill itself, on sampled rows the oracle computes one by one."""
    w = W.get("gqa_s8192_bf16")
    q, k, v = W.make_inputs(w)
    out = _run(w, q, k, v)
    rng = np.random.default_rng(5)
    rows = np.stack([np.zeros(48, dtype=np.int64), rng.integers(0, w.Hq, 48), rng.integers(0, w.Sq, 48)], axis=1)
    rows[0] = (0, 0, 0)
    rows[1] = (0, w.Hq - 1, w.Sq - 1)
    want = oracle.attention_rows(q, k, v, rows, causal=True, scale=w.scale)
    got = out.cpu().double().numpy()[rows[:, 0], rows[:, 2], rows[:, 1]]
    err = np.abs(got - want)
    assert (err <= TOL["bf16"] * (1 + np.abs(want))).all(), err.max()


def test_pair_kernel_lse(force_pair):
    fa = _fa()
    w = W.Workload("pair", 1, 8, 2, 300, 170, 128, causal=True, dtype="bf16", seed=11)
    q, k, v = W.make_inputs(w)
    out, lse = fa.attention(q.cuda(), k.cuda(), v.cuda(), causal=True, scale=w.scale, split=False, return_lse=True)
    torch.cuda.synchronize()
    assert fa.debug_status() == 0
    want = oracle.lse(q, k, causal=True, scale=w.scale)
    got = lse.cpu().double().numpy()
    ninf = np.isneginf(want)
    assert np.array_equal(np.isneginf(got), ninf)
    assert (np.abs(got[~ninf] - want[~ninf]) / (1 + np.abs(want[~ninf]))).max() <= 2e-4
    _check(out, oracle.attention(q, k, v, causal=True, scale=w.scale), "bf16")


def test_pair_kernel_kvcache_capacity(force_pair):
    """K/V read from caches with spare capacity (kv_cap > kv_len): rows past
    kv_len are out of the maps and must not be read."""
    fa = _fa()
    w = W.Workload("pair", 2, 4, 1, 200, 600, 128, causal=True, dtype="f16", seed=21)
    q, k, v = W.make_inputs(w)
    cap = 900
    kc = torch.full((w.B, cap, w.Hkv, w.hd), 1e4, dtype=k.dtype)  # poison past kv_len
    vc = torch.full_like(kc, float("nan"))
    kc[:, : w.Skv] = k
    vc[:, : w.Skv] = v
    out = fa.attention_kvcache(q.cuda(), kc.cuda(), vc.cuda(), w.Skv, causal=True, scale=w.scale, split=False)
    torch.cuda.synchronize()
    assert fa.debug_status() == 0
    _check(out, oracle.attention(q, k, v, causal=True, scale=w.scale), "f16")


@pytest.mark.parametrize("Hq,Hkv,hd", [(4, 2, 128), (6, 2, 128), (4, 1, 64), (4, 1, 256)])
def test_pair_path_falls_back(Hq, Hkv, hd, force_pair):
    """Shapes the pair kernel does not take (groups of 2 or 3, hd 64, hd 256)
    run on the library's choice under the same setting."""
    w = W.Workload("pair", 1, Hq, Hkv, 300, 300, hd, causal=True, dtype="bf16", seed=Hq + hd)
    q, k, v = W.make_inputs(w)
    _check(_run(w, q, k, v), oracle.attention(q, k, v, causal=True, scale=w.scale), "bf16")
