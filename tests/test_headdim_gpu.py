"""Head widths other than 64, 128 and 256 on a GB300.

Any head width that is a multiple of 8 up to 256 runs on the next kernel up
(64, 128 or 256 columns).  The tensor maps describe the true width, so TMA
loads the missing columns of Q, K and V as zeros and clips them from the O
store; zero columns change neither S = Q K^T nor P V.  Every case compares
every output element (and, where asked, the per-row log-sum-exp) with the f64
oracle under the parity tests' tolerance, |o - o_ref| <= tol (1 + |o_ref|),
tol = 2e-3 (f16), 8e-3 (bf16).  The output lives at the start of a larger
NaN-filled buffer: an element not written fails parity, and a write past the
tensor's last row (the padding columns of the last head) leaves a non-NaN in
the guard.
"""
import numpy as np
import pytest
import torch

import oracle
from causal_prefill_flash_gb300 import workloads as W

pytestmark = pytest.mark.gpu

TOL = {"f16": 2e-3, "bf16": 8e-3}
GUARD = 4096  # elements after the output tensor


def _fa():
    import causal_prefill_flash_gb300 as fa
    return fa


def _check(got, want, dtype, what):
    g = got.double().numpy()
    err = np.abs(g - want)
    bad = ~(err <= TOL[dtype] * (1.0 + np.abs(want)))
    assert not bad.any(), f"{what}: {int(bad.sum())} of {err.size} out of tolerance, max err {np.nanmax(err):.3e}"


def _guarded_out(q):
    buf = torch.full((q.numel() + GUARD,), float("nan"), dtype=q.dtype, device="cuda")
    return buf, buf[: q.numel()].view(q.shape)


def _case(B, Hq, Hkv, Sq, Skv, hd, dtype, causal, split=False, lse=False, seed=0):
    fa = _fa()
    w = W.Workload("hd", B, Hq, Hkv, Sq, Skv, hd, causal=causal, dtype=dtype, seed=seed)
    q, k, v = W.make_inputs(w)
    buf, out = _guarded_out(q)
    res = fa.attention(q.cuda(), k.cuda(), v.cuda(), causal=causal, scale=w.scale, out=out, split=split,
                       return_lse=lse)
    torch.cuda.synchronize()
    assert fa.debug_status() == 0, f"kernel watchdog fired: {fa.debug_status():#x}"
    what = f"B{B} H{Hq}/{Hkv} Sq{Sq} Skv{Skv} hd{hd} {dtype} causal{causal} split{split}"
    _check(out.cpu(), oracle.attention(q, k, v, causal=causal, scale=w.scale), dtype, what)
    assert torch.isnan(buf[q.numel():]).all(), f"{what}: write past the output tensor"
    if lse:  # as the log-sum-exp tests: -inf exactly where the oracle has it, else 2e-4 relative
        got = res[1].cpu().double().numpy()
        want = oracle.lse(q, k, causal=causal, scale=w.scale)
        ninf = np.isneginf(want)
        assert np.array_equal(np.isneginf(got), ninf), what
        err = np.abs(got[~ninf] - want[~ninf]) / (1 + np.abs(want[~ninf]))
        assert err.size == 0 or err.max() <= 2e-4, (what, err.max())


# one width on each side of every kernel boundary, and some in between
WIDTHS = [8, 32, 40, 56, 72, 80, 96, 112, 120, 136, 160, 192, 200, 248]


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("hd", WIDTHS)
def test_head_width_causal_ragged(hd, dtype):
    """Two full query tiles and a 44-row tail, GQA head pairs (G = 2)."""
    _case(1, 4, 2, 300, 300, hd, dtype, causal=True, seed=hd)


@pytest.mark.parametrize("hd", [40, 96, 192])
def test_head_width_chunk_and_noncausal(hd):
    """A chunk of 200 rows over 520 keys (bottom-right causal alignment), MHA
    row pairs (G = 1), and the same shape without the mask."""
    _case(2, 3, 3, 200, 520, hd, "f16", causal=True, seed=hd + 1)
    _case(1, 2, 1, 130, 390, hd, "bf16", causal=False, seed=hd + 2)


@pytest.mark.parametrize("hd", [8, 40, 96, 120])
def test_head_width_split_kv_with_lse(hd):
    """The stream-K kernel and its merge (direct 16-byte stores at the true
    row stride) with the log-sum-exp output."""
    _case(1, 2, 1, 128, 4000, hd, "bf16", causal=True, split=True, lse=True, seed=hd + 3)
    _case(1, 4, 2, 300, 300, hd, "f16", causal=True, split=True, lse=True, seed=hd + 4)


def test_head_width_paged_and_cache():
    """A 96-wide head through the paged pool (one-shot and split-KV) and the
    capacity-strided cache."""
    fa = _fa()
    B, Hq, Hkv, Sq, kv_len, hd, page = 2, 4, 2, 150, 650, 96, 256
    w = W.Workload("hdp", B, Hq, Hkv, Sq, kv_len, hd, dtype="f16", seed=96)
    q, k, v = W.make_inputs(w)
    want = oracle.attention(q, k, v, causal=True, scale=w.scale)
    npg = (kv_len + page - 1) // page
    g = torch.Generator(device="cpu")
    g.manual_seed(7)
    nb = B * npg + 2
    perm = torch.randperm(nb, generator=g)[: B * npg].reshape(B, npg).to(torch.int32)
    kp = torch.full((nb, page, Hkv, hd), float("nan"), dtype=k.dtype)
    vp = torch.full_like(kp, float("nan"))
    for b in range(B):
        for p in range(npg):
            n = min(kv_len, (p + 1) * page) - p * page
            kp[perm[b, p], :n] = k[b, p * page: p * page + n]
            vp[perm[b, p], :n] = v[b, p * page: p * page + n]
    for split in (False, True, "persistent"):
        if split == "persistent":
            fa.debug_force_path("persistent")
        try:
            out = fa.attention_paged(q.cuda(), kp.cuda(), vp.cuda(), perm.cuda(), kv_len, causal=True, scale=w.scale,
                                     split=bool(split))
        finally:
            fa.debug_force_path("auto")
        torch.cuda.synchronize()
        assert fa.debug_status() == 0
        _check(out.cpu(), want, "f16", f"paged split{split}")
    cap = 700
    kc = torch.full((B, cap, Hkv, hd), float("nan"), dtype=k.dtype)
    vc = torch.full_like(kc, float("nan"))
    kc[:, :kv_len] = k
    vc[:, :kv_len] = v
    for split in (False, True, "persistent"):
        if split == "persistent":
            fa.debug_force_path("persistent")
        try:
            out = fa.attention_kvcache(q.cuda(), kc.cuda(), vc.cuda(), kv_len, causal=True, scale=w.scale,
                                       split=bool(split))
        finally:
            fa.debug_force_path("auto")
        torch.cuda.synchronize()
        assert fa.debug_status() == 0
        _check(out.cpu(), want, "f16", f"cache split{split}")


def test_unsupported_widths_are_refused():
    fa = _fa()
    for hd in (4, 100, 264):
        qq = torch.zeros(1, 8, 2, hd, dtype=torch.float16, device="cuda")
        with pytest.raises((fa.FaError, ValueError)):
            fa.attention(qq, qq, qq)
    w = torch.zeros(1, 8, 2, 192, dtype=torch.float16, device="cuda")
    with pytest.raises((fa.FaError, ValueError)):
        fa.attention(w, w, w, split=True)  # split-KV: heads up to 128 wide
