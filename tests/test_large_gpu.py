"""Tensors past 2^31 elements, and grid extremes (a GB300 is needed).

B = 1, Hq = 64, Hkv = 8, Sq = Skv = 262144, hd = 128, bf16, causal: Q and O
hold exactly 2^31 elements each (4 GiB), so the rows at the end of the
output lie beyond any 32-bit element offset, and the last query tile walks
2048 KV tiles.  The inputs are drawn on the device from a seeded generator
(~9 GiB in all; only the slices the oracle needs come back to the host).
Run on the one-shot kernel and on the split-KV path.  Sampled rows -- the
first and the last of the tensor among them -- are checked against the f64
oracle, each as its own one-row problem (that query row over its causal
prefix of keys, which under bottom-right alignment is the same row),
together with the per-row log-sum-exp.  Tolerance as in the parity tests:
|o - o_ref| <= 8e-3 (1 + |o_ref|), |lse - lse_ref| <= 2e-4 (1 + |lse_ref|).
"""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu

B, HQ, HKV, S, HD = 1, 64, 8, 262144, 128


def _fa():
    import causal_prefill_flash_gb300 as fa
    return fa


@pytest.mark.parametrize("split", [False, True], ids=["oneshot", "splitkv"])
def test_outputs_beyond_32_bit_offsets(split):
    """split: the split-KV path (stream-K ranges on the persistent kernel,
    partial outputs merged by the merge kernel) on the same tensors."""
    fa = _fa()
    assert B * S * HQ * HD == 2 ** 31
    free, _ = torch.cuda.mem_get_info()
    if free < 12 * 2 ** 30:
        pytest.skip("needs ~12 GiB of free device memory")
    g = torch.Generator(device="cuda")
    g.manual_seed(2 ** 31 - 1)
    q = torch.randn((B, S, HQ, HD), generator=g, device="cuda", dtype=torch.bfloat16)
    k = torch.randn((B, S, HKV, HD), generator=g, device="cuda", dtype=torch.bfloat16)
    v = torch.randn((B, S, HKV, HD), generator=g, device="cuda", dtype=torch.bfloat16)
    scale = 1.0 / np.sqrt(HD)
    out, lse = fa.attention(q, k, v, causal=True, scale=scale, split=split, return_lse=True)
    torch.cuda.synchronize()
    assert fa.debug_status() == 0, f"kernel watchdog fired: {fa.debug_status():#x}"

    rng = np.random.default_rng(31)
    rows = [(0, 0), (HQ - 1, S - 1), (HQ - 1, S - 2), (HQ - 2, S - 1), (7, S - 129), (33, S // 2), (63, 127)]
    rows += [(int(h), int(i)) for h, i in zip(rng.integers(0, HQ, 5), rng.integers(S - 4096, S, 5))]
    k_host, v_host = k.cpu(), v.cpu()
    G = HQ // HKV
    for hq, i in rows:
        hk = hq // G
        q1 = q[0:1, i:i + 1, hq:hq + 1, :].cpu()
        k1 = k_host[0:1, : i + 1, hk:hk + 1, :]
        v1 = v_host[0:1, : i + 1, hk:hk + 1, :]
        want = oracle.attention(q1, k1, v1, causal=True, scale=scale)[0, 0, 0]
        got = out[0, i, hq].float().cpu().double().numpy()
        err = np.abs(got - want)
        assert (err <= 8e-3 * (1 + np.abs(want))).all(), f"row (h{hq}, i{i}): max err {err.max():.3e}"
        want_lse = oracle.lse_rows(q1, k1, np.array([[0, 0, 0]]), causal=True, scale=scale)[0]
        got_lse = float(lse[0, hq, i].item())
        assert abs(got_lse - want_lse) <= 2e-4 * (1 + abs(want_lse)), (hq, i, got_lse, want_lse)


@pytest.mark.parametrize("B,Hq,Hkv,Sq,Skv,hd,dtype", [
    (2048, 2, 1, 7, 7, 128, "f16"),       # thousands of sequences of a few tokens
    (1, 128, 1, 300, 300, 128, "bf16"),   # one KV head for 128 query heads
    (1, 256, 256, 129, 129, 64, "f16"),   # many heads, one row past a tile
    (3, 96, 32, 200, 3000, 8, "bf16"),    # the narrowest heads, GQA 3, chunked
])
def test_extreme_shapes(B, Hq, Hkv, Sq, Skv, hd, dtype):
    """Grid extremes against the oracle on every element (inputs from the
    seeded workload generator), through the library's own path choice."""
    from causal_prefill_flash_gb300 import workloads as W
    fa = _fa()
    w = W.Workload("extreme", B, Hq, Hkv, Sq, Skv, hd, causal=True, dtype=dtype, seed=B + Hq + Sq)
    q, k, v = W.make_inputs(w)
    out = fa.attention(q.cuda(), k.cuda(), v.cuda(), causal=True, scale=w.scale)
    torch.cuda.synchronize()
    assert fa.debug_status() == 0
    want = oracle.attention(q, k, v, causal=True, scale=w.scale)
    got = out.cpu().double().numpy()
    tol = 2e-3 if dtype == "f16" else 8e-3
    err = np.abs(got - want)
    assert (err <= tol * (1 + np.abs(want))).all(), f"max err {err.max():.3e}"
