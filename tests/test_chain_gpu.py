"""Calls whose input is the previous call's output, back to back on one stream
(a GB300 is needed).

Every kernel is launched with programmatic dependent launch: its set-up may
overlap the previous kernel's tail, and it waits (griddepcontrol.wait) before
it reads or writes global memory.  These chains check that ordering: each
stage's input is the previous stage's output, no host synchronisation sits
between the calls, and each stage is compared with the f64 oracle fed the
GPU's own previous output, so a stage that read its input before the previous
kernel had written it fails parity.  Tolerance as in the parity tests:
|o - o_ref| <= tol (1 + |o_ref|), tol = 2e-3 (f16), 8e-3 (bf16).
"""
import numpy as np
import pytest
import torch

import oracle
from causal_prefill_flash_gb300 import workloads as W

pytestmark = pytest.mark.gpu

TOL = {"f16": 2e-3, "bf16": 8e-3}


def _fa():
    import causal_prefill_flash_gb300 as fa
    return fa


def _check(got, want, dtype, what):
    g = got.double().numpy()
    err = np.abs(g - want)
    bad = ~(err <= TOL[dtype] * (1.0 + np.abs(want)))
    assert not bad.any(), f"{what}: {int(bad.sum())} of {err.size} out of tolerance, max err {np.nanmax(err):.3e}"


@pytest.mark.parametrize("split", [False, True, "persistent"], ids=["oneshot", "splitkv", "persistent"])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_output_feeds_the_next_call(dtype, split, request):
    """O1 = attn(Q, K, V); O2 = attn(O1, K, V); O3 = attn(Q, O2, V): the
    second call reads the first's output as its queries, the third the
    second's output as its keys."""
    fa = _fa()
    if split == "persistent":  # the split-KV schedule on the persistent kernel
        request.getfixturevalue("force_persistent")
        split = True
    B, H, S, hd = 1, 8, 700, 128
    w = W.Workload("chain", B, H, H, S, S, hd, dtype=dtype, seed=11)
    q, k, v = (t.cuda() for t in W.make_inputs(w))
    o1 = torch.full_like(q, float("nan"))
    o2 = torch.full_like(q, float("nan"))
    o3 = torch.full_like(q, float("nan"))
    for _ in range(3):  # repeated, so later rounds overlap the previous round's tail too
        fa.attention(q, k, v, causal=True, scale=w.scale, out=o1, split=split)
        fa.attention(o1, k, v, causal=True, scale=w.scale, out=o2, split=split)
        fa.attention(q, o2, v, causal=True, scale=w.scale, out=o3, split=split)
    torch.cuda.synchronize()
    assert fa.debug_status() == 0
    qc, kc, vc = q.cpu(), k.cpu(), v.cpu()
    o1c, o2c = o1.cpu(), o2.cpu()
    _check(o1c, oracle.attention(qc, kc, vc, causal=True, scale=w.scale), dtype, "stage 1")
    _check(o2c, oracle.attention(o1c, kc, vc, causal=True, scale=w.scale), dtype, "stage 2 (queries = stage 1)")
    _check(o3.cpu(), oracle.attention(qc, o2c, vc, causal=True, scale=w.scale), dtype, "stage 3 (keys = stage 2)")


def test_append_then_attend_over_the_cache():
    """fa_kv_append writes the new tokens' rows into the cache and the cache
    attention reads them in the next launch."""
    fa = _fa()
    B, Hq, Hkv, hd, cap, prefix, T = 2, 8, 2, 128, 1024, 500, 200
    g = torch.Generator(device="cpu")
    g.manual_seed(21)
    k_cache = torch.full((B, cap, Hkv, hd), float("nan"), dtype=torch.bfloat16)
    v_cache = torch.full_like(k_cache, float("nan"))
    k_cache[:, :prefix] = torch.randn(B, prefix, Hkv, hd, generator=g).to(torch.bfloat16)
    v_cache[:, :prefix] = torch.randn(B, prefix, Hkv, hd, generator=g).to(torch.bfloat16)
    k_new = torch.randn(B, T, Hkv, hd, generator=g)
    v_new = torch.randn(B, T, Hkv, hd, generator=g)
    q = torch.randn(B, T, Hq, hd, generator=g).to(torch.bfloat16)
    pos = (prefix + torch.arange(T, dtype=torch.int32)).repeat(B, 1).contiguous()
    kc, vc = k_cache.cuda(), v_cache.cuda()
    fa.kv_append(k_new.cuda(), v_new.cuda(), pos.cuda(), kc, vc)
    out = fa.attention_kvcache(q.cuda(), kc, vc, prefix + T, causal=True, scale=hd ** -0.5)
    torch.cuda.synchronize()
    assert fa.debug_status() == 0
    kv_len = prefix + T
    k_all = kc[:, :kv_len].cpu()
    v_all = vc[:, :kv_len].cpu()
    # the appended rows are the f32 rows rounded to bf16 (round to nearest even)
    assert torch.equal(k_all[:, prefix:], k_new.to(torch.bfloat16))
    assert torch.equal(v_all[:, prefix:], v_new.to(torch.bfloat16))
    _check(out.cpu(), oracle.attention(q, k_all, v_all, causal=True, scale=hd ** -0.5), "bf16", "attention over the cache")
