"""Head dimension 256 (fa_prefill256_kernel: one query tile per CTA, P apart
from S in TMEM) against the f64 oracle, element by element, through the C ABI:
tile edges and ragged tails, GQA groups, chunked rows over a cached prefix,
rows that see no key, no mask, both 16-bit types, the cache entry point, and
the entry points that do not take hd 256.  Tolerance as in the parity tests:
|o - o_ref| <= tol (1 + |o_ref|), tol = 2e-3 (f16), 8e-3 (bf16)."""
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


def _case(B, Hq, Hkv, Sq, Skv, dtype, causal=True, seed=0, q_std=1.0):
    fa = _fa()
    w = W.Workload("hd256", B, Hq, Hkv, Sq, Skv, 256, causal=causal, dtype=dtype, seed=seed, q_std=q_std, k_std=q_std)
    q, k, v = W.make_inputs(w)
    out = torch.full_like(q, float("nan")).cuda()
    fa.attention(q.cuda(), k.cuda(), v.cuda(), causal=causal, scale=w.scale, out=out)
    torch.cuda.synchronize()
    assert fa.debug_status() == 0, hex(fa.debug_status())
    got = out.cpu().double().numpy()
    want = oracle.attention(q, k, v, causal=causal, scale=w.scale)
    err = np.abs(got - want) / (1 + np.abs(want))
    assert np.isfinite(got).all() and err.max() <= TOL[dtype], err.max()
    return got


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("S", [1, 2, 127, 128, 129, 255, 256, 300, 640])
def test_square_causal_edges(S, dtype):
    _case(1, 2, 1, S, S, dtype, seed=S)


@pytest.mark.parametrize("Sq,Skv", [(1, 129), (64, 200), (129, 1000), (300, 385)])
def test_chunked_rows_over_a_prefix(Sq, Skv):
    _case(2, 4, 2, Sq, Skv, "bf16", seed=Sq + Skv)


def test_rows_that_see_no_key_are_zero():
    got = _case(1, 2, 2, 300, 40, "f16", seed=3)
    assert np.all(got[:, : 300 - 40] == 0)


@pytest.mark.parametrize("G", [1, 2, 4, 8])
def test_gqa_groups(G):
    _case(2, 8, 8 // G, 200, 200, "f16", seed=10 + G)


def test_no_mask_and_large_scores():
    _case(1, 4, 2, 260, 700, "bf16", causal=False, seed=5)
    _case(1, 2, 2, 300, 300, "f16", seed=6, q_std=3.0)


def test_cache_entry_point_ignores_rows_past_kv_len():
    fa = _fa()
    w = W.Workload("hd256", 2, 4, 2, 130, 500, 256, dtype="bf16", seed=9)
    q, k, v = W.make_inputs(w)
    cap = 700
    kc = torch.full((2, cap, 2, 256), float("nan"), dtype=torch.bfloat16)
    vc = kc.clone()
    kc[:, :500], vc[:, :500] = k, v
    out = fa.attention_kvcache(q.cuda(), kc.cuda(), vc.cuda(), 500, causal=True, scale=w.scale)
    torch.cuda.synchronize()
    got = out.cpu().double().numpy()
    want = oracle.attention(q, k, v, causal=True, scale=w.scale)
    assert np.isfinite(got).all() and (np.abs(got - want) / (1 + np.abs(want))).max() <= TOL["bf16"]


def test_entry_points_without_hd256_say_so():
    fa = _fa()
    q = torch.zeros((1, 128, 2, 256), dtype=torch.float16, device="cuda")
    k = torch.zeros((1, 128, 2, 256), dtype=torch.float16, device="cuda")
    o = torch.empty_like(q)
    ws = torch.zeros(fa.workspace_bytes(128), dtype=torch.uint8, device="cuda")
    assert fa.fa_prefill_ws(q, k, k, o, 1, 2, 2, 128, 128, 256, 1, 0.0625, ws, ws.numel()) == 2
    assert fa.fa_prefill_ws_static(q, k, k, o, 1, 2, 2, 128, 128, 256, 1, 0.0625, 0) == 2
    assert fa.smem_bytes(256) > 0
