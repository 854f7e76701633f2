"""Attention over a paged K/V cache (fa_prefill_paged) on a GB300, through the
C ABI: against the f64 oracle on the K/V the block table gathers
(oracle.gather_pages), and bit for bit against the contiguous entry point on
the same gathered K/V -- the paged path only changes where the producer's TMA
loads point.  Unused pool blocks and the rows of the last page past kv_len
hold NaN, which must not reach the output.  Tolerance as in the parity
tests: |o - o_ref| <= tol (1 + |o_ref|), tol = 2e-3 (f16), 8e-3 (bf16)."""
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


def _paged(k, v, page, seed, spare=3):
    """Scatter contiguous K, V [B, S, Hkv, hd] into NaN-filled pools of pages in
    a shuffled order; returns (k_pool, v_pool, block_table)."""
    B, S, Hkv, hd = k.shape
    npg = (S + page - 1) // page
    nb = B * npg + spare
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    perm = torch.randperm(nb, generator=g)[: B * npg].reshape(B, npg).to(torch.int32)
    kp = torch.full((nb, page, Hkv, hd), float("nan"), dtype=k.dtype)
    vp = torch.full_like(kp, float("nan"))
    for b in range(B):
        for p in range(npg):
            rows = slice(p * page, min(S, (p + 1) * page))
            n = rows.stop - rows.start
            kp[perm[b, p], :n] = k[b, rows]
            vp[perm[b, p], :n] = v[b, rows]
    return kp, vp, perm


CASES = [  # (B, Hq, Hkv, Sq, kv_len, hd, dtype, page)
    (2, 4, 2, 300, 300, 128, "f16", 128),
    (3, 6, 2, 200, 1000, 64, "bf16", 256),
    (1, 8, 8, 129, 700, 128, "bf16", 512),
    (2, 4, 4, 1, 385, 128, "f16", 128),
    (1, 2, 1, 640, 640, 64, "f16", 640),
]


@pytest.fixture(params=[False, True, "persistent"], ids=["oneshot", "splitkv", "persistent"])
def split(request):
    """The one-shot kernel; the split-KV path as the library routes it; and the
    split-KV schedule forced onto the persistent kernel."""
    if request.param != "persistent":
        yield request.param
        return
    request.getfixturevalue("force_persistent")
    yield True


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}_H{}-{}_Sq{}_kv{}_hd{}_{}_p{}".format(*c))
def test_paged_matches_oracle_and_contiguous_path(case, split):
    fa = _fa()
    B, Hq, Hkv, Sq, kv_len, hd, dtype, page = case
    w = W.Workload("case", B, Hq, Hkv, Sq, kv_len, hd, dtype=dtype, seed=kv_len + page)
    q, k, v = W.make_inputs(w)
    kp, vp, table = _paged(k, v, page, seed=page)
    out = fa.attention_paged(q.cuda(), kp.cuda(), vp.cuda(), table.cuda(), kv_len, causal=True, scale=w.scale,
                             split=split)
    ref = fa.attention(q.cuda(), k.cuda(), v.cuda(), causal=True, scale=w.scale, split=split)
    torch.cuda.synchronize()
    assert fa.debug_status() == 0
    assert torch.equal(out, ref)  # same tiles, same kernel: only the load addresses differ
    kg = oracle.gather_pages(kp, table, kv_len, page)
    vg = oracle.gather_pages(vp, table, kv_len, page)
    want = oracle.attention(q, kg, vg, causal=True, scale=w.scale)
    got = out.cpu().double().numpy()
    err = np.abs(got - want) / (1 + np.abs(want))
    assert np.isfinite(got).all() and err.max() <= TOL[dtype], err.max()


def test_paged_full_size_gqa_prompt_sampled_rows():
    """The 8192-token GQA workload through 256-token pages in shuffled order:
    identical to the contiguous path, and sampled rows against the oracle."""
    fa = _fa()
    w = W.get("gqa_s8192_bf16")
    q, k, v = W.make_inputs(w)
    kp, vp, table = _paged(k, v, 256, seed=8)
    out = fa.attention_paged(q.cuda(), kp.cuda(), vp.cuda(), table.cuda(), w.Skv, causal=True, scale=w.scale)
    ref = fa.attention(q.cuda(), k.cuda(), v.cuda(), causal=True, scale=w.scale, split=False)
    torch.cuda.synchronize()
    assert fa.debug_status() == 0
    assert torch.equal(out, ref)
    rows = W.sample_rows(w, 256)
    want = oracle.attention_rows(q, k, v, rows.numpy(), causal=True, scale=w.scale)
    g = out.cpu()[rows[:, 0].long(), rows[:, 2].long(), rows[:, 1].long()].double().numpy()
    assert (np.abs(g - want) / (1 + np.abs(want))).max() <= TOL["bf16"]


def test_paged_long_context_chunk_split_kv():
    """The serving case split-KV exists for: a 128-row chunk over a long paged
    context (few query tiles, long rows).  Split-KV and one-shot agree with the
    oracle on sampled rows; split-KV is bit-identical to its contiguous run."""
    fa = _fa()
    w = W.Workload("case", 1, 16, 4, 128, 9000, 128, seed=31)
    q, k, v = W.make_inputs(w)
    kp, vp, table = _paged(k, v, 256, seed=31)
    dq, dkp, dvp, dt = q.cuda(), kp.cuda(), vp.cuda(), table.cuda()
    assert fa.split_kv_advised(w.B, w.Hq, w.Hkv, w.Sq, w.Skv, True)
    a = fa.attention_paged(dq, dkp, dvp, dt, w.Skv, causal=True, scale=w.scale)             # advised: split-KV
    b = fa.attention_paged(dq, dkp, dvp, dt, w.Skv, causal=True, scale=w.scale, split=False)
    c = fa.attention(dq, k.cuda(), v.cuda(), causal=True, scale=w.scale, split=True)
    torch.cuda.synchronize()
    assert fa.debug_status() == 0
    assert torch.equal(a, c)
    rows = W.sample_rows(w, 256)
    want = oracle.attention_rows(q, k, v, rows.numpy(), causal=True, scale=w.scale)
    for got in (a, b):
        g = got.cpu()[rows[:, 0].long(), rows[:, 2].long(), rows[:, 1].long()].double().numpy()
        assert (np.abs(g - want) / (1 + np.abs(want))).max() <= TOL["f16"]


def test_block_outside_the_pool_is_reported():
    fa = _fa()
    w = W.Workload("case", 1, 2, 2, 64, 300, 128, seed=4)
    q, k, v = W.make_inputs(w)
    kp, vp, table = _paged(k, v, 128, seed=4)
    table[0, 1] = kp.shape[0] + 5  # no such block
    assert fa.debug_status_clear() == 0
    out = fa.attention_paged(q.cuda(), kp.cuda(), vp.cuda(), table.cuda(), 300, causal=True, scale=w.scale)
    torch.cuda.synchronize()
    assert fa.debug_status() & 0xFF == 33
    assert fa.debug_status_clear() == 0
    assert torch.isfinite(out).all()  # the missing page read as zeros, not as memory past the pool
