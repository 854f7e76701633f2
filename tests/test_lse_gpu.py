"""The per-row log-sum-exp output (fa_prefill_ex) of both kernels and every
head dimension against the f64 oracle's definition, lse = log sum_j
exp(scale q.k_j) over the keys a row sees (-inf for none):
|lse - lse_ref| <= 2e-4 (1 + |lse_ref|).  S is accumulated in f32 from the same
16-bit inputs and l sums the f32 exponentials, so the GPU's lse carries only
f32 rounding.  Through the C ABI, with O checked alongside."""
import numpy as np
import pytest
import torch

import oracle
from causal_prefill_flash_gb300 import workloads as W

pytestmark = pytest.mark.gpu

TOL_O = {"f16": 2e-3, "bf16": 8e-3}


def _fa():
    import causal_prefill_flash_gb300 as fa
    return fa


def _check_lse(got, want):
    got = got.cpu().double().numpy()
    ninf = np.isneginf(want)
    assert np.array_equal(np.isneginf(got), ninf)
    err = np.abs(got[~ninf] - want[~ninf]) / (1 + np.abs(want[~ninf]))
    assert err.size == 0 or err.max() <= 2e-4, err.max()


@pytest.mark.parametrize("split", [False, True, "persistent"], ids=["oneshot", "splitkv", "persistent"])
@pytest.mark.parametrize("B,Hq,Hkv,Sq,Skv,hd,dtype,causal", [
    (1, 4, 2, 300, 300, 128, "f16", True),
    (2, 3, 1, 129, 1000, 64, "bf16", True),
    (1, 2, 2, 300, 40, 128, "f16", True),    # rows that see no key
    (1, 4, 4, 200, 700, 128, "bf16", False),
    (1, 2, 1, 260, 260, 256, "bf16", True),
])
def test_lse_matches_oracle(B, Hq, Hkv, Sq, Skv, hd, dtype, causal, split, request):
    fa = _fa()
    if split and hd == 256:
        pytest.skip("split-KV takes hd 64 and 128")
    if split == "persistent":  # the split-KV schedule on the persistent kernel
        request.getfixturevalue("force_persistent")
        split = True
    w = W.Workload("lse", B, Hq, Hkv, Sq, Skv, hd, causal=causal, dtype=dtype, seed=Sq + Skv + hd)
    q, k, v = W.make_inputs(w)
    out, lse = fa.attention(q.cuda(), k.cuda(), v.cuda(), causal=causal, scale=w.scale, split=split,
                            return_lse=True)
    torch.cuda.synchronize()
    assert fa.debug_status() == 0
    _check_lse(lse, oracle.lse(q, k, causal=causal, scale=w.scale))
    want = oracle.attention(q, k, v, causal=causal, scale=w.scale)
    got = out.cpu().double().numpy()
    assert (np.abs(got - want) / (1 + np.abs(want))).max() <= TOL_O[dtype]


def test_lse_of_split_pieces_recombines():
    """The property lse exists for: attention over keys [0, a) and [a, Skv)
    computed separately (non-causal) recombines into the full result with
    weights exp(lse_i - lse)."""
    fa = _fa()
    w = W.Workload("lse", 1, 4, 2, 256, 1000, 128, causal=False, dtype="f16", seed=77)
    q, k, v = (t.cuda() for t in W.make_inputs(w))
    a = 384
    o1, l1 = fa.attention(q, k[:, :a].contiguous(), v[:, :a].contiguous(), causal=False, scale=w.scale, return_lse=True)
    o2, l2 = fa.attention(q, k[:, a:].contiguous(), v[:, a:].contiguous(), causal=False, scale=w.scale, return_lse=True)
    o, l = fa.attention(q, k, v, causal=False, scale=w.scale, return_lse=True)
    torch.cuda.synchronize()
    lt = torch.logaddexp(l1, l2)
    assert (lt - l).abs().max().item() <= 2e-4 * (1 + l.abs().max().item())
    w1 = torch.exp(l1 - lt).transpose(1, 2).unsqueeze(-1)  # [B, Sq, Hq, 1]
    w2 = torch.exp(l2 - lt).transpose(1, 2).unsqueeze(-1)
    comb = o1.float() * w1 + o2.float() * w2
    assert (comb - o.float()).abs().max().item() <= 4e-3


def test_full_size_lse_sampled_rows():
    fa = _fa()
    w = W.get("longctx_chunk128_kv32768")
    q, k, v = W.make_inputs(w)
    out, lse = fa.attention(q.cuda(), k.cuda(), v.cuda(), causal=True, scale=w.scale, return_lse=True)
    torch.cuda.synchronize()
    rows = W.sample_rows(w, 128)
    want = oracle.lse_rows(q, k, rows.numpy(), causal=True, scale=w.scale)
    got = lse.cpu()[rows[:, 0].long(), rows[:, 1].long(), rows[:, 2].long()]
    _check_lse(got, want)
