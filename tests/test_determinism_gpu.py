"""Every kernel path gives bitwise-identical output when a call is repeated on
the same inputs: no atomics in the arithmetic, and split pieces are merged in
a fixed order.  The same call is made four times (a GB300 is needed)."""
import pytest
import torch

from causal_prefill_flash_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _fa():
    import causal_prefill_flash_gb300 as fa
    return fa


PATHS = [  # (name, B, Hq, Hkv, Sq, Skv, hd, dtype, force, split)
    ("oneshot_hd128_rowpairs", 1, 6, 6, 900, 900, 128, "f16", "auto", False),
    ("oneshot_hd128_headpairs", 2, 8, 2, 700, 1100, 128, "bf16", "auto", False),
    ("oneshot_hd64", 2, 8, 2, 800, 800, 64, "f16", "auto", False),
    ("oneshot_hd256", 1, 4, 2, 600, 600, 256, "bf16", "auto", False),
    ("splitkv_pieces", 1, 4, 2, 200, 9000, 128, "bf16", "auto", True),
    ("persistent_whole_units", 1, 16, 4, 1500, 1500, 128, "bf16", "persistent", False),
    ("persistent_streamk_hd64", 2, 16, 4, 1300, 1300, 64, "f16", "persistent", True),
    ("cta_pair", 1, 16, 4, 1200, 1200, 128, "bf16", "pair", False),
]


@pytest.mark.parametrize("case", PATHS, ids=[c[0] for c in PATHS])
def test_repeated_calls_are_bitwise_identical(case):
    fa = _fa()
    name, B, Hq, Hkv, Sq, Skv, hd, dtype, force, split = case
    w = W.Workload(name, B, Hq, Hkv, Sq, Skv, hd, dtype=dtype, seed=Sq + hd)
    q, k, v = (t.cuda() for t in W.make_inputs(w))
    fa.debug_force_path(force)
    try:
        outs = [fa.attention(q, k, v, causal=True, scale=w.scale, split=split).clone() for _ in range(4)]
    finally:
        fa.debug_force_path("auto")
    torch.cuda.synchronize()
    assert fa.debug_status() == 0
    assert not torch.isnan(outs[0]).any()
    for o in outs[1:]:
        assert torch.equal(outs[0], o), f"{name}: a repeated call differs"


def test_paged_is_bitwise_identical_to_contiguous_and_repeatable():
    fa = _fa()
    w = W.Workload("paged", 2, 8, 2, 400, 1000, 128, dtype="f16", seed=9)
    q, k, v = W.make_inputs(w)
    page = 256
    npg = (w.Skv + page - 1) // page
    g = torch.Generator(device="cpu")
    g.manual_seed(4)
    table = torch.randperm(w.B * npg, generator=g).reshape(w.B, npg).to(torch.int32)
    kp = torch.zeros((w.B * npg, page, w.Hkv, w.hd), dtype=k.dtype)
    vp = torch.zeros_like(kp)
    for b in range(w.B):
        for p in range(npg):
            n = min(w.Skv, (p + 1) * page) - p * page
            kp[table[b, p], :n] = k[b, p * page: p * page + n]
            vp[table[b, p], :n] = v[b, p * page: p * page + n]
    dq, kp, vp, table = q.cuda(), kp.cuda(), vp.cuda(), table.cuda()
    outs = [fa.attention_paged(dq, kp, vp, table, w.Skv, causal=True, scale=w.scale, split=False).clone()
            for _ in range(3)]
    contiguous = fa.attention(dq, k.cuda(), v.cuda(), causal=True, scale=w.scale, split=False)
    torch.cuda.synchronize()
    assert fa.debug_status() == 0
    for o in outs[1:]:
        assert torch.equal(outs[0], o)
    assert torch.equal(outs[0], contiguous)
