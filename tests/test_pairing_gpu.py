"""Query-tile pairing of the row-pair grids (MHA and odd GQA groups, two
adjacent 128-row tiles of one head per CTA) when a head has an odd number of
tiles: one tile goes without a partner, tile 0 or the last one, whichever the
host's model of the one-shot grid expects to finish first
(fa_debug_row_pairing); the split-KV paths always leave tile 0 alone.  On the
one-shot kernel (hd 128, and the hd 64 kernel) and on the split-KV path,
every output element and every row's log-sum-exp against the f64 oracle:
|o - o_ref| <= tol (1 + |o_ref|) with tol 2e-3 (f16) / 8e-3 (bf16), and
|lse - lse_ref| <= 2e-4 (1 + |lse_ref|), as in the parity tests."""
import numpy as np
import pytest
import torch

import oracle
from causal_prefill_flash_gb300 import workloads as W

pytestmark = pytest.mark.gpu

TOL_O = {"f16": 2e-3, "bf16": 8e-3}

CASES = [  # B, Hq, Hkv, Sq, Skv, hd, dtype, tile 0 alone on the one-shot grid (None: not asserted)
    (1, 40, 40, 1152, 1152, 128, "f16", True),    # 200 CTAs, ~1.3 waves
    (1, 32, 32, 1152, 1152, 128, "bf16", False),  # 160 CTAs, ~1 wave: the last tile alone
    (1, 48, 16, 1152, 1152, 128, "bf16", True),   # GQA groups of 3
    (2, 20, 20, 1152, 1152, 64, "bf16", True),    # the hd 64 kernel
    (1, 40, 40, 1152, 1152, 64, "f16", True),
    (1, 40, 40, 1100, 1300, 128, "f16", None),    # ragged last tile, 200 keys ahead of the queries
]


def _fa():
    import causal_prefill_flash_gb300 as fa
    return fa


@pytest.mark.parametrize("B,Hq,Hkv,Sq,Skv,hd,dtype,lone", CASES,
                         ids=[f"B{c[0]}H{c[1]}-{c[2]}S{c[3]}x{c[4]}hd{c[5]}{c[6]}" for c in CASES])
def test_odd_tile_counts_match_oracle(B, Hq, Hkv, Sq, Skv, hd, dtype, lone):
    fa = _fa()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    if lone is not None and sms == 152:
        assert fa.debug_row_pairing(B, Hq, Hkv, Sq, Skv, True, sms) == lone
    w = W.Workload("pairing", B, Hq, Hkv, Sq, Skv, hd, causal=True, dtype=dtype, seed=Hq * 7 + Sq + hd)
    q, k, v = W.make_inputs(w)
    want = oracle.attention(q, k, v, causal=True, scale=w.scale)
    want_lse = oracle.lse(q, k, causal=True, scale=w.scale)
    ninf = np.isneginf(want_lse)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    for split in (False, True):
        out, lse = fa.attention(qd, kd, vd, causal=True, scale=w.scale, split=split, return_lse=True)
        torch.cuda.synchronize()
        assert fa.debug_status() == 0, f"split={split}: watchdog {fa.debug_status():#x}"
        got = out.cpu().double().numpy()
        err = np.abs(got - want) / (1 + np.abs(want))
        assert err.max() <= TOL_O[dtype], f"split={split}: max err {err.max():.3e}"
        gl = lse.cpu().double().numpy()
        assert np.array_equal(np.isneginf(gl), ninf)
        lerr = np.abs(gl[~ninf] - want_lse[~ninf]) / (1 + np.abs(want_lse[~ninf]))
        assert lerr.max() <= 2e-4, f"split={split}: lse err {lerr.max():.3e}"
