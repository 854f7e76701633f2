"""The kernels' bounded waits, made to run out on purpose (a GB300 is needed).

Every pipeline wait inside the kernels gives up after a limit (2 s by
default).  A CTA that gives up records a code in the device status word,
raises its abort flag so its other roles stop waiting, waits for the TMA
copies and MMAs it already issued, frees its TMEM and exits: no trap, no
fault.  fa_debug_set_watchdog_ns sets the limit for later launches; at 1 ns
nearly every wait that is not already satisfied runs out.  Each case checks
that such a call returns promptly with a pipeline-wait code in the status
word (never the code of a drain that ran out: the drains have their own
fixed limit), and that the same call then succeeds with the default limit
and matches the f64 oracle, so the context is still usable.
"""
import time

import numpy as np
import pytest
import torch

import oracle
from causal_prefill_flash_gb300 import workloads as W

pytestmark = pytest.mark.gpu

# producer empty, MMA Q / K-V / P / S read, softmax S / O / P V done, a CTA pair's
# forwarder: the codes of the pipeline waits
WAIT_CODES = {1, 3, 4, 5, 7, 8, 10, 11, 13}
WD_DRAIN = 9
TOL = {"f16": 2e-3, "bf16": 8e-3}


def _fa():
    import causal_prefill_flash_gb300 as fa
    return fa


def _paged_call(fa, q, k, v, page, w):
    B, S, Hkv, hd = k.shape
    npg = (S + page - 1) // page
    g = torch.Generator(device="cpu")
    g.manual_seed(3)
    perm = torch.randperm(B * npg + 1, generator=g)[: B * npg].reshape(B, npg).to(torch.int32)
    kp = torch.zeros((B * npg + 1, page, Hkv, hd), dtype=k.dtype)
    vp = torch.zeros_like(kp)
    for b in range(B):
        for p in range(npg):
            n = min(S, (p + 1) * page) - p * page
            kp[perm[b, p], :n] = k[b, p * page: p * page + n]
            vp[perm[b, p], :n] = v[b, p * page: p * page + n]
    kp, vp, perm = kp.cuda(), vp.cuda(), perm.cuda()
    return lambda out: fa.attention_paged(q.cuda(), kp, vp, perm, S, causal=True, scale=w.scale, out=out)


CASES = [  # (name, B, Hq, Hkv, S, hd, dtype, path)
    ("oneshot_hd128", 1, 16, 4, 1500, 128, "bf16", "oneshot"),
    ("oneshot_hd64", 2, 8, 8, 1100, 64, "f16", "oneshot"),
    ("hd256", 1, 4, 2, 900, 256, "bf16", "oneshot"),
    ("split_kv", 1, 8, 2, 2000, 128, "f16", "split"),
    ("paged", 2, 8, 4, 1300, 128, "f16", "paged"),
    ("persistent_hd128", 1, 32, 8, 2200, 128, "bf16", "persistent"),
    ("persistent_ws_hd64", 2, 16, 4, 2300, 64, "f16", "persistent_ws"),
    ("pair_hd128", 1, 16, 4, 1500, 128, "bf16", "pair"),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_waits_that_run_out_are_reported_and_leave_the_context_usable(case):
    fa = _fa()
    name, B, Hq, Hkv, S, hd, dtype, path = case
    w = W.Workload(name, B, Hq, Hkv, S, S, hd, dtype=dtype, seed=hd + S)
    q, k, v = W.make_inputs(w)
    if path == "paged":
        call = _paged_call(fa, q, k, v, 256, w)
    elif path.startswith("persistent") or path == "pair":
        dq, dk, dv = q.cuda(), k.cuda(), v.cuda()

        def call(out):
            fa.debug_force_path("pair" if path == "pair" else "persistent")
            try:
                fa.attention(dq, dk, dv, causal=True, scale=w.scale, out=out, split=path == "persistent_ws")
            finally:
                fa.debug_force_path("auto")
    else:
        dq, dk, dv = q.cuda(), k.cuda(), v.cuda()
        call = lambda out: fa.attention(dq, dk, dv, causal=True, scale=w.scale, out=out, split=(path == "split"))
    out = torch.empty(q.shape, dtype=q.dtype, device="cuda")
    call(out)  # warm-up: build, attributes, schedule
    torch.cuda.synchronize()
    assert fa.debug_status() == 0

    fa.debug_set_watchdog_ns(1)
    try:
        t0 = time.perf_counter()
        call(out)
        torch.cuda.synchronize()
        dt = time.perf_counter() - t0
    finally:
        fa.debug_set_watchdog_ns(0)
    st = fa.debug_status()
    assert st != 0, "no wait ran out at a 1 ns limit"
    assert (st & 0xFF) in WAIT_CODES, f"status {st:#x}: not a pipeline-wait code"
    assert (st & 0xFF) != WD_DRAIN
    assert dt < 1.0, f"an aborting call took {dt:.2f} s (a drain ran to its limit?)"
    assert fa.debug_status_clear() == 0

    out.fill_(float("nan"))
    call(out)
    torch.cuda.synchronize()
    assert fa.debug_status() == 0
    want = oracle.attention(q, k, v, causal=True, scale=w.scale)
    got = out.cpu().double().numpy()
    err = np.abs(got - want)
    assert (err <= TOL[dtype] * (1.0 + np.abs(want))).all(), f"{name}: max err {np.nanmax(err):.3e} after the aborted call"
