"""fa_prefill_ws_static -- the split-KV path with the library's static scratch
and no allocation -- through the C ABI, two calls in a row.

Some callers cannot allocate device memory when they call: an engine whose
device memory is laid out once at start-up (an allocation under peak load may
fail or stall), or a C host that holds only the tensors it is given.  This
entry point serves them; these tests check it like every other path:

* against the f64 oracle, element by element (every element for the small
  cases, a sample of rows the oracle computes one by one for the full-GPU
  grids), with the output at the start of a NaN-filled larger buffer, so an
  unwritten element fails parity and a write past the tensor shows in the
  guard;
* against the caller-workspace entry point fa_prefill_ws on the same inputs
  (same kernel, same schedule, same merge order).

Head widths other than 64 and 128 (8, 40, 96, 120) are included: the tensor
maps must describe the caller's width, or TMA would read the wrong elements
and run past the K/V tensors.

The file name puts it last in collection, so in a full run it follows every
other test (which leave the library's static state -- the per-device set-up
and whatever the scratch holds -- as they please); it must pass both that way
and alone.  Tolerance as in the parity tests:
|o - o_ref| <= tol (1 + |o_ref|), tol = 2e-3 (f16), 8e-3 (bf16).
"""
import numpy as np
import pytest
import torch

import oracle
from causal_prefill_flash_gb300 import workloads as W

pytestmark = pytest.mark.gpu

TOL = {"f16": 2e-3, "bf16": 8e-3}
GUARD = 4096  # elements after the output tensor

# (B, Hq, Hkv, Sq, Skv, hd, dtype, causal): head pairs and row pairs, a
# ragged tail, a cached prefix, no mask, hd 64, narrow and in-between head
# widths, and grids that fill every SM with many split pairs (the largest
# scratch a call can need)
CASES = [
    (1, 4, 2, 1000, 1000, 128, "f16", 1),
    (2, 6, 2, 700, 1300, 64, "bf16", 1),
    (1, 2, 2, 384, 900, 128, "f16", 0),
    (1, 4, 2, 300, 700, 8, "f16", 1),
    (1, 4, 2, 300, 700, 40, "bf16", 1),
    (2, 3, 3, 200, 520, 96, "f16", 1),
    (1, 4, 2, 450, 450, 120, "bf16", 0),
    (1, 32, 8, 2048, 2048, 128, "bf16", 1),
    (1, 32, 32, 2048, 2048, 128, "f16", 1),
]
FULL_ORACLE_LIMIT = 4 * 10**9  # oracle multiply-adds above which only sampled rows are compared


def _fa():
    import causal_prefill_flash_gb300 as fa
    return fa


def _guarded_out(q):
    buf = torch.full((q.numel() + GUARD,), float("nan"), dtype=q.dtype, device="cuda")
    return buf, buf[: q.numel()].view(q.shape)


def _oracle_cmp(got, q, k, v, causal, scale, dtype, what):
    """Every element (small cases) or 96 sampled rows (full grids) against the oracle."""
    B, Sq, Hq, hd = q.shape
    Skv = k.shape[1]
    tol = TOL[dtype]
    if B * Hq * Sq * Skv * hd <= FULL_ORACLE_LIMIT:
        want = oracle.attention(q, k, v, causal=causal, scale=scale)
        g = got.double().numpy()
    else:
        rng = np.random.default_rng(Sq * 31 + Hq)
        rows = np.stack([rng.integers(0, B, 96), rng.integers(0, Hq, 96), rng.integers(0, Sq, 96)], axis=1)
        rows[:4, 2] = [0, Sq - 1, Sq // 2, min(Sq - 1, 127)]
        want = oracle.attention_rows(q, k, v, rows, causal=causal, scale=scale)
        g = got.double().numpy()[rows[:, 0], rows[:, 2], rows[:, 1]]
    err = np.abs(g - want)
    bad = ~(err <= tol * (1.0 + np.abs(want)))
    assert not bad.any(), f"{what}: {int(bad.sum())} of {err.size} out of tolerance, max err {np.nanmax(err):.3e}"


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}_H{}-{}_S{}-{}_hd{}_{}_c{}".format(*c))
def test_static_scratch_matches_oracle_and_workspace_entry_point_twice(case):
    fa = _fa()
    B, Hq, Hkv, Sq, Skv, hd, dtype, causal = case
    w = W.Workload("case", B, Hq, Hkv, Sq, Skv, hd, causal=bool(causal), dtype=dtype, seed=4242 + Sq + hd)
    qc, kc, vc = W.make_inputs(w)
    q, k, v = qc.cuda(), kc.cuda(), vc.cuda()
    bf16 = int(dtype == "bf16")
    # the existing split-KV entry point with a caller workspace
    ws = torch.zeros(fa.workspace_bytes(hd), dtype=torch.uint8, device="cuda")
    ref = torch.full_like(q, float("nan"))
    fn = fa.fa_prefill_ws_bf16 if bf16 else fa.fa_prefill_ws
    assert fn(q, k, v, ref, B, Hq, Hkv, Sq, Skv, hd, causal, w.scale, ws, ws.numel()) == 0
    torch.cuda.synchronize()
    ref = ref.double().cpu()
    outs = [_guarded_out(q) for _ in range(2)]
    for _, o in outs:  # two calls in a row, back to back on one stream
        st = fa.fa_prefill_ws_static(q, k, v, o, B, Hq, Hkv, Sq, Skv, hd, causal, w.scale, bf16)
        assert st == 0, fa.status_string(st)
    torch.cuda.synchronize()
    assert fa.debug_status() == 0, f"kernel watchdog fired: {fa.debug_status():#x}"
    tol = TOL[dtype]
    for i, (buf, o) in enumerate(outs):
        what = f"call {i}, B{B} H{Hq}/{Hkv} Sq{Sq} Skv{Skv} hd{hd} {dtype} causal{causal}"
        got = o.double().cpu()
        assert not torch.isnan(got).any(), f"{what}: unwritten output"
        assert torch.isnan(buf[q.numel():]).all(), f"{what}: write past the output tensor"
        err = ((got - ref).abs() / (1 + ref.abs())).max().item()
        assert err <= tol, f"{what}: max scaled error against fa_prefill_ws {err:.3g} > {tol}"
        _oracle_cmp(o.cpu(), qc, kc, vc, bool(causal), w.scale, dtype, what)


def test_static_scratch_is_the_same_kernel_and_schedule():
    """Same kernel, same schedule, same merge order as fa_prefill_ws: the two
    entry points agree bit for bit."""
    fa = _fa()
    B, Hq, Hkv, Sq, Skv, hd = 1, 32, 8, 2048, 2048, 128
    w = W.Workload("case", B, Hq, Hkv, Sq, Skv, hd, dtype="bf16", seed=777)
    q, k, v = (t.cuda() for t in W.make_inputs(w))
    ws = torch.zeros(fa.workspace_bytes(hd), dtype=torch.uint8, device="cuda")
    a, b = torch.empty_like(q), torch.empty_like(q)
    assert fa.fa_prefill_ws_bf16(q, k, v, a, B, Hq, Hkv, Sq, Skv, hd, 1, w.scale, ws, ws.numel()) == 0
    assert fa.fa_prefill_ws_static(q, k, v, b, B, Hq, Hkv, Sq, Skv, hd, 1, w.scale, 1) == 0
    torch.cuda.synchronize()
    assert fa.debug_status() == 0
    assert torch.equal(a, b)


def test_static_scratch_call_allocates_no_device_memory():
    """After the set-up call, further calls leave the device's free memory and
    torch's allocator untouched."""
    fa = _fa()
    B, Hq, Hkv, Sq, Skv, hd = 1, 8, 8, 1024, 1024, 64
    w = W.Workload("case", B, Hq, Hkv, Sq, Skv, hd, dtype="f16", seed=99)
    q, k, v = (t.cuda() for t in W.make_inputs(w))
    o = torch.empty_like(q)
    assert fa.fa_prefill_ws_static(q, k, v, o, B, Hq, Hkv, Sq, Skv, hd, 1, w.scale, 0) == 0
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    alloc0 = torch.cuda.memory_allocated()
    for _ in range(3):
        assert fa.fa_prefill_ws_static(q, k, v, o, B, Hq, Hkv, Sq, Skv, hd, 1, w.scale, 0) == 0
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert torch.cuda.memory_allocated() == alloc0
    assert free1 == free0
    assert fa.debug_status() == 0
