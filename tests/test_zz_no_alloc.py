"""fa_prefill_ws_static -- the split-KV path with the library's static scratch
and no allocation -- against the caller-workspace entry point fa_prefill_ws,
through the C ABI, two calls in a row.

The file name puts it last in collection, so in a full run it follows every
other test (which leave the library's static state -- the per-device set-up,
the sequence counter and whatever the scratch holds -- as they please); it
must pass both that way and alone.  Tolerance as in the parity tests:
|o - o_ref| <= tol (1 + |o_ref|), tol = 2e-3 (f16), 8e-3 (bf16).
"""
import pytest
import torch

from causal_prefill_flash_gb300 import workloads as W

pytestmark = pytest.mark.gpu

TOL = {"f16": 2e-3, "bf16": 8e-3}

# (B, Hq, Hkv, Sq, Skv, hd, dtype, causal): head pairs and row pairs, a
# ragged tail, a cached prefix, no mask, hd 64, and a grid that fills every
# SM with many split pairs (the largest scratch a call can need)
CASES = [
    (1, 4, 2, 1000, 1000, 128, "f16", 1),
    (2, 6, 2, 700, 1300, 64, "bf16", 1),
    (1, 2, 2, 384, 900, 128, "f16", 0),
    (1, 32, 8, 2048, 2048, 128, "bf16", 1),
    (1, 32, 32, 2048, 2048, 128, "f16", 1),
]


def _fa():
    import causal_prefill_flash_gb300 as fa
    return fa


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}_H{}-{}_S{}-{}_hd{}_{}_c{}".format(*c))
def test_static_scratch_matches_workspace_entry_point_twice(case):
    fa = _fa()
    B, Hq, Hkv, Sq, Skv, hd, dtype, causal = case
    w = W.Workload("case", B, Hq, Hkv, Sq, Skv, hd, dtype=dtype, seed=4242 + Sq + hd)
    q, k, v = (t.cuda() for t in W.make_inputs(w))
    bf16 = int(dtype == "bf16")
    # the reference: the existing split-KV entry point with a caller workspace
    ws = torch.zeros(fa.workspace_bytes(hd), dtype=torch.uint8, device="cuda")
    ref = torch.full_like(q, float("nan"))
    fn = fa.fa_prefill_ws_bf16 if bf16 else fa.fa_prefill_ws
    assert fn(q, k, v, ref, B, Hq, Hkv, Sq, Skv, hd, causal, w.scale, ws, ws.numel()) == 0
    torch.cuda.synchronize()
    ref = ref.double().cpu()
    outs = [torch.full_like(q, float("nan")) for _ in range(2)]
    for o in outs:  # two calls in a row, back to back on one stream
        st = fa.fa_prefill_ws_static(q, k, v, o, B, Hq, Hkv, Sq, Skv, hd, causal, w.scale, bf16)
        assert st == 0, fa.status_string(st)
    torch.cuda.synchronize()
    assert fa.debug_status() == 0, f"kernel watchdog fired: {fa.debug_status():#x}"
    tol = TOL[dtype]
    for i, o in enumerate(outs):
        got = o.double().cpu()
        assert not torch.isnan(got).any(), f"call {i}: unwritten output"
        err = ((got - ref).abs() / (1 + ref.abs())).max().item()
        assert err <= tol, f"call {i}: max scaled error {err:.3g} > {tol}"


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
