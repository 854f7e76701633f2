"""Parity of the CUDA path against the f64 oracle (needs a GB300).

Every comparison is element by element on the same seeded 16-bit inputs:

    |o_gpu - o_ref| <= tol * (1 + |o_ref|),  tol = 2e-3 (f16), 8e-3 (bf16)

where o_gpu is the kernel's 16-bit output upcast and o_ref the oracle's f64
result.  The tolerance covers what the kernel rounds on purpose: P rounded to
16 bits before the P V contraction and O rounded to 16 bits at the end (the
pages note the same f32-regrouping drift between tilings, minfer "53 · r50 —
FA_TKV 32->16 occupancy experiment", section 2).

Small cases compare every output element; the nine workloads at their full
sizes (in the launch configuration the benchmark times) compare a sample of
rows the oracle computes one by one.  Edge cases follow the bug classes the
pages name: tail tiles that need both the local and the global bound (minfer
"28 · r23 — f16-path whole-graph wall decomposition + FA_TKV occupancy raise",
section 2.3), zero-staged rows past the end that must not contribute (same
page, section 3.2), and async-copy ordering (minfer "11 · P5 — prefill gap
session: TM=128 big tiles + FA rewrite", section 3.3), which shows up as
run-to-run differences.
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


def _inputs(B, Hq, Hkv, Sq, Skv, hd, dtype="f16", seed=0, q_std=1.0, k_std=1.0, v_std=1.0):
    w = W.Workload("case", B, Hq, Hkv, Sq, Skv, hd, dtype=dtype, seed=seed,
                   q_std=q_std, k_std=k_std, v_std=v_std)
    return w, W.make_inputs(w)


@pytest.fixture(params=[False, True, "persistent", "persistent_ws"],
                ids=["oneshot", "splitkv", "persistent", "persistent_ws"])
def split(request):
    """Run a parity test through the one-shot kernel, the split-KV path as the
    library routes it (one piece per CTA on the stream-K kernel, several
    segments per CTA on the persistent kernel), and the persistent kernel
    forced: over whole units without a workspace, and over the split-KV
    schedule with one."""
    return request.param


def _run_gpu(q, k, v, causal, scale, fill=float("nan"), split=False):
    fa = _fa()
    dq, dk, dv = q.cuda(), k.cuda(), v.cuda()
    out = torch.full_like(dq, fill)  # NaN-prefilled: an unwritten element fails parity
    if isinstance(split, str):
        fa.debug_force_path("persistent")
        try:
            fa.attention(dq, dk, dv, causal=causal, scale=scale, out=out, split=split == "persistent_ws")
        finally:
            fa.debug_force_path("auto")
    else:
        fa.attention(dq, dk, dv, causal=causal, scale=scale, out=out, split=split)
    torch.cuda.synchronize()
    assert fa.debug_status() == 0, f"kernel watchdog fired: {fa.debug_status():#x}"
    return out.cpu()


def _check(got, want, dtype, what=""):
    g = got.double().numpy() if hasattr(got, "numpy") else got
    err = np.abs(g - want)
    bound = TOL[dtype] * (1.0 + np.abs(want))
    bad = ~(err <= bound)  # NaN counts as bad
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {err.size} elements out of tolerance; "
            f"max err {np.nanmax(err):.3e}; first bad {idx.tolist()} got {g[tuple(idx[0])]} want {want[tuple(idx[0])]}")
    return float(np.max(err)) if err.size else 0.0


def _full_case(B, Hq, Hkv, Sq, Skv, hd, causal=True, dtype="f16", seed=0, split=False, **std):
    w, (q, k, v) = _inputs(B, Hq, Hkv, Sq, Skv, hd, dtype, seed, **std)
    got = _run_gpu(q, k, v, causal, w.scale, split=split)
    want = oracle.attention(q, k, v, causal=causal, scale=w.scale)
    return _check(got, want, dtype, f"B{B} H{Hq}/{Hkv} Sq{Sq} Skv{Skv} hd{hd} causal{causal} {dtype}")


# ------------------------------------------------------------------ small shapes

@pytest.mark.parametrize("hd", [64, 128])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("S", [1, 2, 3, 127, 128, 129, 255, 256, 300])
def test_square_causal_lengths(S, dtype, hd, split):
    _full_case(1, 2, 1, S, S, hd, True, dtype, seed=S, split=split)


@pytest.mark.parametrize("Sq,Skv", [(1, 129), (64, 200), (129, 1000), (200, 513), (384, 385)])
@pytest.mark.parametrize("hd", [64, 128])
def test_chunked_bottom_right(Sq, Skv, hd, split):
    _full_case(2, 4, 2, Sq, Skv, hd, True, "f16", seed=Sq + Skv, split=split)


@pytest.mark.parametrize("Sq,Skv", [(129, 255), (300, 128), (5, 700), (256, 256)])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_non_causal(Sq, Skv, dtype, split):
    _full_case(1, 4, 4, Sq, Skv, 128, False, dtype, seed=7, split=split)


@pytest.mark.parametrize("Sq,Skv", [(300, 40), (256, 129), (130, 1)])
def test_rows_with_no_visible_key_are_zero(Sq, Skv, split):
    """causal with Skv < Sq: rows i < Sq - Skv see no key and must be exactly 0."""
    w, (q, k, v) = _inputs(1, 2, 2, Sq, Skv, 128, "f16", 3)
    got = _run_gpu(q, k, v, True, w.scale, split=split)
    want = oracle.attention(q, k, v, causal=True, scale=w.scale)
    _check(got, want, "f16", "masked rows")
    n0 = Sq - Skv
    assert torch.all(got[:, :n0] == 0)


@pytest.mark.parametrize("G", [1, 2, 4, 8])
def test_gqa_groups(G, split):
    _full_case(2, 8, 8 // G, 257, 257, 128, True, "bf16", seed=G, split=split)


@pytest.mark.parametrize("std", [3.0, 10.0])
def test_large_score_ranges(std, split):
    """Scores with std 9 and 100: the online max subtraction and the lazy
    rescale (and, split, the merge of pieces with different maxima) must keep
    everything finite and exact to tolerance."""
    _full_case(1, 4, 4, 400, 400, 128, True, "f16", seed=int(std), split=split, q_std=std, k_std=std)
    _full_case(1, 4, 4, 400, 400, 64, True, "bf16", seed=int(std), split=split, q_std=std, k_std=std)


def test_scale_is_applied():
    w, (q, k, v) = _inputs(1, 2, 2, 200, 200, 128, "f16", 5)
    for scale in (0.01, 0.3, 2.0):
        got = _run_gpu(q, k, v, True, scale)
        want = oracle.attention(q, k, v, causal=True, scale=scale)
        _check(got, want, "f16", f"scale {scale}")


def test_padding_beyond_skv_never_contributes():
    """K/V rows past Skv inside the caller's allocation hold huge values; the
    kernel reads only [0, Skv) (the tensor map ends there) so they must not leak."""
    fa = _fa()
    B, Hq, Hkv, Sq, Skv, hd = 1, 2, 2, 200, 200, 128
    w, (q, k, v) = _inputs(B, Hq, Hkv, Sq, Skv, hd, "f16", 11)
    big_k = torch.full((B, Skv + 128, Hkv, hd), 6.0e4, dtype=torch.float16)
    big_v = torch.full((B, Skv + 128, Hkv, hd), float("nan"), dtype=torch.float16)
    big_k[:, :Skv] = k
    big_v[:, :Skv] = v
    dq, dk, dv = q.cuda(), big_k.cuda(), big_v.cuda()
    out = torch.full_like(dq, float("nan"))
    st = fa.fa_prefill(dq, dk, dv, out, B, Hq, Hkv, Sq, Skv, hd, 1, w.scale)
    assert st == 0
    torch.cuda.synchronize()
    want = oracle.attention(q, k, v, causal=True, scale=w.scale)
    _check(out.cpu(), want, "f16", "padding")


def test_output_canary_untouched():
    """O sits inside a larger allocation filled with a sentinel: the kernel must
    write exactly B*Sq*Hq*hd elements and nothing around them."""
    fa = _fa()
    B, Hq, Hkv, Sq, Skv, hd = 2, 3, 1, 131, 131, 64
    w, (q, k, v) = _inputs(B, Hq, Hkv, Sq, Skv, hd, "bf16", 12)
    n = B * Sq * Hq * hd
    pad = 4096
    buf = torch.full((n + 2 * pad,), 1234.0, dtype=torch.bfloat16, device="cuda")
    out = buf[pad:pad + n].view(B, Sq, Hq, hd)
    st = fa.fa_prefill_bf16(q.cuda(), k.cuda(), v.cuda(), out, B, Hq, Hkv, Sq, Skv, hd, 1, w.scale)
    assert st == 0
    torch.cuda.synchronize()
    assert torch.all(buf[:pad] == 1234.0) and torch.all(buf[pad + n:] == 1234.0)
    want = oracle.attention(q, k, v, causal=True, scale=w.scale)
    _check(out.cpu(), want, "bf16", "canary")


def test_repeated_runs_are_bitwise_identical():
    fa = _fa()
    w, (q, k, v) = _inputs(2, 8, 2, 700, 700, 128, "f16", 13)
    dq, dk, dv = q.cuda(), k.cuda(), v.cuda()
    first = fa.attention(dq, dk, dv, causal=True, scale=w.scale).clone()
    for _ in range(5):
        again = fa.attention(dq, dk, dv, causal=True, scale=w.scale)
        assert torch.equal(first, again)


def test_empty_inputs():
    fa = _fa()
    # B == 0 and Sq == 0: no-op, FA_OK
    q = torch.zeros((0, 4, 2, 128), dtype=torch.float16, device="cuda")
    k = torch.zeros((0, 4, 2, 128), dtype=torch.float16, device="cuda")
    assert fa.attention(q, k, k).shape == q.shape
    q = torch.zeros((1, 0, 2, 128), dtype=torch.float16, device="cuda")
    k = torch.randn((1, 4, 2, 128), device="cuda").half()
    assert fa.attention(q, k, k).numel() == 0
    # Skv == 0: every row sees no key -> O = 0 (k, v may be null)
    q = torch.randn((1, 5, 2, 128), device="cuda").half()
    k = torch.zeros((1, 0, 2, 128), dtype=torch.float16, device="cuda")
    for causal in (0, 1):
        out = torch.full_like(q, float("nan"))
        assert fa.fa_prefill(q, k, k, out, 1, 2, 2, 5, 0, 128, causal, 0.1) == 0
        torch.cuda.synchronize()
        assert torch.all(out == 0)
        out = fa.attention(q, k, k, causal=bool(causal))
        torch.cuda.synchronize()
        assert torch.all(out == 0)


def test_errors_are_returned_not_hidden():
    fa = _fa()
    q = torch.randn((1, 8, 4, 128), device="cuda").half()
    k = torch.randn((1, 8, 2, 128), device="cuda").half()
    o = torch.empty_like(q)
    assert fa.fa_prefill(q, k, k, o, 1, 4, 3, 8, 8, 128, 1, 0.1) == 1      # Hq % Hkv
    assert fa.fa_prefill(q, k, k, o, 1, 4, 2, 8, 8, 100, 1, 0.1) == 2      # hd
    assert fa.fa_prefill(q.data_ptr() + 2, k, k, o, 1, 4, 2, 8, 8, 128, 1, 0.1) == 3  # alignment
    assert fa.fa_prefill(q, k, k, q, 1, 4, 2, 8, 8, 128, 1, 0.1) == 1      # o aliases q
    assert fa.fa_prefill(q, k, k, o, 1, 4, 2, 8, 8, 128, 1, float("inf")) == 1
    with pytest.raises(fa.FaError):
        fa.attention(q, k[:, :, :1].contiguous().repeat(1, 1, 3, 1), k[:, :, :1].contiguous().repeat(1, 1, 3, 1))


def test_runs_on_a_side_stream():
    fa = _fa()
    w, (q, k, v) = _inputs(1, 4, 4, 333, 333, 128, "f16", 14)
    dq, dk, dv = q.cuda(), k.cuda(), v.cuda()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        out = fa.attention(dq, dk, dv, causal=True, scale=w.scale)
    s.synchronize()
    want = oracle.attention(q, k, v, causal=True, scale=w.scale)
    _check(out.cpu(), want, "f16", "side stream")


# ----------------------------------------------------------- the nine workloads

@pytest.mark.parametrize("idx", range(len(W.WORKLOADS)))
def test_workload_reduced_full_compare(idx, split):
    """Each workload's structure (dtype, GQA ratio, std, chunk offset, hd) at a
    size the oracle finishes in seconds, spanning several tiles and a ragged tail."""
    w = W.WORKLOADS[idx]
    if split and w.hd == 256:
        pytest.skip("split-KV and the persistent kernel take hd 64 and 128")
    if w.Sq == w.Skv:
        small = w.with_(B=1, Hq=min(w.Hq, 8), Hkv=min(w.Hkv, 8) if w.Hq == w.Hkv else 2,
                        Sq=w.Sq % 128 + 2 * 128 if w.Sq % 128 else 3 * 128 - 1,
                        Skv=w.Sq % 128 + 2 * 128 if w.Sq % 128 else 3 * 128 - 1)
    else:  # chunked: keep the offset structure (Skv - Sq >> Sq) at a smaller size
        small = w.with_(B=2, Hq=8, Hkv=2, Sq=160, Skv=1184)
    q, k, v = W.make_inputs(small)
    got = _run_gpu(q, k, v, small.causal, small.scale, split=split)
    want = oracle.attention(q, k, v, causal=small.causal, scale=small.scale)
    _check(got, want, small.dtype, small.name)


@pytest.mark.parametrize("idx", range(len(W.WORKLOADS)))
def test_workload_full_size_sampled_rows(idx, split):
    """The workload at its full size, in the benchmark's launch configuration:
    a sample of output rows (always the first/last rows of the first/last heads)
    against the oracle computed row by row; plus whole-tensor properties."""
    w = W.WORKLOADS[idx]
    if split and w.hd == 256:
        pytest.skip("split-KV and the persistent kernel take hd 64 and 128")
    q, k, v = W.make_inputs(w)
    got = _run_gpu(q, k, v, w.causal, w.scale, split=split)
    assert torch.isfinite(got).all()
    rows = W.sample_rows(w, 384 if w.Skv >= 4096 else 768)
    want = oracle.attention_rows(q, k, v, rows.numpy(), causal=w.causal, scale=w.scale)
    g = got[rows[:, 0].long(), rows[:, 2].long(), rows[:, 1].long()]
    _check(g, want, w.dtype, f"{w.name} sampled rows")
    # row 0 of a square causal case sees only key 0: O = V[0] of its KV head
    if w.causal and w.Sq == w.Skv:
        G = w.Hq // w.Hkv
        v0 = v[:, 0].double().repeat_interleave(G, dim=1)  # [B, Hq, hd]
        _check(got[:, 0], v0.numpy(), w.dtype, "row 0 = v_0")


def test_split_advice_follows_the_grid_fill():
    """The library advises split-KV where the one-shot grid leaves most SMs
    idle and rows are long (the long-context chunk), and -- knowing the head
    width -- for hd 64 grids of more pairs than SMs whose waves leave many SMs
    idle (160 equal pairs on 152 SMs; the chunked hd 64 prefill's 256 pairs);
    not for the workloads below, not at hd 128 or 256."""
    fa = _fa()
    W_ = {w.name: w for w in W.WORKLOADS}
    adv = lambda w: fa.split_kv_advised(w.B, w.Hq, w.Hkv, w.Sq, w.Skv, w.causal)
    adv_hd = lambda w: fa.split_kv_advised(w.B, w.Hq, w.Hkv, w.Sq, w.Skv, w.causal, w.hd)
    assert adv(W_["longctx_chunk128_kv32768"]) and adv_hd(W_["longctx_chunk128_kv32768"])
    for name in ("single_head_s256", "prefill7b_s2048", "ragged_s2659_std3", "gqa_s8192_bf16",
                 "chunked_kv8192_hd128", "chunked_kv8192_hd64", "encoder_s4096_noncausal",
                 "gqa_s4096_hd256_bf16"):
        assert not adv(W_[name]), name
        assert adv_hd(W_[name]) == (name == "chunked_kv8192_hd64" and
                                   torch.cuda.get_device_properties(0).multi_processor_count == 152), name
    # 10 sequences x 16 head pairs of one 128-row tile over 8192 keys: 160 equal
    # pairs, two waves on 152 SMs, the second almost empty
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    if sms == 152:
        assert fa.split_kv_advised(10, 32, 8, 128, 8192, True, 64)
        assert not fa.split_kv_advised(10, 32, 8, 128, 8192, True, 128)


# ------------------------------------------------------ many-CTA / sparse grids

def _sampled_case(B, Hq, Hkv, Sq, Skv, hd, dtype, seed, causal=True, n_rows=512, split=False):
    w, (q, k, v) = _inputs(B, Hq, Hkv, Sq, Skv, hd, dtype, seed)
    got = _run_gpu(q, k, v, causal, w.scale, split=split)
    rows = W.sample_rows(w, n_rows, seed=seed)
    want = oracle.attention_rows(q, k, v, rows.numpy(), causal=causal, scale=w.scale)
    g = got[rows[:, 0].long(), rows[:, 2].long(), rows[:, 1].long()]
    _check(g, want, dtype, f"sampled B{B} H{Hq}/{Hkv} Sq{Sq} Skv{Skv} hd{hd}")
    return got, rows


def test_many_units_with_empty_ones_between(split):
    """Many more CTAs than SMs, most of them with no visible key (causal,
    Skv << Sq): CTAs with nothing to stream write zeros, and every row before
    Sq - Skv must come out exactly 0."""
    Sq, Skv = 8192, 1000
    got, _ = _sampled_case(1, 40, 40, Sq, Skv, 128, "f16", 21, split=split)
    assert torch.all(got[:, : Sq - Skv] == 0)
    assert torch.isfinite(got).all()


def test_odd_gqa_group_pairs_row_tiles_over_rounds(split):
    """G = 3 (odd): a CTA pairs two row tiles of one head (the second may be
    past Sq); B = 4 gives several waves of CTAs."""
    _sampled_case(4, 12, 4, 1000, 1000, 128, "bf16", 22, split=split)


def test_even_gqa_many_rounds_hd64(split):
    _sampled_case(2, 16, 4, 3000, 3000, 64, "f16", 23, split=split)



# --------------------------------------------------------- stream-K specifics

def test_streamk_single_long_row_split_over_many_ctas():
    """One query tile pair over 8192 keys: its 64 KV steps are cut across
    every SM and merged back by the CTA holding KV tile 0."""
    for causal in (True, False):
        _full_case(1, 1, 1, 200, 8192, 128, causal, "f16", seed=31, split=True)
        _full_case(1, 2, 2, 128, 8192, 64, causal, "bf16", seed=32, split=True)


def test_streamk_workspace_reused_across_shapes():
    """The same workspace serves consecutive calls with different shapes (and
    so different splits); flags of an earlier call must never satisfy a later one."""
    cases = [(1, 4, 2, 300, 5000), (1, 1, 1, 64, 9000), (2, 8, 8, 700, 700), (1, 4, 2, 300, 5000)]
    for n, (B, Hq, Hkv, Sq, Skv) in enumerate(cases):
        _full_case(B, Hq, Hkv, Sq, Skv, 128, True, "f16", seed=40 + n, split=True)


def test_streamk_is_bitwise_repeatable_and_matches_oneshot_closely():
    fa = _fa()
    w, (q, k, v) = _inputs(1, 4, 2, 640, 6000, 128, "bf16", 41)
    dq, dk, dv = q.cuda(), k.cuda(), v.cuda()
    a = fa.attention(dq, dk, dv, causal=True, scale=w.scale, split=True).clone()
    for _ in range(4):
        assert torch.equal(a, fa.attention(dq, dk, dv, causal=True, scale=w.scale, split=True))
    b = fa.attention(dq, dk, dv, causal=True, scale=w.scale, split=False)
    assert (a.float() - b.float()).abs().max().item() < 2e-2


def test_streamk_workspace_errors():
    fa = _fa()
    q = torch.randn((1, 8, 4, 128), device="cuda").half()
    k = torch.randn((1, 8, 2, 128), device="cuda").half()
    o = torch.empty_like(q)
    ws = fa.workspace_for(q.device, 128)
    assert fa.fa_prefill_ws(q, k, k, o, 1, 4, 2, 8, 8, 128, 1, 0.1, ws, ws.numel() - 1) == 1
    assert fa.fa_prefill_ws(q, k, k, o, 1, 4, 2, 8, 8, 128, 1, 0.1, ws.data_ptr() + 128, ws.numel() - 256) == 3
    assert fa.fa_prefill_ws(q, k, k, o, 1, 4, 2, 8, 8, 128, 1, 0.1, ws, ws.numel()) == 0
