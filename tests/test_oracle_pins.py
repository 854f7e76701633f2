"""Pins for the f64 oracle: facts fixed by the mathematics, not by the oracle.

Each test is chosen so that a plausible slip in the oracle -- a dropped scale,
a top-left instead of bottom-right causal alignment, an off-by-one in the mask,
a wrong GQA head index, a transposed operand, a missing max subtraction or
normalisation -- fails at least one of them (``test_planted_mistakes_are_caught``
checks that claim for a set of deliberately wrong variants).

The mask rule (a key is visible when it is at or before the query's absolute
position and inside the stored range) follows minfer "28 · r23 — f16-path
whole-graph wall decomposition + FA_TKV occupancy raise", section 3.2; the
fully-masked-row guard follows minfer "53 · r50 — FA_TKV 32->16 occupancy
experiment", section 3.2.
"""
import math
import os
from decimal import Decimal, getcontext
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle


def _rand(shape, seed, scale=1.0):
    g = np.random.default_rng(seed)
    return g.standard_normal(shape) * scale


# --------------------------------------------------------------------------
# 1. exact brute force on tiny integer inputs (rational scores, 50-digit exp)
# --------------------------------------------------------------------------

def _brute_force_exact(q, k, v, causal, scale):
    """O for integer q/k/v with a dyadic scale: rational scores and a
    50-significant-digit decimal exp, one key at a time."""
    getcontext().prec = 50
    B, Sq, Hq, hd = q.shape
    _, Skv, Hkv, _ = k.shape
    G = Hq // Hkv
    out = np.zeros((B, Sq, Hq, hd))
    for b in range(B):
        for h in range(Hq):
            hk = h // G
            for i in range(Sq):
                vis = [j for j in range(Skv) if (not causal) or j <= (Skv - Sq) + i]
                if not vis:
                    continue
                s = {j: scale * sum(Fraction(int(q[b, i, h, d])) * int(k[b, j, hk, d])
                                    for d in range(hd)) for j in vis}
                m = max(s.values())
                e = {j: (Decimal((s[j] - m).numerator) / Decimal((s[j] - m).denominator)).exp()
                     for j in vis}
                z = sum(e.values())
                for d in range(hd):
                    acc = sum(e[j] * int(v[b, j, hk, d]) for j in vis) / z
                    out[b, i, h, d] = float(acc)
    return out


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Sq,Skv", [(4, 4), (3, 5), (5, 3)])
def test_brute_force_exact_tiny(causal, Sq, Skv):
    g = np.random.default_rng(7 + Sq * 10 + Skv)
    q = g.integers(-3, 4, size=(1, Sq, 2, 4)).astype(np.float64)
    k = g.integers(-3, 4, size=(1, Skv, 1, 4)).astype(np.float64)
    v = g.integers(-3, 4, size=(1, Skv, 1, 4)).astype(np.float64)
    scale = Fraction(1, 2)
    want = _brute_force_exact(q, k, v, causal, scale)
    got = oracle.attention(q, k, v, causal=causal, scale=0.5)
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-13)


GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def test_brute_force_4x4_mask_pattern():
    """Sq = Skv = 4, causal: row i averages exactly over keys 0..i when all
    scores tie (q = 0), so O row i = mean(v[0..i]) -- the lower-triangular
    pattern of a square causal mask, worked by hand in the golden fixture."""
    table = np.loadtxt(os.path.join(GOLDEN, "causal_4x4_prefix_mean.txt"), comments="#")
    want = table[:, 1:]
    assert list(table[:, 0]) == [0, 1, 2, 3]
    v = np.arange(16, dtype=np.float64).reshape(1, 4, 1, 4)
    q = np.zeros((1, 4, 1, 4))
    k = np.ones((1, 4, 1, 4))
    got = oracle.attention(q, k, v, causal=True, scale=1.0)[0, :, 0, :]
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-14)


# --------------------------------------------------------------------------
# 2. identical keys: O row i = mean of V over the visible prefix
# --------------------------------------------------------------------------

@pytest.mark.parametrize("Sq,Skv", [(7, 7), (5, 12), (1, 9)])
def test_identical_keys_give_prefix_mean(Sq, Skv):
    B, Hq, Hkv, hd = 2, 4, 2, 8
    q = _rand((B, Sq, Hq, hd), 1)
    kvec = _rand((hd,), 2)
    k = np.broadcast_to(kvec, (B, Skv, Hkv, hd)).copy()
    v = _rand((B, Skv, Hkv, hd), 3)
    got = oracle.attention(q, k, v, causal=True, scale=0.7)
    csum = np.cumsum(v, axis=1)
    off = Skv - Sq
    G = Hq // Hkv
    for i in range(Sq):
        n = off + i + 1
        want = csum[:, n - 1] / n  # [B, Hkv, hd]
        for h in range(Hq):
            np.testing.assert_allclose(got[:, i, h], want[:, h // G], rtol=0, atol=1e-12)
    # non-causal: every row is the mean over all keys
    got_nc = oracle.attention(q, k, v, causal=False, scale=0.7)
    want_nc = v.mean(axis=1)
    for h in range(Hq):
        np.testing.assert_allclose(got_nc[:, :, h], np.broadcast_to(want_nc[:, None, h // G], got_nc[:, :, h].shape),
                                   rtol=0, atol=1e-12)


# --------------------------------------------------------------------------
# 3. one-hot dominant keys: O row i = the V row of its dominant visible key
# --------------------------------------------------------------------------

def test_one_hot_dominant_key():
    Sq = Skv = 12
    hd = 16
    perm = np.random.default_rng(5).permutation(Skv)  # key j points along e_perm[j]
    q = np.zeros((1, Sq, 1, hd))
    k = np.zeros((1, Skv, 1, hd))
    for i in range(Sq):
        q[0, i, 0, i] = 40.0
    for j in range(Skv):
        k[0, j, 0, perm[j]] = 1.0
    v = _rand((1, Skv, 1, hd), 6)
    inv = np.argsort(perm)  # inv[i] = the key whose direction is e_i
    for causal in (False, True):
        got = oracle.attention(q, k, v, causal=causal, scale=1.0)[0, :, 0]
        for i in range(Sq):
            jstar = inv[i]
            if (not causal) or jstar <= i:
                want = v[0, jstar, 0]  # exp(-40) leakage from the other keys
                np.testing.assert_allclose(got[i], want, rtol=0, atol=1e-14 * Skv + 1e-15)
            else:
                # the dominant key is in the future: all visible scores are 0 -> uniform mean
                np.testing.assert_allclose(got[i], v[0, :i + 1, 0].mean(axis=0), rtol=0, atol=1e-13)


# --------------------------------------------------------------------------
# 4. rows of P sum to one; masked entries are exactly zero
# --------------------------------------------------------------------------

def test_probability_rows_sum_to_one_and_respect_mask():
    B, Sq, Skv, Hq, Hkv, hd = 2, 6, 10, 4, 2, 8
    q = _rand((B, Sq, Hq, hd), 11, 3.0)
    k = _rand((B, Skv, Hkv, hd), 12, 3.0)
    off = Skv - Sq
    for b in range(B):
        for h in range(Hq):
            for i in range(Sq):
                p = oracle.probs_row(q, k, b, h, i, causal=True, scale=0.5)
                assert abs(p.sum() - 1.0) < 1e-14
                assert np.all(p >= 0)
                assert np.all(p[off + i + 1:] == 0.0)
                assert np.all(p[:off + i + 1] > 0.0)


# --------------------------------------------------------------------------
# 5. one key: O = v_0 ; causal row 0 of a square case: O = v_0
# --------------------------------------------------------------------------

def test_single_key_returns_that_value():
    q = _rand((3, 1, 2, 8), 21)
    k = _rand((3, 1, 1, 8), 22)
    v = _rand((3, 1, 1, 8), 23)
    for causal in (False, True):
        got = oracle.attention(q, k, v, causal=causal, scale=0.3)
        np.testing.assert_allclose(got, np.repeat(v, 2, axis=2), rtol=0, atol=1e-15)
    q2 = _rand((1, 9, 1, 8), 24)
    k2 = _rand((1, 9, 1, 8), 25)
    v2 = _rand((1, 9, 1, 8), 26)
    got = oracle.attention(q2, k2, v2, causal=True, scale=0.3)
    np.testing.assert_allclose(got[0, 0], v2[0, 0], rtol=0, atol=1e-15)


# --------------------------------------------------------------------------
# 6. GQA equals MHA with K/V repeated per group (contiguous groups)
# --------------------------------------------------------------------------

def test_gqa_equals_repeated_mha():
    B, Sq, Skv, Hq, Hkv, hd = 2, 5, 9, 8, 2, 8
    q = _rand((B, Sq, Hq, hd), 31)
    k = _rand((B, Skv, Hkv, hd), 32)
    v = _rand((B, Skv, Hkv, hd), 33)
    G = Hq // Hkv
    kr = np.repeat(k, G, axis=2)  # head h of the repeat is kv head h // G
    vr = np.repeat(v, G, axis=2)
    for causal in (False, True):
        a = oracle.attention(q, k, v, causal=causal, scale=0.4)
        b = oracle.attention(q, kr, vr, causal=causal, scale=0.4)
        np.testing.assert_allclose(a, b, rtol=0, atol=1e-15)


# --------------------------------------------------------------------------
# 7. chunked prefill = the matching slice of a full causal prefill
# --------------------------------------------------------------------------

def test_chunked_equals_slice_of_full():
    B, S, Hq, Hkv, hd, n_new = 2, 24, 4, 2, 8, 8
    q_full = _rand((B, S, Hq, hd), 41)
    k = _rand((B, S, Hkv, hd), 42)
    v = _rand((B, S, Hkv, hd), 43)
    full = oracle.attention(q_full, k, v, causal=True, scale=0.35)
    chunk = oracle.attention(q_full[:, S - n_new:], k, v, causal=True, scale=0.35)
    np.testing.assert_allclose(chunk, full[:, S - n_new:], rtol=0, atol=1e-15)


# --------------------------------------------------------------------------
# 8. library cross-check: torch SDPA in float64 with an explicit boolean mask
# --------------------------------------------------------------------------

@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Sq,Skv", [(7, 13), (13, 13), (1, 5)])
def test_matches_torch_sdpa_f64(causal, Sq, Skv):
    B, Hq, Hkv, hd = 2, 4, 2, 16
    q = _rand((B, Sq, Hq, hd), 51, 2.0)
    k = _rand((B, Skv, Hkv, hd), 52, 2.0)
    v = _rand((B, Skv, Hkv, hd), 53)
    scale = 0.3
    got = oracle.attention(q, k, v, causal=causal, scale=scale)
    G = Hq // Hkv
    tq = torch.from_numpy(q).permute(0, 2, 1, 3)
    tk = torch.from_numpy(np.repeat(k, G, axis=2)).permute(0, 2, 1, 3)
    tv = torch.from_numpy(np.repeat(v, G, axis=2)).permute(0, 2, 1, 3)
    mask = torch.ones(Sq, Skv, dtype=torch.bool)
    if causal:  # explicit bottom-right mask (is_causal=True would be top-left)
        i = torch.arange(Sq)[:, None]
        j = torch.arange(Skv)[None, :]
        mask = j <= (Skv - Sq) + i
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=mask, scale=scale)
    np.testing.assert_allclose(got, ref.permute(0, 2, 1, 3).numpy(), rtol=0, atol=1e-13)


# --------------------------------------------------------------------------
# 9. shift invariance: adding a constant to every score of a row changes nothing
# --------------------------------------------------------------------------

def test_row_shift_invariance():
    B, Sq, Skv, Hq, hd = 1, 6, 6, 2, 8
    q = _rand((B, Sq, Hq, hd), 61)
    k = _rand((B, Skv, 1, hd), 62)
    k[..., 0] = 1.0  # a constant coordinate: q[..., 0] shifts every score of its row
    v = _rand((B, Skv, 1, hd), 63)
    a = oracle.attention(q, k, v, causal=True, scale=0.5)
    q2 = q.copy()
    q2[..., 0] += np.arange(Sq)[None, :, None] * 7.0 + 100.0
    b = oracle.attention(q2, k, v, causal=True, scale=0.5)
    np.testing.assert_allclose(a, b, rtol=0, atol=1e-12)


# --------------------------------------------------------------------------
# 10. rows that see no key (causal, Skv < Sq) are exactly zero, the rest are not
# --------------------------------------------------------------------------

def test_fully_masked_rows_are_zero():
    B, Sq, Skv, Hq, hd = 1, 6, 3, 2, 8
    q = _rand((B, Sq, Hq, hd), 71)
    k = _rand((B, Skv, 1, hd), 72)
    v = _rand((B, Skv, 1, hd), 73)
    got = oracle.attention(q, k, v, causal=True, scale=0.5)
    off = Skv - Sq  # -3: rows 0..2 see nothing
    for i in range(Sq):
        if off + i < 0:
            assert np.all(got[0, i] == 0.0)
        else:
            assert np.any(got[0, i] != 0.0)
    # row 3 sees exactly key 0
    np.testing.assert_allclose(got[0, 3, 0], v[0, 0, 0], rtol=0, atol=1e-15)


# --------------------------------------------------------------------------
# 11. the scale multiplies the scores before the softmax
# --------------------------------------------------------------------------

def test_scale_applies_to_scores():
    q = _rand((1, 5, 2, 8), 81)
    k = _rand((1, 5, 1, 8), 82)
    v = _rand((1, 5, 1, 8), 83)
    a = oracle.attention(q * 2.0, k, v, causal=True, scale=0.25)
    b = oracle.attention(q, k, v, causal=True, scale=0.5)
    np.testing.assert_allclose(a, b, rtol=0, atol=1e-14)
    c = oracle.attention(q, k, v, causal=True, scale=0.25)
    assert np.max(np.abs(b - c)) > 1e-3


# --------------------------------------------------------------------------
# 12. large score ranges do not overflow (max subtraction)
# --------------------------------------------------------------------------

def test_large_scores_are_stable():
    q = _rand((1, 4, 1, 8), 91, 300.0)
    k = _rand((1, 4, 1, 8), 92, 300.0)
    v = _rand((1, 4, 1, 8), 93)
    got = oracle.attention(q, k, v, causal=True, scale=1.0)
    assert np.all(np.isfinite(got))
    # each row is a convex combination of its visible V rows
    for i in range(4):
        lo = v[0, :i + 1, 0].min(axis=0) - 1e-12
        hi = v[0, :i + 1, 0].max(axis=0) + 1e-12
        assert np.all(got[0, i, 0] >= lo) and np.all(got[0, i, 0] <= hi)


# --------------------------------------------------------------------------
# 13. the row-sampled entry point and the thread count do not change results
# --------------------------------------------------------------------------

def test_rows_entry_point_and_threads_agree():
    B, Sq, Skv, Hq, Hkv, hd = 2, 9, 14, 4, 2, 16
    q = _rand((B, Sq, Hq, hd), 101)
    k = _rand((B, Skv, Hkv, hd), 102)
    v = _rand((B, Skv, Hkv, hd), 103)
    full1 = oracle.attention(q, k, v, causal=True, scale=0.25, nthreads=1)
    full8 = oracle.attention(q, k, v, causal=True, scale=0.25, nthreads=8)
    assert np.array_equal(full1, full8)
    rows = [(b, h, i) for b in range(B) for h in range(Hq) for i in range(Sq)]
    got = oracle.attention_rows(q, k, v, rows, causal=True, scale=0.25, nthreads=3)
    want = np.stack([full1[b, i, h] for (b, h, i) in rows])
    assert np.array_equal(got, want)


def test_bad_arguments_are_rejected():
    q = np.zeros((1, 2, 3, 4))
    k = np.zeros((1, 2, 2, 4))
    with pytest.raises(ValueError):
        oracle.attention(q, k, k)  # Hq % Hkv != 0
    with pytest.raises(ValueError):
        oracle.attention_rows(np.zeros((1, 2, 2, 4)), k, k, [(0, 0, 5)])  # row out of range


# --------------------------------------------------------------------------
# K/V-cache append: IEEE round-to-nearest-even into 16 bits, scattered to
# positions.  The roundings reduce to library conversions (numpy's float32 ->
# float16 and torch's float32 -> bfloat16, both round to nearest even), and
# hand-picked ties fix the tie rule on their own.
# --------------------------------------------------------------------------

def _round_probe_values():
    rng = np.random.default_rng(7)
    bits = rng.integers(0, 2 ** 32, size=60000, dtype=np.uint64).astype(np.uint32)
    rand = bits.view(np.float32)
    rand = rand[~np.isnan(rand)]
    # values around every f16 and bf16 binade, including the subnormal ranges
    scaled = (rng.standard_normal(40000) * np.exp2(rng.integers(-30, 18, size=40000))).astype(np.float32)
    tiny = (rng.standard_normal(20000) * np.exp2(rng.integers(-140, -120, size=20000))).astype(np.float32)
    special = np.array([0.0, -0.0, np.inf, -np.inf, 1.0, -1.0, 65504.0, 65519.996, 65520.0, 65536.0,
                        2.0 ** -24, 2.0 ** -25, 1.5 * 2.0 ** -24, 2.0 ** -14, 2.0 ** -15,
                        1 + 2.0 ** -11, 1 + 3 * 2.0 ** -11, 1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8,
                        np.finfo(np.float32).max, np.finfo(np.float32).tiny, 2.0 ** -149, 2.0 ** -133,
                        2.0 ** -134, 3 * 2.0 ** -135], dtype=np.float32)
    return np.concatenate([rand, scaled, tiny, special, -special])


def test_round_f16_matches_ieee_conversion():
    x = _round_probe_values()
    with np.errstate(over="ignore"):
        want = x.astype(np.float16).view(np.uint16)
    got = oracle.round16_bits(x, bf16=False)
    assert np.array_equal(got, want)


def test_round_bf16_matches_ieee_conversion():
    x = _round_probe_values()
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle.round16_bits(x, bf16=True)
    assert np.array_equal(got, want)


def test_round_ties_go_to_even():
    """Halfway cases, by hand: 1 + 2^-11 lies halfway between 1 and the next
    f16 (1 + 2^-10) and rounds to 1 (even); 1 + 3 2^-11 rounds up to 1 + 2^-9;
    2^-25 (half the smallest f16 subnormal) rounds to 0; 65520 rounds to
    2^16, past the largest f16, so to infinity; likewise for bf16 at 2^-8."""
    f16 = lambda v: int(oracle.round16_bits(np.float32(v), bf16=False))
    bf = lambda v: int(oracle.round16_bits(np.float32(v), bf16=True))
    assert f16(1 + 2.0 ** -11) == 0x3C00 and f16(1 + 3 * 2.0 ** -11) == 0x3C02
    assert f16(2.0 ** -25) == 0x0000 and f16(1.5 * 2.0 ** -24) == 0x0002 and f16(65520.0) == 0x7C00
    assert bf(1 + 2.0 ** -8) == 0x3F80 and bf(1 + 3 * 2.0 ** -8) == 0x3F82
    assert f16(-0.0) == 0x8000 and bf(float("-inf")) == 0xFF80
    assert f16(float("nan")) & 0x7C00 == 0x7C00 and f16(float("nan")) & 0x03FF


def test_kv_append_scatters_rounded_rows_to_positions():
    """Brute force on a tiny cache: every token's K and V row lands, rounded,
    at its position; untouched rows keep their contents; out-of-range
    positions are skipped and counted."""
    rng = np.random.default_rng(11)
    B, T, Hkv, hd, cap = 2, 5, 2, 8, 16
    k_new = (rng.standard_normal((B, T, Hkv, hd)) * 3).astype(np.float32)
    v_new = (rng.standard_normal((B, T, Hkv, hd)) * 3).astype(np.float32)
    pos = np.stack([rng.permutation(cap)[:T] for _ in range(B)]).astype(np.int32)
    pos[1, 2] = cap      # out of range: skipped
    pos[0, 4] = -1       # out of range: skipped
    for bf16 in (False, True):
        kc = np.full((B, cap, Hkv, hd), 0xABCD, dtype=np.uint16)
        vc = np.full((B, cap, Hkv, hd), 0x1234, dtype=np.uint16)
        skipped = oracle.kv_append(k_new, v_new, pos, kc, vc, bf16=bf16)
        assert skipped == 2
        if bf16:
            cvt = lambda a: torch.from_numpy(a).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        else:
            cvt = lambda a: a.astype(np.float16).view(np.uint16)
        wk = np.full_like(kc, 0xABCD)
        wv = np.full_like(vc, 0x1234)
        for b in range(B):
            for t in range(T):
                if 0 <= pos[b, t] < cap:
                    wk[b, pos[b, t]] = cvt(k_new[b, t])
                    wv[b, pos[b, t]] = cvt(v_new[b, t])
        assert np.array_equal(kc, wk) and np.array_equal(vc, wv)


def test_lse_by_brute_force_and_closed_forms():
    """The per-row log-sum-exp: exact on tiny integer inputs (50-digit decimal
    exp and ln of the visible scores), log(n) + s for n identical visible
    scores, s_0 for a row that sees one key, -inf for a row that sees none."""
    getcontext().prec = 50
    rng = np.random.default_rng(12)
    B, Hq, Hkv, Sq, Skv, hd = 1, 2, 1, 3, 5, 4
    q = rng.integers(-3, 4, size=(B, Sq, Hq, hd)).astype(np.float64)
    k = rng.integers(-3, 4, size=(B, Skv, Hkv, hd)).astype(np.float64)
    scale = 0.25
    got = oracle.lse(q, k, causal=True, scale=scale)
    off = Skv - Sq
    for hq in range(Hq):
        for i in range(Sq):
            tot = Decimal(0)
            for j in range(off + i + 1):
                sc = Decimal(scale) * Decimal(int(np.dot(q[0, i, hq], k[0, j, 0])))
                tot += sc.exp()
            assert abs(float(tot.ln()) - got[0, hq, i]) < 1e-12
    # identical keys: row i sees n = off + i + 1 equal scores s
    k2 = np.repeat(k[:, :1], Skv, axis=1)
    got2 = oracle.lse(q, k2, causal=True, scale=scale)
    for hq in range(Hq):
        for i in range(Sq):
            s0 = scale * float(np.dot(q[0, i, hq], k2[0, 0, 0]))
            assert abs(got2[0, hq, i] - (s0 + math.log(off + i + 1))) < 1e-12
    # Sq > Skv: the first rows see nothing; the first row that sees one key gives s_0
    got3 = oracle.lse(q[:, :3], k[:, :2], causal=True, scale=scale)
    assert np.isneginf(got3[0, :, 0]).all() and np.isfinite(got3[0, :, 1:]).all()
    assert abs(got3[0, 0, 1] - scale * float(np.dot(q[0, 1, 0], k[0, 0, 0]))) < 1e-12


def _scatter_to_pages(kc, table, page, nb, fill):
    """The inverse of a paged gather, written as a cache manager fills pages:
    walk each sequence's table entries in order and copy the next `page`
    keys into that block, row by row.  Pool rows no key lands in keep `fill`."""
    B, kv_len = kc.shape[:2]
    pool = np.full((nb, page) + kc.shape[2:], fill)
    for b in range(B):
        src = 0  # next key of sequence b to place
        for entry in table[b]:
            for r in range(page):
                if src >= kv_len:
                    break
                pool[entry, r] = kc[b, src]
                src += 1
    return pool


def test_gather_pages_inverts_a_page_scatter():
    """Scatter contiguous keys into a shuffled pool (the page walk above, which
    never forms j // page or j % page), then gather them back through the block
    table: the result must be the original keys, bit for bit.  Pool rows no key
    was written to hold NaN, so a gather that reads any of them fails.  The
    sizes keep every swapped index in range, so a page/row mix-up gives wrong
    values rather than an index error."""
    rng = np.random.default_rng(3)
    B, kv_len, Hkv, hd, page, max_pages, nb = 2, 14, 2, 3, 4, 5, 12
    kc = rng.standard_normal((B, kv_len, Hkv, hd))
    perm = rng.permutation(nb)
    table = perm[: B * max_pages].reshape(B, max_pages)
    pool = _scatter_to_pages(kc, table, page, nb, np.nan)
    got = oracle.gather_pages(pool, table, kv_len, page)
    assert got.shape == kc.shape
    assert np.array_equal(got, kc)
    # a table that maps both sequences to the same blocks reads the same keys for both
    shared = np.stack([table[0], table[0]])
    pool2 = _scatter_to_pages(kc[:1], shared[:1], page, nb, np.nan)
    got2 = oracle.gather_pages(pool2, shared, kv_len, page)
    assert np.array_equal(got2[0], kc[0]) and np.array_equal(got2[1], kc[0])


# --------------------------------------------------------------------------
# planted mistakes: each wrong variant of the oracle fails at least one pin
# --------------------------------------------------------------------------

def _pin_battery():
    """Every pin above, at fixed arguments, as a list of (name, callable)."""
    return [
        ("brute_force_causal_3x5", lambda: test_brute_force_exact_tiny(True, 3, 5)),
        ("brute_force_causal_5x3", lambda: test_brute_force_exact_tiny(True, 5, 3)),
        ("brute_force_full_4x4", lambda: test_brute_force_exact_tiny(False, 4, 4)),
        ("mask_pattern_4x4", test_brute_force_4x4_mask_pattern),
        ("identical_keys", lambda: test_identical_keys_give_prefix_mean(5, 12)),
        ("one_hot", test_one_hot_dominant_key),
        ("prob_rows", test_probability_rows_sum_to_one_and_respect_mask),
        ("single_key", test_single_key_returns_that_value),
        ("gqa", test_gqa_equals_repeated_mha),
        ("chunked", test_chunked_equals_slice_of_full),
        ("sdpa", lambda: test_matches_torch_sdpa_f64(True, 7, 13)),
        ("shift", test_row_shift_invariance),
        ("masked_rows", test_fully_masked_rows_are_zero),
        ("scale", test_scale_applies_to_scores),
        ("large_scores", test_large_scores_are_stable),
        ("round_f16", test_round_f16_matches_ieee_conversion),
        ("round_bf16", test_round_bf16_matches_ieee_conversion),
        ("round_ties", test_round_ties_go_to_even),
        ("kv_append", test_kv_append_scatters_rounded_rows_to_positions),
        ("lse", test_lse_by_brute_force_and_closed_forms),
        ("gather_pages", test_gather_pages_inverts_a_page_scatter),
    ]


@pytest.mark.parametrize("kind", [k for k in oracle.PLANTED_MISTAKES if k != "none"])
def test_planted_mistakes_are_caught(kind):
    """Plant one mistake in the oracle itself, run every pin, and require that
    at least one pin fails; the correct oracle passes them all."""
    failed = []
    try:
        oracle.plant_mistake(kind)
        for name, pin in _pin_battery():
            try:
                with np.errstate(all="ignore"):
                    pin()
            except AssertionError:
                failed.append(name)
    finally:
        oracle.plant_mistake("none")
    assert failed, f"no pin caught the planted mistake {kind!r}"
    for name, pin in _pin_battery():  # and the restored oracle passes again
        pin()
