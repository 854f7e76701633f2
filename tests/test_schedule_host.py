"""The split-KV work split (host logic, no GPU): fa_debug_schedule returns
what fa_prefill_ws would launch for a shape on a GPU of a given SM count.

Every (query-tile pair, KV step) must belong to exactly one CTA, in order;
with no more pairs than CTAs every CTA computes one piece of one pair, pieces
of a pair are near-equal and none is shorter than 2 steps unless the pair is
whole; sibling pairs of one GQA group with equal lengths are cut at the same
steps (their CTAs then stream the same K/V tiles together); with more pairs
than CTAs the contiguous stream-K ranges carry near-equal cost.  The piece
slot count matches the pieces of the split pairs.
"""
import math

import pytest

SMS = 152
SHAPES = [  # (B, Hq, Hkv, Sq, Skv, causal)
    (1, 32, 8, 128, 32768, True),     # 128-row chunk over a 32K context: 16 pairs
    (1, 1, 1, 256, 256, True),        # one head, one pair of 2 tiles
    (1, 2, 1, 128, 4000, True),       # one GQA pair
    (2, 8, 2, 300, 5000, True),       # ragged rows, GQA
    (1, 4, 4, 1000, 1000, False),     # non-causal MHA row pairs
    (1, 32, 32, 2048, 2048, True),    # 256 pairs: stream-K ranges
    (1, 32, 8, 8192, 8192, True),     # 1024 pairs
    (4, 32, 8, 512, 8192, True),      # chunked prefill, 256 pairs
    (1, 32, 32, 2659, 2659, True),    # odd tile count (tile 0 alone), 352 pairs: stream-K ranges
    (1, 24, 8, 1152, 3000, True),     # GQA 3, odd tile count, keys ahead of the queries
]


@pytest.fixture(scope="module")
def fa():
    import causal_prefill_flash_gb300 as fa
    fa.build()  # a no-op when the library is up to date
    fa.load()
    return fa


def _segments(sc):
    """The CTAs' ranges as lists of (pair, first step, end step)."""
    steps = sc["pair_steps"]
    out = []
    for c in range(sc["ctas"]):
        u, j = sc["cta_pair"][c], sc["cta_step"][c]
        ue, je = sc["cta_pair"][c + 1], sc["cta_step"][c + 1]
        segs = []
        while u < ue or (u == ue and j < je):
            end = je if u == ue else steps[u]
            segs.append((u, j, end))
            u, j = u + 1, 0
        out.append(segs)
    return out


@pytest.mark.parametrize("shape", SHAPES, ids=[f"B{s[0]}H{s[1]}-{s[2]}S{s[3]}x{s[4]}{'c' if s[5] else 'n'}" for s in SHAPES])
def test_every_step_belongs_to_one_cta(fa, shape):
    sc = fa.debug_schedule(*shape, sms=SMS)
    assert 1 <= sc["ctas"] <= min(SMS, 256)
    assert (sc["cta_pair"][0], sc["cta_step"][0]) == (0, 0)
    assert (sc["cta_pair"][-1], sc["cta_step"][-1]) == (sc["pairs"], 0)
    starts = list(zip(sc["cta_pair"], sc["cta_step"]))
    assert all(a < b for a, b in zip(starts, starts[1:])), "CTA ranges must strictly increase"
    covered = {}
    for segs in _segments(sc):
        assert segs, "a CTA with no work"
        for u, j, e in segs:
            assert 0 <= j <= e <= sc["pair_steps"][u]
            for t in range(j, e):
                covered[(u, t)] = covered.get((u, t), 0) + 1
    want = {(u, t) for u, n in enumerate(sc["pair_steps"]) for t in range(n)}
    assert set(covered) == want and all(v == 1 for v in covered.values())


@pytest.mark.parametrize("shape", [s for s in SHAPES if s[3] <= 5000 and s[1] * s[0] * math.ceil(s[3] / 256) <= SMS])
def test_one_piece_per_cta_when_pairs_fit(fa, shape):
    sc = fa.debug_schedule(*shape, sms=SMS)
    assert sc["pairs"] <= SMS and sc["one_segment"]
    segs = _segments(sc)
    assert all(len(s) == 1 for s in segs)
    by_pair = {}
    for (u, j, e), in segs:
        by_pair.setdefault(u, []).append(e - j)
    for u, lens in by_pair.items():
        n = sc["pair_steps"][u]
        if len(lens) > 1:
            assert min(lens) >= 2, "a piece shorter than two KV steps"
            assert max(lens) - min(lens) <= 1, "pieces of one pair are near-equal"
        else:
            assert lens == [n]
    # the next CTA would not have shortened the longest piece by splitting a pair
    # that still allowed it: all pairs are split about equally finely
    longest = max(max(v) for v in by_pair.values())
    for u, lens in by_pair.items():
        n = sc["pair_steps"][u]
        if n // (len(lens) + 1) >= 2 and sc["ctas"] < SMS:
            assert False, "CTAs left unused while a pair could still be split"
        assert math.ceil(n / len(lens)) <= longest
    # split pairs: every pair in more than one piece, one slot per piece
    split = [u for u, lens in by_pair.items() if len(lens) > 1]
    assert sc["split_pairs"] == len(split)
    assert sc["slots"] == sum(len(by_pair[u]) for u in split)


def test_long_context_chunk_cuts_sibling_pairs_alike(fa):
    sc = fa.debug_schedule(1, 32, 8, 128, 32768, True, sms=SMS)
    assert sc["pairs"] == 16 and sc["ctas"] == SMS and sc["one_segment"]
    cuts = {}
    for (u, j, e), in _segments(sc):
        cuts.setdefault(u, []).append(j)
    for u in range(0, 16, 2):  # pairs 2i and 2i+1: the two query-head pairs of one KV head
        assert cuts[u] == cuts[u + 1]
    lens = [e - j for (u, j, e), in _segments(sc)]
    assert max(lens) - min(lens) <= 4  # 256 / 9 vs 256 / 10 steps


@pytest.mark.parametrize("shape", [s for s in SHAPES if s[1] * s[0] * math.ceil(s[3] / 256) > SMS])
def test_stream_k_ranges_carry_equal_cost(fa, shape):
    sc = fa.debug_schedule(*shape, sms=SMS)
    assert not sc["one_segment"] and sc["ctas"] == min(SMS, 256)
    # cost model: 4 per KV step and 8 per segment (quarter steps); every CTA
    # within one pair's cost of the mean
    costs = [sum(4 * (e - j) + 8 for u, j, e in segs) for segs in _segments(sc)]
    mean = sum(costs) / len(costs)
    biggest = 4 * max(sc["pair_steps"]) + 8
    assert max(costs) <= mean + biggest and min(costs) >= mean - biggest


def test_schedule_rejects_bad_shapes(fa):
    for bad in ((0, 8, 2, 128, 128, True), (1, 8, 3, 128, 128, True), (1, 8, 2, 0, 128, True)):
        with pytest.raises(fa.FaError):
            fa.debug_schedule(*bad, sms=SMS)
    with pytest.raises(fa.FaError):
        fa.debug_schedule(1, 8, 2, 128, 128, True, sms=0)


def test_static_scratch_bound_holds_for_every_schedule(fa):
    """fa_prefill_ws_static's documented bound: pieces <= 2 * CTAs - 1, so a
    152-SM GPU needs at most 1048576 + 303 * 1024 * 128 = 40763392 bytes of the
    40 MiB static scratch at hd 128.  A seeded sweep of shapes (GQA and MHA,
    causal and not, chunked and square, tiny to many pairs)."""
    import random
    rng = random.Random(7)
    worst = 0
    for _ in range(300):
        G = rng.choice([1, 2, 4, 8])
        Hkv = rng.choice([1, 2, 4, 8])
        Hq = G * Hkv
        B = rng.choice([1, 1, 2, 4])
        Sq = rng.choice([1, 77, 128, 300, 512, 1000, 2048, 2659])
        Skv = Sq + rng.choice([0, 0, 128, 1000, 7680, 32640])
        causal = rng.random() < 0.8
        sc = fa.debug_schedule(B, Hq, Hkv, Sq, Skv, causal, sms=SMS)
        assert sc["slots"] <= 2 * sc["ctas"] - 1
        need = 1048576 + sc["slots"] * 1024 * 128
        worst = max(worst, need)
        assert need <= 40 * 1024 * 1024
    assert worst <= 40763392


def test_row_pairing_choice(fa):
    """Which tile of a head the one-shot grid leaves without a partner (odd
    tile counts of row pairs): the last one near one wave of CTAs, where the
    longest CTA sets the time, and tile 0 from ~1.5 waves on, where the total
    of the CTAs' KV steps does; nothing when no tile goes alone."""
    assert not fa.debug_row_pairing(1, 32, 32, 2048, 2048, True, SMS)  # even tile count
    assert not fa.debug_row_pairing(1, 32, 8, 2659, 2659, True, SMS)   # head pairs (GQA 4)
    assert not fa.debug_row_pairing(1, 4, 4, 100, 100, True, SMS)      # one tile
    assert not fa.debug_row_pairing(1, 32, 32, 1152, 1152, True, SMS)  # 160 CTAs
    assert fa.debug_row_pairing(1, 40, 40, 1152, 1152, True, SMS)      # 200 CTAs
    assert fa.debug_row_pairing(1, 32, 32, 2659, 2659, True, SMS)      # 352 CTAs
    assert fa.debug_row_pairing(1, 24, 8, 2659, 2659, True, SMS)       # GQA 3, 264 CTAs
    assert not fa.debug_row_pairing(1, 40, 40, 1152, 1152, False, SMS)  # equal CTAs: no gain
    with pytest.raises(fa.FaError):
        fa.debug_row_pairing(1, 3, 2, 100, 100, True, SMS)


def _kv_tiles(Sq, Skv, causal, t):
    off = Skv - Sq
    q_last = min(128 * t + 128, Sq) - 1
    hi = min(Skv, off + q_last + 1) if causal else Skv
    return -(-hi // 128) if hi > 0 else 0


@pytest.mark.parametrize("shape", [(1, 4, 4, 1152, 1152, True), (1, 3, 1, 2659, 2659, True),
                                   (2, 2, 2, 300, 700, True), (1, 2, 2, 1152, 1152, False)])
def test_split_pairs_leave_tile_0_alone(fa, shape):
    """The split-KV paths pair the tiles of an odd count as (0), (1, 2),
    (3, 4), ...: the pairs' KV steps, longest first with the heads inner,
    follow from that pairing alone."""
    B, Hq, Hkv, Sq, Skv, causal = shape
    n_qt = -(-Sq // 128)
    assert n_qt % 2 == 1
    want = []
    for pq in range((n_qt + 1) // 2 - 1, -1, -1):
        tiles = [0] if pq == 0 else [2 * pq - 1, 2 * pq]
        want += [max(_kv_tiles(Sq, Skv, causal, t) for t in tiles)] * (B * Hq)
    assert fa.debug_schedule(B, Hq, Hkv, Sq, Skv, causal, sms=SMS)["pair_steps"] == want


def test_row_pairing_cache_is_consistent(fa):
    """The choice is cached per shape (eight entries): more shapes than
    entries, asked twice in a different order, give the same answers."""
    shapes = [(1, h, h, s, s, True) for h in (24, 32, 40) for s in (1152, 1400, 2432, 2659)]
    first = {sh: fa.debug_row_pairing(*sh, SMS) for sh in shapes}
    again = {sh: fa.debug_row_pairing(*sh, SMS) for sh in reversed(shapes)}
    assert first == again
    assert any(first.values()) and not all(first.values())
