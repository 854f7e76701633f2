"""The K/V ring's barrier-reuse rule, checked on a model (host only).

The one-shot kernel completes V_j and K_{j+1} on one "pair" barrier, reused
every NPB pairs, and at hd 128 frees K_j and V_j with one commit on a
"pair-empty" barrier, reused every NPE pairs.  An mbarrier wait names a phase
only by its parity, so a barrier must never complete two phases while a
waiter still wants the older one.  The kernel's rule: the producer re-arms a
pair barrier only after its previous phase completed, NPB = ceil(NSLOT / 2)
(2 NPB >= NSLOT) and NPE = NSLOT // 2 + 1 (2 NPE > NSLOT).  This model runs
the producer (loads in order into NSLOT slots, each landing after a random
delay), the MMA thread (waits for pair j, then frees its slots after a random
delay) and random thread delays, and checks that no wait ever sees its
barrier two phases ahead and that nothing deadlocks -- for the ring depths the
kernel uses (5 slots at hd 128, 8 at hd 64) -- and that a smaller NPB does
break, so the model can see the failure it guards against.
"""
import heapq
import random

import pytest


def simulate(nslot, npb, npe, n, seed, pair_empty=True):
    """One run over n KV steps; returns None or a description of the fault."""
    rng = random.Random(seed)
    ev, seq = [], [0]

    def push(tm, kind, data):
        seq[0] += 1
        heapq.heappush(ev, (tm, seq[0], kind, data))

    time = 0.0
    full_done = [0] * npb
    empty_done = [0] * npe
    slot_frees = [0] * nslot
    landed, completed = set(), set()
    issued, mma_j, mma_busy, prod_busy = 0, -1, 0.0, 0.0

    def pair_loads(j):
        return [2 * j + 1] + ([2 * j + 2] if 2 * j + 2 < 2 * n else [])

    while True:
        progressed = False
        if issued < 2 * n and time >= prod_busy:  # producer: load `issued`
            i, ok = issued, True
            if i >= nslot:
                if pair_empty:
                    e = (i - nslot) >> 1
                    b, k = e % npe, e // npe
                    if empty_done[b] >= k + 2:
                        return f"pair-empty barrier two phases ahead at load {i}"
                    ok = empty_done[b] == k + 1
                else:
                    ok = slot_frees[i % nslot] >= i // nslot
            if ok and (i & 1):
                pj = (i - 1) >> 1
                if pj >= npb and (pj - npb) not in completed:
                    ok = False
            if ok:
                push(time + rng.random() * rng.choice([0.5, 2.0, 6.0]), "land", i)
                issued += 1
                prod_busy = time + rng.random() * 0.3
                push(prod_busy, "tick", 0)
                progressed = True
        if time >= mma_busy:  # MMA thread
            if mma_j == -1:
                if 0 in landed:  # K_0 arrives with Q
                    mma_j, progressed = 0, True
                    if not pair_empty:
                        push(time + rng.random(), "free_slot", 0)
                    mma_busy = time + rng.random()
                    push(mma_busy, "tick", 0)
            elif mma_j < n:
                j = mma_j
                b, k = j % npb, j // npb
                if full_done[b] >= k + 2:
                    return f"pair barrier two phases ahead at step {j}"
                if full_done[b] == k + 1:
                    if pair_empty:
                        push(time + rng.random() * 3, "free_pair", j)
                    else:
                        push(time + rng.random() * 3, "free_slot", 2 * j + 1)
                        if 2 * j + 2 < 2 * n:
                            push(time + rng.random() * 2, "free_slot", 2 * j + 2)
                    mma_j += 1
                    progressed = True
                    mma_busy = time + rng.random() * 4
                    push(mma_busy, "tick", 0)
            else:
                return None
        if not progressed:
            if not ev:
                return f"deadlock: {issued} loads issued, MMA at step {mma_j}"
            time, _, kind, data = heapq.heappop(ev)
            if kind == "land":
                landed.add(data)
                if data > 0:
                    pj = (data - 1) >> 1
                    if pj not in completed and all(x in landed for x in pair_loads(pj)):
                        completed.add(pj)
                        full_done[pj % npb] += 1
            elif kind == "free_pair":
                empty_done[data % npe] += 1
            elif kind == "free_slot":
                slot_frees[data % nslot] += 1


def kernel_npb(nslot):
    return (nslot + 1) // 2


def kernel_npe(nslot):
    return nslot // 2 + 1


@pytest.mark.parametrize("nslot,pair_empty", [(5, True), (5, False), (8, False), (8, True)])
def test_kernel_rule_never_runs_two_phases_ahead(nslot, pair_empty):
    npb, npe = kernel_npb(nslot), kernel_npe(nslot)
    assert 2 * npb >= nslot and 2 * npe > nslot
    for seed in range(3000):
        fault = simulate(nslot, npb, npe, 1 + seed % 40, seed, pair_empty)
        assert fault is None, f"NSLOT={nslot} seed {seed}: {fault}"


@pytest.mark.parametrize("nslot", [5, 8])
def test_a_smaller_pair_count_does_run_ahead(nslot):
    npb = kernel_npb(nslot) - 1
    faults = [simulate(nslot, npb, kernel_npe(nslot), 1 + seed % 40, seed, False) for seed in range(3000)]
    assert any(f and "two phases ahead" in f for f in faults)
