"""The CTA-pair kernel's load protocol, checked on a model (host only).

Each CTA r of the pair loads Q and its halves of K and V into a ring of NSLOT
slots (load i in slot i % NSLOT: K_0 with Q, then V_j and K_j+1 as pair j).
Its own barriers count only its own copies: the Q barrier and pair barrier
j % NPB, re-armed only after the previous phase completed.  A forwarder in
each CTA waits for those phases and arrives, once per phase, on CTA 0's joint
barrier of the same index, which completes when both CTAs' forwards are in.
Two MMA issuers (tiles A and B) wait for the joint barriers and, when their
MMAs reading a slot have completed, each commit one arrival on that slot's
empty barrier in both CTAs (count 2); a producer reuses a slot after that
phase completed.

An mbarrier wait names a phase by its parity only.  The model runs all of
these with random delays and checks that no wait ever sees its barrier two
phases ahead, that no phase of an empty barrier mixes the commits of two
different loads, and that nothing deadlocks -- for the kernel's ring (6 slots,
3 pair barriers).  It also checks that fewer pair barriers, a producer that
reuses a slot early, or a forwarder that does not wait each do fail, so the
model can see the failures the kernel's rules guard against.
"""
import heapq
import random

import pytest


def simulate(nslot, npb, n, seed, plant=None):
    """One run over n KV steps; returns None or a description of the fault.
    plant: None (the kernel's protocol), "early_reuse" (a producer reuses a
    slot one free early) or "eager_forward" (a forwarder does not wait for
    its own CTA's loads)."""
    rng = random.Random(seed)
    ev, seq = [], [0]

    def push(tm, kind, data):
        seq[0] += 1
        heapq.heappush(ev, (tm, seq[0], kind, data))

    def delay(scale=1.0):
        return rng.random() * rng.choice([0.3, 1.0, 4.0]) * scale

    time = 0.0
    loads = 2 * n  # load 0: K_0 (with Q); 2j+1: V_j; 2j+2: K_j+1
    # per CTA
    issued = [0, 0]
    prod_busy = [0.0, 0.0]
    landed = [set(), set()]
    local_pair_done = [[0] * npb for _ in range(2)]  # completed phases per local pair barrier
    local_q_done = [0, 0]
    pair_complete = [set(), set()]
    empty_done = [[0] * nslot for _ in range(2)]  # completed phases per slot barrier
    empty_arrivals = [[[] for _ in range(nslot)] for _ in range(2)]  # arrivals of the open phase: load index
    fwd_next = [-1, -1]  # -1: the Q barrier next, else the pair index next
    fwd_busy = [0.0, 0.0]
    # CTA 0's joint barriers
    joint_q = [0]  # arrivals (completes at 2)
    joint_pair_done = [0] * npb
    joint_pair_open = [0] * npb  # arrivals in the open phase
    joint_q_done = [False]
    # issuers
    iss_j = [-1, -1]  # -1: waiting for the joint Q barrier
    iss_busy = [0.0, 0.0]
    iss_last_done = [0.0, 0.0]  # completion time of the issuer's latest MMAs (in issue order)

    def pair_loads(j):
        return [2 * j + 1] + ([2 * j + 2] if 2 * j + 2 < loads else [])

    def commit_empty(x, load_i):
        # arrives on the slot's barrier in both CTAs once x's earlier MMAs are done
        t = max(iss_last_done[x], time) + delay(0.5)
        for r in (0, 1):
            push(t, "empty_arrive", (r, load_i))

    while True:
        progressed = False
        for r in (0, 1):  # producers
            i = issued[r]
            if i < loads and time >= prod_busy[r]:
                ok = True
                if i >= nslot:
                    s, k = i % nslot, i // nslot - 1  # phase k of slot s: the frees of load i - nslot
                    if empty_done[r][s] >= k + 2:
                        return f"CTA {r}: empty barrier of slot {s} two phases ahead at load {i}"
                    ok = empty_done[r][s] >= (k if plant == "early_reuse" else k + 1)
                if ok and (i & 1):
                    pj = (i - 1) >> 1
                    if pj >= npb:
                        b, k = pj % npb, (pj - npb) // npb
                        if local_pair_done[r][b] >= k + 2:
                            return f"CTA {r}: pair barrier {b} two phases ahead when re-armed for pair {pj}"
                        ok = local_pair_done[r][b] >= k + 1
                if ok:
                    push(time + delay(2.0), "land", (r, i))
                    issued[r] += 1
                    prod_busy[r] = time + delay(0.3)
                    push(prod_busy[r], "tick", 0)
                    progressed = True
        for r in (0, 1):  # forwarders
            if time < fwd_busy[r]:
                continue
            j = fwd_next[r]
            if j == -1:
                if local_q_done[r] >= 1:
                    push(time + delay(), "joint_q", r)
                    fwd_next[r] = 0
                    fwd_busy[r] = time + delay(0.3)
                    push(fwd_busy[r], "tick", 0)
                    progressed = True
            elif j < n:
                b, k = j % npb, j // npb
                if local_pair_done[r][b] >= k + 2:
                    return f"CTA {r}: forwarder saw pair barrier {b} two phases ahead at pair {j}"
                if plant == "eager_forward" or local_pair_done[r][b] >= k + 1:
                    push(time + delay(), "joint_pair", (r, j))
                    fwd_next[r] = j + 1
                    fwd_busy[r] = time + delay(0.3)
                    push(fwd_busy[r], "tick", 0)
                    progressed = True
        for x in (0, 1):  # MMA issuers
            if time < iss_busy[x]:
                continue
            j = iss_j[x]
            if j == -1:
                if joint_q_done[0]:
                    iss_last_done[x] = max(iss_last_done[x], time) + delay()  # S_X(0)
                    commit_empty(x, 0)  # K_0
                    iss_j[x] = 0
                    iss_busy[x] = time + delay(0.5)
                    push(iss_busy[x], "tick", 0)
                    progressed = True
            elif j < n:
                b, k = j % npb, j // npb
                if joint_pair_done[b] >= k + 2:
                    return f"issuer {x}: joint pair barrier {b} two phases ahead at step {j}"
                if joint_pair_done[b] >= k + 1:
                    # S_X(j+1) and P V_X(j), each after a softmax that takes a while
                    iss_last_done[x] = max(iss_last_done[x], time) + delay(3.0)
                    commit_empty(x, 2 * j + 1)  # V_j
                    if 2 * j + 2 < loads:
                        commit_empty(x, 2 * j + 2)  # K_j+1
                    iss_j[x] = j + 1
                    iss_busy[x] = time + delay(2.0)
                    push(iss_busy[x], "tick", 0)
                    progressed = True
        if all(i >= loads for i in issued) and all(j >= n for j in iss_j) and all(f >= n for f in fwd_next):
            return None
        if not progressed:
            if not ev:
                return f"deadlock: loads {issued}, forwarders {fwd_next}, issuers {iss_j}"
            time, _, kind, data = heapq.heappop(ev)
            if kind == "land":
                r, i = data
                landed[r].add(i)
                if i == 0:
                    local_q_done[r] += 1
                else:
                    pj = (i - 1) >> 1
                    if pj not in pair_complete[r] and all(y in landed[r] for y in pair_loads(pj)):
                        pair_complete[r].add(pj)
                        local_pair_done[r][pj % npb] += 1
            elif kind == "joint_q":
                joint_q[0] += 1
                if joint_q[0] == 2:
                    joint_q_done[0] = True
            elif kind == "joint_pair":
                r, j = data
                b = j % npb
                joint_pair_open[b] += 1
                if joint_pair_open[b] == 2:
                    joint_pair_open[b] = 0
                    joint_pair_done[b] += 1
            elif kind == "empty_arrive":
                r, i = data
                s = i % nslot
                arr = empty_arrivals[r][s]
                arr.append(i)
                if len(arr) == 2:
                    if arr[0] != arr[1]:
                        return f"CTA {r}: a phase of slot {s}'s empty barrier mixed the frees of loads {arr}"
                    arr.clear()
                    empty_done[r][s] += 1


def test_kernel_rule_never_runs_two_phases_ahead():
    nslot, npb = 6, 3  # the kernel's ring: six 16 KB halves, pair j and pair j + 3 share two slots
    for seed in range(2500):
        fault = simulate(nslot, npb, 1 + seed % 40, seed)
        assert fault is None, f"seed {seed}: {fault}"


def test_fewer_pair_barriers_do_run_ahead():
    faults = [simulate(6, 2, 1 + seed % 40, seed) for seed in range(2500)]
    assert any(f and "two phases ahead" in f for f in faults), set(faults)


@pytest.mark.parametrize("plant", ["early_reuse", "eager_forward"])
def test_the_model_sees_a_broken_protocol(plant):
    """A producer that reuses a slot before both issuers freed it, or a
    forwarder that arrives before its CTA's loads landed, is caught."""
    faults = [simulate(6, 3, 1 + seed % 40, seed, plant) for seed in range(800)]
    assert sum(1 for f in faults if f) > 100
