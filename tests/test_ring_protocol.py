"""The shared-memory ring of the TMA-fed kernels, simulated on the host.

One producer issues stages 0, 1, 2, ... into slots k % S: before stage j it waits until the slot's
previous use (stage j - S) has been released, and until stage j - depth has landed. Copies land in
any order. Consumer groups take the stages in turn (stage k goes to group k % G) and wait for stage k
by the parity of the slot's full-barrier phase, as `mbarrier.try_wait.parity` does: the wait passes
when the number of completed phases of the slot has the other parity than stage k's use of it.
That test cannot tell stage k's phase from the phase of stage k - 2S, so it is only sound when the
slot's previous use, stage k - S, has completed by the time the group waits. The kernels keep that
true in one of two ways: S a multiple of G (the group consumed stage k - S itself), or
depth <= S - G (every stage up to k - G - depth has landed before stage k - G was issued).
"""
from __future__ import annotations

import random

import pytest


def false_pass(S: int, G: int, depth: int, n_stages: int, seed: int) -> bool:
    """One random interleaving; True if a consumer passed its wait before its stage had landed."""
    rng = random.Random(seed)
    issued = 0                   # stages issued so far
    landed = set()               # stages whose copies have completed
    phases = [0] * S             # completed full-barrier phases per slot
    released = set()             # stages released by their consumer
    nxt = list(range(G))         # next stage of each group
    while True:
        acts = []
        j = issued
        if j < n_stages and (j < S or (j - S) in released) and (j < depth or (j - depth) in landed):
            acts.append(("issue", j))
        for k in range(issued):
            if k not in landed:
                acts.append(("land", k))
        for g in range(G):
            k = nxt[g]
            if k < n_stages and (phases[k % S] & 1) != ((k // S) & 1):
                acts.append(("consume", g))
        if not acts:
            return False
        kind, v = rng.choice(acts)
        if kind == "issue":
            issued += 1
        elif kind == "land":
            landed.add(v)
            phases[v % S] += 1
        else:
            k = nxt[v]
            if k not in landed:
                return True
            released.add(k)
            nxt[v] += G


def first_false_pass(S, G, depth, runs=400, n_stages=60):
    return next((seed for seed in range(runs) if false_pass(S, G, depth, n_stages, seed)), None)


@pytest.mark.parametrize("S,G,depth", [(12, 3, 6), (6, 3, 6), (9, 3, 6), (11, 2, 4), (5, 2, 2), (8, 1, 8), (4, 2, 4)])
def test_ring_rules_never_pass_early(S, G, depth):
    """Every configuration the launchers allow: S % G == 0 or depth <= S - G."""
    assert S % G == 0 or depth <= S - G
    assert first_false_pass(S, G, depth) is None


@pytest.mark.parametrize("S,G,depth", [(8, 3, 6), (3, 2, 2), (7, 2, 6)])
def test_ring_without_the_rule_can_pass_early(S, G, depth):
    """The configurations the rule excludes: some interleaving lets a group read a stage whose
    copy has not landed (8 slots, 3 groups, depth 6 is the ring the first version of the
    register-resident kernels used)."""
    assert S % G != 0 and depth > S - G
    assert first_false_pass(S, G, depth, runs=4000) is not None
