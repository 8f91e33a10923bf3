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


@pytest.mark.parametrize("S,G,depth", [(12, 3, 6), (6, 3, 6), (9, 3, 6), (11, 2, 4), (5, 2, 2), (8, 1, 8), (4, 2, 4),
                                         (10, 5, 10), (10, 5, 6), (12, 4, 6), (12, 2, 12), (6, 1, 4)])
def test_ring_rules_never_pass_early(S, G, depth):
    """Every configuration the launchers allow: S % G == 0 or depth <= S - G. Among them the rings the
    kernels run: ten stages for five groups with all or six in flight (register-resident rows),
    twelve stages for four groups (narrow fp16 rows), twelve for the prologue's two halves with all
    in flight, six for one group (backward)."""
    assert S % G == 0 or depth <= S - G
    assert first_false_pass(S, G, depth) is None


@pytest.mark.parametrize("S,G,depth", [(8, 3, 6), (3, 2, 2), (7, 2, 6)])
def test_ring_without_the_rule_can_pass_early(S, G, depth):
    """The configurations the rule excludes: some interleaving lets a group read a stage whose
    copy has not landed (8 slots, 3 groups, depth 6 is the ring the first version of the
    register-resident kernels used)."""
    assert S % G != 0 and depth > S - G
    assert first_false_pass(S, G, depth, runs=4000) is not None


# ------------------------------------------------------------------------------------------------
# The work queue (cluster launch control) of the same kernels, simulated on the host.
#
# A grid of `grid` chunks, one per CTA; the first `resident` CTAs start, the others wait to be
# cancelled. A resident CTA keeps kReq requests in flight. The scheduler answers pending requests
# in any order (across CTAs and within one): a request succeeds with a chunk of a CTA that has not
# started while there is one, and fails once there is none. A CTA reads its answers in the order it
# issued them (the response slots are mbarrier phases). Rule of the hardware: no request may follow
# an observed failure.
# ------------------------------------------------------------------------------------------------
def run_queue(grid: int, resident: int, k_req: int, seed: int, take_late: bool, in_order: bool = False):
    """Returns (processed chunk list, rule violations). take_late=True is the kernels' ClcQueue
    (a success read after a failure is taken over); False is the discard-after-failure rule."""
    rng = random.Random(seed)
    pool = list(range(resident, grid))
    processed = list(range(resident))   # every resident CTA processes its own chunk first
    answers = {}                         # (cta, n) -> chunk id or None (failure), once answered
    pending = []                         # (cta, n) issued, not yet answered
    state = {}
    for c in range(resident):
        state[c] = {"issued": k_req, "answered": 0, "failed": False, "done": False, "draining": False}
        pending += [(c, n) for n in range(k_req)]
    violations = 0
    while True:
        acts = [("answer", p) for p in pending
                if not in_order or p[1] == min(n for c, n in pending if c == p[0])]
        for c, st in state.items():
            if not st["done"] and st["answered"] < st["issued"] and (c, st["answered"]) in answers:
                acts.append(("read", c))
            elif not st["done"] and st["answered"] == st["issued"]:
                acts.append(("finish", c))
        if not acts:
            break
        kind, v = rng.choice(acts)
        if kind == "answer":
            pending.remove(v)
            answers[v] = pool.pop(rng.randrange(len(pool))) if pool else None
        elif kind == "finish":
            state[v]["done"] = True
        else:
            st = state[v]
            got = answers[(v, st["answered"])]
            st["answered"] += 1
            if st["draining"]:
                continue                  # discard rule: answers after the first failure are dropped
            if got is None:
                st["failed"] = True
                if not take_late:
                    st["draining"] = True
                continue
            processed.append(got)
            if not st["failed"]:
                pending.append((v, st["issued"]))
                st["issued"] += 1
            elif not take_late:
                violations += 1
    for c, st in state.items():
        if st["answered"] != st["issued"]:
            violations += 1               # a CTA left with a request in flight
    return processed, violations


@pytest.mark.parametrize("grid,resident,k_req", [(40, 8, 2), (17, 16, 2), (100, 3, 3), (9, 9, 2), (64, 12, 1)])
def test_work_queue_processes_every_chunk_once(grid, resident, k_req):
    for seed in range(300):
        done, bad = run_queue(grid, resident, k_req, seed, take_late=True)
        assert bad == 0
        assert sorted(done) == list(range(grid)), (seed, sorted(done))


def test_dropping_late_answers_can_lose_a_chunk():
    """The rule the kernels used before: stop reading at the first failure and discard the answers
    still in flight. When the scheduler answers a later request before an earlier one, a success
    can arrive after a failure, and its chunk is never processed."""
    lost = [s for s in range(2000)
            if sorted(run_queue(40, 8, 2, s, take_late=False)[0]) != list(range(40))]
    assert lost, "no interleaving lost a chunk"


def test_in_order_answers_make_both_rules_agree():
    """If the scheduler answers each CTA's requests in issue order, a failure is followed only by
    failures, so discarding the answers after it loses nothing (what the earlier GPU runs saw)."""
    for seed in range(300):
        done, bad = run_queue(40, 8, 2, seed, take_late=False, in_order=True)
        assert bad == 0 and sorted(done) == list(range(40))
