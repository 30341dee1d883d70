"""Model checks of the kernels' mbarrier ring protocols, on the CPU.

An mbarrier phase wait is a parity test: `try_wait.parity(p)` succeeds once the
phase with parity p has completed, i.e. while the barrier's completed-phase
count has the other parity.  A waiter that is two or more phases behind the
barrier cannot tell its phase from a later one of the same parity, so a ring
protocol is only safe if no waiter can ever test a stage while the stage is
two phases away from the one it wants.

These tests run the prepare kernel's tile ring (one producer, consumer groups
taking tiles round-robin, stage = n % NST) and the attention kernel's K/V ring
(every tile consumed by both MMA warps) under many random schedules and check,
at every successful parity test, that the completed phase is exactly the one
the waiter asked for.  The prepare check also shows why the kernel keeps NST a
multiple of the number of groups: with a stage shared by two groups the
invariant breaks."""
import random

import pytest


class Barrier:
    """Completed-phase counter with the parity test of mbarrier.try_wait."""

    def __init__(self):
        self.done = 0  # phases completed

    def test(self, parity):
        # the phase with this parity has completed iff the count's parity differs
        return (self.done & 1) != parity


def run_prepare_ring(nst, groups, tiles, seed):
    """One producer, `groups` consumer groups; tile n -> stage n % nst, group n % groups.
    Returns the number of parity tests that passed on the wrong phase."""
    rng = random.Random(seed)
    full = [Barrier() for _ in range(nst)]
    empty = [Barrier() for _ in range(nst)]
    pushed = 0
    nxt = [g for g in range(groups)]           # next tile of each group
    holding = [None] * groups                   # tile a group is processing (stage not yet released)
    landed = []                                  # tiles whose copy is in flight
    bad = 0
    while True:
        actions = []
        if pushed < tiles:
            n = pushed
            if empty[n % nst].test(((n // nst) & 1) ^ 1):
                actions.append(("push", n))
        if landed:
            actions.append(("land", None))
        for g in range(groups):
            if holding[g] is not None:
                actions.append(("release", g))
            elif nxt[g] < tiles:
                actions.append(("wait", g))
        if not actions:
            break
        kind, arg = rng.choice(actions)
        if kind == "push":
            landed.append(arg)
            pushed += 1
        elif kind == "land":
            n = landed.pop(rng.randrange(len(landed)))
            full[n % nst].done += 1
        elif kind == "wait":
            g = arg
            n = nxt[g]
            if full[n % nst].test((n // nst) & 1):
                # the completed phase must be this tile's: phase index n // nst
                if full[n % nst].done - 1 != n // nst:
                    bad += 1
                holding[g] = n
                nxt[g] += groups
        elif kind == "release":
            g = arg
            empty[holding[g] % nst].done += 1
            holding[g] = None
        if bad:
            break
    return bad


@pytest.mark.parametrize("nst,groups", [(2, 2), (4, 2), (6, 2), (6, 3)])
def test_prepare_ring_is_safe_when_stages_are_whole_per_group(nst, groups):
    for seed in range(300):
        assert run_prepare_ring(nst, groups, 60, seed) == 0, (nst, groups, seed)


@pytest.mark.parametrize("nst,groups", [(5, 2), (3, 2), (5, 3)])
def test_prepare_ring_breaks_when_a_stage_is_shared(nst, groups):
    assert any(run_prepare_ring(nst, groups, 60, seed) for seed in range(300))


def run_kv_ring(nst, tiles, seed, waiters=2):
    """Attention K/V ring: a producer fills stage n % nst; each of `waiters`
    MMA warps consumes every tile in order and releases it; the stage's empty
    barrier needs one arrival per waiter.  Returns wrong-phase passes."""
    rng = random.Random(seed)
    full = [Barrier() for _ in range(nst)]
    empty_arr = [0] * nst
    empty = [Barrier() for _ in range(nst)]
    pushed, landed, bad = 0, [], 0
    nxt = [0] * waiters
    holding = [None] * waiters
    while True:
        actions = []
        if pushed < tiles and empty[pushed % nst].test(((pushed // nst) & 1) ^ 1):
            actions.append(("push", None))
        if landed:
            actions.append(("land", None))
        for w in range(waiters):
            if holding[w] is not None:
                actions.append(("release", w))
            elif nxt[w] < tiles:
                actions.append(("wait", w))
        if not actions:
            break
        kind, w = rng.choice(actions)
        if kind == "push":
            landed.append(pushed)
            pushed += 1
        elif kind == "land":
            n = landed.pop(rng.randrange(len(landed)))
            full[n % nst].done += 1
        elif kind == "wait":
            n = nxt[w]
            if full[n % nst].test((n // nst) & 1):
                if full[n % nst].done - 1 != n // nst:
                    bad += 1
                holding[w] = n
                nxt[w] += 1
        elif kind == "release":
            s = holding[w] % nst
            empty_arr[s] += 1
            if empty_arr[s] == waiters:
                empty_arr[s] = 0
                empty[s].done += 1
            holding[w] = None
    return bad, min(nxt)


@pytest.mark.parametrize("nst", [2, 3, 4, 5])
def test_attention_kv_ring_is_safe(nst):
    for seed in range(300):
        bad, done = run_kv_ring(nst, 40, seed)
        assert bad == 0 and done == 40, (nst, seed, bad, done)
