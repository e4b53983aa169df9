"""The K-stage ring protocol of the logits kernel, simulated on the CPU.

Producer warp w issues tiles w, w + NP, ... into stage i % S after waiting
for the stage's release by phase parity.  The MMA takes jobs (C per tile) in
order, each once its tile is in its stage and one of ACC accumulators is
free; two epilogue warpgroups take the jobs alternately, each in order, and
a tile's stage is released once every job of the tile has been taken.  A
parity wait cannot tell the release of use u - 1 from that of use u - 2, so a
producer can pass its wait early.  The kernel picks (stages, producers) by a
rule and asserts it at compile time: stages >= producers, and for one-job
tiles some m >= 1 with stages - m * producers even and >= 0.

Random schedules check that every configuration the rule accepts never
passes a wait early and never deadlocks; that configurations it rejects can
pass early (among them the interleaved-cache fault on the MTP shape: two
stages, three producers); and the same when producer warps other than warp 0
hold their tile until their next tile's copies are issued (stages > NP).
"""
import random

import pytest


def rule(stages: int, producers: int, jobs_per_tile: int) -> bool:
    if stages < producers:
        return False
    if jobs_per_tile > 1:
        return True
    return any((stages - m * producers) % 2 == 0 for m in range(1, stages // producers + 1))


def simulate(S, NP, C, ACC, tiles, seed, hold=False):
    """One random interleaving of the roles; returns 'early', 'deadlock' or 'ok'."""
    rnd = random.Random(seed)
    jobs = tiles * C
    released = [0] * S            # completed phases of each stage's release barrier
    full = [False] * tiles        # the tile is in its stage, ready for the MMA
    mma_next = 0                  # next job the MMA issues
    epi_done = [False] * jobs
    jobs_left = [C] * tiles
    wg_next = [0, 1]              # the two warpgroups take jobs 0, 2, 4 ... and 1, 3, 5 ...
    nxt = list(range(NP))         # next tile of each producer warp
    held = [None] * NP            # issued but not yet marked full (holding warps)
    pending = [None] * NP         # a held tile to finish before the warp's next wait
    while True:
        acts = []
        for w in range(NP):
            if pending[w] is not None:
                acts.append(("finish", w))
            elif nxt[w] < tiles:
                i = nxt[w]
                if (released[i % S] & 1) != (((i // S) & 1) ^ 1):   # the parity wait passes
                    acts.append(("issue", w))
            elif held[w] is not None:
                acts.append(("last", w))
        if mma_next < jobs and full[mma_next // C] and (mma_next < ACC or epi_done[mma_next - ACC]):
            acts.append(("mma", None))
        for g in (0, 1):
            if wg_next[g] < jobs and wg_next[g] < mma_next:
                acts.append(("epi", g))
        if not acts:
            return "ok" if all(epi_done) else "deadlock"
        kind, w = rnd.choice(acts)
        if kind == "issue":
            i = nxt[w]
            if released[i % S] < i // S:          # the previous use of the stage is not released
                return "early"
            nxt[w] += NP
            if hold and w != 0:
                pending[w], held[w] = held[w], i
            else:
                full[i] = True
        elif kind == "finish":
            full[pending[w]] = True
            pending[w] = None
        elif kind == "last":
            full[held[w]] = True
            held[w] = None
        elif kind == "mma":
            mma_next += 1
        else:
            a = wg_next[w]
            epi_done[a] = True
            jobs_left[a // C] -= 1
            if jobs_left[a // C] == 0:
                released[(a // C) % S] += 1
            wg_next[w] += 2


CONFIGS = [(S, NP, C) for S in range(2, 9) for NP in (2, 3) for C in (1, 2, 3)]
SEEDS = range(60)


@pytest.mark.parametrize("ACC", [2, 4, 8])
@pytest.mark.parametrize("S,NP,C", [c for c in CONFIGS if rule(*c)])
def test_accepted_rings_never_pass_early_nor_deadlock(S, NP, C, ACC):
    for seed in SEEDS:
        assert simulate(S, NP, C, ACC, tiles=36, seed=seed) == "ok", seed


@pytest.mark.parametrize("S,NP,C", [(2, 3, 2), (2, 3, 1), (4, 3, 1), (5, 2, 1)])
def test_rejected_rings_can_pass_early(S, NP, C):
    # The rule does not count on the accumulators' back-pressure (with two,
    # the MMA of a tile also waits for the epilogue two jobs back, which
    # happens to order 5 stages / 2 producers); with eight it is gone.
    assert not rule(S, NP, C)
    outcomes = {simulate(S, NP, C, 8, tiles=36, seed=seed) for seed in range(600)}
    assert "early" in outcomes, outcomes


@pytest.mark.parametrize("ACC", [2, 8])
@pytest.mark.parametrize("S,NP,C", [c for c in CONFIGS if rule(*c) and c[0] > c[1]])
def test_holding_producers_stay_sound_and_live(S, NP, C, ACC):
    for seed in SEEDS:
        assert simulate(S, NP, C, ACC, tiles=36, seed=seed, hold=True) == "ok", seed


def test_holding_with_as_many_stages_as_producers_can_deadlock():
    # Why holding needs stages > producers: with S = NP a warp holding tile i
    # waits for the release of tile i + NP - S = i, its own unfinished tile.
    outcomes = {simulate(3, 3, 1, 4, tiles=36, seed=seed, hold=True) for seed in range(200)}
    assert "deadlock" in outcomes, outcomes
