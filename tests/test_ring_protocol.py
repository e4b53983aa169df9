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


# ---------------------------------------------------------------- Q slots, two MMA warps
# With two MMA warps (alternate tiles), Q loads (one per request, in order,
# slot q & 1) are released by a barrier of count 2: each MMA warp waits for
# every load in order (also those of requests it has no tile of); at a tile
# of request q it first commits the release of every load before q (waiting
# for any of them it has not waited for yet), then waits for the loads up to
# q; past its last tile it releases the rest it waited for.  The producer issues load q after the release of load
# q - 2.  Parity waits and counted arrivals are simulated exactly: a wait
# passes when the barrier's current phase parity differs from the awaited
# one; an arrival counts toward whatever phase is current.


def simulate_q(tile_req, seed, coupled=False, lookahead=False):
    """tile_req: request index (0, 1, ...) of each tile, non-decreasing, every
    request present.  Returns 'ok', 'early' (a parity wait passed on a phase
    other than the awaited one), 'miscount' (an arrival counted toward
    another load's phase), 'overwrite' (a load reused a slot whose previous
    request an MMA warp still had tiles of) or 'deadlock'.  A warp reads a
    tile's request once the tile has landed.  With `coupled`, one producer
    walks the tiles in order issuing the Q load of each request it enters
    and the copies of the even tiles, so an even tile lands only after the
    Q loads of the requests before it were issued; otherwise Q loads and
    tiles are issued independently.  With `lookahead`, a warp knows the
    request of its next tile without reading it (it walks the tile
    sequence itself): once its tile of request r is done and its next tile
    belongs to a later request q (or it has none), it releases the loads
    before q (those up to r if it has none), waiting first for any it has
    not waited for."""
    rnd = random.Random(seed)
    n_req = tile_req[-1] + 1
    full_ph = [0, 0]          # completed phases of qfull[slot] (loads landed in the slot)
    empty_ph = [0, 0]         # completed phases of qempty[slot]
    empty_arr = [[], []]      # loads the pending arrivals of qempty[slot] were meant for
    issued = 0                # loads issued by the producer
    in_flight = []            # issued, not landed
    tiles = {w: [i for i in range(len(tile_req)) if i % 2 == w] for w in (0, 1)}
    pos = {0: 0, 1: 0}        # next tile of each warp
    waited = {0: 0, 1: 0}     # loads waited for
    done = {0: 0, 1: 0}       # loads released
    finished = {0: False, 1: False}
    walked = 0                # coupled: tiles the producer's walk has passed (and issued, if even)

    def landed(i):
        return not coupled or i % 2 == 1 or i < walked

    while True:
        acts = []
        if issued < n_req:
            j = issued
            may = not coupled or (walked < len(tile_req) and tile_req[walked] == j)
            if may and (j < 2 or (empty_ph[j & 1] & 1) != ((((j - 2) >> 1) & 1))):
                acts.append(("issue",))
        if coupled and walked < len(tile_req) and tile_req[walked] < issued:
            acts.append(("walk",))
        if in_flight:
            acts.append(("land",))
        for w in (0, 1):
            if finished[w]:
                continue
            if lookahead and pos[w] > 0:
                # releases due after the previous tile: loads before the next tile's request
                upto = tile_req[tiles[w][pos[w]]] if pos[w] < len(tiles[w]) else tile_req[tiles[w][pos[w] - 1]] + 1
                if done[w] < upto:
                    if done[w] < waited[w]:
                        acts.append(("release", w))
                    else:
                        j = waited[w]
                        if (full_ph[j & 1] & 1) != ((j >> 1) & 1):
                            acts.append(("wait", w))
                    continue
            if pos[w] < len(tiles[w]):
                if not landed(tiles[w][pos[w]]):
                    continue
                qi = tile_req[tiles[w][pos[w]]]
                if done[w] < qi and done[w] < waited[w]:
                    acts.append(("release", w))
                elif waited[w] <= qi:
                    j = waited[w]
                    if (full_ph[j & 1] & 1) != ((j >> 1) & 1):   # the parity wait passes (early or not)
                        acts.append(("wait", w))
                else:
                    acts.append(("tile", w))
            else:
                acts.append(("finish", w))
        if not acts:
            return "ok" if issued == n_req and all(finished.values()) else "deadlock"
        a = rnd.choice(acts)
        if a[0] == "issue":
            j = issued
            if j >= 2:
                if empty_ph[j & 1] <= (j - 2) >> 1:
                    return "early"
                # the warps' tiles of request j - 2 must all be done
                for w in (0, 1):
                    if pos[w] < len(tiles[w]) and tile_req[tiles[w][pos[w]]] <= j - 2:
                        return "overwrite"
            issued += 1
            in_flight.append(j)
        elif a[0] == "walk":
            walked += 1
        elif a[0] == "land":
            j = in_flight.pop(0)                  # TMA loads of one slot land in order
            full_ph[j & 1] += 1
        elif a[0] == "wait":
            w = a[1]
            j = waited[w]
            if j >= issued or full_ph[j & 1] <= j >> 1:
                return "early"
            waited[w] += 1
        elif a[0] == "release":
            w = a[1]
            j = done[w]
            empty_arr[j & 1].append(j)
            if any(x != empty_ph[j & 1] * 2 + (j & 1) for x in empty_arr[j & 1]):
                return "miscount"
            if len(empty_arr[j & 1]) == 2:
                empty_ph[j & 1] += 1
                empty_arr[j & 1] = []
            done[w] += 1
        elif a[0] == "tile":
            w = a[1]
            pos[w] += 1
        else:
            w = a[1]
            while done[w] < waited[w]:
                j = done[w]
                empty_arr[j & 1].append(j)
                if any(x != empty_ph[j & 1] * 2 + (j & 1) for x in empty_arr[j & 1]):
                    return "miscount"
                if len(empty_arr[j & 1]) == 2:
                    empty_ph[j & 1] += 1
                    empty_arr[j & 1] = []
                done[w] += 1
            finished[w] = True


def _random_tiles(rnd, n_req):
    reqs = []
    for r in range(n_req):
        reqs += [r] * rnd.choice([1, 1, 2, 3, 5])
    return reqs


@pytest.mark.parametrize("n_req", [1, 2, 3, 7, 20])
def test_two_mma_warps_q_slots_sound_and_live(n_req):
    rnd = random.Random(n_req)
    for case in range(40):
        tiles = _random_tiles(rnd, n_req)
        for seed in range(25):
            assert simulate_q(tiles, seed * 1000 + case) == "ok", (tiles, seed)


@pytest.mark.parametrize("n_req", [1, 2, 3, 7, 20])
def test_two_mma_warps_releasing_by_lookahead_live_with_a_coupled_q_producer(n_req):
    # The warp that loads Q also issues the even tiles (waiting for each Q
    # slot's release in order); the MMA warps release a load as soon as their
    # own tiles are past its request, known from their own walk of the tiles.
    rnd = random.Random(100 + n_req)
    for case in range(40):
        tiles = _random_tiles(rnd, n_req)
        for seed in range(25):
            assert simulate_q(tiles, seed * 1000 + case, coupled=True, lookahead=True) == "ok", (tiles, seed)


def test_q_loads_by_a_tile_producer_can_deadlock_with_two_mma_warps():
    # Why the Q loads get a warp of their own: when the warp that loads Q also
    # issues the even tiles, a Q load waiting for the release of load q - 2
    # holds back the next even tile, and the MMA warp of the even tiles reads
    # that tile's request before it releases load q - 2.  Here request 1 is
    # one odd tile: load 2 waits for the even warp to pass request 0, which
    # it does at tile 2, issued after load 2.
    tiles = [0, 1, 2, 2, 3, 3]
    outcomes = {simulate_q(tiles, seed, coupled=True) for seed in range(300)}
    assert outcomes == {"deadlock"}, outcomes
    outcomes = {simulate_q(tiles, seed) for seed in range(300)}
    assert outcomes == {"ok"}, outcomes


def test_releasing_after_waiting_for_the_current_load_deadlocks():
    # A first form: a warp at a tile of request q waited for every load up
    # to q, then released the loads before q.  Load q needs the release of
    # load q - 2, which that warp gives only after waiting for load q.
    tiles = [0, 0, 0, 0, 0, 1, 2, 3]
    assert simulate_q_wait_then_release(tiles) == "deadlock"


def simulate_q_wait_then_release(tile_req):
    """Deterministic schedule of the first form: warp 1 (odd tiles) runs
    ahead; the producer issues whenever it can; loads land at once."""
    n_req = tile_req[-1] + 1
    empty_arr = [0] * n_req
    issued = 0
    tiles = {w: [tile_req[i] for i in range(len(tile_req)) if i % 2 == w] for w in (0, 1)}
    pos = {0: 0, 1: 0}
    waited = {0: 0, 1: 0}
    progress = True
    while progress:
        progress = False
        while issued < n_req and (issued < 2 or empty_arr[issued - 2] == 2):
            issued += 1
            progress = True
        for w in (1, 0):
            if pos[w] < len(tiles[w]):
                qi = tiles[w][pos[w]]
                if qi < issued:                    # waits for loads up to qi, all landed
                    for j in range(waited[w], qi):
                        empty_arr[j] += 1
                    waited[w] = max(waited[w], qi)
                    pos[w] += 1
                    progress = True
    return "ok" if all(pos[w] == len(tiles[w]) for w in (0, 1)) else "deadlock"


def test_releasing_only_at_a_requests_last_tile_deadlocks_with_two_warps():
    # Why every warp releases every load: with the single warp's rule (release
    # at the request's last tile, here by the warp that has it), a barrier of
    # count 2 never completes for a request one warp never touches.
    def simulate_last_tile_rule(tile_req):
        n_req = tile_req[-1] + 1
        arrivals = [0] * n_req
        for i, r in enumerate(tile_req):
            if i == len(tile_req) - 1 or tile_req[i + 1] != r:
                arrivals[r] += 1
        # the producer needs the release of load j - 2 (two arrivals) to issue load j
        return all(arrivals[j - 2] >= 2 for j in range(2, n_req))
    assert not simulate_last_tile_rule([0, 1, 2, 3, 3])
