"""Model check of the reduce kernel's rank-order fold hand-offs (CPU only).

In a block of the fused decompress + reduce, warp p decodes peer p's rows and
folds them into an fp32 row accumulator in rank order.  `zc_decode.cu`
states the protocol beside `fold_barrier`: the accumulator rows form a ring
of two buffers (row r uses buffer j = r mod 2); for row r, warp p > 0 waits
on the named barrier of (pair p - 1, buffer j), which warp p - 1 arrives on
once it has added its row; the last warp rounds and stores, then arrives on
buffer j's mbarrier, and warp 0 waits for that mbarrier's phase (parity
(use - 1) mod 2, use = r div 2) before it writes row r into the buffer.

A named barrier only counts arriving threads, so the protocol is safe only
if a warp never arrives twice on an id before the generation it joined has
completed.  An mbarrier wait on parity P returns once the number of
completed phases has the other parity, so a wait that fell two phases
behind would pass wrongly.  The model runs every warp as its own actor under
random and one-laggard schedules with both semantics and checks freedom from
deadlock, single arrivals per generation and the fold's order: warp p adds
row r after warp p - 1 did, and warp 0 overwrites a buffer only after the
last warp has read it.  Planted mistakes must fail.
"""
from __future__ import annotations

import random

import pytest

BUFS = 2


class ProtocolError(AssertionError):
    pass


def fold_warp(p, k, rows, log, m):
    for r in range(rows):
        j, use = r % BUFS, r // BUFS
        if p > 0:
            yield ("sync", ("pair", p - 1) if m.get("one_id_per_pair") else ("pair", p - 1, j))
        elif k > 1 and use > 0 and not m.get("no_back_edge"):
            parity = (use & 1) if m.get("wrong_parity") else ((use - 1) & 1)
            yield ("mwait", ("done", j), parity)
        log.append(("fold", r, p))
        if p + 1 < k:
            yield ("arrive", ("pair", p) if m.get("one_id_per_pair") else ("pair", p, j))
        else:
            yield ("marrive", ("done", j))


def run(k, rows, seed, m=None, laggard=None):
    m = m or {}
    rng = random.Random(seed)
    log = []
    actors = {p: fold_warp(p, k, rows, log, m) for p in range(k)}
    pending, waiting, done = {}, {}, set()
    named = {}   # id -> [threads arrived, generation, warps arrived]  (64 threads: two warps)
    phases = {}  # mbarrier id -> completed phases (one warp of 32 arrivals completes a phase)

    def fetch(a):
        try:
            pending[a] = next(actors[a])
        except StopIteration:
            done.add(a)

    def phase_done(bid, parity):
        return (phases.get(bid, 0) & 1) != parity

    for a in actors:
        fetch(a)
    while len(done) < len(actors):
        for w, (kind, bid, arg) in list(waiting.items()):
            if kind == "mwait" and phase_done(bid, arg):
                del waiting[w]
                fetch(w)
        runnable = [a for a in actors if a not in done and a not in waiting]
        if not runnable:
            raise ProtocolError(f"deadlock: {sorted(map(str, waiting.items()))}")
        others = [a for a in runnable if a != laggard]
        a = rng.choice(others) if others and (laggard not in runnable or rng.random() > 0.05) else rng.choice(runnable)
        op = pending[a]
        kind, bid = op[0], op[1]
        if kind in ("sync", "arrive"):
            bar = named.setdefault(bid, [0, 0, set()])
            if a in bar[2]:
                raise ProtocolError(f"barrier {bid}: warp {a} arrives twice in generation {bar[1]}")
            bar[2].add(a)
            bar[0] += 32
            if kind == "sync":
                waiting[a] = ("sync", bid, bar[1])
            if bar[0] == 64:
                gen = bar[1]
                bar[0], bar[1], bar[2] = 0, gen + 1, set()
                for w, (wk, wb, wg) in list(waiting.items()):
                    if wk == "sync" and wb == bid and wg == gen:
                        del waiting[w]
                        fetch(w)
            if kind == "arrive":
                fetch(a)
        elif kind == "marrive":
            phases[bid] = phases.get(bid, 0) + 1
            fetch(a)
        else:  # mwait
            if phase_done(bid, op[2]):
                fetch(a)
            else:
                waiting[a] = ("mwait", bid, op[2])
    for bid, bar in named.items():
        if bar[0]:
            raise ProtocolError(f"barrier {bid} left with arrivals of an unfinished generation")
    pos = {e: i for i, e in enumerate(log)}
    for r in range(rows):
        for p in range(1, k):
            if not pos[("fold", r, p - 1)] < pos[("fold", r, p)]:
                raise ProtocolError(f"warp {p} folded row {r} before warp {p - 1}")
        if k > 1 and r + BUFS < rows and not pos[("fold", r, k - 1)] < pos[("fold", r + BUFS, 0)]:
            raise ProtocolError(f"warp 0 overwrote row {r}'s buffer before the last warp read it")
    return log


def sweep(m=None, trials=300):
    rng = random.Random(11)
    for t in range(trials):
        k = rng.randint(1, 8)
        lag = rng.randrange(k) if t % 2 else None
        run(k, rng.randint(1, 9), 500 + t, m, lag)


def test_fold_protocol_is_safe_under_random_schedules():
    sweep()


def test_single_peer_and_single_row():
    for k, rows in ((1, 1), (1, 5), (2, 1), (8, 1), (8, 2), (8, 3)):
        for s in range(40):
            run(k, rows, s)


@pytest.mark.parametrize("mutation", ["one_id_per_pair", "no_back_edge", "wrong_parity"])
def test_planted_fold_mistakes_are_caught(mutation):
    # one_id_per_pair: warp p - 1 can arrive for row r + 1 before warp p has
    # waited for row r; no_back_edge and wrong_parity: warp 0 refills a
    # buffer the last warp has not read yet
    with pytest.raises(ProtocolError):
        sweep({mutation: True}, trials=300)
