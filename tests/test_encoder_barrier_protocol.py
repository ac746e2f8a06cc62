"""Model check of the persistent encoder's named-barrier hand-offs (CPU only).

The encode CTA hands each tile between its roles through hardware named
barriers, one id per image buffer b = i mod 3 (i: the tile's number within
the CTA); `zc_encode.cu` states the protocol beside the barrier ids:

  Parts(b)  the 16 row warps arrive after phase A; the layout warp waits;
  Seg(b)    the layout warp arrives after phase B (which also stages the
            code tables of tile i + 2); the row warps wait after phase A of
            tile i + 1, then run phase D of tile i;
  B(b)      the layout warp arrives after phase B; the store warp waits;
  Img(b)    the row warps arrive after phase D; the store warp waits;
  Free(b)   the store warp arrives once its store has read image b; the row
            warps wait before phase A of tile i + 3.

A named barrier only counts arriving threads: when the count reaches the
expected total the generation completes, releases every thread waiting on
it, and the next arrivals start a new generation.  It cannot tell two
generations' arrivals apart, so a protocol is safe only if no warp can reach
the same id twice before the generation it joined has completed.  This model
runs every warp as a separate actor under random schedules and checks that,
plus freedom from deadlock and the data order the kernel relies on.  Planted
mistakes (in the model, never on a GPU) must fail: among them the early
buffer release of a diagnostic copy of the encoder that hung until its
harness limit.
"""
from __future__ import annotations

import random

import pytest

NB = 3                           # image buffers
ROW_WARPS = 16
PARTS, SEG, B, IMG, FREE = 1, 4, 7, 10, 13
N_ROWS_ROLE = 32 * ROW_WARPS + 32   # kBarThreads: row warps + one role warp
N_B = 64                            # layout + store


class ProtocolError(AssertionError):
    pass


def row_warp(w, n, log, m):
    for i in range(n):
        b = i % NB
        if i >= NB and not m.get("rows_skip_free"):
            yield ("sync", FREE + b, N_ROWS_ROLE)
        log.append(("A", i, w))
        yield ("arrive", PARTS + b, N_ROWS_ROLE)
        if i > 0:
            pb = (i - 1) % NB
            yield ("sync", SEG + pb, N_ROWS_ROLE)
            log.append(("D", i - 1, w))
            yield ("arrive", (IMG if m.get("img_one_id") else IMG + pb), N_ROWS_ROLE)
    if n:
        pb = (n - 1) % NB
        yield ("sync", SEG + pb, N_ROWS_ROLE)
        log.append(("D", n - 1, w))
        yield ("arrive", (IMG if m.get("img_one_id") else IMG + pb), N_ROWS_ROLE)


def layout_warp(n, log, m):
    for i in range(n):
        b = i % NB
        yield ("sync", PARTS + b, N_ROWS_ROLE)
        log.append(("B", i))
        yield ("arrive", SEG + b, N_ROWS_ROLE)
        yield ("arrive", B + b, N_B)


def store_warp(n, log, m):
    for i in range(n):
        b = i % NB
        reuse = i + NB < n
        yield ("sync", B + b, N_B)
        if m.get("free_before_img") and reuse:
            yield ("arrive", FREE + b, N_ROWS_ROLE)
        if not m.get("store_skips_img"):
            yield ("sync", (IMG if m.get("img_one_id") else IMG + b), N_ROWS_ROLE)
        log.append(("S", i))
        if reuse and not m.get("free_before_img"):
            yield ("arrive", FREE + b, N_ROWS_ROLE)


def run(n, seed, m=None, laggard=None):
    """One random schedule of a CTA with n tiles; raises ProtocolError.

    laggard: an actor picked only when nothing else can run, or with
    probability 1/20, so that schedules where one role falls far behind the
    others are explored too."""
    m = m or {}
    rng = random.Random(seed)
    log = []
    actors = {f"row{w}": row_warp(w, n, log, m) for w in range(ROW_WARPS)}
    actors["layout"] = layout_warp(n, log, m)
    actors["store"] = store_warp(n, log, m)
    pending, waiting, done = {}, {}, set()
    bars = {}  # id -> [count, generation, expected, actors arrived in this generation]

    def fetch(a):
        try:
            pending[a] = next(actors[a])
        except StopIteration:
            done.add(a)

    for a in actors:
        fetch(a)
    while len(done) < len(actors):
        runnable = [a for a in actors if a not in done and a not in waiting]
        if not runnable:
            raise ProtocolError(f"deadlock: {sorted(waiting.items())}")
        others = [a for a in runnable if a != laggard]
        a = rng.choice(others) if others and (laggard not in runnable or rng.random() > 0.05) else rng.choice(runnable)
        kind, bid, exp = pending[a]
        bar = bars.setdefault(bid, [0, 0, exp, set()])
        if bar[2] != exp:
            raise ProtocolError(f"barrier {bid} used with counts {bar[2]} and {exp}")
        if a in bar[3]:
            raise ProtocolError(f"barrier {bid}: {a} arrives twice in generation {bar[1]}")
        bar[3].add(a)
        bar[0] += 32
        if kind == "sync":
            waiting[a] = (bid, bar[1])
        if bar[0] == exp:
            gen = bar[1]
            bar[0], bar[1], bar[3] = 0, gen + 1, set()
            for w, (wb, wg) in list(waiting.items()):
                if wb == bid and wg == gen:
                    del waiting[w]
                    fetch(w)
        if kind == "arrive":
            fetch(a)
    for bid, bar in bars.items():
        if bar[0]:
            raise ProtocolError(f"barrier {bid} left with {bar[0]} arrivals of an unfinished generation")
    check_order(n, log)
    return log


def check_order(n, log):
    pos = {e: k for k, e in enumerate(log)}
    for i in range(n):
        for w in range(ROW_WARPS):
            if not pos[("A", i, w)] < pos[("B", i)]:
                raise ProtocolError(f"layout of tile {i} before row warp {w} packed it")
            if not pos[("B", i)] < pos[("D", i, w)]:
                raise ProtocolError(f"row warp {w} placed tile {i} before its layout")
            if not pos[("D", i, w)] < pos[("S", i)]:
                raise ProtocolError(f"tile {i} stored before row warp {w} placed it")
            if i + NB < n and not pos[("S", i)] < pos[("A", i + NB, w)]:
                raise ProtocolError(f"row warp {w} packed tile {i + NB} into an image not yet stored")
            if i >= 2 and not pos[("B", i - 2)] < pos[("A", i, w)]:
                raise ProtocolError(f"row warp {w} packed tile {i} before its code tables were staged")
            if i >= 2 and not pos[("D", i - 2, w)] < pos[("B", i)]:
                raise ProtocolError(f"tables of tile {i + 2} staged over tile {i - 2}'s still in use")


ACTORS = [f"row{w}" for w in range(ROW_WARPS)] + ["layout", "store"]


def sweep(m=None, trials=400):
    rng = random.Random(7)
    for t in range(trials):
        lag = rng.choice(ACTORS) if t % 2 else None
        run(rng.randint(1, 9), 1000 + t, m, lag)


def test_product_protocol_is_safe_under_random_schedules():
    sweep()


def test_single_tile_and_exactly_three_tiles():
    for n in (1, 2, NB, NB + 1):
        for s in range(50):
            run(n, s)


@pytest.mark.parametrize("mutation", ["free_before_img", "store_skips_img", "rows_skip_free", "img_one_id"])
def test_planted_protocol_mistakes_are_caught(mutation):
    # free_before_img is the diagnostic copy that hung: the store warp freed
    # the image before waiting for it, so a row warp's arrival for tile i + 3
    # could land in tile i's generation of Img and complete it early.
    with pytest.raises(ProtocolError):
        sweep({mutation: True}, trials=400)
