"""A model, on the CPU, of the work schedule of the persistent single-kernel
call (k_call.cu), checking that every schedule finishes.

Items come in rounds: round r holds the push of tile r from every sender to
every owner, the reduce of tile r - D of every owner and (unfused) the gather
of tile r - 2D; slots whose tile is out of range are empty and skipped.
Blocks take tickets from one counter, the next one fetched ahead.  A reduce
item needs its tile's P - 1 pushes, a gather item its tile's reduce.  A block
computes one item while it holds the next: if the next item's inputs are
ready it starts it at once, otherwise it first signals the current item and
only then waits.  Blocks advance in random interleavings; a state where no
block can move is a deadlock.  The same model with the wait placed before the
signal (the order to avoid) deadlocks, as a control.
"""
import random

import pytest


def _items(P, tiles, fused, D):
    S = P * (P - 1) + P + (0 if fused else P)
    rounds = tiles + (D if fused else 2 * D)
    out = []
    for r in range(rounds):
        for slot in range(S):
            if slot < P * (P - 1):
                p, oi = divmod(slot, P - 1)
                o = oi + (oi >= p)
                out.append(("push", o, r) if r < tiles else None)
            elif slot < P * (P - 1) + P:
                k = r - D
                out.append(("reduce", slot - P * (P - 1), k) if 0 <= k < tiles else None)
            else:
                k = r - 2 * D
                out.append(("gather", slot - P * (P - 1) - P, k) if 0 <= k < tiles else None)
    return out


def _run(P, tiles, fused, D, nblocks, seed, wait_before_signal=False):
    """True when every item completes, False on a deadlock."""
    rng = random.Random(seed)
    items = _items(P, tiles, fused, D)
    total = len(items)
    counter = [0]
    pushes, reduced, done = {}, {}, set()

    def ready(t):
        kind, o, k = items[t]
        if kind == "push" or (kind == "reduce" and P == 1):
            return True
        if kind == "reduce":
            return pushes.get((o, k), 0) == P - 1
        return reduced.get((o, k), 0) == 1

    def consume(t):
        kind, o, k = items[t]
        if kind == "reduce" and P > 1:
            pushes[(o, k)] = 0
        elif kind == "gather":
            reduced[(o, k)] = 0

    def signal(t):
        kind, o, k = items[t]
        if kind == "push":
            pushes[(o, k)] = pushes.get((o, k), 0) + 1
        elif kind == "reduce" and not fused:
            reduced[(o, k)] = 1
        done.add(t)

    def fetch():
        counter[0] += 1
        return counter[0] - 1

    def take(pre):
        t = pre
        while t < total and items[t] is None:
            t = fetch()
        return (None, total) if t >= total else (t, fetch())

    # states: start | first t pre | run cur pre | next-pending t pre | stuck cur t pre | end
    blocks = [("start",)] * nblocks
    while any(b[0] != "end" for b in blocks):
        movable = [i for i, b in enumerate(blocks)
                   if b[0] in ("start", "run")
                   or (b[0] in ("first", "pending") and ready(b[1]))
                   or (b[0] == "stuck" and ready(b[2]))]
        if not movable:
            return False
        i = rng.choice(movable)
        b = blocks[i]
        if b[0] == "start":
            t, pre = take(fetch())
            blocks[i] = ("end",) if t is None else ("first", t, pre)
        elif b[0] in ("first", "pending"):
            consume(b[1])
            blocks[i] = ("run", b[1], b[2])
        elif b[0] == "stuck":
            consume(b[2])
            signal(b[1])
            blocks[i] = ("run", b[2], b[3])
        else:
            cur, pre = b[1], b[2]
            nxt, pre = take(pre)
            if nxt is not None and not ready(nxt) and wait_before_signal:
                blocks[i] = ("stuck", cur, nxt, pre)
                continue
            pend = nxt is not None and not ready(nxt)
            if nxt is not None and not pend:
                consume(nxt)
            signal(cur)
            blocks[i] = ("end",) if nxt is None else (("pending" if pend else "run"), nxt, pre)
    assert len(done) == sum(1 for x in items if x is not None)
    assert not any(pushes.values()) and not any(reduced.values())   # words back at zero
    return True


def test_every_schedule_finishes():
    for seed in range(1500):
        r = random.Random(seed)
        P = r.choice([1, 2, 3, 4, 8])
        tiles = r.choice([1, 2, 3, 5, 9])
        fused = r.choice([False, True])
        D = min(r.choice([0, 1, 2, 4]), tiles)
        nblocks = r.choice([1, 2, 3, 5, 9, 17])
        assert _run(P, tiles, fused, D, nblocks, seed), (P, tiles, fused, D, nblocks, seed)


@pytest.mark.parametrize("fused", [True, False])
def test_waiting_before_signalling_deadlocks(fused):
    """The control: with two ranks the last push of a tile (rank 1 to owner 0)
    is an input of the first reduce, which comes next; one block that waited
    for that reduce's inputs before signalling the push would block on
    itself."""
    assert not _run(2, 1, fused, 0, 1, 0, wait_before_signal=True)
    assert _run(2, 1, fused, 0, 1, 0)
