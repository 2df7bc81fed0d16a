"""A model, on the CPU, of the work schedule of the persistent single-kernel
call (k_call.cu), checking that every schedule finishes.

Items come in rounds: round r holds the push of tile r from every sender to
every owner, the reduce of tile r - D of every owner and (unfused) the gather
of tile r - 2D; slots whose tile is out of range are empty and skipped.
Blocks take tickets from one counter, the next one fetched ahead.  A reduce
item needs its tile's P - 1 pushes, a gather item its tile's reduce.  A block
holds as many items as its ring has stages (two or three): if the next item's
inputs are ready it issues it at once, otherwise it first signals every item
it holds and only then waits.  Blocks advance in random interleavings; a state
where no block can move is a deadlock.  The same model with the wait placed before the
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


def _run(P, tiles, fused, D, nblocks, seed, stages=2, wait_before_signal=False):
    """True when every item completes, False on a deadlock.  A block holds up
    to `stages` items issued into its ring and not yet signalled; to issue one
    more into a full ring it first lets the oldest finish (signalled at the
    latest just before the block issues or waits)."""
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

    # A block: its state ("start", "run": may take its next ticket, "pending":
    # waits for the inputs of `nxt` holding nothing unsignalled, "stuck": waits
    # for them holding `held` unsignalled, "end"), the tickets in its ring
    # (oldest first), the next ticket it will use, and the one it waits for.
    blocks = [dict(s="start", held=[], pre=None, nxt=None) for _ in range(nblocks)]
    while any(b["s"] != "end" for b in blocks):
        movable = [i for i, b in enumerate(blocks)
                   if b["s"] in ("start", "run")
                   or (b["s"] in ("pending", "stuck") and ready(b["nxt"]))]
        if not movable:
            return False
        b = blocks[rng.choice(movable)]
        if b["s"] == "start":
            b["pre"], b["s"] = fetch(), "run"
        elif b["s"] in ("pending", "stuck"):
            consume(b["nxt"])
            for t in b["held"]:
                signal(t)
            b["held"], b["nxt"], b["s"] = [b["nxt"]], None, "run"
        else:
            freed = b["held"].pop(0) if len(b["held"]) == stages else None
            nxt, b["pre"] = take(b["pre"])
            if nxt is None:
                for t in ([] if freed is None else [freed]) + b["held"]:
                    signal(t)
                b["held"], b["s"] = [], "end"
            elif ready(nxt):
                consume(nxt)
                if freed is not None:
                    signal(freed)
                b["held"].append(nxt)
            else:
                if freed is not None:
                    b["held"].insert(0, freed)
                if not wait_before_signal:
                    for t in b["held"]:
                        signal(t)
                    b["held"] = []
                b["nxt"], b["s"] = nxt, ("stuck" if wait_before_signal else "pending")
    assert len(done) == sum(1 for x in items if x is not None)
    assert not any(pushes.values()) and not any(reduced.values())   # words back at zero
    return True


@pytest.mark.parametrize("stages", [2, 3, 4])
def test_every_schedule_finishes(stages):
    for seed in range(1500):
        r = random.Random(seed)
        P = r.choice([1, 2, 3, 4, 8])
        tiles = r.choice([1, 2, 3, 5, 9])
        fused = r.choice([False, True])
        D = min(r.choice([0, 1, 2, 4]), tiles)
        nblocks = r.choice([1, 2, 3, 5, 9, 17])
        assert _run(P, tiles, fused, D, nblocks, seed, stages), \
            (P, tiles, fused, D, nblocks, seed, stages)


@pytest.mark.parametrize("stages", [2, 3])
@pytest.mark.parametrize("fused", [True, False])
def test_waiting_before_signalling_deadlocks(fused, stages):
    """The control: with two ranks the last push of a tile (rank 1 to owner 0)
    is an input of the first reduce, which comes next; one block that waited
    for that reduce's inputs before signalling the push would block on
    itself."""
    assert not _run(2, 1, fused, 0, 1, 0, stages, wait_before_signal=True)
    assert _run(2, 1, fused, 0, 1, 0, stages)
