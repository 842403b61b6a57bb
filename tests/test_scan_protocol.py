"""CPU model of the hand-off protocol inside kla_scan_kernel
(bayesian_filtering_linear_gb300/csrc/kla_scan_kernel.cuh).

The scan block has producer warps (stage raw tiles with cp.async, build
coefficients, store y) and scanning warps, synchronised only by named
barriers: FULL[b] (producers arrive, scanners wait), EMPTY[b] (scanners
arrive, producers wait), both counting every thread of the block, and one
producer-only barrier. This file restates each role's sequence of barrier
operations and shared-memory accesses in the kernel's order and checks, for
every tile count and many random interleavings, that

* every warp finishes (no deadlock: each wait's barrier generation completes);
* every pair of conflicting accesses to a shared buffer from different warps
  is ordered by the barriers (vector-clock happens-before), counting a
  cp.async copy as a write from its issue until the wait that completes it.

Planted protocol mistakes (a dropped barrier, a buffer reused one step early)
must each be caught, so the checker itself is pinned.

The same checks cover the kernel's MODE 4, whose producers copy each tile's
per-row coefficients (the coefficient pass's output) into coef[b] with
cp.async once the scan has released that buffer, instead of building them.
"""
import random

import pytest

FULL = ("FULL0", "FULL1")
EMPTY = ("EMPTY0", "EMPTY1")
PROD = "PROD"


def producer_ops(ntiles, p, mutant=None):
    """One producer warp `p`. Accesses: ('w'|'r', buffer, part) with part =
    this warp's share, or None for the whole buffer."""
    ops = []

    def stage(n):  # cp.async of tile n into raw[n % 2]: in flight until a wait
        ops.append(("stage", f"raw{n % 2}", p))

    def build(m):
        b = m % 2
        ops.append(("acc", [("r", f"raw{b}", None), ("r", f"kprev{b}", None),
                            ("w", f"coef{b}", p), ("w", f"pj{b}", p), ("w", f"kprev{b ^ 1}", p)]))

    stage(0)
    ops.append(("commit",))
    if ntiles > 1:
        stage(1)
    ops.append(("commit",))  # possibly empty group
    ops.append(("wait", 1))  # all but the newest group landed: tile 0
    ops.append(("sync", PROD))
    build(0)
    ops.append(("arrive", FULL[0]))
    if ntiles > 1:
        ops.append(("wait", 0))
        if mutant != "no_producer_barrier":
            ops.append(("sync", PROD))
        build(1)
        ops.append(("arrive", FULL[1]))
    for n in range(ntiles):
        b = n % 2
        if n + 2 < ntiles and mutant != "stage_after_empty":
            stage(n + 2)
        if mutant != "stage_after_empty":
            ops.append(("commit",))
        if mutant != "no_empty_wait":
            ops.append(("sync", EMPTY[b]))
        if n + 2 < ntiles and mutant == "stage_after_empty":
            stage(n + 2)
        if mutant == "stage_after_empty":
            ops.append(("commit",))
        ops.append(("acc", [("r", f"ypart{b}", None), ("w", "y", p)]))  # store_y(n)
        if n + 2 < ntiles:
            ops.append(("wait", 0))
            ops.append(("sync", PROD))
            build(n + 2)
            ops.append(("arrive", FULL[b]))
    if mutant == "no_empty_wait":
        for n in range(ntiles):  # keep barrier counts balanced
            ops.append(("arrive", EMPTY[n % 2]))
    return ops


def producer_ops_pre(ntiles, p, mutant=None):
    """MODE 4: the producers stage only the per-column inputs (raw[b]) and
    copy the tile's coefficients straight into coef[b]; K of the last token
    (kprev[ntiles % 2]) is written once at the start."""
    ops = []

    def stage_cols(n):
        ops.append(("stage", f"raw{n % 2}", p))

    def fetch(n):  # cp.async of tile n's coefficients into coef[n % 2]
        ops.append(("stage", f"coef{n % 2}", p))

    def cols(m):
        ops.append(("acc", [("r", f"raw{m % 2}", None), ("w", f"pj{m % 2}", p)]))

    ops.append(("acc", [("w", f"kprev{ntiles % 2}", p)]))
    stage_cols(0)
    fetch(0)
    ops.append(("commit",))
    if ntiles > 1:
        stage_cols(1)
        fetch(1)
    ops.append(("commit",))
    ops.append(("wait", 1))
    ops.append(("sync", PROD))
    cols(0)
    ops.append(("arrive", FULL[0]))
    if ntiles > 1:
        ops.append(("wait", 0))
        ops.append(("sync", PROD))
        cols(1)
        ops.append(("arrive", FULL[1]))
    for n in range(ntiles):
        b = n % 2
        if n + 2 < ntiles:
            stage_cols(n + 2)
        ops.append(("commit",))
        if n + 2 < ntiles and mutant == "fetch_before_empty":
            fetch(n + 2)
        ops.append(("sync", EMPTY[b]))
        if n + 2 < ntiles and mutant != "fetch_before_empty":
            fetch(n + 2)
        ops.append(("commit",))
        ops.append(("acc", [("r", f"ypart{b}", None), ("w", "y", p)]))  # store_y(n)
        if n + 2 < ntiles:
            ops.append(("wait", 0))
            ops.append(("sync", PROD))
            cols(n + 2)
            ops.append(("arrive", FULL[b]))
    return ops


def scanner_ops(ntiles, c, mutant=None):
    ops = []
    for n in range(ntiles):
        b = n % 2
        if mutant == "arrive_before_scan":
            ops.append(("sync", FULL[b]))
            ops.append(("arrive", EMPTY[b]))
            ops.append(("acc", [("r", f"coef{b}", None), ("w", f"ypart{b}", c)]))
            continue
        ops.append(("sync", FULL[b]))
        ops.append(("acc", [("r", f"coef{b}", None), ("r", f"pj{b}", None), ("w", f"ypart{b}", c)]))
        ops.append(("arrive", EMPTY[b]))
    ops.append(("acc", [("r", f"kprev{ntiles % 2}", None)]))  # final state reads K of the last token
    return ops


class Race(Exception):
    pass


def run(ntiles, n_prod, n_scan, seed, mutant=None, pre=False):
    """Simulate one interleaving (pre: the MODE 4 producers). Returns True
    when every warp finished; raises Race on an unordered conflicting access."""
    rnd = random.Random(seed)
    progs = [(producer_ops_pre if pre else producer_ops)(ntiles, p, mutant) for p in range(n_prod)]
    progs += [scanner_ops(ntiles, n_prod + c, mutant) for c in range(n_scan)]
    nw = len(progs)
    count = {FULL[0]: nw, FULL[1]: nw, EMPTY[0]: nw, EMPTY[1]: nw, PROD: n_prod}
    clock = [[0] * nw for _ in range(nw)]
    for w in range(nw):
        clock[w][w] = 1
    pc = [0] * nw
    arrivals = {}  # barrier -> (number in, merged clock) of the open generation
    done_gen = {}  # barrier -> completed generations
    released = {}  # (barrier, generation) -> merged clock
    waiting = {}   # warp -> (barrier, generation)
    inflight = {}  # warp -> committed groups, each a list of (buffer, part)
    open_group = {}  # warp -> copies issued since the last commit
    history = {}   # (buffer) -> list of (kind, part, warp, clock)

    def leq(a, b):
        return all(x <= y for x, y in zip(a, b))

    def access(w, kind, buf, part):
        for (k2, part2, w2, c2) in history.get(buf, []):
            if w2 == w or (k2 == "r" and kind == "r"):
                continue
            if part is not None and part2 is not None and part != part2:
                continue  # disjoint shares of the buffer
            if not leq(c2, clock[w]):
                raise Race(f"{kind} of {buf} by warp {w} races {k2} by warp {w2}")
        history.setdefault(buf, []).append((kind, part, w, list(clock[w])))

    def tick(w):
        clock[w][w] += 1

    while True:
        for w in list(waiting):
            bar, g = waiting[w]
            if done_gen.get(bar, 0) > g:
                merged = released[(bar, g)]
                clock[w] = [max(x, y) for x, y in zip(clock[w], merged)]
                del waiting[w]
        runnable = [w for w in range(nw) if pc[w] < len(progs[w]) and w not in waiting]
        if not runnable:
            pending = any(g for w in range(nw) for g in inflight.get(w, [])) or any(open_group.values())
            if pending:
                raise Race("a cp.async copy was never waited for")
            return all(pc[w] == len(progs[w]) for w in range(nw)) and not waiting
        w = rnd.choice(runnable)
        op = progs[w][pc[w]]
        pc[w] += 1
        kind = op[0]
        if kind in ("arrive", "sync"):
            bar = op[1]
            g = done_gen.get(bar, 0)
            n_in, merged = arrivals.get(bar, (0, [0] * nw))
            merged = [max(x, y) for x, y in zip(merged, clock[w])]
            n_in += 1
            if n_in == count[bar]:
                released[(bar, g)] = merged
                done_gen[bar] = g + 1
                arrivals[bar] = (0, [0] * nw)
                if kind == "sync":
                    clock[w] = list(merged)
            else:
                arrivals[bar] = (n_in, merged)
                if kind == "sync":
                    waiting[w] = (bar, g)
            tick(w)
        elif kind == "stage":
            access(w, "w", op[1], op[2])
            open_group.setdefault(w, []).append((op[1], op[2]))
            tick(w)
        elif kind == "commit":
            inflight.setdefault(w, []).append(open_group.pop(w, []))
            tick(w)
        elif kind == "wait":  # every committed group but the newest op[1] has landed
            groups = inflight.get(w, [])
            cut = max(0, len(groups) - op[1])
            for group in groups[:cut]:
                for buf, part in group:  # the copy's bytes land now
                    access(w, "w", buf, part)
            inflight[w] = groups[cut:]
            tick(w)
        else:
            for k2, buf, part in op[1]:
                access(w, k2, buf, part)
            tick(w)


@pytest.mark.parametrize("ntiles", range(1, 8))
@pytest.mark.parametrize("pre", [False, True], ids=["build", "copy"])
def test_protocol_has_no_deadlock_and_no_race(ntiles, pre):
    for seed in range(150):
        assert run(ntiles, n_prod=2, n_scan=3, seed=seed, pre=pre), f"deadlock at {ntiles} tiles, seed {seed}"


def test_copy_mode_fetching_before_the_scan_released_the_buffer_is_caught():
    """The copy of tile n+2's coefficients issued before the EMPTY wait of
    tile n would overwrite coef[b] while the scan still reads it."""
    caught = False
    for seed in range(300):
        try:
            run(5, n_prod=2, n_scan=3, seed=seed, mutant="fetch_before_empty", pre=True)
        except Race:
            caught = True
            break
    assert caught


@pytest.mark.parametrize("mutant", ["no_producer_barrier", "stage_after_empty", "arrive_before_scan",
                                    "no_empty_wait"])
def test_planted_protocol_mistakes_are_caught(mutant):
    caught = False
    for seed in range(300):
        try:
            ok = run(5, n_prod=2, n_scan=3, seed=seed, mutant=mutant)
        except Race:
            caught = True
            break
        if not ok:
            caught = True  # deadlock
            break
    if mutant == "stage_after_empty":
        # Staging tile n+2 after the EMPTY wait is also correct (just later).
        assert not caught
    else:
        assert caught, mutant
