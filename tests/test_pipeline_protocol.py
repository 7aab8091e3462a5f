"""Interleaving model of the pipeline barriers of the two tensor-core kernels (host only, no GPU).

The small-M kernel (nf4_narrow.cuh) and the GEMM-form kernel (nf4_stream.cuh) coordinate their warp
roles with mbarriers that are waited on by phase parity.  A parity wait is correct only while the
barrier is at most one phase from the awaited one: a phase behind, the wait passes at once (a slot is
overwritten or read too early); a phase ahead, it blocks until the next phase (a hang).

Each role runs here as a generator over the kernels' ring indices, barrier counts and release rules.
A seeded scheduler interleaves the roles (each at its own random speed) with copies that land in any
order and MMA commits that complete in issue order per MMA warp, the two MMA warps of the small-M
kernel independently.  At every wait the model asserts the one-phase window; at every fill, A-tile
write and MMA it asserts that the slot holds what the kernel expects; and every run must end (no
deadlock).  The rules of an earlier version of the kernels (a dequant set waiting only for the fills
of its own stages, one release barrier per A slot, no pass over a tile's remaining fills before its
epilogue) are checked to fail, so the model tells a broken protocol from a sound one.
"""
from __future__ import annotations

import random

import pytest


class Violation(Exception):
    pass


class Barrier:
    """An mbarrier: `count` arrivals complete a phase; `phase` counts completed phases."""

    def __init__(self, name: str, count: int):
        self.name, self.count, self.pending, self.phase = name, count, 0, 0

    def arrive(self, n: int = 1) -> None:
        self.pending += n
        if self.pending > self.count:
            raise Violation(f"{self.name}: more arrivals than its count")
        if self.pending == self.count:
            self.pending = 0
            self.phase += 1


def interleave(actors, names, copies, commit_queues, rng, lag):
    """Run the roles to the end.  An actor yields (barrier, phase) for each parity wait.

    copies: list of callables (a copy landing; any order).  commit_queues: lists of callables, each
    completed from its head (the commits of one MMA warp, in issue order)."""
    cur = [None] * len(actors)
    alive = [True] * len(actors)

    def step(i):
        try:
            cur[i] = next(actors[i])
        except StopIteration:
            alive[i] = False

    for i in range(len(actors)):
        step(i)
    speed = [rng.random() ** 2 + 0.02 for _ in actors]
    for _ in range(5_000_000):
        ready = []
        for i, a in enumerate(alive):
            if not a:
                continue
            bar, phase = cur[i]
            passes = (bar.phase & 1) != (phase & 1)  # the hardware's parity test
            if passes and bar.phase != phase + 1:
                raise Violation(f"{names[i]}: wait for phase {phase} of {bar.name} passes at {bar.phase}")
            if not passes and bar.phase != phase:
                raise Violation(f"{names[i]}: wait for phase {phase} of {bar.name} blocks at {bar.phase}")
            if passes:
                ready.append(i)
        events = [(lag, ("copy", k)) for k in range(len(copies))]
        events += [(lag, ("commit", k)) for k, q in enumerate(commit_queues) if q]
        choices = [(speed[i], ("run", i)) for i in ready] + events
        if not choices:
            if any(alive):
                stuck = ", ".join(f"{names[i]}@{cur[i][0].name}/{cur[i][1]}" for i in range(len(actors)) if alive[i])
                raise Violation("deadlock: " + stuck)
            return
        x = rng.random() * sum(w for w, _ in choices)
        for w, (kind, k) in choices:
            x -= w
            if x <= 0:
                break
        if kind == "run":
            step(k)
        elif kind == "copy":
            copies.pop(k)()
        else:
            commit_queues[k].pop(0)()
    raise Violation("no end")


# --------------------------------------------------------------------------------------------------
# small-M kernel: 4 codes load stages (two pipeline stages each), 4 A and x slots, two MMA warps on
# alternate stages, 3 dequant sets of 4 warps (a set takes every third stage), one epilogue set per tile


def small_m(tiles, rng, lag, current=True):
    NA, NL, KS = 4, 4, 3
    KR = NA * KS if current else NA          # release barriers: stage q -> q mod KR
    info, q0, l0 = [], 0, 0
    for nst in tiles:
        info.append((q0, nst, l0))
        q0, l0 = q0 + nst, l0 + (nst + 1) // 2
    Q, LT = q0, l0
    readers = {}
    for (tq0, nst, tl0) in info:
        for kb2 in range(nst):
            readers[tl0 + kb2 // 2] = readers.get(tl0 + kb2 // 2, 0) + 1
    lfull = [Barrier(f"lfull{i}", 1) for i in range(NL)]
    lempty = [Barrier(f"lempty{i}", 4 * KS if current else 8) for i in range(NL)]
    xfull = [Barrier(f"xfull{i}", 1) for i in range(NA)]
    afull = [Barrier(f"afull{i}", 4) for i in range(NA)]
    rel = [Barrier(f"rel{i}", 1) for i in range(KR)]
    dfull = [Barrier(f"dfull{i}", 2) for i in range(KS)]
    dfree = Barrier("dfree", 4)
    codes, xs, a_tiles = [None] * NL, [None] * NA, [[None] * 4 for _ in range(NA)]
    code_reads = {}
    mma_done = set()
    copies, commits = [], [[], []]

    def rel_wait(q):  # the wait for stage q - NA's MMAs before A (or x) slot q mod NA is rewritten
        if current:
            return rel[(q - NA) % KR], (q - NA) // KR
        return rel[q % NA], q // NA - 1

    def codes_producer():
        for L in range(LT):
            if L >= NL:
                yield lempty[L % NL], L // NL - 1
                if code_reads.get(L - NL, 0) != 4 * readers[L - NL]:
                    raise Violation(f"codes load stage {L} refills the slot of {L - NL} before its reads")
            codes[L % NL] = None

            def land(L=L):
                codes[L % NL] = L
                lfull[L % NL].arrive()
            copies.append(land)

    def x_producer():
        for q in range(Q):
            if q >= NA:
                yield rel_wait(q)
                if q - NA not in mma_done:
                    raise Violation(f"x of stage {q} overwrites stage {q - NA} before its MMAs")
            xs[q % NA] = None

            def land(q=q):
                xs[q % NA] = q
                xfull[q % NA].arrive()
            copies.append(land)

    def mma_issuer(e):
        for j, (tq0, nst, _) in enumerate(info):
            if j > 0:
                yield dfree, j - 1
            for q in range(tq0, tq0 + nst):
                if q % 2 != e:
                    continue
                yield xfull[q % NA], q // NA
                yield afull[q % NA], q // NA
                if xs[q % NA] != q or any(a != q for a in a_tiles[q % NA]):
                    raise Violation(f"MMAs of stage {q} read another stage's operands")

                def done(q=q):
                    mma_done.add(q)
                    rel[q % KR].arrive()
                commits[e].append(done)
            commits[e].append(lambda j=j: dfull[j % KS].arrive())

    def dequant_warp(s, w):
        lnext = 0
        for j, (tq0, nst, tl0) in enumerate(info):
            for kb2 in range(nst):
                gq = tq0 + kb2
                if gq % KS != s:
                    continue
                L = tl0 + kb2 // 2
                yield lfull[L % NL], L // NL
                if current:  # pass the load stages of the other sets' stages
                    while lnext < L:
                        yield lfull[lnext % NL], lnext // NL
                        lempty[lnext % NL].arrive()
                        lnext += 1
                if gq >= NA:
                    yield rel_wait(gq)
                if codes[L % NL] != L:
                    raise Violation(f"stage {gq} reads codes slot {L % NL} holding {codes[L % NL]}, not {L}")
                if gq >= NA and gq - NA not in mma_done:
                    raise Violation(f"A tile of stage {gq} overwrites stage {gq - NA} before its MMAs")
                a_tiles[gq % NA][w] = gq
                code_reads[L] = code_reads.get(L, 0) + 1
                afull[gq % NA].arrive()
                if current:
                    lempty[L % NL].arrive()
                    lnext = L + 1
                else:  # weighted: two stages read a load stage, or one at weight 2
                    lempty[L % NL].arrive(1 if nst - 2 * (kb2 // 2) >= 2 else 2)
            if j % KS == s:
                yield dfull[s], j // KS
                if any(q not in mma_done for q in range(tq0, tq0 + nst)):
                    raise Violation(f"epilogue of tile {j} before its MMAs")
                dfree.arrive()
        if current:
            while lnext < LT:
                yield lfull[lnext % NL], lnext // NL
                lempty[lnext % NL].arrive()
                lnext += 1

    actors = [codes_producer(), x_producer(), mma_issuer(0), mma_issuer(1)]
    actors += [dequant_warp(s, w) for s in range(KS) for w in range(4)]
    names = ["codes", "x", "mma0", "mma1"] + [f"set{s}.warp{w}" for s in range(KS) for w in range(4)]
    interleave(actors, names, copies, commits, rng, lag)
    if len(mma_done) != Q:
        raise Violation("the run ended before every stage's MMAs completed")


# --------------------------------------------------------------------------------------------------
# GEMM-form kernel: codes load stages of two pipeline stages, scale tiles of four, x per 64-k
# sub-tile (two per stage), NA A slots, one MMA warp, 4 dequant sets of 4 warps (every fourth stage),
# and every set in every tile's epilogue


def wide(T, tiles, rng, lag, current=True, pass_before_epilogue=True):
    KS = 4
    NA = {64: 6, 128: 6, 256: 4}[T]
    NX = {64: 8, 128: 6, 256: 4}[T]
    NL = 4 if T == 64 else 3
    NSS = 2 if T == 256 else 3
    NR = 2 * NA if current else NA
    info, q0, l0, s0 = [], 0, 0, 0
    for nst in tiles:
        nload, nscale = (2 * nst + 3) // 4, (2 * nst + 7) // 8
        info.append((q0, nst, l0, nload, s0, nscale))
        q0, l0, s0 = q0 + nst, l0 + nload, s0 + nscale
    LT, ST = l0, s0
    readers_l, readers_s = {}, {}
    for (tq0, nst, tl0, _, ts0, _) in info:
        for kb2 in range(nst):
            readers_l[tl0 + kb2 // 2] = readers_l.get(tl0 + kb2 // 2, 0) + 1
            readers_s[ts0 + kb2 // 4] = readers_s.get(ts0 + kb2 // 4, 0) + 1
    lfull = [Barrier(f"lfull{i}", 1) for i in range(NL)]
    lempty = [Barrier(f"lempty{i}", 16 if current else 8) for i in range(NL)]
    sfull = [Barrier(f"sfull{i}", 1) for i in range(NSS)]
    sempty = [Barrier(f"sempty{i}", 16 if current else 48) for i in range(NSS)]
    xfull = [Barrier(f"xfull{i}", 1) for i in range(NX)]
    xempty = [Barrier(f"xempty{i}", 1) for i in range(NX)]
    afull = [Barrier(f"afull{i}", 4) for i in range(NA)]
    arel = [Barrier(f"arel{i}", 1) for i in range(NR)]
    dfull = [Barrier(f"dfull{i}", 1) for i in range(KS)]
    dfree = Barrier("dfree", 16)
    codes, scales, xs = [None] * NL, [None] * NSS, [None] * NX
    a_tiles = [[None] * 4 for _ in range(NA)]
    code_reads, scale_reads = {}, {}
    mma_done, x_done = set(), set()
    copies, commits = [], [[]]

    def producer():
        lq = sq = 0
        for (tq0, nst, *_) in info:
            for kb in range(2 * nst):
                if kb % 4 == 0:
                    L = lq
                    if L >= NL:
                        yield lempty[L % NL], L // NL - 1
                        if code_reads.get(L - NL, 0) != 4 * readers_l[L - NL]:
                            raise Violation(f"codes load stage {L} refills before its slot was read")
                    codes[L % NL] = None

                    def land(L=L):
                        codes[L % NL] = L
                        lfull[L % NL].arrive()
                    copies.append(land)
                    lq += 1
                if kb % 8 == 0:
                    S = sq
                    if S >= NSS:
                        yield sempty[S % NSS], S // NSS - 1
                        if scale_reads.get(S - NSS, 0) != 4 * readers_s[S - NSS]:
                            raise Violation(f"scale tile {S} refills before its slot was read")
                    scales[S % NSS] = None

                    def land(S=S):
                        scales[S % NSS] = S
                        sfull[S % NSS].arrive()
                    copies.append(land)
                    sq += 1

    def x_producer():
        k = 0
        for (tq0, nst, *_) in info:
            for _ in range(2 * nst):
                if k >= NX:
                    yield xempty[k % NX], k // NX - 1
                    if k - NX not in x_done:
                        raise Violation(f"x sub-tile {k} overwrites one not yet read")
                xs[k % NX] = None

                def land(k=k):
                    xs[k % NX] = k
                    xfull[k % NX].arrive()
                copies.append(land)
                k += 1

    def mma_issuer():
        k = 0
        for j, (tq0, nst, *_) in enumerate(info):
            if j > 0:
                yield dfree, j - 1
            for q in range(tq0, tq0 + nst):
                yield afull[q % NA], q // NA
                if any(a != q for a in a_tiles[q % NA]):
                    raise Violation(f"MMAs of stage {q} read another stage's A tile")
                for _ in range(2):
                    yield xfull[k % NX], k // NX
                    if xs[k % NX] != k:
                        raise Violation(f"MMA reads x slot {k % NX} holding {xs[k % NX]}")

                    def xd(k=k):
                        x_done.add(k)
                        xempty[k % NX].arrive()
                    commits[0].append(xd)
                    k += 1

                def done(q=q):
                    mma_done.add(q)
                    arel[q % NR].arrive()
                commits[0].append(done)
            commits[0].append(lambda j=j: dfull[j % KS].arrive())

    def dequant_warp(s, w):
        lnext = snext = 0

        def pass_fills(lend, send):
            nonlocal lnext, snext
            while snext < send:
                yield sfull[snext % NSS], snext // NSS
                sempty[snext % NSS].arrive()
                snext += 1
            while lnext < lend:
                yield lfull[lnext % NL], lnext // NL
                lempty[lnext % NL].arrive()
                lnext += 1

        for j, (tq0, nst, tl0, nload, ts0, nscale) in enumerate(info):
            for kb2 in range((s - tq0 % KS) % KS, nst, KS):
                gq, L, S = tq0 + kb2, tl0 + kb2 // 2, ts0 + kb2 // 4
                if current:
                    yield from pass_fills(L, S)
                yield sfull[S % NSS], S // NSS
                yield lfull[L % NL], L // NL
                if gq >= NA:
                    yield (arel[(gq - NA) % NR], (gq - NA) // NR) if current else (arel[gq % NA], gq // NA - 1)
                if codes[L % NL] != L or scales[S % NSS] != S:
                    raise Violation(f"stage {gq} reads a codes or scale slot that holds another fill")
                if gq >= NA and gq - NA not in mma_done:
                    raise Violation(f"A tile of stage {gq} overwrites stage {gq - NA} before its MMAs")
                a_tiles[gq % NA][w] = gq
                code_reads[L] = code_reads.get(L, 0) + 1
                scale_reads[S] = scale_reads.get(S, 0) + 1
                afull[gq % NA].arrive()
                if current:
                    lempty[L % NL].arrive()
                    sempty[S % NSS].arrive()
                    lnext, snext = L + 1, S + 1
                else:
                    lempty[L % NL].arrive(2 // min(nst - 2 * (kb2 // 2), 2))
                    sempty[S % NSS].arrive(12 // min(nst - 4 * (kb2 // 4), 4))
            if current and pass_before_epilogue:
                yield from pass_fills(tl0 + nload, ts0 + nscale)
            yield dfull[j % KS], j // KS
            if any(q not in mma_done for q in range(tq0, tq0 + nst)):
                raise Violation(f"epilogue of tile {j} before its MMAs")
            dfree.arrive()
        if current and not pass_before_epilogue:
            yield from pass_fills(LT, ST)

    actors = [producer(), x_producer(), mma_issuer()] + [dequant_warp(s, w) for s in range(KS) for w in range(4)]
    names = ["producer", "x", "mma"] + [f"set{s}.warp{w}" for s in range(KS) for w in range(4)]
    interleave(actors, names, copies, commits, rng, lag)
    if len(mma_done) != q0:
        raise Violation("the run ended before every stage's MMAs completed")


LAGS = (0.05, 0.3, 1.0, 3.0)


def _small_m_plan(rng):
    # a CTA's tiles: full tiles of `a` stages and a shorter last tile, or one tile
    a = rng.choice([1, 2, 3, 4, 7, 10, 20])
    n = rng.choice([1, 1, 2, 3, 6])
    return [a] * n + ([rng.randint(1, a)] if rng.random() < 0.5 else [])


@pytest.mark.parametrize("block", range(4))
def test_small_m_protocol_holds(block):
    for t in range(150):
        seed = 1000 * block + t
        rng = random.Random(seed)
        tiles = _small_m_plan(rng)
        try:
            small_m(tiles, rng, rng.choice(LAGS))
        except Violation as v:
            raise AssertionError(f"tiles {tiles}, seed {seed}: {v}")


@pytest.mark.parametrize("T", [64, 128, 256])
def test_wide_protocol_holds(T):
    for t in range(120):
        seed = 7000 + 1000 * T + t
        rng = random.Random(seed)
        tiles = [rng.choice([1, 2, 3, 5, 13, 40]) for _ in range(rng.choice([1, 2, 3, 5]))]
        try:
            wide(T, tiles, rng, rng.choice(LAGS))
        except Violation as v:
            raise AssertionError(f"T {T}, tiles {tiles}, seed {seed}: {v}")


def _first_failure(run, seeds):
    for seed in seeds:
        try:
            run(random.Random(seed), LAGS[seed % len(LAGS)])
        except Violation as v:
            return str(v)
    return None


def test_small_m_one_release_barrier_per_slot_fails():
    """Two MMA warps, one release barrier per A slot: a set's wait can pass a phase early."""
    msg = _first_failure(lambda rng, lag: small_m([20], rng, lag, current=False), range(200))
    assert msg is not None and "passes at" in msg, msg


def test_wide_earlier_rules_fail():
    """Fills waited for only by the sets that read them: a codes or scale wait can pass early."""
    msg = _first_failure(lambda rng, lag: wide(256, [13, 40], rng, lag, current=False), range(400))
    assert msg is not None, "the earlier rules of the GEMM-form kernel were never caught"


def test_wide_epilogue_before_passing_fills_deadlocks():
    """Every set runs every epilogue: waiting for a tile's accumulators before passing the tile's
    remaining fills can hold back a fill that the tile's last stage needs."""
    msg = _first_failure(lambda rng, lag: wide(256, [2, 77, 13, 1, 1], rng, lag, pass_before_epilogue=False),
                         range(200))
    assert msg is not None and "deadlock" in msg, msg
