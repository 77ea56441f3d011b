"""A randomised model of the streaming indexer's per-token synchronisation (no GPU).

The streaming prefill with 32 indexer heads gives each token of a work item to
one epilogue warpgroup of four warps. The warps share the token's candidate
buffer, its count, threshold and cut request, a counter of warps done with the
item, and a four-arrival barrier; they meet only when a reservation overflows
the buffer (a cut) and at the end of an item. This model runs the same control
flow as the kernel with every warp a generator and a random scheduler choosing
which one takes its next shared-memory step, together with the MMA side (an
accumulator ring of four buffers that every epilogue warp must release). It
checks that every schedule ends (no deadlock), that the barrier never runs two
phases ahead of a waiting warp (its parity wait could not tell them apart), and
that each row's final buffer holds its exact top-k. A variant that resets the
row state at the end of an item instead of its start (a race found in review:
a slow warp could read the reset count) must be caught.
"""
import random

import pytest

WARPS = 4      # warps per warpgroup (TMEM lane quadrants)
ACC = 4        # accumulator buffers in the ring


class Barrier:
    def __init__(self):
        self.pending = 0
        self.completed = 0


class Token:
    def __init__(self):
        self.cnt = 0
        self.theta = 0
        self.flag = 0
        self.done = 0
        self.buf = {}
        self.bar = Barrier()


class Deadlock(Exception):
    pass


class Model:
    """n_wg warpgroups (tokens), items of n_tiles tiles, `lanes` keys per warp per tile."""

    def __init__(self, seed, n_wg=2, n_items=3, cap=16, topk=5, lanes=2, reset_at_end=False, defer=True):
        self.rng = random.Random(seed)
        self.n_wg, self.cap, self.topk, self.lanes = n_wg, cap, topk, lanes
        # the kernel's sizes: a warpgroup holds at most 4 x 32 = 128 entries, a
        # cut frees at least 512 slots (else it selects exactly) and an exact
        # cut leaves cap - topk = 2048 free, so the held entries always fit
        self.slack = WARPS * lanes
        assert cap - topk >= self.slack
        self.reset_at_end, self.defer = reset_at_end, defer
        self.tok = [Token() for _ in range(n_wg)]
        self.items = []
        for _ in range(n_items):
            nt = self.rng.randint(1, 9)
            # keys[g][t][w] = [(score, index)] for the lanes of warp w in tile t of token g
            keys = [[[[(self.rng.randint(0, 6), (t * WARPS + w) * lanes + l) for l in range(lanes)]
                      for w in range(WARPS)] for t in range(nt)] for _ in range(n_wg)]
            self.items.append(dict(nt=nt, keys=keys, trivial=self.rng.random() < 0.15))
        self.tile_base = []
        acc = 0
        for it in self.items:
            self.tile_base.append(acc)
            if not it["trivial"]:
                acc += it["nt"]
        self.n_tiles = acc
        self.produced = 0
        self.released = [0] * (self.n_tiles + 1)
        self.results = {}
        self.progress = 0

    # ------------------------------------------------------------------ MMA side
    def mma(self):
        while self.produced < self.n_tiles:
            t = self.produced
            if t >= ACC and self.released[t - ACC] < WARPS * self.n_wg:
                yield
                continue
            self.produced += 1
            self.progress += 1
            yield

    # ------------------------------------------------------------------ one epilogue warp
    def warp(self, g, w):
        S = self.tok[g]
        cap, topk = self.cap, self.topk
        st = dict(phase=0, hold=[], items_done=0)

        def meet():
            B = S.bar
            B.pending += 1
            if B.pending == WARPS:
                B.pending = 0
                B.completed += 1
            yield
            while B.completed <= st["phase"]:
                yield
            # a parity wait cannot tell phase n from n + 2
            assert B.completed == st["phase"] + 1, "barrier ran two phases ahead of a waiting warp"
            st["phase"] += 1

        def cut():
            yield from meet()
            n = min(S.cnt, cap)
            entries = [S.buf[i] for i in range(n)]
            yield
            for _ in range(3):  # key range, histogram, bin scan
                yield from meet()
            order = sorted(entries, key=lambda e: (-e[0], e[1]))
            tk = order[topk - 1][0] if n > topk else 0
            kept = [e for e in entries if e[0] >= tk]
            exact = len(kept) > cap - self.slack
            if exact:
                for _ in range(4):  # exact radix selection
                    yield from meet()
                keep = set(order[:topk])
                kept = [e for e in entries if e in keep]
                tk = order[topk - 1][0]
            for _ in range((n + 7) // 8):  # compaction rounds
                yield from meet()
            if w == 0:
                S.buf = {i: e for i, e in enumerate(kept)}
                S.cnt = len(kept)
                S.theta = tk
                S.flag = 0
            yield
            yield from meet()
            re = [e for e in st["hold"] if e[0] >= tk]
            st["hold"] = []
            if re:
                old = S.cnt
                S.cnt += len(re)
                yield
                for j, e in enumerate(re):
                    assert old + j < cap, "held entries do not fit after a cut"
                    S.buf[old + j] = e
                yield
            yield from meet()
            self.progress += 1

        for ii, item in enumerate(self.items):
            if item["trivial"]:
                continue
            if w == 0 and not self.reset_at_end:
                S.cnt = 0
                S.theta = 0
            yield
            yield from meet()
            for t in range(item["nt"]):
                gt = self.tile_base[ii] + t
                while True:  # wait for the accumulator, serving cut requests first
                    if S.flag:
                        yield from cut()
                        continue
                    if self.produced > gt:
                        break
                    yield
                self.released[gt] += 1
                self.progress += 1
                yield
                theta = S.theta
                yield
                adm = [e for e in item["keys"][g][t][w] if e[0] >= theta]
                if adm:
                    old = S.cnt
                    S.cnt += len(adm)  # one atomic per warp
                    yield
                    for j, e in enumerate(adm):
                        if old + j < cap:
                            S.buf[old + j] = e
                        else:
                            st["hold"].append(e)
                    if old + len(adm) > cap:
                        S.flag = 1
                    yield
            S.done += 1
            st["items_done"] += 1
            yield
            while True:  # the other warps: count first, then the request
                done = S.done
                yield
                flag = S.flag
                yield
                if flag:
                    yield from cut()
                    continue
                if done >= WARPS * st["items_done"]:
                    break
                yield
            assert not st["hold"], "entry held past the end of an item"
            yield from meet()
            n = min(S.cnt, cap)
            yield
            if w == 0:
                self.results[(ii, g)] = [S.buf[i] for i in range(n)]
            if not (n > topk and self.defer):
                for _ in range(3):  # in-kernel selection and sort
                    yield from meet()
            if w == 0 and self.reset_at_end:
                S.cnt = 0
                S.theta = 0
            yield
            yield from meet()
            self.progress += 1

    # ------------------------------------------------------------------ scheduler
    def run(self, max_idle=20000):
        procs = [self.mma()] + [self.warp(g, w) for g in range(self.n_wg) for w in range(WARPS)]
        live = list(range(len(procs)))
        idle, last = 0, -1
        while live:
            i = self.rng.choice(live)
            try:
                next(procs[i])
            except StopIteration:
                live.remove(i)
            if self.progress != last:
                last, idle = self.progress, 0
            else:
                idle += 1
                if idle > max_idle:
                    raise Deadlock("no progress")

    def check(self):
        for ii, item in enumerate(self.items):
            if item["trivial"]:
                continue
            for g in range(self.n_wg):
                allk = [e for t in item["keys"][g] for wl in t for e in wl]
                want = sorted(allk, key=lambda e: (-e[0], e[1]))[:self.topk]
                got = self.results[(ii, g)]
                assert set(want) <= set(got), (ii, g)
                assert len(got) == len(set(got)) and set(got) <= set(allk)


@pytest.mark.parametrize("seed", range(150))
def test_protocol_ends_and_keeps_the_topk(seed):
    m = Model(seed, defer=seed % 2 == 0)
    m.run()
    m.check()


def test_protocol_many_cuts_tight_buffer():
    for seed in range(40):
        m = Model(1000 + seed, n_wg=3, n_items=4, cap=8, topk=3, lanes=1)
        m.run()
        m.check()


def test_model_catches_the_end_of_item_reset():
    """Resetting the count at the end of an item lets a slow warp read the reset
    count and take another path through its meetings: some schedule must fail."""
    failures = 0
    for seed in range(200):
        m = Model(seed, reset_at_end=True, defer=True)
        try:
            m.run()
            m.check()
        except (AssertionError, Deadlock):
            failures += 1
    assert failures > 0
