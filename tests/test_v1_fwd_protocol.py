"""Model check of the V1 forward kernel's barrier protocol (CPU only).

`csrc/v1_fwd.cu` runs each work item on a pair of CTAs whose warps hand
work to each other through mbarriers: a Q/K producer and a V producer, an
MMA issuer, the tensor pipe and the TMA engine (both asynchronous), eight
softmax warps in two warpgroups that meet at a named barrier, and four
epilogue warps per CTA.  Between the two CTAs: each V tile is loaded half
by each CTA with multicast into both, and a V stage is refilled only once
both CTAs' P.V commits (which arrive on both CTAs' barriers) say it is
free; the exchange slot; and the per-row partial sums (one data slot,
barriers by item parity).  An mbarrier wait only compares the parity of the
phase it waits for, so a protocol in which a barrier can complete two
phases before a waiter looks at it hangs or reads the wrong data.

This model gives every warp, the tensor pipe and the TMA engine of both
CTAs its own coroutine, runs them under seeded random interleavings, and
checks:
  * every parity wait returns on exactly the phase it waits for;
  * the O accumulator is overwritten by the next item's first P.V only
    after the epilogue has read it, and rescaled only within its item;
  * the softmax -> epilogue hand-off slot is not overwritten before it was
    read;
  * an exchange slot is rewritten only after the partner has read it, and
    read only while it holds the item being combined;
  * a V stage receives either half of a new tile only after both CTAs'
    P.V MMAs have read the tile it held, and a P.V reads a stage only when
    both halves of its tile have landed there;
  * the partial-sum slot is overwritten only after its value was read;
  * the swapped half maxima of a rare max-raising tile go through the
    hand-off slot only after the epilogue has read it;
  * no interleaving deadlocks.
A second test removes one wait from the model and checks that the model
catches it, so the checks themselves are exercised.
"""
import random

import pytest


class Barrier:
    """An mbarrier: `need` arrivals complete a phase; `done` phases so far."""

    def __init__(self, need):
        self.need = need
        self.count = 0
        self.done = 0

    def arrive(self, k=1):
        self.count += k
        while self.count >= self.need:
            self.count -= self.need
            self.done += 1

    def phase_complete(self, phase):
        # try_wait.parity semantics: only the parity of the current phase is seen
        return (self.done & 1) != (phase & 1)


class Model:
    def __init__(self, items, rnd, drop=None):
        self.items = items
        self.rnd = rnd
        self.drop = drop or set()
        self.errors = []
        self.ctas = [self._cta() for _ in range(2)]

    @staticmethod
    def _cta():
        bars = {}
        for name, need in [("QFULL", 1), ("QEMPTY", 1), ("ORDY", 1), ("ODONE", 1), ("EPI", 256),
                           ("OFREE", 128), ("XRDY", 128), ("SSQ0", 129), ("SSQ1", 129)]:
            bars[name] = Barrier(need)
        for s in range(2):
            # VFULL: the local arm plus both halves' bytes; VEMPTY: both CTAs' P.V commits
            for name, need in [("KFULL", 1), ("KEMPTY", 1), ("VFULL", 3), ("VEMPTY", 2), ("SFULL", 1),
                               ("PFULL", 256)]:
                bars[(name, s)] = Barrier(need)
        return dict(bars=bars, pipe=[], tma=[], o_read=-1, o_item=-1, slot=-1, reading=False,
                    handoff=None, handoff_taken=-1, vhalf=[[-1, -1], [-1, -1]], pv_done=[-1, -1],
                    ssq_val=-1, ssq_read=-1, nb=[0, 0])

    def wait(self, bar, phase, tag):
        while not bar.phase_complete(phase):
            yield
        if bar.done != phase + 1:
            self.errors.append((tag, "woke on phase", bar.done - 1, "waiting for", phase))

    def named_sync(self, c):
        """bar.sync 1, 256: the eight softmax warps of CTA c (count, generation)."""
        nb = self.ctas[c]["nb"]
        gen = nb[1]
        nb[0] += 1
        if nb[0] == 8:
            nb[0] = 0
            nb[1] += 1
        while nb[1] == gen:
            yield

    def trip(self, it, j):
        # a rare tile whose sum leaves the guard: decided by a barrier reduction,
        # so the same for every softmax warp of the CTA
        return j > 0 and random.Random(hash((id(self), it, j)) & 0xffffffff).random() < 0.3

    # ---- asynchronous engines ------------------------------------------------
    def tma_engine(self, c):
        cta = self.ctas[c]
        while True:
            if cta["tma"] and self.rnd.random() < 0.5:
                ev = cta["tma"].pop(self.rnd.randrange(len(cta["tma"])))
                if ev[0] == "Vhalf":  # one half of V tile g multicast into both CTAs
                    _, g, half = ev
                    st = g & 1
                    for d in range(2):
                        dst = self.ctas[d]
                        if g >= 2 and dst["pv_done"][st] < g - 2:
                            self.errors.append(("V stage overwritten before its P.V read it", d, g))
                        dst["vhalf"][st][half] = g
                        dst["bars"][("VFULL", st)].arrive()
                else:
                    cta["bars"][ev].arrive()
            yield

    def tensor_pipe(self, c):
        cta = self.ctas[c]
        while True:
            if cta["pipe"] and self.rnd.random() < 0.5:
                op = cta["pipe"].pop(0)
                if op[0] == "commit":
                    cta["bars"][op[1]].arrive()
                elif op[0] == "commit_mc":  # arrives on the barrier of both CTAs
                    for d in range(2):
                        self.ctas[d]["bars"][op[1]].arrive()
                elif op[0] == "PV":
                    _, it, g, first = op
                    st = g & 1
                    if cta["vhalf"][st] != [g, g]:
                        self.errors.append(("P.V read a V stage without both halves of its tile", c, g,
                                            cta["vhalf"][st]))
                    cta["pv_done"][st] = g
                    if first:
                        if it > 0 and cta["o_read"] < it - 1:
                            self.errors.append(("first P.V overwrote an unread O", c, it))
                        cta["o_item"] = it
            yield

    # ---- warps ------------------------------------------------------------------
    def producer_qk(self, c):
        b = self.ctas[c]["bars"]
        tma = self.ctas[c]["tma"]
        kv = 0
        for it, n in enumerate(self.items):
            if it > 0:
                yield from self.wait(b["QEMPTY"], it - 1, "producer Q")
            tma.append("QFULL")
            for _ in range(n):
                st, use = kv & 1, kv >> 1
                if use > 0:
                    yield from self.wait(b[("KEMPTY", st)], use - 1, "producer K")
                tma.append(("KFULL", st))
                kv += 1
                yield

    def producer_v(self, c):
        b = self.ctas[c]["bars"]
        tma = self.ctas[c]["tma"]
        kv = 0
        for n in self.items:
            for _ in range(n):
                st, use = kv & 1, kv >> 1
                if use > 0 and "producer VEMPTY" not in self.drop:
                    yield from self.wait(b[("VEMPTY", st)], use - 1, "producer V")
                b[("VFULL", st)].arrive()        # the local arm with the whole tile's bytes
                tma.append(("Vhalf", kv, c))     # this CTA's half, multicast to both
                kv += 1
                yield

    def mma(self, c):
        b = self.ctas[c]["bars"]
        pipe = self.ctas[c]["pipe"]
        kv = 0
        for it, n in enumerate(self.items):
            yield from self.wait(b["QFULL"], it, "mma Q")
            for j in range(min(2, n)):
                g = kv + j
                yield from self.wait(b[("KFULL", g & 1)], g >> 1, "mma K")
                pipe += [("S", g), ("commit", ("KEMPTY", g & 1)), ("commit", ("SFULL", g & 1))]
                if j == n - 1:
                    pipe.append(("commit", "QEMPTY"))
            for j in range(n):
                g = kv + j
                st = g & 1
                if j == 0 and it > 0 and "mma OFREE" not in self.drop:
                    yield from self.wait(b["OFREE"], it - 1, "mma OFREE")
                yield from self.wait(b[("PFULL", st)], g >> 1, "mma P")
                yield from self.wait(b[("VFULL", st)], g >> 1, "mma V")
                pipe += [("PV", it, g, j == 0),
                         ("commit", ("VEMPTY", st)) if "multicast VEMPTY" in self.drop
                         else ("commit_mc", ("VEMPTY", st)),
                         ("commit", "ODONE")]
                if j + 2 < n:
                    yield from self.wait(b[("KFULL", (g + 2) & 1)], (g + 2) >> 1, "mma K ahead")
                    pipe += [("S", g + 2), ("commit", ("KEMPTY", st)), ("commit", ("SFULL", st))]
                    if j + 2 == n - 1:
                        pipe.append(("commit", "QEMPTY"))
            pipe.append(("commit", "ORDY"))
            kv += n

    def softmax(self, c, warp):
        cta = self.ctas[c]
        b = cta["bars"]
        kv = 0
        for it, n in enumerate(self.items + [None]):
            yield from self.named_sync(c)  # the stop reduction at an item's start
            if n is None:  # end of the sequence
                if it > 0:
                    yield from self.wait(b["OFREE"], it - 1, "softmax end")
                if warp == 0:
                    cta["handoff"] = ("end", it)
                b["EPI"].arrive(32)
                return
            for j in range(n):
                g = kv + j
                yield from self.wait(b[("SFULL", g & 1)], g >> 1, "softmax S")
                yield from self.named_sync(c)  # first tile: both halves read the row; later: the guard
                if self.trip(it, j):
                    # rare: the half maxima swap through the hand-off slots, then O is rescaled
                    if it > 0 and "softmax rare OFREE" not in self.drop:
                        yield from self.wait(b["OFREE"], it - 1, "softmax rare")
                    if cta["handoff_taken"] < it - 1:
                        self.errors.append(("half maxima overwrote an unread hand-off", c, it))
                    yield from self.named_sync(c)
                    yield from self.wait(b["ODONE"], g - 1, "softmax rescale")
                    if cta["o_item"] != it:
                        self.errors.append(("rescaled O of another item", c, it, cta["o_item"]))
                    yield from self.named_sync(c)
                yield
                b[("PFULL", g & 1)].arrive(32)
            kv += n
            if it > 0 and "softmax OFREE" not in self.drop:
                yield from self.wait(b["OFREE"], it - 1, "softmax hand-off")
            if warp == 0:
                if cta["handoff_taken"] < it - 1:
                    self.errors.append(("hand-off slot overwritten before it was read", c, it))
                cta["handoff"] = ("item", it)
            yield from self.named_sync(c)  # both half sums written before the LSE
            b["EPI"].arrive(32)

    def epilogue(self, c, warp):
        cta, peer = self.ctas[c], self.ctas[1 - c]
        b, pb = cta["bars"], peer["bars"]
        for it in range(len(self.items) + 1):
            yield from self.wait(b["EPI"], it, "epilogue hand-off")
            kind, which = cta["handoff"]
            if which != it:
                self.errors.append(("hand-off slot holds another item", c, it, which))
            if kind == "end":
                return
            yield from self.wait(b["ORDY"], it, "epilogue O ready")
            if cta["o_item"] != it:
                self.errors.append(("O holds another item", c, it, cta["o_item"]))
            if warp == 0:
                if peer["reading"]:
                    self.errors.append(("exchange slot rewritten under the partner's read", c, it))
                cta["slot"] = it
            for _ in range(self.rnd.randint(1, 40)):  # reading O out of TMEM takes a while
                yield
            if warp == 0:
                cta["handoff_taken"] = it
                cta["o_read"] = it
            b["OFREE"].arrive(32)
            pb["XRDY"].arrive(32)
            yield from self.wait(b["XRDY"], it, "epilogue partner slot")
            if warp == 0:
                cta["reading"] = True
                if peer["slot"] != it:
                    self.errors.append(("partner slot holds another item", c, it, peer["slot"]))
            yield
            if warp == 0:
                if peer["slot"] != it:
                    self.errors.append(("partner slot changed during the read", c, it))
                cta["reading"] = False
            parity = it & 1
            if warp == 0:
                b["SSQ%d" % parity].arrive(1)  # the local arrive with the expected bytes
                if peer["ssq_read"] < it - 1:
                    self.errors.append(("partial-sum slot overwritten before it was read", 1 - c, it))
                peer["ssq_val"] = it
            pb["SSQ%d" % parity].arrive(32)    # 32 rows' 4-byte stores into the partner
            yield from self.wait(b["SSQ%d" % parity], it >> 1, "epilogue partial sums")
            if warp == 0:
                if cta["ssq_val"] != it:
                    self.errors.append(("partial-sum slot holds another item", c, it, cta["ssq_val"]))
                cta["ssq_read"] = it
            yield

    def run(self, max_steps=400000):
        actors, engines = [], []
        for c in range(2):
            engines += [self.tma_engine(c), self.tensor_pipe(c)]
            actors += [self.producer_qk(c), self.producer_v(c), self.mma(c)]
            actors += [self.softmax(c, w) for w in range(8)]
            actors += [self.epilogue(c, w) for w in range(4)]
        everyone = engines + actors
        live = set(range(len(engines), len(everyone)))
        steps = 0
        while live and not self.errors:
            k = self.rnd.randrange(len(everyone))
            if k >= len(engines) and k not in live:
                continue
            try:
                next(everyone[k])
            except StopIteration:
                live.discard(k)
            steps += 1
            if steps > max_steps:
                self.errors.append(("deadlock", sorted(live)))
        return self.errors


def _random_items(rnd):
    # key tiles per item: causal items from the diagonal (1 tile) to a few tiles
    return [rnd.choice([1, 1, 2, 3, 5]) for _ in range(rnd.randint(1, 7))]


def test_protocol_holds_under_random_interleavings():
    for seed in range(150):
        rnd = random.Random(seed)
        items = _random_items(rnd)
        errors = Model(items, rnd).run()
        assert not errors, (seed, items, errors[:3])


@pytest.mark.parametrize("dropped", ["mma OFREE", "softmax OFREE", "producer VEMPTY", "multicast VEMPTY",
                                     "softmax rare OFREE"])
def test_model_catches_a_missing_wait(dropped):
    caught = 0
    for seed in range(150):
        rnd = random.Random(seed)
        items = _random_items(rnd)
        if Model(items, rnd, drop={dropped}).run():
            caught += 1
    assert caught > 0, f"dropping the {dropped} wait went unnoticed"
