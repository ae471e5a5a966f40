"""Randomised model of the wide-group tcgen05 decode kernel's barrier protocol.

The kernel (paged_kv_cache_312_gb300/csrc/decode_tc05.cu) hands work between
warps through mbarriers:
  * three load warps; the lead one publishes each item's record and Q;
  * one MMA-issuing warp;
  * SW softmax warps (4 for 32-head items, 8 for 64-head items).
This test replays those warps' waits, arrivals and commits, in the kernel's
order, over modelled barriers. A random scheduler interleaves them with TMA
copies landing in any order, and with a tensor pipe that keeps issue order
only among the MMAs of one accumulator (all the ISA promises across
accumulators). A commit arrives once every MMA issued before it is done.

Checked in every run:
  * S reads the K tile of its key tile (the ring order K0 K1, then K(j+2)
    V(j) pairs, then the last two V) and the Q of its item.
  * P V reads its V tile and the P of its key tile, written by every softmax
    warp.
  * The softmax reads the S of its key tile.
  * Nothing is overwritten while it is still to be read: ring slots, S
    buffers, P buffers (also the vote and partial-sum scratch), O
    (rescale, read-out, the next item's first P V), Q buffers and records.
  * No parity wait falls two phases behind. No run deadlocks.
Mutations that each drop one wait must be caught.
"""
import random

import pytest

KLOAD = 3  # load warps


class Hazard(AssertionError):
    pass


class Barrier:
    def __init__(self, name, count):
        self.name, self.count = name, count
        self.phase = self.arrived = self.tx = 0

    def arrive(self, tx=0):
        self.arrived += 1
        self.tx += tx
        self._advance()

    def complete_tx(self, nbytes):
        self.tx -= nbytes
        self._advance()

    def _advance(self):
        if self.arrived == self.count and self.tx == 0:
            self.phase += 1
            self.arrived = 0

    def done(self, k):
        if self.phase >= k + 2:
            raise Hazard(f"{self.name}: waiter of phase {k} is two phases behind")
        return self.phase > k


def ring_step(i, n):
    """The i-th K or V tile an item's ring carries: ('K' | 'V', tile)."""
    if n == 1:
        return ("K", "V")[i], 0
    if i < 2:
        return "K", i
    if i >= 2 * n - 2:
        return "V", i - n
    m = (i - 2) >> 1
    return ("V", m) if (i - 2) & 1 else ("K", m + 2)


class Model:
    def __init__(self, items, slots, qb, sw, rng, mutation):
        self.items, self.slots, self.qb, self.sw = items, slots, qb, sw
        self.rng, self.mut = rng, mutation
        B = Barrier
        self.full = [B(f"full[{i}]", KLOAD) for i in range(slots)]
        self.empty = [B(f"empty[{i}]", 1) for i in range(slots)]
        self.q_full = [B(f"q_full[{i}]", 1) for i in range(qb)]
        self.q_empty = [B(f"q_empty[{i}]", 1 + sw + KLOAD - 1) for i in range(qb)]
        self.s_full = [B(f"s_full[{i}]", 1) for i in range(2)]
        self.s_free = [B(f"s_free[{i}]", sw) for i in range(2)]
        self.p_full = [B(f"p_full[{i}]", sw) for i in range(2)]
        self.o_done = [B(f"o_done[{i}]", 1) for i in range(2)]
        self.drain = B("drain", 1)
        self.slot_tag, self.slot_readers = [None] * slots, [0] * slots
        self.rec = [None] * qb                # item index (len(items) = the end record)
        self.rec_reads = [0] * qb             # warps that read the record
        self.q_item, self.q_readers = [None] * qb, [0] * qb
        self.s_tag, self.s_reads, self.s_pending = [None, None], [set(), set()], [0, 0]
        self.p_tag, self.p_writers, self.pv_pending = [None, None], [set(), set()], [0, 0]
        self.o_owner, self.o_reads, self.o_pending = None, 0, 0
        self.pipe, self.copies = [], []

    def check(self, cond, what):
        if not cond:
            raise Hazard(what)

    def issue(self, acc, run):
        self.pipe.append({"acc": acc, "run": run})

    def commit(self, bar):
        self.pipe.append({"acc": "commit", "run": bar.arrive})

    def runnable_ops(self):
        out, seen, mma_before = [], set(), False
        for op in self.pipe:
            if op["acc"] == "commit":
                if not mma_before:
                    out.append(op)
                continue
            if op["acc"] not in seen:
                out.append(op)
            seen.add(op["acc"])
            mma_before = True
        return out

    def publish(self, n):
        """The lead load warp writes item n's Q and record into buffer n % QB."""
        b = n % self.qb
        self.check(self.q_readers[b] == 0, f"Q buffer {b} overwritten while an S MMA reads it")
        self.check(self.rec[b] is None or self.rec_reads[b] == self.sw + KLOAD - 1,
                   f"record {b} overwritten before every warp read it")
        self.rec[b], self.rec_reads[b] = n, 0
        if n < len(self.items):
            self.q_item[b] = n


def load_warp(m, lead):
    n = t = 0
    while True:
        b = n % m.qb
        if lead:
            if n >= m.qb and m.mut != "no_q_empty_wait":
                yield ("wait", m.q_empty[b], n // m.qb - 1)
            m.publish(n)
            m.q_full[b].arrive()
        else:
            yield ("wait", m.q_full[b], n // m.qb)
            m.check(m.rec[b] == n, f"load warp read record {m.rec[b]} for item {n}")
            m.rec_reads[b] += 1
            m.q_empty[b].arrive()
        item, n = n, n + 1
        if item == len(m.items):
            return
        nkt = m.items[item]
        for i in range(2 * nkt):
            kv, j = ring_step(i, nkt)
            sl = t % m.slots
            if t >= m.slots:
                yield ("wait", m.empty[sl], t // m.slots - 1)
            m.check(m.slot_readers[sl] == 0, f"slot {sl} reloaded while an MMA reads it")
            m.full[sl].arrive(tx=1)
            m.slot_tag[sl] = None
            m.copies.append((sl, (kv, m.kt0[item] + j)))
            t += 1
            yield ("step",)


def mma_warp(m):
    n = tc = 0
    while True:
        b = n % m.qb
        yield ("wait", m.q_full[b], n // m.qb)
        item, n = m.rec[b], n + 1
        m.check(item == n - 1, f"MMA warp read record {item} for item {n - 1}")
        if item == len(m.items):
            break
        nkt, kt0 = m.items[item], m.kt0[item]

        def take():
            nonlocal tc
            t = tc
            tc += 1
            return ("wait", m.full[t % m.slots], t // m.slots), t % m.slots

        def s_step(kt):
            sb = kt & 1
            if kt >= 2 and m.mut != "no_s_free_wait":
                yield ("wait", m.s_free[sb], (kt - 2) >> 1)
            w, sl = take()
            yield w
            m.slot_readers[sl] += 1
            m.q_readers[b] += 1
            m.s_pending[sb] += 1

            def run(kt=kt, sl=sl, sb=sb, bb=b, it=item):
                m.check(m.slot_tag[sl] == ("K", kt), f"S({kt}) read slot {sl} = {m.slot_tag[sl]}")
                m.check(m.q_item[bb] == it, f"S({kt}) read the Q of item {m.q_item[bb]}")
                m.check(m.s_tag[sb] is None or len(m.s_reads[sb]) == m.sw,
                        f"S({kt}) overwrote S({m.s_tag[sb]}) before every softmax warp read it")
                m.s_tag[sb], m.s_reads[sb] = kt, set()
                m.slot_readers[sl] -= 1
                m.q_readers[bb] -= 1
                m.s_pending[sb] -= 1
            m.issue(f"S{sb}", run)
            m.commit(m.s_full[sb])
            m.commit(m.empty[sl])

        for j in range(min(nkt, 2)):
            yield from s_step(kt0 + j)
        for j in range(nkt):
            kt = kt0 + j
            if j + 2 < nkt:
                yield from s_step(kt + 2)
            sb = kt & 1
            yield ("wait", m.p_full[sb], kt >> 1)
            w, sv = take()
            yield w
            m.slot_readers[sv] += 1
            m.pv_pending[sb] += 1
            m.o_pending += 1

            def run(kt=kt, sv=sv, sb=sb, first=j == 0, it=item):
                m.check(m.slot_tag[sv] == ("V", kt), f"PV({kt}) read slot {sv} = {m.slot_tag[sv]}")
                m.check(m.p_tag[sb] == kt and len(m.p_writers[sb]) == m.sw,
                        f"PV({kt}) read P before every softmax warp wrote it")
                if first:
                    m.check(m.o_owner is None or m.o_reads == m.sw,
                            f"PV({kt}) overwrote O before its read-out")
                    m.o_owner, m.o_reads = it, 0
                m.slot_readers[sv] -= 1
                m.pv_pending[sb] -= 1
                m.o_pending -= 1
            m.issue("O", run)
            m.commit(m.o_done[sb])
            m.commit(m.empty[sv])
        m.commit(m.q_empty[b])
    m.commit(m.drain)
    yield ("wait", m.drain, 0)


def softmax_warp(m, w):
    n = 0

    def write_p_buffer(sb, what):
        m.check(m.pv_pending[sb] == 0, f"{what} written into P buffer {sb} while a P V reads it")

    while True:
        b = n % m.qb
        yield ("wait", m.q_full[b], n // m.qb)
        item, n = m.rec[b], n + 1
        m.check(item == n - 1, f"softmax warp read record {item} for item {n - 1}")
        m.rec_reads[b] += 1
        m.q_empty[b].arrive()
        if item == len(m.items):
            return
        nkt, kt0 = m.items[item], m.kt0[item]
        if nkt == 0:
            continue
        for j in range(nkt):
            kt, sb = kt0 + j, (kt0 + j) & 1
            yield ("wait", m.s_full[sb], kt >> 1)
            m.check(m.s_tag[sb] == kt and m.s_pending[sb] == 0,
                    f"softmax read S({kt}): the buffer holds S({m.s_tag[sb]}) and "
                    f"{m.s_pending[sb]} S MMA(s) still to write it")
            m.s_reads[sb].add(w)
            m.s_free[sb].arrive()
            if kt >= 2 and m.mut != "no_p_free_wait":
                yield ("wait", m.o_done[sb], (kt - 2) >> 1)
            if m.rng.random() < 0.5:  # a score passed the running max: the vote's scratch
                write_p_buffer(sb, "the vote's scratch")
                if j > 0 and m.rng.random() < 0.5:  # the max moved: O is rescaled
                    if m.mut != "no_rescale_wait":
                        yield ("wait", m.o_done[(kt - 1) & 1], (kt - 1) >> 1)
                    m.check(m.o_pending == 0, "O rescaled while a P V accumulates")
            write_p_buffer(sb, f"P({kt})")
            if m.p_tag[sb] != kt:
                m.p_tag[sb], m.p_writers[sb] = kt, set()
            m.p_writers[sb].add(w)
            m.p_full[sb].arrive()
            yield ("step",)
        kl = kt0 + nkt - 1
        if kl >= 1 and m.mut != "no_scratch_wait":
            yield ("wait", m.o_done[(kl - 1) & 1], (kl - 1) >> 1)
        write_p_buffer((kl - 1) & 1, "the partial sums' scratch")
        yield ("wait", m.o_done[kl & 1], kl >> 1)
        m.check(m.o_pending == 0 and m.o_owner == item, "O read out before its last P V")
        m.o_reads += 1


def run_once(items, slots, qb, sw, seed, mutation=None):
    rng = random.Random(seed)
    m = Model(items, slots, qb, sw, rng, mutation)
    m.kt0, acc = [], 0
    for nkt in items:
        m.kt0.append(acc)
        acc += nkt
    agents = ([load_warp(m, True)] + [load_warp(m, False) for _ in range(KLOAD - 1)] +
              [mma_warp(m)] + [softmax_warp(m, w) for w in range(sw)])
    waiting, alive = [None] * len(agents), [True] * len(agents)
    while True:
        choices = [("agent", i) for i in range(len(agents))
                   if alive[i] and (waiting[i] is None or waiting[i][0].done(waiting[i][1]))]
        choices += [("copy", c) for c in range(len(m.copies))]
        choices += [("op", op) for op in m.runnable_ops()]
        if not choices:
            if any(alive):
                raise Hazard("deadlock: " + ", ".join(
                    f"agent {i} waits {w[0].name} phase {w[1]}" for i, w in enumerate(waiting)
                    if alive[i] and w))
            return
        kind, c = rng.choice(choices)
        if kind == "agent":
            waiting[c] = None
            try:
                act = next(agents[c])
                if act[0] == "wait":
                    waiting[c] = (act[1], act[2])
            except StopIteration:
                alive[c] = False
        elif kind == "copy":
            sl, tag = m.copies.pop(c)
            m.slot_tag[sl] = tag
            m.full[sl].complete_tx(1)
        else:
            m.pipe.remove(c)
            c["run"]()


def random_items(rng):
    return [0 if rng.random() < 0.1 else rng.randint(1, 6) for _ in range(rng.randint(1, 5))]


# 32-head items: two Q buffers, four softmax warps, five slots; 64-head items:
# one Q buffer, eight softmax warps, four slots
SHAPES = [pytest.param(5, 2, 4, id="32-head"), pytest.param(4, 1, 8, id="64-head")]


@pytest.mark.parametrize("slots,qb,sw", SHAPES)
def test_wide_decode_protocol_holds_under_random_schedules(slots, qb, sw):
    rng = random.Random(7 + sw)
    for s in range(300):
        run_once(random_items(rng), slots, qb, sw, seed=s)


@pytest.mark.parametrize("mutation", ["no_s_free_wait", "no_p_free_wait", "no_q_empty_wait",
                                      "no_scratch_wait", "no_rescale_wait"])
def test_wide_decode_protocol_model_catches_a_dropped_wait(mutation):
    rng = random.Random(5)
    for s in range(600):
        try:
            run_once(random_items(rng), 5, 2, 4, seed=s, mutation=mutation)
        except Hazard:
            return
    pytest.fail(f"the model missed mutation {mutation}")
