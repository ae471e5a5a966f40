"""Randomised model of the tcgen05 prefill kernel's barrier protocol.

The kernel (paged_kv_cache_312_gb300/csrc/prefill_tc05.cu) runs one load warp,
one MMA-issuing warp and four softmax warps per 128-row query tile (two
tiles, A and B), handing data over through mbarriers.  This test replays that
control flow, the same waits, arrivals and commits in the same order, as
Python agents over modelled barriers. A random scheduler interleaves them
with the asynchronous parts:
  * TMA copies land in any order;
  * the tensor pipe executes MMAs in any order that keeps the MMAs of one
    accumulator in issue order, which is all the ISA promises for different
    accumulators; a commit arrives once every MMA issued before it is done.

Each run checks three things.
  * Every consumer sees what it expects: S reads the K tile and Q of its key
    tile and item; P V reads P of its tile written by all four softmax warps,
    and its V tile; the softmax reads S of its key tile.
  * No buffer is overwritten while a pending MMA still reads it: ring slots,
    the S/P columns, the O accumulator (rescale, read-out, the next item's
    first P V) and the Q buffer.
  * No parity wait falls two phases behind, which a parity bit cannot tell
    apart from the phase it waits for. No run deadlocks.
Mutations that drop one wait each must be caught.  The model runs on the
CPU in a few seconds.
"""
import random

import pytest


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
        """Phase k has completed.  A waiter two phases behind would see the
        parity of phase k again and wait for ever."""
        if self.phase >= k + 2:
            raise Hazard(f"{self.name}: waiter of phase {k} is two phases behind")
        return self.phase > k


class Model:
    """Shared state of one CTA: barriers, buffers, the tensor pipe, copies."""

    def __init__(self, items, slots, rng, mutation=None):
        self.items, self.slots, self.rng, self.mut = items, slots, rng, mutation
        self.full = [Barrier(f"full[{i}]", 1) for i in range(slots)]
        self.empty = [Barrier(f"empty[{i}]", 1) for i in range(slots)]
        self.s_full = [Barrier(f"s_full[{x}]", 1) for x in range(2)]
        self.o_full = [Barrier(f"o_full[{x}]", 1) for x in range(2)]
        self.q_full = [Barrier(f"q_full[{x}]", 4) for x in range(2)]
        self.p_half = [[Barrier(f"p_half[{x}][{h}]", 4) for h in range(2)] for x in range(2)]
        self.drain = Barrier("drain", 1)
        # buffers
        self.slot_tag = [None] * slots           # ('K' | 'V', key tile) that has landed
        self.slot_readers = [0] * slots          # issued MMAs that still read the slot
        self.q_written = [{}, {}]                # item -> warps that wrote their Q rows
        self.q_readers = [0, 0]                  # issued S MMAs still reading Q_x
        self.s_tag = [None, None]                # (item, key tile) of S in tile x's columns
        self.s_pending = [0, 0]                  # issued S MMAs of tile x not yet done
        self.p_written = [[set(), set()], [set(), set()]]  # per half: warps that wrote P
        self.pv_pending = [0, 0]                 # issued P V MMAs of tile x not yet done
        self.o_owner = [None, None]              # item accumulating in O_x
        self.o_reads = [0, 0]                    # warps that read out o_owner's O
        self.pipe = []                           # issued MMAs and commits, in issue order
        self.copies = []                         # TMA copies in flight

    # ------------------------------------------------------------- pipe
    def issue(self, acc, run):
        self.pipe.append({"acc": acc, "run": run})

    def commit(self, bar):
        self.pipe.append({"acc": "commit", "run": bar.arrive})

    def runnable_ops(self):
        """An MMA may run once every earlier MMA on its accumulator has run; a
        commit once every MMA issued before it has.  A commit holds nothing
        back: later MMAs may finish before it arrives."""
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

    # ---------------------------------------------------------- checks
    def check(self, cond, what):
        if not cond:
            raise Hazard(what)


def slot_of(m, t):
    return t % m.slots


def load_warp(m):
    t = 0
    for it, (na, nb) in enumerate(m.items):
        for j in range(max(na, nb)):
            kt = m.kt0[it] + j
            for kv in ("K", "V"):
                sl = slot_of(m, t)
                if t >= m.slots and m.mut != "no_empty_wait":
                    yield ("wait", m.empty[sl], t // m.slots - 1)
                m.check(m.slot_readers[sl] == 0, f"slot {sl} reloaded while an MMA reads it")
                m.full[sl].arrive(tx=1)
                m.slot_tag[sl] = None  # overwritten from now on
                m.copies.append((sl, (kv, kt)))
                t += 1
                yield ("step",)


def mma_warp(m):
    n, nq = [0, 0], [0, 0]
    for it, (na, nb) in enumerate(m.items):
        nkt, kt0 = max(na, nb), m.kt0[it]
        nkt_of = (na, nb)

        def k_ready(kt):
            return ("wait", m.full[slot_of(m, 2 * kt)], 2 * kt // m.slots)

        def v_ready(kt):
            return ("wait", m.full[slot_of(m, 2 * kt + 1)], (2 * kt + 1) // m.slots)

        def issue_s(x, kt, item=it):
            sl = slot_of(m, 2 * kt)
            m.slot_readers[sl] += 1
            m.q_readers[x] += 1
            m.s_pending[x] += 1

            def run():
                m.check(m.slot_tag[sl] == ("K", kt),
                        f"S({x},{kt}) read slot {sl} = {m.slot_tag[sl]}")
                m.check(len(m.q_written[x].get(item, ())) == 4,
                        f"S({x},{kt}) read Q before it landed")
                m.check(m.pv_pending[x] == 0, f"S({x},{kt}) overwrote P that a P V still reads")
                m.s_tag[x] = (item, kt)
                m.p_written[x] = [set(), set()]
                m.slot_readers[sl] -= 1
                m.q_readers[x] -= 1
                m.s_pending[x] -= 1
            m.issue(f"S{x}", run)
            m.commit(m.s_full[x])

        def issue_pv(x, kt, hh, first, item=it):
            sl = slot_of(m, 2 * kt + 1)
            m.slot_readers[sl] += 1
            m.pv_pending[x] += 1

            def run():
                m.check(m.slot_tag[sl] == ("V", kt),
                        f"PV({x},{kt}) read slot {sl} = {m.slot_tag[sl]}")
                m.check(m.s_tag[x] == (item, kt) and len(m.p_written[x][hh]) == 4,
                        f"PV({x},{kt},{hh}) read P before all four warps wrote it")
                if first and hh == 0:
                    m.check(m.o_owner[x] is None or m.o_reads[x] == 4,
                            f"PV({x},{kt}) overwrote O before the read-out")
                    m.o_owner[x], m.o_reads[x] = item, 0
                m.slot_readers[sl] -= 1
                m.pv_pending[x] -= 1
            m.issue(f"O{x}", run)
            if hh == 1:
                m.commit(m.o_full[x])

        yield k_ready(kt0)
        for x in range(2):
            if nkt_of[x] == 0:
                continue
            if m.mut != "no_q_full_wait":
                yield ("wait", m.q_full[x], nq[x])
            if n[x] > 0:
                yield ("wait", m.o_full[x], n[x] - 1)
            nq[x] += 1
            issue_s(x, kt0)
        m.commit(m.empty[slot_of(m, 2 * kt0)])
        for j in range(nkt):
            kt = kt0 + j
            yield v_ready(kt)
            for x in range(2):
                if j >= nkt_of[x]:
                    continue
                half = 0 if m.mut == "test_first_half" else 1
                both = m.p_half[x][half].done(n[x])
                for hh in range(2):
                    if not both:
                        yield ("wait", m.p_half[x][hh], n[x])
                    issue_pv(x, kt, hh, j == 0)
                    yield ("step",)
                n[x] += 1
                if j + 1 >= nkt_of[x]:
                    continue
                yield k_ready(kt + 1)
                if m.mut != "no_o_full_wait":
                    yield ("wait", m.o_full[x], n[x] - 1)
                issue_s(x, kt + 1)
            m.commit(m.empty[slot_of(m, 2 * kt + 1)])
            if j + 1 < nkt:
                m.commit(m.empty[slot_of(m, 2 * kt + 2)])
    m.commit(m.drain)
    yield ("wait", m.drain, 0)


def softmax_warp(m, x, w):
    n = 0
    preloaded = -1

    def write_q(item):
        m.check(m.q_readers[x] == 0, f"Q_{x} overwritten while an S MMA reads it")
        m.q_written[x].setdefault(item, set()).add(w)

    for it, (na, nb) in enumerate(m.items):
        my = (na, nb)[x]
        if my > 0 and preloaded != it:
            write_q(it)
            m.q_full[x].arrive()
        for j in range(my):
            kt = m.kt0[it] + j
            yield ("wait", m.s_full[x], n)
            if j > 0:
                yield ("wait", m.o_full[x], n - 1)
            m.check(m.s_tag[x] == (it, kt) and m.s_pending[x] == 0,
                    f"softmax {x}.{w} read S of {(it, kt)} but found {m.s_tag[x]}")
            if j > 0 and m.rng.random() < 0.5:  # the running max moved: O is rescaled
                m.check(m.pv_pending[x] == 0, f"O_{x} rescaled while a P V accumulates")
            for hh in range(2):
                m.p_written[x][hh].add(w)
                m.p_half[x][hh].arrive()
                yield ("step",)
            n += 1
        if my > 0:
            yield ("wait", m.o_full[x], n - 1)
            nxt = next((v for v in range(it + 1, len(m.items)) if m.items[v][x] > 0), None)
            if nxt is not None:
                write_q(nxt)  # the next item's Q comes in during the read-out
            m.check(m.pv_pending[x] == 0 and m.o_owner[x] == it,
                    f"O_{x} read out before its last P V")
            m.o_reads[x] += 1
            if nxt is not None:
                m.q_full[x].arrive()
                preloaded = nxt
            yield ("step",)


def run_once(items, slots, seed, mutation=None):
    rng = random.Random(seed)
    m = Model(items, slots, rng, mutation)
    m.kt0, acc = [], 0
    for na, nb in items:
        m.kt0.append(acc)
        acc += max(na, nb)
    agents = [load_warp(m), mma_warp(m)] + [softmax_warp(m, x, w) for x in range(2)
                                               for w in range(4)]
    waiting = [None] * len(agents)
    alive = [True] * len(agents)
    while True:
        choices = []
        for i, a in enumerate(agents):
            if alive[i] and (waiting[i] is None or waiting[i][0].done(waiting[i][1])):
                choices.append(("agent", i))
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
    items = []
    for _ in range(rng.randint(1, 4)):
        na = rng.randint(1, 5)
        nb = 0 if rng.random() < 0.2 else rng.randint(na, na + 1)
        items.append((na, nb))
    return items


@pytest.mark.parametrize("slots", [4, 8])
def test_prefill_protocol_holds_under_random_schedules(slots):
    rng = random.Random(1234 + slots)
    for s in range(400):
        run_once(random_items(rng), slots, seed=s)


@pytest.mark.parametrize("mutation", ["no_o_full_wait", "test_first_half", "no_empty_wait",
                                      "no_q_full_wait"])
def test_prefill_protocol_model_catches_a_dropped_wait(mutation):
    rng = random.Random(99)
    for s in range(400):
        try:
            run_once(random_items(rng), 4, seed=s, mutation=mutation)
        except Hazard:
            return
    pytest.fail(f"the model missed mutation {mutation}")
