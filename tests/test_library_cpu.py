"""Host-side checks of libpkv (no GPU): the C ABI loads and exports every
declared symbol, arguments are rejected on the host before any launch, and the
C++ block allocator makes exactly the decisions of the oracle's reference
block manager."""
import ctypes
import os
import random
import re

import numpy as np
import torch
import pytest

import paged_kv_cache_312_gb300 as pkv
from oracle.blockmgr import BlockManager, OutOfBlocks

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built():
    from paged_kv_cache_312_gb300 import build
    build.build()


def declared_functions():
    names = []
    for fn in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if not fn.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", fn)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"^\s*[A-Za-z_][\w\s\*]*?\b(pkv_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_every_declared_symbol_is_exported():
    names = declared_functions()
    assert len(names) >= 20
    handle = ctypes.CDLL(pkv._binding.LIB_PATH)
    for n in names:
        assert hasattr(handle, n), n
    # and the binding knows each one's signature
    assert set(names) <= set(pkv._binding._SIGS)


def test_version_and_error_string():
    L = pkv.lib()
    assert L.pkv_version() == 100
    rc = L.pkv_set_decode_kernel(7)
    assert rc == -2
    assert b"unknown value" in L.pkv_last_error_string()


def _attn(L, **kw):
    a = dict(out=256, q=256, k=256, v=256, bt=256, cl=256, scale=0.1, B=16, Hkv=4, S=2, Hq=8, D=128,
             maxb=4, NB=10, kvdt=2, odt=0, P=0, ws=0, wsb=0)
    a.update(kw)
    P = ctypes.c_void_p
    return L.pkv_paged_decode_attention(P(a["out"]), P(a["q"]), P(a["k"]), P(a["v"]), P(a["bt"]),
                                        P(a["cl"]), a["scale"], a["B"], a["Hkv"], a["S"], a["Hq"],
                                        a["D"], a["maxb"], a["NB"], a["kvdt"], a["odt"], a["P"],
                                        P(a["ws"]), a["wsb"], P(0))


@pytest.mark.parametrize("kw,code", [
    (dict(D=96), -2), (dict(B=12), -2), (dict(Hq=6), -2), (dict(kvdt=5), -3),
    (dict(odt=9), -3), (dict(P=20), -2), (dict(P=32, ws=0), -8), (dict(maxb=0), -2),
    (dict(S=70000), -2), (dict(q=0), -1), (dict(k=8), -10), (dict(scale=float("nan")), -2),
])
def test_decode_rejects_bad_arguments_on_host(kw, code):
    assert _attn(pkv.lib(), **kw) == code


def test_prefill_rejects_bad_arguments_on_host():
    L = pkv.lib()
    P = ctypes.c_void_p

    def call(**kw):
        a = dict(kvdt=2, D=128, B=16, Hq=8, Hkv=2, S=2, maxq=5, q=256)
        a.update(kw)
        return L.pkv_paged_prefill_attention(P(256), P(a["q"]), P(256), P(256), P(256), P(256),
                                             P(256), 0.1, a["B"], a["Hkv"], a["S"], a["Hq"],
                                             a["D"], 4, 10, a["maxq"], a["kvdt"], 0, P(0))
    assert call(kvdt=0) == -4      # fp32 KV not supported
    assert call(D=96) == -2
    assert call(B=4) == -2
    assert call(Hq=7) == -2
    assert call(maxq=-1) == -2
    assert call(q=264) == -10
    assert call(S=0) == 0 and call(maxq=0) == 0


def test_decode_step_rejects_bad_arguments_on_host():
    L = pkv.lib()
    P = ctypes.c_void_p

    def call(**kw):
        a = dict(nk=256, nv=256, D=128, S=2, P=0)
        a.update(kw)
        return L.pkv_decode_step(P(256), P(256), P(a["nk"]), P(a["nv"]), P(256), P(256), P(256),
                                 P(256), 0.1, 16, 4, a["S"], 8, a["D"], 4, 10, 2, 0, a["P"],
                                 P(0), 0, P(0))
    assert call(nk=0) == -1        # new token K missing
    assert call(nv=0) == -1
    assert call(nk=264) == -10     # new_k not 16-byte aligned
    assert call(D=96) == -2        # the attention's own checks still apply
    assert call(P=32) == -8        # split mode without a workspace
    assert call(S=0, nk=0, nv=0) == 0


def test_selftest_rejects_bad_arguments_on_host():
    L = pkv.lib()
    P = ctypes.c_void_p
    assert L.pkv_selftest_bounded_wait(0, P(256), P(0)) == -2
    assert L.pkv_selftest_bounded_wait(70000, P(256), P(0)) == -2
    assert L.pkv_selftest_bounded_wait(4, P(0), P(0)) == -1


def test_decode_with_no_sequences_is_a_no_op():
    assert _attn(pkv.lib(), S=0, out=0, q=0) == 0


def test_workspace_size_formula():
    L = pkv.lib()
    # unsplit: the optional work plan alone (record count, one record per
    # (sequence, query head) at most)
    assert L.pkv_decode_workspace_bytes(8, 32, 128, 32768, 0) == 256 + 8 * 32 * 16
    assert L.pkv_decode_workspace_bytes(8, 32, 128, 32768, -1) == 0
    S, H, P, D = 8, 32, 64, 128
    a = lambda x: (x + 255) // 256 * 256  # noqa: E731
    # counters, (max, sum) and output per partition, the plan's record count
    # and its records (one per possible CTA)
    expect = a(S * H * 4) + a(S * H * P * 8) + a(S * H * P * D * 4) + 256 + S * H * P * 16
    assert L.pkv_decode_workspace_bytes(S, H, D, 32768, 512) == expect


def test_write_and_copy_reject_bad_arguments_on_host():
    L = pkv.lib()
    P = ctypes.c_void_p
    assert L.pkv_kv_write(P(16), P(16), P(16), P(16), P(8), 3, 4, 2, 12, 16, 2, P(0)) == -2
    assert L.pkv_kv_write(P(16), P(16), P(16), P(16), P(8), 3, 4, 2, 64, 16, 7, P(0)) == -3
    assert L.pkv_kv_write(P(16), P(16), P(0), P(16), P(8), 3, 4, 2, 64, 16, 2, P(0)) == -1
    assert L.pkv_kv_write(P(16), P(16), P(24), P(16), P(8), 3, 4, 2, 64, 16, 2, P(0)) == -10
    assert L.pkv_kv_write(P(0), P(0), P(0), P(0), P(0), 0, 4, 2, 64, 16, 2, P(0)) == 0
    assert L.pkv_kv_copy_blocks(P(16), P(16), P(0), 2, 4, 2, 64, 16, 2, P(0)) == -1
    assert L.pkv_kv_copy_blocks(P(0), P(0), P(0), 0, 4, 2, 64, 16, 2, P(0)) == 0


# --------------------------------------------------------------------------
# C++ allocator against the reference block manager
# --------------------------------------------------------------------------

def _same(cpp, ref, seqs):
    for s in seqs:
        assert cpp.table(s) == ref.table(s)
        assert cpp.length(s) == ref.length(s)
    for b in range(ref.num_blocks):
        assert cpp.refcount(b) == ref.refcount(b)
    assert cpp.num_free() == ref.num_free()
    assert cpp.stats() == ref.stats()


def test_allocator_worked_example():
    lengths = [37, 91, 128, 201, 511]
    for B, expect in ((16, 992), (32, 1024)):
        a = pkv.BlockAllocator(100, B)
        for s, n in enumerate(lengths):
            a.add(s, n)
        alloc, valid, used = a.stats()
        assert (alloc, valid, used * B) == (expect, 968, expect)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_allocator_matches_reference_on_random_operations(seed):
    rnd = random.Random(seed)
    NB, B = 48, 4
    order = list(np.random.default_rng(seed).permutation(NB))
    cpp, ref = pkv.BlockAllocator(NB, B, free_order=order), BlockManager(NB, B, free_order=order)
    live, nid = [], 0
    for _ in range(1500):
        op = rnd.random()
        if op < 0.15 or not live:
            n = rnd.randint(0, 10)
            try:
                ref.add(nid, n)
            except OutOfBlocks:
                with pytest.raises(pkv.OutOfBlocks):
                    cpp.add(nid, n)
            else:
                cpp.add(nid, n)
                live.append(nid)
            nid += 1
        elif op < 0.5:
            s = rnd.choice(live)
            try:
                r = ref.append(s)
            except OutOfBlocks:
                with pytest.raises(pkv.OutOfBlocks):
                    cpp.append(s)
            else:
                assert cpp.append(s) == r
        elif op < 0.65:
            s = rnd.choice(live)
            ref.fork(s, nid)
            cpp.fork(s, nid)
            live.append(nid)
            nid += 1
        elif op < 0.85:
            seqs = [rnd.choice(live) for _ in range(rnd.randint(1, 6))]
            try:
                slots, pairs = ref.step_append(seqs)
            except OutOfBlocks:
                with pytest.raises(pkv.OutOfBlocks):
                    cpp.step_append(seqs)
            else:
                cs, cp = cpp.step_append(seqs)
                assert cs.tolist() == slots
                assert [tuple(p) for p in cp.tolist()] == pairs
        else:
            s = live.pop(rnd.randrange(len(live)))
            ref.free_seq(s)
            cpp.free(s)
        _same(cpp, ref, live)


@pytest.mark.parametrize("seed", [0, 1])
def test_swap_matches_reference_between_two_pools(seed):
    rnd = random.Random(100 + seed)
    B = 4
    cg, rg = pkv.BlockAllocator(24, B), BlockManager(24, B)
    cc, rc = pkv.BlockAllocator(10, B), BlockManager(10, B)
    where = {}  # seq -> "gpu" | "cpu"
    nid = 0
    for _ in range(800):
        op = rnd.random()
        on_gpu = [s for s, w in where.items() if w == "gpu"]
        on_cpu = [s for s, w in where.items() if w == "cpu"]
        if op < 0.2 or not where:
            n = rnd.randint(0, 9)
            try:
                rg.add(nid, n)
            except OutOfBlocks:
                with pytest.raises(pkv.OutOfBlocks):
                    cg.add(nid, n)
            else:
                cg.add(nid, n)
                where[nid] = "gpu"
            nid += 1
        elif op < 0.45 and on_gpu:
            s = rnd.choice(on_gpu)
            try:
                r = rg.append(s)
            except OutOfBlocks:
                with pytest.raises(pkv.OutOfBlocks):
                    cg.append(s)
            else:
                assert cg.append(s) == r
        elif op < 0.55 and on_gpu:
            s = rnd.choice(on_gpu)
            rg.fork(s, nid)
            cg.fork(s, nid)
            where[nid] = "gpu"
            nid += 1
        elif op < 0.75 and (on_gpu or on_cpu):
            s = rnd.choice(on_gpu + on_cpu)
            src_r, dst_r, src_c, dst_c = (rg, rc, cg, cc) if where[s] == "gpu" else (rc, rg, cc, cg)
            try:
                pairs = src_r.swap_to(dst_r, s)
            except OutOfBlocks:
                with pytest.raises(pkv.OutOfBlocks):
                    src_c.swap_to(dst_c, s)
            else:
                got = src_c.swap_to(dst_c, s)
                assert [tuple(p) for p in got.tolist()] == pairs
                where[s] = "cpu" if where[s] == "gpu" else "gpu"
        else:
            s = rnd.choice(list(where))
            (rg if where[s] == "gpu" else rc).free_seq(s)
            (cg if where[s] == "gpu" else cc).free(s)
            del where[s]
        _same(cg, rg, [s for s, w in where.items() if w == "gpu"])
        _same(cc, rc, [s for s, w in where.items() if w == "cpu"])
    with pytest.raises(pkv.PkvError):
        cg.swap_to(cg, next(iter(where)) if where else 0)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_prefix_cache_matches_reference(seed):
    rnd = random.Random(200 + seed)
    B = 4
    order = list(np.random.default_rng(seed).permutation(40))
    cpp, ref = pkv.BlockAllocator(40, B, free_order=order), BlockManager(40, B, free_order=order)
    templates = [[rnd.randrange(50) for _ in range(rnd.randint(4, 17))] for _ in range(3)]
    toks = {}
    nid = 0
    for _ in range(1200):
        op = rnd.random()
        live = list(toks)
        if op < 0.3 or not live:
            prompt = rnd.choice(templates)[:rnd.randint(0, 17)] + \
                [rnd.randrange(50) for _ in range(rnd.randint(0, 5))]
            try:
                r = ref.add_cached(nid, prompt)
            except OutOfBlocks:
                with pytest.raises(pkv.OutOfBlocks):
                    cpp.add_cached(nid, prompt)
            else:
                assert cpp.add_cached(nid, prompt) == r
                toks[nid] = list(prompt)
            nid += 1
        elif op < 0.5:
            s = rnd.choice(live)
            n = rnd.randint(0, len(toks[s]))
            assert cpp.register_blocks(s, toks[s][:n]) == ref.register_blocks(s, toks[s][:n])
        elif op < 0.7:
            s = rnd.choice(live)
            try:
                r = ref.append(s)
            except OutOfBlocks:
                with pytest.raises(pkv.OutOfBlocks):
                    cpp.append(s)
            else:
                assert cpp.append(s) == r
                toks[s].append(rnd.randrange(50))
        elif op < 0.78:
            s = rnd.choice(live)
            ref.fork(s, nid)
            cpp.fork(s, nid)
            toks[nid] = list(toks[s])
            nid += 1
        else:
            s = live[rnd.randrange(len(live))]
            ref.free_seq(s)
            cpp.free(s)
            del toks[s]
        _same(cpp, ref, list(toks))
        assert cpp.prefix_cache_stats() == ref.prefix_cache_stats()
        ref.check_invariants()


def test_allocator_errors_leave_state_unchanged():
    a = pkv.BlockAllocator(3, 4)
    a.add(0, 8)
    snap = (a.table(0), a.num_free(), a.stats())
    with pytest.raises(pkv.OutOfBlocks):
        a.add(1, 9)
    with pytest.raises(pkv.PkvError):
        a.add(0, 1)  # exists
    with pytest.raises(pkv.PkvError):
        a.fork(5, 6)  # unknown parent
    with pytest.raises(pkv.PkvError):
        a.free(9)
    assert (a.table(0), a.num_free(), a.stats()) == snap
    with pytest.raises(pkv.PkvError):
        pkv.BlockAllocator(3, 4, free_order=[0, 0, 1])


def test_allocator_dense_tables():
    a = pkv.BlockAllocator(10, 4, free_order=[9, 8, 7, 6, 5, 4, 3, 2, 1, 0])
    a.add(1, 5)
    a.add(2, 0)
    t, l = a.dense_tables([1, 2], 3)
    assert t.tolist() == [[9, 8, -1], [-1, -1, -1]] and l.tolist() == [5, 0]
    with pytest.raises(pkv.PkvError):
        a.dense_tables([1], 1)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_step_append_tables_keeps_dense_tables_equal_to_the_reference(seed):
    # A batch stepped 60 times with the in-place table patching (half of it
    # forked from the other half first, so that shared partial blocks are
    # copied): after every step the patched tables and lengths equal the
    # reference block manager's dense tables, and slots / copy pairs its
    # decisions.
    from workloads import dense_tables
    rnd = random.Random(seed)
    NB, B, W = 400, 4, 6
    order = list(np.random.default_rng(seed).permutation(NB))
    cpp, ref = pkv.BlockAllocator(NB, B, free_order=order), BlockManager(NB, B, free_order=order)
    for s in range(W // 2):
        n = rnd.randint(0, 9)
        cpp.add(s, n)
        ref.add(s, n)
    for s in range(W // 2, W):
        cpp.fork(s - W // 2, s)
        ref.fork(s - W // 2, s)
    batch, maxb = list(range(W)), 40
    seqs = torch.tensor(batch, dtype=torch.int64)
    tables, lens = cpp.dense_tables(batch, maxb)
    slots = torch.empty(W, dtype=torch.int64)
    pairs = torch.empty((W, 2), dtype=torch.int64)
    copies = 0
    for _ in range(60):
        ns = cpp.step_append_tables(seqs, slots, pairs, tables, lens)
        r_slots, r_pairs = ref.step_append(batch)
        copies += ns
        assert slots.tolist() == r_slots
        assert [tuple(p) for p in pairs[:ns].tolist()] == r_pairs
        t_ref, l_ref = dense_tables(ref, batch, maxb)
        assert torch.equal(tables, t_ref) and torch.equal(lens, l_ref)
    assert cpp.stats() == ref.stats()


def test_step_append_tables_with_forks_and_errors():
    from workloads import dense_tables
    rnd = random.Random(7)
    NB, B, W = 300, 4, 5
    order = list(np.random.default_rng(7).permutation(NB))
    cpp, ref = pkv.BlockAllocator(NB, B, free_order=order), BlockManager(NB, B, free_order=order)
    for s in range(W):
        cpp.add(s, 6)
        ref.add(s, 6)
    batch, nid, maxb = list(range(W)), W, 30
    for rnd_sel in range(5):
        # beam re-selection: new beam b forks old beam parent[b]; old beams freed
        parent = [rnd.randrange(W) for _ in range(W)]
        new = list(range(nid, nid + W))
        for b in range(W):
            cpp.fork(batch[parent[b]], new[b])
            ref.fork(batch[parent[b]], new[b])
        for s in batch:
            cpp.free(s)
            ref.free_seq(s)
        batch, nid = new, nid + W
        seqs = torch.tensor(batch, dtype=torch.int64)
        tables, lens = cpp.dense_tables(batch, maxb)
        slots = torch.empty(W, dtype=torch.int64)
        pairs = torch.empty((W, 2), dtype=torch.int64)
        for _ in range(rnd.randint(1, 6)):
            ns = cpp.step_append_tables(seqs, slots, pairs, tables, lens)
            r_slots, r_pairs = ref.step_append(batch)
            assert slots.tolist() == r_slots
            assert [tuple(p) for p in pairs[:ns].tolist()] == r_pairs
            t_ref, l_ref = dense_tables(ref, batch, maxb)
            assert torch.equal(tables, t_ref) and torch.equal(lens, l_ref)
    # a table that would outgrow its row, or a sequence listed twice: refused,
    # nothing changed
    a = pkv.BlockAllocator(20, 4)
    a.add(0, 8)
    a.add(1, 3)
    seqs = torch.tensor([0, 1], dtype=torch.int64)
    tables, lens = a.dense_tables([0, 1], 2)
    slots = torch.empty(2, dtype=torch.int64)
    pairs = torch.empty((2, 2), dtype=torch.int64)
    snap = (a.table(0), a.table(1), a.num_free(), tables.clone(), lens.clone())
    with pytest.raises(pkv.PkvError) as ei:
        a.step_append_tables(seqs, slots, pairs, tables, lens)
    assert ei.value.code == -2
    with pytest.raises(pkv.PkvError) as ei:
        a.step_append_tables(torch.tensor([1, 1], dtype=torch.int64), slots, pairs,
                             tables, lens)
    assert ei.value.code == -9
    assert (a.table(0), a.table(1), a.num_free()) == snap[:3]
    assert torch.equal(tables, snap[3]) and torch.equal(lens, snap[4])


def test_prepared_step_append_tables_matches_the_reference_across_steps():
    # One prepared step, reused over many steps while the batch's contents
    # change in place (beams forked, sequence ids rewritten), gives the
    # reference's slots, copy-on-write pairs, tables and lengths; it keeps
    # its allocator alive.
    from workloads import dense_tables
    rnd = random.Random(11)
    NB, B, W, maxb = 400, 4, 6, 40
    order = list(np.random.default_rng(11).permutation(NB))
    cpp, ref = pkv.BlockAllocator(NB, B, free_order=order), BlockManager(NB, B, free_order=order)
    for s in range(W):
        cpp.add(s, 5 + s)
        ref.add(s, 5 + s)
    batch, nid = list(range(W)), W
    seqs = torch.tensor(batch, dtype=torch.int64)
    tables, lens = cpp.dense_tables(batch, maxb)
    slots = torch.empty(W, dtype=torch.int64)
    pairs = torch.empty((W, 2), dtype=torch.int64)
    step = cpp.prepare_step_append_tables(seqs, slots, pairs, tables, lens)
    del cpp  # the prepared step holds the allocator
    a = step.buffers[0]
    for _ in range(4):
        for _ in range(rnd.randint(1, 5)):
            ns = step()
            r_slots, r_pairs = ref.step_append(batch)
            assert slots.tolist() == r_slots
            assert [tuple(p) for p in pairs[:ns].tolist()] == r_pairs
            t_ref, l_ref = dense_tables(ref, batch, maxb)
            assert torch.equal(tables, t_ref) and torch.equal(lens, l_ref)
        # re-select beams: new ids into the same buffers, tables rewritten in place
        parent = [rnd.randrange(W) for _ in range(W)]
        new = list(range(nid, nid + W))
        for b in range(W):
            a.fork(batch[parent[b]], new[b])
            ref.fork(batch[parent[b]], new[b])
        for s in batch:
            a.free(s)
            ref.free_seq(s)
        batch, nid = new, nid + W
        seqs.copy_(torch.tensor(batch, dtype=torch.int64))
        t_new, l_new = a.dense_tables(batch, maxb)
        tables.copy_(t_new)
        lens.copy_(l_new)


def test_beam_fork_cow_pairs():
    # A width-4 beam over one partial block: three children copy, the last
    # holder writes in place.
    a = pkv.BlockAllocator(16, 4)
    a.add(0, 6)
    for c in (1, 2, 3):
        a.fork(0, c)
    last = a.table(0)[-1]
    assert a.refcount(last) == 4
    slots, pairs = a.step_append([0, 1, 2, 3])
    assert [p[0] for p in pairs.tolist()] == [last, last, last]
    assert a.refcount(last) == 1 and a.table(3)[-1] == last
    assert len(set(slots.tolist())) == 4


def test_grouped_decode_rejects_bad_arguments_on_host():
    L = pkv.lib()
    P = ctypes.c_void_p

    def call(**kw):
        a = dict(nk=256, nv=256, gs=256, G=1, kv=2, Hq=8, Hkv=4, S=2, parts=1, ws=0, wsb=0, mm=0)
        a.update(kw)
        return L.pkv_paged_decode_grouped(P(256), P(256), P(a["nk"]), P(a["nv"]), P(256), P(256),
                                          P(256), P(256), P(a["gs"]), P(256), a["G"], a["mm"],
                                          0.1, 16, a["Hkv"], a["S"], a["Hq"], 128, 4, 10, a["kv"],
                                          0, a["parts"], P(a["ws"]), a["wsb"], P(0))
    need = L.pkv_decode_workspace_bytes(2, 8, 128, 4, 1)
    assert call(gs=0) == -1          # no group table
    assert call(nv=0) == -1          # new_k without new_v
    assert call(G=0) == -2           # fewer than one group
    assert call(G=3) == -2           # more groups than sequences
    assert call(kv=0) == -4          # fp32 KV has no tensor-core path
    assert call(Hq=68) == -4         # 17 query heads per KV head
    assert call(mm=-1) == -2         # a negative member bound
    assert call(nk=0, nv=0, G=0) == -2  # attention only: same group checks
    assert call(parts=65) == -2      # more parts than the kernel takes
    assert call(G=65535, S=65535, Hq=65535, Hkv=65535) == -2  # 2^32 work items
    assert call(parts=4) == -8       # parts need a workspace ...
    assert call(parts=4, ws=256, wsb=need - 1) == -8  # ... of the stated size
    assert call(parts=4, ws=512 + 16, wsb=need) == -10  # ... 256-byte aligned


def _shared_reference(bt, cl, gs, B):
    out = []
    for i in range(len(gs) - 1):
        mem = list(range(gs[i], gs[i + 1]))
        lim = min(cl[s] for s in mem)
        n = 0
        while n < bt.shape[1] and n * B < lim and bt[mem[0], n] >= 0 and \
                all(bt[s, n] == bt[mem[0], n] for s in mem):
            n += 1
        out.append(max(0, min(lim, n * B)))
    return out


def test_group_shared_tokens_against_a_reference():
    rng = np.random.default_rng(5)
    for trial in range(200):
        B = int(rng.choice([8, 16, 32]))
        S = int(rng.integers(1, 12))
        mb = int(rng.integers(1, 10))
        bt = rng.integers(-1, 6, size=(S, mb)).astype(np.int32)
        # groups: consecutive runs; copy a random prefix of the first member's row
        cuts = sorted(set(rng.integers(1, S + 1, size=int(rng.integers(0, 4))).tolist()) | {S})
        gs = [0] + cuts
        for i in range(len(gs) - 1):
            k = int(rng.integers(0, mb + 1))
            for s in range(gs[i] + 1, gs[i + 1]):
                bt[s, :k] = bt[gs[i], :k]
        cl = rng.integers(0, mb * B + 1, size=S).astype(np.int32)
        got = pkv.group_shared_tokens(torch.from_numpy(bt), torch.from_numpy(cl),
                                      torch.tensor(gs, dtype=torch.int32), B)
        assert got.tolist() == _shared_reference(bt, cl, gs, B), (bt, cl, gs, B)
    # the prepared form, reused while the tables change in place, agrees
    rng = np.random.default_rng(6)
    S, mb, B = 8, 6, 16
    bt_t = torch.zeros((S, mb), dtype=torch.int32)
    cl_t = torch.zeros(S, dtype=torch.int32)
    gs_t = torch.tensor([0, 3, 5, 8], dtype=torch.int32)
    out_t = torch.full((3,), -1, dtype=torch.int32)
    step = pkv.prepare_group_shared_tokens(bt_t, cl_t, gs_t, B, out_t)
    for trial in range(50):
        bt = rng.integers(-1, 6, size=(S, mb)).astype(np.int32)
        gs = gs_t.tolist()
        for i in range(len(gs) - 1):
            k = int(rng.integers(0, mb + 1))
            for s in range(gs[i] + 1, gs[i + 1]):
                bt[s, :k] = bt[gs[i], :k]
        cl = rng.integers(0, mb * B + 1, size=S).astype(np.int32)
        bt_t.copy_(torch.from_numpy(bt))
        cl_t.copy_(torch.from_numpy(cl))
        assert step() is out_t
        assert out_t.tolist() == _shared_reference(bt, cl, gs, B)
    with pytest.raises(ValueError):  # buffers must be int32
        pkv.prepare_group_shared_tokens(bt_t.to(torch.int64), cl_t, gs_t, B, out_t)
    with pytest.raises(pkv.PkvError):  # a group past the last sequence
        pkv.group_shared_tokens(torch.zeros(2, 3, dtype=torch.int32),
                                torch.ones(2, dtype=torch.int32),
                                torch.tensor([0, 3], dtype=torch.int32), 16)
