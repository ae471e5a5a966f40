"""Reference block manager (TEST INFRASTRUCTURE): a plain Python model of the
host-side bookkeeping of paged KV memory.

It restates, in the simplest data structures, what the pages describe:

* KV memory is a pool of fixed-size physical blocks of B token positions; a
  sequence keeps a block table mapping its i-th logical block to a physical
  block (aiplusplus page, "core idea" items 1-3).
* Blocks are allocated on demand: a sequence gets blocks for its prompt on
  arrival and one more each time a new token starts a fresh block; any free
  block will do (same page, item 4 and "effects"; lain42 page, "on-demand
  allocation").
* Finished sequences return their blocks at once (aiplusplus page,
  "continuous batching").
* Several block tables may point at one physical block; a reference count
  tracks them, and a branch that writes into a shared block that is not full
  first copies it (copy-on-write) so branches do not overwrite one another
  (auturnal guide section 3; aiplusplus "key techniques" 3; the cayang0802
  page's beam-search example with width 4).

Free-list policy (the pages leave it open): a stack.  The pool starts with
blocks handed out in ``free_order`` (identity if not given); a block whose
count drops to zero is pushed on top and is the next one handed out.  A
sequence releases its blocks from its last logical block to its first.

Automatic prefix caching (cayang0802 walkthrough, prefix caching): a full
block is keyed by a hash of its own tokens and of every token before it; a new
sequence reuses the cached blocks of its longest matching prefix.  The key is
FNV-1a 64-bit (Fowler-Noll-Vo: offset basis 14695981039346656037, prime
1099511628211) over the parent block's key as 8 little-endian bytes (0 for the
first block) followed by the block's token ids as 4 little-endian bytes each;
a hit also compares the stored parent key and tokens.  A registered block
whose count drops to zero stays findable in a least-recently-freed list and is
handed out again (and forgotten) only when the plain free stack is empty.

An operation that runs out of blocks raises ``OutOfBlocks`` and leaves the
state exactly as it was (auturnal guide section 6: OOM must be tested).
"""
from __future__ import annotations

import copy
from collections import OrderedDict

FNV_OFFSET = 14695981039346656037
FNV_PRIME = 1099511628211


def fnv1a64(data: bytes) -> int:
    """FNV-1a, 64-bit: for each byte, xor it in, then multiply by the prime."""
    h = FNV_OFFSET
    for byte in data:
        h = ((h ^ byte) * FNV_PRIME) & 0xFFFFFFFFFFFFFFFF
    return h


def block_key(parent: int, tokens) -> int:
    """FNV-1a over parent (8 bytes LE) and the token ids (4 bytes LE each)."""
    return fnv1a64(parent.to_bytes(8, "little") + b"".join(
        (int(t) & 0xFFFFFFFF).to_bytes(4, "little") for t in tokens))


class OutOfBlocks(Exception):
    pass


class BlockManager:
    def __init__(self, num_blocks: int, block_size: int, free_order=None):
        if num_blocks < 0 or block_size <= 0:
            raise ValueError("bad pool shape")
        order = list(range(num_blocks)) if free_order is None else [int(b) for b in free_order]
        if sorted(order) != list(range(num_blocks)):
            raise ValueError("free_order must be a permutation of the pool")
        self.B = block_size
        self.num_blocks = num_blocks
        self.free = list(reversed(order))  # top of the stack is the end of the list
        self.ref = [0] * num_blocks
        self.tables: dict[int, list[int]] = {}
        self.lens: dict[int, int] = {}
        self.index: dict[int, int] = {}           # key -> block
        self.registered: dict[int, tuple] = {}    # block -> (key, parent key, tokens)
        self.cached: OrderedDict = OrderedDict()  # count-0 registered blocks, oldest first
        self.hits = 0

    # -- primitives ---------------------------------------------------------
    def _pop(self) -> int:
        if self.free:
            b = self.free.pop()
        elif self.cached:
            b, _ = self.cached.popitem(last=False)  # evict the oldest cached block
            self._unregister(b)
        else:
            raise OutOfBlocks()
        assert self.ref[b] == 0
        self.ref[b] = 1
        return b

    def _unregister(self, b: int) -> None:
        key = self.registered.pop(b)[0]
        if self.index.get(key) == b:
            del self.index[key]

    def _release(self, b: int) -> None:
        self.ref[b] -= 1
        assert self.ref[b] >= 0
        if self.ref[b] == 0:
            if b in self.registered:
                self.cached[b] = None
            else:
                self.free.append(b)

    def _atomic(self, fn):
        saved = (list(self.free), list(self.ref), copy.deepcopy(self.tables), dict(self.lens),
                 dict(self.index), dict(self.registered), OrderedDict(self.cached), self.hits)
        try:
            return fn()
        except OutOfBlocks:
            (self.free, self.ref, self.tables, self.lens, self.index, self.registered,
             self.cached, self.hits) = saved
            raise

    # -- public operations --------------------------------------------------
    def add(self, seq: int, prompt_len: int) -> None:
        """New sequence holding prompt_len tokens: ceil(n / B) fresh blocks."""
        if seq in self.tables:
            raise KeyError("sequence exists")
        if prompt_len < 0:
            raise ValueError("negative length")

        def go():
            n_blocks = -(-prompt_len // self.B)
            self.tables[seq] = [self._pop() for _ in range(n_blocks)]
            self.lens[seq] = prompt_len
        self._atomic(go)

    def _append_one(self, seq: int):
        table, p = self.tables[seq], self.lens[seq]
        cow = None
        if p % self.B == 0:
            table.append(self._pop())
        else:
            last = table[-1]
            if self.ref[last] > 1:
                dst = self._pop()
                self._release(last)
                table[-1] = dst
                cow = (last, dst)
        slot = table[p // self.B] * self.B + p % self.B
        self.lens[seq] = p + 1
        return slot, cow

    def append(self, seq: int):
        """Reserve the slot of the sequence's next token; returns (slot, cow)
        where cow is the (src, dst) block pair to copy first, or None."""
        if seq not in self.tables:
            raise KeyError("no such sequence")
        return self._atomic(lambda: self._append_one(seq))

    def step_append(self, seqs):
        """One decode step: append one token to each sequence, in order.
        All or nothing.  Returns (slots, cow_pairs)."""
        for s in seqs:
            if s not in self.tables:
                raise KeyError("no such sequence")

        def go():
            slots, pairs = [], []
            for s in seqs:
                slot, cow = self._append_one(s)
                slots.append(slot)
                if cow is not None:
                    pairs.append(cow)
            return slots, pairs
        return self._atomic(go)

    def fork(self, parent: int, child: int) -> None:
        """The child shares every block of the parent (each count + 1)."""
        if parent not in self.tables:
            raise KeyError("no such parent")
        if child in self.tables:
            raise KeyError("child exists")
        self.tables[child] = list(self.tables[parent])
        self.lens[child] = self.lens[parent]
        for b in self.tables[child]:
            self.ref[b] += 1

    def free_seq(self, seq: int) -> None:
        if seq not in self.tables:
            raise KeyError("no such sequence")
        for b in reversed(self.tables.pop(seq)):
            self._release(b)
        del self.lens[seq]

    def add_cached(self, seq: int, tokens) -> int:
        """New sequence for the prompt `tokens`, reusing the cached blocks of
        its longest prefix of full blocks found in the index; returns the
        number of reused tokens."""
        if seq in self.tables:
            raise KeyError("sequence exists")
        tokens = [int(t) for t in tokens]
        B, n = self.B, len(tokens)

        def go():
            hits, parent = [], 0
            for i in range(n // B):
                blk = tokens[i * B:(i + 1) * B]
                key = block_key(parent, blk)
                b = self.index.get(key)
                if b is None or self.registered[b][1:] != (parent, tuple(blk)):
                    break
                hits.append(b)
                parent = key
            revive = sum(1 for b in hits if self.ref[b] == 0)
            fresh = -(-n // B) - len(hits)
            if fresh > self.num_free() - revive:
                raise OutOfBlocks()
            table = []
            for b in hits:
                if self.ref[b] == 0:
                    del self.cached[b]
                self.ref[b] += 1
                table.append(b)
            table += [self._pop() for _ in range(fresh)]
            self.tables[seq] = table
            self.lens[seq] = n
            self.hits += len(hits)
            return len(hits) * B
        return self._atomic(go)

    def register_blocks(self, seq: int, tokens) -> int:
        """Index the full blocks covering `tokens` (a prefix of the sequence's
        tokens); returns the number of blocks added."""
        if seq not in self.tables:
            raise KeyError("no such sequence")
        tokens = [int(t) for t in tokens]
        if len(tokens) > self.lens[seq]:
            raise ValueError("more tokens than the sequence holds")
        B, parent, added = self.B, 0, 0
        for i in range(len(tokens) // B):
            blk = tuple(tokens[i * B:(i + 1) * B])
            key = block_key(parent, blk)
            b = self.tables[seq][i]
            if b not in self.registered and key not in self.index:
                self.index[key] = b
                self.registered[b] = (key, parent, blk)
                added += 1
            parent = key
        return added

    def prefix_cache_stats(self):
        return self.hits, len(self.index), len(self.cached)

    def swap_to(self, other: "BlockManager", seq: int):
        """Preemption by swapping (aiplusplus section 4; cayang0802
        walkthrough): move `seq` into the pool managed by `other`.  Takes one
        fresh block of `other` per block of the sequence, in table order, then
        releases the sequence here.  Returns the (this block, other block)
        pairs.  All or nothing."""
        if seq not in self.tables:
            raise KeyError("no such sequence")
        if seq in other.tables or other is self:
            raise KeyError("sequence exists in the target")
        if other.B != self.B:
            raise ValueError("block sizes differ")
        table = self.tables[seq]
        if len(table) > other.num_free():
            raise OutOfBlocks()
        moved = [other._pop() for _ in table]
        other.tables[seq] = moved
        other.lens[seq] = self.lens[seq]
        self.free_seq(seq)
        return list(zip(table, moved))

    # -- queries ------------------------------------------------------------
    def table(self, seq: int):
        return list(self.tables[seq])

    def length(self, seq: int) -> int:
        return self.lens[seq]

    def refcount(self, b: int) -> int:
        return self.ref[b]

    def num_free(self) -> int:
        return len(self.free) + len(self.cached)

    def stats(self):
        """(allocated positions = sum over sequences of B * blocks held,
        valid positions = sum of lengths, physical blocks in use)."""
        alloc = sum(self.B * len(t) for t in self.tables.values())
        valid = sum(self.lens.values())
        return alloc, valid, self.num_blocks - self.num_free()

    def check_invariants(self) -> None:
        """Counts match table membership; a free block is unreferenced; no
        block is both free and in a table; tables cover their lengths."""
        count = [0] * self.num_blocks
        for seq, t in self.tables.items():
            assert len(t) == -(-self.lens[seq] // self.B)
            for b in t:
                count[b] += 1
        assert count == self.ref
        free = set(self.free)
        assert len(free) == len(self.free)
        for b in range(self.num_blocks):
            assert (b in free or b in self.cached) == (self.ref[b] == 0)
            assert not (b in free and b in self.cached)
            if b in self.cached:
                assert b in self.registered
        for key, b in self.index.items():
            assert self.registered[b][0] == key
