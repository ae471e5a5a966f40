"""Seeded synthetic inputs for the paged decode path.

This module serves both the oracle and the CUDA path.  It holds none of the
method's arithmetic: it only draws lengths, shuffled physical block ids,
block-table contents and N(0, 1) values rounded to the storage dtype, with the
shapes and distributions of the five decode workloads below.  No public
dataset is involved; all values are synthetic.

Workloads (one transformer layer each):

1. fp32 MHA, 4 heads, head_dim 64, block 16, 5 sequences of 37/91/128/201/511
   tokens (the lengths of the auturnal guide's worked example), pool of 80
   blocks in seeded random order, scale 1/sqrt(64).
2. bf16 MHA, 32 heads, head_dim 128, block 16, 64 sequences, lengths uniform
   on [1, 2048]; each step writes one new token per sequence, then attends.
3. bf16 GQA 64 query / 8 KV heads, head_dim 128, block 16, 256 sequences,
   lengths floor(exp(N(6.3, 0.8))) clipped to [16, 4096].
4. bf16 GQA 32 / 8, head_dim 128, block 32, 8 sequences of 32768 tokens,
   split into 512-token partitions.
5. fp16 MHA, 40 heads, head_dim 128, block 16, 16 groups x 4 beams sharing a
   1024-token prefix per group, private suffixes uniform on [0, 256].

Values are drawn as float32 N(0, 1) by numpy's PCG64 and rounded to the
storage dtype by round-to-nearest-even.  Cache slots that no sequence reaches
(tail positions of last blocks, unreferenced blocks) are filled with NaN so
that a kernel reading them shows up in the results.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

DTYPES = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


@dataclass(frozen=True)
class Workload:
    key: int
    name: str
    dtype: str
    num_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_seqs: int
    lengths: str                 # how context lengths are drawn
    partition_size: int = 0      # 0: one pass per sequence
    writes_new_token: bool = False
    beam_groups: int = 0
    beam_width: int = 0
    prefix_len: int = 0
    fixed_lengths: tuple = field(default_factory=tuple)
    pool_blocks: int = 0         # 0: ceil(1.25 * blocks needed)

    @property
    def torch_dtype(self):
        return DTYPES[self.dtype]

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)


WORKLOADS = {
    1: Workload(1, "fp32-mha4-d64-b16-5seq", "f32", 4, 4, 64, 16, 5, "fixed",
                fixed_lengths=(37, 91, 128, 201, 511), pool_blocks=80),
    2: Workload(2, "bf16-mha32-d128-b16-64seq-u1-2048", "bf16", 32, 32, 128, 16, 64,
                "uniform:1:2048", writes_new_token=True),
    3: Workload(3, "bf16-gqa64x8-d128-b16-256seq-lognormal", "bf16", 64, 8, 128, 16, 256,
                "lognormal:6.3:0.8:16:4096"),
    4: Workload(4, "bf16-gqa32x8-d128-b32-8x32768-split512", "bf16", 32, 8, 128, 32, 8,
                "fixed", fixed_lengths=(32768,) * 8, partition_size=512),
    5: Workload(5, "fp16-mha40-d128-b16-beam16x4-prefix1024", "f16", 40, 40, 128, 16, 64,
                "beam", writes_new_token=True, beam_groups=16, beam_width=4,
                prefix_len=1024),
}


def draw_lengths(w: Workload, rng: np.random.Generator) -> np.ndarray:
    kind = w.lengths.split(":")
    if kind[0] == "fixed":
        return np.array(w.fixed_lengths, dtype=np.int64)
    if kind[0] == "uniform":
        lo, hi = int(kind[1]), int(kind[2])
        return rng.integers(lo, hi + 1, size=w.num_seqs, dtype=np.int64)
    if kind[0] == "lognormal":
        mu, sigma, lo, hi = float(kind[1]), float(kind[2]), int(kind[3]), int(kind[4])
        x = np.floor(np.exp(rng.normal(mu, sigma, size=w.num_seqs)))
        return np.clip(x, lo, hi).astype(np.int64)
    if kind[0] == "beam":
        suffix = rng.integers(0, 257, size=w.num_seqs, dtype=np.int64)
        return w.prefix_len + suffix
    raise ValueError(w.lengths)


def normal_values(rng: np.random.Generator, shape, dtype: torch.dtype) -> torch.Tensor:
    x = rng.standard_normal(size=shape, dtype=np.float32)
    return torch.from_numpy(x).to(dtype)


def blocks_for(length: int, block_size: int) -> int:
    """Number of table entries a sequence of `length` tokens occupies."""
    return -(-int(length) // block_size)


@dataclass
class DecodeCase:
    """Inputs of one decode step, all on the host."""
    workload: Workload
    lengths: np.ndarray          # context length per sequence (new token included)
    q: torch.Tensor              # [S, Hq, D]
    k_cache: torch.Tensor        # [NB, Hkv, B, D]
    v_cache: torch.Tensor
    block_tables: torch.Tensor   # int32 [S, max_blocks]: sequential pagination, -1 unused
    context_lens: torch.Tensor   # int32 [S]
    pool_order: np.ndarray       # physical ids in hand-out order
    new_key: torch.Tensor | None = None    # [S, Hkv, D] token written this step
    new_value: torch.Tensor | None = None

    @property
    def num_blocks(self) -> int:
        return self.k_cache.shape[0]


def make_decode_case(w: Workload, seed: int = 0, lengths=None, num_seqs=None,
                     poison: bool = True, pool_blocks=None) -> DecodeCase:
    """Random paged cache for workload w.

    block_tables hands out the shuffled pool in sequence order (sequence s
    takes the next blocks_for(L_s) ids).  Workloads that write a new token
    each step draw it as new_key/new_value; callers that build their tables
    through a block allocator instead should poison with `poison_unused`.
    """
    rng = np.random.default_rng(seed)
    if lengths is None:
        lengths = draw_lengths(w, rng)
        if num_seqs is not None:
            lengths = lengths[:num_seqs]
    lengths = np.asarray(lengths, dtype=np.int64)
    S = len(lengths)
    B, Hkv, D, Hq = w.block_size, w.num_kv_heads, w.head_dim, w.num_heads
    need = [blocks_for(n, B) for n in lengths]
    total = int(sum(need))
    NB = pool_blocks or w.pool_blocks or max(1, math.ceil(1.25 * total))
    if NB < total:
        raise ValueError("pool too small")
    maxb = max(1, max(need, default=1))
    order = rng.permutation(NB)
    tables = np.full((S, maxb), -1, dtype=np.int32)
    cur = 0
    for s in range(S):
        tables[s, :need[s]] = order[cur:cur + need[s]]
        cur += need[s]

    dt = w.torch_dtype
    k_cache = normal_values(rng, (NB, Hkv, B, D), dt)
    v_cache = normal_values(rng, (NB, Hkv, B, D), dt)
    q = normal_values(rng, (S, Hq, D), dt)
    new_key = new_value = None
    if w.writes_new_token:
        new_key = normal_values(rng, (S, Hkv, D), dt)
        new_value = normal_values(rng, (S, Hkv, D), dt)
    tables_t = torch.from_numpy(tables)
    if poison:
        filled = lengths - (1 if w.writes_new_token else 0)
        poison_unused(k_cache, v_cache, tables_t, filled)
    return DecodeCase(w, lengths, q, k_cache, v_cache, tables_t,
                      torch.from_numpy(lengths.astype(np.int32)), order, new_key, new_value)


def poison_unused(k_cache: torch.Tensor, v_cache: torch.Tensor, tables, filled) -> None:
    """NaN into every cache slot that does not hold one of the first filled[s]
    tokens of some sequence s (tables: [S, max_blocks], -1 = unused)."""
    NB, _, B, _ = k_cache.shape
    valid = np.zeros((NB, B), dtype=bool)
    tables = np.asarray(tables)
    for s in range(tables.shape[0]):
        n = int(filled[s])
        for i in range(blocks_for(n, B)):
            valid[tables[s, i], :min(B, n - i * B)] = True
    bad = torch.from_numpy(~valid)[:, None, :, None]
    k_cache.masked_fill_(bad, float("nan"))
    v_cache.masked_fill_(bad, float("nan"))


def dense_tables(manager, seqs, max_blocks=None):
    """int32 [n, max_blocks] tables (-1 unused) and int32 lengths read from a
    block manager exposing table(seq) and length(seq)."""
    rows = [manager.table(s) for s in seqs]
    mb = max_blocks or max(1, max(len(r) for r in rows))
    t = torch.full((len(rows), mb), -1, dtype=torch.int32)
    for i, r in enumerate(rows):
        if r:
            t[i, :len(r)] = torch.tensor(r, dtype=torch.int32)
    lens = torch.tensor([manager.length(s) for s in seqs], dtype=torch.int32)
    return t, lens


def write_step_schedule(manager, lengths):
    """Drive a block manager to the state of a decode step in which sequence
    s already holds lengths[s] - 1 tokens and one more is appended for each
    sequence.  Returns (slots int64 [S], cow pairs, tables, lens)."""
    S = len(lengths)
    for s in range(S):
        manager.add(s, int(lengths[s]) - 1)
    slots, pairs = manager.step_append(list(range(S)))
    tables, lens = dense_tables(manager, range(S))
    return (torch.as_tensor(slots, dtype=torch.int64).reshape(-1),
            torch.as_tensor(pairs, dtype=torch.int64).reshape(-1, 2), tables, lens)


def beam_parents(rng: np.random.Generator, groups: int, width: int) -> np.ndarray:
    """Seeded beam re-selection: each beam of each group picks a parent beam of
    the same group uniformly at random.  Returns [groups, width]."""
    return rng.integers(0, width, size=(groups, width), dtype=np.int64)


@dataclass
class BeamCase:
    """Beam-search workload: per group a shared prompt, per beam a private
    suffix, then one decode step after a seeded re-selection of parents."""
    workload: Workload
    suffix: np.ndarray           # [groups * width] suffix lengths
    parents: np.ndarray          # [groups, width] parent beam of each new beam
    prefix_k: torch.Tensor       # [groups, prefix, Hkv, D]
    prefix_v: torch.Tensor
    suffix_k: list               # per beam [suffix, Hkv, D]
    suffix_v: list
    q: torch.Tensor              # [groups * width, Hq, D]
    new_key: torch.Tensor        # [groups * width, Hkv, D]
    new_value: torch.Tensor
    pool_blocks: int
    pool_order: np.ndarray


def make_beam_case(w: Workload, seed: int = 0, groups=None, prefix_len=None) -> BeamCase:
    rng = np.random.default_rng(seed)
    G = groups or w.beam_groups
    W = w.beam_width
    P = w.prefix_len if prefix_len is None else prefix_len
    B, Hkv, D, Hq = w.block_size, w.num_kv_heads, w.head_dim, w.num_heads
    suffix = rng.integers(0, 257, size=G * W, dtype=np.int64)
    parents = beam_parents(rng, G, W)
    need = G * blocks_for(P, B) + sum(blocks_for(P + n + 1, B) - blocks_for(P, B) + 1
                                      for n in suffix)
    NB = max(1, math.ceil(1.25 * need))
    order = rng.permutation(NB)
    dt = w.torch_dtype
    prefix_k = normal_values(rng, (G, P, Hkv, D), dt)
    prefix_v = normal_values(rng, (G, P, Hkv, D), dt)
    suffix_k = [normal_values(rng, (int(n), Hkv, D), dt) for n in suffix]
    suffix_v = [normal_values(rng, (int(n), Hkv, D), dt) for n in suffix]
    q = normal_values(rng, (G * W, Hq, D), dt)
    new_key = normal_values(rng, (G * W, Hkv, D), dt)
    new_value = normal_values(rng, (G * W, Hkv, D), dt)
    return BeamCase(w, suffix, parents, prefix_k, prefix_v, suffix_k, suffix_v, q, new_key,
                    new_value, NB, order)


def beam_setup_schedule(manager, case: BeamCase):
    """Drive a block manager through the beam workload's history: each group's
    prompt is appended token by token to a root sequence, the root is forked
    into `width` beams (prompt blocks shared, count = width) and freed, and
    each beam appends its private suffix.  Returns the slots of the prompt
    tokens [groups, prefix] and of each beam's suffix tokens (list)."""
    G, W = case.parents.shape
    P = case.prefix_k.shape[1]
    roots = [10_000 + g for g in range(G)]
    for r in roots:
        manager.add(r, 0)
    prefix_slots = torch.empty((G, P), dtype=torch.int64)
    for p in range(P):
        slots, pairs = manager.step_append(roots)
        assert len(pairs) == 0
        prefix_slots[:, p] = torch.as_tensor(slots, dtype=torch.int64).reshape(-1)
    for g in range(G):
        for b in range(W):
            manager.fork(roots[g], g * W + b)
        manager.free_seq(roots[g])
    suffix_slots = [[] for _ in range(G * W)]
    remaining = [int(n) for n in case.suffix]
    while any(remaining):
        active = [i for i in range(G * W) if remaining[i] > 0]
        slots, pairs = manager.step_append(active)
        assert len(pairs) == 0
        for i, sl in zip(active, torch.as_tensor(slots).reshape(-1).tolist()):
            suffix_slots[i].append(sl)
            remaining[i] -= 1
    return prefix_slots, [torch.tensor(x, dtype=torch.int64) for x in suffix_slots]


def beam_step_schedule(manager, case: BeamCase):
    """Beam re-selection and one decode step: new beam b of group g is forked
    from old beam parents[g, b], the old beams are freed, and every new beam
    appends one token (a beam appending into a still-shared partial block
    gets a copy first).  Returns (new beam ids, slots, cow pairs, tables, lens)."""
    G, W = case.parents.shape
    new_ids = [20_000 + i for i in range(G * W)]
    for g in range(G):
        for b in range(W):
            manager.fork(g * W + int(case.parents[g, b]), new_ids[g * W + b])
    for i in range(G * W):
        manager.free_seq(i)
    slots, pairs = manager.step_append(new_ids)
    tables, lens = dense_tables(manager, new_ids)
    return (new_ids, torch.as_tensor(slots, dtype=torch.int64).reshape(-1),
            torch.as_tensor(pairs, dtype=torch.int64).reshape(-1, 2), tables, lens)
