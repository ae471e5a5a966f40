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
    q: torch.Tensor              # [S, Hq, D]
    k_cache: torch.Tensor        # [NB, Hkv, B, D]
    v_cache: torch.Tensor
    block_tables: torch.Tensor   # int32 [S, max_blocks], unused entries -1
    context_lens: torch.Tensor   # int32 [S]
    new_key: torch.Tensor | None = None    # [S, Hkv, D] token written this step
    new_value: torch.Tensor | None = None
    pool_order: np.ndarray | None = None   # physical ids in hand-out order

    @property
    def num_blocks(self) -> int:
        return self.k_cache.shape[0]


def make_decode_case(w: Workload, seed: int = 0, lengths=None, max_blocks=None,
                     poison: bool = True, num_seqs=None) -> DecodeCase:
    """Random paged cache for workload w.

    Sequences receive physical blocks from a seeded shuffle of the pool, in
    sequence order.  When the workload writes a new token each step, the
    token at position context_len - 1 is drawn as new_key/new_value and its
    cache slot is left poisoned: the step's write must fill it.
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
    NB = w.pool_blocks if w.pool_blocks else max(1, math.ceil(1.25 * total))
    if NB < total:
        raise ValueError("pool too small")
    maxb = max_blocks if max_blocks is not None else max(1, max(need, default=1))
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
    if poison:
        valid = np.zeros((NB, B), dtype=bool)
        for s in range(S):
            n = int(lengths[s]) - (1 if w.writes_new_token else 0)
            for i in range(need[s]):
                valid[tables[s, i], :max(0, min(B, n - i * B))] = True
        bad = torch.from_numpy(~valid)[:, None, :, None].expand(NB, Hkv, B, D)
        k_cache[bad] = float("nan")
        v_cache[bad] = float("nan")
    return DecodeCase(w, q, k_cache, v_cache, torch.from_numpy(tables),
                      torch.from_numpy(lengths.astype(np.int32)), new_key, new_value,
                      order)


def beam_parents(rng: np.random.Generator, groups: int, width: int) -> np.ndarray:
    """Seeded beam re-selection: each beam of each group picks a parent beam of
    the same group uniformly at random.  Returns [groups, width]."""
    return rng.integers(0, width, size=(groups, width), dtype=np.int64)
