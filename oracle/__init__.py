"""Paged-KV oracle (TEST INFRASTRUCTURE).

Plain, slow, obviously correct CPU restatement of what the PagedAttention
decode path computes, in float64.  Only ``tests/``, ``__graft_entry__.smoke``
and the CPU-baseline leg of ``bench.py`` may import it; the product package
never does, and the two share no code: the oracle widens stored bf16/fp16/fp32
values itself (oracle.c), indexes the cache with its own arithmetic and calls
nothing in ``paged_kv_cache_312_gb300``.

What each function follows (pages on "Efficient Memory Management for Large
Language Model Serving with PagedAttention", Kwon et al. 2023):

* ``paged_decode_attention`` -- aiplusplus page, "core idea" items 1-4 and
  "key techniques" 1 (block table lookup assembles scattered K/V blocks);
  auturnal guide section 1 (paging changes storage, not what attention reads)
  and its verification protocol (compare with a contiguous-KV baseline).
* ``paged_prefill_attention`` -- the same attention for several new query
  tokens per sequence, each causal over the sequence's tokens up to its own
  position (cayang0802 walkthrough, recomputation: a whole prompt's KV is
  produced in one parallel pass).
* ``kv_write`` -- cayang0802 page, KV-cache paragraph: only the new token's
  K and V are computed and stored; slot = block * B + offset (core idea 3).
* ``kv_copy_blocks`` -- auturnal guide section 3 and aiplusplus "key
  techniques" 3: a branch that must modify a shared, not-full block first
  gets a private copy (copy-on-write).
* ``kv_swap_blocks`` -- aiplusplus section 4 and the cayang0802 walkthrough
  (preemption by swapping): blocks move between the GPU pool and a CPU pool.
* ``kv_bytes`` / ``allocated_positions`` / ``tail_waste`` /
  ``position_utilisation`` -- auturnal guide Eq. (1), (2), (3).
* ``decode_partitions`` / ``lse_combine`` -- the split-context form: softmax
  over a union of disjoint token ranges rebuilt from per-range maxima, sums
  and unnormalised outputs (the pages are silent on splitting; this is the
  plain log-sum-exp identity).

Every function is pinned by tests/test_oracle_pins.py against values the pages
print, closed forms, library routines or brute force; none is "parity
unpinned".
"""
from __future__ import annotations

import ctypes
import math
import os

import numpy as np
import torch

from . import build as _build

__all__ = [
    "DTYPE_CODE", "paged_decode_attention", "paged_prefill_attention", "kv_write", "kv_copy_blocks",
    "kv_swap_blocks", "slot_for_position", "kv_bytes", "allocated_positions", "tail_waste",
    "position_utilisation", "fixed_reservation_positions", "gather_sequence",
    "decode_partitions", "lse_combine", "widen",
]

DTYPE_CODE = {torch.float32: 0, torch.float16: 1, torch.bfloat16: 2}

_lib = None


def _load():
    global _lib
    if _lib is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        P, I, I64, D = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_double
        lib.orc_widen.argtypes = [P, I, I64, P]
        lib.orc_kv_write.argtypes = [P, P, P, P, P, I, I, I, I, I, I]
        lib.orc_kv_copy_blocks.argtypes = [P, P, P, I, I, I, I, I, I]
        lib.orc_kv_swap_blocks.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I]
        lib.orc_paged_prefill_attention.argtypes = [
            P, P, P, P, I, P, P, P, D, I, I, I, I, I, I, I, I]
        lib.orc_paged_decode_attention.argtypes = [
            P, P, P, P, I, P, P, D, I, I, I, I, I, I, I, I]
        for f in (lib.orc_widen, lib.orc_kv_write, lib.orc_kv_copy_blocks,
                  lib.orc_kv_swap_blocks, lib.orc_paged_decode_attention,
                  lib.orc_paged_prefill_attention):
            f.restype = ctypes.c_int
        _lib = lib
    return _lib


def _cpu(t: torch.Tensor) -> torch.Tensor:
    if t.device.type != "cpu":
        raise ValueError("the oracle takes host tensors")
    return t.contiguous()


def widen(t: torch.Tensor) -> np.ndarray:
    """Stored f32/f16/bf16 values widened exactly to float64 (same shape)."""
    t = _cpu(t)
    out = np.empty(t.shape, dtype=np.float64)
    rc = _load().orc_widen(t.data_ptr(), DTYPE_CODE[t.dtype], t.numel(),
                           out.ctypes.data)
    if rc != 0:
        raise ValueError("orc_widen failed: %d" % rc)
    return out


def paged_decode_attention(q, k_cache, v_cache, block_tables, context_lens, scale,
                           block_size, num_kv_heads, nthreads=1) -> np.ndarray:
    """out[s, h, :] = softmax_i(scale * q[s,h] . k_i) v_i over the sequence's
    logical tokens i < context_lens[s], reached through block_tables[s].

    q: [S, Hq, D]; k_cache/v_cache: [NB, Hkv, B, D] (same dtype as q);
    block_tables: int32 [S, max_blocks]; context_lens: int32 [S].
    Returns float64 [S, Hq, D].
    """
    q, k_cache, v_cache = _cpu(q), _cpu(k_cache), _cpu(v_cache)
    bt = _cpu(block_tables).to(torch.int32)
    cl = _cpu(context_lens).to(torch.int32)
    S, Hq, D = q.shape
    NB = k_cache.shape[0]
    if k_cache.dtype != q.dtype or v_cache.dtype != q.dtype:
        raise ValueError("q, k_cache and v_cache must share a dtype")
    out = np.empty((S, Hq, D), dtype=np.float64)
    rc = _load().orc_paged_decode_attention(
        out.ctypes.data, q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
        DTYPE_CODE[q.dtype], bt.data_ptr(), cl.data_ptr(), float(scale),
        int(block_size), int(num_kv_heads), S, Hq, D, bt.shape[1], NB, int(nthreads))
    if rc != 0:
        raise ValueError("orc_paged_decode_attention failed: %d" % rc)
    return out


def paged_prefill_attention(q, k_cache, v_cache, block_tables, context_lens, query_start,
                            scale, block_size, num_kv_heads, nthreads=1) -> np.ndarray:
    """Multi-token (prefill) attention over paged KV: rows query_start[s] ..
    query_start[s+1]-1 of q ([rows, Hq, D]) are the last qn_s tokens of
    sequence s; row t of s sits at position L_s - qn_s + t and attends to the
    sequence's tokens 0 .. L_s - qn_s + t (causal).  Returns float64
    [rows, Hq, D].  (cayang0802 walkthrough: the KV of a whole prompt can be
    computed in one parallel pass -- the prefill that recomputation relies
    on.)"""
    q, k_cache, v_cache = _cpu(q), _cpu(k_cache), _cpu(v_cache)
    bt = _cpu(block_tables).to(torch.int32)
    cl = _cpu(context_lens).to(torch.int32)
    qs = _cpu(query_start).to(torch.int32)
    R, Hq, D = q.shape
    S = cl.numel()
    out = np.full((R, Hq, D), np.nan, dtype=np.float64)
    rc = _load().orc_paged_prefill_attention(
        out.ctypes.data, q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
        DTYPE_CODE[q.dtype], bt.data_ptr(), cl.data_ptr(), qs.data_ptr(), float(scale),
        int(block_size), int(num_kv_heads), S, Hq, D, bt.shape[1], k_cache.shape[0],
        int(nthreads))
    if rc != 0:
        raise ValueError("orc_paged_prefill_attention failed: %d" % rc)
    return out


def kv_write(k_cache, v_cache, key, value, slot_mapping, block_size):
    """In place: k_cache/v_cache[slot // B, :, slot % B, :] = key/value[t] for
    every token t whose slot is >= 0."""
    for t in (k_cache, v_cache):
        if not t.is_contiguous():
            raise ValueError("cache must be contiguous")
    key, value = _cpu(key), _cpu(value)
    sm = _cpu(slot_mapping).to(torch.int64)
    NB, Hkv, B, D = k_cache.shape
    rc = _load().orc_kv_write(k_cache.data_ptr(), v_cache.data_ptr(), key.data_ptr(),
                              value.data_ptr(), sm.data_ptr(), sm.numel(), NB, Hkv, D,
                              int(block_size), DTYPE_CODE[k_cache.dtype])
    if rc != 0:
        raise ValueError("orc_kv_write failed: %d" % rc)


def decode_step(q, new_k, new_v, k_cache, v_cache, block_tables, context_lens, scale,
                block_size, num_kv_heads, nthreads=1):
    """One decode step ([CAY] KV-cache paragraph): in place, the new token of
    sequence s (new_k/new_v[s]) is stored at position context_lens[s] - 1,
    i.e. at slot_for_position(table row, L - 1) ([AIPP] core idea 3-4); then
    the step's query attends over the updated cache.  Returns that output.
    A sequence with no tokens, or whose table entry for the new position is
    not a block of the cache, gets no write."""
    NB = k_cache.shape[0]
    lens = _cpu(context_lens).tolist()
    tables = _cpu(block_tables)
    slots = []
    for s, L in enumerate(lens):
        ok = L > 0 and (L - 1) // block_size < tables.shape[1]
        if ok:
            blk = int(tables[s, (L - 1) // block_size])
            ok = 0 <= blk < NB
        slots.append(slot_for_position(tables[s].tolist(), L - 1, block_size) if ok else -1)
    kv_write(k_cache, v_cache, new_k, new_v, torch.tensor(slots, dtype=torch.int64), block_size)
    return paged_decode_attention(q, k_cache, v_cache, block_tables, context_lens, scale,
                                  block_size, num_kv_heads, nthreads=nthreads)


def kv_copy_blocks(k_cache, v_cache, pairs):
    """In place: for each (src, dst) row of pairs, in order, the whole physical
    block dst of K and V becomes a copy of block src."""
    pr = _cpu(pairs).to(torch.int64).reshape(-1, 2).contiguous()
    NB, Hkv, B, D = k_cache.shape
    rc = _load().orc_kv_copy_blocks(k_cache.data_ptr(), v_cache.data_ptr(), pr.data_ptr(),
                                    pr.shape[0], NB, Hkv, D, B, DTYPE_CODE[k_cache.dtype])
    if rc != 0:
        raise ValueError("orc_kv_copy_blocks failed: %d" % rc)


def kv_swap_blocks(dst_k, dst_v, src_k, src_v, pairs):
    """In place: for each (src, dst) row of pairs, block dst of the
    destination pools becomes a copy of block src of the source pools."""
    for t in (dst_k, dst_v):
        if not t.is_contiguous():
            raise ValueError("pools must be contiguous")
    src_k, src_v = _cpu(src_k), _cpu(src_v)
    pr = _cpu(pairs).to(torch.int64).reshape(-1, 2).contiguous()
    NS_, Hkv, B, D = src_k.shape
    rc = _load().orc_kv_swap_blocks(dst_k.data_ptr(), dst_v.data_ptr(), src_k.data_ptr(),
                                    src_v.data_ptr(), pr.data_ptr(), pr.shape[0], NS_,
                                    dst_k.shape[0], Hkv, D, B, DTYPE_CODE[src_k.dtype])
    if rc != 0:
        raise ValueError("orc_kv_swap_blocks failed: %d" % rc)


def slot_for_position(table_row, position: int, block_size: int) -> int:
    """Physical slot of logical token `position`: the table entry of logical
    block position // B, times B, plus the offset position % B."""
    return int(table_row[position // block_size]) * block_size + position % block_size


# ---- allocation arithmetic (auturnal guide, Eq. (1)-(3)) -------------------

def kv_bytes(layers: int, tokens: int, kv_heads: int, head_dim: int, elem_bytes: int) -> int:
    """Eq. (1): M_KV = 2 * L * n * h_KV * d_h * b (the 2 is key plus value)."""
    return 2 * layers * tokens * kv_heads * head_dim * elem_bytes


def allocated_positions(n: int, block_size: int) -> int:
    """Eq. (2): A_B(n) = B * ceil(n / B)."""
    return block_size * (-(-n // block_size))


def tail_waste(n: int, block_size: int) -> int:
    """Eq. (2): W_B(n) = A_B(n) - n, the unused positions of the last block."""
    return allocated_positions(n, block_size) - n


def fixed_reservation_positions(lengths, max_len: int) -> int:
    """Positions held when every request reserves max_len contiguously."""
    return max_len * len(lengths)


def position_utilisation(lengths, block_size: int) -> float:
    """Eq. (3): U = sum n_i / sum B * ceil(n_i / B)."""
    return sum(lengths) / sum(allocated_positions(n, block_size) for n in lengths)


# ---- split-context form (log-sum-exp identity) -----------------------------

def gather_sequence(cache: torch.Tensor, table_row, length: int) -> np.ndarray:
    """Logical [length, Hkv, D] float64 copy of one sequence's K or V."""
    NB, Hkv, B, D = cache.shape
    out = np.empty((length, Hkv, D), dtype=np.float64)
    for i in range(length):
        blk = int(table_row[i // B])
        if not 0 <= blk < NB:
            raise ValueError("block id out of range")
        out[i] = widen(cache[blk, :, i % B, :])
    return out


def decode_partitions(q_row: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float,
                      partition: int):
    """Per partition p of tokens [p*P, min((p+1)*P, L)): the max score m_p,
    the sum l_p = sum exp(z_i - m_p) and the unnormalised O_p = sum
    exp(z_i - m_p) v_i, for one query head (q_row: [D]; K, V: [L, D])."""
    L = K.shape[0]
    parts = []
    for start in range(0, L, partition):
        z = scale * (K[start:start + partition] @ q_row)
        m = float(z.max())
        w = np.exp(z - m)
        parts.append((m, float(w.sum()), w @ V[start:start + partition]))
    return parts


def lse_combine(parts) -> np.ndarray:
    """Combine per-partition (m_p, l_p, O_p): with M = max m_p and
    w_p = exp(m_p - M), out = sum w_p O_p / sum w_p l_p."""
    M = max(m for m, _, _ in parts)
    num = sum(math.exp(m - M) * O for m, _, O in parts)
    den = sum(math.exp(m - M) * l for m, l, _ in parts)
    return num / den


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)
