"""Pins of the oracle to things other than itself (CPU only).

Each test checks the oracle against a value the pages print, a closed form, a
library routine or brute force, chosen so that a plausible slip (dropped term,
wrong sign, swapped index, transposed operand, wrong head grouping) fails.
"""
import json
import math
import os
import random

import numpy as np
import pytest
import torch

import oracle
from oracle.blockmgr import BlockManager, OutOfBlocks, block_key, fnv1a64
from workloads import WORKLOADS, make_decode_case, normal_values

pytestmark = pytest.mark.filterwarnings("ignore")


# --------------------------------------------------------------------------
# Allocation arithmetic: the worked example printed by the auturnal guide.
# --------------------------------------------------------------------------

@pytest.fixture(scope="module")
def worked(golden_dir):
    with open(os.path.join(golden_dir, "alloc_worked_example.json")) as f:
        return json.load(f)


def test_worked_example_positions(worked):
    lengths = worked["lengths"]
    assert sum(lengths) == worked["valid_positions"]
    assert oracle.fixed_reservation_positions(
        lengths, worked["fixed_reservation_max_len"]) == worked["fixed_reservation_positions"]
    for B, expect in worked["paged_positions"].items():
        assert sum(oracle.allocated_positions(n, int(B)) for n in lengths) == expect


def test_worked_example_utilisation(worked):
    lengths = worked["lengths"]
    pr = worked["utilisation_percent_printed"]
    fixed = sum(lengths) / worked["fixed_reservation_positions"]
    assert round(100 * fixed, 2) == pr["fixed512"]
    for B in ("16", "32"):
        assert round(100 * oracle.position_utilisation(lengths, int(B)), 2) == pr[B]


def test_tail_waste_bounds():
    # Eq. (2): the last block wastes at most B - 1 positions; none when B | n.
    for B in (1, 4, 16, 32):
        for n in range(0, 200):
            w = oracle.tail_waste(n, B)
            assert 0 <= w <= B - 1
            assert (w == 0) == (n % B == 0)


def test_worked_example_through_block_manager(worked):
    for B, expect in worked["paged_positions"].items():
        bm = BlockManager(200, int(B))
        for s, n in enumerate(worked["lengths"]):
            bm.add(s, n)
        alloc, valid, used = bm.stats()
        assert (alloc, valid) == (expect, worked["valid_positions"])
        assert used * int(B) == expect
        bm.check_invariants()


def test_eq1_matches_tensor_bytes():
    # Eq. (1) with n = all pool positions equals the bytes of the K and V pools.
    w = WORKLOADS[1]
    case = make_decode_case(w, seed=0)
    NB, Hkv, B, D = case.k_cache.shape
    total = case.k_cache.numel() * case.k_cache.element_size() * 2
    assert oracle.kv_bytes(1, NB * B, Hkv, D, 4) == total == 80 * 2 * 4 * 16 * 64 * 4
    # ... and with n = 968 attended tokens it is the ~1.98 MB the workload reads.
    assert oracle.kv_bytes(1, 968, 4, 64, 4) == 1_982_464


# --------------------------------------------------------------------------
# Widening of stored values: every bit pattern against torch's conversion.
# --------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
def test_widen_all_16bit_patterns(dtype):
    bits = torch.arange(-32768, 32768, dtype=torch.int32).to(torch.int16)
    vals = bits.view(dtype)
    got = oracle.widen(vals)
    ref = vals.to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_widen_spot_values():
    h = torch.tensor([0x3C00, 0x0001, 0x7BFF, 0xC000 - 65536, 0x0400], dtype=torch.int16)
    got = oracle.widen(h.view(torch.float16))
    assert list(got) == [1.0, 2.0 ** -24, 65504.0, -2.0, 2.0 ** -14]
    b = torch.tensor([0x3F80, 0x4049, 0xBF80 - 65536], dtype=torch.int16)
    got = oracle.widen(b.view(torch.bfloat16))
    assert list(got) == [1.0, 3.140625, -1.0]


# --------------------------------------------------------------------------
# Attention: library routine, brute force, closed forms, invariances.
# --------------------------------------------------------------------------

def _scatter_case(Kl, Vl, block_size, NB, dtype, seed, Hq):
    """Page contiguous per-sequence K/V ([L, Hkv, D] float tensors) into a
    random pool; returns (k_cache, v_cache, tables, lens)."""
    rng = np.random.default_rng(seed)
    S = len(Kl)
    Hkv, D = Kl[0].shape[1], Kl[0].shape[2]
    need = [-(-k.shape[0] // block_size) for k in Kl]
    maxb = max(1, max(need))
    order = rng.permutation(NB)
    k_cache = torch.full((NB, Hkv, block_size, D), float("nan"), dtype=dtype)
    v_cache = torch.full_like(k_cache, float("nan"))
    tables = torch.full((S, maxb), -1, dtype=torch.int32)
    cur = 0
    for s in range(S):
        for j in range(need[s]):
            blk = int(order[cur]); cur += 1
            tables[s, j] = blk
            lo, hi = j * block_size, min((j + 1) * block_size, Kl[s].shape[0])
            k_cache[blk, :, :hi - lo, :] = Kl[s][lo:hi].transpose(0, 1).to(dtype)
            v_cache[blk, :, :hi - lo, :] = Vl[s][lo:hi].transpose(0, 1).to(dtype)
    lens = torch.tensor([k.shape[0] for k in Kl], dtype=torch.int32)
    return k_cache, v_cache, tables, lens


def _random_logical(seed, S, Lmax, Hkv, D, dtype, Lmin=1):
    g = torch.Generator().manual_seed(seed)
    lens = torch.randint(Lmin, Lmax + 1, (S,), generator=g).tolist()
    Kl = [torch.randn(n, Hkv, D, generator=g).to(dtype) for n in lens]
    Vl = [torch.randn(n, Hkv, D, generator=g).to(dtype) for n in lens]
    return Kl, Vl


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16, torch.float16])
@pytest.mark.parametrize("Hq,Hkv", [(4, 4), (8, 2), (6, 1)])
def test_attention_matches_sdpa(dtype, Hq, Hkv):
    S, D, B = 4, 32, 8
    Kl, Vl = _random_logical(1 + Hq, S, 70, Hkv, D, dtype)
    q = torch.randn(S, Hq, D, generator=torch.Generator().manual_seed(7)).to(dtype)
    kc, vc, bt, cl = _scatter_case(Kl, Vl, B, 40, dtype, seed=3, Hq=Hq)
    scale = 0.37
    got = oracle.paged_decode_attention(q, kc, vc, bt, cl, scale, B, Hkv)
    for s in range(S):
        qs = q[s].to(torch.float64)[None, :, None, :]
        ks = Kl[s].to(torch.float64).transpose(0, 1)[None]
        vs = Vl[s].to(torch.float64).transpose(0, 1)[None]
        ref = torch.nn.functional.scaled_dot_product_attention(
            qs, ks, vs, scale=scale, enable_gqa=True)[0, :, 0, :].numpy()
        np.testing.assert_allclose(got[s], ref, rtol=1e-12, atol=1e-12)


def test_attention_brute_force_high_precision():
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 40
    S, Hq, Hkv, D, B = 3, 4, 2, 8, 4
    Kl, Vl = _random_logical(11, S, 40, Hkv, D, torch.float32)
    q = torch.randn(S, Hq, D, generator=torch.Generator().manual_seed(5))
    kc, vc, bt, cl = _scatter_case(Kl, Vl, B, 40, torch.float32, seed=9, Hq=Hq)
    scale = 1 / math.sqrt(D)
    got = oracle.paged_decode_attention(q, kc, vc, bt, cl, scale, B, Hkv)
    G = Hq // Hkv
    for s in range(S):
        K = Kl[s].tolist(); V = Vl[s].tolist(); L = len(K)
        for h in range(Hq):
            g = h // G
            # no max subtraction: exp of the raw scores, in 40 digits
            w = [mpmath.exp(mpmath.mpf(scale) * mpmath.fsum(
                mpmath.mpf(q[s, h, d].item()) * mpmath.mpf(K[i][g][d]) for d in range(D)))
                for i in range(L)]
            den = mpmath.fsum(w)
            for d in range(D):
                ref = mpmath.fsum(w[i] * mpmath.mpf(V[i][g][d]) for i in range(L)) / den
                assert abs(got[s, h, d] - float(ref)) <= 1e-12


def test_single_token_returns_its_value_exactly():
    w = WORKLOADS[1]
    case = make_decode_case(w, seed=2, lengths=[1, 1, 1])
    out = oracle.paged_decode_attention(case.q, case.k_cache, case.v_cache, case.block_tables,
                                        case.context_lens, w.scale, w.block_size, w.num_kv_heads)
    for s in range(3):
        blk = int(case.block_tables[s, 0])
        v0 = case.v_cache[blk, :, 0, :].to(torch.float64).numpy()
        assert np.array_equal(out[s], v0)


def test_zero_scale_and_equal_keys_give_mean_of_values():
    S, Hq, Hkv, D, B = 2, 4, 4, 16, 16
    Kl, Vl = _random_logical(21, S, 50, Hkv, D, torch.float32, Lmin=20)
    q = torch.randn(S, Hq, D)
    kc, vc, bt, cl = _scatter_case(Kl, Vl, B, 20, torch.float32, seed=1, Hq=Hq)
    out = oracle.paged_decode_attention(q, kc, vc, bt, cl, 0.0, B, Hkv)
    for s in range(S):
        np.testing.assert_allclose(out[s], Vl[s].double().mean(0).numpy(), rtol=1e-13, atol=1e-14)
    # all keys equal (any scale): weights equal again
    Ke = [k[:1].expand_as(k).clone() for k in Kl]
    kc, vc, bt, cl = _scatter_case(Ke, Vl, B, 20, torch.float32, seed=1, Hq=Hq)
    out = oracle.paged_decode_attention(q, kc, vc, bt, cl, 0.9, B, Hkv)
    for s in range(S):
        np.testing.assert_allclose(out[s], Vl[s].double().mean(0).numpy(), rtol=1e-13, atol=1e-14)


def test_dominant_key_selects_its_value():
    D, Hkv, B, L = 8, 1, 4, 13
    K = torch.zeros(L, Hkv, D)
    V = torch.randn(L, Hkv, D)
    j = 9
    K[j, 0, 0] = 1.0
    q = torch.zeros(1, 1, D)
    q[0, 0, 0] = 1.0
    kc, vc, bt, cl = _scatter_case([K], [V], B, 8, torch.float32, seed=4, Hq=1)
    out = oracle.paged_decode_attention(q, kc, vc, bt, cl, 800.0, B, Hkv)
    np.testing.assert_allclose(out[0, 0], V[j, 0].double().numpy(), rtol=0, atol=1e-300)


def test_gqa_equals_mha_with_duplicated_kv_heads():
    S, Hq, Hkv, D, B = 3, 8, 2, 16, 8
    Kl, Vl = _random_logical(31, S, 45, Hkv, D, torch.bfloat16)
    q = torch.randn(S, Hq, D).to(torch.bfloat16)
    kc, vc, bt, cl = _scatter_case(Kl, Vl, B, 30, torch.bfloat16, seed=2, Hq=Hq)
    gqa = oracle.paged_decode_attention(q, kc, vc, bt, cl, 0.25, B, Hkv)
    G = Hq // Hkv
    Kd = [k.repeat_interleave(G, dim=1) for k in Kl]
    Vd = [v.repeat_interleave(G, dim=1) for v in Vl]
    kc, vc, bt, cl = _scatter_case(Kd, Vd, B, 30, torch.bfloat16, seed=2, Hq=Hq)
    mha = oracle.paged_decode_attention(q, kc, vc, bt, cl, 0.25, B, Hq)
    assert np.array_equal(gqa, mha)


def test_invariant_to_physical_permutation_and_block_size():
    S, Hq, Hkv, D = 4, 4, 2, 16
    Kl, Vl = _random_logical(41, S, 100, Hkv, D, torch.float16)
    q = torch.randn(S, Hq, D).to(torch.float16)
    outs = []
    for B, NB, seed in ((16, 40, 1), (16, 40, 2), (32, 20, 3), (8, 70, 4)):
        kc, vc, bt, cl = _scatter_case(Kl, Vl, B, NB, torch.float16, seed=seed, Hq=Hq)
        outs.append(oracle.paged_decode_attention(q, kc, vc, bt, cl, 0.125, B, Hkv))
    for o in outs[1:]:
        assert np.array_equal(o, outs[0])


def test_shared_prefix_equals_duplicated_prefix():
    # Two sequences whose first two blocks are the same physical blocks versus
    # private copies of the same contents.
    B, Hkv, D, Hq = 4, 2, 8, 2
    g = torch.Generator().manual_seed(8)
    prefix_k = torch.randn(8, Hkv, D, generator=g)
    prefix_v = torch.randn(8, Hkv, D, generator=g)
    tails = [(torch.randn(n, Hkv, D, generator=g), torch.randn(n, Hkv, D, generator=g)) for n in (3, 6)]
    Kl = [torch.cat([prefix_k, t[0]]) for t in tails]
    Vl = [torch.cat([prefix_v, t[1]]) for t in tails]
    q = torch.randn(2, Hq, D, generator=g)
    kc, vc, bt, cl = _scatter_case(Kl, Vl, B, 12, torch.float32, seed=5, Hq=Hq)
    dup = oracle.paged_decode_attention(q, kc, vc, bt, cl, 0.3, B, Hkv)
    shared = bt.clone()
    # point sequence 1's prefix entries at sequence 0's physical blocks
    shared[1, :2] = bt[0, :2]
    kc2, vc2 = kc.clone(), vc.clone()
    for j in range(2):
        kc2[int(bt[1, j])] = float("nan")
        vc2[int(bt[1, j])] = float("nan")
    out = oracle.paged_decode_attention(q, kc2, vc2, shared, cl, 0.3, B, Hkv)
    assert np.array_equal(out, dup)


def test_poison_outside_context_has_no_effect():
    w = WORKLOADS[1]
    case = make_decode_case(w, seed=4)
    assert torch.isnan(case.k_cache).any()
    a = oracle.paged_decode_attention(case.q, case.k_cache, case.v_cache, case.block_tables,
                                      case.context_lens, w.scale, w.block_size, w.num_kv_heads)
    assert np.isfinite(a).all()
    kc = torch.nan_to_num(case.k_cache, nan=1e30)
    vc = torch.nan_to_num(case.v_cache, nan=-7.0)
    b = oracle.paged_decode_attention(case.q, kc, vc, case.block_tables, case.context_lens,
                                      w.scale, w.block_size, w.num_kv_heads)
    assert np.array_equal(a, b)


def test_zero_length_gives_zero_row():
    w = WORKLOADS[1]
    case = make_decode_case(w, seed=1, lengths=[0, 5])
    out = oracle.paged_decode_attention(case.q, case.k_cache, case.v_cache, case.block_tables,
                                        case.context_lens, w.scale, w.block_size, w.num_kv_heads)
    assert np.array_equal(out[0], np.zeros_like(out[0]))
    assert np.isfinite(out[1]).all()


def test_bad_block_id_is_rejected():
    w = WORKLOADS[1]
    case = make_decode_case(w, seed=1, lengths=[20])
    bt = case.block_tables.clone()
    bt[0, 1] = 80
    with pytest.raises(ValueError):
        oracle.paged_decode_attention(case.q, case.k_cache, case.v_cache, bt, case.context_lens,
                                      w.scale, w.block_size, w.num_kv_heads)


def test_threads_do_not_change_bits():
    w = WORKLOADS[1]
    case = make_decode_case(w, seed=6)
    args = (case.q, case.k_cache, case.v_cache, case.block_tables, case.context_lens,
            w.scale, w.block_size, w.num_kv_heads)
    assert np.array_equal(oracle.paged_decode_attention(*args, nthreads=1),
                          oracle.paged_decode_attention(*args, nthreads=3))


# --------------------------------------------------------------------------
# Prefill (several query tokens per sequence, causal).
# --------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_prefill_matches_sdpa_with_causal_mask(dtype):
    S, Hq, Hkv, D, B = 3, 6, 2, 16, 8
    Kl, Vl = _random_logical(61, S, 60, Hkv, D, dtype, Lmin=10)
    lens = [k.shape[0] for k in Kl]
    qn = [lens[0], 3, 1]  # a whole prompt, a 3-token chunk, one token
    starts = torch.tensor([0, qn[0], qn[0] + qn[1], sum(qn)], dtype=torch.int32)
    g = torch.Generator().manual_seed(4)
    q = torch.randn(sum(qn), Hq, D, generator=g).to(dtype)
    kc, vc, bt, cl = _scatter_case(Kl, Vl, B, 40, dtype, seed=8, Hq=Hq)
    out = oracle.paged_prefill_attention(q, kc, vc, bt, cl, starts, 0.3, B, Hkv)
    for s in range(S):
        L, n = lens[s], qn[s]
        rows = q[starts[s]:starts[s + 1]].to(torch.float64).transpose(0, 1)[None]  # [1,Hq,n,D]
        mask = torch.arange(L)[None, :] <= (L - n + torch.arange(n))[:, None]     # [n, L]
        ref = torch.nn.functional.scaled_dot_product_attention(
            rows, Kl[s].double().transpose(0, 1)[None], Vl[s].double().transpose(0, 1)[None],
            attn_mask=mask, scale=0.3, enable_gqa=True)[0].transpose(0, 1).numpy()
        np.testing.assert_allclose(out[starts[s]:starts[s + 1]], ref, rtol=1e-12, atol=1e-12)


def test_prefill_last_row_is_decode_and_first_row_is_v0():
    w = WORKLOADS[1]
    case = make_decode_case(w, seed=3, lengths=[40, 17])
    L = case.context_lens.tolist()
    g = torch.Generator().manual_seed(2)
    q = torch.randn(sum(L), 4, 64, generator=g)
    starts = torch.tensor([0, L[0], L[0] + L[1]], dtype=torch.int32)
    out = oracle.paged_prefill_attention(q, case.k_cache, case.v_cache, case.block_tables,
                                         case.context_lens, starts, w.scale, 16, 4)
    last = torch.stack([q[L[0] - 1], q[L[0] + L[1] - 1]])
    dec = oracle.paged_decode_attention(last, case.k_cache, case.v_cache, case.block_tables,
                                        case.context_lens, w.scale, 16, 4)
    assert np.array_equal(out[[L[0] - 1, L[0] + L[1] - 1]], dec)
    v0 = case.v_cache[int(case.block_tables[0, 0]), :, 0, :].double().numpy()
    assert np.array_equal(out[0], v0)
    with pytest.raises(ValueError):  # more query rows than context
        oracle.paged_prefill_attention(q[:50], case.k_cache, case.v_cache, case.block_tables,
                                       case.context_lens, torch.tensor([0, 41, 50]), 0.1, 16, 4)


# --------------------------------------------------------------------------
# Split-context form: log-sum-exp combination equals the one-pass result.
# --------------------------------------------------------------------------

@pytest.mark.parametrize("P", [1, 7, 32, 512, 10_000])
def test_lse_combine_equals_one_pass(P):
    S, Hq, Hkv, D, B = 2, 4, 2, 16, 16
    Kl, Vl = _random_logical(51, S, 300, Hkv, D, torch.bfloat16, Lmin=100)
    q = torch.randn(S, Hq, D).to(torch.bfloat16)
    kc, vc, bt, cl = _scatter_case(Kl, Vl, B, 60, torch.bfloat16, seed=6, Hq=Hq)
    full = oracle.paged_decode_attention(q, kc, vc, bt, cl, 0.2, B, Hkv)
    G = Hq // Hkv
    for s in range(S):
        K = oracle.gather_sequence(kc, bt[s], int(cl[s]))
        V = oracle.gather_sequence(vc, bt[s], int(cl[s]))
        assert np.array_equal(K, Kl[s].double().numpy())
        for h in range(Hq):
            parts = oracle.decode_partitions(q[s, h].double().numpy(), K[:, h // G], V[:, h // G],
                                             0.2, P)
            assert len(parts) == -(-int(cl[s]) // P)
            np.testing.assert_allclose(oracle.lse_combine(parts), full[s, h], rtol=1e-12,
                                       atol=1e-13)


def _merged_state(parts):
    # one (max, sum, unnormalised output) for a run of partitions: the state
    # a single partition over their union would have
    M = max(m for m, _, _ in parts)
    w = [np.exp(m - M) for m, _, _ in parts]
    return (M, sum(wi * l for wi, (_, l, _) in zip(w, parts)),
            sum(wi * O for wi, (_, _, O) in zip(w, parts)))


@pytest.mark.parametrize("P,fan", [(16, 4), (7, 4), (32, 3), (1, 2)])
def test_two_level_lse_merge_equals_the_flat_one(P, fan):
    # merging runs of `fan` consecutive partitions first, then the runs'
    # states (the tensor-core kernel's order with one partition per warp,
    # four to a CTA), is the same log-sum-exp identity regrouped: it equals
    # the flat merge and the one-pass softmax to rounding; with an empty run
    # (max -inf) it still does
    S, Hq, Hkv, D, B = 2, 4, 2, 16, 16
    Kl, Vl = _random_logical(53, S, 300, Hkv, D, torch.bfloat16, Lmin=100)
    q = torch.randn(S, Hq, D).to(torch.bfloat16)
    kc, vc, bt, cl = _scatter_case(Kl, Vl, B, 60, torch.bfloat16, seed=7, Hq=Hq)
    full = oracle.paged_decode_attention(q, kc, vc, bt, cl, 0.2, B, Hkv)
    G = Hq // Hkv
    for s in range(S):
        K = oracle.gather_sequence(kc, bt[s], int(cl[s]))
        V = oracle.gather_sequence(vc, bt[s], int(cl[s]))
        for h in range(Hq):
            parts = oracle.decode_partitions(q[s, h].double().numpy(), K[:, h // G], V[:, h // G],
                                             0.2, P)
            runs = [_merged_state(parts[i:i + fan]) for i in range(0, len(parts), fan)]
            runs.append((-np.inf, 0.0, np.zeros(D)))  # a run with no tokens
            two = oracle.lse_combine(runs)
            np.testing.assert_allclose(two, oracle.lse_combine(parts), rtol=1e-12, atol=1e-13)
            np.testing.assert_allclose(two, full[s, h], rtol=1e-12, atol=1e-13)


# --------------------------------------------------------------------------
# Cache write and copy-on-write copy.
# --------------------------------------------------------------------------

def test_kv_write_round_trip_through_gather():
    B, Hkv, D, NB = 8, 3, 16, 30
    bm = BlockManager(NB, B, free_order=np.random.default_rng(0).permutation(NB))
    g = torch.Generator().manual_seed(3)
    lens = [13, 1, 29]
    kc = torch.full((NB, Hkv, B, D), float("nan"), dtype=torch.bfloat16)
    vc = torch.full_like(kc, float("nan"))
    logical = {}
    for s, n in enumerate(lens):
        bm.add(s, 0)
        K = torch.randn(n, Hkv, D, generator=g).to(torch.bfloat16)
        V = torch.randn(n, Hkv, D, generator=g).to(torch.bfloat16)
        slots = torch.tensor([bm.append(s)[0] for _ in range(n)], dtype=torch.int64)
        oracle.kv_write(kc, vc, K, V, slots, B)
        logical[s] = (K, V)
    for s, n in enumerate(lens):
        table = bm.table(s)
        assert np.array_equal(oracle.gather_sequence(kc, table, n), logical[s][0].double().numpy())
        assert np.array_equal(oracle.gather_sequence(vc, table, n), logical[s][1].double().numpy())
    # exactly sum(lens) * Hkv * D elements were written in each cache
    assert int((~torch.isnan(kc)).sum()) == sum(lens) * Hkv * D


def test_kv_write_skips_negative_slots_and_rejects_out_of_range():
    B, Hkv, D, NB = 4, 2, 8, 5
    kc = torch.zeros(NB, Hkv, B, D)
    vc = torch.zeros_like(kc)
    key = torch.ones(3, Hkv, D)
    oracle.kv_write(kc, vc, key, key, torch.tensor([-1, -5, -1]), B)
    assert not kc.any() and not vc.any()
    with pytest.raises(ValueError):
        oracle.kv_write(kc, vc, key[:1], key[:1], torch.tensor([NB * B]), B)


def test_decode_step_appends_at_position_then_attends():
    # The decode step stores each new token at position L-1 through the table
    # and attends over the sequence with it: against plain softmax attention
    # over the gathered sequence with the new row put in by hand.
    from workloads import Workload
    w = Workload(0, "step", "f32", 4, 2, 64, 16, 4, "fixed", writes_new_token=True)
    case = make_decode_case(w, seed=12, lengths=[1, 16, 17, 40])
    k, v = case.k_cache.clone(), case.v_cache.clone()
    out = oracle.decode_step(case.q, case.new_key, case.new_value, k, v, case.block_tables,
                             case.context_lens, w.scale, 16, 2)
    for s, L in enumerate(case.lengths):
        K = oracle.gather_sequence(k, case.block_tables[s].tolist(), int(L))
        V = oracle.gather_sequence(v, case.block_tables[s].tolist(), int(L))
        assert np.array_equal(K[L - 1], case.new_key[s].double().numpy())
        assert np.array_equal(V[L - 1], case.new_value[s].double().numpy())
        for hq in range(4):
            g = hq // 2
            sc = K[:, g, :] @ case.q[s, hq].double().numpy() * w.scale
            p_ = np.exp(sc - sc.max())
            ref = (p_[:, None] * V[:, g, :]).sum(0) / p_.sum()
            assert np.abs(out[s, hq] - ref).max() < 1e-12


def test_slot_for_position_agrees_with_block_manager():
    bm = BlockManager(50, 16, free_order=np.random.default_rng(1).permutation(50))
    bm.add(0, 0)
    slots = [bm.append(0)[0] for _ in range(100)]
    table = bm.table(0)
    assert slots == [oracle.slot_for_position(table, p, 16) for p in range(100)]
    assert len(set(slots)) == 100


def test_copy_blocks_in_order_and_untouched_rest():
    NB, Hkv, B, D = 6, 2, 4, 8
    g = torch.Generator().manual_seed(4)
    kc = torch.randn(NB, Hkv, B, D, generator=g).to(torch.float16)
    vc = torch.randn(NB, Hkv, B, D, generator=g).to(torch.float16)
    k0, v0 = kc.clone(), vc.clone()
    oracle.kv_copy_blocks(kc, vc, torch.tensor([[1, 4], [4, 5]]))
    assert torch.equal(kc[4], k0[1]) and torch.equal(vc[4], v0[1])
    assert torch.equal(kc[5], k0[1]) and torch.equal(vc[5], v0[1])  # chain: pair order
    for b in (0, 1, 2, 3):
        assert torch.equal(kc[b], k0[b]) and torch.equal(vc[b], v0[b])


def test_cow_isolation_between_beams():
    # Parent and child share a partial last block; the child's append copies it
    # first, so writing the child's token leaves the parent's output unchanged.
    B, Hkv, D, Hq, NB = 4, 2, 8, 2, 12
    bm = BlockManager(NB, B)
    g = torch.Generator().manual_seed(12)
    kc = torch.full((NB, Hkv, B, D), float("nan"))
    vc = torch.full_like(kc, float("nan"))
    bm.add(0, 0)
    n = 6
    K = torch.randn(n, Hkv, D, generator=g)
    V = torch.randn(n, Hkv, D, generator=g)
    oracle.kv_write(kc, vc, K, V, torch.tensor([bm.append(0)[0] for _ in range(n)]), B)
    bm.fork(0, 1)
    last = bm.table(0)[-1]
    assert bm.refcount(last) == 2
    q = torch.randn(2, Hq, D, generator=g)

    def attend(seqs):
        maxb = max(len(bm.table(s)) for s in seqs)
        bt = torch.full((len(seqs), maxb), -1, dtype=torch.int32)
        for i, s in enumerate(seqs):
            bt[i, :len(bm.table(s))] = torch.tensor(bm.table(s))
        cl = torch.tensor([bm.length(s) for s in seqs], dtype=torch.int32)
        return oracle.paged_decode_attention(q[:len(seqs)], kc, vc, bt, cl, 0.4, B, Hkv)

    before = attend([0])
    slot, cow = bm.append(1)
    assert cow is not None and cow[0] == last and bm.refcount(last) == 1
    oracle.kv_copy_blocks(kc, vc, torch.tensor([cow]))
    newk = torch.randn(1, Hkv, D, generator=g)
    oracle.kv_write(kc, vc, newk, newk, torch.tensor([slot]), B)
    assert np.array_equal(attend([0]), before)
    # child sees parent's 6 tokens + its own, as a contiguous baseline would
    Kc = torch.cat([K, newk]).double().numpy()
    child_k = oracle.gather_sequence(kc, bm.table(1), 7)
    assert np.array_equal(child_k, Kc)
    bm.check_invariants()


def test_swap_out_and_back_preserves_every_sequence():
    # Preemption by swapping: a sequence's blocks move to a CPU pool and back
    # into other GPU blocks; its logical K/V and its attention are unchanged,
    # and the sequences that shared its prefix keep theirs.
    B, Hkv, D, Hq = 4, 2, 8, 4
    gpu, cpu = BlockManager(20, B, free_order=list(range(19, -1, -1))), BlockManager(12, B)
    g = torch.Generator().manual_seed(21)
    kc = torch.full((20, Hkv, B, D), float("nan"))
    vc = torch.full_like(kc, float("nan"))
    hk = torch.full((12, Hkv, B, D), float("nan"))
    hv = torch.full_like(hk, float("nan"))
    K = torch.randn(11, Hkv, D, generator=g)
    V = torch.randn(11, Hkv, D, generator=g)
    gpu.add(0, 0)
    oracle.kv_write(kc, vc, K[:9], V[:9], torch.tensor([gpu.append(0)[0] for _ in range(9)]), B)
    gpu.fork(0, 1)  # 1 shares 0's blocks
    slot, cow = gpu.append(1)
    oracle.kv_copy_blocks(kc, vc, torch.tensor([cow]))
    oracle.kv_write(kc, vc, K[9:10], V[9:10], torch.tensor([slot]), B)
    q = torch.randn(1, Hq, D, generator=g)

    def attend(mgr, kcache, vcache, seq):
        bt = torch.tensor([mgr.table(seq)], dtype=torch.int32)
        cl = torch.tensor([mgr.length(seq)], dtype=torch.int32)
        return oracle.paged_decode_attention(q, kcache, vcache, bt, cl, 0.3, B, Hkv)

    before0, before1 = attend(gpu, kc, vc, 0), attend(gpu, kc, vc, 1)
    pairs = gpu.swap_to(cpu, 1)
    assert [p[0] for p in pairs] == gpu.table(0)[:2] + [cow[1]]
    oracle.kv_swap_blocks(hk, hv, kc, vc, torch.tensor(pairs))
    gpu.check_invariants()
    cpu.check_invariants()
    assert np.array_equal(attend(cpu, hk, hv, 1), before1)   # readable from the CPU pool
    assert np.array_equal(attend(gpu, kc, vc, 0), before0)   # sharer untouched
    back = cpu.swap_to(gpu, 1)
    oracle.kv_swap_blocks(kc, vc, hk, hv, torch.tensor(back))
    assert np.array_equal(attend(gpu, kc, vc, 1), before1)
    expect = torch.cat([K[:9], K[9:10]]).double().numpy()
    assert np.array_equal(oracle.gather_sequence(kc, gpu.table(1), 10), expect)
    assert cpu.num_free() == 12
    gpu.check_invariants()
    with pytest.raises(OutOfBlocks):
        gpu.swap_to(BlockManager(1, B), 0)  # needs 3 blocks
    assert gpu.length(0) == 9


# --------------------------------------------------------------------------
# Automatic prefix caching (hash of a block and everything before it).
# --------------------------------------------------------------------------

def test_fnv1a64_published_vectors():
    # Test vectors of the FNV-1a 64-bit hash (Fowler/Noll/Vo reference list).
    assert fnv1a64(b"") == 0xcbf29ce484222325
    assert fnv1a64(b"a") == 0xaf63dc4c8601ec8c
    assert fnv1a64(b"foobar") == 0x85944171f73967e8


def test_block_key_depends_on_every_preceding_token():
    a = block_key(0, [1, 2, 3, 4])
    assert a != block_key(0, [1, 2, 3, 5])
    assert block_key(a, [9, 9, 9, 9]) != block_key(block_key(0, [1, 2, 3, 5]), [9, 9, 9, 9])
    assert block_key(0, [-1, 0, 0, 0]) == fnv1a64(bytes(8) + b"\xff\xff\xff\xff" + bytes(12))


def test_prefix_cache_reuses_blocks_and_keeps_outputs():
    # Sequence 1 shares 2 full blocks of prompt with sequence 0 and differs in
    # the third: it reuses exactly those 2 blocks, only its own tokens are
    # written, and its attention equals attention over a fresh full copy.
    B, Hkv, D, Hq = 4, 2, 8, 2
    mgr = BlockManager(16, B)
    g = torch.Generator().manual_seed(33)
    tok0 = [5, 6, 7, 8, 9, 10, 11, 12, 13, 14]
    tok1 = tok0[:8] + [99, 98, 97]
    K = {t: torch.randn(Hkv, D, generator=g) for t in set(tok0 + tok1)}  # KV of a token
    kc = torch.full((16, Hkv, B, D), float("nan"))
    vc = torch.full_like(kc, float("nan"))

    def write(seq, tokens, start):
        table = mgr.table(seq)
        slots = torch.tensor([oracle.slot_for_position(table, p, B)
                              for p in range(start, len(tokens))])
        ks = torch.stack([K[t] for t in tokens[start:]])
        oracle.kv_write(kc, vc, ks, -ks, slots, B)

    assert mgr.add_cached(0, tok0) == 0
    write(0, tok0, 0)
    assert mgr.register_blocks(0, tok0) == 2
    reused = mgr.add_cached(1, tok1)
    assert reused == 8 and mgr.table(1)[:2] == mgr.table(0)[:2]
    assert mgr.table(1)[2] != mgr.table(0)[2]
    write(1, tok1, reused)
    q = torch.randn(1, Hq, D, generator=g)
    bt = torch.tensor([mgr.table(1)], dtype=torch.int32)
    out = oracle.paged_decode_attention(q, kc, vc, bt, torch.tensor([11], dtype=torch.int32),
                                        0.5, B, Hkv)
    ks = torch.stack([K[t] for t in tok1])  # [11, Hkv, D]
    ref = torch.nn.functional.scaled_dot_product_attention(
        q.double()[:, :, None, :].transpose(0, 1), ks.double().transpose(0, 1)[:, None],
        -ks.double().transpose(0, 1)[:, None], scale=0.5)
    np.testing.assert_allclose(out[0], ref[:, 0, 0, :].numpy(), rtol=1e-12, atol=1e-12)
    assert mgr.prefix_cache_stats() == (2, 2, 0)
    mgr.check_invariants()


def test_prefix_cache_keeps_freed_blocks_until_the_pool_runs_dry():
    B = 2
    mgr = BlockManager(6, B)
    t = [1, 2, 3, 4, 5]
    mgr.add_cached(0, t)
    mgr.register_blocks(0, t)
    kept = mgr.table(0)[:2]
    mgr.free_seq(0)
    assert mgr.num_free() == 6 and mgr.prefix_cache_stats()[2] == 2
    assert mgr.add_cached(1, t) == 4 and mgr.table(1)[:2] == kept  # revived
    mgr.free_seq(1)
    # released last to first: the cached list holds block 1 (oldest), block 0
    mgr.add(2, 10)  # 5 blocks: the 4 plain free ones, then block 1 is evicted
    assert mgr.prefix_cache_stats()[1:] == (1, 1)
    assert kept[1] in mgr.table(2) and kept[0] not in mgr.table(2)
    mgr.free_seq(2)
    assert mgr.add_cached(3, t) == 2 and mgr.table(3)[0] == kept[0]  # block 0 survived
    mgr.check_invariants()
    with pytest.raises(OutOfBlocks):
        mgr.add_cached(4, [7] * 12)
    assert mgr.table(3)[0] == kept[0]


# --------------------------------------------------------------------------
# Block manager: random model check of its invariants, OOM atomicity.
# --------------------------------------------------------------------------

def test_block_manager_random_operations_keep_invariants():
    rnd = random.Random(0)
    bm = BlockManager(64, 4, free_order=list(np.random.default_rng(2).permutation(64)))
    live, next_id = [], 0
    for _ in range(3000):
        op = rnd.random()
        try:
            if op < 0.15 or not live:
                bm.add(next_id, rnd.randint(0, 12)); live.append(next_id); next_id += 1
            elif op < 0.6:
                s = rnd.choice(live)
                before = bm.table(s)
                slot, cow = bm.append(s)
                after = bm.table(s)
                if cow is not None:
                    # a copy target is fresh and private
                    assert bm.refcount(cow[1]) == 1 and cow[0] == before[-1]
                assert slot // 4 == after[(bm.length(s) - 1) // 4]
                assert bm.refcount(after[-1]) == 1  # written block is never shared
            elif op < 0.75:
                s = rnd.choice(live)
                bm.fork(s, next_id); live.append(next_id); next_id += 1
            elif op < 0.85:
                seqs = rnd.sample(live, min(len(live), 4))
                bm.step_append(seqs)
            else:
                s = live.pop(rnd.randrange(len(live)))
                bm.free_seq(s)
        except OutOfBlocks:
            pass
        bm.check_invariants()


def test_block_manager_oom_leaves_state_unchanged():
    bm = BlockManager(3, 4)
    bm.add(0, 8)  # 2 blocks
    snap = (bm.table(0), bm.num_free(), bm.stats())
    with pytest.raises(OutOfBlocks):
        bm.add(1, 9)  # needs 3
    assert (bm.table(0), bm.num_free(), bm.stats()) == snap
    bm.add(1, 1)
    bm.append(1); bm.append(1); bm.append(1)
    with pytest.raises(OutOfBlocks):
        bm.step_append([1, 0])  # seq 1 would need a fresh block, seq 0 too
    assert bm.length(1) == 4 and bm.length(0) == 8
    bm.check_invariants()
