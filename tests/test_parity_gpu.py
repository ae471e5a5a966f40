"""GPU parity: the CUDA path (through the C ABI) against the oracle.

Cache writes and block copies must match bit for bit; attention outputs must
be within max-abs 2e-3 of the oracle for 16-bit KV and 1e-5 for fp32 KV (fp32
output).  Cases span several 16-token tiles, ragged tails, empty sequences,
bad ids, every block size / head_dim / group size the kernels support, both
decode kernels, the split-context path, and the full-size workloads through
the benchmark's own step (every sequence checked)."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_312_gb300 as pkv
from oracle.blockmgr import BlockManager
from workloads import (WORKLOADS, Workload, beam_setup_schedule, beam_step_schedule,
                       make_beam_case, make_decode_case, poison_unused, write_step_schedule)

pytestmark = pytest.mark.gpu

TOL16, TOL32 = 2e-3, 1e-5
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    pkv.device_status(reset=True)
    yield
    pkv.set_decode_kernel(pkv.KERNEL_AUTO)


@pytest.fixture(autouse=True)
def clean_status():
    pkv.device_status(reset=True)
    yield


def tol(dtype):
    return TOL32 if dtype == torch.float32 else TOL16


def bits(t):
    t = t.cpu().contiguous()
    return t.view(torch.int32) if t.element_size() == 4 else t.view(torch.int16)


def gpu_decode(q, kc, vc, bt, cl, scale, B, Hkv, P=0, out_dtype=torch.float32, kernel=None,
               plan=False):
    """Decode attention through the C ABI; `plan` gives an unsplit launch the
    optional workspace (the work plan: longest sequence first).  Split
    launches always take a workspace (and so a plan)."""
    if kernel is not None:
        pkv.set_decode_kernel(kernel)
    try:
        S, Hq, D = q.shape
        out = torch.full((S, Hq, D), float("nan"), dtype=out_dtype, device=DEV)
        ws = None
        if P or plan:
            n = pkv.decode_workspace_bytes(S, Hq, D, bt.shape[1] * B, P)
            ws = torch.empty(n, dtype=torch.uint8, device=DEV)
        pkv.paged_decode_attention(out, q.to(DEV), kc, vc, bt.to(DEV), cl.to(DEV), scale, B, Hkv,
                                   partition_size=P, workspace=ws)
        torch.cuda.synchronize()
        return out
    finally:
        pkv.set_decode_kernel(pkv.KERNEL_AUTO)


def max_err(out, ref):
    return float(np.abs(out.cpu().double().numpy() - ref).max())


# --------------------------------------------------------------------------
# kv_write / kv_copy_blocks: bit-exact
# --------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", [torch.float32, torch.float16, torch.bfloat16])
@pytest.mark.parametrize("B,D,Hkv", [(8, 64, 3), (16, 128, 8), (32, 128, 2)])
def test_kv_write_bit_exact(dtype, B, D, Hkv):
    NB, T = 23, 150
    g = torch.Generator().manual_seed(B + D)
    kc = torch.randn(NB, Hkv, B, D, generator=g).to(dtype)
    vc = torch.randn(NB, Hkv, B, D, generator=g).to(dtype)
    key = torch.randn(T, Hkv, D, generator=g).to(dtype)
    val = torch.randn(T, Hkv, D, generator=g).to(dtype)
    slots = torch.randperm(NB * B, generator=g)[:T].to(torch.int64)
    slots[::7] = -1  # padding tokens
    dk, dv = kc.to(DEV), vc.to(DEV)
    pkv.kv_write(dk, dv, key.to(DEV), val.to(DEV), slots.to(DEV))
    oracle.kv_write(kc, vc, key, val, slots, B)
    torch.cuda.synchronize()
    assert torch.equal(bits(dk), bits(kc)) and torch.equal(bits(dv), bits(vc))
    assert pkv.device_status() == 0


def test_kv_write_out_of_range_slot_is_flagged_and_skipped():
    NB, Hkv, B, D = 4, 2, 16, 64
    kc = torch.zeros(NB, Hkv, B, D, dtype=torch.bfloat16, device=DEV)
    vc = torch.zeros_like(kc)
    key = torch.ones(2, Hkv, D, dtype=torch.bfloat16, device=DEV)
    slots = torch.tensor([NB * B, 5], dtype=torch.int64, device=DEV)
    pkv.kv_write(kc, vc, key, key, slots)
    assert pkv.device_status() & 4
    assert float(kc.float().sum()) == Hkv * D  # only slot 5 was written
    assert float(kc[0, :, 5].float().sum()) == Hkv * D


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16, torch.float32])
def test_copy_blocks_bit_exact(dtype):
    NB, Hkv, B, D = 40, 4, 16, 128
    g = torch.Generator().manual_seed(3)
    kc = torch.randn(NB, Hkv, B, D, generator=g).to(dtype)
    vc = torch.randn(NB, Hkv, B, D, generator=g).to(dtype)
    perm = torch.randperm(NB, generator=g)
    pairs = torch.stack([perm[:12], perm[12:24]], dim=1).to(torch.int64)
    dk, dv = kc.to(DEV), vc.to(DEV)
    pkv.kv_copy_blocks(dk, dv, pairs.to(DEV))
    oracle.kv_copy_blocks(kc, vc, pairs)
    torch.cuda.synchronize()
    assert torch.equal(bits(dk), bits(kc)) and torch.equal(bits(dv), bits(vc))
    bad = torch.tensor([[0, NB]], dtype=torch.int64, device=DEV)
    pkv.kv_copy_blocks(dk, dv, bad)
    assert pkv.device_status() & 8
    assert torch.equal(bits(dk), bits(kc))


# --------------------------------------------------------------------------
# decode attention on small cases (several tiles, ragged tails, empty rows)
# --------------------------------------------------------------------------

RAGGED = [0, 1, 7, 15, 16, 17, 33, 100, 129, 300, 513]

SMALL = [  # dtype, Hq, Hkv, D, B
    ("bf16", 8, 1, 128, 16), ("bf16", 32, 4, 128, 16), ("bf16", 16, 16, 128, 16),
    ("f16", 8, 4, 128, 8), ("bf16", 4, 2, 64, 32), ("f16", 16, 4, 64, 16),
    ("bf16", 6, 2, 128, 32), ("f16", 12, 12, 64, 8), ("bf16", 16, 2, 64, 8),
    ("f32", 8, 2, 128, 16), ("f32", 4, 4, 64, 32), ("bf16", 32, 2, 128, 16),
    # wide groups: two n8 column tiles (G = 10, 12), head slices (G = 32: 2 x
    # 16; G = 40: 14 + 14 + 12 columns)
    ("f16", 20, 2, 128, 32), ("bf16", 12, 1, 64, 16), ("bf16", 32, 1, 64, 16),
    ("f16", 40, 1, 128, 8),
]


@pytest.mark.parametrize("kernel", [pkv.KERNEL_AUTO, pkv.KERNEL_CUDA_CORE])
@pytest.mark.parametrize("P", [0, 16, 64])
@pytest.mark.parametrize("dt,Hq,Hkv,D,B", SMALL)
def test_decode_small(dt, Hq, Hkv, D, B, P, kernel):
    # P = 16 splits the 513-token context into 33 partitions: the tensor-core
    # kernel then gives each warp a partition of its own (groups of four, the
    # last one partial); P = 64 (9 partitions) spreads each over all warps
    w = Workload(0, "small", dt, Hq, Hkv, D, B, len(RAGGED), "fixed")
    case = make_decode_case(w, seed=Hq * 7 + B + D, lengths=RAGGED)
    if P and P % B:
        pytest.skip("partition must be a multiple of the block size")
    kc, vc = case.k_cache.to(DEV), case.v_cache.to(DEV)
    out = gpu_decode(case.q, kc, vc, case.block_tables, case.context_lens, w.scale, B, Hkv, P=P,
                     kernel=kernel)
    ref = oracle.paged_decode_attention(case.q, case.k_cache, case.v_cache, case.block_tables,
                                        case.context_lens, w.scale, B, Hkv)
    assert pkv.device_status() == 0
    assert max_err(out, ref) <= tol(w.torch_dtype)
    assert torch.equal(out[0].cpu(), torch.zeros_like(out[0].cpu()))  # length-0 row


@pytest.mark.parametrize("dt,Hq,Hkv,D,B", SMALL)
def test_unsplit_work_plan_matches_oracle_and_the_unplanned_call(dt, Hq, Hkv, D, B):
    # An unsplit call with the optional workspace runs its CTAs longest
    # sequence first (the work plan); the lengths are shuffled so that the
    # plan reorders them.  Each (sequence, KV head) is still one CTA doing the
    # same arithmetic, so the output equals the unplanned call's bit for bit.
    w = Workload(0, "plan", dt, Hq, Hkv, D, B, len(RAGGED), "fixed")
    lengths = list(np.random.default_rng(Hq + D + B).permutation(RAGGED + [2049, 5, 0]))
    case = make_decode_case(w, seed=Hq * 3 + B + D, lengths=lengths)
    kc, vc = case.k_cache.to(DEV), case.v_cache.to(DEV)
    planned = gpu_decode(case.q, kc, vc, case.block_tables, case.context_lens, w.scale, B, Hkv,
                         plan=True)
    assert pkv.device_status() == 0
    plain = gpu_decode(case.q, kc, vc, case.block_tables, case.context_lens, w.scale, B, Hkv)
    ref = oracle.paged_decode_attention(case.q, case.k_cache, case.v_cache, case.block_tables,
                                        case.context_lens, w.scale, B, Hkv)
    assert max_err(planned, ref) <= tol(w.torch_dtype)
    assert torch.equal(planned, plain)
    for s_, n in enumerate(lengths):
        if n == 0:
            assert not planned[s_].any()


@pytest.mark.parametrize("B", [8, 16, 32])
@pytest.mark.parametrize("G", [1, 4, 8, 16, 64])
@pytest.mark.parametrize("D", [64, 128])
def test_sweep_points(B, G, D):
    # every point of the block-size / GQA / head-dim sweep, at a small size
    # and in both launch configurations the sweep times: one pass per
    # (sequence, KV head) and 2048-token partitions, each with the work plan
    import bench
    w = bench.sweep_workload(B, G, D)
    case = make_decode_case(w, seed=B * 100 + G * 10 + D, lengths=[1, 700, 2100, 1500, 4100])
    kc, vc = case.k_cache.to(DEV), case.v_cache.to(DEV)
    ref = oracle.paged_decode_attention(case.q, case.k_cache, case.v_cache, case.block_tables,
                                        case.context_lens, w.scale, B, 8)
    for P in (0, 2048):
        out = gpu_decode(case.q, kc, vc, case.block_tables, case.context_lens, w.scale, B, 8,
                         P=P, plan=True)
        assert pkv.device_status() == 0
        assert max_err(out, ref) <= TOL16, P


def test_workload1_fp32():
    w = WORKLOADS[1]
    for seed in (0, 1, 2):
        case = make_decode_case(w, seed=seed)
        kc, vc = case.k_cache.to(DEV), case.v_cache.to(DEV)
        out = gpu_decode(case.q, kc, vc, case.block_tables, case.context_lens, w.scale,
                         w.block_size, w.num_kv_heads)
        ref = oracle.paged_decode_attention(case.q, case.k_cache, case.v_cache, case.block_tables,
                                            case.context_lens, w.scale, w.block_size,
                                            w.num_kv_heads)
        assert max_err(out, ref) <= TOL32


@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float16])
def test_16bit_outputs(out_dtype):
    # The output is rounded once to its dtype: allow the attention tolerance
    # plus one unit of rounding at the reference's magnitude.
    w = Workload(0, "o", "bf16", 16, 4, 128, 16, 6, "fixed")
    case = make_decode_case(w, seed=5, lengths=[1, 5, 40, 77, 200, 333])
    kc, vc = case.k_cache.to(DEV), case.v_cache.to(DEV)
    for P in (0, 32):
        out = gpu_decode(case.q, kc, vc, case.block_tables, case.context_lens, w.scale, 16, 4,
                         P=P, out_dtype=out_dtype)
        ref = oracle.paged_decode_attention(case.q, case.k_cache, case.v_cache,
                                            case.block_tables, case.context_lens, w.scale, 16, 4)
        rel = 2.0 ** -8 if out_dtype == torch.bfloat16 else 2.0 ** -11
        diff = np.abs(out.cpu().double().numpy() - ref)
        assert (diff <= TOL16 + rel * np.abs(ref)).all()


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_output_base_not_16_byte_aligned(out_dtype):
    # the decode kernel stores four outputs at a time only from a 16-byte
    # aligned base; one element past an aligned base takes the scalar stores
    w = Workload(0, "ua", "bf16", 16, 2, 128, 16, 4, "fixed")
    case = make_decode_case(w, seed=21, lengths=[1, 50, 300, 1000])
    kc, vc = case.k_cache.to(DEV), case.v_cache.to(DEV)
    ref = oracle.paged_decode_attention(case.q, case.k_cache, case.v_cache, case.block_tables,
                                        case.context_lens, w.scale, 16, 2)
    n = case.q.numel()
    for P in (0, 64):
        big = torch.full((n + 1,), float("nan"), dtype=out_dtype, device=DEV)
        out = big[1:].view(case.q.shape)
        assert out.data_ptr() % 16 != 0
        ws = None
        if P:
            nb = pkv.decode_workspace_bytes(4, 16, 128, case.block_tables.shape[1] * 16, P)
            ws = torch.empty(nb, dtype=torch.uint8, device=DEV)
        pkv.paged_decode_attention(out, case.q.to(DEV), kc, vc, case.block_tables.to(DEV),
                                   case.context_lens.to(DEV), w.scale, 16, 2,
                                   partition_size=P, workspace=ws)
        torch.cuda.synchronize()
        assert pkv.device_status() == 0
        assert torch.isnan(big[:1].float()).all()  # nothing written before the view
        rel = 0.0 if out_dtype == torch.float32 else 2.0 ** -8
        diff = np.abs(out.float().cpu().double().numpy() - ref)
        assert (diff <= TOL16 + rel * np.abs(ref)).all(), P


def test_bad_block_id_and_length_are_flagged():
    w = Workload(0, "bad", "bf16", 8, 2, 128, 16, 3, "fixed")
    case = make_decode_case(w, seed=9, lengths=[40, 40, 40])
    bt = case.block_tables.clone()
    bt[1, 1] = case.num_blocks + 5
    cl = case.context_lens.clone()
    cl[2] = bt.shape[1] * 16 + 1
    kc, vc = case.k_cache.to(DEV), case.v_cache.to(DEV)
    for kernel, plan, P in ((pkv.KERNEL_AUTO, False, 0), (pkv.KERNEL_CUDA_CORE, False, 0),
                            (pkv.KERNEL_AUTO, True, 0), (pkv.KERNEL_AUTO, True, 16)):
        out = gpu_decode(case.q, kc, vc, bt, cl, w.scale, 16, 2, kernel=kernel, plan=plan, P=P)
        st = pkv.device_status()
        assert st & 1 and st & 2
        ref = oracle.paged_decode_attention(case.q[:1], case.k_cache, case.v_cache, bt[:1],
                                            cl[:1], w.scale, 16, 2)
        assert max_err(out[:1], ref) <= TOL16  # the healthy sequence is unaffected
        assert torch.isfinite(out[1]).all()


def test_split_matches_one_pass_and_kernels_agree():
    w = Workload(0, "split", "bf16", 32, 8, 128, 16, 5, "fixed")
    case = make_decode_case(w, seed=11, lengths=[1000, 1, 513, 512, 2049])
    kc, vc = case.k_cache.to(DEV), case.v_cache.to(DEV)
    ref = oracle.paged_decode_attention(case.q, case.k_cache, case.v_cache, case.block_tables,
                                        case.context_lens, w.scale, 16, 8)
    for P in (0, 16, 256, 512, 4096):
        for kernel in (pkv.KERNEL_AUTO, pkv.KERNEL_CUDA_CORE):
            out = gpu_decode(case.q, kc, vc, case.block_tables, case.context_lens, w.scale, 16, 8,
                             P=P, kernel=kernel)
            assert max_err(out, ref) <= TOL16, (P, kernel)


@pytest.mark.parametrize("Hq", [16, 32, 64])
def test_split_with_thousands_of_partitions(Hq):
    # 1500 and 1875 partitions of 16 tokens: more merge weights than the
    # decode kernel keeps in shared memory, so the merge recomputes them;
    # G = 8, 16 (two column tiles) and 32 (two head slices)
    w = Workload(0, "many", "bf16", Hq, 2, 128, 16, 3, "fixed")
    case = make_decode_case(w, seed=13, lengths=[24000, 30000, 17])
    kc, vc = case.k_cache.to(DEV), case.v_cache.to(DEV)
    ref = oracle.paged_decode_attention(case.q, case.k_cache, case.v_cache, case.block_tables,
                                        case.context_lens, w.scale, 16, 2)
    for P in (16, 32, 4096):
        out = gpu_decode(case.q, kc, vc, case.block_tables, case.context_lens, w.scale, 16, 2,
                         P=P)
        assert pkv.device_status() == 0
        assert max_err(out, ref) <= TOL16, P


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16, torch.float32])
@pytest.mark.parametrize("pairs_on_host", [False, True])
def test_swap_blocks_to_pinned_host_and_back(dtype, pairs_on_host):
    # Device pool -> pinned host pool -> other device blocks, bit-exact, with
    # the pair list either on the GPU or in pinned host memory.
    NB, NH, Hkv, B, D = 30, 12, 4, 16, 128
    g = torch.Generator().manual_seed(7)
    kc = torch.randn(NB, Hkv, B, D, generator=g).to(dtype)
    vc = torch.randn(NB, Hkv, B, D, generator=g).to(dtype)
    hk = torch.zeros(NH, Hkv, B, D, dtype=dtype).pin_memory()
    hv = torch.zeros(NH, Hkv, B, D, dtype=dtype).pin_memory()
    out_pairs = torch.tensor([[3, 0], [17, 5], [29, 11], [0, 2]], dtype=torch.int64)
    in_pairs = torch.tensor([[0, 20], [5, 21], [11, 1], [2, 4]], dtype=torch.int64)
    place = (lambda t: t.pin_memory()) if pairs_on_host else (lambda t: t.to(DEV))
    dk, dv = kc.to(DEV), vc.to(DEV)
    pkv.kv_swap_blocks(hk, hv, dk, dv, place(out_pairs))
    torch.cuda.synchronize()
    rk, rv = torch.zeros_like(hk), torch.zeros_like(hv)
    oracle.kv_swap_blocks(rk, rv, kc, vc, out_pairs)
    assert torch.equal(bits(hk), bits(rk)) and torch.equal(bits(hv), bits(rv))
    pkv.kv_swap_blocks(dk, dv, hk, hv, place(in_pairs))
    torch.cuda.synchronize()
    oracle.kv_swap_blocks(kc, vc, rk, rv, in_pairs)
    assert torch.equal(bits(dk), bits(kc)) and torch.equal(bits(dv), bits(vc))
    assert pkv.device_status() == 0
    pkv.kv_swap_blocks(hk, hv, dk, dv, place(torch.tensor([[NB, 0]], dtype=torch.int64)))
    assert pkv.device_status() & 8
    assert torch.equal(bits(hk), bits(rk))


def test_swap_round_trip_keeps_attention():
    # A sequence swapped out to a host pool by the allocator and the swap
    # kernel, then back into other device blocks, attends exactly as before.
    w = Workload(0, "swap", "bf16", 16, 4, 128, 16, 5, "fixed")
    case = make_decode_case(w, seed=3, lengths=[100, 300, 17, 512, 64])
    NB = case.num_blocks
    gpu = pkv.BlockAllocator(NB + 40, 16, free_order=list(case.pool_order) + list(range(NB, NB + 40)))
    for s, n in enumerate(case.lengths):
        gpu.add(s, int(n))
    bt0, cl = gpu.dense_tables(range(5), case.block_tables.shape[1])
    assert torch.equal(bt0, case.block_tables)
    kc = torch.cat([case.k_cache, torch.zeros(40, 4, 16, 128, dtype=torch.bfloat16)]).to(DEV)
    vc = torch.cat([case.v_cache, torch.zeros(40, 4, 16, 128, dtype=torch.bfloat16)]).to(DEV)
    before = gpu_decode(case.q, kc, vc, bt0, cl, w.scale, 16, 4)
    host = pkv.BlockAllocator(64, 16)
    hk = torch.zeros(64, 4, 16, 128, dtype=torch.bfloat16).pin_memory()
    hv = torch.zeros_like(hk).pin_memory()
    pkv.kv_swap_blocks(hk, hv, kc, vc, gpu.swap_to(host, 3).to(DEV))
    gpu.add(99, 64)  # another sequence takes some of the freed blocks meanwhile
    pkv.kv_swap_blocks(kc, vc, hk, hv, host.swap_to(gpu, 3).to(DEV))
    bt1, cl1 = gpu.dense_tables(range(5), case.block_tables.shape[1])
    assert not torch.equal(bt1[3], bt0[3])
    after = gpu_decode(case.q, kc, vc, bt1, cl1, w.scale, 16, 4)
    assert pkv.device_status() == 0
    assert torch.equal(before, after)


def test_prefix_cached_sequence_attends_like_a_fresh_one():
    # Sequence 1 reuses sequence 0's cached prompt blocks; only its own tokens
    # are written on the GPU.  Its attention must equal the oracle's over a
    # cache where every token of sequence 1 was written afresh.
    B, Hkv, D, Hq = 16, 4, 128, 16
    g = torch.Generator().manual_seed(9)
    vocab = 64
    KV = torch.randn(vocab, 2, Hkv, D, generator=g).to(torch.bfloat16)  # K/V of a token id
    tok0 = torch.randint(0, vocab, (300,), generator=g).tolist()
    tok1 = tok0[:256] + torch.randint(0, vocab, (37,), generator=g).tolist()
    mgr = pkv.BlockAllocator(64, B)
    kc = torch.full((64, Hkv, B, D), float("nan"), dtype=torch.bfloat16, device=DEV)
    vc = torch.full_like(kc, float("nan"))

    def write(seq, tokens, start):
        table = mgr.table(seq)
        slots = torch.tensor([oracle.slot_for_position(table, p, B)
                              for p in range(start, len(tokens))], dtype=torch.int64)
        kv = KV[torch.tensor(tokens[start:])]
        pkv.kv_write(kc, vc, kv[:, 0].contiguous().to(DEV), kv[:, 1].contiguous().to(DEV),
                     slots.to(DEV))

    assert mgr.add_cached(0, tok0) == 0
    write(0, tok0, 0)
    assert mgr.register_blocks(0, tok0) == 300 // B
    reused = mgr.add_cached(1, tok1)
    assert reused == 256
    write(1, tok1, reused)
    q = torch.randn(1, Hq, D, generator=g).to(torch.bfloat16)
    bt = torch.tensor([mgr.table(1)], dtype=torch.int32)
    cl = torch.tensor([len(tok1)], dtype=torch.int32)
    out = gpu_decode(q, kc, vc, bt, cl, D ** -0.5, B, Hkv)
    # fresh: every token of sequence 1 written into its own blocks on the host
    fk = torch.full((64, Hkv, B, D), float("nan"), dtype=torch.bfloat16)
    fv = torch.full_like(fk, float("nan"))
    fresh_table = list(range(-(-len(tok1) // B)))
    kv = KV[torch.tensor(tok1)]
    oracle.kv_write(fk, fv, kv[:, 0].contiguous(), kv[:, 1].contiguous(),
                    torch.tensor([oracle.slot_for_position(fresh_table, p, B)
                                  for p in range(len(tok1))]), B)
    ref = oracle.paged_decode_attention(q, fk, fv, torch.tensor([fresh_table], dtype=torch.int32),
                                        cl, D ** -0.5, B, Hkv)
    assert pkv.device_status() == 0
    assert max_err(out, ref) <= TOL16


# --------------------------------------------------------------------------
# maximum sizes: the most sequences a call takes (65535), tiny contexts
# --------------------------------------------------------------------------

def test_decode_and_decode_step_at_the_sequence_limit():
    S, B = 65535, 8
    w = Workload(0, "max-seqs", "bf16", 2, 1, 64, B, S, "fixed", writes_new_token=True)
    rng = np.random.default_rng(33)
    lengths = rng.integers(1, 3 * B + 1, size=S)
    case = make_decode_case(w, seed=34, lengths=lengths.tolist())
    kc, vc = case.k_cache.to(DEV), case.v_cache.to(DEV)
    out = torch.empty(case.q.shape, dtype=torch.float32, device=DEV)
    pkv.decode_step(out, case.q.to(DEV), case.new_key.to(DEV), case.new_value.to(DEV), kc, vc,
                    case.block_tables.to(DEV), case.context_lens.to(DEV), w.scale, B, 1)
    torch.cuda.synchronize()
    k_ref, v_ref = case.k_cache.clone(), case.v_cache.clone()
    ref = oracle.decode_step(case.q, case.new_key, case.new_value, k_ref, v_ref,
                             case.block_tables, case.context_lens, w.scale, B, 1,
                             nthreads=oracle.default_threads())
    assert pkv.device_status() == 0
    assert torch.equal(bits(kc), bits(k_ref)) and torch.equal(bits(vc), bits(v_ref))
    assert max_err(out, ref) <= TOL16
    # plain attention over the updated cache, split into one-block partitions
    n = pkv.decode_workspace_bytes(S, 2, 64, case.block_tables.shape[1] * B, B)
    ws = torch.empty(n, dtype=torch.uint8, device=DEV)
    out2 = torch.empty_like(out)
    pkv.paged_decode_attention(out2, case.q.to(DEV), kc, vc, case.block_tables.to(DEV),
                               case.context_lens.to(DEV), w.scale, B, 1, partition_size=B,
                               workspace=ws)
    torch.cuda.synchronize()
    assert pkv.device_status() == 0
    assert max_err(out2, ref) <= TOL16


# --------------------------------------------------------------------------
# bounded waits: a wait that nothing completes gives up, flags, and the
# context stays usable (no fault, nothing left in flight)
# --------------------------------------------------------------------------

def test_bounded_waits_give_up_flag_and_leave_the_context_usable():
    import time
    n = 600  # more CTAs than one wait: they must stop on the first one's flag
    drained = torch.zeros(1, dtype=torch.int32, device=DEV)
    t0 = time.time()
    pkv.selftest_bounded_wait(n, drained)
    torch.cuda.synchronize()
    elapsed = time.time() - t0
    st = pkv.device_status(reset=True)
    assert st & 16  # PKV_STATUS_TIMEOUT
    assert int(drained.item()) == n
    assert elapsed < 10.0, elapsed
    # the same context still computes correct attention
    w = Workload(0, "after", "bf16", 8, 2, 128, 16, 3, "fixed")
    case = make_decode_case(w, seed=3, lengths=[5, 100, 300])
    out = gpu_decode(case.q, case.k_cache.to(DEV), case.v_cache.to(DEV), case.block_tables,
                     case.context_lens, w.scale, 16, 2)
    ref = oracle.paged_decode_attention(case.q, case.k_cache, case.v_cache, case.block_tables,
                                        case.context_lens, w.scale, 16, 2)
    assert pkv.device_status() == 0
    assert max_err(out, ref) <= TOL16


# --------------------------------------------------------------------------
# decode step: append the new token, then attend (one call)
# --------------------------------------------------------------------------

STEP_CASES = [  # dtype, Hq, Hkv, D, B, partition
    ("bf16", 32, 32, 128, 16, 0), ("bf16", 32, 8, 128, 16, 64), ("f16", 16, 2, 64, 8, 0),
    ("bf16", 8, 1, 128, 32, 32), ("f16", 8, 8, 128, 16, 512),
    ("bf16", 32, 2, 128, 16, 0), ("f16", 48, 2, 64, 8, 32),  # G = 16, G = 24 (2 slices)
    ("bf16", 16, 4, 128, 16, 16),  # 16-token partitions: one per warp, four to a CTA
    ("f32", 4, 4, 64, 16, 0),  # CUDA-core kernel path
]


@pytest.mark.parametrize("plan", [False, True])
@pytest.mark.parametrize("dt,Hq,Hkv,D,B,P", STEP_CASES)
def test_decode_step_matches_oracle(dt, Hq, Hkv, D, B, P, plan):
    # the new position's slot holds NaN until the step writes it; lengths put
    # the new token first in a block, last in a block, mid-block, alone.
    # `plan` gives an unsplit step the optional workspace (the work plan)
    if plan and P:
        pytest.skip("a split step always has the plan")
    w = Workload(0, "step", dt, Hq, Hkv, D, B, 6, "fixed", writes_new_token=True)
    lengths = [1, B, B + 1, 3 * B - 5, 700, 2049]
    case = make_decode_case(w, seed=Hq + B + P, lengths=lengths)
    kc, vc = case.k_cache.to(DEV), case.v_cache.to(DEV)
    out = torch.full(case.q.shape, float("nan"), dtype=torch.float32, device=DEV)
    ws = None
    if P or plan:
        n = pkv.decode_workspace_bytes(6, Hq, D, case.block_tables.shape[1] * B, P)
        ws = torch.empty(n, dtype=torch.uint8, device=DEV)
    pkv.decode_step(out, case.q.to(DEV), case.new_key.to(DEV), case.new_value.to(DEV), kc, vc,
                    case.block_tables.to(DEV), case.context_lens.to(DEV), w.scale, B, Hkv,
                    partition_size=P, workspace=ws)
    torch.cuda.synchronize()
    k_ref, v_ref = case.k_cache.clone(), case.v_cache.clone()
    ref = oracle.decode_step(case.q, case.new_key, case.new_value, k_ref, v_ref,
                             case.block_tables, case.context_lens, w.scale, B, Hkv)
    assert pkv.device_status() == 0
    # the cache is bit-exact (NaN slots elsewhere compared as bits)
    assert torch.equal(bits(kc), bits(k_ref)) and torch.equal(bits(vc), bits(v_ref))
    assert max_err(out, ref) <= tol(w.torch_dtype)


@pytest.mark.parametrize("P", [0, 512])
def test_back_to_back_steps_see_each_others_writes(P):
    # Two decode steps back to back on one stream, one workspace, no
    # synchronisation between them: the second appends its token at the next
    # position, attends over the cache the first one appended to, and takes
    # the first one's bf16 output as its queries.  Each decode launch starts
    # while the kernel before it runs, so it must read the cache and q only
    # after waiting for that kernel.
    B = 16
    lengths = [5, 17, 700, 2049, 1001, 35]  # the next position stays in the last block
    w = Workload(0, "chain", "bf16", 32, 8, 128, B, len(lengths), "fixed",
                 writes_new_token=True)
    case = make_decode_case(w, seed=31, lengths=lengths)
    S, Hq, D = case.q.shape
    g = torch.Generator().manual_seed(7)
    nk2 = torch.randn(S, 8, D, generator=g).to(torch.bfloat16)
    nv2 = torch.randn(S, 8, D, generator=g).to(torch.bfloat16)
    kc, vc = case.k_cache.to(DEV), case.v_cache.to(DEV)
    bt = case.block_tables.to(DEV)
    cl1, cl2 = case.context_lens.to(DEV), (case.context_lens + 1).to(DEV)
    out1 = torch.full((S, Hq, D), float("nan"), dtype=torch.bfloat16, device=DEV)
    out2 = torch.full((S, Hq, D), float("nan"), dtype=torch.float32, device=DEV)
    ws = torch.empty(pkv.decode_workspace_bytes(S, Hq, D, case.block_tables.shape[1] * B, P),
                     dtype=torch.uint8, device=DEV)
    pkv.decode_step(out1, case.q.to(DEV), case.new_key.to(DEV), case.new_value.to(DEV), kc, vc,
                    bt, cl1, w.scale, B, 8, partition_size=P, workspace=ws)
    pkv.decode_step(out2, out1, nk2.to(DEV), nv2.to(DEV), kc, vc, bt, cl2, w.scale, B, 8,
                    partition_size=P, workspace=ws)
    torch.cuda.synchronize()
    assert pkv.device_status() == 0
    k_ref, v_ref = case.k_cache.clone(), case.v_cache.clone()
    ref1 = oracle.decode_step(case.q, case.new_key, case.new_value, k_ref, v_ref,
                              case.block_tables, case.context_lens, w.scale, B, 8)
    q2 = out1.cpu()  # the first step's output, as the second step took it
    assert max_err(q2.float(), ref1) <= TOL16 + 2 ** -8 * float(np.abs(ref1).max())
    ref2 = oracle.decode_step(q2, nk2, nv2, k_ref, v_ref, case.block_tables,
                              case.context_lens + 1, w.scale, B, 8)
    assert torch.equal(bits(kc), bits(k_ref)) and torch.equal(bits(vc), bits(v_ref))
    assert max_err(out2, ref2) <= TOL16


def test_decode_step_equals_write_then_attend_and_flags_bad_block():
    w = Workload(0, "step2", "bf16", 16, 4, 128, 16, 3, "fixed", writes_new_token=True)
    case = make_decode_case(w, seed=5, lengths=[33, 64, 200])
    bt = case.block_tables.clone()
    kc1, vc1 = case.k_cache.to(DEV), case.v_cache.to(DEV)
    kc2, vc2 = kc1.clone(), vc1.clone()
    out1 = torch.empty(case.q.shape, dtype=torch.float32, device=DEV)
    out2 = torch.empty_like(out1)
    q, nk, nv = case.q.to(DEV), case.new_key.to(DEV), case.new_value.to(DEV)
    pkv.decode_step(out1, q, nk, nv, kc1, vc1, bt.to(DEV), case.context_lens.to(DEV),
                    w.scale, 16, 4)
    slots = torch.tensor([oracle.slot_for_position(bt[s].tolist(), int(L) - 1, 16)
                          for s, L in enumerate(case.lengths)], dtype=torch.int64)
    pkv.kv_write(kc2, vc2, nk, nv, slots.to(DEV))
    pkv.paged_decode_attention(out2, q, kc2, vc2, bt.to(DEV), case.context_lens.to(DEV),
                               w.scale, 16, 4)
    torch.cuda.synchronize()
    assert torch.equal(bits(kc1), bits(kc2)) and torch.equal(bits(vc1), bits(vc2))
    assert torch.equal(out1, out2)  # same kernel, same inputs: same bits
    assert pkv.device_status() == 0
    # a table entry out of range at the new position: no write, flagged
    bt[1, (64 - 1) // 16] = case.num_blocks + 3
    kc3, vc3 = case.k_cache.to(DEV), case.v_cache.to(DEV)
    pkv.decode_step(out1, q, nk, nv, kc3, vc3, bt.to(DEV), case.context_lens.to(DEV),
                    w.scale, 16, 4)
    torch.cuda.synchronize()
    assert pkv.device_status() & 1
    ref0 = oracle.decode_step(case.q[:1], case.new_key[:1], case.new_value[:1],
                              case.k_cache.clone(), case.v_cache.clone(), bt[:1],
                              case.context_lens[:1], w.scale, 16, 4)
    assert max_err(out1[:1], ref0) <= TOL16  # the healthy sequence is unaffected


# --------------------------------------------------------------------------
# paged prefill (causal multi-token queries)
# --------------------------------------------------------------------------

PREFILL_KERNELS = [pytest.param(pkv.PREFILL_TCGEN05, id="tcgen05"),
                   pytest.param(pkv.PREFILL_WARP_MMA, id="warp_mma")]


def gpu_prefill(q, kc, vc, bt, cl, qs, scale, B, Hkv, out_dtype=torch.float32,
                kernel=pkv.PREFILL_TCGEN05):
    pkv.set_prefill_kernel(kernel)
    try:
        out = torch.full(q.shape, float("nan"), dtype=out_dtype, device=DEV)
        qn = (qs[1:] - qs[:-1]).tolist()
        pkv.paged_prefill_attention(out, q.to(DEV), kc, vc, bt.to(DEV), cl.to(DEV), qs.to(DEV),
                                    scale, B, Hkv, max_query_len=max(qn + [0]))
        torch.cuda.synchronize()
        return out
    finally:
        pkv.set_prefill_kernel(pkv.PREFILL_TCGEN05)


PREFILL = [  # dtype, Hq, Hkv, D, B
    ("bf16", 8, 2, 128, 16), ("f16", 4, 4, 128, 32), ("bf16", 16, 2, 64, 8),
    ("f16", 6, 3, 64, 16), ("bf16", 32, 8, 128, 32), ("bf16", 8, 1, 128, 8),
]


@pytest.mark.parametrize("kernel", PREFILL_KERNELS)
@pytest.mark.parametrize("dt,Hq,Hkv,D,B", PREFILL)
def test_prefill_small(dt, Hq, Hkv, D, B, kernel):
    # whole prompts, chunks of longer contexts, single tokens, an empty query
    # set; lengths off every tile boundary
    lengths = [1, 17, 64, 65, 200, 300, 129, 40]
    qn = [1, 17, 64, 65, 77, 1, 128, 0]
    w = Workload(0, "prefill", dt, Hq, Hkv, D, B, len(lengths), "fixed")
    case = make_decode_case(w, seed=Hq + D + B, lengths=lengths)
    qs = torch.tensor([0] + list(np.cumsum(qn)), dtype=torch.int32)
    g = torch.Generator().manual_seed(5)
    q = torch.randn(int(qs[-1]), Hq, D, generator=g).to(w.torch_dtype)
    kc, vc = case.k_cache.to(DEV), case.v_cache.to(DEV)
    out = gpu_prefill(q, kc, vc, case.block_tables, case.context_lens, qs, w.scale, B, Hkv,
                      kernel=kernel)
    ref = oracle.paged_prefill_attention(q, case.k_cache, case.v_cache, case.block_tables,
                                         case.context_lens, qs, w.scale, B, Hkv)
    assert pkv.device_status() == 0
    assert max_err(out, ref) <= TOL16


def test_prefill_many_items_per_persistent_cta():
    # 64 sequences x 32 heads of short prompts: about 14 work items per CTA of
    # the persistent kernel, so every query tile crosses many item boundaries;
    # items with an empty second tile, one-row prompts and no-query sequences
    # are mixed in
    rng = np.random.default_rng(17)
    S = 64
    lengths = rng.integers(1, 400, size=S)
    qn = np.minimum(lengths, rng.choice([0, 1, 7, 128, 129, 255, 256, 300], size=S))
    w = Workload(0, "prefill-many", "bf16", 32, 8, 128, 8, S, "fixed")
    case = make_decode_case(w, seed=18, lengths=lengths.tolist())
    qs = torch.tensor([0] + list(np.cumsum(qn)), dtype=torch.int32)
    q = torch.randn(int(qs[-1]), 32, 128, generator=torch.Generator().manual_seed(9)).to(
        torch.bfloat16)
    kc, vc = case.k_cache.to(DEV), case.v_cache.to(DEV)
    out = gpu_prefill(q, kc, vc, case.block_tables, case.context_lens, qs, w.scale, 8, 8)
    ref = oracle.paged_prefill_attention(q, case.k_cache, case.v_cache, case.block_tables,
                                         case.context_lens, qs, w.scale, 8, 8,
                                         nthreads=oracle.default_threads())
    assert pkv.device_status() == 0
    assert max_err(out, ref) <= TOL16


@pytest.mark.parametrize("kernel", PREFILL_KERNELS)
def test_prefill_long_prompts_and_16bit_out(kernel):
    w = Workload(0, "prefill-long", "bf16", 16, 4, 128, 16, 3, "fixed")
    lengths = [1500, 777, 2048]
    qn = [1500, 300, 1024]
    case = make_decode_case(w, seed=77, lengths=lengths)
    qs = torch.tensor([0] + list(np.cumsum(qn)), dtype=torch.int32)
    q = torch.randn(int(qs[-1]), 16, 128, generator=torch.Generator().manual_seed(6)).to(
        torch.bfloat16)
    kc, vc = case.k_cache.to(DEV), case.v_cache.to(DEV)
    ref = oracle.paged_prefill_attention(q, case.k_cache, case.v_cache, case.block_tables,
                                         case.context_lens, qs, w.scale, 16, 4,
                                         nthreads=oracle.default_threads())
    out = gpu_prefill(q, kc, vc, case.block_tables, case.context_lens, qs, w.scale, 16, 4,
                      kernel=kernel)
    assert max_err(out, ref) <= TOL16
    out16 = gpu_prefill(q, kc, vc, case.block_tables, case.context_lens, qs, w.scale, 16, 4,
                        out_dtype=torch.bfloat16, kernel=kernel)
    diff = np.abs(out16.cpu().double().numpy() - ref)
    assert (diff <= TOL16 + 2.0 ** -8 * np.abs(ref)).all()
    assert pkv.device_status() == 0


@pytest.mark.parametrize("kernel", PREFILL_KERNELS)
def test_prefill_last_row_equals_decode_and_bad_lengths_flag(kernel):
    w = Workload(0, "pd", "f16", 8, 2, 128, 16, 2, "fixed")
    case = make_decode_case(w, seed=8, lengths=[333, 90])
    qn = [40, 90]
    qs = torch.tensor([0, 40, 130], dtype=torch.int32)
    q = torch.randn(130, 8, 128, generator=torch.Generator().manual_seed(1)).to(torch.float16)
    kc, vc = case.k_cache.to(DEV), case.v_cache.to(DEV)
    out = gpu_prefill(q, kc, vc, case.block_tables, case.context_lens, qs, w.scale, 16, 2,
                      kernel=kernel)
    dec = gpu_decode(torch.stack([q[39], q[129]]), kc, vc, case.block_tables, case.context_lens,
                     w.scale, 16, 2)
    assert float((out[[39, 129]] - dec).abs().max()) <= 2 * TOL16
    bad = torch.tensor([0, 40, 130 + 300], dtype=torch.int32)  # 390 rows for a 90-token context
    q2 = torch.zeros(430, 8, 128, dtype=torch.float16)
    out2 = torch.zeros(430, 8, 128, dtype=torch.float32, device=DEV)
    pkv.set_prefill_kernel(kernel)
    try:
        pkv.paged_prefill_attention(out2, q2.to(DEV), kc, vc, case.block_tables.to(DEV),
                                    case.context_lens.to(DEV), bad.to(DEV), w.scale, 16, 2,
                                    max_query_len=390)
    finally:
        pkv.set_prefill_kernel(pkv.PREFILL_TCGEN05)
    assert pkv.device_status() & 2
    assert not out2[40:].any()


@pytest.mark.parametrize("kernel", PREFILL_KERNELS)
def test_prefill_nan_poison_and_bad_block(kernel):
    # Unused cache slots hold NaN: outputs stay finite and match the oracle.
    # A table entry out of range is skipped (its keys masked) and flagged.
    w = Workload(0, "pp", "bf16", 8, 2, 128, 16, 2, "fixed")
    case = make_decode_case(w, seed=31, lengths=[70, 200])
    poison_unused(case.k_cache, case.v_cache, case.block_tables, case.context_lens)
    qs = torch.tensor([0, 70, 70 + 150], dtype=torch.int32)
    q = torch.randn(220, 8, 128, generator=torch.Generator().manual_seed(2)).to(torch.bfloat16)
    kc, vc = case.k_cache.to(DEV), case.v_cache.to(DEV)
    out = gpu_prefill(q, kc, vc, case.block_tables, case.context_lens, qs, w.scale, 16, 2,
                      kernel=kernel)
    ref = oracle.paged_prefill_attention(q, case.k_cache, case.v_cache, case.block_tables,
                                         case.context_lens, qs, w.scale, 16, 2)
    assert torch.isfinite(out).all()
    assert max_err(out, ref) <= TOL16
    assert pkv.device_status() == 0
    bt = case.block_tables.clone()
    bt[1, 2] = case.num_blocks + 5  # tokens 32..47 of sequence 1
    out_bad = gpu_prefill(q, kc, vc, bt, case.context_lens, qs, w.scale, 16, 2, kernel=kernel)
    assert pkv.device_status() & 1
    assert torch.isfinite(out_bad).all()
    assert max_err(out_bad[:70], ref[:70]) <= TOL16  # the healthy sequence is unaffected


@pytest.mark.parametrize("kernel", PREFILL_KERNELS)
@pytest.mark.parametrize("B", [8, 16, 32])
def test_prefill_bad_block_keys_are_masked_exactly(B, kernel):
    # A table entry out of range: the kernel flags it, masks that block's keys
    # and attends to the rest.  Each expected row comes from the oracle's
    # partition form: the runs of visible keys before and after the bad block,
    # merged by their log-sum-exp.
    Hq, Hkv, D, L, qn = 8, 2, 128, 200, 150
    w = Workload(0, "pb", "bf16", Hq, Hkv, D, B, 1, "fixed")
    case = make_decode_case(w, seed=41 + B, lengths=[L])
    qs = torch.tensor([0, qn], dtype=torch.int32)
    q = torch.randn(qn, Hq, D, generator=torch.Generator().manual_seed(3)).to(torch.bfloat16)
    bad = 2  # logical block 2: keys [2B, 3B)
    bt = case.block_tables.clone()
    bt[0, bad] = case.num_blocks + 7
    pkv.device_status(reset=True)
    out = gpu_prefill(q, case.k_cache.to(DEV), case.v_cache.to(DEV), bt, case.context_lens, qs,
                      w.scale, B, Hkv, kernel=kernel)
    assert pkv.device_status() & 1
    pkv.device_status(reset=True)
    K = oracle.gather_sequence(case.k_cache, case.block_tables[0], L)
    V = oracle.gather_sequence(case.v_cache, case.block_tables[0], L)
    Q = oracle.widen(q)
    got = out.double().cpu().numpy()
    lo, hi = bad * B, (bad + 1) * B
    worst = 0.0
    for t in range(qn):
        pos = L - qn + t
        for h in range(Hq):
            g = h // (Hq // Hkv)
            parts = []
            for a, b in ((0, min(lo, pos + 1)), (hi, pos + 1)):
                if b > a:
                    parts += oracle.decode_partitions(Q[t, h], K[a:b, g], V[a:b, g], w.scale,
                                                      b - a)
            worst = max(worst, float(np.abs(got[t, h] - oracle.lse_combine(parts)).max()))
    assert worst <= TOL16


def test_nan_poison_and_physical_permutation():
    # Same logical data paged twice with different physical ids: same output.
    w = Workload(0, "perm", "f16", 16, 4, 128, 16, 4, "fixed")
    a = make_decode_case(w, seed=21, lengths=[50, 129, 7, 260])
    perm = torch.randperm(a.num_blocks, generator=torch.Generator().manual_seed(1))
    kc2 = torch.empty_like(a.k_cache)
    vc2 = torch.empty_like(a.v_cache)
    kc2[perm] = a.k_cache
    vc2[perm] = a.v_cache
    bt2 = torch.where(a.block_tables >= 0, perm[a.block_tables.clamp(min=0).long()].int(),
                      a.block_tables)
    o1 = gpu_decode(a.q, a.k_cache.to(DEV), a.v_cache.to(DEV), a.block_tables, a.context_lens,
                    w.scale, 16, 4)
    o2 = gpu_decode(a.q, kc2.to(DEV), vc2.to(DEV), bt2, a.context_lens, w.scale, 16, 4)
    assert torch.isfinite(o1).all()
    assert torch.equal(o1, o2)


# --------------------------------------------------------------------------
# full-size workloads, in the launch configuration the benchmark times
# --------------------------------------------------------------------------

def full_oracle(q, kc_host, vc_host, bt, cl, w):
    """The oracle's output for every sequence and query head of the batch."""
    return oracle.paged_decode_attention(q, kc_host, vc_host, bt, cl, w.scale, w.block_size,
                                         w.num_kv_heads, nthreads=oracle.default_threads())


_STEPS = {}


def bench_steps(key):
    """The benchmark's host inputs of workload `key` (seed 0), built twice:
    tables from the library's allocator (what the GPU gets) and from the
    oracle's own block manager (what the oracle gets).  One workload is kept
    at a time."""
    import bench
    if key not in _STEPS:
        _STEPS.clear()
        _STEPS[key] = (bench.Step(key, 0, pkv.BlockAllocator), bench.Step(key, 0, BlockManager))
    return _STEPS[key]


@pytest.mark.parametrize("key,grouped,parts", [
    pytest.param(2, False, 1, id="w2-decode_step"),
    pytest.param(3, False, 1, id="w3-gqa"),
    pytest.param(4, False, 1, id="w4-long-context-split"),
    pytest.param(5, True, 1, id="w5-beam-groups"),
    pytest.param(5, True, 2, id="w5-beam-groups-2-parts"),
    pytest.param(5, False, 1, id="w5-ungrouped-decode_step"),
])
def test_full_size_step_as_benchmarked(key, grouped, parts):
    # The very calls bench.py times (its GpuStep: copy-on-write copies, then
    # one decode call that appends each sequence's new token and attends, in
    # the benchmark's launch configuration), at full size, on the benchmark's
    # inputs.  Every output element of every sequence is checked against the
    # oracle, and both caches bit for bit.
    import bench
    st, st_ref = bench_steps(key)
    w = st.w
    assert torch.equal(st.tables, st_ref.tables) and torch.equal(st.lens, st_ref.lens)
    assert torch.equal(st.pairs, st_ref.pairs)
    if st.slots is not None:
        assert torch.equal(st.slots, st_ref.slots)
    g = bench.GpuStep(pkv, st, DEV, grouped, parts)
    g.out.fill_(float("nan"))
    g.run()
    torch.cuda.synchronize()
    assert pkv.device_status() == 0
    # the oracle's step on its own copy of the cache
    kh, vh = st_ref.k_cache.clone(), st_ref.v_cache.clone()
    B = w.block_size
    if st_ref.setup_slots is not None:
        oracle.kv_write(kh, vh, st_ref.setup_keys, st_ref.setup_vals, st_ref.setup_slots, B)
    if st_ref.pairs.shape[0]:
        oracle.kv_copy_blocks(kh, vh, st_ref.pairs)
    if st_ref.slots is not None:
        oracle.kv_write(kh, vh, st_ref.new_key, st_ref.new_value, st_ref.slots, B)
    assert torch.equal(bits(g.kc), bits(kh)) and torch.equal(bits(g.vc), bits(vh))
    ref = full_oracle(st_ref.q, kh, vh, st_ref.tables, st_ref.lens, w)
    out = g.out.cpu().double().numpy()
    assert np.isfinite(out).all()
    err = np.abs(out - ref)
    worst = np.unravel_index(int(err.argmax()), err.shape)
    assert float(err.max()) <= TOL16, ("max abs error %g at (seq, head, d) = %s" %
                                       (float(err.max()), worst))
    # running the step again (its copies and writes are idempotent) gives the
    # same output bits: no state leaks from one launch to the next
    first = g.out.clone()
    g.run()
    torch.cuda.synchronize()
    assert pkv.device_status() == 0
    assert torch.equal(first, g.out)
    del g


def test_workload2_write_then_attend_full_size():
    import bench
    w = WORKLOADS[2]
    case = make_decode_case(w, seed=0, poison=False)
    ref_mgr = BlockManager(case.num_blocks, w.block_size, free_order=case.pool_order)
    gpu_mgr = pkv.BlockAllocator(case.num_blocks, w.block_size, free_order=case.pool_order)
    slots_r, pairs_r, bt_r, cl_r = write_step_schedule(ref_mgr, case.lengths)
    slots, pairs, bt, cl = write_step_schedule(gpu_mgr, case.lengths)
    assert torch.equal(slots, slots_r) and torch.equal(bt, bt_r) and pairs.numel() == 0
    poison_unused(case.k_cache, case.v_cache, bt, case.lengths - 1)
    kc, vc = case.k_cache.to(DEV), case.v_cache.to(DEV)
    P = bench.launch_partition(w, bt.shape[1])
    pkv.kv_write(kc, vc, case.new_key.to(DEV), case.new_value.to(DEV), slots.to(DEV))
    out = gpu_decode(case.q, kc, vc, bt, cl, w.scale, w.block_size, w.num_kv_heads, P=P)
    assert pkv.device_status() == 0
    oracle.kv_write(case.k_cache, case.v_cache, case.new_key, case.new_value, slots_r,
                    w.block_size)
    assert torch.equal(bits(kc), bits(case.k_cache)) and torch.equal(bits(vc), bits(case.v_cache))
    ref = full_oracle(case.q, case.k_cache, case.v_cache, bt_r, cl_r, w)
    assert max_err(out, ref) <= TOL16


def test_workload5_beam_step_full_size():
    import bench
    w = WORKLOADS[5]
    case = make_beam_case(w, seed=0)
    ref_mgr = BlockManager(case.pool_blocks, w.block_size, free_order=case.pool_order)
    gpu_mgr = pkv.BlockAllocator(case.pool_blocks, w.block_size, free_order=case.pool_order)
    host = {}
    for name, mgr in (("ref", ref_mgr), ("gpu", gpu_mgr)):
        pre, suf = beam_setup_schedule(mgr, case)
        host[name] = (pre, suf) + beam_step_schedule(mgr, case)
    pre, suf, ids, slots, pairs, bt, cl = host["gpu"]
    pre_r, suf_r, ids_r, slots_r, pairs_r, bt_r, cl_r = host["ref"]
    assert torch.equal(pre, pre_r) and all(torch.equal(a, b) for a, b in zip(suf, suf_r))
    assert torch.equal(slots, slots_r) and torch.equal(pairs, pairs_r) and torch.equal(bt, bt_r)
    assert pairs.shape[0] > 0  # re-selection shares partial blocks: copies happen

    NB, Hkv, B, D = case.pool_blocks, w.num_kv_heads, w.block_size, w.head_dim
    G, W = case.parents.shape
    kh = torch.full((NB, Hkv, B, D), float("nan"), dtype=torch.float16)
    vh = torch.full_like(kh, float("nan"))
    keys = torch.cat([case.prefix_k.reshape(-1, Hkv, D)] + case.suffix_k)
    vals = torch.cat([case.prefix_v.reshape(-1, Hkv, D)] + case.suffix_v)
    all_slots = torch.cat([pre.reshape(-1)] + suf)
    kc, vc = kh.to(DEV), vh.to(DEV)
    # history (setup), then the timed step: CoW copy, write, attend
    pkv.kv_write(kc, vc, keys.to(DEV), vals.to(DEV), all_slots.to(DEV))
    pkv.kv_copy_blocks(kc, vc, pairs.to(DEV))
    pkv.kv_write(kc, vc, case.new_key.to(DEV), case.new_value.to(DEV), slots.to(DEV))
    P = bench.launch_partition(w, bt.shape[1])
    out = gpu_decode(case.q, kc, vc, bt, cl, w.scale, B, Hkv, P=P)
    assert pkv.device_status() == 0
    oracle.kv_write(kh, vh, keys, vals, torch.cat([pre_r.reshape(-1)] + suf_r), B)
    oracle.kv_copy_blocks(kh, vh, pairs_r)
    oracle.kv_write(kh, vh, case.new_key, case.new_value, slots_r, B)
    assert torch.equal(bits(kc), bits(kh)) and torch.equal(bits(vc), bits(vh))
    ref = full_oracle(case.q, kh, vh, bt_r, cl_r, w)
    assert max_err(out, ref) <= TOL16
    # isolation: each beam sees its parent's history plus its own new token
    g0 = 0
    for b in range(W):
        par = g0 * W + int(case.parents[g0, b])
        n = int(case.suffix[par])
        K = oracle.gather_sequence(kh, bt_r[b].tolist(), int(cl_r[b]))
        expect = torch.cat([case.prefix_k[g0], case.suffix_k[par], case.new_key[b:b + 1]])
        assert int(cl_r[b]) == w.prefix_len + n + 1
        assert np.array_equal(K, expect.double().numpy())


# --------------------------------------------------------------------------
# Beam groups: sequences sharing a prefix of physical blocks, attended by one
# CTA per (group, KV head) that reads each shared tile once
# --------------------------------------------------------------------------

def make_group_case(dt, Hq, Hkv, D, B, groups, seed, step):
    """groups: list of (shared blocks, [tail tokens per member]).  Members of
    a group hold the same first `shared blocks` ids, then blocks of their own
    for the tail; unused slots are NaN.  With step, each member's last token
    is the new one (its slot NaN until the step writes it)."""
    g = torch.Generator().manual_seed(seed)
    dtype = {"bf16": torch.bfloat16, "f16": torch.float16}[dt]
    rows, lens = [], []
    nxt = 0
    for nsh, tails in groups:
        shared_ids = list(range(nxt, nxt + nsh))
        nxt += nsh
        for t in tails:
            own = -(-t // B)
            rows.append(shared_ids + list(range(nxt, nxt + own)))
            nxt += own
            lens.append(nsh * B + t)
    NB = nxt + 3
    perm = torch.randperm(NB, generator=g).tolist()  # physical ids in shuffled order
    S = len(rows)
    mb = max(len(r) for r in rows)
    bt = torch.full((S, mb), -1, dtype=torch.int32)
    for s, r in enumerate(rows):
        bt[s, :len(r)] = torch.tensor([perm[i] for i in r], dtype=torch.int32)
    cl = torch.tensor(lens, dtype=torch.int32)
    kc = torch.randn(NB, Hkv, B, D, generator=g).to(dtype)
    vc = torch.randn(NB, Hkv, B, D, generator=g).to(dtype)
    # NaN in every slot no sequence attends (and in the new tokens' slots)
    used = torch.zeros(NB, B, dtype=torch.bool)
    for s in range(S):
        n = int(cl[s]) - (1 if step else 0)
        for i in range(n):
            used[int(bt[s, i // B]), i % B] = True
    unused = (~used)[:, None, :, None].expand_as(kc)
    kc[unused] = float("nan")
    vc[unused] = float("nan")
    q = torch.randn(S, Hq, D, generator=g).to(dtype)
    nk = torch.randn(S, Hkv, D, generator=g).to(dtype)
    nv = torch.randn(S, Hkv, D, generator=g).to(dtype)
    gs = [0]
    for _, tails in groups:
        gs.append(gs[-1] + len(tails))
    return q, kc, vc, bt, cl, torch.tensor(gs, dtype=torch.int32), nk, nv


GROUP_CASES = [  # dtype, Hq, Hkv, D, B, groups (shared blocks, member tails)
    ("f16", 8, 8, 128, 16, [(64, [1, 40, 256, 0]), (3, [17, 1]), (0, [5, 9, 100]), (10, [33])]),
    ("bf16", 4, 4, 64, 8, [(5, [1, 2, 3, 4, 5, 6, 7, 8]), (12, [60, 0])]),
    ("bf16", 16, 8, 128, 32, [(4, [16, 33, 1, 64]), (2, [31])]),
    ("f16", 8, 2, 128, 16, [(9, [7, 70]), (1, [1, 2])]),
    ("bf16", 16, 2, 64, 16, [(3, [50])]),  # G = 8: one member per group
    # two n8 column tiles: 12 columns (G = 2 x 6), 16 (G = 4 x 4), 16 (G = 1 x
    # 16 members), and G = 16 alone
    ("bf16", 8, 4, 64, 16, [(6, [3, 9, 17, 40, 1, 2]), (1, [5, 5])]),
    ("f16", 16, 4, 128, 16, [(12, [5, 30, 1, 64]), (2, [7])]),
    ("bf16", 4, 4, 128, 32, [(3, list(range(1, 17)))]),
    ("f16", 32, 2, 64, 8, [(20, [9]), (0, [3])]),
]


def group_ws(q, parts):
    S, Hq, D = q.shape
    if parts <= 1:
        return None
    return torch.empty(pkv.decode_workspace_bytes(S, Hq, D, parts, 1), dtype=torch.uint8,
                       device=DEV)


@pytest.mark.parametrize("parts", [1, 2, 5])
@pytest.mark.parametrize("step", [False, True])
@pytest.mark.parametrize("dt,Hq,Hkv,D,B,groups", GROUP_CASES)
def test_beam_groups_match_oracle(dt, Hq, Hkv, D, B, groups, step, parts):
    # parts > 1 cuts each group's stage list over that many CTAs (some runs
    # empty when a group has fewer stages), merged inside the launch
    if step:  # a decode step needs a new token in each member's own tail
        groups = [(nsh, [max(t, 1) for t in tails]) for nsh, tails in groups]
    q, kc, vc, bt, cl, gs, nk, nv = make_group_case(dt, Hq, Hkv, D, B, groups, seed=Hq + B + D,
                                                    step=step)
    scale = D ** -0.5
    sh = pkv.group_shared_tokens(bt, cl, gs, B)
    for i, (nsh, tails) in enumerate(groups):  # the helper finds the shared blocks
        expect = min(nsh * B, min(nsh * B + t for t in tails)) if len(tails) > 1 else \
            nsh * B + tails[0]
        assert int(sh[i]) == expect
    kd, vd = kc.to(DEV), vc.to(DEV)
    out = torch.full(q.shape, float("nan"), dtype=torch.float32, device=DEV)
    pkv.paged_decode_grouped(out, q.to(DEV), kd, vd, bt.to(DEV), cl.to(DEV), gs.to(DEV),
                             sh.to(DEV), scale, B, Hkv,
                             new_k=nk.to(DEV) if step else None,
                             new_v=nv.to(DEV) if step else None,
                             parts=parts, workspace=group_ws(q, parts))
    torch.cuda.synchronize()
    assert pkv.device_status() == 0
    if step:
        k_ref, v_ref = kc.clone(), vc.clone()
        ref = oracle.decode_step(q, nk, nv, k_ref, v_ref, bt, cl, scale, B, Hkv)
        assert torch.equal(bits(kd), bits(k_ref)) and torch.equal(bits(vd), bits(v_ref))
    else:
        ref = oracle.paged_decode_attention(q, kc, vc, bt, cl, scale, B, Hkv)
    assert max_err(out, ref) <= TOL16


def test_beam_groups_equal_ungrouped_step_and_flag_oversized_groups():
    groups = [(20, [3, 90, 1, 17]), (6, [40, 41])]
    q, kc, vc, bt, cl, gs, nk, nv = make_group_case("f16", 8, 8, 128, 16, groups, seed=3,
                                                    step=True)
    sh = pkv.group_shared_tokens(bt, cl, gs, 16)
    k1, v1 = kc.to(DEV), vc.to(DEV)
    k2, v2 = k1.clone(), v1.clone()
    o1 = torch.empty(q.shape, dtype=torch.float32, device=DEV)
    o2 = torch.empty_like(o1)
    pkv.paged_decode_grouped(o1, q.to(DEV), k1, v1, bt.to(DEV), cl.to(DEV), gs.to(DEV),
                             sh.to(DEV), 128 ** -0.5, 16, 8, new_k=nk.to(DEV), new_v=nv.to(DEV))
    pkv.decode_step(o2, q.to(DEV), nk.to(DEV), nv.to(DEV), k2, v2, bt.to(DEV), cl.to(DEV),
                    128 ** -0.5, 16, 8)
    torch.cuda.synchronize()
    assert pkv.device_status() == 0
    assert torch.equal(bits(k1), bits(k2)) and torch.equal(bits(v1), bits(v2))
    assert float((o1 - o2).abs().max()) <= TOL16
    # nine members with two query heads each (G = 2) need 18 > 16 columns; six
    # need 12, more than one tile holds when max_members = 4 picks the
    # one-tile kernel: either way the group is skipped and flagged
    for members, max_members in ((9, None), (6, 4)):
        q6, kc6, vc6, bt6, cl6, gs6, _, _ = make_group_case(
            "f16", 16, 8, 128, 16, [(4, list(range(1, members + 1)))], seed=4, step=False)
        out = torch.full(q6.shape, 7.0, dtype=torch.float32, device=DEV)
        pkv.paged_decode_grouped(out, q6.to(DEV), kc6.to(DEV), vc6.to(DEV), bt6.to(DEV),
                                 cl6.to(DEV), gs6.to(DEV),
                                 pkv.group_shared_tokens(bt6, cl6, gs6, 16).to(DEV),
                                 128 ** -0.5, 16, 8, max_members=max_members)
        torch.cuda.synchronize()
        assert pkv.device_status() & 2  # bad context length / group
        assert bool((out == 7.0).all())  # nothing written for the skipped group
        pkv.device_status(reset=True)
    # the same six with the default bound take the two-tile kernel
    out = torch.full(q6.shape, float("nan"), dtype=torch.float32, device=DEV)
    pkv.paged_decode_grouped(out, q6.to(DEV), kc6.to(DEV), vc6.to(DEV), bt6.to(DEV),
                             cl6.to(DEV), gs6.to(DEV),
                             pkv.group_shared_tokens(bt6, cl6, gs6, 16).to(DEV),
                             128 ** -0.5, 16, 8)
    torch.cuda.synchronize()
    assert pkv.device_status() == 0
    ref = oracle.paged_decode_attention(q6, kc6, vc6, bt6, cl6, 128 ** -0.5, 16, 8)
    assert max_err(out, ref) <= TOL16


@pytest.mark.parametrize("parts,hint", [(1, True), (2, False)])
def test_workload5_grouped_step_full_size(parts, hint):
    # the benchmark's beam step through the beam-group call: CoW copy, then
    # one launch that appends every beam's new token and attends the group
    # (the bench's launch: one CTA a group and KV head, the one-tile kernel
    # picked by the beam width as member bound; and each group's stages over
    # two CTAs on the two-tile kernel the default bound picks)
    w = WORKLOADS[5]
    case = make_beam_case(w, seed=1)
    mgr = pkv.BlockAllocator(case.pool_blocks, w.block_size, free_order=case.pool_order)
    pre, suf = beam_setup_schedule(mgr, case)
    ids, slots, pairs, bt, cl = beam_step_schedule(mgr, case)
    NB, Hkv, B, D = case.pool_blocks, w.num_kv_heads, w.block_size, w.head_dim
    G, W = case.parents.shape
    kh = torch.full((NB, Hkv, B, D), float("nan"), dtype=torch.float16)
    vh = torch.full_like(kh, float("nan"))
    keys = torch.cat([case.prefix_k.reshape(-1, Hkv, D)] + case.suffix_k)
    vals = torch.cat([case.prefix_v.reshape(-1, Hkv, D)] + case.suffix_v)
    all_slots = torch.cat([pre.reshape(-1)] + suf)
    oracle.kv_write(kh, vh, keys, vals, all_slots, B)
    oracle.kv_copy_blocks(kh, vh, pairs)
    kc, vc = kh.to(DEV), vh.to(DEV)  # history and copies in place; new tokens not yet
    gs = torch.arange(0, G * W + 1, W, dtype=torch.int32)
    sh = pkv.group_shared_tokens(bt, cl, gs, B)
    assert int(sh.min()) >= w.prefix_len  # every group shares at least its prompt
    out = torch.full(case.q.shape, float("nan"), dtype=torch.float32, device=DEV)
    pkv.paged_decode_grouped(out, case.q.to(DEV), kc, vc, bt.to(DEV), cl.to(DEV), gs.to(DEV),
                             sh.to(DEV), w.scale, B, Hkv, new_k=case.new_key.to(DEV),
                             new_v=case.new_value.to(DEV), parts=parts,
                             workspace=group_ws(case.q, parts), max_members=W if hint else None)
    torch.cuda.synchronize()
    assert pkv.device_status() == 0
    oracle.kv_write(kh, vh, case.new_key, case.new_value, slots, B)
    assert torch.equal(bits(kc), bits(kh)) and torch.equal(bits(vc), bits(vh))
    ref = full_oracle(case.q, kh, vh, bt, cl, w)
    assert max_err(out, ref) <= TOL16
    assert bool(torch.isfinite(out).all())


@pytest.mark.parametrize("parts", [16, 64])
def test_parallel_sampling_of_one_long_prompt_over_many_parts(parts):
    # one group: four samples share a 4096-token prompt (256 blocks) and hold
    # tails of their own; 16 or 64 CTAs a KV head split the 260-odd stages
    groups = [(256, [1, 16, 7, 12])]
    q, kc, vc, bt, cl, gs, _, _ = make_group_case("bf16", 32, 8, 128, 16, groups, seed=21,
                                                  step=False)
    sh = pkv.group_shared_tokens(bt, cl, gs, 16)
    assert int(sh[0]) == 4096  # the prompt's blocks
    out = torch.full(q.shape, float("nan"), dtype=torch.float32, device=DEV)
    pkv.paged_decode_grouped(out, q.to(DEV), kc.to(DEV), vc.to(DEV), bt.to(DEV), cl.to(DEV),
                             gs.to(DEV), sh.to(DEV), 128 ** -0.5, 16, 8, parts=parts,
                             workspace=group_ws(q, parts))
    torch.cuda.synchronize()
    assert pkv.device_status() == 0
    ref = oracle.paged_decode_attention(q, kc, vc, bt, cl, 128 ** -0.5, 16, 8)
    assert max_err(out, ref) <= TOL16


@pytest.mark.parametrize("parts", [1, 4])
def test_beam_groups_empty_members_and_uncovered_sequences(parts):
    # a member with no tokens gets a zero row; sequences outside every group
    # are not touched
    groups = [(2, [0, 30, 5]), (0, [0]), (3, [7, 9])]
    q, kc, vc, bt, cl, gs, _, _ = make_group_case("bf16", 8, 8, 128, 16, groups, seed=8,
                                                  step=False)
    cl = cl.clone()
    cl[0] = 0  # first member of group 0: empty
    gs_part = gs[:3].clone()  # groups 0 and 1 only; group 2's sequences uncovered
    sh = pkv.group_shared_tokens(bt, cl, gs_part, 16)
    assert int(sh[0]) == 0  # the empty member shares nothing
    out = torch.full(q.shape, 5.0, dtype=torch.float32, device=DEV)
    pkv.paged_decode_grouped(out, q.to(DEV), kc.to(DEV), vc.to(DEV), bt.to(DEV), cl.to(DEV),
                             gs_part.to(DEV), sh.to(DEV), 128 ** -0.5, 16, 8, parts=parts,
                             workspace=group_ws(q, parts))
    torch.cuda.synchronize()
    assert pkv.device_status() == 0
    ref = oracle.paged_decode_attention(q, kc, vc, bt, cl, 128 ** -0.5, 16, 8)
    covered = int(gs_part[-1])
    assert max_err(out[:covered], ref[:covered]) <= TOL16
    assert bool((out[0] == 0).all())
    assert bool((out[covered:] == 5.0).all())


# dtype, Hq, Hkv, B, members per group, decode step, parts (all head_dim 128)
WAVE_CASES = [
    ("f16", 32, 32, 16, 4, True, 1),    # one n8 tile (4 columns)
    ("bf16", 64, 32, 32, 3, False, 2),  # G = 2, 6 columns; two CTAs a group and KV head
    ("bf16", 32, 16, 8, 6, True, 1),    # G = 2, 12 columns: two tiles
    ("f16", 16, 16, 16, 16, False, 3),  # 16 members: two tiles, three CTAs
]


@pytest.mark.parametrize("dt,Hq,Hkv,B,members,step,parts", WAVE_CASES)
def test_beam_groups_over_more_than_one_wave(dt, Hq, Hkv, B, members, step, parts):
    # groups x KV heads x parts is about 4.5 CTAs a SM (a wave holds three),
    # with ragged shared prefixes and tails: CTAs of the second wave reuse the
    # shared memory and counters' neighbours of the first
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    n = -(-(9 * sms // 2) // (Hkv * parts))
    assert 3 * sms < n * Hkv * parts <= 6 * sms
    g = torch.Generator().manual_seed(Hq + members)
    groups = []
    for _ in range(n):
        nsh = int(torch.randint(0, 7, (1,), generator=g))
        tails = torch.randint(1 if step else 0, 41, (members,), generator=g).tolist()
        groups.append((nsh, tails))
    q, kc, vc, bt, cl, gs, nk, nv = make_group_case(dt, Hq, Hkv, 128, B, groups, seed=members,
                                                    step=step)
    scale = 128 ** -0.5
    sh = pkv.group_shared_tokens(bt, cl, gs, B)
    kd, vd = kc.to(DEV), vc.to(DEV)
    out = torch.full(q.shape, float("nan"), dtype=torch.float32, device=DEV)
    pkv.paged_decode_grouped(out, q.to(DEV), kd, vd, bt.to(DEV), cl.to(DEV), gs.to(DEV),
                             sh.to(DEV), scale, B, Hkv,
                             new_k=nk.to(DEV) if step else None,
                             new_v=nv.to(DEV) if step else None,
                             parts=parts, workspace=group_ws(q, parts), max_members=members)
    torch.cuda.synchronize()
    assert pkv.device_status() == 0
    if step:
        k_ref, v_ref = kc.clone(), vc.clone()
        ref = oracle.decode_step(q, nk, nv, k_ref, v_ref, bt, cl, scale, B, Hkv)
        assert torch.equal(bits(kd), bits(k_ref)) and torch.equal(bits(vd), bits(v_ref))
    else:
        ref = oracle.paged_decode_attention(q, kc, vc, bt, cl, scale, B, Hkv)
    assert max_err(out, ref) <= TOL16
    assert bool(torch.isfinite(out).all())


# --------------------------------------------------------------------------
# The work plan itself, and the calls replayed from a CUDA graph
# --------------------------------------------------------------------------

def _align256(x):
    return (x + 255) // 256 * 256


@pytest.mark.parametrize("P", [0, 64, 512])
def test_work_plan_records_cover_every_cta_once_longest_first(P):
    # The plan's records (in the workspace, as include/pkv.h lays it out):
    # one per CTA with work, each (sequence, KV head x head slice, partition
    # group) exactly once, sequences in non-increasing order of length
    # (counting-sort buckets are exact below 2048 tokens), the head slices of
    # one group adjacent.
    rng = np.random.default_rng(P + 5)
    lengths = [int(x) for x in rng.permutation([0, 1, 17, 300, 700, 1500, 2000, 64, 65, 999])]
    Hq, Hkv, D, B = 48, 2, 128, 16  # G = 24: two head slices of 12
    w = Workload(0, "plan", "bf16", Hq, Hkv, D, B, len(lengths), "fixed")
    case = make_decode_case(w, seed=3, lengths=lengths)
    S = len(lengths)
    maxb = case.block_tables.shape[1]
    n = pkv.decode_workspace_bytes(S, Hq, D, maxb * B, P)
    ws = torch.zeros(n, dtype=torch.uint8, device=DEV)
    out = torch.empty((S, Hq, D), dtype=torch.float32, device=DEV)
    pkv.paged_decode_attention(out, case.q.to(DEV), case.k_cache.to(DEV), case.v_cache.to(DEV),
                               case.block_tables.to(DEV), case.context_lens.to(DEV), w.scale, B,
                               Hkv, partition_size=P, workspace=ws)
    torch.cuda.synchronize()
    assert pkv.device_status() == 0
    if P == 0:
        count_off, items_off = 0, 256
        groups = [1] * S
    else:
        nP = -(-maxb * B // P)
        ml = _align256(S * Hq * 4)
        o = ml + _align256(S * Hq * nP * 8)
        count_off = o + _align256(S * Hq * nP * D * 4)
        items_off = count_off + 256
        cta_parts = 4 if (P <= 512 and nP >= 16) else 1
        groups = [-(-max(1, -(-L // P)) // cta_parts) for L in lengths]
    host = ws.cpu()
    count = int(host[count_off:count_off + 4].view(torch.int32)[0])
    HS = 2
    assert count == sum(Hkv * HS * g for g in groups)
    rec = host[items_off:items_off + count * 16].view(torch.int32).view(count, 4).tolist()
    seen = set()
    for s_, L, gh, grp in rec:
        assert L == lengths[s_] and 0 <= gh < Hkv * HS and 0 <= grp < groups[s_]
        seen.add((s_, gh, grp))
    assert len(seen) == count
    order = [r[0] for r in rec]
    firsts = list(dict.fromkeys(order))  # sequences in plan order
    assert sorted(firsts) == list(range(S))
    assert [lengths[s_] for s_ in firsts] == sorted(lengths, reverse=True)
    for i in range(0, count, HS):  # slices of one (sequence, KV head, group) adjacent
        a, b = rec[i], rec[i + 1]
        assert a[0] == b[0] and a[3] == b[3] and a[2] // HS == b[2] // HS
    ref = oracle.paged_decode_attention(case.q, case.k_cache, case.v_cache, case.block_tables,
                                        case.context_lens, w.scale, B, Hkv)
    assert max_err(out, ref) <= TOL16


def _plan_pieces(items, slots, cmax):
    # the plan's choice of pieces per sequence for near-equal contexts: the
    # fewest whose CTAs fill their last wave to 95 %, else the fullest
    best, best_ctas, best_room = 1, 0, 1
    for c in range(1, cmax + 1):
        ctas = items * c
        room = -(-ctas // slots) * slots
        if 100 * ctas >= 95 * room:
            return c
        if ctas * best_room > best_ctas * room:
            best, best_ctas, best_room = c, ctas, room
    return best


# dtype, Hq, Hkv, D, B, context lengths, partition tokens, decode step
PIECE_CASES = [
    ("bf16", 32, 8, 128, 32, [8000, 8600, 8301, 8450], 512, False),  # partitions a warp
    ("bf16", 8, 8, 64, 16, [3000, 3100, 3071], 256, True),           # 32-token stages, append
    ("f16", 48, 2, 128, 16, [1950, 2048, 2000, 1999, 2040], 1024, False),  # head slices
    ("bf16", 32, 8, 128, 16, [4096] * 39 + [0], 512, True),          # many, and an empty one
]


@pytest.mark.parametrize("dt,Hq,Hkv,D,B,lengths,P,step", PIECE_CASES)
def test_split_near_equal_contexts_in_equal_pieces(dt, Hq, Hkv, D, B, lengths, P, step):
    # Contexts within 10 % of the same stage count: the plan cuts each into
    # the same number of equal runs of stages (pieces), as many as fill the
    # GPU's waves, instead of partition groups; the records say so and the
    # result is unchanged.
    S = len(lengths)
    w = Workload(0, "pieces", dt, Hq, Hkv, D, B, S, "fixed", writes_new_token=step)
    case = make_decode_case(w, seed=S + D, lengths=lengths)
    maxb = case.block_tables.shape[1]
    nP = -(-maxb * B // P)
    n = pkv.decode_workspace_bytes(S, Hq, D, maxb * B, P)
    ws = torch.zeros(n, dtype=torch.uint8, device=DEV)
    out = torch.full((S, Hq, D), float("nan"), dtype=torch.float32, device=DEV)
    kc, vc = case.k_cache.to(DEV), case.v_cache.to(DEV)
    if step:
        pkv.decode_step(out, case.q.to(DEV), case.new_key.to(DEV), case.new_value.to(DEV), kc,
                        vc, case.block_tables.to(DEV), case.context_lens.to(DEV), w.scale, B,
                        Hkv, partition_size=P, workspace=ws)
    else:
        pkv.paged_decode_attention(out, case.q.to(DEV), kc, vc, case.block_tables.to(DEV),
                                   case.context_lens.to(DEV), w.scale, B, Hkv, partition_size=P,
                                   workspace=ws)
    torch.cuda.synchronize()
    assert pkv.device_status() == 0
    # the records
    G = Hq // Hkv
    HS = -(-G // 16)
    cta_parts = 4 if (P <= 512 and nP >= 16) else 1
    max_groups = -(-nP // cta_parts)
    ST = 32 if D == 64 else 16
    nst = [-(-L // ST) for L in lengths if L > 0]
    assert 10 * max(nst) <= 11 * min(nst)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    cmax = min(min(-(-L // P) for L in lengths if L > 0), max_groups, 64)
    pieces = _plan_pieces(len(nst) * Hkv * HS, 3 * sms, cmax)
    ml = _align256(S * Hq * 4)
    o = ml + _align256(S * Hq * nP * 8)
    count_off = o + _align256(S * Hq * nP * D * 4)
    host = ws.cpu()
    count = int(host[count_off:count_off + 4].view(torch.int32)[0])
    per = [pieces if L > 0 else 1 for L in lengths]
    assert count == sum(Hkv * HS * c for c in per)
    rec = host[count_off + 256:count_off + 256 + count * 16].view(torch.int32).view(count, 4)
    seen = set()
    for s_, L, gh, wv in rec.tolist():
        assert L == lengths[s_] and 0 <= gh < Hkv * HS
        assert wv & (1 << 30)  # a piece
        i, c = wv & 0x7FFF, (wv >> 15) & 0x7FFF
        assert c == per[s_] and 0 <= i < c
        seen.add((s_, gh, i))
    assert len(seen) == count
    # the result
    if step:
        k_ref, v_ref = case.k_cache.clone(), case.v_cache.clone()
        ref = oracle.decode_step(case.q, case.new_key, case.new_value, k_ref, v_ref,
                                 case.block_tables, case.context_lens, w.scale, B, Hkv,
                                 nthreads=oracle.default_threads())
        assert torch.equal(bits(kc), bits(k_ref)) and torch.equal(bits(vc), bits(v_ref))
    else:
        ref = oracle.paged_decode_attention(case.q, case.k_cache, case.v_cache,
                                            case.block_tables, case.context_lens, w.scale, B,
                                            Hkv, nthreads=oracle.default_threads())
    assert max_err(out, ref) <= TOL16
    assert bool(torch.isfinite(out).all())


# dtype, Hq, Hkv, D, B (the items per sequence: Hkv x head slices)
SHALLOW_CASES = [
    ("bf16", 16, 16, 128, 16),
    ("f16", 64, 8, 64, 32),
    ("bf16", 96, 8, 128, 8),   # G = 12: two column tiles
    ("f16", 32, 32, 64, 8),
    ("bf16", 48, 2, 128, 32),  # G = 24: two head slices
]


@pytest.mark.parametrize("plan", [False, True])
@pytest.mark.parametrize("dt,Hq,Hkv,D,B", SHALLOW_CASES)
def test_unsplit_launch_of_many_items(dt, Hq, Hkv, D, B, plan):
    # An unsplit launch of more items (sequence x KV head x head slice) than
    # two waves of three CTAs a SM keeps 2-stage rings, three CTAs a SM; fewer
    # items (every other small test) get 3-stage rings, two a SM.  Short
    # ragged contexts, some empty, with and without the work plan.
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    HS = -(-(Hq // Hkv) // 16)
    S = -(-(13 * sms) // (2 * Hkv * HS))
    assert S * Hkv * HS > 6 * sms
    rng = np.random.default_rng(S + D + B)
    lengths = [int(x) for x in rng.integers(0, 300, size=S)]
    w = Workload(0, "shallow", dt, Hq, Hkv, D, B, S, "fixed")
    case = make_decode_case(w, seed=D + B, lengths=lengths)
    ws = None
    if plan:
        n = pkv.decode_workspace_bytes(S, Hq, D, case.block_tables.shape[1] * B, 0)
        ws = torch.empty(n, dtype=torch.uint8, device=DEV)
    out = torch.full((S, Hq, D), float("nan"), dtype=torch.float32, device=DEV)
    pkv.paged_decode_attention(out, case.q.to(DEV), case.k_cache.to(DEV), case.v_cache.to(DEV),
                               case.block_tables.to(DEV), case.context_lens.to(DEV), w.scale, B,
                               Hkv, workspace=ws)
    torch.cuda.synchronize()
    assert pkv.device_status() == 0
    ref = oracle.paged_decode_attention(case.q, case.k_cache, case.v_cache, case.block_tables,
                                        case.context_lens, w.scale, B, Hkv,
                                        nthreads=oracle.default_threads())
    assert max_err(out, ref) <= TOL16
    assert bool(torch.isfinite(out).all())


@pytest.mark.parametrize("call", ["unsplit", "split", "step", "grouped", "f32_split"])
def test_query_and_output_in_pinned_host_memory(call):
    # q and out may be pinned host memory: the kernel loads q and stores the
    # output rows over the host link; the result is the same bits as with
    # device tensors
    lengths = [1, 700, 33, 2049, 0, 1500]
    dt = "f32" if call == "f32_split" else "bf16"  # fp32: the CUDA-core kernel and its merge
    w = Workload(0, "hostout", dt, 32, 8, 128, 16, len(lengths), "fixed",
                 writes_new_token=(call == "step"))
    case = make_decode_case(w, seed=77, lengths=lengths)
    S, Hq, D = case.q.shape
    maxb = case.block_tables.shape[1]
    outs = []
    for host in (False, True):
        kc, vc = case.k_cache.to(DEV), case.v_cache.to(DEV)
        q = case.q.pin_memory() if host else case.q.to(DEV)
        bt, cl = case.block_tables.to(DEV), case.context_lens.to(DEV)
        out = torch.full((S, Hq, D), float("nan"), dtype=torch.float32)
        out = out.pin_memory() if host else out.to(DEV)
        if call == "grouped":
            gs = torch.tensor([0, 2, 3, 6], dtype=torch.int32)
            sh = pkv.group_shared_tokens(case.block_tables, case.context_lens, gs, 16)
            pkv.paged_decode_grouped(out, q, kc, vc, bt, cl, gs.to(DEV), sh.to(DEV), w.scale, 16,
                                     8)
        elif call == "step":
            pkv.decode_step(out, q, case.new_key.to(DEV), case.new_value.to(DEV), kc, vc, bt, cl,
                            w.scale, 16, 8)
        else:
            P = 512 if call in ("split", "f32_split") else 0
            ws = torch.empty(pkv.decode_workspace_bytes(S, Hq, D, maxb * 16, P),
                             dtype=torch.uint8, device=DEV)
            pkv.paged_decode_attention(out, q, kc, vc, bt, cl, w.scale, 16, 8, partition_size=P,
                                       workspace=ws)
        torch.cuda.synchronize()
        assert pkv.device_status() == 0
        outs.append(out.cpu())
    assert torch.equal(outs[0], outs[1])
    if call == "step":
        k_ref, v_ref = case.k_cache.clone(), case.v_cache.clone()
        ref = oracle.decode_step(case.q, case.new_key, case.new_value, k_ref, v_ref,
                                 case.block_tables, case.context_lens, w.scale, 16, 8)
    else:
        ref = oracle.paged_decode_attention(case.q, case.k_cache, case.v_cache, case.block_tables,
                                            case.context_lens, w.scale, 16, 8)
    assert max_err(outs[1], ref) <= (TOL32 if dt == "f32" else TOL16)


def _relayout(case, B_new, seed):
    """The same logical K/V of every sequence in a fresh pool of block size
    B_new, in a random physical order, unused slots NaN."""
    S = len(case.lengths)
    _, Hkv, B, D = case.k_cache.shape
    g = torch.Generator().manual_seed(seed)
    need = [-(-int(L) // B_new) for L in case.lengths]
    NB = sum(need) + 5
    perm = torch.randperm(NB, generator=g)
    maxb = max(max(need), 1)
    tables = torch.full((S, maxb), -1, dtype=torch.int32)
    kc = torch.full((NB, Hkv, B_new, D), float("nan"), dtype=case.k_cache.dtype)
    vc = torch.full_like(kc, float("nan"))
    nxt = 0
    for s_, L in enumerate(case.lengths):
        L = int(L)
        pos = torch.arange(L)
        old = case.block_tables[s_, (pos // B).long()].long()
        ks = case.k_cache[old, :, (pos % B).long()]  # [L, Hkv, D]
        vs = case.v_cache[old, :, (pos % B).long()]
        ids = perm[nxt:nxt + need[s_]]
        nxt += need[s_]
        tables[s_, :need[s_]] = ids.to(torch.int32)
        new = ids[(pos // B_new).long()]
        kc[new, :, (pos % B_new).long()] = ks
        vc[new, :, (pos % B_new).long()] = vs
    return kc, vc, tables


@pytest.mark.parametrize("D,P", [(128, 0), (128, 512), (64, 0), (64, 256)])
def test_paging_changes_storage_not_output_bits(D, P):
    # Paging changes where K/V live, not what attention reads: the same
    # logical K/V in pools of block size 8, 16 and 32, each in its own random
    # physical order, give the decode kernel's output bit for bit (a stage
    # holds the same tokens at every block size), within the tolerance of
    # the oracle.
    lengths = [1, 15, 16, 17, 300, 1000, 2049, 513]
    w = Workload(0, "paging", "bf16", 32, 8, D, 16, len(lengths), "fixed")
    case = make_decode_case(w, seed=D + P, lengths=lengths)
    S, Hq, _ = case.q.shape
    outs = []
    for i, Bn in enumerate((16, 8, 32, 16)):
        kc, vc, bt = _relayout(case, Bn, seed=i + 1)
        out = torch.full((S, Hq, D), float("nan"), dtype=torch.float32, device=DEV)
        ws = None
        if P:
            ws = torch.empty(pkv.decode_workspace_bytes(S, Hq, D, bt.shape[1] * Bn, P),
                             dtype=torch.uint8, device=DEV)
        pkv.paged_decode_attention(out, case.q.to(DEV), kc.to(DEV), vc.to(DEV), bt.to(DEV),
                                   case.context_lens.to(DEV), w.scale, Bn, 8, partition_size=P,
                                   workspace=ws)
        torch.cuda.synchronize()
        assert pkv.device_status() == 0
        outs.append(out.cpu())
    for o in outs[1:]:
        assert torch.equal(o, outs[0])
    ref = oracle.paged_decode_attention(case.q, case.k_cache, case.v_cache, case.block_tables,
                                        case.context_lens, w.scale, 16, 8)
    assert max_err(outs[0], ref) <= TOL16


def _random_decode_config(i):
    """Configuration i of the seeded random sweep: dtype, heads, head_dim, block size,
    lengths (ragged, or near-equal so that a split call gets pieces), split, plan, step."""
    r = np.random.default_rng(1000 + i)
    dt = ["bf16", "f16"][int(r.integers(2))]
    Hkv = int(r.choice([1, 2, 4, 8]))
    G = int(r.choice([1, 2, 4, 6, 8, 12, 16, 24, 32]))
    D = int(r.choice([64, 128]))
    B = int(r.choice([8, 16, 32]))
    S = int(r.integers(1, 24))
    if r.random() < 0.4:  # near-equal contexts
        base = int(r.integers(40, 900))
        lengths = [base + int(x) for x in r.integers(0, max(1, base // 12), size=S)]
    else:
        lengths = [int(x) for x in r.integers(0, 1200, size=S)]
    P = int(r.choice([0, 0, 0, B, 2 * B, 8 * B, 16 * B]))
    plan = bool(r.integers(2)) if P == 0 else True
    step = bool(r.integers(2))
    if step:
        lengths = [max(1, L) for L in lengths]
    return dt, Hkv * G, Hkv, D, B, lengths, P, plan, step


@pytest.mark.parametrize("i", range(40))
def test_random_decode_configurations(i):
    # Seeded random configurations crossing the launch choices (work plan or
    # not, partition groups or pieces, deep or 2-stage rings, one or two
    # column tiles or head slices, decode step or attention) against the oracle.
    dt, Hq, Hkv, D, B, lengths, P, plan, step = _random_decode_config(i)
    w = Workload(0, "random", dt, Hq, Hkv, D, B, len(lengths), "fixed", writes_new_token=step)
    case = make_decode_case(w, seed=i, lengths=lengths)
    S = len(lengths)
    kc, vc = case.k_cache.to(DEV), case.v_cache.to(DEV)
    out = torch.full((S, Hq, D), float("nan"), dtype=torch.float32, device=DEV)
    ws = None
    if P or plan:
        ws = torch.empty(pkv.decode_workspace_bytes(S, Hq, D, case.block_tables.shape[1] * B, P),
                         dtype=torch.uint8, device=DEV)
    args = (case.block_tables.to(DEV), case.context_lens.to(DEV), w.scale, B, Hkv)
    if step:
        pkv.decode_step(out, case.q.to(DEV), case.new_key.to(DEV), case.new_value.to(DEV), kc, vc,
                        *args, partition_size=P, workspace=ws)
    else:
        pkv.paged_decode_attention(out, case.q.to(DEV), kc, vc, *args, partition_size=P,
                                   workspace=ws)
    torch.cuda.synchronize()
    assert pkv.device_status() == 0
    if step:
        k_ref, v_ref = case.k_cache.clone(), case.v_cache.clone()
        ref = oracle.decode_step(case.q, case.new_key, case.new_value, k_ref, v_ref,
                                 case.block_tables, case.context_lens, w.scale, B, Hkv)
        assert torch.equal(bits(kc), bits(k_ref)) and torch.equal(bits(vc), bits(v_ref))
    else:
        ref = oracle.paged_decode_attention(case.q, case.k_cache, case.v_cache,
                                            case.block_tables, case.context_lens, w.scale, B,
                                            Hkv)
    assert max_err(out, ref) <= TOL16, (dt, Hq, Hkv, D, B, P, plan, step)
    assert bool(torch.isfinite(out).all())


def test_decode_calls_replayed_from_a_cuda_graph():
    # The decode calls (split with the plan, unsplit with the plan, the decode
    # step) captured once in a CUDA graph and replayed: each replay matches the
    # oracle, also after the inputs are rewritten in place between replays.
    w = Workload(0, "graph", "bf16", 32, 8, 128, 16, 6, "fixed", writes_new_token=True)
    lengths = [1, 16, 17, 700, 2049, 300]
    case = make_decode_case(w, seed=11, lengths=lengths)
    S, Hq, D = case.q.shape
    maxb = case.block_tables.shape[1]
    kc, vc = case.k_cache.to(DEV), case.v_cache.to(DEV)
    q, bt, cl = case.q.to(DEV), case.block_tables.to(DEV), case.context_lens.to(DEV)
    nk, nv = case.new_key.to(DEV), case.new_value.to(DEV)
    outs = [torch.empty((S, Hq, D), dtype=torch.float32, device=DEV) for _ in range(3)]
    wss = [torch.empty(pkv.decode_workspace_bytes(S, Hq, D, maxb * 16, P), dtype=torch.uint8,
                       device=DEV) for P in (128, 0, 0)]

    def body(sm):
        pkv.decode_step(outs[2], q, nk, nv, kc, vc, bt, cl, w.scale, 16, 8, partition_size=0,
                        workspace=wss[2], stream=sm)
        pkv.paged_decode_attention(outs[0], q, kc, vc, bt, cl, w.scale, 16, 8,
                                   partition_size=128, workspace=wss[0], stream=sm)
        pkv.paged_decode_attention(outs[1], q, kc, vc, bt, cl, w.scale, 16, 8,
                                   partition_size=0, workspace=wss[1], stream=sm)

    side = torch.cuda.Stream(DEV)
    side.wait_stream(torch.cuda.current_stream(DEV))
    with torch.cuda.stream(side):
        body(side)
    torch.cuda.current_stream(DEV).wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side, capture_error_mode="thread_local"):
        body(side)
    k_ref, v_ref = case.k_cache.clone(), case.v_cache.clone()
    q_host = case.q.clone()
    for rep in range(2):
        for o in outs:
            o.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert pkv.device_status() == 0
        ref = oracle.decode_step(q_host, case.new_key, case.new_value, k_ref.clone(),
                                 v_ref.clone(), case.block_tables, case.context_lens, w.scale,
                                 16, 8)
        for o in outs:
            assert max_err(o, ref) <= TOL16, rep
        # new queries, written in place: the next replay reads them
        q_host = torch.randn(q_host.shape, generator=torch.Generator().manual_seed(rep)) \
            .to(torch.bfloat16)
        q.copy_(q_host)


# --------------------------------------------------------------------------
# Wide query-head groups (G a multiple of 32, head_dim 128, unsplit): the
# tcgen05 kernel, against the oracle and against the head-slice kernel
# --------------------------------------------------------------------------

WIDE_LENGTHS = [1, 127, 128, 129, 0, 700, 2049, 4100, 255, 33]


def wide_decode(case, w, kc, vc, which, plan, out_dtype=torch.float32, q=None, out=None):
    pkv.set_wide_group_kernel(which)
    try:
        return gpu_decode(case.q if q is None else q, kc, vc, case.block_tables,
                          case.context_lens, w.scale, w.block_size, w.num_kv_heads,
                          out_dtype=out_dtype, plan=plan)
    finally:
        pkv.set_wide_group_kernel(pkv.WIDE_TCGEN05)


@pytest.mark.parametrize("dt,G,Hkv,B", [("bf16", 32, 2, 16), ("f16", 32, 1, 8),
                                         ("bf16", 64, 2, 32), ("f16", 96, 1, 16),
                                         ("bf16", 32, 8, 8), ("f16", 64, 1, 8),
                                         ("bf16", 128, 1, 16)])
@pytest.mark.parametrize("plan", [False, True])
def test_wide_groups_tcgen05_match_oracle_and_head_slices(dt, G, Hkv, B, plan):
    # ragged lengths around the 128-token tile (1, 127, 128, 129, ...), an
    # empty sequence, NaN in every unused cache slot; with and without the
    # work plan (records taken through the kernel's counter)
    w = Workload(0, "wide", dt, G * Hkv, Hkv, 128, B, len(WIDE_LENGTHS), "fixed")
    case = make_decode_case(w, seed=G + B + Hkv, lengths=WIDE_LENGTHS)
    kc, vc = case.k_cache.to(DEV), case.v_cache.to(DEV)
    ref = oracle.paged_decode_attention(case.q, case.k_cache, case.v_cache, case.block_tables,
                                        case.context_lens, w.scale, B, Hkv)
    for which in (pkv.WIDE_TCGEN05, pkv.WIDE_HEAD_SLICES):
        out = wide_decode(case, w, kc, vc, which, plan)
        assert pkv.device_status() == 0, which
        assert max_err(out, ref) <= TOL16, which
        assert torch.equal(out[4].cpu(), torch.zeros_like(out[4].cpu()))  # length 0


@pytest.mark.parametrize("plan", [False, True])
def test_wide_groups_many_items_per_cta(plan):
    # 600 items (300 sequences x 2 KV heads) over at most one CTA a SM: each
    # CTA runs several items back to back through both Q buffers, among them
    # one-token and empty ones
    lengths = [int(x) for x in np.random.default_rng(4).integers(0, 600, size=300)]
    lengths[:5] = [1, 0, 0, 1, 128]
    w = Workload(0, "wide_many", "bf16", 64, 2, 128, 16, len(lengths), "fixed")
    case = make_decode_case(w, seed=8, lengths=lengths)
    kc, vc = case.k_cache.to(DEV), case.v_cache.to(DEV)
    ref = oracle.paged_decode_attention(case.q, case.k_cache, case.v_cache, case.block_tables,
                                        case.context_lens, w.scale, 16, 2)
    out = wide_decode(case, w, kc, vc, pkv.WIDE_TCGEN05, plan)
    assert pkv.device_status() == 0
    assert max_err(out, ref) <= TOL16


@pytest.mark.parametrize("G", [32, 64])
@pytest.mark.parametrize("rising", [True, False])
def test_wide_groups_running_max_moves(rising, G):
    # keys scaled up (or down) along each context, so that the per-head max
    # rises by more than the 2^8 margin several times mid-sequence (O^T and
    # the partial sums are then rescaled) -- or is set by the first tile;
    # G = 64 runs one 64-head item, two halves with a running max each
    lengths = [2049, 900, 3000]
    w = Workload(0, "wide_max", "bf16", G, 1, 128, 16, len(lengths), "fixed")
    case = make_decode_case(w, seed=31, lengths=lengths)
    kc = case.k_cache.float()
    for s, L in enumerate(lengths):
        for pos in range(L):
            f = 1.0 + 7.0 * pos / L
            kc[case.block_tables[s, pos // 16], :, pos % 16] *= f if rising else 8.0 / f
    case.k_cache.copy_(kc.to(case.k_cache.dtype))
    dk, dv = case.k_cache.to(DEV), case.v_cache.to(DEV)
    ref = oracle.paged_decode_attention(case.q, case.k_cache, case.v_cache, case.block_tables,
                                        case.context_lens, w.scale, 16, 1)
    out = wide_decode(case, w, dk, dv, pkv.WIDE_TCGEN05, True)
    assert pkv.device_status() == 0
    assert max_err(out, ref) <= TOL16


@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float16])
def test_wide_groups_16bit_outputs(out_dtype):
    # rounded once to the output dtype, as in test_16bit_outputs
    w = Workload(0, "wide_o", "bf16", 64, 2, 128, 16, 4, "fixed")
    case = make_decode_case(w, seed=6, lengths=[5, 300, 129, 1000])
    kc, vc = case.k_cache.to(DEV), case.v_cache.to(DEV)
    ref = oracle.paged_decode_attention(case.q, case.k_cache, case.v_cache, case.block_tables,
                                        case.context_lens, w.scale, 16, 2)
    out = wide_decode(case, w, kc, vc, pkv.WIDE_TCGEN05, False, out_dtype=out_dtype)
    rel = 2.0 ** -8 if out_dtype == torch.bfloat16 else 2.0 ** -11
    diff = np.abs(out.cpu().double().numpy() - ref)
    assert (diff <= TOL16 + rel * np.abs(ref)).all()


def test_wide_groups_bad_block_and_length_are_flagged():
    w = Workload(0, "wide_bad", "bf16", 32, 1, 128, 16, 3, "fixed")
    case = make_decode_case(w, seed=19, lengths=[300, 300, 300])
    bt = case.block_tables.clone()
    bt[1, 3] = case.num_blocks + 5
    cl = case.context_lens.clone()
    cl[2] = bt.shape[1] * 16 + 1
    kc, vc = case.k_cache.to(DEV), case.v_cache.to(DEV)
    ref = oracle.paged_decode_attention(case.q[:1], case.k_cache, case.v_cache, bt[:1], cl[:1],
                                        w.scale, 16, 1)
    for plan in (False, True):
        pkv.set_wide_group_kernel(pkv.WIDE_TCGEN05)
        out = gpu_decode(case.q, kc, vc, bt, cl, w.scale, 16, 1, plan=plan)
        st = pkv.device_status(reset=True)
        assert st & 1 and st & 2
        assert max_err(out[:1], ref) <= TOL16  # the healthy sequence is unaffected
        assert torch.isfinite(out[1]).all()
        assert torch.equal(out[2].cpu(), torch.zeros_like(out[2].cpu()))


@pytest.mark.parametrize("plan", [False, True])
def test_wide_groups_decode_step(plan):
    # the step's append runs first (a kernel of its own), then the tcgen05
    # kernel attends over the new token too; the cache is bit-exact
    lengths = [1, 16, 17, 129, 700, 2049]
    w = Workload(0, "wide_step", "bf16", 64, 2, 128, 16, len(lengths), "fixed",
                 writes_new_token=True)
    case = make_decode_case(w, seed=23, lengths=lengths)
    kc, vc = case.k_cache.to(DEV), case.v_cache.to(DEV)
    out = torch.full(case.q.shape, float("nan"), dtype=torch.float32, device=DEV)
    ws = None
    if plan:
        n = pkv.decode_workspace_bytes(len(lengths), 64, 128, case.block_tables.shape[1] * 16, 0)
        ws = torch.empty(n, dtype=torch.uint8, device=DEV)
    pkv.decode_step(out, case.q.to(DEV), case.new_key.to(DEV), case.new_value.to(DEV), kc, vc,
                    case.block_tables.to(DEV), case.context_lens.to(DEV), w.scale, 16, 2,
                    workspace=ws)
    torch.cuda.synchronize()
    k_ref, v_ref = case.k_cache.clone(), case.v_cache.clone()
    ref = oracle.decode_step(case.q, case.new_key, case.new_value, k_ref, v_ref,
                             case.block_tables, case.context_lens, w.scale, 16, 2)
    assert pkv.device_status() == 0
    assert torch.equal(bits(kc), bits(k_ref)) and torch.equal(bits(vc), bits(v_ref))
    assert max_err(out, ref) <= TOL16


def test_wide_groups_query_and_output_in_pinned_host_memory():
    # q read and the output written over the host link: the same bits as
    # with device tensors
    lengths = [1, 700, 33, 2049, 0]
    w = Workload(0, "wide_host", "bf16", 32, 2, 128, 16, len(lengths), "fixed")
    case = make_decode_case(w, seed=41, lengths=lengths)
    kc, vc = case.k_cache.to(DEV), case.v_cache.to(DEV)
    S, Hq, D = case.q.shape
    outs = []
    for host in (False, True):
        q = case.q.pin_memory() if host else case.q.to(DEV)
        out = torch.full((S, Hq, D), float("nan"), dtype=torch.float32)
        out = out.pin_memory() if host else out.to(DEV)
        pkv.paged_decode_attention(out, q, kc, vc, case.block_tables.to(DEV),
                                   case.context_lens.to(DEV), w.scale, 16, 2)
        torch.cuda.synchronize()
        outs.append(out.cpu())
    assert pkv.device_status() == 0
    assert torch.equal(bits(outs[0]), bits(outs[1]))


def test_wide_groups_unaligned_query_takes_head_slices():
    # q 4-byte but not 16-byte aligned: the call runs the head-slice kernel
    # (the tcgen05 kernel reads q in 16-byte pieces) with the same result
    lengths = [40, 300, 129]
    w = Workload(0, "wide_ua", "bf16", 32, 1, 128, 16, len(lengths), "fixed")
    case = make_decode_case(w, seed=43, lengths=lengths)
    kc, vc = case.k_cache.to(DEV), case.v_cache.to(DEV)
    ref = oracle.paged_decode_attention(case.q, case.k_cache, case.v_cache, case.block_tables,
                                        case.context_lens, w.scale, 16, 1)
    n = case.q.numel()
    big = torch.empty(n + 2, dtype=case.q.dtype, device=DEV)
    q = big[2:].view(case.q.shape)
    q.copy_(case.q.to(DEV))
    assert q.data_ptr() % 16 != 0 and q.data_ptr() % 4 == 0
    out = gpu_decode(q, kc, vc, case.block_tables, case.context_lens, w.scale, 16, 1)
    assert pkv.device_status() == 0
    assert max_err(out, ref) <= TOL16


@pytest.mark.parametrize("Hq", [64, 128])
def test_wide_groups_back_to_back_steps_see_each_others_writes(Hq):
    # As test_back_to_back_steps_see_each_others_writes, for G = 32 and 64 on
    # the tcgen05 kernel: append kernel, work plan and persistent kernel, all
    # dependent launches, twice on one stream and one workspace (the plan
    # zeroes the kernel's record counter again before the second launch)
    B, Hkv = 16, 2
    lengths = [5, 17, 700, 2049, 1001, 35]
    w = Workload(0, "wide_chain", "bf16", Hq, Hkv, 128, B, len(lengths), "fixed",
                 writes_new_token=True)
    case = make_decode_case(w, seed=37, lengths=lengths)
    S, _, D = case.q.shape
    g = torch.Generator().manual_seed(9)
    nk2 = torch.randn(S, Hkv, D, generator=g).to(torch.bfloat16)
    nv2 = torch.randn(S, Hkv, D, generator=g).to(torch.bfloat16)
    kc, vc = case.k_cache.to(DEV), case.v_cache.to(DEV)
    bt = case.block_tables.to(DEV)
    cl1, cl2 = case.context_lens.to(DEV), (case.context_lens + 1).to(DEV)
    out1 = torch.full((S, Hq, D), float("nan"), dtype=torch.bfloat16, device=DEV)
    out2 = torch.full((S, Hq, D), float("nan"), dtype=torch.float32, device=DEV)
    ws = torch.empty(pkv.decode_workspace_bytes(S, Hq, D, case.block_tables.shape[1] * B, 0),
                     dtype=torch.uint8, device=DEV)
    pkv.decode_step(out1, case.q.to(DEV), case.new_key.to(DEV), case.new_value.to(DEV), kc, vc,
                    bt, cl1, w.scale, B, Hkv, workspace=ws)
    pkv.decode_step(out2, out1, nk2.to(DEV), nv2.to(DEV), kc, vc, bt, cl2, w.scale, B, Hkv,
                    workspace=ws)
    torch.cuda.synchronize()
    assert pkv.device_status() == 0
    k_ref, v_ref = case.k_cache.clone(), case.v_cache.clone()
    ref1 = oracle.decode_step(case.q, case.new_key, case.new_value, k_ref, v_ref,
                              case.block_tables, case.context_lens, w.scale, B, Hkv)
    q2 = out1.cpu()
    assert max_err(q2.float(), ref1) <= TOL16 + 2 ** -8 * float(np.abs(ref1).max())
    ref2 = oracle.decode_step(q2, nk2, nv2, k_ref, v_ref, case.block_tables,
                              case.context_lens + 1, w.scale, B, Hkv)
    assert torch.equal(bits(kc), bits(k_ref)) and torch.equal(bits(vc), bits(v_ref))
    assert max_err(out2, ref2) <= TOL16


def test_wide_groups_split_decode_step_and_back_to_back():
    # G = 32: two split decode steps back to back on one workspace (split
    # launches of wide groups run head slices with the in-launch merge); the
    # plan zeroes the merge counters again before the second
    B, Hkv, Hq, P = 16, 2, 64, 256
    lengths = [5, 17, 700, 2049, 1001, 35]
    w = Workload(0, "wide_split_step", "bf16", Hq, Hkv, 128, B, len(lengths), "fixed",
                 writes_new_token=True)
    case = make_decode_case(w, seed=53, lengths=lengths)
    S, _, D = case.q.shape
    g = torch.Generator().manual_seed(11)
    nk2 = torch.randn(S, Hkv, D, generator=g).to(torch.bfloat16)
    nv2 = torch.randn(S, Hkv, D, generator=g).to(torch.bfloat16)
    kc, vc = case.k_cache.to(DEV), case.v_cache.to(DEV)
    bt = case.block_tables.to(DEV)
    cl1, cl2 = case.context_lens.to(DEV), (case.context_lens + 1).to(DEV)
    out1 = torch.full((S, Hq, D), float("nan"), dtype=torch.bfloat16, device=DEV)
    out2 = torch.full((S, Hq, D), float("nan"), dtype=torch.float32, device=DEV)
    ws = torch.empty(pkv.decode_workspace_bytes(S, Hq, D, case.block_tables.shape[1] * B, P),
                     dtype=torch.uint8, device=DEV)
    pkv.decode_step(out1, case.q.to(DEV), case.new_key.to(DEV), case.new_value.to(DEV), kc, vc,
                    bt, cl1, w.scale, B, Hkv, partition_size=P, workspace=ws)
    pkv.decode_step(out2, out1, nk2.to(DEV), nv2.to(DEV), kc, vc, bt, cl2, w.scale, B, Hkv,
                    partition_size=P, workspace=ws)
    torch.cuda.synchronize()
    assert pkv.device_status() == 0
    k_ref, v_ref = case.k_cache.clone(), case.v_cache.clone()
    ref1 = oracle.decode_step(case.q, case.new_key, case.new_value, k_ref, v_ref,
                              case.block_tables, case.context_lens, w.scale, B, Hkv)
    q2 = out1.cpu()
    assert max_err(q2.float(), ref1) <= TOL16 + 2 ** -8 * float(np.abs(ref1).max())
    ref2 = oracle.decode_step(q2, nk2, nv2, k_ref, v_ref, case.block_tables,
                              case.context_lens + 1, w.scale, B, Hkv)
    assert torch.equal(bits(kc), bits(k_ref)) and torch.equal(bits(vc), bits(v_ref))
    assert max_err(out2, ref2) <= TOL16


def test_wide_groups_split_bad_block_is_flagged():
    w = Workload(0, "wide_split_bad", "bf16", 64, 1, 128, 16, 3, "fixed")
    case = make_decode_case(w, seed=59, lengths=[1500, 1500, 1500])
    bt = case.block_tables.clone()
    bt[1, 40] = case.num_blocks + 5  # in the second 512-token partition
    kc, vc = case.k_cache.to(DEV), case.v_cache.to(DEV)
    ref = oracle.paged_decode_attention(case.q[:1], case.k_cache, case.v_cache, bt[:1],
                                        case.context_lens[:1], w.scale, 16, 1)
    out = gpu_decode(case.q, kc, vc, bt, case.context_lens, w.scale, 16, 1, P=512)
    assert pkv.device_status(reset=True) & 1
    assert max_err(out[:1], ref) <= TOL16
    assert torch.isfinite(out[1]).all()


def test_wide_groups_in_a_cuda_graph():
    # a wide-group decode step (append kernel, work plan, persistent tcgen05
    # kernel) captured once as a CUDA graph and replayed: each replay zeroes
    # the record counter again and gives the same result as a direct call
    lengths = [1, 700, 129, 2049]
    w = Workload(0, "wide_graph", "bf16", 64, 2, 128, 16, len(lengths), "fixed",
                 writes_new_token=True)
    case = make_decode_case(w, seed=61, lengths=lengths)
    S, Hq, D = case.q.shape
    kc, vc = case.k_cache.to(DEV), case.v_cache.to(DEV)
    q, nk, nv = case.q.to(DEV), case.new_key.to(DEV), case.new_value.to(DEV)
    bt, cl = case.block_tables.to(DEV), case.context_lens.to(DEV)
    ws = torch.empty(pkv.decode_workspace_bytes(S, Hq, D, case.block_tables.shape[1] * 16, 0),
                     dtype=torch.uint8, device=DEV)
    out = torch.full((S, Hq, D), float("nan"), dtype=torch.float32, device=DEV)
    stream = torch.cuda.Stream(DEV)
    stream.wait_stream(torch.cuda.current_stream(DEV))
    # a separate cache for the warm-up call outside the capture (it appends
    # the new tokens too)
    kw, vw = case.k_cache.to(DEV), case.v_cache.to(DEV)
    with torch.cuda.stream(stream):
        pkv.decode_step(out, q, nk, nv, kw, vw, bt, cl, w.scale, 16, 2, workspace=ws,
                        stream=stream)
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream, capture_error_mode="thread_local"):
        pkv.decode_step(out, q, nk, nv, kc, vc, bt, cl, w.scale, 16, 2, workspace=ws,
                        stream=stream)
    k_ref, v_ref = case.k_cache.clone(), case.v_cache.clone()
    ref = oracle.decode_step(case.q, case.new_key, case.new_value, k_ref, v_ref,
                             case.block_tables, case.context_lens, w.scale, 16, 2)
    for _ in range(2):
        out.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert pkv.device_status() == 0
        assert max_err(out, ref) <= TOL16
    assert torch.equal(bits(kc), bits(k_ref)) and torch.equal(bits(vc), bits(v_ref))
