"""The allocation-free split-context decode entry point.

pkv_paged_decode_attention_noalloc serves callers that cannot allocate device
memory (plugins run inside a host framework's execute step, serving loops
whose memory another allocator owns, latency-critical code that cannot afford
cudaMalloc).  Its partition scratch is a fixed array inside the library.  This
test calls it through the C ABI twice in a row, on two different batches, and
checks each result against the regular entry point with a caller workspace,
within the attention tolerance of the other GPU tests; it also checks that a
request larger than the fixed array is refused.  It must pass in a fresh
process and after the other tests (the file name makes pytest collect it
last)."""
import numpy as np
import pytest
import torch

import paged_kv_cache_312_gb300 as pkv
from workloads import Workload, make_decode_case

pytestmark = pytest.mark.gpu

TOL16 = 2e-3
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    pkv.set_decode_kernel(pkv.KERNEL_AUTO)


def _case(seed, lengths, Hq, Hkv, B, dt):
    w = Workload(0, "noalloc", dt, Hq, Hkv, 128, B, len(lengths), "fixed")
    c = make_decode_case(w, seed=seed, lengths=lengths)
    return w, c


def _with_workspace(w, c, P):
    S, Hq, D = c.q.shape
    out = torch.empty((S, Hq, D), dtype=torch.float32, device=DEV)
    n = pkv.decode_workspace_bytes(S, Hq, D, c.block_tables.shape[1] * w.block_size, P)
    ws = torch.empty(n, dtype=torch.uint8, device=DEV)
    pkv.paged_decode_attention(out, c.q.to(DEV), c.k_cache.to(DEV), c.v_cache.to(DEV),
                               c.block_tables.to(DEV), c.context_lens.to(DEV), w.scale,
                               w.block_size, w.num_kv_heads, partition_size=P, workspace=ws)
    torch.cuda.synchronize()
    return out


def _noalloc(w, c, P):
    S, Hq, D = c.q.shape
    out = torch.full((S, Hq, D), float("nan"), dtype=torch.float32, device=DEV)
    pkv.paged_decode_attention_noalloc(out, c.q.to(DEV), c.k_cache.to(DEV), c.v_cache.to(DEV),
                                       c.block_tables.to(DEV), c.context_lens.to(DEV), w.scale,
                                       w.block_size, w.num_kv_heads, P)
    torch.cuda.synchronize()
    return out


def test_noalloc_matches_workspace_entry_point_twice_in_a_row():
    pkv.device_status(reset=True)
    # first call: GQA 32/8, block 32, long and ragged contexts, 512-token parts
    w1, c1 = _case(1, [4000, 1, 513, 2047, 0, 3100], 32, 8, 32, "bf16")
    # second call: other shapes, so the array holds the first call's leftovers
    w2, c2 = _case(2, [100, 1500, 64, 999, 777, 3, 2048, 1025], 16, 16, 16, "f16")
    got1 = _noalloc(w1, c1, 512)
    got2 = _noalloc(w2, c2, 256)
    ref1 = _with_workspace(w1, c1, 512)
    ref2 = _with_workspace(w2, c2, 256)
    assert pkv.device_status() == 0
    for got, ref in ((got1, ref1), (got2, ref2)):
        assert torch.isfinite(got).all()
        err = float((got.double() - ref.double()).abs().max())
        assert err <= TOL16, err


def test_noalloc_refuses_requests_beyond_its_scratch():
    S, Hq, D, B = 64, 64, 128, 16
    maxb = 4096  # 65536-token contexts, 16-token partitions: far beyond 16 MiB
    need = pkv.decode_workspace_bytes(S, Hq, D, maxb * B, 16)
    assert need > pkv.NOALLOC_SCRATCH_BYTES
    q = torch.zeros((S, Hq, D), dtype=torch.bfloat16, device=DEV)
    out = torch.zeros((S, Hq, D), dtype=torch.float32, device=DEV)
    kc = torch.zeros((4, 8, B, D), dtype=torch.bfloat16, device=DEV)
    bt = torch.zeros((S, maxb), dtype=torch.int32, device=DEV)
    cl = torch.zeros((S,), dtype=torch.int32, device=DEV)
    with pytest.raises(pkv.PkvError) as ei:
        pkv.paged_decode_attention_noalloc(out, q, kc, kc, bt, cl, 0.1, B, 8, 16)
    assert ei.value.code == -8 and "fixed array holds" in str(ei.value)
    with pytest.raises(pkv.PkvError) as ei:
        pkv.paged_decode_attention_noalloc(out, q, kc, kc, bt, cl, 0.1, B, 8, 0)
    assert ei.value.code == -2
    assert not out.any()
