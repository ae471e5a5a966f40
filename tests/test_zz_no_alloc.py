"""The allocation-free split-context decode entry point.

pkv_paged_decode_attention_noalloc serves callers that cannot allocate device
memory: a plugin run inside a host framework's execute step (where the
framework forbids allocation), a serving loop whose device memory another
allocator carved up at start-up, or latency-critical code that cannot afford
cudaMalloc and its possible device-wide synchronisation.  Its partition
scratch is a fixed array inside the library.

The test calls it through the C ABI several times in a row, on batches of
different shapes (so each call finds the previous call's leftovers in the
array), and checks every result against the oracle (fp64, within the
attention tolerance of the other GPU tests) and against the regular entry
point with a caller workspace.  The cases reach every layout the scratch
takes: partitions spread over a CTA's four warps, one partition per warp
(short partitions of long contexts), head slices of a wide query-head group,
the CUDA-core kernel with its separate log-sum-exp merge (fp32 KV), and the
equal pieces the work plan cuts near-equal contexts into.  It
also checks that a request larger than the array is refused, and that a
malformed request gets the same code as from the workspace entry point.  It
must pass in a fresh process and after the other tests (the file name makes
pytest collect it last)."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_312_gb300 as pkv
from workloads import Workload, make_decode_case

pytestmark = pytest.mark.gpu

TOL16, TOL32 = 2e-3, 1e-5
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    pkv.set_decode_kernel(pkv.KERNEL_AUTO)


# dtype, Hq, Hkv, D, B, context lengths, partition tokens, what it reaches
CASES = [
    ("bf16", 32, 8, 128, 32, [4000, 1, 513, 2047, 0, 3100], 512, "partitions over four warps"),
    ("f16", 16, 16, 128, 16, [100, 1500, 64, 999, 777, 3, 2048, 1025], 256, "MHA"),
    ("bf16", 16, 4, 128, 16, [2048, 3000, 17, 1200, 2100], 32, "one partition per warp"),
    ("bf16", 48, 2, 128, 16, [1500, 700, 2100, 16], 256, "head slices of a 24-head group"),
    ("f32", 8, 2, 64, 16, [1000, 33, 600, 0, 257], 128, "CUDA-core kernel + separate merge"),
    ("bf16", 32, 8, 128, 32, [4096, 4000, 4050, 3990], 512, "pieces of near-equal contexts"),
]


def _case(i, dt, Hq, Hkv, D, B, lengths):
    w = Workload(0, "noalloc", dt, Hq, Hkv, D, B, len(lengths), "fixed")
    return w, make_decode_case(w, seed=100 + i, lengths=lengths)


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


def test_noalloc_matches_oracle_and_workspace_entry_point_call_after_call():
    pkv.device_status(reset=True)
    cases = [(_case(i, *c[:6]), c[6]) for i, c in enumerate(CASES)]
    for (w, c), P in cases:  # the scratch need of every case fits the array
        need = pkv.decode_workspace_bytes(c.q.shape[0], w.num_heads, w.head_dim,
                                          c.block_tables.shape[1] * w.block_size, P)
        assert 0 < need <= pkv.NOALLOC_SCRATCH_BYTES
    # back to back, each call on the array the previous one left behind
    got = [_noalloc(w, c, P) for (w, c), P in cases]
    assert pkv.device_status() == 0
    for ((w, c), P), g, spec in zip(cases, got, CASES):
        tol = TOL32 if w.dtype == "f32" else TOL16
        ref = oracle.paged_decode_attention(c.q, c.k_cache, c.v_cache, c.block_tables,
                                            c.context_lens, w.scale, w.block_size,
                                            w.num_kv_heads, nthreads=oracle.default_threads())
        assert bool(torch.isfinite(g).all()), spec[7]
        err = float(np.abs(g.cpu().double().numpy() - ref).max())
        assert err <= tol, (spec[7], err)
        ws = _with_workspace(w, c, P)
        assert float((g - ws).abs().max()) <= tol, spec[7]
    # and once more on the first batch, after every other layout has used the array
    (w, c), P = cases[0]
    again = _noalloc(w, c, P)
    assert pkv.device_status() == 0
    assert float((again - got[0]).abs().max()) <= TOL16


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
    # malformed and oversized at once (a partition that is not a whole number
    # of blocks): the shape error, as from the workspace entry point
    with pytest.raises(pkv.PkvError) as ei:
        pkv.paged_decode_attention_noalloc(out, q, kc, kc, bt, cl, 0.1, B, 8, 24)
    assert ei.value.code == -2 and "multiple of" in str(ei.value)
    assert not out.any()
