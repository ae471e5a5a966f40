"""bench.py on the host: the reference arm's JSON line (the oracle timed on
the host cores) and the launch rules the GPU arm uses, without a GPU."""
import json
import os
import subprocess
import sys

import pytest
import torch

import bench
from workloads import WORKLOADS

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_contract_line():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "3",
                        "--warmup", "3"], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    assert d["unit"] == "GB/s" and d["higher_is_better"] is True
    assert d["steps"] == 3 and d["warmup"] == 3 and d["n_gpus"] == 1
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert d["config"]["workload"] == WORKLOADS[2].name
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1
    e = d["e2e"]
    assert e["value"] == d["value"] and e["unit"] == d["unit"]
    assert e["h2d_bytes_per_step"] == 0 and e["d2h_bytes_per_step"] == 0
    # the same workload description as the GPU arm's line (whose Step builds
    # its tables with the library's allocator: host code, no GPU needed)
    import paged_kv_cache_312_gb300 as pkv
    assert d["config"] == bench.config_of(bench.Step(2, 0, pkv.BlockAllocator), False, 1, 1)
    assert cb["cpu_model"]


def test_warmup_below_three_is_refused():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--warmup", "2"],
                       cwd=ROOT, capture_output=True, text=True, timeout=120)
    assert r.returncode != 0 and "--warmup" in r.stderr


@pytest.mark.parametrize("key", [2, 3, 4, 5])
def test_launch_partition_rule(key):
    # a workload's own split if it names one; else one pass while every
    # context fits in 2048 tokens, 2048-token partitions beyond
    w = WORKLOADS[key]
    for max_blocks in (1, 2048 // w.block_size, 2048 // w.block_size + 1, 32768 // w.block_size):
        P = bench.launch_partition(w, max_blocks)
        if w.partition_size:
            assert P == w.partition_size
        elif max_blocks * w.block_size <= 2048:
            assert P == 0
        else:
            assert P == 2048


def test_ragged_batches_run_unsplit_with_the_work_plan():
    # workload 3's lognormal lengths are ragged (the longest far above the
    # mean): one pass per (sequence, KV head), longest first; workload 2's
    # uniform lengths are not; a split launch always has the plan
    import numpy as np
    from workloads import draw_lengths
    for key, expect_ragged in ((2, False), (3, True), (4, False)):
        w = WORKLOADS[key]
        # the lengths make_decode_case draws first from the same seed
        lens = draw_lengths(w, np.random.default_rng(0)).tolist()
        assert bench.ragged(lens) == expect_ragged
        maxb = -(-max(lens) // w.block_size)
        P = bench.launch_partition(w, maxb, lens)
        assert bench.work_plan(w, lens, P) == (expect_ragged or P > 0)
        if expect_ragged:
            assert P == 0
    assert bench.ragged([1, 1, 1, 10]) and not bench.ragged([5, 5, 5, 5])


def test_sweep_workloads_cover_the_sweep_grid():
    seen = set()
    for B in bench.SWEEP_BLOCKS:
        for G in bench.SWEEP_GROUPS:
            for D in bench.SWEEP_DIMS:
                w = bench.sweep_workload(B, G, D)
                assert (w.block_size, w.num_heads // w.num_kv_heads, w.head_dim) == (B, G, D)
                assert w.num_kv_heads == 8 and w.dtype == "bf16"
                seen.add(w.name)
    assert len(seen) == len(bench.SWEEP_BLOCKS) * len(bench.SWEEP_GROUPS) * len(bench.SWEEP_DIMS)


def test_cpu_baseline_compares_the_gpu_output_with_the_oracle():
    # The CPU-baseline leg computes the oracle's output for the sequences it
    # times; given the GPU step's output it reports the largest difference.
    # Here the "GPU output" is the oracle's own (difference 0) and then that
    # output with one element moved by 0.25.
    import numpy as np
    import oracle
    import paged_kv_cache_312_gb300 as pkv
    st = bench.Step(1, 0, pkv.BlockAllocator)
    w = st.w
    ref = torch.from_numpy(np.asarray(oracle.paged_decode_attention(
        st.q, st.k_cache, st.v_cache, st.tables, st.lens, w.scale, w.block_size,
        w.num_kv_heads))).float()
    cb = bench.cpu_baseline(st, 0.2, ref)
    g = cb["gpu_output_vs_oracle"]
    assert g["sequences"] == g["of"] == st.q.shape[0]
    assert g["max_abs_err"] < 1e-6 and g["bound"] == 1e-5
    bad = ref.clone()
    bad[2, 1, 5] += 0.25
    g = bench.cpu_baseline(st, 0.2, bad)["gpu_output_vs_oracle"]
    assert abs(g["max_abs_err"] - 0.25) < 1e-6
