"""Benchmark of the paged decode step on GB300.

Default workload: bf16 MHA decode step, 32 heads x head_dim 128, block 16,
64 sequences with context lengths uniform on [1, 2048]; one step = each
sequence's new token appended to the cache and paged decode attention over
its context, in one decode-step call (the append runs inside the attention
launch).  The
metric is KV bytes the attention must read (sum_s L_s * 2 * Hkv * D * 2) per
second, with decode steps/s beside it.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload 2..5]
  python bench.py --impl reference ...   # the CPU oracle on the host cores

Under torchrun (N > 1) every rank runs the same workload on its own GPU with
no collective on the data path (sequences shard across GPUs with nothing to
exchange); the time is the max over ranks and the value the sum.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from workloads import (WORKLOADS, Workload, make_beam_case, make_decode_case,  # noqa: E402
                       poison_unused, write_step_schedule, beam_setup_schedule,
                       beam_step_schedule)

METRIC = "paged decode attention KV GB/s (% of GB300 HBM peak), decode steps/sec"
FALLBACK_HBM_GBS = 6800.0

# DRAM bytes (read + write) per launch of the tensor-core decode kernel from
# one ncu capture of each workload's launch, valid only while the kernel
# source hashes to `source_sha`.
TRAFFIC = {"source_sha": "be889194e7ba1bac",
           "bytes_per_launch": {"2": 1109357056, "3": 800045312, "4": 1077338624,
                                "5": 486553088}}


def launch_partition(w, max_blocks: int, lens=None) -> int:
    """Partition size (tokens) the benchmark launches a workload with: the
    workload's own split if it names one; one pass per (sequence, KV head)
    for a ragged batch (see `work_plan`: longest first, a long context
    starts at once and needs no split) or while every context fits in 2048
    tokens; 2048-token partitions beyond (so that a few long contexts do not
    finish last; with the work plan ordering the launch, they measured
    faster than 1024-token ones at every point of the sweep)."""
    if w.partition_size:
        return w.partition_size
    if lens is not None and ragged(lens):
        return 0
    return 0 if max_blocks * w.block_size <= 2048 else 2048


def ragged(lens) -> bool:
    """A batch whose longest context is more than three times the mean."""
    L = [int(x) for x in lens]
    return len(L) > 0 and max(L) > 3 * (sum(L) / len(L))


def work_plan(w, lens, P: int) -> bool:
    """Whether the benchmark gives a launch the library's work plan (a
    workspace): always for split launches (the library plans every split
    launch of up to 4096 sequences), and for unsplit ones when the batch is
    ragged, so that its long sequences start first.  A host scheduler knows
    its lengths and can make the same choice."""
    return P > 0 or ragged(lens)


def kernel_sha() -> str:
    """Hash of the decode kernel's sources, comments and blank space left out
    (the traffic figures above hold only for the code they were captured
    from)."""
    h = hashlib.sha256()
    for name in ("decode_tc.cu", "decode_wide.cu", "decode_deep.cu", "decode_group.cu",
                 "decode_plan.cu", "decode_tc.cuh", "tc_common.cuh"):
        text = open(os.path.join(ROOT, "paged_kv_cache_312_gb300", "csrc", name)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        h.update("".join(text.split()).encode())
    return h.hexdigest()[:16]


# ---------------------------------------------------------------------------
# workload set-up (host), shared by both arms
# ---------------------------------------------------------------------------

class Step:
    """Host tensors of one decode step of a workload, plus its byte counts."""

    def __init__(self, key: int, seed: int, allocator_cls, partition=None):
        w = WORKLOADS[key]
        self.w = w
        self.pairs = torch.zeros((0, 2), dtype=torch.int64)
        self.slots = None
        self.new_key = self.new_value = None
        if key == 5:
            case = make_beam_case(w, seed=seed)
            mgr = allocator_cls(case.pool_blocks, w.block_size, free_order=case.pool_order)
            pre, suf = beam_setup_schedule(mgr, case)
            _, self.slots, self.pairs, self.tables, self.lens = beam_step_schedule(mgr, case)
            NB, Hkv, B, D = case.pool_blocks, w.num_kv_heads, w.block_size, w.head_dim
            self.k_cache = torch.full((NB, Hkv, B, D), float("nan"), dtype=w.torch_dtype)
            self.v_cache = torch.full_like(self.k_cache, float("nan"))
            self.setup_slots = torch.cat([pre.reshape(-1)] + suf)
            self.setup_keys = torch.cat([case.prefix_k.reshape(-1, Hkv, D)] + case.suffix_k)
            self.setup_vals = torch.cat([case.prefix_v.reshape(-1, Hkv, D)] + case.suffix_v)
            self.q, self.new_key, self.new_value = case.q, case.new_key, case.new_value
            self.unique_blocks = int(mgr.stats()[2])
            self.pool_order = case.pool_order
        else:
            case = make_decode_case(w, seed=seed, poison=not w.writes_new_token)
            self.k_cache, self.v_cache, self.q = case.k_cache, case.v_cache, case.q
            self.pool_order = case.pool_order
            self.setup_slots = None
            if w.writes_new_token:
                mgr = allocator_cls(case.num_blocks, w.block_size, free_order=case.pool_order)
                self.slots, self.pairs, self.tables, self.lens = write_step_schedule(
                    mgr, case.lengths)
                poison_unused(self.k_cache, self.v_cache, self.tables, case.lengths - 1)
                self.new_key, self.new_value = case.new_key, case.new_value
            else:
                self.tables, self.lens = case.block_tables, case.context_lens
            self.unique_blocks = None
        self.P = launch_partition(w, self.tables.shape[1], self.lens) if partition is None \
            else partition
        # the beam workload runs through the beam-group call, which has no plan
        self.plan = self.unique_blocks is None and work_plan(w, self.lens.tolist(), self.P)
        if self.slots is not None:
            # the step's new tokens sit at position L-1 of each sequence (what
            # the decode-step call writes, through the table)
            for s_, (row, n) in enumerate(zip(self.tables.tolist(), self.lens.tolist())):
                want = row[(n - 1) // w.block_size] * w.block_size + (n - 1) % w.block_size
                assert int(self.slots[s_]) == want, "step slot is not position L-1"
        L = self.lens.to(torch.int64)
        b = w.torch_dtype.itemsize
        self.kv_bytes = int(L.sum()) * 2 * w.num_kv_heads * w.head_dim * b
        # beam workload: K and V of every physical block in use, counted once
        self.unique_bytes = None if self.unique_blocks is None else \
            self.unique_blocks * w.num_kv_heads * w.block_size * w.head_dim * 2 * b
        S = L.numel()
        io = S * w.num_heads * w.head_dim * (b + 4) + int((L + w.block_size - 1).div(
            w.block_size, rounding_mode="floor").sum()) * 4 + S * 4
        self.attn_bytes = self.kv_bytes + io  # KV + q + fp32 out + table entries + lens
        if self.slots is not None:  # the decode step also reads and stores the new K/V
            self.attn_bytes += 2 * 2 * S * w.num_kv_heads * w.head_dim * b


class GpuStep:
    """Device side of one decode step of a workload, as the benchmark times
    it: the cache on the device (the beam history written into it), the
    step's inputs packed in one pinned host buffer and one device buffer
    (views per tensor), the fp32 output, the workspace, and run(), the calls
    of one step: the copy-on-write copies (if any), then one decode call that
    appends each sequence's new token and attends (beam groups: one CTA per
    group and KV head)."""

    def __init__(self, pkv, st: Step, dev, grouped: bool, gparts: int = 1):
        w = st.w
        self.pkv, self.st, self.w, self.dev = pkv, st, w, dev
        self.grouped, self.gparts = grouped, gparts
        self.kc, self.vc = st.k_cache.to(dev), st.v_cache.to(dev)
        if st.setup_slots is not None:  # beam history
            pkv.kv_write(self.kc, self.vc, st.setup_keys.to(dev), st.setup_vals.to(dev),
                         st.setup_slots.to(dev))
        self.has_write = st.slots is not None
        inputs = [st.q, st.tables, st.lens, st.pairs]
        if self.has_write:
            inputs += [st.new_key, st.new_value]
        if grouped:
            S_ = st.q.shape[0]
            gstart = torch.arange(0, S_ + 1, w.beam_width, dtype=torch.int32)
            shared = pkv.group_shared_tokens(st.tables, st.lens, gstart, w.block_size)
            inputs += [gstart, shared]
        self.h_pack, views = pack_inputs(inputs, dev)
        self.q, self.bt, self.cl, self.pairs = views[:4]
        # q in the pinned pack (the pack's first tensor), and where the rest starts
        qn = st.q.numel() * st.q.element_size()
        self.h_q = self.h_pack[:qn].view(st.q.dtype).view(st.q.shape)
        self.rest_off = (qn + 255) // 256 * 256
        self.nk = self.nv = None
        if self.has_write:
            self.nk, self.nv = views[4:6]
        if grouped:
            self.gs, self.sh = views[-3:-1]
        self.d_pack = views[-1]
        S, Hq, D = self.q.shape
        self.out = torch.empty((S, Hq, D), dtype=torch.float32, device=dev)
        self.ws = None
        if st.P or (st.plan and not grouped):
            # split scratch, or (unsplit) the optional work plan
            self.ws = torch.empty(pkv.decode_workspace_bytes(S, Hq, D,
                                                             self.bt.shape[1] * w.block_size,
                                                             st.P),
                                  dtype=torch.uint8, device=dev)
        elif gparts > 1:
            self.ws = torch.empty(pkv.decode_workspace_bytes(S, Hq, D, gparts, 1),
                                  dtype=torch.uint8, device=dev)
        self.stream = torch.cuda.current_stream(dev)
        # one decode kernel per call, the append fused in (split mode also
        # merges inside it); a call with a workspace on the ungrouped path
        # first runs the one-CTA work-plan kernel (beam groups split over
        # several CTAs zero their counters with a memset, not a kernel)
        plan_kernel = (st.P > 0 or st.plan) and not grouped
        self.launches_per_step = (1 if self.pairs.shape[0] else 0) + 1 + (1 if plan_kernel else 0)

    def run(self, ev=None, stream=None, out=None, q=None):
        """One step on `stream` (default self.stream); `ev`, if given, is
        recorded between the copy-on-write copies and the decode call; `out`
        and `q` (default self.out, self.q) may be pinned host memory."""
        pkv, w, st = self.pkv, self.w, self.st
        sm = self.stream if stream is None else stream
        out = self.out if out is None else out
        q = self.q if q is None else q
        if self.pairs.shape[0]:
            pkv.kv_copy_blocks(self.kc, self.vc, self.pairs, stream=sm)
        if ev is not None:
            ev.record(sm)
        if self.grouped:  # append the new tokens and attend, one CTA per (group, KV head)
            pkv.paged_decode_grouped(out, q, self.kc, self.vc, self.bt, self.cl,
                                     self.gs, self.sh, w.scale, w.block_size, w.num_kv_heads,
                                     new_k=self.nk, new_v=self.nv, parts=self.gparts,
                                     workspace=self.ws, max_members=w.beam_width, stream=sm)
        elif self.has_write:  # append the new tokens and attend, one call
            pkv.decode_step(out, q, self.nk, self.nv, self.kc, self.vc, self.bt,
                            self.cl, w.scale, w.block_size, w.num_kv_heads, partition_size=st.P,
                            workspace=self.ws, stream=sm)
        else:
            pkv.paged_decode_attention(out, q, self.kc, self.vc, self.bt, self.cl,
                                       w.scale, w.block_size, w.num_kv_heads,
                                       partition_size=st.P, workspace=self.ws, stream=sm)


# ---------------------------------------------------------------------------
# clocks sampled while the timed region runs
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self, t_begin=None, t_end=None, t_load_end=None):
        """Stops sampling; summarises the samples taken between host wall
        times t_begin and t_load_end (the timed region and the same steps
        kept running after it), or t_end without a load window, or else all
        samples."""
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                ts = time.mktime(time.strptime(f[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                ts += float("0." + f[0].split(".")[1]) if "." in f[0] else 0.0
                rows.append((ts, float(f[1]), float(f[2]),
                             {n for n, v in zip(names, f[5:9]) if v.lower() == "active"}))
            except (ValueError, IndexError):
                continue
        if t_load_end is not None:
            inside = [r for r in rows if t_begin - 0.05 <= r[0] <= t_load_end + 0.05]
            window = "timed region and the same steps run on, untimed, for %.1f s after it" % (
                t_load_end - t_end)
        else:
            inside = [r for r in rows
                      if t_begin is None or t_begin - 0.05 <= r[0] <= t_end + 0.05]
            window = "timed region"
        if not inside:
            window = "around the timed region"
        use = inside or rows
        if not use:
            return None
        reasons = set().union(*[r[3] for r in use])
        return {"sm_mhz": statistics.median(r[1] for r in use),
                "sm_max_mhz": max(r[2] for r in use), "reasons": sorted(reasons),
                "samples": len(use), "window": window}


def max_over_ranks(x: float, world: int) -> float:
    """Largest value of x over the ranks of the default process group (the
    job's time is that of its slowest GPU)."""
    if world <= 1:
        return x
    t = torch.tensor([x], dtype=torch.float64)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

EXTRA_WORKLOADS = (3, 4, 5)
NOMINAL_HBM_GBS = 7900.0  # GB300 HBM3e nominal bandwidth (context beside the measured peak)


def step_kind(st, grouped: bool, gparts: int) -> str:
    w = st.w
    return (("cow-copy + " if st.pairs.shape[0] else "") +
            ("paged_decode_grouped (beam groups of %d: shared prompt blocks read once per "
             "group; each group's stages over %d CTA(s) a KV head, merged in the launch; new "
             "tokens appended inside the attention launch)" % (w.beam_width, gparts)
             if grouped else
             "decode_step (new tokens appended inside the attention launch)"
             if st.slots is not None else "paged_decode_attention"))


def config_of(st, grouped: bool, gparts: int, world: int) -> dict:
    """The `config` object of a workload's line (the same on both arms)."""
    w = st.w
    cfg = {"workload": w.name, "num_seqs": int(st.q.shape[0]), "num_heads": w.num_heads,
           "num_kv_heads": w.num_kv_heads, "head_dim": w.head_dim, "block_size": w.block_size,
           "partition_size": st.P, "work_plan": bool(st.plan and not grouped),
           "kv_bytes_per_step": st.kv_bytes,
           "group_parts": gparts if grouped else None,
           "step": step_kind(st, grouped, gparts),
           "l2": "inputs larger than L2 (KV %.2f GB vs 129 MB L2), no flush" % (st.kv_bytes / 1e9),
           "parallelism": "replicas" if world > 1 else "single GPU"}
    if st.unique_blocks is not None:
        cfg["unique_kv_bytes"] = st.unique_bytes
    return cfg


def measure(pkv, st, args, rank, world, local_rank, steps, warmup, grouped, gparts,
            e2e_alloc=False):
    """Times one workload's step on this rank's GPU: K steps back to back
    between two events (the value), then K more with events around each
    decode call (the roofline), then end to end through the public API from
    pinned host buffers.  Returns the workload's line (without cpu_baseline)."""
    w = st.w
    dev = torch.device("cuda", local_rank)
    g = GpuStep(pkv, st, dev, grouped, gparts)
    step, stream, out = g.run, g.stream, g.out
    S, Hq, D = out.shape
    for _ in range(warmup):
        step()
    torch.cuda.synchronize(dev)
    assert pkv.device_status() == 0

    # ---- device-timed region: K steps back to back, one event on each side
    # (the per-step events of the roofline pass below would add gaps)
    clocks = ClockSampler(local_rank) if rank == 0 else None
    time.sleep(0.3 if clocks else 0)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    wall0 = time.time()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for i in range(steps):
        step()
    t1.record(stream)
    torch.cuda.synchronize(dev)
    wall1 = time.time()
    # clocks under this load: a short timed region (K steps of 0.1-0.2 ms)
    # holds no nvidia-smi sample (one every 100 ms), so the same step keeps
    # running, untimed, for 0.4 s after it while the sampler runs on
    wall2 = None
    if clocks:
        while time.time() - wall1 < 0.4:
            for _ in range(50):
                step()
            torch.cuda.synchronize(dev)
        wall2 = time.time()
    clk = clocks.stop(wall0, wall1, wall2) if clocks else None
    total_ms = t0.elapsed_time(t1)
    if world > 1:
        torch.distributed.barrier()
    total_ms = max_over_ranks(total_ms, world)
    ms_per_step = total_ms / steps
    assert pkv.device_status() == 0

    # ---- roofline pass: the same K steps with events around each decode
    # call, for that kernel's own average duration
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    mids = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    torch.cuda.synchronize(dev)
    for i in range(steps):
        starts[i].record(stream)
        step(mids[i])
        ends[i].record(stream)
    torch.cuda.synchronize(dev)
    attn_ms = [mids[i].elapsed_time(ends[i]) for i in range(steps)]
    copy_ms = [starts[i].elapsed_time(mids[i]) for i in range(steps)]
    assert pkv.device_status() == 0

    # ---- end to end through the public API with pinned host buffers: every
    # step copies its inputs to the device (one packed copy), runs the calls,
    # reads the output back and synchronises
    e2e = None
    if not args.no_e2e:
        e2e = end_to_end(g, st, dev, max(1, min(steps, 50)), graphs=not args.no_graph)
    launches = g.launches_per_step
    g_pairs = int(g.pairs.shape[0])  # copy-on-write copies in the step
    gpu_out = g.out.cpu()  # the step's output, for the oracle comparison of the CPU baseline
    del g
    torch.cuda.empty_cache()

    peak, peak_src = measured_peaks()
    # A step that is one decode call (no copy-on-write copies) is timed by the
    # back-to-back region itself: events between the calls would stop a
    # call's work plan from reading its lengths while the previous call's
    # last CTAs run.  Otherwise the per-call events of the roofline pass.
    isolated_avg = statistics.mean(attn_ms)
    one_call = g_pairs == 0
    attn_avg = ms_per_step if one_call else isolated_avg
    # beam groups: the bytes the launch must read are the physical blocks in
    # use, each once (shared prompt blocks included once), not the logical
    # KV of every beam
    alg_bytes = st.attn_bytes if st.unique_bytes is None else \
        st.attn_bytes - st.kv_bytes + st.unique_bytes
    achieved = alg_bytes / (attn_avg * 1e-3) / 1e9
    value = st.kv_bytes * world / (ms_per_step * 1e-3) / 1e9
    sha = kernel_sha()
    tr = TRAFFIC["bytes_per_launch"].get(str(w.key)) if TRAFFIC["source_sha"] == sha else None
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": steps, "warmup": warmup, "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": w.dtype, "data": "synthetic (seeded N(0,1) values, shuffled block pool)",
        "config": config_of(st, grouped, gparts, world),
        "steps_per_s": round(1e3 / ms_per_step, 2),
        "pct_hbm_peak": round(100 * value / world / peak, 2),
        "pct_nominal_hbm_peak": round(100 * value / world / NOMINAL_HBM_GBS, 2),
        "clocks": clk,
        "e2e": e2e,
        "gpu_launches": launches * steps,
        "roofline": {"bound": "hbm", "kernel": ("paged_decode_grouped" if grouped else
                                                "decode_step" if st.slots is not None else
                                                "paged_decode_attention") +
                     (" call: tensor-core decode kernel with in-kernel log-sum-exp merge" +
                      (" (+ work-plan kernel)" if not grouped else " (+ counter memset)")
                      if st.P or gparts > 1 else
                      " (tensor-core kernel + work-plan kernel)" if st.plan and not grouped else
                      " (tensor-core kernel)"),
                     "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4),
                     "frac_of_nominal": round(achieved / NOMINAL_HBM_GBS, 4),
                     "traffic": tr, "traffic_source_sha": sha if tr is not None else None,
                     "algorithmic_bytes_per_launch": alg_bytes,
                     "algorithmic_bytes": "unique KV (every physical block in use once) + q + "
                                          "fp32 out + table entries + new K/V"
                     if st.unique_bytes is not None else
                     "KV of every attended token + q + fp32 out + table entries" +
                     (" + new K/V" if st.slots is not None else ""),
                     "avg_launch_ms": round(attn_avg, 5),
                     "avg_launch_timing": "the timed region (K back-to-back decode calls "
                                          "between two events)" if one_call else
                                          "events around each decode call",
                     "avg_launch_ms_events_around_each_call": round(isolated_avg, 5),
                     "peak_source": "%s (MEASURED_PEAKS.json hbm_gbs); nominal %.0f GB/s" %
                     (peak_src, NOMINAL_HBM_GBS)
                     if peak_src == "measured" else "fallback 6.8 TB/s"},
    }
    # each kernel of the step on its own (events around it): the copy-on-write
    # copies, and the decode call (the append of the new K/V runs inside it)
    line["step_kernels_ms"] = {
        "kv_copy_blocks": round(statistics.mean(copy_ms), 5) if g_pairs else None,
        "copy_pairs": g_pairs,
        "decode_call": round(isolated_avg, 5),
        "decode_call_kernels": ("work plan + " if launches - (1 if g_pairs else 0) == 2 else "") +
                               "tensor-core decode" +
                               (" (new K/V appended inside)" if st.slots is not None else ""),
        "timing": "events around each kernel (adds the gaps the back-to-back region avoids)"}
    line["_gpu_out"] = gpu_out
    if st.unique_blocks is not None:
        line["pct_hbm_peak_unique_bytes"] = round(
            100 * st.unique_bytes / (attn_avg * 1e-3) / 1e9 / peak, 2)
    if st.slots is not None and rank == 0:
        line["host_allocator"] = host_allocator_timing(st, pkv, grouped)
        if e2e_alloc and not args.no_e2e and not grouped:
            ka = max(1, min(steps, 50))
            ea = e2e_with_allocator(pkv, st, dev, ka, graphs=not args.no_graph)
            ed = e2e_with_allocator(pkv, st, dev, ka, graphs=not args.no_graph, direct=True)
            ea["direct_io"] = {k_: ed[k_] for k_ in ("value", "unit", "ms_per_step",
                                                       "host_plan_us_per_step", "what")}
            line["e2e_with_allocator"] = ea
    return line


def run_gpu(args, rank, world, local_rank):
    import paged_kv_cache_312_gb300 as pkv
    import __graft_entry__

    __graft_entry__.build()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    cpu = rank == 0 and world == 1 and not args.no_cpu_baseline
    st = Step(args.workload, args.seed + rank, pkv.BlockAllocator,  # independent problems
              partition=args.partition)
    # beam groups: the beams of a group (consecutive sequences) attend their
    # shared prompt blocks in one CTA per (group, KV head)
    grouped = st.unique_blocks is not None and not args.ungrouped
    gparts = args.group_parts if grouped else 1
    line = measure(pkv, st, args, rank, world, local_rank, args.steps, args.warmup, grouped,
                   gparts, e2e_alloc=True)
    gout = line.pop("_gpu_out")
    if cpu:
        line["cpu_baseline"] = cpu_baseline(st, args.cpu_budget, gout)
    del st, gout
    extra = [] if args.extra in ("", "none") else [int(x) for x in args.extra.split(",")]
    if extra:
        line["workloads"] = {}
    for key in extra:
        if key == args.workload:
            continue
        # the other workloads, each in its own launch configuration (the
        # beam workload through the beam-group call), K steps after W warm-up
        sx = Step(key, args.seed + rank, pkv.BlockAllocator)
        gx = sx.unique_blocks is not None
        lx = measure(pkv, sx, args, rank, world, local_rank, args.steps, args.warmup, gx, 1)
        for k_ in ("metric", "higher_is_better", "scaling", "vs_baseline", "n_gpus", "data"):
            lx.pop(k_, None)
        gx_out = lx.pop("_gpu_out")
        if cpu:
            lx["cpu_baseline"] = cpu_baseline(sx, args.cpu_budget_extra, gx_out)
        line["workloads"][str(key)] = lx
        del sx
    if rank == 0 and world == 1 and args.workload == 2 and not args.no_wide:
        # wide query-head groups on their tcgen05 kernel (the sweep workload's
        # G = 32 and 64 points), attention call only
        line["wide_groups"] = wide_group_points(pkv, args.steps, args.warmup, args.seed)
    return line


def end_to_end(g, st, dev, k, graphs=True):
    """End to end through the public API from pinned host buffers: every
    step copies its inputs to the device (one packed copy), runs the step's
    library calls, copies the fp32 output back and synchronises.  With
    `graphs`, the copy, the calls and the read-back are captured once from
    those public calls as a CUDA graph, and each step is one graph launch
    (the copies still move every step's bytes); the plain form, one API call
    after the other, is timed beside it."""
    S, Hq, D = g.out.shape
    h_out = torch.empty((S, Hq, D), dtype=torch.float32).pin_memory()
    res = {"h2d_bytes_per_step": int(g.h_pack.numel()),
           "d2h_bytes_per_step": int(h_out.numel() * h_out.element_size()), "steps": k,
           "inputs": "q, block tables, lengths, CoW pairs, new K/V in one pinned buffer"}

    def body(sm):
        g.d_pack.copy_(g.h_pack, non_blocking=True)
        g.run(stream=sm)
        h_out.copy_(g.out, non_blocking=True)

    def timed(fn, sm):
        torch.cuda.synchronize(dev)
        w0 = time.perf_counter()
        for _ in range(k):
            fn()
            sm.synchronize()
        return (time.perf_counter() - w0) / k

    def body_direct(sm):
        # the output rows go straight to pinned host memory from the kernel
        # (NVLink-C2C stores as each CTA finishes): no copy after the launch
        g.d_pack.copy_(g.h_pack, non_blocking=True)
        g.run(stream=sm, out=h_out)

    def body_direct_io(sm):
        # q read in place from the pinned pack by the kernel as well: only the
        # rest of the pack (tables, lengths, pairs, new K/V) is copied
        g.d_pack[g.rest_off:].copy_(g.h_pack[g.rest_off:], non_blocking=True)
        g.run(stream=sm, out=h_out, q=g.h_q)

    plain_s = timed(lambda: body(g.stream), g.stream)
    res["api_calls_ms_per_step"] = round(plain_s * 1e3, 4)
    res["api_calls_value"] = round(st.kv_bytes / plain_s / 1e9, 2)
    e2e_s, how = plain_s, "one public API call after the other, every step"
    copied = h_out.clone()  # the step's output as the D2H copy brought it back
    h_out.fill_(float("nan"))
    direct_s = timed(lambda: body_direct(g.stream), g.stream)
    assert torch.equal(h_out, copied), "direct output differs from the copied-back output"
    direct_how = "one public API call after the other, every step"
    if graphs:
        graph = capture_step_graph(body, dev)
        if graph is not None:
            cur = torch.cuda.current_stream(dev)
            graph.replay()
            e2e_s = timed(graph.replay, cur)
            how = ("the step's public API calls (H2D copy, library calls, D2H copy) captured "
                   "once as a CUDA graph, one graph launch per step")
        graph_d = capture_step_graph(body_direct, dev)
        if graph_d is not None:
            cur = torch.cuda.current_stream(dev)
            graph_d.replay()
            direct_s = min(direct_s, timed(graph_d.replay, cur))
            direct_how = "the better of the plain calls and their CUDA graph"
    h_out.fill_(float("nan"))
    io_s = timed(lambda: body_direct_io(g.stream), g.stream)
    assert torch.equal(h_out, copied), "direct-io output differs from the copied-back output"
    io_how = "one public API call after the other, every step"
    if graphs:
        graph_io = capture_step_graph(body_direct_io, dev)
        if graph_io is not None:
            cur = torch.cuda.current_stream(dev)
            graph_io.replay()
            io_s = min(io_s, timed(graph_io.replay, cur))
            io_how = "the better of the plain calls and their CUDA graph"
    res.update({"value": round(st.kv_bytes / e2e_s / 1e9, 2), "unit": "GB/s",
                "ms_per_step": round(e2e_s * 1e3, 4), "how": how})
    res["direct_io"] = {
        "value": round(st.kv_bytes / io_s / 1e9, 2), "unit": "GB/s",
        "ms_per_step": round(io_s * 1e3, 4),
        "h2d_bytes_per_step": res["h2d_bytes_per_step"],
        "d2h_bytes_per_step": res["d2h_bytes_per_step"],
        "how": "q read by the decode kernel from pinned host memory and the fp32 output "
               "written there (NVLink-C2C); the other inputs copied; " + io_how}
    # the same step with the output written to pinned host memory by the
    # decode kernel itself: the same bytes cross NVLink-C2C, during the
    # launch instead of after it
    res["direct_output"] = {
        "value": round(st.kv_bytes / direct_s / 1e9, 2), "unit": "GB/s",
        "ms_per_step": round(direct_s * 1e3, 4),
        "h2d_bytes_per_step": res["h2d_bytes_per_step"],
        "d2h_bytes_per_step": res["d2h_bytes_per_step"],
        "how": "inputs copied as above; the decode call writes its fp32 output to pinned "
               "host memory directly (NVLink-C2C stores from the kernel), then the host "
               "synchronises; " + direct_how}
    return res


def capture_step_graph(body, dev):
    """CUDA graph of body(stream), captured on a side stream after two
    eager runs there; None if capture is refused."""
    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(side):
        for _ in range(2):
            body(side)
    torch.cuda.current_stream(dev).wait_stream(side)
    torch.cuda.synchronize(dev)
    graph = torch.cuda.CUDAGraph()
    try:
        with torch.cuda.graph(graph, stream=side, capture_error_mode="thread_local"):
            body(side)
    except RuntimeError as e:
        sys.stderr.write("graph capture refused (%s); e2e uses the plain calls\n" % e)
        torch.cuda.synchronize(dev)
        return None
    torch.cuda.synchronize(dev)
    return graph


def e2e_with_allocator(pkv, st, dev, k, graphs=True, direct=False):
    """End to end with the host side of every step in the timed region, as a
    serving loop runs it: the library's allocator reserves each sequence's
    next slot (pkv_step_append_tables: new blocks, copy-on-write decisions)
    and patches the batch's block tables and lengths in place; they go into
    one of two pinned input buffers, which is copied to the device with the
    step's q and new K/V; the step runs (append + attention); the fp32 output
    is copied back and the host waits for it.  The host plans step i+1 while
    the device runs step i (the allocator needs only the lengths, not the
    step's output).  Each step's copies and calls are one CUDA graph launch
    (one graph per input buffer, captured from the public calls).  Lengths
    grow one token a step per sequence, as in serving, so the tables get
    spare columns and the KV bytes are summed over the steps.  With `direct`,
    the decode call reads q from the pinned input buffer and writes its output
    to pinned host memory itself (NVLink-C2C), and only the rest of the
    buffer is copied."""
    w = st.w
    B = w.block_size
    S = st.q.shape[0]
    L0 = st.lens.to(torch.int64) - 1  # tokens held before the first timed step
    a = pkv.BlockAllocator(st.k_cache.shape[0], B, free_order=st.pool_order)
    for s_ in range(S):
        a.add(s_, int(L0[s_]))
    seqs = torch.arange(S, dtype=torch.int64)
    maxb = int((L0.max() + k + B - 1) // B) + 1
    tables, lens = a.dense_tables(range(S), maxb)  # kept current by the allocator
    pairs = torch.zeros((S, 2), dtype=torch.int64)
    slots = torch.empty(S, dtype=torch.int64)
    kc, vc = st.k_cache.to(dev), st.v_cache.to(dev)
    out = torch.empty((S, w.num_heads, w.head_dim), dtype=torch.float32, device=dev)
    h_out = torch.empty(out.shape, dtype=torch.float32).pin_memory()
    bufs = []
    for _ in range(2):
        h_pack, views = pack_inputs([st.q, tables, torch.zeros_like(lens), pairs, st.new_key,
                                     st.new_value], dev)
        b_ = dict(zip(("q", "bt", "cl", "pairs_d", "nk", "nv", "d_pack"), views))
        b_["h_pack"] = h_pack
        offs, total = [], 0
        for t in (st.q, tables, lens, pairs):
            offs.append(total)
            total += (t.numel() * t.element_size() + 255) // 256 * 256
        b_["h_tables"] = h_pack[offs[1]:offs[1] + tables.numel() * 4].view(torch.int32) \
            .view(S, maxb)
        b_["h_lens"] = h_pack[offs[2]:offs[2] + S * 4].view(torch.int32)
        b_["h_pairs"] = h_pack[offs[3]:offs[3] + S * 16].view(torch.int64).view(S, 2)
        b_["h_q"] = h_pack[:st.q.numel() * st.q.element_size()].view(st.q.dtype).view(st.q.shape)
        b_["rest"] = offs[1]
        bufs.append(b_)

    def body(b_, sm, n_pairs=0):
        if direct:
            b_["d_pack"][b_["rest"]:].copy_(b_["h_pack"][b_["rest"]:], non_blocking=True)
        else:
            b_["d_pack"].copy_(b_["h_pack"], non_blocking=True)
        if n_pairs:
            pkv.kv_copy_blocks(kc, vc, b_["pairs_d"][:n_pairs], stream=sm)
        pkv.decode_step(h_out if direct else out, b_["h_q"] if direct else b_["q"], b_["nk"],
                        b_["nv"], kc, vc, b_["bt"], b_["cl"], w.scale, B, w.num_kv_heads,
                        partition_size=0, stream=sm)
        if not direct:
            h_out.copy_(out, non_blocking=True)

    # captured while the lengths are 0: the capture's runs write and read nothing
    for b_ in bufs:
        b_["graph"] = capture_step_graph(lambda sm, b_=b_: body(b_, sm), dev) if graphs else None
    stream = torch.cuda.current_stream(dev)
    kv_tok = 2 * w.num_kv_heads * w.head_dim * w.torch_dtype.itemsize
    graphed = all(b_["graph"] is not None for b_ in bufs)

    step_append = a.prepare_step_append_tables(seqs, slots, pairs, tables, lens)

    def plan(b_):
        """Host side of the next step into input buffer b_ (its count of CoW pairs)."""
        n = step_append()
        b_["h_tables"].copy_(tables)
        b_["h_lens"].copy_(lens)
        if n:
            b_["h_pairs"][:n].copy_(pairs[:n])
        return n

    kv_total, t_plan = 0, 0.0
    torch.cuda.synchronize(dev)
    w0 = time.perf_counter()
    ta = time.perf_counter()
    n_pairs = plan(bufs[0])
    t_plan += time.perf_counter() - ta
    for i in range(k):
        b_ = bufs[i % 2]
        if n_pairs or not graphed:  # copies to make first: this step runs call by call
            body(b_, stream, n_pairs)
        else:
            b_["graph"].replay()
        kv_total += int(L0.sum() + (i + 1) * S) * kv_tok
        if i + 1 < k:  # plan the next step while this one runs
            ta = time.perf_counter()
            n_pairs = plan(bufs[(i + 1) % 2])
            t_plan += time.perf_counter() - ta
        stream.synchronize()
    dt = time.perf_counter() - w0
    assert pkv.device_status() == 0
    assert torch.isfinite(h_out).all()
    del kc, vc
    torch.cuda.empty_cache()
    return {"value": round(kv_total / dt / 1e9, 2), "unit": "GB/s",
            "ms_per_step": round(dt / k * 1e3, 4), "steps": k,
            "h2d_bytes_per_step": int(bufs[0]["h_pack"].numel()),
            "d2h_bytes_per_step": int(h_out.numel() * 4),
            "host_plan_us_per_step": round(t_plan / k * 1e6, 2),
            "graphs": graphed,
            "what": "pkv_step_append_tables (slots, new blocks, CoW decisions; tables and "
                    "lengths patched in place) for step i+1 on the host while the device runs "
                    "step i; per step " +
                    ("one H2D copy of the pinned inputs but q, decode_step reading q from and "
                     "writing its output to pinned host memory" if direct else
                     "one H2D copy of the pinned inputs + decode_step + output D2H") +
                    " + synchronise; lengths grow one token a step"}


def pack_inputs(tensors, dev):
    """One pinned host buffer holding every tensor (256-byte aligned), and the
    device copy of it: returns (host buffer, [device view per tensor...,
    device buffer])."""
    offs, total = [], 0
    for t in tensors:
        offs.append(total)
        total += (t.numel() * t.element_size() + 255) // 256 * 256
    host = torch.zeros(max(total, 256), dtype=torch.uint8).pin_memory()
    for t, o in zip(tensors, offs):
        n = t.numel() * t.element_size()
        if n:
            host[o:o + n].copy_(t.contiguous().reshape(-1).view(torch.uint8))
    buf = host.to(dev)
    views = []
    for t, o in zip(tensors, offs):
        n = t.numel() * t.element_size()
        views.append(buf[o:o + n].view(t.dtype).view(t.shape))
    return host, views + [buf]


def host_allocator_timing(st, pkv, grouped=False, steps=256):
    """Host side of a decode step (a1/a2) through the C ABI:
    pkv_step_append_tables for every sequence (slot mapping, new blocks,
    copy-on-write decisions), which keeps the dense block tables and lengths
    the device calls take current in place (and, for beam groups, the shared
    prefix of each group found from those tables).  Timed over `steps`
    consecutive steps from the workload's lengths, in a pool with room for
    them; mean microseconds per step.  The headline form is the prepared
    call a serving loop makes on its reused staging buffers
    (prepare_step_append_tables); beside it, the same step with its buffers
    checked on every call, and the earlier form, pkv_step_append plus a dense
    read-back of every table."""
    w = st.w
    lens = st.lens.tolist()
    S, B = len(lens), w.block_size
    need = sum((n + steps + B - 1) // B for n in lens)
    maxb = max((n + steps + B - 1) // B for n in lens)
    gstart = torch.arange(0, S + 1, max(1, w.beam_width), dtype=torch.int32)
    res = {}
    for form in ("prepared", "patched", "dense"):
        a = pkv.BlockAllocator(need + S, B)
        for i, n in enumerate(lens):
            a.add(i, max(0, n - 1))
        seqs = torch.arange(S, dtype=torch.int64)
        tables, tl = a.dense_tables(range(S), maxb)
        slots = torch.empty(S, dtype=torch.int64)
        pairs = torch.empty((S, 2), dtype=torch.int64)
        step = a.prepare_step_append_tables(seqs, slots, pairs, tables, tl)
        shared = torch.zeros(gstart.numel() - 1, dtype=torch.int32)
        group_step = pkv.prepare_group_shared_tokens(tables, tl, gstart, B, shared)
        t0 = time.perf_counter()
        for _ in range(steps):
            if form == "prepared":
                step()
                if grouped:
                    group_step()
                continue
            if form == "patched":
                a.step_append_tables(seqs, slots, pairs, tables, tl)
            else:
                a.step_append(range(S))
                tables, tl = a.dense_tables(range(S), maxb)
            if grouped:
                pkv.group_shared_tokens(tables, tl, gstart, B)
        res[form] = (time.perf_counter() - t0) / steps * 1e6
    return {"us_per_step": round(res["prepared"], 2), "steps": steps, "sequences": S,
            "what": "pkv_step_append_tables for every sequence (tables and lengths patched in "
                    "place; the prepared call on reused buffers)" +
                    (" + shared prefix per beam group" if grouped else ""),
            "us_per_step_checked_call": round(res["patched"], 2),
            "us_per_step_dense_readback": round(res["dense"], 2)}


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu part")):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.machine()


def _oracle_rate(st, kc, vc, budget_s, threads, gpu_out=None, err=None):
    """Passes of the oracle over the step's sequences (copies, write and
    attention) with `threads` threads until `budget_s` of CPU time is used:
    (KV GB/s, bytes, seconds, passes, chunk).  With `gpu_out` (the GPU step's
    output), each sequence the first pass computes is compared with it,
    outside the timed region: err gets the largest absolute difference and
    the number of sequences compared."""
    import oracle
    w = st.w
    S = st.q.shape[0]
    done_bytes, t_used, passes = 0, 0.0, 0
    chunk = max(1, min(S, 4 * threads))
    L = st.lens.to(torch.int64)
    while t_used < budget_s and passes < 100:
        for c0 in range(0, S, chunk):
            idx = torch.arange(c0, min(S, c0 + chunk))
            t = time.perf_counter()
            if c0 == 0:
                if st.pairs.shape[0]:
                    oracle.kv_copy_blocks(kc, vc, st.pairs)
                if st.slots is not None:
                    oracle.kv_write(kc, vc, st.new_key, st.new_value, st.slots, w.block_size)
            ref = oracle.paged_decode_attention(st.q[idx], kc, vc, st.tables[idx], st.lens[idx],
                                                w.scale, w.block_size, w.num_kv_heads,
                                                nthreads=threads)
            t_used += time.perf_counter() - t
            if gpu_out is not None and passes == 0:
                d = np.abs(gpu_out[idx].double().numpy() - np.asarray(ref)).max()
                err["max_abs_err"] = max(err.get("max_abs_err", 0.0), float(d))
                err["sequences"] = err.get("sequences", 0) + len(idx)
            done_bytes += int(L[idx].sum()) * 2 * w.num_kv_heads * w.head_dim * \
                w.torch_dtype.itemsize
            if t_used >= budget_s:
                break
        passes += 1
    return done_bytes / t_used / 1e9, done_bytes, t_used, passes, chunk


def cpu_baseline(st, budget_s=8.0, gpu_out=None):
    """Time the oracle (as it stands) on this host's cores on a bounded sample
    of the same step: passes over the step's sequences (write + attention)
    until the budget is used, on every core, then on one core (a third of
    the budget).  With the GPU step's output, the sequences the oracle
    computed are compared with it (max abs error beside the timing)."""
    import oracle
    w = st.w
    n = os.cpu_count() or 1
    kc, vc = st.k_cache.clone(), st.v_cache.clone()
    if st.setup_slots is not None:
        oracle.kv_write(kc, vc, st.setup_keys, st.setup_vals, st.setup_slots, w.block_size)
    err = {}
    v, nb, t, passes, chunk = _oracle_rate(st, kc, vc, budget_s, n, gpu_out, err)
    v1, nb1, t1, _, _ = _oracle_rate(st, kc, vc, max(1.0, budget_s / 3), 1)
    out = {"value": round(v, 4), "unit": "GB/s", "cores": n, "kind": "oracle",
            "cpu_model": cpu_model(),
            "sample": "%.2f GB of the step's KV (%d pass(es) over chunks of %d sequences, "
                      "fp64 C oracle, %d threads, %.1f s)" % (nb / 1e9, passes, chunk, n, t),
            "single_core": {"value": round(v1, 4), "unit": "GB/s", "cores": 1,
                            "sample": "%.2f GB of the step's KV, 1 thread, %.1f s" %
                                      (nb1 / 1e9, t1)}}
    if err:
        out["gpu_output_vs_oracle"] = {
            "max_abs_err": err["max_abs_err"], "sequences": err["sequences"],
            "of": int(st.q.shape[0]), "bound": 1e-5 if w.dtype == "f32" else 2e-3}
    return out


SWEEP_BLOCKS = (8, 16, 32)
SWEEP_GROUPS = (1, 4, 8, 16, 32, 64)
SWEEP_DIMS = (64, 128)


def sweep_workload(B: int, G: int, D: int) -> Workload:
    """The block-size / GQA / head-dim sweep: bf16, 8 KV heads, 64 sequences
    with contexts uniform on [1024, 4096] (0.34-0.67 GB of KV, beyond L2)."""
    return Workload(0, "sweep-b%d-g%d-d%d" % (B, G, D), "bf16", 8 * G, 8, D, B, 64,
                    "uniform:1024:4096")


def time_decode_call(pkv, call, steps, warmup, stream, dev):
    """Mean ms of `call` over `steps` back-to-back launches on `stream` (CUDA
    events around them), after `warmup` untimed ones."""
    for _ in range(warmup):
        call()
    torch.cuda.synchronize(dev)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(steps):
        call()
    t1.record(stream)
    torch.cuda.synchronize(dev)
    assert pkv.device_status() == 0
    return t0.elapsed_time(t1) / steps


def wide_group_points(pkv, steps, warmup, seed=0):
    """The sweep workload at G = 32 and 64 (block 16, head_dim 128, unsplit with
    the work plan): the decode kernel for wide query-head groups, as a
    fraction of the measured copy peak (KV bytes once per (token, KV head))."""
    dev = torch.device("cuda", torch.cuda.current_device())
    stream = torch.cuda.current_stream(dev)
    peak, _ = measured_peaks()
    B, D = 16, 128
    base = sweep_workload(B, 64, D)
    case = make_decode_case(base, seed=seed)
    kc, vc = case.k_cache.to(dev), case.v_cache.to(dev)
    bt, cl = case.block_tables.to(dev), case.context_lens.to(dev)
    kv = int(case.context_lens.to(torch.int64).sum()) * 2 * 8 * D * 2
    res = {}
    for G in (32, 64):
        w = sweep_workload(B, G, D)
        q = case.q[:, :w.num_heads].contiguous().to(dev)
        S = q.shape[0]
        out = torch.empty((S, w.num_heads, D), dtype=torch.float32, device=dev)
        ws = torch.empty(pkv.decode_workspace_bytes(S, w.num_heads, D, bt.shape[1] * B, 0),
                         dtype=torch.uint8, device=dev)

        def call():
            pkv.paged_decode_attention(out, q, kc, vc, bt, cl, w.scale, B, 8, partition_size=0,
                                       workspace=ws, stream=stream)
        ms = time_decode_call(pkv, call, steps, warmup, stream, dev)
        res[str(G)] = {"kernel": "decode_tc05 (tcgen05, %d heads an item)" % (64 if G % 64 == 0
                                                                               else 32),
                       "query_heads": w.num_heads, "kv_heads": 8, "head_dim": D,
                       "block_size": B, "sequences": S, "kv_bytes": kv,
                       "attn_ms": round(ms, 5), "attn_gbs": round(kv / (ms * 1e-3) / 1e9, 1),
                       "frac_of_measured_peak": round(kv / (ms * 1e-3) / 1e9 / peak, 4)}
    del kc, vc
    return res


def run_sweep(args):
    """Attention GB/s over B x G x D, one JSON line per point, plus the
    allocation side of the same trade-off for the drawn lengths: table entries
    (indirection) and position utilisation (tail waste), Eq. (2)-(3).  Each
    point is timed in two launch configurations, both with the work plan
    (longest sequence first): one pass per (sequence, KV head), and 2048-token
    partitions; the line gives both and the better one (`--partition` times
    that one configuration alone)."""
    import paged_kv_cache_312_gb300 as pkv
    import __graft_entry__

    __graft_entry__.build()
    dev = torch.device("cuda", 0)
    peak, _ = measured_peaks()
    stream = torch.cuda.current_stream(dev)
    wide = {"tcgen05": pkv.WIDE_TCGEN05, "head_slices": pkv.WIDE_HEAD_SLICES}[args.wide_kernel]
    pkv.set_wide_group_kernel(wide)
    blocks, groups, dims = SWEEP_BLOCKS, SWEEP_GROUPS, SWEEP_DIMS
    if args.sweep_point:
        pb, pg, pd = (int(x) for x in args.sweep_point.split(","))
        blocks, groups, dims = (pb,), (pg,), (pd,)
    launches = (0, 2048) if args.partition is None else (args.partition,)
    for B in blocks:
        for D in dims:
            base = sweep_workload(B, max(groups), D)
            case = make_decode_case(base, seed=args.seed)
            kc, vc = case.k_cache.to(dev), case.v_cache.to(dev)
            bt, cl = case.block_tables.to(dev), case.context_lens.to(dev)
            L = case.context_lens.to(torch.int64)
            kv = int(L.sum()) * 2 * 8 * D * 2
            entries = int(((L + B - 1) // B).sum())
            alloc = entries * B
            for G in groups:
                w = sweep_workload(B, G, D)
                q = case.q[:, :w.num_heads].contiguous().to(dev)
                S = q.shape[0]
                out = torch.empty((S, w.num_heads, D), dtype=torch.float32, device=dev)
                timed = {}
                for P in launches:
                    # the optional workspace gives an unsplit launch the plan too
                    ws = torch.empty(pkv.decode_workspace_bytes(S, w.num_heads, D,
                                                                bt.shape[1] * B, P),
                                     dtype=torch.uint8, device=dev)

                    def call():
                        pkv.paged_decode_attention(out, q, kc, vc, bt, cl, w.scale, B, 8,
                                                   partition_size=P, workspace=ws, stream=stream)
                    timed[P] = time_decode_call(pkv, call, args.steps, args.warmup, stream, dev)
                best = min(timed, key=timed.get)
                ms = timed[best]
                line = {"sweep": {"block_size": B, "group": G, "head_dim": D,
                                  "num_heads": w.num_heads, "num_kv_heads": 8,
                                  "partition_size": best, "work_plan": True,
                                  "wide_group_kernel": args.wide_kernel},
                        "attn_ms": round(ms, 5), "kv_bytes": kv,
                        "attn_gbs": round(kv / (ms * 1e-3) / 1e9, 1),
                        "frac_of_measured_peak": round(kv / (ms * 1e-3) / 1e9 / peak, 4),
                        "by_partition_size": {str(P): round(kv / (t * 1e-3) / 1e9 / peak, 4)
                                              for P, t in timed.items()},
                        "table_entries": entries,
                        "position_utilisation": round(int(L.sum()) / alloc, 5),
                        "tail_waste_positions": alloc - int(L.sum())}
                print(json.dumps(line), flush=True)


def measured_bf16_tflops():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]), "measured burst cuBLAS bf16"
    except (OSError, KeyError, ValueError):
        return 1900.0, "fallback 1.9 PFLOP/s"


def run_prefill(args):
    """Paged prefill: 16 sequences whose whole 2048-token prompts attend
    causally over the paged cache (bf16, 32 query / 8 KV heads x 128, block
    16).  Reports attention TFLOP/s (4 * D per query head per attended key)
    against the measured dense bf16 tensor peak."""
    import paged_kv_cache_312_gb300 as pkv
    import __graft_entry__

    __graft_entry__.build()
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream(dev)
    S, L, Hq, Hkv, D, B = 16, 2048, 32, 8, 128, 16
    w = Workload(0, "prefill-bf16-32x8-d128-b16-16x2048", "bf16", Hq, Hkv, D, B, S, "fixed",
                 fixed_lengths=(L,) * S)
    case = make_decode_case(w, seed=args.seed)
    kc, vc = case.k_cache.to(dev), case.v_cache.to(dev)
    bt, cl = case.block_tables.to(dev), case.context_lens.to(dev)
    qs = torch.arange(0, (S + 1) * L, L, dtype=torch.int32, device=dev)
    q = torch.randn(S * L, Hq, D, device=dev).to(torch.bfloat16)
    out = torch.empty(S * L, Hq, D, dtype=torch.bfloat16, device=dev)

    def call():
        pkv.paged_prefill_attention(out, q, kc, vc, bt, cl, qs, w.scale, B, Hkv,
                                    max_query_len=L, stream=stream)
    keys = S * L * (L + 1) // 2  # attended (query, key) pairs per head
    flops = 4 * D * Hq * keys
    peak, src = measured_bf16_tflops()
    steps = max(1, min(args.steps, 50))
    for name, kernel in (("tcgen05", pkv.PREFILL_TCGEN05), ("warp_mma", pkv.PREFILL_WARP_MMA)):
        pkv.set_prefill_kernel(kernel)
        for _ in range(args.warmup):
            call()
        torch.cuda.synchronize(dev)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(steps):
            call()
        b.record(stream)
        torch.cuda.synchronize(dev)
        assert pkv.device_status() == 0
        ms = a.elapsed_time(b) / steps
        tf = flops / (ms * 1e-3) / 1e12
        print(json.dumps({"prefill": {"workload": w.name, "query_tokens": S * L, "causal": True,
                                      "kernel": name},
                          "ms": round(ms, 4), "tflops": round(tf, 1),
                          "roofline": {"bound": "tensor", "achieved": round(tf, 1), "peak": peak,
                                       "unit": "TFLOP/s", "frac": round(tf / peak, 4),
                                       "peak_source": src},
                          "kv_bytes": int(case.context_lens.sum()) * 2 * Hkv * D * 2}),
              flush=True)
    pkv.set_prefill_kernel(pkv.PREFILL_TCGEN05)


def run_sampling(args):
    """Parallel sampling of one long prompt: n = 4 samples share every block
    of an L-token prompt (L = 8192 and 32768; bf16, 32 query / 8 KV heads x
    128, block 16) and each holds one private block of 1-16 tokens.  Times
    the ungrouped split decode (1024-token partitions) against the beam-group
    call with each group's stages over 1, 8, 32 and 64 CTAs a KV head, each
    call on its own after an L2 flush.  GB/s count the unique KV bytes (the
    prompt once)."""
    import paged_kv_cache_312_gb300 as pkv
    import __graft_entry__

    __graft_entry__.build()
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream(dev)
    peak, _ = measured_peaks()
    n, Hq, Hkv, D, B = 4, 32, 8, 128, 16
    gen = torch.Generator(device=dev)
    rng = np.random.default_rng(args.seed)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    for Lp in (8192, 32768):
        gen.manual_seed(args.seed + Lp)
        nbp = Lp // B
        NB = nbp + n
        perm = torch.from_numpy(rng.permutation(NB).astype(np.int32))
        tails = rng.integers(1, B + 1, size=n)
        bt = torch.empty((n, nbp + 1), dtype=torch.int32)
        for s_ in range(n):
            bt[s_, :nbp] = perm[:nbp]
            bt[s_, nbp] = perm[nbp + s_]
        cl = torch.tensor([Lp + int(t) for t in tails], dtype=torch.int32)
        kc = torch.randn((NB, Hkv, B, D), generator=gen, device=dev).to(torch.bfloat16)
        vc = torch.randn((NB, Hkv, B, D), generator=gen, device=dev).to(torch.bfloat16)
        q = torch.randn((n, Hq, D), generator=gen, device=dev).to(torch.bfloat16)
        gs = torch.tensor([0, n], dtype=torch.int32)
        sh = pkv.group_shared_tokens(bt, cl, gs, B)
        btd, cld, gsd, shd = bt.to(dev), cl.to(dev), gs.to(dev), sh.to(dev)
        unique = (Lp + int(tails.sum())) * 2 * Hkv * D * 2
        P = 1024
        ws_u = torch.empty(pkv.decode_workspace_bytes(n, Hq, D, (nbp + 1) * B, P),
                           dtype=torch.uint8, device=dev)
        ref = torch.empty((n, Hq, D), dtype=torch.float32, device=dev)
        calls = [("ungrouped, %d-token partitions" % P, 0,
                  lambda o: pkv.paged_decode_attention(o, q, kc, vc, btd, cld, D ** -0.5, B, Hkv,
                                                       partition_size=P, workspace=ws_u,
                                                       stream=stream))]
        for parts in (1, 8, 32, 64):
            ws_g = torch.empty(pkv.decode_workspace_bytes(n, Hq, D, parts, 1),
                               dtype=torch.uint8, device=dev) if parts > 1 else None
            calls.append(("grouped, %d part(s)" % parts, parts,
                          lambda o, parts=parts, ws_g=ws_g: pkv.paged_decode_grouped(
                              o, q, kc, vc, btd, cld, gsd, shd, D ** -0.5, B, Hkv, parts=parts,
                              workspace=ws_g, max_members=n, stream=stream)))
        calls[0][2](ref)
        for name, parts, fn in calls:
            out = torch.empty_like(ref)
            for _ in range(args.warmup):
                fn(out)
            torch.cuda.synchronize(dev)
            # each call timed on its own, after a 256 MB write that flushes L2
            k = min(args.steps, 200)
            evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(k)]
            for a_, b_ in evs:
                flush.zero_()
                a_.record(stream)
                fn(out)
                b_.record(stream)
            torch.cuda.synchronize(dev)
            assert pkv.device_status() == 0
            ms = statistics.mean(a_.elapsed_time(b_) for a_, b_ in evs)
            print(json.dumps({"sampling": {"samples": n, "prompt_tokens": Lp, "call": name,
                                           "parts": parts, "num_heads": Hq, "num_kv_heads": Hkv,
                                           "head_dim": D, "block_size": B},
                              "ms": round(ms, 5), "unique_kv_bytes": unique,
                              "unique_gbs": round(unique / (ms * 1e-3) / 1e9, 1),
                              "frac_of_measured_peak": round(unique / (ms * 1e-3) / 1e9 / peak, 4),
                              "max_abs_diff_vs_ungrouped": float((out - ref).abs().max())}),
                  flush=True)
        del kc, vc


# NVIDIA's published NVLink-C2C bandwidth of the Grace-Blackwell superchip:
# 900 GB/s bidirectional, 450 GB/s each way (context: the box's measured
# copy-engine rate is the achievable reference)
C2C_NOMINAL_GBS_PER_DIRECTION = 450.0


def run_swap(args):
    """Preemption by swapping: move every block of 64 sequences x 2048 tokens
    (bf16, 8 KV heads x 128) from the device cache to a pinned host pool and
    back with kv_swap_blocks, block pairs shuffled on both sides, for block
    sizes 8 / 16 / 32; then both directions at once (half the blocks out
    while the other half comes in, two streams).  Reference: a plain copy of
    the same bytes between one contiguous device buffer and one pinned host
    buffer (torch copy_, the copy engines over NVLink-C2C), one way and both
    ways at once.  Fractions are also given of the nominal C2C rate."""
    import paged_kv_cache_312_gb300 as pkv
    import __graft_entry__

    __graft_entry__.build()
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream(dev)
    S, L, Hkv, D = 64, 2048, 8, 128
    total = S * L * Hkv * D * 2 * 2  # K and V, bf16
    s1, s2 = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def timed(fn, reps):
        for _ in range(3):
            fn()
        torch.cuda.synchronize(dev)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(reps):
            fn()
        b.record(stream)
        torch.cuda.synchronize(dev)
        return a.elapsed_time(b) / reps

    def both(fn_out, fn_in):
        """fn_out on stream s1 and fn_in on stream s2, started together; the
        main stream waits for both."""
        def run():
            s1.wait_stream(stream)
            s2.wait_stream(stream)
            fn_out(s1)
            fn_in(s2)
            stream.wait_stream(s1)
            stream.wait_stream(s2)
        return run

    flat_d = torch.empty(total, dtype=torch.uint8, device=dev)
    flat_h = torch.empty(total, dtype=torch.uint8).pin_memory()
    half = total // 2
    ref = {"out": total / (timed(lambda: flat_h.copy_(flat_d, non_blocking=True), 10) * 1e-3)
           / 1e9,
           "in": total / (timed(lambda: flat_d.copy_(flat_h, non_blocking=True), 10) * 1e-3)
           / 1e9}

    def ce_out(sm):
        with torch.cuda.stream(sm):
            flat_h[:half].copy_(flat_d[:half], non_blocking=True)

    def ce_in(sm):
        with torch.cuda.stream(sm):
            flat_d[half:].copy_(flat_h[half:], non_blocking=True)
    ref["both"] = total / (timed(both(ce_out, ce_in), 10) * 1e-3) / 1e9
    del flat_d, flat_h
    rng = np.random.default_rng(args.seed)
    for B in (8, 16, 32):
        nb = S * L // B
        kd = torch.randn(nb, Hkv, B, D, device=dev).to(torch.bfloat16)
        vd = torch.randn(nb, Hkv, B, D, device=dev).to(torch.bfloat16)
        kh = torch.empty(nb, Hkv, B, D, dtype=torch.bfloat16).pin_memory()
        vh = torch.empty(nb, Hkv, B, D, dtype=torch.bfloat16).pin_memory()
        pairs = torch.from_numpy(np.stack([rng.permutation(nb), rng.permutation(nb)], 1))
        out_pairs = pairs.to(dev)
        in_pairs = pairs[:, [1, 0]].contiguous().to(dev)
        ms_out = timed(lambda: pkv.kv_swap_blocks(kh, vh, kd, vd, out_pairs, stream=stream), 10)
        ms_in = timed(lambda: pkv.kv_swap_blocks(kd, vd, kh, vh, in_pairs, stream=stream), 10)
        # both ways at once: the first half of the pairs out, the second half in
        h_out_pairs = out_pairs[:nb // 2].contiguous()
        h_in_pairs = in_pairs[nb // 2:].contiguous()
        ms_both = timed(both(
            lambda sm: pkv.kv_swap_blocks(kh, vh, kd, vd, h_out_pairs, stream=sm),
            lambda sm: pkv.kv_swap_blocks(kd, vd, kh, vh, h_in_pairs, stream=sm)), 10)
        assert pkv.device_status() == 0
        for key, direction, ms in (("out", "out (device -> pinned host)", ms_out),
                                   ("in", "in (pinned host -> device)", ms_in),
                                   ("both", "both at once (half the blocks each way)", ms_both)):
            gbs = total / (ms * 1e-3) / 1e9
            nominal = C2C_NOMINAL_GBS_PER_DIRECTION * (2 if key == "both" else 1)
            print(json.dumps({"swap": {"block_size": B, "direction": direction,
                                       "blocks": nb, "block_bytes": Hkv * B * D * 2 * 2},
                              "bytes": total, "ms": round(ms, 4), "gbs": round(gbs, 1),
                              "reference_copy_gbs": round(ref[key], 1),
                              "frac_of_reference": round(gbs / ref[key], 3),
                              "c2c_nominal_gbs": nominal,
                              "frac_of_c2c_nominal": round(gbs / nominal, 3)}), flush=True)
        del kd, vd, kh, vh


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", type=int, default=2, choices=[2, 3, 4, 5])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--partition", type=int, default=None,
                    help="partition size in tokens (default: the workload's launch setting)")
    ap.add_argument("--impl", default="gpu", choices=["gpu", "reference"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-graph", action="store_true",
                    help="e2e: one public API call after the other instead of a captured graph")
    ap.add_argument("--ungrouped", action="store_true",
                    help="beam workload: attend every beam on its own (decode_step) instead of "
                         "one CTA per beam group")
    ap.add_argument("--group-parts", type=int, default=1,
                    help="beam workload: CTAs that share one beam group's stages for a KV head")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-wide", action="store_true",
                    help="leave out the wide query-head group points (G = 32, 64 on the sweep "
                         "workload) that the default line carries in `wide_groups`")
    ap.add_argument("--cpu-budget", type=float, default=8.0,
                    help="seconds of oracle time for the headline workload's CPU baseline")
    ap.add_argument("--cpu-budget-extra", type=float, default=3.0,
                    help="seconds of oracle time for each extra workload's CPU baseline")
    ap.add_argument("--extra", default=None,
                    help="comma-separated workloads measured after the headline one, into the "
                         "line's `workloads` object (default 3,4,5 with workload 2, else none; "
                         "'none' for none)")
    ap.add_argument("--prefill", action="store_true",
                    help="paged prefill throughput (one JSON line; not the benchmark line)")
    ap.add_argument("--swap", action="store_true",
                    help="device <-> pinned host block swap throughput (one JSON line per "
                         "block size and direction; not the benchmark line)")
    ap.add_argument("--sampling", action="store_true",
                    help="parallel sampling of one long prompt: ungrouped split decode against "
                         "the beam-group call over several part counts (one JSON line per call; "
                         "not the benchmark line)")
    ap.add_argument("--sweep", action="store_true",
                    help="block size x GQA group x head_dim sweep of the attention call "
                         "(one JSON line per point; not the benchmark line)")
    ap.add_argument("--sweep-point", default=None, metavar="B,G,D",
                    help="with --sweep: time only this block size, group and head_dim")
    ap.add_argument("--wide-kernel", default="tcgen05", choices=("tcgen05", "head_slices"),
                    help="with --sweep: kernel of unsplit launches with G a multiple of 32 at "
                         "head_dim 128 (the tcgen05 kernel, or head slices on mma.sync)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.extra is None:
        args.extra = ",".join(str(k) for k in EXTRA_WORKLOADS) if args.workload == 2 else ""

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.sweep:
        run_sweep(args)
        return
    if args.sampling:
        run_sampling(args)
        return
    if args.swap:
        run_swap(args)
        return
    if args.prefill:
        run_prefill(args)
        return
    if args.impl == "reference":
        if rank != 0:
            return
        line = run_reference(args)
        print(json.dumps(line), flush=True)
        return

    if world > 1:
        torch.distributed.init_process_group("gloo")
    line = run_gpu(args, rank, world, local_rank)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()


def run_reference(args):
    """The oracle as it stands, timed on the host cores over K steps of a
    bounded sample of the workload (the sample is a fixed subset of the step's
    sequences chosen to keep each step to a few seconds)."""
    import oracle
    from oracle.blockmgr import BlockManager  # the oracle's own block manager builds the tables

    st = Step(args.workload, args.seed, BlockManager, partition=args.partition)
    w = st.w
    n = os.cpu_count() or 1
    kc, vc = st.k_cache.clone(), st.v_cache.clone()
    if st.setup_slots is not None:
        oracle.kv_write(kc, vc, st.setup_keys, st.setup_vals, st.setup_slots, w.block_size)
    S = st.q.shape[0]
    L = st.lens.to(torch.int64)
    # bounded sample: time one pass over a few sequences, then keep a prefix of
    # the step's sequences sized so that the whole run (warm-up and timed
    # steps) takes about two minutes, and no step more than 2 s
    t = time.perf_counter()
    oracle.paged_decode_attention(st.q[:min(S, n)], kc, vc, st.tables[:min(S, n)],
                                  st.lens[:min(S, n)], w.scale, w.block_size, w.num_kv_heads,
                                  nthreads=n)
    per_seq = (time.perf_counter() - t) / min(S, n)
    step_budget = min(2.0, 120.0 / max(1, args.steps + args.warmup))
    m = int(max(1, min(S, step_budget / max(per_seq, 1e-6))))
    idx = torch.arange(m)
    sample_bytes = int(L[idx].sum()) * 2 * w.num_kv_heads * w.head_dim * w.torch_dtype.itemsize

    def step():
        if st.pairs.shape[0]:
            oracle.kv_copy_blocks(kc, vc, st.pairs)
        if st.slots is not None:
            oracle.kv_write(kc, vc, st.new_key, st.new_value, st.slots, w.block_size)
        oracle.paged_decode_attention(st.q[idx], kc, vc, st.tables[idx], st.lens[idx], w.scale,
                                      w.block_size, w.num_kv_heads, nthreads=n)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = (time.perf_counter() - t0) / args.steps
    value = sample_bytes / dt / 1e9
    sample = "%d of %d sequences of the step (%.3f GB of KV per step), fp64 C oracle" % (
        m, S, sample_bytes / 1e9)
    return {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
            "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_of(st, st.unique_blocks is not None and not args.ungrouped,
                                args.group_parts if st.unique_blocks is not None and
                                not args.ungrouped else 1,
                                int(os.environ.get("WORLD_SIZE", "1"))),
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": n,
                             "kind": "oracle", "cpu_model": cpu_model(), "sample": sample},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


if __name__ == "__main__":
    main()
