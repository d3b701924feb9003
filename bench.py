#!/usr/bin/env python
"""Benchmark of the paged-attention hot path on GB300.

One step = one pass of the decode hot path over one batch: append this step's
new K/V rows into the paged cache (paged_kv_store) and run paged attention over
every query (paged_attn_forward_split with the library's split heuristic, which
launches the split-KV decode kernel and, when splits > 1, the LSE merge).  The
schedule is built and uploaded once before timing (it is reused while the
schedule is unchanged).  The end-to-end leg replays one CUDA graph per step:
pinned host-to-device copies of the step's inputs, pa_plan_advance (the
schedule moves one position on, on the device), the append, the attention and
the device-to-host copy of the output.

Main line: the Llama-3-8B-like GQA decode layer -- 64 sequences, one query each,
Hq=32, Hkv=8, D=Dv=128, page_size=16, contexts U[512, 8192], bf16, shuffled
pages.  Its KV working set (~1.1 GB) exceeds the 129 MB L2, so no flush is
needed between steps.  Metric: KV-cache bytes the step must read (sum over
queries of visible keys x Hkv x (D + Dv) x 2 B) per second, plus queries/s.

Secondary measurements (same JSON line, key "workloads"): long-context split
decode (contexts 32K..128K, Hq=64, split sweep), mixed chunked prefill +
decode (TFLOP/s on causal-visible pairs), and MLA decode (TFLOP/s and KV GB/s).

--impl reference times the fp64 CPU oracle on the host cores on bounded samples
of the same workload (there is no other implementation to compare with).
Multi-GPU: independent replicas (no exchange step exists), weak scaling; a
multi-rank run times the decode workloads only (see secondary_for_run).
"""
from __future__ import annotations

import argparse
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged decode KV GB/s (% HBM peak), queries/s; prefill/MLA TFLOP/s"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


# ----------------------------------------------------------------- helpers --

def visible_counts(case) -> np.ndarray:
    if case.causal:
        return case.query_pos.astype(np.int64) + 1
    return case.seq_lens[case.query_seq].astype(np.int64)


def kv_bytes(case, first: int = 0) -> int:
    """Algorithmic K/V bytes: each query's visible keys (queries first.. on), each KV head read once."""
    elt = torch.empty((), dtype=case.dtype).element_size()
    n = int(visible_counts(case)[first:].sum())
    if case.is_mla:
        return n * (case.d + case.p) * elt
    return n * case.hkv * (case.d + case.dv) * elt


def attn_flops(case, first: int = 0, count: int | None = None) -> int:
    """Multiply-add flops over causal-visible (query, key) pairs (of queries first..first+count-1)."""
    vc = visible_counts(case)
    n = int(vc[first:None if count is None else first + count].sum())
    if case.is_mla:
        return n * case.hq * (2 * (case.d + case.p) + 2 * case.d)
    return n * case.hq * (2 * case.d + 2 * case.dv)


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            d = json.load(open(path))
            hbm = d.get("hbm_gbs") or d.get("hbm_GBps")
            bf16 = d.get("bf16_tflops")
            bf16s = d.get("bf16_tflops_sustained") or bf16
            if hbm and bf16:
                return {"hbm_gbs": float(hbm), "bf16_tflops": float(bf16), "bf16_tflops_sustained": float(bf16s),
                        "source": "measured"}
        except Exception:
            pass
    return {"hbm_gbs": FALLBACK_HBM_GBS, "bf16_tflops": FALLBACK_BF16_TFLOPS,
            "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def profile_traffic(name: str, source_files):
    """dram bytes per launch recorded in profiles/<name>.md, if the kernel source is unchanged."""
    import hashlib
    path = os.path.join(ROOT, "profiles", name + ".md")
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", text)
    h = re.search(r"source_sha256:\s*([0-9a-f]+)", text)
    if not m or not h:
        return None
    sha = hashlib.sha256()
    for f in source_files:
        sha.update(open(os.path.join(ROOT, f), "rb").read())
    if sha.hexdigest()[:16] != h.group(1)[:16]:
        return None
    return float(m.group(1))


class ClockSampler:
    """nvidia-smi clock / throttle samples taken while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.tmp = None

    def start(self):
        try:
            self.tmp = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.tmp, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.tmp.flush()
        rows = [r.split(",") for r in open(self.tmp.name).read().strip().splitlines() if r.strip()]
        os.unlink(self.tmp.name)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
            except ValueError:
                continue
            for name, val in zip(names, r[5:9]):
                if val.strip().lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_info():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(x: float, world: int, device) -> float:
    """Largest value over the ranks (device: where the collective's tensor lives)."""
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_step: float, steps: int, local_ms: float, world: int, device) -> tuple:
    """Weak scaling over independent replicas: every rank processes `units_per_step`
    per step; the job time is the slowest rank's.  Returns (units per second, max ms)."""
    total_ms = max_over_ranks(local_ms, world, device)
    return world * units_per_step * steps / (total_ms / 1e3), total_ms


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# -------------------------------------------------------------- GPU steps --

class DecodeStep:
    """Resident inputs, plan, workspace and the two calls of one step."""

    def __init__(self, case, device, splits=None):
        import paged_kv_attention_20_gb300 as pka
        self.pka = pka
        self.case = case
        self.dc = case.to(device)
        self.plan = pka.paged_attn_plan(case.seq_lens, case.block_table, case.query_seq, case.query_pos,
                                        case.page_size, case.num_pages, device=device)
        sms = torch.cuda.get_device_properties(device).multi_processor_count
        if splits:
            self.splits = splits
        elif case.is_mla:
            self.splits = pka.paged_mla_split_heuristic(self.plan, case.hq, sms)
        else:
            self.splits = pka.paged_attn_split_heuristic(self.plan, case.hq, case.hkv, sms)
        self.ws = pka.make_workspace(self.plan, case.hq, case.dv, max(self.splits, 1), device)
        self.out = torch.empty(case.num_queries, case.hq, case.dv, dtype=case.dtype, device=device)

    def store(self):
        d = self.dc
        self.pka.paged_kv_store(self.plan, d.new_k, d.new_v, d.k_cache, d.v_cache)

    def attend(self):
        d = self.dc
        if self.case.is_mla:
            self.pka.paged_mla_forward(self.plan, d.q, d.qp, d.k_cache, d.v_cache, self.case.scale,
                                       causal=self.case.causal, workspace=self.ws, splits=self.splits,
                                       out=self.out)
        else:
            self.pka.paged_attn_forward_split(self.plan, d.q, d.k_cache, d.v_cache, self.case.scale,
                                              self.splits, workspace=self.ws, causal=self.case.causal,
                                              out=self.out)

    def kernels_per_step(self) -> int:
        return 2 + (1 if self.splits > 1 else 0) + (1 if (self.plan.n_tiles and not self.case.is_mla) else 0)


def time_step(step: DecodeStep, steps: int, warmup: int, world: int, device, sampler=None):
    """K steps back to back between two events (nothing recorded between the
    kernels, so each launch may overlap the tail of the one before it), then
    a separate pass of up to 200 steps with events around the append, the
    attention call and its main kernel for the per-kernel breakdown."""
    for _ in range(warmup):
        step.store()
        step.attend()
    torch.cuda.synchronize(device)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize(device)
    if sampler:
        sampler.start()
    t0.record()
    for _ in range(steps):
        step.store()
        step.attend()
    t1.record()
    torch.cuda.synchronize(device)
    clocks = sampler.stop() if sampler else None
    barrier(world)
    total = t0.elapsed_time(t1)
    nb = min(steps, 200)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(nb)]
    for e in evs:              # create the CUDA events before use
        for ev in e:
            ev.record()
    torch.cuda.synchronize(device)
    for i in range(nb):
        evs[i][0].record()
        step.store()
        evs[i][1].record()
        step.pka.time_next_kernel(evs[i][3], evs[i][4])   # brackets the main attention kernel
        step.attend()
        evs[i][2].record()
    torch.cuda.synchronize(device)
    store_ms = [e[0].elapsed_time(e[1]) for e in evs]
    attn_ms = [e[1].elapsed_time(e[2]) for e in evs]
    kern_ms = [e[3].elapsed_time(e[4]) for e in evs]
    return total, store_ms, attn_ms, kern_ms, clocks


def soak_clocks(step: DecodeStep, device, seconds=1.0):
    sampler = ClockSampler(device.index or 0).start()
    time.sleep(0.2)
    t_end = time.time() + seconds
    while time.time() < t_end:
        for _ in range(20):
            step.store()
            step.attend()
        torch.cuda.synchronize(device)
    c = sampler.stop()
    c["window"] = "load soak right after the timed region"
    return c


def _pipelined_e2e(step, names, host_src, device, steps: int, warmup: int, pre=None):
    """Replays a step through the public API from host buffers, software-
    pipelined as a serving loop runs it.  Two CUDA graphs alternate.  Graph p
    runs `pre` (if any), paged_kv_store and the attention on device input set
    p into device output p; beside it, on two more streams (one per copy
    direction), it copies the next step's inputs from pinned host set 1-p into
    device set 1-p and the previous step's output from device output 1-p into
    pinned host buffer 1-p.
    The host enqueues step i+1, then waits for step i.  Every step thus moves
    one step's inputs host-to-device and one output device-to-host, and both
    copies overlap a step's kernels; the timed region ends with the copy of
    the last step's output.  Returns (seconds for `steps` steps, the last
    output on the host)."""
    import copy
    base = step.dc
    dsets = [base, copy.copy(base)]
    for k in names:
        setattr(dsets[1], k, getattr(base, k).clone())
    douts = [step.out, torch.empty_like(step.out)]
    hsets = [{k: host_src[k].pin_memory() for k in names} for _ in range(2)]
    outs = [torch.empty(step.out.shape, dtype=step.out.dtype).pin_memory() for _ in range(2)]
    stream = torch.cuda.current_stream(device)
    h2d, d2h = torch.cuda.Stream(device), torch.cuda.Stream(device)   # one per copy direction

    def body(p):
        cur = torch.cuda.current_stream(device)
        h2d.wait_stream(cur)
        d2h.wait_stream(cur)
        with torch.cuda.stream(h2d):
            for k in names:
                getattr(dsets[1 - p], k).copy_(hsets[1 - p][k], non_blocking=True)
        with torch.cuda.stream(d2h):
            outs[1 - p].copy_(douts[1 - p], non_blocking=True)
        step.dc, step.out = dsets[p], douts[p]
        if pre:
            pre()
        step.store()
        step.attend()
        cur.wait_stream(h2d)
        cur.wait_stream(d2h)

    side = torch.cuda.Stream(device)
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        for k in names:
            getattr(dsets[0], k).copy_(hsets[0][k], non_blocking=True)
        body(0)                      # kernel attributes are set outside capture (first `pre`)
    stream.wait_stream(side)
    torch.cuda.synchronize(device)
    graphs = [torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()]
    for p in range(2):
        with torch.cuda.graph(graphs[p]):
            body(p)
    evs = [torch.cuda.Event(), torch.cuda.Event()]

    def run(n, first):
        if n == 0:
            return first
        prev = None
        for i in range(n):
            p = (first + i) % 2
            graphs[p].replay()
            evs[p].record(stream)
            if prev is not None:
                evs[prev].synchronize()      # step i-1 done (and step i-2's output on the host)
            prev = p
        evs[prev].synchronize()
        return (prev + 1) % 2

    nxt = run(warmup, 1)             # the eager step used set 0 and filled set 1
    last = (nxt + 1) % 2
    t = time.perf_counter()
    nxt = run(steps, nxt)
    last = (nxt + 1) % 2
    outs[last].copy_(douts[last], non_blocking=True)
    stream.synchronize()
    dt = time.perf_counter() - t
    step.dc, step.out = dsets[last], douts[last]
    return dt, outs[last].clone()


PIPELINE_MODE = ("two CUDA graphs alternate; graph p runs the step on device set p while two more streams "
                 "copy the next step's inputs from pinned host set 1-p and the previous step's output "
                 "into pinned host buffer 1-p; the host enqueues step i+1 before waiting for step i; the "
                 "timed region ends with the copy of the last output")


def e2e_leg(case, device, steps: int, warmup: int):
    """Same metric through the public API with host buffers, run as a decode
    loop replays its attention layer: each step copies its inputs (q, the
    position query for MLA, and the new cache rows) from pinned host memory,
    runs pa_plan_advance (every query moves one position on, on the device),
    the append and the attention (split GQA, or MLA), and copies the output
    back to pinned host memory; steps are software-pipelined (_pipelined_e2e).
    The case is the given decode workload with its pages reserved for the
    positions the loop reaches; the KV bytes (and, for MLA, the flops) are
    counted per step as the histories grow.  The last step is checked against
    the same attention called directly."""
    import workloads
    import paged_kv_attention_20_gb300 as pka
    total = warmup + steps + 2
    ctx = [int(n) for n in case.seq_lens]
    grown = workloads.build_case(case.name + "_loop", case.meta["seed"], [n + total for n in ctx],
                                 [(i, n - 1) for i, n in enumerate(ctx)], case.hq, case.hkv, case.d,
                                 case.p if case.is_mla else case.dv, case.page_size, case.dtype, case.scale,
                                 mla_p=case.p)
    step = DecodeStep(grown, device)
    names = ("q", "qp", "new_k", "new_v") if grown.is_mla else ("q", "new_k", "new_v")
    src = {k: getattr(grown, k) for k in names}
    h2d = sum(t.numel() * t.element_size() for t in src.values())
    d2h = step.out.numel() * step.out.element_size()
    dt, last = _pipelined_e2e(step, names, src, device, steps, warmup,
                              pre=lambda: pka.paged_attn_plan_advance(step.plan))
    done = 1 + warmup                # advances so far (the eager step and the warm-up replays)
    # positions during timed step i: ctx - 1 + done + 1 + i; keys seen: that + 1
    elt = grown.new_k.element_size()
    if grown.is_mla:
        per_tok = (grown.d + grown.p) * elt
        per_key_flops = grown.hq * (2 * (grown.d + grown.p) + 2 * grown.d)
    else:
        per_tok = grown.hkv * (grown.d + grown.dv) * elt
        per_key_flops = grown.hq * (2 * grown.d + 2 * grown.dv)
    keys = sum(sum(ctx) + len(ctx) * (done + 1 + i) for i in range(steps))
    step.attend()                    # the same attention on the state the last step left
    torch.cuda.synchronize(device)
    if not torch.equal(step.out.cpu(), last) or pka.device_status() != 0:
        raise RuntimeError("graph-replayed decode step differs from the direct call")
    what = "paged_mla_forward" if grown.is_mla else "paged_attn_forward_split"
    res = {"value": keys * per_tok / dt / 1e9, "unit": "GB/s", "h2d_bytes_per_step": int(h2d),
           "d2h_bytes_per_step": int(d2h), "ms_per_step": dt / steps * 1e3, "splits": step.splits,
           "mode": f"per step: pinned H2D of {', '.join(names)}; pa_plan_advance (schedule on the device); "
                   f"paged_kv_store; {what}; D2H of the output into pinned memory; {PIPELINE_MODE}"}
    if grown.is_mla:
        res.update(value=keys * per_key_flops / dt / 1e12, unit="TFLOP/s", kv_gbs=keys * per_tok / dt / 1e9)
    return res


def e2e_static_leg(case, device, steps: int, warmup: int):
    """The mixed prefill + decode call end to end through the public API with
    host buffers: each step copies its q and new K/V rows from pinned host
    memory, runs the append and the attention (prefill tiles and decode items)
    and copies the output back to pinned host memory; steps are software-
    pipelined (_pipelined_e2e).  The schedule is uploaded once (a serving step
    would stage a new one with pa_plan_stage, which a graph can hold as well);
    every step appends the same rows at the same positions, so the flops per
    step are the workload's.  The last step is checked against the same
    attention called directly."""
    import paged_kv_attention_20_gb300 as pka
    step = DecodeStep(case, device)
    names = ("q", "new_k", "new_v")
    src = {k: getattr(case, k) for k in names}
    h2d = sum(t.numel() * t.element_size() for t in src.values())
    d2h = step.out.numel() * step.out.element_size()
    dt, last = _pipelined_e2e(step, names, src, device, steps, warmup)
    step.attend()
    torch.cuda.synchronize(device)
    if not torch.equal(step.out.cpu(), last) or pka.device_status() != 0:
        raise RuntimeError("graph-replayed mixed step differs from the direct call")
    fl = attn_flops(case)
    return {"value": fl * steps / dt / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h), "ms_per_step": dt / steps * 1e3, "splits": step.splits,
            "mode": "per step: pinned H2D of q, new_k, new_v; paged_kv_store; paged_attn_forward_split "
                    f"(prefill tiles + decode items); D2H of the output into pinned memory; {PIPELINE_MODE}"}


DECODE_ONLY = ("long", "gqa")


def secondary_for_run(requested: str, world: int) -> list:
    """Secondary workloads a run measures.  A multi-rank run (one replica per
    GPU) keeps to the decode workloads, whose kernels read only their own
    GPU's memory through plain per-CTA TMA loads: it launches no prefill and
    no MLA kernel, so no thread-block-cluster kernel runs in a job that spans
    several GPUs."""
    which = [w for w in requested.split(",") if w]
    if world > 1:
        which = [w for w in which if w in DECODE_ONLY]
    return which


def secondary(device, warmup: int, steps: int, peaks, which, cpu=True):
    """Long-context split decode, mixed prefill + decode, MLA decode (one entry each);
    with cpu=True each entry also carries the oracle timed on the host cores over
    the same inputs (cpu_baseline, in the entry's own unit)."""
    import workloads
    res = {}
    hbm, tc = peaks["hbm_gbs"], peaks["bf16_tflops"]
    if "long" in which:
        res.update(_long_context(device, warmup, steps, hbm, cpu))
    if "gqa" in which:
        res.update(_split_sweep(workloads.gqa_decode_bf16(), "gqa_decode_bf16_split_sweep",
                                "64 seqs ctx U[512,8192], Hq=32, Hkv=8, D=128, ps=16, bf16",
                                (None, 1, 2, 3, 4, 8), device, warmup, steps, hbm))
    for name, maker in (("mixed_prefill_decode_bf16", workloads.mixed_prefill_decode_bf16),
                        ("mla_decode_bf16", workloads.mla_decode_bf16)):
        if name.split("_")[0] not in which:
            continue
        case = maker()
        st = DecodeStep(case, device)
        for _ in range(warmup):
            st.store()
            st.attend()
        torch.cuda.synchronize(device)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(steps):
            st.attend()
        e1.record()
        torch.cuda.synchronize(device)
        ms = e0.elapsed_time(e1) / steps
        # the call's main kernel alone (prefill tiles / MLA), events recorded by the library
        kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        for i in range(steps):
            st.pka.time_next_kernel(*kev[i])
            st.attend()
        torch.cuda.synchronize(device)
        kms = sum(a.elapsed_time(b) for a, b in kev) / steps
        fl = attn_flops(case)
        res[name] = {"queries": case.num_queries, "splits": st.splits, "ms": ms, "flops": fl,
                     "tflops": fl / ms / 1e9, "frac_bf16_peak": fl / ms / 1e9 / tc,
                     "prefill_tiles": st.plan.n_tiles, "decode_items": st.plan.n_decode}
        if case.is_mla:
            res[name].update(kernel_ms=kms, kernel_tflops=fl / kms / 1e9, kernel_frac_bf16_peak=fl / kms / 1e9 / tc,
                             kv_gbs=kv_bytes(case) / ms / 1e6, frac_hbm=kv_bytes(case) / ms / 1e6 / hbm)
            res[name]["e2e"] = e2e_leg(case, device, steps=max(10, steps), warmup=warmup)
        else:
            # prefill chunks are the first n_prefill * chunk queries.  In the call the decode items
            # (HBM-bound) run beside the prefill kernel on a share of the SMs, so the prefill
            # kernel is also timed alone, on the whole GPU, over a plan of the same chunks only
            npq = case.meta["n_prefill"] * case.meta["chunk"]
            pfl = attn_flops(case, 0, npq)
            pcase = maker(n_decode=0)
            pst = DecodeStep(pcase, device)
            for _ in range(warmup):
                pst.attend()
            pev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
            for i in range(steps):
                pst.pka.time_next_kernel(*pev[i])
                pst.attend()
            torch.cuda.synchronize(device)
            pkms = sum(a.elapsed_time(b) for a, b in pev) / steps
            del pst, pcase
            res[name].update(prefill_kernel_ms=pkms, prefill_flops=pfl, prefill_kernel_tflops=pfl / pkms / 1e9,
                             prefill_kernel_frac_bf16_peak=pfl / pkms / 1e9 / tc,
                             prefill_kernel_ms_in_call=kms, decode_kv_bytes=kv_bytes(case, npq),
                             note="ms and tflops cover the whole call: the prefill kernel with the decode items "
                                  "(HBM-bound) beside it on a share of the SMs; prefill_kernel_* is the prefill "
                                  "kernel alone on the whole GPU over the same chunks (a plan without the decode "
                                  "items), prefill_kernel_ms_in_call the same kernel inside the mixed call")
            res[name]["e2e"] = e2e_static_leg(case, device, steps=max(10, steps), warmup=warmup)
        if cpu:
            label = "MLA decode workload" if case.is_mla else "mixed prefill + decode workload"
            res[name]["cpu_baseline"] = cpu_baseline(case, label, unit="TFLOP/s")
        del st, case
        torch.cuda.empty_cache()
    return res


def _long_context(device, warmup, steps, hbm, cpu=False):
    import workloads
    case = workloads.long_context_decode_bf16()
    res = _split_sweep(case, "long_context_split_decode_bf16",
                       "4 seqs ctx {32K,64K,96K,128K}, Hq=64, Hkv=8, D=128, ps=16, bf16",
                       (None, 1, 4, 8, 16, 32, 64), device, warmup, steps, hbm)
    if cpu:
        res["long_context_split_decode_bf16"]["cpu_baseline"] = cpu_baseline(case, "long-context decode workload")
    return res


def _split_sweep(c3, name, desc, counts, device, warmup, steps, hbm):
    res = {}
    sweep = {}
    for s in counts:
        st = DecodeStep(c3, device, splits=s)
        for _ in range(warmup):
            st.attend()
        torch.cuda.synchronize(device)
        # calls back to back (nothing between them), then the main kernel alone
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(steps):
            st.attend()
        e1.record()
        torch.cuda.synchronize(device)
        ms = e0.elapsed_time(e1) / steps
        kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        for a, b in kev:
            a.record()
            b.record()
        for i in range(steps):
            st.pka.time_next_kernel(*kev[i])
            st.attend()
        torch.cuda.synchronize(device)
        kms = statistics.mean(a.elapsed_time(b) for a, b in kev)
        sweep["heuristic" if s is None else str(s)] = {"splits": st.splits, "ms": ms,
                                                        "kv_gbs": kv_bytes(c3) / ms / 1e6, "kernel_ms": kms,
                                                        "kernel_kv_gbs": kv_bytes(c3) / kms / 1e6}
        del st
    best = max(sweep.values(), key=lambda r: r["kv_gbs"])
    h = sweep["heuristic"]
    res[name] = {
        "config": desc,
        "kv_bytes": kv_bytes(c3), "heuristic_splits": h["splits"], "ms": h["ms"], "kv_gbs": h["kv_gbs"],
        "frac_hbm": h["kv_gbs"] / hbm, "best_splits": best["splits"], "best_kv_gbs": best["kv_gbs"],
        "sweep": sweep}
    del c3
    torch.cuda.empty_cache()
    return res


# ------------------------------------------------------------- CPU oracle --

def oracle_rows_rate(case, rows, nthreads=0):
    """Run the oracle on flat (q*Hq+h) rows; return (seconds, algorithmic KV bytes covered)."""
    dt, b, _ = oracle_rows_work(case, rows, nthreads)
    return dt, b


def oracle_rows_work(case, rows, nthreads=0):
    """Run the oracle on flat (q*Hq+h) rows; return (seconds, algorithmic KV bytes, flops) those
    rows account for: each row's share of its query's KV bytes (kv_bytes) and its own flops
    over its causal-visible keys (attn_flops)."""
    import oracle
    q_of = np.asarray(rows) // case.hq
    n = float(visible_counts(case)[q_of].sum())
    elt = torch.empty((), dtype=case.dtype).element_size()
    t = time.perf_counter()
    if case.is_mla:
        oracle.attention(case.q, case.k_cache, case.k_cache, case.seq_lens, case.block_table, case.query_seq,
                         case.query_pos, case.scale, qp=case.qp, kp_cache=case.v_cache, rows=rows,
                         nthreads=nthreads)
        per_key_bytes = (case.d + case.p) * elt / case.hq          # one shared latent head per query
        per_key_flops = 2 * (case.d + case.p) + 2 * case.d
    else:
        oracle.attention(case.q, case.k_cache, case.v_cache, case.seq_lens, case.block_table, case.query_seq,
                         case.query_pos, case.scale, rows=rows, nthreads=nthreads)
        per_key_bytes = case.hkv * (case.d + case.dv) * elt / case.hq   # each KV head once per query
        per_key_flops = 2 * case.d + 2 * case.dv
    return time.perf_counter() - t, n * per_key_bytes, n * per_key_flops


def cpu_baseline(case, label="GQA decode workload", unit="GB/s", budget_s=12.0):
    """The oracle, as it stands, on all host cores over a bounded, evenly spaced
    sample of the workload's (query, head) rows, reported in `unit` (GB/s of
    algorithmic KV bytes, or TFLOP/s over causal-visible pairs; both figures are
    given).  When the whole workload takes well under the budget it is repeated
    so the figure covers about `budget_s` seconds of work."""
    import oracle
    threads = oracle.threads()
    nrows = case.num_queries * case.hq
    probe = np.unique(np.linspace(0, nrows - 1, min(nrows, max(threads, 32))).astype(np.int64))
    t, _, _ = oracle_rows_work(case, probe)
    want = int(min(nrows, max(len(probe), len(probe) * budget_s / max(t, 1e-6))))
    rows = np.unique(np.linspace(0, nrows - 1, want).astype(np.int64))
    t, b, f = oracle_rows_work(case, rows)
    passes = 1
    while len(rows) == nrows and t < 0.66 * budget_s and passes < 1000:
        dt, db, df = oracle_rows_work(case, rows)
        t, b, f, passes = t + dt, b + db, f + df, passes + 1
    what = (f"{passes} passes over all {nrows} (query, head) rows of the {label}"
            if len(rows) == nrows else
            f"{len(rows)} of {nrows} (query, head) rows of the {label}, evenly spaced")
    gbs, tflops = b / t / 1e9, f / t / 1e12
    return {"value": gbs if unit == "GB/s" else tflops, "unit": unit, "cores": threads, "kind": "oracle",
            "kv_gbs": gbs, "tflops": tflops, "seconds": t,
            "sample": f"{what}; {t:.1f} s on {threads} threads"}


def reference_arm(args, rank, world):
    """The oracle as the reference implementation: bounded samples per step, host cores."""
    if world > 1 and rank != 0:
        return
    import oracle
    import workloads
    case = workloads.gqa_decode_bf16()
    threads = oracle.threads()
    nrows = case.num_queries * case.hq
    probe = np.arange(min(nrows, max(threads, 32)))
    t, _ = oracle_rows_rate(case, probe)
    per_row = t / len(probe)
    budget = 150.0 / max(1, args.steps + args.warmup)
    k = int(max(threads, min(nrows, budget / max(per_row, 1e-9))))
    k = min(k, nrows)
    times, bytes_ = [], []
    for i in range(args.warmup + args.steps):
        rows = (np.arange(k) * 97 + i * k) % nrows
        rows = np.unique(rows)
        dt, b = oracle_rows_rate(case, rows)
        if i >= args.warmup:
            times.append(dt)
            bytes_.append(b)
    value = sum(bytes_) / sum(times) / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": sum(times) / len(times) * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": "gqa_decode_bf16: 64 seqs x 1 query, Hq=32, Hkv=8, D=Dv=128, ps=16, "
                                   "ctx U[512,8192], bf16 inputs", "l2": "inputs larger than L2"},
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": threads, "kind": "oracle",
                             "sample": f"{k} (query, head) rows per step of the same workload"},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)


def profile_run(args):
    """A few un-timed steps of one workload, for ncu captures of one kernel."""
    import paged_kv_attention_20_gb300 as pka
    import workloads
    pka.build()
    device = torch.device("cuda", 0)
    n = args.profile_seqs
    if args.profile == "gqa":
        case = workloads.gqa_decode_bf16(num_seqs=n or 64)
    elif args.profile == "long":
        case = workloads.long_context_decode_bf16()
    elif args.profile == "prefill":
        case = workloads.mixed_prefill_decode_bf16(n_prefill=n or 8, n_decode=0 if n else 120)
    elif args.profile == "mla":
        case = workloads.mla_decode_bf16(num_seqs=n or 128)
    else:
        # decode loop with the schedule advanced on the device each step: the GQA
        # decode workload with pages reserved for the positions the loop reaches
        base = workloads.gqa_decode_bf16(num_seqs=n or 64)
        ctx = [int(x) for x in base.seq_lens]
        grow = args.profile_iters + 2
        case = workloads.build_case("gqa_decode_loop", base.meta["seed"], [x + grow for x in ctx],
                                    [(i, x - 1) for i, x in enumerate(ctx)], base.hq, base.hkv, base.d, base.dv,
                                    base.page_size, base.dtype, base.scale)
    step = DecodeStep(case, device, splits=args.splits)
    for _ in range(args.profile_iters):
        if args.profile == "advance":
            pka.paged_attn_plan_advance(step.plan)
        step.store()
        step.attend()
    torch.cuda.synchronize(device)
    print(json.dumps({"profile": args.profile, "queries": case.num_queries, "splits": step.splits,
                      "kv_bytes": kv_bytes(case), "device_status": pka.device_status()}))


# -------------------------------------------------------------------- main --

def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--secondary", default="long,mixed,mla",
                    help="comma list of secondary workloads: long, gqa, mixed, mla ('' for none)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--splits", type=int, default=None, help="override the split heuristic")
    ap.add_argument("--profile", choices=["gqa", "long", "prefill", "mla", "advance"], default=None,
                    help="run a few un-timed steps of one workload (for ncu captures) and exit")
    ap.add_argument("--profile-seqs", type=int, default=0,
                    help="with --profile: number of sequences (0 = the full workload)")
    ap.add_argument("--profile-iters", type=int, default=3)
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    rank, world, local = dist_info()
    if args.profile:
        profile_run(args)
        return

    if args.impl == "reference":
        reference_arm(args, rank, world)
        return

    import paged_kv_attention_20_gb300 as pka
    import workloads
    pka.build()
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)

    peaks = measured_peaks()
    case = workloads.gqa_decode_bf16()
    step = DecodeStep(case, device, splits=args.splits)
    sampler = ClockSampler(device.index or 0) if rank == 0 else None
    local_ms, store_ms, attn_ms, kern_ms, clocks = time_step(step, args.steps, args.warmup, world, device, sampler)
    kvb = kv_bytes(case)
    rate, total_ms = whole_job_rate(kvb, args.steps, local_ms, world, device)
    if rank == 0 and clocks is not None and clocks.get("samples", 0) < 3:
        clocks = soak_clocks(step, device)

    ms_per_step = total_ms / args.steps
    value = rate / 1e9
    attn_mean = statistics.mean(attn_ms)
    kern_mean = statistics.mean(kern_ms)
    achieved = kvb / (kern_mean / 1e3) / 1e9
    traffic = profile_traffic("decode_tma_gqa_decode_bf16",
                              ["paged_kv_attention_20_gb300/csrc/decode_tma.cu"])

    if rank != 0:
        barrier(world)
        return
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "gqa_decode_bf16: 64 seqs x 1 decode query, Hq=32, Hkv=8, D=Dv=128, "
                               "page_size=16, ctx U[512,8192] (seed 2), shuffled pages, bf16, fp32 accumulate",
                   "step": "paged_kv_store + paged_attn_forward_split (heuristic splits) on resident inputs",
                   "splits": step.splits, "kv_bytes_per_step": kvb, "queries_per_step": case.num_queries,
                   "l2": "inputs larger than L2 (KV working set ~1.1 GB > 129 MB)",
                   "parallelism": f"replicas x{world}"},
        "queries_per_s": world * case.num_queries * args.steps / (total_ms / 1e3),
        "frac_hbm_peak": value / world / peaks["hbm_gbs"],
        "kernel_ms": {"store": statistics.mean(store_ms), "attention_call": attn_mean, "decode_kernel": kern_mean},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": achieved / peaks["hbm_gbs"], "traffic": traffic,
                     "kernel": "decode_tma_kernel<bf16,128,4>, timed alone with CUDA events recorded by the library around its launch",
                     "peak_source": f"{peaks['source']} HBM copy bandwidth"},
        "clocks": clocks,
        "gpu_launches": args.steps * step.kernels_per_step(),
    }
    del step
    torch.cuda.empty_cache()
    line["e2e"] = e2e_leg(case, device, steps=max(10, min(args.steps, 200)), warmup=args.warmup)
    which = secondary_for_run(args.secondary, world)
    if which:
        line["workloads"] = secondary(device, args.warmup, 20, peaks, which, cpu=not args.no_cpu_baseline)
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(case)
    print(json.dumps(line), flush=True)
    barrier(world)


if __name__ == "__main__":
    main()
