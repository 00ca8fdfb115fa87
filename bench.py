"""Benchmark of the single-GPU MoE layer forward (tokens/s on a B300).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME]

A step is one pass of the whole hot path (route, slot assignment, dispatch,
expert FFN, combine) over one batch of T synthetic tokens of the workload
(default: the largest one, the Mixtral 8x7B layer shape: T=32768, d=4096,
8 experts, top-2, ffn=14336, no capacity limit), inputs and weights resident
in HBM.  The L2 cache is flushed (a 2 x L2 write) before every timed step,
outside the step's events.

Printed (rank 0, one JSON line): tokens/s over the timed steps (max over
ranks of the device time), the per-call breakdown from a second, identical
loop that times each C-ABI call with events on the launching stream, the
roofline of the dominant call (the expert FFN, against the measured bf16
tensor peak), the end-to-end figure through moe_layer_forward with pinned
host buffers and the copies inside the timed region, SM clocks sampled
during the timed loop, and the CPU oracle on a bounded sample.

Multi-GPU (torchrun): every rank runs its own independent layer instance
(replicas: the layer forward has no cross-GPU exchange here), value = total
tokens of all ranks / max-over-ranks time, "scaling": "weak".

--impl reference times the CPU oracle (the only reference this method has)
on the same workload, each step a bounded sample, on rank 0 only.
"""
from __future__ import annotations

import argparse
import ctypes
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import moe_inputs  # noqa: E402

DEFAULT_WORKLOAD = "mixtral_8x7b"
METRIC = "MoE layer forward tokens/sec on 1 B300; % of HBM BW / BF16 tensor peak"
# DRAM bytes (read + write) of one expert-FFN launch per workload, as ncu
# measured them on the current kernel (dram__bytes_read.sum +
# dram__bytes_write.sum of one launch); a workload without a capture of the
# current kernel has no entry and reports null
FFN_DRAM_BYTES = {"mixtral_8x7b": 16541366272 + 2411979520}
# a launch at least this long runs under the board's power limit: its
# roofline takes the sustained bf16 peak, shorter ones the burst peak
SUSTAINED_MS = 2.0


def _peaks():
    """(HBM GB/s, bf16 burst TFLOP/s, bf16 sustained TFLOP/s, source)."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            pk = json.load(f)
        return pk["hbm_gbs"], pk["bf16_tflops"], pk.get("bf16_tflops_sustained", pk["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6400.0, 1800.0, 1400.0, "fallback"


def workload_config(wl, C, kept, dropped, world):
    """The `config` object of both arms' JSON lines (identical keys and values
    for the same workload)."""
    return {"workload": wl.name, "T": wl.T, "d": wl.d, "E": wl.E, "D": wl.D, "k": wl.k, "ffn": wl.ffn,
            "capacity_factor": wl.capacity_factor, "act": wl.act, "C_expert": C, "kept": kept,
            "dropped": dropped, "parallelism": f"replicas x{world}",
            "l2": "flushed before every timed step (2 x L2 write)"}


# ---------------------------------------------------------------- clocks --
class ClockSampler:
    """nvidia-smi SM clocks and throttle reasons, sampled every 200 ms."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.out = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=self.out, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        self.out.flush()
        self.out.seek(0)
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.out.read().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        os.unlink(self.out.name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# --------------------------------------------------------- multi-rank --
def replica_workload(wl, rank: int):
    """Each rank runs an independent layer instance (replicas): same shapes,
    inputs drawn with a rank-specific seed."""
    return wl.with_(seed=wl.seed + 1000 * rank)


def max_over_ranks(value: float, world: int, device) -> float:
    """The largest of every rank's value (all ranks get it); the identity on one rank."""
    if world == 1:
        return float(value)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(tokens_per_rank: int, world: int, steps: int, max_total_ms: float) -> float:
    """Whole-job throughput: tokens of all ranks over the slowest rank's time."""
    return world * tokens_per_rank * steps / (max_total_ms * 1e-3)


# ------------------------------------------------------------ our path --
def run_ours(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist
    import expert_parallelism_gemm_b300 as moe

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    wl = moe_inputs.WORKLOADS[args.workload]
    inp = moe_inputs.make_inputs(replica_workload(wl, rank), device=dev)
    p = moe.problem_of(wl)
    C, C_shard, rows_max = moe.moe_capacity(p)
    ws = moe.alloc_workspace(p, dev)
    wsb = ws.numel()
    y = torch.empty(wl.T, wl.d, dtype=inp.x.dtype, device=dev)
    stream = torch.cuda.current_stream(dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush_buf = torch.empty(max(2 * l2, 256 << 20), dtype=torch.uint8, device=dev)

    def flush():
        flush_buf.fill_(1)

    def step():
        moe.moe_layer_forward(p, inp.x, inp.Wg, inp.bias, inp.W1, inp.W3, inp.W2, None, y, ws, wsb,
                              stream)

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)

    # ---- warm-up
    for _ in range(args.warmup):
        flush()
        step()
    torch.cuda.synchronize(dev)
    status = moe.moe_device_status(ws, stream)
    if status != moe.MOE_OK:
        raise RuntimeError(f"device status after warm-up: {moe.moe_status_string(status)}")

    # ---- timed steps (device time, events on the launching stream)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    with ClockSampler(local_rank) as clk:
        barrier()
        for i in range(args.steps):
            flush()
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        barrier()
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    total_ms_max = max_over_ranks(sum(step_ms), world, dev)
    status = moe.moe_device_status(ws, stream)
    if status != moe.MOE_OK:
        raise RuntimeError(f"device status after timed steps: {moe.moe_status_string(status)}")

    # ---- per-call breakdown: the same step as five C-ABI calls, events between
    i32, f32 = torch.int32, torch.float32
    idx = torch.empty(wl.T, wl.k, dtype=i32, device=dev)
    gate = torch.empty(wl.T, wl.k, dtype=f32, device=dev)
    slot = torch.empty(wl.T, wl.k, dtype=i32, device=dev)
    cr, ck = torch.empty(wl.E, dtype=i32, device=dev), torch.empty(wl.E, dtype=i32, device=dev)
    off = torch.empty(wl.E + 1, dtype=i32, device=dev)
    so, sr, sov = (torch.empty(n, dtype=i32, device=dev) for n in (wl.D + 1, wl.D, wl.D))
    row_token = torch.empty(max(rows_max, 1), dtype=i32, device=dev)
    dropped = torch.empty(1, dtype=i32, device=dev)
    xd = torch.empty(max(rows_max, 1), wl.d, dtype=inp.x.dtype, device=dev)
    yd = torch.empty(max(rows_max, 1), wl.d, dtype=inp.x.dtype, device=dev)
    by_token = wl.k >= 2 and wl.T * wl.d * inp.x.element_size() > l2 // 2
    calls = ["route", "assign", "dispatch", "expert_ffn", "combine"]
    call_fns = [
        lambda: moe.moe_route(p, inp.x, inp.Wg, inp.bias, idx, gate, None, ws, wsb, None),
        lambda: moe.moe_assign_slots(p, idx, slot, cr, ck, off, so, sr, sov, row_token, dropped, ws, wsb,
                                     None),
        # the form moe_layer_forward uses: token-major for k >= 2 when x is
        # larger than half the L2 (each x row read once for all its slots),
        # expert-major otherwise
        (lambda: moe.moe_dispatch_by_token(p, inp.x, idx, slot, off, xd, None)) if by_token else
        (lambda: moe.moe_dispatch(p, inp.x, row_token, off, xd, None)),
        lambda: moe.moe_expert_ffn(p, xd, off, inp.W1, inp.W3, inp.W2, yd, ws, wsb, None),
        lambda: moe.moe_combine(p, yd, idx, slot, off, gate, None, y, None),
    ]
    for _ in range(max(1, args.warmup)):
        flush()
        for fn in call_fns:
            fn()
    torch.cuda.synchronize(dev)
    # Each call (stream None: torch's current stream, which is the capture
    # stream inside torch.cuda.graph) is captured in a CUDA graph of its own and replayed between
    # events, so the times are the calls' device time (no Python or ctypes
    # overhead between the events); the calls replay in step order, so every
    # call reads what the previous one wrote, and L2 is flushed before each.
    graphs = []
    for fn in call_fns:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        graphs.append(g)
    torch.cuda.synchronize(dev)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2 * len(calls))] for _ in range(args.steps)]
    barrier()
    for i in range(args.steps):
        for j, g in enumerate(graphs):
            flush()
            evs[i][2 * j].record(stream)
            g.replay()
            evs[i][2 * j + 1].record(stream)
    barrier()
    per_call = {c: statistics.mean(e[2 * j].elapsed_time(e[2 * j + 1]) for e in evs)
                for j, c in enumerate(calls)}
    status = moe.moe_device_status(ws, stream)
    if status != moe.MOE_OK:
        raise RuntimeError(f"device status after the per-call loop: {moe.moe_status_string(status)}")
    kept = int(off[-1].item())
    n_dropped = int(dropped.item())

    # ---- routing statistics (load-balancing term, entropy, drops, imbalance)
    # from the router's probabilities: one captured call, timed like the others
    probs = torch.empty(wl.T, wl.E, dtype=f32, device=dev)
    moe.moe_route(p, inp.x, inp.Wg, inp.bias, idx, gate, probs, ws, wsb, None)
    stats = torch.empty(moe.MOE_NUM_STATS, dtype=f32, device=dev)
    mean_prob = torch.empty(wl.E, dtype=f32, device=dev)
    stats_fn = lambda: moe.moe_routing_stats(p, probs, cr, ck, stats, mean_prob, ws, wsb, None)
    stats_fn()
    torch.cuda.synchronize(dev)
    g_stats = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_stats):
        stats_fn()
    st_ev = []
    for _ in range(args.steps):
        flush()
        a_ev, b_ev = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a_ev.record(stream)
        g_stats.replay()
        b_ev.record(stream)
        st_ev.append((a_ev, b_ev))
    torch.cuda.synchronize(dev)
    stats_ms = statistics.mean(a_ev.elapsed_time(b_ev) for a_ev, b_ev in st_ev)
    stats_vals = stats.cpu().tolist()

    # ---- a shared expert as wide as a routed one over every token (the
    # layer option of moe_layer_forward_shared), timed alone like the calls
    shared_ms = shared_layer_ms = None
    if wl.dtype == "bf16" and wl.act == "swiglu":
        swl = wl.with_(ffn_shared=wl.ffn)
        sp = moe.problem_of(swl)
        sws = moe.alloc_workspace(sp, dev)
        sin = moe_inputs.make_inputs(replica_workload(swl, rank), device=dev)
        ys = torch.empty(wl.T, wl.d, dtype=inp.x.dtype, device=dev)
        sh_fn = lambda: moe.moe_shared_expert_ffn(sp, sin.x, sin.Ws1, sin.Ws3, sin.Ws2, ys, sws, sws.numel(),
                                                  None)
        sh_fn()
        torch.cuda.synchronize(dev)
        g_sh = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_sh):
            sh_fn()
        sh_ev = []
        for _ in range(args.steps):
            flush()
            a_ev, b_ev = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a_ev.record(stream)
            g_sh.replay()
            b_ev.record(stream)
            sh_ev.append((a_ev, b_ev))
        torch.cuda.synchronize(dev)
        shared_ms = statistics.mean(a_ev.elapsed_time(b_ev) for a_ev, b_ev in sh_ev)
        if moe.moe_device_status(sws, stream) != moe.MOE_OK:
            raise RuntimeError("device status after the shared-expert loop")
        # the whole layer with that shared expert (its FFN overlaps the routed
        # FFN's last tiles), against the routed layer and the shared FFN apart
        ys_layer = torch.empty(wl.T, wl.d, dtype=inp.x.dtype, device=dev)
        shl_fn = lambda: moe.moe_layer_forward_shared(sp, sin.x, sin.Wg, sin.bias, sin.W1, sin.W3, sin.W2, sin.Ws1,
                                                      sin.Ws3, sin.Ws2, None, ys_layer, sws, sws.numel(), None)
        shl_fn()
        torch.cuda.synchronize(dev)
        g_shl = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_shl):
            shl_fn()
        shl_ev = []
        for _ in range(args.steps):
            flush()
            a_ev, b_ev = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a_ev.record(stream)
            g_shl.replay()
            b_ev.record(stream)
            shl_ev.append((a_ev, b_ev))
        torch.cuda.synchronize(dev)
        shared_layer_ms = statistics.mean(a_ev.elapsed_time(b_ev) for a_ev, b_ev in shl_ev)
        if moe.moe_device_status(sws, stream) != moe.MOE_OK:
            raise RuntimeError("device status after the shared-layer loop")
        del sin, sws, ys, ys_layer, g_sh, g_shl

    def time_layer_variant(vwl, what):
        """One whole moe_layer_forward of a layer variant per graph replay;
        returns (mean ms, the variant's workspace)."""
        vp = moe.problem_of(vwl)
        vws = moe.alloc_workspace(vp, dev)
        fn = lambda: moe.moe_layer_forward(vp, inp.x, inp.Wg, inp.bias, inp.W1, inp.W3, inp.W2, None, y, vws,
                                           vws.numel(), None)
        fn()
        torch.cuda.synchronize(dev)
        g_v = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_v):
            fn()
        v_ev = []
        for _ in range(args.steps):
            flush()
            a_ev, b_ev = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a_ev.record(stream)
            g_v.replay()
            b_ev.record(stream)
            v_ev.append((a_ev, b_ev))
        torch.cuda.synchronize(dev)
        if moe.moe_device_status(vws, stream) != moe.MOE_OK:
            raise RuntimeError(f"device status after the {what} loop")
        return statistics.mean(a_ev.elapsed_time(b_ev) for a_ev, b_ev in v_ev), vws

    # ---- the same layer with expert-choice routing (each expert takes its
    # C highest-scoring tokens)
    ewl = wl.with_(expert_choice=True)
    ec_ms, ews = time_layer_variant(ewl, "expert-choice")
    ec_rows = ewl.E * moe.moe_capacity(moe.problem_of(ewl))[0]
    del ews

    # ---- the same layer with overflow rerouting to the next-best expert
    rr_ms, rr_stats = None, None
    if 2 * wl.k <= wl.E:
        rwl = wl.with_(reroute=True)
        rr_ms, rws = time_layer_variant(rwl, "rerouting")
        rp = moe.problem_of(rwl)
        rr_stats = {n: int(moe.workspace_view(rws, rp, n, torch.int32, 1).item()) for n in ("rerouted", "dropped")}
        rr_stats["kept"] = int(moe.workspace_view(rws, rp, "expert_offsets", torch.int32, wl.E + 1)[-1].item())
        del rws

    # ---- end to end through moe_layer_forward_host: every step copies its x
    # in from page-locked host memory (moe_host_alloc) and its y back out.
    # Serial: one step per call, L2 flushed before each.  Pipelined (the e2e
    # value): K steps in one call, step i's input copy overlapping step i-1's
    # layer and step i-2's output copy on the library's copy streams; no L2
    # flush there, as x arrives from the host every step and the 176 MB of
    # expert weights the layer streams exceed L2.
    eb_ = inp.x.element_size()
    nbytes = wl.T * wl.d * eb_
    hx = [moe.moe_host_alloc(nbytes) for _ in range(2)]
    hy = [moe.moe_host_alloc(nbytes) for _ in range(2)]
    # written by one thread: host lines left dirty in many cores' caches by a
    # multi-threaded fill made every later copy from them ~5x slower here
    x_bytes = inp.x.cpu().contiguous().view(torch.uint8).numpy().reshape(-1)
    for a in hx:
        np.copyto(np.ctypeslib.as_array((ctypes.c_uint8 * nbytes).from_address(a)), x_bytes)
    stg_bytes = moe.moe_host_staging_size(p)
    staging = torch.empty(stg_bytes, dtype=torch.uint8, device=dev)

    def host_run(n):
        moe.moe_layer_forward_host(p, [hx[i % 2] for i in range(n)], inp.Wg, inp.bias, inp.W1, inp.W3, inp.W2,
                                   [hy[i % 2] for i in range(n)], staging, stg_bytes, ws, wsb, stream)

    for _ in range(max(1, args.warmup)):
        flush()
        host_run(1)
    e_s = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    e_e = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    barrier()
    for i in range(args.steps):
        flush()
        e_s[i].record(stream)
        host_run(1)
        e_e[i].record(stream)
    barrier()
    e2e_serial_ms_max = max_over_ranks(sum(a.elapsed_time(b) for a, b in zip(e_s, e_e)), world, dev)

    host_run(max(3, args.warmup))
    barrier()
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    host_run(args.steps)
    t_end.record(stream)
    barrier()
    e2e_ms_max = max_over_ranks(t_start.elapsed_time(t_end), world, dev)
    y_last = moe.host_tensor(hy[(args.steps - 1) % 2], (wl.T, wl.d), inp.x.dtype).clone()
    for a in hx + hy:
        moe.moe_host_free(a)
    if moe.moe_device_status(ws, stream) != moe.MOE_OK:
        raise RuntimeError("device status after the end-to-end loops")
    step()
    torch.cuda.synchronize(dev)
    if not torch.equal(y_last, y.cpu()):
        raise RuntimeError("end-to-end output differs from the device step's output")

    out = None
    if rank == 0:
        eb = 2 if wl.dtype == "bf16" else 4
        hbm_gbs, bf16_burst, bf16_sust, peak_src = _peaks()
        sustained = per_call["expert_ffn"] >= SUSTAINED_MS
        bf16_tf = bf16_sust if sustained else bf16_burst
        mats = 3 if wl.act == "swiglu" else 2
        ffn_flops = 2.0 * mats * wl.d * wl.ffn * kept
        ffn_s = per_call["expert_ffn"] * 1e-3
        achieved_tf = ffn_flops / ffn_s / 1e12
        n_exp_used = int((ck > 0).sum().item())
        route_bytes = wl.T * wl.d * eb + wl.E * wl.d * eb + wl.T * wl.k * 8
        disp_tokens = int((slot >= 0).any(dim=1).sum().item())
        dispatch_bytes = disp_tokens * wl.d * eb + kept * wl.d * eb
        combine_bytes = kept * wl.d * eb + wl.T * wl.d * eb + wl.T * wl.k * 12
        weight_bytes = mats * wl.d * wl.ffn * eb * n_exp_used
        # the expert FFN's DRAM floor: each used expert's weights once, plus xd
        # read, h written and read back, yd written, per kept row
        ffn_bytes = weight_bytes + kept * (2 * wl.d + 2 * wl.ffn) * eb
        hbm_bound = ffn_bytes / (hbm_gbs * 1e9) > ffn_flops / (bf16_tf * 1e12)
        gb = lambda b, ms: b / (ms * 1e-3) / 1e9
        kernels = {
            "route": {"ms": per_call["route"], "GB_s": gb(route_bytes, per_call["route"]),
                      "frac_hbm": gb(route_bytes, per_call["route"]) / hbm_gbs},
            "assign": {"ms": per_call["assign"]},
            "dispatch": {"ms": per_call["dispatch"], "GB_s": gb(dispatch_bytes, per_call["dispatch"]),
                         "frac_hbm": gb(dispatch_bytes, per_call["dispatch"]) / hbm_gbs,
                         "form": "moe_dispatch_by_token" if by_token else "moe_dispatch"},
            "expert_ffn": {"ms": per_call["expert_ffn"], "TFLOP_s": achieved_tf,
                           "frac_bf16": achieved_tf / bf16_tf,
                           "weight_GB_s": gb(weight_bytes, per_call["expert_ffn"]),
                           "GB_s": gb(ffn_bytes, per_call["expert_ffn"]),
                           "frac_hbm": gb(ffn_bytes, per_call["expert_ffn"]) / hbm_gbs},
            "combine": {"ms": per_call["combine"], "GB_s": gb(combine_bytes, per_call["combine"]),
                        "frac_hbm": gb(combine_bytes, per_call["combine"]) / hbm_gbs},
            "shared_expert_ffn": None if shared_ms is None else {
                "ms": shared_ms, "ffn_shared": wl.ffn,
                "TFLOP_s": 2.0 * mats * wl.d * wl.ffn * wl.T / (shared_ms * 1e-3) / 1e12,
                "frac_bf16": 2.0 * mats * wl.d * wl.ffn * wl.T / (shared_ms * 1e-3) / (bf16_tf * 1e12),
                "layer_ms": shared_layer_ms,
                "note": "ms: moe_shared_expert_ffn alone; layer_ms: moe_layer_forward_shared, graph replay"},
            "expert_choice_layer": {"ms": ec_ms, "tokens_per_s": wl.T / (ec_ms * 1e-3), "rows": ec_rows,
                                    "note": "whole moe_layer_forward with expert-choice routing, graph replay"},
            "reroute_layer": None if rr_ms is None else dict(
                ms=rr_ms, tokens_per_s=wl.T / (rr_ms * 1e-3), **rr_stats,
                note="whole moe_layer_forward with overflow rerouting, graph replay"),
            "routing_stats": {"ms": stats_ms, "GB_s": gb(wl.T * wl.E * 4 + 8 * wl.E, stats_ms),
                              "aux": stats_vals[0], "entropy": stats_vals[1], "drop": stats_vals[2],
                              "imbalance": stats_vals[3]},
        }
        value = job_tokens_per_s(wl.T, world, args.steps, total_ms_max)
        clocks = clk.summary()
        out = {
            "metric": METRIC,
            "value": value,
            "unit": "tokens/s",
            "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": total_ms_max / args.steps,
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": wl.dtype,
            "data": "synthetic (seeded torch generator on the device; random-init weights)",
            "config": workload_config(wl, C, kept, n_dropped, world),
            "roofline": ffn_roofline(hbm_bound, achieved_tf, bf16_tf, bf16_burst, bf16_sust,
                                     gb(ffn_bytes, per_call["expert_ffn"]), hbm_gbs, ffn_bytes, kept,
                                     FFN_DRAM_BYTES.get(wl.name),
                                     (f"{peak_src} bf16 sustained (a {per_call['expert_ffn']:.1f} ms launch "
                                      f"runs under the power limit)" if sustained else f"{peak_src} bf16 burst"),
                                     peak_src, mats),
            "kernels": kernels,
            "e2e": {"value": job_tokens_per_s(wl.T, world, args.steps, e2e_ms_max), "unit": "tokens/s",
                    "h2d_bytes_per_step": wl.T * wl.d * eb, "d2h_bytes_per_step": wl.T * wl.d * eb,
                    "ms_per_step": e2e_ms_max / args.steps,
                    "api": "moe_layer_forward_host: K steps, x copied in from page-locked host memory and y "
                           "copied out every step, copies of neighbouring steps overlapping the layer",
                    "serial": {"value": job_tokens_per_s(wl.T, world, args.steps, e2e_serial_ms_max),
                               "ms_per_step": e2e_serial_ms_max / args.steps,
                               "note": "one step per moe_layer_forward_host call, L2 flushed before each"}},
            "gpu_launches": args.steps * launches_per_step(wl),
            "clocks": clocks,
        }
    return out


def ffn_roofline(hbm_bound, achieved_tf, bf16_tf, bf16_burst, bf16_sust, achieved_gbs, hbm_gbs, ffn_bytes,
                 kept, traffic, tensor_src, peak_src, mats):
    """The expert FFN launch against whichever floor is higher for this shape:
    the tensor pipe (flops / bf16 peak) or HBM (its algorithmic bytes / copy
    bandwidth).  Experts with few rows each stream their weights faster than
    the MMAs on them can finish, and are HBM-bound."""
    kernel = "moe_expert_ffn (one persistent tcgen05 launch: gate/up + down)"
    both = {"frac_burst": achieved_tf / bf16_burst, "frac_sustained": achieved_tf / bf16_sust,
            "tflops": achieved_tf, "gbs": achieved_gbs, "frac_hbm": achieved_gbs / hbm_gbs}
    if hbm_bound:
        return {"kernel": kernel, "bound": "hbm", "achieved": achieved_gbs, "peak": hbm_gbs, "unit": "GB/s",
                "frac": achieved_gbs / hbm_gbs, "traffic": traffic, "peak_source": f"{peak_src} HBM copy",
                **both, "algorithmic": f"{mats}*d*ffn*b per used expert + (2*d + 2*ffn)*b per kept row "
                                       f"({ffn_bytes} B, {kept} rows)"}
    return {"kernel": kernel, "bound": "tensor", "achieved": achieved_tf, "peak": bf16_tf, "unit": "TFLOP/s",
            "frac": achieved_tf / bf16_tf, "traffic": traffic, "peak_source": tensor_src,
            **both, "algorithmic": f"2*{mats}*d*ffn flops per kept row x {kept} rows"}


def launches_per_step(wl) -> int:
    """Kernels of one moe_layer_forward, as the library counts them."""
    import expert_parallelism_gemm_b300 as moe
    return moe.moe_layer_launch_count(moe.problem_of(wl))


# -------------------------------------------------------------- oracle --
def oracle_sample_step(wl, cpu_inp, n_tokens, rng, want_slots=False):
    """One bounded oracle step: routing and slots for all T tokens, then the
    expert FFN and combine of n_tokens sampled tokens.  Returns
    (seconds for routing, seconds for the sample, tokens in the sample), and
    the slot assignment as a fourth item with want_slots."""
    import oracle
    t0 = time.perf_counter()
    g, _, idx, gate = oracle.route(cpu_inp.x, cpu_inp.Wg, cpu_inp.bias, wl.k, want_probs=False)
    slots = oracle.assign(idx, wl.E, wl.D, wl.capacity_factor)
    t1 = time.perf_counter()
    toks = rng.choice(wl.T, size=min(n_tokens, wl.T), replace=False)
    oracle.token_outputs(toks, cpu_inp.x, idx, slots.slot_pos, gate, cpu_inp.W1, cpu_inp.W3,
                         cpu_inp.W2, oracle.act_code(wl.act))
    t2 = time.perf_counter()
    if want_slots:
        return t1 - t0, t2 - t1, len(toks), slots
    return t1 - t0, t2 - t1, len(toks)


def oracle_tokens_per_s(wl, route_s, sample_s, n):
    # the whole layer's time: routing of all T tokens plus T/n times the sample
    return wl.T / (route_s + sample_s * wl.T / n)


def oracle_cores():
    n = os.environ.get("OMP_NUM_THREADS")
    return int(n) if n else len(os.sched_getaffinity(0))


def cpu_baseline(wl, budget_s=12.0):
    cpu = moe_inputs.make_inputs(wl, device="cpu")
    rng = np.random.default_rng(0)
    # size the sample to the budget from a calibration run; a small sample
    # parallelises poorly over the host's threads and overstates the cost per
    # token, so the size is corrected once more from the first sized run
    r_s, s_s, n = oracle_sample_step(wl, cpu, min(wl.T, 128), rng)
    for _ in range(2):
        per_tok = s_s / max(n, 1)
        n_next = int(max(16, min(wl.T, (budget_s - r_s) / max(per_tok, 1e-6))))
        r_s, s_s, n = oracle_sample_step(wl, cpu, n_next, rng)
        if r_s + s_s >= 0.5 * budget_s or n >= wl.T:
            break
    out = {"value": oracle_tokens_per_s(wl, r_s, s_s, n), "unit": "tokens/s", "cores": oracle_cores(),
           "kind": "oracle",
           "sample": (f"the whole layer, all {wl.T} tokens ({r_s + s_s:.1f} s of CPU work)" if n >= wl.T else
                      f"routing + slots of all {wl.T} tokens, expert FFN + combine of {n} random tokens, "
                      f"extrapolated to {wl.T} ({r_s + s_s:.1f} s of CPU work)")}
    # the same on one thread, on a smaller sample sized from the run above
    one = single_thread_oracle(wl, cpu, rng, per_tok=s_s / max(n, 1) * oracle_cores(), budget_s=budget_s / 3)
    if one is not None:
        out["single_core"] = one
    return out


def _set_omp_threads(n: int) -> bool:
    import ctypes.util
    name = ctypes.util.find_library("gomp") or "libgomp.so.1"
    try:
        ctypes.CDLL(name).omp_set_num_threads(int(n))
        return True
    except OSError:
        return False


def single_thread_oracle(wl, cpu, rng, per_tok, budget_s):
    """The oracle's tokens/s on one OpenMP thread (routing + slots of all T
    tokens, FFN + combine of a sample), or None if the runtime is not found."""
    if not _set_omp_threads(1):
        return None
    try:
        n1 = int(max(8, min(wl.T, budget_s / max(per_tok, 1e-6))))
        r_s, s_s, n = oracle_sample_step(wl, cpu, n1, rng)
    finally:
        _set_omp_threads(oracle_cores())
    return {"value": oracle_tokens_per_s(wl, r_s, s_s, n), "unit": "tokens/s", "cores": 1,
            "sample": f"routing + slots of all {wl.T} tokens, expert FFN + combine of {n} random tokens, "
                      f"extrapolated to {wl.T} ({r_s + s_s:.1f} s on one thread)"}


def run_reference(args, rank):
    """The oracle as it stands, on the host's cores: every step routes and
    assigns all T tokens and runs the expert FFN and combine of a random token
    sample sized so the whole run takes a few minutes.  ms_per_step is the
    measured wall time of a step; the layer time the oracle would need for all
    T tokens (the sample extrapolated linearly) gives `value` and is printed
    as extrapolated_ms_per_layer."""
    if rank != 0:
        return None
    wl = moe_inputs.WORKLOADS[args.workload]
    cpu = moe_inputs.make_inputs(wl, device="cpu")
    rng = np.random.default_rng(0)
    r_s, s_s, n = oracle_sample_step(wl, cpu, 8, rng)
    per_tok = s_s / max(n, 1)
    # about 150 s for all warm-up and timed steps together, at least 8 tokens a step
    step_budget = max(r_s + 8 * per_tok, 150.0 / (args.steps + args.warmup))
    n_step = int(max(8, min(wl.T, (step_budget - r_s) / max(per_tok, 1e-6))))
    for _ in range(args.warmup):
        oracle_sample_step(wl, cpu, n_step, rng)
    rs, ss = 0.0, 0.0
    t_start = time.perf_counter()
    for _ in range(args.steps):
        a, b, n, slots = oracle_sample_step(wl, cpu, n_step, rng, want_slots=True)
        rs += a
        ss += b
    wall_ms = 1e3 * (time.perf_counter() - t_start) / args.steps
    value = oracle_tokens_per_s(wl, rs / args.steps, ss / args.steps, n)
    sample = (f"each step: routing + slots of all {wl.T} tokens, expert FFN + combine of {n} random "
              f"tokens; value extrapolated to all {wl.T} tokens")
    kept = int(slots.expert_offsets[-1])
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": wall_ms,
            "extrapolated_ms_per_layer": 1e3 * wl.T / value,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": wl.dtype,
            "data": "synthetic (seeded torch generator on the host)",
            "config": workload_config(wl, int(slots.C), kept, int(slots.dropped), 1),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": oracle_cores(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(moe_inputs.WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        out = run_reference(args, rank)
        if out is not None:
            print(json.dumps(out), flush=True)
        return 0

    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    out = run_ours(args, rank, world, local_rank)
    if rank == 0:
        # the oracle baseline is timed on rank 0 of a one-GPU run only
        if not args.no_cpu_baseline and world == 1:
            out["cpu_baseline"] = cpu_baseline(moe_inputs.WORKLOADS[args.workload])
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
