"""Benchmark: causal bf16 attention forward + backward on one GB300.

Step = one pass of the hot path over one batch: ``attn_fwd`` (O, LSE) and
``attn_bwd`` (row terms, dq/dk/dv) of causal self-attention, bf16,
B=4, S=4096, H=16, D=128 (16384 tokens per batch, the S>=4096 point of the
head-dim-128 sweep).  The LSE merge and the fp32 path are timed in the same
run as auxiliary lines (``aux``).  Throughput counts algorithmic flops:
forward 4*D*N_vis, backward 10*D*N_vis (five GEMM-shaped products including
the recompute of S), N_vis = exact number of visible (query, key) pairs.

``--impl reference`` times the float64 CPU oracle on a bounded sample of the
same workload instead (the reference arm; the oracle is test
infrastructure, used here only as that baseline).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = dict(B=4, S=4096, H=16, D=128, window=(-1, 0))
# DRAM bytes (read + write) per launch of the dominant kernel on this workload,
# from a one-kernel ncu capture of this command (dram__bytes metrics; see
# profiles/); None when the kernel changed after the capture.
TRAFFIC = {"bwd_fused": 626503168}
METRIC = "attention TFLOP/s fwd+bwd (bf16 causal) and % of GB300 dense BF16 tensor peak"


def n_visible(S, window):
    wl, wr = window
    n = 0
    for i in range(S):
        lo = 0 if wl < 0 else max(0, i - wl)
        hi = S - 1 if wr < 0 else min(S - 1, i + wr)
        n += max(0, hi - lo + 1)
    return n


def flops(B, S, H, D, window):
    nv = n_visible(S, window) * B * H
    return 4.0 * D * nv, 10.0 * D * nv, nv


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index, period_ms=10):
        self.index = index
        self.period_ms = period_ms
        self.proc = None
        self.lines = []
        self.marks = {}

    def mark(self, name):
        """Remembers how many samples had arrived at this point."""
        self.marks[name] = len(self.lines)

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", str(self.period_ms)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        out = {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
               "reasons": sorted(reasons), "samples": len(sm),
               "span": "from the start of the timed region through the per-kernel region and the "
                       "end-to-end leg, every %d ms" % self.period_ms}
        if "region1_start" in self.marks and "region1_end" in self.marks:
            out["samples_in_timed_region"] = self.marks["region1_end"] - self.marks["region1_start"]
        return out


def dist_setup(args, backend="nccl"):
    """Rank, world size and local rank from the torchrun environment; one
    process group per job (NCCL across GPUs; gloo for the CPU tests)."""
    import torch
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, ws):
    """The slowest rank's time: the job is done when every rank is."""
    if ws == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(ws, flops_per_rank_step, ms_per_step):
    """Whole-job TFLOP/s: every rank processes its own (weak-scaled) batch of
    flops_per_rank_step in each step, and a step takes ms_per_step (the max
    over ranks)."""
    return ws * flops_per_rank_step / (ms_per_step * 1e-3) / 1e12


def run_ours(args):
    import torch
    import scaled_dot_product_03_gb300 as gb
    from scaled_dot_product_03_gb300 import build as libbuild
    from scaled_dot_product_03_gb300 import inputs

    ws, rank, local = dist_setup(args)
    libbuild.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    B, S, H, D, win = (WORKLOAD[k] for k in ("B", "S", "H", "D", "window"))
    if args.shape:
        B, S, H, D = (int(x) for x in args.shape.split(","))
    prob = inputs.dense(B, S, H, D, window=win, seed=rank)
    d = prob.to(dev)
    q, k, v, dout = d.q, d.k, d.v, d.dout
    scale = d.scale
    o = torch.empty_like(q)
    lse = torch.empty(B, H, S, dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    wsb = gb.attn_bwd_workspace_size(q, k, scale=scale, window=win)
    work = torch.empty(wsb, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(ev=None):
        if ev:
            ev[0].record(stream)
        gb.attn_fwd(q, k, v, scale=scale, window=win, out=o, lse=lse)
        if ev:
            ev[1].record(stream)
        gb.attn_bwd(dout, q, k, v, o, lse, scale=scale, window=win, dq=dq, dk=dk, dv=dv,
                    workspace=work)
        if ev:
            ev[2].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    gb.check_device_error()
    # Timed region 1 (the reported value): K steps bracketed only by two
    # events, a barrier and a synchronize.  nvidia-smi samples the clocks from
    # here through region 2 and the end-to-end leg, so that a short region 1
    # still has a clock record around it (its own samples are counted apart).
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clk = ClockSampler(local).__enter__()
    time.sleep(0.05)
    barrier(ws)
    torch.cuda.synchronize()
    clk.mark("region1_start")
    start.record(stream)
    for i in range(args.steps):
        step()
    end.record(stream)
    torch.cuda.synchronize()
    clk.mark("region1_end")
    barrier(ws)
    gb.check_device_error()
    ms_total = max_over_ranks(start.elapsed_time(end), ws)
    # Timed region 2 (the breakdown): the same K steps with every kernel
    # launch bracketed by CUDA events on its own stream (the library's
    # per-launch timing hook) and the forward / backward split by events.
    # Recording those events costs ~2% of a step, so it stays out of region 1.
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    barrier(ws)
    torch.cuda.synchronize()
    gb.profile_begin(8 * args.steps)
    for i in range(args.steps):
        step(evs[i])
    torch.cuda.synchronize()
    launches = gb.profile_read(8 * args.steps)
    barrier(ws)
    gb.check_device_error()
    fwd_ms = [e[0].elapsed_time(e[1]) for e in evs]
    bwd_ms = [e[1].elapsed_time(e[2]) for e in evs]
    f_fwd, f_bwd, nvis = flops(B, S, H, D, win)
    ms_step = ms_total / args.steps
    tflops = job_throughput(ws, f_fwd + f_bwd, ms_step)
    peaks, src = measured_peaks()
    peak_bf16 = peaks.get("bf16_tflops_sustained" if args.steps * ms_step > 2000 else "bf16_tflops")
    # per-kernel launch statistics; flops each kernel executes and the part of
    # them that belongs to the algorithm's count (4 + 10 D N_vis per step)
    # (bwd_fused: S, dP, dV, dK and the dQ share, each pair once; the
    # deterministic two-kernel backward splits them as bwd_dkdv + bwd_dq and
    # recomputes S and dP in the second)
    exec_flops = {"fwd": 4.0 * D * nvis, "bwd_fused": 10.0 * D * nvis,
                  "bwd_dkdv": 8.0 * D * nvis, "bwd_dq": 6.0 * D * nvis}
    alg_flops = {"fwd": 4.0 * D * nvis, "bwd_fused": 10.0 * D * nvis,
                 "bwd_dkdv": 8.0 * D * nvis, "bwd_dq": 2.0 * D * nvis}
    kern = {}
    for name, ms in launches:
        kern.setdefault(name, []).append(ms)
    kernels = {}
    for name, lst in kern.items():
        m = statistics.mean(lst)
        kernels[name] = {"launches": len(lst), "mean_ms": round(m, 4),
                         "share": round(sum(lst) / max(1e-9, sum(sum(v) for v in kern.values())), 4)}
        if name in exec_flops:
            kernels[name]["executed_tflops"] = round(exec_flops[name] / (m * 1e-3) / 1e12, 1)
            kernels[name]["algorithmic_tflops"] = round(alg_flops[name] / (m * 1e-3) / 1e12, 1)
    # HBM-bound kernels: algorithmic bytes per launch and achieved GB/s
    # (preprocess: reads O and dO, writes delta and clears the fp32 dq
    # accumulator; convert: reads the accumulator, writes dq)
    elt, rows = 2, B * H * S
    hbm_bytes = {"bwd_preprocess": rows * (2 * D * elt + 4 + 4 * D),
                 "bwd_dq_convert": rows * (4 * D + D * elt)}
    for name, nbytes in hbm_bytes.items():
        if name in kernels:
            gbs = nbytes / (kernels[name]["mean_ms"] * 1e-3) / 1e9
            kernels[name].update({"algorithmic_bytes": nbytes, "GB/s": round(gbs, 1),
                                  "hbm_frac": round(gbs / peaks["hbm_gbs"], 4)})
    dominant = max(kern, key=lambda k: sum(kern[k]))

    # ------------------------------------------------------------- end to end
    # through the public API with host buffers: every step copies its q, k, v,
    # dO in from pinned host memory, runs fwd + bwd, and copies dq, dk, dv
    # (and the loss-side O) back.  As in a training loop that prefetches,
    # the steps are pipelined on three streams over two device buffer sets:
    # step i's copy-in (stream s_in) overlaps step i-1's compute, and its
    # copy-out (stream s_out) overlaps step i+1's compute.  A set's inputs
    # (q, k, v, dO) are refilled once the compute two steps back has read
    # them, and its outputs (dq, dk, dv, O) rewritten once that step's
    # copy-out has read them, so copies in both directions run back to back
    # and the link sets the pace.  Every step's copies lie inside the timed
    # region.
    hq = [t.cpu().pin_memory() for t in (prob.q, prob.k, prob.v, prob.dout)]
    h2d = sum(t.numel() * t.element_size() for t in hq)
    sets = []
    for n in range(2):
        bufs = dict(q=q, k=k, v=v, dout=dout, o=o, lse=lse, dq=dq, dk=dk, dv=dv) if n == 0 else \
            {name: torch.empty_like(t) for name, t in
             dict(q=q, k=k, v=v, dout=dout, o=o, lse=lse, dq=dq, dk=dk, dv=dv).items()}
        bufs["hout"] = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in (q, k, v, q)]
        sets.append(bufs)
    d2h = sum(t.numel() * t.element_size() for t in sets[0]["hout"])
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = {key: [torch.cuda.Event() for _ in range(2)] for key in ("in", "comp", "out")}
    for n in range(2):
        ev["comp"][n].record(stream)
        ev["out"][n].record(s_out)

    def e2e_step(i):
        b, n = sets[i % 2], i % 2
        s_in.wait_event(ev["comp"][n])         # set n's inputs read by step i-2
        with torch.cuda.stream(s_in):
            for src_t, dst_t in zip(hq, (b["q"], b["k"], b["v"], b["dout"])):
                dst_t.copy_(src_t, non_blocking=True)
        ev["in"][n].record(s_in)
        stream.wait_event(ev["in"][n])
        stream.wait_event(ev["out"][n])        # set n's outputs copied out by step i-2
        gb.attn_fwd(b["q"], b["k"], b["v"], scale=scale, window=win, out=b["o"], lse=b["lse"])
        gb.attn_bwd(b["dout"], b["q"], b["k"], b["v"], b["o"], b["lse"], scale=scale, window=win,
                    dq=b["dq"], dk=b["dk"], dv=b["dv"], workspace=work)
        ev["comp"][n].record(stream)
        s_out.wait_event(ev["comp"][n])
        with torch.cuda.stream(s_out):
            for src_t, dst_t in zip((b["dq"], b["dk"], b["dv"], b["o"]), b["hout"]):
                dst_t.copy_(src_t, non_blocking=True)
        ev["out"][n].record(s_out)

    e2e_ms = float("nan")
    if not args.no_e2e:
        for i in range(max(2, args.warmup)):
            e2e_step(i)
        torch.cuda.synchronize()
        s2, e2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(ws)
        s2.record(stream)
        s_in.wait_event(s2)                    # no copy starts before the clock
        for i in range(args.steps):
            e2e_step(i)
        for n in range(2):                     # every copy-out done
            stream.wait_event(ev["out"][n])
        e2.record(stream)
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks(s2.elapsed_time(e2), ws) / args.steps
        # the results are those of the device-resident step
        assert torch.equal(sets[0]["o"], sets[1]["o"]) or args.steps < 2
    e2e_tflops = job_throughput(ws, f_fwd + f_bwd, e2e_ms) if e2e_ms == e2e_ms else None
    clk.__exit__(None, None, None)

    aux = aux_lines(gb, inputs, dev, peaks) if rank == 0 and not args.no_aux else {}
    if rank == 0 and not args.no_aux:
        aux["causal_fwd_bwd_sweep"] = sweep_lines(gb, inputs, dev, peaks["bf16_tflops"])
        aux.update(workload_lines(gb, inputs, dev, peaks["bf16_tflops"]))
        aux.update(head_dim_and_mqa_lines(gb, inputs, dev, peaks["bf16_tflops"]))
    cpu = cpu_baseline(args) if rank == 0 and ws == 1 and not args.no_cpu else None

    if rank != 0:
        return None
    fwd_mean = statistics.mean(fwd_ms)
    bwd_mean = statistics.mean(bwd_ms)
    dom_ms = kernels[dominant]["mean_ms"]
    dom_flops = alg_flops.get(dominant, 0.0)
    achieved = dom_flops / (dom_ms * 1e-3) / 1e12
    line = {
        "metric": METRIC,
        "value": round(tflops, 2),
        "unit": "TFLOP/s",
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic: seeded N(0,1) q, k, v, dO on the CPU generator",
        "config": {"workload": "causal self-attention fwd+bwd, bf16, B=%d S=%d H=%d D=%d" % (
            B, S, H, D), "B": B, "S": S, "H": H, "D": D, "window": list(win),
            "parallelism": "replicas" if ws > 1 else "single-gpu",
            "l2": "inputs larger than L2 (q,k,v,o,dO,dq,dk,dv = %d MB)" % (
                8 * q.numel() * 2 // 2**20),
            "flops_per_step": f_fwd + f_bwd, "n_visible_pairs": nvis},
        "pct_of_peak": round(100.0 * tflops / ws / peak_bf16, 2),
        "peak_tflops": peak_bf16, "peak_source": src,
        "fwd_ms": round(fwd_mean, 4), "bwd_ms": round(bwd_mean, 4),
        "fwd_tflops": round(f_fwd / (fwd_mean * 1e-3) / 1e12, 2),
        "bwd_tflops": round(f_bwd / (bwd_mean * 1e-3) / 1e12, 2),
        "bwd_tflops_without_recompute": round(0.8 * f_bwd / (bwd_mean * 1e-3) / 1e12, 2),
        "roofline": {"bound": "tensor", "kernel": dominant, "achieved": round(achieved, 2),
                     "peak": peak_bf16, "unit": "TFLOP/s",
                     "frac": round(achieved / peak_bf16, 4),
                     "traffic": TRAFFIC.get(dominant), "peak_source": src,
                     "algorithmic_flops_per_launch": dom_flops},
        "kernels": kernels,
        "clocks": clk.summary(),
        "ms_per_step_x_sm_ghz": (round(ms_step * clk.summary()["sm_mhz"] / 1000.0, 4)
                                 if clk.summary()["sm_mhz"] else None),
        "e2e": {"value": None if e2e_tflops is None else round(e2e_tflops, 2), "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(e2e_ms, 4),
                "overlap": "step i+1's copy-in and step i-1's copy-out overlap step i's compute "
                           "(two device buffer sets; compute, copy-in and copy-out streams)"},
        "gpu_launches": len(launches),
        "timing": "value: K steps between two events (region 1); kernels, fwd_ms, bwd_ms and the "
                  "roofline: a second K-step region with per-launch events (the same launches)",
        "cpu_baseline": cpu,
        "aux": aux,
    }
    return line


def sweep_lines(gb, inputs, dev, peak):
    """fwd+bwd TFLOP/s of the causal bf16 sequence-length sweep (16384 tokens
    per batch, H=16, D=128) and of the B=8 S=1024 D=64 case."""
    import torch
    res = {}
    cases = [(16384 // S, S, 16, 128) for S in (1024, 2048, 4096, 8192, 16384)] + [(8, 1024, 16, 64)]
    for (B, S, H, D) in cases:
        d = inputs.dense(B, S, H, D, seed=3, dout_seed=4).to(dev)
        o, lse = gb.attn_fwd(d.q, d.k, d.v, scale=d.scale, window=(-1, 0))
        dq, dk, dv = torch.empty_like(d.q), torch.empty_like(d.k), torch.empty_like(d.v)
        work = torch.empty(gb.attn_bwd_workspace_size(d.q, d.k, scale=d.scale, window=(-1, 0)),
                           dtype=torch.uint8, device=dev)

        def one():
            gb.attn_fwd(d.q, d.k, d.v, scale=d.scale, window=(-1, 0), out=o, lse=lse)
            gb.attn_bwd(d.dout, d.q, d.k, d.v, o, lse, scale=d.scale, window=(-1, 0), dq=dq, dk=dk,
                        dv=dv, workspace=work)
        for _ in range(3):
            one()
        n = 20
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        s0.record()
        for _ in range(n):
            one()
        s1.record()
        torch.cuda.synchronize()
        ms = s0.elapsed_time(s1) / n
        f_fwd, f_bwd, _ = flops(B, S, H, D, (-1, 0))
        tf = (f_fwd + f_bwd) / (ms * 1e-3) / 1e12
        res["B%d_S%d_H%d_D%d" % (B, S, H, D)] = {"ms": round(ms, 4), "TFLOP/s": round(tf, 1),
                                                 "pct_of_peak": round(100 * tf / peak, 2)}
        del d, o, lse, dq, dk, dv, work
    return res


def _time_steps(one, n, flush=None):
    """Mean ms of ``one()`` over n calls after 3 warm-up calls.  With a flush
    buffer, the buffer is overwritten before every call (outside the timed
    events) so that each call starts with a cold L2."""
    import torch
    for _ in range(3):
        one()
    torch.cuda.synchronize()
    if flush is None:
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s0.record()
        for _ in range(n):
            one()
        s1.record()
        torch.cuda.synchronize()
        return s0.elapsed_time(s1) / n
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(n)]
    for a, b in ev:
        flush.fill_(1.0)
        a.record()
        one()
        b.record()
    torch.cuda.synchronize()
    return sum(a.elapsed_time(b) for a, b in ev) / n


def workload_lines(gb, inputs, dev, peak):
    """fwd+bwd TFLOP/s on the packed THD workload (16 causal sequences of
    U[128, 4096] tokens, 32 query heads over 8 KV heads, D=128), on that
    workload under the emulated context-parallel ring (CP = 4), on a causal
    sliding window (1023, 0) over S=16384, and the S=1024 sweep point with
    the L2 flushed before every step."""
    import torch
    out = {}

    def fwd_bwd(d, window, extra):
        o, lse = gb.attn_fwd(d.q, d.k, d.v, scale=d.scale, window=window, **extra)
        dq, dk, dv = torch.empty_like(d.q), torch.empty_like(d.k), torch.empty_like(d.v)
        work = torch.empty(gb.attn_bwd_workspace_size(d.q, d.k, scale=d.scale, window=window,
                                                      **extra), dtype=torch.uint8, device=dev)

        def fwd():
            gb.attn_fwd(d.q, d.k, d.v, scale=d.scale, window=window, out=o, lse=lse, **extra)

        def step():
            fwd()
            gb.attn_bwd(d.dout, d.q, d.k, d.v, o, lse, scale=d.scale, window=window, dq=dq,
                        dk=dk, dv=dv, workspace=work, **extra)
        return fwd, step

    def line(name, fl_fwd, fl_bwd, ms_fwd, ms_step):
        tf = (fl_fwd + fl_bwd) / (ms_step * 1e-3) / 1e12
        return {"workload": name, "ms": round(ms_step, 4), "TFLOP/s": round(tf, 1),
                "pct_of_peak": round(100 * tf / peak, 2), "fwd_ms": round(ms_fwd, 4),
                "fwd_TFLOP/s": round(fl_fwd / (ms_fwd * 1e-3) / 1e12, 1)}

    d = inputs.varlen().to(dev)
    lens = (d.cu_seqlens_q[1:] - d.cu_seqlens_q[:-1]).tolist()
    nvis = sum(L * (L + 1) // 2 for L in lens) * d.Hq
    extra = dict(cu_seqlens_q=d.cu_seqlens_q, cu_seqlens_kv=d.cu_seqlens_kv,
                 max_seqlen_q=d.Sq, max_seqlen_kv=d.Skv)
    fwd, step = fwd_bwd(d, (-1, 0), extra)
    out["varlen_thd"] = line("bf16 THD causal, %d sequences U[128,4096] (T=%d), Hq=32 Hkv=8 "
                             "D=128" % (len(lens), sum(lens)), 4.0 * 128 * nvis,
                             10.0 * 128 * nvis, _time_steps(fwd, 20), _time_steps(step, 20))
    del fwd, step

    # The same batch under the load-balanced context-parallel split, CP = 4,
    # every rank's ring emulated on this GPU: each sequence padded to a
    # multiple of 2 CP rows, the ring forward (pair attentions merged by LSE)
    # and its backward (pair backward with the merged O and LSE, fp32 sums).
    # The ring plans its calls on the host from cu_seqlens every call.
    from scaled_dot_product_03_gb300 import cp
    cp_size = 4
    pads = [0]
    for L in lens:
        pads.append(pads[-1] + -(-L // (2 * cp_size)) * (2 * cp_size))
    rows = torch.cat([torch.arange(pads[b], pads[b] + L) for b, L in enumerate(lens)]).to(dev)

    def padded(t):
        z = torch.zeros((pads[-1],) + tuple(t.shape[1:]), dtype=t.dtype, device=dev)
        z[rows] = t
        return z
    qp, kp, vp, dop = padded(d.q), padded(d.k), padded(d.v), padded(d.dout)
    pad_d = torch.tensor(pads, dtype=torch.int32, device=dev)

    def cp_fwd():
        return cp.ring_attention_fwd(qp, kp, vp, d.cu_seqlens_q, pad_d, cp_size, causal=True, scale=d.scale)

    def cp_step():
        o_r, l_r = cp_fwd()
        cp.ring_attention_bwd(dop, qp, kp, vp, o_r, l_r, d.cu_seqlens_q, pad_d, cp_size, causal=True,
                              scale=d.scale)
    out["cp_ring_thd"] = line("the THD workload above under CP=4 (sequences padded to multiples of 8 rows, "
                              "T=%d), every rank's ring emulated on one GPU" % pads[-1], 4.0 * 128 * nvis,
                              10.0 * 128 * nvis, _time_steps(cp_fwd, 5), _time_steps(cp_step, 5))
    del d, qp, kp, vp, dop

    B, S, H, D, win = 1, 16384, 16, 128, (1023, 0)
    d = inputs.dense(B, S, H, D, window=win, seed=3, dout_seed=4).to(dev)
    fwd, step = fwd_bwd(d, win, {})
    f_fwd, f_bwd, _ = flops(B, S, H, D, win)
    out["sliding_window"] = line("bf16 window (1023, 0), B=1 S=16384 H=16 D=128", f_fwd, f_bwd,
                                 _time_steps(fwd, 20), _time_steps(step, 20))
    del d, fwd, step

    B, S, H, D = 16, 1024, 16, 128
    d = inputs.dense(B, S, H, D, seed=3, dout_seed=4).to(dev)
    fwd, step = fwd_bwd(d, (-1, 0), {})
    flush = torch.empty(256 * 2**20 // 4, dtype=torch.float32, device=dev)
    f_fwd, f_bwd, _ = flops(B, S, H, D, (-1, 0))
    out["causal_s1024_l2_flushed"] = line(
        "bf16 causal B=16 S=1024 H=16 D=128, 256 MB written before every step", f_fwd, f_bwd,
        _time_steps(fwd, 20, flush), _time_steps(step, 20, flush))
    del d, fwd, step, flush
    return out


def kernel_breakdown(gb, step, n=5):
    """Mean live duration (ms) of each kernel kind over n profiled calls of
    step(), from the library's per-launch timing hook."""
    import torch
    step()
    torch.cuda.synchronize()
    gb.profile_begin(64 * n)
    for _ in range(n):
        step()
    torch.cuda.synchronize()
    per = {}
    for name, ms in gb.profile_read(64 * n):
        per.setdefault(name, []).append(ms)
    return {k: round(sum(v) / n, 4) for k, v in per.items()}


def head_dim_and_mqa_lines(gb, inputs, dev, peak):
    """fwd / fwd+bwd TFLOP/s of: the page-1 workload (fp16, 16 query heads
    over one KV head, packed strided views, S=2048) and causal bf16
    multi-query attention against multi-head at equal flops (B2 S4096 H16
    D128); head dims 32, 96 (padded tensor-core kernels) and 256 (forward
    only) on causal bf16 B4 S4096 H16; the D=64 workload with its per-kernel
    breakdown."""
    import torch
    out = {}

    def measure(name, d, window, bwd=True, breakdown=False):
        o, lse = gb.attn_fwd(d.q, d.k, d.v, scale=d.scale, window=window)
        fwd = lambda: gb.attn_fwd(d.q, d.k, d.v, scale=d.scale, window=window, out=o, lse=lse)
        lens = [d.Sq] * d.B
        nvis = sum(n_visible(L, window) for L in lens) * d.Hq
        f_fwd, f_bwd = 4.0 * d.D * nvis, 10.0 * d.D * nvis
        ms_f = _time_steps(fwd, 20)
        line = {"workload": name, "fwd_ms": round(ms_f, 4),
                "fwd_TFLOP/s": round(f_fwd / (ms_f * 1e-3) / 1e12, 1),
                "fwd_pct_of_peak": round(100 * f_fwd / (ms_f * 1e-3) / 1e12 / peak, 2)}
        step = fwd
        if bwd:
            dq, dk, dv = torch.empty_like(d.q), torch.empty_like(d.k), torch.empty_like(d.v)
            work = torch.empty(max(1, gb.attn_bwd_workspace_size(d.q, d.k, scale=d.scale, window=window)),
                               dtype=torch.uint8, device=dev)

            def step():
                fwd()
                gb.attn_bwd(d.dout, d.q, d.k, d.v, o, lse, scale=d.scale, window=window, dq=dq, dk=dk,
                            dv=dv, workspace=work)
            ms = _time_steps(step, 20)
            tf = (f_fwd + f_bwd) / (ms * 1e-3) / 1e12
            line.update({"ms": round(ms, 4), "TFLOP/s": round(tf, 1), "pct_of_peak": round(100 * tf / peak, 2)})
        if breakdown:
            line["kernels_ms"] = kernel_breakdown(gb, step)
        return line

    d = inputs.page1(scale=0.1, dout_seed=5).to(dev)
    assert d.q.stride() == (1152, 1152, 64, 1)
    out["page1_mqa_fp16_strided"] = measure(
        "fp16 causal S=2048, 16 query heads over 1 KV head, D=64, packed sb(h+2h_g)d views", d, (-1, 0),
        breakdown=True)
    del d
    for hkv in (1, 16):
        d = inputs.dense(2, 4096, 16, 128, Hkv=hkv, seed=3, dout_seed=4).to(dev)
        out["causal_B2_S4096_H16_D128_Hkv%d" % hkv] = measure(
            "bf16 causal B=2 S=4096, 16 query heads over %d KV heads, D=128" % hkv, d, (-1, 0),
            breakdown=(hkv == 1))
        del d
    for D in (32, 96, 256):
        d = inputs.dense(4, 4096, 16, D, seed=3, dout_seed=4 if D != 256 else None).to(dev)
        out["causal_B4_S4096_H16_D%d" % D] = measure(
            "bf16 causal B=4 S=4096 H=16 D=%d%s" % (D, " (forward only)" if D == 256 else
                                                    " (on the %d-wide kernels)" % (64 if D == 32 else 128)),
            d, (-1, 0), bwd=D != 256)
        del d
    d = inputs.dense(8, 1024, 16, 64, seed=3, dout_seed=4).to(dev)
    out["causal_B8_S1024_H16_D64"] = measure("bf16 causal B=8 S=1024 H=16 D=64", d, (-1, 0), breakdown=True)
    del d
    return out


def aux_lines(gb, inputs, dev, peaks):
    """LSE merge (HBM-bound) and fp32 forward+backward, timed on their own."""
    import torch
    out = {}
    B, S, H, D = 4, 4096, 16, 128
    g = torch.Generator().manual_seed(5)
    o1 = torch.randn(B, S, H, D, generator=g).bfloat16().to(dev)
    o2 = torch.randn(B, S, H, D, generator=g).bfloat16().to(dev)
    l1 = torch.randn(B, H, S, generator=g).to(dev)
    l2 = torch.randn(B, H, S, generator=g).to(dev)
    oo, lo = torch.empty_like(o1), torch.empty_like(l1)
    for _ in range(3):
        gb.attn_merge_lse(o1, l1, o2, l2, out=oo, lse_out=lo)
    torch.cuda.synchronize()
    n = 20
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record()
    for _ in range(n):
        gb.attn_merge_lse(o1, l1, o2, l2, out=oo, lse_out=lo)
    e.record()
    torch.cuda.synchronize()
    ms = s.elapsed_time(e) / n
    nbytes = 3 * o1.numel() * 2 + 3 * l1.numel() * 4
    gbs = nbytes / (ms * 1e-3) / 1e9
    out["merge"] = {"workload": "bf16 B=4 S=4096 H=16 D=128", "ms": round(ms, 4),
                    "GB/s": round(gbs, 1), "bound": "hbm", "peak_gbs": peaks["hbm_gbs"],
                    "frac": round(gbs / peaks["hbm_gbs"], 4), "algorithmic_bytes": nbytes}
    # its backward: reads o1, o2, dO, lse1, lse2, dLSE; writes dO1, dO2, dLSE1, dLSE2
    dout_m = torch.randn(B, S, H, D, generator=g).bfloat16().to(dev)
    dl_m = torch.randn(B, H, S, generator=g).to(dev)
    gr = [torch.empty_like(o1), torch.empty_like(l1), torch.empty_like(o2), torch.empty_like(l2)]
    for _ in range(3):
        gb.attn_merge_lse_bwd(o1, l1, o2, l2, dout_m, dl_m, do1=gr[0], dlse1=gr[1], do2=gr[2],
                              dlse2=gr[3])
    torch.cuda.synchronize()
    s.record()
    for _ in range(n):
        gb.attn_merge_lse_bwd(o1, l1, o2, l2, dout_m, dl_m, do1=gr[0], dlse1=gr[1], do2=gr[2],
                              dlse2=gr[3])
    e.record()
    torch.cuda.synchronize()
    ms = s.elapsed_time(e) / n
    nbytes = 5 * o1.numel() * 2 + 5 * l1.numel() * 4
    gbs = nbytes / (ms * 1e-3) / 1e9
    out["merge_bwd"] = {"workload": "bf16 B=4 S=4096 H=16 D=128", "ms": round(ms, 4),
                        "GB/s": round(gbs, 1), "bound": "hbm", "peak_gbs": peaks["hbm_gbs"],
                        "frac": round(gbs / peaks["hbm_gbs"], 4), "algorithmic_bytes": nbytes}
    del dout_m, dl_m, gr
    # the bitwise-reproducible backward (deterministic=True) on the workload
    wp = inputs.dense(B, S, H, D, window=(-1, 0), seed=7).to(dev)
    o, lse = gb.attn_fwd(wp.q, wp.k, wp.v, scale=wp.scale, window=(-1, 0))
    for _ in range(3):
        gb.attn_bwd(wp.dout, wp.q, wp.k, wp.v, o, lse, scale=wp.scale, window=(-1, 0),
                    deterministic=True)
    torch.cuda.synchronize()
    s.record()
    for _ in range(n):
        gb.attn_bwd(wp.dout, wp.q, wp.k, wp.v, o, lse, scale=wp.scale, window=(-1, 0),
                    deterministic=True)
    e.record()
    torch.cuda.synchronize()
    ms = s.elapsed_time(e) / n
    _, f_bwd, _ = flops(B, S, H, D, (-1, 0))
    out["bwd_deterministic"] = {"workload": "bf16 causal bwd B=4 S=4096 H=16 D=128, two kernels",
                                "ms": round(ms, 4),
                                "TFLOP/s": round(f_bwd / (ms * 1e-3) / 1e12, 1)}
    del wp, o, lse
    prob = inputs.page3().to(dev)
    for _ in range(3):
        o, lse = gb.attn_fwd(prob.q, prob.k, prob.v, scale=prob.scale)
        gb.attn_bwd(prob.dout, prob.q, prob.k, prob.v, o, lse, scale=prob.scale)
    torch.cuda.synchronize()
    s.record()
    for _ in range(n):
        o, lse = gb.attn_fwd(prob.q, prob.k, prob.v, scale=prob.scale)
        gb.attn_bwd(prob.dout, prob.q, prob.k, prob.v, o, lse, scale=prob.scale)
    e.record()
    torch.cuda.synchronize()
    ms = s.elapsed_time(e) / n
    f_fwd, f_bwd, _ = flops(1, 512, 4, 64, (-1, -1))
    # FFMA peak derived from the unit counts: SMs x 128 fp32 lanes x 2 flops
    # x the maximum SM clock of MEASURED_PEAKS.json
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    ffma_peak = sms * 128 * 2 * peaks.get("sm_max_mhz", 2070.0) * 1e6 / 1e12
    tf32 = (f_fwd + f_bwd) / (ms * 1e-3) / 1e12
    out["fp32_page3"] = {"workload": "fp32 fwd+bwd B=1 S=512 H=4 D=64 non-causal",
                         "ms": round(ms, 4), "TFLOP/s": round(tf32, 3),
                         "bound": "alu", "ffma_peak_tflops": round(ffma_peak, 1),
                         "ffma_peak_source": "derived: %d SMs x 128 lanes x 2 flops x max SM clock" % sms,
                         "frac": round(tf32 / ffma_peak, 4),
                         "kernels_ms": kernel_breakdown(gb, lambda: gb.attn_bwd(
                             prob.dout, prob.q, prob.k, prob.v, *gb.attn_fwd(prob.q, prob.k, prob.v,
                                                                             scale=prob.scale),
                             scale=prob.scale))}
    return out


def cpu_sample_units(heads=2):
    return dict(B=1, S=WORKLOAD["S"], H=heads, D=WORKLOAD["D"], window=WORKLOAD["window"])


def run_oracle_sample(seed=0, heads=2):
    """Oracle fwd + bwd on the bounded sample (2 heads of one batch item of
    the workload, all rows).  Returns (seconds, flops)."""
    import oracle
    from scaled_dot_product_03_gb300 import inputs
    sm = cpu_sample_units(heads)
    prob = inputs.dense(sm["B"], sm["S"], sm["H"], sm["D"], window=sm["window"], seed=seed)
    f64 = lambda t: t.to("cpu").double().contiguous().reshape(-1, t.shape[2], t.shape[3]).numpy()
    q, k, v, do = f64(prob.q), f64(prob.k), f64(prob.v), f64(prob.dout)
    cu = oracle.dense_cu(sm["B"], sm["S"])
    t0 = time.perf_counter()
    oracle.attn_fwd(q, k, v, cu, cu, prob.scale, prob.window)
    oracle.attn_bwd(q, k, v, do, cu, cu, prob.scale, prob.window)
    dt = time.perf_counter() - t0
    f_fwd, f_bwd, _ = flops(sm["B"], sm["S"], sm["H"], sm["D"], sm["window"])
    return dt, f_fwd + f_bwd


def cpu_baseline(args):
    import oracle
    oracle.build()
    dt, fl = run_oracle_sample(heads=6)
    return {"value": round(fl / dt / 1e12, 6), "unit": "TFLOP/s", "cores": oracle.num_threads(),
            "kind": "oracle",
            "sample": "float64 oracle fwd+bwd on 6 heads x 4096 rows of one batch item "
                      "(causal, D=128); %.1f s" % dt}


def run_reference(args):
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return None
    import oracle
    oracle.build()
    for _ in range(args.warmup):
        run_oracle_sample()
    times, fl = [], 0
    for i in range(args.steps):
        dt, fl = run_oracle_sample()
        times.append(dt)
    total = sum(times)
    value = fl * args.steps / total / 1e12
    B, S, H, D, win = (WORKLOAD[k] for k in ("B", "S", "H", "D", "window"))
    sm = cpu_sample_units()
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * total / args.steps, 2), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "causal self-attention fwd+bwd, bf16, B=%d S=%d H=%d D=%d" % (
            B, S, H, D), "B": B, "S": S, "H": H, "D": D, "window": list(win)},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s",
                         "cores": oracle.num_threads(), "kind": "oracle",
                         "sample": "each step: float64 oracle fwd+bwd on %d heads x %d rows of "
                                   "one batch item of the workload" % (sm["H"], sm["S"])},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


# Small workloads, one per kernel, for profiler captures (one kernel per
# capture, a few launches): name -> (description, builder).  Each builder
# returns a callable running the case once; the captured kernel is named in
# the profile summaries.
def _profile_cases():
    import torch
    import scaled_dot_product_03_gb300 as gb
    from scaled_dot_product_03_gb300 import inputs
    dev = torch.device("cuda", 0)

    def fwd_bwd(prob, window=(-1, 0), det=False, extra=None):
        d = prob.to(dev)
        extra = extra or {}
        o, lse = gb.attn_fwd(d.q, d.k, d.v, scale=d.scale, window=window, **extra)
        dq, dk, dv = torch.empty_like(d.q), torch.empty_like(d.k), torch.empty_like(d.v)
        work = torch.empty(max(1, gb.attn_bwd_workspace_size(d.q, d.k, scale=d.scale, window=window,
                                                             deterministic=det, **extra)),
                           dtype=torch.uint8, device=dev)

        def run():
            gb.attn_fwd(d.q, d.k, d.v, scale=d.scale, window=window, out=o, lse=lse, **extra)
            if d.dout is not None:
                gb.attn_bwd(d.dout, d.q, d.k, d.v, o, lse, scale=d.scale, window=window, dq=dq, dk=dk, dv=dv,
                            workspace=work, deterministic=det, **extra)
        return run

    def merge():
        g = torch.Generator().manual_seed(5)
        B, S, H, D = 4, 4096, 16, 128
        o1, o2, do = (torch.randn(B, S, H, D, generator=g).bfloat16().to(dev) for _ in range(3))
        l1, l2, dl = (torch.randn(B, H, S, generator=g).to(dev) for _ in range(3))
        oo, lo = torch.empty_like(o1), torch.empty_like(l1)
        gr = [torch.empty_like(o1), torch.empty_like(l1), torch.empty_like(o2), torch.empty_like(l2)]

        def run():
            gb.attn_merge_lse(o1, l1, o2, l2, out=oo, lse_out=lo)
            gb.attn_merge_lse_bwd(o1, l1, o2, l2, do, dl, do1=gr[0], dlse1=gr[1], do2=gr[2], dlse2=gr[3])
        return run

    def partition():
        from scaled_dot_product_03_gb300 import _lib
        import ctypes
        lens = [262144] * 64
        pads = [0]
        for L in lens:
            pads.append(pads[-1] + L)
        pad = torch.tensor(pads, dtype=torch.int32, device=dev)
        out = torch.empty(pads[-1] // 4, dtype=torch.int32, device=dev)
        lib = _lib.load()

        def run():
            _lib.check(lib.attn_thd_partitioned_indices(pad.data_ptr(), len(lens), pads[-1], 4, 1, out.data_ptr(),
                                                         ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)))
        return run

    return {
        "causal_bf16_b2_s8192_h8_d128": ("tc_fwd<bf16,128>, single-pass backward, preprocess, dq convert",
                                         lambda: fwd_bwd(inputs.dense(2, 8192, 8, 128, seed=3, dout_seed=4))),
        "causal_bf16_b2_s8192_h8_d128_det": ("the two-kernel backward (tc_bwd_dkdv, tc_bwd_dq)",
                                             lambda: fwd_bwd(inputs.dense(2, 8192, 8, 128, seed=3, dout_seed=4),
                                                             det=True)),
        "causal_bf16_b8_s1024_h16_d64": ("tc_fwd<bf16,64>, single-pass backward at D=64",
                                         lambda: fwd_bwd(inputs.dense(8, 1024, 16, 64, seed=3, dout_seed=4))),
        "causal_bf16_b2_s4096_h16_d128_mqa": ("query-head split and the dK/dV reduce (one KV head)",
                                              lambda: fwd_bwd(inputs.dense(2, 4096, 16, 128, Hkv=1, seed=3,
                                                                           dout_seed=4))),
        "causal_fp16_b1_s2048_h16_hkv1_d64_page1": ("the page-1 multi-query workload: single pass at D=64 "
                                                    "with 16 query-head splits, dK/dV reduce",
                                                    lambda: fwd_bwd(inputs.page1(scale=0.1, dout_seed=5))),
        "causal_bf16_b1_s8192_h8_d256": ("tc_fwd<bf16,256> (forward only)",
                                         lambda: fwd_bwd(inputs.dense(1, 8192, 8, 256, seed=3, dout_seed=None))),
        "fp32_causal_b4_s2048_h16_d64": ("FFMA forward, dq and dk/dv kernels",
                                         lambda: fwd_bwd(inputs.dense(4, 2048, 16, 64, dtype=torch.float32, seed=3,
                                                                      dout_seed=4))),
        "merge_bf16_b4_s4096_h16_d128": ("LSE merge and its backward", merge),
        "thd_partition_64x262144_cp4": ("THD context-parallel partition (rank 1 of 4)", partition),
    }


def run_profile_case(name, repeats):
    """Runs one profiling workload `repeats` times (no timing, no output but
    a line naming the case); for profiler captures of one kernel."""
    import torch
    from scaled_dot_product_03_gb300 import build as libbuild
    import scaled_dot_product_03_gb300 as gb
    libbuild.build()
    cases = _profile_cases()
    if name not in cases:
        raise SystemExit("unknown profile case %r (known: %s)" % (name, ", ".join(sorted(cases))))
    desc, make = cases[name]
    run = make()
    for _ in range(repeats):
        run()
    torch.cuda.synchronize()
    gb.check_device_error()
    print("profile case %s (%s): %d runs" % (name, desc, repeats))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-aux", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end leg")
    ap.add_argument("--shape", default=None,
                    help="B,S,H,D of the causal workload (default: the headline workload)")
    ap.add_argument("--profile-case", default=None,
                    help="run one small per-kernel workload for a profiler capture and exit")
    ap.add_argument("--repeats", type=int, default=3, help="runs of --profile-case")
    args = ap.parse_args()
    if args.profile_case:
        run_profile_case(args.profile_case, args.repeats)
        return
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    line = run_reference(args) if args.impl == "reference" else run_ours(args)
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
