#!/usr/bin/env python3
"""Benchmark of the packed width-4 causal depthwise convolution + SiLU on GB300.

One step = one pass of the whole hot path over one batch of synthetic input:
the forward (y from x) and the backward (dx, dweight, dbias from x and dy; two
launches, the second programmatically dependent). The default workload is the
linear-attention short-conv shape S = 65536 packed tokens, C = 6144 channels
(q|k|v, 3 x 2048), uniform document lengths in [1, 8192] with 3 empty
documents, FP32 weight and bias, BF16 x / dy, SiLU' at the BF16-rounded
preactivation.

Printed JSON (one line, rank 0):
  value        fwd+bwd achieved HBM GB/s = compulsory bytes (fwd: read x, write y;
               bwd: read x and dy, write dx, plus the partial rows written and
               read) / device time, inputs resident in HBM; inputs (805 MB each)
               exceed the 129 MB L2, so no flush is needed between steps.
  e2e          the same metric through the public API with pinned host buffers,
               host->device copies of the step's inputs and device->host copies
               of its outputs inside the timed region.
  roofline     backward call (its main kernel dominates the step) against the
               measured HBM copy bandwidth, and against the library's own
               streaming kernel moving the same bytes (ceiling_gbs).
  ceiling      vcd_stream_copy (include/vcd_stream.h) timed on the workload's
               own buffers: the forward's traffic (read x, write y) and the
               backward's (read x and dy, write dx) with no arithmetic.
  routes       every workload and SiLU' policy the operation is specified on,
               forward and backward timed the same way, and the exactness-guarded
               routes beside them (--no-sweep skips it).
  cpu_baseline the FP64 oracle (test infrastructure, single-threaded C) timed on
               a bounded slice of the same workload, and the same slice split
               by channels over every host core.

Multi-GPU (torchrun, N > 1): every rank runs an independent replica on its own
GPU (the operation has no exchange step); value sums the ranks' bytes over the
slowest rank's time.
"""
import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

METRIC = "fwd/bwd achieved HBM GB/s (% of GB300 peak) and Mtokens/s at S=65536, C=6144"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0

# ncu DRAM traffic (read + write bytes per launch) of the backward main kernel on
# the default workload, keyed by the SHA-256 of the kernel sources it was taken
# on (comments and blank space stripped, so only code changes count); a changed
# kernel reports traffic null until it is profiled again. Taken on the same
# workload at S = 16384 (a capture small enough for ncu's replay) and scaled by
# the 4x units of S = 65536 (traffic is proportional to tokens).
NCU_TRAFFIC = {"23535773b6930b8c": 4 * 579.377408e6}
KERNEL_SOURCES = ["varlen_causal_depthwise_gb300/csrc/vcd_bwd.cu",
                  "varlen_causal_depthwise_gb300/csrc/vcd_device.cuh",
                  "varlen_causal_depthwise_gb300/csrc/vcd_dfloat.cuh",
                  "varlen_causal_depthwise_gb300/csrc/vcd_kernels.h",
                  "varlen_causal_depthwise_gb300/csrc/vcd_plan.h"]


def strip_comments(src):
    """C/C++ source without comments and with blank space collapsed (string and
    character literals kept as they are)."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c in "\"'":
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            i = src.find("\n", i)
            i = n if i < 0 else i
        elif src.startswith("/*", i):
            i = src.find("*/", i + 2)
            i = n if i < 0 else i + 2
            out.append(" ")
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def kernel_sha():
    h = hashlib.sha256()
    for p in KERNEL_SOURCES:
        with open(os.path.join(ROOT, p), encoding="utf-8") as f:
            h.update(strip_comments(f.read()).encode())
    return h.hexdigest()[:16]


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.window = None    # (t0, t1) wall-clock seconds of the timed region

    def mark(self, t0, t1):
        self.window = (t0, t1)

    def __enter__(self):
        self.nvml = NvmlSampler(self.gpu).__enter__()
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.nvml.__exit__()
        self.out = ""
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in (self.out or "").splitlines():
            f = [v.strip() for v in line.split(",")]
            if len(f) < 10:
                continue
            try:
                ts = time.mktime(time.strptime(f[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                ts += float("0." + f[0].split(".")[1]) if "." in f[0] else 0.0
                clk, cmax = float(f[2]), float(f[3])
            except (ValueError, IndexError):
                continue
            if self.window and not (self.window[0] - 0.25 <= ts <= self.window[1] + 0.25):
                continue
            sm.append(clk)
            mx.append(cmax)
            for n, v in zip(names, f[6:10]):
                if v.lower() == "active":
                    reasons.add(n)
        n_smi = len(sm)
        if self.window:
            nsm, nreasons = self.nvml.in_window(*self.window)
            sm += nsm
            reasons |= nreasons
            if self.nvml.max_mhz:
                mx.append(self.nvml.max_mhz)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm), "samples_nvidia_smi": n_smi,
                "samples_nvml": len(sm) - n_smi}


class NvmlSampler:
    """SM clock and clock-event reasons read through NVML (ctypes, read-only
    queries) every ~2 ms on a host thread, so that a timed region of a few
    milliseconds still gets several samples. Silently empty where NVML is
    missing; the nvidia-smi sampler runs beside it."""
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown"}

    def __init__(self, gpu_index, period_s=0.002):
        self.gpu, self.period = gpu_index, period_s
        self.samples, self.max_mhz = [], None
        self._stop = None

    def __enter__(self):
        import ctypes
        import threading

        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                return self
            h = ctypes.c_void_p()
            if nv.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(self.gpu), ctypes.byref(h)) != 0:
                return self
            reasons = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                getattr(nv, "nvmlDeviceGetCurrentClocksThrottleReasons")
        except (OSError, AttributeError):
            return self
        mx = ctypes.c_uint()
        if nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:
            self.max_mhz = float(mx.value)
        self._nv, self._stop = nv, threading.Event()

        def poll():
            clk, rs = ctypes.c_uint(), ctypes.c_ulonglong()
            while not self._stop.is_set():
                if nv.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk)) == 0 and \
                        reasons(h, ctypes.byref(rs)) == 0:
                    self.samples.append((time.time(), float(clk.value), int(rs.value)))
                self._stop.wait(self.period)

        self._thread = threading.Thread(target=poll, daemon=True)
        self._thread.start()
        return self

    def __exit__(self, *exc):
        if self._stop is not None:
            self._stop.set()
            self._thread.join(timeout=5)
            self._nv.nvmlShutdown()

    def in_window(self, t0, t1):
        sm, reasons = [], set()
        for ts, clk, rs in self.samples:
            if t0 <= ts <= t1:
                sm.append(clk)
                reasons.update(n for bit, n in self.REASONS.items() if rs & bit)
        return sm, reasons


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def reduce_max(value, device):
    """Largest `value` over all ranks (the slowest rank sets the job's time)."""
    import torch.distributed as dist

    if not dist.is_available() or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def vcd_call_bytes(w, policy):
    """Partial-row bytes the backward call writes (and its reduce reads back):
    the exact workspace need of this call's launch shape."""
    import varlen_causal_depthwise_gb300 as vcd

    return vcd.conv1d_bwd_call_workspace_size(w.S, w.C, w.num_docs, policy, w.bias is not None)


def compulsory_bytes(S, C, partial_bytes):
    E = S * C
    fwd = 4 * E
    bwd = 6 * E + 2 * partial_bytes
    return fwd, bwd


def run_ours(args):
    import torch.distributed as dist

    import varlen_causal_depthwise_gb300 as vcd
    from varlen_causal_depthwise_gb300 import synth

    ws, rank, local = dist_env()
    if ws > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    recipe = synth.RECIPES[args.config]
    w = synth.make(args.config, device=dev, S=args.S)
    S, C = w.S, w.C
    policy = args.policy or recipe.policies[0]
    nws = vcd.conv1d_bwd_workspace_size(S, C)
    wsp = torch.empty(nws, dtype=torch.uint8, device=dev)
    y = torch.empty_like(w.x)
    dx = torch.empty_like(w.x)
    dW = torch.empty(C, 4, dtype=w.weight.dtype, device=dev)
    dB = None if w.bias is None else torch.empty(C, dtype=w.bias.dtype, device=dev)
    stream = torch.cuda.current_stream(dev)

    if args.exact:
        wsp = torch.empty(vcd.conv1d_bwd_exact_workspace_size(S, C), dtype=torch.uint8, device=dev)

    def fwd():
        if args.exact:
            vcd.conv1d_fwd_exact(w.x, w.weight, w.cu_seqlens, w.bias, y=y, stream=stream)
        else:
            vcd.conv1d_fwd(w.x, w.weight, w.cu_seqlens, w.bias, y=y, stream=stream)

    def bwd():
        entry = vcd.conv1d_bwd_exact if args.exact else vcd.conv1d_bwd
        entry(w.x, w.dy, w.weight, w.cu_seqlens, w.bias, policy, dx=dx, dweight=dW, dbias=dB,
              workspace=wsp, stream=stream)

    for _ in range(args.warmup):
        fwd()
        bwd()
    torch.cuda.synchronize(dev)

    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    with ClockSampler(local) as clk:
        time.sleep(0.5)                 # let the sampler start
        if ws > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)
        wall0 = time.time()
        t_start = torch.cuda.Event(enable_timing=True)
        t_end = torch.cuda.Event(enable_timing=True)
        t_start.record(stream)
        for i in range(K):
            ev[i][0].record(stream)
            fwd()
            ev[i][1].record(stream)
            bwd()
            ev[i][2].record(stream)
        t_end.record(stream)
        torch.cuda.synchronize(dev)
        clk.mark(wall0, time.time())
        if ws > 1:
            dist.barrier()
    total_ms = t_start.elapsed_time(t_end)
    fwd_ms = [e[0].elapsed_time(e[1]) for e in ev]
    bwd_ms = [e[1].elapsed_time(e[2]) for e in ev]
    total_ms = reduce_max(total_ms, dev)
    extra = {"ceiling": ceiling_leg(w, y, dx, stream, 20)}
    if not args.no_sweep and rank == 0:
        extra["routes"] = sweep_leg(dev, 20, measured_peak()[0])

    # ---- end to end: pinned host buffers through the public API ----
    if args.no_e2e:
        return finish(args, w, S, C, policy, nws, K, total_ms, fwd_ms, bwd_ms, clk, None, ws, rank,
                      extra)
    e2e = e2e_pipelined(w, policy, K, dev, vcd)
    e2e = (reduce_max(e2e[0], dev),) + e2e[1:]
    return finish(args, w, S, C, policy, nws, K, total_ms, fwd_ms, bwd_ms, clk, e2e, ws, rank,
                  extra)


def time_events(fn, iters, stream, flush=None):
    """Median device time (us) of fn() over iters runs, CUDA events on `stream`;
    flush() (not timed) runs before each when given."""
    out = []
    for _ in range(iters):
        if flush is not None:
            flush()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        out.append((a, b))
    torch.cuda.synchronize()
    return 1e3 * statistics.median(a.elapsed_time(b) for a, b in out)


def ceiling_leg(w, y, dx, stream, iters):
    """The library's streaming kernel over the workload's own buffers: the
    forward's traffic (x -> y) and the backward's (x, dy -> dx), each at the
    best of 1, 2 and 4 CTAs of 512 threads per SM."""
    from varlen_causal_depthwise_gb300 import binding

    E = w.x.numel()
    res = {}
    for leg, args, nbytes in (("fwd_mix", (w.x, y, None), 4 * E),
                              ("bwd_mix", (w.x, dx, w.dy), 6 * E)):
        best = None
        for bps in (1, 2, 4):
            fn = lambda: binding.stream_copy(args[0], args[1], args[2], bps, stream)
            for _ in range(3):
                fn()
            us = time_events(fn, iters, stream)
            if best is None or us < best[0]:
                best = (us, bps)
        res[leg] = {"us_median": round(best[0], 2), "blocks_per_sm": best[1], "bytes": nbytes,
                    "gbs": round(nbytes / (best[0] * 1e-6) / 1e9, 1)}
    return res


def sweep_leg(dev, iters, peak):
    """Forward and backward of every specified workload and policy, timed on
    their own inputs; workloads whose tensors fit in L2 several times over are
    timed with L2 flushed before each call."""
    import varlen_causal_depthwise_gb300 as vcd
    from varlen_causal_depthwise_gb300 import synth

    stream = torch.cuda.current_stream(dev)
    scrub = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    flush = lambda: scrub.fill_(1)
    out = {}
    for name, recipe in synth.RECIPES.items():
        w = synth.make(name, device=dev)
        S, C = w.S, w.C
        small = 2 * S * C < 4 * (128 << 20)
        y = torch.empty_like(w.x)
        dx = torch.empty_like(w.x)
        ws = torch.empty(vcd.conv1d_bwd_workspace_size(S, C), dtype=torch.uint8, device=dev)
        dW = torch.empty(C, 4, dtype=w.weight.dtype, device=dev)
        dB = None if w.bias is None else torch.empty(C, dtype=w.bias.dtype, device=dev)
        fwd = lambda: vcd.conv1d_fwd(w.x, w.weight, w.cu_seqlens, w.bias, y=y, stream=stream)
        fwd_x = lambda: vcd.conv1d_fwd_exact(w.x, w.weight, w.cu_seqlens, w.bias, y=y,
                                             stream=stream)
        for _ in range(3):
            fwd()
            fwd_x()
        f_us = time_events(fwd, iters, stream, flush if small else None)
        fx_us = time_events(fwd_x, iters, stream, flush if small else None)
        fwd_b = 4 * S * C
        wsx = torch.empty(vcd.conv1d_bwd_exact_workspace_size(S, C), dtype=torch.uint8, device=dev)
        for pol in recipe.policies:
            bwd = lambda: vcd.conv1d_bwd(w.x, w.dy, w.weight, w.cu_seqlens, w.bias, pol, dx=dx,
                                         dweight=dW, dbias=dB, workspace=ws, stream=stream)
            bwd_x = lambda: vcd.conv1d_bwd_exact(w.x, w.dy, w.weight, w.cu_seqlens, w.bias, pol,
                                                 dx=dx, dweight=dW, dbias=dB, workspace=wsx,
                                                 stream=stream)
            for _ in range(3):
                bwd()
                bwd_x()
            b_us = time_events(bwd, iters, stream, flush if small else None)
            bx_us = time_events(bwd_x, iters, stream, flush if small else None)
            bwd_b = compulsory_bytes(S, C, vcd_call_bytes(w, pol))[1]
            row = {"S": S, "C": C, "docs": w.num_docs, "policy": pol,
                   "l2": "flushed before each call" if small else "inputs larger than L2"}
            # the exactness-guarded routes (conv1d_fwd_exact / conv1d_bwd_exact) moving
            # the same compulsory bytes: their cost against the plain ones
            for d, us, nb in (("fwd", f_us, fwd_b), ("bwd", b_us, bwd_b),
                              ("fwd_exact", fx_us, fwd_b), ("bwd_exact", bx_us, bwd_b)):
                gbs = nb / (us * 1e-6) / 1e9
                row[d] = {"us_median": round(us, 2), "gbs": round(gbs, 1),
                          "frac_of_measured": round(gbs / peak, 4),
                          "frac_of_8tbs_nominal": round(gbs / NOMINAL_HBM_GBS, 4),
                          "mtokens_per_s": round(S / (us * 1e-6) / 1e6, 2)}
            out[f"{name}/{pol}"] = row
        del w, y, dx, ws, wsx
        torch.cuda.empty_cache()
    return out


def e2e_pipelined(w, policy, K, dev, vcd):
    """Steps through the public API with host buffers: every step copies its
    inputs (x, dy, weight, bias, cu_seqlens) from pinned host memory, runs the
    forward and backward, and copies y, dx, dweight, dbias back to pinned host
    memory. Three streams and two buffer sets let step i's compute overlap the
    copy-in of step i+1 and the copy-out of step i-1; each step's own copies
    are all inside the timed region. Returns (ms per step, H2D bytes, D2H bytes)."""
    S, C = w.S, w.C
    Ke = max(4, min(K, 12))
    h_in = [[t.cpu().pin_memory() for t in (w.x, w.dy)] for _ in range(2)]
    h_par = [t.cpu().pin_memory() for t in (w.weight, w.bias, w.cu_seqlens) if t is not None]
    d_in = [[torch.empty_like(w.x), torch.empty_like(w.dy)] for _ in range(2)]
    d_par = [[torch.empty_like(t) for t in (w.weight, w.bias, w.cu_seqlens) if t is not None]
             for _ in range(2)]
    outs = [[torch.empty_like(w.x), torch.empty_like(w.x), torch.empty(C, 4, dtype=w.weight.dtype, device=dev)]
            + ([torch.empty(C, dtype=w.bias.dtype, device=dev)] if w.bias is not None else [])
            for _ in range(2)]
    h_out = [[torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in o] for o in outs]
    wsp = [torch.empty(vcd.conv1d_bwd_workspace_size(S, C), dtype=torch.uint8, device=dev)
           for _ in range(2)]
    s_in, s_cmp, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = lambda: torch.cuda.Event()
    in_done, cmp_done, out_done = [ev(), ev()], [ev(), ev()], [ev(), ev()]
    h2d = sum(t.numel() * t.element_size() for t in h_in[0] + h_par)
    d2h = sum(t.numel() * t.element_size() for t in h_out[0])

    def step(i):
        b = i % 2
        with torch.cuda.stream(s_in):
            if i >= 2:
                s_in.wait_event(cmp_done[b])          # step i-2 finished reading set b
            for h, d in zip(h_in[b] + h_par, d_in[b] + d_par[b]):
                d.copy_(h, non_blocking=True)
            in_done[b].record(s_in)
        with torch.cuda.stream(s_cmp):
            s_cmp.wait_event(in_done[b])
            if i >= 2:
                s_cmp.wait_event(out_done[b])         # step i-2's results are out
            x, dy = d_in[b]
            par = d_par[b]
            weight, cu = par[0], par[-1]
            bias = par[1] if w.bias is not None else None
            y, dx, dW = outs[b][:3]
            dB = outs[b][3] if w.bias is not None else None
            vcd.conv1d_fwd(x, weight, cu, bias, y=y, stream=s_cmp)
            vcd.conv1d_bwd(x, dy, weight, cu, bias, policy, dx=dx, dweight=dW, dbias=dB,
                           workspace=wsp[b], stream=s_cmp)
            cmp_done[b].record(s_cmp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(cmp_done[b])
            for d, h in zip(outs[b], h_out[b]):
                h.copy_(d, non_blocking=True)
            out_done[b].record(s_out)

    for i in range(2):
        step(i)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    for i in range(Ke):
        step(i)
    s_out.wait_event(out_done[(Ke - 1) % 2])
    e1.record(s_out)
    torch.cuda.synchronize(dev)
    return e0.elapsed_time(e1) / Ke, h2d, d2h


def finish(args, w, S, C, policy, nws, K, total_ms, fwd_ms, bwd_ms, clk, e2e, ws, rank, extra):
    import torch.distributed as dist

    # the partial rows this call writes and reads back (the workspace size
    # query is the maximum over routes and launch shapes)
    fwd_b, bwd_b = compulsory_bytes(S, C, vcd_call_bytes(w, policy))
    step_b = fwd_b + bwd_b
    ms_step = total_ms / K
    peak, peak_kind = measured_peak()
    fwd_us = 1e3 * statistics.median(fwd_ms)
    bwd_us = 1e3 * statistics.median(bwd_ms)
    bwd_mean_us = 1e3 * statistics.mean(bwd_ms)
    clocks = clk.summary()

    ceil = extra["ceiling"]

    def direction(nbytes, us, mix):
        gbs = nbytes / (us * 1e-6) / 1e9
        return {"us_median": round(us, 2), "gbs": round(gbs, 1),
                "frac_of_measured": round(gbs / peak, 4),
                "frac_of_own_ceiling": round(gbs / ceil[mix]["gbs"], 4),
                "frac_of_8tbs_nominal": round(gbs / NOMINAL_HBM_GBS, 4),
                "mtokens_per_s": round(S / (us * 1e-6) / 1e6, 2),
                "bytes": nbytes}

    value = ws * step_b / (ms_step * 1e-3) / 1e9
    sha = kernel_sha()
    tr = NCU_TRAFFIC.get(sha)
    bwd_achieved = bwd_b / (bwd_mean_us * 1e-6) / 1e9
    out = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "GB/s",
        "n_gpus": ws,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": f"{args.config}: S={S}, C={C}, {w.num_docs} docs, "
                               f"weight {str(w.weight.dtype)[6:]}, "
                               f"bias {'none' if w.bias is None else str(w.bias.dtype)[6:]}, "
                               f"SiLU' policy {policy}, BF16 x/dy/y/dx"
                               + (", exactness-guarded routes" if args.exact else ""),
                   "S": S, "C": C, "num_docs": w.num_docs, "policy": policy,
                   "parallelism": f"replicas x{ws}",
                   "l2": "inputs larger than L2 (no flush needed)"},
        "detail": {"fwd": direction(fwd_b, fwd_us, "fwd_mix"),
                   "bwd": direction(bwd_b, bwd_us, "bwd_mix"),
                   "step": {"gbs": round(step_b / (ms_step * 1e-3) / 1e9, 1),
                            "mtokens_per_s": round(S / (ms_step * 1e-3) / 1e6, 2),
                            "frac_of_measured": round(step_b / (ms_step * 1e-3) / 1e9 / peak, 4)}},
        "roofline": {"kernel": "conv1d_bwd (main + dependent reduce)", "bound": "hbm",
                     "achieved": round(bwd_achieved, 1), "peak": peak,
                     "peak_kind": peak_kind, "unit": "GB/s",
                     "frac": round(bwd_achieved / peak, 4),
                     "ceiling_gbs": ceil["bwd_mix"]["gbs"],
                     "frac_of_ceiling": round(bwd_achieved / ceil["bwd_mix"]["gbs"], 4),
                     "frac_of_8tbs_nominal": round(bwd_achieved / NOMINAL_HBM_GBS, 4),
                     "traffic": tr, "algorithmic_bytes": bwd_b},
        "ceiling": ceil,
        "e2e": None if e2e is None else {
            "value": round(ws * step_b / (e2e[0] * 1e-3) / 1e9, 1), "unit": "GB/s",
            "ms_per_step": round(e2e[0], 3), "h2d_bytes_per_step": e2e[1],
            "d2h_bytes_per_step": e2e[2]},
        "gpu_launches": (4 if args.exact else 3) * K,
        **({"routes": extra["routes"]} if "routes" in extra else {}),
        "clocks": clocks,
        "kernel_sha": sha,
    }
    if rank == 0 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(w, policy, args.cpu_tokens)
    if ws > 1:
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(out), flush=True)


def oracle_slice(w, tokens):
    """The first `tokens` tokens of the workload as a CPU problem of its own
    (documents cut at the slice end)."""
    import numpy as np

    from varlen_causal_depthwise_gb300 import synth

    n = min(tokens, w.S)
    lens, tot = [], 0
    for L in w.lengths:
        if tot >= n:
            break
        take = min(L, n - tot)
        lens.append(take)
        tot += take
    cu = synth.cu_from_lengths(lens)
    x = w.x[:n].cpu()
    dy = w.dy[:n].cpu()
    return x, dy, w.weight.cpu(), None if w.bias is None else w.bias.cpu(), cu, n, np


def oracle_channel_sharded(x, dy, W, b, cu, policy, nthreads):
    """The oracle, as it is, on channel slices in nthreads host threads (its
    C calls release the interpreter lock; channels are independent, so the
    values are those of one call over all channels)."""
    import concurrent.futures

    import oracle

    C = x.shape[1]
    bounds = [C * i // nthreads for i in range(nthreads + 1)]

    def job(i):
        c0, c1 = bounds[i], bounds[i + 1]
        if c1 <= c0:
            return
        xs, gs = x[:, c0:c1].contiguous(), dy[:, c0:c1].contiguous()
        bs = None if b is None else b[c0:c1]
        oracle.fwd(xs, W[c0:c1], cu, bs)
        oracle.bwd(xs, gs, W[c0:c1], cu, bs, policy)

    oracle.load()
    with concurrent.futures.ThreadPoolExecutor(nthreads) as ex:
        list(ex.map(job, range(nthreads)))


def cpu_baseline(w, policy, tokens):
    import oracle

    x, dy, W, b, cu, n, _ = oracle_slice(w, tokens)
    t0 = time.perf_counter()
    oracle.fwd(x, W, cu, b)
    oracle.bwd(x, dy, W, cu, b, policy)
    dt = time.perf_counter() - t0
    fwd_b, bwd_b = compulsory_bytes(n, w.C, 0)
    nproc = os.cpu_count() or 1
    t0 = time.perf_counter()
    oracle_channel_sharded(x, dy, W, b, cu, policy, nproc)
    dt_all = time.perf_counter() - t0
    return {"value": round((fwd_b + bwd_b) / dt / 1e9, 5), "unit": "GB/s", "cores": 1,
            "kind": "oracle", "seconds": round(dt, 2),
            "mtokens_per_s": round(n / dt / 1e6, 6), "host_nproc": nproc,
            "sample": f"first {n} tokens x all {w.C} channels of the same workload, "
                      f"fwd + bwd ({policy}), single-threaded FP64 C",
            "all_cores": {"value": round((fwd_b + bwd_b) / dt_all / 1e9, 5), "unit": "GB/s",
                          "cores": nproc, "seconds": round(dt_all, 2),
                          "mtokens_per_s": round(n / dt_all / 1e6, 6),
                          "sample": f"the same slice split by channels over {nproc} threads"}}


def ref_tokens(args, C):
    """Tokens per step of the reference arm: --ref-tokens, else 96 tokens cut
    down (to 16 at least) so that --steps steps of the single-threaded FP64
    oracle take about a minute (about 2.7 ms per token at C = 6144, in
    proportion to C)."""
    if args.ref_tokens is not None:
        return args.ref_tokens
    per_token_s = 2.7e-3 * C / 6144
    return int(max(16, min(96, 60.0 / (max(args.steps, 1) * per_token_s))))


def run_reference(args):
    ws, rank, local = dist_env()
    if rank != 0:
        return
    from varlen_causal_depthwise_gb300 import synth
    import oracle

    recipe = synth.RECIPES[args.config]
    policy = recipe.policies[0]
    # inputs drawn on the GPU when there is one (faster; the oracle still runs on
    # the host cores), else on the CPU
    w = synth.make(args.config, device="cuda" if torch.cuda.is_available() else "cpu")
    x, dy, W, b, cu, n, _ = oracle_slice(w, ref_tokens(args, w.C))
    del w.x, w.dy
    for _ in range(args.warmup):
        oracle.fwd(x[:8], W, synth.cu_from_lengths([8]), b)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle.fwd(x, W, cu, b)
        oracle.bwd(x, dy, W, cu, b, policy)
        times.append(time.perf_counter() - t0)
    dt = statistics.median(times)
    fwd_b, bwd_b = compulsory_bytes(n, w.C, 0)
    v = round((fwd_b + bwd_b) / dt / 1e9, 5)
    out = {"impl": "reference", "metric": METRIC, "value": v, "unit": "GB/s", "n_gpus": ws,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 2),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
           "data": "synthetic",
           "config": {"workload": f"{args.config}: S={w.S}, C={w.C} (bounded slice: first {n} "
                                  f"tokens per step)", "S": w.S, "C": w.C},
           "cpu_baseline": {"value": v, "unit": "GB/s", "cores": 1, "kind": "oracle",
                            "sample": f"first {n} tokens x {w.C} channels, fwd + bwd ({policy})"},
           "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="linattn",
                    choices=["tiny", "mid", "linattn", "boundary", "large"])
    ap.add_argument("--cpu-tokens", type=int, default=4096,
                    help="tokens of the workload the CPU-baseline oracle leg processes")
    ap.add_argument("--ref-tokens", type=int, default=None,
                    help="tokens per step of the reference (oracle) arm (default: 96, fewer "
                         "when --steps is large, so the arm's K steps take about a minute)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end leg")
    ap.add_argument("--exact", action="store_true",
                    help="time the exactness-guarded routes (conv1d_fwd_exact, conv1d_bwd_exact)")
    ap.add_argument("--no-sweep", action="store_true",
                    help="skip the per-workload / per-policy timings (routes)")
    ap.add_argument("--S", type=int, default=None,
                    help="scale the workload to S tokens (same recipe); profiling runs only")
    ap.add_argument("--policy", choices=["bf16", "fp32"], default=None,
                    help="SiLU' policy (default: the workload's own)")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
