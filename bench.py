#!/usr/bin/env python3
"""Benchmark of the attention BoB hot path on synthetic bf16 inputs.

One step = the whole hot path over one batch: attention forward, first
backward and the two-pass BoB.  The metric is the BoB call (its ms/call and
counted TFLOP/s, and the fraction of the BF16 tensor peak), so ``value`` is
the BoB call's whole-job TFLOP/s, timed with CUDA events around every BoB
call inside the K timed steps; the step's own time and TFLOP/s sit beside it.

Default workload: B=2, H=16, N=16384, d=128, tau=1/sqrt(128) (the wide-head
d=128 case on which the >=40%-of-BF16-peak target is stated).  After the
headline it runs, untimed by the headline clock: a per-kernel profiling repeat
of the same K steps, the BoB call on every other benchmark configuration
("vs N": the GPT-2-Small shape, the long-context sweep N = 4096 ... 262144,
the peaky d=128 batch), the four-pass ablation, and the end-to-end BoB call
from pinned host buffers.  Prints ONE JSON line on rank 0.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME] [--no-sweep] [--causal]

FLOPs counted per head (2 N^2 d per N x N x d GEMM): forward 4 N^2 d (S, PV),
first backward 10 N^2 d (S, dP, dV, dQ, dK), BoB 38 N^2 d (19 GEMMs over the
two passes).  Inputs are larger than L2, so no L2 flush is needed between
steps.

--impl reference times the fp64 CPU oracle (the reference arm: there is no
runnable reference implementation), on a bounded sample of the same workload.
Multi-GPU: replicas only (heads are independent; no collective on the data
path) - each rank runs the full workload on its own GPU, value = total work of
all ranks / max time over ranks.  --gpus must equal the launcher's WORLD_SIZE.
"""

from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "attn BoB ms/call and TFLOP/s vs N (bf16, d=64/128); % of BF16 tensor peak"
FLOPS_FWD, FLOPS_BWD, FLOPS_BOB = 4, 10, 38   # x N^2 d per head
DEFAULT_WORKLOAD = "wide_head_b2h16_n16384_d128"
# The other benchmark configurations, timed on the BoB call after the headline.
SWEEP = ("gpt2s_b8h12_n1024_d64",
         "long_context_b1h1_d64@N=4096", "long_context_b1h1_d64@N=16384", "long_context_b1h1_d64@N=65536",
         "long_context_b1h1_d64@N=131072", "long_context_b1h1_d64@N=262144",
         "peaky_b4h32_n8192_d128")
# Counted GEMMs (2 N^2 d FLOPs each, per head) attributed to each kernel: the
# 38 N^2 d of BoB = pass 1 (11: S, dP, C, B x2, U1 x2, U2, W, Y x2) + pass 2
# (8).  At d <= 64 pass 1 is one sweep (bob_pass1: all 11).  At d > 64 it runs
# as two sweeps: U1-and-Y (the five score GEMMs + U1 x2 + Y x2 = 9) and Z (one
# GEMM doing the work of U2 and W: 2); the recomputed S and dP of the Z sweep
# are not counted.  Forward 2 (S, PV; the second P V product of the hi/lo
# split of P is not counted); first backward 5 (S, dP, dQ in the row kernel,
# dV, dK in the column kernel; the column kernel's recomputed S and dP are not
# counted).
COUNTED_GEMMS = {"bob_pass1": 11, "bob_pass1_u1y": 9, "bob_pass1_z": 2, "bob_pass2": 8,
                 "attn_fwd": 2, "attn_bwd_dq": 3, "attn_bwd_dkdv": 2}


def executed_gemms(d):
    """GEMMs of 2 N^2 d the kernels execute per head and BoB call: the 19
    counted plus recomputed score tiles and split operands.  Two-pass at
    d <= 64: one-sweep pass 1 (11 + the lo term of P o B) and pass 2 (8); at
    d > 64: U1-and-Y (9 + 1), Z (3: S, dP recomputed, Z) and pass 2 (8).
    Four-pass: alpha (S, B: 3), E (5), rows (9), pass 2 (8)."""
    return {"four_pass": 25, "two_pass": 20 if d <= 64 else 21}


def bob_kernels(d):
    """The launches of one BoB call at head size d."""
    return ("bob_pass1", "bob_pass2") if d <= 64 else ("bob_pass1_u1y", "bob_pass1_z", "bob_pass2")
# Resident rows of one CTA: the query-row block of pass 1 (B_r) and the key
# block of pass 2 (B_c) of every BoB kernel.
BLOCK_ROWS = 128


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return p["hbm_gbs"], p["bf16_tflops"], p["bf16_tflops_sustained"], "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def check_gpus(requested, world_size):
    """--gpus N must match the number of ranks the launcher started (one per
    GPU); a mismatch would silently time another number of replicas."""
    if requested != world_size:
        raise SystemExit(f"bench.py: --gpus {requested} but WORLD_SIZE={world_size}; launch N > 1 with "
                         f"torchrun --nproc-per-node {requested}")


class _Nvml:
    """Read-only NVML queries through ctypes (libnvidia-ml ships with the
    driver): SM clock, its maximum and the active clock-event reasons."""
    SM = 1                                                  # NVML_CLOCK_SM
    BITS = {"sw_power_cap": 0x4, "hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20, "hw_thermal_slowdown": 0x40}

    def __init__(self, index):
        import ctypes
        self.c = ctypes
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        self.lib, self.h = lib, ctypes.c_void_p()
        if lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(index), ctypes.byref(self.h)) != 0:
            raise OSError("no NVML handle")
        self.reasons_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            lib.nvmlDeviceGetCurrentClocksThrottleReasons
        self.sample()

    def max_sm(self):
        v = self.c.c_uint()
        return float(v.value) if self.lib.nvmlDeviceGetMaxClockInfo(self.h, self.SM, self.c.byref(v)) == 0 else 0.0

    def sample(self):
        clk, r = self.c.c_uint(), self.c.c_ulonglong()
        if self.lib.nvmlDeviceGetClockInfo(self.h, self.SM, self.c.byref(clk)) != 0:
            raise OSError("nvmlDeviceGetClockInfo failed")
        self.reasons_fn(self.h, self.c.byref(r))
        return float(clk.value), [n for n, bit in self.BITS.items() if r.value & bit]


class Clocks:
    """SM clock and throttle reasons sampled DURING the timed region: an NVML
    poller thread (every 2 ms, so short regions get samples too), else
    nvidia-smi -lms 200.  The samples are kept in clocks_rank<i>.csv in the
    folder named by $FBOB_CLOCK_DIR (default: the current directory)."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.nvml = None
        self.path = os.path.join(os.environ.get("FBOB_CLOCK_DIR") or os.getcwd(), f"clocks_rank{index}.csv")

    def start(self):
        os.makedirs(os.path.dirname(self.path), exist_ok=True)
        try:
            self.nvml = _Nvml(self.index)
        except Exception:
            self.nvml = None
        if self.nvml is not None:
            import threading
            self.samples, self.halt, self.live = [], threading.Event(), threading.Event()

            def poll():
                while not self.halt.is_set():
                    if self.live.is_set():
                        try:
                            self.samples.append(self.nvml.sample())
                        except Exception:
                            return
                    self.halt.wait(0.002)

            self.thread = threading.Thread(target=poll, daemon=True)
            self.thread.start()
            return
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def begin(self):
        """The timed region starts now (the NVML poller records from here on)."""
        if self.nvml is not None:
            self.live.set()

    def stop(self):
        if self.nvml is not None:
            self.halt.set()
            self.thread.join(timeout=5)
            mx = self.nvml.max_sm()
            with open(self.path, "w") as f:
                f.write("sm_mhz,sm_max_mhz,reasons\n")
                for clk, rs in self.samples:
                    f.write(f"{clk:.0f},{mx:.0f},{'|'.join(rs)}\n")
            if not self.samples:
                return None
            reasons = sorted({n for _, rs in self.samples for n in rs})
            return {"sm_mhz": statistics.median(c for c, _ in self.samples), "sm_max_mhz": mx, "reasons": reasons,
                    "samples": len(self.samples), "source": "nvml"}
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, mx, reasons = [], 0.0, set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = max(mx, float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm), "source": "nvidia-smi"}


class Chain:
    """Device buffers of one workload and the three calls of the hot path."""

    def __init__(self, fb, torch, w, dev, causal, host=None):
        import attn_inputs
        self.fb, self.w, self.cz = fb, w, dict(causal=causal)
        self.host = attn_inputs.make_inputs(w, pin_memory=True) if host is None else host
        self.x = {k: v.to(dev) for k, v in self.host.items()}
        shp = (w.B, w.H, w.N, w.d)
        f32 = dict(dtype=torch.float32, device=dev)
        self.O, self.dQ, self.dK, self.dV = (torch.empty(shp, **f32) for _ in range(4))
        self.g = [torch.empty(shp, **f32) for _ in range(4)]
        self.L, self.D = torch.empty(shp[:3], **f32), torch.empty(shp[:3], **f32)
        self.ws = torch.empty(shp[:3] + (2,), **f32)

    def fwd_bwd(self):
        fb, x, w = self.fb, self.x, self.w
        fb.attn_fwd(x["Q"], x["K"], x["V"], w.tau, self.O, self.L, **self.cz)
        fb.attn_bwd(x["Q"], x["K"], x["V"], self.O, x["dO"], self.L, w.tau, self.dQ, self.dK, self.dV, self.D,
                    **self.cz)

    def bob(self, entry=None, x=None, O=None, L=None, D=None, g=None):
        fb, w = self.fb, self.w
        x = self.x if x is None else x
        g = self.g if g is None else g
        (entry or fb.attn_bob)(x["Q"], x["K"], x["V"], self.O if O is None else O, x["dO"],
                               self.L if L is None else L, self.D if D is None else D,
                               x["UQ"], x["UK"], x["UV"], w.tau, *g, self.ws, **self.cz)

    def step(self):
        self.fwd_bwd()
        self.bob()


def time_calls(torch, stream, fn, n, warmup=2):
    """Mean ms of n back-to-back calls of fn (CUDA events on the launching stream)."""
    for _ in range(warmup):
        fn()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(n):
        fn()
    e1.record(stream)
    e1.synchronize()
    return e0.elapsed_time(e1) / n


def run_ours(args, w):
    import torch
    import torch.distributed as dist

    import attn_inputs
    import exact_second_order_attn_gb300 as fb

    ws, rank, local = dist_env()
    check_gpus(args.gpus, ws)
    if ws > 1:
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    fb.load()
    stream = torch.cuda.current_stream()

    def barrier():
        if ws > 1:
            dist.barrier()
        torch.cuda.synchronize()

    def max_over_ranks(v):
        return reduce_max(v, ws, dev)

    torch.cuda.reset_peak_memory_stats()
    ch = Chain(fb, torch, w, dev, args.causal)
    for _ in range(args.warmup):
        ch.step()
    fb.device_status()

    # ---- headline: K steps (fwd + bwd + BoB), each BoB call bracketed by events
    clocks = Clocks(local)
    clocks.start()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    barrier()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks.begin()
    t0.record(stream)
    for b0, b1 in ev:
        ch.fwd_bwd()
        b0.record(stream)
        ch.bob()
        b1.record(stream)
    t1.record(stream)
    barrier()
    clk = clocks.stop()
    step_ms = max_over_ranks(t0.elapsed_time(t1) / args.steps)
    bob_ms = max_over_ranks(statistics.mean(b0.elapsed_time(b1) for b0, b1 in ev))
    fb.device_status()
    peak_mem = int(torch.cuda.max_memory_allocated())

    # ---- per-kernel times: a second timed repeat of the same K steps with the
    # library's per-launch CUDA events (kept out of the headline region)
    fb.fbob_profile_report()          # drop anything recorded so far
    fb.fbob_profile_enable(True)
    barrier()
    for _ in range(args.steps):
        ch.step()
    barrier()
    fb.fbob_profile_enable(False)
    kernels = fb.fbob_profile_report()
    launches_per_step = sum(v[0] for v in kernels.values()) / args.steps
    fb.device_status()

    heads = w.B * w.H
    # causal: every GEMM covers the N (N + 1) / 2 unmasked (query, key) pairs
    pairs = causal_fraction(w.N) if args.causal else 1.0
    unit = w.N * w.N * w.d * heads * pairs
    flops_step = (FLOPS_FWD + FLOPS_BWD + FLOPS_BOB) * unit
    flops_bob = FLOPS_BOB * unit
    hbm, pk, pk_sus, pk_kind = peaks()
    value = job_tflops(ws, flops_bob, bob_ms)
    sweep = run_sweep(args, fb, torch, dev, stream, pk, w) if args.sweep else None

    # ---- ablation: the same BoB on the four-pass schedule (alpha, E, rows, columns)
    nb = max(3, args.steps)
    four_ms = max_over_ranks(time_calls(torch, stream, lambda: ch.bob(fb.fbob_attn_bob_four_pass), nb))
    fb.device_status()

    # ---- end to end through the public API from pinned host buffers
    e2e = run_e2e(args, fb, torch, dev, stream, ch, flops_bob, ws, max_over_ranks, barrier)
    fb.device_status()

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 3), "unit": "TFLOP/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(step_ms, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded iid Gaussian, bf16 inputs, fp32 accumulation and outputs)",
            "value_basis": "the BoB call (pass 1 + pass 2): counted 38 N^2 d per head / its mean time, "
                           "CUDA events around each BoB call of the K timed steps",
            "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d, "tau": w.tau,
                       "causal": bool(args.causal),
                       "step": "fwd + first bwd + BoB (pass 1 + pass 2)",
                       "flops_per_step": flops_step,
                       "flop_count": "52 N^2 d per head per step (fwd 4, bwd 10, BoB 38)"
                                     + (", times (N+1)/(2N) for the causal mask" if args.causal else ""),
                       "l2": "inputs (%.0f MB) larger than the 129 MB L2; no flush"
                             % (sum(v.numel() * v.element_size() for v in ch.host.values()) / 1e6),
                       "parallelism": f"replicas x{ws}"},
            "bob": {"ms_per_call": round(bob_ms, 4), "tflops": round(flops_bob / (bob_ms * 1e-3) / 1e12, 3),
                    "frac_of_peak": round(flops_bob / (bob_ms * 1e-3) / 1e12 / pk, 4), "peak_tflops": pk,
                    "peak_kind": f"{pk_kind} burst (bf16_tflops)", "counted_flops": flops_bob},
            "step": {"ms": round(step_ms, 4), "tflops": round(job_tflops(ws, flops_step, step_ms), 3)},
            # the two-pass schedule against the four-pass one it collapses (same counted
            # 38 N^2 d; executed GEMMs per head in the json)
            "ablation_four_pass": {"ms_per_call": round(four_ms, 4),
                                   "tflops_counted": round(flops_bob / (four_ms * 1e-3) / 1e12, 3),
                                   "two_pass_ms_per_call": round(bob_ms, 4),
                                   "two_pass_speedup": round(four_ms / bob_ms, 3),
                                   "gemms_executed_per_head": executed_gemms(w.d)},
            "e2e": e2e,
            # our kernels launched in the timed region: K steps x the launches per
            # step the library recorded in the profiling repeat
            "gpu_launches": int(round(launches_per_step * args.steps)),
            # no N x N tensor exists: the process's peak device allocation (inputs,
            # outputs, workspace, all on the caller's side) beside one fp32 N x N score matrix
            "memory": {"peak_allocated_bytes": peak_mem, "one_nxn_fp32_bytes": 4 * w.N * w.N * heads},
            "clocks": clk,
        }
        line["kernels"] = {k: {"launches": v[0], "avg_ms": round(v[1] / v[0], 4)} for k, v in kernels.items()}
        line["kernel_timing"] = "a second timed repeat of the K steps with per-launch CUDA events on the launching stream"
        line["roofline"] = roofline(w, kernels, pk_sus, pairs)
        line["bob"]["ledger"] = bob_ledger(w, pairs)
        if sweep is not None:
            line["sweep"] = sweep
        line["cpu_baseline"] = cpu_baseline(w, args, head0(ch.host))
        print(json.dumps(line), flush=True)
    if ws > 1:
        dist.destroy_process_group()


def run_sweep(args, fb, torch, dev, stream, peak, headline):
    """BoB ms/call, counted TFLOP/s, fraction of the burst peak and the peak
    device allocation of every other benchmark configuration ("vs N"), each
    after fwd + bwd produced its O, L, D; 3 warm-up calls, then enough calls
    for about a quarter of a second (at least 5)."""
    import attn_inputs
    out = []
    for name in SWEEP:
        w = attn_inputs.WORKLOADS[name]
        if w.name == headline.name:
            continue
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        torch.cuda.reset_peak_memory_stats()
        base = torch.cuda.memory_allocated()
        ch = Chain(fb, torch, w, dev, args.causal)
        ch.fwd_bwd()
        one = time_calls(torch, stream, ch.bob, 1, warmup=3)
        n = max(5, min(200, int(250.0 / max(one, 1e-3))))
        ms = time_calls(torch, stream, ch.bob, n, warmup=0)
        fb.device_status()
        # per-kernel times: a separate repeat with the library's per-launch events
        fb.fbob_profile_report()
        fb.fbob_profile_enable(True)
        for _ in range(3):
            ch.bob()
        torch.cuda.synchronize()
        fb.fbob_profile_enable(False)
        kern = {k: round(v[1] / v[0], 4) for k, v in fb.fbob_profile_report().items()}
        pairs = causal_fraction(w.N) if args.causal else 1.0
        flops = FLOPS_BOB * w.N * w.N * w.d * w.B * w.H * pairs
        tf = flops / (ms * 1e-3) / 1e12
        out.append({"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d, "calls": n,
                    "ms_per_call": round(ms, 4), "tflops": round(tf, 3), "frac_of_peak": round(tf / peak, 4),
                    "kernel_avg_ms": kern,
                    "peak_allocated_bytes": int(torch.cuda.max_memory_allocated() - base),
                    "one_nxn_fp32_bytes": 4 * w.N * w.N * w.B * w.H})
        del ch
    return out


def run_e2e(args, fb, torch, dev, stream, ch, flops_bob, ws, max_over_ranks, barrier):
    """The BoB call end to end through the public API from pinned host buffers:
    every step copies that step's inputs (Q, K, V, dO, UQ, UK, UV, O, L, D)
    host -> device and the four gradients device -> host.  Pipelined: two
    device buffer sets; the copy-in of step k+1 and the copy-out of step k run
    on two copy streams while step k+1 / k computes.  The serial variant (copy
    in, call, copy out, one after another) is timed too."""
    names = ("Q", "K", "V", "dO", "UQ", "UK", "UV")
    h_in = dict(ch.host)
    for k, t in (("O", ch.O), ("L", ch.L), ("D", ch.D)):
        h_in[k] = t.cpu().pin_memory()
    h_out = [[torch.empty(g.shape, dtype=torch.float32, pin_memory=True) for g in ch.g] for _ in range(2)]
    d_in = [{k: torch.empty_like(v, device=dev) for k, v in h_in.items()} for _ in range(2)]
    d_out = [[torch.empty_like(g) for g in ch.g] for _ in range(2)]
    h2d = sum(v.numel() * v.element_size() for v in h_in.values())
    d2h = sum(t.numel() * t.element_size() for t in h_out[0])
    cin, cout = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = lambda: torch.cuda.Event()   # noqa: E731

    def call(b):
        x = {k: d_in[b][k] for k in names}
        ch.bob(x=x, O=d_in[b]["O"], L=d_in[b]["L"], D=d_in[b]["D"], g=d_out[b])

    def pipelined(n):
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e_in, e_done, e_out = [ev(), ev()], [None, None], [None, None]
        start.record(stream)
        cin.wait_event(start)

        def copy_in(b):
            with torch.cuda.stream(cin):
                for k, v in h_in.items():
                    d_in[b][k].copy_(v, non_blocking=True)
                e_in[b].record(cin)

        copy_in(0)
        for k in range(n):
            b = k % 2
            stream.wait_event(e_in[b])
            if e_out[b] is not None:
                stream.wait_event(e_out[b])      # d_out[b] copied out (step k - 2)
            call(b)
            e_done[b] = ev()
            e_done[b].record(stream)
            if k + 1 < n:
                nb = (k + 1) % 2
                if e_done[nb] is not None:
                    cin.wait_event(e_done[nb])   # step k - 1 no longer reads d_in[nb]
                copy_in(nb)
            cout.wait_event(e_done[b])
            with torch.cuda.stream(cout):
                for hdst, src in zip(h_out[b], d_out[b]):
                    hdst.copy_(src, non_blocking=True)
                e_out[b] = ev()
                e_out[b].record(cout)
        for e in e_out:
            if e is not None:
                stream.wait_event(e)
        end.record(stream)
        end.synchronize()
        return start.elapsed_time(end) / n

    def serial(n):
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(stream)
        for _ in range(n):
            for k, v in h_in.items():
                d_in[0][k].copy_(v, non_blocking=True)
            call(0)
            for hdst, src in zip(h_out[0], d_out[0]):
                hdst.copy_(src, non_blocking=True)
        end.record(stream)
        end.synchronize()
        return start.elapsed_time(end) / n

    pipelined(2)
    barrier()
    ms = max_over_ranks(pipelined(args.steps))
    barrier()
    serial(1)
    ms_serial = max_over_ranks(serial(args.steps))
    # the copied-out gradients equal the device-side call's on the same inputs
    ch.bob()
    torch.cuda.synchronize()
    same = all(torch.equal(h.to(dev), g) for h, g in zip(h_out[0], ch.g))   # the serial run's last copy-out
    return {"value": round(job_tflops(ws, flops_bob, ms), 3), "unit": "TFLOP/s", "ms_per_call": round(ms, 4),
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "call": "fbob_attn_bob from pinned host buffers (inputs Q, K, V, dO, UQ, UK, UV, O, L, D in, "
                    "gQ, gK, gV, gdO out)",
            "overlap": "double-buffered: copy-in of step k+1 and copy-out of step k on two copy streams "
                       "while the compute stream runs",
            "serial": {"ms_per_call": round(ms_serial, 4), "value": round(job_tflops(ws, flops_bob, ms_serial), 3)},
            "outputs_match_device_call": bool(same)}


def run_once(args, w):
    """Profiler target: the same step as the timed loop, run warmup + 1 times."""
    import torch

    import attn_inputs
    import exact_second_order_attn_gb300 as fb
    fb.load()
    x = {k: v.cuda() for k, v in attn_inputs.make_inputs(w).items()}
    for _ in range(args.warmup + 1):
        O, L = fb.attn_fwd(x["Q"], x["K"], x["V"], w.tau)
        dQ, dK, dV, D = fb.attn_bwd(x["Q"], x["K"], x["V"], O, x["dO"], L, w.tau)
        fb.attn_bob(x["Q"], x["K"], x["V"], O, x["dO"], L, D, x["UQ"], x["UK"], x["UV"], w.tau)
    fb.device_status()
    torch.cuda.synchronize()
    print(f"once ok: {w.name}")


def reduce_max(v, world_size, device):
    """Max of a per-rank float over all ranks (the slowest replica sets the time)."""
    if world_size == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(world_size, flops_per_rank_step, step_ms):
    """Whole-job throughput: every replica does the same work; time is the max."""
    return world_size * flops_per_rank_step / (step_ms * 1e-3) / 1e12


def kernel_source_hash():
    """Hash of the tensor-core kernel sources; DRAM counters taken with other
    sources are stale."""
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "exact_second_order_attn_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        if f.startswith("tc_") or f == "tmap.cu":
            h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


def causal_fraction(N):
    """Share of (query, key) pairs a causal mask keeps: N (N + 1) / 2 of N^2."""
    return (N + 1) / (2.0 * N)


def kernel_bytes(name, N, d, br=BLOCK_ROWS):
    """(ledger, compulsory) HBM bytes of one head for a BoB kernel, bf16 inputs
    and fp32 O / L / D / (alpha, E) / outputs.

    ledger: the transfer count of the pages' Theorem 4.3 (evolve.pub review,
    Strengths, "Theory honestly scoped"), split by kernel and evaluated at the
    resident block of BLOCK_ROWS rows: every row block re-reads the streamed
    tensors of all N rows.  compulsory: every tensor the kernel touches read
    or written once."""
    Nd, N2 = N * d, N * N / br
    if name == "bob_pass1":
        # the one-sweep pass 1: resident Q, UQ, dO, O, L, D; streams K, UK, V, UV;
        # writes gQ, gdO, (alpha, E)
        res, stream, out = 6 * Nd + 4 * Nd + 8 * N, 8 * d * N2, 8 * Nd + 8 * N
        return res + stream + out, res + 8 * Nd + out
    if name == "bob_pass1_u1y":
        # resident Q, UQ, dO (bf16), O, L, D; streams K, UK, V, UV; writes U1 (gQ), gdO, (alpha, E)
        res, stream, out = 6 * Nd + 4 * Nd + 8 * N, 8 * d * N2, 8 * Nd + 8 * N
        return res + stream + out, res + 8 * Nd + out
    if name == "bob_pass1_z":
        # resident Q, dO, U1 (gQ), L, D, (alpha, E); streams K, V; writes gQ
        res, stream, out = 4 * Nd + 4 * Nd + 16 * N, 4 * d * N2, 4 * Nd
        return res + stream + out, res + 4 * Nd + out
    if name == "bob_pass2":
        # resident K, UK, V, UV; streams Q, UQ, dO, L, D, (alpha, E); writes gK, gV
        res, stream, out = 8 * Nd, (6 * d + 16) * N2, 8 * Nd
        return res + stream + out, res + 6 * Nd + 16 * N + out
    return None, None


def bob_ledger(w, pairs=1.0):
    """The pages' HBM transfer ledger for one BoB call (evolve.pub review,
    Strengths, "Theory honestly scoped": Theorem 4.3, Q = 12Nd + 4N +
    4dN^2/B_r + (3d+4)N^2/B_c words per head), in bytes for bf16 inputs and
    fp32 O / vectors / outputs, at B_r = B_c = BLOCK_ROWS, beside the same
    count for the kernels as built (at d > 64 pass 1 runs as two sweeps: the
    Z sweep streams K, V once more and round-trips U1), and measured DRAM
    bytes per call when the committed counters match the current sources."""
    N, d, h = w.N, w.d, w.B * w.H
    br = bc = BLOCK_ROWS
    pages = h * (34 * N * d + 16 * N + 8 * d * N * N / br + (6 * d + 16) * N * N / bc)
    kern = bob_kernels(d)
    built = sum(kernel_bytes(k, N, d)[0] for k in kern) * h
    comp = sum(kernel_bytes(k, N, d)[1] for k in kern) * h
    measured = None
    rec = _traffic_record(w, pairs)
    if rec is not None:
        got = [rec["kernels"].get(k) for k in kern]
        if all(g is not None for g in got):
            measured = sum(g["bytes_per_launch"] * h / g["heads"] for g in got)
    out = {"formula": "Theorem 4.3: 12Nd + 4N + 4dN^2/B_r + (3d+4)N^2/B_c words per head",
           "B_r": br, "B_c": bc, "pages_ledger_bytes": pages, "kernels_ledger_bytes": built,
           "compulsory_bytes": comp, "measured_dram_bytes": measured}
    if measured is not None:
        out["measured_over_ledger"] = round(measured / built, 4)
        out["measured_over_compulsory"] = round(measured / comp, 4)
    return out


def _traffic_record(w, pairs):
    """The committed per-kernel DRAM counters, if they were taken on the
    current sources at this N and d without the causal mask."""
    try:
        with open(os.path.join(ROOT, "profiles", "dram_traffic.json")) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    if pairs != 1.0 or rec.get("source_hash") != kernel_source_hash():
        return None
    ks = {k: v for k, v in rec.get("kernels", {}).items() if v.get("d") == w.d and v.get("N") == w.N}
    return {**rec, "kernels": ks}


def roofline(w, kernels, peak, pairs=1.0):
    """Roofline of the dominant kernel (largest share of the step): counted
    FLOPs per launch / its average launch time (CUDA events recorded by the
    library on the launching stream in the profiling repeat of the K steps),
    against the sustained bf16 peak (the kernel runs inside a long step).
    traffic = DRAM bytes per launch from the committed ncu counters, scaled
    from their profiling workload by the number of heads, or null if the
    kernels changed since; beside it the kernel's ledger and compulsory
    bytes."""
    if not kernels:
        return None
    name, (n, total, _, _) = max(kernels.items(), key=lambda kv: kv[1][1])
    avg_ms = total / n
    heads = w.B * w.H
    flops = COUNTED_GEMMS.get(name, 0) * 2 * w.N * w.N * w.d * heads * pairs
    achieved = flops / (avg_ms * 1e-3) / 1e12
    traffic = None
    rec = _traffic_record(w, pairs)
    if rec is not None and name in rec["kernels"]:
        k = rec["kernels"][name]
        traffic = k["bytes_per_launch"] * heads / k["heads"]
    ledger, comp = kernel_bytes(name, w.N, w.d)
    out = {"kernel": name, "bound": "tensor", "achieved": round(achieved, 3), "peak": peak,
           "unit": "TFLOP/s", "frac": round(achieved / peak, 4), "traffic": traffic,
           "avg_launch_ms": round(avg_ms, 4), "counted_flops_per_launch": flops,
           "peak_source": "MEASURED_PEAKS.json bf16_tflops_sustained (kernel timed inside the step)"}
    if ledger is not None and pairs == 1.0:
        out["ledger_bytes"] = ledger * heads
        out["compulsory_bytes"] = comp * heads
        if traffic is not None:
            out["traffic_over_ledger"] = round(traffic / (ledger * heads), 4)
            out["traffic_over_compulsory"] = round(traffic / (comp * heads), 4)
    return out


def head0(inp):
    return {k: v[0, 0].double().numpy() for k, v in inp.items()}


def oracle_sample(w, x, rows, causal=False):
    """One bounded sample of the workload on the CPU oracle: query rows
    [0, rows) of head (0, 0) through forward, first backward and BoB (each
    row block's work is exactly rows/N of the head's; with the causal mask
    the sampled rows keep rows (rows + 1) / 2 (query, key) pairs)."""
    import numpy as np

    import oracle.attention as orc
    r = slice(0, rows)
    q = np.arange(rows) if causal else None
    t = time.perf_counter()
    orc.attn_fwd_head(x["Q"][r], x["K"], x["V"], w.tau, q)
    orc.attn_bwd_rows(x["Q"][r], x["K"], x["V"], x["dO"][r], w.tau, q)
    orc.bob_rows(x["Q"][r], x["K"], x["V"], x["dO"][r], x["UQ"][r], x["UK"], x["UV"], w.tau, q)
    return time.perf_counter() - t


def sample_pairs(w, rows, causal):
    return rows * (rows + 1) / 2 if causal else rows * w.N


def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        return max((i.get("num_threads", 0) for i in threadpool_info()), default=os.cpu_count())
    except Exception:
        return int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))


def cpu_baseline(w, args, x):
    rows = args.baseline_rows
    secs = oracle_sample(w, x, rows, args.causal)
    flops = (FLOPS_FWD + FLOPS_BWD + FLOPS_BOB) * sample_pairs(w, rows, args.causal) * w.d
    return {"value": round(flops / secs / 1e12, 6), "unit": "TFLOP/s", "cores": blas_threads(),
            "kind": "oracle", "seconds": round(secs, 3),
            "sample": f"query rows [0,{rows}) of head (0,0) of {w.name}: fwd + first bwd + BoB rows, "
                      f"fp64 numpy, = {rows}/{w.N * w.B * w.H} of one step's work"}


def run_reference(args, w):
    ws, rank, _ = dist_env()
    check_gpus(args.gpus, ws)
    if rank != 0:
        return
    import attn_inputs
    x = head0(attn_inputs.make_inputs(w))
    for _ in range(args.warmup):
        oracle_sample(w, x, args.cpu_rows, args.causal)
    times = [oracle_sample(w, x, args.cpu_rows, args.causal) for _ in range(args.steps)]
    secs = statistics.mean(times)
    flops = (FLOPS_FWD + FLOPS_BWD + FLOPS_BOB) * sample_pairs(w, args.cpu_rows, args.causal) * w.d
    value = flops / secs / 1e12
    cb = {"value": round(value, 6), "unit": "TFLOP/s", "cores": blas_threads(), "kind": "oracle",
          "sample": f"query rows [0,{args.cpu_rows}) of head (0,0) of {w.name} per step"}
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s",
            "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(secs * 1e3, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d, "causal": bool(args.causal),
                       "step": "fwd + first bwd + BoB on the sampled rows"},
            "cpu_baseline": cb,
            "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    import attn_inputs
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1, help="GPUs = ranks; must equal the launcher's WORLD_SIZE")
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(attn_inputs.WORKLOADS))
    ap.add_argument("--cpu-rows", type=int, default=None,
                    help="query rows of one head per reference-arm step (CPU oracle); "
                         "default 2048 * 16384 / N (a fixed amount of oracle work), at most N")
    ap.add_argument("--baseline-rows", type=int, default=None,
                    help="query rows of one head in the cpu_baseline sample; "
                         "default 16384 * 16384 / N (about ten seconds of oracle work), at most N")
    ap.add_argument("--causal", action="store_true",
                    help="causal mask (query i attends to keys j <= i); counted FLOPs scale by (N+1)/(2N)")
    ap.add_argument("--no-sweep", dest="sweep", action="store_false",
                    help="skip the BoB timings of the other benchmark configurations")
    ap.add_argument("--once", action="store_true",
                    help="run --warmup + 1 steps and exit without timing (for profiler captures)")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    w = attn_inputs.WORKLOADS[args.workload]
    # the oracle's cost per query row grows with N: size its samples by work, not rows
    if args.cpu_rows is None:
        args.cpu_rows = min(w.N, max(64, 2048 * 16384 // w.N))
    if args.baseline_rows is None:
        args.baseline_rows = min(w.N, max(128, 16384 * 16384 // w.N))
    if args.impl == "reference":
        run_reference(args, w)
    elif args.once:
        run_once(args, w)
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()
