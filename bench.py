#!/usr/bin/env python
"""Benchmark of the W4A16 MoE layer forward on GB300.

One step = one forward call per batch size of the workload (default: the
decode sweep M in {1, 9, 90} of an E=384, H=7168, I=2048, top-8, INT4 g32
layer), inputs already resident in HBM, L2 flushed before every call.  The
headline value is that workload's tokens/s; the same run also times the rest
of the metric's M range (the plateau M = 256-1024, the Zipf prefill M = 4096
and 16384, the second layer shape E=128 M = 1-2048) the same way and reports
each under ``other_workloads``.  Every row also gives the µs/call with all
timed calls of its batch size back to back (``us_per_call_alone``), next to
the step's interleaved calls.

  python bench.py [--gpus N] [--steps K] [--warmup W]
                  [--config decode|plateau|prefill|second|toy|e256|group128]
                  [--extra plateau,prefill,second|none]
                  [--small-batch-kernel five|one] [--impl ours|reference]

Prints one JSON line (rank 0).  ``--impl reference`` times the plain CPU
oracle on a bounded sample of the same workload instead.  Under torchrun
(N > 1) every rank runs an independent replica of the workload on its own GPU
(the layer forward has no exchange step); the time is the max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = ("MoE layer µs/call & tokens/s vs M (1–16384); HBM GB/s or tensor-pipe % of peak")
CONFIGS = {"decode": synth.DECODE, "plateau": synth.PLATEAU, "prefill": synth.PREFILL,
           "second": synth.SECOND, "toy": synth.TOY, "e256": synth.E256,
           "group128": synth.GROUP128}
# The pages' sweep on one RTX PRO 6000 (sm_120), context only: ms per call.
PAGES_MS = {1: 0.151, 9: 1.18, 90: 5.19, 256: 7.02, 512: 7.01, 1024: 7.02}
KERNELS = ["align", "gather", "gemm_gate_up", "gemm_down", "combine"]
# small batches (at most 128 slots): one kernel aligns and gathers
SMALL_KERNELS = ["align_gather", None, "gemm_gate_up", "gemm_down", "combine"]
FUSED_KERNEL = "decode_fused"   # opt-in: the whole layer in one kernel

# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum, one ncu pass,
# caches flushed by ncu before each launch) of the gate+up GEMM launches of
# the decode sweep, from one capture of the kernel sources whose SHA-256 is
# given (see the profile named there; the hash covers the sources' code with
# comments and blank lines removed).  For any other source the figure no
# longer describes the kernel and the bench reports traffic as null.
TRAFFIC_CAPTURE = {
    "kernel": "gemm_gate_up",
    "sources_sha256": "bd099faca5e098c8f0b518a325138edde1d2ed479ece9339616085d52d719294",
    "workload": "decode_e384_h7168_i2048_top8",
    "bytes_per_launch": {1: 132329216 + 2752768, 9: 1091149312 + 1076736,
                         90: 5559584512 + 2606592},
    "profile": "profiles/dram_gemm_gate_up_decode_e384_m1_9_90.md",
}
KERNEL_SOURCES = ["gemm_tc.cu", "gemm_tc.h", "tc_common.cuh", "sm100.cuh", "moe_internal.h",
                  "device_common.cuh", "decode.cu", "decode.h"]


def code_only(text):
    """C/C++ source without its comments: // and /* */ comments removed
    (string and character literals kept as they are), each line stripped,
    blank lines dropped.  Editing a comment leaves it unchanged; editing
    code does not."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        elif c in "\"'":
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        else:
            out.append(c)
            i += 1
    lines = (line.strip() for line in "".join(out).split("\n"))
    return "\n".join(line for line in lines if line)


def kernel_sources_sha256():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "quantized_moe_expert_align_gb300", "csrc")
    for name in KERNEL_SOURCES:
        path = os.path.join(csrc, name)
        if os.path.exists(path):
            with open(path, encoding="utf-8") as f:
                h.update(name.encode() + b"\0" + code_only(f.read()).encode() + b"\0")
    return h.hexdigest()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(path))
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


def expert_bytes(L):
    """Algorithmic bytes of one expert's codes + bf16 scales (at the layer's
    scale group), for w13 and w2."""
    w13 = 2 * L.I * L.H // 2 + 2 * L.I * (L.H // L.group) * 2
    w2 = L.H * L.I // 2 + L.H * (L.I // L.group) * 2
    return w13, w2


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.idx = device_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


def max_over_ranks(value, device="cpu"):
    """The largest of every rank's ``value`` (the job's time is its slowest
    replica's); ``value`` itself without an initialised multi-rank group."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(tokens_per_step, steps, world, ms):
    """Whole-job tokens/s: every replica processed the same tokens in at
    most ``ms`` (max over ranks)."""
    return world * tokens_per_step * steps / (ms / 1e3)


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def oracle_sample(wl, batches, max_slots):
    """A bounded sample of the workload for the oracle: from each batch, the
    first tokens up to a share of ``max_slots`` slots."""
    per = max(1, max_slots // max(1, len(batches)))
    out = []
    for M, (x, ids, w) in batches.items():
        t = max(1, min(M, per // wl.layer.k))
        out.append((M, x[:t], ids[:t], w[:t]))
    return out


def run_oracle(wl, host_w, sample):
    import oracle
    L = wl.layer
    tok = 0
    t0 = time.perf_counter()
    for _, x, ids, w in sample:
        oracle.forward(x, ids, w, *host_w, L.E, L.H, L.I)
        tok += x.shape[0]
    return tok, time.perf_counter() - t0


def make_batches(wl, seed=0):
    L = wl.layer
    out = {}
    for M in wl.Ms:
        x = synth.hidden(M, L.H, seed)
        ids, w = synth.routing(M, L, seed, zipf_s=wl.zipf_s)
        out[M] = (x, ids, w)
    return out


def describe_sample(sample, wl):
    parts = [f"{x.shape[0]} of {M} tokens" for M, x, _, _ in sample]
    return (f"{wl.name}: " + ", ".join(parts) + " (oracle in fp64, all k slots of each "
            "sampled token)")


def reference_arm(args, wl):
    world, rank, _ = dist_setup()
    if rank != 0:
        return 0
    import oracle
    oracle.build()
    L = wl.layer
    batches = make_batches(wl)
    touched = sorted(set(int(e) for _, ids, _ in batches.values() for e in np.unique(ids)))
    host_w = synth.layer_weights(L, 0, experts=touched)
    sample = oracle_sample(wl, batches, max_slots=8 * len(wl.Ms))
    for _ in range(args.warmup):
        run_oracle(wl, host_w, sample)
    tok, secs = 0, 0.0
    for _ in range(args.steps):
        t, s = run_oracle(wl, host_w, sample)
        tok += t
        secs += s
    value = tok / secs
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * secs / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl.name, "Ms": list(wl.Ms), "E": L.E, "H": L.H, "I": L.I,
                   "k": L.k, "group": L.group, "parallelism": "none (host CPU)"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": oracle.num_threads(),
                         "kind": "oracle", "sample": describe_sample(sample, wl)},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def layer_rows(wl, batches, call_ms, kernel_ms, hbm_peak, tf_peak, alone_ms=None):
    """Per batch size: µs/call, tokens/s, active experts and the fraction of
    roofline = max(touched experts' weight bytes / HBM copy rate,
    6·M·k·H·I / dense fp16 peak) over the measured time; with ``alone_ms``
    also the µs/call and fraction of the calls timed one batch size at a
    time."""
    L = wl.layer
    b13, b2 = expert_bytes(L)
    rows = []
    for M in wl.Ms:
        active = int(np.unique(batches[M][1]).size)
        roof_bytes = active * (b13 + b2)
        flops = 6.0 * M * L.k * L.H * L.I
        t_hbm = roof_bytes / (hbm_peak * 1e9)
        t_tc = flops / (tf_peak * 1e12)
        t_roof_ms = 1e3 * max(t_hbm, t_tc)
        k_ms, mode = kernel_ms[M]
        names = {"one": [FUSED_KERNEL], "small": SMALL_KERNELS}.get(mode, KERNELS)
        rows.append({
            "M": M, "active_experts": active,
            "us_per_call": round(1e3 * call_ms[M], 2),
            "tokens_per_s": round(M / (call_ms[M] / 1e3), 1),
            "bound": "hbm" if t_hbm >= t_tc else "tensor",
            "roofline_bytes": roof_bytes, "roofline_flops": flops,
            "roofline_us": round(1e3 * t_roof_ms, 2),
            "frac_of_roofline": round(t_roof_ms / call_ms[M], 4),
            "kernel_ms": {n: round(float(v), 5) for n, v in zip(names, k_ms) if n},
            "us_per_call_profiled": round(1e3 * float(k_ms.sum()), 2),
            "pages_ms_rtx_pro_6000": PAGES_MS.get(M) if L.E == 384 else None,
        })
        if alone_ms is not None:
            rows[-1]["us_per_call_alone"] = round(1e3 * alone_ms[M], 2)
            rows[-1]["frac_of_roofline_alone"] = round(t_roof_ms / alone_ms[M], 4)
    return rows


class Bench:
    """The library loaded on this rank's GPU, plus what every workload's
    timing shares: the stream, an L2-flush buffer and prepacked layers."""

    def __init__(self, local):
        import torch
        import quantized_moe_expert_align_gb300 as moe
        from quantized_moe_expert_align_gb300 import build as lib_build
        self.torch, self.moe = torch, moe
        lib_build.build()
        moe.load()
        self.stream = torch.cuda.current_stream()
        l2 = torch.cuda.get_device_properties(local).L2_cache_size
        self.flush = torch.empty(max(2 * l2, 256 << 20), dtype=torch.uint8, device="cuda")
        self.layers = {}

    def dev(self, a):
        return self.torch.from_numpy(np.ascontiguousarray(a)).cuda()

    def layer(self, L):
        """(host canonical weights, prepacked w13, prepacked w2) of layer L."""
        if L not in self.layers:
            moe, torch = self.moe, self.torch
            host_w = synth.layer_weights(L, 0)
            q, s = self.dev(host_w[0]), self.dev(host_w[1].view(np.int16))
            p13 = moe.prepack(moe.MOE_PACK_W13, q, s)
            del q, s
            q, s = self.dev(host_w[2]), self.dev(host_w[3].view(np.int16))
            p2 = moe.prepack(moe.MOE_PACK_W2, q, s)
            del q, s
            torch.cuda.synchronize()
            torch.cuda.empty_cache()
            self.layers[L] = (host_w, p13, p2)
        return self.layers[L]

    def device_batches(self, wl, batches):
        torch, L = self.torch, wl.layer
        out = {}
        for M, (x, ids, w) in batches.items():
            out[M] = (self.dev(x.view(np.int16)).view(torch.bfloat16), self.dev(ids), self.dev(w),
                      torch.empty((M, L.H), dtype=torch.bfloat16, device="cuda"))
        return out

    def caller(self, wl, devb, ws):
        moe, L = self.moe, wl.layer
        _, p13, p2 = self.layer(L)

        def call(M):
            x, ids, w, out = devb[M]
            st = moe.moe_w4a16_forward(x, ids, w, p13, p2, out, M, L.k, L.E, L.H, L.I,
                                       ws.buf, self.stream)
            if st != moe.MOE_OK:
                raise moe.MoeError(st, "moe_w4a16_forward")
        return call

    def timed(self, fn, Ms, steps):
        """Per M, the device time (ms) of each of ``steps`` calls fn(M), CUDA
        events on the launching stream around each call, L2 flushed (a
        write of 2x L2) before every call, outside the events."""
        torch = self.torch
        ev = {M: [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in range(steps)] for M in Ms}
        for i in range(steps):
            for M in Ms:
                self.flush.zero_()
                ev[M][i][0].record(self.stream)
                fn(M)
                ev[M][i][1].record(self.stream)
        torch.cuda.synchronize()
        return {M: [a.elapsed_time(b) for a, b in ev[M]] for M in Ms}

    def timed_alone(self, fn, Ms, steps):
        """As timed, but all ``steps`` calls of one batch size back to back
        before the next size (the step interleaves the sizes)."""
        return {M: self.timed(fn, [M], steps)[M] for M in Ms}

    def kernel_times(self, wl, devb, ws, reps):
        """Per M: (mean ms of each library kernel, the path: "five" kernels,
        "small" -- four, one aligning and gathering -- or "one" for the opt-in
        single kernel) -- events between kernels
        (moe_w4a16_forward_profiled), L2 flushed before every call.  The
        single kernel's time is the first entry."""
        torch, moe, L = self.torch, self.moe, wl.layer
        _, p13, p2 = self.layer(L)
        per = {M: np.zeros(5) for M in wl.Ms}
        fused = {}
        for _ in range(reps):
            for M in wl.Ms:
                x, ids, w, out = devb[M]
                evs = [torch.cuda.Event(enable_timing=True) for _ in range(6)]
                self.flush.zero_()
                st = moe.moe_w4a16_forward_profiled(x, ids, w, p13, p2, out, M, L.k, L.E, L.H,
                                                    L.I, ws.buf, evs, self.stream)
                if st != moe.MOE_OK:
                    raise moe.MoeError(st, "moe_w4a16_forward_profiled")
                fused[M] = {1: "one", 4: "small"}.get(moe.moe_w4a16_get_diag()["kernels_launched"],
                                                     "five")
                torch.cuda.synchronize()
                per[M] += np.array([evs[i].elapsed_time(evs[i + 1]) for i in range(5)])
        return {M: (per[M][:1] if fused[M] == "one" else per[M]) / reps for M in wl.Ms}, fused

    def check_status(self, ws, what):
        moe = self.moe
        st, detail = moe.moe_w4a16_get_device_status(ws.buf)
        if st != moe.MOE_OK:
            raise moe.MoeError(st, f"{what}: device status (detail {detail})")


def extra_sweep(bench, wl, args, local, hbm_peak, tf_peak):
    """One more workload of the metric's M range, timed like the headline
    sweep (per call, L2 flushed before each), with its own clock record."""
    torch, moe, L = bench.torch, bench.moe, wl.layer
    batches = make_batches(wl)
    devb = bench.device_batches(wl, batches)
    ws = moe.Workspace(max(wl.Ms), L.k, L.E, L.H, L.I, "cuda")
    call = bench.caller(wl, devb, ws)
    for M in wl.Ms:
        call(M)
    bench.check_status(ws, wl.name)
    for _ in range(args.warmup):
        for M in wl.Ms:
            call(M)
    torch.cuda.synchronize()
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    ms = bench.timed(call, wl.Ms, args.steps)
    alone = bench.timed_alone(call, wl.Ms, args.steps)
    clocks = sampler.stop()
    call_ms = {M: float(np.mean(v)) for M, v in ms.items()}
    alone_ms = {M: float(np.mean(v)) for M, v in alone.items()}
    k_ms, fused = bench.kernel_times(wl, devb, ws, max(3, min(args.steps, 10)))
    bench.check_status(ws, wl.name)
    rows = layer_rows(wl, batches, call_ms, {M: (k_ms[M], fused[M]) for M in wl.Ms}, hbm_peak,
                      tf_peak, alone_ms)
    del devb, ws
    torch.cuda.empty_cache()
    return {"workload": wl.name, "E": L.E, "H": L.H, "I": L.I, "k": L.k, "group": L.group,
            "routing": "zipf(1.1)-biased" if wl.zipf_s else "uniform",
            "timed_calls_per_M": args.steps, "clocks": clocks, "rows": rows}


def our_arm(args, wl):
    import torch
    import torch.distributed as dist

    world, rank, local = dist_setup()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    bench = Bench(local)
    moe = bench.moe
    L = wl.layer
    hbm_peak, tf_peak, peak_kind = peaks()
    host_w, p13, p2 = bench.layer(L)

    batches = make_batches(wl)
    ws = moe.Workspace(max(wl.Ms), L.k, L.E, L.H, L.I, "cuda")
    devb = bench.device_batches(wl, batches)
    stream = bench.stream
    flush = bench.flush
    call = bench.caller(wl, devb, ws)
    dev = bench.dev

    # correctness gate before timing (device status of the last call)
    for M in wl.Ms:
        call(M)
    bench.check_status(ws, "first forward")
    for _ in range(args.warmup):
        for M in wl.Ms:
            call(M)
    torch.cuda.synchronize()

    # ---- timed region: K steps of one call per M; device time per call,
    # L2 flushed before every call (outside the events) ----
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    ms = bench.timed(call, wl.Ms, args.steps)
    if world > 1:
        dist.barrier()
    # (each batch size alone, for the sweep rows; not part of the step)
    alone = bench.timed_alone(call, wl.Ms, args.steps)
    clocks = sampler.stop()
    call_ms = {M: float(np.mean(v)) for M, v in ms.items()}
    alone_ms = {M: float(np.mean(v)) for M, v in alone.items()}
    total_ms = max_over_ranks(sum(sum(v) for v in ms.values()), "cuda")
    tokens_per_step = sum(wl.Ms)
    value = job_value(tokens_per_step, args.steps, world, total_ms)
    launches_per_step = 0
    for M in wl.Ms:   # kernels per call differ with M (the router's, the large alignment)
        call(M)
        launches_per_step += moe.moe_w4a16_get_diag()["kernels_launched"]
    torch.cuda.synchronize()
    gpu_launches = launches_per_step * args.steps

    # ---- per-kernel durations (events between the library's kernels) ----
    per_kernel, fused = bench.kernel_times(wl, devb, ws, max(3, min(args.steps, 10)))

    # ---- router front-end: logits -> ids, weights and alignment alone
    # (moe_route_align), and the whole layer from logits
    # (moe_w4a16_forward_routed, L2 flushed before each call as in the timed
    # steps); same logits as the batches' routing.  A device-side sleep first
    # lets the host queue the calls ahead of the GPU, so that the events time
    # the kernels, not the host's launch latency.
    router = {}
    reps = max(5, min(args.steps, 20))
    for M in wl.Ms:
        x, ids, w, out = devb[M]
        lg = dev(synth.logits(M, L.E, seed=0, zipf_s=wl.zipf_s))
        r_ids = torch.empty((M, L.k), dtype=torch.int32, device="cuda")
        r_w = torch.empty((M, L.k), dtype=torch.float32, device="cuda")
        cnt = torch.empty(L.E, dtype=torch.int32, device="cuda")
        off = torch.empty(L.E + 1, dtype=torch.int32, device="cuda")
        perm = torch.empty(M * L.k, dtype=torch.int32, device="cuda")
        inv = torch.empty(M * L.k, dtype=torch.int32, device="cuda")
        aws = torch.empty(max(moe.moe_align_workspace_size(M, L.k, L.E), 256),
                          dtype=torch.uint8, device="cuda")

        def route_call():
            st = moe.moe_route_align(lg, M, L.k, L.E, r_ids, r_w, cnt, off, perm, inv, aws, stream)
            if st != moe.MOE_OK:
                raise moe.MoeError(st, "moe_route_align")

        def layer_call():
            st = moe.moe_w4a16_forward_routed(x, lg, p13, p2, out, r_ids, r_w, M, L.k, L.E,
                                              L.H, L.I, ws.buf, stream)
            if st != moe.MOE_OK:
                raise moe.MoeError(st, "moe_w4a16_forward_routed")

        route_call()
        layer_call()
        torch.cuda.synchronize()
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(2 + 2 * reps)]
        torch.cuda._sleep(4_000_000)
        ev[0].record(stream)
        for _ in range(reps):
            route_call()
        ev[1].record(stream)
        for r in range(reps):
            flush.zero_()
            ev[2 + 2 * r].record(stream)
            layer_call()
            ev[3 + 2 * r].record(stream)
        torch.cuda.synchronize()
        t_route = ev[0].elapsed_time(ev[1]) / reps
        t_layer = float(np.mean([ev[2 + 2 * r].elapsed_time(ev[3 + 2 * r]) for r in range(reps)]))
        bench.check_status(ws, "routed forward")
        if not torch.equal(r_ids, ids):
            raise RuntimeError(f"routed ids differ from the batch's routing at M={M}")
        nbytes = M * L.E * 4 + M * L.k * 8
        router[M] = {"route_align_us": round(1e3 * t_route, 2),
                     "route_align_timing": f"mean of {reps} back-to-back calls, warm L2",
                     "route_bytes": nbytes,
                     "route_gbs": round(nbytes / (t_route / 1e3) / 1e9, 1),
                     "us_per_call_from_logits": round(1e3 * t_layer, 2)}

    # ---- the same forward captured once in a CUDA graph and replayed (a
    # decode loop without host launch overhead); L2 flushed before each
    # replay, as in the timed steps ----
    graph_us = {}
    for M in wl.Ms:
        x, ids, w, out = devb[M]
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            st = moe.moe_w4a16_forward(x, ids, w, p13, p2, out, M, L.k, L.E, L.H, L.I, ws.buf)
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        if st != moe.MOE_OK:
            raise moe.MoeError(st, "moe_w4a16_forward")
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            st = moe.moe_w4a16_forward(x, ids, w, p13, p2, out, M, L.k, L.E, L.H, L.I, ws.buf)
        if st != moe.MOE_OK:
            raise moe.MoeError(st, "moe_w4a16_forward (capture)")
        graph.replay()
        torch.cuda.synchronize()
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(2 * reps)]
        for r in range(reps):
            flush.zero_()
            ev[2 * r].record(stream)
            graph.replay()
            ev[2 * r + 1].record(stream)
        torch.cuda.synchronize()
        graph_us[M] = round(1e3 * float(np.mean([ev[2 * r].elapsed_time(ev[2 * r + 1])
                                                   for r in range(reps)])), 2)
        del graph
    bench.check_status(ws, "graph replay")

    # roofline of the dominant kernel (the most device time over the sweep):
    # its algorithmic bytes -- the touched experts' codes + scales it streams
    # (w13 for the gate+up GEMM, w2 for the down GEMM, both for the single
    # small-batch kernel) -- over its mean launch duration
    b13, b2 = expert_bytes(L)
    sweep = layer_rows(wl, batches, call_ms, {M: (per_kernel[M], fused[M]) for M in wl.Ms},
                       hbm_peak, tf_peak, alone_ms)
    per_name = {}
    for row in sweep:
        M = row["M"]
        active = row["active_experts"]
        unit_bytes = {FUSED_KERNEL: b13 + b2, "gemm_gate_up": b13, "gemm_down": b2}
        for name, ms_ in row["kernel_ms"].items():
            if name in unit_bytes:
                acc = per_name.setdefault(name, [0.0, 0.0, 0, unit_bytes[name]])
                acc[0] += active * unit_bytes[name]
                acc[1] += ms_
                acc[2] += 1
        row["router"] = router[M]
        row["us_per_call_graph"] = graph_us[M]
        row["frac_of_roofline_profiled"] = round(row["roofline_us"] / row["us_per_call_profiled"], 4)
    dom = max(per_name, key=lambda nm: per_name[nm][1])
    dom_bytes, dom_ms, dom_launches, dom_unit = per_name[dom]
    achieved = dom_bytes / (dom_ms / 1e3) / 1e9
    traffic = None
    tc = TRAFFIC_CAPTURE
    dom_Ms = [row["M"] for row in sweep if dom in row["kernel_ms"]]
    if (tc["sources_sha256"] == kernel_sources_sha256() and tc["workload"] == wl.name
            and tc["kernel"] == dom and all(M in tc["bytes_per_launch"] for M in dom_Ms)):
        traffic = float(np.mean([tc["bytes_per_launch"][M] for M in dom_Ms]))

    # ---- end to end through the C ABI: pinned host inputs and output.  A
    # call's inputs (hidden, ids, weights) sit packed in one pinned buffer and
    # go over in one copy to one device buffer whose slices are the call's
    # arguments; the output comes back in one copy.  Timed per call, L2
    # flushed before each, like the device-resident steps. ----
    host = {}
    h2d = d2h = 0

    def up16(v):
        return (v + 15) // 16 * 16

    for M, (x, ids, w) in batches.items():
        parts = [np.ascontiguousarray(x).view(np.uint8).reshape(-1),
                 np.ascontiguousarray(ids).view(np.uint8).reshape(-1),
                 np.ascontiguousarray(w).view(np.uint8).reshape(-1)]
        offs, total = [], 0
        for p_ in parts:
            offs.append(total)
            total = up16(total + p_.size)
        packed = np.zeros(total, np.uint8)
        for o, p_ in zip(offs, parts):
            packed[o:o + p_.size] = p_
        hbuf = torch.from_numpy(packed).pin_memory()
        dbuf = torch.empty(total, dtype=torch.uint8, device="cuda")
        dx = dbuf[offs[0]:offs[0] + parts[0].size].view(torch.bfloat16).view(M, L.H)
        did = dbuf[offs[1]:offs[1] + parts[1].size].view(torch.int32).view(M, L.k)
        dw = dbuf[offs[2]:offs[2] + parts[2].size].view(torch.float32).view(M, L.k)
        hout = torch.empty((M, L.H), dtype=torch.int16).pin_memory()
        host[M] = (hbuf, dbuf, dx, did, dw, hout)
        h2d += sum(p_.size for p_ in parts)
        d2h += hout.numel() * 2

    def e2e_call(M):
        hbuf, dbuf, dx, did, dw, hout = host[M]
        out = devb[M][3]
        dbuf.copy_(hbuf, non_blocking=True)
        st = moe.moe_w4a16_forward(dx, did, dw, p13, p2, out, M, L.k, L.E, L.H, L.I, ws.buf,
                                   stream)
        if st != moe.MOE_OK:
            raise moe.MoeError(st, "moe_w4a16_forward")
        hout.copy_(out.view(torch.int16), non_blocking=True)

    # the packed copies reproduce the device-resident inputs: same outputs
    ref_out = {}
    for M in wl.Ms:
        call(M)
        ref_out[M] = devb[M][3].view(torch.int16).clone()
    for M in wl.Ms:
        e2e_call(M)
    torch.cuda.synchronize()
    for M in wl.Ms:
        if not torch.equal(host[M][5], ref_out[M].cpu()):
            raise RuntimeError(f"end-to-end output differs at M={M}")
    e_ms = bench.timed(e2e_call, wl.Ms, args.steps)
    e2e_ms = max_over_ranks(sum(sum(v) for v in e_ms.values()), "cuda")
    e2e = {"value": job_value(tokens_per_step, args.steps, world, e2e_ms), "unit": "tokens/s",
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
           "timing": "per call, L2 flushed before each; copies inside the events"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        oracle.build()
        sample = oracle_sample(wl, batches, max_slots=args.cpu_slots)
        tok, secs = run_oracle(wl, host_w, sample)
        cpu = {"value": tok / secs, "unit": "tokens/s", "cores": oracle.num_threads(),
               "kind": "oracle", "sample": describe_sample(sample, wl)}

    # ---- the rest of the metric's M range: the other workloads, each timed
    # the same way (the headline value stays the decode sweep) ----
    del devb, host
    torch.cuda.empty_cache()
    extras = []
    for name in args.extra:
        xwl = CONFIGS[name]
        if xwl is wl:
            continue
        extras.append(extra_sweep(bench, xwl, args, local, hbm_peak, tf_peak))

    pages = [PAGES_MS.get(M) for M in wl.Ms]
    vs = None
    if L.E == 384 and all(p is not None for p in pages):
        vs = value / (tokens_per_step / (sum(pages) / 1e3))

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": total_ms / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": vs, "dtype": "f16 MMA operands, f32 accumulate (int4 weights)",
            "data": "synthetic",
            "config": {"workload": wl.name, "Ms": list(wl.Ms), "E": L.E, "H": L.H, "I": L.I,
                       "k": L.k, "group": L.group,
                       "routing": "zipf(1.1)-biased" if wl.zipf_s else "uniform",
                       "l2": "flushed before every call (write of 2x L2, outside the events)",
                       "small_batch_kernel": args.small_batch_kernel,
                       "parallelism": f"replicas x{world}",
                       "vs_baseline_ref": "pages' sweep on one RTX PRO 6000 (sm_120): context"},
            "clocks": clocks, "e2e": e2e, "gpu_launches": gpu_launches,
            "roofline": {"bound": "hbm", "kernel": dom, "achieved": achieved,
                         "peak": hbm_peak, "unit": "GB/s", "frac": achieved / hbm_peak,
                         "peak_source": f"{peak_kind} hbm_gbs", "traffic": traffic,
                         "algorithmic_bytes_per_launch": dom_bytes / dom_launches,
                         "launches_averaged": {"Ms": dom_Ms, "count": dom_launches},
                         "traffic_source": tc["profile"] if traffic is not None else None,
                         "algorithmic_bytes_per_unit": dom_unit,
                         "unit_of_work": "active expert (codes + scales the kernel streams)"},
            "cpu_baseline": cpu, "sweep": sweep, "other_workloads": extras,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", choices=sorted(CONFIGS), default="decode")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-slots", type=int, default=800,
                    help="slots the CPU-baseline oracle sample covers")
    ap.add_argument("--small-batch-kernel", choices=["five", "one"], default="five",
                    help="batches of at most 128 slots: the five kernels (default) or the "
                         "opt-in single kernel (MOE_W4A16_DECODE_FUSED=1)")
    ap.add_argument("--extra", default=None,
                    help="comma-separated further workloads timed in the same run "
                         "(default with the decode sweep: plateau,prefill,second; "
                         "'none' for none)")
    args = ap.parse_args()
    if args.extra is None:
        args.extra = "plateau,prefill,second" if args.config == "decode" else "none"
    args.extra = [] if args.extra == "none" else [e for e in args.extra.split(",") if e]
    for e in args.extra:
        if e not in CONFIGS:
            ap.error(f"--extra: unknown workload {e!r}")
    if args.warmup < 3 and args.impl == "ours":
        ap.error("--warmup must be >= 3")
    wl = CONFIGS[args.config]
    if args.small_batch_kernel == "one":
        os.environ["MOE_W4A16_DECODE_FUSED"] = "1"   # read by the library at its first call
    if args.impl == "reference":
        return reference_arm(args, wl)
    return our_arm(args, wl)


if __name__ == "__main__":
    sys.exit(main())
