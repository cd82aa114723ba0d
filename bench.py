#!/usr/bin/env python3
"""Benchmark of one XPress Jacobi draft pass on GB300 (one JSON line on rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference]

Workload: N=32 blocks of B=16 slots, V=152064, D=3584, R=512, H=1536 (the
serving-scale pass), seeded synthetic inputs (no trained weights or hidden
states exist here).  A step is one whole pass through the C ABI
(xp_jacobi_pass: latent stage, tcgen05 readout with the fused add + argmax
written into blk), inputs resident in HBM.  The metric is microseconds per
pass (lower is better); the add-argmax leg (480 x 152064 base + bias) is
reported beside it in GB/s and as a fraction of the measured HBM peak.

Also reported: `roofline` for the dominant kernel (the readout, timed alone
with CUDA events), `e2e` (the same pass through the Python binding with host
buffers, host<->device copies inside the timed region), `cpu_baseline` (the
CPU oracle on a bounded sample, scaled to one pass), SM clocks sampled during
the run.  `--impl reference` times the CPU oracle as the reference arm.

With N > 1 (torchrun, one process per GPU) every rank runs an independent
replica: the pass does not shard, there is no collective on the data path,
and the time is the maximum over ranks.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from speculative_decoding_gb300 import synth  # noqa: E402

METRIC = "µs per Jacobi pass & add-argmax HBM GB/s (% of roofline) at N=32,B=16,V=152064"
SHAPE = synth.SERVE
PEAKS = os.path.join(ROOT, "MEASURED_PEAKS.json")
PROFILE = os.path.join(ROOT, "profiles", "readout_argmax_N32_B16_V152064.md")
READOUT_SRC = os.path.join(ROOT, "speculative_decoding_gb300", "csrc", "xp_readout.cu")


# nominal figures of the part (context beside the measured denominators)
NOMINAL_HBM_GBS = 8000.0
NOMINAL_BF16_TFLOPS = 2250.0


def peaks():
    if os.path.exists(PEAKS):
        with open(PEAKS) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


def readout_bytes(shape) -> int:
    """Algorithmic bytes of one readout launch: W2 once, base once, the latent once."""
    return shape.R * shape.V * 2 + shape.rows * shape.V * 2 + shape.rows * shape.R * 2


def readout_flops(shape) -> float:
    return 2.0 * shape.rows * shape.V * shape.R


def pass_bytes(shape) -> int:
    """Algorithmic bytes of one pass: every weight and input read once (only
    the embedding rows the tokens touch), the latent written and read once,
    the new tokens written."""
    N, B, V, D, R, H = shape.N, shape.B, shape.V, shape.D, shape.R, shape.H
    bf16 = (D * R + 2 * R * H + H * R + R * V      # W_lat, Wg, Wu, Wd, W2
            + N * B * D + N * B * R + N * (B - 1) * V)  # gathered E rows, hcache, base
    mixer = 4 * B * B * R                           # L, fp32
    tokens_in = 8 * (N * B + N)                     # blk, am1
    lat = 2 * (2 * N * (B - 1) * R)                 # bf16 latent: written, then read
    return 2 * bf16 + mixer + tokens_in + lat + 8 * N * (B - 1)


def pass_flops(shape) -> float:
    N, B, V, D, R, H = shape.N, shape.B, shape.V, shape.D, shape.R, shape.H
    return 2.0 * N * B * D * R + 2.0 * N * (B - 1) * (2 * R * H + H * R) + 2.0 * N * (B - 1) * R * V


def traffic_from_profile():
    """dram bytes per readout launch from the committed ncu summary, if it was
    taken on the current readout source (else None)."""
    if not os.path.exists(PROFILE):
        return None
    text = open(PROFILE).read()
    m = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text)
    h = re.search(r"source_sha256:\s*([0-9a-f]{64})", text)
    if not m or not h:
        return None
    cur = hashlib.sha256(open(READOUT_SRC, "rb").read()).hexdigest()
    return float(m.group(1)) if cur == h.group(1) else None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 100 ms."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.samples = []
        self.proc = None
        self.index = index

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "100", "-i", str(self.index)], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 9:
                self.samples.append((time.time(), parts))

    def wait_first(self, limit_s: float = 5.0):
        """Block until nvidia-smi has printed its first sample (or the limit)."""
        t_end = time.time() + limit_s
        while self.proc and not self.samples and time.time() < t_end:
            time.sleep(0.05)

    def stop(self):
        """End the sampling (the samples taken so far stay)."""
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=2)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.proc = None

    def __exit__(self, *a):
        self.stop()

    def summary(self, t0, t1):
        inside = [p for (t, p) in self.samples if t0 - 0.25 <= t <= t1 + 0.25] or [p for (_, p) in self.samples]
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm = [float(p[1]) for p in inside if p[1].replace(".", "").isdigit()]
        mx = [float(p[2]) for p in inside if p[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for p in inside for i in range(4) if p[5 + i].lower() == "active"})
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(inside)}


# ---------------------------------------------------------------------------
# CPU oracle baseline (bounded sample, scaled to one pass)
# ---------------------------------------------------------------------------

def oracle_sample(d, shape, budget_s: float = 12.0):
    import oracle

    oracle.build()
    threads = oracle.num_threads()
    blk, N, B = d["blk"], shape.N, shape.B
    # latent: time groups of `threads` blocks (the oracle is parallel over blocks)
    t_blocks, nb = 0.0, 0
    while nb < N and (nb < 1 or t_blocks < budget_s * 0.3):
        hi = min(N, nb + threads)
        t0 = time.perf_counter()
        lat = oracle.latent(blk, d["am1"], d["hcache"], d["E"], d["W_lat"], d["L"], d["Wg"], d["Wu"], d["Wd"],
                            blocks=(nb, hi))
        t_blocks += time.perf_counter() - t0
        nb = hi
    flat = lat.reshape(-1, shape.R)
    t_rows, nr = 0.0, 0
    while nr < shape.rows and (nr < 1 or t_rows < budget_s * 0.7):
        t0 = time.perf_counter()
        oracle.row_logits(flat[nr % (B - 1)], d["W2"], d["base"][nr])
        t_rows += time.perf_counter() - t0
        nr += 1
    us = (t_blocks / nb * N + t_rows / nr * shape.rows) * 1e6
    sample = (f"oracle latent for {nb} of {N} blocks and readout+add+argmax for {nr} of {shape.rows} rows "
              f"({t_blocks + t_rows:.1f} s), scaled to the whole pass")
    return us, threads, sample


# ---------------------------------------------------------------------------
# reference arm: the CPU oracle
# ---------------------------------------------------------------------------

def max_over_ranks(values, world: int, device) -> list:
    """Each timing's maximum over the ranks (an all-reduce MAX; identity on
    one rank)."""
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    if world > 1:
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def whole_job_per_pass(us: float, passes_per_rank: int, world: int) -> float:
    """µs per pass of the whole job: every rank ran passes_per_rank independent
    passes (replicas) within the max-over-ranks time us."""
    return us / (passes_per_rank * world)


def workload_config(world: int) -> dict:
    """The `config` object of both arms' JSON lines."""
    return {"workload": SHAPE.name, "N": SHAPE.N, "B": SHAPE.B, "V": SHAPE.V, "D": SHAPE.D, "R": SHAPE.R,
            "H": SHAPE.H, "parallelism": "replicas" if world > 1 else "single GPU",
            "l2": "inputs larger than L2 (W2 + base = 302 MB per pass; two sets of per-pass inputs alternate)"}


def run_reference(args, world):
    d = synth.pass_inputs(SHAPE)
    oracle_sample(d, SHAPE, budget_s=0.0)  # warm-up: builds the oracle, one block and one row
    per = []
    sample = ""
    threads = 1
    for _ in range(args.steps):
        us, threads, sample = oracle_sample(d, SHAPE, budget_s=min(12.0, 150.0 / max(1, args.steps)))
        per.append(us)
    value = float(np.median(per))
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 1), "unit": "us/pass", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(value / 1e3, 3),
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": workload_config(world),
        "cpu_baseline": {"value": round(value, 1), "unit": "us/pass", "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 1), "unit": "us/pass", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# GB300 arm
# ---------------------------------------------------------------------------

def dev_bf16(bits, device):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def events_time(stream, fn, steps):
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(steps):
        fn(i)
    e1.record(stream)
    e1.synchronize()
    return e0.elapsed_time(e1) * 1e3  # microseconds


def run_gb300(args, rank, world, local_rank):
    from speculative_decoding_gb300 import build as xbuild
    from speculative_decoding_gb300 import xpress

    if not torch.cuda.is_available():
        raise RuntimeError("bench.py needs a CUDA GPU")
    xbuild.build()
    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    stream = torch.cuda.current_stream()
    hbm_peak, tf_peak, peak_kind = peaks()
    sh = SHAPE
    N, B, V, D, R, H = sh.N, sh.B, sh.V, sh.D, sh.R, sh.H

    d = synth.pass_inputs(sh)
    # second set of per-pass inputs, alternated between steps
    d2 = synth.pass_inputs(synth.PassShape(sh.name, N, B, V, D, R, H, sh.seed + 100), with_embedding=False)
    w = {k: dev_bf16(d[k], device) for k in ("E", "W_lat", "Wg", "Wu", "Wd")}
    w["W2t"] = dev_bf16(np.ascontiguousarray(d["W2"].T), device)  # readout weight, vocabulary-major [V, R]
    L = torch.from_numpy(d["L"]).to(device)
    sets = []
    for src in (d, d2):
        sets.append(dict(hcache=dev_bf16(src["hcache"], device), base=dev_bf16(src["base"], device),
                         am1=torch.from_numpy(src["am1"]).to(device), blk0=torch.from_numpy(src["blk"]).to(device),
                         blk=torch.from_numpy(src["blk"]).to(device)))
    ws = xpress.workspace(xpress.jacobi_workspace_size(N, B, V, D, R, H), device)

    def step(i):
        s = sets[i & 1]
        xpress.jacobi_pass(s["blk"], s["am1"], s["hcache"], w["E"], w["W_lat"], L, w["Wg"], w["Wu"], w["Wd"],
                           w["W2t"], s["base"], ws)

    def reset():
        for s in sets:
            s["blk"].copy_(s["blk0"])

    # ---- the timed passes
    with ClockSampler(local_rank) as clk:
        clk.wait_first()
        for i in range(args.warmup):
            step(i)
        # keep the GPU under the same load for ~0.6 s more (untimed), so that
        # the 100 ms clock samples around the short timed region see it loaded
        t_soak = time.time() + 0.6
        i = args.warmup
        while time.time() < t_soak:
            for _ in range(64):
                step(i)
                i += 1
            torch.cuda.synchronize()
        reset()
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        t0 = time.time()
        us = events_time(stream, step, args.steps)
        torch.cuda.synchronize()
        t1 = time.time()
        if world > 1:
            torch.distributed.barrier()
        if xpress.read_error(ws) != 0:
            raise RuntimeError("device-side error bits set during the timed passes")
        clocks = clk.summary(t0, t1)
        # the clocks are those of the timed passes: the sampler (an nvidia-smi
        # process polling the driver) stops before the other legs
        clk.stop()

        # ---- the dominant kernel alone: the readout with its fused epilogue
        lat = torch.empty((N, B - 1, R), dtype=torch.bfloat16, device=device)
        lws = xpress.workspace(xpress.latent_workspace_size(N, B, D, R, H), device)
        s0 = sets[0]
        xpress.latent_pass(s0["blk"], s0["am1"], s0["hcache"], w["E"], w["W_lat"], L, w["Wg"], w["Wu"], w["Wd"],
                           lat, lws)
        lat2 = lat.view(-1, R)
        rws = xpress.workspace(xpress.readout_workspace_size(sh.rows, V), device)
        rblk = [s["blk"].clone() for s in sets]

        def ro(i):
            xpress.readout_argmax(lat2, w["W2t"], sets[i & 1]["base"], rblk[i & 1], rws)

        for i in range(max(3, args.warmup)):
            ro(i)
        ro_us = events_time(stream, ro, args.steps) / args.steps

        # ---- the add-argmax leg: 480 x 152064 base + bias
        aa = synth.argmax_inputs(synth.ARGMAX_ROWS, synth.ARGMAX_V, 32, 16, seed=synth.ARGMAX_SEED, tie_frac=0.01)
        ab, ac = dev_bf16(aa["base"], device), dev_bf16(aa["bias"], device)
        ablk = torch.from_numpy(aa["blk"]).to(device)
        aws = xpress.workspace(xpress.add_argmax_workspace_size(synth.ARGMAX_ROWS, synth.ARGMAX_V), device)

        def am(i):
            xpress.add_argmax(ab, ac, ablk, aws)

        for i in range(max(3, args.warmup)):
            am(i)
        aa_us = events_time(stream, am, args.steps) / args.steps
        aa_bytes = synth.ARGMAX_ROWS * synth.ARGMAX_V * 4

        # ---- latency floor: one block (N=1, B=16, same model dims), the pass
        # captured once in a CUDA graph and replayed (inputs stay resident)
        fa = synth.pass_activations(synth.FLOOR)
        f_in = dict(hcache=dev_bf16(fa["hcache"], device), base=dev_bf16(fa["base"], device),
                    am1=torch.from_numpy(fa["am1"]).to(device), blk=torch.from_numpy(fa["blk"]).to(device))
        fws = xpress.workspace(xpress.jacobi_workspace_size(1, B, V, D, R, H), device)

        def floor_pass():
            xpress.jacobi_pass(f_in["blk"], f_in["am1"], f_in["hcache"], w["E"], w["W_lat"], L, w["Wg"], w["Wu"],
                               w["Wd"], w["W2t"], f_in["base"], fws)

        for _ in range(3):
            floor_pass()
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            floor_pass()
        graph.replay()
        torch.cuda.synchronize()
        floor_reps = 10000
        floor_us = events_time(stream, lambda i: graph.replay(), floor_reps) / floor_reps
        # the median of single replays, each between its own pair of events
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(1000)]
        for e0, e1 in ev:
            e0.record(stream)
            graph.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        floor_med = float(np.median([e0.elapsed_time(e1) * 1e3 for e0, e1 in ev]))
        if xpress.read_error(fws) != 0:
            raise RuntimeError("device-side error bits set in the latency-floor replays")

        # ---- multi-pass: N=64, B=16, passes to the fixpoint (at most 8), all
        # enqueued at once (xp_jacobi_fixpoint), no host round trip
        xa = synth.pass_activations(synth.FIXPOINT)
        x_in = dict(hcache=dev_bf16(xa["hcache"], device), base=dev_bf16(xa["base"], device),
                    am1=torch.from_numpy(xa["am1"]).to(device), blk0=torch.from_numpy(xa["blk"]).to(device))
        x_blk = x_in["blk0"].clone()
        xws = xpress.workspace(xpress.jacobi_workspace_size(synth.FIXPOINT.N, B, V, D, R, H), device)
        x_passes = torch.zeros(1, dtype=torch.int32, device=device)

        def fixpoint(i):
            x_blk.copy_(x_in["blk0"])
            xpress.jacobi_fixpoint(x_blk, x_in["am1"], x_in["hcache"], w["E"], w["W_lat"], L, w["Wg"], w["Wu"],
                                   w["Wd"], w["W2t"], x_in["base"], xws, x_passes, max_passes=8)

        fixpoint(0)
        torch.cuda.synchronize()
        fx_reps = max(3, min(20, args.steps))
        fx_us = events_time(stream, fixpoint, fx_reps) / fx_reps
        fx_passes = int(x_passes.item())
        # the same call captured in a CUDA graph: one conditional while node
        # whose body is one pass, so only the passes needed run
        fx_graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(fx_graph):
            fixpoint(0)
        x_passes.zero_()
        fx_graph.replay()
        torch.cuda.synchronize()
        if int(x_passes.item()) != fx_passes:
            raise RuntimeError("the captured fixpoint ran a different number of passes")
        fxg_us = events_time(stream, lambda i: fx_graph.replay(), fx_reps) / fx_reps
        if xpress.read_error(xws) != 0:
            raise RuntimeError("device-side error bits set in the multi-pass runs")

        # ---- the same pass in the GEMM-MLP schedule (do_mlp = 0: bf16 g, v
        # and residual), same inputs alternating
        def gemm_step(i):
            s = sets[i & 1]
            xpress.jacobi_pass(s["blk"], s["am1"], s["hcache"], w["E"], w["W_lat"], L, w["Wg"], w["Wu"], w["Wd"],
                               w["W2t"], s["base"], ws, do_mlp=False)

        reset()
        for i in range(max(3, args.warmup)):
            gemm_step(i)
        gm_us = events_time(stream, gemm_step, args.steps) / args.steps
        if xpress.read_error(ws) != 0:
            raise RuntimeError("device-side error bits set in the GEMM-MLP passes")

        # ---- the pages' own embedding layout: E already at the latent width
        # (D = R = 512, W_lat [R, R]); everything else as in the pass
        e_pp = dev_bf16(synth.normal_bf16(sh.seed + 200, 1, (V, R), 0.02), device)
        wl_pp = dev_bf16(synth.normal_bf16(sh.seed + 200, 2, (R, R), 1.0 / math.sqrt(R)), device)
        pws = xpress.workspace(xpress.jacobi_workspace_size(N, B, V, R, R, H), device)

        def pp_step(i):
            s = sets[i & 1]
            xpress.jacobi_pass(s["blk"], s["am1"], s["hcache"], e_pp, wl_pp, L, w["Wg"], w["Wu"], w["Wd"],
                               w["W2t"], s["base"], pws)

        reset()
        for i in range(max(3, args.warmup)):
            pp_step(i)
        pp_us = events_time(stream, pp_step, args.steps) / args.steps
        if xpress.read_error(pws) != 0:
            raise RuntimeError("device-side error bits set in the D = R passes")
        pp_shape = synth.PassShape("pp", N, B, V, R, R, H, 0)

        # ---- end to end through the binding, host buffers, copies inside.
        # Every step copies its inputs from pinned host memory and reads its
        # result back; the copies run on their own streams (the large base
        # split over several, so several copy engines share it), double
        # buffered, so step i+1's inputs stream in while pass i runs.
        host = [dict(hcache=torch.from_numpy(src["hcache"].view(np.int16)).view(torch.bfloat16).pin_memory(),
                     base=torch.from_numpy(src["base"].view(np.int16)).view(torch.bfloat16).pin_memory(),
                     am1=torch.from_numpy(src["am1"]).pin_memory(), blk=torch.from_numpy(src["blk"]).pin_memory(),
                     out=torch.empty((N, B), dtype=torch.int64).pin_memory()) for src in (d, d2)]
        bufs = [dict(hcache=torch.empty_like(sets[0]["hcache"]), base=torch.empty_like(sets[0]["base"]),
                     am1=torch.empty_like(sets[0]["am1"]), blk=torch.empty_like(sets[0]["blk"])) for _ in range(2)]
        n_cs = 4
        copy_streams = [torch.cuda.Stream(device) for _ in range(n_cs)]
        landed = [[torch.cuda.Event() for _ in range(n_cs)] for _ in range(2)]
        freed = [torch.cuda.Event() for _ in range(2)]
        rows_per = (sh.rows + n_cs - 1) // n_cs

        def issue_copy(i):
            h, bf = host[i & 1], bufs[i & 1]
            for c, cs in enumerate(copy_streams):
                if i >= 2:
                    cs.wait_event(freed[i & 1])  # the pass that last read this buffer is done
                with torch.cuda.stream(cs):
                    r0, r1 = c * rows_per, min(sh.rows, (c + 1) * rows_per)
                    if r0 < r1:
                        bf["base"][r0:r1].copy_(h["base"][r0:r1], non_blocking=True)
                    if c == 0:
                        for k in ("hcache", "am1", "blk"):
                            bf[k].copy_(h[k], non_blocking=True)
                landed[i & 1][c].record(cs)

        def e2e_step(i):
            bf = bufs[i & 1]
            for ev in landed[i & 1]:
                stream.wait_event(ev)
            xpress.jacobi_pass(bf["blk"], bf["am1"], bf["hcache"], w["E"], w["W_lat"], L, w["Wg"], w["Wu"],
                               w["Wd"], w["W2t"], bf["base"], ws)
            host[i & 1]["out"].copy_(bf["blk"], non_blocking=True)
            freed[i & 1].record(stream)
            issue_copy(i + 1)

        def e2e_run(steps):
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for cs in copy_streams:
                cs.wait_event(e0)
            issue_copy(0)
            for i in range(steps):
                e2e_step(i)
            e1.record(stream)
            torch.cuda.synchronize()
            return e0.elapsed_time(e1) * 1e3

        e2e_run(max(3, args.warmup))
        e2e_us = e2e_run(args.steps) / args.steps
        if xpress.read_error(ws) != 0:
            raise RuntimeError("device-side error bits set in the end-to-end passes")
        h2d = sum(host[0][k].numel() * host[0][k].element_size() for k in ("hcache", "base", "am1", "blk"))
        d2h = host[0]["out"].numel() * 8

        # the host link alone: the same copies (same four streams, same split)
        # with no pass between them, back to back
        def link_run(steps):
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for cs in copy_streams:
                cs.wait_event(e0)
            for i in range(steps):
                issue_copy(i)
                for ev in landed[i & 1]:
                    stream.wait_event(ev)
                freed[i & 1].record(stream)
            e1.record(stream)
            torch.cuda.synchronize()
            return e0.elapsed_time(e1) * 1e3

        link_run(3)
        link_us = link_run(args.steps) / args.steps

    us, ro_us, aa_us, e2e_us, link_us = max_over_ranks([us, ro_us, aa_us, e2e_us, link_us], world, device)
    if rank != 0:
        return
    per_pass = whole_job_per_pass(us, args.steps, world)
    e2e_per_pass = whole_job_per_pass(e2e_us * args.steps, args.steps, world)
    ro_achieved = readout_bytes(sh) / ro_us / 1e3  # GB/s
    cpu = None
    if world == 1:
        cpu_us, cores, sample = oracle_sample(d, sh)
        cpu = {"value": round(cpu_us, 1), "unit": "us/pass", "cores": cores, "kind": "oracle", "sample": sample}
    line = {
        "metric": METRIC,
        "value": round(per_pass, 2),
        "unit": "us/pass",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(us / args.steps / 1e3, 4),
        "higher_is_better": False,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded; random weights of the stated shapes)",
        "config": workload_config(world),
        "pass": {"us": round(per_pass, 2), "passes_per_s": round(1e6 / per_pass, 1),
                 "rows_V_per_s": round(sh.rows * V / per_pass * 1e6, 1),
                 "roofline_us": round(max(pass_bytes(sh) / hbm_peak / 1e3, pass_flops(sh) / tf_peak / 1e6), 2),
                 "frac_of_roofline": round(max(pass_bytes(sh) / hbm_peak / 1e3,
                                               pass_flops(sh) / tf_peak / 1e6) / per_pass, 3),
                 "frac_of_nominal_roofline": round(max(pass_bytes(sh) / NOMINAL_HBM_GBS / 1e3,
                                                       pass_flops(sh) / NOMINAL_BF16_TFLOPS / 1e6) / per_pass, 3)},
        "latency_floor": {"workload": "pass N=1 B=16 V=152064 D=3584 R=512 H=1536, CUDA graph replay",
                          "replays": floor_reps, "us_per_pass": round(floor_us, 2),
                          "median_us_single_replay": round(floor_med, 2)},
        "multipass": {"workload": "fixpoint N=64 B=16 V=152064 D=3584 R=512 H=1536, at most 8 passes",
                      "passes": fx_passes, "us_per_call": round(fx_us, 2),
                      "us_per_pass": round(fx_us / max(1, fx_passes), 2),
                      "graph_us_per_call": round(fxg_us, 2),
                      "graph_us_per_pass": round(fxg_us / max(1, fx_passes), 2)},
        "gemm_mlp": {"workload": sh.name + ", GEMM-MLP schedule (do_mlp = 0)", "us_per_pass": round(gm_us, 2)},
        "preprojected": {"workload": f"pass N={N} B={B} V={V} D={R} R={R} H={H} (E at the latent width)",
                         "us_per_pass": round(pp_us, 2),
                         "roofline_us": round(max(pass_bytes(pp_shape) / hbm_peak / 1e3,
                                                  pass_flops(pp_shape) / tf_peak / 1e6), 2)},
        "add_argmax": {"workload": "rows=480 V=152064 base+bias bf16", "us": round(aa_us, 2),
                       "GBps": round(aa_bytes / aa_us / 1e3, 1),
                       "frac": round(aa_bytes / aa_us / 1e3 / hbm_peak, 3), "peak": f"{peak_kind} {hbm_peak} GB/s",
                       "frac_of_nominal": round(aa_bytes / aa_us / 1e3 / NOMINAL_HBM_GBS, 3),
                       "rows_V_per_s": round(synth.ARGMAX_ROWS * synth.ARGMAX_V / aa_us * 1e6, 1)},
        "roofline": {"kernel": "readout_argmax_kernel", "bound": "hbm", "achieved": round(ro_achieved, 1),
                     "peak": hbm_peak, "unit": "GB/s", "frac": round(ro_achieved / hbm_peak, 3),
                     "traffic": traffic_from_profile(), "us_per_launch": round(ro_us, 2),
                     "algorithmic_bytes": readout_bytes(sh),
                     "tflops": round(readout_flops(sh) / ro_us / 1e6, 1), "peak_kind": peak_kind,
                     "frac_of_nominal": round(ro_achieved / NOMINAL_HBM_GBS, 3)},
        "cpu_baseline": cpu,
        "e2e": {"value": round(e2e_per_pass, 2), "unit": "us/pass", "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h),
                "link": {"what": "the same pinned host-to-device copies alone, back to back (four streams)",
                         "us_per_step": round(link_us, 2), "GBps": round(h2d / link_us / 1e3, 1),
                         "e2e_frac_of_link": round(link_us / (e2e_us), 3)}},
        "gpu_launches": 4 * args.steps,
        "clocks": clocks,
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            run_reference(args, world)
        return
    if world > 1:
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl")
    try:
        run_gb300(args, rank, world, local_rank)
    finally:
        if world > 1:
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
