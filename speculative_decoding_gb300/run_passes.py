"""Run Jacobi passes on the synthetic model at a chosen batch and time them.

    python -m speculative_decoding_gb300.run_passes --N 64 --passes 4
    python -m speculative_decoding_gb300.run_passes --N 64 --fixpoint 8

Model dimensions B=16, V=152064, D=3584, R=512, H=1536 (overridable), weights
and activations from the seeded generators in ``synth``; each timed call
starts from the same blk.  Prints one line per repetition: microseconds per
call, and the passes a fixpoint call ran.  A small fixed launch sequence, so
that a profiler can capture one kernel of one shape with few launches before
it.
"""

import argparse

import numpy as np
import torch

from . import synth, xpress


def _bf16(bits, device):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def main(argv=None) -> None:
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--N", type=int, default=32, help="sequences in the batch")
    ap.add_argument("--B", type=int, default=16, help="block size (tokens per sequence, slot 0 included)")
    ap.add_argument("--V", type=int, default=152064)
    ap.add_argument("--D", type=int, default=3584)
    ap.add_argument("--R", type=int, default=512)
    ap.add_argument("--H", type=int, default=1536)
    ap.add_argument("--seed", type=int, default=4)
    ap.add_argument("--passes", type=int, default=1, help="single passes per call (host loop)")
    ap.add_argument("--fixpoint", type=int, default=0, help="if > 0: one xp_jacobi_fixpoint call, this many passes at most")
    ap.add_argument("--warmup", type=int, default=2, help="untimed calls first")
    ap.add_argument("--reps", type=int, default=3, help="timed calls")
    args = ap.parse_args(argv)

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    sh = synth.PassShape(f"N={args.N} B={args.B}", args.N, args.B, args.V, args.D, args.R, args.H, args.seed)
    d = synth.pass_inputs(sh)
    w = {k: _bf16(d[k], dev) for k in ("E", "W_lat", "Wg", "Wu", "Wd", "hcache", "base")}
    W2t = _bf16(np.ascontiguousarray(d["W2"].T), dev)
    L = torch.from_numpy(d["L"]).to(dev)
    am1 = torch.from_numpy(d["am1"]).to(dev)
    blk0 = torch.from_numpy(d["blk"]).to(dev)
    blk = blk0.clone()
    ws = xpress.workspace(xpress.jacobi_workspace_size(args.N, args.B, args.V, args.D, args.R, args.H), dev)
    passes = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream()

    def call():
        blk.copy_(blk0)
        if args.fixpoint > 0:
            xpress.jacobi_fixpoint(blk, am1, w["hcache"], w["E"], w["W_lat"], L, w["Wg"], w["Wu"], w["Wd"], W2t,
                                   w["base"], ws, passes, max_passes=args.fixpoint)
        else:
            for _ in range(args.passes):
                xpress.jacobi_pass(blk, am1, w["hcache"], w["E"], w["W_lat"], L, w["Wg"], w["Wu"], w["Wd"], W2t,
                                   w["base"], ws)

    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize()
    for r in range(args.reps):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        call()
        e1.record(stream)
        e1.synchronize()
        line = f"N={args.N} B={args.B}: {e0.elapsed_time(e1) * 1e3:.1f} us per call"
        if args.fixpoint > 0:
            line += f", {int(passes.item())} passes"
        else:
            line += f", {args.passes} passes"
        print(line, flush=True)
    if xpress.read_error(ws) != 0:
        raise RuntimeError("device-side error bits set")


if __name__ == "__main__":
    main()
