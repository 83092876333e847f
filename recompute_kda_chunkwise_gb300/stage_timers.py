"""Per-stage cycle counts of the tensor-core kernels (tracing build).

    python -m recompute_kda_chunkwise_gb300.stage_timers [--workload NAME] [--iters N]

Builds the library with the kernels' stage timers compiled in
(``build.build(stage_timers=True)``, a separate ``_build_stage_timers``
directory; the default library is untouched), runs kda_fwd + kda_bwd of one
seeded workload N times on cuda:0 and prints, per kernel and per CTA role, the
mean clock64 cycles of each stage per chunk step, from the last iteration.

Thread 0 of every CTA reads clock64 at each stage mark and adds the cycles since
its previous mark to that stage (shared-memory counters, written out once when
the CTA exits). Each mark closes the stage it names, so waits are counted in
the stage that ends with them. The marks add a few instructions per stage to
thread 0; the kernels run somewhat slower in the tracing build, so compare the
shares, not the absolute times.

Roles: forward main CTAs (one per (sequence, head) item) and helper CTAs
(split mode, the spare SMs); backward reverse CTAs and helper CTAs (split
mode) or reverse CTAs that rebuild inline.
"""
from __future__ import annotations

import argparse
import ctypes

import numpy as np
import torch

from . import build as kbuild
from . import kda as K
from .inputs import WORKLOADS, make_inputs

ROWS = 512  # CTA rows of the device arrays (kStageCtas)

FWD_STAGES = ["state update, output", "loop top", "q/k/g TMA wait", "row norms", "gate, cumulative decay",
              "block references", "operand tiles", "Abar|M tf32 rounds", "Abar, M readout", "inverse",
              "v -> fp16, W/U products", "-W tile", "helper hand-off stores", "handed chunk wait",
              "U~ and H^T part of O", "Kbar^T U~ and M U~", "next handed chunk fetch"]
BWD_STAGES = ["helper job claim", "segment hand-off wait", "checkpoint load", "next tiles issue",
              "state bulk store issue", "tiles wait", "top barrier", "norms, gate", "cumsum, operand tiles",
              "helper matrices wait", "next dO issue", "Abar/M tiles", "inverse", "W/U",
              "U~ MMA", "dU~ MMA", "U~/dU~ readout", "rebuild MMA", "state update", "dM, dU~V^T tiles",
              "state MMAs", "[E] dH, dgamma, readouts", "[D1]", "[D2]", "[F] 16x128 products",
              "dG cumsum", "norm row dots", "outputs"]


def _table(title, rows, names):
    rows = rows[rows[:, 31] > 0]
    if len(rows) == 0:
        return []
    steps = rows[:, 31].sum()
    tot = rows[:, :31].sum()
    per_cta = rows[:, :31].sum(axis=1)  # cycles each CTA spent from its first mark to its last
    out = [f"{title}: {len(rows)} CTAs, {steps / len(rows):.0f} steps per CTA, "
           f"{tot / steps:.0f} cycles per step; cycles per CTA min / mean / max "
           f"{per_cta.min() / 1e6:.1f} / {per_cta.mean() / 1e6:.1f} / {per_cta.max() / 1e6:.1f} M",
           "", "| stage | cycles per step | share |", "|---|---:|---:|"]
    for i, n in enumerate(names):
        v = rows[:, i].sum()
        if v > 0:
            out.append(f"| {n} | {v / steps:.0f} | {100 * v / tot:.1f}% |")
    return out + [""]


def measure(w, iters=3):
    """Runs kda_fwd + kda_bwd of workload w `iters` times with the tracing
    build and returns (forward rows, backward rows, (fwd ms, bwd ms) of the
    last iteration); rows are [CTA][32] cycle sums (slot 31: steps)."""
    lib_path = kbuild.build(stage_timers=True)
    if K._lib is not None and K._lib._name != lib_path:
        raise RuntimeError("the default KDA library is already loaded in this process: "
                           "run the stage timers in a process of their own")
    K.load_library(lib_path)
    lib = K._lib
    for fn in (lib.kda_fwd_stage_timers, lib.kda_bwd_stage_timers):
        fn.argtypes = [ctypes.c_void_p, ctypes.c_int]
        fn.restype = ctypes.c_int
    assert w.D == 128 and w.dtype == "bf16" and w.gates != "channel", "a KDA workload of the tensor-core kernels"
    inp = make_inputs(w, device="cuda")
    p = K.make_problem(w.total_tokens, w.num_seqs, w.H, w.D, inp["q"].dtype, inp["cu_seqlens"])
    call = [inp[n] for n in ["q", "k", "v", "g", "beta", "A_log", "dt_bias", "cu_seqlens"]]
    ws = torch.empty(K.workspace_bytes(p), dtype=torch.uint8, device="cuda")
    times = (0.0, 0.0)
    for _ in range(iters):
        torch.cuda.synchronize()
        assert lib.kda_fwd_stage_timers(None, 1) == 0 and lib.kda_bwd_stage_timers(None, 1) == 0
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        ev[0].record()
        o, ctx = K.kda_fwd(*call)
        ev[1].record()
        K.kda_bwd(*call, inp["dO"], ctx, workspace=ws)
        ev[2].record()
        torch.cuda.synchronize()
        times = (ev[0].elapsed_time(ev[1]), ev[1].elapsed_time(ev[2]))
    fb = np.zeros(ROWS * 32, dtype=np.uint64)
    bb = np.zeros(ROWS * 32, dtype=np.uint64)
    assert lib.kda_fwd_stage_timers(fb.ctypes.data, 0) == 0 and lib.kda_bwd_stage_timers(bb.ctypes.data, 0) == 0
    return fb.reshape(ROWS, 32).astype(np.float64), bb.reshape(ROWS, 32).astype(np.float64), times


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--workload", default="mbs1_8k_h96_d128_bf16")
    ap.add_argument("--iters", type=int, default=3)
    args = ap.parse_args(argv)
    w = WORKLOADS[args.workload]
    fb, bb, times = measure(w, args.iters)
    items = w.num_seqs * w.H
    lines = [f"workload {w.name}: forward {times[0]:.3f} ms, backward {times[1]:.3f} ms "
             f"(tracing build, last of {args.iters} iterations)", ""]
    lines += _table("forward main CTAs", fb[:items], FWD_STAGES)
    lines += _table("forward helper CTAs", fb[items:], FWD_STAGES)
    lines += _table("backward reverse CTAs", bb[:min(items, ROWS)], BWD_STAGES)
    lines += _table("backward helper CTAs", bb[items:], BWD_STAGES)
    print("\n".join(lines))


if __name__ == "__main__":
    main()
