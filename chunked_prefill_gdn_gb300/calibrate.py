"""Measures the auto-CP planner's step costs on the GPU at hand.

The intra-card sequence-parallel paragraph of the FlashQLA talk
"Qwen系列模型线性注意力高性能优化实践" models a split sequence as
T = lambda1 L + lambda2 N / L and takes the lambdas from the hardware.  The
library's planner uses the wave-aware form of that model (gdn_plan_costs in
include/gdn.h); this module times the library's own passes through the C ABI,
with CUDA events on the launching stream, and fits the four costs:

  chunk_step_us  slope of the fused output pass over the chunk count, one full
                 wave of (sequence, head) units, CP off
  state_step_us, scan_step_us, pass_us
                 least squares of the correction stage (correction pass + scan)
                 over forced segment lengths, on one long sequence whose heads
                 all need correction matrices: time = state_step * (waves x
                 longest item) + scan_step * (segments - 1) + pass

The step counts of every measured plan are read back from the workspace (the
device planner may merge segments), so the fit uses the plan that ran.

    python -m chunked_prefill_gdn_gb300.calibrate [out.json]

writes the table as JSON; placed at chunked_prefill_gdn_gb300/plan_costs.json
it is what the package hands the library when it loads it.
"""
from __future__ import annotations

import datetime
import json
import statistics
import sys

import numpy as np
import torch

from . import (CP_FORCE, CP_OFF, STAGE_CORRECTION, STAGE_FUSED, STAGE_INVERSE, STAGE_PREP, chunk_fwd,
               default_options, gdn_plan_query, gdn_workspace_query, BF16, workspace_for)
from .inputs import CONFIGS, make_inputs

FLUSH_BYTES = 512 << 20


def _timed(fn, flush, reps):
    """Median over reps of one call, CUDA events on the current stream, the L2
    flushed (a write larger than L2) before each."""
    stream = torch.cuda.current_stream()
    times = []
    for i in range(reps):
        flush.fill_(i & 0xFF)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        b.synchronize()
        times.append(a.elapsed_time(b) * 1e3)   # microseconds
    return statistics.median(times)


def _run(inp, opts, ws):
    return chunk_fwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["initial_state"], inp["cu_seqlens"],
                     inp["scale"], opts=opts, workspace=ws)


def _num_items(inp, ws, opts):
    q = inp["q"]
    B, T, H, dk = q.shape
    lay = gdn_workspace_query(B, T, H, dk, inp["v"].shape[-1], B, 0, BF16, opts)
    torch.cuda.synchronize()
    return ws[lay.num_items:lay.num_items + 16].view(torch.int32).cpu().tolist()


def measure(device="cuda", reps=5, verbose=False):
    dev = torch.device(device)
    if dev.index is None:
        dev = torch.device("cuda", torch.cuda.current_device())
    torch.cuda.set_device(dev)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    pre = STAGE_PREP | STAGE_INVERSE

    # ---- chunk_step_us: the output pass over one full wave of units, CP off
    H = 8
    B = -(-sms // H)
    fused_points = []
    for nc in (32, 64, 96):
        cfg = CONFIGS[1].scaled(B=B, T=64 * nc, H=H)
        inp = make_inputs(cfg, dev)
        o_ws = default_options(cp_mode=CP_OFF)
        ws = workspace_for(inp["q"], inp["v"], None, o_ws)
        _run(inp, default_options(cp_mode=CP_OFF, stages=pre), ws)
        only = default_options(cp_mode=CP_OFF, stages=STAGE_FUSED)
        _run(inp, only, ws)
        fused_points.append((nc, _timed(lambda: _run(inp, only, ws), flush, reps)))
        del inp, ws
    x = np.array([p[0] for p in fused_points], dtype=np.float64)
    y = np.array([p[1] for p in fused_points], dtype=np.float64)
    chunk_step, fused_fixed = np.polyfit(x, y, 1)

    # ---- the correction stage: one sequence, every head with alpha == 1
    nc = 1024
    cfg = CONFIGS[2].scaled(T=64 * nc, H=H, zero_gate_heads=tuple(range(H)))
    inp = make_inputs(cfg, dev)
    units = H
    rows, rhs, corr_points = [], [], []
    max_ns = max(3, min(64, (sms + 3 * units) // (2 * units)))   # pass 1 stays within one wave
    for ns in sorted({3, 4, 6, 8, max(3, max_ns // 2), max_ns}):
        L = -(-nc // ns)
        o_ws = default_options(cp_mode=CP_FORCE, chunks_per_segment=L)
        ws = workspace_for(inp["q"], inp["v"], None, o_ws)
        _run(inp, default_options(cp_mode=CP_FORCE, chunks_per_segment=L, stages=pre), ws)
        only = default_options(cp_mode=CP_FORCE, chunks_per_segment=L, stages=STAGE_CORRECTION)
        _run(inp, only, ws)
        t = _timed(lambda: _run(inp, only, ws), flush, reps)
        items2, items1 = _num_items(inp, ws, o_ws)[:2]
        ns_eff = items2 // units                       # every head split alike
        L_eff = -(-nc // ns_eff)
        waves1 = -(-items1 // sms)
        rows.append([waves1 * L_eff, ns_eff - 1, 1.0])
        rhs.append(t)
        corr_points.append({"segments": ns_eff, "chunks_per_segment": L_eff, "pass1_items": items1, "us": t})
        del ws
    sol, *_ = np.linalg.lstsq(np.array(rows), np.array(rhs), rcond=None)
    state_step, scan_step, pass_fixed = (float(v) for v in sol)

    costs = {"chunk_step_us": float(chunk_step), "state_step_us": max(state_step, 1e-3),
             "scan_step_us": max(scan_step, 0.0), "pass_us": max(pass_fixed, 0.0)}
    out = {"device": torch.cuda.get_device_name(dev), "sm_count": sms,
           "measured_utc": datetime.datetime.now(datetime.timezone.utc).isoformat(timespec="seconds"),
           "costs": costs,
           "fit": {"fused_pass": {"points_chunks_us": fused_points, "fixed_us": float(fused_fixed),
                                  "units": B * H},
                   "correction_stage": {"points": corr_points, "units": units, "chunks": nc}},
           "method": "CUDA events around single stages of gdn_chunk_fwd (opts.stages), L2 flushed, median of %d"
                     % reps}
    if verbose:
        print(json.dumps(out, indent=1))
    return out


def main(argv):
    out = measure(verbose=True)
    if len(argv) > 1:
        with open(argv[1], "w") as f:
            json.dump(out, f, indent=1)
            f.write("\n")


if __name__ == "__main__":
    main(sys.argv)
