#!/usr/bin/env python3
"""GDN chunked-prefill forward benchmark (tokens/s and % of roofline).

One step = one full forward pass (gate -> inverse -> [correction + scan] ->
fused) over the layer workload B=4, T=8192, H=32, dk=dv=128 (bf16 q/k/v, fp32
gates), inputs resident in HBM.  Prints one JSON line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the fp64 CPU oracle (the checker the CUDA path is
pinned to) on a bounded sample of the same workload, on the host cores.
With N > 1 (torchrun) every rank runs its own replica: the path shards over
independent (sequence, head) units and has no exchange step.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC_PREFIX = "GDN chunked-prefill fwd tokens/s & % roofline"
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
FLUSH_BYTES = 512 << 20          # > 129 MB L2
CLOCK_QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
               "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
               "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


def load_peaks():
    try:
        with open(PEAKS_FILE) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def shape_label(cfg):
    """The workload's shape as the metric names it, e.g. B=4,T=8192,H=32,d=128
    (packed batches: N sequences, T total tokens)."""
    d = "d=%d" % cfg.dk if cfg.dk == cfg.dv else "dk=%d,dv=%d" % (cfg.dk, cfg.dv)
    if cfg.varlen:
        return "N=%d varlen,T=%d,H=%d,%s" % (cfg.n_seqs, cfg.T, cfg.H, d)
    return "B=%d,T=%d,H=%d,%s" % (cfg.B, cfg.T, cfg.H, d)


def metric_for(cfg):
    return "%s (%s)" % (METRIC_PREFIX, shape_label(cfg))


def workload_label(cfg):
    return "GDN fwd %s %s %s" % (cfg.name, shape_label(cfg).replace(",", " "), cfg.dtype)


def input_bytes(cfg):
    """Bytes of the step's inputs resident in HBM (q, k, v, g, beta, initial state)."""
    e = 2 if cfg.dtype == "bf16" else 4
    th = cfg.total_tokens * cfg.H
    n = th * ((2 * cfg.dk + cfg.dv) * e + 8)
    if cfg.s0_std is not None:
        n += cfg.num_seqs * cfg.H * cfg.dk * cfg.dv * 4
    return n


def algorithmic_work(cfg):
    """Bytes and FLOPs the path must move / issue (per-token-head figures times
    token-heads, plus the states)."""
    e = 2 if cfg.dtype == "bf16" else 4
    th = cfg.total_tokens * cfg.H
    per_th_bytes = (2 * cfg.dk + cfg.dv) * e + cfg.dv * e + 8
    state = cfg.num_seqs * cfg.H * cfg.dk * cfg.dv * 4
    nbytes = th * per_th_bytes + state * (2 if cfg.s0_std is not None else 1)
    flops = th * (6 * cfg.dk * cfg.dv + 4 * 64 * (cfg.dk + cfg.dv))
    return nbytes, flops, per_th_bytes


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), "--query-gpu=" + CLOCK_QUERY,
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
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
            self.fh.close()

    def summary(self):
        if self.proc is None or not self.path:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        power = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows), "power_w_max": max(power) if power else None}


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def replica_throughput(total_ms, steps, tokens_per_rank, dist=None, device="cpu"):
    """Whole-job throughput of N independent replicas: the job's time is the
    slowest rank's (max over ranks), and every rank processed tokens_per_rank.
    Returns (ms per step, tokens/s of the whole job)."""
    import torch
    ws = 1
    if dist is not None:
        ws = dist.get_world_size()
        t = torch.tensor([float(total_ms)], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        total_ms = float(t.item())
    ms_per_step = total_ms / steps
    return ms_per_step, tokens_per_rank * ws / (ms_per_step * 1e-3)


def reference_arm(args, cfg):
    """The fp64 oracle on the host cores, on a bounded sample of the workload."""
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle
    from chunked_prefill_gdn_gb300.inputs import make_inputs
    inp = make_inputs(cfg.scaled(B=1), "cpu")      # one sequence of the layer batch
    heads = list(range(args.ref_heads))
    step_times = []
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        oracle.gdn_reference(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["initial_state"],
                             inp["cu_seqlens"], scale=inp["scale"], heads=heads)
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            step_times.append(dt)
    per = statistics.mean(step_times)
    token_heads = cfg.T * len(heads)
    value = token_heads / per / cfg.H                  # tokens/s of the full-width layer
    sample = "%s x %d of %d heads (all %d tokens, all %d value rows) per step" % (
        "all %d packed sequences" % cfg.n_seqs if cfg.varlen else "1 of %d sequences" % cfg.B,
        len(heads), cfg.H, cfg.T, cfg.dv)
    line = {
        "impl": "reference", "metric": metric_for(cfg), "value": value, "unit": "tokens/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": per * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": workload_label(cfg),
                   "global_batch": cfg.B, "seq_len": cfg.T, "heads": cfg.H, "head_dim": cfg.dk,
                   "parallelism": "host cores (OpenMP)", "sample": sample},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": oracle.oracle_threads(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def cpu_baseline(cfg, budget_s):
    """Oracle throughput on the host cores (tokens/s of the full-width layer) on a
    bounded sample: whole (sequence, head) units of the workload, added until the
    estimated run time reaches budget_s; the whole workload is the upper bound."""
    import oracle
    from chunked_prefill_gdn_gb300.inputs import make_inputs
    inp = make_inputs(cfg.scaled(B=1), "cpu")
    t0 = time.perf_counter()
    oracle.gdn_reference(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["initial_state"],
                         inp["cu_seqlens"], scale=inp["scale"], heads=[0])
    per_unit = max(time.perf_counter() - t0, 1e-4)       # one head of one sequence
    units = int(min(cfg.B * cfg.H, max(1, budget_s / per_unit)))
    nseq = min(cfg.B, -(-units // cfg.H))
    done = 0
    elapsed = 0.0
    for b in range(nseq):
        heads = list(range(min(cfg.H, units - done)))
        if not heads:
            break
        seq_inp = inp if b == 0 else make_inputs(cfg.scaled(B=1, seed=cfg.seed + 1000 + b), "cpu")
        t0 = time.perf_counter()
        oracle.gdn_reference(seq_inp["q"], seq_inp["k"], seq_inp["v"], seq_inp["g"], seq_inp["beta"],
                             seq_inp["initial_state"], seq_inp["cu_seqlens"], scale=seq_inp["scale"], heads=heads)
        elapsed += time.perf_counter() - t0
        done += len(heads)
    value = cfg.T * done / elapsed / cfg.H
    return {"value": value, "unit": "tokens/s", "cores": oracle.oracle_threads(), "kind": "oracle",
            "sample": "%d (%s, head) units of %d (T=%d each, all %d value rows), %.1f s" % (
                done, "packed batch of %d sequences" % cfg.n_seqs if cfg.varlen else "sequence",
                cfg.B * cfg.H, cfg.T, cfg.dv, elapsed)}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", type=int, default=1, help="workload index (1 = the layer shape)")
    ap.add_argument("--kernel", default="auto", choices=["auto", "tc", "simt"])
    ap.add_argument("--cp", default="auto", choices=["auto", "off", "force"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-qk-l2norm", action="store_true", help="skip timing the optional q/k normalisation pass")
    ap.add_argument("--no-backward", action="store_true", help="skip timing the backward pass")
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--ref-heads", type=int, default=2, help="heads per reference-arm step")
    ap.add_argument("--override", action="append", default=[],
                    help="workload field override, e.g. B=1 (profiling runs on smaller cases)")
    args = ap.parse_args()

    from chunked_prefill_gdn_gb300.inputs import CONFIGS
    cfg = CONFIGS[args.config]
    if args.override:
        kw = {}
        for item in args.override:
            key, val = item.split("=", 1)
            kw[key] = type(getattr(cfg, key))(val) if getattr(cfg, key) is not None else int(val)
        cfg = cfg.scaled(**kw)
    if args.impl == "reference":
        reference_arm(args, cfg)
        return

    import torch
    import chunked_prefill_gdn_gb300 as gdn
    from chunked_prefill_gdn_gb300 import build as lib_build
    from chunked_prefill_gdn_gb300.inputs import make_inputs

    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        dist = None
    dev = torch.device("cuda", local if ws > 1 else 0)
    torch.cuda.set_device(dev)
    if rank == 0:
        lib_build.build()
    if dist is not None:
        dist.barrier()
    gdn.load_library()

    kernel = {"auto": gdn.KERNEL_AUTO, "tc": gdn.KERNEL_TC, "simt": gdn.KERNEL_SIMT}[args.kernel]
    cp = {"auto": gdn.CP_AUTO, "off": gdn.CP_OFF, "force": gdn.CP_FORCE}[args.cp]
    opts = gdn.default_options(kernel=kernel, cp_mode=cp)
    inp = make_inputs(cfg, dev)
    q, k, v, g, beta = inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"]
    s0, cu, scale = inp["initial_state"], inp["cu_seqlens"], inp["scale"]
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    N = cfg.num_seqs
    dtc = gdn.BF16 if q.dtype == torch.bfloat16 else gdn.F32
    plan = gdn.gdn_plan_query(B, T, H, dk, dv, N, cu is not None, dtc, opts)
    out = torch.empty(B, T, H, dv, dtype=q.dtype, device=dev)
    fs = torch.empty(N, H, dk, dv, dtype=torch.float32, device=dev)
    wsp = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device=dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    ev_fb = torch.cuda.Event(enable_timing=True)
    ev_fe = torch.cuda.Event(enable_timing=True)
    ev_fb.record(stream)
    ev_fe.record(stream)
    opts.prof_begin = ev_fb.cuda_event
    opts.prof_end = ev_fe.cuda_event

    def step():
        gdn.chunk_fwd(q, k, v, g, beta, s0, cu, scale, opts=opts, out=out, final_state=fs, workspace=wsp,
                      stream=stream)

    for _ in range(max(3, args.warmup)):
        step()
    st = gdn.gdn_chunk_fwd_check(ctypes_ptr(wsp), ctypes_ptr_stream(stream))
    if st != 0:
        raise SystemExit("device check failed: %s" % gdn.gdn_status_string(st))
    torch.cuda.synchronize(dev)

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    fused_ms = []
    with ClockSampler(dev.index if dev.index is not None else 0) as clocks:
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize(dev)
        for i in range(args.steps):
            flush.fill_(i & 0xFF)                       # untimed: evict the previous step from L2
            starts[i].record(stream)
            step()
            ends[i].record(stream)
            ev_fe.synchronize()
            fused_ms.append(ev_fb.elapsed_time(ev_fe))
        torch.cuda.synchronize(dev)
        if dist is not None:
            dist.barrier()
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    ms_per_step, value = replica_throughput(sum(step_ms), args.steps, cfg.total_tokens, dist, dev)

    peaks, peak_src = load_peaks()
    nbytes, flops, per_th = algorithmic_work(cfg)
    fused_avg_ms = statistics.mean(fused_ms)
    achieved = nbytes / (fused_avg_ms * 1e-3) / 1e9
    t_hbm = nbytes / (peaks["hbm_gbs"] * 1e9)
    t_tc = flops / (peaks["bf16_tflops"] * 1e12)
    roof_ms = max(t_hbm, t_tc) * 1e3
    kname = "tc" if plan.kernel == gdn.KERNEL_TC else "simt"
    traffic = recorded_traffic(kname, workload_label(cfg), bool(plan.cp_enabled))
    launches_per_step = plan.launches

    result = {
        "metric": metric_for(cfg), "value": value, "unit": "tokens/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if cfg.dtype == "bf16" else "f32", "data": "synthetic",
        "config": {"workload": workload_label(cfg),
                   "global_batch": B * ws, "seq_len": T, "heads": H, "head_dim": dk,
                   "parallelism": "replicas" if ws > 1 else "single GPU",
                   "l2": "flushed between timed steps (%d MB write); inputs %d MB (%s L2)" % (
                       FLUSH_BYTES >> 20, input_bytes(cfg) // 10 ** 6,
                       "exceed" if input_bytes(cfg) > 129 * 10 ** 6 else "fit in"),
                   "fused_kernel": kname, "cp": bool(plan.cp_enabled)},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": achieved / peaks["hbm_gbs"], "traffic": traffic,
                     "kernel": "fused output pass (%s)" % kname, "kernel_ms": fused_avg_ms,
                     "alg_bytes_per_launch": nbytes, "peak_source": peak_src},
        "path_roofline": {"roofline_ms": roof_ms, "t_hbm_ms": t_hbm * 1e3, "t_tensor_ms": t_tc * 1e3,
                          "measured_ms": ms_per_step, "frac": roof_ms / ms_per_step,
                          "alg_bytes": nbytes, "alg_flops": flops, "peak_source": peak_src},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks.summary(),
    }
    if not args.no_qk_l2norm:
        result["qk_l2norm"] = qk_l2norm_measure(gdn, torch, q, k, flush, stream, peaks, peak_src)
    if not args.no_backward:
        result["backward"] = backward_measure(gdn, torch, inp, cfg, flush, stream)
    if not args.no_e2e:
        result["e2e"] = e2e_measure(gdn, torch, inp, cfg, opts, dev, args)
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(cfg, args.cpu_budget)
    if rank == 0:
        print(json.dumps(result), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def ctypes_ptr(t):
    import ctypes
    return ctypes.c_void_p(t.data_ptr())


def ctypes_ptr_stream(s):
    import ctypes
    return ctypes.c_void_p(s.cuda_stream)


TRAFFIC_FILE = os.path.join(ROOT, "profiles", "fused_pass_traffic.json")


def recorded_traffic(kname, workload, cp):
    """DRAM bytes per launch of the fused output pass from an ncu capture of
    this exact kernel source on this workload (profiles/fused_pass_traffic.json,
    one record per (kernel, source, workload)); None when no such capture
    exists, e.g. after the kernel changed."""
    try:
        with open(TRAFFIC_FILE) as f:
            records = json.load(f)
    except (OSError, ValueError):
        return None
    sha = kernel_source_sha(kname)
    for r in records:
        if (r.get("kernel") == kname and r.get("source_sha") == sha and r.get("workload") == workload
                and bool(r.get("cp", False)) == cp):
            return r.get("dram_bytes_per_launch")
    return None


def kernel_source_sha(kname):
    import hashlib
    path = os.path.join(ROOT, "chunked_prefill_gdn_gb300", "csrc", "fused_tc.cu" if kname == "tc" else "fused_simt.cu")
    with open(path, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def qk_l2norm_measure(gdn, torch, q, k, flush, stream, peaks, peak_src, iters=10):
    """The optional q/k L2 normalisation pass (opts.qk_l2norm; not part of the
    timed step, whose inputs arrive normalised) timed alone on this workload's
    q and k: CUDA events around each launch, L2 flushed before each one.
    Algorithmic bytes: q and k read once and written once."""
    qo, ko = torch.empty_like(q), torch.empty_like(k)
    for _ in range(3):
        gdn.qk_l2norm(q, k, qo, ko, stream=stream)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(iters)]
    for i, (a, b) in enumerate(evs):
        flush.fill_((i + 7) & 0xFF)
        a.record(stream)
        gdn.qk_l2norm(q, k, qo, ko, stream=stream)
        b.record(stream)
    torch.cuda.synchronize(q.device)
    ms = statistics.mean(a.elapsed_time(b) for a, b in evs)
    nbytes = 2 * (q.numel() + k.numel()) * q.element_size()
    achieved = nbytes / (ms * 1e-3) / 1e9
    return {"kernel": "qk_l2norm_kernel (gdn_qk_l2norm)", "bound": "hbm", "kernel_ms": ms,
            "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
            "alg_bytes_per_launch": nbytes, "launches": iters, "peak_source": peak_src,
            "note": "optional step in front of the path (opts.qk_l2norm = 1); not inside the timed step"}


# FP32 CUDA-core peak of a GB300 at its maximum SM clock: 152 SMs x 128 FP32
# lanes x 2 flops (FMA) x 2.07 GHz.
FP32_ALU_TFLOPS = 152 * 128 * 2 * 2.07e9 / 1e12
# Dense tf32 tensor peak: the measured bf16 peak times the nominal tf32 / bf16
# ratio (1.1 / 2.25 PFLOP/s dense).
TF32_NOMINAL_RATIO = 1.1 / 2.25


def backward_flops(dk, dv, chunks, H):
    """Algorithmic flops of the chunked backward (2 per multiply-add), per
    (chunk, head) with C = 64: the forward pieces it needs once (K K^T, the
    triangular inverse, X = K S0, U = T B, the state update) and the backward
    products (Q K^T, Q S0, K dS, dU, dB, dM, dA, the five dK terms, the two dQ
    terms, the two dS0 terms); a short last chunk counts as a whole one."""
    C = 64
    fwd = C * C * dk + C ** 3 / 3 + C * dk * dv + C * C * dv + C * dk * dv
    bwd = (C * C * dk + 2 * C * dk * dv + 4 * C * C * dv + 3 * C * C * dk + 2 * C * dk * dv
           + C * C * dk + C * dk * dv + 2 * C * dk * dv)
    return 2.0 * (fwd + bwd) * chunks * H


def backward_measure(gdn, torch, inp, cfg, flush, stream, iters=3):
    """The backward pass (chunk_bwd: gdn_chunk_bwd, with the automatic
    sequence-parallel plan) on this workload with seeded upstream gradients:
    CUDA events around each call, L2 flushed before each.  Reported against the
    dense tf32 tensor peak for the tensor-core backward (the default; every
    product a kind::tf32 MMA), or the FP32 CUDA-core peak for the CUDA-core one."""
    from chunked_prefill_gdn_gb300.inputs import make_grad_inputs
    grads = make_grad_inputs(cfg, inp["q"].device)
    do, dsf = grads["do"], grads["d_final_state"]
    q = inp["q"]
    B, T, H, dk = q.shape
    dv = inp["v"].shape[-1]
    from chunked_prefill_gdn_gb300.seqpar import backward_segments
    segments = backward_segments(q, inp["v"]) if inp["cu_seqlens"] is None else 1

    def run(check=False):
        return gdn.chunk_bwd(q, inp["k"], inp["v"], inp["g"], inp["beta"], do, inp["initial_state"],
                             inp["cu_seqlens"], inp["scale"], dsf, stream=stream, check=check)
    run(check=True)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(iters)]
    for i, (a, b) in enumerate(evs):
        flush.fill_((i + 11) & 0xFF)
        a.record(stream)
        run()
        b.record(stream)
    torch.cuda.synchronize(q.device)
    ms = statistics.mean(a.elapsed_time(b) for a, b in evs)
    if inp["cu_seqlens"] is not None:
        lens = inp["cu_seqlens"].cpu().diff().tolist()
        chunks = sum(-(-n // 64) for n in lens)
    else:
        chunks = B * -(-T // 64)
    flops = backward_flops(dk, dv, chunks, H)
    achieved = flops / (ms * 1e-3) / 1e12
    slices = dv // 32
    passes = 1 if segments == 1 else 2
    extra = 0 if segments == 1 else 7
    if gdn.gdn_get_backward_kernel() != gdn.KERNEL_SIMT:
        seg_note = ("; with segments > 1 each sequence is cut into that many segments (forward maps and scan, "
                    "each segment's local state-gradient map by the reverse recurrence alone, the reverse "
                    "gradient scan, then the backward per segment); timed on its own, not inside the forward step")
        peak = load_peaks()[0]["bf16_tflops"] * TF32_NOMINAL_RATIO
        return {"kernel": "bwd_tc_chain_kernel + bwd_tc_chunk_kernel (gdn_chunk_bwd)", "ms": ms,
                "segments": segments, "tokens_per_s": cfg.total_tokens / (ms * 1e-3), "bound": "tensor",
                "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak, "alg_flops": flops,
                "launches": iters * ((4 if segments == 1 else 3 + 4) + extra),
                "peak_source": "measured bf16 peak x nominal tf32/bf16 ratio (1.1/2.25)",
                "note": "every product a tcgen05 kind::tf32 MMA (fp32 operands, fp32 accumulation): a chain "
                        "kernel per (sequence, head) for the state and state-gradient recurrences, then one CTA "
                        "per (chunk, head) for dq, dk, dg, dbeta; plus the sequence prep and the per-chunk "
                        "inverse" + seg_note}
    seg_note = ("; with segments > 1 each sequence is cut into that many segments (forward maps and scan, a "
                "local backward, the reverse gradient scan, the backward per segment: two backward passes); timed on "
                "its own, not inside the forward step")
    return {"kernel": "bwd_kernel + bwd_reduce_kernel (gdn_chunk_bwd)", "ms": ms, "segments": segments,
            "tokens_per_s": cfg.total_tokens / (ms * 1e-3), "bound": "alu", "achieved": achieved,
            "peak": FP32_ALU_TFLOPS, "unit": "TFLOP/s", "frac": achieved / FP32_ALU_TFLOPS,
            "alg_flops": flops,
            "launches": iters * ((3 + (4 if slices > 1 else 0)) * passes + extra),
            "peak_source": "derived: 152 SMs x 128 FP32 lanes x 2 x 2.07 GHz",
            "note": "Gram products on tcgen05 (bf16, d=128), the other products fp32 on CUDA cores; one CTA per "
                    "(32 value columns, head, sequence or segment)" + seg_note}


def e2e_measure(gdn, torch, inp, cfg, opts, dev, args):
    """Same metric through gdn_chunk_fwd_host: pinned host inputs copied in,
    the pass, o and final_state copied out, all inside the timed region."""
    import ctypes
    host = {k: (v.cpu().pin_memory() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    B, T, H, dk = host["q"].shape
    dv = host["v"].shape[-1]
    N = cfg.num_seqs
    o = torch.empty(B, T, H, dv, dtype=host["q"].dtype, pin_memory=True)
    fs = torch.empty(N, H, dk, dv, dtype=torch.float32, pin_memory=True)
    dtc = gdn.BF16 if host["q"].dtype == torch.bfloat16 else gdn.F32
    e2e_opts = gdn.default_options(kernel=opts.kernel, cp_mode=opts.cp_mode)
    nbuf = gdn.gdn_chunk_fwd_host_buffer_size(B, T, H, dk, dv, N, host["cu_seqlens"] is not None,
                                              host["initial_state"] is not None, dtc, e2e_opts)
    buf = torch.empty(nbuf, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def once():
        gdn.chunk_fwd_host(host["q"], host["k"], host["v"], host["g"], host["beta"], host["initial_state"],
                           host["cu_seqlens"], host["scale"], opts=e2e_opts, out=o, final_state=fs,
                           device_buffer=buf, stream=stream, device=dev)

    for _ in range(2):
        once()
    steps = max(3, min(args.steps, 10))
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    for _ in range(steps):
        once()
    dt = (time.perf_counter() - t0) / steps
    el = host["q"].element_size()
    h2d = sum(host[k].numel() * host[k].element_size() for k in ("q", "k", "v", "g", "beta"))
    if host["initial_state"] is not None:
        h2d += host["initial_state"].numel() * 4
    if host["cu_seqlens"] is not None:
        h2d += host["cu_seqlens"].numel() * 4
    d2h = o.numel() * el + fs.numel() * 4
    link = host_link_rates(torch, dev, max(h2d, d2h))
    copy_ms = (h2d / link["h2d_gbs"] + d2h / link["d2h_gbs"]) / 1e6
    return {"value": cfg.total_tokens / dt, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": dt * 1e3, "steps": steps,
            "api": "gdn_chunk_fwd_host (pinned host buffers, synchronous per step)",
            "link_gbs_h2d": link["h2d_gbs"], "link_gbs_d2h": link["d2h_gbs"],
            "link_gbs_both": link["both_gbs"],
            "copy_floor_ms_serial": copy_ms,
            "copy_floor_ms_overlapped": (h2d + d2h) / link["both_gbs"] / 1e6,
            "link_note": "one pinned cudaMemcpyAsync of %d MB each way (and both at once on two streams), CUDA "
                         "events, best of %d" % (link["bytes"] // 10 ** 6, link["reps"])}


def host_link_rates(torch, dev, nbytes, reps=5):
    """Plain pinned host<->device copy rates on this machine: one large
    cudaMemcpyAsync each way (torch copy_), timed with CUDA events, best of
    `reps`; and both directions at once on two streams (bytes of both / time)."""
    nbytes = int(min(max(nbytes, 64 << 20), 1 << 30))
    h_src = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    h_dst = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    d_a = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    d_b = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    s1 = torch.cuda.Stream(dev)
    s2 = torch.cuda.Stream(dev)

    def timed(fn, stream):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        best = float("inf")
        for _ in range(reps):
            torch.cuda.synchronize(dev)
            a.record(stream)
            fn()
            b.record(stream)
            torch.cuda.synchronize(dev)
            best = min(best, a.elapsed_time(b))
        return best

    with torch.cuda.stream(s1):
        h2d_ms = timed(lambda: d_a.copy_(h_src, non_blocking=True), s1)
        d2h_ms = timed(lambda: h_dst.copy_(d_a, non_blocking=True), s1)

    def both():
        ev = torch.cuda.Event()
        ev.record(s1)
        s2.wait_event(ev)
        with torch.cuda.stream(s2):
            h_dst.copy_(d_b, non_blocking=True)
        d_a.copy_(h_src, non_blocking=True)
        ev2 = torch.cuda.Event()
        ev2.record(s2)
        s1.wait_event(ev2)

    with torch.cuda.stream(s1):
        both_ms = timed(both, s1)
    return {"h2d_gbs": nbytes / h2d_ms / 1e6, "d2h_gbs": nbytes / d2h_ms / 1e6,
            "both_gbs": 2 * nbytes / both_ms / 1e6, "bytes": nbytes, "reps": reps}


if __name__ == "__main__":
    main()
