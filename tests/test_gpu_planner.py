"""The auto-CP planner on the GPU: its plan, under the measured cost table,
against a sweep of forced segment counts on the two workloads that split
(one long sequence with 8 heads; the 1M-token sliding-window mix with 16
heads).  The talk's auto-CP paragraph derives the segment length from a cost
model with lambdas measured on the hardware; the bar here is that the plan it
picks runs within 5% of the best segment count in the sweep."""
import json
import os
import statistics

import pytest
import torch

import chunked_prefill_gdn_gb300 as gdn
from chunked_prefill_gdn_gb300.inputs import CONFIGS, make_inputs

pytestmark = pytest.mark.gpu

FLUSH_BYTES = 512 << 20


def timed_ms(inp, opts, flush, reps=7):
    ws = gdn.workspace_for(inp["q"], inp["v"], inp["cu_seqlens"], opts)

    def run():
        gdn.chunk_fwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["initial_state"],
                      inp["cu_seqlens"], inp["scale"], opts=opts, workspace=ws)
    run()
    run()
    stream = torch.cuda.current_stream()
    times = []
    for i in range(reps):
        flush.fill_(i & 0xFF)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        run()
        b.record(stream)
        b.synchronize()
        times.append(a.elapsed_time(b))
    st = gdn.gdn_chunk_fwd_check(gdn._ptr(ws), torch.cuda.current_stream().cuda_stream)
    assert st == 0, gdn.gdn_status_string(st)
    return statistics.median(times)


@pytest.mark.parametrize("idx", [2, 4])
def test_auto_plan_within_5pct_of_the_best_swept(idx):
    cfg = CONFIGS[idx]
    inp = make_inputs(cfg, "cuda")
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    B, T, H, dk = inp["q"].shape
    info = gdn.gdn_plan_query(B, T, H, dk, dk, B, 0, gdn.BF16, gdn.default_options())
    assert info.cp_enabled == 1
    nc = -(-T // 64)
    t_auto = timed_ms(inp, gdn.default_options(), flush)
    ns_auto = -(-nc // info.chunks_per_segment)
    sweep = sorted({2, 4, 8, 12, 16, 24, 32, 48, max(2, ns_auto // 2), ns_auto, 2 * ns_auto})
    results = {}
    for ns in sweep:
        L = -(-nc // ns)
        results[ns] = timed_ms(inp, gdn.default_options(cp_mode=gdn.CP_FORCE, chunks_per_segment=L), flush)
    best_ns = min(results, key=results.get)
    path = os.environ.get("GDN_PLANNER_SWEEP")
    if path:
        c = gdn.gdn_get_plan_costs()
        with open(path, "a") as f:
            f.write(json.dumps({"workload": idx, "name": cfg.name, "auto_segments": ns_auto,
                                "auto_chunks_per_segment": info.chunks_per_segment, "auto_ms": t_auto,
                                "sweep_ms": {str(k): v for k, v in results.items()}, "best_segments": best_ns,
                                "costs_us": [c.chunk_step_us, c.state_step_us, c.scan_step_us, c.pass_us]}) + "\n")
    assert t_auto <= 1.05 * results[best_ns], (
        "auto plan (%d segments of %d chunks) %.3f ms; best swept %d segments %.3f ms; sweep %s" % (
            ns_auto, info.chunks_per_segment, t_auto, best_ns, results[best_ns],
            {k: round(v, 3) for k, v in results.items()}))
