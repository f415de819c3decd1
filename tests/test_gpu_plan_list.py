"""The device planner's work list against a model of it on the CPU.

The planner decides, per (sequence, head), how a sequence is cut into
segments (the talk "Qwen系列模型线性注意力高性能优化实践", intra-card CP and auto-CP
paragraphs), which segments restart from zero after a look-back window (its
sliding-window paragraph: a head whose gate is not identically one forgets an
old state after a finite number of chunks) and which take the exact
correction-matrix path (heads with alpha identically 1, windows longer than the
walk bound, or no sliding).  That is index work, so the output pass's items are
compared field by field.  The model takes the head flags and the chunk totals
from the oracle (fp64) and the segment rule, the window rule and the
correction-segment cost model as the library states them; a window decided by
floating point may differ by one chunk only where the fp64 walk sits within
fp32 rounding of ln(eps)."""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import gate
import chunked_prefill_gdn_gb300 as gdn
from chunked_prefill_gdn_gb300.inputs import CONFIGS, make_inputs

from gpu_helpers import gpu_run, seq_bounds, to_device

pytestmark = pytest.mark.gpu

C = 64
ITEM_OUTPUT, FROM_INITIAL, FROM_ZERO, FROM_SLOT, WRITE_FINAL = 1, 2, 4, 16, 32
MAX_LOOKBACK = 256


def ceil_div(a, b):
    return -(-a // b)


def walk(tot, c_begin, ln_eps, max_walk):
    """Chunks to step back from c_begin (the oracle's rule), -1 past max_walk;
    also the partial sums, for the rounding check."""
    acc, w, sums = 0.0, 0, []
    while w < c_begin:
        if w >= max_walk:
            return -1, sums
        acc += float(tot[c_begin - 1 - w])
        sums.append(acc)
        w += 1
        if acc <= ln_eps:
            break
    return w, sums


def correction_cost(ns, nc, ns0, n_m, n_s, grid, state_ratio, scan_ratio):
    ls = (nc + ns0 - 1) // ns0 + (4 if n_s > 0 else 0)
    lm = (nc + ns - 1) // ns
    it1 = n_m * (2 * ns - 3)
    it2 = n_m * ns + n_s * ns0
    return (float((it1 + grid - 1) // grid) * lm * state_ratio +
            float((it2 + grid - 1) // grid) * max(lm, ls if n_s > 0 else 0) + scan_ratio * ns)


def model_items(cu, H, flags, totals, L, ln_eps, sliding, varlen, grid):
    """Items of the output pass, in list order, and the pass-1 / scan counts."""
    N = len(cu) - 1
    ncs = [ceil_div(int(cu[n + 1]) - int(cu[n]), C) for n in range(N)]
    order = sorted(range(N), key=lambda n: (-ncs[n], n))          # longest first, stable
    units = N * H
    ns_m = 0
    if not varlen and units > 0:
        nc = ncs[0]
        ns0 = ceil_div(nc, L) if nc > L else 1
        l0 = max(1, ceil_div(nc, ns0))
        ns0 = ceil_div(nc, l0) if nc > 0 else 1
        if ns0 > 2:
            n_m = sum(1 for n in range(N) for h in range(H) if not (flags[n, h] and sliding))
            n_s = units - n_m
            if n_m > 0 and grid > 0:
                costs = gdn.gdn_get_plan_costs()
                sr = float(np.float32(costs.state_step_us) / np.float32(costs.chunk_step_us))
                cr = float(np.float32(costs.scan_step_us) / np.float32(costs.chunk_step_us))
                cand = {ns: correction_cost(ns, nc, ns0, n_m, n_s, grid, sr, cr) for ns in range(2, ns0)}
                if cand:
                    cmin = min(cand.values())
                    best = max(ns for ns, c in cand.items() if c == cmin)
                    c0 = correction_cost(ns0, nc, ns0, n_m, n_s, grid, sr, cr)
                    ns_m = best if cmin < 0.95 * c0 else 0
    max_walk = min(L, MAX_LOOKBACK)
    items, walks, n1, nscan = [], [], 0, 0
    o2 = os_ = 0
    for u in range(units):
        n, h = order[u // H], u % H
        nc = ncs[n]
        ns = ceil_div(nc, L) if nc > L else 1
        lu = max(1, ceil_div(nc, ns))
        ns = ceil_div(nc, lu) if nc > 0 else 1
        flagged = bool(flags[n, h])
        if ns_m > 0 and ns > ns_m and not (flagged and sliding):
            lu = ceil_div(nc, ns_m)
            ns = ceil_div(nc, lu)
        mpath = ns > 1 and not (flagged and sliding)
        wins = {}
        if ns > 1 and not mpath:
            for j in range(1, ns):
                wins[j] = walk(totals[n][:, h], j * lu, ln_eps, max_walk)
            mpath = any(w < 0 for w, _ in wins.values())
        for j in range(ns):
            c_begin, c_end = j * lu, min(nc, (j + 1) * lu)
            f = ITEM_OUTPUT | (WRITE_FINAL if j == ns - 1 else 0)
            c_start, slot = c_begin, -1
            if j == 0:
                f |= FROM_INITIAL
            elif mpath:
                f |= FROM_SLOT
                slot = os_ + j - 1
            else:
                w, sums = wins[j]
                c_start = c_begin - w
                f |= FROM_INITIAL if c_start == 0 else FROM_ZERO
                walks.append((o2 + j, sums))
            items.append((n, h, c_begin, c_end, c_start, f, slot))
        o2 += ns
        if mpath:
            n1 += 2 * ns - 3
            os_ += ns - 1
            nscan += 1
    return items, walks, (len(items), n1, nscan)


def lpt_reorder(items, G):
    """Packed sequences with more items than CTAs: the list reordered so that
    the fused pass's snake order (round r: item r G + c, or r G + G - 1 - c in
    odd rounds) deals it out longest first, by rounds of G, each item to the
    least-loaded group (ties: lower index), the groups with an item in the last
    round on that round's first snake positions."""
    n = len(items)
    if n <= G:
        return list(items)
    ln = [max(0, it[3] - it[4]) for it in items]
    by_rank = sorted(range(n), key=lambda i: (-ln[i], i))
    load = [0] * G
    group = [0] * n
    rounds = -(-n // G)
    for r in range(rounds):
        cta_at = sorted(range(G), key=lambda c: (load[c], c))
        for k in range(G):
            j = r * G + k
            if j < n:
                group[j] = cta_at[k]
                load[cta_at[k]] += ln[by_rank[j]]
    last = rounds - 1
    rem = n - last * G
    has = [0] * G
    for j in range(last * G, n):
        has[group[j]] = 1
    phys = [0] * G
    for c in range(G):
        before = sum(1 for m in range(c) if has[m] == has[c])
        pos = before if has[c] else rem + before
        phys[c] = G - 1 - pos if last & 1 else pos
    out = [None] * n
    for j in range(n):
        r, cp = j // G, phys[group[j]]
        out[r * G + (G - 1 - cp if r & 1 else cp)] = items[by_rank[j]]
    return out


def near_threshold(sums, ln_eps, w_dev):
    """The device's window differs from the fp64 walk only by where the running
    sum crosses ln(eps): accept it when that sum is within fp32 rounding."""
    k = min(w_dev, len(sums)) - 1
    cand = [s for s in sums[max(0, k - 1):k + 2]]
    return any(abs(s - ln_eps) <= 1e-5 * max(1.0, abs(ln_eps)) for s in cand)


CASES = {
    # one long sequence, two heads with alpha == 1 (correction matrices, the
    # segment count searched by the cost model), two decaying heads whose
    # windows exceed the walk bound of 5 chunks or fit it
    "long_L5": (CONFIGS[2].scaled(T=4133, H=4, zero_gate_heads=(0, 1)), 5, 1),
    # windows up to ~18 chunks walked in several rounds of eight lanes
    "long_L24": (CONFIGS[2].scaled(T=12000, H=4, zero_gate_heads=(0,)), 24, 1),
    # packed sequences of unequal length, longest first
    "varlen_L5": (CONFIGS[3].scaled(T=6000, H=4, n_seqs=9), 5, 1),
    # no sliding: every split head through correction matrices
    "mix_nosliding": (CONFIGS[4].scaled(T=5000, H=5, zero_gate_heads=(0, 1)), 7, 0),
    # more items than CTAs on packed sequences: the list dealt out longest first
    "varlen_many": (CONFIGS[3].scaled(T=40000, H=4, n_seqs=64), 3, 1),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_planner_work_list_matches_the_model(name):
    cfg, L, sliding = CASES[name]
    inp = to_device(make_inputs(cfg, "cpu"))
    opts = gdn.default_options(cp_mode=gdn.CP_FORCE, chunks_per_segment=L, sliding=sliding)
    ws = gdn.workspace_for(inp["q"], inp["v"], inp["cu_seqlens"], opts)
    gpu_run(inp, opts, workspace=ws)
    q, v = inp["q"], inp["v"]
    B, T, H, dk = q.shape
    cu = seq_bounds(inp)
    varlen = inp["cu_seqlens"] is not None
    N = len(cu) - 1
    dt = gdn.BF16 if q.dtype == torch.bfloat16 else gdn.F32
    info = gdn.gdn_plan_query(B, T, H, dk, v.shape[-1], N, varlen, dt, opts)
    lay = gdn.gdn_workspace_query(B, T, H, dk, v.shape[-1], N, varlen, dt, opts)
    num = ws[lay.num_items:lay.num_items + 16].view(torch.int32).tolist()
    dev = ws[lay.items:lay.items + 32 * num[0]].view(torch.int32).view(num[0], 8).cpu().numpy()

    g = oracle.to_f64(inp["g"]).reshape(-1, H)
    flags = gate.head_flags(g, cu)
    tot_all = gate.chunk_totals(g, cu, C)                          # [chunks, H], sequences in order
    totals, c0 = [], 0
    for n in range(N):
        nc = ceil_div(int(cu[n + 1]) - int(cu[n]), C)
        totals.append(tot_all[c0:c0 + nc])
        c0 += nc
    ln_eps = float(np.float32(math.log(np.float32(opts.sw_eps))))
    assert info.cp_enabled == 1
    items, walks, counts = model_items(cu, H, flags, totals, info.chunks_per_segment, ln_eps, sliding, varlen,
                                       info.grid_fused)
    if varlen:
        # (the look-back allowance below is by list position: map it through the reordering)
        pos_of = {id(it): j for j, it in enumerate(items)}
        items = lpt_reorder(items, info.grid_fused)
        moved = {pos_of[id(it)]: j for j, it in enumerate(items)}
        walks = [(moved[j], sums) for j, sums in walks]

    # every case has correction units; the sliding ones also restart segments from zero
    assert counts[1] > 0 and counts[2] > 0
    assert (not sliding) or any(it[5] & FROM_ZERO for it in items)
    assert tuple(num[:3]) == counts
    slack = {}
    for idx, sums in walks:
        slack[idx] = sums
    for i, (ref, got) in enumerate(zip(items, dev.tolist())):
        seq, head, c_begin, c_end, c_start, flg, slot = got[:7]
        assert (seq, head, c_begin, c_end, slot) == (ref[0], ref[1], ref[2], ref[3], ref[6]), (i, ref, got)
        if (c_start, flg) != (ref[4], ref[5]):
            # only a window, and only where the fp64 walk meets ln(eps) within rounding
            assert i in slack and near_threshold(slack[i], ln_eps, c_begin - c_start), (i, ref, got)
