"""Shared helpers for the GPU parity tests: run the CUDA path through the C ABI
and compare with the fp64 oracle on the same inputs."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import chunked_prefill_gdn_gb300 as gdn
from chunked_prefill_gdn_gb300.inputs import make_inputs

# Parity bar: relative L2 error and max-abs error on o and final_state.
REL_L2 = 5e-3
MAX_ABS = 2e-2


def to_device(inp, device="cuda"):
    out = dict(inp)
    for k in ("q", "k", "v", "g", "beta", "initial_state", "cu_seqlens"):
        if out.get(k) is not None:
            out[k] = out[k].to(device).contiguous()
    return out


def gpu_run(inp, opts=None, **kw):
    o, sf = gdn.chunk_fwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp.get("initial_state"),
                          inp.get("cu_seqlens"), inp["scale"], opts=opts, check=True, **kw)
    torch.cuda.synchronize()
    return o, sf


def errors(x, ref):
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    d = x - ref
    rel = float(np.linalg.norm(d) / max(np.linalg.norm(ref), 1e-300))
    return rel, float(np.abs(d).max()) if d.size else 0.0


def assert_close(name, x, ref, rel_tol=REL_L2, abs_tol=MAX_ABS):
    rel, mab = errors(x, ref)
    assert np.isfinite(x).all(), "%s has non-finite values" % name
    assert rel <= rel_tol and mab <= abs_tol, "%s: rel-L2 %.3e (tol %.1e), max-abs %.3e (tol %.1e)" % (
        name, rel, rel_tol, mab, abs_tol)
    return rel, mab


def seq_bounds(inp):
    q = inp["q"]
    if inp.get("cu_seqlens") is not None:
        cu = inp["cu_seqlens"].cpu().numpy().astype(np.int64)
    else:
        B, T = q.shape[:2]
        cu = np.arange(B + 1, dtype=np.int64) * T
    return cu


def sampled_reference(inp, seqs, heads, rows=None):
    """Oracle on a subset, slicing on the device first so only the sampled
    sequences and heads travel to the host.  Returns (o_ref [T_sel,H_sel,dv_sel],
    sf_ref [N_sel,H_sel,dk,dv_sel], token index array)."""
    cu = seq_bounds(inp)
    flat = lambda t: t.reshape(-1, *t.shape[2:])
    idx = np.concatenate([np.arange(cu[n], cu[n + 1]) for n in seqs])
    tidx = torch.as_tensor(idx, device=inp["q"].device)
    hidx = torch.as_tensor(list(heads), device=inp["q"].device)
    take = lambda t: flat(t).index_select(0, tidx).index_select(1, hidx)
    q, k, v = take(inp["q"]), take(inp["k"]), take(inp["v"])
    g, b = take(inp["g"]), take(inp["beta"])
    if rows is not None:
        v = v[..., list(rows)]
    s0 = None
    if inp.get("initial_state") is not None:
        s0 = inp["initial_state"][list(seqs)][:, list(heads)]
        if rows is not None:
            s0 = s0[..., list(rows)]
    lens = [int(cu[n + 1] - cu[n]) for n in seqs]
    cu_sel = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    o, sf = oracle.gdn_reference(q, k, v, g, b, s0, cu_sel, scale=inp["scale"])
    return o, sf, idx


def gpu_sampled(o_gpu, sf_gpu, inp, seqs, heads, rows, idx):
    flat = o_gpu.reshape(-1, *o_gpu.shape[2:])
    tidx = torch.as_tensor(idx, device=o_gpu.device)
    o = flat.index_select(0, tidx)[:, list(heads)]
    sf = sf_gpu[list(seqs)][:, list(heads)]
    if rows is not None:
        o = o[..., list(rows)]
        sf = sf[..., list(rows)]
    return oracle.to_f64(o), oracle.to_f64(sf)


def full_reference(inp):
    return oracle.gdn_reference(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp.get("initial_state"),
                                inp.get("cu_seqlens"), scale=inp["scale"])
