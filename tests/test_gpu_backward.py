"""GPU parity of the backward pass (gdn_chunk_bwd through the C ABI) against the
oracle's gradients: oracle/backward.py, whose token-level form is pinned to
central finite differences of the forward oracle and whose chunked form is
pinned to the token-level one (test_oracle_backward.py).

Bar: relative L2 error <= 5e-3 (the forward's) and max-abs error <= 2e-2 times
max(1, max |reference|) for every gradient — the gradients reach tens, so the
forward's absolute 2e-2 is applied relative to their scale.  Inputs are
bf16- or fp32-exact on both sides.  The tensor-core backward (the default)
reads its fp32 operands as tf32 (a CPU simulation of that rounding puts every
gradient near 4e-4 relative); the CUDA-core backward computes in fp32 (~1e-7)."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from oracle.backward import gdn_backward_chunked, gdn_backward_reference
import chunked_prefill_gdn_gb300 as gdn
from chunked_prefill_gdn_gb300 import build as gdn_build
from chunked_prefill_gdn_gb300.inputs import CONFIGS, make_grad_inputs, make_inputs

from gpu_helpers import errors, to_device

pytestmark = pytest.mark.gpu

NAMES = ("dq", "dk", "dv", "dg", "dbeta", "d_initial_state")
REL_L2 = 5e-3
MAX_ABS_REL = 2e-2


@pytest.fixture(scope="module", autouse=True)
def lib():
    gdn_build.build()
    return gdn.load_library()


def check(name, got, ref):
    got = oracle.to_f64(got).reshape(ref.shape)
    assert np.isfinite(got).all(), "%s has non-finite values" % name
    rel, mab = errors(got, ref)
    bound = MAX_ABS_REL * max(1.0, float(np.abs(ref).max()))
    path = os.environ.get("GDN_BWD_MARGINS")
    if path:   # the margins of every checked gradient, absolute error included
        with open(path, "a") as f:
            f.write(json.dumps({"test": os.environ.get("PYTEST_CURRENT_TEST", "").split(" ")[0], "grad": name,
                                "rel_l2": rel, "max_abs": mab, "max_ref": float(np.abs(ref).max()),
                                "max_abs_bound": bound}) + "\n")
    assert rel <= REL_L2 and mab <= bound, "%s: rel-L2 %.3e (tol %.1e), max-abs %.3e (tol %.2e)" % (
        name, rel, REL_L2, mab, bound)


def run_bwd(inp, grads, **kw):
    out = gdn.chunk_bwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], grads["do"], inp.get("initial_state"),
                        inp.get("cu_seqlens"), inp["scale"], grads.get("d_final_state"), check=True, **kw)
    torch.cuda.synchronize()
    return out


def reference(inp, grads):
    return gdn_backward_reference(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp.get("initial_state"),
                                  inp.get("cu_seqlens"), scale=inp["scale"], do=grads["do"],
                                  d_final_state=grads.get("d_final_state"))


def with_initial_state(inp, std=0.1, seed=77):
    cfg = inp["config"]
    gen = torch.Generator().manual_seed(seed)
    N = inp["cu_seqlens"].numel() - 1 if inp.get("cu_seqlens") is not None else cfg.B
    out = dict(inp)
    out["initial_state"] = std * torch.randn(N, cfg.H, cfg.dk, cfg.dv, generator=gen)
    return out


def packed_case(lens, H, dk, dv, dtype, seed):
    """Packed sequences of the given lengths (zero and one allowed)."""
    cfg = CONFIGS[0].scaled(B=1, T=int(sum(lens)), H=H, dk=dk, dv=dv, dtype=dtype, seed=seed, gate="decay",
                            a_range=(-3.0, -1.0))
    inp = make_inputs(cfg, "cpu")
    cu = torch.zeros(len(lens) + 1, dtype=torch.int32)
    cu[1:] = torch.tensor(lens).cumsum(0).to(torch.int32)
    inp["cu_seqlens"] = cu
    inp = with_initial_state(inp, seed=seed)
    gen = torch.Generator().manual_seed(seed + 5)
    grads = dict(do=torch.randn(1, cfg.T, H, dv, generator=gen).to(inp["q"].dtype),
                 d_final_state=0.1 * torch.randn(len(lens), H, dk, dv, generator=gen))
    return inp, grads


def batched_case(cfg, s0=True):
    inp = make_inputs(cfg, "cpu")
    if s0:
        inp = with_initial_state(inp, seed=cfg.seed + 3)
    return inp, make_grad_inputs(cfg, "cpu")


CASES = {
    # tiny fp32 workload, dk = dv = 32: one slice, no reduction
    "tiny_f32": lambda: batched_case(CONFIGS[0]),
    # layer head sizes (four 32-column slices), a ragged last chunk (200 = 3 x 64 + 8)
    "layer_ragged_bf16": lambda: batched_case(CONFIGS[1].scaled(B=2, T=200, H=2)),
    # packed: an empty sequence, a one-token sequence, chunk-aligned and ragged ones
    "varlen_edges_f32": lambda: packed_case([70, 0, 1, 130, 64], H=3, dk=64, dv=32, dtype="f32", seed=21),
    # dk 32 / dv 64 (two slices), no initial state
    "dk32_dv64_bf16": lambda: batched_case(CONFIGS[1].scaled(B=3, T=100, H=2, dk=32, dv=64), s0=False),
}


@pytest.fixture
def bwd_kernel(request):
    """Selects the backward's kernels for one test, then restores the default."""
    gdn.gdn_set_backward_kernel(request.param)
    yield request.param
    gdn.gdn_set_backward_kernel(gdn.KERNEL_AUTO)


@pytest.mark.parametrize("bwd_kernel", [gdn.KERNEL_TC, gdn.KERNEL_SIMT], ids=["tc", "simt"], indirect=True)
@pytest.mark.parametrize("name", list(CASES))
def test_backward_matches_oracle(name, bwd_kernel):
    inp, grads = CASES[name]()
    ref = reference(inp, grads)
    got = run_bwd(to_device(inp), {k: v.cuda() for k, v in grads.items()})
    for n, x, r in zip(NAMES, got, ref):
        check("%s/%s" % (name, n), x, r)


@pytest.mark.parametrize("name", ["layer_ragged_bf16", "varlen_edges_f32", "dk32_dv64_bf16"])
def test_state_grad_alone_equals_backward(name):
    """gdn_chunk_state_grad (the reverse recurrence alone, which the
    sequence-parallel backward uses for each segment's local map) gives the
    tensor-core backward's d_initial_state bit for bit."""
    inp, grads = CASES[name]()
    d_inp, d_grads = to_device(inp), {k: v.cuda() for k, v in grads.items()}
    gdn.gdn_set_backward_kernel(gdn.KERNEL_TC)
    full = run_bwd(d_inp, d_grads)[5]
    alone = gdn.chunk_state_grad(d_inp["q"], d_inp["k"], d_inp["g"], d_inp["beta"], d_grads["do"],
                                 d_inp.get("cu_seqlens"), d_inp["scale"], d_grads.get("d_final_state"), check=True)
    torch.cuda.synchronize()
    assert torch.equal(full, alone)


def test_backward_of_zero_upstream_is_zero():
    inp, grads = batched_case(CONFIGS[1].scaled(B=1, T=130, H=2))
    grads = {k: torch.zeros_like(v) for k, v in grads.items()}
    for x in run_bwd(to_device(inp), {k: v.cuda() for k, v in grads.items()}):
        assert torch.count_nonzero(x).item() == 0


def test_backward_is_deterministic():
    """Partials are added in a fixed order: two calls agree bit for bit."""
    inp, grads = batched_case(CONFIGS[1].scaled(B=2, T=300, H=4))
    d_inp, d_grads = to_device(inp), {k: v.cuda() for k, v in grads.items()}
    a = run_bwd(d_inp, d_grads)
    b = run_bwd(d_inp, d_grads)
    for n, x, y in zip(NAMES, a, b):
        assert torch.equal(x, y), n


def test_backward_reports_bad_cu_seqlens():
    """A decreasing cu_seqlens is caught on the device (each CTA checks its own
    sequence's bounds before any access) and reported by the check call."""
    inp, grads = packed_case([40, 40, 40], H=2, dk=32, dv=32, dtype="f32", seed=3)
    inp["cu_seqlens"] = torch.tensor([0, 50, 40, 120], dtype=torch.int32)
    with pytest.raises(gdn.GdnError) as ei:
        run_bwd(to_device(inp), {k: v.cuda() for k, v in grads.items()})
    assert ei.value.status == 5


def test_backward_full_layer_sampled():
    """The full layer workload (B=4, T=8192, H=32, dk=dv=128, bf16) in one call;
    three (sequence, head) pairs are checked against the chunked oracle over
    their whole 8192 tokens."""
    cfg = CONFIGS[1]
    inp = make_inputs(cfg, "cuda")
    grads = make_grad_inputs(cfg, "cuda")
    got = run_bwd(inp, grads)
    for n, h in [(0, 0), (2, 17), (3, 31)]:
        sl = lambda t: t[n:n + 1, :, h:h + 1].cpu()
        ref = gdn_backward_chunked(sl(inp["q"]), sl(inp["k"]), sl(inp["v"]), sl(inp["g"]), sl(inp["beta"]), None,
                                   None, scale=inp["scale"], do=sl(grads["do"]),
                                   d_final_state=grads["d_final_state"][n:n + 1, h:h + 1].cpu())
        for name, x, r in zip(NAMES, got, ref):
            x = x[n:n + 1, h:h + 1] if name == "d_initial_state" else x[n:n + 1, :, h:h + 1]
            check("layer n=%d h=%d %s" % (n, h, name), x.cpu(), r)


@pytest.mark.parametrize("name", ["tiny_f32", "layer_bf16"])
def test_autograd_entry_matches_oracle(name):
    """chunk_gated_delta_rule under autograd: loss.backward() through the
    forward and backward kernels gives the oracle's gradients for q, k, v, g,
    beta and the initial state (bf16 gradients carry one more rounding)."""
    cfg = CONFIGS[0] if name == "tiny_f32" else CONFIGS[1].scaled(B=1, T=150, H=2)
    inp = with_initial_state(make_inputs(cfg, "cpu"), seed=9)
    names = ("q", "k", "v", "g", "beta", "initial_state")
    leaves = {n: inp[n].cuda().clone().requires_grad_() for n in names}
    o, sf = gdn.chunk_gated_delta_rule(leaves["q"], leaves["k"], leaves["v"], leaves["g"], leaves["beta"],
                                       scale=inp["scale"], initial_state=leaves["initial_state"],
                                       output_final_state=True)
    gen = torch.Generator().manual_seed(4)
    w_o = torch.randn(o.shape, generator=gen).to(o.dtype)
    w_s = 0.1 * torch.randn(sf.shape, generator=gen)
    loss = (o.float() * w_o.cuda().float()).sum() + (sf * w_s.cuda()).sum()
    loss.backward()
    torch.cuda.synchronize()
    ref = gdn_backward_reference(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["initial_state"], None,
                                 scale=inp["scale"], do=w_o, d_final_state=w_s)
    for n, r in zip(names, ref):
        assert leaves[n].grad is not None and leaves[n].grad.dtype == leaves[n].dtype, n
        check("%s/%s" % (name, n), leaves[n].grad.float().cpu(), r)


# ---------------------------------------------- sequence-parallel backward

def test_grad_scan_walks_back():
    """gdn_state_grad_scan: out[R-1] = ds_last, out[r] = out[r+1] M(r+1)^T +
    ds*(r+1), in the stored (transposed) layout of states and maps."""
    R, N, H, d = 4, 2, 3, 32
    g = torch.Generator().manual_seed(3)
    ds_star = 0.1 * torch.randn(R, N, H, d, d, generator=g)
    m = torch.eye(d).expand(R, N, H, d, d) * 0.9 + 0.02 * torch.randn(R, N, H, d, d, generator=g)
    last = torch.randn(N, H, d, d, generator=g)
    out = gdn.state_grad_scan(ds_star.cuda(), m.cuda().contiguous(), last.cuda())
    torch.cuda.synchronize()
    # math layout: stored X[j][i] = S[i][j], stored M_st[b][a] = M[a][b]
    S = lambda x: x.double().transpose(-1, -2)
    Mm = lambda x: x.double().transpose(-1, -2)
    ref = [None] * R
    Y = S(last)
    ref[R - 1] = Y
    for r in range(R - 2, -1, -1):
        Y = Y @ Mm(m[r + 1]).transpose(-1, -2) + S(ds_star[r + 1])
        ref[r] = Y
    got = out.double().cpu().transpose(-1, -2)
    np.testing.assert_allclose(got.numpy(), torch.stack(ref).numpy(), rtol=1e-4, atol=1e-5)


@pytest.mark.parametrize("dtype,d,segments", [("f32", 64, 4), ("bf16", 128, 5)])
def test_segmented_backward_matches_oracle(dtype, d, segments):
    """The backward with every sequence cut into segments (forward maps, start
    states by scan, a local backward per segment, end gradients by the reverse
    scan, the backward per segment) against the oracle's gradients."""
    cfg = CONFIGS[1].scaled(B=2, T=700, H=2, dk=d, dv=d, dtype=dtype, s0_std=0.05)
    inp = make_inputs(cfg, "cpu")
    grads = make_grad_inputs(cfg, "cpu")
    dev = to_device(inp)
    got = run_bwd(dev, {k: v.cuda() for k, v in grads.items()}, segments=segments)
    ref = reference(inp, grads)
    for name, x, r in zip(NAMES, got, ref):
        check(name, x, r)


def test_segmented_backward_long_sequence_matches_unsegmented():
    """One long sequence with few heads (the shape whose backward runs on few
    CTAs): the automatic plan splits it, and its gradients agree with the
    whole-sequence backward within the backward's bar.  (Not bit for bit: the
    segments' start states come from the forward's tcgen05 correction pass,
    with its bf16 operands, where the whole-sequence backward recomputes every
    state in fp32; the two differ by ~1e-3 relative.)"""
    cfg = CONFIGS[2].scaled(T=16384, H=2, zero_gate_heads=(0,))
    inp = to_device(make_inputs(cfg, "cpu"))
    grads = {k: v.cuda() for k, v in make_grad_inputs(cfg, "cpu").items()}
    from chunked_prefill_gdn_gb300.seqpar import backward_segments
    assert backward_segments(inp["q"], inp["v"]) > 1
    seg = run_bwd(inp, grads)
    whole = run_bwd(inp, grads, segments=1)
    for name, a, b in zip(NAMES, seg, whole):
        check(name, a, oracle.to_f64(b))
