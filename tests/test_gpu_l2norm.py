"""GPU parity of the q/k L2 normalisation: gdn_qk_l2norm element by element
against the oracle's fp64 normalisation, and the forward pass with
opts.qk_l2norm = 1 on un-normalised inputs against the oracle's recurrence on
the oracle-normalised q and k.

Element bar: the device sums squares in fp32 and rounds once to the output
type, so a bf16 result is within 2^-8 of the exact value relative to it (one
rounding) plus the fp32 error of the sum and the reciprocal square root; fp32
results are within 1e-5 relative.  The forward pass keeps the parity bar of the
other GPU tests (relative L2 <= 5e-3, max-abs <= 2e-2)."""
import numpy as np
import pytest
import torch

import oracle
from oracle.norm import l2_normalize, l2_normalize_backward
import chunked_prefill_gdn_gb300 as gdn
from chunked_prefill_gdn_gb300 import build as gdn_build
from chunked_prefill_gdn_gb300.inputs import CONFIGS, make_inputs

from gpu_helpers import assert_close, full_reference, gpu_run, to_device

pytestmark = pytest.mark.gpu

TOL = {"bf16": 2.0 ** -8 + 2e-6, "f32": 1e-5}
TORCH = {"bf16": torch.bfloat16, "f32": torch.float32}


@pytest.fixture(scope="module", autouse=True)
def lib():
    gdn_build.build()
    return gdn.load_library()


def raw_rows(shape, dtype, seed):
    """Rows whose norms spread over about four decades, plus a zero row and a
    row of tiny norm (where eps matters)."""
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(*shape, generator=g) * torch.exp(2.0 * torch.randn(*shape[:-1], 1, generator=g))
    flat = x.view(-1, shape[-1])
    flat[0] = 0.0
    flat[1] = 1e-4
    return x.to(TORCH[dtype])


def check_rows(y, x, dtype):
    ref = l2_normalize(oracle.to_f64(x))
    got = oracle.to_f64(y)
    err = np.abs(got - ref)
    assert np.all(err <= TOL[dtype] * np.abs(ref) + 1e-30), "max rel %.3e" % float(
        np.max(err / np.maximum(np.abs(ref), 1e-30)))


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("dk", [32, 64, 128])
def test_qk_l2norm_matches_oracle(dtype, dk):
    # 1237 tokens x 3 heads: rows not a multiple of the 32 a block takes per step
    q = raw_rows((1237, 3, dk), dtype, seed=dk).cuda()
    k = raw_rows((1237, 3, dk), dtype, seed=dk + 1).cuda()
    qn, kn = gdn.qk_l2norm(q, k)
    torch.cuda.synchronize()
    check_rows(qn, q, dtype)
    check_rows(kn, k, dtype)
    assert torch.all(qn.view(-1, dk)[0] == 0)


def test_qk_l2norm_in_place_and_one_sided():
    q = raw_rows((777, 2, 128), "bf16", seed=5).cuda()
    k = raw_rows((777, 2, 128), "bf16", seed=6).cuda()
    qn, kn = gdn.qk_l2norm(q, k)
    q2, k2 = q.clone(), k.clone()
    gdn.qk_l2norm(q2, k2, q_out=q2, k_out=k2)           # in place
    only_k = gdn.qk_l2norm(None, k)[1]                  # q absent
    torch.cuda.synchronize()
    assert torch.equal(q2, qn) and torch.equal(k2, kn) and torch.equal(only_k, kn)


def unnormalise(inp, seed):
    """Scale every q and k row by a positive factor in [0.25, 4]: the forward
    pass with qk_l2norm = 1 must undo it."""
    g = torch.Generator().manual_seed(seed)
    out = dict(inp)
    for name in ("q", "k"):
        t = inp[name]
        s = torch.exp(torch.empty(*t.shape[:-1], 1).uniform_(-1.386, 1.386, generator=g))
        out[name] = (t.float() * s.to(t.device)).to(t.dtype).contiguous()
    return out


def oracle_normalised(inp):
    ref_inp = dict(inp)
    for name in ("q", "k"):
        ref_inp[name] = l2_normalize(oracle.to_f64(inp[name]))
    return full_reference(ref_inp)


@pytest.mark.parametrize("name,cfg,kw", [
    ("tiny_f32", CONFIGS[0], {}),
    ("layer_ragged_tc", CONFIGS[1].scaled(B=2, T=1000, H=4), {}),
    ("layer_ragged_cp", CONFIGS[1].scaled(B=2, T=1000, H=4), dict(cp_mode=gdn.CP_FORCE, chunks_per_segment=5)),
    ("varlen", CONFIGS[3].scaled(T=3000, H=3, n_seqs=5), {}),
])
def test_forward_with_qk_l2norm(name, cfg, kw):
    inp = unnormalise(to_device(make_inputs(cfg, "cpu")), seed=11)
    q_before, k_before = inp["q"].clone(), inp["k"].clone()
    o_ref, sf_ref = oracle_normalised(inp)
    o, sf = gpu_run(inp, gdn.default_options(qk_l2norm=1, **kw))
    assert torch.equal(inp["q"], q_before) and torch.equal(inp["k"], k_before)   # caller's tensors untouched
    assert_close("o", oracle.to_f64(o).reshape(o_ref.shape), o_ref)
    assert_close("final_state", oracle.to_f64(sf), sf_ref)


def test_forward_qk_l2norm_is_a_no_op_on_unit_rows():
    """Inputs that are already unit-norm give the same result with and without
    the option, to within the bf16 rounding of the re-normalised copies."""
    inp = to_device(make_inputs(CONFIGS[1].scaled(B=1, T=700, H=2), "cpu"))
    o0, sf0 = gpu_run(inp, gdn.default_options())
    o1, sf1 = gpu_run(inp, gdn.default_options(qk_l2norm=1))
    assert_close("o", oracle.to_f64(o1), oracle.to_f64(o0))
    assert_close("final_state", oracle.to_f64(sf1), oracle.to_f64(sf0))


def test_host_entry_streams_with_normalisation():
    """The host-buffer entry point with opts.qk_l2norm = 1 on a problem large
    enough to go through in parts (each part normalises its own slice into its
    workspace copies) gives the device entry point's result bit for bit."""
    cfg = CONFIGS[1].scaled(B=4, T=2048, H=32)
    inp = unnormalise(make_inputs(cfg, "cpu"), seed=5)
    opts = gdn.default_options(qk_l2norm=1)
    pinned = {k: (v.pin_memory() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    o_h, sf_h = gdn.chunk_fwd_host(pinned["q"], pinned["k"], pinned["v"], pinned["g"], pinned["beta"],
                                   pinned["initial_state"], pinned["cu_seqlens"], inp["scale"], opts=opts)
    o_d, sf_d = gpu_run(to_device(inp), opts)
    assert torch.equal(o_h, o_d.cpu()) and torch.equal(sf_h, sf_d.cpu())


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("dk", [32, 64, 128])
def test_qk_l2norm_backward_matches_oracle(dtype, dk):
    """gdn_qk_l2norm_bwd element by element against the oracle's closed form,
    on rows whose norms spread over decades, a zero row and a tiny-norm row.
    fp32 arithmetic: each element within 1e-5 of its row's scale
    max|dy| / n + max|x| |x . dy| / n^3."""
    x = raw_rows((1237, 3, dk), dtype, seed=dk + 10).cuda()
    g = torch.Generator().manual_seed(dk)
    dy = torch.randn(1237, 3, dk, generator=g).cuda()
    dx = gdn.qk_l2norm_backward(x, dy)
    dy2 = dy.clone()
    gdn.qk_l2norm_backward(x, dy2, dx=dy2)                     # in place
    torch.cuda.synchronize()
    assert torch.equal(dx, dy2)
    x64, dy64 = oracle.to_f64(x), oracle.to_f64(dy)
    ref = l2_normalize_backward(x64, dy64)
    n = np.sqrt(np.sum(x64 * x64, axis=-1, keepdims=True) + 1e-6)
    row_scale = (np.abs(dy64).max(axis=-1, keepdims=True) / n +
                 np.abs(x64).max(axis=-1, keepdims=True) * np.abs(np.sum(x64 * dy64, axis=-1, keepdims=True)) / n ** 3)
    err = np.abs(oracle.to_f64(dx) - ref)
    assert np.all(err <= 1e-5 * row_scale), "max %.3e of row scale" % float(np.max(err / row_scale))


@pytest.mark.parametrize("name,cfg", [
    ("tiny_f32", CONFIGS[0]),
    ("layer_bf16", CONFIGS[1].scaled(B=1, T=150, H=2)),
])
def test_autograd_with_in_kernel_normalisation(name, cfg):
    """chunk_gated_delta_rule(use_qk_l2norm_in_kernel=True) under autograd on
    un-normalised q and k: the gradients equal the oracle's chain — exact
    normalisation, the recurrence's gradients on the normalised rows, then the
    normalisation's backward — within the parity bar (the device's normalised
    copies are rounded to the input dtype, as in the forward test above)."""
    from oracle.backward import gdn_backward_reference
    inp = unnormalise(make_inputs(cfg, "cpu"), seed=13)
    names = ("q", "k", "v", "g", "beta")
    leaves = {n: inp[n].cuda().clone().requires_grad_() for n in names}
    o, sf = gdn.chunk_gated_delta_rule(leaves["q"], leaves["k"], leaves["v"], leaves["g"], leaves["beta"],
                                       scale=inp["scale"], output_final_state=True, use_qk_l2norm_in_kernel=True)
    gen = torch.Generator().manual_seed(6)
    w_o = torch.randn(o.shape, generator=gen).to(o.dtype)
    w_s = 0.1 * torch.randn(sf.shape, generator=gen)
    ((o.float() * w_o.cuda().float()).sum() + (sf * w_s.cuda()).sum()).backward()
    torch.cuda.synchronize()
    q64, k64 = oracle.to_f64(inp["q"]), oracle.to_f64(inp["k"])
    qn, kn = l2_normalize(q64), l2_normalize(k64)
    dqn, dkn, dv, dg, db, _ = gdn_backward_reference(qn, kn, inp["v"], inp["g"], inp["beta"], None, None,
                                                     scale=inp["scale"], do=w_o, d_final_state=w_s)
    ref = dict(q=l2_normalize_backward(q64.reshape(dqn.shape), dqn), k=l2_normalize_backward(k64.reshape(dkn.shape), dkn),
               v=dv, g=dg, beta=db)
    for n in names:
        got = oracle.to_f64(leaves[n].grad).reshape(ref[n].shape)
        assert np.isfinite(got).all(), n
        rel = np.linalg.norm(got - ref[n]) / np.linalg.norm(ref[n])
        mab = np.abs(got - ref[n]).max()
        assert rel <= 5e-3 and mab <= 2e-2 * max(1.0, np.abs(ref[n]).max()), "%s %s: rel %.3e max-abs %.3e" % (
            name, n, rel, mab)
