"""Inter-card sequence parallelism on the GPU, its ranks emulated one after
another on one device (the ranks' kernels never wait on one another, so they
can run in turn): each slice's map through gdn_chunk_transition, the scan of
start states through gdn_state_scan, each slice's pass from its start state,
against the single pass over the whole sequences and against the oracle."""
import numpy as np
import pytest
import torch

import oracle
import chunked_prefill_gdn_gb300 as gdn
from chunked_prefill_gdn_gb300.inputs import CONFIGS, make_inputs

from gpu_helpers import assert_close, full_reference, gpu_run, to_device

pytestmark = pytest.mark.gpu


def _split(T, R):
    edges = [round(T * r / R) for r in range(R + 1)]
    return list(zip(edges[:-1], edges[1:]))


def test_transition_is_the_slice_map():
    """S* = the slice's end state from zero; M = its end state from the
    identity with zero values (the oracle's token recurrence)."""
    cfg = CONFIGS[1].scaled(B=2, T=300, H=3)
    inp = to_device(make_inputs(cfg, "cpu"))
    s_star, m = gdn.chunk_transition(inp["k"], inp["v"], inp["g"], inp["beta"], check=True)
    torch.cuda.synchronize()
    _, s_ref = oracle.gdn_reference(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], None, None,
                                    scale=inp["scale"])
    eye = np.broadcast_to(np.eye(128), (2, 3, 128, 128)).copy()
    _, m_ref = oracle.gdn_reference(inp["q"], inp["k"], torch.zeros(2, 300, 3, 128), inp["g"], inp["beta"], eye,
                                    None, scale=inp["scale"])
    assert_close("s_star", oracle.to_f64(s_star), s_ref)
    assert_close("m", oracle.to_f64(m), m_ref)


def test_state_scan_composes_maps():
    R, N, H, d = 4, 2, 3, 64
    g = torch.Generator().manual_seed(7)
    s_star = 0.1 * torch.randn(R, N, H, d, d, generator=g)
    m = torch.eye(d).expand(R, N, H, d, d) * 0.9 + 0.02 * torch.randn(R, N, H, d, d, generator=g)
    s0 = torch.randn(N, H, d, d, generator=g)
    out = gdn.state_scan(s_star.cuda(), m.cuda().contiguous(), s0.cuda())
    torch.cuda.synchronize()
    X = s0.double()
    ref = [X]
    for r in range(R - 1):
        X = torch.einsum("nhjm,nhmi->nhji", m[r].double(), X) + s_star[r].double()
        ref.append(X)
    np.testing.assert_allclose(out.double().cpu().numpy(), torch.stack(ref).numpy(), rtol=1e-4, atol=1e-5)


CASES = {
    "layer_bf16_3ranks": (CONFIGS[1].scaled(B=2, T=3000, H=4, s0_std=0.02), 3, None),
    "long_alpha1_4ranks": (CONFIGS[2].scaled(T=8192, H=4, zero_gate_heads=(0, 1)), 4, None),
    "fp32_d64_2ranks": (CONFIGS[0].scaled(B=3, T=701, H=2, dk=64, dv=64, s0_std=0.1), 2, None),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_emulated_ranks_match_the_single_pass(name):
    cfg, R, _ = CASES[name]
    inp = to_device(make_inputs(cfg, "cpu"))
    T = inp["q"].shape[1]
    maps, slices = [], []
    for a, b in _split(T, R):
        sl = {n: inp[n][:, a:b].contiguous() for n in ("q", "k", "v", "g", "beta")}
        slices.append(sl)
        maps.append(gdn.chunk_transition(sl["k"], sl["v"], sl["g"], sl["beta"], check=True))
    s_start = gdn.state_scan(torch.stack([s for s, _ in maps]), torch.stack([m for _, m in maps]),
                             inp["initial_state"])
    outs = []
    for r, sl in enumerate(slices):
        o, s_end = gdn.chunk_fwd(sl["q"], sl["k"], sl["v"], sl["g"], sl["beta"], s_start[r].contiguous(), None,
                                 inp["scale"], check=True)
        outs.append(o)
    torch.cuda.synchronize()
    o_par = torch.cat(outs, dim=1)
    o_one, s_one = gpu_run(inp)
    o_ref, s_ref = full_reference(inp)
    assert_close("o", oracle.to_f64(o_par).reshape(o_ref.shape), o_ref)
    assert_close("final_state", oracle.to_f64(s_end), s_ref)
    # and close to the single pass on one card (same kernels, other split points)
    assert_close("o vs one card", oracle.to_f64(o_par), oracle.to_f64(o_one), 5e-3, 2e-2)
