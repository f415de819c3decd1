"""Inter-card sequence parallelism, host side: the rank bookkeeping and the
exchange of chunked_prefill_gdn_gb300.seqpar, run as gloo ranks on the CPU.
The three compute steps are the oracle's here (the fp64 token recurrence: the
map of a slice is its end state from zero with the values, and from the
identity with zero values), so every rank's slice of o and the last rank's end
state must equal the oracle's single pass over the whole sequences to
rounding.  The GPU steps are tested in tests/test_gpu_seqpar.py."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
from chunked_prefill_gdn_gb300.inputs import CONFIGS, make_inputs
from chunked_prefill_gdn_gb300.seqpar import SeqParOps, chunk_fwd_sequence_parallel


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _oracle_ops(scale):
    def transition(k, v, g, beta, cu):
        B, T, H, dk = k.shape
        N = B if cu is None else cu.numel() - 1
        _, s_star = oracle.gdn_reference(k, k, v, g, beta, None, cu, scale=scale)
        eye = np.broadcast_to(np.eye(dk), (N, H, dk, dk)).copy()
        _, m = oracle.gdn_reference(k, k, torch.zeros(B, T, H, dk, dtype=torch.float64), g, beta, eye, cu,
                                    scale=scale)
        return torch.from_numpy(s_star), torch.from_numpy(m)

    def scan(s_star, m, s0):
        # stored layout X[j][i] = S[i][j]: X(r+1) = M^T-stored(r) X(r) + X*(r)
        X = torch.zeros_like(s_star[0]) if s0 is None else s0.to(torch.float64)
        out = [X]
        for r in range(s_star.shape[0] - 1):
            X = torch.einsum("nhjm,nhmi->nhji", m[r], X) + s_star[r]
            out.append(X)
        return torch.stack(out)

    def forward(q, k, v, g, beta, s_start, cu, scale_, opts):
        o, sf = oracle.gdn_reference(q, k, v, g, beta, s_start, cu, scale=scale_)
        return torch.from_numpy(o), torch.from_numpy(sf)

    return SeqParOps(transition, scan, forward)


def _split(T, R):
    edges = [round(T * r / R) for r in range(R + 1)]
    return list(zip(edges[:-1], edges[1:]))


def _rank(rank, world, port, outdir, T):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        cfg = CONFIGS[0].scaled(B=2, T=T, H=2, dk=16, dv=16, s0_std=0.3)
        inp = make_inputs(cfg, "cpu")
        a, b = _split(T, world)[rank]
        sl = {n: inp[n][:, a:b].contiguous() for n in ("q", "k", "v", "g", "beta")}
        o, s_end = chunk_fwd_sequence_parallel(sl["q"], sl["k"], sl["v"], sl["g"], sl["beta"], inp["initial_state"],
                                               None, inp["scale"], ops=_oracle_ops(inp["scale"]))
        np.save(os.path.join(outdir, "o%d.npy" % rank), o.numpy())
        np.save(os.path.join(outdir, "s%d.npy" % rank), s_end.numpy())
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_ranks_reassemble_the_single_pass(tmp_path, world):
    T = 157                      # slices of 78/79 or 52/53 tokens: none ends on a chunk boundary
    mp.spawn(_rank, args=(world, _free_port(), str(tmp_path), T), nprocs=world, join=True)
    cfg = CONFIGS[0].scaled(B=2, T=T, H=2, dk=16, dv=16, s0_std=0.3)
    inp = make_inputs(cfg, "cpu")
    o_ref, s_ref = oracle.gdn_reference(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["initial_state"],
                                        None, scale=inp["scale"])
    o_ref = o_ref.reshape(2, T, 2, 16)
    for r, (a, b) in enumerate(_split(T, world)):
        o = np.load(tmp_path / ("o%d.npy" % r)).reshape(2, b - a, 2, 16)
        np.testing.assert_allclose(o, o_ref[:, a:b], rtol=1e-9, atol=1e-11)
    s_last = np.load(tmp_path / ("s%d.npy" % (world - 1)))
    np.testing.assert_allclose(s_last, s_ref, rtol=1e-9, atol=1e-11)
