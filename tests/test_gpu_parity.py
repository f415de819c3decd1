"""GPU parity: the CUDA path, called through the C ABI, against the fp64 oracle
on the same seeded inputs.  Bar: relative L2 <= 5e-3 and max-abs <= 2e-2 on o
and final_state.

Reduced cases keep each workload's distributions but shrink it so the oracle
finishes in seconds while still spanning many chunks, a ragged last chunk and
several segments; the full-size cases run each workload in the bench's launch
configuration and compare every element of o and final_state with the oracle
(one head at a time on the host).
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import chunked, gate
import chunked_prefill_gdn_gb300 as gdn
from chunked_prefill_gdn_gb300.inputs import CONFIGS, make_inputs

from gpu_helpers import (assert_close, full_reference, gpu_run, gpu_sampled, sampled_reference, seq_bounds,
                         to_device)

pytestmark = pytest.mark.gpu

KERNELS = {"auto": gdn.KERNEL_AUTO, "simt": gdn.KERNEL_SIMT}


def opts_for(kernel="auto", **kw):
    return gdn.default_options(kernel=KERNELS[kernel], **kw)


REDUCED = {
    "tiny": CONFIGS[0],
    "layer_ragged": CONFIGS[1].scaled(B=2, T=1000, H=4),
    "long_cp": CONFIGS[2].scaled(T=4133, H=4, zero_gate_heads=(0, 1)),
    "varlen": CONFIGS[3].scaled(T=6000, H=4, n_seqs=9),
    "mix_cp": CONFIGS[4].scaled(T=5000, H=5, zero_gate_heads=(0, 1)),
    # the same mix in fp32 (kind::tf32 kernels): look-back restarts, correction
    # matrices and the scan through the tf32 state
    "mix_cp_f32": CONFIGS[4].scaled(T=3000, H=5, zero_gate_heads=(0, 1), dtype="f32"),
}


@pytest.mark.parametrize("kernel", ["auto", "simt"])
@pytest.mark.parametrize("name", sorted(REDUCED))
@pytest.mark.parametrize("cp", ["off", "force"])
def test_reduced_parity(name, cp, kernel):
    cfg = REDUCED[name]
    inp = to_device(make_inputs(cfg, "cpu"))
    o_ref, sf_ref = full_reference(inp)
    kw = dict(cp_mode=gdn.CP_OFF) if cp == "off" else dict(cp_mode=gdn.CP_FORCE, chunks_per_segment=5)
    o, sf = gpu_run(inp, opts_for(kernel, **kw))
    B, T, H, dv = o.shape
    assert_close("o", oracle.to_f64(o).reshape(B * T, H, dv), o_ref)
    assert_close("final_state", oracle.to_f64(sf), sf_ref)


def test_cp_forced_without_sliding():
    """Every split head through correction matrices and the scan."""
    inp = to_device(make_inputs(REDUCED["mix_cp"], "cpu"))
    o_ref, sf_ref = full_reference(inp)
    o, sf = gpu_run(inp, opts_for(cp_mode=gdn.CP_FORCE, chunks_per_segment=7, sliding=0))
    assert_close("o", oracle.to_f64(o).reshape(o_ref.shape), o_ref)
    assert_close("final_state", oracle.to_f64(sf), sf_ref)


@pytest.mark.parametrize("T", [1, 63, 64, 65, 129])
def test_short_and_ragged_lengths(T):
    inp = to_device(make_inputs(CONFIGS[1].scaled(B=3, T=T, H=2, s0_std=0.02), "cpu"))
    o_ref, sf_ref = full_reference(inp)
    o, sf = gpu_run(inp)
    assert_close("o", oracle.to_f64(o).reshape(o_ref.shape), o_ref)
    assert_close("final_state", oracle.to_f64(sf), sf_ref)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_varlen_with_empty_and_tiny_sequences(dtype):
    """Packed sequences of lengths 0, 1, 64, 200 and 3 with an initial state
    (bf16: the kind::f16 kernels; fp32: the kind::tf32 fused kernel and the
    tf32-Gram inverse)."""
    lens = [0, 1, 64, 0, 200, 3, 0]
    cfg = CONFIGS[1].scaled(B=1, T=sum(lens), H=3, s0_std=0.02, dtype=dtype)
    inp = make_inputs(cfg, "cpu")
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32)
    inp["cu_seqlens"] = cu
    inp["initial_state"] = 0.02 * torch.randn(len(lens), 3, 128, 128, generator=torch.Generator().manual_seed(5))
    inp = to_device(inp)
    o_ref, sf_ref = full_reference(inp)
    o, sf = gpu_run(inp)
    assert_close("o", oracle.to_f64(o).reshape(o_ref.shape), o_ref)
    assert_close("final_state", oracle.to_f64(sf), sf_ref)
    # empty sequences hand their initial state straight through
    for n in (0, 3, 6):
        assert torch.equal(sf[n], inp["initial_state"][n])


@pytest.mark.parametrize("d", [32, 64, 128])
def test_head_sizes_fp32(d):
    cfg = CONFIGS[0].scaled(T=300, H=3, dk=d, dv=d, s0_std=0.1)
    inp = to_device(make_inputs(cfg, "cpu"))
    o_ref, sf_ref = full_reference(inp)
    o, sf = gpu_run(inp, opts_for(cp_mode=gdn.CP_FORCE, chunks_per_segment=2))
    assert_close("o", oracle.to_f64(o).reshape(o_ref.shape), o_ref)
    assert_close("final_state", oracle.to_f64(sf), sf_ref)


@pytest.mark.parametrize("cp", ["off", "force"])
@pytest.mark.parametrize("dk,dv", [(32, 32), (64, 64), (64, 128), (32, 64), (128, 32)])
def test_bf16_small_head_sizes_run_on_tcgen05(dk, dv, cp):
    """bf16 head sizes 32 and 64, and mixed ones, run on the tcgen05 kernels,
    zero-padded to 128 by the TMA (features past dk or dv read as zeros, which
    leaves the real rows and columns of the state exact); compared with the
    oracle.  With CP forced the correction matrices (dk x dk) and segment
    starts (dk x dv) go through the padded state too."""
    cfg = CONFIGS[1].scaled(B=2, T=333, H=3, dk=dk, dv=dv, s0_std=0.05)
    inp = to_device(make_inputs(cfg, "cpu"))
    info = gdn.gdn_plan_query(2, 333, 3, dk, dv, 2, 0, gdn.BF16, opts_for("auto"))
    assert info.kernel == gdn.KERNEL_TC
    kw = dict(cp_mode=gdn.CP_OFF) if cp == "off" else dict(cp_mode=gdn.CP_FORCE, chunks_per_segment=2, sliding=0)
    o_ref, sf_ref = full_reference(inp)
    o, sf = gpu_run(inp, opts_for("auto", **kw))
    assert_close("o", oracle.to_f64(o).reshape(o_ref.shape), o_ref)
    assert_close("final_state", oracle.to_f64(sf), sf_ref)


@pytest.mark.parametrize("cp", ["off", "force"])
@pytest.mark.parametrize("dk,dv", [(32, 32), (64, 64), (128, 128), (32, 128), (128, 64)])
def test_fp32_runs_on_tcgen05_tf32(dk, dv, cp):
    """fp32 inputs run on the kind::tf32 kernel (the plan reports the tcgen05
    kernel), compared with the oracle over several chunks, a ragged last chunk,
    an initial state and, with CP forced, the correction matrices and segment
    starts; and with the CUDA-core kernel on the same inputs."""
    cfg = CONFIGS[0].scaled(B=2, T=333, H=3, dk=dk, dv=dv, s0_std=0.1)
    inp = to_device(make_inputs(cfg, "cpu"))
    info = gdn.gdn_plan_query(2, 333, 3, dk, dv, 2, 0, gdn.F32, opts_for("auto"))
    assert info.kernel == gdn.KERNEL_TC
    kw = dict(cp_mode=gdn.CP_OFF) if cp == "off" else dict(cp_mode=gdn.CP_FORCE, chunks_per_segment=2, sliding=0)
    o_ref, sf_ref = full_reference(inp)
    o, sf = gpu_run(inp, opts_for("auto", **kw))
    assert_close("o", oracle.to_f64(o).reshape(o_ref.shape), o_ref)
    assert_close("final_state", oracle.to_f64(sf), sf_ref)
    o_si, sf_si = gpu_run(inp, opts_for("simt", **kw))
    assert_close("o vs CUDA-core", oracle.to_f64(o), oracle.to_f64(o_si))
    assert_close("final_state vs CUDA-core", oracle.to_f64(sf), oracle.to_f64(sf_si))


def test_unequal_head_sizes():
    cfg = CONFIGS[1].scaled(B=2, T=150, H=2, dk=128, dv=64, s0_std=0.02)
    inp = to_device(make_inputs(cfg, "cpu"))
    o_ref, sf_ref = full_reference(inp)
    o, sf = gpu_run(inp, opts_for(cp_mode=gdn.CP_FORCE, chunks_per_segment=1, sliding=0))
    assert_close("o", oracle.to_f64(o).reshape(o_ref.shape), o_ref)
    assert_close("final_state", oracle.to_f64(sf), sf_ref)


def test_resume_two_calls_equal_one():
    inp = to_device(make_inputs(CONFIGS[1].scaled(B=1, T=700, H=2), "cpu"))
    o, sf = gpu_run(inp)
    cut = 320
    a = dict(inp, q=inp["q"][:, :cut].contiguous(), k=inp["k"][:, :cut].contiguous(), v=inp["v"][:, :cut].contiguous(),
             g=inp["g"][:, :cut].contiguous(), beta=inp["beta"][:, :cut].contiguous())
    oa, sfa = gpu_run(a)
    b = dict(inp, q=inp["q"][:, cut:].contiguous(), k=inp["k"][:, cut:].contiguous(), v=inp["v"][:, cut:].contiguous(),
             g=inp["g"][:, cut:].contiguous(), beta=inp["beta"][:, cut:].contiguous(), initial_state=sfa)
    ob, sfb = gpu_run(b)
    assert_close("o", oracle.to_f64(torch.cat([oa, ob], 1)), oracle.to_f64(o), 2e-3, 1e-2)
    assert_close("final_state", oracle.to_f64(sfb), oracle.to_f64(sf), 2e-3, 1e-2)


def test_cp_off_is_deterministic():
    inp = to_device(make_inputs(CONFIGS[1].scaled(B=2, T=500, H=4), "cpu"))
    o1, s1 = gpu_run(inp, opts_for(cp_mode=gdn.CP_OFF))
    o2, s2 = gpu_run(inp, opts_for(cp_mode=gdn.CP_OFF))
    assert torch.equal(o1, o2) and torch.equal(s1, s2)


@pytest.mark.parametrize("cols", [1, 6, 16])
def test_inverse_overlap_is_bit_identical(cols):
    """The fused pass computing the inverse of the last `cols` chunk columns on
    the SMs its units leave idle (one cooperative launch; each such column's T1
    is loaded once its ready count says all units are in memory) gives the
    same bits as the separate inverse launch; 16 columns is every column of
    these sequences, including the ragged last one."""
    inp = to_device(make_inputs(CONFIGS[1].scaled(B=2, T=1000, H=8), "cpu"))
    B, T, H, dk = inp["q"].shape
    info = gdn.gdn_plan_query(B, T, H, dk, dk, B, 0, gdn.BF16, opts_for(cp_mode=gdn.CP_OFF, inverse_overlap=cols))
    assert info.overlap_columns == min(cols, 16)
    o0, s0 = gpu_run(inp, opts_for(cp_mode=gdn.CP_OFF, inverse_overlap=-1))
    o1, s1 = gpu_run(inp, opts_for(cp_mode=gdn.CP_OFF, inverse_overlap=cols))
    assert torch.equal(o0, o1) and torch.equal(s0, s1)
    if cols == 16:
        o_ref, sf_ref = full_reference(inp)
        assert_close("o", oracle.to_f64(o1).reshape(B * T, H, -1), o_ref)
        assert_close("final_state", oracle.to_f64(s1), sf_ref)


# ----------------------------------------------------------- intermediates

def _workspace_views(inp, ws, opts=None):
    q, v = inp["q"], inp["v"]
    B, T, H, dk = q.shape
    cu = inp.get("cu_seqlens")
    N = B if cu is None else cu.numel() - 1
    dt = gdn.BF16 if q.dtype == torch.bfloat16 else gdn.F32
    lay = gdn.gdn_workspace_query(B, T, H, dk, v.shape[-1], N, cu is not None, dt, opts)
    total_T = B * T
    info = gdn.gdn_plan_query(B, T, H, dk, v.shape[-1], N, cu is not None, dt, opts)

    def view(off, n, dtype):
        esz = torch.tensor([], dtype=dtype).element_size()
        return ws[off:off + n * esz].view(dtype)

    return dict(
        G=view(lay.gate_cumsum, H * total_T, torch.float32).view(H, total_T),
        flags=view(lay.head_flags, N * H, torch.int32).view(N, H),
        tprime=view(lay.tprime, H * total_T * 64, q.dtype).view(H, total_T, 64),
        totals=view(lay.chunk_totals, H * info.max_chunks, torch.float32).view(H, info.max_chunks),
        num_chunks=int(view(lay.num_chunks, 1, torch.int32).item()),
        chunks=view(lay.chunk_table, 4 * info.max_chunks, torch.int32).view(info.max_chunks, 4),
        items=view(lay.items, 8 * info.max_items, torch.int32).view(info.max_items, 8),
        num_items=view(lay.num_items, 4, torch.int32).tolist(),
    )


def gate_scaled_tprime(Tp, G, beta, cu, C):
    """T1 = T' diag(c1) per chunk and head, from the oracle's T' and chunk-local
    gate cumsum G: the factored gate Gamma_rm = a_r b_m around the midpoint G* of
    the chunk's first and last cumsum gives c1_m = b_m beta_m, b_m = exp(G* - G_m);
    a chunk whose last cumsum is below -80 keeps Gamma element-wise instead:
    T1 = (Gamma ⊙ T') diag(beta)."""
    out = np.zeros_like(Tp)
    for n in range(len(cu) - 1):
        for t0 in range(int(cu[n]), int(cu[n + 1]), C):
            L = min(C, int(cu[n + 1]) - t0)
            for h in range(Tp.shape[1]):
                Gc, bc = G[t0:t0 + L, h], beta[t0:t0 + L, h]
                blk = Tp[t0:t0 + L, h, :L]
                if Gc[-1] < -80.0:
                    gam = np.exp(np.minimum(Gc[:, None] - Gc[None, :], 0.0))
                    out[t0:t0 + L, h, :L] = blk * gam * bc[None, :]
                else:
                    b = np.exp(0.5 * (Gc[0] + Gc[-1]) - Gc)
                    out[t0:t0 + L, h, :L] = blk * (b * bc)[None, :]
    return out


def test_planner_gives_correction_heads_fewer_segments_when_a_wave_is_saved():
    """With 16 CTAs, 3 heads with alpha == 1 and 5 decaying heads split into 16
    segments, pass 1 would need six waves of 4-chunk items; the device planner's
    per-pass model gives the alpha == 1 heads fewer, longer segments (the
    decaying heads keep 16), and the result still matches the oracle."""
    cfg = CONFIGS[2].scaled(T=4096, H=8, zero_gate_heads=(0, 1, 2))
    inp = to_device(make_inputs(cfg, "cpu"))
    opts = gdn.default_options(cp_mode=gdn.CP_FORCE, chunks_per_segment=4, sm_count=16)
    ws = gdn.workspace_for(inp["q"], inp["v"], None, opts)
    o, sf = gpu_run(inp, opts, workspace=ws)
    views = _workspace_views(inp, ws, opts)
    items = views["items"][:views["num_items"][0]].cpu().numpy()
    per_head = {h: int((items[:, 1] == h).sum()) for h in range(8)}
    assert all(per_head[h] == 16 for h in range(3, 8)), per_head
    assert all(2 <= per_head[h] < 16 for h in range(3)), per_head
    o_ref, sf_ref = full_reference(inp)
    assert_close("o", oracle.to_f64(o).reshape(o_ref.shape), o_ref)
    assert_close("final_state", oracle.to_f64(sf), sf_ref)


@pytest.mark.parametrize("case", ["varlen", "equal"])
def test_gate_and_inverse_intermediates(case):
    """G, chunk totals, head flags and T1 in the workspace after a call, for
    packed sequences and for equal ones without a split (whose work list the
    sequence-prep kernel writes itself)."""
    if case == "varlen":
        cfg = CONFIGS[3].scaled(T=3000, H=3, n_seqs=5, zero_gate_heads=(1,))
    else:
        cfg = CONFIGS[1].scaled(B=3, T=1000, H=3)
    inp = to_device(make_inputs(cfg, "cpu"))
    H = inp["q"].shape[2]
    opts = gdn.default_options(cp_mode=gdn.CP_OFF) if case == "equal" else None
    ws = gdn.workspace_for(inp["q"], inp["v"], inp["cu_seqlens"], opts)
    gpu_run(inp, opts, workspace=ws)
    views = _workspace_views(inp, ws, opts)
    cu = seq_bounds(inp)
    g = oracle.to_f64(inp["g"]).reshape(-1, H)
    # chunk-local cumsum of the gate
    G_ref = gate.chunk_local_cumsum(g, cu, 64)
    assert np.abs(oracle.to_f64(views["G"]).T - G_ref).max() < 1e-4
    nck = views["num_chunks"]
    table = gate.chunk_table(cu, 64)
    assert nck == len(table)
    # the chunk table entry by entry: (sequence, first token, length, chunk index in the sequence)
    ref_rows = [(n, t0, ln, (t0 - int(cu[n])) // 64) for n, t0, ln in table]
    assert views["chunks"][:nck].cpu().numpy().tolist() == [list(r) for r in ref_rows]
    if case == "equal":
        # the work list the sequence-prep kernel writes: one whole-sequence item per (sequence, head)
        N = len(cu) - 1
        nc = [-(-(int(cu[n + 1]) - int(cu[n])) // 64) for n in range(N)]
        assert views["num_items"][:3] == [N * H, 0, 0]
        want = [[n, h, 0, nc[n], 0, 1 | 2 | 32, -1, 0] for n in range(N) for h in range(H)]
        assert views["items"][:N * H].cpu().numpy().tolist() == want
    # chunk totals and head flags
    tot_ref = gate.chunk_totals(g, cu, 64)
    assert np.abs(oracle.to_f64(views["totals"][:, :nck]).T - tot_ref).max() < 1e-4
    assert views["flags"].cpu().numpy().tolist() == gate.head_flags(g, cu).tolist()
    # T' rows against the fp64 inverse (bf16 storage).  The tcgen05 path stores
    # the gate-scaled T1 = T' diag(c1) that its fused kernel multiplies by.
    beta = oracle.to_f64(inp["beta"]).reshape(-1, H)
    Tp_ref = chunked.inverse_rows(oracle.to_f64(inp["k"]).reshape(-1, H, 128), beta, cu, 64)
    Tp_ref = gate_scaled_tprime(Tp_ref, G_ref, beta, cu, 64)
    Tp = oracle.to_f64(views["tprime"]).transpose(1, 0, 2)
    # element-wise: bf16 storage of entries that the gate scaling can make large
    assert (np.abs(Tp - Tp_ref) / (1.0 + np.abs(Tp_ref))).max() < 2e-2
    assert np.linalg.norm(Tp - Tp_ref) / np.linalg.norm(Tp_ref) < 4e-3


def test_bad_cu_seqlens_is_reported_not_faulted():
    cfg = CONFIGS[3].scaled(T=1000, H=2, n_seqs=4)
    inp = to_device(make_inputs(cfg, "cpu"))
    bad = inp["cu_seqlens"].clone()
    bad[2] = bad[1] - 5            # decreasing
    with pytest.raises(gdn.GdnError) as e:
        gdn.chunk_fwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], None, bad, inp["scale"], check=True)
    assert e.value.status == 5
    bad = inp["cu_seqlens"].clone()
    bad[-1] = 999                  # does not cover the tokens
    with pytest.raises(gdn.GdnError) as e:
        gdn.chunk_fwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], None, bad, inp["scale"], check=True)
    assert e.value.status == 5
    # the context is still usable afterwards
    o, sf = gpu_run(inp)
    assert torch.isfinite(o.float()).all()


@pytest.mark.parametrize("kernel", ["auto", "simt"])
@pytest.mark.parametrize("cp", ["off", "force"])
def test_zero_beta_only_decays_the_initial_state(kernel, cp):
    """beta = 0 everywhere: no token writes the state, so S_t = (prod alpha) S_0
    and o_t = scale gamma_t S_0 q_t, on every path (both fused kernels, with and
    without the segment split)."""
    cfg = CONFIGS[1].scaled(B=2, T=700, H=3, s0_std=0.5)
    inp = to_device(make_inputs(cfg, "cpu"))
    inp["beta"] = torch.zeros_like(inp["beta"])
    kw = dict(cp_mode=gdn.CP_OFF) if cp == "off" else dict(cp_mode=gdn.CP_FORCE, chunks_per_segment=3)
    o, sf = gpu_run(inp, opts_for(kernel, **kw))
    g = oracle.to_f64(inp["g"])                                   # [B, T, H]
    G = np.cumsum(g, axis=1)
    s0 = oracle.to_f64(inp["initial_state"])                      # [B, H, dk, dv], [j][i] = S[i][j]
    q = oracle.to_f64(inp["q"])                                   # [B, T, H, dk]
    o_ref = inp["scale"] * np.exp(G)[..., None] * np.einsum("bthj,bhji->bthi", q, s0)
    sf_ref = np.exp(G[:, -1])[..., None, None] * s0
    assert_close("o", oracle.to_f64(o), o_ref)
    assert_close("final_state", oracle.to_f64(sf), sf_ref)


def test_orthonormal_keys_with_full_writes_store_the_values_exactly():
    """alpha = 1, beta = 1 and orthonormal keys (T <= dk): each token overwrites
    the state along its key, so the final state maps every key to its value,
    S_T k_t = v_t (fp32, CUDA-core kernel), whatever the initial state."""
    T, dk = 32, 32
    cfg = CONFIGS[0].scaled(T=T, H=2, s0_std=0.3)
    inp = make_inputs(cfg, "cpu")
    g = torch.Generator().manual_seed(7)
    for h in range(2):
        qmat, _ = torch.linalg.qr(torch.randn(dk, dk, generator=g, dtype=torch.float64))
        inp["k"][0, :, h, :] = qmat[:, :T].T.to(torch.float32)      # rows: orthonormal keys
    inp["g"] = torch.zeros_like(inp["g"])
    inp["beta"] = torch.ones_like(inp["beta"])
    inp = to_device(inp)
    _, sf = gpu_run(inp, opts_for("simt", cp_mode=gdn.CP_OFF))
    S = oracle.to_f64(sf)[0]                                      # [H, dk, dv], [j][i] = S[i][j]
    k = oracle.to_f64(inp["k"])[0]                                # [T, H, dk]
    v = oracle.to_f64(inp["v"])[0]                                # [T, H, dv]
    recalled = np.einsum("hji,thj->thi", S, k)                    # S_T k_t
    assert np.abs(recalled - v).max() < 2e-4


def test_many_heads_span_several_gate_groups():
    """H = 70: the gate kernel takes heads in groups of 64, so a second, partial
    group; 3 x 70 units fill more than one wave of the persistent passes."""
    cfg = CONFIGS[1].scaled(B=3, T=200, H=70, s0_std=0.02)
    inp = to_device(make_inputs(cfg, "cpu"))
    o_ref, sf_ref = full_reference(inp)
    o, sf = gpu_run(inp, opts_for(cp_mode=gdn.CP_OFF))
    assert_close("o", oracle.to_f64(o).reshape(o_ref.shape), o_ref)
    assert_close("final_state", oracle.to_f64(sf), sf_ref)


@pytest.mark.parametrize("cp", ["off", "force"])
def test_stages_run_separately_equal_one_call(cp):
    """opts.stages: the prep and inverse stages in one call and the correction
    and fused stages in a second call on the same workspace give the one-call
    result bit for bit (each stage reads only what earlier stages left in the
    workspace)."""
    cfg = CONFIGS[3].scaled(T=3000, H=3, n_seqs=5, s0_std=0.02)
    inp = to_device(make_inputs(cfg, "cpu"))
    kw = dict(cp_mode=gdn.CP_OFF) if cp == "off" else dict(cp_mode=gdn.CP_FORCE, chunks_per_segment=4)
    ws = gdn.workspace_for(inp["q"], inp["v"], inp["cu_seqlens"], gdn.default_options(**kw))
    o1, sf1 = gpu_run(inp, gdn.default_options(**kw), workspace=ws)
    o1, sf1 = o1.clone(), sf1.clone()
    gpu_run(inp, gdn.default_options(stages=gdn.STAGE_PREP | gdn.STAGE_INVERSE, **kw), workspace=ws)
    o2, sf2 = gpu_run(inp, gdn.default_options(stages=gdn.STAGE_CORRECTION | gdn.STAGE_FUSED, **kw), workspace=ws)
    assert torch.equal(o1, o2) and torch.equal(sf1, sf2)


def test_bounded_wait_runs_out_and_reports_timeout():
    """GDN_DEBUG_TIMEOUT_PROBE: the tcgen05 fused pass's tile producer signals
    nothing, so every bounded wait of that pass runs out (about 2 s) without a
    fault or a hang; the call reports GDN_ERR_TIMEOUT through the device check,
    and the next call on the same workspace is unaffected."""
    cfg = CONFIGS[1].scaled(B=1, T=300, H=2)
    inp = to_device(make_inputs(cfg, "cpu"))
    ws = gdn.workspace_for(inp["q"], inp["v"])
    with pytest.raises(gdn.GdnError) as e:
        gpu_run(inp, gdn.default_options(cp_mode=gdn.CP_OFF, kernel=gdn.KERNEL_TC, debug_checks=1), workspace=ws)
    assert e.value.status == 6
    o, sf = gpu_run(inp, gdn.default_options(cp_mode=gdn.CP_OFF, kernel=gdn.KERNEL_TC), workspace=ws)
    o_ref, sf_ref = full_reference(inp)
    assert_close("o", oracle.to_f64(o).reshape(o_ref.shape), o_ref)
    assert_close("final_state", oracle.to_f64(sf), sf_ref)


def test_host_buffer_entry_point():
    inp = make_inputs(CONFIGS[3].scaled(T=2500, H=2, n_seqs=3, s0_std=0.02), "cpu")
    pinned = {k: (v.pin_memory() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    o, sf = gdn.chunk_fwd_host(pinned["q"], pinned["k"], pinned["v"], pinned["g"], pinned["beta"],
                               pinned["initial_state"], pinned["cu_seqlens"], inp["scale"])
    o_ref, sf_ref = full_reference(inp)
    assert_close("o", oracle.to_f64(o).reshape(o_ref.shape), o_ref)
    assert_close("final_state", oracle.to_f64(sf), sf_ref)


@pytest.mark.parametrize("case", ["batched", "varlen"])
def test_host_entry_streams_large_problems_in_parts(case):
    """Above 64 MB of input the host-buffer entry point copies, runs and copies
    back in parts on three streams (batched: two 1024-token pieces of each of
    the four sequences, the state handed on through the device buffer; varlen:
    eight groups of whole sequences); every part keeps the whole problem's
    plan, so the result equals the device entry point's bit for bit."""
    if case == "batched":
        cfg = CONFIGS[1].scaled(B=4, T=2048, H=32, s0_std=0.02)     # 203 MB of input, eight parts
    else:
        cfg = CONFIGS[3].scaled(T=65536, H=16, n_seqs=13, s0_std=0.02)
    inp = make_inputs(cfg, "cpu")
    pinned = {k: (v.pin_memory() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    o, sf = gdn.chunk_fwd_host(pinned["q"], pinned["k"], pinned["v"], pinned["g"], pinned["beta"],
                               pinned["initial_state"], pinned["cu_seqlens"], inp["scale"])
    dev = to_device(inp)
    o_d, sf_d = gpu_run(dev)
    assert torch.equal(o, o_d.cpu()) and torch.equal(sf, sf_d.cpu())
    # and a sampled check against the oracle
    cu = seq_bounds(inp)
    seqs, heads, rows = [0, len(cu) - 2], [0, cfg.H - 1], [0, 77]
    o_ref, sf_ref, idx = sampled_reference(inp, seqs, heads, rows)
    o_s, sf_s = gpu_sampled(o, sf, inp, seqs, heads, rows, idx)
    assert_close("o", o_s, o_ref)
    assert_close("final_state", sf_s, sf_ref)


# ---------------------------------------------- full sizes, every output

def full_size_errors(inp, o, sf):
    """Every (sequence, head, value row) of a full-size run against the oracle,
    one head at a time (so the fp64 copies stay a few GB even for the 1M-token
    workload).  Returns whole-tensor rel-L2 and max-abs for o and final_state,
    plus the worst head's rel-L2 for each (a diagnostic)."""
    cu = inp.get("cu_seqlens")
    cu = cu.cpu() if cu is not None else None
    H = inp["q"].shape[2]
    acc = {"o": [0.0, 0.0, 0.0, 0.0], "final_state": [0.0, 0.0, 0.0, 0.0]}   # |d|^2, |ref|^2, max|d|, worst head
    for h in range(H):
        sl = lambda t: t[:, :, h:h + 1].contiguous().cpu()
        s0 = inp.get("initial_state")
        s0h = s0[:, h:h + 1].contiguous().cpu() if s0 is not None else None
        o_ref, sf_ref = oracle.gdn_reference(sl(inp["q"]), sl(inp["k"]), sl(inp["v"]), sl(inp["g"]),
                                             sl(inp["beta"]), s0h, cu, scale=inp["scale"])
        got = {"o": oracle.to_f64(o[:, :, h:h + 1]).reshape(o_ref.shape), "final_state": oracle.to_f64(sf[:, h:h + 1])}
        for name, ref in (("o", o_ref), ("final_state", sf_ref)):
            x = got[name]
            assert np.isfinite(x).all(), "%s head %d has non-finite values" % (name, h)
            d = x - ref
            a = acc[name]
            dd, rr = float((d * d).sum()), float((ref * ref).sum())
            a[0] += dd
            a[1] += rr
            a[2] = max(a[2], float(np.abs(d).max()) if d.size else 0.0)
            a[3] = max(a[3], (dd / rr) ** 0.5 if rr > 0 else 0.0)
        del o_ref, sf_ref, got
    return {name: {"rel_l2": (a[0] / a[1]) ** 0.5 if a[1] > 0 else 0.0, "max_abs": a[2], "worst_head_rel_l2": a[3]}
            for name, a in acc.items()}


@pytest.mark.parametrize("idx", [0, 1, 2, 3, 4])
def test_full_size_every_output(idx):
    """Each workload at its full size, in the bench's launch configuration,
    compared with the oracle on every element of o and final_state.  With
    GDN_PARITY_MARGINS set to a file name, the errors are also appended there
    as one JSON line per workload (the margin table)."""
    import json
    import os
    import time
    cfg = CONFIGS[idx]
    inp = make_inputs(cfg, "cuda")
    o, sf = gpu_run(inp)
    t0 = time.time()
    err = full_size_errors(inp, o, sf)
    path = os.environ.get("GDN_PARITY_MARGINS")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps({"workload": idx, "name": cfg.name, "B": cfg.B, "T": cfg.T, "H": cfg.H,
                                "dk": cfg.dk, "dv": cfg.dv, "dtype": cfg.dtype,
                                "n_seqs": cfg.num_seqs, "oracle_s": time.time() - t0, **err}) + "\n")
    for name in ("o", "final_state"):
        e = err[name]
        assert e["rel_l2"] <= 5e-3 and e["max_abs"] <= 2e-2, "%s: %s" % (name, e)


def test_tcgen05_kernel_matches_cuda_core_kernel():
    """The tcgen05 kernel and the CUDA-core kernel follow the same chunked
    algebra; on a layer-shaped case they agree far inside the oracle bar."""
    cfg = CONFIGS[1].scaled(B=2, T=777, H=3, s0_std=0.02)
    inp = to_device(make_inputs(cfg, "cpu"))
    info = gdn.gdn_plan_query(2, 777, 3, 128, 128, 2, 0, gdn.BF16, opts_for("auto"))
    assert info.kernel == gdn.KERNEL_TC
    o_tc, s_tc = gpu_run(inp, opts_for("auto", cp_mode=gdn.CP_FORCE, chunks_per_segment=3))
    o_si, s_si = gpu_run(inp, opts_for("simt", cp_mode=gdn.CP_FORCE, chunks_per_segment=3))
    assert_close("o", oracle.to_f64(o_tc), oracle.to_f64(o_si), 4e-3, 2e-2)
    assert_close("final_state", oracle.to_f64(s_tc), oracle.to_f64(s_si), 4e-3, 2e-2)


@pytest.mark.parametrize("kernel", ["auto", "simt"])
def test_extreme_gates_take_the_exact_form(kernel):
    """Heads whose gate cumsum falls far within a chunk (per-token |g| up to
    ~4) exercise the element-wise Gamma path; other heads stay factored."""
    cfg = CONFIGS[1].scaled(B=2, T=330, H=4, a_range=(-3.0, 1.5), s0_std=0.02)
    inp = to_device(make_inputs(cfg, "cpu"))
    o_ref, sf_ref = full_reference(inp)
    o, sf = gpu_run(inp, opts_for(kernel, cp_mode=gdn.CP_FORCE, chunks_per_segment=2))
    assert_close("o", oracle.to_f64(o).reshape(o_ref.shape), o_ref)
    assert_close("final_state", oracle.to_f64(sf), sf_ref)
