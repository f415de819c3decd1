"""Host-side tests of the C ABI (no GPU needed): the library loads, exports
every function include/gdn.h declares, plans sensibly and rejects bad
arguments before any launch."""
import ctypes
import os
import re

import pytest

import chunked_prefill_gdn_gb300 as gdn
from chunked_prefill_gdn_gb300 import build as gdn_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    gdn_build.build()
    return gdn.load_library()


def declared_functions():
    names = []
    for h in os.listdir(os.path.join(ROOT, "include")):
        if not h.endswith(".h"):
            continue
        src = open(os.path.join(ROOT, "include", h)).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        names += re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*(gdn_[a-z0-9_]+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert "gdn_chunk_fwd" in names and len(names) >= 9
    for n in names:
        assert hasattr(lib, n), n


def test_version_and_status_strings(lib):
    assert "sm_103a" in gdn.gdn_version()
    assert gdn.gdn_status_string(0) == "GDN_OK"
    assert gdn.gdn_status_string(5) == "GDN_ERR_DEVICE_CHECK"


def test_option_struct_layout(lib):
    assert ctypes.sizeof(gdn.GdnOptions) == 64
    o = gdn.default_options()
    assert o.cp_mode == gdn.CP_AUTO and o.sliding == 1 and abs(o.sw_eps - 2 ** -24) < 1e-12


def plan(*a, **kw):
    opts = gdn.default_options(**kw) if kw else None
    return gdn.gdn_plan_query(*a, opts=opts)


def test_plan_layer_shape_runs_without_cp(lib):
    p = plan(4, 8192, 32, 128, 128, 4, 0, gdn.BF16, sm_count=152)
    assert p.cp_enabled == 0 and p.max_chunks == 512 and p.max_items == 128


def test_plan_few_long_sequences_split(lib):
    p = plan(1, 131072, 8, 128, 128, 1, 0, gdn.BF16, sm_count=152)
    assert p.cp_enabled == 1
    segs = -(-2048 // p.chunks_per_segment)
    assert 8 * segs <= 152 * 2 and segs >= 10
    assert p.max_cp_slots >= 8 * (segs - 1)


def test_plan_cp_modes(lib):
    off = plan(1, 131072, 8, 128, 128, 1, 0, gdn.BF16, sm_count=152, cp_mode=gdn.CP_OFF)
    assert off.cp_enabled == 0 and off.max_cp_slots == 0
    force = plan(4, 8192, 32, 128, 128, 4, 0, gdn.BF16, sm_count=152, cp_mode=gdn.CP_FORCE,
                 chunks_per_segment=16)
    assert force.cp_enabled == 1 and force.chunks_per_segment == 16
    assert force.max_items >= 4 * 32 * 8


def test_plan_inverse_overlap(lib):
    """The fused pass takes over the inverse of the last chunk columns only
    when asked (inverse_overlap = k > 0), and only for equal sequences without
    a split on the tcgen05 kernels with idle SMs; k is capped at the columns."""
    q = lambda B, T, H, **kw: plan(B, T, H, 128, 128, B, 0, gdn.BF16, sm_count=152, **kw)
    assert q(4, 8192, 32).overlap_columns == 0                               # off by default
    assert q(4, 8192, 32, inverse_overlap=-1).overlap_columns == 0
    on = q(4, 8192, 32, inverse_overlap=7)
    assert on.overlap_columns == 7 and on.grid_fused == 152
    assert q(4, 8192, 32, inverse_overlap=500).overlap_columns == 128
    assert q(8, 8192, 32, inverse_overlap=7).overlap_columns == 0           # no idle SM
    assert q(4, 8192, 32, inverse_overlap=7, cp_mode=gdn.CP_FORCE).overlap_columns == 0
    assert q(4, 8192, 32, inverse_overlap=7, kernel=gdn.KERNEL_SIMT).overlap_columns == 0
    assert plan(1, 8192, 32, 128, 128, 4, 1, gdn.BF16, sm_count=152, inverse_overlap=7).overlap_columns == 0
    assert plan(4, 8192, 32, 128, 128, 4, 0, gdn.F32, sm_count=152, inverse_overlap=7).overlap_columns == 0


def test_plan_counts_the_launches_of_a_call(lib):
    """seqprep, gate, inverse, fused pass; a planner launch unless the sequences
    are equal and unsplit; the correction pass and scan with a split; the
    normalisation pass when asked for."""
    assert plan(4, 8192, 32, 128, 128, 4, 0, gdn.BF16, sm_count=152).launches == 4
    assert plan(4, 8192, 32, 128, 128, 4, 0, gdn.BF16, sm_count=152, qk_l2norm=1).launches == 5
    assert plan(1, 131072, 8, 128, 128, 1, 0, gdn.BF16, sm_count=152).launches == 7
    assert plan(1, 4096, 4, 128, 128, 3, 1, gdn.BF16, sm_count=152, cp_mode=gdn.CP_OFF).launches == 5


def test_plan_kernel_choice_by_head_size(lib):
    """Head sizes 32, 64 or 128 (any pair) take the tcgen05 kernels: kind::f16
    for bf16, kind::tf32 for fp32; the CUDA-core kernel only when asked."""
    for dk in (32, 64, 128):
        for dv in (32, 64, 128):
            assert plan(2, 256, 2, dk, dv, 2, 0, gdn.BF16).kernel == gdn.KERNEL_TC
            assert plan(2, 256, 2, dk, dv, 2, 0, gdn.F32).kernel == gdn.KERNEL_TC
            assert plan(2, 256, 2, dk, dv, 2, 0, gdn.F32, kernel=gdn.KERNEL_SIMT).kernel == gdn.KERNEL_SIMT


def test_plan_varlen_capacity_bounds(lib):
    p = plan(1, 262144, 16, 128, 128, 64, 1, gdn.BF16, sm_count=152)
    assert p.max_chunks == 262144 // 64 + 64
    L = p.chunks_per_segment
    assert p.max_items >= 16 * 64 and p.max_cp_slots == 16 * (-(-p.max_chunks // L))


def test_plan_rejects_bad_shapes(lib):
    with pytest.raises(gdn.GdnError):
        plan(1, 100, 2, 48, 64, 1, 0, gdn.BF16)       # unsupported head size
    with pytest.raises(gdn.GdnError):
        plan(2, 100, 2, 64, 64, 2, 1, gdn.BF16)       # varlen needs B == 1
    with pytest.raises(gdn.GdnError):
        plan(1, 100, 0, 64, 64, 1, 0, gdn.BF16)


def test_workspace_size_grows_with_tokens(lib):
    a = gdn.gdn_chunk_fwd_workspace_size(1, 1000, 4, 128, 128, 1, 0, gdn.BF16)
    b = gdn.gdn_chunk_fwd_workspace_size(1, 2000, 4, 128, 128, 1, 0, gdn.BF16)
    assert 0 < a < b
    assert gdn.gdn_chunk_fwd_workspace_size(1, 10, 4, 48, 128, 1, 0, gdn.BF16) == 0


def test_host_argument_errors_before_launch(lib):
    """Null or misaligned pointers and a short workspace are rejected on the
    host; these calls never reach the GPU."""
    fake = ctypes.c_void_p(1 << 20)
    mis = ctypes.c_void_p((1 << 20) + 4)
    args = dict(q=fake, k=fake, v=fake, g=fake, b=fake)
    ws = gdn.gdn_chunk_fwd_workspace_size(1, 256, 2, 32, 32, 1, 0, gdn.F32)

    def call(q=fake, o=fake, sf=fake, wsp=fake, wsb=ws):
        return gdn.gdn_chunk_fwd(q, fake, fake, fake, fake, None, None, 1, 0.0, 1, 256, 2, 32, 32, gdn.F32,
                                 o, sf, wsp, wsb, None, None)
    assert call(q=None) == 1
    assert call(q=mis) == 1
    assert call(sf=None) == 1
    assert call(wsb=ws - 1) == 3
    assert gdn.gdn_chunk_fwd(fake, fake, fake, fake, fake, None, None, 1, 0.0, 1, 256, 2, 48, 32, gdn.F32,
                             fake, fake, fake, ws, None, None) == 2


def test_qk_l2norm_option_and_workspace(lib):
    o = gdn.default_options()
    assert o.qk_l2norm == 0 and ctypes.sizeof(gdn.GdnOptions) == 64
    T, H, dk = 1000, 4, 128
    plain = gdn.gdn_chunk_fwd_workspace_size(1, T, H, dk, 128, 1, 0, gdn.BF16, gdn.default_options(sm_count=152))
    normed = gdn.gdn_chunk_fwd_workspace_size(1, T, H, dk, 128, 1, 0, gdn.BF16,
                                              gdn.default_options(sm_count=152, qk_l2norm=1))
    copy = -(-T * H * dk * 2 // 256) * 256            # one bf16 copy of q (or k), 256-byte aligned
    assert normed - plain == 2 * copy
    with pytest.raises(gdn.GdnError):
        gdn.gdn_plan_query(1, T, H, dk, 128, 1, 0, gdn.BF16, gdn.default_options(qk_l2norm=2))


def test_qk_l2norm_argument_errors_before_launch(lib):
    """gdn_qk_l2norm rejects bad sizes, dtypes, alignment and NULL pairings on
    the host, and zero rows enqueue nothing; none of these reach the GPU."""
    fake = ctypes.c_void_p(1 << 20)
    mis = ctypes.c_void_p((1 << 20) + 8)
    f = gdn.gdn_qk_l2norm
    assert f(fake, fake, fake, fake, 10, 48, gdn.BF16, 0.0, None) == 1      # dk
    assert f(fake, fake, fake, fake, -1, 128, gdn.BF16, 0.0, None) == 1     # rows
    assert f(fake, fake, fake, fake, 10, 128, 7, 0.0, None) == 1            # dtype
    assert f(mis, fake, fake, fake, 10, 128, gdn.BF16, 0.0, None) == 1      # alignment
    assert f(fake, None, fake, fake, 10, 128, gdn.BF16, 0.0, None) == 1     # k NULL, k_out not
    assert f(fake, fake, None, fake, 10, 128, gdn.BF16, 0.0, None) == 1     # q_out NULL, q not
    assert f(fake, fake, fake, fake, 0, 128, gdn.BF16, 0.0, None) == 0      # nothing to do


def test_backward_workspace_size(lib):
    """The backward's workspace holds the chunk start states and, above 32 value
    columns, the per-slice partial sums; bad shapes give 0."""
    a = gdn.gdn_chunk_bwd_workspace_size(1, 1000, 4, 128, 32, 1, 0, gdn.BF16)
    b = gdn.gdn_chunk_bwd_workspace_size(1, 2000, 4, 128, 32, 1, 0, gdn.BF16)
    c = gdn.gdn_chunk_bwd_workspace_size(1, 2000, 4, 128, 128, 1, 0, gdn.BF16)
    assert 0 < a < b < c
    # states: (T/64 + N) slots of H x dk x dv fp32 at least
    assert b >= (2000 // 64 + 1) * 4 * 128 * 32 * 4
    # partials of dq, dk (4 slices each) on top of the states for dv = 128
    assert c >= (2000 // 64 + 1) * 4 * 128 * 128 * 4 + 2 * 4 * 2000 * 4 * 128 * 4
    assert gdn.gdn_chunk_bwd_workspace_size(1, 10, 4, 48, 128, 1, 0, gdn.BF16) == 0
    assert gdn.gdn_chunk_bwd_workspace_size(2, 10, 4, 64, 64, 2, 1, gdn.BF16) == 0    # varlen needs B == 1
    assert gdn.gdn_chunk_bwd_workspace_size(1, 10, 4, 64, 64, 70000, 1, gdn.BF16) == 0


def test_backward_argument_errors_before_launch(lib):
    """Null or misaligned pointers, unsupported head sizes and a short workspace
    are rejected on the host; these calls never reach the GPU."""
    fake = ctypes.c_void_p(1 << 20)
    mis = ctypes.c_void_p((1 << 20) + 4)
    ws = gdn.gdn_chunk_bwd_workspace_size(1, 256, 2, 32, 64, 1, 0, gdn.F32)

    def call(q=fake, do=fake, dq=fake, wsp=fake, wsb=ws, dk=32, dv=64):
        return gdn.gdn_chunk_bwd(q, fake, fake, fake, fake, None, None, 1, 0.0, 1, 256, 2, dk, dv, gdn.F32,
                                 do, None, dq, fake, fake, fake, fake, None, wsp, wsb, None)
    assert call(q=None) == 1
    assert call(do=None) == 1
    assert call(dq=None) == 1
    assert call(dq=mis) == 1
    assert call(wsp=None) == 1
    assert call(wsb=ws - 1) == 3
    assert call(dk=48) == 2
    assert call(dv=16) == 2
    assert gdn.gdn_chunk_bwd_check(None, None) == 1


def test_qk_l2norm_backward_argument_errors_before_launch(lib):
    """Sizes, dtype, NULL and misaligned pointers are rejected on the host (no
    GPU is touched); zero rows is a no-op."""
    fake = ctypes.c_void_p(1 << 20)
    mis = ctypes.c_void_p((1 << 20) + 4)
    assert gdn.gdn_qk_l2norm_bwd(fake, fake, fake, 10, 48, gdn.BF16, 0.0, None) == 1
    assert gdn.gdn_qk_l2norm_bwd(fake, fake, fake, 10, 64, 7, 0.0, None) == 1
    assert gdn.gdn_qk_l2norm_bwd(fake, None, fake, 10, 64, gdn.BF16, 0.0, None) == 1
    assert gdn.gdn_qk_l2norm_bwd(fake, fake, mis, 10, 64, gdn.BF16, 0.0, None) == 1
    assert gdn.gdn_qk_l2norm_bwd(fake, fake, fake, -1, 64, gdn.BF16, 0.0, None) == 1
    assert gdn.gdn_qk_l2norm_bwd(None, None, None, 0, 64, gdn.BF16, 0.0, None) == 0


def test_binding_rejects_mismatched_shapes_before_the_library():
    """The C ABI sees plain pointers, so the binding checks every tensor's shape
    against q's and v's first (a short k or state would otherwise be read out
    of bounds on the device); these raise on the host, before any CUDA call.
    The tensors here live on the CPU, so a call that passes the shape checks
    stops at the device check instead (the control below)."""
    import torch
    q = torch.zeros(1, 8, 2, 32)
    v = torch.zeros(1, 8, 2, 64)
    g = torch.zeros(1, 8, 2)
    good = dict(q=q, k=q, v=v, g=g, beta=g)
    with pytest.raises(ValueError, match="CUDA"):                                   # control
        gdn.chunk_fwd(q, q, v, g, g)
    with pytest.raises(ValueError, match="CUDA"):
        gdn.chunk_bwd(q, q, v, g, g, torch.zeros(1, 8, 2, 64))
    cases = [
        dict(k=torch.zeros(1, 8, 2, 16)),
        dict(v=torch.zeros(1, 7, 2, 64)),
        dict(g=torch.zeros(1, 8, 3)),
        dict(beta=torch.zeros(8, 2)),
    ]
    for bad in cases:
        a = dict(good, **bad)
        with pytest.raises(ValueError, match="shape"):
            gdn.chunk_fwd(a["q"], a["k"], a["v"], a["g"], a["beta"])
    with pytest.raises(ValueError, match="initial_state has shape"):
        gdn.chunk_fwd(q, q, v, g, g, initial_state=torch.zeros(1, 2, 32, 32))
    with pytest.raises(ValueError, match="out has shape"):
        gdn.chunk_fwd(q, q, v, g, g, out=torch.zeros(1, 8, 2, 32))
    with pytest.raises(ValueError, match="cu_seqlens"):
        gdn.chunk_fwd(q, q, v, g, g, cu_seqlens=torch.zeros(1, dtype=torch.int32))
    with pytest.raises(ValueError, match="do has shape"):
        gdn.chunk_bwd(q, q, v, g, g, torch.zeros(1, 8, 2, 32))                       # do like o
    with pytest.raises(ValueError, match="d_final_state has shape"):
        gdn.chunk_bwd(q, q, v, g, g, torch.zeros(1, 8, 2, 64), d_final_state=torch.zeros(2, 2, 32, 64))
    with pytest.raises(ValueError, match="beta has shape"):
        gdn.chunk_fwd_host(q, q, v, g, torch.zeros(1, 8, 1))


def test_binding_rejects_wrong_dtypes_before_the_library():
    """A tensor of the wrong element type would be read or written past its end
    by the kernels (an fp32 state written into a bf16 buffer, an int64
    cu_seqlens read as int32 pairs), so the binding checks every dtype first.
    These tensors are on the CPU, so passing the dtype checks would stop at the
    placement check instead (the control)."""
    import torch
    q = torch.zeros(1, 8, 2, 32, dtype=torch.bfloat16)
    v = torch.zeros(1, 8, 2, 64, dtype=torch.bfloat16)
    g = torch.zeros(1, 8, 2)
    with pytest.raises(ValueError, match="CUDA"):                                   # control
        gdn.chunk_fwd(q, q, v, g, g)
    cases = [
        dict(final_state=torch.zeros(1, 2, 32, 64, dtype=torch.bfloat16)),
        dict(out=torch.zeros(1, 8, 2, 64, dtype=torch.float32)),
        dict(initial_state=torch.zeros(1, 2, 32, 64, dtype=torch.float64)),
        dict(cu_seqlens=torch.tensor([0, 8], dtype=torch.int64)),
        dict(workspace=torch.zeros(16, dtype=torch.int32)),
    ]
    for kw in cases:
        with pytest.raises(TypeError, match=next(iter(kw))):
            gdn.chunk_fwd(q, q, v, g, g, **kw)
    with pytest.raises(TypeError, match="g must be"):
        gdn.chunk_fwd(q, q, v, g.double(), g)
    with pytest.raises(TypeError, match="v must be"):
        gdn.chunk_fwd(q, q, v.float(), g, g)
    with pytest.raises(TypeError, match="do must be"):
        gdn.chunk_bwd(q, q, v, g, g, torch.zeros(1, 8, 2, 64))
    with pytest.raises(TypeError, match="d_final_state must be"):
        gdn.chunk_bwd(q, q, v, g, g, torch.zeros(1, 8, 2, 64, dtype=torch.bfloat16),
                      d_final_state=torch.zeros(1, 2, 32, 64, dtype=torch.bfloat16))
    with pytest.raises(TypeError, match="final_state must be"):
        gdn.chunk_fwd_host(q, q, v, g, g, final_state=torch.zeros(1, 2, 32, 64, dtype=torch.bfloat16))


def test_binding_placement_check():
    """Every tensor handed to a device entry point must live on q's device, and
    every tensor of the host-buffer entry point in host memory: the library
    receives bare pointers.  Without a GPU here the device rule is exercised on
    the 'meta' device type (same code path: type first, then the device, then
    contiguity)."""
    import torch
    meta = torch.empty(4, 4, device="meta")
    cpu = torch.zeros(4, 4)
    gdn._check_placement("meta", meta.device, dict(a=meta, b=None))
    with pytest.raises(ValueError, match="initial_state must be a contiguous META tensor"):
        gdn._check_placement("meta", meta.device, dict(q=meta, initial_state=cpu))
    with pytest.raises(ValueError, match="cu_seqlens must be a contiguous CUDA tensor"):
        gdn._check_placement("cuda", None, dict(cu_seqlens=cpu))
    with pytest.raises(ValueError, match="contiguous"):
        gdn._check_placement("cpu", cpu.device, dict(x=cpu.t()))
    # the host-buffer entry point: a device-side (here: meta) input is refused
    q = torch.zeros(1, 8, 2, 32)
    v = torch.zeros(1, 8, 2, 64)
    g = torch.zeros(1, 8, 2)
    with pytest.raises(ValueError, match="initial_state must be a contiguous CPU tensor"):
        gdn.chunk_fwd_host(q, q, v, g, g, initial_state=torch.empty(1, 2, 32, 64, device="meta"))
    with pytest.raises(ValueError, match="device_buffer must be a contiguous CUDA tensor"):
        gdn.chunk_fwd_host(q, q, v, g, g, device_buffer=torch.zeros(16, dtype=torch.uint8))


def test_plan_costs_roundtrip_and_validation(lib):
    """The planner's measured step costs can be read, replaced and restored;
    bad tables are refused without touching the current one."""
    orig = gdn.gdn_get_plan_costs()
    try:
        c = gdn.GdnPlanCosts(2.0, 1.0, 0.5, 10.0)
        gdn.gdn_set_plan_costs(c)
        got = gdn.gdn_get_plan_costs()
        assert (got.chunk_step_us, got.state_step_us, got.scan_step_us, got.pass_us) == (2.0, 1.0, 0.5, 10.0)
        for bad in (gdn.GdnPlanCosts(0.0, 1.0, 0.5, 1.0), gdn.GdnPlanCosts(1.0, -1.0, 0.5, 1.0),
                    gdn.GdnPlanCosts(float("nan"), 1.0, 0.5, 1.0), gdn.GdnPlanCosts(1.0, 1.0, -0.1, 1.0)):
            with pytest.raises(gdn.GdnError):
                gdn.gdn_set_plan_costs(bad)
        assert gdn.gdn_get_plan_costs().chunk_step_us == 2.0
        gdn.gdn_set_plan_costs(None)                     # the library's built-in table
        d = gdn.gdn_get_plan_costs()
        assert d.chunk_step_us > 0 and d.state_step_us > 0 and d.scan_step_us >= 0
    finally:
        gdn.gdn_set_plan_costs(orig)


def test_auto_cp_boundary_is_a_curve(lib):
    """The talk's enabling-condition paragraph: in the plane of (sequence, head)
    units and sequence length, the region where auto CP pays is bounded by a
    curve, not by a threshold on either axis.  The planner's boundary: more
    units leave fewer idle SMs, so the least length that splits grows with the
    unit count and no length does once the units fill the SMs; and the plan
    query agrees with the boundary on both sides of it."""
    sms = 152
    mins = {u: gdn.gdn_auto_cp_min_chunks(u, sms) for u in (1, 2, 4, 8, 16, 24, 32, 48, 64, 96, 128, 151, 152, 300)}
    assert mins[152] == 0 and mins[300] == 0
    on = [u for u, m in sorted(mins.items()) if m > 0]
    assert on and on[0] == 1
    assert all(mins[a] <= mins[b] for a, b in zip(on, on[1:])), mins
    assert mins[on[-1]] > mins[1]                        # the curve rises before it ends
    for u in (1, 8, 32):
        nc = mins[u]
        H = 8 if u % 8 == 0 else u
        B = u // H
        p_on = gdn.gdn_plan_query(B, 64 * nc, H, 128, 128, B, 0, gdn.BF16, gdn.default_options(sm_count=sms))
        p_off = gdn.gdn_plan_query(B, 64 * (nc - 1), H, 128, 128, B, 0, gdn.BF16,
                                   gdn.default_options(sm_count=sms))
        assert p_on.cp_enabled == 1 and p_off.cp_enabled == 0, (u, nc)
    # a dearer scan (lambda2) pushes the boundary to longer sequences
    orig = gdn.gdn_get_plan_costs()
    try:
        gdn.gdn_set_plan_costs(gdn.GdnPlanCosts(orig.chunk_step_us, orig.state_step_us, 20 * orig.scan_step_us + 5,
                                                orig.pass_us))
        assert gdn.gdn_auto_cp_min_chunks(8, sms) > mins[8]
    finally:
        gdn.gdn_set_plan_costs(orig)


def test_transition_and_scan_argument_errors_before_launch(lib):
    """gdn_chunk_transition and gdn_state_scan reject bad sizes, NULL or
    misaligned pointers, a short workspace and an output that overlaps an
    input on the host; none of these calls reaches the GPU."""
    fake = ctypes.c_void_p(1 << 20)
    mis = ctypes.c_void_p((1 << 20) + 4)
    ws = gdn.gdn_chunk_transition_workspace_size(1, 256, 2, 32, 32, 1, 0, gdn.F32)
    assert ws > 0
    assert gdn.gdn_chunk_transition_workspace_size(1, 256, 2, 48, 32, 1, 0, gdn.F32) == 0

    def tr(k=fake, s=fake, m=fake, wsp=fake, wsb=ws, dk=32):
        return gdn.gdn_chunk_transition(k, fake, fake, fake, None, 1, 1, 256, 2, dk, 32, gdn.F32, s, m, wsp, wsb,
                                        None)
    assert tr(k=None) == 1
    assert tr(k=mis) == 1
    assert tr(s=None) == 1
    assert tr(m=mis) == 1
    assert tr(wsp=None) == 1
    assert tr(wsb=ws - 1) == 3
    assert tr(dk=48) == 2
    sc = gdn.gdn_state_scan
    base = 1 << 24
    p = lambda off: ctypes.c_void_p(base + off)
    n = 3 * 1 * 2 * 32 * 32 * 4                    # bytes of the s_star / s_start stacks (R=3, N=1, H=2, d=32)
    assert sc(None, p(0), p(n), 0, 1, 2, 32, 32, p(2 * n), None) == 1           # R
    assert sc(None, p(0), p(n), 3, 1, 2, 48, 32, p(2 * n), None) == 2           # dk
    assert sc(None, None, p(n), 3, 1, 2, 32, 32, p(2 * n), None) == 1           # s_star NULL
    assert sc(None, p(0), p(n), 3, 1, 2, 32, 32, None, None) == 1               # out NULL
    assert sc(None, p(4), p(n), 3, 1, 2, 32, 32, p(2 * n), None) == 1           # misaligned
    assert sc(None, p(0), p(n), 3, 1, 2, 32, 32, p(n // 2), None) == 1          # out overlaps s_star
    assert sc(p(2 * n + 64), p(0), p(n), 3, 1, 2, 32, 32, p(2 * n), None) == 1  # out overlaps s0
