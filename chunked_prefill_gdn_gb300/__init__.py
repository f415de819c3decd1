"""GB300 (sm_103a) Gated Delta Network chunked-prefill forward pass.

A thin ctypes binding over the C ABI in include/gdn.h: every function here only
marshals arguments; all of the computation runs in the library's CUDA kernels.
There is no CPU fallback: when the library is missing or cannot load, every
call raises.

    o, final_state = chunk_fwd(q, k, v, g, beta, initial_state=None,
                               cu_seqlens=None, scale=None)
    dq, dk, dv, dg, dbeta, d_initial_state = chunk_bwd(q, k, v, g, beta, do, ...)
    o, final_state = chunk_gated_delta_rule(q, k, v, g, beta, ...)   # autograd

q, k [B,T,H,dk] and v [B,T,H,dv] in bf16 or fp32, g and beta [B,T,H] fp32,
initial_state [N,H,dk,dv] fp32, cu_seqlens int32 [N+1] (then B = 1), all on
the same CUDA device.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

from . import build as _build

__all__ = [
    "GdnOptions", "GdnPlanInfo", "GdnPlanCosts", "GdnWorkspaceLayout", "WORK_ITEM_DTYPE",
    "gdn_set_plan_costs", "gdn_get_plan_costs", "gdn_auto_cp_min_chunks",
    "gdn_chunk_transition_workspace_size", "gdn_chunk_transition", "gdn_state_scan", "chunk_transition",
    "state_scan", "gdn_state_grad_scan", "state_grad_scan",
    "load_library", "library_path", "default_options",
    "gdn_default_options", "gdn_plan_query", "gdn_chunk_fwd_workspace_size", "gdn_workspace_query",
    "gdn_chunk_fwd", "gdn_chunk_fwd_check", "gdn_chunk_fwd_host_buffer_size", "gdn_chunk_fwd_host",
    "gdn_chunk_fwd_static", "gdn_qk_l2norm", "qk_l2norm", "gdn_qk_l2norm_bwd", "qk_l2norm_backward",
    "gdn_chunk_bwd_workspace_size", "gdn_chunk_bwd", "gdn_chunk_bwd_check", "chunk_bwd",
    "gdn_set_backward_kernel", "gdn_get_backward_kernel", "gdn_chunk_state_grad", "chunk_state_grad",
    "chunk_gated_delta_rule",
    "gdn_status_string", "gdn_version", "gdn_last_error_detail", "chunk_fwd", "chunk_fwd_host", "workspace_for", "GdnError",
    "CP_AUTO", "CP_OFF", "CP_FORCE", "KERNEL_AUTO", "KERNEL_TC", "KERNEL_SIMT", "BF16", "F32",
    "STAGE_PREP", "STAGE_INVERSE", "STAGE_CORRECTION", "STAGE_FUSED",
]

BF16, F32 = 0, 1
CP_AUTO, CP_OFF, CP_FORCE = 0, 1, 2
KERNEL_AUTO, KERNEL_TC, KERNEL_SIMT = 0, 1, 2
STAGE_PREP, STAGE_INVERSE, STAGE_CORRECTION, STAGE_FUSED = 1, 2, 4, 8
STATUS = {0: "GDN_OK", 1: "GDN_ERR_INVALID_ARG", 2: "GDN_ERR_UNSUPPORTED", 3: "GDN_ERR_WORKSPACE",
          4: "GDN_ERR_CUDA", 5: "GDN_ERR_DEVICE_CHECK", 6: "GDN_ERR_TIMEOUT"}


class GdnError(RuntimeError):
    def __init__(self, status: int, where: str = ""):
        self.status = status
        detail = ""
        if status == 4 and _lib is not None:
            detail = _lib.gdn_last_error_detail().decode()
        super().__init__("%s%s%s" % (STATUS.get(status, "status %d" % status), (" in " + where) if where else "",
                                     (" (" + detail + ")") if detail else ""))


class GdnOptions(ctypes.Structure):
    _fields_ = [("cp_mode", ctypes.c_int32), ("kernel", ctypes.c_int32),
                ("chunks_per_segment", ctypes.c_int32), ("sliding", ctypes.c_int32),
                ("sw_eps", ctypes.c_float), ("sm_count", ctypes.c_int32),
                ("stages", ctypes.c_int32), ("debug_checks", ctypes.c_int32),
                ("prof_begin", ctypes.c_void_p), ("prof_end", ctypes.c_void_p),
                ("qk_l2norm", ctypes.c_int32), ("inverse_overlap", ctypes.c_int32),
                ("reserved", ctypes.c_int32 * 2)]


class GdnPlanInfo(ctypes.Structure):
    _fields_ = [("kernel", ctypes.c_int32), ("cp_enabled", ctypes.c_int32),
                ("chunks_per_segment", ctypes.c_int32), ("max_chunks", ctypes.c_int32),
                ("max_items", ctypes.c_int32), ("max_cp_slots", ctypes.c_int32),
                ("sm_count", ctypes.c_int32), ("grid_fused", ctypes.c_int32),
                ("overlap_columns", ctypes.c_int32), ("launches", ctypes.c_int32),
                ("workspace_bytes", ctypes.c_size_t)]


class GdnPlanCosts(ctypes.Structure):
    _fields_ = [("chunk_step_us", ctypes.c_float), ("state_step_us", ctypes.c_float),
                ("scan_step_us", ctypes.c_float), ("pass_us", ctypes.c_float)]


class GdnWorkspaceLayout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in ("error_word", "gate_cumsum", "chunk_totals", "head_flags",
                                              "tprime", "chunk_table", "num_chunks", "items", "num_items",
                                              "total")]


# field order of gdn_work_item (eight int32)
WORK_ITEM_DTYPE = ("seq", "head", "c_begin", "c_end", "c_start", "flags", "slot", "pad")

_lib = None


def library_path() -> str:
    return _build.LIB


def load_library(build_if_missing: bool = False):
    """Load the CUDA library (raises when it is absent and not built)."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.LIB
    if not os.path.exists(path):
        if not build_if_missing:
            raise RuntimeError("GDN CUDA library not built: %s (run __graft_entry__.build() or "
                               "python chunked_prefill_gdn_gb300/build.py)" % path)
        _build.build()
    lib = ctypes.CDLL(path)
    vp, sz, i32, f32 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_float
    opt = ctypes.POINTER(GdnOptions)
    lib.gdn_default_options.argtypes = [opt]
    lib.gdn_default_options.restype = None
    lib.gdn_plan_query.argtypes = [i32] * 7 + [i32, opt, ctypes.POINTER(GdnPlanInfo)]
    lib.gdn_plan_query.restype = i32
    lib.gdn_chunk_fwd_workspace_size.argtypes = [i32] * 7 + [i32, opt]
    lib.gdn_chunk_fwd_workspace_size.restype = sz
    lib.gdn_workspace_query.argtypes = [i32] * 7 + [i32, opt, ctypes.POINTER(GdnWorkspaceLayout)]
    lib.gdn_workspace_query.restype = i32
    fwd_args = [vp, vp, vp, vp, vp, vp, vp, i32, f32, i32, i32, i32, i32, i32, i32, vp, vp, vp, sz, opt, vp]
    lib.gdn_chunk_fwd.argtypes = fwd_args
    lib.gdn_chunk_fwd.restype = i32
    lib.gdn_chunk_fwd_check.argtypes = [vp, vp]
    lib.gdn_chunk_fwd_check.restype = i32
    lib.gdn_chunk_fwd_host_buffer_size.argtypes = [i32] * 8 + [i32, opt]
    lib.gdn_chunk_fwd_host_buffer_size.restype = sz
    lib.gdn_chunk_fwd_host.argtypes = fwd_args
    lib.gdn_chunk_fwd_host.restype = i32
    lib.gdn_chunk_fwd_static.argtypes = fwd_args[:17] + [vp, opt, vp]
    lib.gdn_chunk_fwd_static.restype = i32
    lib.gdn_qk_l2norm.argtypes = [vp, vp, vp, vp, ctypes.c_int64, i32, i32, ctypes.c_float, vp]
    lib.gdn_qk_l2norm.restype = i32
    lib.gdn_qk_l2norm_bwd.argtypes = [vp, vp, vp, ctypes.c_int64, i32, i32, ctypes.c_float, vp]
    lib.gdn_qk_l2norm_bwd.restype = i32
    lib.gdn_chunk_bwd_workspace_size.argtypes = [i32] * 8
    lib.gdn_chunk_bwd_workspace_size.restype = sz
    lib.gdn_chunk_bwd.argtypes = [vp] * 7 + [i32, f32] + [i32] * 6 + [vp] * 8 + [vp, sz, vp]
    lib.gdn_chunk_bwd.restype = i32
    lib.gdn_chunk_bwd_check.argtypes = [vp, vp]
    lib.gdn_chunk_bwd_check.restype = i32
    lib.gdn_chunk_state_grad.argtypes = [vp] * 5 + [i32, f32] + [i32] * 6 + [vp] * 4 + [sz, vp]
    lib.gdn_chunk_state_grad.restype = i32
    lib.gdn_set_backward_kernel.argtypes = [i32]
    lib.gdn_set_backward_kernel.restype = i32
    lib.gdn_get_backward_kernel.argtypes = []
    lib.gdn_get_backward_kernel.restype = i32
    lib.gdn_chunk_transition_workspace_size.argtypes = [i32] * 8
    lib.gdn_chunk_transition_workspace_size.restype = sz
    lib.gdn_chunk_transition.argtypes = [vp, vp, vp, vp, vp, i32] + [i32] * 6 + [vp, vp, vp, sz, vp]
    lib.gdn_chunk_transition.restype = i32
    lib.gdn_state_scan.argtypes = [vp, vp, vp] + [i32] * 5 + [vp, vp]
    lib.gdn_state_scan.restype = i32
    lib.gdn_state_grad_scan.argtypes = [vp, vp, vp] + [i32] * 5 + [vp, vp]
    lib.gdn_state_grad_scan.restype = i32
    lib.gdn_set_plan_costs.argtypes = [ctypes.POINTER(GdnPlanCosts)]
    lib.gdn_set_plan_costs.restype = i32
    lib.gdn_get_plan_costs.argtypes = [ctypes.POINTER(GdnPlanCosts)]
    lib.gdn_get_plan_costs.restype = None
    lib.gdn_auto_cp_min_chunks.argtypes = [i32, i32]
    lib.gdn_auto_cp_min_chunks.restype = i32
    lib.gdn_status_string.argtypes = [i32]
    lib.gdn_status_string.restype = ctypes.c_char_p
    lib.gdn_version.argtypes = []
    lib.gdn_version.restype = ctypes.c_char_p
    lib.gdn_last_error_detail.argtypes = []
    lib.gdn_last_error_detail.restype = ctypes.c_char_p
    _lib = lib
    _apply_measured_costs(lib)
    return lib


PLAN_COSTS_FILE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "plan_costs.json")


def _apply_measured_costs(lib):
    """The planner's step costs measured by the calibrate module on this kind
    of GPU (plan_costs.json next to this file), when present; the library's
    built-in table otherwise."""
    if not os.path.exists(PLAN_COSTS_FILE):
        return
    import json
    with open(PLAN_COSTS_FILE) as f:
        c = json.load(f)["costs"]
    costs = GdnPlanCosts(*(float(c[k]) for k in ("chunk_step_us", "state_step_us", "scan_step_us", "pass_us")))
    st = lib.gdn_set_plan_costs(ctypes.byref(costs))
    if st != 0:
        raise GdnError(st, "gdn_set_plan_costs (%s)" % PLAN_COSTS_FILE)


def default_options(**kw) -> GdnOptions:
    o = GdnOptions()
    load_library().gdn_default_options(ctypes.byref(o))
    for k, v in kw.items():
        setattr(o, k, v)
    return o


# ----------------------------------------------------------- raw C-ABI names

def gdn_default_options(opts: GdnOptions) -> None:
    load_library().gdn_default_options(ctypes.byref(opts))


def gdn_plan_query(B, T, H, dk, dv, n_seqs, varlen, dtype, opts=None) -> GdnPlanInfo:
    info = GdnPlanInfo()
    st = load_library().gdn_plan_query(B, T, H, dk, dv, n_seqs, int(varlen), dtype,
                                       ctypes.byref(opts) if opts is not None else None, ctypes.byref(info))
    if st != 0:
        raise GdnError(st, "gdn_plan_query")
    return info


def gdn_chunk_fwd_workspace_size(B, T, H, dk, dv, n_seqs, varlen, dtype, opts=None) -> int:
    return int(load_library().gdn_chunk_fwd_workspace_size(B, T, H, dk, dv, n_seqs, int(varlen), dtype,
                                                            ctypes.byref(opts) if opts is not None else None))


def gdn_workspace_query(B, T, H, dk, dv, n_seqs, varlen, dtype, opts=None) -> GdnWorkspaceLayout:
    lay = GdnWorkspaceLayout()
    st = load_library().gdn_workspace_query(B, T, H, dk, dv, n_seqs, int(varlen), dtype,
                                            ctypes.byref(opts) if opts is not None else None, ctypes.byref(lay))
    if st != 0:
        raise GdnError(st, "gdn_workspace_query")
    return lay


def gdn_chunk_fwd(*args) -> int:
    return int(load_library().gdn_chunk_fwd(*args))


def gdn_chunk_fwd_check(workspace_ptr, stream_ptr) -> int:
    return int(load_library().gdn_chunk_fwd_check(workspace_ptr, stream_ptr))


def gdn_chunk_fwd_host_buffer_size(B, T, H, dk, dv, n_seqs, varlen, has_initial_state, dtype, opts=None) -> int:
    return int(load_library().gdn_chunk_fwd_host_buffer_size(
        B, T, H, dk, dv, n_seqs, int(varlen), int(has_initial_state), dtype,
        ctypes.byref(opts) if opts is not None else None))


def gdn_chunk_fwd_host(*args) -> int:
    return int(load_library().gdn_chunk_fwd_host(*args))


def gdn_chunk_fwd_static(*args) -> int:
    """gdn_chunk_fwd without a workspace argument: the scratch is the library's
    fixed 64 MiB device array (for callers that must not allocate)."""
    return int(load_library().gdn_chunk_fwd_static(*args))


def gdn_qk_l2norm(*args) -> int:
    return int(load_library().gdn_qk_l2norm(*args))


def gdn_qk_l2norm_bwd(*args) -> int:
    return int(load_library().gdn_qk_l2norm_bwd(*args))


def gdn_chunk_bwd_workspace_size(B, T, H, dk, dv, n_seqs, varlen, dtype) -> int:
    return int(load_library().gdn_chunk_bwd_workspace_size(B, T, H, dk, dv, n_seqs, int(varlen), dtype))


def gdn_chunk_bwd(*args) -> int:
    return int(load_library().gdn_chunk_bwd(*args))


def gdn_chunk_bwd_check(workspace_ptr, stream_ptr) -> int:
    return int(load_library().gdn_chunk_bwd_check(workspace_ptr, stream_ptr))


def gdn_chunk_state_grad(*args) -> int:
    return int(load_library().gdn_chunk_state_grad(*args))


def gdn_set_backward_kernel(kernel) -> None:
    """KERNEL_AUTO / KERNEL_TC: the tensor-core backward (default);
    KERNEL_SIMT: the CUDA-core backward.  Process-wide, for later calls."""
    st = int(load_library().gdn_set_backward_kernel(int(kernel)))
    if st != 0:
        raise GdnError(st, "gdn_set_backward_kernel")


def gdn_get_backward_kernel() -> int:
    return int(load_library().gdn_get_backward_kernel())


def gdn_chunk_transition_workspace_size(B, T, H, dk, dv, n_seqs, varlen, dtype) -> int:
    return int(load_library().gdn_chunk_transition_workspace_size(B, T, H, dk, dv, n_seqs, int(varlen), dtype))


def gdn_chunk_transition(*args) -> int:
    return int(load_library().gdn_chunk_transition(*args))


def gdn_state_scan(*args) -> int:
    return int(load_library().gdn_state_scan(*args))


def gdn_state_grad_scan(*args) -> int:
    return int(load_library().gdn_state_grad_scan(*args))


def gdn_set_plan_costs(costs: Optional[GdnPlanCosts]) -> None:
    st = load_library().gdn_set_plan_costs(ctypes.byref(costs) if costs is not None else None)
    if st != 0:
        raise GdnError(st, "gdn_set_plan_costs")


def gdn_get_plan_costs() -> GdnPlanCosts:
    c = GdnPlanCosts()
    load_library().gdn_get_plan_costs(ctypes.byref(c))
    return c


def gdn_auto_cp_min_chunks(units: int, sms: int) -> int:
    return int(load_library().gdn_auto_cp_min_chunks(units, sms))


def gdn_status_string(status: int) -> str:
    return load_library().gdn_status_string(status).decode()


def gdn_version() -> str:
    return load_library().gdn_version().decode()


def gdn_last_error_detail() -> str:
    return load_library().gdn_last_error_detail().decode()


# ---------------------------------------------------------------- tensor API

def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float32:
        return F32
    raise TypeError("q/k/v must be bfloat16 or float32, got %s" % t.dtype)


def _ptr(t: Optional[torch.Tensor]):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _shape(q, v, cu_seqlens):
    if q.dim() != 4:
        raise ValueError("q must be [B, T, H, dk]")
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    if cu_seqlens is not None:
        if B != 1:
            raise ValueError("cu_seqlens needs B == 1")
        N = cu_seqlens.numel() - 1
    else:
        N = B
    return B, T, H, dk, dv, N


def _expect(name, t, shape):
    if t is not None and tuple(t.shape) != tuple(shape):
        raise ValueError("%s has shape %s, expected %s" % (name, tuple(t.shape), tuple(shape)))


def _check_shapes(q, k, v, g, beta, initial_state=None, cu_seqlens=None):
    """Every input's shape against q's and v's, before any pointer reaches the
    library (which sees plain pointers and cannot check them); returns
    (B, T, H, dk, dv, N)."""
    if v.dim() != 4:
        raise ValueError("v must be [B, T, H, dv]")
    if cu_seqlens is not None and (cu_seqlens.dim() != 1 or cu_seqlens.numel() < 2):
        raise ValueError("cu_seqlens must be 1-D with at least two entries")
    B, T, H, dk, dv, N = _shape(q, v, cu_seqlens)
    _expect("k", k, (B, T, H, dk))
    _expect("v", v, (B, T, H, dv))
    _expect("g", g, (B, T, H))
    _expect("beta", beta, (B, T, H))
    _expect("initial_state", initial_state, (N, H, dk, dv))
    return B, T, H, dk, dv, N


def _check_dtypes(named, dtypes):
    """Each given tensor's dtype against the one the C ABI expects for it (a
    wrong element size would make the kernels read or write past its end)."""
    for name, t in named.items():
        if t is not None and t.dtype != dtypes[name]:
            raise TypeError("%s must be %s, got %s" % (name, dtypes[name], t.dtype))


def _check_placement(kind, device, named):
    """Every given tensor contiguous, of device type `kind` ("cuda" for the
    device entry points, "cpu" for the host-buffer one) and, when `device` is
    given, on that device: the library receives bare pointers and would
    dereference a host pointer on the GPU (or a pointer into another GPU's
    memory) without any way to tell."""
    for name, t in named.items():
        if t is None:
            continue
        if t.device.type != kind:
            raise ValueError("%s must be a contiguous %s tensor, got one on %s" % (
                name, "CUDA" if kind == "cuda" else kind.upper(), t.device))
        if device is not None and t.device != device:
            raise ValueError("%s is on %s but q is on %s" % (name, t.device, device))
        if not t.is_contiguous():
            raise ValueError("%s must be a contiguous %s tensor" % (name, "CUDA" if kind == "cuda" else kind.upper()))


def workspace_for(q, v, cu_seqlens=None, opts: Optional[GdnOptions] = None) -> torch.Tensor:
    B, T, H, dk, dv, N = _shape(q, v, cu_seqlens)
    n = gdn_chunk_fwd_workspace_size(B, T, H, dk, dv, N, cu_seqlens is not None, _dtype_code(q), opts)
    if n == 0:
        raise GdnError(1, "gdn_chunk_fwd_workspace_size")
    return torch.empty(n, dtype=torch.uint8, device=q.device)


def chunk_fwd(q, k, v, g, beta, initial_state=None, cu_seqlens=None, scale=None,
              opts: Optional[GdnOptions] = None, out=None, final_state=None, workspace=None,
              stream: Optional[torch.cuda.Stream] = None, check: bool = False):
    """GDN chunked-prefill forward on the GPU; returns (o, final_state)."""
    B, T, H, dk, dv, N = _check_shapes(q, k, v, g, beta, initial_state, cu_seqlens)
    _expect("out", out, (B, T, H, dv))
    _expect("final_state", final_state, (N, H, dk, dv))
    dt = _dtype_code(q)
    f32 = torch.float32
    _check_dtypes(dict(k=k, v=v, g=g, beta=beta, initial_state=initial_state, cu_seqlens=cu_seqlens, out=out,
                       final_state=final_state, workspace=workspace),
                  dict(k=q.dtype, v=q.dtype, g=f32, beta=f32, initial_state=f32, cu_seqlens=torch.int32,
                       out=q.dtype, final_state=f32, workspace=torch.uint8))
    _check_placement("cuda", None, dict(q=q))
    _check_placement("cuda", q.device, dict(k=k, v=v, g=g, beta=beta, initial_state=initial_state,
                                            cu_seqlens=cu_seqlens, out=out, final_state=final_state,
                                            workspace=workspace))
    with torch.cuda.device(q.device):
        if out is None:
            out = torch.empty(B, T, H, dv, dtype=q.dtype, device=q.device)
        if final_state is None:
            final_state = torch.empty(N, H, dk, dv, dtype=torch.float32, device=q.device)
        if workspace is None:
            workspace = workspace_for(q, v, cu_seqlens, opts)
        stream = stream if stream is not None else torch.cuda.current_stream(q.device)
        st = gdn_chunk_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(initial_state), _ptr(cu_seqlens),
                           N, float(scale) if scale is not None else 0.0, B, T, H, dk, dv, dt,
                           _ptr(out), _ptr(final_state), _ptr(workspace), workspace.numel(),
                           ctypes.byref(opts) if opts is not None else None, ctypes.c_void_p(stream.cuda_stream))
        if st != 0:
            raise GdnError(st, "gdn_chunk_fwd")
        if check:
            st = gdn_chunk_fwd_check(_ptr(workspace), ctypes.c_void_p(stream.cuda_stream))
            if st != 0:
                raise GdnError(st, "device check")
    return out, final_state


def chunk_transition(k, v, g, beta, cu_seqlens=None, workspace=None, stream: Optional[torch.cuda.Stream] = None,
                     check: bool = False):
    """The affine map of each (sequence, head) of this slice on the state,
    S_end = S_start M + S*, through gdn_chunk_transition; returns fp32
    (s_star [N, H, dk, dv], m [N, H, dk, dk]) in the library's state layout."""
    B, T, H, dk, dv, N = _check_shapes(k, k, v, g, beta, None, cu_seqlens)
    dt = _dtype_code(k)
    f32 = torch.float32
    _check_dtypes(dict(v=v, g=g, beta=beta, cu_seqlens=cu_seqlens, workspace=workspace),
                  dict(v=k.dtype, g=f32, beta=f32, cu_seqlens=torch.int32, workspace=torch.uint8))
    _check_placement("cuda", None, dict(k=k))
    _check_placement("cuda", k.device, dict(v=v, g=g, beta=beta, cu_seqlens=cu_seqlens, workspace=workspace))
    with torch.cuda.device(k.device):
        s_star = torch.empty(N, H, dk, dv, dtype=f32, device=k.device)
        m = torch.empty(N, H, dk, dk, dtype=f32, device=k.device)
        if workspace is None:
            n = gdn_chunk_transition_workspace_size(B, T, H, dk, dv, N, cu_seqlens is not None, dt)
            if n == 0:
                raise GdnError(1, "gdn_chunk_transition_workspace_size")
            workspace = torch.empty(n, dtype=torch.uint8, device=k.device)
        stream = stream if stream is not None else torch.cuda.current_stream(k.device)
        st = gdn_chunk_transition(_ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(cu_seqlens), N, B, T, H, dk, dv, dt,
                                  _ptr(s_star), _ptr(m), _ptr(workspace), workspace.numel(),
                                  ctypes.c_void_p(stream.cuda_stream))
        if st != 0:
            raise GdnError(st, "gdn_chunk_transition")
        if check:
            st = gdn_chunk_fwd_check(_ptr(workspace), ctypes.c_void_p(stream.cuda_stream))
            if st != 0:
                raise GdnError(st, "device check")
    return s_star, m


def state_scan(s_star, m, s0=None, stream: Optional[torch.cuda.Stream] = None):
    """Start states of R consecutive slices from their maps (s_star
    [R, N, H, dk, dv], m [R, N, H, dk, dk], rank-major) through gdn_state_scan:
    out[0] = s0 (or zero), out[r + 1] = out[r] M_r + S*_r."""
    if s_star.dim() != 5 or m.dim() != 5:
        raise ValueError("s_star must be [R, N, H, dk, dv] and m [R, N, H, dk, dk]")
    R, N, H, dk, dv = s_star.shape
    _expect("m", m, (R, N, H, dk, dk))
    _expect("s0", s0, (N, H, dk, dv))
    f32 = torch.float32
    _check_dtypes(dict(s_star=s_star, m=m, s0=s0), dict(s_star=f32, m=f32, s0=f32))
    _check_placement("cuda", None, dict(s_star=s_star))
    _check_placement("cuda", s_star.device, dict(m=m, s0=s0))
    with torch.cuda.device(s_star.device):
        out = torch.empty_like(s_star)
        stream = stream if stream is not None else torch.cuda.current_stream(s_star.device)
        st = gdn_state_scan(_ptr(s0), _ptr(s_star), _ptr(m), R, N, H, dk, dv, _ptr(out),
                            ctypes.c_void_p(stream.cuda_stream))
        if st != 0:
            raise GdnError(st, "gdn_state_scan")
    return out


def state_grad_scan(ds_star, m, ds_last=None, stream: Optional[torch.cuda.Stream] = None):
    """End-state gradients of R consecutive slices from each slice's own
    start-state gradient (ds_star [R, N, H, dk, dv]) and map (m [R, N, H, dk,
    dk]) through gdn_state_grad_scan: out[R - 1] = ds_last (or zero),
    out[r] = out[r + 1] M_{r+1}^T + ds_star[r + 1]."""
    if ds_star.dim() != 5 or m.dim() != 5:
        raise ValueError("ds_star must be [R, N, H, dk, dv] and m [R, N, H, dk, dk]")
    R, N, H, dk, dv = ds_star.shape
    _expect("m", m, (R, N, H, dk, dk))
    _expect("ds_last", ds_last, (N, H, dk, dv))
    f32 = torch.float32
    _check_dtypes(dict(ds_star=ds_star, m=m, ds_last=ds_last), dict(ds_star=f32, m=f32, ds_last=f32))
    _check_placement("cuda", None, dict(ds_star=ds_star))
    _check_placement("cuda", ds_star.device, dict(m=m, ds_last=ds_last))
    with torch.cuda.device(ds_star.device):
        out = torch.empty_like(ds_star)
        stream = stream if stream is not None else torch.cuda.current_stream(ds_star.device)
        st = gdn_state_grad_scan(_ptr(ds_last), _ptr(ds_star), _ptr(m), R, N, H, dk, dv, _ptr(out),
                                 ctypes.c_void_p(stream.cuda_stream))
        if st != 0:
            raise GdnError(st, "gdn_state_grad_scan")
    return out


def qk_l2norm(q=None, k=None, q_out=None, k_out=None, eps: float = 0.0,
              stream: Optional[torch.cuda.Stream] = None):
    """Unit-L2-norm rows of q and/or k ([..., dk], contiguous CUDA tensors of one
    dtype) through gdn_qk_l2norm; returns (q_hat, k_hat) (None where not given).
    Pass q_out=q / k_out=k to normalise in place."""
    ref = q if q is not None else k
    if ref is None:
        return None, None
    for t in (q, k):
        if t is not None and (not t.is_cuda or not t.is_contiguous() or t.dtype != ref.dtype
                              or t.shape != ref.shape):
            raise ValueError("q and k must be contiguous CUDA tensors of one shape and dtype")
    for name, t in (("q_out", q_out), ("k_out", k_out)):
        if t is not None and (t.dtype != ref.dtype or t.shape != ref.shape):
            raise ValueError("%s must have the inputs' shape and dtype" % name)
    _check_placement("cuda", ref.device, dict(q=q, k=k, q_out=q_out, k_out=k_out))
    dk = ref.shape[-1]
    rows = ref.numel() // dk
    with torch.cuda.device(ref.device):
        if q is not None and q_out is None:
            q_out = torch.empty_like(q)
        if k is not None and k_out is None:
            k_out = torch.empty_like(k)
        stream = stream if stream is not None else torch.cuda.current_stream(ref.device)
        st = gdn_qk_l2norm(_ptr(q), _ptr(k), _ptr(q_out), _ptr(k_out), rows, dk, _dtype_code(ref), float(eps),
                           ctypes.c_void_p(stream.cuda_stream))
        if st != 0:
            raise GdnError(st, "gdn_qk_l2norm")
    return q_out, k_out


def qk_l2norm_backward(x, dy, dx=None, eps: float = 0.0, stream: Optional[torch.cuda.Stream] = None):
    """fp32 gradient of the rows x (the tensor qk_l2norm normalised) from the
    fp32 gradient dy of their normalised copies, through gdn_qk_l2norm_bwd.
    Pass dx=dy to overwrite dy."""
    for name, t in (("x", x), ("dy", dy)):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("%s must be a contiguous CUDA tensor" % name)
    if dy.dtype != torch.float32 or dy.shape != x.shape:
        raise ValueError("dy must be float32 with x's shape")
    if dx is not None and (dx.dtype != torch.float32 or dx.shape != x.shape):
        raise ValueError("dx must be float32 with x's shape")
    _check_placement("cuda", x.device, dict(dy=dy, dx=dx))
    dk = x.shape[-1]
    with torch.cuda.device(x.device):
        if dx is None:
            dx = torch.empty_like(dy)
        stream = stream if stream is not None else torch.cuda.current_stream(x.device)
        st = gdn_qk_l2norm_bwd(_ptr(x), _ptr(dy), _ptr(dx), x.numel() // dk, dk, _dtype_code(x), float(eps),
                               ctypes.c_void_p(stream.cuda_stream))
        if st != 0:
            raise GdnError(st, "gdn_qk_l2norm_bwd")
    return dx


def chunk_fwd_host(q, k, v, g, beta, initial_state=None, cu_seqlens=None, scale=None,
                   opts: Optional[GdnOptions] = None, out=None, final_state=None, device_buffer=None,
                   stream: Optional[torch.cuda.Stream] = None, device=None):
    """The same pass for CPU (ideally pinned) tensors through gdn_chunk_fwd_host:
    the library copies inputs in, runs, copies results out and syncs."""
    B, T, H, dk, dv, N = _check_shapes(q, k, v, g, beta, initial_state, cu_seqlens)
    _expect("out", out, (B, T, H, dv))
    _expect("final_state", final_state, (N, H, dk, dv))
    dt = _dtype_code(q)
    f32 = torch.float32
    _check_dtypes(dict(k=k, v=v, g=g, beta=beta, initial_state=initial_state, cu_seqlens=cu_seqlens, out=out,
                       final_state=final_state, device_buffer=device_buffer),
                  dict(k=q.dtype, v=q.dtype, g=f32, beta=f32, initial_state=f32, cu_seqlens=torch.int32,
                       out=q.dtype, final_state=f32, device_buffer=torch.uint8))
    _check_placement("cpu", None, dict(q=q, k=k, v=v, g=g, beta=beta, initial_state=initial_state,
                                       cu_seqlens=cu_seqlens, out=out, final_state=final_state))
    if device_buffer is not None:
        device = device_buffer.device if device is None else torch.device(device)
        _check_placement("cuda", device, dict(device_buffer=device_buffer))
    device = torch.device(device or "cuda")
    if device.type != "cuda":
        raise ValueError("device must be a CUDA device, got %s" % device)
    with torch.cuda.device(device):
        if out is None:
            out = torch.empty(B, T, H, dv, dtype=q.dtype, pin_memory=True)
        if final_state is None:
            final_state = torch.empty(N, H, dk, dv, dtype=torch.float32, pin_memory=True)
        if device_buffer is None:
            n = gdn_chunk_fwd_host_buffer_size(B, T, H, dk, dv, N, cu_seqlens is not None,
                                               initial_state is not None, dt, opts)
            device_buffer = torch.empty(n, dtype=torch.uint8, device=device)
        stream = stream if stream is not None else torch.cuda.current_stream(device)
        st = gdn_chunk_fwd_host(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(initial_state),
                                _ptr(cu_seqlens), N, float(scale) if scale is not None else 0.0, B, T, H, dk, dv, dt,
                                _ptr(out), _ptr(final_state), _ptr(device_buffer), device_buffer.numel(),
                                ctypes.byref(opts) if opts is not None else None,
                                ctypes.c_void_p(stream.cuda_stream))
        if st != 0:
            raise GdnError(st, "gdn_chunk_fwd_host")
    return out, final_state


def chunk_bwd(q, k, v, g, beta, do, initial_state=None, cu_seqlens=None, scale=None, d_final_state=None,
              workspace=None, stream: Optional[torch.cuda.Stream] = None, check: bool = False, segments=None):
    """Gradients of sum <o, do> + <final_state, d_final_state> through
    gdn_chunk_bwd; returns fp32 (dq, dk, dv, dg, dbeta, d_initial_state).
    segments: None lets the backward's sequence-parallel plan decide how many
    segments each sequence is cut into (batched input only; see seqpar), 1
    runs each (sequence, head) whole, n > 1 forces n segments."""
    if workspace is None and cu_seqlens is None and segments != 1:
        from .seqpar import backward_segments, chunk_bwd_segmented
        ns = segments if segments is not None else backward_segments(q, v)
        if ns > 1:
            return chunk_bwd_segmented(q, k, v, g, beta, do, initial_state, scale, d_final_state, ns,
                                       stream=stream, check=check)
    B, T, H, dk, dv, N = _check_shapes(q, k, v, g, beta, initial_state, cu_seqlens)
    _expect("do", do, (B, T, H, dv))
    _expect("d_final_state", d_final_state, (N, H, dk, dv))
    dt = _dtype_code(q)
    f32, dev = torch.float32, q.device
    _check_dtypes(dict(k=k, v=v, do=do, g=g, beta=beta, initial_state=initial_state, cu_seqlens=cu_seqlens,
                       d_final_state=d_final_state, workspace=workspace),
                  dict(k=q.dtype, v=q.dtype, do=q.dtype, g=f32, beta=f32, initial_state=f32,
                       cu_seqlens=torch.int32, d_final_state=f32, workspace=torch.uint8))
    _check_placement("cuda", None, dict(q=q))
    _check_placement("cuda", dev, dict(k=k, v=v, g=g, beta=beta, do=do, initial_state=initial_state,
                                       cu_seqlens=cu_seqlens, d_final_state=d_final_state, workspace=workspace))
    with torch.cuda.device(dev):
        dq = torch.empty(B, T, H, dk, dtype=f32, device=dev)
        dk_ = torch.empty(B, T, H, dk, dtype=f32, device=dev)
        dv_ = torch.empty(B, T, H, dv, dtype=f32, device=dev)
        dg = torch.empty(B, T, H, dtype=f32, device=dev)
        db = torch.empty(B, T, H, dtype=f32, device=dev)
        ds0 = torch.empty(N, H, dk, dv, dtype=f32, device=dev)
        if workspace is None:
            n = gdn_chunk_bwd_workspace_size(B, T, H, dk, dv, N, cu_seqlens is not None, dt)
            if n == 0:
                raise GdnError(1, "gdn_chunk_bwd_workspace_size")
            workspace = torch.empty(n, dtype=torch.uint8, device=dev)
        stream = stream if stream is not None else torch.cuda.current_stream(dev)
        st = gdn_chunk_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(initial_state), _ptr(cu_seqlens),
                           N, float(scale) if scale is not None else 0.0, B, T, H, dk, dv, dt,
                           _ptr(do), _ptr(d_final_state), _ptr(dq), _ptr(dk_), _ptr(dv_), _ptr(dg), _ptr(db),
                           _ptr(ds0), _ptr(workspace), workspace.numel(), ctypes.c_void_p(stream.cuda_stream))
        if st != 0:
            raise GdnError(st, "gdn_chunk_bwd")
        if check:
            st = gdn_chunk_bwd_check(_ptr(workspace), ctypes.c_void_p(stream.cuda_stream))
            if st != 0:
                raise GdnError(st, "device check")
    return dq, dk_, dv_, dg, db, ds0


def chunk_state_grad(q, k, g, beta, do, cu_seqlens=None, scale=None, d_final_state=None, dv=None,
                     workspace=None, stream: Optional[torch.cuda.Stream] = None, check: bool = False):
    """The initial state's gradient alone (gdn_chunk_state_grad): what
    chunk_bwd returns as d_initial_state, without the other gradients.  dv
    (the value head size) defaults to do's last dimension."""
    for name, t in (("q", q), ("k", k), ("g", g), ("beta", beta), ("do", do)):
        if t is None:
            raise ValueError("%s is required" % name)
    B, T, H, dk = q.shape
    dv = do.shape[-1] if dv is None else dv
    N = cu_seqlens.numel() - 1 if cu_seqlens is not None else B
    for name, t, shape in (("k", k, (B, T, H, dk)), ("g", g, (B, T, H)), ("beta", beta, (B, T, H)),
                           ("do", do, (B, T, H, dv))):
        _expect(name, t, shape)
    _expect("d_final_state", d_final_state, (N, H, dk, dv))
    dt = _dtype_code(q)
    f32, dev = torch.float32, q.device
    _check_dtypes(dict(k=k, do=do, g=g, beta=beta, cu_seqlens=cu_seqlens, d_final_state=d_final_state,
                       workspace=workspace),
                  dict(k=q.dtype, do=q.dtype, g=f32, beta=f32, cu_seqlens=torch.int32, d_final_state=f32,
                       workspace=torch.uint8))
    _check_placement("cuda", None, dict(q=q))
    _check_placement("cuda", dev, dict(k=k, g=g, beta=beta, do=do, cu_seqlens=cu_seqlens,
                                       d_final_state=d_final_state, workspace=workspace))
    with torch.cuda.device(dev):
        ds0 = torch.empty(N, H, dk, dv, dtype=f32, device=dev)
        if workspace is None:
            n = gdn_chunk_bwd_workspace_size(B, T, H, dk, dv, N, cu_seqlens is not None, dt)
            if n == 0:
                raise GdnError(1, "gdn_chunk_bwd_workspace_size")
            workspace = torch.empty(n, dtype=torch.uint8, device=dev)
        stream = stream if stream is not None else torch.cuda.current_stream(dev)
        st = gdn_chunk_state_grad(_ptr(q), _ptr(k), _ptr(g), _ptr(beta), _ptr(cu_seqlens), N,
                                  float(scale) if scale is not None else 0.0, B, T, H, dk, dv, dt, _ptr(do),
                                  _ptr(d_final_state), _ptr(ds0), _ptr(workspace), workspace.numel(),
                                  ctypes.c_void_p(stream.cuda_stream))
        if st != 0:
            raise GdnError(st, "gdn_chunk_state_grad")
        if check:
            st = gdn_chunk_bwd_check(_ptr(workspace), ctypes.c_void_p(stream.cuda_stream))
            if st != 0:
                raise GdnError(st, "device check")
    return ds0


class _ChunkGDN(torch.autograd.Function):
    """gdn_chunk_fwd forward, gdn_chunk_bwd backward (the fp32 gradients of q,
    k, v are handed back in the inputs' dtype).  With norm_qk, q and k are first
    normalised by gdn_qk_l2norm, and their gradients go back through
    gdn_qk_l2norm_bwd in fp32."""

    @staticmethod
    def forward(ctx, q, k, v, g, beta, initial_state, cu_seqlens, scale, opts, norm_qk):
        qn, kn = qk_l2norm(q, k) if norm_qk else (q, k)
        o, final_state = chunk_fwd(qn, kn, v, g, beta, initial_state, cu_seqlens, scale, opts=opts)
        ctx.save_for_backward(q, k, qn, kn, v, g, beta, initial_state, cu_seqlens)
        ctx.scale = scale
        ctx.norm_qk = norm_qk
        return o, final_state

    @staticmethod
    def backward(ctx, do, d_final_state):
        q, k, qn, kn, v, g, beta, initial_state, cu_seqlens = ctx.saved_tensors
        if do is None:
            do = torch.zeros(*q.shape[:-1], v.shape[-1], dtype=q.dtype, device=q.device)
        dq, dk, dv, dg, dbeta, ds0 = chunk_bwd(
            qn, kn, v, g, beta, do.contiguous(), initial_state, cu_seqlens, ctx.scale,
            d_final_state.contiguous() if d_final_state is not None else None)
        if ctx.norm_qk:
            qk_l2norm_backward(q, dq, dx=dq)
            qk_l2norm_backward(k, dk, dx=dk)
        dt = q.dtype
        return (dq.to(dt), dk.to(dt), dv.to(dt), dg, dbeta, (ds0 if initial_state is not None else None),
                None, None, None, None)


def chunk_gated_delta_rule(q, k, v, g, beta, scale=None, initial_state=None, output_final_state=False,
                           cu_seqlens=None, use_qk_l2norm_in_kernel=False, cp_mode=CP_AUTO):
    """The high-level entry point with autograd: o (and the final state when
    output_final_state) from q, k [B,T,H,dk], v [B,T,H,dv] (bf16 or fp32), the
    log-decay gate g and beta [B,T,H] (fp32), an optional initial state
    [N,H,dk,dv] (fp32) and cu_seqlens (int32, packed batch with B = 1).
    Gradients flow to q, k, v, g, beta and the initial state through
    gdn_chunk_bwd.  use_qk_l2norm_in_kernel normalises q and k first: inside
    the forward pass (opts.qk_l2norm) when no gradient is needed, else by
    gdn_qk_l2norm in front of it, with gdn_qk_l2norm_bwd on the way back."""
    needs_grad = torch.is_grad_enabled() and any(
        t is not None and t.requires_grad for t in (q, k, v, g, beta, initial_state))
    q, k, v, g, beta = (t.contiguous() for t in (q, k, v, g, beta))
    if initial_state is not None:
        initial_state = initial_state.contiguous()
    in_pass = bool(use_qk_l2norm_in_kernel) and not needs_grad
    opts = default_options(qk_l2norm=1 if in_pass else 0, cp_mode=cp_mode)
    o, final_state = _ChunkGDN.apply(q, k, v, g, beta, initial_state, cu_seqlens, scale, opts,
                                     bool(use_qk_l2norm_in_kernel) and needs_grad)
    return o, (final_state if output_final_state else None)
