"""GPU test of gdn_chunk_fwd_static, the entry point that allocates nothing.

Some callers cannot allocate device memory while they run: a server that gives
all of HBM to its own pool at start-up and forbids allocation on the request
path, or a plugin that only receives tensors from a host framework.  For them
the library keeps a fixed 64 MiB scratch array per device and runs the same
forward pass with it in place of a caller workspace.

The test calls that entry point through the C ABI twice in a row, on two
different problems (so the second call finds the first call's leftovers in the
shared array), and checks both results against gdn_chunk_fwd with a workspace
of its own: the two entry points run the same kernels with the same plan, so
the results must agree bit for bit (and within the parity tolerance of the
other GPU tests, which that implies).  The file name makes pytest collect it
last.
"""
import ctypes

import pytest
import torch

import chunked_prefill_gdn_gb300 as gdn
from chunked_prefill_gdn_gb300 import build as gdn_build
from chunked_prefill_gdn_gb300.inputs import CONFIGS, make_inputs

from gpu_helpers import MAX_ABS, REL_L2, assert_close, oracle, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    gdn_build.build()
    return gdn.load_library()


def _p(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def run_static(inp, device_status=None):
    q, v = inp["q"], inp["v"]
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    cu = inp.get("cu_seqlens")
    N = cu.numel() - 1 if cu is not None else B
    o = torch.full((B, T, H, dv), float("nan"), dtype=q.dtype, device=q.device)
    sf = torch.full((N, H, dk, dv), float("nan"), dtype=torch.float32, device=q.device)
    dt = gdn.BF16 if q.dtype == torch.bfloat16 else gdn.F32
    stream = torch.cuda.current_stream()
    st = gdn.gdn_chunk_fwd_static(_p(q), _p(inp["k"]), _p(v), _p(inp["g"]), _p(inp["beta"]),
                                  _p(inp.get("initial_state")), _p(cu), N, float(inp["scale"]),
                                  B, T, H, dk, dv, dt, _p(o), _p(sf), _p(device_status), None,
                                  ctypes.c_void_p(stream.cuda_stream))
    return st, o, sf


def run_workspace(inp):
    o, sf = gdn.chunk_fwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp.get("initial_state"),
                          inp.get("cu_seqlens"), inp["scale"], check=True)
    torch.cuda.synchronize()
    return o, sf


def problems():
    # a ragged bf16 batch with an initial state (tcgen05 fused kernel) ...
    a = CONFIGS[1].scaled(B=2, T=1000, H=4, s0_std=0.02)
    # ... then a packed varlen fp32 batch (CUDA-core fused kernel, CP on)
    b = CONFIGS[3].scaled(T=3000, H=3, n_seqs=5, dtype="f32", len_mu=6.0, len_max=1500)
    return [to_device(make_inputs(a, "cpu")), to_device(make_inputs(b, "cpu"))]


def test_static_scratch_matches_workspace_entry_point_twice(lib):
    first, second = problems()
    # call 1: NULL status pointer, the call syncs and returns the device status
    st1, o1, sf1 = run_static(first)
    assert st1 == 0, gdn.gdn_status_string(st1)
    # call 2, right after: the status word is copied to a device int32
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    st2, o2, sf2 = run_static(second, device_status=status)
    assert st2 == 0, gdn.gdn_status_string(st2)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for inp, o, sf in ((first, o1, sf1), (second, o2, sf2)):
        o_ref, sf_ref = run_workspace(inp)
        assert_close("o", oracle.to_f64(o), oracle.to_f64(o_ref), REL_L2, MAX_ABS)
        assert_close("final_state", oracle.to_f64(sf), oracle.to_f64(sf_ref), REL_L2, MAX_ABS)
        assert torch.equal(o, o_ref) and torch.equal(sf, sf_ref)


def test_static_scratch_rejects_oversized_problem(lib):
    # B=4, T=8192, H=32 needs about 132 MiB of scratch: refused before any launch
    q = torch.empty(1, dtype=torch.bfloat16, device="cuda")
    st = gdn.gdn_chunk_fwd_static(_p(q), _p(q), _p(q), _p(q), _p(q), None, None, 4, 0.0,
                                  4, 8192, 32, 128, 128, gdn.BF16, _p(q), _p(q), None, None, None)
    assert gdn.gdn_status_string(st) == "GDN_ERR_WORKSPACE"
    assert "static scratch" in gdn.gdn_last_error_detail()
