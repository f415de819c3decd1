"""fp64 CPU oracle for the GDN chunked-prefill forward pass.

TEST INFRASTRUCTURE ONLY.  Only tests/, the package-root smoke() check and the
CPU-baseline leg of bench.py may import this package.  The CUDA library never
does, and this package imports nothing from the library.

Contents
  gdn_reference      the token-by-token recurrence (C, fp64, OpenMP) — the
                     definition every CUDA result is compared against
  gate               chunk-local gate cumsum, head flags, look-back windows
  chunked            the chunked (WY) method written plainly in numpy fp64:
                     used to pin the recurrence and the pages' algebra

Parity pins: see tests/test_oracle_pins.py (closed forms, invariants, brute
force against the chunked algebra, planted-mistake sensitivity).
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import numpy as np

from . import build as _build

__all__ = ["gdn_reference", "oracle_threads", "to_f64", "flatten_batch"]

_lib = None


def _load():
    global _lib
    if _lib is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        dp = ctypes.POINTER(ctypes.c_double)
        lib.gdn_oracle_fwd.restype = ctypes.c_int
        lib.gdn_oracle_fwd.argtypes = [dp, dp, dp, dp, dp, dp,
                                       ctypes.POINTER(ctypes.c_int64), ctypes.c_int, ctypes.c_int,
                                       ctypes.c_int, ctypes.c_int, ctypes.c_double, ctypes.c_int,
                                       ctypes.c_int, ctypes.c_int, dp, dp]
        lib.gdn_oracle_max_threads.restype = ctypes.c_int
        _lib = lib
    return _lib


def oracle_threads() -> int:
    """OpenMP threads the oracle runs with."""
    return int(_load().gdn_oracle_max_threads())


def to_f64(x) -> np.ndarray:
    """Exact upcast of a torch tensor (any float dtype, any device) or array."""
    if x is None:
        return None
    try:
        import torch
        if isinstance(x, torch.Tensor):
            return x.detach().to("cpu", torch.float64).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(x, dtype=np.float64)


def flatten_batch(q, k, v, g, beta, cu_seqlens):
    """[B,T,H,d] -> packed [B*T,H,d] plus int64 cu_seqlens [N+1]."""
    q, k, v, g, beta = (to_f64(a) for a in (q, k, v, g, beta))
    if q.ndim == 4:
        B, T = q.shape[:2]
        q = q.reshape(B * T, *q.shape[2:])
        k = k.reshape(B * T, *k.shape[2:])
        v = v.reshape(B * T, *v.shape[2:])
        g = g.reshape(B * T, -1)
        beta = beta.reshape(B * T, -1)
        if cu_seqlens is None:
            cu = np.arange(B + 1, dtype=np.int64) * T
        else:
            if B != 1:
                raise ValueError("cu_seqlens needs B == 1")
            cu = to_f64(cu_seqlens).astype(np.int64)
    else:
        cu = (np.array([0, q.shape[0]], dtype=np.int64) if cu_seqlens is None
              else to_f64(cu_seqlens).astype(np.int64))
    return q, k, v, g, beta, cu


def gdn_reference(q, k, v, g, beta, initial_state=None, cu_seqlens=None, scale=None,
                  heads: Optional[Sequence[int]] = None, rows: Optional[Sequence[int]] = None,
                  seqs: Optional[Sequence[int]] = None, threads: int = 0, mutation: int = 0,
                  row_block: Optional[int] = None):
    """The GDN forward pass in fp64, token by token.

    Inputs may be torch tensors or numpy arrays in the library's layouts
    (q,k [B,T,H,dk] or packed [T,H,dk]; v [.., dv]; g, beta [.., H];
    initial_state [N,H,dk,dv] or None; cu_seqlens [N+1] or None).
    scale defaults to dk ** -0.5.

    `seqs`, `heads` and `rows` select a subset of sequences, heads and value
    rows (state rows evolve independently, so a subset is computed exactly as in
    the full problem).  Returns (o, final_state) as float64 arrays:
    o [T_sel, H_sel, dv_sel] packed over the selected sequences,
    final_state [N_sel, H_sel, dk, dv_sel].
    """
    q, k, v, g, beta, cu = flatten_batch(q, k, v, g, beta, cu_seqlens)
    s0 = to_f64(initial_state)
    n_seqs = len(cu) - 1
    H, dk = q.shape[1], q.shape[2]
    if scale is None:
        scale = dk ** -0.5
    if seqs is not None:
        seqs = list(seqs)
        idx = np.concatenate([np.arange(cu[n], cu[n + 1]) for n in seqs]) if seqs else np.zeros(0, np.int64)
        lens = [int(cu[n + 1] - cu[n]) for n in seqs]
        q, k, v, g, beta = q[idx], k[idx], v[idx], g[idx], beta[idx]
        cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
        if s0 is not None:
            s0 = s0[seqs]
        n_seqs = len(seqs)
    if heads is not None:
        heads = list(heads)
        q, k, v, g, beta = q[:, heads], k[:, heads], v[:, heads], g[:, heads], beta[:, heads]
        if s0 is not None:
            s0 = s0[:, heads]
        H = len(heads)
    if rows is not None:
        rows = list(rows)
        v = v[:, :, rows]
        if s0 is not None:
            s0 = s0[..., rows]
    dv = v.shape[2]
    q, k, v, g, beta = (np.ascontiguousarray(a, dtype=np.float64) for a in (q, k, v, g, beta))
    if s0 is not None:
        s0 = np.ascontiguousarray(s0, dtype=np.float64)
    cu = np.ascontiguousarray(cu, dtype=np.int64)
    o = np.zeros((q.shape[0], H, dv), dtype=np.float64)
    sf = np.zeros((n_seqs, H, dk, dv), dtype=np.float64)
    if row_block is None:
        # enough tasks to keep every thread busy even with few heads
        nt = max(1, threads or oracle_threads())
        units = max(1, n_seqs * H)
        blocks_per_unit = max(1, -(-4 * nt // units))
        row_block = max(1, dv // blocks_per_unit)
    lib = _load()
    dp = ctypes.POINTER(ctypes.c_double)

    def p(a):
        return a.ctypes.data_as(dp) if a is not None else None

    rc = lib.gdn_oracle_fwd(p(q), p(k), p(v), p(g), p(beta), p(s0),
                            cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), n_seqs, H, dk, dv,
                            float(scale), int(row_block), int(threads), int(mutation), p(o), p(sf))
    if rc != 0:
        raise RuntimeError("gdn_oracle_fwd failed with code %d" % rc)
    return o, sf
