"""The backward pass of the GDN recurrence, in fp64 (oracle side).

TEST INFRASTRUCTURE ONLY.

The talk "Qwen系列模型线性注意力高性能优化实践" reports a backward pass for the
chunked prefill (its backward paragraph: gradients of q, k, v, the gate and
beta, with the dA + dA^T terms merged); it prints no formulas.  This module
restates the gradients of the recurrence itself, token by token, from the
chain rule — the definition a chunked CUDA backward has to reproduce.

Forward (math orientation, S is dv x dk; per sequence and head):

    A_t = alpha_t (I - beta_t k_t k_t^T),     alpha_t = exp(g_t)
    S_t = S_{t-1} A_t + beta_t v_t k_t^T,     o_t = scale S_t q_t

Given upstream gradients do_t and dS_T (the final state's), let G_t be the total
gradient of the loss with respect to S_t.  Walking t = T .. 1:

    G_t   = G_{t+1} A_{t+1}^T + scale do_t q_t^T          (G_{T+1} A^T := dS_T)
    dq_t  = scale S_t^T do_t
    dv_t  = beta_t G_t k_t
    dA_t  = S_{t-1}^T G_t                                  (dk x dk)
    dbeta_t = v_t^T G_t k_t - alpha_t k_t^T dA_t k_t
    dk_t  = beta_t G_t^T v_t - alpha_t beta_t (dA_t + dA_t^T) k_t
    dg_t  = alpha_t (tr dA_t - beta_t k_t^T dA_t k_t)
    dS_0  = G_1 A_1^T

Loss convention: L = sum_t <o_t, do_t> + <S_T, dS_T>, so these are exact
derivatives of L (the tests pin them to central finite differences of the
forward oracle).  The states S_0 .. S_T are kept, so this is for small cases.
Layouts are the library's: q, k [.., T, H, dk]; v, o [.., T, H, dv]; g, beta
[.., T, H]; states [N, H, dk, dv] with element [j][i] = S[i][j].
"""
from __future__ import annotations

import numpy as np

from . import flatten_batch, to_f64

__all__ = ["gdn_backward_reference"]


def _unit_backward(q, k, v, g, beta, S0, do, dST, scale):
    """One sequence and head.  q, k: [T, dk]; v, do: [T, dv]; g, beta: [T];
    S0, dST: [dv, dk] (math orientation).  Returns dq, dk, dv, dg, dbeta, dS0."""
    T, dk = q.shape
    dv = v.shape[1]
    alpha = np.exp(g)
    # forward, keeping every state
    S = np.empty((T + 1, dv, dk))
    S[0] = S0
    A = np.empty((T, dk, dk))
    for t in range(T):
        A[t] = alpha[t] * (np.eye(dk) - beta[t] * np.outer(k[t], k[t]))
        S[t + 1] = S[t] @ A[t] + beta[t] * np.outer(v[t], k[t])
    dq = np.zeros((T, dk))
    dk_ = np.zeros((T, dk))
    dv_ = np.zeros((T, dv))
    dg = np.zeros(T)
    db = np.zeros(T)
    G = dST.copy()                       # gradient with respect to S_T, before o_T's term
    for t in range(T - 1, -1, -1):       # token t here is t + 1 in the docstring
        St, Sprev = S[t + 1], S[t]
        G = G + scale * np.outer(do[t], q[t])
        dq[t] = scale * St.T @ do[t]
        dv_[t] = beta[t] * (G @ k[t])
        dA = Sprev.T @ G
        kdak = k[t] @ dA @ k[t]
        db[t] = v[t] @ G @ k[t] - alpha[t] * kdak
        dk_[t] = beta[t] * (G.T @ v[t]) - alpha[t] * beta[t] * ((dA + dA.T) @ k[t])
        dg[t] = alpha[t] * (np.trace(dA) - beta[t] * kdak)
        G = G @ A[t].T
    return dq, dk_, dv_, dg, db, G


def gdn_backward_reference(q, k, v, g, beta, initial_state=None, cu_seqlens=None, scale=None, do=None,
                           d_final_state=None):
    """Gradients of L = sum <o, do> + <final_state, d_final_state> with respect
    to q, k, v, g, beta and the initial state, in fp64.

    Inputs as gdn_reference (torch tensors or arrays, batched [B, T, ...] or
    packed with cu_seqlens); do like o; d_final_state like the final state (or
    None for zero).  Returns (dq, dk, dv, dg, dbeta, d_initial_state), the first
    five packed [total_T, H, ...], the last [N, H, dk, dv] ([j][i] = dS[i][j])."""
    qf, kf, vf, gf, bf, cu = flatten_batch(q, k, v, g, beta, cu_seqlens)
    do_f = to_f64(do)
    if do_f.ndim == 4:
        do_f = do_f.reshape(-1, *do_f.shape[2:])
    H, dk = qf.shape[1], qf.shape[2]
    dv = vf.shape[2]
    N = len(cu) - 1
    if scale is None:
        scale = dk ** -0.5
    s0 = to_f64(initial_state)
    dsT = to_f64(d_final_state)
    out = [np.zeros_like(qf), np.zeros_like(kf), np.zeros_like(vf), np.zeros_like(gf), np.zeros_like(bf),
           np.zeros((N, H, dk, dv))]
    for n in range(N):
        a, b = int(cu[n]), int(cu[n + 1])
        for h in range(H):
            S0 = s0[n, h].T if s0 is not None else np.zeros((dv, dk))
            dST = dsT[n, h].T if dsT is not None else np.zeros((dv, dk))
            r = _unit_backward(qf[a:b, h], kf[a:b, h], vf[a:b, h], gf[a:b, h], bf[a:b, h], S0,
                               do_f[a:b, h], dST, scale)
            out[0][a:b, h], out[1][a:b, h], out[2][a:b, h] = r[0], r[1], r[2]
            out[3][a:b, h], out[4][a:b, h] = r[3], r[4]
            out[5][n, h] = r[5].T
    return tuple(out)
