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

__all__ = ["gdn_backward_reference", "gdn_backward_chunked"]


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


# ----------------------------------------------------------------------------
# The same gradients in the chunked (WY) form: the algebra a chunked backward
# kernel runs, written out one chunk at a time (math orientation, S dv x dk).
#
# Forward of one chunk (C tokens, start state S0, chunk-local G = cumsum g,
# gamma = exp(G), Gamma_ri = exp(G_r - G_i), e_i = gamma_C / gamma_i):
#     A  = strictlower(diag(beta) (Gamma ⊙ K K^T)),  T = (I + A)^{-1}
#     B  = diag(beta) (V - D_gamma K S0^T),           U = T B
#     M  = Gamma ⊙ tril(Q K^T)                        (diagonal included)
#     O  = scale (D_gamma Q S0^T + M U)
#     S_C = gamma_C S0 + U^T D_e K
# Backward, given dO and dS_C (all by the chain rule):
#     dU = scale M^T dO + D_e K dS_C^T          dM = scale dO U^T (lower part)
#     dB = T^T dU                               dA = -dB U^T (strictly lower part)
#     dV = diag(beta) dB                        dX = -diag(beta) dB,  X = D_gamma K S0^T
#     P  = dA ⊙ Gamma ⊙ beta_r (strictly lower), R = dM ⊙ Gamma (lower)
#     dK = P K + P^T K + R^T Q + D_gamma dX S0 + D_e U dS_C
#     dQ = R K + scale D_gamma dO S0
#     dS0 = scale dO^T D_gamma Q + dX^T D_gamma K + gamma_C dS_C      (to the chunk before)
#     dbeta_r = (V - X)_r . dB_r + sum_{i<r} dA_ri Gamma_ri k_r.k_i
#     dG from every place G enters (Gamma, gamma, gamma_C, e), then dg = the
#     reverse cumsum of dG inside the chunk.
# The merged P K + P^T K is the "dA + dA^T" of the talk's backward paragraph.
# ----------------------------------------------------------------------------

def _chunk_backward(q, k, v, g, beta, S0, dO, dSC, scale):
    """One chunk.  q, k: [C, dk]; v, dO: [C, dv]; g, beta: [C]; S0, dSC: [dv, dk].
    Returns dq, dk, dv, dg, dbeta, dS0."""
    C = q.shape[0]
    G = np.cumsum(g)
    gam = np.exp(G)
    gC = gam[-1]
    Gam = np.exp(G[:, None] - G[None, :])
    low = np.tril(np.ones((C, C)), -1)            # strictly lower
    lowd = np.tril(np.ones((C, C)))               # lower with the diagonal
    KK = k @ k.T
    A = low * (beta[:, None] * Gam * KK)
    T = np.linalg.inv(np.eye(C) + A)
    X = gam[:, None] * (k @ S0.T)                  # D_gamma K S0^T
    B = beta[:, None] * (v - X)
    U = T @ B
    QK = q @ k.T
    M = lowd * Gam * QK
    e = gC / gam
    # backward
    dU = scale * M.T @ dO + e[:, None] * (k @ dSC.T)
    dM = lowd * (scale * dO @ U.T)
    dB = T.T @ dU
    dA = low * (-dB @ U.T)
    dV = beta[:, None] * dB
    dX = -beta[:, None] * dB
    P = dA * Gam * beta[:, None]
    R = dM * Gam
    dK = P @ k + P.T @ k + R.T @ q + gam[:, None] * (dX @ S0) + e[:, None] * (U @ dSC)
    dQ = R @ k + scale * gam[:, None] * (dO @ S0)
    dS0 = scale * dO.T @ (gam[:, None] * q) + dX.T @ (gam[:, None] * k) + gC * dSC
    dbeta = np.sum((v - X) * dB, axis=1) + np.sum(dA * Gam * KK, axis=1)
    # gradient with respect to G (then g)
    dGam = low * dA * beta[:, None] * KK + dM * QK          # where Gamma enters A and M
    dG = np.sum(dGam * Gam, axis=1) - np.sum(dGam * Gam, axis=0)
    dgam = scale * np.sum(dO * (q @ S0.T), axis=1) + np.sum(dX * (k @ S0.T), axis=1)   # D_gamma in O and X
    dG += dgam * gam
    de = np.sum(U * (k @ dSC.T), axis=1)                    # e_i = exp(G_C - G_i)
    dG -= de * e
    dG[-1] += np.sum(de * e) + gC * np.sum(dSC * S0)         # e's numerator and gamma_C S0
    dg = np.cumsum(dG[::-1])[::-1]
    return dQ, dK, dV, dg, dbeta, dS0


def gdn_backward_chunked(q, k, v, g, beta, initial_state=None, cu_seqlens=None, scale=None, do=None,
                         d_final_state=None, C: int = 64):
    """gdn_backward_reference computed chunk by chunk in the WY form: the chunk
    start states come from a forward sweep, then the chunks are walked in
    reverse, each passing dS0 to the one before.  Same arguments and results."""
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
        starts = list(range(a, b, C))
        for h in range(H):
            S = s0[n, h].T.copy() if s0 is not None else np.zeros((dv, dk))
            chunk_S0 = []
            for t0 in starts:                            # forward: the state at each chunk start
                chunk_S0.append(S.copy())
                for t in range(t0, min(t0 + C, b)):
                    At = np.exp(gf[t, h]) * (np.eye(dk) - bf[t, h] * np.outer(kf[t, h], kf[t, h]))
                    S = S @ At + bf[t, h] * np.outer(vf[t, h], kf[t, h])
            dS = dsT[n, h].T.copy() if dsT is not None else np.zeros((dv, dk))
            for ci in range(len(starts) - 1, -1, -1):
                t0 = starts[ci]
                t1 = min(t0 + C, b)
                r = _chunk_backward(qf[t0:t1, h], kf[t0:t1, h], vf[t0:t1, h], gf[t0:t1, h], bf[t0:t1, h],
                                    chunk_S0[ci], do_f[t0:t1, h], dS, scale)
                out[0][t0:t1, h], out[1][t0:t1, h], out[2][t0:t1, h] = r[0], r[1], r[2]
                out[3][t0:t1, h], out[4][t0:t1, h] = r[3], r[4]
                dS = r[5]
            out[5][n, h] = dS.T
    return tuple(out)
