"""The chunked (WY) form of the GDN forward pass, written plainly in numpy fp64.

TEST INFRASTRUCTURE ONLY.  These functions restate, one step at a time, the
algebra the FlashQLA talk ("Qwen系列模型线性注意力高性能优化实践") describes, so
the tests can pin the token-by-token oracle to an independent algorithm and pin
each rewrite the CUDA path relies on:

  four-step paragraph   per chunk: (1) K K^T and its inverse, (2) W and U,
                        (3) the chunk-to-chunk state recurrence, (4) the output
  Gamma paragraph       Gamma_{ri} = gamma_r / gamma_i = exp(G_r - G_i)
  Gamma-extraction ¶    (I + A)^{-1} = Gamma ⊙ (I + A')^{-1}, A' without Gamma
  forward-merge ¶       U = T diag(beta) (V - D_gamma K S0^T)  ("V minus S first")
  difference ¶          the chunk map is affine in S0: S_end = S0 M + S*
  compute-for-memory ¶  segments keep only their last (S*, M); a scan over
                        segments; a second pass recomputes S and O
  sliding-window ¶      a head with alpha != 1 restarts from zero a window back

Derivation (ours; the pages state the steps only in prose).  Within a chunk with
start state S0 (dv x dk), G = cumsum(g), gamma = exp(G):
    u_r = beta_r (v_r - gamma_r S0 k_r - sum_{i<r} Gamma_ri (k_r.k_i) u_i)
 => (I + A) U = diag(beta) (V - D_gamma K S0^T),  A_ri = beta_r Gamma_ri k_r.k_i (i<r)
    O  = scale (D_gamma Q S0^T + (Gamma ⊙ tril(Q K^T)) U)
    S_C = gamma_C S0 + U^T diag(gamma_C / gamma) K
All arrays here use the math orientation: S is dv x dk.
"""
from __future__ import annotations

import numpy as np

from .gate import lookback_chunks

__all__ = ["wy_forward", "chunk_inverse", "inverse_rows", "correction_product",
           "cp_forward", "sliding_forward"]


def _strict_lower(x):
    return np.tril(x, -1)


def _gamma_matrix(G):
    """Gamma_{ri} = exp(G_r - G_i) for i <= r, 0 above the diagonal."""
    L = len(G)
    D = G[:, None] - G[None, :]
    out = np.exp(np.where(np.tril(np.ones((L, L), dtype=bool)), D, -np.inf))
    return out


def chunk_inverse(Kc, bc, G=None):
    """(I + A)^{-1} for one chunk.  With G given, A carries Gamma (the plain form);
    with G None, A' = diag(beta) strictlower(K K^T) (the Gamma-free form)."""
    L = Kc.shape[0]
    KK = _strict_lower(Kc @ Kc.T)
    if G is not None:
        KK = KK * _gamma_matrix(G)
    A = bc[:, None] * KK
    return np.linalg.solve(np.eye(L) + A, np.eye(L))


def inverse_rows(k, beta, cu, C):
    """T' = (I + diag(beta) strictlower(K K^T))^{-1} for every chunk and head,
    stored by token: out[t, h, :len] is row (t - t0) of its chunk's T'."""
    k = np.asarray(k, dtype=np.float64)
    beta = np.asarray(beta, dtype=np.float64)
    T, H, _ = k.shape
    out = np.zeros((T, H, C))
    for n in range(len(cu) - 1):
        for t0 in range(int(cu[n]), int(cu[n + 1]), C):
            L = min(C, int(cu[n + 1]) - t0)
            for h in range(H):
                out[t0:t0 + L, h, :L] = chunk_inverse(k[t0:t0 + L, h], beta[t0:t0 + L, h])
    return out


def wy_forward(q, k, v, g, beta, S0, scale, C, gamma_extraction=True, merged=True,
               want_output=True):
    """One sequence, one head.  q,k [T,dk]; v [T,dv]; g, beta [T]; S0 [dv,dk].
    Returns (o [T,dv], S_T [dv,dk])."""
    T = q.shape[0]
    dv = v.shape[1]
    S = np.array(S0, dtype=np.float64, copy=True)
    o = np.zeros((T, dv))
    for t0 in range(0, T, C):
        sl = slice(t0, min(T, t0 + C))
        Kc, Qc, Vc, gc, bc = k[sl], q[sl], v[sl], g[sl], beta[sl]
        G = np.cumsum(gc)
        gam = np.exp(G)
        Gam = _gamma_matrix(G)
        # step 1: the inverse
        if gamma_extraction:
            Tm = Gam * chunk_inverse(Kc, bc)
        else:
            Tm = chunk_inverse(Kc, bc, G)
        # step 2: W and U
        if merged:
            U = Tm @ (bc[:, None] * (Vc - gam[:, None] * (Kc @ S.T)))
        else:
            W = Tm @ ((bc * gam)[:, None] * Kc)
            U_tilde = Tm @ (bc[:, None] * Vc)
            U = U_tilde - W @ S.T
        # step 4 (uses the chunk's start state)
        if want_output:
            o[sl] = scale * (gam[:, None] * (Qc @ S.T) + (Gam * (Qc @ Kc.T)) @ U)
        # step 3: the state recurrence
        S = gam[-1] * S + U.T @ (np.exp(G[-1] - G)[:, None] * Kc)
    return o, S


def correction_product(k, g, beta):
    """M = prod_t alpha_t (I - beta_t k_t k_t^T), multiplied on the right in
    token order (dk x dk)."""
    dk = k.shape[1]
    M = np.eye(dk)
    for t in range(k.shape[0]):
        M = M @ (np.exp(g[t]) * (np.eye(dk) - beta[t] * np.outer(k[t], k[t])))
    return M


def _segments(nc, L):
    return [(c, min(nc, c + L)) for c in range(0, nc, L)]


def cp_forward(q, k, v, g, beta, S0, scale, C, L):
    """Sequence parallelism with correction matrices, one sequence and head.

    Segments of L chunks.  Pass 1: segment 0 runs from S0 to its true end state;
    every later segment j (but the last) runs twice from a wrong start: the
    values V from S = 0 give S*_j, and zero values from S = I give M_j (the
    correction matrix is the recurrence itself with v = 0 started from I).  Only
    each segment's final pair is kept.  A scan S_{j+1} = S_j M_j + S*_j gives
    every segment's exact start; pass 2 recomputes S and O from those starts."""
    T, dk = k.shape
    dv = v.shape[1]
    nc = -(-T // C)
    segs = _segments(nc, L)
    starts = [np.array(S0, dtype=np.float64)]
    for j, (c0, c1) in enumerate(segs[:-1]):
        sl = slice(c0 * C, min(T, c1 * C))
        if j == 0:
            _, S_end = wy_forward(q[sl], k[sl], v[sl], g[sl], beta[sl], S0, scale, C, want_output=False)
        else:
            _, S_star = wy_forward(q[sl], k[sl], v[sl], g[sl], beta[sl], np.zeros((dv, dk)), scale, C,
                                   want_output=False)
            _, M = wy_forward(q[sl], k[sl], np.zeros((sl.stop - sl.start, dk)), g[sl], beta[sl],
                              np.eye(dk), scale, C, want_output=False)
            S_end = starts[-1] @ M + S_star
        starts.append(S_end)
    o = np.zeros((T, dv))
    S = None
    for (c0, c1), S_start in zip(segs, starts):
        sl = slice(c0 * C, min(T, c1 * C))
        o[sl], S = wy_forward(q[sl], k[sl], v[sl], g[sl], beta[sl], S_start, scale, C)
    return o, S


def sliding_forward(q, k, v, g, beta, S0, scale, C, L, ln_eps):
    """Sliding-window restart, one sequence and head: segment j (starting at
    chunk c0 > 0) restarts from S = 0 at chunk c0 - w, with w the look-back
    window for ln_eps, and runs state-only up to c0; a window that reaches the
    sequence start begins from S0 instead (exact)."""
    T, dk = k.shape
    dv = v.shape[1]
    nc = -(-T // C)
    totals = np.array([g[c * C:min(T, (c + 1) * C)].sum() for c in range(nc)])
    o = np.zeros((T, dv))
    S = None
    for c0, c1 in _segments(nc, L):
        w = lookback_chunks(totals, c0, ln_eps) if c0 > 0 else 0
        b = c0 - w
        S_b = np.array(S0, dtype=np.float64) if b == 0 else np.zeros((dv, dk))
        if w:
            sl = slice(b * C, c0 * C)
            _, S_b = wy_forward(q[sl], k[sl], v[sl], g[sl], beta[sl], S_b, scale, C, want_output=False)
        sl = slice(c0 * C, min(T, c1 * C))
        o[sl], S = wy_forward(q[sl], k[sl], v[sl], g[sl], beta[sl], S_b, scale, C)
    return o, S
