"""Gate-side quantities of the chunked method, in fp64 (oracle side).

TEST INFRASTRUCTURE ONLY.

* chunk-local inclusive cumsum of the log gate: chunks of C tokens start at
  each sequence's first token; G_r = sum_{j <= r} g_j inside a chunk.  The talk
  ("Qwen系列模型线性注意力高性能优化实践", SFU paragraph) keeps the gate product
  in log space so that gamma_s / gamma_t = exp(G_s - G_t) never divides by a
  vanishing gamma.
* per-chunk totals G_C (the last valid row of each chunk).
* per (sequence, head) flag: alpha not identically 1, i.e. some g != 0
  (sliding-window paragraph: a head whose forget gate is not identically one has
  a finite window).
* look-back window: for a segment starting at chunk c0, the least number w of
  whole chunks before c0 such that the summed chunk totals of chunks
  c0-w .. c0-1 are <= ln(eps); w stops at the sequence start (then the restart
  is exact).
"""
from __future__ import annotations

import math

import numpy as np

__all__ = ["chunk_local_cumsum", "chunk_totals", "head_flags", "lookback_chunks", "chunk_table"]


def chunk_table(cu, C):
    """List of (seq, t0, length) for every chunk, sequences in order."""
    out = []
    for n in range(len(cu) - 1):
        for t0 in range(int(cu[n]), int(cu[n + 1]), C):
            out.append((n, t0, min(C, int(cu[n + 1]) - t0)))
    return out


def chunk_local_cumsum(g, cu, C):
    """g [T, H] (packed) -> G [T, H], inclusive cumsum restarted at every chunk."""
    g = np.asarray(g, dtype=np.float64)
    G = np.zeros_like(g)
    for _, t0, ln in chunk_table(cu, C):
        G[t0:t0 + ln] = np.cumsum(g[t0:t0 + ln], axis=0)
    return G


def chunk_totals(g, cu, C):
    """[num_chunks, H]: sum of g over each chunk."""
    g = np.asarray(g, dtype=np.float64)
    return np.stack([g[t0:t0 + ln].sum(axis=0) for _, t0, ln in chunk_table(cu, C)])


def head_flags(g, cu):
    """[N, H] int: 1 when some g != 0 in that sequence and head."""
    g = np.asarray(g)
    return np.stack([(g[int(cu[n]):int(cu[n + 1])] != 0).any(axis=0).astype(np.int32)
                     for n in range(len(cu) - 1)])


def lookback_chunks(totals_of_seq, c0, ln_eps):
    """totals_of_seq [nc] (one head) -> whole chunks to step back from chunk c0."""
    acc = 0.0
    w = 0
    while w < c0:
        acc += float(totals_of_seq[c0 - 1 - w])
        w += 1
        if acc <= ln_eps:
            break
    return w
