"""Inter-card sequence parallelism: one long batch of sequences split along
time over the ranks of a process group, one GPU per rank.

The FlashQLA talk "Qwen系列模型线性注意力高性能优化实践" describes intra-card
sequence parallelism in three steps (each segment's affine map, a scan over
segments, the recompute from exact starts) and notes that the algorithm does
not tell cards from segments; its timeline paragraph lists inter-card sequence
parallelism as the natural extension.  Here the segments are the ranks:

  1. every rank: (S*_r, M_r) = the affine map of its slice on the state,
     S_end = S_start M_r + S*_r                   (gdn_chunk_transition)
  2. all ranks: all-gather of the maps             (the process group's collective)
  3. every rank: s_start = the scan of the maps   (gdn_state_scan)
  4. every rank: its slice from its start state   (gdn_chunk_fwd)

Rank r holds tokens [r T / R, (r + 1) T / R) of every sequence (any split
works: each rank passes its own slice; with cu_seqlens, sequence n's slice on
every rank is the n-th packed sequence of that rank).  The exchange per rank is
one map per (sequence, head): dk x dv + dk x dk fp32.  Every rank gets its
slice of o; the last rank's end state is the sequences' final state.

All arithmetic runs in the library's CUDA kernels; this module only calls them
and the collective.
"""
from __future__ import annotations

from typing import Callable, NamedTuple, Optional

import torch


class SeqParOps(NamedTuple):
    """The three compute steps (so the exchange and the rank bookkeeping can
    be tested apart from the GPU)."""
    transition: Callable   # (k, v, g, beta, cu_seqlens) -> (s_star, m)
    scan: Callable         # (s_star [R,...], m [R,...], s0) -> s_start [R,...]
    forward: Callable      # (q, k, v, g, beta, s_start, cu_seqlens, scale, opts) -> (o, s_end)


def _library_ops() -> SeqParOps:
    from . import chunk_fwd, chunk_transition, state_scan

    def forward(q, k, v, g, beta, s_start, cu_seqlens, scale, opts):
        return chunk_fwd(q, k, v, g, beta, s_start, cu_seqlens, scale, opts=opts, check=True)

    return SeqParOps(transition=lambda k, v, g, beta, cu: chunk_transition(k, v, g, beta, cu, check=True),
                     scan=lambda s, m, s0: state_scan(s, m, s0), forward=forward)


def chunk_fwd_sequence_parallel(q, k, v, g, beta, initial_state=None, cu_seqlens=None, scale=None, group=None,
                                opts=None, ops: Optional[SeqParOps] = None):
    """This rank's part of a GDN forward pass whose sequences are split along
    time over the ranks of `group` (torch.distributed; one rank per GPU).
    q, k, v, g, beta (and cu_seqlens) are this rank's slice; initial_state is
    the sequences' initial state, the same tensor (or None) on every rank.
    Returns (o of this slice, the state at the end of this slice); on the last
    rank that state is the sequences' final state."""
    import torch.distributed as dist
    ops = ops or _library_ops()
    R = dist.get_world_size(group)
    r = dist.get_rank(group)
    s_star, m = ops.transition(k, v, g, beta, cu_seqlens)
    all_s = [torch.empty_like(s_star) for _ in range(R)]
    all_m = [torch.empty_like(m) for _ in range(R)]
    dist.all_gather(all_s, s_star.contiguous(), group=group)
    dist.all_gather(all_m, m.contiguous(), group=group)
    s_start = ops.scan(torch.stack(all_s), torch.stack(all_m), initial_state)[r].contiguous()
    return ops.forward(q, k, v, g, beta, s_start, cu_seqlens, scale, opts)
