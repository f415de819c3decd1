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


# ---------------------------------------------------------------------------
# Sequence parallelism in the backward pass, on one GPU.
#
# The talk's results paragraph has the backward split with the same
# segment scheme as the forward.  One CTA of the backward kernel walks a whole
# (sequence, head, 32 value columns): a batch with few of them leaves SMs idle
# while each walks every chunk (one sequence of 2,048 chunks with 8 heads: 32
# CTAs).  Cut each sequence into NS segments at chunk boundaries:
#
#   1. the segments' forward maps (S*, M)           gdn_chunk_transition
#   2. their start states, forward scan             gdn_state_scan
#   3. each segment's backward with a zero end
#      gradient -> its own start gradient ds*       gdn_chunk_bwd
#   4. every segment's end gradient, reverse scan   gdn_state_grad_scan
#      ds_end(j) = ds_end(j+1) M(j+1)^T + ds*(j+1)
#   5. each segment's backward from its start state
#      with its end gradient: the gradients         gdn_chunk_bwd
#
# Step 5 is exact for every token (the loss restricted to a segment and its
# future is a function of the segment's start state through the segment's
# map), and segment 0's start gradient is the initial state's.  Steps 3 and 5
# are two backward passes over the tokens, run on NS times as many CTAs.

kMinSegmentChunks = 16   # a segment of the backward spans at least 1,024 tokens


def backward_segments(q, v, sms=None) -> int:
    """Segments per sequence for the backward of a batched input: the count
    that minimises waves x longest segment for the two passes, against one
    pass over whole sequences; 1 unless splitting saves a tenth (the maps,
    the scans and the allocations cost about 1-2% of a pass)."""
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    if sms is None:
        sms = torch.cuda.get_device_properties(q.device).multi_processor_count if q.is_cuda else 152
    ctas = B * H * max(1, dv // 32)
    nc = -(-T // 64)
    if ctas >= sms or nc < 16:
        return 1
    cost1 = -(-ctas // sms) * nc
    best, best_cost = 1, float(cost1)
    for ns in range(2, nc // kMinSegmentChunks + 1):
        L = -(-nc // ns)
        ns_eff = -(-nc // L)
        cost = 2.0 * (-(-ctas * ns_eff // sms)) * L
        if cost < 0.98 * best_cost:          # among near-equal plans, the fewest segments
            best, best_cost = ns_eff, cost
    return best if best_cost < 0.9 * cost1 else 1


def chunk_bwd_segmented(q, k, v, g, beta, do, initial_state, scale, d_final_state, segments,
                        stream=None, check=False):
    """chunk_bwd with every sequence of a batched input cut into `segments`
    segments at chunk boundaries (steps above); returns what chunk_bwd does."""
    from . import (KERNEL_SIMT, chunk_bwd, chunk_state_grad, chunk_transition, gdn_get_backward_kernel,
                   state_grad_scan, state_scan)
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    nc = -(-T // 64)
    L = -(-nc // segments)
    NS = -(-nc // L)
    seg_len = 64 * L
    dev = q.device
    edges = [min(T, j * seg_len) for j in range(NS)] + [T]
    cu = torch.tensor([b * T + e for b in range(B) for e in edges[:-1]] + [B * T], dtype=torch.int32, device=dev)
    pack = lambda t: t.reshape(1, B * T, *t.shape[2:])
    qp, kp, vp, gp, bp, dop = (pack(t) for t in (q, k, v, g, beta, do))
    # rank-major views: segment (b, j) is packed sequence b NS + j
    to_rm = lambda t: t.reshape(B, NS, *t.shape[1:]).transpose(0, 1).contiguous()
    from_rm = lambda t: t.transpose(0, 1).reshape(B * NS, *t.shape[2:]).contiguous()
    s_star, m = chunk_transition(kp, vp, gp, bp, cu, stream=stream, check=check)
    m_rm = to_rm(m)
    s_start = from_rm(state_scan(to_rm(s_star), m_rm, initial_state, stream=stream))
    # each segment's local map: the state gradient back from a zero end gradient
    # (the reverse recurrence alone; the CUDA-core backward when it is selected)
    if gdn_get_backward_kernel() == KERNEL_SIMT:
        ds_local = chunk_bwd(qp, kp, vp, gp, bp, dop, s_start, cu, scale, None, stream=stream, check=check,
                             segments=1)[5]
    else:
        ds_local = chunk_state_grad(qp, kp, gp, bp, dop, cu, scale, None, dv=dv, stream=stream, check=check)
    ds_end = from_rm(state_grad_scan(to_rm(ds_local), m_rm, d_final_state, stream=stream))
    dq, dk_, dv_, dg, db, ds0 = chunk_bwd(qp, kp, vp, gp, bp, dop, s_start, cu, scale, ds_end, stream=stream,
                                          check=check, segments=1)
    unpack = lambda t: t.reshape(B, T, *t.shape[2:])
    return (unpack(dq), unpack(dk_), unpack(dv_), unpack(dg), unpack(db),
            ds0.reshape(B, NS, H, dk, dv)[:, 0].contiguous())
