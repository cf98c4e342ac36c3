"""One problem split over several processes (one per GPU), through torch.distributed.

The work separates two ways:

* **Heads.**  The (b, h) heads are independent problems.  Rank r takes a contiguous range of
  the flattened B*H heads (``head_range``) and runs the forward on it; no data crosses
  ranks.

* **Sequence.**  Rank r takes a contiguous range of rows of every head
  (``sequence_range``).  The one exchange is the carried state of the chunked order
  ("attention と線形の間", section 2: the state before a chunk is the sum of the earlier
  chunks' phi(K)^T V), taken at segment granularity.  Every rank computes its segment's own
  total T_r = sum_t w_t phi(k_t) v_t^T and zeta_r = sum_t w_t phi(k_t) (``la_chunked_state``;
  w_t = 1, or gamma^(rows after t in the segment) with the Retention decay), the ranks
  all-gather the totals (``gather_totals``), and rank r starts its own pass from the
  exclusive prefix P_r = sum_{r' < r} gamma^(rows of segments r'+1 .. r-1) T_r'
  (``la_state_combine`` applied in rank order, then ``la_chunked_fwd_init``).  In exact
  arithmetic the concatenated rows equal one pass over the whole sequence.

The collective runs on device tensors under NCCL and on host copies under gloo.  The
arithmetic of every step runs in the library's kernels; this module only moves the fp32
totals between processes.
"""
from __future__ import annotations

import math


def head_range(n_heads: int, world: int, rank: int) -> tuple[int, int]:
    """Rank `rank`'s contiguous share [h0, h1) of n_heads heads: sizes differ by at most 1,
    lower ranks take the larger shares.  Empty when there are more ranks than heads."""
    if world <= 0 or not 0 <= rank < world or n_heads < 0:
        raise ValueError("need world > 0, 0 <= rank < world, n_heads >= 0")
    base, extra = divmod(n_heads, world)
    h0 = rank * base + min(rank, extra)
    return h0, h0 + base + (1 if rank < extra else 0)


def sequence_range(L: int, world: int, rank: int, align: int = 64) -> tuple[int, int]:
    """Rank `rank`'s contiguous rows [t0, t1) of a length-L sequence.  Boundaries fall on
    multiples of `align` (a chunk size), so each segment's chunks are chunks of the whole
    sequence; the last rank takes the ragged end."""
    if world <= 0 or not 0 <= rank < world or L < 0 or align <= 0:
        raise ValueError("need world > 0, 0 <= rank < world, L >= 0, align > 0")
    blocks = math.ceil(L / align)
    b0, b1 = head_range(blocks, world, rank)
    return min(L, b0 * align), min(L, b1 * align)


def gather_totals(S, z, rows: int, group=None):
    """All-gather every rank's segment total: returns ([S_0 .. S_{n-1}], [z_0 ..] or None,
    [rows_0 ..]) in rank order, on S's device.  S [B, H, D, dv] and z [B, H, D] (or None on
    every rank) share one float dtype; every rank passes the same shapes.  Work queued on
    the current stream that produces S and z is complete before they are shipped."""
    import torch
    import torch.distributed as dist
    world = dist.get_world_size(group)
    on_dev = dist.get_backend(group) == "nccl"
    dev = S.device
    move = (lambda t: t) if on_dev else (lambda t: t.cpu())
    ship_dev = dev if on_dev else torch.device("cpu")
    flat = [move(S.contiguous().reshape(-1))]
    if z is not None:
        flat.append(move(z.contiguous().reshape(-1)))
    flat.append(torch.tensor([float(rows)], dtype=S.dtype, device=ship_dev))
    payload = torch.cat(flat)
    parts = [torch.empty_like(payload) for _ in range(world)]
    dist.all_gather(parts, payload, group=group)
    nS = S.numel()
    nz = 0 if z is None else z.numel()
    Ss = [p[:nS].reshape(S.shape).to(dev) for p in parts]
    zs = None if z is None else [p[nS:nS + nz].reshape(z.shape).to(dev) for p in parts]
    rws = [int(p[-1].item()) for p in parts]
    return Ss, zs, rws


def sequence_parallel_fwd(q, k, v, group=None, C=64, feature_map="identity", omega=None,
                          normalize=False, gamma=1.0):
    """This rank's rows of a causal forward whose sequence is cut across the ranks of
    `group` in rank order: q, k [B, H, Lr, dk] and v [B, H, Lr, dv] are this rank's segment
    of the same heads on every rank (CUDA tensors).  Returns this rank's output rows
    [B, H, Lr, dv]; concatenated in rank order they are the forward over the whole sequence
    (plain mask, or the Retention decay for gamma < 1).  Runs on the current stream."""
    import torch
    import torch.distributed as dist

    from . import (LA_OK, LAError, chunked_fwd_init, chunked_state, la_state_combine)
    rank = dist.get_rank(group)
    B, H, Lr, _ = k.shape
    dv = v.shape[-1]
    stream = torch.cuda.current_stream(q.device).cuda_stream
    S, z = chunked_state(k, v, feature_map=feature_map, omega=omega, gamma=gamma,
                         normalize=normalize, stream=stream)
    Ss, zs, rows = gather_totals(S, z, Lr, group)
    D = S.shape[2]
    P = torch.zeros_like(S)
    Pz = torch.zeros_like(z) if z is not None else None
    for r in range(rank):
        # P <- gamma^(rows of segment r) P + T_r: the earlier prefix decays over segment r
        factor = 1.0 if gamma == 1.0 else float(gamma) ** rows[r]
        rc = la_state_combine(P.data_ptr(), Pz.data_ptr() if Pz is not None else None,
                              Ss[r].data_ptr(), zs[r].data_ptr() if zs is not None else None,
                              B, H, D, dv, factor, stream)
        if rc != LA_OK:
            raise LAError(rc, "la_state_combine")
    return chunked_fwd_init(q, k, v, P, Pz, C=C, feature_map=feature_map, omega=omega,
                            normalize=normalize, gamma=gamma, stream=stream)
