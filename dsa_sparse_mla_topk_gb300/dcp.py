"""Decode context parallelism (DCP) for DSA sparse MLA: the KV positions of a
context are sharded round-robin over G ranks and one exchange step merges
the ranks' work.

"GLM-5.3 Optimizations, Part 2: PCP, DCP, and Hybrid HiSparse on 16 H200s",
DCP: the KV cache of a long context is split by token across the ranks of a
group, so that each holds 1/G of it.  For DSA this needs two exchanges:

1. selection: rank r owns the positions p with p % G == r (local index
   p // G).  Every position the global top-k picks is among its owner's local
   top-k, so the union of the G local top-k lists (all-gathered as (score,
   position) candidates) contains the global selection; reselecting the k best
   candidates with the same tie rule (score descending, position ascending)
   gives exactly the single-rank result;
2. attention: each rank runs the Partial over the selected positions it owns
   (two KV splits, fp32 partials with their log-sum-exp) and the ranks
   all-gather the partials, which merge exactly as the Combine step does.

The exchange logic here is plain torch.distributed over the ranks' tensors;
the compute steps are the library's kernels (``dsa_topk_select``,
``dsa_sparse_mla_fwd``, ``dsa_combine``) unless other implementations with the
same contract are passed in.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Callable

import torch
import torch.distributed as dist


def owned_positions(num_positions: int, rank: int, world: int) -> torch.Tensor:
    """Global positions a rank holds, in local order (local index j = p // G)."""
    return torch.arange(rank, num_positions, world, dtype=torch.int64)


def local_q_pos(q_pos: torch.Tensor, rank: int, world: int) -> torch.Tensor:
    """Local index of the last position a query sees on this rank, -1 when it
    sees none there (q_pos < rank)."""
    qp = q_pos.to(torch.int64)
    return torch.where(qp >= rank, torch.div(qp - rank, world, rounding_mode="floor"), torch.full_like(qp, -1))


@dataclass
class Compute:
    """The three compute steps.  topk(scores, q_pos, k) -> int32 idx [num_q, k]
    (ascending, -1 padded; rows with q_pos < 0 select nothing); partial(idx) ->
    (o_part fp32 [2, num_q, H, d_latent], lse_part [2, num_q, H]) over this
    rank's pool; combine(o_part, lse_part) -> (out, lse)."""
    topk: Callable
    partial: Callable
    combine: Callable


def library_compute(q, kv, kv_scale, block_table, q_req, *, d_latent, d_rope, page_size, softmax_scale,
                    stream=None) -> Compute:
    """The library's kernels on this rank's device and KV pool."""
    import dsa_sparse_mla_topk_gb300 as dsa

    def topk(scores, q_pos, k):
        out = torch.full((scores.shape[0], k), -1, dtype=torch.int32, device=scores.device)
        rows = q_pos >= 0  # rows that see nothing on this rank keep -1
        if bool(rows.any()):
            sel = rows.nonzero().flatten()
            out[sel] = dsa.topk_select(scores[sel].contiguous(), q_pos[sel].to(torch.int32).contiguous(), k,
                                       stream=stream)
        return out

    def partial(idx):
        return dsa.sparse_mla_fwd(q, kv, kv_scale, block_table, q_req, idx.contiguous(), d_latent=d_latent,
                                  d_rope=d_rope, page_size=page_size, softmax_scale=softmax_scale, num_splits=2,
                                  stream=stream)

    def combine(o_part, lse_part):
        return dsa.combine(o_part.contiguous(), lse_part.contiguous(), stream=stream)

    return Compute(topk, partial, combine)


def _all_gather(t: torch.Tensor, world: int, group=None) -> torch.Tensor:
    if world == 1:
        return t.unsqueeze(0)
    parts = [torch.empty_like(t) for _ in range(world)]
    dist.all_gather(parts, t.contiguous(), group=group)
    return torch.stack(parts)


def dcp_sparse_mla_topk(scores_local: torch.Tensor, q_pos: torch.Tensor, k: int, compute: Compute, *, group=None):
    """One DCP pass on this rank.  ``scores_local`` [num_q, ld_local] holds the
    indexer scores of this rank's positions (column j = global position
    j * G + rank); ``q_pos`` the global positions of the query tokens.
    Returns (out, lse, idx) with idx the global selection (ascending, -1
    padded), identical on every rank."""
    # without a process group this is a group of one (every position local)
    world = dist.get_world_size(group) if dist.is_initialized() else 1
    rank = dist.get_rank(group) if dist.is_initialized() else 0
    num_q = q_pos.shape[0]
    dev = scores_local.device
    # 1. local selection -> (score, global position) candidates of every rank
    lq = local_q_pos(q_pos, rank, world).to(dev)
    idx_l = compute.topk(scores_local, lq, k).to(torch.int64)
    valid = idx_l >= 0
    cand_pos = torch.where(valid, idx_l * world + rank, torch.full_like(idx_l, -1))
    cand_score = torch.where(valid, torch.gather(scores_local, 1, idx_l.clamp_min(0)),
                             torch.full(idx_l.shape, float("-inf"), dtype=scores_local.dtype, device=dev))
    all_pos = _all_gather(cand_pos, world, group).permute(1, 0, 2).reshape(num_q, world * k)
    all_score = _all_gather(cand_score, world, group).permute(1, 0, 2).reshape(num_q, world * k)
    # 2. reselect: candidates in ascending position (invalid ones last), so that
    #    the top-k kernel's tie rule (lower index) is the position rule
    key = torch.where(all_pos >= 0, all_pos, torch.full_like(all_pos, torch.iinfo(torch.int64).max))
    order = torch.argsort(key, dim=1)
    pos_sorted = torch.gather(all_pos, 1, order)
    score_sorted = torch.gather(all_score, 1, order).contiguous()
    n_valid = (all_pos >= 0).sum(dim=1)
    sel = compute.topk(score_sorted, (n_valid - 1).to(torch.int32), k).to(torch.int64)
    idx = torch.where(sel >= 0, torch.gather(pos_sorted, 1, sel.clamp_min(0)), torch.full_like(sel, -1))
    # 3. attention over the selected positions this rank owns (local indices)
    mine = (idx >= 0) & (idx % world == rank)
    idx_mine = torch.where(mine, torch.div(idx, world, rounding_mode="floor"), torch.full_like(idx, -1))
    o_part, lse_part = compute.partial(idx_mine.to(torch.int32))
    # 4. exchange the partials and merge them all
    o_all = _all_gather(o_part, world, group).reshape(world * o_part.shape[0], *o_part.shape[1:])
    l_all = _all_gather(lse_part, world, group).reshape(world * lse_part.shape[0], *lse_part.shape[1:])
    out, lse = compute.combine(o_all, l_all)
    return out, lse, idx.to(torch.int32)
