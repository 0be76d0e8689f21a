"""Context-parallel attention: the keys of a sequence are split across ranks.

Rank r of the process group holds all queries and the r-th contiguous block
of keys and values. Each rank computes its part (softmax over its own keys,
with that part's logsumexp), the parts are exchanged once (all-gather), and
every rank folds them with the block merge of the "FlashAttention + Triton"
page (section 2.3, in LSE form), which is exact: the result equals attention
over the whole key set. With NCCL the exchange moves B*H*N*(d+1) fp32 values
per rank.

The compute steps are the library's kernels (fa_fwd_partial, fa_merge). The
``partial`` and ``merge`` arguments exist so that the exchange logic can be
exercised on CPU process groups (gloo) with stand-ins for the kernels.
"""
from __future__ import annotations


def shard_bounds(n_keys: int, world_size: int, rank: int) -> tuple[int, int]:
    """Key rows [lo, hi) of `rank` when n_keys are split into world_size
    contiguous blocks whose sizes differ by at most one (earlier ranks larger)."""
    if world_size < 1 or not 0 <= rank < world_size or n_keys < 0:
        raise ValueError("bad shard request")
    base, extra = divmod(n_keys, world_size)
    lo = rank * base + min(rank, extra)
    return lo, lo + base + (1 if rank < extra else 0)


def context_parallel_attention(q, k_local, v_local, group=None, scale: float | None = None, *,
                               partial=None, merge=None):
    """O, LSE of attention of q [B, H, N, d] over the keys held by all ranks of
    `group`, in rank order; this rank holds k_local, v_local [B, H, N_r, d]
    (N_r may be 0). Returns the full (O in q's dtype, LSE fp32) on every rank."""
    import torch
    import torch.distributed as dist
    from . import attention_partial, merge_partials

    partial = partial or attention_partial
    merge = merge or merge_partials
    o_p, l_p = partial(q, k_local, v_local, scale=scale)
    world = dist.get_world_size(group)
    o_all = [torch.empty_like(o_p) for _ in range(world)]
    l_all = [torch.empty_like(l_p) for _ in range(world)]
    dist.all_gather(o_all, o_p.contiguous(), group=group)
    dist.all_gather(l_all, l_p.contiguous(), group=group)
    return merge(torch.stack(o_all), torch.stack(l_all), dtype=q.dtype)
