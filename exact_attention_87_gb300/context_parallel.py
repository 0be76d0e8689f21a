"""Context-parallel attention: the keys of a sequence are split across ranks.

Rank r of the process group holds all queries and the r-th contiguous block
of keys and values. Each rank computes its part (softmax over its own keys,
with that part's logsumexp), the parts are exchanged once (all-gather), and
every rank folds them with the block merge of the "FlashAttention + Triton"
page (section 2.3, in LSE form), which is exact: the result equals attention
over the whole key set.

Two exchanges (``exchange=``), with R = B*H*N rows and G ranks:
  "all_gather"  every rank receives every part and merges all R rows: each
                rank sends R*(d+1) fp32 values and holds G of them
                (G*R*(d+1)*4 bytes; 8.6 GB for B=8, H=32, N=4096, d=128 on 8
                ranks);
  "all_to_all"  the R rows are split into G contiguous blocks; rank r
                receives every part's rows of block r only (one all-to-all),
                merges them, and, with gather=True, the merged blocks (in q's
                dtype, plus LSE) are all-gathered. Each rank holds about
                R*(d+1)*4 bytes of parts (one part's worth) plus the merged
                result, whatever G is.

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
                               exchange: str = "all_gather", gather: bool = True, partial=None, merge=None,
                               o_dtype=None):
    """O, LSE of attention of q [B, H, N, d] over the keys held by all ranks of
    `group`, in rank order; this rank holds k_local, v_local [B, H, N_r, d]
    (N_r may be 0). Returns the full (O in q's dtype, LSE fp32) on every rank;
    with exchange="all_to_all" and gather=False, returns (lo, hi, O_rows,
    LSE_rows) instead: this rank's merged rows [lo, hi) of the B*H*N rows in
    memory order (shard_bounds(B*H*N, G, rank)), O_rows [hi - lo, d]. o_dtype
    is the dtype `merge` returns O in (default q's, as the library's merge
    does): a rank with no rows makes its empty block in it."""
    import torch
    import torch.distributed as dist
    from . import attention_partial, merge_partials

    partial = partial or attention_partial
    merge = merge or merge_partials
    o_p, l_p = partial(q, k_local, v_local, scale=scale)
    world = dist.get_world_size(group)
    if exchange == "all_gather":
        o_all = [torch.empty_like(o_p) for _ in range(world)]
        l_all = [torch.empty_like(l_p) for _ in range(world)]
        dist.all_gather(o_all, o_p.contiguous(), group=group)
        dist.all_gather(l_all, l_p.contiguous(), group=group)
        return merge(torch.stack(o_all), torch.stack(l_all), dtype=q.dtype)
    if exchange != "all_to_all":
        raise ValueError(f"unknown exchange {exchange!r}")
    rank = dist.get_rank(group)
    B, H, N, d = q.shape
    rows = B * H * N
    bounds = [shard_bounds(rows, world, r) for r in range(world)]
    width = bounds[0][1] - bounds[0][0]  # the largest block (earlier ranks are larger)
    o_flat, l_flat = o_p.reshape(rows, d), l_p.reshape(rows)
    # Row block r of this rank's part goes to rank r (blocks padded to `width`;
    # padding rows carry LSE = -inf and are never read).
    send_o = torch.zeros((world * width, d), dtype=o_p.dtype, device=o_p.device)
    send_l = torch.full((world * width,), float("-inf"), dtype=l_p.dtype, device=l_p.device)
    for r, (lo, hi) in enumerate(bounds):
        send_o[r * width: r * width + hi - lo] = o_flat[lo:hi]
        send_l[r * width: r * width + hi - lo] = l_flat[lo:hi]
    recv_o, recv_l = torch.empty_like(send_o), torch.empty_like(send_l)
    dist.all_to_all_single(recv_o, send_o, group=group)
    dist.all_to_all_single(recv_l, send_l, group=group)
    lo, hi = bounds[rank]
    n = hi - lo
    # Block s of what arrived is rank s's part for rows [lo, hi).
    if n > 0:
        parts_o = recv_o.view(world, width, d)[:, :n].contiguous().view(world, 1, 1, n, d)
        parts_l = recv_l.view(world, width)[:, :n].contiguous().view(world, 1, 1, n)
        o_r, l_r = merge(parts_o, parts_l, dtype=q.dtype)
        o_r, l_r = o_r.reshape(n, d), l_r.reshape(n)
    else:  # more ranks than rows: this rank merges none
        o_r = torch.empty((0, d), dtype=o_dtype or q.dtype, device=q.device)
        l_r = torch.empty((0,), dtype=l_p.dtype, device=q.device)
    if not gather:
        return lo, hi, o_r, l_r
    o_pad = torch.zeros((width, d), dtype=o_r.dtype, device=o_r.device)
    l_pad = torch.zeros((width,), dtype=l_r.dtype, device=l_r.device)
    o_pad[:n], l_pad[:n] = o_r, l_r
    o_all = torch.empty((world * width, d), dtype=o_r.dtype, device=o_r.device)
    l_all = torch.empty((world * width,), dtype=l_r.dtype, device=l_r.device)
    dist.all_gather_into_tensor(o_all, o_pad, group=group)
    dist.all_gather_into_tensor(l_all, l_pad, group=group)
    idx = torch.cat([torch.arange(r * width, r * width + b - a, device=o_all.device)
                     for r, (a, b) in enumerate(bounds)])
    return o_all.index_select(0, idx).reshape(B, H, N, d), l_all.index_select(0, idx).reshape(B, H, N)
