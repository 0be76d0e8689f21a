"""Head-parallel attention: the B*H problems of one forward pass split across ranks.

Every (batch, head) pair is an independent attention problem (the pages'
outer loop runs over them with no exchange), so one forward pass shards
across G GPUs without any communication: rank r takes a contiguous block of
the B*H problems in memory order (``head_bounds``), runs the kernel on that
slice (a [1, H_r, N, d] view of the [B*H, N, d] arrays) and owns that block
of O and LSE. Only when one device must hold the whole result does an
all-gather of O and LSE assemble it (the one collective; blocks are padded to
the largest block for it).

The compute step is the library's kernel (``attention``). The ``attention_fn``
argument exists so that the sharding and exchange logic can be exercised on
CPU process groups (gloo) with a stand-in for the kernel.
"""
from __future__ import annotations


def head_bounds(B: int, H: int, world_size: int, rank: int) -> tuple[int, int]:
    """Problems [lo, hi) of `rank`, numbered b*H + h, when the B*H problems are
    split into world_size contiguous blocks whose sizes differ by at most one
    (earlier ranks larger)."""
    if B < 1 or H < 1 or world_size < 1 or not 0 <= rank < world_size:
        raise ValueError("bad shard request")
    n = B * H
    base, extra = divmod(n, world_size)
    lo = rank * base + min(rank, extra)
    return lo, lo + base + (1 if rank < extra else 0)


def head_slice(t, lo: int, hi: int):
    """Problems [lo, hi) of a [B, H, ...] tensor as a [1, hi - lo, ...] view
    (contiguous: the problems are consecutive in memory)."""
    flat = t.reshape((t.shape[0] * t.shape[1],) + tuple(t.shape[2:]))
    return flat[lo:hi].unsqueeze(0)


def head_parallel_attention(q, k, v, group=None, scale: float | None = None, gather: bool = False, *,
                            attention_fn=None, o_dtype=None):
    """This rank's block of attention(q, k, v) for q, k, v [B, H, N, d] (the
    same tensors on every rank; contiguous). Returns (lo, hi, O_r, LSE_r) with
    O_r [1, hi - lo, N, d] and LSE_r [1, hi - lo, N] for problems [lo, hi);
    with gather=True, returns the whole (O [B, H, N, d], LSE [B, H, N]) on
    every rank instead (one all-gather). o_dtype is the dtype attention_fn
    returns O in (default q's, as the library's kernel does): a rank with no
    problem makes its empty block in it."""
    import torch
    import torch.distributed as dist
    from . import attention

    attention_fn = attention_fn or attention
    world = dist.get_world_size(group) if dist.is_initialized() else 1
    rank = dist.get_rank(group) if dist.is_initialized() else 0
    B, H, N, d = q.shape
    lo, hi = head_bounds(B, H, world, rank)
    if hi > lo:
        o_r, l_r = attention_fn(head_slice(q, lo, hi), head_slice(k, lo, hi), head_slice(v, lo, hi), scale=scale)
    else:  # more ranks than problems: this rank has none
        o_r = torch.empty((1, 0, N, d), dtype=o_dtype or q.dtype, device=q.device)
        l_r = torch.empty((1, 0, N), dtype=torch.float32, device=q.device)
    if not gather:
        return lo, hi, o_r, l_r
    if world == 1:
        return o_r.reshape(B, H, N, d), l_r.reshape(B, H, N)
    width = -(-B * H // world)  # the largest block
    o_pad = torch.zeros((width, N, d), dtype=o_r.dtype, device=o_r.device)
    l_pad = torch.zeros((width, N), dtype=l_r.dtype, device=l_r.device)
    o_pad[: hi - lo] = o_r[0]
    l_pad[: hi - lo] = l_r[0]
    o_all = torch.empty((world * width, N, d), dtype=o_r.dtype, device=o_r.device)
    l_all = torch.empty((world * width, N), dtype=l_r.dtype, device=l_r.device)
    dist.all_gather_into_tensor(o_all, o_pad, group=group)
    dist.all_gather_into_tensor(l_all, l_pad, group=group)
    rows = [r * width + i for r in range(world) for i in range(head_bounds(B, H, world, r)[1]
                                                                - head_bounds(B, H, world, r)[0])]
    idx = torch.tensor(rows, device=o_all.device)
    return o_all.index_select(0, idx).reshape(B, H, N, d), l_all.index_select(0, idx).reshape(B, H, N)
