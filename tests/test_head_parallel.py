"""Head parallelism: the B*H independent problems of one forward pass split across ranks.

CPU tests check the partition (every problem on exactly one rank, blocks
differing by at most one) and, on gloo ranks (world size 2 and 3, one case
with more ranks than problems), that each rank's block and the gathered whole
equal attention over every problem; the kernel cannot run there, so the
oracle stands in for it (``attention_fn=``). GPU tests run the library's
kernel on a rank's slice (a view of the whole arrays) and the whole path
through a one-rank NCCL group.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

import oracle
from exact_attention_87_gb300.head_parallel import head_bounds, head_slice
from workloads import make_qkv


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_head_bounds_cover_every_problem_once():
    for B, H in [(1, 1), (1, 2), (2, 3), (8, 32), (3, 7)]:
        for world in (1, 2, 3, 4, 8, 13):
            bounds = [head_bounds(B, H, world, r) for r in range(world)]
            assert bounds[0][0] == 0 and bounds[-1][1] == B * H
            for (a, b), (c, _) in zip(bounds, bounds[1:]):
                assert b == c and a <= b
            sizes = [b - a for a, b in bounds]
            assert max(sizes) - min(sizes) <= 1
    with pytest.raises(ValueError):
        head_bounds(2, 2, 2, 2)


def test_head_slice_is_a_view_of_consecutive_problems():
    t = torch.arange(2 * 3 * 4 * 2).reshape(2, 3, 4, 2)
    s = head_slice(t, 2, 5)
    assert s.shape == (1, 3, 4, 2) and s.data_ptr() == t[0, 2].data_ptr()
    assert torch.equal(s[0, 0], t[0, 2]) and torch.equal(s[0, 1], t[1, 0]) and torch.equal(s[0, 2], t[1, 1])


def _oracle_attention(q, k, v, scale=None):
    """Stand-in for the kernel on CPU ranks: the oracle on the slice."""
    o, lse = oracle.attn(q, k, v, scale=scale, nthreads=1)
    return torch.from_numpy(o), torch.from_numpy(lse).to(torch.float32)


def _worker(rank, world, port, B, H, out):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import torch.distributed as dist
    from exact_attention_87_gb300.head_parallel import head_parallel_attention
    from workloads import make_qkv
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    q, k, v = make_qkv(B, H, 40, 16, "f16", sigma_qk=2.0, seed=5, wid=15000 + B * H)
    lo, hi, o_r, l_r = head_parallel_attention(q, k, v, scale=0.3, attention_fn=_oracle_attention,
                                               o_dtype=torch.float64)
    o, lse = head_parallel_attention(q, k, v, scale=0.3, gather=True, attention_fn=_oracle_attention,
                                     o_dtype=torch.float64)
    out[rank] = (lo, hi, o_r.numpy(), l_r.numpy(), o.numpy(), lse.numpy())
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("world,B,H", [(2, 2, 3), (3, 1, 5), (3, 1, 2)])
def test_blocks_and_gathered_whole_on_cpu_ranks(world, B, H):
    """(3, 1, 2): the third rank has no problem at all."""
    port = _free_port()
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(world, port, B, H, out), nprocs=world, join=True)
    q, k, v = make_qkv(B, H, 40, 16, "f16", sigma_qk=2.0, seed=5, wid=15000 + B * H)
    o_ref, lse_ref = oracle.attn(q, k, v, scale=0.3)
    o_flat, l_flat = o_ref.reshape(B * H, 40, 16), lse_ref.reshape(B * H, 40)
    covered = []
    for r in range(world):
        lo, hi, o_r, l_r, o, lse = out[r]
        assert (lo, hi) == head_bounds(B, H, world, r)
        np.testing.assert_allclose(o_r[0], o_flat[lo:hi], rtol=0, atol=1e-12)
        np.testing.assert_allclose(l_r[0], l_flat[lo:hi], rtol=0, atol=2e-6 * max(1.0, np.abs(l_flat).max()))
        np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse, lse_ref, rtol=0, atol=2e-6 * max(1.0, np.abs(lse_ref).max()))
        covered += list(range(lo, hi))
    assert covered == list(range(B * H))


@pytest.mark.gpu
def test_rank_slices_through_the_kernel_equal_the_whole_pass():
    """Every rank's slice, run through the kernel on a [1, H_r, N, d] view,
    gives the rows of the whole pass bit for bit (same kernel, same tiles)."""
    import exact_attention_87_gb300 as fa
    fa.build()
    q, k, v = (t.cuda() for t in make_qkv(2, 5, 700, 128, "bf16", sigma_qk=3.0, seed=6, wid=15100))
    o, lse = fa.attention(q, k, v)
    torch.cuda.synchronize()
    of, lf = o.reshape(10, 700, 128), lse.reshape(10, 700)
    world = 3
    for r in range(world):
        lo, hi = head_bounds(2, 5, world, r)
        o_r, l_r = fa.attention(head_slice(q, lo, hi), head_slice(k, lo, hi), head_slice(v, lo, hi))
        torch.cuda.synchronize()
        assert torch.equal(o_r[0], of[lo:hi]) and torch.equal(l_r[0], lf[lo:hi])
    assert fa.fa_get_device_status() == fa.FA_OK


@pytest.mark.gpu
def test_head_parallel_through_a_one_rank_nccl_group():
    import datetime
    import torch.distributed as dist
    import exact_attention_87_gb300 as fa
    from parity_util import compare
    from exact_attention_87_gb300.head_parallel import head_parallel_attention
    fa.build()
    q, k, v = make_qkv(2, 4, 600, 128, "bf16", sigma_qk=3.0, seed=7, wid=15200)
    dist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{_free_port()}", rank=0, world_size=1,
                            timeout=datetime.timedelta(seconds=120))
    try:
        o, lse = head_parallel_attention(q.cuda(), k.cuda(), v.cuda(), gather=True)
        torch.cuda.synchronize()
    finally:
        dist.destroy_process_group()
    assert fa.fa_get_device_status() == fa.FA_OK
    o_ref, lse_ref = oracle.attn(q, k, v)
    res = compare(o.cpu().double().numpy(), lse.cpu().double().numpy(), o_ref, lse_ref, "bf16")
    assert res["ok"], res
