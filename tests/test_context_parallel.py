"""Context parallelism: keys split across ranks, parts merged after one exchange.

CPU tests (gloo, world size 2 and 3) check the exchange logic of both
exchanges (all-gather of the parts; all-to-all of row blocks, then a gather of
the merged blocks): rank order, shapes, an empty key shard, a rank with no
rows, and that every rank ends with attention over the whole key set. The kernels cannot run there, so the part and merge steps are
the oracle's (``partial=`` / ``merge=`` of context_parallel_attention).
GPU tests check the kernels themselves: fa_fwd_partial against the oracle on
one key shard, shards merged by fa_merge against attention over all keys, and
the whole path through a one-rank NCCL group.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

import oracle
from exact_attention_87_gb300.context_parallel import shard_bounds
from workloads import make_qkv


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_shard_bounds_cover_the_keys_once():
    for n in (0, 1, 5, 128, 1000, 4097):
        for world in (1, 2, 3, 4, 7):
            bounds = [shard_bounds(n, world, r) for r in range(world)]
            assert bounds[0][0] == 0 and bounds[-1][1] == n
            for (a, b), (c, _) in zip(bounds, bounds[1:]):
                assert b == c and a <= b
            sizes = [b - a for a, b in bounds]
            assert max(sizes) - min(sizes) <= 1
    with pytest.raises(ValueError):
        shard_bounds(10, 2, 2)


def _oracle_partial(q, k, v, scale=None):
    """Stand-in for attention_partial on CPU: the oracle over this rank's keys."""
    B, H, N, d = q.shape
    if k.shape[2] == 0:
        return torch.zeros((B, H, N, d), dtype=torch.float64), torch.full((B, H, N), float("-inf"), dtype=torch.float64)
    o, lse = oracle.attn(q, k, v, scale=scale, nthreads=1)
    return torch.from_numpy(o), torch.from_numpy(lse)


def _oracle_merge(o_parts, lse_parts, dtype=None):
    o, lse = oracle.merge(o_parts.numpy(), lse_parts.numpy())
    return torch.from_numpy(o), torch.from_numpy(lse)


def _worker(rank, world, port, N, out):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import torch.distributed as dist
    from exact_attention_87_gb300.context_parallel import context_parallel_attention, shard_bounds
    from workloads import make_qkv
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    q, k, v = make_qkv(2, 3, N, 16, "f16", sigma_qk=2.0, seed=4, wid=12000 + N)
    lo, hi = shard_bounds(N, world, rank)
    o, lse = context_parallel_attention(q, k[:, :, lo:hi].contiguous(), v[:, :, lo:hi].contiguous(), scale=0.3,
                                        partial=_oracle_partial, merge=_oracle_merge)
    out[rank] = (o.numpy(), lse.numpy())
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("world,N", [(2, 37), (3, 2), (3, 100)])
def test_exchange_on_cpu_ranks_gives_attention_over_all_keys(world, N):
    """(3, 2): one rank holds no key at all."""
    port = _free_port()
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(world, port, N, out), nprocs=world, join=True)
    q, k, v = make_qkv(2, 3, N, 16, "f16", sigma_qk=2.0, seed=4, wid=12000 + N)
    o_ref, lse_ref = oracle.attn(q, k, v, scale=0.3)
    for r in range(world):
        o, lse = out[r]
        np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse, lse_ref, rtol=0, atol=1e-12)


# ---------------------------------------------------------------------------
# GPU: the kernels
# ---------------------------------------------------------------------------

def _gpu():
    import exact_attention_87_gb300 as fa
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    fa.build()
    fa.lib()
    return fa


@pytest.mark.gpu
@pytest.mark.parametrize("B,H,Nq,Nk,d,dtype,sig", [
    (1, 2, 300, 129, 128, "bf16", 3.0),
    (2, 1, 1000, 700, 64, "f16", 1.0),
    (1, 3, 64, 1, 128, "f16", 1.0),
    (1, 1, 257, 2048, 128, "bf16", 2.0),
    (1, 2, 300, 129, 256, "bf16", 3.0),
    (2, 1, 200, 1000, 256, "f16", 1.0),
])
def test_partial_against_oracle_on_one_key_shard(B, H, Nq, Nk, d, dtype, sig):
    """Normalised fp32 O of one part: max error 1e-2, cosine 0.999 (P is
    rounded to the input type before P V, as in the whole pass); LSE within
    1e-4 * max(1, |LSE|)."""
    fa = _gpu()
    q, _, _ = make_qkv(B, H, Nq, d, dtype, sigma_qk=sig, seed=6, wid=12100 + Nq)
    _, k, v = make_qkv(B, H, Nk, d, dtype, sigma_qk=sig, seed=7, wid=12200 + Nk)
    o_p, l_p = fa.attention_partial(q.cuda(), k.cuda(), v.cuda())
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == fa.FA_OK
    o_ref, lse_ref = oracle.attn(q, k, v)
    o = o_p.cpu().double().numpy()
    lse = l_p.cpu().double().numpy()
    assert np.abs(o - o_ref).max() <= 1e-2
    cos = float((o * o_ref).sum() / np.sqrt((o * o).sum() * (o_ref * o_ref).sum()))
    assert cos >= 0.999
    assert np.all(np.abs(lse - lse_ref) <= 1e-4 * np.maximum(1.0, np.abs(lse_ref)))


@pytest.mark.gpu
@pytest.mark.parametrize("B,H,N,d,dtype,sig,parts", [
    (1, 2, 1000, 128, "bf16", 3.0, 2),
    (2, 2, 777, 64, "f16", 1.0, 3),
    (1, 1, 4096, 128, "bf16", 3.0, 4),
    (1, 2, 130, 128, "f16", 1.0, 5),   # shards of 26 keys
    (1, 2, 1000, 256, "bf16", 3.0, 3),
])
def test_shards_merged_equal_attention_over_all_keys(B, H, N, d, dtype, sig, parts):
    from parity_util import compare
    fa = _gpu()
    q, k, v = make_qkv(B, H, N, d, dtype, sigma_qk=sig, seed=8, wid=12300 + N + parts)
    qc, kc, vc = q.cuda(), k.cuda(), v.cuda()
    o_parts, l_parts = [], []
    for r in range(parts):
        lo, hi = shard_bounds(N, parts, r)
        o_p, l_p = fa.attention_partial(qc, kc[:, :, lo:hi].contiguous(), vc[:, :, lo:hi].contiguous())
        o_parts.append(o_p)
        l_parts.append(l_p)
    o, lse = fa.merge_partials(torch.stack(o_parts), torch.stack(l_parts), dtype=q.dtype)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == fa.FA_OK
    o_ref, lse_ref = oracle.attn(q, k, v)
    res = compare(o.cpu().double().numpy(), lse.cpu().double().numpy(), o_ref, lse_ref, dtype)
    assert res["ok"], res


@pytest.mark.gpu
def test_merge_of_empty_parts():
    """A part with LSE = -inf adds nothing; a row whose parts are all -inf gets O = 0, LSE = -inf."""
    fa = _gpu()
    B, H, N, d = 1, 2, 50, 64
    g = torch.Generator().manual_seed(3)
    o_parts = torch.randn((3, B, H, N, d), generator=g, dtype=torch.float32)
    l_parts = torch.randn((3, B, H, N), generator=g, dtype=torch.float32)
    l_parts[1] = float("-inf")
    l_parts[:, 0, 1, 7] = float("-inf")
    o, lse = fa.merge_partials(o_parts.cuda(), l_parts.cuda(), dtype=torch.float16)
    torch.cuda.synchronize()
    o, lse = o.cpu().double().numpy(), lse.cpu().double().numpy()
    o_ref, lse_ref = oracle.merge(o_parts[[0, 2]].numpy(), l_parts[[0, 2]].numpy())
    keep = np.ones((B, H, N), dtype=bool)
    keep[0, 1, 7] = False
    assert np.abs(o - o_ref)[keep].max() <= 2e-3 * max(1.0, np.abs(o_ref[keep]).max())
    assert np.abs(lse - lse_ref)[keep].max() <= 1e-4 * max(1.0, np.abs(lse_ref[keep]).max())
    assert np.all(o[0, 1, 7] == 0.0) and lse[0, 1, 7] == -np.inf


def _worker_a2a(rank, world, port, B, H, N, out):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import torch.distributed as dist
    from exact_attention_87_gb300.context_parallel import context_parallel_attention, shard_bounds
    from workloads import make_qkv
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    q, k, v = make_qkv(B, H, N, 16, "f16", sigma_qk=2.0, seed=4, wid=12500 + N)
    lo, hi = shard_bounds(N, world, rank)
    kw = dict(scale=0.3, exchange="all_to_all", partial=_oracle_partial, merge=_oracle_merge, o_dtype=torch.float64)
    kl, vl = k[:, :, lo:hi].contiguous(), v[:, :, lo:hi].contiguous()
    rlo, rhi, o_r, l_r = context_parallel_attention(q, kl, vl, gather=False, **kw)
    o, lse = context_parallel_attention(q, kl, vl, gather=True, **kw)
    out[rank] = (rlo, rhi, o_r.numpy(), l_r.numpy(), o.numpy(), lse.numpy())
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("world,B,H,N", [(2, 2, 3, 37), (3, 1, 2, 5), (3, 1, 1, 2)])
def test_all_to_all_exchange_on_cpu_ranks(world, B, H, N):
    """The memory-bounded exchange: each rank merges its block of the B*H*N
    rows from every part, then the merged blocks are gathered. (3, 1, 1, 2):
    two rows on three ranks, so one rank merges none (and one holds no key)."""
    from exact_attention_87_gb300.context_parallel import shard_bounds
    port = _free_port()
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_worker_a2a, args=(world, port, B, H, N, out), nprocs=world, join=True)
    q, k, v = make_qkv(B, H, N, 16, "f16", sigma_qk=2.0, seed=4, wid=12500 + N)
    o_ref, lse_ref = oracle.attn(q, k, v, scale=0.3)
    rows_o, rows_l = o_ref.reshape(-1, 16), lse_ref.reshape(-1)
    covered = []
    for r in range(world):
        rlo, rhi, o_r, l_r, o, lse = out[r]
        assert (rlo, rhi) == shard_bounds(B * H * N, world, r)
        np.testing.assert_allclose(o_r, rows_o[rlo:rhi], rtol=0, atol=1e-12)
        np.testing.assert_allclose(l_r, rows_l[rlo:rhi], rtol=0, atol=1e-12)
        np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse, lse_ref, rtol=0, atol=1e-12)
        covered += list(range(rlo, rhi))
    assert covered == list(range(B * H * N))


@pytest.mark.gpu
@pytest.mark.parametrize("exchange", ["all_gather", "all_to_all"])
def test_context_parallel_through_a_one_rank_nccl_group(exchange):
    import datetime
    import torch.distributed as dist
    from parity_util import compare
    from exact_attention_87_gb300.context_parallel import context_parallel_attention
    fa = _gpu()
    q, k, v = make_qkv(2, 4, 600, 128, "bf16", sigma_qk=3.0, seed=9, wid=12400)
    dist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{_free_port()}", rank=0, world_size=1,
                            timeout=datetime.timedelta(seconds=120))
    try:
        o, lse = context_parallel_attention(q.cuda(), k.cuda(), v.cuda(), exchange=exchange)
        torch.cuda.synchronize()
    finally:
        dist.destroy_process_group()
    assert fa.fa_get_device_status() == fa.FA_OK
    o_ref, lse_ref = oracle.attn(q, k, v)
    res = compare(o.cpu().double().numpy(), lse.cpu().double().numpy(), o_ref, lse_ref, "bf16")
    assert res["ok"], res
