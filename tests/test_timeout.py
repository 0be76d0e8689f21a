"""Bounded waits: a barrier that is never completed makes the kernel give up,
report FA_ERR_DEVICE_TIMEOUT through the status word, drain its own work and
exit; the context stays usable. The failure is injected on the producer side
(one V tile is never loaded): no GPU fault, trap or endless loop is involved,
and every wait has a short limit (2e7 cycles, about 10 ms).
"""
import pytest
import torch

import exact_attention_87_gb300 as fa
import oracle
from parity_util import compare
from workloads import make_qkv

pytestmark = pytest.mark.gpu


def test_injected_missing_tile_times_out_and_recovers():
    from exact_attention_87_gb300 import testing
    q, k, v = make_qkv(1, 2, 512, 128, "bf16", seed=8, wid=8000)
    qc, kc, vc = q.cuda(), k.cuda(), v.cuda()
    assert testing.device_status() == 0
    testing.attention(qc, kc, vc, inject=1, wait_limit_cycles=20_000_000)
    torch.cuda.synchronize()
    where = testing.last_timeout_where()
    assert where != 0, "no wait recorded a timeout"
    assert testing.device_status() == fa.FA_ERR_DEVICE_TIMEOUT
    assert testing.device_status() == 0  # cleared by the read
    # the context is still usable: a normal call gives correct results
    o, lse, _, _ = testing.attention(qc, kc, vc)
    torch.cuda.synchronize()
    assert testing.device_status() == 0
    o_ref, lse_ref = oracle.attn(q, k, v)
    res = compare(o.cpu().double().numpy(), lse.cpu().double().numpy(), o_ref, lse_ref, "bf16")
    assert res["ok"], res
