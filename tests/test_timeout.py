"""Bounded waits: a barrier that is never completed makes the kernel give up,
report FA_ERR_DEVICE_TIMEOUT through the status word, drain its own work and
exit; the context stays usable. The failure is injected on the producer side
(one V or dO tile is never loaded): no GPU fault, trap or endless loop is involved,
and every wait has a short limit (2e7 cycles, about 10 ms).
"""
import pytest
import torch

import exact_attention_87_gb300 as fa
import oracle
from parity_util import compare
from workloads import make_qkv

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("d", [128, 256])
def test_injected_missing_tile_times_out_and_recovers(d):
    from exact_attention_87_gb300 import testing
    q, k, v = make_qkv(1, 2, 512, d, "bf16", seed=8, wid=8000)
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


@pytest.mark.parametrize("d", [128, 256])
def test_backward_injected_missing_tile_times_out_and_recovers(d):
    """The backward kernel (at d = 256 the dK/dQ kernel): dO of the first Q
    tile is never loaded."""
    from exact_attention_87_gb300 import testing
    from workloads import make_dout
    q, k, v = (t.cuda() for t in make_qkv(1, 2, 512, d, "bf16", seed=8, wid=8001))
    do = make_dout(1, 2, 512, d, "bf16", seed=8, wid=8001).cuda()
    o, lse = fa.attention(q, k, v)
    torch.cuda.synchronize()
    assert testing.device_status() == 0
    testing.attention_backward(q, k, v, o, lse, do, inject=1, wait_limit_cycles=20_000_000)
    torch.cuda.synchronize()
    assert testing.last_timeout_where() != 0
    assert testing.device_status() == fa.FA_ERR_DEVICE_TIMEOUT
    assert testing.device_status() == 0
    # still usable, and the same result as the product library
    dq, dk, dv, _ = testing.attention_backward(q, k, v, o, lse, do)
    ref = fa.attention_backward(q, k, v, o, lse, do)
    torch.cuda.synchronize()
    assert testing.device_status() == 0
    assert torch.equal(dk, ref[1]) and torch.equal(dv, ref[2])
    assert (dq.float() - ref[0].float()).abs().max().item() <= 1e-2 * ref[0].float().abs().max().item()


def test_backward_timeline_respects_dependencies():
    """clock64 stamps of the testing build: every MMA is issued after the
    softmax arrival it depends on (same SM clock within one CTA)."""
    from exact_attention_87_gb300 import testing
    from workloads import make_dout
    N = 1024
    q, k, v = (t.cuda() for t in make_qkv(1, 8, N, 128, "bf16", seed=9, wid=8002))
    do = make_dout(1, 8, N, 128, "bf16", seed=9, wid=8002).cuda()
    o, lse = fa.attention(q, k, v)
    _, _, _, tl = testing.attention_backward(q, k, v, o, lse, do, timeline=True)
    torch.cuda.synchronize()
    assert testing.device_status() == 0
    ev = {n: i for i, n in enumerate(testing.BWD_EVENTS)}
    t = tl.cpu().numpy().astype("int64")
    nq = N // 128
    for c in range(testing.TRACE_CTAS):
        for i in range(nq):
            assert t[c, ev["dV_issued"], i] >= t[c, ev["sm_P_arrived"], i] > 0
            assert t[c, ev["dK_issued"], i] >= t[c, ev["sm_dS_arrived"], i] > 0
            assert t[c, ev["sm_dQ_ready"], i] >= t[c, ev["dQ_issued"], i] > 0
            assert t[c, ev["sm_S_ready"], i] > 0 and t[c, ev["sm_dP_ready"], i] > 0
