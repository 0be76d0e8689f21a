"""Tile-by-tile statistics of the kernel against the oracle's online model.

The dataflow page's validation layer 2 (section 4.1): print each block's
running max and running sum and compare them with the reference softmax. The
kernel moves its reference max lazily and warp-wide, so the comparable
quantity is the running logsumexp m + ln l after each key tile, which does
not depend on when the reference moved; the reference max itself must never
decrease, never exceed the true running max, and never trail it by more than
the threshold (15 in log2 units: P, taken against the reference, stays
<= 2^15).
"""
import numpy as np
import pytest
import torch

import oracle
from workloads import make_qkv, rising_norm_order

pytestmark = pytest.mark.gpu
LN2 = float(np.log(2.0))
THRESHOLD_LOG2 = 15  # the lazy-rescale threshold of the product build


@pytest.mark.parametrize("N,d,dtype,sig,rising", [
    (700, 128, "bf16", 3.0, True),
    (512, 128, "f16", 1.0, False),
    (300, 64, "bf16", 3.0, True),
])
def test_running_statistics_match_online_model(N, d, dtype, sig, rising):
    from exact_attention_87_gb300 import testing
    q, k, v = make_qkv(1, 2, N, d, dtype, sigma_qk=sig, seed=4, wid=7000 + N)
    if rising:
        k, v = rising_norm_order(k, v)
    o, lse, st, _ = testing.attention(q.cuda(), k.cuda(), v.cuda(), stats=True)
    torch.cuda.synchronize()
    assert testing.device_status() == 0
    st = st.cpu().double().numpy()            # [B,H,N,nkv,2]
    m_k, l_k = st[..., 0], st[..., 1]
    _, _, m_eager, l_eager = oracle.attn_online(q, k, v, block_n=testing.kv_tile(d), tau=0.0, trace=True)
    run_lse_ref = m_eager + np.log(l_eager)
    run_lse_k = m_k + np.log(l_k)
    tol = 1e-4 * np.maximum(1.0, np.abs(run_lse_ref))
    assert np.all(np.abs(run_lse_k - run_lse_ref) <= tol), float(np.abs(run_lse_k - run_lse_ref).max())
    eps = 1e-4 * np.maximum(1.0, np.abs(m_eager))
    assert np.all(np.diff(m_k, axis=-1) >= -eps[..., 1:])        # never decreases
    assert np.all(m_k <= m_eager + eps)                           # a max of scores seen so far
    assert np.all(m_eager - m_k <= THRESHOLD_LOG2 * LN2 + eps)    # trails by at most the threshold
    # the final tile's statistics give the LSE output
    np.testing.assert_allclose(run_lse_k[..., -1], lse.cpu().double().numpy(), rtol=0, atol=4e-3)


@pytest.mark.parametrize("N,d,dtype", [(700, 128, "bf16"), (300, 64, "f16")])
def test_eager_threshold_reference_max_is_the_running_max(N, d, dtype):
    """With the rescale threshold at 0 (testing build) a warp moves its
    reference max whenever any of its rows' max grows, and then every row
    takes its own running max: after each tile the kernel's m equals the
    online model's eager running max, and m + ln l its running logsumexp."""
    from exact_attention_87_gb300 import testing
    q, k, v = make_qkv(1, 2, N, d, dtype, sigma_qk=3.0, seed=6, wid=7100 + N)
    k, v = rising_norm_order(k, v)
    o, lse, st = testing.attention_debug(q.cuda(), k.cuda(), v.cuda(), tau=0.0, stats=True)
    torch.cuda.synchronize()
    assert testing.device_status() == 0
    st = st.cpu().double().numpy()
    m_k, l_k = st[..., 0], st[..., 1]
    _, _, m_eager, l_eager = oracle.attn_online(q, k, v, block_n=testing.kv_tile(d), tau=0.0, trace=True)
    eps = 1e-4 * np.maximum(1.0, np.abs(m_eager))
    assert np.all(np.abs(m_k - m_eager) <= eps), float(np.abs(m_k - m_eager).max())
    run_lse_ref = m_eager + np.log(l_eager)
    assert np.all(np.abs(m_k + np.log(l_k) - run_lse_ref) <= 1e-4 * np.maximum(1.0, np.abs(run_lse_ref)))
