"""Host-side helpers of bench.py that need no GPU: the L2 policy and the
per-step distribution."""
import bench


def test_l2_policy_flushes_only_inputs_that_fit_in_l2():
    flush, note = bench.l2_policy(805_306_368)            # B=8 H=32 N=4096 d=128 bf16: Q, K, V
    assert flush == 0 and "larger than L2" in note
    flush, note = bench.l2_policy(3 * 33_554_432)         # B=1 H=8 N=16384 d=128 bf16: 100.7 MB
    assert flush == bench.FLUSH_BYTES and flush > bench.L2_BYTES and "flushed" in note


def test_step_distribution_percentiles():
    d = bench.step_distribution([5.0, 1.0, 3.0, 2.0, 4.0])
    assert d == {"median": 3.0, "p10": 1.4, "p90": 4.6, "n": 5}
    d = bench.step_distribution([2.5])
    assert d["median"] == d["p10"] == d["p90"] == 2.5
