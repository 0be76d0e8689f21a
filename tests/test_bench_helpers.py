"""Host-side helpers of bench.py that need no GPU: the L2 policy, the
per-step distribution, the code key of the recorded traffic and the name of
the kernel a timed launch runs."""
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


def test_code_of_drops_comments_and_blank_lines_only():
    src = "int a; // note\n\n/* block\n   comment */ int b;\n  x = 1;   // more\n"
    assert bench.code_of(src) == "int a;\n int b;\n  x = 1;"
    # an edit of comments alone leaves the code (and so the recorded traffic's key) unchanged
    assert bench.code_of(src.replace("note", "a longer note")) == bench.code_of(src)
    assert bench.code_of(src.replace("x = 1", "x = 2")) != bench.code_of(src)


def test_kernel_names_of_the_timed_launches():
    from workloads import WORKLOADS
    W = WORKLOADS
    # d = 128, N <= 4096, N a multiple of 256: the persistent form (causal too, N a multiple of 512)
    assert bench.fwd_kernel_name(W["b8h32n4096d128_bf16_qk3"]) == "fa_fwd_persist_kernel<128,bf16>"
    assert bench.fwd_kernel_name(W["b8h32n4096d128_bf16_qk3"], causal=True) == "fa_fwd_persist_kernel<128,bf16>"
    # the streamed tail runs on it as well
    assert bench.fwd_kernel_name(W["b8h12n2048d128_f16"], launches=2, streamed=True) == \
        "fa_fwd_persist_kernel<128,f16>"
    # longer sequences: one CTA per unit (here under the key-range tail plan)
    assert bench.fwd_kernel_name(W["b1h8n16384d128_bf16"], launches=3) == "fa_fwd_f16_kernel<128,bf16>"
    # d = 64: persistent when unmasked, one CTA per unit with the causal mask
    assert bench.fwd_kernel_name(W["b8h32n4096d64_bf16"]) == "fa_fwd_persist_kernel<64,bf16>"
    assert bench.fwd_kernel_name(W["b8h32n4096d64_bf16"], causal=True) == "fa_fwd_f16_kernel<64,bf16>"
    assert bench.fwd_kernel_name(W["b4h16n4096d256_bf16"]) == "fa_fwd_d256_kernel<bf16>"
    assert bench.fwd_kernel_name(W["b1h1n64d64_f32"]) == "fa_fwd_f32_kernel<64>"
