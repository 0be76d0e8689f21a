"""Masked forward pass (causal, per-batch key lengths): GPU parity against the
oracle's masked definition, including rows with no key to see."""
import numpy as np
import pytest
import torch

import exact_attention_87_gb300 as fa
import oracle
from parity_util import compare
from workloads import make_qkv

pytestmark = pytest.mark.gpu


def run(q, k, v, causal, klen, num_splits=1):
    kl = torch.tensor(klen, dtype=torch.int32, device="cuda") if klen is not None else None
    o, lse = fa.attention(q.cuda(), k.cuda(), v.cuda(), causal=causal, seqlens_k=kl, num_splits=num_splits)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == fa.FA_OK
    return o.cpu().double().numpy(), lse.cpu().double().numpy()


def check(q, k, v, dtype, causal=False, klen=None, num_splits=1):
    o, lse = run(q, k, v, causal, klen, num_splits)
    o_ref, lse_ref = oracle.attn_masked(q, k, v, causal=causal, klen=klen)
    empty = np.isneginf(lse_ref)
    assert np.all(o[empty] == 0) and np.all(np.isneginf(lse[empty]))
    res = compare(o[~empty], lse[~empty], o_ref[~empty], lse_ref[~empty], dtype)
    assert res["ok"], res


@pytest.mark.parametrize("B,H,N,d,dtype", [
    (1, 2, 1000, 128, "bf16"),
    (2, 3, 513, 128, "f16"),
    (1, 2, 777, 64, "bf16"),
    (1, 1, 129, 64, "f16"),
    (1, 2, 300, 128, "f32"),
    (2, 1, 200, 64, "f32"),
])
def test_causal(B, H, N, d, dtype):
    # the fp32 gate (1e-5) is stated for unit-variance inputs; 16-bit cases use sigma 2
    q, k, v = make_qkv(B, H, N, d, dtype, sigma_qk=1.0 if dtype == "f32" else 2.0, seed=40, wid=13000 + N + d)
    check(q, k, v, dtype, causal=True)


@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("f16", 64), ("f32", 128)])
def test_key_lengths(dtype, d):
    B, H, N = 5, 2, 700
    q, k, v = make_qkv(B, H, N, d, dtype, seed=41, wid=13100 + d)
    check(q, k, v, dtype, klen=[700, 1, 129, 256, 0])


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_causal_with_key_lengths(dtype):
    B, H, N, d = 3, 2, 600, 128
    q, k, v = make_qkv(B, H, N, d, dtype, sigma_qk=1.0 if dtype == "f32" else 2.0, seed=42, wid=13200)
    check(q, k, v, dtype, causal=True, klen=[600, 300, 77])


def test_padded_keys_need_not_be_finite():
    """Keys beyond a batch's length may be anything (their scores are replaced
    by -inf); values there only need to be finite (they get weight 0)."""
    B, H, N, d = 2, 2, 400, 128
    q, k, v = make_qkv(B, H, N, d, "bf16", seed=43, wid=13300)
    klen = [250, 400]
    o_ref, lse_ref = oracle.attn_masked(q, k, v, klen=klen)
    k2, v2 = k.clone(), v.clone()
    k2[0, :, 250:] = float("nan")
    v2[0, :, 250:] = 3.0e38
    o, lse = run(q, k2, v2, False, klen)
    res = compare(o, lse, o_ref, lse_ref, "bf16")
    assert res["ok"], res


@pytest.mark.parametrize("d,dtype", [(128, "bf16"), (64, "f16"), (256, "bf16")])
@pytest.mark.parametrize("splits", [2, 3, 0])
@pytest.mark.parametrize("causal,klen", [(True, None), (False, [700, 1, 129, 256, 0]),
                                         (True, [600, 300, 77, 0, 700])], ids=["causal", "lengths", "both"])
def test_masks_with_split_kv(d, dtype, splits, causal, klen):
    """fa_fwd_splitkv_ex: key ranges that a row's masks leave empty contribute
    nothing, rows with no key anywhere get O = 0 and LSE = -inf."""
    B, H, N = 5, 2, 700
    q, k, v = make_qkv(B, H, N, d, dtype, sigma_qk=2.0, seed=44, wid=13400 + d + splits)
    check(q, k, v, dtype, causal=causal, klen=klen, num_splits=splits)


@pytest.mark.parametrize("splits", [0, 3])
@pytest.mark.parametrize("causal", [False, True])
def test_padded_long_sequence_batch_split(causal, splits):
    """The padded variable-length batch with few heads and long sequences
    (the Triton page, section 5.1): B=4 H=1 N=4096 with key lengths 4096,
    3000, 0 and 2500 (64 work units on 152 SMs, which the automatic plan
    splits), split automatically and three ways."""
    B, H, N, d = 4, 1, 4096, 128
    klen = [4096, 3000, 0, 2500]
    q, k, v = make_qkv(B, H, N, d, "bf16", sigma_qk=1.5, seed=45, wid=13500 + causal)
    if splits == 0:
        assert fa.fa_fwd_splitkv_num_splits(B, H, N, d) > 1
    check(q, k, v, "bf16", causal=causal, klen=klen, num_splits=splits)


@pytest.mark.parametrize("B,H,N,dtype", [
    (3, 52, 1024, "bf16"),   # 624 units: 312 heavy/light pairs, two or three per CTA
    (2, 40, 2048, "f16"),    # 640 units of 8 Q blocks per head
])
def test_causal_persistent_several_pairs_per_cta(B, H, N, dtype):
    """The persistent causal form (d = 128, N a multiple of 512): each CTA
    walks several heavy/light pairs of Q blocks, with the barrier phases
    carried across them; every output against the oracle."""
    q, k, v = make_qkv(B, H, N, 128, dtype, sigma_qk=2.0, seed=42, wid=13300 + N)
    check(q, k, v, dtype, causal=True)
