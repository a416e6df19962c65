"""The whole forward (ulysses_dist_attn_fwd), unfused and fused, against the oracle's
explicit pipeline; fused and unfused must agree bit for bit."""
import random

import pytest
import torch

import oracle
import sequence_attention_seq_gb300 as uly
from gpu_util import assert_close, bits_equal, device_ok, need_gpu
from sequence_attention_seq_gb300.inputs import seq_shards_qkv

pytestmark = pytest.mark.gpu

CASES = [
    # P, b, s, hq, hkv, d, causal
    (2, 1, 256, 4, 2, 64, True),
    (4, 2, 512, 8, 8, 128, False),
    (4, 2, 512, 8, 8, 128, True),
    (8, 1, 1024, 16, 8, 128, True),
    (1, 1, 384, 2, 1, 128, True),      # P = 1: plain attention
    (16, 1, 2048, 16, 16, 64, True),   # 16 ranks: the fused forward's small parameter block
]


@pytest.mark.parametrize("P,b,s,hq,hkv,d,causal", CASES)
def test_dist_attn_fwd_bf16(P, b, s, hq, hkv, d, causal):
    need_gpu()
    qs, ks, vs = seq_shards_qkv(P, b, s, hq, hkv, d, torch.bfloat16, seed=P * 11 + s)
    qd, kd, vd = [t.cuda() for t in qs], [t.cuda() for t in ks], [t.cuda() for t in vs]
    unfused = uly.ulysses_dist_attn_fwd(qd, kd, vd, causal, fused=False)
    fused = uly.ulysses_dist_attn_fwd(qd, kd, vd, causal, fused=True)
    torch.cuda.synchronize()
    device_ok()
    want = oracle.dist_attn_fwd(qs, ks, vs, causal)
    for j in range(P):
        assert_close(unfused[j], want[j], torch.bfloat16, f"unfused rank {j}")
        assert bits_equal(fused[j], unfused[j]), f"fused != unfused on rank {j}"


def test_dist_attn_fwd_ragged_unfused_only():
    """(s/P) % 128 != 0: the fused path declines, the unfused path handles the ragged tail."""
    need_gpu()
    P, b, s, hq, hkv, d = 2, 1, 200, 4, 4, 128
    qs, ks, vs = seq_shards_qkv(P, b, s, hq, hkv, d, torch.bfloat16, seed=3)
    qd, kd, vd = [t.cuda() for t in qs], [t.cuda() for t in ks], [t.cuda() for t in vs]
    with pytest.raises(uly.UlyssesError):
        uly.ulysses_dist_attn_fwd(qd, kd, vd, True, fused=True)
    out = uly.ulysses_dist_attn_fwd(qd, kd, vd, True, fused=False)
    torch.cuda.synchronize()
    want = oracle.dist_attn_fwd(qs, ks, vs, True)
    for j in range(P):
        assert_close(out[j], want[j], torch.bfloat16, f"rank {j}")
    device_ok()


def test_repeat_calls_are_deterministic():
    need_gpu()
    qs, ks, vs = seq_shards_qkv(4, 1, 1024, 8, 4, 128, torch.bfloat16, seed=21)
    qd, kd, vd = [t.cuda() for t in qs], [t.cuda() for t in ks], [t.cuda() for t in vs]
    a = uly.ulysses_dist_attn_fwd(qd, kd, vd, True, fused=True)
    b = uly.ulysses_dist_attn_fwd(qd, kd, vd, True, fused=True)
    torch.cuda.synchronize()
    for x, y in zip(a, b):
        assert bits_equal(x, y)
    device_ok()


@pytest.mark.parametrize("P,b,s,hq,hkv,d,causal", [
    (32, 1, 4096, 32, 32, 64, True),    # more ranks than the small parameter block holds
    (64, 1, 8192, 64, 64, 128, False),  # the most ranks any call takes
])
def test_dist_attn_fwd_many_ranks(P, b, s, hq, hkv, d, causal):
    """The fused forward over 32 and 64 ranks (one tensor map per rank buffer) gives the
    unfused forward's bits, and sampled rows match the oracle."""
    need_gpu()
    qs, ks, vs = seq_shards_qkv(P, b, s, hq, hkv, d, torch.bfloat16, seed=P + s)
    qd, kd, vd = [t.cuda() for t in qs], [t.cuda() for t in ks], [t.cuda() for t in vs]
    unfused = uly.ulysses_dist_attn_fwd(qd, kd, vd, causal, fused=False)
    fused = uly.ulysses_dist_attn_fwd(qd, kd, vd, causal, fused=True)
    torch.cuda.synchronize()
    device_ok()
    for j in range(P):
        assert bits_equal(fused[j], unfused[j]), f"fused != unfused on rank {j}"
    rng = random.Random(P)
    S = s // P
    samples = sorted({(rng.randrange(P), 0, rng.choice([0, S - 1, rng.randrange(S)]), h) for h in range(hq)})
    want = oracle.dist_attn_rows(qs, ks, vs, causal, samples)
    got = torch.stack([fused[j][bb, t, gh] for (j, bb, t, gh) in samples])
    assert_close(got, want, torch.bfloat16, f"P={P} sampled rows")
