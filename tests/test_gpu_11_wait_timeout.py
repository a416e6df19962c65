"""The failure path of the bounded device waits, exercised without a fault: a wait on a
barrier that nothing completes gives up after its limit, the device error word reports the
timeout, every later kernel of the library exits at once while the word is set, and after
the word is cleared the context runs the forward correctly again."""
import pytest
import torch

import oracle
import sequence_attention_seq_gb300 as uly
from gpu_util import assert_close, device_ok, need_gpu
from sequence_attention_seq_gb300.inputs import seq_shards_qkv

pytestmark = pytest.mark.gpu


def test_wait_gives_up_and_context_stays_usable():
    need_gpu()
    P, b, s, hq, hkv, d = 2, 1, 256, 4, 2, 128
    qs, ks, vs = seq_shards_qkv(P, b, s, hq, hkv, d, torch.bfloat16, seed=3)
    qd, kd, vd = [t.cuda() for t in qs], [t.cuda() for t in ks], [t.cuda() for t in vs]
    device_ok()
    try:
        uly.ulysses_wait_selftest(limit_ns=50_000_000)  # 50 ms
        # reading without clearing: the timeout stays reported
        assert uly.ulysses_device_status(clear=False) == uly.ULY_ERR_TIMEOUT
        # while the word is set, the attention kernels exit without writing their output
        sentinel = [torch.full((b, s // P, hq, d), 7.0, dtype=torch.bfloat16, device="cuda") for _ in range(P)]
        uly.ulysses_dist_attn_fwd(qd, kd, vd, True, fused=True, out_seq=sentinel)
        assert uly.ulysses_device_status(clear=True) == uly.ULY_ERR_TIMEOUT
        for t in sentinel:
            assert bool((t == 7.0).all()), "a kernel ran while the error word was set"
    finally:
        uly.ulysses_device_status(clear=True)
    # cleared: the same forward runs and is correct
    out = uly.ulysses_dist_attn_fwd(qd, kd, vd, True, fused=True)
    torch.cuda.synchronize()
    device_ok()
    want = oracle.dist_attn_fwd(qs, ks, vs, causal=True)
    for j in range(P):
        assert_close(out[j], want[j], torch.bfloat16, f"rank {j}")


def test_wait_selftest_argument_limits():
    need_gpu()
    for bad in (0, 999, 10**10 + 1):
        with pytest.raises(uly.UlyssesError) as e:
            uly.ulysses_wait_selftest(limit_ns=bad)
        assert e.value.status == uly.ULY_ERR_INVALID_ARG
    device_ok()
