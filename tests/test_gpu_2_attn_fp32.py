"""fp32 path (fp32 FMA attention) against the fp64 oracle: max-abs <= 1e-5."""
import pytest
import torch

import oracle
import sequence_attention_seq_gb300 as uly
from gpu_util import assert_close, device_ok, need_gpu
from sequence_attention_seq_gb300.inputs import global_qkv, seq_shards_qkv, shard_seq

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("causal", [False, True])
def test_tiny_configuration_end_to_end(causal):
    """P=2, b=1, s=64, h=4 MHA, d=16, fp32 N(0,1) from seed 0: exchange #1, attention with
    scale 1/sqrt(d), exchange #2."""
    need_gpu()
    qs, ks, vs = seq_shards_qkv(2, 1, 64, 4, 4, 16, torch.float32, seed=0)
    out = uly.ulysses_dist_attn_fwd([t.cuda() for t in qs], [t.cuda() for t in ks], [t.cuda() for t in vs],
                                    causal=causal, fused=False)
    torch.cuda.synchronize()
    want = oracle.dist_attn_fwd(qs, ks, vs, causal)
    for g, w in zip(out, want):
        assert_close(g, w, torch.float32, "tiny")
    device_ok()


@pytest.mark.parametrize("P,b,s,hq,hkv,d,causal", [
    (1, 1, 1, 1, 1, 16, False),      # a single token
    (2, 1, 98, 4, 2, 4, True),       # ragged tiles, grouped K/V
    (2, 2, 130, 4, 4, 64, False),
    (4, 1, 256, 8, 4, 128, True),
    (1, 1, 70, 2, 1, 256, True),     # the largest head dim
    (2, 1, 66, 2, 2, 36, False),     # d not a power of two
])
def test_local_attention_fp32(P, b, s, hq, hkv, d, causal):
    need_gpu()
    q, k, v = global_qkv(b, s, hq, hkv, d, torch.float32, seed=s + d)
    q_head = oracle.seq2head(shard_seq(q, P))
    k_head = oracle.seq2head(shard_seq(k, P))
    v_head = oracle.seq2head(shard_seq(v, P))
    out = uly.ulysses_local_attention([t.cuda() for t in q_head], [t.cuda() for t in k_head],
                                      [t.cuda() for t in v_head], causal)
    torch.cuda.synchronize()
    for r in range(P):
        assert_close(out[r], oracle.attention(q_head[r], k_head[r], v_head[r], causal), torch.float32, f"rank {r}")
    device_ok()
