"""bf16 tensor-core attention (tcgen05) against the fp64 oracle:
max-abs <= 1.5e-2 and mean-abs <= 2e-3, on shapes that span several 128-row tiles and
ragged tails."""
import pytest
import torch

import oracle
import sequence_attention_seq_gb300 as uly
from gpu_util import assert_close, device_ok, need_gpu
from sequence_attention_seq_gb300.inputs import global_qkv, shard_seq

pytestmark = pytest.mark.gpu

CASES = [
    # P, b, s, hq, hkv, d, causal
    (1, 1, 128, 1, 1, 128, False),   # one tile
    (1, 1, 128, 1, 1, 128, True),
    (1, 1, 128, 1, 1, 64, False),
    (2, 1, 384, 4, 4, 128, False),   # several tiles
    (2, 1, 384, 4, 4, 128, True),
    (2, 2, 320, 4, 2, 64, True),     # ragged tail, grouped K/V
    (2, 2, 320, 4, 2, 64, False),
    (4, 1, 512, 16, 4, 128, True),   # 4 query heads per K/V head
    (1, 1, 1, 1, 1, 64, False),      # one token
    (2, 1, 1000, 2, 2, 128, True),   # ragged, several tiles
    (3, 1, 771, 3, 3, 64, False),
]


@pytest.mark.parametrize("P,b,s,hq,hkv,d,causal", CASES)
def test_local_attention_bf16(P, b, s, hq, hkv, d, causal):
    need_gpu()
    q, k, v = global_qkv(b, s, hq, hkv, d, torch.bfloat16, seed=s * 3 + d)
    q_head = oracle.seq2head(shard_seq(q, P))
    k_head = oracle.seq2head(shard_seq(k, P))
    v_head = oracle.seq2head(shard_seq(v, P))
    out = uly.ulysses_local_attention([t.cuda() for t in q_head], [t.cuda() for t in k_head],
                                      [t.cuda() for t in v_head], causal)
    torch.cuda.synchronize()
    device_ok()
    for r in range(P):
        assert_close(out[r], oracle.attention(q_head[r], k_head[r], v_head[r], causal), torch.bfloat16, f"rank {r}")


def test_large_scores_rescaling():
    """Scores that grow along the key axis force the running maximum up many times (the
    output rescale path), and a huge score spike must dominate its row."""
    need_gpu()
    s, d = 640, 128
    g = torch.Generator().manual_seed(5)
    q = torch.randn(1, s, 1, d, generator=g)
    k = torch.randn(1, s, 1, d, generator=g) * torch.linspace(0.2, 4.0, s).view(1, s, 1, 1)
    v = torch.randn(1, s, 1, d, generator=g)
    q, k, v = q.bfloat16(), k.bfloat16(), v.bfloat16()
    for causal in (False, True):
        out = uly.ulysses_local_attention([q.cuda()], [k.cuda()], [v.cuda()], causal)
        torch.cuda.synchronize()
        assert_close(out[0], oracle.attention(q, k, v, causal), torch.bfloat16, f"causal={causal}")
    device_ok()
