"""All-to-all #1 / #2 kernels against the oracle: bit-exact (the exchanges are bit copies)."""
import pytest
import torch

import oracle
import sequence_attention_seq_gb300 as uly
from gpu_util import bits_equal, need_gpu
from sequence_attention_seq_gb300.inputs import random_bits, shard_seq

pytestmark = pytest.mark.gpu

SMALL = [
    # P, b, s, h, d, dtype          (run = (h/P)*d*e bytes; 16-B vectors down to 2-B)
    (2, 1, 64, 4, 16, torch.float32),     # the tiny configuration
    (1, 1, 8, 2, 8, torch.bfloat16),      # P = 1
    (3, 2, 9, 6, 5, torch.bfloat16),      # 20-B runs, odd everything
    (5, 1, 15, 10, 7, torch.float32),     # 56-B runs
    (4, 3, 12, 4, 1, torch.bfloat16),     # 2-B runs
    (8, 1, 64, 64, 4, torch.bfloat16),
    (16, 2, 256, 32, 64, torch.bfloat16),
    (64, 1, 128, 64, 128, torch.bfloat16),  # P at its maximum, 256-B runs
    (4, 2, 4096, 8, 128, torch.bfloat16),
]


@pytest.mark.parametrize("P,b,s,h,d,dtype", SMALL)
def test_exchanges_bit_exact(P, b, s, h, d, dtype):
    need_gpu()
    x = random_bits((b, s, h, d), dtype, seed=P * 7 + s)
    shards = shard_seq(x, P)
    dev = [t.cuda() for t in shards]
    got = uly.ulysses_a2a_seq2head(dev)
    torch.cuda.synchronize()
    want = oracle.seq2head(shards)
    for g, w in zip(got, want):
        assert bits_equal(g.cpu(), w)
    y = [random_bits((b, s, h // P, d), dtype, seed=100 + r) for r in range(P)]
    got2 = uly.ulysses_a2a_head2seq([t.cuda() for t in y])
    torch.cuda.synchronize()
    want2 = oracle.head2seq(y)
    for g, w in zip(got2, want2):
        assert bits_equal(g.cpu(), w)


SWEEP_S = [8192, 32768, 131072, 262144]
SWEEP_P = [2, 4, 8, 16, 32, 64]


@pytest.mark.parametrize("s", SWEEP_S)
@pytest.mark.parametrize("P", SWEEP_P)
def test_permute_sweep_full_size(P, s):
    """bf16 [P][1, s/P, 64, 128] uniform random bits at the sweep's full sizes: the round trip
    is the identity bit for bit, and a slice of the head dim (the exchange commutes with
    slicing d) matches the oracle bit for bit."""
    need_gpu()
    h, d = 64, 128
    dev = [random_bits((1, s // P, h, d), torch.bfloat16, seed=j, device="cuda") for j in range(P)]
    head = uly.ulysses_a2a_seq2head(dev)
    back = uly.ulysses_a2a_head2seq(head)
    torch.cuda.synchronize()
    for a, c in zip(dev, back):
        assert bits_equal(a, c)
    cols = slice(37, 39)
    want = oracle.seq2head([t[..., cols].cpu() for t in dev])
    for g, w in zip(head, want):
        assert bits_equal(g[..., cols].cpu(), w)
    want2 = oracle.head2seq([t[..., cols].cpu() for t in head])
    for g, w in zip(back, want2):
        assert bits_equal(g[..., cols].cpu(), w)
