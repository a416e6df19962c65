"""The per-process halves of the exchange (ulysses_a2a_pack / ulysses_a2a_unpack) on the GPU.

(1) Each kernel produces exactly the block layout the multi-process exchange is defined by
    (the reshapes of test_multirank_a2a_cpu.py, which the gloo test checks against the
    oracle), bit for bit.
(2) P ranks emulated on one GPU: every rank packs, the blocks are swapped as the
    all-to-all would (block r of rank j's send buffer becomes block j of rank r's receive
    buffer), every rank unpacks: the result equals ulysses_a2a_seq2head (and, back,
    ulysses_a2a_head2seq) bit for bit.
(3) The forward, and the training forward and backward, over a process group of one rank
    (the only group one GPU can form) run the whole multi-process path and equal the
    single-process calls bit for bit."""

import pytest
import torch

import sequence_attention_seq_gb300 as uly
from gpu_util import bits_equal, device_ok, need_gpu
from sequence_attention_seq_gb300.inputs import random_bits, seq_shards_qkv
from test_multirank_a2a_cpu import _pack, _unpack

pytestmark = pytest.mark.gpu

SHAPES = [
    # P, b, s, h, d, dtype
    (4, 2, 512, 8, 128, torch.bfloat16),
    (3, 3, 96, 6, 64, torch.float32),
    (8, 1, 1024, 64, 128, torch.bfloat16),
    (1, 2, 256, 4, 64, torch.bfloat16),
    (2, 1, 64, 2, 20, torch.bfloat16),   # runs of 40 bytes: 8-byte vectors
]


@pytest.mark.parametrize("P,b,s,h,d,dt", SHAPES)
def test_pack_unpack_layouts(P, b, s, h, d, dt):
    need_gpu()
    S = s // P
    seq = random_bits((b, S, h, d), dt, seed=P + s, device="cuda")
    head = random_bits((b, s, h // P, d), dt, seed=P + s + 1, device="cuda")
    blocks = random_bits((P, b, S, h // P, d), dt, seed=P + s + 2, device="cuda")
    got = [uly.ulysses_a2a_pack(seq, 0, P), uly.ulysses_a2a_pack(head, 1, P),
           uly.ulysses_a2a_unpack(blocks, 0), uly.ulysses_a2a_unpack(blocks, 1)]
    want = [_pack(seq, 0, P), _pack(head, 1, P), _unpack(blocks, 0), _unpack(blocks, 1)]
    torch.cuda.synchronize()
    device_ok()
    for n, (g, w) in enumerate(zip(got, want)):
        assert g.shape == w.shape and bits_equal(g, w.contiguous()), f"layout {n}"


@pytest.mark.parametrize("P,b,s,h,d,dt", SHAPES)
def test_emulated_exchange_equals_the_device_exchange(P, b, s, h, d, dt):
    need_gpu()
    S = s // P
    shards = [random_bits((b, S, h, d), dt, seed=10 * j + s, device="cuda") for j in range(P)]
    sends = [uly.ulysses_a2a_pack(x, 0, P) for x in shards]
    heads = [uly.ulysses_a2a_unpack(torch.stack([sends[j][r] for j in range(P)]), 0) for r in range(P)]
    want = uly.ulysses_a2a_seq2head(shards)
    sends = [uly.ulysses_a2a_pack(x, 1, P) for x in heads]
    back = [uly.ulysses_a2a_unpack(torch.stack([sends[r][j] for r in range(P)]), 1) for j in range(P)]
    torch.cuda.synchronize()
    device_ok()
    for r in range(P):
        assert bits_equal(heads[r], want[r]), f"seq -> head, rank {r}"
    for j in range(P):
        assert bits_equal(back[j], shards[j]), f"round trip, rank {j}"
    assert all(bits_equal(x, y) for x, y in zip(uly.ulysses_a2a_head2seq(heads), back))


def test_multi_process_forward_on_one_rank():
    need_gpu()
    import socket

    import torch.distributed as dist

    from sequence_attention_seq_gb300.inputs import global_grad
    from sequence_attention_seq_gb300.multi import (ulysses_dist_attn_bwd_multi, ulysses_dist_attn_fwd_lse_multi,
                                                    ulysses_dist_attn_fwd_multi)

    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    torch.cuda.set_device(0)
    dist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{port}", rank=0, world_size=1)
    try:
        qs, ks, vs = seq_shards_qkv(1, 2, 384, 4, 2, 128, torch.bfloat16, seed=4, device="cuda")
        for causal in (False, True):
            got = ulysses_dist_attn_fwd_multi(qs[0], ks[0], vs[0], causal)
            want = uly.ulysses_dist_attn_fwd(qs, ks, vs, causal)[0]
            torch.cuda.synchronize()
            assert bits_equal(got, want), f"causal={causal}"
            # training: forward with statistics, then the backward through both exchanges
            do = global_grad(2, 384, 4, 128, torch.bfloat16, seed=5, device="cuda")
            o_m, saved = ulysses_dist_attn_fwd_lse_multi(qs[0], ks[0], vs[0], causal)
            g_m = ulysses_dist_attn_bwd_multi(do, saved, causal)
            o_s, lse_s = uly.ulysses_dist_attn_fwd_lse(qs, ks, vs, causal)
            g_s = uly.ulysses_dist_attn_bwd(qs, ks, vs, o_s, [do], lse_s, causal)
            torch.cuda.synchronize()
            assert bits_equal(o_m, o_s[0]) and bits_equal(saved[4], lse_s[0])
            for name, a, c in zip(("dq", "dk", "dv"), g_m, g_s):
                assert bits_equal(a, c[0]), f"{name} causal={causal}"
    finally:
        dist.destroy_process_group()
    device_ok()
