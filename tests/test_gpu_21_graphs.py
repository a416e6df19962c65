"""The forward (unfused and fused), the training forward and backward, and the exchanges
captured in a CUDA graph and replayed: every replay gives the bits of the same calls made
eagerly.  The calls only enqueue kernels on the given stream (no synchronisation, no
allocation in the library), so a graph can hold a whole step for shapes where launch cost
matters.  (The no-allocation entry point is not covered here.)"""
import pytest
import torch

import sequence_attention_seq_gb300 as uly
from gpu_util import bits_equal, device_ok, need_gpu
from sequence_attention_seq_gb300.inputs import global_grad, seq_shards_qkv, shard_seq

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("P,b,s,hq,hkv,d,causal", [(4, 1, 512, 8, 4, 128, True), (2, 2, 256, 4, 2, 64, False)])
def test_graph_replay_gives_the_eager_bits(P, b, s, hq, hkv, d, causal):
    need_gpu()
    qs, ks, vs = seq_shards_qkv(P, b, s, hq, hkv, d, torch.bfloat16, seed=s + P, device="cuda")
    dos = shard_seq(global_grad(b, s, hq, d, torch.bfloat16, seed=s + P + 1, device="cuda"), P)

    def step():
        o_u = uly.ulysses_dist_attn_fwd(qs, ks, vs, causal, fused=False)
        o_f = uly.ulysses_dist_attn_fwd(qs, ks, vs, causal, fused=True)
        o, lse = uly.ulysses_dist_attn_fwd_lse(qs, ks, vs, causal, fused=True)
        g = uly.ulysses_dist_attn_bwd(qs, ks, vs, o, dos, lse, causal, fused=True)
        heads = uly.ulysses_a2a_seq2head(qs)
        back = uly.ulysses_a2a_head2seq(heads)
        return [*o_u, *o_f, *o, *lse, *g[0], *g[1], *g[2], *heads, *back]

    want = step()
    torch.cuda.synchronize()
    device_ok()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # warm-up on the capturing stream
        step()
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        got = step()
    for _ in range(2):
        for x in got:
            x.zero_()
        graph.replay()
        torch.cuda.synchronize()
        device_ok()
        for n, (a, c) in enumerate(zip(got, want)):
            assert bits_equal(a, c), f"result {n}"
