"""DistributedAttention (sequence_attention_seq_gb300/attention.py) on the GPU.

(1) With the library's kernels, the module's output and its autograd gradients are the bits
    of the direct calls (ulysses_dist_attn_fwd_lse, ulysses_dist_attn_bwd).
(2) The differentiable exchanges are exact: a local attention that returns 2q gives 2q
    back in seq layout, and gradients 2 dO for Q and zeros for the unused K and V.
(3) With a local attention written in PyTorch (fp32), output and gradients match the same
    attention applied to the global tensors ("DeepSpeed-Ulysses 深度解析", section "核心设计"
    steps 3-5: each rank's heads see the whole sequence; the exchanges' backward is the
    swapped exchange).
(4) One rank per process: over a one-rank NCCL group the module gives the one-GPU module's
    bits (several ranks are checked on CPU in test_multirank_module_cpu.py)."""
import math

import pytest
import torch

import sequence_attention_seq_gb300 as uly
from gpu_util import bits_equal, device_ok, need_gpu
from sequence_attention_seq_gb300.attention import DistributedAttention, head_to_seq, seq_to_head
from sequence_attention_seq_gb300.inputs import global_grad, global_qkv, shard_seq

pytestmark = pytest.mark.gpu


def _leaves(xs):
    return [x.cuda().requires_grad_() for x in xs]


def torch_attention(causal):
    """Plain attention in PyTorch on [b, s, heads, d] tensors, K/V heads shared by
    h_q/h_kv consecutive query heads."""
    def f(q, k, v):
        g = q.shape[2] // k.shape[2]
        k, v = k.repeat_interleave(g, dim=2), v.repeat_interleave(g, dim=2)
        sc = torch.einsum("bqhd,bkhd->bhqk", q, k) / math.sqrt(q.shape[3])
        if causal:
            s = q.shape[1]
            sc = sc.masked_fill(torch.ones(s, s, dtype=torch.bool, device=q.device).triu(1), float("-inf"))
        return torch.einsum("bhqk,bkhd->bqhd", torch.softmax(sc, dim=-1), v)
    return f


@pytest.mark.parametrize("P,b,s,hq,hkv,d,causal,fused", [
    (4, 1, 512, 8, 4, 128, True, None),    # fused kernels chosen
    (2, 2, 384, 4, 2, 64, False, None),    # (s/P) % 128 != 0: unfused
    (4, 1, 512, 8, 4, 128, False, False),  # unfused by request
    (4, 1, 512, 8, 2, 64, True, None),     # replicated K/V heads
])
def test_kernels_module_gives_the_direct_calls_bits(P, b, s, hq, hkv, d, causal, fused):
    need_gpu()
    q, k, v = global_qkv(b, s, hq, hkv, d, torch.bfloat16, seed=s + P)
    do = global_grad(b, s, hq, d, torch.bfloat16, seed=s + P + 1)
    qs, ks, vs = (_leaves(shard_seq(x, P)) for x in (q, k, v))
    dos = [t.cuda() for t in shard_seq(do, P)]
    att = DistributedAttention(causal=causal, fused=fused)
    o = att(qs, ks, vs)
    grads = torch.autograd.grad(o, qs + ks + vs, grad_outputs=dos)
    fz = ((s // P) % 128 == 0) if fused is None else fused
    qd, kd, vd = ([x.detach() for x in xs] for xs in (qs, ks, vs))
    o_d, lse = uly.ulysses_dist_attn_fwd_lse(qd, kd, vd, causal, fused=fz)
    g_d = uly.ulysses_dist_attn_bwd(qd, kd, vd, o_d, dos, lse, causal, fused=fz)
    torch.cuda.synchronize()
    device_ok()
    for j in range(P):
        assert bits_equal(o[j], o_d[j]), f"output, rank {j}"
    for n, name in enumerate(("dq", "dk", "dv")):
        for j in range(P):
            assert bits_equal(grads[n * P + j], g_d[n][j]), f"{name}, rank {j}"


def test_differentiable_exchanges_are_exact():
    need_gpu()
    P, b, s, h, d = 4, 2, 256, 8, 64
    q, k, v = global_qkv(b, s, h, h, d, torch.bfloat16, seed=3)
    do = global_grad(b, s, h, d, torch.bfloat16, seed=4)
    qs, ks, vs = (_leaves(shard_seq(x, P)) for x in (q, k, v))
    dos = [t.cuda() for t in shard_seq(do, P)]
    att = DistributedAttention(local_attention=lambda a, b_, c: a * 2.0)
    o = att(qs, ks, vs)
    grads = torch.autograd.grad(o, qs + ks + vs, grad_outputs=dos, allow_unused=True)
    torch.cuda.synchronize()
    device_ok()
    for j in range(P):
        assert bits_equal(o[j], qs[j].detach() * 2.0)
        assert bits_equal(grads[j], dos[j] * 2.0)
        for g in (grads[P + j], grads[2 * P + j]):
            assert g is None or not g.any()
    # the functions alone: head_to_seq(seq_to_head(x)) == x, gradient passed back unchanged
    xs = _leaves(shard_seq(q, P))
    back = head_to_seq(seq_to_head(xs))
    gx = torch.autograd.grad(back, xs, grad_outputs=dos)
    assert all(bits_equal(a, b_.detach()) for a, b_ in zip(back, xs))
    assert all(bits_equal(a, b_) for a, b_ in zip(gx, dos))


@pytest.mark.parametrize("P,b,s,hq,hkv,causal", [(4, 1, 256, 8, 4, True), (2, 2, 192, 4, 2, False)])
def test_custom_local_attention_matches_global_attention(P, b, s, hq, hkv, causal):
    need_gpu()
    d = 32
    q, k, v = global_qkv(b, s, hq, hkv, d, torch.float32, seed=s)
    do = global_grad(b, s, hq, d, torch.float32, seed=s + 1)
    f = torch_attention(causal)
    qs, ks, vs = (_leaves(shard_seq(x, P)) for x in (q, k, v))
    dos = [t.cuda() for t in shard_seq(do, P)]
    o = DistributedAttention(local_attention=f)(qs, ks, vs)
    grads = torch.autograd.grad(o, qs + ks + vs, grad_outputs=dos)
    qg, kg, vg = (x.cuda().requires_grad_() for x in (q, k, v))
    og = f(qg, kg, vg)
    want = torch.autograd.grad(og, (qg, kg, vg), grad_outputs=do.cuda())
    torch.cuda.synchronize()
    device_ok()
    assert (torch.cat(o, dim=1) - og).abs().max().item() <= 1e-5
    for n, name in enumerate(("dq", "dk", "dv")):
        got = torch.cat(grads[n * P:(n + 1) * P], dim=1)
        assert (got - want[n]).abs().max().item() <= 1e-4, name


def test_module_over_a_process_group_of_one_rank():
    need_gpu()
    import socket

    import torch.distributed as dist

    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    torch.cuda.set_device(0)
    dist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{port}", rank=0, world_size=1)
    try:
        b, s, hq, hkv, d = 2, 384, 4, 2, 128
        q, k, v = global_qkv(b, s, hq, hkv, d, torch.bfloat16, seed=8)
        do = global_grad(b, s, hq, d, torch.bfloat16, seed=9).cuda()
        for causal in (False, True):
            q1, k1, v1 = _leaves([q])[0], _leaves([k])[0], _leaves([v])[0]
            o1 = DistributedAttention(group=dist.group.WORLD, causal=causal)(q1, k1, v1)
            g1 = torch.autograd.grad(o1, (q1, k1, v1), grad_outputs=do)
            q2, k2, v2 = _leaves([q]), _leaves([k]), _leaves([v])
            o2 = DistributedAttention(causal=causal, fused=False)(q2, k2, v2)
            g2 = torch.autograd.grad(o2, q2 + k2 + v2, grad_outputs=[do])
            torch.cuda.synchronize()
            assert bits_equal(o1, o2[0])
            for a, c in zip(g1, g2):
                assert bits_equal(a, c)
        # fp32: the forward only (the fp32 kernels have no backward)
        q, k, v = global_qkv(1, 128, 2, 2, 64, torch.float32, seed=10)
        qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
        o1 = DistributedAttention(group=dist.group.WORLD, causal=True)(qd, kd, vd)
        o2 = uly.ulysses_dist_attn_fwd([qd], [kd], [vd], True)
        torch.cuda.synchronize()
        assert bits_equal(o1, o2[0])
    finally:
        dist.destroy_process_group()
    device_ok()
