"""DistributedAttention with one rank per process (sequence_attention_seq_gb300/attention.py)
over gloo groups of 2 and 4 CPU ranks, with a local attention written in PyTorch.

The per-process exchange kernels are replaced on CPU by their definitions (the block
layouts of test_multirank_a2a_cpu.py, which the GPU test checks the kernels against); the
autograd composition is the module's own: all-to-all #1 on Q, K, V, the local attention,
all-to-all #2, and in the backward each exchange's reverse ("DeepSpeed-Ulysses 深度解析",
section "核心设计：沿序列切分 + 两次 All-to-All": the backward swaps the split and gather
dimensions).  Every rank's output and gradients must equal, in float64, the same attention
applied to the global tensors and differentiated by autograd on one process."""
import datetime
import math
import os
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _attention(causal):
    def f(q, k, v):
        g = q.shape[2] // k.shape[2]
        k, v = k.repeat_interleave(g, dim=2), v.repeat_interleave(g, dim=2)
        sc = torch.einsum("bqhd,bkhd->bhqk", q, k) / math.sqrt(q.shape[3])
        if causal:
            s = q.shape[1]
            sc = sc.masked_fill(torch.ones(s, s, dtype=torch.bool).triu(1), float("-inf"))
        return torch.einsum("bhqk,bkhd->bqhd", torch.softmax(sc, dim=-1), v)
    return f


def _run(rank, world, port, shape):
    import torch.distributed as dist

    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    from sequence_attention_seq_gb300 import multi
    from sequence_attention_seq_gb300.attention import DistributedAttention
    from test_multirank_a2a_cpu import _pack, _unpack

    multi.ulysses_a2a_pack = lambda x, direction, P, stream=None: _pack(x, direction, P)
    multi.ulysses_a2a_unpack = lambda r, direction, stream=None: _unpack(r, direction).contiguous()

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world, timeout=datetime.timedelta(seconds=60))
    b, s, hq, hkv, d, causal = shape
    g = torch.Generator().manual_seed(5)
    q, k, v, do = (torch.randn((b, s, h, d), generator=g, dtype=torch.float64) for h in (hq, hkv, hkv, hq))
    S = s // world
    mine = [x[:, rank * S:(rank + 1) * S].clone().requires_grad_() for x in (q, k, v)]
    f = _attention(causal)
    o = DistributedAttention(local_attention=f, group=dist.group.WORLD)(*mine)
    grads = torch.autograd.grad(o, mine, grad_outputs=do[:, rank * S:(rank + 1) * S].contiguous())
    qg, kg, vg = (x.clone().requires_grad_() for x in (q, k, v))
    og = f(qg, kg, vg)
    want = torch.autograd.grad(og, (qg, kg, vg), grad_outputs=do)
    sl = slice(rank * S, (rank + 1) * S)
    err = {"o": (o - og[:, sl]).abs().max().item()}
    for name, a, w in zip(("dq", "dk", "dv"), grads, want):
        err[name] = (a - w[:, sl]).abs().max().item()
    dist.destroy_process_group()
    return err


def _worker(rank, world, port, shape, out):
    # a failing rank reports at once (its peers' collectives then time out after 60 s)
    try:
        out.put((rank, _run(rank, world, port, shape)))
    except Exception as e:  # noqa: BLE001
        out.put((rank, {f"error: {e!r}": float("inf")}))


@pytest.mark.parametrize("world,shape", [
    (2, (1, 32, 4, 2, 8, True)),
    (2, (2, 16, 2, 2, 4, False)),
    (4, (1, 32, 8, 4, 8, True)),
])
def test_module_over_gloo(world, shape):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 30400 + (os.getpid() * 7 + world + shape[1]) % 1000
    procs = [ctx.Process(target=_worker, args=(r, world, port, shape, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted((q.get(timeout=180) for _ in procs), key=lambda x: x[0])
    for p in procs:
        p.join(timeout=300)
        assert p.exitcode == 0
    for rank, err in res:
        bad = {k: e for k, e in err.items() if not e <= 1e-12}
        assert not bad, f"rank {rank}: {bad}"
