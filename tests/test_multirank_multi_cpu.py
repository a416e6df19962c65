"""The multi-process Ulysses forward and backward (sequence_attention_seq_gb300/multi.py) over
gloo process groups of 2 and 4 CPU ranks.

On one GPU the process group has a single rank, so every exchange there is the identity and
a swapped direction or a misplaced block would go unseen.  Here the composition itself is
checked at several ranks: multi.py's exchanges run over the process group, with the
per-process kernels and the local attention replaced on CPU by their definitions -- the
block layouts of ulysses_a2a_pack / ulysses_a2a_unpack (the reshapes that
test_multirank_a2a_cpu.py checks against the oracle, and that the GPU test checks the kernels
against) and the oracle's local attention, statistics and backward.  Each rank's output and
gradients must equal the oracle's single-process Ulysses pipeline for that rank
("DeepSpeed-Ulysses 深度解析", section "核心设计" steps 3-5; "02 · DeepSpeed-Ulysses",
section 5 for the backward)."""
import datetime
import os
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(rank, world, port, shape):
    import torch.distributed as dist

    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import oracle
    from sequence_attention_seq_gb300 import multi
    from test_multirank_a2a_cpu import _pack, _unpack

    # the per-process kernels and the local attention by their definitions, on CPU
    multi.ulysses_a2a_pack = lambda x, direction, P, stream=None: _pack(x, direction, P)
    multi.ulysses_a2a_unpack = lambda r, direction, stream=None: _unpack(r, direction).contiguous()
    multi.ulysses_local_attention = lambda q, k, v, causal: [oracle.attention(q[0], k[0], v[0], causal)]

    def fwd_lse(q, k, v, causal):
        return [oracle.attention(q[0], k[0], v[0], causal)], [oracle.attention_lse(q[0], k[0], causal)]

    def bwd(q, k, v, o, do, lse, causal):
        dq, dk, dv = oracle.attention_bwd(q[0], k[0], v[0], do[0].to(q[0].dtype), causal)
        return [dq], [dk], [dv]

    multi.ulysses_local_attention_fwd_lse = fwd_lse
    multi.ulysses_local_attention_bwd = bwd

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world, timeout=datetime.timedelta(seconds=60))
    b, s, hq, hkv, d, causal = shape
    g = torch.Generator().manual_seed(11)
    q = torch.randn((b, s, hq, d), generator=g)
    k = torch.randn((b, s, hkv, d), generator=g)
    v = torch.randn((b, s, hkv, d), generator=g)
    do = torch.randn((b, s, hq, d), generator=g)
    S = s // world
    shard = lambda x: [x[:, j * S:(j + 1) * S].contiguous() for j in range(world)]  # noqa: E731
    qs, ks, vs, dos = shard(q), shard(k), shard(v), shard(do)

    o = multi.ulysses_dist_attn_fwd_multi(qs[rank], ks[rank], vs[rank], causal)
    want_o = oracle.dist_attn_fwd(qs, ks, vs, causal)[rank]
    o2, saved = multi.ulysses_dist_attn_fwd_lse_multi(qs[rank], ks[rank], vs[rank], causal)
    grads = multi.ulysses_dist_attn_bwd_multi(dos[rank], saved, causal)
    want_g = [x[rank] for x in oracle.dist_attn_bwd(qs, ks, vs, dos, causal)]
    ok = {"o": torch.equal(o, want_o), "o_training": torch.equal(o2, want_o),
          "shapes": [tuple(x.shape) for x in grads] == [tuple(x.shape) for x in want_g]}
    for name, got, want in zip(("dq", "dk", "dv"), grads, want_g):
        ok[name] = torch.equal(got, want)
    dist.destroy_process_group()
    return ok


def _worker(rank, world, port, shape, out):
    # a failing rank reports at once (its peers' collectives then time out after 60 s)
    try:
        out.put((rank, _run(rank, world, port, shape)))
    except Exception as e:  # noqa: BLE001
        out.put((rank, {f"error: {e!r}": False}))


@pytest.mark.parametrize("world,shape", [
    (2, (1, 64, 4, 2, 8, True)),    # grouped K/V heads (2 query heads per K/V head), causal
    (2, (2, 32, 2, 2, 4, False)),
    (4, (1, 64, 8, 4, 8, True)),
])
def test_multi_process_forward_and_backward_gloo(world, shape):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29800 + (os.getpid() * 3 + world + shape[1]) % 1000
    procs = [ctx.Process(target=_worker, args=(r, world, port, shape, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted((q.get(timeout=180) for _ in procs), key=lambda x: x[0])
    for p in procs:
        p.join(timeout=300)
        assert p.exitcode == 0
    for rank, ok in res:
        bad = [k for k, v in ok.items() if not v]
        assert not bad, f"rank {rank}: {bad} differ from the oracle's Ulysses pipeline"
