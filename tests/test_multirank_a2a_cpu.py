"""The exchange across processes, on CPU (gloo): every rank packs its shard into P send
blocks in the layout ulysses_a2a_pack produces (block i = heads [i*h/P, (i+1)*h/P) of the
rank's tokens), one equal-split all_to_all_single moves them, and the blocks are placed in
the layout ulysses_a2a_unpack produces (block j at tokens [j*s/P, (j+1)*s/P)).  The result
must be the oracle's all-to-all #1 for that rank, and the reverse exchange must give the
rank's shard back ("大模型分布式训练通信原语及其应用", section 5 "AllToAll（全交换）";
"DeepSpeed-Ulysses 深度解析", step 3).  The GPU test of the pack and unpack kernels checks
that they produce exactly these layouts."""
import os
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _pack(x, direction, P):
    if direction == 0:  # seq shard [b, S, h, d] -> [P, b, S, h/P, d]
        b, S, h, d = x.shape
        return x.reshape(b, S, P, h // P, d).permute(2, 0, 1, 3, 4).contiguous()
    b, s, H, d = x.shape  # head shard [b, s, H, d] -> [P, b, s/P, H, d]
    return x.reshape(b, P, s // P, H, d).permute(1, 0, 2, 3, 4).contiguous()


def _unpack(r, direction):
    P, b, S, H, d = r.shape
    if direction == 0:  # block j at tokens [j*S, (j+1)*S)
        return r.permute(1, 0, 2, 3, 4).reshape(b, P * S, H, d)
    return r.permute(1, 2, 0, 3, 4).reshape(b, S, P * H, d)  # block r at heads [r*H, (r+1)*H)


def _worker(rank, world, port, shape, out):
    import torch.distributed as dist

    sys.path.insert(0, ROOT)
    import oracle

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    b, s, h, d = shape
    g = torch.Generator().manual_seed(7)
    x = torch.randn((b, s, h, d), generator=g, dtype=torch.float64)
    S = s // world
    shards = [x[:, j * S:(j + 1) * S].contiguous() for j in range(world)]
    send = _pack(shards[rank], 0, world)
    recv = torch.empty_like(send)
    dist.all_to_all_single(recv, send)
    head = _unpack(recv, 0)
    want = oracle.seq2head(shards)[rank]
    ok_fwd = torch.equal(head, want)
    send = _pack(head, 1, world)
    recv = torch.empty_like(send)
    dist.all_to_all_single(recv, send)
    ok_back = torch.equal(_unpack(recv, 1), shards[rank])
    out.put((rank, ok_fwd, ok_back))
    dist.destroy_process_group()


@pytest.mark.parametrize("world,shape", [(2, (2, 64, 4, 8)), (3, (1, 96, 6, 4))])
def test_exchange_across_processes_gloo(world, shape):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29600 + (os.getpid() + world) % 1000
    procs = [ctx.Process(target=_worker, args=(r, world, port, shape, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=180) for _ in procs)
    for p in procs:
        p.join(timeout=180)
        assert p.exitcode == 0
    for rank, ok_fwd, ok_back in res:
        assert ok_fwd, f"rank {rank}: the exchange differs from the oracle's all-to-all #1"
        assert ok_back, f"rank {rank}: the reverse exchange did not restore the shard"
