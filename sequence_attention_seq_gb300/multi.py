"""Ulysses across GPUs: one process per GPU, one sequence-parallel rank per process.

"DeepSpeed-Ulysses 深度解析", section "构建序列并行通信组": DistributedAttention runs over a
sequence-parallel process group of P ranks; section "核心设计：沿序列切分 + 两次
All-to-All", steps 3-5: all-to-all #1 on Q, K and V, the local attention of the rank's
heads, all-to-all #2 on the output.  Each exchange here is the library's pack kernel (the
rank's P send blocks), one equal-split all-to-all of those blocks over the process group
("大模型分布式训练通信原语及其应用", section 5 "AllToAll（全交换）": block i goes to
rank i, blocks arrive in sending-rank order), and the library's unpack kernel.  Every step
of the computation runs in the library's kernels; torch.distributed (NCCL between GPUs)
only moves the blocks.

Layout: this rank holds tokens [rank*s/P, (rank+1)*s/P) of every head (seq shard
[b, s/P, h, d]); between the exchanges it holds heads [rank*h/P, (rank+1)*h/P) of every
token (head shard [b, s, h/P, d]).  Both head counts must be multiples of P: each rank
holds whole K/V heads.
"""
from __future__ import annotations

import torch
import torch.distributed as dist

from . import (ulysses_a2a_pack, ulysses_a2a_unpack, ulysses_local_attention, ulysses_local_attention_bwd,
               ulysses_local_attention_fwd_lse)

__all__ = ["exchange", "ulysses_dist_attn_fwd_multi", "ulysses_dist_attn_fwd_lse_multi",
           "ulysses_dist_attn_bwd_multi"]


def exchange(x, direction, group=None, stream=None):
    """This rank's part of all-to-all #1 (direction 0: seq shard -> head shard) or #2
    (direction 1: head shard -> seq shard) over the process group."""
    P = dist.get_world_size(group)
    send = ulysses_a2a_pack(x, direction, P, stream=stream)
    recv = torch.empty_like(send)
    dist.all_to_all_single(recv, send, group=group)  # ordered after the pack on the current stream
    return ulysses_a2a_unpack(recv, direction, stream=stream)


def ulysses_dist_attn_fwd_multi(q, k, v, causal, group=None):
    """The Ulysses forward with one rank per process: q [b, s/P, h_q, d], k and v
    [b, s/P, h_kv, d] (this rank's tokens, all heads) -> o [b, s/P, h_q, d]."""
    P = dist.get_world_size(group)
    hq, hkv = q.shape[2], k.shape[2]
    if hq % P or hkv % P:
        raise ValueError(f"h_q={hq} and h_kv={hkv} must be multiples of the {P} ranks")
    qh, kh, vh = (exchange(x, 0, group) for x in (q, k, v))
    (oh,) = ulysses_local_attention([qh], [kh], [vh], causal)
    return exchange(oh, 1, group)


def ulysses_dist_attn_fwd_lse_multi(q, k, v, causal, group=None):
    """The forward for training: returns (o [b, s/P, h_q, d], saved), saved holding what the
    backward needs -- this rank's head shards of Q, K, V and O and the natural-log
    log-sum-exp [b, h_q/P, s] of its heads' rows."""
    P = dist.get_world_size(group)
    if q.shape[2] % P or k.shape[2] % P:
        raise ValueError(f"h_q={q.shape[2]} and h_kv={k.shape[2]} must be multiples of the {P} ranks")
    qh, kh, vh = (exchange(x, 0, group) for x in (q, k, v))
    (oh,), (lse,) = ulysses_local_attention_fwd_lse([qh], [kh], [vh], causal)
    return exchange(oh, 1, group), (qh, kh, vh, oh, lse)


def ulysses_dist_attn_bwd_multi(do, saved, causal, group=None):
    """The backward ("02 · DeepSpeed-Ulysses", section 5: the backward of all-to-all #2 is
    all-to-all #1 and the reverse): dO [b, s/P, h_q, d] of this rank's tokens and the saved
    forward state -> (dq, dk, dv) in this rank's seq layout."""
    qh, kh, vh, oh, lse = saved
    doh = exchange(do, 0, group)
    (dqh,), (dkh,), (dvh,) = ulysses_local_attention_bwd([qh], [kh], [vh], [oh], [doh], [lse], causal)
    return tuple(exchange(g, 1, group) for g in (dqh, dkh, dvh))
