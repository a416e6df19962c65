"""DistributedAttention as a PyTorch module with autograd.

"DeepSpeed-Ulysses 深度解析", section "核心设计：沿序列切分 + 两次 All-to-All" (last
paragraph): the all-to-all is a differentiable operation whose backward is the same
exchange with the split and gather dimensions swapped; section "两行代码替换注意力": the
module wraps a local attention and runs it between the two exchanges.

The P sequence-parallel ranks run either on one GPU, as P tensors (lists of P seq-layout
tensors [b, s/P, heads, d] in and out), or one per process over a torch.distributed
process group (this rank's seq-layout tensor in and out).  The local attention is either
the library's kernels (local_attention=None: the forward with statistics, then the
attention backward; on one GPU the exchanges can be folded into the kernels' tile
addressing), or any callable local_attention(q, k, v) on head-layout tensors
[b, s, heads, d] -> [b, s, heads, d], which autograd differentiates, placed between the
library's exchange kernels wrapped as autograd functions.  Every exchange and every
built-in attention step runs in the library's kernels; PyTorch provides autograd, memory
and, across processes, the collective that moves the exchange's blocks.
"""
from __future__ import annotations

import torch

from . import (ulysses_a2a_head2seq, ulysses_a2a_seq2head, ulysses_dist_attn_bwd, ulysses_dist_attn_fwd,
               ulysses_dist_attn_fwd_lse)

__all__ = ["DistributedAttention", "seq_to_head", "head_to_seq"]


def _filled(grads, meta):
    """Gradients of a list of outputs, zeros for the outputs that received none."""
    shape, dtype, device = meta
    return [torch.zeros(shape, dtype=dtype, device=device) if g is None else g.contiguous() for g in grads]


class _SeqToHead(torch.autograd.Function):
    """All-to-all #1 over P tensors on one GPU; its backward is all-to-all #2."""

    @staticmethod
    def forward(ctx, *xs):
        outs = ulysses_a2a_seq2head([x.contiguous() for x in xs])
        ctx.meta = (outs[0].shape, outs[0].dtype, outs[0].device)
        return tuple(outs)

    @staticmethod
    def backward(ctx, *grads):
        return tuple(ulysses_a2a_head2seq(_filled(grads, ctx.meta)))


class _HeadToSeq(torch.autograd.Function):
    """All-to-all #2 over P tensors on one GPU; its backward is all-to-all #1."""

    @staticmethod
    def forward(ctx, *xs):
        outs = ulysses_a2a_head2seq([x.contiguous() for x in xs])
        ctx.meta = (outs[0].shape, outs[0].dtype, outs[0].device)
        return tuple(outs)

    @staticmethod
    def backward(ctx, *grads):
        return tuple(ulysses_a2a_seq2head(_filled(grads, ctx.meta)))


def seq_to_head(xs):
    """Differentiable all-to-all #1 over P tensors on one GPU: [b, s/P, h, d] -> [b, s, h/P, d]."""
    return list(_SeqToHead.apply(*xs))


def head_to_seq(xs):
    """Differentiable all-to-all #2 over P tensors on one GPU: [b, s, h/P, d] -> [b, s/P, h, d]."""
    return list(_HeadToSeq.apply(*xs))


def _fused_fits(P, S, dtype, backward):
    """Shapes the fused kernels take: bf16, (s/P) % 128 == 0, at most 64 ranks (48 backward)."""
    return dtype == torch.bfloat16 and S % 128 == 0 and P <= (48 if backward else 64)


class _Kernels(torch.autograd.Function):
    """The library's whole forward over P tensors on one GPU, and its backward."""

    @staticmethod
    def forward(ctx, causal, fused, P, *qkv):
        q, k, v = list(qkv[:P]), list(qkv[P:2 * P]), list(qkv[2 * P:])
        S, dtype = q[0].shape[1], q[0].dtype
        use_fused = _fused_fits(P, S, dtype, False) if fused is None else bool(fused)
        ctx.P, ctx.causal, ctx.fused = P, causal, fused
        if dtype != torch.bfloat16:  # the fp32 kernels have no backward
            ctx.trainable = False
            return tuple(ulysses_dist_attn_fwd(q, k, v, causal, fused=use_fused))
        ctx.trainable = True
        o, lse = ulysses_dist_attn_fwd_lse(q, k, v, causal, fused=use_fused)
        ctx.save_for_backward(*q, *k, *v, *o, *lse)
        return tuple(o)

    @staticmethod
    def backward(ctx, *do):
        if not ctx.trainable:
            raise RuntimeError("DistributedAttention: the library's backward kernels are bf16 only")
        P = ctx.P
        t = ctx.saved_tensors
        q, k, v, o, lse = (list(t[i * P:(i + 1) * P]) for i in range(5))
        S = q[0].shape[1]
        use_fused = _fused_fits(P, S, q[0].dtype, True) if ctx.fused is None else bool(ctx.fused)
        dq, dk, dv = ulysses_dist_attn_bwd(q, k, v, o, _filled(do, (o[0].shape, o[0].dtype, o[0].device)), lse,
                                           ctx.causal, fused=use_fused)
        return (None, None, None, *dq, *dk, *dv)


class _Exchange(torch.autograd.Function):
    """This rank's part of an exchange over a process group (direction 0: all-to-all #1,
    1: all-to-all #2); its backward is the exchange in the other direction."""

    @staticmethod
    def forward(ctx, x, direction, group):
        from .multi import exchange

        ctx.direction, ctx.group = direction, group
        return exchange(x.contiguous(), direction, group)

    @staticmethod
    def backward(ctx, g):
        from .multi import exchange

        return exchange(g.contiguous(), 1 - ctx.direction, ctx.group), None, None


class _KernelsMulti(torch.autograd.Function):
    """The library's forward with one rank per process, and its backward."""

    @staticmethod
    def forward(ctx, causal, group, q, k, v):
        from .multi import ulysses_dist_attn_fwd_lse_multi, ulysses_dist_attn_fwd_multi

        ctx.causal, ctx.group = causal, group
        q, k, v = q.contiguous(), k.contiguous(), v.contiguous()
        ctx.trainable = q.dtype == torch.bfloat16
        if not ctx.trainable:  # the fp32 kernels have no backward
            return ulysses_dist_attn_fwd_multi(q, k, v, causal, group)
        o, saved = ulysses_dist_attn_fwd_lse_multi(q, k, v, causal, group)
        ctx.save_for_backward(*saved)
        return o

    @staticmethod
    def backward(ctx, do):
        from .multi import ulysses_dist_attn_bwd_multi

        if not ctx.trainable:
            raise RuntimeError("DistributedAttention: the library's backward kernels are bf16 only")
        dq, dk, dv = ulysses_dist_attn_bwd_multi(do.contiguous(), ctx.saved_tensors, ctx.causal, ctx.group)
        return None, None, dq, dk, dv


class DistributedAttention(torch.nn.Module):
    """Ulysses attention over P sequence-parallel ranks.

    local_attention: None for the library's kernels (bf16 with d in {64, 128} for training;
        fp32 forward only), else a callable (q, k, v) -> o on head-layout tensors
        [b, s, heads, d]; it applies its own mask and scale.  With a callable, the K/V head
        count must be a multiple of P (the exchanges split every tensor's heads P ways).
    group: None for P ranks on one GPU (forward takes lists of P tensors and returns one),
        else a torch.distributed process group with one rank per process (forward takes
        this rank's tensors and returns one).
    causal: the causal mask of the library's kernels (ignored with a callable).
    fused: one GPU, library kernels: fold both exchanges into the attention kernels; None
        chooses them wherever they take the shape.
    """

    def __init__(self, local_attention=None, group=None, causal=False, fused=None):
        super().__init__()
        self.local_attention = local_attention
        self.group = group
        self.causal = bool(causal)
        self.fused = fused

    def forward(self, q, k, v):
        if self.group is None:
            P = len(q)
            if len(k) != P or len(v) != P:
                raise ValueError(f"{P} query tensors but {len(k)} key and {len(v)} value tensors")
            if self.local_attention is None:
                return list(_Kernels.apply(self.causal, self.fused, P, *q, *k, *v))
            qh, kh, vh = seq_to_head(q), seq_to_head(k), seq_to_head(v)
            return head_to_seq([self.local_attention(a, b_, c) for a, b_, c in zip(qh, kh, vh)])
        if self.local_attention is None:
            return _KernelsMulti.apply(self.causal, self.group, q, k, v)
        qh, kh, vh = (_Exchange.apply(x, 0, self.group) for x in (q, k, v))
        return _Exchange.apply(self.local_attention(qh, kh, vh), 1, self.group)
