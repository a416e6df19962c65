"""Seeded synthetic inputs shared by the tests, the oracle checks and the benchmark.

This module only draws numbers and slices them into per-rank shards; it holds none of
the method's arithmetic (no all-to-all, no attention).  Both the CUDA path and the
oracle consume what it returns.

Conventions (the pages fix no generator, so these are this library's choice):

* Gaussian inputs: ``torch.Generator(device).manual_seed(seed)``, then
  ``torch.randn`` in float32 for the *global* Q ``[b, s, h_q, d]``, then K and V
  ``[b, s, h_kv, d]``, in that order, then a round-to-nearest-even cast to the I/O
  dtype.  Small cases draw on the CPU generator; very large cases may draw on a CUDA
  generator (same recipe, different stream of numbers) so they are not limited by host
  RNG speed.
* Uniform random bits (permute-only workloads): ``torch.randint`` over the full
  16-bit (or 32-bit) range, reinterpreted as the element type.
* Output gradients (backward): ``torch.randn`` in float32 for the global dO
  ``[b, s, h_q, d]`` from a generator of its own, then the same cast.
* Sequence sharding (the input layout of DistributedAttention): rank ``j`` holds the
  contiguous token block ``[j*s/P, (j+1)*s/P)`` of every batch row, all heads.
"""
from __future__ import annotations

import torch

__all__ = ["global_qkv", "global_grad", "shard_seq", "random_bits", "seq_shards_qkv", "empty_like_shards"]


def global_qkv(b, s, h_q, h_kv, d, dtype=torch.bfloat16, seed=0, device="cpu"):
    """Return global (unsharded) Q [b,s,h_q,d], K and V [b,s,h_kv,d] drawn N(0,1)."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    q = torch.randn((b, s, h_q, d), generator=g, dtype=torch.float32, device=device)
    k = torch.randn((b, s, h_kv, d), generator=g, dtype=torch.float32, device=device)
    v = torch.randn((b, s, h_kv, d), generator=g, dtype=torch.float32, device=device)
    return q.to(dtype), k.to(dtype), v.to(dtype)


def global_grad(b, s, h_q, d, dtype=torch.bfloat16, seed=0, device="cpu"):
    """Return a global output gradient dO [b,s,h_q,d] drawn N(0,1) (its own generator and
    seed, so it does not disturb the Q/K/V stream)."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return torch.randn((b, s, h_q, d), generator=g, dtype=torch.float32, device=device).to(dtype)


def shard_seq(x, P):
    """Split a global [b, s, ...] tensor into P contiguous per-rank token blocks."""
    s = x.shape[1]
    if s % P:
        raise ValueError(f"s={s} is not divisible by P={P}")
    n = s // P
    return [x[:, j * n:(j + 1) * n].contiguous() for j in range(P)]


def seq_shards_qkv(P, b, s, h_q, h_kv, d, dtype=torch.bfloat16, seed=0, device="cpu"):
    """Per-rank seq-partitioned Q, K, V lists, each entry [b, s/P, heads, d]."""
    q, k, v = global_qkv(b, s, h_q, h_kv, d, dtype, seed, device)
    return shard_seq(q, P), shard_seq(k, P), shard_seq(v, P)


def random_bits(shape, dtype=torch.bfloat16, seed=0, device="cpu"):
    """Uniform random bit patterns reinterpreted as ``dtype`` (NaNs and infs included)."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    if dtype in (torch.bfloat16, torch.float16):
        raw = torch.randint(-32768, 32768, shape, generator=g, dtype=torch.int16, device=device)
    elif dtype == torch.float32:
        raw = torch.randint(-(2 ** 31), 2 ** 31, shape, generator=g, dtype=torch.int32, device=device)
    else:
        raise ValueError(f"unsupported dtype {dtype}")
    return raw.view(dtype)


def empty_like_shards(shape, P, dtype, device):
    """P freshly allocated tensors of one shape (caller-owned output buffers)."""
    return [torch.empty(shape, dtype=dtype, device=device) for _ in range(P)]
