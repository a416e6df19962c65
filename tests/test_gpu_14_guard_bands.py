"""Guard bands: every output, statistics array and workspace of the library sits inside a
larger buffer whose margins hold a known byte pattern, and the margins must come back
unchanged.  This catches a kernel writing past the end (or before the start) of what it
owns, in the cases most likely to do so: ragged last tiles, head sub-ranges, the
replicated-K/V partial sums, the two-level layout and the fused paths over more rank
buffers than the small parameter block holds.  The results themselves are
checked elsewhere; here only that nothing else was touched."""
import pytest
import torch

import sequence_attention_seq_gb300 as uly
from gpu_util import device_ok, need_gpu
from sequence_attention_seq_gb300.inputs import global_grad, global_qkv, shard_seq

pytestmark = pytest.mark.gpu

GUARD = 64 * 1024  # bytes on each side: more than one 128-row bf16 tile of a 128-wide head
PATTERN = 0xA5


class Guarded:
    """Hands out tensors inside guard bands and checks the bands afterwards."""

    def __init__(self):
        self.blocks = []

    def tensor(self, shape, dtype):
        n = torch.Size(shape).numel() * torch.empty((), dtype=dtype).element_size()
        body = (n + 255) // 256 * 256
        raw = torch.full((GUARD + body + GUARD,), PATTERN, dtype=torch.uint8, device="cuda")
        self.blocks.append((raw, n))
        return raw[GUARD:GUARD + n].view(dtype).view(shape)

    def like(self, xs):
        return [self.tensor(x.shape, x.dtype) for x in xs]

    def bytes(self, n):
        return self.tensor((max(n, 1),), torch.uint8)

    def check(self, what):
        torch.cuda.synchronize()
        for i, (raw, n) in enumerate(self.blocks):
            head, tail = raw[:GUARD], raw[GUARD + n:]
            assert bool((head == PATTERN).all()), f"{what}: buffer {i} written before its start"
            assert bool((tail == PATTERN).all()), f"{what}: buffer {i} written past its end"


def _seq(P, b, s, hq, hkv, d, dt, seed):
    q, k, v = global_qkv(b, s, hq, hkv, d, dt, seed=seed)
    return [[t.cuda() for t in shard_seq(x, P)] for x in (q, k, v)]


@pytest.mark.parametrize("P,b,s,hq,hkv,d,dt", [
    (2, 1, 200, 4, 2, 128, torch.bfloat16),   # ragged: s/P = 100 rows
    (4, 2, 512, 8, 8, 64, torch.bfloat16),
    (4, 1, 512, 8, 2, 128, torch.bfloat16),   # replicated K/V heads (h_kv < P)
    (2, 1, 96, 4, 4, 32, torch.float32),      # the fp32 kernel
    (32, 1, 4096, 32, 32, 64, torch.bfloat16),  # fused over 32 rank buffers: the wide parameter block
])
def test_forward_paths_stay_inside(P, b, s, hq, hkv, d, dt):
    need_gpu()
    qs, ks, vs = _seq(P, b, s, hq, hkv, d, dt, seed=s + d)
    for causal in (False, True):
        g = Guarded()
        qh = uly.ulysses_a2a_seq2head(qs, out_head=g.like([torch.empty(b, s, hq // P, d, dtype=dt)] * P))
        uly.ulysses_a2a_head2seq(qh, out_seq=g.like(qs))
        ws = g.bytes(uly.ulysses_dist_attn_workspace_bytes(P, b, s, hq, hkv, d, dt, False))
        uly.ulysses_dist_attn_fwd(qs, ks, vs, causal, fused=False, out_seq=g.like(qs), workspace=ws)
        if dt == torch.bfloat16 and (s // P) % 128 == 0:
            uly.ulysses_dist_attn_fwd(qs, ks, vs, causal, fused=True, out_seq=g.like(qs))
        if dt == torch.bfloat16:
            lse = [g.tensor((b, hq // P, s), torch.float32) for _ in range(P)]
            ws = g.bytes(uly.ulysses_dist_attn_workspace_bytes(P, b, s, hq, hkv, d, dt, False))
            uly.ulysses_dist_attn_fwd_lse(qs, ks, vs, causal, out_seq=g.like(qs), lse=lse, workspace=ws)
            if (hq // P) % 2 == 0:
                ws = g.bytes(uly.ulysses_dist_attn_overlap_workspace_bytes(P, b, s, hq, hkv, d, dt, 2))
                uly.ulysses_dist_attn_fwd_overlap(qs, ks, vs, causal, n_chunks=2, out_seq=g.like(qs), workspace=ws)
        g.check(f"forward causal={causal}")
        device_ok()


@pytest.mark.parametrize("P,b,s,hq,hkv,d,fused", [
    (2, 1, 200, 4, 2, 128, False),    # ragged last tile
    (4, 2, 512, 8, 8, 64, True),
    (4, 1, 512, 8, 2, 128, False),    # replicated K/V: fp32 partial sums in the workspace
    (4, 8, 320, 32, 16, 64, False),   # several work items per CTA
    (24, 1, 3072, 24, 24, 64, True),  # fused over 24 rank buffers: the wide parameter block
])
def test_backward_stays_inside(P, b, s, hq, hkv, d, fused):
    need_gpu()
    qs, ks, vs = _seq(P, b, s, hq, hkv, d, torch.bfloat16, seed=3 * s + d)
    dos = [t.cuda() for t in shard_seq(global_grad(b, s, hq, d, torch.bfloat16, seed=s), P)]
    for causal in (False, True):
        o, lse = uly.ulysses_dist_attn_fwd_lse(qs, ks, vs, causal, fused=fused)
        g = Guarded()
        grads = (g.like(qs), g.like(ks), g.like(vs))
        ws = g.bytes(uly.ulysses_attn_bwd_workspace_bytes(P, b, s, hq, hkv, d, torch.bfloat16, True, fused))
        uly.ulysses_dist_attn_bwd(qs, ks, vs, o, dos, lse, causal, grads=grads, workspace=ws, fused=fused)
        g.check(f"backward causal={causal}")
        device_ok()


def test_two_level_stays_inside():
    need_gpu()
    Pu, Pr, b, s, hq, hkv, d = 2, 2, 1, 512, 4, 2, 128
    P = Pu * Pr
    qs, ks, vs = _seq(P, b, s, hq, hkv, d, torch.bfloat16, seed=9)
    dos = [t.cuda() for t in shard_seq(global_grad(b, s, hq, d, torch.bfloat16, seed=10), P)]
    for causal in (False, True):
        g = Guarded()
        ws = g.bytes(uly.ulysses_usp_workspace_bytes(Pu, Pr, b, s, hq, hkv, d, torch.bfloat16))
        uly.ulysses_usp_attn_fwd(qs, ks, vs, causal, Pu, Pr, out_seq=g.like(qs), workspace=ws)
        o, lse = uly.ulysses_usp_attn_fwd_lse(qs, ks, vs, causal, Pu, Pr)
        grads = (g.like(qs), g.like(ks), g.like(vs))
        ws = g.bytes(uly.ulysses_usp_bwd_workspace_bytes(Pu, Pr, b, s, hq, hkv, d, torch.bfloat16))
        uly.ulysses_usp_attn_bwd(qs, ks, vs, o, dos, lse, causal, Pu, Pr, grads=grads, workspace=ws)
        g.check(f"two-level causal={causal}")
        device_ok()
