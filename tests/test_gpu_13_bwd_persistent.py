"""The backward kernels with several work items per CTA.  For short sequences (non-causal,
or causal with at most 64 tiles and every unit's tiles in L2) the dK/dV and dQ kernels
keep one CTA per SM and walk their items; at each item boundary the next item's fixed tiles
load and its first products run while the current item's accumulators are stored.  The
small parity cases give every CTA at most one item, so these shapes are sized to give
each CTA several: ragged last tiles, query heads sharing a K/V head, both head dims, both
masks, the local and the fused distributed backward, against the oracle's attention
backward ("02 · DeepSpeed-Ulysses", section 5) and bit for bit between repeat calls."""
import pytest
import torch

import oracle
import sequence_attention_seq_gb300 as uly
from gpu_util import assert_close_grad, bits_equal, device_ok, need_gpu
from sequence_attention_seq_gb300.inputs import global_grad, global_qkv, shard_seq

pytestmark = pytest.mark.gpu

LOCAL_CASES = [
    # P, b, s, hq, hkv, d, causal; items over at most 152 CTAs
    (4, 8, 320, 32, 16, 64, True),   # ragged last tile, 2 query heads per K/V head: 384 dK/dV, 768 dQ items
    (2, 8, 384, 16, 16, 128, True),  # 384 dK/dV and dQ items
]


def _cuda(xs):
    return [x.cuda() for x in xs]


@pytest.mark.parametrize("P,b,s,hq,hkv,d,causal", LOCAL_CASES)
def test_local_backward_many_items(P, b, s, hq, hkv, d, causal):
    need_gpu()
    q, k, v = global_qkv(b, s, hq, hkv, d, torch.bfloat16, seed=11 * s + d)
    do = global_grad(b, s, hq, d, torch.bfloat16, seed=11 * s + d + 1)
    qh, kh, vh, doh = (oracle.seq2head(shard_seq(x, P)) for x in (q, k, v, do))
    qd, kd, vd, dod = _cuda(qh), _cuda(kh), _cuda(vh), _cuda(doh)
    o, lse = uly.ulysses_local_attention_fwd_lse(qd, kd, vd, causal)
    g1 = uly.ulysses_local_attention_bwd(qd, kd, vd, o, dod, lse, causal)
    g2 = uly.ulysses_local_attention_bwd(qd, kd, vd, o, dod, lse, causal)
    torch.cuda.synchronize()
    device_ok()
    for r in range(P):
        want = oracle.attention_bwd(qh[r], kh[r], vh[r], doh[r], causal)
        for name, got, again, ref in zip(("dq", "dk", "dv"), g1, g2, want):
            assert_close_grad(got[r], ref, f"{name} rank {r}")
            assert bits_equal(got[r], again[r]), f"{name} rank {r}: repeat call differs"


@pytest.mark.parametrize("causal", [True, False])
def test_fused_backward_many_items(causal):
    # fused: one launch over global heads, 4 x 16 units x 4 tiles = 256 dK/dV and dQ items
    need_gpu()
    P, b, s, hq, hkv, d = 4, 4, 512, 16, 16, 64
    q, k, v = global_qkv(b, s, hq, hkv, d, torch.bfloat16, seed=31 + causal)
    do = global_grad(b, s, hq, d, torch.bfloat16, seed=32 + causal)
    qs, ks, vs, dos = (shard_seq(x, P) for x in (q, k, v, do))
    qd, kd, vd, dod = _cuda(qs), _cuda(ks), _cuda(vs), _cuda(dos)
    o, lse = uly.ulysses_dist_attn_fwd_lse(qd, kd, vd, causal, fused=True)
    fused = uly.ulysses_dist_attn_bwd(qd, kd, vd, o, dod, lse, causal, fused=True)
    plain = uly.ulysses_dist_attn_bwd(qd, kd, vd, o, dod, lse, causal, fused=False)
    torch.cuda.synchronize()
    device_ok()
    want = oracle.attention_bwd(q, k, v, do, causal)
    for name, got, other, ref in zip(("dq", "dk", "dv"), fused, plain, want):
        ref_s = shard_seq(ref, P)
        for j in range(P):
            assert_close_grad(got[j], ref_s[j], f"{name} rank {j}")
            assert bits_equal(got[j], other[j]), f"{name} rank {j}: fused and unfused differ"
