"""Pins for the oracle's two-level forward (Ulysses inside groups of Pu ranks, ring across Pr
groups; "长上下文训练中的 SP 与 CP", section "组合与配置：区分算法组合和并行维度", "Ulysses + Ring"
subsection; "02 · DeepSpeed-Ulysses", section 4 "a2a+p2p 分层 CP").  The ring's online-softmax
merge and causal block skipping are checked against full attention computed by a library
routine; the degenerate sizes reduce to Ulysses (Pr = 1) and to a pure ring (Pu = 1)."""
import pytest
import torch
import torch.nn.functional as F

import oracle
from sequence_attention_seq_gb300.inputs import global_qkv, shard_seq


def _full_attention(q, k, v, causal):
    g = q.shape[2] // k.shape[2]
    kk = k.double().repeat_interleave(g, dim=2)
    vv = v.double().repeat_interleave(g, dim=2)
    o = F.scaled_dot_product_attention(q.double().transpose(1, 2), kk.transpose(1, 2), vv.transpose(1, 2),
                                       is_causal=causal)
    return o.transpose(1, 2)


@pytest.mark.parametrize("Pu,Pr,b,s,hq,hkv,d,causal", [
    (2, 2, 1, 16, 4, 2, 8, True), (2, 2, 2, 16, 4, 4, 8, False), (4, 2, 1, 32, 8, 4, 4, True),
    (2, 4, 1, 32, 2, 2, 6, True), (1, 4, 1, 16, 2, 1, 4, True), (3, 2, 1, 18, 6, 3, 5, False)])
def test_usp_equals_full_attention(Pu, Pr, b, s, hq, hkv, d, causal):
    q, k, v = global_qkv(b, s, hq, hkv, d, torch.float64, seed=s + Pu * 7 + Pr)
    P = Pu * Pr
    out = oracle.usp_fwd(shard_seq(q, P), shard_seq(k, P), shard_seq(v, P), causal, Pu, Pr)
    want = _full_attention(q, k, v, causal)
    assert torch.allclose(torch.cat(out, 1), want, atol=1e-12, rtol=0)


@pytest.mark.parametrize("causal", [False, True])
def test_usp_with_one_ring_group_is_ulysses(causal):
    P, b, s, hq, hkv, d = 4, 1, 32, 8, 4, 8
    qs, ks, vs = (shard_seq(x, P) for x in global_qkv(b, s, hq, hkv, d, torch.float32, seed=3))
    a = oracle.usp_fwd(qs, ks, vs, causal, P, 1)
    b2 = oracle.dist_attn_fwd(qs, ks, vs, causal)
    for x, y in zip(a, b2):
        assert torch.allclose(x, y, atol=1e-13, rtol=0)


def test_usp_matches_ulysses_for_every_split():
    """The same 8 ranks split 8x1, 4x2, 2x4, 1x8 all give the Ulysses output."""
    P, b, s, hq, hkv, d = 8, 1, 64, 8, 8, 4
    qs, ks, vs = (shard_seq(x, P) for x in global_qkv(b, s, hq, hkv, d, torch.bfloat16, seed=9))
    want = oracle.dist_attn_fwd(qs, ks, vs, True)
    for Pu, Pr in ((8, 1), (4, 2), (2, 4), (1, 8)):
        got = oracle.usp_fwd(qs, ks, vs, True, Pu, Pr)
        for x, y in zip(got, want):
            assert torch.allclose(x, y, atol=1e-12, rtol=0), (Pu, Pr)


def test_first_segment_causal_sees_only_itself():
    """Causal: ring group 0's queries depend only on segment 0 -- changing every later K/V
    block leaves their output unchanged (those blocks are skipped, not merged as zeros)."""
    Pu, Pr, b, s, hq, d = 2, 2, 1, 16, 2, 4
    q, k, v = global_qkv(b, s, hq, hq, d, torch.float64, seed=1)
    P = Pu * Pr
    out1 = oracle.usp_fwd(shard_seq(q, P), shard_seq(k, P), shard_seq(v, P), True, Pu, Pr)
    k2, v2 = k.clone(), v.clone()
    k2[:, s // 2:] += 5.0
    v2[:, s // 2:] -= 3.0
    out2 = oracle.usp_fwd(shard_seq(q, P), shard_seq(k2, P), shard_seq(v2, P), True, Pu, Pr)
    for j in range(Pu):  # ranks of ring group 0 hold the first half of the tokens
        assert torch.equal(out1[j], out2[j])
    assert not torch.equal(out1[Pu], out2[Pu])


def test_scaled_256k_example_shapes():
    """The 256K-token, Ulysses 4 x Ring 2 example scaled by 1/1024: 8 ranks hold 32 tokens
    each; after the exchange inside each four-rank group every rank holds its group's 128
    tokens for a quarter of the heads, and the two groups cover the 256 tokens."""
    Pu, Pr, b, s, h, d = 4, 2, 1, 256, 8, 2
    q = torch.arange(b * s * h * d, dtype=torch.float64).reshape(b, s, h, d)
    qs = shard_seq(q, Pu * Pr)
    assert all(x.shape == (b, 32, h, d) for x in qs)
    qh = oracle.usp_group_exchange(qs, Pu)
    for j, x in enumerate(qh):
        g, u = divmod(j, Pu)
        assert x.shape == (b, 128, h // Pu, d)
        want = q[:, g * 128:(g + 1) * 128, u * (h // Pu):(u + 1) * (h // Pu)]
        assert torch.equal(x, want)
