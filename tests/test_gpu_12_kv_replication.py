"""Fewer K/V heads than ranks (P a multiple of h_kv, e.g. one K/V head for all ranks): every
K/V head is replicated on the P/h_kv ranks whose query heads use it.  The forward (unfused,
fused, fp32) and the training path against the oracle's attention on the global tensors,
which is what replicated Ulysses must compute; fused, unfused and overlapped forwards bit
for bit; the unfused backward sums the replicas' dK/dV."""
import pytest
import torch

import oracle
import sequence_attention_seq_gb300 as uly
from gpu_util import (GRAD_MEAN, assert_close, assert_close_grad, assert_grad_within_rounding, bits_equal,
                      device_ok, need_gpu)
from sequence_attention_seq_gb300.inputs import global_grad, global_qkv, shard_seq

pytestmark = pytest.mark.gpu

CASES = [
    # P, b, s, hq, hkv, d, causal
    (4, 1, 512, 8, 2, 128, True),    # two K/V heads, each on two ranks
    (4, 2, 512, 4, 1, 128, False),   # one K/V head on every rank (multi-query)
    (8, 1, 1024, 8, 1, 64, True),
    (2, 1, 384, 4, 1, 128, True),    # ragged last tile
    (8, 1, 1024, 16, 4, 128, False),
]


def _inputs(P, b, s, hq, hkv, d, dt, seed):
    q, k, v = global_qkv(b, s, hq, hkv, d, dt, seed=seed)
    return q, k, v, [shard_seq(x, P) for x in (q, k, v)]


@pytest.mark.parametrize("P,b,s,hq,hkv,d,causal", CASES)
def test_replicated_kv_forward(P, b, s, hq, hkv, d, causal):
    need_gpu()
    q, k, v, (qs, ks, vs) = _inputs(P, b, s, hq, hkv, d, torch.bfloat16, seed=s + P + hkv)
    qd, kd, vd = ([t.cuda() for t in x] for x in (qs, ks, vs))
    unfused = uly.ulysses_dist_attn_fwd(qd, kd, vd, causal, fused=False)
    fused = uly.ulysses_dist_attn_fwd(qd, kd, vd, causal, fused=True) if (s // P) % 128 == 0 else None
    torch.cuda.synchronize()
    device_ok()
    want = shard_seq(oracle.attention(q, k, v, causal), P)
    for j in range(P):
        assert_close(unfused[j], want[j], torch.bfloat16, f"unfused rank {j}")
        if fused is not None:
            assert bits_equal(fused[j], unfused[j]), f"fused != unfused, rank {j}"


def test_replicated_kv_forward_fp32():
    need_gpu()
    P, b, s, hq, hkv, d = 4, 1, 128, 4, 1, 32
    q, k, v, (qs, ks, vs) = _inputs(P, b, s, hq, hkv, d, torch.float32, seed=3)
    out = uly.ulysses_dist_attn_fwd([t.cuda() for t in qs], [t.cuda() for t in ks], [t.cuda() for t in vs], True)
    torch.cuda.synchronize()
    device_ok()
    want = shard_seq(oracle.attention(q, k, v, True), P)
    for j in range(P):
        assert_close(out[j], want[j], torch.float32, f"rank {j}")


@pytest.mark.parametrize("P,b,s,hq,hkv,d,causal", [(4, 1, 512, 8, 2, 128, True), (4, 1, 512, 4, 1, 64, False),
                                                     (8, 1, 1024, 8, 1, 128, True),
                                                     # 192 dK/dV items: several per CTA of the persistent kernel
                                                     (8, 8, 384, 16, 2, 64, True)])
@pytest.mark.parametrize("fused", [False, True])
def test_replicated_kv_training(P, b, s, hq, hkv, d, causal, fused):
    need_gpu()
    if fused and (s // P) % 128:
        pytest.skip("the fused kernels need s/P to be a multiple of 128")
    q, k, v, (qs, ks, vs) = _inputs(P, b, s, hq, hkv, d, torch.bfloat16, seed=21 + s)
    do = global_grad(b, s, hq, d, torch.bfloat16, seed=22 + s)
    qd, kd, vd = ([t.cuda() for t in x] for x in (qs, ks, vs))
    dod = [t.cuda() for t in shard_seq(do, P)]
    o, lse = uly.ulysses_dist_attn_fwd_lse(qd, kd, vd, causal, fused=fused)
    dq, dk, dv = uly.ulysses_dist_attn_bwd(qd, kd, vd, o, dod, lse, causal, fused=fused)
    torch.cuda.synchronize()
    device_ok()
    # statistics per head rank, laid side by side: [b, hq, s]
    err = (torch.cat([x.cpu().double() for x in lse], dim=1) - oracle.attention_lse(q, k, causal)).abs().max().item()
    assert err <= 2e-4, f"lse max-abs {err:.3e}"
    gq, gk, gv = oracle.attention_bwd(q, k, v, do, causal)
    mags = oracle.attention_bwd_magnitudes(q, k, v, do, causal) if hq // hkv > 4 else None
    for n, (name, got, ref) in enumerate((("dq", dq, gq), ("dk", dk, gk), ("dv", dv, gv))):
        want = shard_seq(ref, P)
        for j in range(P):
            if name != "dq" and mags is not None:
                # dK/dV of a K/V head shared by more than 4 query heads: the bound scales with
                # the magnitude of the summed terms (see gpu_util)
                assert_grad_within_rounding(got[j], want[j], shard_seq(mags[n], P)[j], f"{name} rank {j}",
                                            mean_tol=GRAD_MEAN)
            else:
                assert_close_grad(got[j], want[j], f"{name} rank {j}")


@pytest.mark.parametrize("P,b,s,hq,hkv,d,causal,n_chunks", [(4, 1, 512, 8, 2, 128, True, 2),
                                                              (4, 2, 512, 16, 1, 64, False, 4),
                                                              (8, 1, 1024, 16, 2, 128, True, 2),
                                                              (2, 1, 384, 4, 1, 128, True, 1)])
def test_replicated_kv_overlap(P, b, s, hq, hkv, d, causal, n_chunks):
    # the overlapped forward: every chunk shares the rank's one K/V head; same bits as the
    # unfused forward
    need_gpu()
    _, _, _, (qs, ks, vs) = _inputs(P, b, s, hq, hkv, d, torch.bfloat16, seed=5 + n_chunks)
    qd, kd, vd = ([t.cuda() for t in x] for x in (qs, ks, vs))
    over = uly.ulysses_dist_attn_fwd_overlap(qd, kd, vd, causal, n_chunks=n_chunks)
    plain = uly.ulysses_dist_attn_fwd(qd, kd, vd, causal, fused=False)
    torch.cuda.synchronize()
    device_ok()
    for j in range(P):
        assert bits_equal(over[j], plain[j]), f"rank {j}: overlapped != unfused"


USP_CASES = [
    # Pu, Pr, b, s, hq, hkv, d, causal: fewer K/V heads than Ulysses ranks in every group
    (4, 2, 1, 1024, 8, 2, 128, True),    # each K/V head on 2 ranks of a group
    (4, 2, 1, 1024, 4, 1, 64, False),    # one K/V head for the whole group
    (2, 2, 2, 512, 4, 1, 128, True),
]


@pytest.mark.parametrize("Pu,Pr,b,s,hq,hkv,d,causal", USP_CASES)
def test_replicated_kv_two_level(Pu, Pr, b, s, hq, hkv, d, causal):
    # the two-level layout with replicated K/V heads: forward against the oracle's attention
    # on the global tensors and bit for bit against plain Ulysses over the same ranks (which
    # replicates too); the training path against the oracle's attention backward
    need_gpu()
    P = Pu * Pr
    q, k, v, (qs, ks, vs) = _inputs(P, b, s, hq, hkv, d, torch.bfloat16, seed=41 + s + Pu)
    do = global_grad(b, s, hq, d, torch.bfloat16, seed=42 + s + Pu)
    qd, kd, vd = ([t.cuda() for t in x] for x in (qs, ks, vs))
    dod = [t.cuda() for t in shard_seq(do, P)]
    out = uly.ulysses_usp_attn_fwd(qd, kd, vd, causal, Pu, Pr)
    # plain Ulysses over all P ranks needs P | h_q (the two-level split only Pu | h_q)
    plain = uly.ulysses_dist_attn_fwd(qd, kd, vd, causal, fused=False) if hq % P == 0 else None
    o, lse = uly.ulysses_usp_attn_fwd_lse(qd, kd, vd, causal, Pu, Pr)
    dq, dk, dv = uly.ulysses_usp_attn_bwd(qd, kd, vd, o, dod, lse, causal, Pu, Pr)
    torch.cuda.synchronize()
    device_ok()
    want = shard_seq(oracle.attention(q, k, v, causal), P)
    for j in range(P):
        assert_close(out[j], want[j], torch.bfloat16, f"rank {j}")
        if plain is not None:
            assert bits_equal(out[j], plain[j]), f"rank {j}: two-level != plain Ulysses"
        assert bits_equal(o[j], out[j]), f"rank {j}: the statistics store changed the output"
    gq, gk, gv = oracle.attention_bwd(q, k, v, do, causal)
    for name, got, ref in (("dq", dq, gq), ("dk", dk, gk), ("dv", dv, gv)):
        want = shard_seq(ref, P)
        for j in range(P):
            assert_close_grad(got[j], want[j], f"{name} rank {j}")
