"""Training on the two-level (Ulysses x Ring) layout: the forward with its softmax statistics
and the backward, against the oracle's attention backward on the global tensors (the
two-level split changes where tokens and heads live, not what is computed), and bit for bit
against the plain Ulysses training path over the same ranks where that path accepts the shape."""
import pytest
import torch

import oracle
import sequence_attention_seq_gb300 as uly
from gpu_util import assert_close, assert_close_grad, bits_equal, device_ok, need_gpu
from sequence_attention_seq_gb300.inputs import global_grad, global_qkv, shard_seq

pytestmark = pytest.mark.gpu

CASES = [
    # Pu, Pr, b, s, hq, hkv, d, causal
    (2, 2, 1, 512, 4, 4, 128, True),     # P | h_kv: also bitwise against plain Ulysses
    (2, 2, 2, 512, 4, 2, 64, False),
    (2, 4, 1, 1024, 4, 2, 128, True),    # h_kv < P: only the two-level split accepts it
    (1, 2, 1, 256, 2, 1, 128, True),     # ring only
    (4, 1, 1, 512, 8, 4, 64, True),      # Ulysses only
    (4, 2, 1, 1024, 8, 8, 128, False),   # P | h_kv
    (4, 8, 1, 1024, 4, 4, 64, True),     # 32 rank buffers: the wide parameter block
]


def _inputs(P, b, s, hq, hkv, d, seed):
    q, k, v = global_qkv(b, s, hq, hkv, d, torch.bfloat16, seed=seed)
    do = global_grad(b, s, hq, d, torch.bfloat16, seed=seed + 1)
    return q, k, v, do, [shard_seq(x, P) for x in (q, k, v, do)]


@pytest.mark.parametrize("Pu,Pr,b,s,hq,hkv,d,causal", CASES)
def test_usp_training_against_oracle(Pu, Pr, b, s, hq, hkv, d, causal):
    need_gpu()
    P = Pu * Pr
    q, k, v, do, (qs, ks, vs, dos) = _inputs(P, b, s, hq, hkv, d, seed=s + 3 * Pu + Pr)
    qd, kd, vd, dod = ([t.cuda() for t in x] for x in (qs, ks, vs, dos))
    o, lse = uly.ulysses_usp_attn_fwd_lse(qd, kd, vd, causal, Pu, Pr)
    dq, dk, dv = uly.ulysses_usp_attn_bwd(qd, kd, vd, o, dod, lse, causal, Pu, Pr)
    torch.cuda.synchronize()
    device_ok()
    # the forward output and the statistics: O from the oracle, L = log sum exp of scaled scores
    want_o = shard_seq(oracle.attention(q, k, v, causal), P)
    for j in range(P):
        assert_close(o[j], want_o[j], torch.bfloat16, f"o rank {j}")
    want_lse = oracle.attention_lse(q, k, causal)  # [b, hq, s]
    got_lse = torch.cat([x.cpu().double() for x in lse], dim=1)
    err = (got_lse - want_lse).abs().max().item()
    assert err <= 2e-4, f"lse max-abs {err:.3e}"
    # the gradients of the global attention, split into the seq layout of every rank
    gq, gk, gv = oracle.attention_bwd(q, k, v, do, causal)
    for name, got, ref in (("dq", dq, gq), ("dk", dk, gk), ("dv", dv, gv)):
        want = shard_seq(ref, P)
        for j in range(P):
            assert_close_grad(got[j], want[j], f"{name} rank {j}")


@pytest.mark.parametrize("Pu,Pr,hkv,causal", [(2, 2, 4, True), (4, 2, 8, False), (2, 4, 8, True)])
def test_usp_training_matches_plain_ulysses_bitwise(Pu, Pr, hkv, causal):
    need_gpu()
    P, b, s, hq, d = Pu * Pr, 1, 1024, 8, 128
    _, _, _, _, (qs, ks, vs, dos) = _inputs(P, b, s, hq, hkv, d, seed=7)
    qd, kd, vd, dod = ([t.cuda() for t in x] for x in (qs, ks, vs, dos))
    o_u, lse_u = uly.ulysses_usp_attn_fwd_lse(qd, kd, vd, causal, Pu, Pr)
    g_u = uly.ulysses_usp_attn_bwd(qd, kd, vd, o_u, dod, lse_u, causal, Pu, Pr)
    o_p, lse_p = uly.ulysses_dist_attn_fwd_lse(qd, kd, vd, causal)
    g_p = uly.ulysses_dist_attn_bwd(qd, kd, vd, o_p, dod, lse_p, causal)
    torch.cuda.synchronize()
    device_ok()
    for j in range(P):
        assert bits_equal(o_u[j], o_p[j]), f"o rank {j}"
    # both hold [b, heads of the unit or rank, s]: laid side by side they are [b, hq, s]
    assert bits_equal(torch.cat(lse_u, dim=1), torch.cat(lse_p, dim=1))
    for name, a, c in zip(("dq", "dk", "dv"), g_u, g_p):
        for j in range(P):
            assert bits_equal(a[j], c[j]), f"{name} rank {j}"


def test_usp_backward_deterministic():
    need_gpu()
    Pu, Pr, b, s, hq, hkv, d = 2, 2, 1, 512, 4, 2, 128
    _, _, _, _, (qs, ks, vs, dos) = _inputs(Pu * Pr, b, s, hq, hkv, d, seed=11)
    qd, kd, vd, dod = ([t.cuda() for t in x] for x in (qs, ks, vs, dos))
    o, lse = uly.ulysses_usp_attn_fwd_lse(qd, kd, vd, True, Pu, Pr)
    a = uly.ulysses_usp_attn_bwd(qd, kd, vd, o, dod, lse, True, Pu, Pr)
    c = uly.ulysses_usp_attn_bwd(qd, kd, vd, o, dod, lse, True, Pu, Pr)
    torch.cuda.synchronize()
    device_ok()
    for x, y in zip(a, c):
        for j in range(Pu * Pr):
            assert bits_equal(x[j], y[j])


def test_usp_training_argument_errors():
    need_gpu()
    Pu, Pr, b, s, hq, hkv, d = 2, 2, 1, 512, 4, 2, 128
    _, _, _, _, (qs, ks, vs, dos) = _inputs(Pu * Pr, b, s, hq, hkv, d, seed=13)
    qd, kd, vd, dod = ([t.cuda() for t in x] for x in (qs, ks, vs, dos))
    o, lse = uly.ulysses_usp_attn_fwd_lse(qd, kd, vd, False, Pu, Pr)
    with pytest.raises(ValueError):  # rank count does not match Pu x Pr
        uly.ulysses_usp_attn_bwd(qd, kd, vd, o, dod, lse, False, Pu, 3)
    with pytest.raises(ValueError):  # one statistics array per Ulysses unit
        uly.ulysses_usp_attn_bwd(qd, kd, vd, o, dod, lse[:1], False, Pu, Pr)
    with pytest.raises(uly.UlyssesError) as e:  # too small a workspace
        uly.ulysses_usp_attn_bwd(qd, kd, vd, o, dod, lse, False, Pu, Pr,
                                 workspace=torch.empty(256, dtype=torch.uint8, device="cuda"))
    assert e.value.status == uly.ULY_ERR_INVALID_ARG
    with pytest.raises(uly.UlyssesError) as e:  # a gradient buffer aliasing an input
        uly.ulysses_usp_attn_bwd(qd, kd, vd, o, dod, lse, False, Pu, Pr,
                                 grads=(qd, [torch.empty_like(x) for x in kd], [torch.empty_like(x) for x in vd]))
    assert e.value.status == uly.ULY_ERR_INVALID_ARG
    # (s/Pr) % 128 != 0: no kernel for it
    _, _, _, _, (q2, k2, v2, d2) = _inputs(4, 1, 320, 4, 2, 128, seed=17)
    q2, k2, v2, d2 = ([t.cuda() for t in x] for x in (q2, k2, v2, d2))
    with pytest.raises(uly.UlyssesError) as e:
        uly.ulysses_usp_attn_fwd_lse(q2, k2, v2, False, 2, 2)
    assert e.value.status == uly.ULY_ERR_UNSUPPORTED
    # fp32 has no training kernels
    q3, k3, v3 = ([t.float() for t in x] for x in (qd, kd, vd))
    with pytest.raises(uly.UlyssesError) as e:
        uly.ulysses_usp_attn_fwd_lse(q3, k3, v3, False, Pu, Pr)
    assert e.value.status == uly.ULY_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    device_ok()
