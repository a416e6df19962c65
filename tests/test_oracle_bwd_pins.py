"""Pins for the oracle's backward: attention gradients against float64 autograd through a
library routine and against central finite differences; the log-sum-exp against
torch.logsumexp; the exchange backward as the adjoint of the exchange; the whole Ulysses
backward against single-device autograd ("02 · DeepSpeed-Ulysses", section 5: each
all-to-all's backward is the all-to-all with the split axes swapped, and the local
attention's backward is the ordinary one)."""
import pytest
import torch
import torch.nn.functional as F

import oracle
from sequence_attention_seq_gb300.inputs import global_qkv, shard_seq


def _autograd(q, k, v, do, causal):
    g = q.shape[2] // k.shape[2]
    q = q.double().detach().requires_grad_()
    k = k.double().detach().requires_grad_()
    v = v.double().detach().requires_grad_()
    kk = k.repeat_interleave(g, dim=2)
    vv = v.repeat_interleave(g, dim=2)
    o = F.scaled_dot_product_attention(q.transpose(1, 2), kk.transpose(1, 2), vv.transpose(1, 2), is_causal=causal)
    o = o.transpose(1, 2)
    o.backward(do.double())
    return q.grad, k.grad, v.grad


@pytest.mark.parametrize("b,s,hq,hkv,d,causal", [
    (1, 9, 2, 2, 4, False), (2, 13, 4, 2, 8, True), (1, 16, 4, 1, 5, True), (1, 7, 3, 3, 6, False)])
def test_backward_vs_autograd(b, s, hq, hkv, d, causal):
    gen = torch.Generator().manual_seed(s * 7 + d)
    q = torch.randn(b, s, hq, d, generator=gen, dtype=torch.float64)
    k = torch.randn(b, s, hkv, d, generator=gen, dtype=torch.float64)
    v = torch.randn(b, s, hkv, d, generator=gen, dtype=torch.float64)
    do = torch.randn(b, s, hq, d, generator=gen, dtype=torch.float64)
    dq, dk, dv = oracle.attention_bwd(q, k, v, do, causal)
    rq, rk, rv = _autograd(q, k, v, do, causal)
    for a, r in ((dq, rq), (dk, rk), (dv, rv)):
        assert torch.allclose(a, r, atol=1e-11, rtol=0)


def test_backward_vs_finite_differences():
    gen = torch.Generator().manual_seed(3)
    b, s, hq, hkv, d = 1, 5, 2, 1, 3
    q = torch.randn(b, s, hq, d, generator=gen, dtype=torch.float64)
    k = torch.randn(b, s, hkv, d, generator=gen, dtype=torch.float64)
    v = torch.randn(b, s, hkv, d, generator=gen, dtype=torch.float64)
    do = torch.randn(b, s, hq, d, generator=gen, dtype=torch.float64)
    for causal in (False, True):
        dq, dk, dv = oracle.attention_bwd(q, k, v, do, causal)

        def loss(qq, kk, vv):
            return float((oracle.attention(qq, kk, vv, causal) * do).sum())

        eps = 1e-6
        for x, grad, idx in ((q, dq, 0), (k, dk, 1), (v, dv, 2)):
            flat = x.view(-1)
            for n in range(0, flat.numel(), 2):
                keep = flat[n].item()
                flat[n] = keep + eps
                up = loss(q, k, v)
                flat[n] = keep - eps
                dn = loss(q, k, v)
                flat[n] = keep
                assert abs((up - dn) / (2 * eps) - grad.view(-1)[n].item()) < 1e-6, (causal, idx, n)


@pytest.mark.parametrize("causal", [False, True])
def test_lse_vs_logsumexp(causal):
    gen = torch.Generator().manual_seed(5)
    b, s, hq, hkv, d = 2, 11, 4, 2, 8
    q = torch.randn(b, s, hq, d, generator=gen, dtype=torch.float64)
    k = torch.randn(b, s, hkv, d, generator=gen, dtype=torch.float64)
    lse = oracle.attention_lse(q, k, causal)
    kk = k.repeat_interleave(hq // hkv, dim=2)
    sc = torch.einsum("bihc,bjhc->bhij", q, kk) / d ** 0.5
    if causal:
        sc = sc.masked_fill(torch.ones(s, s, dtype=torch.bool).triu(1), float("-inf"))
    assert torch.allclose(lse, torch.logsumexp(sc, dim=-1), atol=1e-12, rtol=0)


@pytest.mark.parametrize("P,b,s,h,d", [(2, 1, 8, 4, 3), (4, 2, 16, 8, 2), (3, 1, 9, 6, 4)])
def test_exchange_backward_is_its_adjoint(P, b, s, h, d):
    """<seq2head(x), y> == <x, head2seq(y)>: the backward of each exchange is the other one."""
    gen = torch.Generator().manual_seed(P + s)
    x = [torch.randn(b, s // P, h, d, generator=gen, dtype=torch.float64) for _ in range(P)]
    y = [torch.randn(b, s, h // P, d, generator=gen, dtype=torch.float64) for _ in range(P)]
    lhs = sum(float((a * c).sum()) for a, c in zip(oracle.seq2head(x), y))
    rhs = sum(float((a * c).sum()) for a, c in zip(x, oracle.head2seq(y)))
    assert abs(lhs - rhs) < 1e-9


@pytest.mark.parametrize("P,b,s,hq,hkv,d,causal", [(2, 1, 16, 4, 2, 4, True), (4, 1, 16, 8, 4, 3, False)])
def test_dist_backward_equals_single_device(P, b, s, hq, hkv, d, causal):
    q, k, v = global_qkv(b, s, hq, hkv, d, torch.float32, seed=P + s)
    do = torch.randn(b, s, hq, d, generator=torch.Generator().manual_seed(1)).float()
    dq, dk, dv = oracle.dist_attn_bwd(shard_seq(q, P), shard_seq(k, P), shard_seq(v, P), shard_seq(do, P), causal)
    rq, rk, rv = _autograd(q, k, v, do, causal)
    assert torch.allclose(torch.cat(dq, 1), rq, atol=1e-9, rtol=0)
    assert torch.allclose(torch.cat(dk, 1), rk, atol=1e-9, rtol=0)
    assert torch.allclose(torch.cat(dv, 1), rv, atol=1e-9, rtol=0)


@pytest.mark.parametrize("b,s,hq,hkv,d,causal", [(2, 13, 4, 2, 8, True), (1, 11, 2, 2, 6, False),
                                                 (1, 16, 4, 1, 5, True)])
def test_backward_rows_vs_autograd(b, s, hq, hkv, d, causal):
    """The per-row gradient evaluation against float64 autograd, rows and heads spread out."""
    gen = torch.Generator().manual_seed(s + 100 * d)
    q = torch.randn(b, s, hq, d, generator=gen, dtype=torch.float64)
    k = torch.randn(b, s, hkv, d, generator=gen, dtype=torch.float64)
    v = torch.randn(b, s, hkv, d, generator=gen, dtype=torch.float64)
    do = torch.randn(b, s, hq, d, generator=gen, dtype=torch.float64)
    rq, rk, rv = _autograd(q, k, v, do, causal)
    qsm = [(bb, i, hh) for bb in range(b) for i in (0, s // 2, s - 1) for hh in (0, hq - 1)]
    ksm = [(bb, j, kh) for bb in range(b) for j in (0, s // 3, s - 1) for kh in range(hkv)]
    dq, dk, dv = oracle.attention_bwd_rows(q, k, v, do, causal, qsm, ksm)
    for n, (bb, i, hh) in enumerate(qsm):
        assert torch.allclose(dq[n], rq[bb, i, hh], atol=1e-11, rtol=0)
    for n, (bb, j, kh) in enumerate(ksm):
        assert torch.allclose(dk[n], rk[bb, j, kh], atol=1e-11, rtol=0)
        assert torch.allclose(dv[n], rv[bb, j, kh], atol=1e-11, rtol=0)


# ---------------------------------------------------------------- term magnitudes
# oracle.attention_bwd_magnitudes: per gradient element, the sum of the absolute values of
# its terms (dS_ij widened by P_ij E_i), the quantity a rounding-error bound scales with.

def _autograd_scores(q, k, v, do, causal):
    """P and dS = dL/dS of one head, from float64 autograd through softmax (a library
    routine); q, do [s, d], k, v [s, d]."""
    d = q.shape[-1]
    sc = (q.double() @ k.double().T / d ** 0.5).detach().requires_grad_()
    if causal:
        mask = torch.ones(sc.shape, dtype=torch.bool).tril()
        p = torch.softmax(sc.masked_fill(~mask, float("-inf")), dim=-1)
    else:
        p = torch.softmax(sc, dim=-1)
    o = p @ v.double()
    (o * do.double()).sum().backward()
    return p.detach(), sc.grad, o.detach()


@pytest.mark.parametrize("b,s,hq,hkv,d,causal", [(1, 9, 2, 2, 4, False), (2, 13, 4, 2, 8, True),
                                                 (1, 16, 4, 1, 5, True)])
def test_magnitudes_vs_autograd_scores(b, s, hq, hkv, d, causal):
    gen = torch.Generator().manual_seed(41 + s)
    q = torch.randn(b, s, hq, d, generator=gen, dtype=torch.float64)
    k = torch.randn(b, s, hkv, d, generator=gen, dtype=torch.float64)
    v = torch.randn(b, s, hkv, d, generator=gen, dtype=torch.float64)
    do = torch.randn(b, s, hq, d, generator=gen, dtype=torch.float64)
    mq, mk, mv = oracle.attention_bwd_magnitudes(q, k, v, do, causal)
    g = hq // hkv
    wk = torch.zeros_like(mk)
    wv = torch.zeros_like(mv)
    for bb in range(b):
        for hh in range(hq):
            kh = hh // g
            p, ds, o = _autograd_scores(q[bb, :, hh], k[bb, :, kh], v[bb, :, kh], do[bb, :, hh], causal)
            e = (do[bb, :, hh].abs() * (o.abs() + p @ v[bb, :, kh].abs())).sum(-1, keepdim=True)
            w = ds.abs() + p * e
            want_q = w @ k[bb, :, kh].abs() / d ** 0.5
            assert torch.allclose(mq[bb, :, hh], want_q, atol=1e-10, rtol=1e-10)
            wk[bb, :, kh] += w.T @ q[bb, :, hh].abs() / d ** 0.5
            wv[bb, :, kh] += p.T @ do[bb, :, hh].abs()
    assert torch.allclose(mk, wk, atol=1e-10, rtol=1e-10)
    assert torch.allclose(mv, wv, atol=1e-10, rtol=1e-10)


@pytest.mark.parametrize("causal", [False, True])
def test_magnitudes_bound_the_gradients(causal):
    """Triangle inequality: each magnitude is at least the gradient it belongs to."""
    gen = torch.Generator().manual_seed(5)
    b, s, hq, hkv, d = 2, 11, 4, 2, 6
    q, k, v = (torch.randn(b, s, h, d, generator=gen, dtype=torch.float64) for h in (hq, hkv, hkv))
    do = torch.randn(b, s, hq, d, generator=gen, dtype=torch.float64)
    dq, dk, dv = oracle.attention_bwd(q, k, v, do, causal)
    mq, mk, mv = oracle.attention_bwd_magnitudes(q, k, v, do, causal)
    for grad, mag in ((dq, mq), (dk, mk), (dv, mv)):
        assert (mag >= grad.abs() - 1e-12).all()


def test_magnitudes_closed_forms():
    gen = torch.Generator().manual_seed(9)
    d = 7
    # one token: P = 1, dS = dO.v - dO.O = 0, E = 2 sum_c |dO_c||v_c|
    q, k, v, do = (torch.randn(1, 1, 1, d, generator=gen, dtype=torch.float64) for _ in range(4))
    mq, mk, mv = oracle.attention_bwd_magnitudes(q, k, v, do, False)
    e = 2 * (do.abs() * v.abs()).sum()
    assert torch.allclose(mv, do.abs(), atol=1e-14)
    assert torch.allclose(mq, e * k.abs() / d ** 0.5, atol=1e-13)
    assert torch.allclose(mk, e * q.abs() / d ** 0.5, atol=1e-13)
    # non-negative dO: every dV term is non-negative, so the magnitude is dV itself
    s = 10
    q, k, v = (torch.randn(1, s, 2, d, generator=gen, dtype=torch.float64) for _ in range(3))
    do = torch.randn(1, s, 2, d, generator=gen, dtype=torch.float64).abs()
    for causal in (False, True):
        _, _, dv = oracle.attention_bwd(q, k, v, do, causal)
        _, _, mv = oracle.attention_bwd_magnitudes(q, k, v, do, causal)
        assert torch.allclose(mv, dv, atol=1e-12)
    # zero values: O = 0, dP = 0, so dS = 0 and E = 0
    mq, mk, _ = oracle.attention_bwd_magnitudes(q, k, torch.zeros_like(v), do, True)
    assert mq.abs().max().item() == 0.0 and mk.abs().max().item() == 0.0
