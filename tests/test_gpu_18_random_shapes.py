"""Seeded random shapes through the whole Ulysses forward and backward, against the oracle.

The fixed cases elsewhere pick shapes by hand; here a seeded generator draws them: rank
counts 1-8 including odd ones, ragged sequence tails, up to 16 query heads per K/V head (4
in the training cases), K/V heads split over the ranks or replicated on them (P a multiple
of h_kv), d in {64, 128}, both masks.  Every case compares the unfused forward with the
oracle's pipeline and, where the fused kernel takes the shape ((s/P) % 128 == 0), the fused
forward bit for bit with the unfused one; the training cases do the same for dQ, dK and dV
(with replicated K/V heads the two paths sum dK/dV in different orders, so there each is
checked against the oracle instead) ("DeepSpeed-Ulysses 深度解析", section "核心设计"
steps 3-5; "02 · DeepSpeed-Ulysses", section 5).  The later tests draw fp32, overlapped and
two-level cases the same way.  Sizes stay small enough for the oracle to finish each case
in a few seconds."""
import random

import pytest
import torch

import oracle
import sequence_attention_seq_gb300 as uly
from gpu_util import assert_close, assert_close_grad, bits_equal, device_ok, need_gpu
from sequence_attention_seq_gb300.inputs import global_grad, global_qkv, shard_seq

pytestmark = pytest.mark.gpu


def _draw(rng, max_tokens):
    """One shape: (P, b, s, hq, hkv, d, causal)."""
    P = rng.choice([1, 2, 3, 4, 6, 8])
    d = rng.choice([64, 128])
    b = rng.choice([1, 2])
    rep = [x for x in (1, 2, 4) if x < P and P % x == 0]
    if rep and rng.random() < 0.35:
        hkv = rng.choice(rep)              # replicated: each K/V head on P/h_kv ranks
        hq = P * rng.choice([1, 2])        # a multiple of P (and so of h_kv)
    else:
        hkv = P * rng.choice([1, 2])       # split over the ranks
        hq = hkv * rng.choice([1, 2, 4])
    if rng.random() < 0.35:
        S = 128 * rng.randint(1, max(1, max_tokens // (128 * P)))  # a shape the fused kernel takes
    else:
        S = rng.randint(1, max(1, max_tokens // P))                 # ragged
    return P, b, P * S, hq, hkv, d, rng.random() < 0.5


def _cases(seed, n, max_tokens, budget, max_group):
    rng = random.Random(seed)
    out = []
    while len(out) < n:
        P, b, s, hq, hkv, d, causal = _draw(rng, max_tokens)
        if hq // hkv > max_group or b * hq * s * s * d > budget:  # group size; oracle work
            continue
        out.append((P, b, s, hq, hkv, d, causal))
    return out


FWD = _cases(seed=2024, n=40, max_tokens=1024, budget=1 << 30, max_group=16)
# the gradient bound of assert_close_grad holds for at most 4 query heads per K/V head
BWD = _cases(seed=4048, n=16, max_tokens=768, budget=1 << 29, max_group=4)


def _want_fwd(q, k, v, qs, ks, vs, P, causal):
    """The oracle's exchange pipeline where the K/V heads split over the ranks; with
    replicated K/V heads (which the oracle's exchange does not take), its attention over the
    global tensors, which replicated Ulysses must equal (the two agree where both apply)."""
    if k.shape[2] % P == 0:
        return oracle.dist_attn_fwd(qs, ks, vs, causal)
    return shard_seq(oracle.attention(q, k, v, causal), P)


@pytest.mark.parametrize("P,b,s,hq,hkv,d,causal", FWD)
def test_random_forward(P, b, s, hq, hkv, d, causal):
    need_gpu()
    q, k, v = global_qkv(b, s, hq, hkv, d, torch.bfloat16, seed=s * 7 + hq + d)
    qs, ks, vs = shard_seq(q, P), shard_seq(k, P), shard_seq(v, P)
    qd, kd, vd = [t.cuda() for t in qs], [t.cuda() for t in ks], [t.cuda() for t in vs]
    unfused = uly.ulysses_dist_attn_fwd(qd, kd, vd, causal, fused=False)
    fused = uly.ulysses_dist_attn_fwd(qd, kd, vd, causal, fused=True) if (s // P) % 128 == 0 else None
    torch.cuda.synchronize()
    device_ok()
    want = _want_fwd(q, k, v, qs, ks, vs, P, causal)
    for j in range(P):
        assert_close(unfused[j], want[j], torch.bfloat16, f"rank {j}")
        if fused is not None:
            assert bits_equal(fused[j], unfused[j]), f"fused != unfused on rank {j}"


@pytest.mark.parametrize("P,b,s,hq,hkv,d,causal", BWD)
def test_random_backward(P, b, s, hq, hkv, d, causal):
    need_gpu()
    q, k, v = global_qkv(b, s, hq, hkv, d, torch.bfloat16, seed=s * 5 + hkv + d)
    do = global_grad(b, s, hq, d, torch.bfloat16, seed=s + 3)
    qs, ks, vs, dos = (shard_seq(x, P) for x in (q, k, v, do))
    qd, kd, vd, dod = ([t.cuda() for t in x] for x in (qs, ks, vs, dos))
    o, lse = uly.ulysses_dist_attn_fwd_lse(qd, kd, vd, causal)
    grads = uly.ulysses_dist_attn_bwd(qd, kd, vd, o, dod, lse, causal)
    fused = None
    if (s // P) % 128 == 0:
        fused = uly.ulysses_dist_attn_bwd(qd, kd, vd, o, dod, lse, causal, fused=True)
    torch.cuda.synchronize()
    device_ok()
    if hkv % P == 0:
        want = oracle.dist_attn_bwd(qs, ks, vs, dos, causal)
    else:  # replicated K/V heads: the gradients of attention over the global tensors
        want = [shard_seq(x, P) for x in oracle.attention_bwd(q, k, v, do, causal)]
    for name, got, ref, fz in zip(("dq", "dk", "dv"), grads, want, fused or (None,) * 3):
        for j in range(P):
            assert_close_grad(got[j], ref[j], f"{name} rank {j}")
            if fz is None:
                continue
            if hkv % P == 0 or name == "dq":
                assert bits_equal(fz[j], got[j]), f"fused {name} != unfused on rank {j}"
            else:  # replicated K/V heads: the two paths sum dK/dV in different orders
                assert_close_grad(fz[j], ref[j], f"fused {name} rank {j}")


def test_the_draw_covers_the_shape_classes():
    """The seeded draw reaches the classes it is meant to (needs no GPU)."""
    cases = FWD + BWD
    assert any(P in (3, 6) for P, *_ in cases)
    assert any((s // P) % 128 == 0 and P > 1 for P, _, s, *_ in cases)
    assert any((s // P) % 128 for P, _, s, *_ in cases)
    assert any(hkv < P for P, _, _, _, hkv, *_ in cases)
    assert any(hq > hkv for _, _, _, hq, hkv, *_ in cases)
    assert any(c for *_, c in cases) and any(not c for *_, c in cases)


def _fp32_cases(seed, n):
    rng = random.Random(seed)
    out = []
    while len(out) < n:
        P = rng.choice([1, 2, 3, 4])
        hkv = P * rng.choice([1, 2])
        hq = hkv * rng.choice([1, 2])
        d = 4 * rng.randint(1, 64)            # any multiple of 4 up to 256
        s = P * rng.randint(1, 160 // P)
        if hq * s * s * d <= 1 << 26:
            out.append((P, 1, s, hq, hkv, d, rng.random() < 0.5))
    return out


@pytest.mark.parametrize("P,b,s,hq,hkv,d,causal", _fp32_cases(seed=77, n=10))
def test_random_forward_fp32(P, b, s, hq, hkv, d, causal):
    """The fp32 path (any d that is a multiple of 4) against the oracle at 1e-5."""
    need_gpu()
    q, k, v = global_qkv(b, s, hq, hkv, d, torch.float32, seed=s + d)
    qs, ks, vs = shard_seq(q, P), shard_seq(k, P), shard_seq(v, P)
    out = uly.ulysses_dist_attn_fwd([t.cuda() for t in qs], [t.cuda() for t in ks], [t.cuda() for t in vs], causal)
    torch.cuda.synchronize()
    device_ok()
    want = oracle.dist_attn_fwd(qs, ks, vs, causal)
    for j in range(P):
        assert_close(out[j], want[j], torch.float32, f"rank {j}")


def _overlap_cases(seed, n):
    """Drawn FWD-style shapes with a valid head-group count for the overlapped forward."""
    rng = random.Random(seed)
    out = []
    for P, b, s, hq, hkv, d, causal in _cases(seed, 4 * n, 1024, 1 << 29, 16):
        Hq, Hk = hq // P, max(1, hkv // P)
        chunks = [c for c in (1, 2, 3, 4, 6, 8) if Hq % c == 0 and (Hk % c == 0 or c % Hk == 0)]
        if chunks:
            out.append((P, b, s, hq, hkv, d, causal, rng.choice(chunks)))
        if len(out) == n:
            break
    return out


@pytest.mark.parametrize("P,b,s,hq,hkv,d,causal,n_chunks", _overlap_cases(seed=91, n=10))
def test_random_overlap(P, b, s, hq, hkv, d, causal, n_chunks):
    """The overlapped forward gives the unfused forward's bits for every drawn shape."""
    need_gpu()
    q, k, v = global_qkv(b, s, hq, hkv, d, torch.bfloat16, seed=s + n_chunks)
    qd, kd, vd = ([t.cuda() for t in shard_seq(x, P)] for x in (q, k, v))
    over = uly.ulysses_dist_attn_fwd_overlap(qd, kd, vd, causal, n_chunks=n_chunks)
    plain = uly.ulysses_dist_attn_fwd(qd, kd, vd, causal, fused=False)
    torch.cuda.synchronize()
    device_ok()
    for j in range(P):
        assert bits_equal(over[j], plain[j]), f"rank {j}: overlapped != unfused"


def _usp_cases(seed, n):
    rng = random.Random(seed)
    out = []
    while len(out) < n:
        Pu, Pr = rng.choice([1, 2, 3, 4]), rng.choice([1, 2, 3, 4])
        P = Pu * Pr
        d = rng.choice([64, 128])
        if rng.random() < 0.3 and Pu > 1:
            hkv = rng.choice([x for x in (1, 2) if Pu % x == 0 and x < Pu] or [Pu])
            hq = Pu * rng.choice([1, 2])
        else:
            hkv = Pu * rng.choice([1, 2])
            hq = hkv * rng.choice([1, 2, 4])
        s = Pr * 128 * rng.randint(1, max(1, 768 // (128 * Pr)))  # (s/Pr) % 128 == 0
        if s % P or hq * s * s * d > 1 << 29 or hq // hkv > 4:
            continue
        out.append((Pu, Pr, 1, s, hq, hkv, d, rng.random() < 0.5))
    return out


@pytest.mark.parametrize("Pu,Pr,b,s,hq,hkv,d,causal", _usp_cases(seed=123, n=10))
def test_random_two_level(Pu, Pr, b, s, hq, hkv, d, causal):
    """The two-level forward and training path: forward against the oracle's explicit ring
    (or, with replicated K/V heads, its attention over the global tensors), bit for bit
    against plain Ulysses where that call takes the shape; gradients against the oracle."""
    need_gpu()
    P = Pu * Pr
    q, k, v = global_qkv(b, s, hq, hkv, d, torch.bfloat16, seed=s + 3 * Pu + Pr)
    do = global_grad(b, s, hq, d, torch.bfloat16, seed=s + 1)
    qs, ks, vs, dos = (shard_seq(x, P) for x in (q, k, v, do))
    qd, kd, vd, dod = ([t.cuda() for t in x] for x in (qs, ks, vs, dos))
    out = uly.ulysses_usp_attn_fwd(qd, kd, vd, causal, Pu, Pr)
    plain = uly.ulysses_dist_attn_fwd(qd, kd, vd, causal) if hq % P == 0 and hkv % P == 0 else None
    o, lse = uly.ulysses_usp_attn_fwd_lse(qd, kd, vd, causal, Pu, Pr)
    grads = uly.ulysses_usp_attn_bwd(qd, kd, vd, o, dod, lse, causal, Pu, Pr)
    torch.cuda.synchronize()
    device_ok()
    want = oracle.usp_fwd(qs, ks, vs, causal, Pu, Pr) if hkv % Pu == 0 else shard_seq(
        oracle.attention(q, k, v, causal), P)
    for j in range(P):
        assert_close(out[j], want[j], torch.bfloat16, f"rank {j}")
        assert bits_equal(o[j], out[j]), f"rank {j}: the forward with statistics changed the output"
        if plain is not None:
            assert bits_equal(out[j], plain[j]), f"rank {j}: two-level != plain Ulysses"
    ref = [shard_seq(x, P) for x in oracle.attention_bwd(q, k, v, do, causal)]
    for name, got, r in zip(("dq", "dk", "dv"), grads, ref):
        for j in range(P):
            assert_close_grad(got[j], r[j], f"{name} rank {j}")
