"""Pins for the CPU oracle: the oracle is checked against what the pages and the
mathematics fix, never against itself or against the CUDA library.

* all-to-all: the printed two-rank AllToAll example, the two-rank block example, the
  4-rank/16-token/8-head shape example, the communication-volume table, the global-view
  definition of the exchange, round-trip identities and P=1;
* attention: a library routine (PyTorch float64 scaled_dot_product_attention) on the
  global tensors, closed forms (s=1, Q=0, constant V, first causal row), invariances
  (key shift, causality) and the per-row evaluation against the full pipeline.
"""
import json
import os

import pytest
import torch
import torch.nn.functional as F

import oracle
from sequence_attention_seq_gb300.inputs import global_qkv, random_bits, shard_seq


def _load(golden_dir, name):
    with open(os.path.join(golden_dir, name)) as f:
        return json.load(f)


# ----------------------------------------------------------------------------- all-to-all

def test_alltoall_two_rank_example(golden_dir):
    g = _load(golden_dir, "alltoall_two_rank.json")
    labels = sorted({x for row in g["before"].values() for x in row})
    code = {lab: n + 1 for n, lab in enumerate(labels)}
    chunk = lambda lab: torch.full((3,), code[lab], dtype=torch.int32)  # noqa: E731
    before = [[chunk(x) for x in g["before"][f"rank{i}"]] for i in range(2)]
    after = oracle.all_to_all(before)
    for j in range(2):
        got = [int(c[0]) for c in after[j]]
        assert got == [code[x] for x in g["after"][f"rank{j}"]]


def _block_tagged(P, b, s, h, d):
    """Global tensor whose element value encodes (token segment i, head group j, unique id)."""
    S, H = s // P, h // P
    idx = torch.arange(b * s * h * d, dtype=torch.int64).reshape(b, s, h, d)
    seg = (torch.arange(s) // S).view(1, s, 1, 1)
    grp = (torch.arange(h) // H).view(1, 1, h, 1)
    return (seg * 1_000_000 + grp * 100_000 + idx).to(torch.int64)


def test_rank0_block_two_rank_example(golden_dir):
    g = _load(golden_dir, "rank0_block_two_rank.json")
    P, b, s, h, d = g["P"], 1, 6, 4, 3
    S, H = s // P, h // P
    X = _block_tagged(P, b, s, h, d)
    out = oracle.seq2head(shard_seq(X, P))
    r0 = out[0]
    seg = r0 // 1_000_000
    grp = (r0 // 100_000) % 10
    # rank 0 holds [X_{0,0}; X_{1,0}] along the sequence axis
    for n, (i, j) in enumerate(g["rank0_after_seq_order"]):
        blk = slice(n * S, (n + 1) * S)
        assert torch.all(seg[:, blk] == i) and torch.all(grp[:, blk] == j)
    keep_i, keep_j = g["rank0_keeps"]
    assert torch.equal(r0[:, :S], X[:, keep_i * S:(keep_i + 1) * S, keep_j * H:(keep_j + 1) * H])
    recv_i, recv_j = g["rank0_receives"]
    assert torch.equal(r0[:, S:], X[:, recv_i * S:(recv_i + 1) * S, recv_j * H:(recv_j + 1) * H])
    # X_{0,1} left rank 0: it sits at the front of rank 1's output
    si, sj = g["rank0_sends"]
    assert torch.equal(out[1][:, :S], X[:, si * S:(si + 1) * S, sj * H:(sj + 1) * H])


def test_shape_example_4x16x8(golden_dir):
    g = _load(golden_dir, "shape_example_4x16x8.json")
    P, s, h, d_h = g["P"], g["tokens"], g["heads"], 5
    x = random_bits((1, s, h, d_h), torch.bfloat16, seed=3)
    shards = shard_seq(x, P)
    assert list(shards[0].shape[1:3]) == g["per_rank_before"]
    out = oracle.seq2head(shards)
    for o, sh in zip(out, shards):
        assert list(o.shape[1:3]) == g["per_rank_after"]
        assert o.numel() == sh.numel() == g["elements_per_rank_in_units_of_d_h"] * d_h


@pytest.mark.parametrize("P,b,s,h,d", [(2, 1, 8, 4, 3), (4, 2, 16, 8, 2), (8, 1, 64, 16, 4), (3, 2, 9, 6, 5)])
def test_seq2head_matches_global_view(P, b, s, h, d):
    """Rank r ends with head group r of the whole sequence (page 02 · DeepSpeed-Ulysses,
    section 2: every card holds all tokens of heads/cp heads), in global token order."""
    x = random_bits((b, s, h, d), torch.bfloat16, seed=P * 100 + s)
    out = oracle.seq2head(shard_seq(x, P))
    H = h // P
    for r in range(P):
        assert torch.equal(out[r].view(torch.int16), x[:, :, r * H:(r + 1) * H].contiguous().view(torch.int16))


@pytest.mark.parametrize("P,b,s,h,d,dtype", [
    (1, 1, 4, 2, 3, torch.bfloat16), (2, 1, 64, 4, 16, torch.float32), (4, 2, 32, 8, 8, torch.bfloat16),
    (8, 1, 64, 64, 4, torch.bfloat16), (16, 1, 32, 16, 2, torch.float32), (5, 3, 15, 10, 7, torch.bfloat16)])
def test_round_trips_are_identity(P, b, s, h, d, dtype):
    x = random_bits((b, s, h, d), dtype, seed=7 + P)
    shards = shard_seq(x, P)
    back = oracle.head2seq(oracle.seq2head(shards))
    for a, c in zip(shards, back):
        assert a.shape == c.shape and a.view(torch.uint8).equal(c.view(torch.uint8))
    y = [random_bits((b, s, h // P, d), dtype, seed=50 + r) for r in range(P)]
    again = oracle.seq2head(oracle.head2seq(y))
    for a, c in zip(y, again):
        assert a.view(torch.uint8).equal(c.view(torch.uint8))


def test_p1_is_identity():
    x = random_bits((2, 8, 4, 3), torch.bfloat16, seed=11)
    assert oracle.seq2head([x])[0].view(torch.int16).equal(x.view(torch.int16))
    assert oracle.head2seq([x])[0].view(torch.int16).equal(x.view(torch.int16))


def _foreign_elements(P, b, s, h, d):
    """Elements that each rank holds after all-to-all #1 but did not hold before."""
    S = s // P
    tagged = [torch.full((b, S, h, d), j, dtype=torch.int16) for j in range(P)]
    out = oracle.seq2head(tagged)
    return [int((o != r).sum()) for r, o in enumerate(out)], [o.numel() for o in out]


@pytest.mark.parametrize("P,b,s,h,d", [(2, 1, 8, 4, 2), (4, 2, 16, 8, 3), (8, 1, 64, 16, 2)])
def test_volume_per_rank(P, b, s, h, d):
    """Per-rank elements crossing ranks = (P-1) N h d / P^2 and element count is preserved
    ("Ulysses vs Ring Attention", section 2; "02 · DeepSpeed-Ulysses", section 3)."""
    foreign, counts = _foreign_elements(P, b, s, h, d)
    assert all(c == b * s * h * d // P for c in counts)
    assert all(f * P * P == (P - 1) * b * s * h * d for f in foreign)
    # page 1's form: (s/cp) * heads * d * (cp-1)/cp
    assert all(f * P == b * (s // P) * h * d * (P - 1) for f in foreign)


def test_volume_table_entries(golden_dir):
    g = _load(golden_dir, "volume_table.json")
    h, d = g["h"], g["d"]
    for P_str, per_tok in g["per_tensor_per_token"].items():
        P = int(P_str)
        s = 2 * P
        foreign, _ = _foreign_elements(P, 1, s, h, d)
        assert all(f == per_tok * s for f in foreign)
    for P_str, per_tok in g["four_tensors_per_token"].items():
        P = int(P_str)
        s = 2 * P
        foreign, _ = _foreign_elements(P, 1, s, h, d)
        # Q, K, V through exchange #1 and O back through exchange #2 move equal volumes
        o_head = [torch.full((1, s, h // P, d), r, dtype=torch.int16) for r in range(P)]
        back = oracle.head2seq(o_head)
        foreign_o = [int((o != j).sum()) for j, o in enumerate(back)]
        assert all(3 * f + fo == per_tok * s for f, fo in zip(foreign, foreign_o))


# ----------------------------------------------------------------------------- attention

def _sdpa_global(q, k, v, causal):
    """Library routine on global [b, s, h, d] float64 tensors; K/V heads repeated so that
    query head i reads K/V head i // (h_q / h_kv)."""
    g = q.shape[2] // k.shape[2]
    qq = q.double().permute(0, 2, 1, 3)
    kk = k.double().repeat_interleave(g, dim=2).permute(0, 2, 1, 3)
    vv = v.double().repeat_interleave(g, dim=2).permute(0, 2, 1, 3)
    o = F.scaled_dot_product_attention(qq, kk, vv, is_causal=causal)
    return o.permute(0, 2, 1, 3).contiguous()


@pytest.mark.parametrize("b,s,hq,hkv,d,causal", [
    (1, 17, 2, 2, 8, False), (2, 33, 4, 2, 16, True), (1, 40, 8, 1, 4, True), (2, 9, 3, 3, 5, False)])
def test_local_attention_vs_library(b, s, hq, hkv, d, causal):
    g = torch.Generator().manual_seed(s * 31 + d)
    q = torch.randn(b, s, hq, d, generator=g, dtype=torch.float64)
    k = torch.randn(b, s, hkv, d, generator=g, dtype=torch.float64)
    v = torch.randn(b, s, hkv, d, generator=g, dtype=torch.float64)
    got = oracle.attention(q, k, v, causal)
    assert torch.allclose(got, _sdpa_global(q, k, v, causal), atol=1e-12, rtol=0)


@pytest.mark.parametrize("P,b,s,hq,hkv,d,causal,dtype", [
    (2, 1, 64, 4, 4, 16, False, torch.float32),
    (2, 1, 64, 4, 4, 16, True, torch.float32),
    (4, 2, 32, 8, 4, 8, True, torch.bfloat16),
    (4, 1, 48, 8, 8, 4, False, torch.bfloat16),
    (8, 1, 64, 16, 8, 4, True, torch.bfloat16),
    (2, 1, 32, 8, 4, 8, True, torch.bfloat16)])
def test_ulysses_equals_single_device_attention(P, b, s, hq, hkv, d, causal, dtype):
    """Heads are independent, so the three exchanges plus per-rank attention equal plain
    attention over the whole sequence ("02 · DeepSpeed-Ulysses", section 1)."""
    q, k, v = global_qkv(b, s, hq, hkv, d, dtype, seed=P + s)
    out = oracle.dist_attn_fwd(shard_seq(q, P), shard_seq(k, P), shard_seq(v, P), causal)
    ref = _sdpa_global(q, k, v, causal)
    assert torch.allclose(torch.cat(out, dim=1), ref, atol=1e-12, rtol=0)


def test_single_token_returns_v():
    g = torch.Generator().manual_seed(1)
    q, k, v = (torch.randn(1, 1, 2, 6, generator=g, dtype=torch.float64) for _ in range(3))
    for causal in (False, True):
        assert torch.equal(oracle.attention(q, k, v, causal), v)


def test_zero_query_gives_mean_and_prefix_mean():
    g = torch.Generator().manual_seed(2)
    s, d = 12, 5
    q = torch.zeros(1, s, 1, d, dtype=torch.float64)
    k = torch.randn(1, s, 1, d, generator=g, dtype=torch.float64)
    v = torch.randn(1, s, 1, d, generator=g, dtype=torch.float64)
    full = oracle.attention(q, k, v, False)
    assert torch.allclose(full[0, :, 0], v[0, :, 0].mean(0).expand(s, d), atol=1e-14, rtol=0)
    causal = oracle.attention(q, k, v, True)
    prefix = torch.cumsum(v[0, :, 0], 0) / torch.arange(1, s + 1, dtype=torch.float64).unsqueeze(1)
    assert torch.allclose(causal[0, :, 0], prefix, atol=1e-14, rtol=0)


def test_constant_values_and_first_causal_row():
    g = torch.Generator().manual_seed(3)
    q, k = (torch.randn(1, 10, 2, 4, generator=g, dtype=torch.float64) for _ in range(2))
    c = torch.tensor([0.5, -2.0, 3.25, 1.0], dtype=torch.float64)
    v = c.expand(1, 10, 2, 4).contiguous()
    assert torch.allclose(oracle.attention(q, k, v, False), v, atol=1e-14, rtol=0)
    v2 = torch.randn(1, 10, 2, 4, generator=g, dtype=torch.float64)
    out = oracle.attention(q, k, v2, True)
    assert torch.equal(out[:, 0], v2[:, 0])


def test_key_shift_invariance_and_causality():
    g = torch.Generator().manual_seed(4)
    q, k, v = (torch.randn(1, 16, 2, 8, generator=g, dtype=torch.float64) for _ in range(3))
    u = torch.randn(1, 1, 2, 8, generator=g, dtype=torch.float64)
    for causal in (False, True):
        a = oracle.attention(q, k, v, causal)
        b = oracle.attention(q, k + u, v, causal)
        assert torch.allclose(a, b, atol=1e-12, rtol=0)
    base = oracle.attention(q, k, v, True)
    k2, v2 = k.clone(), v.clone()
    k2[:, 9:] += 5.0
    v2[:, 9:] -= 3.0
    pert = oracle.attention(q, k2, v2, True)
    assert torch.equal(base[:, :9], pert[:, :9])
    assert not torch.allclose(base[:, 9:], pert[:, 9:])


@pytest.mark.parametrize("P,b,s,hq,hkv,d,causal", [(4, 2, 32, 8, 4, 8, True), (2, 1, 24, 4, 2, 6, False)])
def test_row_evaluation_matches_pipeline(P, b, s, hq, hkv, d, causal):
    q, k, v = global_qkv(b, s, hq, hkv, d, torch.bfloat16, seed=9)
    qs, ks, vs = shard_seq(q, P), shard_seq(k, P), shard_seq(v, P)
    full = oracle.dist_attn_fwd(qs, ks, vs, causal)
    S = s // P
    samples = [(j, bb, t, gh) for j in range(P) for bb in range(b) for t in (0, S - 1) for gh in (0, hq - 1, hq // 2)]
    rows = oracle.dist_attn_rows(qs, ks, vs, causal, samples)
    for n, (j, bb, t, gh) in enumerate(samples):
        assert torch.allclose(rows[n], full[j][bb, t, gh], atol=1e-14, rtol=0)
