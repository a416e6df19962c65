"""The forward kernel's persistent paths, against the oracle.

(1) Several work items per CTA.  The forward launches min(items, SMs) CTAs, and each walks
    its items in snake order, continuing its barrier phases, loading the next item's Q as
    soon as the last S product has read the current one, and handing O back to the MMA
    warp after the epilogue.  With more than two items per SM every CTA runs at least
    two items; the whole output is compared with the oracle element by element, fused and
    unfused, both masks, grouped heads (4 query heads per K/V head).
(2) Several causal bands.  When the K and V of all (rank, batch, K/V head) units exceed
    L2, causal items run in bands of units (heaviest first inside a band).  At s = 16384
    with 32 heads of d = 128 every unit holds 8 MiB of K and V, so the 32 units form six
    bands; sampled rows cover the first and last unit of every band, the first and last
    query tile, diagonal tiles and the rank boundary.

Causal rule: "长上下文训练中的 SP 与 CP", Ring Attention section, causal paragraph (key j
visible iff j <= i); the pipeline: "DeepSpeed-Ulysses 深度解析", steps 3-5."""
import random

import pytest
import torch

import oracle
import sequence_attention_seq_gb300 as uly
from gpu_util import assert_close, bits_equal, device_ok, need_gpu
from sequence_attention_seq_gb300.inputs import seq_shards_qkv

pytestmark = pytest.mark.gpu


def _sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_forward_many_items_per_cta(d, causal):
    need_gpu()
    P, b, s, hq, hkv = 4, 4, 512, 48, 12
    n_pairs = (s // 128 + 1) // 2
    assert b * hq * n_pairs > 2 * _sms()  # every CTA runs at least two items
    qs, ks, vs = seq_shards_qkv(P, b, s, hq, hkv, d, torch.bfloat16, seed=100 + d + int(causal))
    qd, kd, vd = [t.cuda() for t in qs], [t.cuda() for t in ks], [t.cuda() for t in vs]
    unfused = uly.ulysses_dist_attn_fwd(qd, kd, vd, causal, fused=False)
    fused = uly.ulysses_dist_attn_fwd(qd, kd, vd, causal, fused=True)
    torch.cuda.synchronize()
    device_ok()
    want = oracle.dist_attn_fwd(qs, ks, vs, causal)
    for j in range(P):
        assert_close(unfused[j], want[j], torch.bfloat16, f"unfused rank {j}")
        assert bits_equal(fused[j], unfused[j]), f"fused != unfused on rank {j}"


def _band_samples(P, S, heads, band_units, n_random, seed):
    s = P * S
    rng = random.Random(seed)
    edges = sorted({h for base in range(0, heads, band_units) for h in (base, min(base + band_units, heads) - 1)})
    tokens = [0, 1, 127, 128, S - 1, S, s - 128, s - 1]  # first/last query tile, rank boundary
    picks = set()
    for h in edges:
        for tok in tokens:
            picks.add((tok // S, 0, tok % S, h))
        k = rng.randrange(1, s // 128)
        for tok in (128 * k, 128 * k + 127):  # a diagonal tile's first and last row
            picks.add((tok // S, 0, tok % S, h))
    while len(picks) < len(edges) * 10 + n_random:
        tok = rng.randrange(s)
        picks.add((tok // S, 0, tok % S, rng.randrange(heads)))
    return sorted(picks), edges


def test_forward_causal_bands():
    need_gpu()
    P, b, s, hq, hkv, d = 2, 1, 16384, 32, 32, 128
    unit_kv = 2 * s * d * 2
    assert unit_kv * b * hkv > 129 * 2 ** 20  # the units' K/V exceed L2: several bands
    band_units = (48 * 2 ** 20) // unit_kv  # the kernel's band size at this shape
    qd, kd, vd = seq_shards_qkv(P, b, s, hq, hkv, d, torch.bfloat16, seed=7, device="cuda")
    fused = uly.ulysses_dist_attn_fwd(qd, kd, vd, True, fused=True)
    unfused = uly.ulysses_dist_attn_fwd(qd, kd, vd, True, fused=False)
    torch.cuda.synchronize()
    device_ok()
    for j in range(P):
        assert bits_equal(fused[j], unfused[j]), f"fused != unfused on rank {j}"
    samples, edges = _band_samples(P, s // P, hq, band_units, 140, seed=11)
    assert len(samples) >= 256 and len(edges) >= 10
    qc, kc, vc = [t.cpu() for t in qd], [t.cpu() for t in kd], [t.cpu() for t in vd]
    want = oracle.dist_attn_rows(qc, kc, vc, True, samples)
    got = torch.stack([fused[j][bb, t, gh] for (j, bb, t, gh) in samples])
    assert_close(got, want, torch.bfloat16, "banded causal rows")
