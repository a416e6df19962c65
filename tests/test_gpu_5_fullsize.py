"""The measured attention workloads at their full sizes, in the launch configuration the
benchmark times: sampled output rows against the oracle's per-row evaluation (exact per
row), and fused == unfused bit for bit over every output element.  Every query head is
sampled at least once; Long's causal items run in bands of one head each, and its samples
include every sampled head's first and last query tile (the last and the first item of
that head's band)."""
import random

import pytest
import torch

import oracle
import sequence_attention_seq_gb300 as uly
from gpu_util import assert_close, bits_equal, device_ok, need_gpu
from sequence_attention_seq_gb300.inputs import seq_shards_qkv

pytestmark = pytest.mark.gpu

CONFIGS = {
    # name: (P, b, s, hq, hkv, d, causal list, rows sampled)
    "dit_mha": (4, 2, 4096, 32, 32, 128, (False, True), 64),
    "gqa_causal": (8, 1, 32768, 32, 8, 128, (True,), 128),
    "long_causal": (8, 1, 131072, 64, 64, 128, (True,), 96),
}


def _samples(P, b, S, hq, n, seed):
    rng = random.Random(seed)
    picks = set()
    edges = [0, 1, 127, 128, S // 2, S - 129, S - 1]
    for h in range(hq):  # every head once, at a random token
        picks.add((rng.randrange(P), rng.randrange(b), rng.randrange(S), h))
    for h in rng.sample(range(hq), min(8, hq)):  # first and last query tile of some heads
        picks.add((0, rng.randrange(b), rng.randrange(128), h))
        picks.add((P - 1, rng.randrange(b), S - 1 - rng.randrange(128), h))
    while len(picks) < n:
        j = rng.randrange(P)
        t = rng.choice(edges) if rng.random() < 0.5 else rng.randrange(S)
        picks.add((j, rng.randrange(b), t, rng.randrange(hq)))
    return sorted(picks)


@pytest.mark.parametrize("name", list(CONFIGS))
def test_full_size_sampled_rows(name):
    need_gpu()
    P, b, s, hq, hkv, d, causals, nrows = CONFIGS[name]
    qd, kd, vd = seq_shards_qkv(P, b, s, hq, hkv, d, torch.bfloat16, seed=0, device="cuda")
    qc, kc, vc = [t.cpu() for t in qd], [t.cpu() for t in kd], [t.cpu() for t in vd]
    samples = _samples(P, b, s // P, hq, nrows, seed=len(name))
    for causal in causals:
        fused = uly.ulysses_dist_attn_fwd(qd, kd, vd, causal, fused=True)
        unfused = uly.ulysses_dist_attn_fwd(qd, kd, vd, causal, fused=False)
        torch.cuda.synchronize()
        device_ok()
        for j in range(P):
            assert bits_equal(fused[j], unfused[j]), f"{name}: fused != unfused on rank {j}"
        want = oracle.dist_attn_rows(qc, kc, vc, causal, samples)
        got = torch.stack([fused[j][bb, t, gh] for (j, bb, t, gh) in samples])
        assert_close(got, want, torch.bfloat16, f"{name} causal={causal}")
        del fused, unfused
